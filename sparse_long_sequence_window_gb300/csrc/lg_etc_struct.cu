// ETC global-local attention with relative-position labels and per-instance
// masks, on the 5th-generation tensor cores: "ETC: Encoding Long and
// Structured Inputs in Transformers", section 3.4, "Relative Position
// Encoding" (a learnable vector a^K_l per relation label and head, added to
// the key; the appendix's trick of computing q_i . a^K_l for every label once
// and gathering one scalar per edge) and "Global-Local Attention" (the four
// pieces' logits e_ij = q_i (k_j + a^K_ij)^T / sqrt(d) - (1 - M_ij) C with
// C = 10000, the l2l piece only for |i - j| <= r clamped to valid indices,
// one softmax over g2g + g2l for a global query and one over l2g + l2l for a
// long query; per-instance binary masks M).
//
// Each edge carries one code byte: the label in bits 0..6 and 1 - M_ij in
// bit 7.  Three kernels:
//  * es_pack_kernel lays the caller's four code arrays out as one 128 x 128
//    byte block per (query tile, key tile) in the order the attention kernel
//    visits them (rows of 128 bytes, 16-byte chunks XOR-swizzled by the row,
//    so that the softmax threads read them from shared memory without bank
//    conflicts), and checks the labels against the vocabulary;
//  * es_qa_kernel computes qa_il = s log2(e) q_i . a^K_l for every query row
//    and label, stored label-major per 128-row tile (qa[l][row]), so that a
//    softmax thread gathers its row's value of any label conflict-free;
//  * es_attn_kernel: one CTA per (instance, head, 128-row query tile) with
//    warp 0 loading tiles (TMA for q, k, v; bulk copies for the code blocks
//    and qa), warp 1 owning tensor memory and issuing the MMAs from one lane,
//    and warps 4..7 the softmax (one thread per row).  S = Q K^T lands in one
//    of two TMEM buffers, so the QK of tile j + 2 is issued right after the PV
//    of tile j and runs while the softmax works on tile j + 1; the softmax adds
//    qa[label], applies the blocked edges' -C (exactly, see the softmax),
//    keeps a running maximum (O rescaled in TMEM only when it grows by more
//    than 2^8), writes P (bf16) over its S and the MMA warp accumulates
//    O += P V with P read from TMEM.
// Long query tiles visit the band key tiles [t0 - r, t0 + 127 + r] and then
// the global key tiles; global query tiles the global key tiles and then every
// long key tile.  Global query tiles come first in the grid (they are the
// long units).
#include <math.h>

#include <algorithm>
#include <mutex>

#include "lg_internal.h"
#include "lg_ptx.cuh"

namespace lg {
namespace {

constexpr int kEsThreads = 256;
constexpr int kEsMaxDevices = 64;
constexpr int kEsMaxLabels = 64;
constexpr int kCodeTile = 128 * 128;                // bytes of one (query tile, key tile) code block
constexpr long long kEsDrainCap = 4000000000LL;     // fixed bound of waits for already-issued async work
constexpr float kEsMaskC = 10000.f;

struct EsGeom {
  int B, H, L, G, r;
  int n_lq, n_gq;          // long / global query tiles (= long / global key tiles)
  int band_max;            // most band key tiles of a long query tile
  int steps_l, steps_g;    // key tiles of a long / global query tile (the code-block stride)
  long long blocks_per_b;  // code blocks of one instance
};

// Band key tiles of long query tile tq: first key band_lo, n_band tiles.
__host__ __device__ inline void es_band(int L, int r, int tq, int& band_lo, int& n_band) {
  const int t0 = tq * 128;
  const int last = t0 + 127 < L - 1 ? t0 + 127 : L - 1;
  band_lo = t0 - r > 0 ? t0 - r : 0;
  const int band_hi = last + r < L - 1 ? last + r : L - 1;
  n_band = (band_hi - band_lo) / 128 + 1;
}

EsGeom es_geom(int B, int H, int L, int G, int r) {
  EsGeom g{};
  g.B = B; g.H = H; g.L = L; g.G = G; g.r = r;
  g.n_lq = (L + 127) / 128;
  g.n_gq = (G + 127) / 128;
  g.band_max = 0;
  for (int tq = 0; tq < g.n_lq; ++tq) {
    int lo, nb;
    es_band(L, r, tq, lo, nb);
    g.band_max = std::max(g.band_max, nb);
  }
  g.steps_l = g.band_max + g.n_gq;
  g.steps_g = g.n_gq + g.n_lq;
  g.blocks_per_b = static_cast<long long>(g.n_gq) * g.steps_g + static_cast<long long>(g.n_lq) * g.steps_l;
  return g;
}

// First code block of a query tile of instance b.
__host__ __device__ inline long long es_block(const EsGeom& g, int b, bool glob, int tq) {
  return static_cast<long long>(b) * g.blocks_per_b +
         (glob ? static_cast<long long>(tq) * g.steps_g
               : static_cast<long long>(g.n_gq) * g.steps_g + static_cast<long long>(tq) * g.steps_l);
}

// ---------------------------------------------------------------- code blocks

struct EsPackParams {
  EsGeom g;
  const uint8_t* l2l;   // [B, L, 2r + 1] or NULL
  const uint8_t* l2g;   // [B, L, G] or NULL
  const uint8_t* g2l;   // [B, G, L] or NULL
  const uint8_t* g2g;   // [B, G, G] or NULL
  uint8_t* codes;
  int n_labels;         // labels are checked against it when > 0
  int* status;
};

// One thread per 16-byte chunk of a block (16 edges of one row).
__global__ void __launch_bounds__(256) es_pack_kernel(const EsPackParams p) {
  const EsGeom& g = p.g;
  const long long total = static_cast<long long>(g.B) * g.blocks_per_b * (kCodeTile / 16);
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int chunk = static_cast<int>(idx % (kCodeTile / 16));
    const long long blk = idx / (kCodeTile / 16);
    const int b = static_cast<int>(blk / g.blocks_per_b);
    long long rem = blk % g.blocks_per_b;
    const int row = chunk >> 3;
    const int k = (chunk & 7) ^ (row & 7);   // logical 16-column group stored in this physical chunk
    const bool glob = rem < static_cast<long long>(g.n_gq) * g.steps_g;
    int tq, j;
    if (glob) {
      tq = static_cast<int>(rem / g.steps_g); j = static_cast<int>(rem % g.steps_g);
    } else {
      rem -= static_cast<long long>(g.n_gq) * g.steps_g;
      tq = static_cast<int>(rem / g.steps_l); j = static_cast<int>(rem % g.steps_l);
    }
    // piece: 0 none, 1 l2l, 2 l2g, 3 g2l, 4 g2g; key0: first key of the tile
    int piece = 0, key0 = 0, key_n = 0;
    const int qi = tq * 128 + row;
    if (glob) {
      if (qi < g.G) {
        if (j < g.n_gq) { piece = 4; key0 = j * 128; key_n = g.G; }
        else { piece = 3; key0 = (j - g.n_gq) * 128; key_n = g.L; }
      }
    } else if (qi < g.L) {
      int band_lo, n_band;
      es_band(g.L, g.r, tq, band_lo, n_band);
      if (j < n_band) { piece = 1; key0 = band_lo + j * 128; key_n = g.L; }
      else if (j - n_band < g.n_gq) { piece = 2; key0 = (j - n_band) * 128; key_n = g.G; }
    }
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    bool bad = false;
    if (piece != 0) {
      const uint8_t* src = piece == 1 ? p.l2l : piece == 2 ? p.l2g : piece == 3 ? p.g2l : p.g2g;
      for (int e = 0; e < 16; ++e) {
        const int kj = key0 + 16 * k + e;
        if (kj >= key_n) continue;
        uint32_t c = 0;
        if (piece == 1) {
          const int t = kj - qi;
          if (t < -g.r || t > g.r) continue;   // outside the band: not an edge
          if (src) c = src[(static_cast<size_t>(b) * g.L + qi) * (2 * g.r + 1) + (t + g.r)];
        } else if (src) {
          const size_t rows = piece == 2 ? g.L : g.G, cols = piece == 2 ? g.G : (piece == 3 ? g.L : g.G);
          c = src[(static_cast<size_t>(b) * rows + qi) * cols + kj];
        }
        if (p.n_labels > 0 && static_cast<int>(c & 127u) >= p.n_labels) bad = true;
        w[e >> 2] |= c << (8 * (e & 3));
      }
    }
    if (bad) atomicOr(p.status, ST_BAD_CODE);
    reinterpret_cast<uint4*>(p.codes)[idx] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------- qa = s log2(e) q . a^K_l

struct EsQaParams {
  const __nv_bfloat16* q_l;   // [BH, L, D]
  const __nv_bfloat16* q_g;   // [BH, G, D]
  const __nv_bfloat16* rel;   // [H, V, D]
  float* qa;                  // [BH][n_gq + n_lq][V][128]
  int H, L, G, D, V, n_gq, n_lq;
  long long total;            // BH * (n_gq + n_lq) * V * 128
  float c;
};

__global__ void __launch_bounds__(256) es_qa_kernel(const EsQaParams p) {
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < p.total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(idx & 127);
    long long t = idx >> 7;
    const int l = static_cast<int>(t % p.V); t /= p.V;
    const int tile = static_cast<int>(t % (p.n_gq + p.n_lq));
    const long long bh = t / (p.n_gq + p.n_lq);
    const bool glob = tile < p.n_gq;
    const int row = (glob ? tile : tile - p.n_gq) * 128 + r;
    float acc = 0.f;
    if (row < (glob ? p.G : p.L)) {
      const uint4* q = reinterpret_cast<const uint4*>(glob ? p.q_g + (bh * p.G + row) * p.D : p.q_l + (bh * p.L + row) * p.D);
      const uint4* a = reinterpret_cast<const uint4*>(p.rel + (static_cast<size_t>(bh % p.H) * p.V + l) * p.D);
      for (int x = 0; x < p.D / 8; ++x) {
        const uint4 qv = __ldg(q + x), av = __ldg(a + x);
        const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[e]));
          const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
          acc = fmaf(qf.x, af.x, acc);
          acc = fmaf(qf.y, af.y, acc);
        }
      }
    }
    p.qa[idx] = acc * p.c;
  }
}

// ---------------------------------------------------------------- attention

struct EsParams {
  CUtensorMap mQl, mKl, mVl, mQg, mKg, mVg;   // {D, rows, BH}, 128-row boxes
  CUtensorMap sOl, sOg;                       // output stores, 32-row boxes
  EsGeom g;
  const uint8_t* codes;
  const float* qa;
  float* lse_l;
  float* lse_g;
  int* status;
  long long wait_cap;
  int withhold;
  int V;
  float scale_log2;
};

template <int D>
struct EsCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kStage = 2 * kTile + kCodeTile;   // K, V, code block
  static constexpr int kOffStage = kTile;                // after Q
  static constexpr int kOffQa = kTile + 2 * kStage;
  static constexpr int kOffMisc = kOffQa + kEsMaxLabels * 512;
  static constexpr int kSmem = kOffMisc + 256 + 1024;    // + alignment slack
};

template <int D>
__device__ __forceinline__ void es_load_tile(const CUtensorMap* map, int y0, int bh, uint32_t dst, uint32_t bar) {
#pragma unroll
  for (int blk = 0; blk < D / 64; ++blk) tma_load_3d(dst + blk * (128 * 128), map, bar, blk * 64, y0, bh);
}

template <int D, bool BIAS>
__global__ void __launch_bounds__(kEsThreads, 1) es_attn_kernel(const __grid_constant__ EsParams p) {
  using C = EsCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t sQ = sb, sQa = sb + C::kOffQa;
  auto stage = [&](int st) { return sb + C::kOffStage + st * C::kStage; };
  unsigned char* misc = smem + C::kOffMisc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  enum { B_QF = 0, B_KVF = 1, B_KVE = 3, B_SF = 5, B_PF = 7, B_PV = 9, B_DONE = 10, NB = 11 };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 132);
  auto bar = [&](int i) { return smem_addr(&bars[i]); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) mbar_init(bar(i), (i == B_PF || i == B_PF + 1) ? 128 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();
  const long long cap = p.wait_cap;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.status, ST_TIMEOUT);
  };

  // ---- the unit: (instance, head, query tile); global query tiles first
  const EsGeom& g = p.g;
  const int BH = g.B * g.H;
  const int u = blockIdx.x;
  const bool glob = u < BH * g.n_gq;
  const int bh = glob ? u / g.n_gq : (u - BH * g.n_gq) / g.n_lq;
  const int tq = glob ? u % g.n_gq : (u - BH * g.n_gq) % g.n_lq;
  const int b = bh / g.H;
  int band_lo = 0, n_band = 0;
  if (!glob) es_band(g.L, g.r, tq, band_lo, n_band);
  const int n_steps = glob ? g.steps_g : n_band + g.n_gq;
  const uint8_t* codes = p.codes + es_block(g, b, glob, tq) * kCodeTile;
  constexpr uint32_t kTS = 0, kTO = 256;   // S buffers at columns 0 and 128, O at 256

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0 && !p.withhold) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar(B_QF), C::kTile + (BIAS ? p.V * 512 : 0));
      es_load_tile<D>(glob ? &p.mQg : &p.mQl, tq * 128, bh, sQ, bar(B_QF));
      if (BIAS) {
        const float* qa = p.qa + (static_cast<size_t>(bh) * (g.n_gq + g.n_lq) + (glob ? tq : g.n_gq + tq)) * p.V * 128;
        bulk_load_1d(sQa, qa, p.V * 512, bar(B_QF));
      }
      for (int j = 0; j < n_steps; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(bar(B_KVE + st), ((j >> 1) - 1) & 1, abort_flag, cap)) { fail(); ok = false; break; }
        bool kglob;
        int y;
        if (glob) { kglob = j < g.n_gq; y = kglob ? j * 128 : (j - g.n_gq) * 128; }
        else { kglob = j >= n_band; y = kglob ? (j - n_band) * 128 : band_lo + j * 128; }
        const uint32_t dst = stage(st);
        mbar_arrive_expect_tx(bar(B_KVF + st), C::kStage);
        es_load_tile<D>(kglob ? &p.mKg : &p.mKl, y, bh, dst, bar(B_KVF + st));
        es_load_tile<D>(kglob ? &p.mVg : &p.mVl, y, bh, dst + C::kTile, bar(B_KVF + st));
        bulk_load_1d(dst + 2 * C::kTile, codes + static_cast<size_t>(j) * kCodeTile, kCodeTile, bar(B_KVF + st));
        issued = j + 1;
      }
      // Drain: every load issued here has landed before the CTA exits.
      mbar_wait(bar(B_QF), 0, nullptr, kEsDrainCap);
      for (int x = max(0, issued - 2); x < issued; ++x) mbar_wait(bar(B_KVF + (x & 1)), (x >> 1) & 1, nullptr, kEsDrainCap);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdSS = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdTS = idesc_bf16_f32(128, D, true);
    const bool leader = elect_one();
    const uint64_t dQd = sdesc_sw128(sQ, 16, 1024);
    bool ok = true;
    auto wait_or_fail = [&](int bb, int parity) -> bool {
      if (__all_sync(0xffffffffu, mbar_wait(bar(bb), parity, abort_flag, cap))) return true;
      if (leader) fail();
      ok = false;
      return false;
    };
    // S_{j mod 2} = Q K_j^T
    auto issue_qk = [&](int j) -> bool {
      if (!wait_or_fail(B_KVF + (j & 1), (j >> 1) & 1)) return false;
      tc_fence_after();
      if (leader) {
        const uint64_t dk = sdesc_sw128(stage(j & 1), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
          umma_bf16_ss(tmem + kTS + 128 * (j & 1), dQd + o, dk + o, kIdSS, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_SF + (j & 1)));
      }
      __syncwarp();
      return true;
    };
    if (wait_or_fail(B_QF, 0) && issue_qk(0) && (n_steps < 2 || issue_qk(1))) {
      for (int j = 0; j < n_steps; ++j) {
        if (!wait_or_fail(B_PF + (j & 1), (j >> 1) & 1)) break;
        tc_fence_after();
        if (leader) {
          // O += P_j V_j, P_j (bf16) read from the first 64 columns of S_{j mod 2}
          const uint64_t dv = sdesc_sw128(stage(j & 1) + C::kTile, 128 * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ts(tmem + kTO, tmem + kTS + 128 * (j & 1) + kk * 8, dv + kk * 128, kIdTS, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(B_PV));
          umma_commit(bar(B_KVE + (j & 1)));
        }
        __syncwarp();
        if (j + 2 < n_steps && !issue_qk(j + 2)) break;
      }
    }
    if (leader) umma_commit(bar(B_DONE));   // also: every MMA issued here has completed before TMEM is released
    __syncwarp();
    if (!ok) mbar_wait(bar(B_DONE), 0, nullptr, kEsDrainCap);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int qi = tq * 128 + r;
    const bool valid = qi < (glob ? g.G : g.L);
    const float cs = p.scale_log2;
    const int vmax = p.V - 1;
    // The -C of a blocked edge never enters the fp32 logits: while a row has
    // seen only blocked edges ("blocked frame") their weights are exp2(x - m)
    // of the unshifted logits (the common -C cancels); once it has an allowed
    // edge, blocked edges weigh exp(-10000 + ...) = 0 and the mass gathered in
    // the blocked frame is scaled by exp(-C) = 0.  C is subtracted from the
    // LSE of a row whose every edge is blocked.  Blocked edges are tagged in
    // the lowest mantissa bit of their logit (a 1-ulp change).
    bool has_allowed = false;
    float m_use = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_steps; ++j) {
      // this row's keys in tile j: columns [lo, hi]
      int lo = 0, hi;
      if (glob) {
        hi = j < g.n_gq ? min(127, g.G - 1 - j * 128) : min(127, g.L - 1 - (j - g.n_gq) * 128);
      } else if (j < n_band) {
        const int k0 = band_lo + j * 128;
        lo = max(qi - g.r, 0) - k0;
        hi = min(qi + g.r, g.L - 1) - k0;
      } else {
        hi = min(127, g.G - 1 - (j - n_band) * 128);
      }
      if (!valid) { lo = 1; hi = 0; }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SF + (j & 1)), (j >> 1) & 1, abort_flag, cap))) {
        fail(); ok = false; break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + kTS + 128 * (j & 1);
      const uint32_t crow = stage(j & 1) + 2 * C::kTile + r * 128;
      float x[128];
      float ta = -INFINITY, tb = -INFINITY;   // tile maxima over allowed / blocked edges
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float s[32];
        tmem_ld32(tS + 32 * c4, s);
        uint32_t cw[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t a = crow + ((((2 * c4 + h) ^ (r & 7))) << 4);
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(cw[4 * h]), "=r"(cw[4 * h + 1]), "=r"(cw[4 * h + 2]), "=r"(cw[4 * h + 3])
                       : "r"(a));
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = 32 * c4 + e;
          const uint32_t code = (cw[e >> 2] >> (8 * (e & 3))) & 0xFFu;
          float v = s[e] * cs;
          if (BIAS) {
            const int label = min(static_cast<int>(code & 127u), vmax);
            float qa;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(qa) : "r"(sQa + (label * 128 + r) * 4));
            v += qa;
          }
          const uint32_t blk = code >> 7;
          v = __uint_as_float((__float_as_uint(v) & ~1u) | blk);
          const bool member = col >= lo && col <= hi;
          x[col] = member ? v : -INFINITY;
          ta = fmaxf(ta, (member && !blk) ? v : -INFINITY);
          tb = fmaxf(tb, (member && blk) ? v : -INFINITY);
        }
      }
      const bool now_allowed = has_allowed || ta > -INFINITY;
      const float tmax = now_allowed ? ta : tb;
      const bool leave_blocked_frame = now_allowed && !has_allowed && l_run > 0.f;
      // lazy rescale: move the running maximum only when it grows by more than 2^8
      const bool grow = leave_blocked_frame || tmax > m_use + 8.f;
      const float m_new = grow ? tmax : m_use;
      const float f = grow ? (leave_blocked_frame ? 0.f : exp2f(m_use - m_new)) : 1.f;   // 0 when m_use is -inf
      const bool rescale_o = grow && l_run > 0.f;
      l_run *= f;
      m_use = m_new;
      has_allowed = now_allowed;
      if (__any_sync(0xffffffffu, rescale_o)) {
        // PV_{j-1} must have completed before O is read and written (PV_{j-2} has: QK_j came after it)
        if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(B_PV), (j - 1) & 1, abort_flag, cap))) {
          fail(); ok = false; break;
        }
        tc_fence_after();
        const float fo = rescale_o ? f : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_off + kTO + 32 * c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= fo;
          tmem_st32(tmem + lane_off + kTO + 32 * c, o);
        }
      }
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      float sum = 0.f;
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = x[32 * wd + 2 * i], x1 = x[32 * wd + 2 * i + 1];
          float p0 = ex2_approx(x0 - m_sub), p1 = ex2_approx(x1 - m_sub);
          p0 = (has_allowed && (__float_as_uint(x0) & 1u)) ? 0.f : p0;
          p1 = (has_allowed && (__float_as_uint(x1) & 1u)) ? 0.f : p1;
          sum += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16_nowait(tS + 16 * wd, pk);   // P over the S columns already read
      }
      l_run += sum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PF + (j & 1)));
    }
    if (ok) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DONE), 0, abort_flag, cap))) {
        fail();
      } else {
        tc_fence_after();
        const float inv = (valid && l_run > 0.f) ? 1.f / l_run : 0.f;
        // stage 32 rows x 64 columns per warp in the (now idle) first K tile and store with TMA
        const uint32_t st = stage(0) + (warp - 4) * 4096;
        const int y0 = tq * 128 + 32 * (warp & 3);
#pragma unroll 1
        for (int half = 0; half < D / 64; ++half) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            float o[32];
            tmem_ld32(tmem + lane_off + kTO + half * 64 + cc * 32, o);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int ci = cc * 4 + c;
              st_shared_v4(st + lane * 128 + ((ci ^ (lane & 7)) << 4), pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                           pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                           pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                           pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(glob ? &p.sOg : &p.sOl, st, half * 64, y0, bh);
            bulk_commit_group();
          }
        }
        if (valid) {
          const float lse = (m_use + __log2f(l_run)) * 0.6931471805599453f - (has_allowed ? 0.f : kEsMaskC);
          if (glob) p.lse_g[static_cast<size_t>(bh) * g.G + qi] = lse;
          else p.lse_l[static_cast<size_t>(bh) * g.L + qi] = lse;
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BIAS>
cudaError_t es_prepare() {
  static std::mutex mu;
  static bool done[kEsMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kEsMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(es_attn_kernel<D, BIAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, EsCfg<D>::kSmem);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

template <int D, bool BIAS>
cudaError_t es_launch(const EsParams& p, int units, cudaStream_t s) {
  cudaError_t e = es_prepare<D, BIAS>();
  if (e != cudaSuccess) return e;
  return launch_kernel(es_attn_kernel<D, BIAS>, dim3(static_cast<unsigned>(units)), dim3(kEsThreads), EsCfg<D>::kSmem,
                       s, false, p);
}

bool es_aligned(const void* x, size_t a) { return (reinterpret_cast<uintptr_t>(x) % a) == 0; }
size_t es_rup(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct EsLayout {
  size_t codes = 0, qa = 0, total = 0;
};

EsLayout es_layout(const EsGeom& g, int n_labels) {
  EsLayout w;
  size_t off = kStatusBytes;
  w.codes = off;
  off += es_rup(static_cast<size_t>(g.B) * g.blocks_per_b * kCodeTile, 256);
  w.qa = off;
  if (n_labels > 0)
    off += es_rup(static_cast<size_t>(g.B) * g.H * (g.n_gq + g.n_lq) * n_labels * 128 * 4, 256);
  w.total = off;
  return w;
}

lg_status es_check(int B, int H, int L, int G, int D, int radius, int n_labels, lg_dtype dt) {
  if (B < 1 || H < 1 || L < 1 || G < 1 || radius < 0 || n_labels < 0) return LG_ERR_INVALID_ARG;
  if (dt != LG_BF16 && dt != LG_F32) return LG_ERR_INVALID_ARG;
  if (dt != LG_BF16 || (D != 64 && D != 128) || n_labels > kEsMaxLabels) return LG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * (static_cast<long long>(L) + G) > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((L + 127) / 128 + (G + 127) / 128) > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  return LG_OK;
}

}  // namespace
}  // namespace lg

using namespace lg;

extern "C" {

size_t lg_etc_struct_attn_fwd_workspace_size(int B, int H, int L, int G, int D, int radius, int n_labels, lg_dtype dt) {
  if (es_check(B, H, L, G, D, radius, n_labels, dt) != LG_OK) return 0;
  return es_layout(es_geom(B, H, L, G, radius), n_labels).total;
}

lg_status lg_etc_struct_attn_fwd(const void* q_l, const void* k_l, const void* v_l, const void* q_g, const void* k_g,
                                 const void* v_g, void* out_l, void* out_g, float* lse_l, float* lse_g,
                                 const void* rel_k, int n_labels, const uint8_t* code_l2l, const uint8_t* code_l2g,
                                 const uint8_t* code_g2l, const uint8_t* code_g2g, lg_dtype dt, int B, int H, int L,
                                 int G, int D, int radius, float scale, void* workspace, size_t workspace_bytes,
                                 lg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  lg_status st = es_check(B, H, L, G, D, radius, n_labels, dt);
  if (st != LG_OK) return st;
  if ((rel_k == nullptr) != (n_labels == 0)) return LG_ERR_INVALID_ARG;
  const void* t16[] = {q_l, k_l, v_l, q_g, k_g, v_g, out_l, out_g};
  for (const void* x : t16)
    if (x == nullptr || !es_aligned(x, 16)) return LG_ERR_INVALID_ARG;
  if (!lse_l || !lse_g || !es_aligned(lse_l, 4) || !es_aligned(lse_g, 4)) return LG_ERR_INVALID_ARG;
  if (rel_k != nullptr && !es_aligned(rel_k, 16)) return LG_ERR_INVALID_ARG;
  const EsGeom geom = es_geom(B, H, L, G, radius);
  const EsLayout lay = es_layout(geom, n_labels);
  if (workspace == nullptr || !es_aligned(workspace, 256) || workspace_bytes < lay.total) return LG_ERR_WORKSPACE;
  if (!encode_fn()) return LG_ERR_CUDA;

  const int BH = B * H;
  const float s = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  EsParams p{};
  if (!encode_map(&p.mQl, q_l, D, L, BH, 1) || !encode_map(&p.mKl, k_l, D, L, BH, 1) ||
      !encode_map(&p.mVl, v_l, D, L, BH, 1) || !encode_map(&p.mQg, q_g, D, G, BH, 1) ||
      !encode_map(&p.mKg, k_g, D, G, BH, 1) || !encode_map(&p.mVg, v_g, D, G, BH, 1) ||
      !encode_store_map(&p.sOl, out_l, D, L, BH, 1) || !encode_store_map(&p.sOg, out_g, D, G, BH, 1))
    return LG_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) return LG_ERR_CUDA;
  const long long cap_blocks = 16LL * device_sm_count();

  EsPackParams pp{};
  pp.g = geom;
  pp.l2l = code_l2l; pp.l2g = code_l2g; pp.g2l = code_g2l; pp.g2g = code_g2g;
  pp.codes = reinterpret_cast<uint8_t*>(ws + lay.codes);
  pp.n_labels = n_labels;
  pp.status = status;
  const long long pack_threads = static_cast<long long>(B) * geom.blocks_per_b * (kCodeTile / 16);
  if (launch_kernel(es_pack_kernel, dim3(static_cast<unsigned>(std::min((pack_threads + 255) / 256, cap_blocks))),
                    dim3(256), 0, stream, false, pp) != cudaSuccess)
    return LG_ERR_CUDA;
  if (n_labels > 0) {
    EsQaParams qp{};
    qp.q_l = static_cast<const __nv_bfloat16*>(q_l);
    qp.q_g = static_cast<const __nv_bfloat16*>(q_g);
    qp.rel = static_cast<const __nv_bfloat16*>(rel_k);
    qp.qa = reinterpret_cast<float*>(ws + lay.qa);
    qp.H = H; qp.L = L; qp.G = G; qp.D = D; qp.V = n_labels; qp.n_gq = geom.n_gq; qp.n_lq = geom.n_lq;
    qp.total = static_cast<long long>(BH) * (geom.n_gq + geom.n_lq) * n_labels * 128;
    qp.c = s * 1.4426950408889634f;
    if (launch_kernel(es_qa_kernel, dim3(static_cast<unsigned>(std::min((qp.total + 255) / 256, cap_blocks))),
                      dim3(256), 0, stream, false, qp) != cudaSuccess)
      return LG_ERR_CUDA;
  }
  p.g = geom;
  p.codes = pp.codes;
  p.qa = reinterpret_cast<const float*>(ws + lay.qa);
  p.lse_l = lse_l;
  p.lse_g = lse_g;
  p.status = status;
  p.wait_cap = wait_cap_cycles();
  p.withhold = withhold_for_test();
  p.V = n_labels > 0 ? n_labels : 1;
  p.scale_log2 = s * 1.4426950408889634f;
  const int units = BH * (geom.n_gq + geom.n_lq);
  cudaError_t e = prof_mark(stream, true);
  if (e == cudaSuccess) {
    if (D == 64) e = n_labels > 0 ? es_launch<64, true>(p, units, stream) : es_launch<64, false>(p, units, stream);
    else e = n_labels > 0 ? es_launch<128, true>(p, units, stream) : es_launch<128, false>(p, units, stream);
  }
  if (e == cudaSuccess) e = prof_mark(stream, false);
  return e == cudaSuccess ? LG_OK : LG_ERR_CUDA;
}

}  // extern "C"
