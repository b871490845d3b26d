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
// bit 7.  Two kernels:
//  * es_pack_kernel lays the caller's four code arrays out as one 128 x 128
//    byte block per (query tile, key tile) in the order the attention kernel
//    visits them (rows of 128 bytes, 16-byte chunks XOR-swizzled by the row,
//    so that the softmax threads read them from shared memory without bank
//    conflicts), and checks the labels against the vocabulary;
//  * es_attn_kernel: one CTA per (instance, head, 128-row query tile) with
//    warp 0 loading tiles (TMA for q, k, v and a^K; bulk copies for the code
//    blocks), warp 1 owning tensor memory and issuing the MMAs from one lane,
//    and warps 4..11 the softmax: two threads per row, one per 64-column half
//    of the tile, which exchange their tile maxima through shared memory
//    (two warps per sub-partition, half the serial work each).  S = Q K^T lands in one
//    of two TMEM buffers, so the QK of tile j + 2 is issued right after the PV
//    of tile j and runs while the softmax works on tile j + 1; the softmax adds
//    qa[label], applies the blocked edges' -C (exactly, see the softmax),
//    keeps a running maximum (O rescaled in TMEM only when it grows by more
//    than 2^8), writes P (bf16) over its S and the MMA warp accumulates
//    O += P V with P read from TMEM.  With a relative term, one more MMA per
//    unit gives qa_il = q_i . a^K_l for the tile's rows and every label (the
//    appendix's q a^K table, M = 128, N = labels rounded up to 16, K = D); the
//    softmax threads move it, times s log2(e), from TMEM into a shared-memory
//    table stored label-major ([label][row]), so a thread gathers its row's
//    value of any label without bank conflicts.
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

constexpr int kEsThreads = 384;   // warp 0 loads, warp 1 MMA, warps 4..11 softmax (two column halves)
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

// One thread per 16-byte chunk of a block (16 edges of one row); four CTAs of
// 256 threads per block, so the block index is blockIdx.x / 4.
__global__ void __launch_bounds__(256) es_pack_kernel(const EsPackParams p) {
  const EsGeom& g = p.g;
  {
    const int blk = static_cast<int>(blockIdx.x >> 2);
    const int chunk = static_cast<int>((blockIdx.x & 3) * 256 + threadIdx.x);
    const long long idx = static_cast<long long>(blk) * (kCodeTile / 16) + chunk;
    const int bpb = static_cast<int>(g.blocks_per_b);
    const int b = blk / bpb;
    int rem = blk - b * bpb;
    const int row = chunk >> 3;
    const int k = (chunk & 7) ^ (row & 7);   // logical 16-column group stored in this physical chunk
    const bool glob = rem < g.n_gq * g.steps_g;
    int tq, j;
    if (glob) {
      tq = rem / g.steps_g; j = rem - tq * g.steps_g;
    } else {
      rem -= g.n_gq * g.steps_g;
      tq = rem / g.steps_l; j = rem - tq * g.steps_l;
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
    const uint8_t* src = piece == 1 ? p.l2l : piece == 2 ? p.l2g : piece == 3 ? p.g2l : p.g2g;
    const int kj0 = key0 + 16 * k;
    // A whole chunk of a g2g, l2g or g2l row whose bytes are 16-byte aligned: one load.
    const size_t vcols = piece == 2 ? g.G : (piece == 3 ? g.L : g.G);
    const size_t vrows = piece == 2 ? g.L : g.G;
    const bool vec = piece >= 2 && src != nullptr && kj0 + 16 <= key_n && vcols % 16 == 0 &&
                     (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    if (vec) {
      const uint4 x = *reinterpret_cast<const uint4*>(src + (static_cast<size_t>(b) * vrows + qi) * vcols + kj0);
      w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
      if (p.n_labels > 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (static_cast<int>((w[e >> 2] >> (8 * (e & 3))) & 127u) >= p.n_labels) bad = true;
      }
    } else if (piece != 0) {
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

// ---------------------------------------------------------------- attention

struct EsParams {
  CUtensorMap mQl, mKl, mVl, mQg, mKg, mVg;   // {D, rows, BH}, 128-row boxes
  CUtensorMap sOl, sOg;                       // output stores, 32-row boxes
  EsGeom g;
  CUtensorMap mA;                             // a^K viewed as {D, V, H}, boxes of Vp rows
  const uint8_t* codes;
  float* lse_l;
  float* lse_g;
  int* status;
  long long wait_cap;
  int withhold;
  int V, Vp;                                  // labels, and labels rounded up to 16 (the MMA's N)
  float scale_log2;
};

template <int D>
struct EsCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kStage = 2 * kTile + kCodeTile;   // K, V, code block
  static constexpr int kOffStage = kTile;                // after Q
  static constexpr int kOffMisc = kTile + 2 * kStage;    // barriers, then the softmax halves' exchange area
  static constexpr int kMisc = 8192;
  static constexpr int kOffQa = kOffMisc + kMisc;        // q . a^K of the tile's rows, [label][row]
  static constexpr int kMaxLabels = D == 64 ? kEsMaxLabels : 40;   // what fits in 227 KB next to D = 128 tiles
  // D = 64: the table has a row for every 7-bit label, so that any code byte's label reads
  // inside it without a clamp (labels past the vocabulary are reported by the packing kernel);
  // D = 128: kMaxLabels rows, the label clamped.
  static constexpr int kTableLabels = D == 64 ? 128 : kMaxLabels;
  static constexpr int kSmem = kOffQa + kTableLabels * 512 + 1024;   // + alignment slack
};

// Bits e of a 32-column chunk with lo <= e <= hi (any lo, hi; empty when lo > hi).
__device__ __forceinline__ uint32_t es_range_bits(int lo, int hi) {
  const int a = max(lo, 0), b = min(hi, 31);
  if (a > b) return 0u;
  const uint32_t upper = (b >= 31) ? 0xFFFFFFFFu : ((1u << (b + 1)) - 1u);
  return upper & ~((1u << a) - 1u);
}

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
  enum { B_QF = 0, B_KVF = 1, B_KVE = 3, B_SF = 5, B_PF = 7, B_PV = 9, B_DONE = 10, B_QAF = 11, NB = 12 };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 132);
  // exchange between the two column halves of a row: tile maxima [parity][half][row] (allowed
  // edges, all edges), and the final partial sums [half][row]
  float* x_allowed = reinterpret_cast<float*>(misc + 256);
  float* x_all = x_allowed + 512;
  float* x_sum = x_all + 512;
  auto bar = [&](int i) { return smem_addr(&bars[i]); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) mbar_init(bar(i), (i == B_PF || i == B_PF + 1) ? 256 : 1);
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
  // TMEM: S buffers at columns 0 and 128 (P of keys 0..63 over columns 0..31, of keys 64..127 over
  // columns 64..95, each inside the S columns its own softmax half reads), O at 256
  constexpr uint32_t kTS = 0, kTO = 256, kTQA = 256 + D;   // q . a^K of the tile's rows after O

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0 && !p.withhold) {
      int issued = 0;
      mbar_arrive_expect_tx(bar(B_QF), C::kTile + (BIAS ? p.Vp * D * 2 : 0));
      es_load_tile<D>(glob ? &p.mQg : &p.mQl, tq * 128, bh, sQ, bar(B_QF));
      if (BIAS) {
        // a^K of this head, Vp rows (rows past V zero-filled), staged in the q . a^K region until
        // the MMA that reads it has completed
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk) tma_load_3d(sQa + blk * p.Vp * 128, &p.mA, bar(B_QF), blk * 64, 0, bh % g.H);
      }
      for (int j = 0; j < n_steps; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(bar(B_KVE + st), ((j >> 1) - 1) & 1, abort_flag, cap)) { fail(); break; }
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
    bool q_ready = wait_or_fail(B_QF, 0);
    if (BIAS && q_ready) {
      // qa = Q a^K^T (M = 128, N = Vp, K = D) into TMEM columns kTQA..kTQA + Vp
      tc_fence_after();
      if (leader) {
        const uint32_t kIdQA = idesc_bf16_f32(128, p.Vp, false);
        const uint64_t dA = sdesc_sw128(sQa, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oq = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
          const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * (p.Vp * 128) + (kk & 3) * 32) >> 4);
          umma_bf16_ss(tmem + kTQA, dQd + oq, dA + oa, kIdQA, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_QAF));
      }
      __syncwarp();
    }
    if (q_ready && issue_qk(0) && (n_steps < 2 || issue_qk(1))) {
      for (int j = 0; j < n_steps; ++j) {
        if (!wait_or_fail(B_PF + (j & 1), (j >> 1) & 1)) break;
        tc_fence_after();
        if (leader) {
          // O += P_j V_j; keys 16 kk .. 16 kk + 15 of P at columns 8 kk (kk < 4) or 64 + 8 (kk - 4)
          const uint64_t dv = sdesc_sw128(stage(j & 1) + C::kTile, 128 * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ts(tmem + kTO, tmem + kTS + 128 * (j & 1) + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8), dv + kk * 128,
                         kIdTS, (j > 0 || kk > 0) ? 1u : 0u);
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
    // ------------------------------------------------------------ softmax (two column halves per row) + epilogue
    const int half = (warp - 4) >> 2;        // warps 4..7: columns 0..63; warps 8..11: columns 64..127
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int qi = tq * 128 + r;
    const bool valid = qi < (glob ? g.G : g.L);
    const float cs = p.scale_log2;
    const int vmax = p.V - 1;
    const uint32_t qa_row = sQa + r * 4;     // this row's entry of label 0 in the q . a^K table
    // The -C of a blocked edge never enters the fp32 logits: while a row has
    // seen only blocked edges ("blocked frame") their weights are exp2(x - m)
    // of the unshifted logits (the common -C cancels); once it has an allowed
    // edge, blocked edges weigh exp(-10000 + ...) = 0 and the mass gathered in
    // the blocked frame is scaled by exp(-C) = 0.  C is subtracted from the
    // LSE of a row whose every edge is blocked.  Blocked edges are tagged in
    // the lowest mantissa bit of their logit (a 1-ulp change).  Both halves of
    // a row take the same decisions from the exchanged tile maxima.
    bool has_allowed = false, has_mass = false;
    float m_use = -INFINITY, l_half = 0.f;
    bool ok = true;
    if (BIAS) {
      // this row's q . a^K from TMEM, times s log2(e), into the table [label][row] that replaces a^K
      // in shared memory (the MMA that read a^K has completed); half h moves labels 32 h .. 32 h + 31
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_QAF), 0, abort_flag, cap))) { fail(); ok = false; }
      if (ok && 32 * half < p.Vp) {
        tc_fence_after();
        float qa[32];
        tmem_ld32(tmem + lane_off + kTQA + 32 * half, qa);
        float* tab = reinterpret_cast<float*>(smem + C::kOffQa);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (32 * half + e < p.V) tab[(32 * half + e) * 128 + r] = qa[e] * cs;
      }
      named_bar_sync(2 + (warp & 3), 64);   // the two warps on these rows
    }
    for (int j = 0; j < n_steps; ++j) {
      // this row's keys in tile j: columns [lo, hi] of the full tile
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
      // After a failed wait a warp keeps taking the named barriers below (without waits or work),
      // so that every softmax thread takes each of them the same number of times.
      if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_SF + (j & 1)), (j >> 1) & 1, abort_flag, cap))) {
        fail(); ok = false;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + kTS + 128 * (j & 1);
      const uint32_t crow = stage(j & 1) + 2 * C::kTile + r * 128;
      float x[64];
      float ta = -INFINITY, tall = -INFINITY;   // maxima over this half's allowed / member edges
      uint32_t blk_any = 0u;                    // blocked bits of this row's code bytes
#pragma unroll
      for (int c2 = 0; c2 < 2 && ok; ++c2) {
        const int c4 = 2 * half + c2;          // 32-column chunk of the tile
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
        for (int k = 0; k < 8; ++k) blk_any |= cw[k];
        // this row's keys of the chunk as a bit mask (one bit test per edge below)
        const uint32_t kmask = es_range_bits(lo - 32 * c4, hi - 32 * c4);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint32_t wv = cw[e >> 2];
          const int kByte = 8 * (e & 3);   // a constant once the loop is unrolled
          float v;
          if (BIAS) {
            // the label's table row: (label << 9) taken straight from the code word
            uint32_t off;
            if constexpr (D == 64) {
              off = (kByte >= 9 ? (wv >> (kByte - 9)) : (wv << (9 - kByte))) & (127u << 9);
            } else {
              off = min((wv >> kByte) & 127u, static_cast<uint32_t>(vmax)) << 9;
            }
            float qa;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(qa) : "r"(qa_row + off));
            v = fmaf(s[e], cs, qa);
          } else {
            v = s[e] * cs;
          }
          const uint32_t blk = (wv >> (kByte + 7)) & 1u;
          v = __uint_as_float((__float_as_uint(v) & ~1u) | blk);
          const float xv = ((kmask >> e) & 1u) ? v : -INFINITY;
          x[32 * c2 + e] = xv;
          tall = fmaxf(tall, xv);
        }
      }
      // The maximum over the allowed edges differs only where a code byte is blocked (tagged
      // logits: lowest bit 1); taken in a second loop only for such warps.
      ta = tall;
      if (__any_sync(0xffffffffu, (blk_any & 0x80808080u) != 0u)) {
        ta = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e) ta = fmaxf(ta, (__float_as_uint(x[e]) & 1u) ? -INFINITY : x[e]);
      }
      // combine the two halves' maxima
      x_allowed[(j & 1) * 256 + half * 128 + r] = ta;
      x_all[(j & 1) * 256 + half * 128 + r] = tall;
      named_bar_sync(2 + (warp & 3), 64);   // the two warps on these rows
      ta = fmaxf(ta, x_allowed[(j & 1) * 256 + (1 - half) * 128 + r]);
      tall = fmaxf(tall, x_all[(j & 1) * 256 + (1 - half) * 128 + r]);
      if (!ok) continue;
      const bool now_allowed = has_allowed || ta > -INFINITY;
      const float tmax = now_allowed ? ta : tall;   // in the blocked frame every member is blocked
      const bool leave_blocked_frame = now_allowed && !has_allowed && has_mass;
      // lazy rescale: move the running maximum only when it grows by more than 2^8
      const bool grow = leave_blocked_frame || tmax > m_use + 8.f;
      const float m_new = grow ? tmax : m_use;
      const float f = grow ? (leave_blocked_frame ? 0.f : exp2f(m_use - m_new)) : 1.f;   // 0 when m_use is -inf
      const bool rescale_o = grow && has_mass;
      l_half *= f;
      m_use = m_new;
      has_allowed = now_allowed;
      has_mass = has_mass || tall > -INFINITY;
      if (__any_sync(0xffffffffu, rescale_o)) {
        // PV_{j-1} must have completed before O is read and written (PV_{j-2} has: QK_j came after it);
        // each half rescales its own D / 2 columns of O
        if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(B_PV), (j - 1) & 1, abort_flag, cap))) {
          fail(); ok = false; continue;
        }
        tc_fence_after();
        const float fo = rescale_o ? f : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          float o[32];
          const uint32_t ta_o = tmem + lane_off + kTO + half * (D / 2) + 32 * c;
          tmem_ld32(ta_o, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= fo;
          tmem_st32(ta_o, o);
        }
      }
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      const uint64_t negm2 = f2_pack(-m_sub, -m_sub);
      const uint32_t tag = has_allowed ? 1u : 0u;   // blocked edges weigh 0 once the row has an allowed one
      uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
      for (int wd = 0; wd < 2; ++wd) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = x[32 * wd + 2 * i], x1 = x[32 * wd + 2 * i + 1];
          float a0, a1;
          f2_unpack(f2_add(f2_pack(x0, x1), negm2), a0, a1);
          float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
          p0 = (__float_as_uint(x0) & tag) ? 0.f : p0;
          p1 = (__float_as_uint(x1) & tag) ? 0.f : p1;
          sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16_nowait(tS + 64 * half + 16 * wd, pk);   // P of this half's keys over its own S columns
      }
      float s0, s1, s2, s3;
      f2_unpack(sum2[0], s0, s1);
      f2_unpack(sum2[1], s2, s3);
      l_half += (s0 + s1) + (s2 + s3);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PF + (j & 1)));
    }
    // the row's sum: both halves' partial sums
    x_sum[half * 128 + r] = l_half;
    named_bar_sync(2 + (warp & 3), 64);   // the two warps on these rows
    const float l_run = l_half + x_sum[(1 - half) * 128 + r];
    if (ok) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DONE), 0, abort_flag, cap))) {
        fail();
      } else if (D == 128 || half == 0) {
        tc_fence_after();
        const float inv = (valid && l_run > 0.f) ? 1.f / l_run : 0.f;
        // stage 32 rows x 64 columns per warp in the (now idle) first K tile and store with TMA;
        // D = 128: half h stores columns 64 h .. 64 h + 63
        const uint32_t st = stage(0) + (warp - 4) * 4096;
        const int y0 = tq * 128 + 32 * (warp & 3);
        const int col0 = D == 128 ? 64 * half : 0;
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          float o[32];
          tmem_ld32(tmem + lane_off + kTO + col0 + cc * 32, o);
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
          tma_store_3d(glob ? &p.sOg : &p.sOl, st, col0, y0, bh);
          bulk_commit_group();
        }
        if (valid && half == 0) {
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
  size_t codes = 0, total = 0;
};

EsLayout es_layout(const EsGeom& g) {
  EsLayout w;
  size_t off = kStatusBytes;
  w.codes = off;
  off += es_rup(static_cast<size_t>(g.B) * g.blocks_per_b * kCodeTile, 256);
  w.total = off;
  return w;
}

// a^K [H, V, D] bf16 viewed as {D, V, H} for loads of Vp rows x 64 columns
// (rows past V zero-filled), the B operand of the q . a^K contraction.
bool es_encode_rel(CUtensorMap* m, const void* rel, int D, int V, int Vp, int H) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(H)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(V) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(Vp), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(rel), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

lg_status es_check(int B, int H, int L, int G, int D, int radius, int n_labels, lg_dtype dt) {
  if (B < 1 || H < 1 || L < 1 || G < 1 || radius < 0 || n_labels < 0) return LG_ERR_INVALID_ARG;
  if (dt != LG_BF16 && dt != LG_F32) return LG_ERR_INVALID_ARG;
  if (dt != LG_BF16 || (D != 64 && D != 128)) return LG_ERR_UNSUPPORTED;
  if (n_labels > (D == 64 ? EsCfg<64>::kMaxLabels : EsCfg<128>::kMaxLabels)) return LG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * (static_cast<long long>(L) + G) > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((L + 127) / 128 + (G + 127) / 128) > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  {
    // the code blocks of one call are indexed with 32-bit integers, four packing CTAs per block
    const EsGeom g = es_geom(B, H, L, G, radius);
    if (static_cast<long long>(B) * g.blocks_per_b * 4 > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  }
  return LG_OK;
}

}  // namespace
}  // namespace lg

using namespace lg;

extern "C" {

size_t lg_etc_struct_attn_fwd_workspace_size(int B, int H, int L, int G, int D, int radius, int n_labels, lg_dtype dt) {
  if (es_check(B, H, L, G, D, radius, n_labels, dt) != LG_OK) return 0;
  return es_layout(es_geom(B, H, L, G, radius)).total;
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
  const EsLayout lay = es_layout(geom);
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

  EsPackParams pp{};
  pp.g = geom;
  pp.l2l = code_l2l; pp.l2g = code_l2g; pp.g2l = code_g2l; pp.g2g = code_g2g;
  pp.codes = reinterpret_cast<uint8_t*>(ws + lay.codes);
  pp.n_labels = n_labels;
  pp.status = status;
  const long long pack_ctas = static_cast<long long>(B) * geom.blocks_per_b * 4;
  if (launch_kernel(es_pack_kernel, dim3(static_cast<unsigned>(pack_ctas)), dim3(256), 0, stream, false, pp) !=
      cudaSuccess)
    return LG_ERR_CUDA;
  p.g = geom;
  p.codes = pp.codes;
  p.lse_l = lse_l;
  p.lse_g = lse_g;
  p.status = status;
  p.wait_cap = wait_cap_cycles();
  p.withhold = withhold_for_test();
  p.V = n_labels > 0 ? n_labels : 1;
  p.Vp = (p.V + 15) / 16 * 16;
  if (n_labels > 0 && !es_encode_rel(&p.mA, rel_k, D, n_labels, p.Vp, H)) return LG_ERR_CUDA;
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
