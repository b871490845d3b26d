// bf16 window + dilation + global attention, backward pass, on the
// 5th-generation tensor cores (tcgen05 MMA with TMEM accumulators, TMA loads).
//
// The gradients are the chain rule of the forward's masked softmax, with P
// recomputed from the saved LSE instead of a second softmax pass:
//   P = exp(s q k^T - LSE) on the allowed pairs (0 elsewhere),
//   dV = P^T dO,  dP = dO V^T,  Delta_i = sum_d dO_id O_id,
//   dS = P o (dP - Delta),  dQ = s dS K,  dK = s dS^T Q.
// The pages train with this attention and take these gradients through it:
// "LONGNET: Scaling Transformers to 1,000,000,000 Tokens", section 3.4,
// "Distributed Training Algorithm" (gradients of the keys and values), and
// "Longformer: The Long-Document Transformer", "Autoregressive Language
// Modeling Configuration" (activations recomputed in the backward pass).
// The mask is the forward's: "Longformer", section 3.4, "Sliding Window
// Attention", "Dilated Sliding Window Attention", "Global Attention"; and
// "ETC: Encoding Long and Structured Inputs in Transformers", section 3.4,
// "Global-Local Attention".
//
// Two kernels, one CTA per work unit (384 threads: warp 0 loads tiles with
// TMA, warp 1 owns TMEM and issues the MMAs from one elected lane, warps 4..11
// are two elementwise warpgroups, one thread per TMEM lane in each, taking the
// two 64-column halves of every tile):
//  * bwd_q_kernel: TMEM rows are 128 queries.  Per key tile: S = Q K^T and
//    dP = dO V^T (TMEM; S alternates between two buffers, so S of the next key
//    tile is computed during this tile's elementwise step), then the warpgroups
//    write dS (bf16) over S, then dQ += dS K (A operand read from TMEM).  Band units: a query tile of one
//    dilation residue class against its band key tiles and the global-key
//    tiles (global keys inside the band masked there, as in the forward).
//    Global-row units: 128 global queries against a split of all key tiles,
//    writing partial sums of dQ.
//  * bwd_kv_kernel: TMEM rows are 128 keys.  Per query tile: S^T = K Q^T and
//    dP^T = V dO^T (at D = 64 S^T alternates between two buffers as S does
//    above), then the warpgroups write P^T over S^T and dS^T over dP^T, then
//    dV += P^T dO and dK += dS^T Q.  Band units: a key tile of one
//    residue class against the query tiles whose windows reach it and the
//    global-query tiles (a global row whose band already holds the key is
//    masked there, so every pair counts once).  Global-key units: 128 global
//    keys against a split of all query tiles, writing partial sums of dK, dV.
// Partials simply add (P comes from the final LSE, so no rescaling); a
// reduce kernel sums them and scatters the global rows' dQ, dK, dV, after
// the band units wrote theirs.  Dilated residue classes are read and
// written through tensor maps with element stride d, as in the forward.
#include <math.h>

#include <atomic>

#include "lg_internal.h"
#include "lg_ptx.cuh"

namespace lg {

// Class stride of the class-major vectors: class c of a head with dilation d
// starts at c * M (16-byte aligned).
__host__ __device__ int bwd_class_stride(int N, int d) {
  const int n = (N + d - 1) / d;
  return (n + 3) / 4 * 4;
}
int bwd_cm(int N) { return (N + 4 * LG_MAX_BF16_DILATION + 128 + 3) / 4 * 4; }

namespace {

constexpr int kBwdThreads = 384;   // warp 0 TMA, warp 1 MMA, warps 4..11 elementwise (two column halves)
constexpr long long kBwdDrainCap = 4000000000LL;   // fixed bound of waits for already-issued async work
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ __forceinline__ int rows_per_load_b(int d) { return d <= 2 ? 128 : (d <= 4 ? 64 : 32); }

// TMA loads of one 128-row tile (D / 64 blocks of 64 columns, 128-byte swizzle).
template <int D>
__device__ __forceinline__ void load_tile_b(const CUtensorMap* map, int d, int y0, int bh, uint32_t dst, uint32_t bar) {
  const int R = rows_per_load_b(d);
#pragma unroll
  for (int blk = 0; blk < D / 64; ++blk)
    for (int piece = 0; piece < 128 / R; ++piece)
      tma_load_3d(dst + blk * (128 * 128) + piece * R * 128, map, bar, blk * 64, y0 + piece * R * d, bh);
}

__device__ __forceinline__ uint32_t range_bits_b(int lo, int hi, int base) {
  const int a = max(lo - base, 0), b = min(hi - base, 31);
  if (a > b) return 0u;
  const uint32_t upper = (b >= 31) ? 0xFFFFFFFFu : ((1u << (b + 1)) - 1u);
  return upper & ~((1u << a) - 1u);
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Residue class and first step of class-major tile x of one head (classes
// c = 0..d-1 in order, ceil(n_c / 128) tiles each).
__device__ __forceinline__ void class_tile(int N, int d, int x, int& c, int& t0, int& n_c) {
  c = 0; t0 = 0; n_c = N;
  for (int cc = 0; cc < d; ++cc) {
    const int n = (N - cc + d - 1) / d;
    const int nt = (n + 127) / 128;
    if (x < nt) { c = cc; t0 = x * 128; n_c = n; return; }
    x -= nt;
  }
}

// A work unit: the 128 rows of this CTA (own side) and its tiles of the other side.
struct BUnit {
  int grow;            // 1: global rows (q) / global keys (kv) against a split of the other side
  int bh;
  int c, n_c, t0;      // band: residue class, class length, first step of the own tile
  int band_lo, n_band; // band: first class step of the other side's band tiles, their count
  int gt;              // grow: tile of the global side
  int x0;              // grow: first other-side tile of the split
  int n_tiles;         // other-side tiles
};

// Band tiles of the other side: kv units (keys) see the queries in
// [u - w_right, u + w_left]; q units (queries) see the keys in
// [t - w_left, t + w_right].
__device__ BUnit decode_bwd_unit(const BwdParams& p, int u, bool kv) {
  BUnit w{};
  if (u < p.n_grow) {
    w.grow = 1;
    const int split = u % p.n_splits;
    int r = u / p.n_splits;
    w.gt = r % p.n_gt;
    r /= p.n_gt;
    const int hi = r % p.n_heads, b = r / p.n_heads;
    w.bh = b * p.H + p.heads[hi];
    w.x0 = split * p.split;
    w.n_tiles = min(p.split, p.other_tiles - w.x0);
    return w;
  }
  const int v = u - p.n_grow;
  const int tile = v % p.tiles_per_head;
  const int r = v / p.tiles_per_head;
  const int hi = r % p.n_heads, b = r / p.n_heads;
  w.bh = b * p.H + p.heads[hi];
  class_tile(p.N, p.d, tile, w.c, w.t0, w.n_c);
  const int before = kv ? p.wr : p.wl, after = kv ? p.wl : p.wr;
  const int t_last = min(w.t0 + 127, w.n_c - 1);
  // a multiple of 4 steps: the tile's 128 lse2 / delta values are read with a
  // bulk copy, whose source must be 16-byte aligned
  w.band_lo = max(0, w.t0 - before) & ~3;
  const int band_hi = min(w.n_c - 1, t_last + after);
  w.n_band = (band_hi - w.band_lo) / 128 + 1;
  w.n_tiles = w.n_band + p.n_gt;
  return w;
}

// Where other-side tile j of unit w comes from.  kind: 0 band tile (class c,
// steps from s0), 1 global-side tile (global index g0), 2 class tile of a
// grow unit (class c, steps from s0).  y: row coordinate in the tensor map;
// vec: offset of its 128 lse2 / delta values (kv kernel).
struct OTile {
  int kind, c, s0, n_c, g0, y;
  size_t vec;
};

__device__ __forceinline__ OTile other_tile(const BwdParams& p, const BUnit& w, int j) {
  OTile o{};
  if (!w.grow) {
    if (j < w.n_band) {
      o.kind = 0; o.c = w.c; o.n_c = w.n_c; o.s0 = w.band_lo + j * 128;
      o.y = o.c + p.d * o.s0;
      o.vec = static_cast<size_t>(w.bh) * p.CM + static_cast<size_t>(o.c) * p.M + o.s0;
    } else {
      o.kind = 1; o.g0 = (j - w.n_band) * 128;
      o.y = o.g0;
      o.vec = static_cast<size_t>(w.bh) * p.gpad + o.g0;
    }
    return o;
  }
  int x = w.x0 + j;
  if (p.etc && x < p.n_gt) {
    o.kind = 1; o.g0 = x * 128; o.y = o.g0;
    o.vec = static_cast<size_t>(w.bh) * p.gpad + o.g0;
    return o;
  }
  if (p.etc) x -= p.n_gt;
  o.kind = 2;
  class_tile(p.N, p.d, x, o.c, o.s0, o.n_c);
  o.y = o.c + p.d * o.s0;
  o.vec = static_cast<size_t>(w.bh) * p.CM + static_cast<size_t>(o.c) * p.M + o.s0;
  return o;
}

// Keep mask (4 words of 32 columns) of one row against other-side tile o.
//  band tile: columns [lo, hi] (the caller computes them);
//  global tile: columns below the global count, minus [ca, cb) (the
//    Longformer global rows/keys already counted in the band; for d > 1 only
//    those on the row's stride lattice: `lattice_pos`, checked per column);
//  class tile of a grow unit: the rows of the class.
struct KeepMask {
  uint32_t w[4];
  bool any_partial;   // warp-uniform: some row of the warp keeps part of the tile
};

__device__ __forceinline__ KeepMask make_keep(int lo, int hi, int ca, int cb, const int* gidx, int g0, int d,
                                              int lattice_pos) {
  KeepMask k;
  k.any_partial = __any_sync(0xffffffffu, (lo > 0) | (hi < 127) | (ca < cb));
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) k.w[wd] = 0xFFFFFFFFu;
  if (k.any_partial) {
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) k.w[wd] = range_bits_b(lo, hi, 32 * wd);
    if (ca < cb) {
      if (d == 1) {
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) k.w[wd] &= ~range_bits_b(ca, cb - 1, 32 * wd);
      } else {
        for (int c = ca; c < cb; ++c) {
          if ((__ldg(gidx + g0 + c) - lattice_pos) % d == 0) {
            const uint32_t bit = 1u << (c & 31);
            if ((c >> 5) == 0) k.w[0] &= ~bit;
            else if ((c >> 5) == 1) k.w[1] &= ~bit;
            else if ((c >> 5) == 2) k.w[2] &= ~bit;
            else k.w[3] &= ~bit;
          }
        }
      }
    }
  }
  return k;
}

__device__ __forceinline__ uint32_t keep_word(const KeepMask& k, int wd) {
  return wd == 0 ? k.w[0] : (wd == 1 ? k.w[1] : (wd == 2 ? k.w[2] : k.w[3]));
}

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kVecBytes = 1024;   // 128 lse2 + 128 delta (kv kernel stages)
  // q kernel: Q, dO, then two stages of (K, V)
  static constexpr int kQSmem = 6 * kTileBytes;
  // kv kernel: K, V, then two stages of (Q, dO, vectors)
  static constexpr int kKVStage = 2 * kTileBytes + kVecBytes;
  static constexpr int kKVSmem = 2 * kTileBytes + 2 * kKVStage;
  static constexpr int kMisc = 256;
  static constexpr int kQTotal = kQSmem + kMisc + 1024;
  static constexpr int kKVTotal = kKVSmem + kMisc + 1024;
};

// Shared pieces of the two kernels' epilogues: 32 rows x 64 columns of an
// fp32 TMEM accumulator, times `mul`, to bf16 in a swizzled staging buffer
// and out through a TMA store.
template <int D>
__device__ __forceinline__ void store_rows_tma(const CUtensorMap* map, uint32_t stage, uint32_t tacc, float mul,
                                               int y0, int bh, int lane, int col_half) {
  // D = 128: this warp stores the 64 columns of col_half; D = 64: all 64 columns
#pragma unroll 1
  for (int half = D == 128 ? col_half : 0; half < (D == 128 ? col_half + 1 : 1); ++half) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      float o[32];
      tmem_ld32(tacc + half * 64 + cc * 32, o);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int ci = cc * 4 + c;
        st_shared_v4(stage + lane * 128 + ((ci ^ (lane & 7)) << 4), pack_bf16x2(o[8 * c] * mul, o[8 * c + 1] * mul),
                     pack_bf16x2(o[8 * c + 2] * mul, o[8 * c + 3] * mul),
                     pack_bf16x2(o[8 * c + 4] * mul, o[8 * c + 5] * mul),
                     pack_bf16x2(o[8 * c + 6] * mul, o[8 * c + 7] * mul));
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(map, stage, half * 64, y0, bh);
      bulk_commit_group();
    }
  }
}

// fp32 partial sums of one row from one or two TMEM accumulators (tacc_b,
// dst_b: the second, or 0 / NULL), 32 columns of each per iteration.  The
// warp-collective TMEM loads run in every lane, and the warp reconverges
// after the stores of the valid rows before the next loads.  (Reading two
// accumulators in two separate loops gave the first one's values twice.)
template <int D>
__device__ __forceinline__ void store_partial_rows(float* dst_a, uint32_t tacc_a, float* dst_b, uint32_t tacc_b,
                                                   bool valid, int c_begin, int c_end) {
#pragma unroll 1
  for (int cc = c_begin; cc < c_end; ++cc) {
    float oa[32], ob[32];
    tmem_ld32(tacc_a + cc * 32, oa);
    if (dst_b != nullptr) tmem_ld32(tacc_b + cc * 32, ob);
    if (valid) {
      float4* a4 = reinterpret_cast<float4*>(dst_a) + 8 * cc;
#pragma unroll
      for (int k = 0; k < 8; ++k) a4[k] = make_float4(oa[4 * k], oa[4 * k + 1], oa[4 * k + 2], oa[4 * k + 3]);
      if (dst_b != nullptr) {
        float4* b4 = reinterpret_cast<float4*>(dst_b) + 8 * cc;
#pragma unroll
        for (int k = 0; k < 8; ++k) b4[k] = make_float4(ob[4 * k], ob[4 * k + 1], ob[4 * k + 2], ob[4 * k + 3]);
      }
    }
    __syncwarp();
  }
}

// ======================================================================== dQ

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_q_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t sQ = sb, sdO = sb + C::kTileBytes, sKV = sb + 2 * C::kTileBytes;
  unsigned char* misc = smem + C::kQSmem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  enum { B_QF = 0, B_KVF = 1, B_KVE = 3, B_SR = 5, B_PR = 6, B_DONE = 7, NB = 8 };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 132);
  auto bar = [&](int i) { return smem_addr(&bars[i]); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) mbar_init(bar(i), i == B_PR ? 256 : 1);
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
  const BUnit w = decode_bwd_unit(p, blockIdx.x, false);
  // S of key tile j in buffer j & 1 (columns 0 or 384): S of tile j + 1 is computed while
  // the elementwise warps work on tile j, and only dP of tile j + 1 waits for them.
  constexpr uint32_t kTS = 0, kTdP = 128, kTdQ = 256, kTS1 = 384;
  auto s_col = [&](int j) -> uint32_t { return (j & 1) ? kTS1 : kTS; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar(B_QF), 2 * C::kTileBytes);
      if (w.grow) {
        load_tile_b<D>(&p.mQG, 1, w.gt * 128, w.bh, sQ, bar(B_QF));
        load_tile_b<D>(&p.mdOG, 1, w.gt * 128, w.bh, sdO, bar(B_QF));
      } else {
        load_tile_b<D>(&p.mQ, p.d, w.c + p.d * w.t0, w.bh, sQ, bar(B_QF));
        load_tile_b<D>(&p.mdO, p.d, w.c + p.d * w.t0, w.bh, sdO, bar(B_QF));
      }
      for (int j = 0; j < w.n_tiles && ok; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(bar(B_KVE + st), ((j >> 1) - 1) & 1, abort_flag, cap)) { fail(); ok = false; break; }
        const OTile o = other_tile(p, w, j);
        const bool glob = o.kind == 1;
        const uint32_t dst = sKV + st * 2 * C::kTileBytes;
        mbar_arrive_expect_tx(bar(B_KVF + st), 2 * C::kTileBytes);
        load_tile_b<D>(glob ? &p.mKG : &p.mK, glob ? 1 : p.d, o.y, w.bh, dst, bar(B_KVF + st));
        load_tile_b<D>(glob ? &p.mVG : &p.mV, glob ? 1 : p.d, o.y, w.bh, dst + C::kTileBytes, bar(B_KVF + st));
        issued = j + 1;
      }
      // Drain: every load issued here has landed before the CTA exits.
      mbar_wait(bar(B_QF), 0, nullptr, kBwdDrainCap);
      for (int x = max(0, issued - 2); x < issued; ++x) mbar_wait(bar(B_KVF + (x & 1)), (x >> 1) & 1, nullptr, kBwdDrainCap);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdSS = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdTS = idesc_bf16_f32(128, D, true);
    constexpr uint64_t kStage = (2 * C::kTileBytes) >> 4;
    const bool leader = elect_one();
    const uint64_t dQd = sdesc_sw128(sQ, 16, 1024), ddO = sdesc_sw128(sdO, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024), dV0 = sdesc_sw128(sKV + C::kTileBytes, 16, 1024);
    const uint64_t dKmn0 = sdesc_sw128(sKV, 128 * 128, 1024);
    bool ok = true;
    auto wait_or_fail = [&](int b, int parity) -> bool {
      if (__all_sync(0xffffffffu, mbar_wait(bar(b), parity, abort_flag, cap))) return true;
      if (leader) fail();
      ok = false;
      return false;
    };
    // S(j) = Q K(j)^T into buffer j & 1; dP(j) = dO V(j)^T; dQ += dS(j) K(j) with dS(j) read
    // from S(j)'s buffer.  Order per tile: S(j + 1) (its buffer was last read by dQ(j - 1),
    // issued before it), then, once the elementwise warps are done with tile j, dQ(j) and
    // dP(j + 1) (dP's columns are free again), then the commit that S(j + 1) and dP(j + 1)
    // are ready.
    auto s_mmas = [&](int j) {
      const uint64_t dk = dK0 + (j & 1) * kStage;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
        umma_bf16_ss(tmem + s_col(j), dQd + o, dk + o, kIdSS, kk > 0 ? 1u : 0u);
      }
    };
    auto dp_mmas = [&](int j) {
      const uint64_t dv = dV0 + (j & 1) * kStage;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
        umma_bf16_ss(tmem + kTdP, ddO + o, dv + o, kIdSS, kk > 0 ? 1u : 0u);
      }
    };
    if (wait_or_fail(B_QF, 0) && w.n_tiles > 0 && wait_or_fail(B_KVF, 0)) {
      tc_fence_after();
      if (leader) {
        s_mmas(0);
        dp_mmas(0);
        umma_commit(bar(B_SR));
      }
      __syncwarp();
      for (int j = 0; j < w.n_tiles; ++j) {
        const int st = j & 1;
        const bool next = j + 1 < w.n_tiles;
        if (next) {
          if (!wait_or_fail(B_KVF + (st ^ 1), ((j + 1) >> 1) & 1)) break;
          tc_fence_after();
          if (leader) s_mmas(j + 1);
          __syncwarp();
        }
        if (!wait_or_fail(B_PR, j & 1)) break;
        tc_fence_after();
        if (leader) {
          const uint64_t dkm = dKmn0 + st * kStage;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ts(tmem + kTdQ, tmem + s_col(j) + kk * 8 + (kk >= 4 ? 32 : 0), dkm + kk * 128, kIdTS,
                         (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(B_KVE + st));
          if (next) {
            dp_mmas(j + 1);
            umma_commit(bar(B_SR));
          }
        }
        __syncwarp();
      }
    }
    if (leader) umma_commit(bar(B_DONE));   // also: every MMA issued here has completed before TMEM is released
    __syncwarp();
    if (!ok) mbar_wait(bar(B_DONE), 0, nullptr, kBwdDrainCap);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise warpgroups + epilogue
    // Two threads per row: warps 4..7 take columns 0..63, warps 8..11 columns 64..127 (every
    // element is independent: P and dS need only per-row and per-column constants).  Each half
    // writes its packed bf16 results inside its own S / dP columns (columns 32 h.. + 0..31).
    const int half = (warp - 4) >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tdP = tmem + lane_off + kTdP, tdQ = tmem + lane_off + kTdQ;
    bool valid;
    float lse2r, deltar;
    int t = 0, pos = 0;
    if (w.grow) {
      const int gr = w.gt * 128 + r;
      valid = gr < p.n_glob;
      lse2r = valid ? p.lse2g[static_cast<size_t>(w.bh) * p.gpad + gr] : 0.f;
      deltar = valid ? p.deltag[static_cast<size_t>(w.bh) * p.gpad + gr] : 0.f;
    } else {
      t = w.t0 + r;
      pos = w.c + p.d * t;
      valid = t < w.n_c;
      const size_t ix = static_cast<size_t>(w.bh) * p.CM + static_cast<size_t>(w.c) * p.M + t;
      lse2r = valid ? p.lse2[ix] : 0.f;
      deltar = valid ? p.delta[ix] : 0.f;
    }
    // Global keys inside this row's band (Longformer): list indices [g_a, g_b).
    int g_a = 0, g_b = 0;
    if (!w.grow && !p.etc && p.n_glob > 0 && valid) {
      const long long a = static_cast<long long>(pos) - static_cast<long long>(p.d) * p.wl;
      const long long b = static_cast<long long>(pos) + static_cast<long long>(p.d) * p.wr + 1;
      g_a = __ldg(p.gcount + (a < 0 ? 0 : (a > p.N ? p.N : a)));
      g_b = __ldg(p.gcount + (b < 0 ? 0 : (b > p.N ? p.N : b)));
    }
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2), nl2 = f2_pack(-lse2r, -lse2r);
    const uint64_t nd2 = f2_pack(-deltar, -deltar);
    bool ok = true;
    for (int j = 0; j < w.n_tiles; ++j) {
      const OTile o = other_tile(p, w, j);
      int lo = 0, hi = 127, ca = 0, cb = 0;
      if (o.kind == 0) {
        lo = t - p.wl - o.s0;
        hi = min(t + p.wr, o.n_c - 1) - o.s0;
      } else if (o.kind == 1) {
        hi = min(128, p.n_glob - o.g0) - 1;
        if (!w.grow && !p.etc) { ca = max(g_a - o.g0, 0); cb = min(g_b - o.g0, 128); }
      } else {
        hi = min(128, o.n_c - o.s0) - 1;
      }
      const KeepMask km = make_keep(lo, hi, ca, cb, p.gidx, o.g0, p.d, pos);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SR), j & 1, abort_flag, cap))) { fail(); ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + s_col(j);
#pragma unroll 1
      for (int wd = 2 * half; wd < 2 * half + 2; ++wd) {
        uint32_t sr[32], dr[32];
        tmem_ld32_nowait(tS + 32 * wd, sr);
        tmem_ld32_nowait(tdP + 32 * wd, dr);
        tmem_wait_ld();
        const uint32_t kw = keep_word(km, wd);
        const bool full = !km.any_partial || __all_sync(0xffffffffu, kw == 0xFFFFFFFFu);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1, d0, d1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), c2, nl2), x0, x1);
          const uint64_t pp = f2_pack(ex2_approx(x0), ex2_approx(x1));
          const uint64_t dd = f2_add(f2_pack(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1])), nd2);
          f2_unpack(f2_mul(pp, dd), d0, d1);
          if (!full) {
            d0 = ((kw >> (2 * i)) & 1u) ? d0 : 0.f;
            d1 = ((kw >> (2 * i + 1)) & 1u) ? d1 : 0.f;
          }
          pk[i] = pack_bf16x2(d0, d1);
        }
        tmem_st16_nowait(tS + 16 * wd + 32 * half, pk);   // dS over this half's S columns, already read
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PR));
    }
    if (ok) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DONE), 0, abort_flag, cap))) {
        fail();
      } else {
        tc_fence_after();
        if (w.grow) {
          const size_t prow = (static_cast<size_t>(w.bh) * p.n_glob + w.gt * 128 + r) * p.ns_stride + w.x0 / p.split;
          const int c0 = half * (D / 64), c1 = c0 + D / 64;   // this half's 32-column chunks
          store_partial_rows<D>(p.part_a + prow * D, tdQ, nullptr, 0u, valid, c0, c1);
        } else {
          const uint32_t stage = sKV + (warp - 4) * 4096;
          const int y0 = w.c + p.d * (w.t0 + 32 * (warp & 3));
          if (D == 128 || half == 0) store_rows_tma<D>(&p.sA, stage, tdQ, p.scale, y0, w.bh, lane, half);
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

// ======================================================================== dK, dV

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kv_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t sK = sb, sV = sb + C::kTileBytes, sQS = sb + 2 * C::kTileBytes;  // stage st at sQS + st * kKVStage
  unsigned char* misc = smem + C::kKVSmem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  enum { B_KVF = 0, B_QF = 1, B_QE = 3, B_SR = 5, B_PR = 6, B_DONE = 7, NB = 8 };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 132);
  auto bar = [&](int i) { return smem_addr(&bars[i]); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) mbar_init(bar(i), i == B_PR ? 256 : 1);
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
  const BUnit w = decode_bwd_unit(p, blockIdx.x, true);
  constexpr uint32_t kTS = 0, kTdP = 128, kTdV = 256, kTdK = 256 + D;
  // D = 64 leaves columns 384..511 free: S^T of query tile j in buffer j & 1 (columns 0 or
  // 384), so S^T of tile j + 1 is computed while the elementwise warps work on tile j.
  // D = 128 fills the 512 columns and keeps one buffer.
  constexpr bool kDB = D == 64;
  constexpr uint32_t kTS1 = 384;
  auto s_col = [&](int j) -> uint32_t { return (kDB && (j & 1)) ? kTS1 : kTS; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar(B_KVF), 2 * C::kTileBytes);
      if (w.grow) {
        load_tile_b<D>(&p.mKG, 1, w.gt * 128, w.bh, sK, bar(B_KVF));
        load_tile_b<D>(&p.mVG, 1, w.gt * 128, w.bh, sV, bar(B_KVF));
      } else {
        load_tile_b<D>(&p.mK, p.d, w.c + p.d * w.t0, w.bh, sK, bar(B_KVF));
        load_tile_b<D>(&p.mV, p.d, w.c + p.d * w.t0, w.bh, sV, bar(B_KVF));
      }
      for (int j = 0; j < w.n_tiles && ok; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(bar(B_QE + st), ((j >> 1) - 1) & 1, abort_flag, cap)) { fail(); ok = false; break; }
        const OTile o = other_tile(p, w, j);
        const bool glob = o.kind == 1;
        const uint32_t dst = sQS + st * C::kKVStage;
        if (o.vec & 3) {   // a bulk copy needs a 16-byte aligned source: never issue a misaligned one
          atomicOr(p.status, ST_INTERNAL);
          *abort_flag = 1;
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(B_QF + st), 2 * C::kTileBytes + C::kVecBytes);
        load_tile_b<D>(glob ? &p.mQG : &p.mQ, glob ? 1 : p.d, o.y, w.bh, dst, bar(B_QF + st));
        load_tile_b<D>(glob ? &p.mdOG : &p.mdO, glob ? 1 : p.d, o.y, w.bh, dst + C::kTileBytes, bar(B_QF + st));
        bulk_load_1d(dst + 2 * C::kTileBytes, (glob ? p.lse2g : p.lse2) + o.vec, 512, bar(B_QF + st));
        bulk_load_1d(dst + 2 * C::kTileBytes + 512, (glob ? p.deltag : p.delta) + o.vec, 512, bar(B_QF + st));
        issued = j + 1;
      }
      mbar_wait(bar(B_KVF), 0, nullptr, kBwdDrainCap);
      for (int x = max(0, issued - 2); x < issued; ++x) mbar_wait(bar(B_QF + (x & 1)), (x >> 1) & 1, nullptr, kBwdDrainCap);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdSS = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdTS = idesc_bf16_f32(128, D, true);
    constexpr uint64_t kStage = C::kKVStage >> 4;
    const bool leader = elect_one();
    const uint64_t dK = sdesc_sw128(sK, 16, 1024), dV = sdesc_sw128(sV, 16, 1024);
    const uint64_t dQ0 = sdesc_sw128(sQS, 16, 1024), ddO0 = sdesc_sw128(sQS + C::kTileBytes, 16, 1024);
    const uint64_t dQmn0 = sdesc_sw128(sQS, 128 * 128, 1024), ddOmn0 = sdesc_sw128(sQS + C::kTileBytes, 128 * 128, 1024);
    bool ok = true;
    auto wait_or_fail = [&](int b, int parity) -> bool {
      if (__all_sync(0xffffffffu, mbar_wait(bar(b), parity, abort_flag, cap))) return true;
      if (leader) fail();
      ok = false;
      return false;
    };
    // S^T(j) = K Q(j)^T into buffer s_col(j); dP^T(j) = V dO(j)^T; then dV += P^T(j) dO(j)
    // and dK += dS^T(j) Q(j) with P^T and dS^T read from TMEM.  D = 64 issues S^T(j + 1)
    // before waiting for the elementwise warps on tile j (its buffer was last read by
    // dV(j - 1), issued before it), and dP^T(j + 1) after dV(j) and dK(j).
    auto st_mmas = [&](int j) {
      const uint64_t dq = dQ0 + (j & 1) * kStage;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
        umma_bf16_ss(tmem + s_col(j), dK + o, dq + o, kIdSS, kk > 0 ? 1u : 0u);
      }
    };
    auto dpt_mmas = [&](int j) {
      const uint64_t ddo = ddO0 + (j & 1) * kStage;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
        umma_bf16_ss(tmem + kTdP, dV + o, ddo + o, kIdSS, kk > 0 ? 1u : 0u);
      }
    };
    auto grad_mmas = [&](int j) {
      const int st = j & 1;
      const uint64_t qm = dQmn0 + st * kStage, om = ddOmn0 + st * kStage;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_bf16_ts(tmem + kTdV, tmem + s_col(j) + kk * 8 + (kk >= 4 ? 32 : 0), om + kk * 128, kIdTS,
                     (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_bf16_ts(tmem + kTdK, tmem + kTdP + kk * 8 + (kk >= 4 ? 32 : 0), qm + kk * 128, kIdTS,
                     (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit(bar(B_QE + st));
    };
    if (wait_or_fail(B_KVF, 0)) {
      if constexpr (kDB) {
        if (w.n_tiles > 0 && wait_or_fail(B_QF, 0)) {
          tc_fence_after();
          if (leader) {
            st_mmas(0);
            dpt_mmas(0);
            umma_commit(bar(B_SR));
          }
          __syncwarp();
          for (int j = 0; j < w.n_tiles; ++j) {
            const bool next = j + 1 < w.n_tiles;
            if (next) {
              if (!wait_or_fail(B_QF + ((j + 1) & 1), ((j + 1) >> 1) & 1)) break;
              tc_fence_after();
              if (leader) st_mmas(j + 1);
              __syncwarp();
            }
            if (!wait_or_fail(B_PR, j & 1)) break;
            tc_fence_after();
            if (leader) {
              grad_mmas(j);
              if (next) {
                dpt_mmas(j + 1);
                umma_commit(bar(B_SR));
              }
            }
            __syncwarp();
          }
        }
      } else {
        for (int j = 0; j < w.n_tiles; ++j) {
          const int st = j & 1;
          if (!wait_or_fail(B_QF + st, (j >> 1) & 1)) break;
          tc_fence_after();
          if (leader) {
            st_mmas(j);
            dpt_mmas(j);
            umma_commit(bar(B_SR));
          }
          __syncwarp();
          if (!wait_or_fail(B_PR, j & 1)) break;
          tc_fence_after();
          if (leader) grad_mmas(j);
          __syncwarp();
        }
      }
    }
    if (leader) umma_commit(bar(B_DONE));
    __syncwarp();
    if (!ok) mbar_wait(bar(B_DONE), 0, nullptr, kBwdDrainCap);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise warpgroups + epilogue
    // Two threads per row: warps 4..7 take columns 0..63, warps 8..11 columns 64..127 (every
    // element is independent: P and dS need only per-row and per-column constants).  Each half
    // writes its packed bf16 results inside its own S / dP columns (columns 32 h.. + 0..31).
    const int half = (warp - 4) >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tdP = tmem + lane_off + kTdP;
    bool valid;
    int u = 0, pos = 0;
    if (w.grow) {
      valid = w.gt * 128 + r < p.n_glob;
    } else {
      u = w.t0 + r;
      pos = w.c + p.d * u;
      valid = u < w.n_c;
    }
    // Global rows whose band already holds this key (Longformer): list
    // indices [g_a, g_b) of the positions in [pos - d*w_right, pos + d*w_left].
    int g_a = 0, g_b = 0;
    if (!w.grow && !p.etc && p.n_glob > 0 && valid) {
      const long long a = static_cast<long long>(pos) - static_cast<long long>(p.d) * p.wr;
      const long long b = static_cast<long long>(pos) + static_cast<long long>(p.d) * p.wl + 1;
      g_a = __ldg(p.gcount + (a < 0 ? 0 : (a > p.N ? p.N : a)));
      g_b = __ldg(p.gcount + (b < 0 ? 0 : (b > p.N ? p.N : b)));
    }
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int j = 0; j < w.n_tiles; ++j) {
      const int st = j & 1;
      const OTile o = other_tile(p, w, j);
      int lo = 0, hi = 127, ca = 0, cb = 0;
      if (o.kind == 0) {
        lo = u - p.wr - o.s0;
        hi = min(u + p.wl, o.n_c - 1) - o.s0;
      } else if (o.kind == 1) {
        hi = min(128, p.n_glob - o.g0) - 1;
        if (!w.grow && !p.etc) { ca = max(g_a - o.g0, 0); cb = min(g_b - o.g0, 128); }
      } else {
        hi = min(128, o.n_c - o.s0) - 1;
      }
      const KeepMask km = make_keep(lo, hi, ca, cb, p.gidx, o.g0, p.d, pos);
      // the stage's lse2 / delta vectors, and S^T, dP^T
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_QF + st), (j >> 1) & 1, abort_flag, cap)) ||
          !__all_sync(0xffffffffu, mbar_wait(bar(B_SR), j & 1, abort_flag, cap))) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + s_col(j);
      const float* vl = reinterpret_cast<const float*>(smem + 2 * C::kTileBytes + st * C::kKVStage + 2 * C::kTileBytes);
      const float* vd = vl + 128;
#pragma unroll 1
      for (int wd = 2 * half; wd < 2 * half + 2; ++wd) {
        uint32_t sr[32], dr[32];
        tmem_ld32_nowait(tS + 32 * wd, sr);
        tmem_ld32_nowait(tdP + 32 * wd, dr);
        tmem_wait_ld();
        const uint32_t kw = keep_word(km, wd);
        const bool full = !km.any_partial || __all_sync(0xffffffffu, kw == 0xFFFFFFFFu);
        uint32_t pkp[16], pks[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 l2 = *reinterpret_cast<const float2*>(vl + 32 * wd + 2 * i);
          const float2 dl = *reinterpret_cast<const float2*>(vd + 32 * wd + 2 * i);
          float x0, x1, p0, p1, d0, d1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), c2,
                           f2_pack(-l2.x, -l2.y)),
                    x0, x1);
          p0 = ex2_approx(x0);
          p1 = ex2_approx(x1);
          const uint64_t dd = f2_add(f2_pack(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1])),
                                     f2_pack(-dl.x, -dl.y));
          f2_unpack(f2_mul(f2_pack(p0, p1), dd), d0, d1);
          if (!full) {
            const bool k0 = (kw >> (2 * i)) & 1u, k1 = (kw >> (2 * i + 1)) & 1u;
            p0 = k0 ? p0 : 0.f;
            p1 = k1 ? p1 : 0.f;
            d0 = k0 ? d0 : 0.f;
            d1 = k1 ? d1 : 0.f;
          }
          pkp[i] = pack_bf16x2(p0, p1);
          pks[i] = pack_bf16x2(d0, d1);
        }
        tmem_st16_nowait(tS + 16 * wd + 32 * half, pkp);    // P^T over this half's S^T columns, already read
        tmem_st16_nowait(tdP + 16 * wd + 32 * half, pks);   // dS^T over this half's dP^T columns, already read
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PR));
    }
    if (ok) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DONE), 0, abort_flag, cap))) {
        fail();
      } else {
        tc_fence_after();
        const uint32_t tdV = tmem + lane_off + kTdV, tdK = tmem + lane_off + kTdK;
        if (w.grow) {
          const size_t prow = (static_cast<size_t>(w.bh) * p.n_glob + w.gt * 128 + r) * p.ns_stride + w.x0 / p.split;
          const int c0 = half * (D / 64), c1 = c0 + D / 64;   // this half's 32-column chunks
          store_partial_rows<D>(p.part_a + prow * D, tdK, p.part_b + prow * D, tdV, valid, c0, c1);
        } else {
          // staging: the first stage's Q tile (every load has landed and been consumed)
          const uint32_t stage = sQS + (warp - 4) * 4096;
          const int y0 = w.c + p.d * (w.t0 + 32 * (warp & 3));
          if (D == 128 || half == 0) {
            store_rows_tma<D>(&p.sA, stage, tdK, p.scale, y0, w.bh, lane, half);
            store_rows_tma<D>(&p.sB, stage, tdV, 1.f, y0, w.bh, lane, half);
          }
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

// ======================================================================== prep and reduce

// One thread per (b, h, row): Delta = sum_d dO * O and lse2 = LSE * log2(e),
// stored class-major; rows of global positions also go to the gathered
// global-side arrays (with their dO row).  ETC: the global-side rows come
// from their own inputs (rows bh * N .. are the long input, then the global
// input's rows follow in the row index).
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdPrepParams p) {
  grid_dep_launch();
  // one thread per row: Delta = <dO, O> with 16-byte loads, LSE * log2(e), written class-major
  const long long n_main = static_cast<long long>(p.BH) * p.N;
  const long long n_rows = n_main + (p.etc ? static_cast<long long>(p.BH) * p.n_glob : 0);
  const int q8 = p.D / 8;
  for (long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; row < n_rows;
       row += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool gside = row >= n_main;   // ETC global input row
    int bh, i;
    const __nv_bfloat16 *o, *dO;
    float lse;
    if (!gside) {
      bh = static_cast<int>(row / p.N);
      i = static_cast<int>(row - static_cast<long long>(bh) * p.N);
      o = p.out + row * p.D;
      dO = p.dout + row * p.D;
      lse = p.lse[row];
    } else {
      const long long g = row - n_main;
      bh = static_cast<int>(g / p.n_glob);
      i = static_cast<int>(g - static_cast<long long>(bh) * p.n_glob);
      o = p.out_g + g * p.D;
      dO = p.dout_g + g * p.D;
      lse = p.lse_g[g];
    }
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
    for (int x = 0; x < q8; ++x) {
      const uint4 va = __ldg(reinterpret_cast<const uint4*>(o) + x), vb = __ldg(reinterpret_cast<const uint4*>(dO) + x);
      const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
        const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
        a0 = fmaf(fa.x, fb.x, a0);
        a1 = fmaf(fa.y, fb.y, a1);
      }
    }
    const float acc = a0 + a1;
    const float l2 = lse * kLog2e;
    if (gside) {
      p.lse2g[static_cast<size_t>(bh) * p.gpad + i] = l2;
      p.deltag[static_cast<size_t>(bh) * p.gpad + i] = acc;
      continue;
    }
    const int d = p.dil[bh % p.H];
    const int M = bwd_class_stride(p.N, d);
    const int cls = i % d;
    const size_t ix = static_cast<size_t>(bh) * p.CM + static_cast<size_t>(cls) * M + (i - cls) / d;
    p.lse2[ix] = l2;
    p.delta[ix] = acc;
    if (p.gidx != nullptr) {
      const int gi = __ldg(p.gcount + i);
      if (__ldg(p.gcount + i + 1) != gi) {   // position i is global number gi
        p.lse2g[static_cast<size_t>(bh) * p.gpad + gi] = l2;
        p.deltag[static_cast<size_t>(bh) * p.gpad + gi] = acc;
        uint4* dst = reinterpret_cast<uint4*>(p.dog + (static_cast<size_t>(bh) * p.n_glob + gi) * p.D);
        for (int x = 0; x < q8; ++x) dst[x] = __ldg(reinterpret_cast<const uint4*>(dO) + x);
      }
    }
  }
}

// One block per (b, h, global row): sums the partials over the splits,
// scales, rounds to bf16 and writes the row (scattered to its position).
__global__ void bwd_reduce_kernel(const BwdReduceParams p) {
  grid_dep_wait();
  const long long row = blockIdx.x;
  const int bh = static_cast<int>(row / p.n_glob), r = static_cast<int>(row % p.n_glob);
  const int pos = p.gidx ? p.gidx[r] : r;
  if (pos < 0 || pos >= p.n_rows_out) return;
  for (int col = threadIdx.x; col < p.D; col += blockDim.x) {
    float a = 0.f, b = 0.f;
    for (int s = 0; s < p.n_splits; ++s) {
      const size_t ix = (static_cast<size_t>(row) * p.n_splits + s) * p.D + col;
      a += p.part_a[ix];
      if (p.part_b) b += p.part_b[ix];
    }
    const size_t o = (static_cast<size_t>(bh) * p.n_rows_out + pos) * p.D + col;
    reinterpret_cast<__nv_bfloat16*>(p.out_a)[o] = __float2bfloat16_rn(a * p.scale_a);
    if (p.out_b) reinterpret_cast<__nv_bfloat16*>(p.out_b)[o] = __float2bfloat16_rn(b * p.scale_b);
  }
}

template <int D>
cudaError_t set_smem_attrs() {
  cudaError_t e = cudaFuncSetAttribute(bwd_q_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kQTotal);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bwd_kv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kKVTotal);
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdPrepParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.BH) * p.N + (p.etc ? static_cast<long long>(p.BH) * p.n_glob : 0);
  long long blocks = (rows + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  if (blocks < 1) blocks = 1;
  bwd_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
  return cudaGetLastError();
}

namespace {
// Shared-memory attributes are per device: set once for each (device, D).
std::atomic<unsigned> g_bwd_attr_done[64];
}

static cudaError_t ensure_bwd_attrs(int D) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned bit = D == 64 ? 1u : 2u;
  if (g_bwd_attr_done[dev].load() & bit) return cudaSuccess;
  e = D == 64 ? set_smem_attrs<64>() : set_smem_attrs<128>();
  if (e == cudaSuccess) g_bwd_attr_done[dev].fetch_or(bit);
  return e;
}

cudaError_t launch_bwd_q(const BwdParams& p, cudaStream_t s) {
  const long long units = static_cast<long long>(p.n_grow) + p.n_band;
  if (units <= 0) return cudaSuccess;
  cudaError_t e = ensure_bwd_attrs(p.D);
  if (e != cudaSuccess) return e;
  if (p.D == 64)
    return launch_kernel(bwd_q_kernel<64>, dim3(static_cast<unsigned>(units)), dim3(kBwdThreads), BwdCfg<64>::kQTotal, s,
                         true, p);
  return launch_kernel(bwd_q_kernel<128>, dim3(static_cast<unsigned>(units)), dim3(kBwdThreads), BwdCfg<128>::kQTotal, s,
                       true, p);
}

cudaError_t launch_bwd_kv(const BwdParams& p, cudaStream_t s) {
  const long long units = static_cast<long long>(p.n_grow) + p.n_band;
  if (units <= 0) return cudaSuccess;
  cudaError_t e = ensure_bwd_attrs(p.D);
  if (e != cudaSuccess) return e;
  if (p.D == 64)
    return launch_kernel(bwd_kv_kernel<64>, dim3(static_cast<unsigned>(units)), dim3(kBwdThreads), BwdCfg<64>::kKVTotal,
                         s, true, p);
  return launch_kernel(bwd_kv_kernel<128>, dim3(static_cast<unsigned>(units)), dim3(kBwdThreads), BwdCfg<128>::kKVTotal,
                       s, true, p);
}

cudaError_t launch_bwd_reduce(const BwdReduceParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.BH) * p.n_glob;
  if (rows <= 0) return cudaSuccess;
  return launch_kernel(bwd_reduce_kernel, dim3(static_cast<unsigned>(rows)), dim3(128), 0, s, true, p);
}

}  // namespace lg
