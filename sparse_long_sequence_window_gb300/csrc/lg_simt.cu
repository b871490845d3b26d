// fp32 window + dilation + global attention forward on the CUDA cores.
//
// This is the exact-precision path (fp32 inputs, fp32 FMA, no TF32).  The
// keys are those of "Longformer: The Long-Document Transformer", section
// 3.4, "Sliding Window Attention", "Dilated Sliding Window Attention" and
// "Global Attention": a band row takes the keys i + d*t inside [0, N), then
// the global keys that are not already in its band; a global query row takes
// every key.  For the ETC call ("ETC: Encoding Long and Structured Inputs in
// Transformers", section 3.4, "Global-Local Attention") a long row takes its
// |i - j| <= r long keys and the G global keys; a global row takes all G + L
// keys.  Longformer with separate global projections ("Separate Linear
// Projections for Local vs. Global Attention"): a global row is q_glob[i]
// against k_glob, v_glob of every token; the other rows use q, k, v.
//
// Every block stages its keys in shared memory and computes from there
// (below): band rows in tiles of eight consecutive steps of one residue class,
// one row per warp; a global row in one block whose warps split each staged
// pass of keys.  Each warp keeps an online softmax (running max m and sum l)
// over chunks of 32 keys, merged across the lanes with warp shuffles.
#include <math.h>

#include "lg_internal.h"

namespace lg {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ bool is_global_pos(const int* gidx, int n, int pos) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = __ldg(gidx + mid);
    if (v == pos) return true;
    if (v < pos) lo = mid + 1; else hi = mid - 1;
  }
  return false;
}

__device__ __forceinline__ bool in_band(int i, int j, int d, int wl, int wr) {
  const int diff = j - i;
  if (diff % d != 0) return false;
  const int t = diff / d;
  return t >= -wl && t <= wr;
}

// ---------------------------------------------------------------- band-row tiles
//
// A band tile is kTileRows consecutive steps t0.. of one residue class c of
// one (b, h), one row per warp.  The block stages the keys of the rows'
// windows (class steps [t0 - wl, t0 + kTileRows - 1 + wr]), and then the
// global keys, in shared memory, simt_super_keys(D) keys at a time, with
// eight independent 16-byte loads per thread in flight (four of K, four of V): K row-major with rows
// padded by four floats (lane j's 16-byte reads of key j fall in distinct
// banks) and V row-major.  Each warp then runs its row's online softmax over
// chunks of 32 staged keys: one key per lane for the scores (16-byte loads of
// q and k), one 16-byte group of output columns per lane for P V.

constexpr int kTileRows = kWarps;

__host__ __device__ inline int simt_super_keys(int D) {
  const int k = (12288 / D) / 32 * 32;   // K and V of a pass in about 96 KB
  return k > 256 ? 256 : k;
}

size_t simt_band_smem(int D) {
  const int S = simt_super_keys(D);
  return static_cast<size_t>(S * (D + 4) + S * D + kTileRows * D) * sizeof(float);
}

struct RowPart4 {
  float m, l;
  float4 o;       // unnormalised output, columns 4 lane .. 4 lane + 3
};

// Online softmax of one row over n staged keys (chunks of 32); member(k) says
// whether staged key k belongs to the row.
template <typename Member>
__device__ __forceinline__ void staged_keys(RowPart4& rp, const float4* ks, const float4* vs, const float4* qs, int n,
                                            int D, float scale, int lane, Member member) {
  const int q4 = D / 4;
  for (int sub = 0; sub < n; sub += 32) {
    const int k = sub + lane;
    const bool mem = k < n && member(k);
    if (!__any_sync(0xffffffffu, mem)) continue;
    float s = -INFINITY;
    if (mem) {
      const float4* kr = ks + k * (q4 + 1);
      float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
      for (int x = 0; x < q4; ++x) {
        const float4 qv = qs[x], kv = kr[x];
        a0 = fmaf(qv.x, kv.x, a0);
        a1 = fmaf(qv.y, kv.y, a1);
        a0 = fmaf(qv.z, kv.z, a0);
        a1 = fmaf(qv.w, kv.w, a1);
      }
      s = (a0 + a1) * scale;
    }
    const float m_new = fmaxf(rp.m, warp_max(s));
    const float corr = expf(rp.m - m_new);
    const float pj = mem ? expf(s - m_new) : 0.f;
    rp.l = rp.l * corr + warp_sum(pj);
    rp.o.x *= corr; rp.o.y *= corr; rp.o.z *= corr; rp.o.w *= corr;
    // P V without branches on the weights (a key outside the row has weight 0,
    // and every staged row is readable), so consecutive keys' shuffles and
    // loads issue back to back
    const int last = min(32, n - sub);
    const int col = lane < q4 ? lane : 0;
#pragma unroll 8
    for (int src = 0; src < last; ++src) {
      const float pb = __shfl_sync(0xffffffffu, pj, src);
      const float4 v = vs[(sub + src) * q4 + col];
      rp.o.x = fmaf(pb, v.x, rp.o.x);
      rp.o.y = fmaf(pb, v.y, rp.o.y);
      rp.o.z = fmaf(pb, v.z, rp.o.z);
      rp.o.w = fmaf(pb, v.w, rp.o.w);
    }
    rp.m = m_new;
  }
}

// Stages keys [0, n) of a pass: row(k) is the key's row in ksrc / vsrc.
template <typename Row>
__device__ __forceinline__ void stage_keys(float4* ks, float4* vs, const float* ksrc, const float* vsrc, int n, int D,
                                           Row row) {
  constexpr int kBatch = 4;
  const int q4 = D / 4;
  const int per = blockDim.x / q4;                       // keys per sweep of the block
  const int k_off = threadIdx.x / q4, x4 = threadIdx.x - k_off * q4;
  if (k_off >= per) return;
  for (int k = k_off; k < n; k += kBatch * per) {
    float4 kv[kBatch], vv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int kk = k + u * per;
      if (kk < n) {
        const size_t r = static_cast<size_t>(row(kk)) * D;
        kv[u] = __ldg(reinterpret_cast<const float4*>(ksrc + r) + x4);
        vv[u] = __ldg(reinterpret_cast<const float4*>(vsrc + r) + x4);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int kk = k + u * per;
      if (kk < n) {
        ks[kk * (q4 + 1) + x4] = kv[u];
        vs[kk * q4 + x4] = vv[u];
      }
    }
  }
}

template <bool ETC>
__device__ void band_tile(const SimtParams& p, int tile, float* dyn) {
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, D = p.D;
  const int per_batch = p.tile_start[p.H];
  const int b = tile / per_batch;
  int rem = tile - b * per_batch;
  int h = 0;
  while (h + 1 < p.H && p.tile_start[h + 1] <= rem) ++h;
  rem -= p.tile_start[h];
  const int d = ETC ? 1 : p.dil[h];
  int c = 0, n_c = 0, t0 = 0;
  for (c = 0; c < d; ++c) {
    n_c = (N - c + d - 1) / d;
    const int nt = (n_c + kTileRows - 1) / kTileRows;
    if (rem < nt) { t0 = rem * kTileRows; break; }
    rem -= nt;
  }
  const int bh = b * p.H + h;
  const int S = simt_super_keys(D);
  float4* ks = reinterpret_cast<float4*>(dyn);
  float4* vs = ks + S * (D / 4 + 1);
  float4* qs = vs + S * (D / 4) + wib * (D / 4);
  const int t = t0 + wib;
  const int i = c + d * t;
  bool active = t < n_c;
  if (active && !ETC && p.n_glob > 0 && is_global_pos(p.gidx, p.n_glob, i)) active = false;   // a global-row block's
  if (active && lane < D / 4)
    qs[lane] = __ldg(reinterpret_cast<const float4*>(p.q + (static_cast<size_t>(bh) * N + i) * D) + lane);
  const int r_lo = max(0, t - p.wl), r_hi = min(n_c - 1, t + p.wr);
  RowPart4 rp;
  rp.m = -INFINITY;
  rp.l = 0.f;
  rp.o = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* kb = p.k + static_cast<size_t>(bh) * N * D;
  const float* vb = p.v + static_cast<size_t>(bh) * N * D;
  // band keys: class steps [lo, hi] of the tile's windows
  const int lo = max(0, t0 - p.wl), hi = min(n_c - 1, t0 + kTileRows - 1 + p.wr);
  for (int k0 = lo; k0 <= hi; k0 += S) {
    const int n = min(S, hi - k0 + 1);
    __syncthreads();   // the previous pass is no longer read (and qs is written)
    stage_keys(ks, vs, kb, vb, n, D, [&](int k) { return c + d * (k0 + k); });
    __syncthreads();
    if (active)
      staged_keys(rp, ks, vs, qs, n, D, p.scale, lane, [&](int k) { return k0 + k >= r_lo && k0 + k <= r_hi; });
  }
  // global keys (Longformer: the positions outside the row's band; ETC: the separate global input)
  for (int g0 = 0; g0 < p.n_glob; g0 += S) {
    const int n = min(S, p.n_glob - g0);
    __syncthreads();
    if (ETC) {
      stage_keys(ks, vs, p.kg + static_cast<size_t>(bh) * p.n_glob * D, p.vg + static_cast<size_t>(bh) * p.n_glob * D,
                 n, D, [&](int k) { return g0 + k; });
    } else {
      // a position outside [0, N) (a bad list, reported by the prep kernel) stages row 0 and is no key
      stage_keys(ks, vs, kb, vb, n, D, [&](int k) {
        const int pos = __ldg(p.gidx + g0 + k);
        return (pos >= 0 && pos < N) ? pos : 0;
      });
    }
    __syncthreads();
    if (active)
      staged_keys(rp, ks, vs, qs, n, D, p.scale, lane, [&](int k) {
        if (ETC) return true;
        const int pos = __ldg(p.gidx + g0 + k);
        return pos >= 0 && pos < N && !in_band(i, pos, d, p.wl, p.wr);
      });
  }
  if (active) {
    const float inv_l = 1.f / rp.l;
    if (lane < D / 4)
      reinterpret_cast<float4*>(p.out + (static_cast<size_t>(bh) * N + i) * D)[lane] =
          make_float4(rp.o.x * inv_l, rp.o.y * inv_l, rp.o.z * inv_l, rp.o.w * inv_l);
    if (lane == 0) p.lse[static_cast<size_t>(bh) * N + i] = rp.m + logf(rp.l);
  }
}

// A global row (one block): every key of its list, staged pass after pass as
// for the band tiles; warp w takes the w-th eighth of each pass, and the eight
// partial (m, l, O) are combined by their softmax denominators ("LONGNET:
// Scaling Transformers to 1,000,000,000 Tokens", section 3.4, "Mixture of
// Dilated Attentions": one joint softmax over the union of the parts).
// Longformer: the keys are every position, with the global rows' own
// projections; ETC: the G global keys, then the L long keys.
template <bool ETC>
__device__ void grow_row(const SimtParams& p, int blk, float* dyn) {
  __shared__ float pm[kWarps], pl[kWarps];
  __shared__ float4 po[kWarps][32];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, D = p.D;
  const int bh = blk / p.n_glob;
  const int gi = blk % p.n_glob;
  int i;
  const float* qrow;
  if (ETC) {
    i = gi;
    qrow = p.qg + (static_cast<size_t>(bh) * p.n_glob + gi) * D;
  } else {
    i = __ldg(p.gidx + gi);
    if (i < 0 || i >= N) return;   // a bad list is reported by the prep kernel; nothing is written
    qrow = p.qgl + (static_cast<size_t>(bh) * N + i) * D;   // the global rows' query projection
  }
  const int S = simt_super_keys(D);
  float4* ks = reinterpret_cast<float4*>(dyn);
  float4* vs = ks + S * (D / 4 + 1);
  float4* qs = vs + S * (D / 4);   // the row's query (one copy for the block)
  if (threadIdx.x < D / 4) qs[threadIdx.x] = __ldg(reinterpret_cast<const float4*>(qrow) + threadIdx.x);
  RowPart4 rp;
  rp.m = -INFINITY;
  rp.l = 0.f;
  rp.o = make_float4(0.f, 0.f, 0.f, 0.f);
  const long long n_keys = ETC ? static_cast<long long>(p.n_glob) + N : N;
  const float* kl = (ETC ? p.k : p.kgl) + static_cast<size_t>(bh) * N * D;
  const float* vl = (ETC ? p.v : p.vgl) + static_cast<size_t>(bh) * N * D;
  for (long long k0 = 0; k0 < n_keys; k0 += S) {
    const int n = static_cast<int>(n_keys - k0 < S ? n_keys - k0 : S);
    __syncthreads();
    if (ETC && k0 < p.n_glob) {
      // a pass may straddle the global and long keys: stage the two parts separately
      const int ng = min(n, p.n_glob - static_cast<int>(k0));
      stage_keys(ks, vs, p.kg + static_cast<size_t>(bh) * p.n_glob * D, p.vg + static_cast<size_t>(bh) * p.n_glob * D,
                 ng, D, [&](int k) { return static_cast<int>(k0) + k; });
      if (n > ng)
        stage_keys(ks + ng * (D / 4 + 1), vs + ng * (D / 4), kl, vl, n - ng, D, [&](int k) { return k; });
    } else {
      const int first = static_cast<int>(k0 - (ETC ? p.n_glob : 0));
      stage_keys(ks, vs, kl, vl, n, D, [&](int k) { return first + k; });
    }
    __syncthreads();
    const int slice = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
    const int s_lo = wib * slice, s_hi = min(n, s_lo + slice);
    if (s_lo < s_hi)
      staged_keys(rp, ks + s_lo * (D / 4 + 1), vs + s_lo * (D / 4), qs, s_hi - s_lo, D, p.scale, lane,
                  [](int) { return true; });
  }
  if (lane == 0) { pm[wib] = rp.m; pl[wib] = rp.l; }
  po[wib][lane] = rp.o;
  __syncthreads();
  if (wib != 0) return;
  float m = -INFINITY;
  for (int w = 0; w < kWarps; ++w) m = fmaxf(m, pm[w]);
  float l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int w = 0; w < kWarps; ++w) {
    const float f = pm[w] == -INFINITY ? 0.f : expf(pm[w] - m);
    l += f * pl[w];
    const float4 x = po[w][lane];
    o.x = fmaf(f, x.x, o.x); o.y = fmaf(f, x.y, o.y); o.z = fmaf(f, x.z, o.z); o.w = fmaf(f, x.w, o.w);
  }
  const float inv_l = 1.f / l;
  float* orow = ETC ? p.out_g + (static_cast<size_t>(bh) * p.n_glob + i) * D : p.out + (static_cast<size_t>(bh) * N + i) * D;
  float* lrow = ETC ? p.lse_g + static_cast<size_t>(bh) * p.n_glob + i : p.lse + static_cast<size_t>(bh) * N + i;
  if (lane < D / 4) reinterpret_cast<float4*>(orow)[lane] = make_float4(o.x * inv_l, o.y * inv_l, o.z * inv_l, o.w * inv_l);
  if (lane == 0) *lrow = m + logf(l);
}

// Blocks [0, n_grow_blocks): one global row each.  The other blocks: band
// tiles of eight rows (a Longformer row that is global is left to its
// global-row block).
template <bool ETC>
__global__ void __launch_bounds__(kWarps * 32, 2) simt_attn_kernel(const SimtParams p, int n_grow_blocks) {
  extern __shared__ float4 dyn4[];
  float* dyn = reinterpret_cast<float*>(dyn4);
  if (!ETC) {
    // the global list must be strictly increasing inside [0, N); every read of it is guarded, so
    // the other blocks need not wait for this check
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < p.n_glob; r += gridDim.x * blockDim.x) {
      const int pos = __ldg(p.gidx + r);
      if (pos < 0 || pos >= p.N || (r > 0 && __ldg(p.gidx + r - 1) >= pos)) atomicOr(p.status, ST_GLOBAL_IDX);
    }
  }
  if (static_cast<int>(blockIdx.x) < n_grow_blocks) grow_row<ETC>(p, static_cast<int>(blockIdx.x), dyn);
  else band_tile<ETC>(p, static_cast<int>(blockIdx.x) - n_grow_blocks, dyn);
}

}  // namespace

cudaError_t launch_simt(const SimtParams& p_in, cudaStream_t s) {
  SimtParams p = p_in;
  long long per_batch = 0;
  for (int h = 0; h < p.H; ++h) {
    p.tile_start[h] = static_cast<int>(per_batch);
    const int d = p.etc ? 1 : p.dil[h];
    for (int c = 0; c < d && c < p.N; ++c) per_batch += ((p.N - c + d - 1) / d + kTileRows - 1) / kTileRows;
    if (per_batch > 0x3fffffffLL) return cudaErrorInvalidValue;
  }
  p.tile_start[p.H] = static_cast<int>(per_batch);
  const long long grow_blocks = static_cast<long long>(p.BH) * p.n_glob;
  const long long blocks = grow_blocks + (p.BH / p.H) * per_batch;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t smem = simt_band_smem(p.D);
  cudaError_t e = p.etc ? cudaFuncSetAttribute(simt_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem))
                        : cudaFuncSetAttribute(simt_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (p.etc)
    simt_attn_kernel<true><<<static_cast<unsigned>(blocks), kWarps * 32, smem, s>>>(p, static_cast<int>(grow_blocks));
  else
    simt_attn_kernel<false><<<static_cast<unsigned>(blocks), kWarps * 32, smem, s>>>(p, static_cast<int>(grow_blocks));
  return cudaGetLastError();
}

}  // namespace lg
