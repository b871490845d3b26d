// fp32 window + dilation + global attention forward on the CUDA cores.
//
// This is the exact-precision path (fp32 inputs, fp32 FMA, no TF32).  A
// row's candidate keys are enumerated in chunks of 32, one key per lane:
// band steps t (keys i + d*t inside [0, N)), then the global keys that are
// not already in the band ("Longformer: The Long-Document Transformer",
// section 3.4, "Sliding Window Attention", "Dilated Sliding Window
// Attention", "Global Attention").  A global query row takes every key.  For
// the ETC call ("ETC: Encoding Long and Structured Inputs in Transformers",
// section 3.4, "Global-Local Attention") a long row takes its |i - j| <= r
// long keys and the G global keys; a global row takes all G + L keys.  Each
// chunk updates an online softmax (running max m and sum l) merged across
// the lanes with warp shuffles.
//
// Longformer with separate global projections ("Separate Linear Projections
// for Local vs. Global Attention"): a global row is q_glob[i] against
// k_glob, v_glob of every token; the other rows use q, k, v throughout.
//
// Work split: a band row is one warp (eight rows per block).  A global row,
// which takes every key, is one block of eight warps: warp w takes the w-th
// eighth of the key list, and the block combines the eight partial
// (m, l, O) by their softmax denominators ("LONGNET: Scaling Transformers to
// 1,000,000,000 Tokens", section 3.4, "Mixture of Dilated Attentions": one
// joint softmax over the union of the parts).  In the P V step the 32 keys
// of a chunk are taken without branches (a missing key has weight 0 and
// points at a valid row), so the value loads of consecutive keys are
// independent and issue together.
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

// One query row (or, for a global row, one slice of its key list) in one warp.
struct RowPart {
  float m, l;     // running max and sum (natural-log units of the scaled logits)
  float o[4];     // unnormalised output, columns lane + 32 r
};

// Runs the online softmax of row (bh, i) over candidates [c_lo, c_hi) of its
// key list.  qs: the row's query in shared memory.
template <bool ETC>
__device__ RowPart row_part(const SimtParams& p, int bh, int i, bool grow_row, int d, long long c_lo, long long c_hi,
                            const float* qs, int lane, const float* kmain, const float* vmain) {
  const int N = p.N, D = p.D;
  int t_lo = 0, n_band = 0;
  if (!grow_row) {
    t_lo = max(-p.wl, -(i / d));
    const int t_hi = min(p.wr, (N - 1 - i) / d);
    n_band = max(0, t_hi - t_lo + 1);
  }
  const float* kl = kmain + static_cast<size_t>(bh) * N * D;
  const float* vl = vmain + static_cast<size_t>(bh) * N * D;
  const float* kgl = ETC ? p.kg + static_cast<size_t>(bh) * p.n_glob * D : nullptr;
  const float* vgl = ETC ? p.vg + static_cast<size_t>(bh) * p.n_glob * D : nullptr;
  RowPart rp;
  rp.m = -INFINITY;
  rp.l = 0.f;
#pragma unroll
  for (int r = 0; r < 4; ++r) rp.o[r] = 0.f;
  for (long long base = c_lo; base < c_hi; base += 32) {
    const long long c = base + lane;
    // key row of this lane: >= 0 long/main row, < -1 global-input row (-2 - r), -1 none
    int key = -1;
    if (c < c_hi) {
      if (grow_row) {
        if (ETC) key = (c < p.n_glob) ? -2 - static_cast<int>(c) : static_cast<int>(c - p.n_glob);
        else key = static_cast<int>(c);
      } else if (c < n_band) {
        key = i + d * (t_lo + static_cast<int>(c));
      } else {
        const int jj = static_cast<int>(c - n_band);
        if (ETC) {
          key = -2 - jj;
        } else {
          const int pos = __ldg(p.gidx + jj);
          if (pos >= 0 && pos < N && !in_band(i, pos, d, p.wl, p.wr)) key = pos;
        }
      }
    }
    float s = -INFINITY;
    if (key != -1) {
      const float* kr = key >= 0 ? kl + static_cast<size_t>(key) * D : kgl + static_cast<size_t>(-2 - key) * D;
      float acc = 0.f;
      // unrolled so that the row's loads issue together rather than one per step
#pragma unroll 8
      for (int x = 0; x < D; x += 4) {
        const float4 kv = __ldg(reinterpret_cast<const float4*>(kr + x));
        acc = fmaf(qs[x], kv.x, acc);
        acc = fmaf(qs[x + 1], kv.y, acc);
        acc = fmaf(qs[x + 2], kv.z, acc);
        acc = fmaf(qs[x + 3], kv.w, acc);
      }
      s = acc * p.scale;
    }
    const float cmax = warp_max(s);
    const float m_new = fmaxf(rp.m, cmax);
    if (m_new == -INFINITY) continue;
    const float corr = expf(rp.m - m_new);
    const float pj = (key != -1) ? expf(s - m_new) : 0.f;
    rp.l = rp.l * corr + warp_sum(pj);
#pragma unroll
    for (int r = 0; r < 4; ++r) rp.o[r] *= corr;
    // P V without branches: a missing key has weight 0 and reads row 0.
    const float* vsafe = key >= 0 ? vl + static_cast<size_t>(key) * D
                                  : (key < -1 ? vgl + static_cast<size_t>(-2 - key) * D : vl);
#pragma unroll 8
    for (int src = 0; src < 32; ++src) {
      const float pb = __shfl_sync(0xffffffffu, pj, src);
      const float* vr = reinterpret_cast<const float*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(vsafe), src));
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int x = lane + 32 * r;
        if (x < D) rp.o[r] = fmaf(pb, __ldg(vr + x), rp.o[r]);
      }
    }
    rp.m = m_new;
  }
  return rp;
}

template <bool ETC>
__device__ __forceinline__ void write_row(const SimtParams& p, int bh, int i, bool gside, const RowPart& rp, int lane) {
  const int D = p.D, N = p.N;
  const float inv_l = 1.f / rp.l;
  float* orow;
  float* lrow;
  if (ETC && gside) {
    orow = p.out_g + (static_cast<size_t>(bh) * p.n_glob + i) * D;
    lrow = p.lse_g + static_cast<size_t>(bh) * p.n_glob + i;
  } else {
    orow = p.out + (static_cast<size_t>(bh) * N + i) * D;
    lrow = p.lse + static_cast<size_t>(bh) * N + i;
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int x = lane + 32 * r;
    if (x < D) orow[x] = rp.o[r] * inv_l;
  }
  if (lane == 0) *lrow = rp.m + logf(rp.l);
}

// Blocks [0, n_grow_blocks): one global row each, its key list split over the
// eight warps.  The other blocks: eight band rows each, one per warp (a
// Longformer row that is global is left to its global-row block).
template <bool ETC>
__global__ void __launch_bounds__(kWarps * 32) simt_attn_kernel(const SimtParams p, int n_grow_blocks) {
  __shared__ float sq[kWarps][128];
  __shared__ float pm[kWarps], pl[kWarps];
  __shared__ float po[kWarps][128];
  const int wib = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = p.N, D = p.D;

  if (static_cast<int>(blockIdx.x) < n_grow_blocks) {
    // ---- one global row per block
    const int bh = blockIdx.x / p.n_glob;
    const int gi = blockIdx.x % p.n_glob;
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
    for (int x = lane; x < D; x += 32) sq[wib][x] = qrow[x];
    __syncwarp();
    const long long n_cand = ETC ? static_cast<long long>(p.n_glob) + N : N;
    const long long seg = ((n_cand + kWarps - 1) / kWarps + 31) / 32 * 32;
    const long long c_lo = wib * seg, c_hi = min(n_cand, c_lo + seg);
    const RowPart rp = row_part<ETC>(p, bh, i, true, 1, c_lo, c_hi, sq[wib], lane, ETC ? p.k : p.kgl, ETC ? p.v : p.vgl);
    if (lane == 0) {
      pm[wib] = rp.m;
      pl[wib] = rp.l;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int x = lane + 32 * r;
      if (x < D) po[wib][x] = rp.o[r];
    }
    __syncthreads();
    if (wib != 0) return;
    RowPart all;
    all.m = -INFINITY;
    for (int w = 0; w < kWarps; ++w) all.m = fmaxf(all.m, pm[w]);
    all.l = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) all.o[r] = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float f = pm[w] == -INFINITY ? 0.f : expf(pm[w] - all.m);
      all.l += f * pl[w];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int x = lane + 32 * r;
        if (x < D) all.o[r] = fmaf(f, po[w][x], all.o[r]);
      }
    }
    write_row<ETC>(p, bh, i, true, all, lane);
    return;
  }

  // ---- band rows, one per warp
  const long long row_id = static_cast<long long>(blockIdx.x - n_grow_blocks) * kWarps + wib;
  if (row_id >= static_cast<long long>(p.BH) * N) return;
  const int bh = static_cast<int>(row_id / N);
  const int i = static_cast<int>(row_id % N);
  if (!ETC && p.n_glob > 0 && is_global_pos(p.gidx, p.n_glob, i)) return;
  const int d = ETC ? 1 : p.dil[bh % p.H];
  const float* qrow = p.q + (static_cast<size_t>(bh) * N + i) * D;
  for (int x = lane; x < D; x += 32) sq[wib][x] = qrow[x];
  __syncwarp();
  const int t_lo = max(-p.wl, -(i / d));
  const int t_hi = min(p.wr, (N - 1 - i) / d);
  const long long n_cand = static_cast<long long>(max(0, t_hi - t_lo + 1)) + p.n_glob;
  const RowPart rp = row_part<ETC>(p, bh, i, false, d, 0, n_cand, sq[wib], lane, p.k, p.v);
  write_row<ETC>(p, bh, i, false, rp, lane);
}

}  // namespace

cudaError_t launch_simt(const SimtParams& p, cudaStream_t s) {
  const long long band_rows = static_cast<long long>(p.BH) * p.N;
  const long long grow_blocks = static_cast<long long>(p.BH) * p.n_glob;
  const long long blocks = grow_blocks + (band_rows + kWarps - 1) / kWarps;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.etc)
    simt_attn_kernel<true><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p, static_cast<int>(grow_blocks));
  else
    simt_attn_kernel<false><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p, static_cast<int>(grow_blocks));
  return cudaGetLastError();
}

}  // namespace lg
