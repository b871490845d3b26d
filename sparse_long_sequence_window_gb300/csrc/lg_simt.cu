// fp32 window + dilation + global attention forward on the CUDA cores.
//
// This is the exact-precision path (fp32 inputs, fp32 FMA, no TF32).  One
// warp owns one query row.  The row's candidate keys are enumerated in
// chunks of 32, one key per lane: band steps t (keys i + d*t inside [0, N)),
// then the global keys that are not already in the band ("Longformer: The
// Long-Document Transformer", section 3.4, "Sliding Window Attention",
// "Dilated Sliding Window Attention", "Global Attention").  A global query
// row enumerates every key.  For the ETC call ("ETC: Encoding Long and
// Structured Inputs in Transformers", section 3.4, "Global-Local Attention")
// a long row enumerates its |i - j| <= r long keys and the G global keys; a
// global row enumerates all G + L keys.  Each chunk updates an online softmax
// (running max m and sum l) merged across the lanes with warp shuffles.
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

template <bool ETC>
__global__ void __launch_bounds__(kWarps * 32) simt_attn_kernel(const SimtParams p) {
  __shared__ float sq[kWarps][128];
  const int wib = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row_id = static_cast<long long>(blockIdx.x) * kWarps + wib;
  const int N = p.N, D = p.D;
  const long long n_rows_long = static_cast<long long>(p.BH) * N;
  const long long n_rows = ETC ? n_rows_long + static_cast<long long>(p.BH) * p.n_glob : n_rows_long;
  if (row_id >= n_rows) return;

  // ---- which row, and its candidate list
  bool grow_row;  // query attends to every key
  int bh, i;
  if (ETC && row_id >= n_rows_long) {
    const long long g = row_id - n_rows_long;
    bh = static_cast<int>(g / p.n_glob);
    i = static_cast<int>(g % p.n_glob);
    grow_row = true;
  } else {
    bh = static_cast<int>(row_id / N);
    i = static_cast<int>(row_id % N);
    grow_row = !ETC && p.n_glob > 0 && is_global_pos(p.gidx, p.n_glob, i);
  }
  const int h = bh % p.H;
  const int d = ETC ? 1 : p.dil[h];
  const float* qrow = (ETC && grow_row) ? p.qg + (static_cast<size_t>(bh) * p.n_glob + i) * D
                                        : p.q + (static_cast<size_t>(bh) * N + i) * D;
  for (int x = lane; x < D; x += 32) sq[wib][x] = qrow[x];
  __syncwarp();

  // band step range of a band row
  int t_lo = 0, n_band = 0;
  if (!grow_row) {
    t_lo = max(-p.wl, -(i / d));
    const int t_hi = min(p.wr, (N - 1 - i) / d);
    n_band = max(0, t_hi - t_lo + 1);
  }
  long long n_cand;
  if (grow_row) n_cand = ETC ? static_cast<long long>(p.n_glob) + N : N;
  else n_cand = static_cast<long long>(n_band) + p.n_glob;

  const float* kl = p.k + static_cast<size_t>(bh) * N * D;
  const float* vl = p.v + static_cast<size_t>(bh) * N * D;
  const float* kgl = ETC ? p.kg + static_cast<size_t>(bh) * p.n_glob * D : nullptr;
  const float* vgl = ETC ? p.vg + static_cast<size_t>(bh) * p.n_glob * D : nullptr;

  float m = -INFINITY, l = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  for (long long base = 0; base < n_cand; base += 32) {
    const long long c = base + lane;
    // key row of this lane: >= 0 long/main row, < -1 global-input row (-2 - r), -1 none
    int key = -1;
    if (c < n_cand) {
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
      for (int x = 0; x < D; x += 4) {
        const float4 kv = *reinterpret_cast<const float4*>(kr + x);
        acc = fmaf(sq[wib][x], kv.x, acc);
        acc = fmaf(sq[wib][x + 1], kv.y, acc);
        acc = fmaf(sq[wib][x + 2], kv.z, acc);
        acc = fmaf(sq[wib][x + 3], kv.w, acc);
      }
      s = acc * p.scale;
    }
    const float cmax = warp_max(s);
    const float m_new = fmaxf(m, cmax);
    if (m_new == -INFINITY) continue;
    const float corr = expf(m - m_new);
    const float pj = (key != -1) ? expf(s - m_new) : 0.f;
    l = l * corr + warp_sum(pj);
#pragma unroll
    for (int r = 0; r < 4; ++r) o[r] *= corr;
    for (int src = 0; src < 32; ++src) {
      const float pb = __shfl_sync(0xffffffffu, pj, src);
      const int kb = __shfl_sync(0xffffffffu, key, src);
      if (pb == 0.f) continue;
      const float* vr = kb >= 0 ? vl + static_cast<size_t>(kb) * D : vgl + static_cast<size_t>(-2 - kb) * D;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int x = lane + 32 * r;
        if (x < D) o[r] = fmaf(pb, vr[x], o[r]);
      }
    }
    m = m_new;
  }

  const float inv_l = 1.f / l;
  float* orow;
  float* lrow;
  if (ETC && grow_row) {
    orow = p.out_g + (static_cast<size_t>(bh) * p.n_glob + i) * D;
    lrow = p.lse_g + static_cast<size_t>(bh) * p.n_glob + i;
  } else {
    orow = p.out + (static_cast<size_t>(bh) * N + i) * D;
    lrow = p.lse + static_cast<size_t>(bh) * N + i;
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int x = lane + 32 * r;
    if (x < D) orow[x] = o[r] * inv_l;
  }
  if (lane == 0) *lrow = m + logf(l);
}

}  // namespace

cudaError_t launch_simt(const SimtParams& p, cudaStream_t s) {
  long long rows = static_cast<long long>(p.BH) * p.N;
  if (p.etc) rows += static_cast<long long>(p.BH) * p.n_glob;
  const long long blocks = (rows + kWarps - 1) / kWarps;
  if (blocks <= 0) return cudaSuccess;
  if (p.etc) simt_attn_kernel<true><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  else simt_attn_kernel<false><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lg
