// fp32 backward of window + dilation + global attention on the CUDA cores
// (fp32 FMA, no TF32): the exact-precision path of the backward pass.
//
// The chain rule of the forward's masked softmax ("Longformer: The
// Long-Document Transformer", section 3.4, "Sliding Window Attention",
// "Dilated Sliding Window Attention", "Global Attention"; "ETC: Encoding Long
// and Structured Inputs in Transformers", section 3.4, "Global-Local
// Attention"), with P recomputed from the saved LSE:
//   P_ij = exp(s q_i.k_j - LSE_i),  dP_ij = dO_i.v_j,  Delta_i = dO_i.O_i,
//   dS_ij = P_ij (dP_ij - Delta_i),
//   dQ_i = s sum_j dS_ij k_j,  dK_j = s sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i.
// One warp per query row enumerates the row's allowed keys exactly as the
// fp32 forward does (band steps, then the global keys not in the band; a
// global row takes every key), 32 keys at a time with one key per lane.  dQ
// stays in registers; dK and dV rows are accumulated with atomic adds into
// outputs the host zeroed.
#include <math.h>

#include "lg_internal.h"

namespace lg {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ bool is_global_b(const int* gidx, int n, int pos) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = __ldg(gidx + mid);
    if (v == pos) return true;
    if (v < pos) lo = mid + 1; else hi = mid - 1;
  }
  return false;
}

__device__ __forceinline__ bool in_band_b(int i, int j, int d, int wl, int wr) {
  const int diff = j - i;
  if (diff % d != 0) return false;
  const int t = diff / d;
  return t >= -wl && t <= wr;
}

// Delta_i = sum_d dO_id O_id for every query row (ETC: long rows, then global rows).
__global__ void __launch_bounds__(kWarps * 32) simt_delta_kernel(const SimtBwdParams p) {
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + wib;
  const long long n_main = static_cast<long long>(p.BH) * p.N;
  const long long n_rows = n_main + (p.etc ? static_cast<long long>(p.BH) * p.n_glob : 0);
  if (row >= n_rows) return;
  const float* o = row < n_main ? p.out + row * p.D : p.out_g + (row - n_main) * p.D;
  const float* g = row < n_main ? p.dout + row * p.D : p.dout_g + (row - n_main) * p.D;
  float acc = 0.f;
  for (int x = lane; x < p.D; x += 32) acc = fmaf(o[x], g[x], acc);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) p.delta[row] = acc;
}

template <bool ETC>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_kernel(const SimtBwdParams p) {
  __shared__ float sq[kWarps][128];
  __shared__ float sg[kWarps][128];
  const int wib = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row_id = static_cast<long long>(blockIdx.x) * kWarps + wib;
  const int N = p.N, D = p.D;
  const long long n_rows_long = static_cast<long long>(p.BH) * N;
  const long long n_rows = ETC ? n_rows_long + static_cast<long long>(p.BH) * p.n_glob : n_rows_long;
  if (row_id >= n_rows) return;

  bool grow_row;   // the query attends to every key
  int bh, i;
  if (ETC && row_id >= n_rows_long) {
    const long long g = row_id - n_rows_long;
    bh = static_cast<int>(g / p.n_glob);
    i = static_cast<int>(g % p.n_glob);
    grow_row = true;
  } else {
    bh = static_cast<int>(row_id / N);
    i = static_cast<int>(row_id % N);
    grow_row = !ETC && p.n_glob > 0 && is_global_b(p.gidx, p.n_glob, i);
  }
  const int h = bh % p.H;
  const int d = ETC ? 1 : p.dil[h];
  const bool gside = ETC && grow_row;   // an ETC global-input row
  const size_t qoff = gside ? (static_cast<size_t>(bh) * p.n_glob + i) * D : (static_cast<size_t>(bh) * N + i) * D;
  const float* qrow = (gside ? p.qg : p.q) + qoff;
  const float* grow = (gside ? p.dout_g : p.dout) + qoff;
  for (int x = lane; x < D; x += 32) {
    sq[wib][x] = qrow[x];
    sg[wib][x] = grow[x];
  }
  __syncwarp();
  const float lse = gside ? p.lse_g[static_cast<size_t>(bh) * p.n_glob + i] : p.lse[static_cast<size_t>(bh) * N + i];
  const float delta = p.delta[gside ? n_rows_long + static_cast<size_t>(bh) * p.n_glob + i
                                    : static_cast<size_t>(bh) * N + i];

  int t_lo = 0, n_band = 0;
  if (!grow_row) {
    t_lo = max(-p.wl, -(i / d));
    const int t_hi = min(p.wr, (N - 1 - i) / d);
    n_band = max(0, t_hi - t_lo + 1);
  }
  long long n_cand;
  if (grow_row) n_cand = ETC ? static_cast<long long>(p.n_glob) + N : N;
  else n_cand = static_cast<long long>(n_band) + p.n_glob;

  const size_t base_l = static_cast<size_t>(bh) * N * D;
  const size_t base_g = ETC ? static_cast<size_t>(bh) * p.n_glob * D : 0;
  float dq[4] = {0.f, 0.f, 0.f, 0.f};
  for (long long base = 0; base < n_cand; base += 32) {
    const long long c = base + lane;
    int key = -1;   // >= 0: main row; < -1: ETC global-input row (-2 - r); -1: none
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
          if (pos >= 0 && pos < N && !in_band_b(i, pos, d, p.wl, p.wr)) key = pos;
        }
      }
    }
    float pj = 0.f, ds = 0.f;
    if (key != -1) {
      const float* kr = key >= 0 ? p.k + base_l + static_cast<size_t>(key) * D : p.kg + base_g + static_cast<size_t>(-2 - key) * D;
      const float* vr = key >= 0 ? p.v + base_l + static_cast<size_t>(key) * D : p.vg + base_g + static_cast<size_t>(-2 - key) * D;
      float s = 0.f, dp = 0.f;
#pragma unroll 8
      for (int x = 0; x < D; x += 4) {
        const float4 kv = __ldg(reinterpret_cast<const float4*>(kr + x));
        const float4 vv = __ldg(reinterpret_cast<const float4*>(vr + x));
        s = fmaf(sq[wib][x], kv.x, s); s = fmaf(sq[wib][x + 1], kv.y, s);
        s = fmaf(sq[wib][x + 2], kv.z, s); s = fmaf(sq[wib][x + 3], kv.w, s);
        dp = fmaf(sg[wib][x], vv.x, dp); dp = fmaf(sg[wib][x + 1], vv.y, dp);
        dp = fmaf(sg[wib][x + 2], vv.z, dp); dp = fmaf(sg[wib][x + 3], vv.w, dp);
      }
      pj = expf(s * p.scale - lse);
      ds = pj * (dp - delta);
    }
    for (int src = 0; src < 32; ++src) {
      const int kb = __shfl_sync(0xffffffffu, key, src);
      const float pb = __shfl_sync(0xffffffffu, pj, src);
      const float db = __shfl_sync(0xffffffffu, ds, src);
      if (kb == -1) continue;
      const size_t ko = kb >= 0 ? base_l + static_cast<size_t>(kb) * D : base_g + static_cast<size_t>(-2 - kb) * D;
      const float* kr = (kb >= 0 ? p.k : p.kg) + ko;
      float* dkr = (kb >= 0 ? p.dk : p.dk_g) + ko;
      float* dvr = (kb >= 0 ? p.dv : p.dv_g) + ko;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int x = lane + 32 * r;
        if (x < D) {
          dq[r] = fmaf(db, kr[x], dq[r]);
          atomicAdd(dkr + x, p.scale * db * sq[wib][x]);
          atomicAdd(dvr + x, pb * sg[wib][x]);
        }
      }
    }
  }
  float* dqr = (gside ? p.dq_g : p.dq) + qoff;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int x = lane + 32 * r;
    if (x < D) dqr[x] = dq[r] * p.scale;
  }
}

}  // namespace

cudaError_t launch_simt_bwd(const SimtBwdParams& p, cudaStream_t s) {
  long long rows = static_cast<long long>(p.BH) * p.N;
  if (p.etc) rows += static_cast<long long>(p.BH) * p.n_glob;
  const long long blocks = (rows + kWarps - 1) / kWarps;
  if (blocks <= 0) return cudaSuccess;
  simt_delta_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.etc) simt_bwd_kernel<true><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  else simt_bwd_kernel<false><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lg
