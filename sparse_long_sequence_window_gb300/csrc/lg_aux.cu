// Support kernels of the bf16 path:
//  * prep: checks that the global positions are strictly increasing and inside
//    [0, N) (a bad list sets a status bit; nothing outside the tensors is
//    touched), gathers the global tokens' q, k, v rows into contiguous
//    [BH, g, D] buffers that the tensor-core kernel reads with TMA, and
//    tabulates gcount[x] = number of global positions below x for x in
//    [0, N] (one binary search per entry), so that a query row finds the
//    global keys inside its band with two loads.
//  * merge: combines the partial softmax statistics of the global-query rows
//    over the key splits.  With m = max_p m_p: l = sum_p 2^{m_p - m} l_p,
//    O = sum_p 2^{m_p - m} acc_p / l, LSE = (m + log2 l) ln 2 (statistics are
//    kept in log2 units).  This is the softmax-denominator weighting of
//    "LONGNET: Scaling Transformers to 1,000,000,000 Tokens", section 3.4,
//    "Mixture of Dilated Attentions", which equals one joint softmax over the
//    union of the key splits (see merge_block_kernel and merge_warp_kernel).
#include <math.h>

#include "lg_internal.h"

namespace lg {
namespace {

__global__ void prep_kernel(const PrepParams p) {
  grid_dep_launch();   // the next kernel of the call may start
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthreads = gridDim.x * blockDim.x;
  for (int r = tid; r < p.n_glob; r += nthreads) {
    const int pos = p.gidx[r];
    bool bad = pos < 0 || pos >= p.N;
    if (r > 0 && p.gidx[r - 1] >= pos) bad = true;
    if (bad) atomicOr(p.status, ST_GLOBAL_IDX);
  }
  if (p.gcount != nullptr) {
    for (int x = tid; x <= p.N; x += nthreads) {
      int lo = 0, hi = p.n_glob;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (p.gidx[mid] < x) lo = mid + 1; else hi = mid;
      }
      p.gcount[x] = lo;
    }
  }
  if (p.q == nullptr) return;
  const int lane = threadIdx.x & 31;
  const int chunks = p.D / 8;  // 16-byte pieces of a row
  const long long total = static_cast<long long>(p.BH) * p.n_glob;
  for (long long wid = tid >> 5; wid < total; wid += nthreads >> 5) {
    const int bh = static_cast<int>(wid / p.n_glob);
    const int r = static_cast<int>(wid % p.n_glob);
    const int pos = p.gidx[r];
    const bool ok = pos >= 0 && pos < p.N;
    if (lane < chunks) {
      const size_t src = (static_cast<size_t>(bh) * p.N + (ok ? pos : 0)) * p.D + lane * 8;
      const size_t dst = (static_cast<size_t>(bh) * p.n_glob + r) * p.D + lane * 8;
      const uint4 zero = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(p.qg + dst) = ok ? *reinterpret_cast<const uint4*>(p.q + src) : zero;
      *reinterpret_cast<uint4*>(p.kg + dst) = ok ? *reinterpret_cast<const uint4*>(p.k + src) : zero;
      *reinterpret_cast<uint4*>(p.vg + dst) = ok ? *reinterpret_cast<const uint4*>(p.v + src) : zero;
    }
  }
}

// Many partials per row (long sequences): one block of 128 threads per global row.  Pass 1: the row's maximum and
// sum over the partials (threads stride over the partials, block
// reductions).  Pass 2: the weights 2^(m_p - m) of a chunk of partials go to
// shared memory and each thread accumulates one output column over the
// chunk (for D = 64, two groups of threads take alternate partials and add
// up at the end), so the loads of consecutive partials are independent.
constexpr int kMergeThreads = 128;
constexpr int kMergeChunk = 1024;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_block_kernel(const MergeParams p, int bf16_out) {
  constexpr int G = kMergeThreads / D;  // thread groups over the partials
  __shared__ float wgt[kMergeChunk];
  __shared__ float red[kMergeThreads / 32];
  __shared__ float part[G > 1 ? G * D : 1];
  const long long row_id = blockIdx.x;
  const int bh = static_cast<int>(row_id / p.n_glob);
  const int r = static_cast<int>(row_id % p.n_glob);
  const int tid = threadIdx.x, lane = tid & 31, wrp = tid >> 5;
  grid_dep_wait();     // the partials are written by the tensor-core kernel before this one
  const size_t base = static_cast<size_t>(row_id) * p.n_splits;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + base;

  float m = -INFINITY;
  for (int s = tid; s < p.n_splits; s += kMergeThreads) m = fmaxf(m, ml[s].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[wrp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float l = 0.f;
  for (int s = tid; s < p.n_splits; s += kMergeThreads) {
    const float2 v = ml[s];
    if (v.x != -INFINITY) l += exp2f(v.x - m) * v.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) red[wrp] = l;
  __syncthreads();
  l = red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) l += red[w];

  const int col = tid % D, grp = tid / D;
  float acc = 0.f;
  for (int c0 = 0; c0 < p.n_splits; c0 += kMergeChunk) {
    const int n = min(kMergeChunk, p.n_splits - c0);
    __syncthreads();
    for (int s = tid; s < n; s += kMergeThreads) {
      const float2 v = ml[c0 + s];
      wgt[s] = (v.x == -INFINITY) ? 0.f : exp2f(v.x - m);  // empty partials hold no sums
    }
    __syncthreads();
    const float* a = p.part_acc + (base + c0) * D + col;
#pragma unroll 4
    for (int s = grp; s < n; s += G) {
      const float wv = wgt[s];
      if (wv != 0.f) acc = fmaf(wv, a[static_cast<size_t>(s) * D], acc);
    }
  }
  if (G > 1) {
    part[grp * D + col] = acc;
    __syncthreads();
    if (grp != 0) return;
#pragma unroll
    for (int g2 = 1; g2 < G; ++g2) acc += part[g2 * D + col];
  }
  const int row = p.gidx ? p.gidx[r] : r;
  if (row < 0 || row >= p.N_out) return;
  const float inv_l = 1.f / l;
  const size_t orow = (static_cast<size_t>(bh) * p.N_out + row) * D;
  if (bf16_out) reinterpret_cast<__nv_bfloat16*>(p.out)[orow + col] = __float2bfloat16_rn(acc * inv_l);
  else reinterpret_cast<float*>(p.out)[orow + col] = acc * inv_l;
  if (col == 0) p.lse[static_cast<size_t>(bh) * p.N_out + row] = (m + log2f(l)) * 0.6931471805599453f;
}

// Few partials per row (and many rows, as for ETC's global rows): one warp
// per global row, kMergeRows rows per block, lane i owning the D/32 adjacent
// output columns starting at i * D/32.  Pass 1 (lanes strided over the
// partials, then warp reductions): the row's maximum m and its sum l.  Pass 2:
// every lane walks the partials in order, reading each (m_p, l_p) (one address
// for the whole warp) and its own columns of acc_p (one coalesced row of D
// floats across the warp).  A partial whose split held no allowed key has
// m_p = -inf and an accumulator that was never written: it is skipped (the
// same decision in every lane).  No block-wide barrier: a row costs a few
// dependent loads, not two block reductions.
constexpr int kMergeRows = 8;
constexpr int kMergeWarpMaxParts = 8;    // above this the per-partial chain of one warp is too long

template <int D>
__global__ void __launch_bounds__(32 * kMergeRows) merge_warp_kernel(const MergeParams p, int bf16_out) {
  constexpr int C = D / 32;   // columns per lane
  static_assert(C == 2 || C == 4, "D = 64 or 128");
  const int lane = threadIdx.x & 31;
  const long long row_id = static_cast<long long>(blockIdx.x) * kMergeRows + (threadIdx.x >> 5);
  grid_dep_wait();     // the partials are written by the tensor-core kernel before this one
  if (row_id >= static_cast<long long>(p.BH) * p.n_glob) return;
  const int bh = static_cast<int>(row_id / p.n_glob);
  const int r = static_cast<int>(row_id % p.n_glob);
  const size_t base = static_cast<size_t>(row_id) * p.n_splits;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + base;

  float m = -INFINITY;
  for (int s = lane; s < p.n_splits; s += 32) m = fmaxf(m, ml[s].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
  for (int s = lane; s < p.n_splits; s += 32) {
    const float2 v = ml[s];
    if (v.x != -INFINITY) l += exp2f(v.x - m) * v.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);

  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  const float* a = p.part_acc + base * D + lane * C;
  for (int s = 0; s < p.n_splits; ++s) {
    const float2 v = ml[s];
    if (v.x == -INFINITY) continue;
    const float wv = exp2f(v.x - m);
    if constexpr (C == 2) {
      const float2 x = *reinterpret_cast<const float2*>(a + static_cast<size_t>(s) * D);
      acc[0] = fmaf(wv, x.x, acc[0]);
      acc[1] = fmaf(wv, x.y, acc[1]);
    } else {
      const float4 x = *reinterpret_cast<const float4*>(a + static_cast<size_t>(s) * D);
      acc[0] = fmaf(wv, x.x, acc[0]);
      acc[1] = fmaf(wv, x.y, acc[1]);
      acc[2] = fmaf(wv, x.z, acc[2]);
      acc[3] = fmaf(wv, x.w, acc[3]);
    }
  }
  const int row = p.gidx ? p.gidx[r] : r;
  if (row < 0 || row >= p.N_out) return;
  const float inv_l = 1.f / l;
  const size_t orow = (static_cast<size_t>(bh) * p.N_out + row) * D + lane * C;
  if (bf16_out) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + orow;
#pragma unroll
    for (int c = 0; c < C; c += 2)
      *reinterpret_cast<__nv_bfloat162*>(o + c) = __floats2bfloat162_rn(acc[c] * inv_l, acc[c + 1] * inv_l);
  } else {
    float* o = reinterpret_cast<float*>(p.out) + orow;
#pragma unroll
    for (int c = 0; c < C; ++c) o[c] = acc[c] * inv_l;
  }
  if (lane == 0) p.lse[static_cast<size_t>(bh) * p.N_out + row] = (m + log2f(l)) * 0.6931471805599453f;
}

}  // namespace

cudaError_t launch_prep(const PrepParams& p, cudaStream_t s) {
  if (p.n_glob <= 0) return cudaSuccess;
  long long work = p.q ? static_cast<long long>(p.BH) * p.n_glob * 32 : p.n_glob;
  if (p.gcount != nullptr && work < static_cast<long long>(p.N) + 1) work = static_cast<long long>(p.N) + 1;
  long long nb = (work + 255) / 256;
  int blocks = static_cast<int>(nb < 4096 ? nb : 4096);
  if (blocks < 1) blocks = 1;
  prep_kernel<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, int bf16_out, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.BH) * p.n_glob;
  if (rows <= 0) return cudaSuccess;
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.n_splits <= kMergeWarpMaxParts) {
    const unsigned blocks = static_cast<unsigned>((rows + kMergeRows - 1) / kMergeRows);
    if (p.D == 64) return launch_kernel(merge_warp_kernel<64>, dim3(blocks), dim3(32 * kMergeRows), 0, s, true, p, bf16_out);
    if (p.D == 128) return launch_kernel(merge_warp_kernel<128>, dim3(blocks), dim3(32 * kMergeRows), 0, s, true, p, bf16_out);
    return cudaErrorInvalidValue;
  }
  const unsigned blocks = static_cast<unsigned>(rows);
  if (p.D == 64) return launch_kernel(merge_block_kernel<64>, dim3(blocks), dim3(kMergeThreads), 0, s, true, p, bf16_out);
  if (p.D == 128) return launch_kernel(merge_block_kernel<128>, dim3(blocks), dim3(kMergeThreads), 0, s, true, p, bf16_out);
  return cudaErrorInvalidValue;
}

}  // namespace lg
