// LongNet dilated attention on the tensor-core kernel: "LONGNET: Scaling
// Transformers to 1,000,000,000 Tokens", section 3.4, "Dilated Attention:
// Core Mechanism", "Mixture of Dilated Attentions" and "Multi-Head Dilated
// Attention: Offset Mechanism".
//
// Pattern (w, r) on head h keeps the rows i w + s, i w + s + r, ... (s = h mod
// r) of every segment [i w, (i + 1) w) and runs dense attention among the
// kept rows of each segment: block-diagonal attention over the kept rows,
// which the tensor-core kernel runs in its segment mode.  Two layouts:
//  * strided (r divides w, r <= 8): the kept rows of a head are one dilation
//    residue class (c = s, stride r) and segment i is the block [i B, (i + 1)
//    B) of its steps, B = w / r; the kernel reads them in place through the
//    stride-r tensor maps and writes O_k at the rows' own positions.
//  * packed (any other r): a gather kernel packs each head's kept rows
//    segment after segment (seg_block(w, r, s) rows per full segment) into
//    dense buffers; the kernel runs with stride 1 over them and writes O_k
//    packed the same way.
// Each pattern writes its own (O_k, LSE_k) for its kept rows into the
// workspace; the mix kernel then combines the patterns of every row by their
// softmax denominators: LSE = ln sum_k exp(LSE_k) over the patterns that
// keep the row, O = sum_k exp(LSE_k - LSE) O_k (a row no pattern keeps gets
// O = 0, LSE = -inf).
#include <math.h>

#include <algorithm>

#include "lg_internal.h"

namespace lg {
namespace {

constexpr int kMaxPatterns = 16;

bool strided_layout(int w, int r) { return r <= LG_MAX_BF16_DILATION && w % r == 0; }

// Packed rows of the longest head of pattern (w, r) (heads differ by offset).
int packed_rows(int H, int N, int w, int r) {
  int m = 0;
  for (int h = 0; h < std::min(H, r); ++h) m = std::max(m, seg_class_len(N, w, r, h % r));
  return m;
}

struct GatherParams {
  const uint4* src[3];   // q, k, v [BH, N, D]
  uint4* dst[3];         // packed [BH, P, D]; rows past a head's kept rows are zero
  int H, N, P, chunks;   // chunks: 16-byte pieces of a row (D / 8)
  int w, r;
  long long total;       // BH * P * chunks
};

// One thread per 16-byte piece of a packed row of q, k and v.
__global__ void __launch_bounds__(256) longnet_gather_kernel(const GatherParams g) {
  grid_dep_launch();
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < g.total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int x = static_cast<int>(idx % g.chunks);
    const long long prow = idx / g.chunks;
    const int t_p = static_cast<int>(prow % g.P);
    const long long bh = prow / g.P;
    const int s = static_cast<int>(bh % g.H) % g.r;
    const int L = seg_block(g.w, g.r, s);
    long long pos = -1;
    if (L > 0) {
      const int seg = t_p / L;
      pos = static_cast<long long>(seg) * g.w + s + static_cast<long long>(t_p - seg * L) * g.r;
      if (pos >= g.N) pos = -1;
    }
    const long long from = (bh * g.N + pos) * g.chunks + x;
#pragma unroll
    for (int a = 0; a < 3; ++a) g.dst[a][idx] = pos >= 0 ? __ldg(g.src[a] + from) : make_uint4(0, 0, 0, 0);
  }
}

struct MixParams {
  const __nv_bfloat16* o[kMaxPatterns];   // O_k [BH, rows_k, D] (rows the pattern keeps are valid)
  const float* l[kMaxPatterns];           // LSE_k [BH, rows_k]
  int w[kMaxPatterns], r[kMaxPatterns];
  int rows[kMaxPatterns];                 // rows_k: N (strided layout) or the packed length
  int packed[kMaxPatterns];
  int n_pat, H, BH, N, D;
  __nv_bfloat16* out;
  float* lse;
};

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One thread per row and kMixCols columns (D / kMixCols threads per row,
// adjacent): the pattern membership arithmetic once per pattern in 32-bit
// integers, then kMixCols / 8 16-byte loads of the pattern's output.  The
// patterns that keep the row are merged online (running max of LSE_k).  The
// parameter block is read in place (__grid_constant__): its per-pattern arrays
// are indexed by a runtime k.  32 columns keep the accumulator at 32 registers,
// so that enough warps are resident to cover the load latency (64 columns per
// thread held 97 registers, two blocks per SM, and the kernel was
// latency-bound at a third of DRAM bandwidth).
constexpr int kMixCols = 32;

template <int D>
__global__ void __launch_bounds__(256) longnet_mix_kernel(const __grid_constant__ MixParams p) {
  grid_dep_wait();   // the patterns' kernels came before
  constexpr int kParts = D / kMixCols;
  constexpr int kVec = kMixCols / 8;   // 16-byte pieces per thread
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= static_cast<long long>(p.BH) * p.N * kParts) return;
  const int part = static_cast<int>(tid % kParts);
  const int row = static_cast<int>(tid / kParts);   // BH * N < 2^31
  const int i = row % p.N;
  const int bh = row / p.N;
  const int h = bh % p.H;
  float acc[kMixCols];
#pragma unroll
  for (int c = 0; c < kMixCols; ++c) acc[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int k = 0; k < p.n_pat; ++k) {
    const int w = p.w[k], r = p.r[k], s = h % r;
    const int seg = i / w, rel = i - seg * w - s;
    if (rel < 0 || rel % r != 0) continue;
    const long long src = p.packed[k] ? static_cast<long long>(bh) * p.rows[k] +
                                            static_cast<long long>(seg) * seg_block(w, r, s) + rel / r
                                      : row;
    const uint4* o = reinterpret_cast<const uint4*>(p.o[k] + src * D + part * kMixCols);
    uint4 v[kVec];
#pragma unroll
    for (int x = 0; x < kVec; ++x) v[x] = __ldg(o + x);
    const float lk = __ldg(p.l[k] + src);
    if (lk > m) {   // new running maximum: rescale what is accumulated
      const float f = exp2f((m - lk) * 1.4426950408889634f);
      l *= f;
#pragma unroll
      for (int c = 0; c < kMixCols; ++c) acc[c] *= f;
      m = lk;
    }
    const float wgt = exp2f((lk - m) * 1.4426950408889634f);
    l += wgt;
#pragma unroll
    for (int x = 0; x < kVec; ++x) {
      const uint32_t vw[4] = {v[x].x, v[x].y, v[x].z, v[x].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vw[e]));
        acc[8 * x + 2 * e] = fmaf(wgt, f2.x, acc[8 * x + 2 * e]);
        acc[8 * x + 2 * e + 1] = fmaf(wgt, f2.y, acc[8 * x + 2 * e + 1]);
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<long long>(row) * D + part * kMixCols);
#pragma unroll
  for (int x = 0; x < kVec; ++x)
    dst[x] = make_uint4(pack_bf16x2_rn(acc[8 * x] * inv, acc[8 * x + 1] * inv),
                        pack_bf16x2_rn(acc[8 * x + 2] * inv, acc[8 * x + 3] * inv),
                        pack_bf16x2_rn(acc[8 * x + 4] * inv, acc[8 * x + 5] * inv),
                        pack_bf16x2_rn(acc[8 * x + 6] * inv, acc[8 * x + 7] * inv));
  if (part == 0) p.lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
}

bool aligned_ln(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t rup_ln(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct LnLayout {
  size_t o[kMaxPatterns] = {}, l[kMaxPatterns] = {};
  int rows[kMaxPatterns] = {};
  bool fused = false;                 // every pattern in one tensor-core launch
  size_t gather[kMaxPatterns][3] = {};  // packed q, k, v of each packed pattern (one shared set unless fused)
  size_t units = 0, max_units = 0, total = 0;
};

// One launch for all patterns when their tensor maps fit the slots of one
// launch and the per-pattern head tables fit the launch parameters.
bool fused_call(int H, int n_pat) { return n_pat <= kMaxPatternSlots && H <= kMaxFusedHeads; }

// Work units of a launch, at most: per head and pattern ceil(rows / 256)
// (rows <= N, the pattern's kept rows of the longest head), and half as many
// again for the split tail; one pattern per launch, or all of them (fused).
LnLayout ln_layout(int BH, int H, int N, int D, int n_pat, const int32_t* seg_w, const int32_t* seg_r) {
  LnLayout w;
  w.fused = fused_call(H, n_pat);
  size_t off = kStatusBytes;
  int p_max = 0;
  size_t per_head_max = 0, per_head_sum = 0;
  for (int k = 0; k < n_pat; ++k) {
    const bool strided = strided_layout(seg_w[k], seg_r[k]);
    w.rows[k] = strided ? N : std::max(1, packed_rows(H, N, seg_w[k], seg_r[k]));
    if (!strided) p_max = std::max(p_max, w.rows[k]);
    w.o[k] = off; off += rup_ln(static_cast<size_t>(BH) * w.rows[k] * D * 2, 256);
    w.l[k] = off; off += rup_ln(static_cast<size_t>(BH) * w.rows[k] * 4, 256);
    const size_t per_head = (static_cast<size_t>(w.rows[k]) + 255) / 256;
    per_head_max = std::max(per_head_max, per_head);
    per_head_sum += per_head;
  }
  // Packed q, k, v: a set per packed pattern when fused (all are read by the
  // one launch); otherwise one set of the longest size, which every packed
  // pattern uses in turn.
  size_t shared[3] = {0, 0, 0};
  if (!w.fused && p_max > 0) {
    for (int a = 0; a < 3; ++a) {
      shared[a] = off;
      off += rup_ln(static_cast<size_t>(BH) * p_max * D * 2, 256);
    }
  }
  for (int k = 0; k < n_pat; ++k) {
    if (strided_layout(seg_w[k], seg_r[k])) continue;
    for (int a = 0; a < 3; ++a) {
      if (w.fused) {
        w.gather[k][a] = off;
        off += rup_ln(static_cast<size_t>(BH) * w.rows[k] * D * 2, 256);
      } else {
        w.gather[k][a] = shared[a];
      }
    }
  }
  w.units = off;
  const size_t per_head = w.fused ? per_head_sum : per_head_max;
  w.max_units = static_cast<size_t>(BH) * per_head + static_cast<size_t>(BH) * per_head / 2 + 1;
  off += rup_ln(w.max_units * 64, 256);
  w.total = off;
  return w;
}


lg_status check_patterns(int n_pat, const int32_t* seg_w, const int32_t* seg_r) {
  if (n_pat < 1 || seg_w == nullptr || seg_r == nullptr) return LG_ERR_INVALID_ARG;
  if (n_pat > kMaxPatterns) return LG_ERR_UNSUPPORTED;
  for (int k = 0; k < n_pat; ++k)
    if (seg_w[k] < 1 || seg_r[k] < 1) return LG_ERR_INVALID_ARG;
  return LG_OK;
}

bool shape_ok(int B, int H, int N, int D, lg_dtype dt) {
  return B >= 1 && H >= 1 && N >= 1 && dt == LG_BF16 && (D == 64 || D == 128) && H <= LG_MAX_HEADS &&
         static_cast<long long>(B) * H * N <= (1LL << 31) - 1;
}

}  // namespace
}  // namespace lg

using namespace lg;

extern "C" {

size_t lg_longnet_attn_fwd_workspace_size(int B, int H, int N, int D, int n_patterns, const int32_t* seg_w,
                                          const int32_t* seg_r, lg_dtype dt) {
  if (!shape_ok(B, H, N, D, dt) || check_patterns(n_patterns, seg_w, seg_r) != LG_OK) return 0;
  return ln_layout(B * H, H, N, D, n_patterns, seg_w, seg_r).total;
}

int64_t lg_longnet_count_pairs(int N, int n_patterns, const int32_t* seg_w, const int32_t* seg_r, int causal, int head) {
  if (N < 1 || head < 0 || (causal != 0 && causal != 1) || check_patterns(n_patterns, seg_w, seg_r) != LG_OK) return -1;
  int64_t total = 0;
  for (int k = 0; k < n_patterns; ++k) {
    const long long w = seg_w[k], r = seg_r[k], s = head % r;
    for (long long a = 0; a < N; a += w) {
      const long long end = std::min<long long>(a + w, N);
      const long long n = a + s < end ? (end - 1 - (a + s)) / r + 1 : 0;
      total += causal ? n * (n + 1) / 2 : n * n;
    }
  }
  return total;
}

lg_status lg_longnet_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, lg_dtype dt, int B,
                              int H, int N, int D, int n_patterns, const int32_t* seg_w, const int32_t* seg_r,
                              int causal, float scale, void* workspace, size_t workspace_bytes, lg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // ---- argument checks (nothing is launched on failure)
  if (B < 1 || H < 1 || N < 1 || (causal != 0 && causal != 1)) return LG_ERR_INVALID_ARG;
  if (dt != LG_BF16 && dt != LG_F32) return LG_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D, dt)) return LG_ERR_UNSUPPORTED;
  lg_status st = check_patterns(n_patterns, seg_w, seg_r);
  if (st != LG_OK) return st;
  if (!q || !k || !v || !out || !lse) return LG_ERR_INVALID_ARG;
  if (!aligned_ln(q, 16) || !aligned_ln(k, 16) || !aligned_ln(v, 16) || !aligned_ln(out, 16) || !aligned_ln(lse, 4))
    return LG_ERR_INVALID_ARG;
  const size_t need = lg_longnet_attn_fwd_workspace_size(B, H, N, D, n_patterns, seg_w, seg_r, dt);
  if (workspace == nullptr || !aligned_ln(workspace, 256) || workspace_bytes < need) return LG_ERR_WORKSPACE;
  if (!encode_fn()) return LG_ERR_CUDA;

  const int BH = B * H;
  const float s = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  const LnLayout lay = ln_layout(BH, H, N, D, n_patterns, seg_w, seg_r);
  if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) return LG_ERR_CUDA;

  // Packs pattern pk's kept rows of q, k, v into its gather buffers; src gets their addresses.
  auto gather = [&](int pk, const void* (&src)[3]) -> bool {
    GatherParams g{};
    for (int a = 0; a < 3; ++a) {
      g.src[a] = static_cast<const uint4*>(src[a]);
      g.dst[a] = reinterpret_cast<uint4*>(ws + lay.gather[pk][a]);
      src[a] = ws + lay.gather[pk][a];
    }
    g.H = H; g.N = N; g.P = lay.rows[pk]; g.chunks = D / 8; g.w = seg_w[pk]; g.r = seg_r[pk];
    g.total = static_cast<long long>(BH) * lay.rows[pk] * g.chunks;
    const long long blocks = std::min<long long>((g.total + 255) / 256, 16LL * device_sm_count());
    // plain launch: it waits for every kernel before it (the previous pattern's
    // kernel reads the shared buffers until it completes)
    return launch_kernel(longnet_gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, false, g) ==
           cudaSuccess;
  };
  // Band units of pattern (w, r) per head, prefix over the heads in hs[0..H].
  auto head_units = [&](int w, int r, bool strided, int* hs) {
    int start = 0;
    for (int h = 0; h < H; ++h) {
      const int sh = h % r;
      const int n_c = strided ? (N - sh + r - 1) / r : seg_class_len(N, w, r, sh);
      hs[h] = start;
      start += n_c > 0 ? (n_c + 2 * kTileM - 1) / (2 * kTileM) : 0;
    }
    hs[H] = start;
    return start;
  };
  auto common = [&](auto& tp) {
    tp.mapQg = tp.mapQ[0]; tp.mapKg = tp.mapK[0]; tp.mapVg = tp.mapV[0];
    tp.mapKgr = tp.mapK[0]; tp.mapVgr = tp.mapV[0];
    tp.seg_n = N;
    tp.seg_causal = causal;
    tp.status = status;
    tp.wait_cap = wait_cap_cycles();
    tp.withhold = withhold_for_test();
    tp.scale_log2 = s * 1.4426950408889634f;
    tp.BH = BH; tp.H = H; tp.D = D; tp.wl = 0; tp.wr = 0; tp.n_glob = 0; tp.etc = 0;
    tp.grow_split = 1;
    tp.units = ws + lay.units;
  };

  if (lay.fused) {
    // Every pattern in one launch, pattern k in slot k: the CTAs claim the
    // units of all patterns from one counter, so a pattern with few or
    // uneven units (the last segments' units of a causal block are the
    // longest) no longer ends its own launch on a few busy SMs.
    TcParamsLn tp{};
    tp.n_pat = n_patterns;
    long long units = 0;
    for (int pk = 0; pk < n_patterns; ++pk) {
      const int w = seg_w[pk], r = seg_r[pk];
      const bool strided = strided_layout(w, r);
      const int d = strided ? r : 1;
      const int rows = lay.rows[pk];
      const void* src[3] = {q, k, v};
      if (!strided && !gather(pk, src)) return LG_ERR_CUDA;
      if (!encode_map(&tp.mapQ[pk], src[0], D, rows, BH, d) || !encode_map(&tp.mapK[pk], src[1], D, rows, BH, d) ||
          !encode_map(&tp.mapV[pk], src[2], D, rows, BH, d) ||
          !encode_store_map(&tp.mapO[pk], ws + lay.o[pk], D, rows, BH, d))
        return LG_ERR_CUDA;
      tp.slot_dil[pk] = d;
      tp.pat_w[pk] = w; tp.pat_r[pk] = r; tp.pat_packed[pk] = strided ? 0 : 1; tp.pat_rows[pk] = rows;
      tp.pat_lse[pk] = reinterpret_cast<float*>(ws + lay.l[pk]);
      tp.pat_unit_start[pk] = static_cast<int>(units);
      units += static_cast<long long>(B) * head_units(w, r, strided, tp.pat_head_unit_start[pk]);
    }
    tp.pat_unit_start[n_patterns] = static_cast<int>(units);
    for (int sl = n_patterns; sl < kMaxPatternSlots; ++sl) {
      tp.mapQ[sl] = tp.mapQ[0]; tp.mapK[sl] = tp.mapK[0]; tp.mapV[sl] = tp.mapV[0]; tp.mapO[sl] = tp.mapO[0];
      tp.slot_dil[sl] = 1;
    }
    common(tp);
    tp.N = N;
    tp.lse = tp.pat_lse[0];
    tp.unit_counter = status + 1;
    const long long tail = tail_split(units, units);
    tp.n_tail_split = static_cast<int>(tail);
    units += tail;
    if (units > static_cast<long long>(lay.max_units)) return LG_ERR_WORKSPACE;
    if (prof_mark(stream, true) != cudaSuccess || launch_tc(tp, static_cast<int>(units), stream, true) != cudaSuccess ||
        prof_mark(stream, false) != cudaSuccess)
      return LG_ERR_CUDA;
  } else {
    for (int pk = 0; pk < n_patterns; ++pk) {
      const int w = seg_w[pk], r = seg_r[pk];
      const bool strided = strided_layout(w, r);
      const int d = strided ? r : 1;          // stride of the kernel's tensor maps
      const int rows = lay.rows[pk];          // rows of the kernel's tensors (N, or the packed length)
      const void* src[3] = {q, k, v};
      if (!strided && !gather(pk, src)) return LG_ERR_CUDA;
      TcParams tp{};
      if (!encode_map(&tp.mapQ[0], src[0], D, rows, BH, d) || !encode_map(&tp.mapK[0], src[1], D, rows, BH, d) ||
          !encode_map(&tp.mapV[0], src[2], D, rows, BH, d) ||
          !encode_store_map(&tp.mapO[0], ws + lay.o[pk], D, rows, BH, d))
        return LG_ERR_CUDA;
      for (int sl = 0; sl < kMaxSlots; ++sl) {
        tp.mapQ[sl] = tp.mapQ[0]; tp.mapK[sl] = tp.mapK[0]; tp.mapV[sl] = tp.mapV[0]; tp.mapO[sl] = tp.mapO[0];
        tp.slot_dil[sl] = d;
      }
      tp.seg_w = w; tp.seg_r = r; tp.seg_packed = strided ? 0 : 1;
      for (int h = 0; h < H; ++h) {
        tp.head_slot[h] = 0;
        tp.head_class[h] = 0;
      }
      const int start = head_units(w, r, strided, tp.head_unit_start);
      tp.band_units_per_batch = start;
      common(tp);
      tp.N = rows;
      tp.out = ws + lay.o[pk];
      tp.lse = reinterpret_cast<float*>(ws + lay.l[pk]);
      tp.unit_counter = status + 1 + pk;   // one zeroed word of the status area per launch
      const long long band_units = static_cast<long long>(B) * start;
      const long long tail = tail_split(band_units, band_units);
      tp.n_tail_split = static_cast<int>(tail);
      const long long units = band_units + tail;
      if (units > static_cast<long long>(lay.max_units)) return LG_ERR_WORKSPACE;
      // The unit table of a later pattern may not overwrite the one the previous
      // pattern's kernel reads: chained only after the memset or a gather (which
      // itself waited for that kernel).
      if (prof_mark(stream, true) != cudaSuccess ||
          launch_tc(tp, static_cast<int>(units), stream, pk == 0 || !strided) != cudaSuccess ||
          prof_mark(stream, false) != cudaSuccess)
        return LG_ERR_CUDA;
    }
  }
  MixParams mp{};
  for (int pk = 0; pk < n_patterns; ++pk) {
    mp.o[pk] = reinterpret_cast<const __nv_bfloat16*>(ws + lay.o[pk]);
    mp.l[pk] = reinterpret_cast<const float*>(ws + lay.l[pk]);
    mp.w[pk] = seg_w[pk]; mp.r[pk] = seg_r[pk]; mp.rows[pk] = lay.rows[pk];
    mp.packed[pk] = strided_layout(seg_w[pk], seg_r[pk]) ? 0 : 1;
  }
  mp.n_pat = n_patterns; mp.H = H; mp.BH = BH; mp.N = N; mp.D = D;
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.lse = lse;
  const long long rows = static_cast<long long>(BH) * N;
  const unsigned blocks = static_cast<unsigned>((rows * (D / kMixCols) + 255) / 256);
  if (launch_kernel(D == 64 ? longnet_mix_kernel<64> : longnet_mix_kernel<128>, dim3(blocks), dim3(256), 0, stream, true,
                    mp) != cudaSuccess)
    return LG_ERR_CUDA;
  return LG_OK;
}

}  // extern "C"
