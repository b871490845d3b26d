// Host side of the backward entry points declared in include/lg_attn.h:
// argument checks, workspace layout, the split of the global rows' and
// global keys' work, tensor maps and the kernel launches.
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <vector>

#include "lg_internal.h"

using namespace lg;

namespace {

bool aligned_b(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t rup(size_t x, size_t a) { return (x + a - 1) / a * a; }
int cdiv_b(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_b() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

int rows_per_load_host(int d) { return d <= 2 ? 128 : (d <= 4 ? 64 : 32); }

// bf16 [rows, D] slices of BH as {D, rows, BH}; load maps: boxes of
// rows_per_load(d) * d rows (element stride d); store maps: 32 * d rows.
bool encode_b(CUtensorMap* m, const void* base, int D, int rows, int BH, int d, bool store) {
  auto fn = encode_fn_b();
  if (!fn) return false;
  const int R = store ? 32 : rows_per_load_host(d);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(R * d), 1};
  cuuint32_t estr[3] = {1, static_cast<cuuint32_t>(d), 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  store ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Class-major 128-step tiles of one head with dilation d.
int tiles_for(int N, int d) {
  int t = 0;
  for (int c = 0; c < d && c < N; ++c) t += cdiv_b((N - c + d - 1) / d, 128);
  return t;
}

// Other-side tiles per split of the global rows' / keys' work: at least 4,
// and few enough that a row has at most 32 partials.
int bwd_split(int other_tiles) { return std::max(4, cdiv_b(other_tiles, 32)); }

struct BwdLayout {
  size_t lse2 = 0, delta = 0, qg = 0, kg = 0, vg = 0, dog = 0, lse2g = 0, deltag = 0, cnt = 0;
  size_t pq = 0, pk = 0, pv = 0, total = kStatusBytes;
  int CM = 0, gpad = 0, ns = 0;
};

// gather: Longformer (gathered global rows and the gcount table); max_tiles:
// the most other-side tiles a global row or key may have (sizes the partials).
BwdLayout bwd_layout(int BH, int N, int D, int g, bool gather, int max_tiles) {
  BwdLayout w;
  size_t off = kStatusBytes;
  w.CM = bwd_cm(N);
  w.lse2 = off; off += rup(static_cast<size_t>(BH) * w.CM * 4, 256);
  w.delta = off; off += rup(static_cast<size_t>(BH) * w.CM * 4, 256);
  if (g > 0) {
    w.gpad = static_cast<int>(rup(g, 128));
    const size_t gb = rup(static_cast<size_t>(BH) * g * D * 2, 256);
    if (gather) {
      w.qg = off; off += gb;
      w.kg = off; off += gb;
      w.vg = off; off += gb;
      w.dog = off; off += gb;
      w.cnt = off; off += rup((static_cast<size_t>(N) + 1) * 4, 256);
    }
    w.lse2g = off; off += rup(static_cast<size_t>(BH) * w.gpad * 4, 256);
    w.deltag = off; off += rup(static_cast<size_t>(BH) * w.gpad * 4, 256);
    // partial slots per row: bwd_split gives at most 32 splits, and at most
    // ceil(tiles / 4) (a bound that grows with the tile count)
    w.ns = std::min(32, cdiv_b(max_tiles, 4));
    const size_t pb = rup(static_cast<size_t>(BH) * g * w.ns * D * 4, 256);
    w.pq = off; off += pb;
    w.pk = off; off += pb;
    w.pv = off; off += pb;
  }
  w.total = off;
  return w;
}

bool valid_dt_b(lg_dtype dt) { return dt == LG_F32 || dt == LG_BF16; }

lg_status check_d_b(lg_dtype dt, int D) {
  if (dt == LG_BF16) return (D == 64 || D == 128) ? LG_OK : LG_ERR_UNSUPPORTED;
  return (D >= 4 && D <= 128 && D % 4 == 0) ? LG_OK : LG_ERR_UNSUPPORTED;
}

// The per-launch part of BwdParams shared by the q and kv launches of one dilation.
struct Group {
  int d;
  std::vector<int> heads;
};

std::vector<Group> dilation_groups(const int32_t* dilation, int H) {
  std::vector<Group> g;
  for (int h = 0; h < H; ++h) {
    auto it = std::find_if(g.begin(), g.end(), [&](const Group& x) { return x.d == dilation[h]; });
    if (it == g.end()) g.push_back(Group{dilation[h], {h}});
    else it->heads.push_back(h);
  }
  return g;
}

// Launches the kv then q kernels for every dilation group, then the reduces.
// main_*: main-side tensors [BH, N, D]; glob_*: global-side tensors [BH, g, D]
// (gathered or the ETC inputs).
lg_status run_bwd_kernels(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dv,
                          const void* qg, const void* kg, const void* vg, const void* dog, void* dq_g, void* dk_g,
                          void* dv_g, int B, int H, int N, int D, int wl, int wr, const int32_t* dilation, int etc,
                          const int32_t* gidx, int g, float s, unsigned char* ws, const BwdLayout& lay,
                          cudaStream_t stream) {
  const int BH = B * H;
  const std::vector<Group> groups = dilation_groups(dilation, H);
  const int n_gt = g > 0 ? cdiv_b(g, 128) : 0;
  for (int pass = 0; pass < 2; ++pass) {   // 0: kv kernel (dK, dV), 1: q kernel (dQ)
    const bool kv = pass == 0;
    for (const Group& grp : groups) {
      BwdParams bp{};
      const int d = grp.d;
      if (!encode_b(&bp.mQ, q, D, N, BH, d, false) || !encode_b(&bp.mK, k, D, N, BH, d, false) ||
          !encode_b(&bp.mV, v, D, N, BH, d, false) || !encode_b(&bp.mdO, dout, D, N, BH, d, false))
        return LG_ERR_CUDA;
      if (g > 0) {
        if (!encode_b(&bp.mQG, qg, D, g, BH, 1, false) || !encode_b(&bp.mKG, kg, D, g, BH, 1, false) ||
            !encode_b(&bp.mVG, vg, D, g, BH, 1, false) || !encode_b(&bp.mdOG, dog, D, g, BH, 1, false))
          return LG_ERR_CUDA;
      } else {
        bp.mQG = bp.mQ; bp.mKG = bp.mK; bp.mVG = bp.mV; bp.mdOG = bp.mdO;
      }
      if (kv) {
        if (!encode_b(&bp.sA, dk, D, N, BH, d, true) || !encode_b(&bp.sB, dv, D, N, BH, d, true)) return LG_ERR_CUDA;
      } else {
        if (!encode_b(&bp.sA, dq, D, N, BH, d, true)) return LG_ERR_CUDA;
        bp.sB = bp.sA;
      }
      bp.lse2 = reinterpret_cast<const float*>(ws + lay.lse2);
      bp.delta = reinterpret_cast<const float*>(ws + lay.delta);
      bp.lse2g = g > 0 ? reinterpret_cast<const float*>(ws + lay.lse2g) : nullptr;
      bp.deltag = g > 0 ? reinterpret_cast<const float*>(ws + lay.deltag) : nullptr;
      bp.gidx = etc ? nullptr : gidx;
      bp.gcount = (!etc && g > 0) ? reinterpret_cast<const int*>(ws + lay.cnt) : nullptr;
      bp.part_a = g > 0 ? reinterpret_cast<float*>(ws + (kv ? lay.pk : lay.pq)) : nullptr;
      bp.part_b = g > 0 ? reinterpret_cast<float*>(ws + lay.pv) : nullptr;
      bp.status = reinterpret_cast<int*>(ws);
      bp.wait_cap = wait_cap_cycles();
      bp.scale = s;
      bp.scale_log2 = s * 1.4426950408889634f;
      bp.B = B; bp.H = H; bp.N = N; bp.D = D; bp.wl = wl; bp.wr = wr; bp.d = d; bp.n_glob = g; bp.etc = etc;
      bp.CM = lay.CM; bp.M = bwd_class_stride(N, d); bp.gpad = lay.gpad;
      bp.n_heads = static_cast<int>(grp.heads.size());
      for (int x = 0; x < bp.n_heads; ++x) bp.heads[x] = grp.heads[x];
      bp.tiles_per_head = tiles_for(N, d);
      bp.n_gt = n_gt;
      bp.other_tiles = (etc ? n_gt : 0) + bp.tiles_per_head;
      bp.split = bwd_split(bp.other_tiles);
      bp.n_splits = g > 0 ? cdiv_b(bp.other_tiles, bp.split) : 1;
      bp.ns_stride = std::max(1, lay.ns);
      if (g > 0 && bp.n_splits > lay.ns) return LG_ERR_WORKSPACE;
      const long long n_grow = g > 0 ? static_cast<long long>(B) * bp.n_heads * n_gt * bp.n_splits : 0;
      const long long n_band = static_cast<long long>(B) * bp.n_heads * bp.tiles_per_head;
      if (n_grow + n_band > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
      bp.n_grow = static_cast<int>(n_grow);
      bp.n_band = static_cast<int>(n_band);
      const cudaError_t e = kv ? launch_bwd_kv(bp, stream) : launch_bwd_q(bp, stream);
      if (e != cudaSuccess) return LG_ERR_CUDA;
    }
  }
  if (g > 0) {
    // Each row's partials over the splits: the splits of every dilation group
    // share n_splits = ns_used (the same other-side tile count per head only
    // when the dilations agree), so the reduce takes the largest and unused
    // slots were never written: they are cleared before the kernels run.
    BwdReduceParams rk{};
    rk.part_a = reinterpret_cast<const float*>(ws + lay.pk);
    rk.part_b = reinterpret_cast<const float*>(ws + lay.pv);
    rk.out_a = etc ? dk_g : dk;
    rk.out_b = etc ? dv_g : dv;
    rk.gidx = etc ? nullptr : gidx;
    rk.BH = BH; rk.n_glob = g; rk.n_rows_out = etc ? g : N; rk.D = D; rk.n_splits = lay.ns;
    rk.scale_a = s; rk.scale_b = 1.f;
    if (launch_bwd_reduce(rk, stream) != cudaSuccess) return LG_ERR_CUDA;
    BwdReduceParams rq = rk;
    rq.part_a = reinterpret_cast<const float*>(ws + lay.pq);
    rq.part_b = nullptr;
    rq.out_a = etc ? dq_g : dq;
    rq.out_b = nullptr;
    rq.scale_a = s;
    if (launch_bwd_reduce(rq, stream) != cudaSuccess) return LG_ERR_CUDA;
  }
  return LG_OK;
}

}  // namespace

extern "C" {

size_t lg_attn_bwd_workspace_size(int B, int H, int N, int D, int n_global, lg_dtype dt) {
  if (B < 1 || H < 1 || N < 1 || D < 1 || n_global < 0 || n_global > N || !valid_dt_b(dt)) return 0;
  if (dt == LG_F32) return kStatusBytes + rup(static_cast<size_t>(B) * H * N * 4, 256);
  return bwd_layout(B * H, N, D, n_global, true, cdiv_b(N, 128) + LG_MAX_BF16_DILATION).total;
}

size_t lg_etc_attn_bwd_workspace_size(int B, int H, int L, int G, int D, lg_dtype dt) {
  if (B < 1 || H < 1 || L < 1 || G < 1 || D < 1 || !valid_dt_b(dt)) return 0;
  if (dt == LG_F32) return kStatusBytes + rup(static_cast<size_t>(B) * H * (static_cast<size_t>(L) + G) * 4, 256);
  return bwd_layout(B * H, L, D, G, false, cdiv_b(L, 128) + cdiv_b(G, 128)).total;
}

lg_status lg_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
                      void* dq, void* dk, void* dv, lg_dtype dt, int B, int H, int N, int D, int w_left, int w_right,
                      const int32_t* dilation, int causal, const int32_t* global_idx, int n_global, float scale,
                      void* workspace, size_t workspace_bytes, lg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // ---- argument checks (nothing is launched on failure): those of the forward
  // on q, k, v, out, lse, plus the gradient tensors and this call's workspace.
  lg_status st = validate_fwd_args(q, k, v, out, lse, dt, B, H, N, D, w_left, w_right, dilation, causal, global_idx,
                                   n_global, true);
  if (st != LG_OK) return st;
  if (!dout || !dq || !dk || !dv) return LG_ERR_INVALID_ARG;
  if (!aligned_b(dout, 16) || !aligned_b(dq, 16) || !aligned_b(dk, 16) || !aligned_b(dv, 16)) return LG_ERR_INVALID_ARG;
  const size_t need = lg_attn_bwd_workspace_size(B, H, N, D, n_global, dt);
  if (need == 0) return LG_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned_b(workspace, 256) || workspace_bytes < need) return LG_ERR_WORKSPACE;

  const int BH = B * H;
  const int wl = std::min(w_left, N);
  const int wr = causal ? 0 : std::min(w_right, N);
  const float s = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) return LG_ERR_CUDA;

  if (dt == LG_F32) {
    SimtBwdParams sp{};
    sp.q = static_cast<const float*>(q); sp.k = static_cast<const float*>(k); sp.v = static_cast<const float*>(v);
    sp.out = static_cast<const float*>(out); sp.lse = lse; sp.dout = static_cast<const float*>(dout);
    sp.dq = static_cast<float*>(dq); sp.dk = static_cast<float*>(dk); sp.dv = static_cast<float*>(dv);
    sp.delta = reinterpret_cast<float*>(ws + kStatusBytes);
    sp.gidx = global_idx; sp.status = status;
    sp.BH = BH; sp.H = H; sp.N = N; sp.D = D; sp.wl = wl; sp.wr = wr; sp.n_glob = n_global; sp.etc = 0; sp.scale = s;
    for (int h = 0; h < H; ++h) sp.dil[h] = dilation[h];
    const size_t nbytes = static_cast<size_t>(BH) * N * D * 4;
    if (cudaMemsetAsync(dk, 0, nbytes, stream) != cudaSuccess || cudaMemsetAsync(dv, 0, nbytes, stream) != cudaSuccess)
      return LG_ERR_CUDA;
    PrepParams pp{};
    pp.gidx = global_idx; pp.n_glob = n_global; pp.N = N; pp.status = status; pp.BH = BH; pp.D = D;
    if (launch_prep(pp, stream) != cudaSuccess) return LG_ERR_CUDA;
    return launch_simt_bwd(sp, stream) == cudaSuccess ? LG_OK : LG_ERR_CUDA;
  }

  if (!encode_fn_b()) return LG_ERR_CUDA;
  const BwdLayout lay = bwd_layout(BH, N, D, n_global, true, cdiv_b(N, 128) + LG_MAX_BF16_DILATION);
  // The class-major vectors start at zero (their padding is read for masked
  // columns), and so do the global side's vectors and partial sums (a row's
  // unused partial slots take part in the reduce).
  if (cudaMemsetAsync(ws + lay.lse2, 0, 2 * (lay.delta - lay.lse2), stream) != cudaSuccess) return LG_ERR_CUDA;
  if (n_global > 0) {
    if (cudaMemsetAsync(ws + lay.lse2g, 0, lay.total - lay.lse2g, stream) != cudaSuccess) return LG_ERR_CUDA;
    PrepParams pp{};
    pp.gidx = global_idx; pp.n_glob = n_global; pp.N = N; pp.status = status; pp.BH = BH; pp.D = D;
    pp.q = static_cast<const __nv_bfloat16*>(q); pp.k = static_cast<const __nv_bfloat16*>(k);
    pp.v = static_cast<const __nv_bfloat16*>(v);
    pp.qg = reinterpret_cast<__nv_bfloat16*>(ws + lay.qg); pp.kg = reinterpret_cast<__nv_bfloat16*>(ws + lay.kg);
    pp.vg = reinterpret_cast<__nv_bfloat16*>(ws + lay.vg);
    pp.gcount = reinterpret_cast<int*>(ws + lay.cnt);
    if (launch_prep(pp, stream) != cudaSuccess) return LG_ERR_CUDA;
  }
  BwdPrepParams bp{};
  bp.out = static_cast<const __nv_bfloat16*>(out); bp.dout = static_cast<const __nv_bfloat16*>(dout); bp.lse = lse;
  bp.gidx = n_global > 0 ? global_idx : nullptr;
  for (int h = 0; h < H; ++h) bp.dil[h] = dilation[h];
  bp.dog = n_global > 0 ? reinterpret_cast<__nv_bfloat16*>(ws + lay.dog) : nullptr;
  bp.lse2 = reinterpret_cast<float*>(ws + lay.lse2); bp.delta = reinterpret_cast<float*>(ws + lay.delta);
  bp.lse2g = n_global > 0 ? reinterpret_cast<float*>(ws + lay.lse2g) : nullptr;
  bp.deltag = n_global > 0 ? reinterpret_cast<float*>(ws + lay.deltag) : nullptr;
  bp.gcount = n_global > 0 ? reinterpret_cast<int*>(ws + lay.cnt) : nullptr;
  bp.status = status;
  bp.BH = BH; bp.H = H; bp.N = N; bp.D = D; bp.n_glob = n_global; bp.CM = lay.CM; bp.gpad = lay.gpad; bp.etc = 0;
  if (launch_bwd_prep(bp, stream) != cudaSuccess) return LG_ERR_CUDA;
  return run_bwd_kernels(q, k, v, dout, dq, dk, dv, ws + lay.qg, ws + lay.kg, ws + lay.vg, ws + lay.dog, nullptr,
                         nullptr, nullptr, B, H, N, D, wl, wr, dilation, 0, global_idx, n_global, s, ws, lay, stream);
}

lg_status lg_etc_attn_bwd(const void* q_l, const void* k_l, const void* v_l, const void* q_g, const void* k_g,
                          const void* v_g, const void* out_l, const void* out_g, const float* lse_l, const float* lse_g,
                          const void* dout_l, const void* dout_g, void* dq_l, void* dk_l, void* dv_l, void* dq_g,
                          void* dk_g, void* dv_g, lg_dtype dt, int B, int H, int L, int G, int D, int radius,
                          float scale, void* workspace, size_t workspace_bytes, lg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!valid_dt_b(dt) || B < 1 || H < 1 || L < 1 || G < 1 || radius < 0) return LG_ERR_INVALID_ARG;
  if (H > LG_MAX_HEADS) return LG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * (static_cast<long long>(L) + G) > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  const void* ptrs[18] = {q_l, k_l, v_l, q_g, k_g, v_g, out_l, out_g, dout_l, dout_g,
                          dq_l, dk_l, dv_l, dq_g, dk_g, dv_g, lse_l, lse_g};
  for (int x = 0; x < 18; ++x)
    if (ptrs[x] == nullptr || !aligned_b(ptrs[x], x < 16 ? 16 : 4)) return LG_ERR_INVALID_ARG;
  lg_status st = check_d_b(dt, D);
  if (st != LG_OK) return st;
  const size_t need = lg_etc_attn_bwd_workspace_size(B, H, L, G, D, dt);
  if (workspace == nullptr || !aligned_b(workspace, 256) || workspace_bytes < need) return LG_ERR_WORKSPACE;

  const int BH = B * H;
  const int r = std::min(radius, L);
  const float s = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) return LG_ERR_CUDA;

  if (dt == LG_F32) {
    SimtBwdParams sp{};
    sp.q = static_cast<const float*>(q_l); sp.k = static_cast<const float*>(k_l); sp.v = static_cast<const float*>(v_l);
    sp.qg = static_cast<const float*>(q_g); sp.kg = static_cast<const float*>(k_g); sp.vg = static_cast<const float*>(v_g);
    sp.out = static_cast<const float*>(out_l); sp.out_g = static_cast<const float*>(out_g);
    sp.lse = lse_l; sp.lse_g = lse_g;
    sp.dout = static_cast<const float*>(dout_l); sp.dout_g = static_cast<const float*>(dout_g);
    sp.dq = static_cast<float*>(dq_l); sp.dk = static_cast<float*>(dk_l); sp.dv = static_cast<float*>(dv_l);
    sp.dq_g = static_cast<float*>(dq_g); sp.dk_g = static_cast<float*>(dk_g); sp.dv_g = static_cast<float*>(dv_g);
    sp.delta = reinterpret_cast<float*>(ws + kStatusBytes);
    sp.status = status;
    sp.BH = BH; sp.H = H; sp.N = L; sp.D = D; sp.wl = r; sp.wr = r; sp.n_glob = G; sp.etc = 1; sp.scale = s;
    for (int h = 0; h < H; ++h) sp.dil[h] = 1;
    const size_t nl = static_cast<size_t>(BH) * L * D * 4, ng = static_cast<size_t>(BH) * G * D * 4;
    if (cudaMemsetAsync(dk_l, 0, nl, stream) != cudaSuccess || cudaMemsetAsync(dv_l, 0, nl, stream) != cudaSuccess ||
        cudaMemsetAsync(dk_g, 0, ng, stream) != cudaSuccess || cudaMemsetAsync(dv_g, 0, ng, stream) != cudaSuccess)
      return LG_ERR_CUDA;
    return launch_simt_bwd(sp, stream) == cudaSuccess ? LG_OK : LG_ERR_CUDA;
  }

  if (!encode_fn_b()) return LG_ERR_CUDA;
  const BwdLayout lay = bwd_layout(BH, L, D, G, false, cdiv_b(L, 128) + cdiv_b(G, 128));
  if (cudaMemsetAsync(ws + lay.lse2, 0, lay.total - lay.lse2, stream) != cudaSuccess) return LG_ERR_CUDA;
  BwdPrepParams bp{};
  bp.out = static_cast<const __nv_bfloat16*>(out_l); bp.dout = static_cast<const __nv_bfloat16*>(dout_l); bp.lse = lse_l;
  bp.out_g = static_cast<const __nv_bfloat16*>(out_g); bp.dout_g = static_cast<const __nv_bfloat16*>(dout_g);
  bp.lse_g = lse_g;
  bp.gidx = nullptr;
  for (int h = 0; h < H; ++h) bp.dil[h] = 1;
  bp.lse2 = reinterpret_cast<float*>(ws + lay.lse2); bp.delta = reinterpret_cast<float*>(ws + lay.delta);
  bp.lse2g = reinterpret_cast<float*>(ws + lay.lse2g); bp.deltag = reinterpret_cast<float*>(ws + lay.deltag);
  bp.status = status;
  bp.BH = BH; bp.H = H; bp.N = L; bp.D = D; bp.n_glob = G; bp.CM = lay.CM; bp.gpad = lay.gpad; bp.etc = 1;
  if (launch_bwd_prep(bp, stream) != cudaSuccess) return LG_ERR_CUDA;
  std::vector<int32_t> ones(H, 1);
  return run_bwd_kernels(q_l, k_l, v_l, dout_l, dq_l, dk_l, dv_l, q_g, k_g, v_g, dout_g, dq_g, dk_g, dv_g, B, H, L, D,
                         r, r, ones.data(), 1, nullptr, G, s, ws, lay, stream);
}

}  // extern "C"
