// Host side of the C ABI declared in include/lg_attn.h: argument checks, the
// work schedule (band tiles per dilation residue class, splits of the
// global-query rows), TMA tensor-map encoding and the kernel launches.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "lg_internal.h"

namespace lg {
int tc_rows_per_load(int d);
}

namespace lg {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// bf16 tensor viewed as {D, rows, BH}; the row dimension strided by `d`
// (d rows apart) with boxes of rows_per_load(d) rows of 64 columns.
bool encode_map(CUtensorMap* m, const void* base, int D, int rows, int BH, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int R = (d == 0) ? kTileM : tc_rows_per_load(d);
  const int stride = d == 0 ? 1 : d;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(R * stride), 1};
  cuuint32_t estr[3] = {1, static_cast<cuuint32_t>(stride), 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 output viewed as {D, rows, BH} for tiled stores of 32 rows x 64
// columns, the rows `d` apart (element stride d along the row dimension, a
// box of 32*d rows: the 32 rows of one dilation residue class).
bool encode_store_map(CUtensorMap* m, void* base, int D, int rows, int BH, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(32 * d), 1};
  cuuint32_t estr[3] = {1, static_cast<cuuint32_t>(d), 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Band units at the end of a launch of `units` units to split in two
// one-tile units each: the last round of a persistent launch (units mod grid
// units) when splitting it still leaves at most one item per CTA; 0 otherwise.
long long grow_tail_cap(const TcParams& tp) {
  if (tp.n_grow_units == 0 || !tp.grow_interleave) return 1LL << 40;
  // the units after the last key split's global-row units in the last (batch, head) block
  const long long nb = tp.head_unit_start[tp.H] - tp.head_unit_start[tp.H - 1];
  return nb > 0 ? nb - nb * (tp.n_splits - 1) / tp.n_splits : 0;
}

long long tail_split(long long units, long long band_units) {
  const long long grid = std::min<long long>(units, device_sm_count());
  if (grid <= 0 || units <= grid) return 0;
  const long long last = units % grid;
  return (last > 0 && last <= grid - last && last <= band_units) ? last : 0;
}

// ------------------------------------------------------------------ profiling

struct Profiler {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> events;
  size_t used = 0;
};
Profiler& prof() {
  static Profiler p;
  return p;
}

cudaError_t prof_mark(cudaStream_t s, bool start) {
  Profiler& p = prof();
  if (!p.on) return cudaSuccess;
  if (start) {
    if (p.used == p.events.size()) {
      cudaEvent_t a, b;
      cudaError_t e = cudaEventCreate(&a);
      if (e != cudaSuccess) return e;
      e = cudaEventCreate(&b);
      if (e != cudaSuccess) return e;
      p.events.emplace_back(a, b);
    }
    return cudaEventRecord(p.events[p.used].first, s);
  }
  cudaError_t e = cudaEventRecord(p.events[p.used].second, s);
  ++p.used;
  return e;
}

}  // namespace lg

using namespace lg;

namespace {

// ------------------------------------------------------------------ helpers

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Cap of the bounded work waits and the timeout-test switch (lg_debug_timeout_test).
std::atomic<long long> g_wait_cap_override{0};
std::atomic<int> g_withhold{0};

// Band work units of one head: pairs of 128-step query tiles in each residue class.
int band_units_for(int N, int d) {
  int units = 0;
  for (int c = 0; c < d && c < N; ++c) {
    const int n_c = (N - c + d - 1) / d;
    units += cdiv(n_c, 2 * kTileM);
  }
  return units;
}

// Global-query rows: 128-row tiles against splits of the key tiles; the two
// warpgroups of a unit take alternate key tiles, so each split leaves two
// partial slots per row.
struct GrowPlan {
  int n_gtiles = 0, n_key_tiles = 0, n_splits = 0, n_parts = 0, split = 0;
};

// Fewest key tiles per split the workspace is sized for: rows of up to 64 key
// tiles may be split into 8-tile pieces, up to 256 into 16, longer rows keep
// 32-tile splits.
int min_grow_split(int key_tiles) { return key_tiles <= 64 ? 8 : key_tiles <= 256 ? 16 : kGrowSplitMax; }

// The splits of a row of key_tiles key tiles into pieces of about `split`
// tiles (clamped to [min_grow_split, kGrowSplitMax]), evened out so that the
// pieces differ by at most two tiles.  split = 0 gives the finest plan, the
// one the workspace is sized for; any other plan has no more splits.
GrowPlan grow_plan(int n_glob, int key_tiles, int split) {
  GrowPlan g;
  if (n_glob <= 0) return g;
  split = std::max(min_grow_split(key_tiles), std::min(kGrowSplitMax, split));
  g.n_gtiles = cdiv(n_glob, kTileM);
  g.n_key_tiles = key_tiles;
  const int n = cdiv(key_tiles, split);
  g.split = std::min(kGrowSplitMax, 2 * cdiv(cdiv(key_tiles, n), 2));
  g.n_splits = cdiv(key_tiles, g.split);
  g.n_parts = 2 * g.n_splits;
  return g;
}

// Key tiles per split for a launch: a global-row unit (split / 2 key tiles per
// warpgroup) should take no longer than a band unit (band_tiles key tiles per
// query tile) or than an SM's average share of the launch, whichever is
// longer, so that the few global-row units do not end after everything else.
int choose_grow_split(long long band_units, int band_tiles, long long grow_blocks, int key_tiles) {
  const double work = static_cast<double>(band_units) * band_tiles +
                      static_cast<double>(grow_blocks) * key_tiles / 2.0;   // in key tiles per warpgroup
  const double per_sm = work / std::max(1, device_sm_count());
  const double len = std::max(static_cast<double>(band_tiles), per_sm);
  return static_cast<int>(std::min(2.0 * len, static_cast<double>(kGrowSplitMax)));
}

struct WsLayout {
  size_t qg = 0, kg = 0, vg = 0, cnt = 0, acc = 0, ml = 0, units = 0, max_units = 0, total = kStatusBytes;
};

// Work units of one tensor-core launch, at most: band units (per head at most
// ceil(rows / 256) plus one per residue class) and the global-row units.
long long max_units(int BH, int rows, int max_dil, const GrowPlan& g) {
  return static_cast<long long>(BH) * (cdiv(rows, 2 * kTileM) + max_dil) +
         static_cast<long long>(BH) * g.n_gtiles * g.n_splits;
}

// gather (Longformer): gathered global rows and the gcount table of N + 1 ints.
// Then the partial sums of the global rows and the unit table (16 ints per unit).
WsLayout ws_layout(int BH, int n_glob, int D, int n_splits, bool gather, int N, long long units) {
  WsLayout w;
  size_t off = kStatusBytes;
  if (n_glob > 0) {
    const size_t gbytes = round_up(static_cast<size_t>(BH) * n_glob * D * 2, 256);
    if (gather) {
      w.qg = off; off += gbytes;
      w.kg = off; off += gbytes;
      w.vg = off; off += gbytes;
      w.cnt = off; off += round_up((static_cast<size_t>(N) + 1) * 4, 256);
    }
    w.acc = off; off += round_up(static_cast<size_t>(BH) * n_glob * n_splits * D * 4, 256);
    w.ml = off; off += round_up(static_cast<size_t>(BH) * n_glob * n_splits * 2 * 4, 256);
  }
  w.units = off;
  w.max_units = static_cast<size_t>(units) + static_cast<size_t>(units) / 2;   // room for the tail split
  off += round_up(w.max_units * 64, 256);
  w.total = off;
  return w;
}

lg_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LG_OK : LG_ERR_CUDA; }

bool valid_dt(lg_dtype dt) { return dt == LG_F32 || dt == LG_BF16; }

lg_status check_d(lg_dtype dt, int D) {
  if (dt == LG_BF16) return (D == 64 || D == 128) ? LG_OK : LG_ERR_UNSUPPORTED;
  return (D >= 4 && D <= 128 && D % 4 == 0) ? LG_OK : LG_ERR_UNSUPPORTED;
}

}  // namespace

// ==================================================================== ABI

extern "C" {

const char* lg_status_string(lg_status s) {
  switch (s) {
    case LG_OK: return "LG_OK";
    case LG_ERR_INVALID_ARG: return "LG_ERR_INVALID_ARG: an argument is outside its documented range";
    case LG_ERR_UNSUPPORTED: return "LG_ERR_UNSUPPORTED: valid arguments this build does not run";
    case LG_ERR_CUDA: return "LG_ERR_CUDA: a CUDA call or kernel launch failed";
    case LG_ERR_TIMEOUT: return "LG_ERR_TIMEOUT: a bounded device wait ran out";
    case LG_ERR_WORKSPACE: return "LG_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case LG_ERR_GLOBAL_IDX: return "LG_ERR_GLOBAL_IDX: global positions not strictly increasing or out of range";
  }
  return "unknown lg_status";
}

const char* lg_version(void) { return "0.1.0 sm_103a"; }

size_t lg_attn_fwd_workspace_size(int B, int H, int N, int D, int n_global, lg_dtype dt) {
  if (B < 1 || H < 1 || N < 1 || D < 1 || n_global < 0 || n_global > N || !valid_dt(dt)) return 0;
  if (dt == LG_F32) return kStatusBytes;
  const GrowPlan g = grow_plan(n_global, cdiv(N, kTileN), 0);
  return ws_layout(B * H, n_global, D, g.n_parts, true, N, max_units(B * H, N, LG_MAX_BF16_DILATION, g)).total;
}

size_t lg_etc_attn_fwd_workspace_size(int B, int H, int L, int G, int D, lg_dtype dt) {
  if (B < 1 || H < 1 || L < 1 || G < 1 || D < 1 || !valid_dt(dt)) return 0;
  if (dt == LG_F32) return kStatusBytes;
  const GrowPlan g = grow_plan(G, cdiv(G, kTileN) + cdiv(L, kTileN), 0);
  return ws_layout(B * H, G, D, g.n_parts, false, 0, max_units(B * H, L, 1, g)).total;
}

}  // extern "C"

namespace lg {

long long wait_cap_cycles() {
  const long long v = g_wait_cap_override.load(std::memory_order_relaxed);
  return v > 0 ? v : 2000000000LL;  // about one second at the SM clock
}

int withhold_for_test() { return g_withhold.load(std::memory_order_relaxed); }

// Every argument check of lg_attn_fwd but the workspace, on sizes and
// pointers only (no CUDA call).  per_call_head_limit: refuse H >
// LG_MAX_HEADS (the host-memory entry point splits larger problems into
// groups of at most that many slices).
lg_status validate_fwd_args(const void* q, const void* k, const void* v, const void* out, const float* lse,
                            lg_dtype dt, int B, int H, int N, int D, int w_left, int w_right,
                            const int32_t* dilation, int causal, const int32_t* global_idx, int n_global,
                            bool per_call_head_limit) {
  if (!valid_dt(dt) || B < 1 || H < 1 || N < 1 || w_left < 0 || w_right < 0 || (causal != 0 && causal != 1) ||
      n_global < 0 || n_global > N || dilation == nullptr)
    return LG_ERR_INVALID_ARG;
  if (per_call_head_limit && H > LG_MAX_HEADS) return LG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * N > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  if (!q || !k || !v || !out || !lse) return LG_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return LG_ERR_INVALID_ARG;
  if (n_global > 0 && (global_idx == nullptr || !aligned(global_idx, 4))) return LG_ERR_INVALID_ARG;
  for (int h = 0; h < H; ++h)
    if (dilation[h] < 1) return LG_ERR_INVALID_ARG;
  lg_status st = check_d(dt, D);
  if (st != LG_OK) return st;
  if (dt == LG_BF16)
    for (int h = 0; h < H; ++h)
      if (dilation[h] > LG_MAX_BF16_DILATION) return LG_ERR_UNSUPPORTED;
  return LG_OK;
}

lg_status validate_fwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                       lg_dtype dt, int B, int H, int N, int D, int w_left, int w_right, const int32_t* dilation,
                       int causal, const int32_t* global_idx, int n_global, const void* workspace,
                       size_t workspace_bytes, bool per_call_head_limit) {
  const lg_status st = validate_fwd_args(q, k, v, out, lse, dt, B, H, N, D, w_left, w_right, dilation, causal,
                                         global_idx, n_global, per_call_head_limit);
  if (st != LG_OK) return st;
  const size_t need = lg_attn_fwd_workspace_size(B, H, N, D, n_global, dt);
  if (need == 0) return LG_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return LG_ERR_WORKSPACE;
  return LG_OK;
}

}  // namespace lg

namespace {

// The Longformer forward; qgl / kgl / vgl: the global rows' separate
// projections (all three, or none: then q, k, v serve the global rows too).
lg_status attn_fwd_impl(const void* q, const void* k, const void* v, const void* qgl, const void* kgl,
                        const void* vgl, void* out, float* lse, lg_dtype dt, int B, int H, int N, int D, int w_left,
                        int w_right, const int32_t* dilation, int causal, const int32_t* global_idx, int n_global,
                        float scale, void* workspace, size_t workspace_bytes, lg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // ---- argument checks (nothing is launched on failure)
  lg_status st = validate_fwd(q, k, v, out, lse, dt, B, H, N, D, w_left, w_right, dilation, causal, global_idx,
                              n_global, workspace, workspace_bytes, true);
  if (st != LG_OK) return st;
  if (qgl == nullptr) { qgl = q; kgl = k; vgl = v; }

  const int BH = B * H;
  const int wl = std::min(w_left, N);
  const int wr = causal ? 0 : std::min(w_right, N);
  const float s = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);

  cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, stream);
  if (e != cudaSuccess) return LG_ERR_CUDA;

  if (dt == LG_F32) {
    SimtParams sp{};   // the kernel itself checks the global list (one launch per call)
    sp.status = status;
    sp.q = static_cast<const float*>(q); sp.k = static_cast<const float*>(k); sp.v = static_cast<const float*>(v);
    sp.out = static_cast<float*>(out); sp.lse = lse; sp.gidx = global_idx;
    sp.qgl = static_cast<const float*>(qgl); sp.kgl = static_cast<const float*>(kgl);
    sp.vgl = static_cast<const float*>(vgl);
    sp.BH = BH; sp.H = H; sp.N = N; sp.D = D; sp.wl = wl; sp.wr = wr; sp.n_glob = n_global; sp.etc = 0;
    sp.scale = s;
    for (int h = 0; h < H; ++h) sp.dil[h] = dilation[h];
    if ((e = prof_mark(stream, true)) != cudaSuccess) return LG_ERR_CUDA;
    if ((e = launch_simt(sp, stream)) != cudaSuccess) return LG_ERR_CUDA;
    return cuda_status(prof_mark(stream, false));
  }

  // ---- bf16 tensor-core path
  if (!encode_fn()) return LG_ERR_CUDA;
  GrowPlan gp;
  const bool interleave = grow_interleave_for(4LL * BH * N * D);   // K and V, bf16
  if (n_global > 0) {
    long long band_units = 0;
    for (int h = 0; h < H; ++h) band_units += band_units_for(N, dilation[h]);
    band_units *= B;
    const int band_tiles = std::min(cdiv(static_cast<long long>(wl) + wr + kTileM, kTileN) + 1, cdiv(N, kTileN)) + cdiv(n_global, kTileN);
    // interleaved global-row units are sized like a band unit (2 x band_tiles key tiles), so that
    // the rounds stay even; first-placed ones may be longer
    gp = grow_plan(n_global, cdiv(N, kTileN),
                   interleave ? 2 * band_tiles
                              : choose_grow_split(band_units, band_tiles, static_cast<long long>(BH) * cdiv(n_global, kTileM),
                                                  cdiv(N, kTileN)));
  }
  const WsLayout lay = ws_layout(BH, n_global, D, gp.n_parts, true, N, max_units(BH, N, LG_MAX_BF16_DILATION, gp));
  __nv_bfloat16* qg = reinterpret_cast<__nv_bfloat16*>(ws + lay.qg);
  __nv_bfloat16* kg = reinterpret_cast<__nv_bfloat16*>(ws + lay.kg);
  __nv_bfloat16* vg = reinterpret_cast<__nv_bfloat16*>(ws + lay.vg);
  if (n_global > 0) {
    PrepParams pp{};
    pp.gidx = global_idx; pp.n_glob = n_global; pp.N = N; pp.status = status; pp.BH = BH; pp.D = D;
    pp.q = static_cast<const __nv_bfloat16*>(qgl); pp.k = static_cast<const __nv_bfloat16*>(k);
    pp.v = static_cast<const __nv_bfloat16*>(v);
    pp.qg = qg; pp.kg = kg; pp.vg = vg;
    pp.gcount = reinterpret_cast<int*>(ws + lay.cnt);
    if ((e = launch_prep(pp, stream)) != cudaSuccess) return LG_ERR_CUDA;
  }

  // distinct dilations other than 1, in groups that fit the slots beside d = 1
  std::vector<int> others;
  for (int h = 0; h < H; ++h)
    if (dilation[h] != 1 && std::find(others.begin(), others.end(), dilation[h]) == others.end())
      others.push_back(dilation[h]);
  std::sort(others.begin(), others.end());
  const int n_groups = std::max(1, cdiv(static_cast<long long>(others.size()), kMaxSlots - 1));
  static_assert(1 + (LG_MAX_HEADS + kMaxSlots - 2) / (kMaxSlots - 1) <= static_cast<int>(kStatusBytes / sizeof(int)),
                "one unit counter per launch fits in the status area");

  TcParams tp;  // filled per launch (a few KB; calls from several host threads keep their own)
  for (int grp = 0; grp < n_groups; ++grp) {
    tp = TcParams{};
    int slot_d[kMaxSlots] = {1, 0, 0, 0};
    int n_slots = 1;
    for (size_t x = grp * (kMaxSlots - 1); x < others.size() && n_slots < kMaxSlots; ++x) slot_d[n_slots++] = others[x];
    for (int sl = 0; sl < n_slots; ++sl) {
      tp.slot_dil[sl] = slot_d[sl];
      tp.slot_units[sl] = band_units_for(N, slot_d[sl]);
      if (!encode_map(&tp.mapQ[sl], q, D, N, BH, slot_d[sl]) || !encode_map(&tp.mapK[sl], k, D, N, BH, slot_d[sl]) ||
          !encode_map(&tp.mapV[sl], v, D, N, BH, slot_d[sl]) || !encode_store_map(&tp.mapO[sl], out, D, N, BH, slot_d[sl]))
        return LG_ERR_CUDA;
    }
    for (int sl = n_slots; sl < kMaxSlots; ++sl) {
      tp.slot_dil[sl] = 1;
      tp.mapQ[sl] = tp.mapQ[0]; tp.mapK[sl] = tp.mapK[0]; tp.mapV[sl] = tp.mapV[0]; tp.mapO[sl] = tp.mapO[0];
    }
    if (n_global > 0) {
      if (!encode_map(&tp.mapQg, qg, D, n_global, BH, 0) || !encode_map(&tp.mapKg, kg, D, n_global, BH, 0) ||
          !encode_map(&tp.mapVg, vg, D, n_global, BH, 0) || !encode_map(&tp.mapKgr, kgl, D, N, BH, 1) ||
          !encode_map(&tp.mapVgr, vgl, D, N, BH, 1))
        return LG_ERR_CUDA;
    } else {
      tp.mapQg = tp.mapQ[0]; tp.mapKg = tp.mapK[0]; tp.mapVg = tp.mapV[0];
      tp.mapKgr = tp.mapK[0]; tp.mapVgr = tp.mapV[0];
    }
    int start = 0;
    for (int h = 0; h < H; ++h) {
      tp.head_unit_start[h] = start;
      int sl = -1;
      if (dilation[h] == 1) sl = (grp == 0) ? 0 : -1;
      else
        for (int x = 1; x < n_slots; ++x)
          if (slot_d[x] == dilation[h]) sl = x;
      tp.head_slot[h] = sl < 0 ? 255 : static_cast<unsigned char>(sl);
      if (sl >= 0) start += tp.slot_units[sl];
    }
    tp.head_unit_start[H] = start;
    tp.band_units_per_batch = start;
    for (int h = 0; h < H; ++h) tp.head_class[h] = -1;
    tp.seg_w = 0;
    tp.seg_causal = 0;
    tp.out = out; tp.lse = lse;
    tp.part_acc = reinterpret_cast<float*>(ws + lay.acc);
    tp.part_ml = reinterpret_cast<float*>(ws + lay.ml);
    tp.gidx = global_idx; tp.gcount = n_global > 0 ? reinterpret_cast<const int*>(ws + lay.cnt) : nullptr;
    tp.status = status; tp.wait_cap = wait_cap_cycles(); tp.withhold = withhold_for_test();
    tp.unit_counter = status + 1 + grp;   // one zeroed word of the status area per launch
    tp.scale_log2 = s * 1.4426950408889634f;
    tp.BH = BH; tp.H = H; tp.N = N; tp.D = D; tp.wl = wl; tp.wr = wr; tp.n_glob = n_global; tp.etc = 0;
    tp.n_gtiles = gp.n_gtiles; tp.n_splits = gp.n_splits; tp.n_parts = gp.n_parts;
    tp.n_key_tiles_grow = gp.n_key_tiles; tp.grow_split = std::max(1, gp.split);
    tp.n_grow_units = (grp == 0 && n_global > 0) ? BH * gp.n_gtiles * gp.n_splits : 0;
    tp.grow_interleave = interleave ? 1 : 0;
    const long long base_units = static_cast<long long>(tp.n_grow_units) + static_cast<long long>(B) * start;
    tp.n_tail_split = static_cast<int>(std::min(tail_split(base_units, static_cast<long long>(B) * start), grow_tail_cap(tp)));
    const long long units = base_units + tp.n_tail_split;
    if (units > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
    if (units > static_cast<long long>(lay.max_units)) return LG_ERR_WORKSPACE;
    tp.units = ws + lay.units;
    if ((e = prof_mark(stream, true)) != cudaSuccess) return LG_ERR_CUDA;
    // A later group's table may not overwrite the table the previous group's kernel reads.
    if ((e = launch_tc(tp, static_cast<int>(units), stream, grp == 0)) != cudaSuccess) return LG_ERR_CUDA;
    if ((e = prof_mark(stream, false)) != cudaSuccess) return LG_ERR_CUDA;
  }
  if (n_global > 0) {
    MergeParams mp{};
    mp.part_acc = reinterpret_cast<const float*>(ws + lay.acc);
    mp.part_ml = reinterpret_cast<const float*>(ws + lay.ml);
    mp.out = out; mp.lse = lse; mp.gidx = global_idx;
    mp.BH = BH; mp.N_out = N; mp.D = D; mp.n_glob = n_global; mp.n_splits = gp.n_parts;
    if ((e = launch_merge(mp, 1, stream)) != cudaSuccess) return LG_ERR_CUDA;
  }
  return LG_OK;
}

}  // namespace

extern "C" {

lg_status lg_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, lg_dtype dt, int B,
                      int H, int N, int D, int w_left, int w_right, const int32_t* dilation, int causal,
                      const int32_t* global_idx, int n_global, float scale, void* workspace,
                      size_t workspace_bytes, lg_stream_t stream) {
  return attn_fwd_impl(q, k, v, nullptr, nullptr, nullptr, out, lse, dt, B, H, N, D, w_left, w_right, dilation,
                       causal, global_idx, n_global, scale, workspace, workspace_bytes, stream);
}

lg_status lg_attn_fwd_gproj(const void* q, const void* k, const void* v, const void* q_glob, const void* k_glob,
                            const void* v_glob, void* out, float* lse, lg_dtype dt, int B, int H, int N, int D,
                            int w_left, int w_right, const int32_t* dilation, int causal,
                            const int32_t* global_idx, int n_global, float scale, void* workspace,
                            size_t workspace_bytes, lg_stream_t stream) {
  if (q_glob == nullptr || k_glob == nullptr || v_glob == nullptr) return LG_ERR_INVALID_ARG;
  if (!aligned(q_glob, 16) || !aligned(k_glob, 16) || !aligned(v_glob, 16)) return LG_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, q_glob, k_glob, v_glob, out, lse, dt, B, H, N, D, w_left, w_right, dilation,
                       causal, global_idx, n_global, scale, workspace, workspace_bytes, stream);
}

lg_status lg_etc_attn_fwd(const void* q_l, const void* k_l, const void* v_l, const void* q_g, const void* k_g,
                          const void* v_g, void* out_l, void* out_g, float* lse_l, float* lse_g, lg_dtype dt, int B,
                          int H, int L, int G, int D, int radius, float scale, void* workspace, size_t workspace_bytes,
                          lg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!valid_dt(dt) || B < 1 || H < 1 || L < 1 || G < 1 || radius < 0) return LG_ERR_INVALID_ARG;
  if (H > LG_MAX_HEADS) return LG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * (static_cast<long long>(L) + G) > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  const void* ptrs[10] = {q_l, k_l, v_l, q_g, k_g, v_g, out_l, out_g, lse_l, lse_g};
  for (int x = 0; x < 10; ++x)
    if (ptrs[x] == nullptr || !aligned(ptrs[x], x < 8 ? 16 : 4)) return LG_ERR_INVALID_ARG;
  lg_status st = check_d(dt, D);
  if (st != LG_OK) return st;
  const size_t need = lg_etc_attn_fwd_workspace_size(B, H, L, G, D, dt);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return LG_ERR_WORKSPACE;

  const int BH = B * H;
  const int r = std::min(radius, L);
  const float s = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, stream);
  if (e != cudaSuccess) return LG_ERR_CUDA;

  if (dt == LG_F32) {
    SimtParams sp{};
    sp.q = static_cast<const float*>(q_l); sp.k = static_cast<const float*>(k_l); sp.v = static_cast<const float*>(v_l);
    sp.qg = static_cast<const float*>(q_g); sp.kg = static_cast<const float*>(k_g);
    sp.vg = static_cast<const float*>(v_g);
    sp.out = static_cast<float*>(out_l); sp.lse = lse_l; sp.out_g = static_cast<float*>(out_g); sp.lse_g = lse_g;
    sp.BH = BH; sp.H = H; sp.N = L; sp.D = D; sp.wl = r; sp.wr = r; sp.n_glob = G; sp.etc = 1; sp.scale = s;
    for (int h = 0; h < H; ++h) sp.dil[h] = 1;
    if ((e = prof_mark(stream, true)) != cudaSuccess) return LG_ERR_CUDA;
    if ((e = launch_simt(sp, stream)) != cudaSuccess) return LG_ERR_CUDA;
    return cuda_status(prof_mark(stream, false));
  }

  if (!encode_fn()) return LG_ERR_CUDA;
  const int key_tiles_g = cdiv(G, kTileN) + cdiv(L, kTileN);
  const int band_tiles = std::min(cdiv(2LL * r + kTileM, kTileN) + 1, cdiv(L, kTileN)) + cdiv(G, kTileN);
  const bool interleave = grow_interleave_for(4LL * BH * (static_cast<long long>(L) + G) * D);
  const GrowPlan gp = grow_plan(G, key_tiles_g,
                                interleave ? 2 * band_tiles
                                           : choose_grow_split(static_cast<long long>(BH) * band_units_for(L, 1),
                                                               band_tiles, static_cast<long long>(BH) * cdiv(G, kTileM),
                                                               key_tiles_g));
  const WsLayout lay = ws_layout(BH, G, D, gp.n_parts, false, 0, max_units(BH, L, 1, gp));
  TcParams tp{};
  if (!encode_map(&tp.mapQ[0], q_l, D, L, BH, 1) || !encode_map(&tp.mapK[0], k_l, D, L, BH, 1) ||
      !encode_map(&tp.mapV[0], v_l, D, L, BH, 1) || !encode_map(&tp.mapQg, q_g, D, G, BH, 0) ||
      !encode_map(&tp.mapKg, k_g, D, G, BH, 0) || !encode_map(&tp.mapVg, v_g, D, G, BH, 0) ||
      !encode_store_map(&tp.mapO[0], out_l, D, L, BH, 1))
    return LG_ERR_CUDA;
  for (int sl = 1; sl < kMaxSlots; ++sl) {
    tp.mapQ[sl] = tp.mapQ[0]; tp.mapK[sl] = tp.mapK[0]; tp.mapV[sl] = tp.mapV[0]; tp.mapO[sl] = tp.mapO[0];
    tp.slot_dil[sl] = 1;
  }
  tp.mapKgr = tp.mapK[0];
  tp.mapVgr = tp.mapV[0];
  tp.slot_dil[0] = 1;
  tp.slot_units[0] = band_units_for(L, 1);
  for (int h = 0; h < H; ++h) {
    tp.head_slot[h] = 0;
    tp.head_unit_start[h] = h * tp.slot_units[0];
  }
  tp.head_unit_start[H] = H * tp.slot_units[0];
  tp.band_units_per_batch = H * tp.slot_units[0];
  for (int h = 0; h < H; ++h) tp.head_class[h] = -1;
  tp.seg_w = 0;
  tp.seg_causal = 0;
  tp.out = out_l; tp.lse = lse_l;
  tp.part_acc = reinterpret_cast<float*>(ws + lay.acc);
  tp.part_ml = reinterpret_cast<float*>(ws + lay.ml);
  tp.gidx = nullptr; tp.status = status; tp.wait_cap = wait_cap_cycles(); tp.withhold = withhold_for_test();
  tp.unit_counter = status + 1;
  tp.scale_log2 = s * 1.4426950408889634f;
  tp.BH = BH; tp.H = H; tp.N = L; tp.D = D; tp.wl = r; tp.wr = r; tp.n_glob = G; tp.etc = 1;
  tp.n_gtiles = gp.n_gtiles; tp.n_splits = gp.n_splits; tp.n_parts = gp.n_parts;
  tp.n_key_tiles_grow = gp.n_key_tiles; tp.grow_split = std::max(1, gp.split);
  tp.n_grow_units = BH * gp.n_gtiles * gp.n_splits;
  tp.grow_interleave = interleave ? 1 : 0;
  const long long band_units = static_cast<long long>(B) * tp.band_units_per_batch;
  tp.n_tail_split = static_cast<int>(
      std::min(tail_split(static_cast<long long>(tp.n_grow_units) + band_units, band_units), grow_tail_cap(tp)));
  const long long units = static_cast<long long>(tp.n_grow_units) + band_units + tp.n_tail_split;
  if (units > (1LL << 31) - 1) return LG_ERR_UNSUPPORTED;
  if (units > static_cast<long long>(lay.max_units)) return LG_ERR_WORKSPACE;
  tp.units = ws + lay.units;
  if ((e = prof_mark(stream, true)) != cudaSuccess) return LG_ERR_CUDA;
  if ((e = launch_tc(tp, static_cast<int>(units), stream, true)) != cudaSuccess) return LG_ERR_CUDA;
  if ((e = prof_mark(stream, false)) != cudaSuccess) return LG_ERR_CUDA;
  MergeParams mp{};
  mp.part_acc = reinterpret_cast<const float*>(ws + lay.acc);
  mp.part_ml = reinterpret_cast<const float*>(ws + lay.ml);
  mp.out = out_g; mp.lse = lse_g; mp.gidx = nullptr;
  mp.BH = BH; mp.N_out = G; mp.D = D; mp.n_glob = G; mp.n_splits = gp.n_parts;
  if ((e = launch_merge(mp, 1, stream)) != cudaSuccess) return LG_ERR_CUDA;
  return LG_OK;
}

lg_status lg_query_status(const void* workspace, lg_stream_t stream_) {
  if (workspace == nullptr) return LG_ERR_WORKSPACE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return LG_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LG_ERR_CUDA;
  if (word != 0 && cudaMemset(const_cast<void*>(workspace), 0, sizeof(int)) != cudaSuccess) return LG_ERR_CUDA;
  if (word & ST_INTERNAL) return LG_ERR_CUDA;
  if (word & ST_TIMEOUT) return LG_ERR_TIMEOUT;
  if (word & ST_GLOBAL_IDX) return LG_ERR_GLOBAL_IDX;
  if (word & ST_BAD_CODE) return LG_ERR_INVALID_ARG;
  return LG_OK;
}

int64_t lg_count_pairs(int N, int w_left, int w_right, int dilation, int causal, const int32_t* global_idx_host,
                       int n_global) {
  if (N < 1 || w_left < 0 || w_right < 0 || dilation < 1 || n_global < 0 || n_global > N ||
      (n_global > 0 && global_idx_host == nullptr))
    return -1;
  const long long d = dilation;
  const long long wl = std::min(w_left, N), wr = causal ? 0 : std::min(w_right, N);
  std::vector<unsigned char> is_g(N, 0);
  for (int x = 0; x < n_global; ++x) {
    const int p = global_idx_host[x];
    if (p < 0 || p >= N || is_g[p]) return -1;
    is_g[p] = 1;
  }
  // hits[i] = global keys inside the band of row i: walk each global key's band column.
  std::vector<int> hits(N, 0);
  for (int x = 0; x < n_global; ++x) {
    const long long j = global_idx_host[x];
    for (long long t = -wl; t <= wr; ++t) {
      const long long i = j - d * t;
      if (i >= 0 && i < N) ++hits[i];
    }
  }
  int64_t total = 0;
  for (long long i = 0; i < N; ++i) {
    if (is_g[i]) { total += N; continue; }
    // band keys i + d*t, t in [-wl, wr], inside [0, N)
    const long long t_lo = std::max(-wl, -(i / d));
    const long long t_hi = std::min(wr, (N - 1 - i) / d);
    const long long band = std::max(0LL, t_hi - t_lo + 1);
    total += band + (n_global - hits[i]);
  }
  return total;
}

int64_t lg_etc_count_pairs(int L, int G, int radius) {
  if (L < 1 || G < 0 || radius < 0) return -1;
  int64_t band = 0;
  for (long long i = 0; i < L; ++i) {
    const long long lo = std::max(0LL, i - radius), hi = std::min<long long>(L - 1, i + radius);
    band += hi - lo + 1;
  }
  return band + static_cast<int64_t>(L) * G + static_cast<int64_t>(G) * (G + L);
}

lg_status lg_debug_timeout_test(int withhold, long long wait_cap_cycles) {
  if (withhold != 0 && withhold != 1) return LG_ERR_INVALID_ARG;
  g_withhold.store(withhold, std::memory_order_relaxed);
  g_wait_cap_override.store(wait_cap_cycles > 0 ? wait_cap_cycles : 0, std::memory_order_relaxed);
  return LG_OK;
}

lg_status lg_profile_begin(void) {
  Profiler& p = prof();
  p.on = true;
  p.used = 0;
  return LG_OK;
}

lg_status lg_profile_end(float* total_ms, int* launches) {
  Profiler& p = prof();
  float sum = 0.f;
  for (size_t x = 0; x < p.used; ++x) {
    if (cudaEventSynchronize(p.events[x].second) != cudaSuccess) return LG_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.events[x].first, p.events[x].second) != cudaSuccess) return LG_ERR_CUDA;
    sum += ms;
  }
  if (total_ms) *total_ms = sum;
  if (launches) *launches = static_cast<int>(p.used);
  p.on = false;
  p.used = 0;
  return LG_OK;
}

}  // extern "C"
