// Internal declarations shared by the CUDA translation units of liblg_attn.
// Not part of the public ABI (that is include/lg_attn.h).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/lg_attn.h"

namespace lg {

// Device status word bits (workspace offset 0).  The host maps the highest
// set bit to an lg_status.
enum : int {
  ST_GLOBAL_IDX = 1 << 0,
  ST_TIMEOUT = 1 << 1,
  ST_INTERNAL = 1 << 2,   // an internal invariant failed on the device; the work was abandoned
  ST_BAD_CODE = 1 << 3,   // an ETC relative-position label outside the vocabulary
};

constexpr size_t kStatusBytes = 256;     // status area at the head of every workspace
constexpr int kTileM = 128;              // query rows per tile (tcgen05 M)
constexpr int kTileN = 128;              // keys per tile
constexpr int kGrowSplitMax = 32;        // most key tiles per split of a global-query row block (two partials)
constexpr int kMaxSlots = 4;             // distinct dilations per tensor-core launch (slot 0 is d = 1)
constexpr int kMaxPatternSlots = 8;      // LongNet patterns sharing one launch (a slot each)
constexpr int kMaxFusedHeads = 32;       // heads of a LongNet call whose patterns share one launch

// ---------------------------------------------------------------- launch chaining
// The kernels of one call run back to back on one stream.  A kernel launched
// with programmatic stream serialization may start while its predecessor is
// still running (its prologue overlaps the predecessor's tail and the launch
// latency); it calls grid_dep_wait() before it touches anything the
// predecessor writes, and that wait returns once the predecessor has completed
// and its memory is visible.  A chained kernel also waits before it exits, so
// that its completion implies its predecessors'.  grid_dep_launch() lets the
// successor launch early.  Both are no-ops when there is no such predecessor
// or successor.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch on stream s, chained to the stream's previous kernel when `chained`.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool chained,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = chained ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- fp32 CUDA-core path

struct SimtParams {
  const float* q; const float* k; const float* v;   // [BH, N, D] (ETC: long input, N = L)
  const float* qg; const float* kg; const float* vg; // ETC only: global input [BH, G, D]
  float* out; float* lse;                           // [BH, N, D], [BH, N]
  float* out_g; float* lse_g;                       // ETC only
  const int* gidx;                                   // Longformer global positions (device)
  const float* qgl; const float* kgl; const float* vgl;  // Longformer global rows: their projections (= q, k, v if shared)
  int BH, H, N, D;
  int wl, wr;                                        // wr already 0 when causal
  int n_glob;                                        // Longformer: g; ETC: G
  int etc;
  float scale;
  int dil[LG_MAX_HEADS];
  int tile_start[LG_MAX_HEADS + 1];  // prefix over heads of the band-row tiles of one batch
  int* status;                       // device status word (Longformer: a bad global list is reported here)
};

// fp32 backward on the CUDA cores: one warp per query row; dQ written, dK and
// dV accumulated with atomic adds into zeroed outputs.
struct SimtBwdParams {
  const float* q; const float* k; const float* v; const float* out; const float* lse; const float* dout;
  const float* qg; const float* kg; const float* vg; const float* out_g; const float* lse_g; const float* dout_g;
  float* dq; float* dk; float* dv;                   // [BH, N, D]
  float* dq_g; float* dk_g; float* dv_g;             // ETC only: [BH, G, D]
  float* delta;                                      // workspace: [BH, N] (+ [BH, G] for ETC)
  const int* gidx;
  int* status;
  int BH, H, N, D;
  int wl, wr;
  int n_glob;
  int etc;
  float scale;
  int dil[LG_MAX_HEADS];
};

// ---------------------------------------------------------------- bf16 tensor-core path

// One launch covers all batches and the heads whose dilation has a slot here.
// Work units: first the global-query row units (gtile, split) per (b, h), then
// the band units (dilation residue class c, query tile) per (b, h).
// S slots of tensor maps.  The window and ETC paths use S = kMaxSlots, which
// keeps the block within the 4 KB that a launch passes without an extra copy
// of its parameters; the one launch of several LongNet patterns uses
// TcParamsLn below.
template <int S>
struct TcParamsT {
  static constexpr bool kPatterns = false;
  CUtensorMap mapQ[S];           // main q/k/v viewed as {D, N, BH}, rows strided by the slot's dilation
  CUtensorMap mapK[S];
  CUtensorMap mapV[S];
  CUtensorMap mapQg, mapKg, mapVg;  // global side {D, g, BH}: gathered rows (Longformer) or q_g/k_g/v_g (ETC)
  CUtensorMap mapO[S];            // output {D, N, BH}, boxes of 32 rows x 64 columns, rows strided by the slot's dilation
  CUtensorMap mapKgr, mapVgr;     // keys / values of the global-row units over the main sequence {D, N, BH}
                                  // (the separate global projections, or the main k / v)
  void* out;                      // bf16 [BH, N, D]
  float* lse;                     // [BH, N]
  float* part_acc;                // [BH, n_glob, n_parts, D] unnormalised partial outputs
  float* part_ml;                 // [BH, n_glob, n_parts, 2] partial (max, sum), max in log2 units
  void* units;                    // [n_units, 16] int unit records (workspace), written before the kernel
  const int* gidx;                // Longformer global positions (device), for band de-duplication
  const int* gcount;              // Longformer: gcount[x] = number of global positions < x, x in [0, N]
  int* status;
  int* unit_counter;              // units claimed so far (zeroed before the launch)
  int grow_split;                 // key tiles per split of a global-query row block
  int n_tail_split;               // last band units split into two one-tile units each
  int grow_interleave;            // 1: global-row units interleaved with their head's band units
  long long wait_cap;             // clock64 cycles a bounded wait may spin
  int withhold;                   // test of the timeout path: issue no TMA load and no MMA
  float scale_log2;               // scale * log2(e)
  int BH, H, N, D;                // N = L for ETC
  int wl, wr;                     // wr already 0 when causal
  int n_glob;                     // g (Longformer) or G (ETC)
  int etc;
  int n_grow_units;               // global-query row units (placed first)
  int n_gtiles;                   // query tiles of the global rows
  int n_splits;                   // key splits of the global rows
  int n_parts;                    // partial slots per global row (two per split)
  int n_key_tiles_grow;           // key tiles of one global row block (ETC: ceil(G/128) + ceil(L/128))
  int band_units_per_batch;
  int slot_dil[S];
  int slot_units[S];              // band units of one head with this slot's dilation
  unsigned char head_slot[LG_MAX_HEADS];  // 255: head not in this launch
  signed char head_class[LG_MAX_HEADS];   // >= 0: the one residue class this head computes (LongNet offset); -1: all
  // Segment mode (LongNet dilated attention), seg_w > 0: pattern (seg_w,
  // seg_r) over a sequence of seg_n tokens; a row sees the keys of its
  // segment's block (seg_block).  seg_packed = 0: the tensors are the
  // original [BH, N, D] ones, read in class h mod seg_r with stride seg_r;
  // 1: they hold each head's kept rows packed segment after segment
  // (N = the packed length, class 0, stride 1).
  int seg_w, seg_r, seg_n, seg_packed;
  int seg_causal;                 // segment mode: only keys at or before the query
  int head_unit_start[LG_MAX_HEADS + 1];  // prefix of band units over heads (one batch)
};
using TcParams = TcParamsT<kMaxSlots>;

// Several LongNet patterns in one launch (seg_n, seg_causal as above): pattern
// k uses slot k (its tensor maps and slot_dil[k]); its units are
// [pat_unit_start[k], pat_unit_start[k + 1]) of the table, per batch in the
// head order of pat_head_unit_start[k]; its LSE rows go to pat_lse[k],
// pat_rows[k] rows per (b, h) (N, or the packed length).
struct TcParamsLn : TcParamsT<kMaxPatternSlots> {
  static constexpr bool kPatterns = true;
  int n_pat;
  int pat_unit_start[kMaxPatternSlots + 1];
  int pat_w[kMaxPatternSlots], pat_r[kMaxPatternSlots], pat_packed[kMaxPatternSlots], pat_rows[kMaxPatternSlots];
  float* pat_lse[kMaxPatternSlots];
  int pat_head_unit_start[kMaxPatternSlots][kMaxFusedHeads + 1];
};

// LongNet pattern (w, r), head offset s = h mod r: the kept rows of segment i
// are i w + s + t r, 0 <= t < seg_block (those below N).  seg_class_len: the
// kept rows of one head over the sequence (the packed length).
__host__ __device__ inline int seg_block(int w, int r, int s) { return w > s ? (w - s + r - 1) / r : 0; }
__host__ __device__ inline int seg_class_len(int N, int w, int r, int s) {
  const int n_full = N / w, rest = N - n_full * w;
  return n_full * seg_block(w, r, s) + (rest > s ? (rest - s + r - 1) / r : 0);
}

struct MergeParams {
  const float* part_acc; const float* part_ml;
  void* out; float* lse;          // Longformer: out/lse of the main tensor; ETC: out_g/lse_g
  const int* gidx;                // Longformer: scatter rows; NULL for ETC (row r -> row r)
  int BH, N_out, D, n_glob, n_splits;
};

struct PrepParams {
  const int* gidx; int n_glob; int N;
  const __nv_bfloat16* q; const __nv_bfloat16* k; const __nv_bfloat16* v;  // NULL: validate only
                                                                            // (q: the global rows' query projection)
  __nv_bfloat16* qg; __nv_bfloat16* kg; __nv_bfloat16* vg;                 // [BH, g, D]
  int* gcount;                                                              // [N + 1] or NULL
  int BH, D;
  int* status;
};

// ---------------------------------------------------------------- bf16 backward (tensor cores)

// One launch of a backward tensor-core kernel covers the heads of one
// dilation (all batches).  The two kernels share this block:
//  * the q kernel: rows of TMEM are queries; band units are 128-step query
//    tiles of one residue class against their band key tiles and the
//    global-key tiles (dQ written); global-row units are a tile of global
//    queries against one split of all key tiles (partial dQ in `part_a`).
//  * the kv kernel: rows of TMEM are keys; band units are 128-step key tiles
//    of one residue class against the query tiles whose windows reach them
//    and the global-query tiles (dK, dV written); global-key units are a tile
//    of global keys against one split of all query tiles (partial dK in
//    `part_a`, dV in `part_b`).
// "Global" is the Longformer global set (rows gathered by the prep kernel)
// or, for ETC, the separate global input.  Class-major vectors: lse2 / delta
// of (b, h) position c + d*t at [bh * CM + c * M + t].
struct BwdParams {
  CUtensorMap mQ, mK, mV, mdO;      // main input {D, N, BH}, rows strided by d
  CUtensorMap mQG, mKG, mVG, mdOG;  // global side {D, g, BH}
  CUtensorMap sA, sB;               // store maps of the main outputs, rows strided by d (q: dQ; kv: dK, dV)
  const float* lse2;                // LSE * log2(e), class-major [BH][CM]
  const float* delta;               // rowsum(dO * O), class-major [BH][CM]
  const float* lse2g;               // [BH][gpad] of the global rows
  const float* deltag;              // [BH][gpad]
  const int* gidx;                  // Longformer global positions (device); NULL for ETC
  const int* gcount;                // Longformer: gcount[x] = number of global positions < x
  float* part_a;                    // grow-unit partials [BH * g][n_splits][D] (q: dQ; kv: dK)
  float* part_b;                    // kv: dV partials
  int* status;
  long long wait_cap;
  float scale, scale_log2;          // s and s * log2(e)
  int B, H, N, D, wl, wr, d, n_glob, etc, CM, M, gpad;
  int n_heads;                      // heads of this launch
  int heads[LG_MAX_HEADS];
  int tiles_per_head;               // class-major 128-step tiles of one (b, h)
  int n_gt;                         // tiles of the global side
  int n_splits, split;              // grow units: splits of the other side's tiles, tiles per split
  int ns_stride;                    // partial slots per row in part_a / part_b (>= n_splits; unused slots stay 0)
  int other_tiles;                  // tiles of the other side for grow units
  int n_grow, n_band;               // units of this launch (grow units first)
};

struct BwdPrepParams {
  const __nv_bfloat16* out; const __nv_bfloat16* dout; const float* lse;  // main [BH, N, D], [BH, N]
  const __nv_bfloat16* q; const __nv_bfloat16* k; const __nv_bfloat16* v;  // Longformer: gathered at gidx
  const int* gidx;                  // NULL: no gather (ETC or no globals)
  int dil[LG_MAX_HEADS];            // per head dilation
  __nv_bfloat16* qg; __nv_bfloat16* kg; __nv_bfloat16* vg; __nv_bfloat16* dog;  // [BH, g, D]
  float* lse2; float* delta;        // class-major [BH][CM]
  float* lse2g; float* deltag;      // [BH][gpad] (Longformer: gathered rows; ETC: from the global-side inputs)
  const __nv_bfloat16* out_g; const __nv_bfloat16* dout_g; const float* lse_g;  // ETC global side
  int* gcount;                      // [N + 1] or NULL
  int* status;
  int BH, H, N, D, n_glob, CM, gpad, etc;
};

struct BwdReduceParams {
  const float* part_a; const float* part_b;  // [BH * g][n_splits][D]
  void* out_a; void* out_b;                  // bf16 [BH, n_rows_out, D] (b may be NULL)
  const int* gidx;                           // scatter rows (Longformer) or NULL (row r -> r)
  int BH, n_glob, n_rows_out, D, n_splits;
  float scale_a, scale_b;
};

// Host-side launchers (each defined next to its kernel).
cudaError_t launch_simt(const SimtParams& p, cudaStream_t s);
cudaError_t launch_simt_bwd(const SimtBwdParams& p, cudaStream_t s);
// The unit-table kernel and the tensor-core kernel; the table kernel is
// chained to the stream's previous kernel when chain_table (not when that
// kernel may still read the unit table), the tensor-core kernel always is.
cudaError_t launch_tc(const TcParams& p, int n_units, cudaStream_t s, bool chain_table);
cudaError_t launch_tc(const TcParamsLn& p, int n_units, cudaStream_t s, bool chain_table);
cudaError_t launch_merge(const MergeParams& p, int bf16_out, cudaStream_t s);
cudaError_t launch_prep(const PrepParams& p, cudaStream_t s);
cudaError_t launch_bwd_prep(const BwdPrepParams& p, cudaStream_t s);
cudaError_t launch_bwd_q(const BwdParams& p, cudaStream_t s);
cudaError_t launch_bwd_kv(const BwdParams& p, cudaStream_t s);
cudaError_t launch_bwd_reduce(const BwdReduceParams& p, cudaStream_t s);
__host__ __device__ int bwd_class_stride(int N, int d);   // M: class stride of the class-major vectors
int bwd_cm(int N);                     // CM: per-(b, h) length of the class-major vectors
size_t tc_smem_bytes(int D);
// bf16 tensor maps of [BH, rows, D] as {D, rows, BH}: load maps with boxes of
// rows_per_load(d) * d rows (element stride d; d = 0: plain 128-row boxes),
// store maps with boxes of 32 * d rows.
bool encode_map(CUtensorMap* m, const void* base, int D, int rows, int BH, int d);
bool encode_store_map(CUtensorMap* m, void* base, int D, int rows, int BH, int d);
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
// Cap of the bounded work waits (clock64 cycles) and the timeout-test switch,
// as set by lg_debug_timeout_test (default: about one second, no withholding).
long long wait_cap_cycles();
int withhold_for_test();
// Every argument check of lg_attn_fwd but the workspace (sizes, values, pointers).
lg_status validate_fwd_args(const void* q, const void* k, const void* v, const void* out, const float* lse,
                            lg_dtype dt, int B, int H, int N, int D, int w_left, int w_right,
                            const int32_t* dilation, int causal, const int32_t* global_idx, int n_global,
                            bool per_call_head_limit);
// Every argument check of lg_attn_fwd (sizes, values, pointers, workspace),
// without any CUDA call.  per_call_head_limit: also refuse H > LG_MAX_HEADS
// (one kernel call); the host-memory entry point splits larger problems.
lg_status validate_fwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                       lg_dtype dt, int B, int H, int N, int D, int w_left, int w_right, const int32_t* dilation,
                       int causal, const int32_t* global_idx, int n_global, const void* workspace,
                       size_t workspace_bytes, bool per_call_head_limit);
int device_sm_count();
long long device_l2_bytes();
// Whether a launch interleaves its global-row units with the band units: when
// K and V of the launch (kv_bytes) are over four times the L2, the global rows'
// own pass over every key would otherwise be read from HBM a second time.  (At
// about twice the L2, measured, placing the long global-row units first wins.)
inline bool grow_interleave_for(long long kv_bytes) { return kv_bytes > 4 * device_l2_bytes(); }
// Band units of a launch of `units` units to split into one-tile halves (the last round).
long long tail_split(long long units, long long band_units);
// The tail split may only take band units: with global-row units interleaved,
// at most the band units after the last head's last key split.
long long grow_tail_cap(const TcParams& tp);
// Profiling of the tensor-core launches (lg_profile_begin/end): events around a launch.
cudaError_t prof_mark(cudaStream_t s, bool start);  // SMs of the current device (cached per device)

}  // namespace lg
