// bf16 window + dilation + global attention forward on the 5th-generation
// tensor cores (tcgen05 MMA with TMEM accumulators, TMA operand loads).
//
// Method: "Longformer: The Long-Document Transformer", section 3.4 ("Sliding
// Window Attention", "Dilated Sliding Window Attention", "Global Attention",
// causal mode from "Autoregressive Language Modeling Configuration"), and
// "ETC: Encoding Long and Structured Inputs in Transformers", section 3.4
// ("Global-Local Attention", "Softmax unification").
//
// The kernel is persistent: one CTA per SM claims the work units of a table
// built before the launch one at a time from a global counter.  A unit has
// two 128-row query tiles (q = 0, 1), each owned by its own softmax
// warpgroup, against a list of 128-key tiles:
//  * Band unit: query steps t0 .. t0+255 of one dilation residue class c
//    (positions c + d*t).  Inside a class the dilated window is the contiguous
//    step range [t - w_left, t + w_right]; the key tiles are the contiguous
//    class rows intersecting the union of the two tiles' windows, fetched by
//    TMA with an element stride of d along the row dimension (the dilation is
//    folded into the TMA coordinates).  Each K/V tile is loaded once and used
//    by both query tiles (a query tile skips tiles outside its own windows).
//    The global-key tiles follow; a global key already inside a row's band is
//    masked there (it counts once).
//  * Global-row unit: 128 global queries against one split of all keys; the
//    two query tiles hold the same rows and take alternate key tiles, and
//    each writes partial softmax statistics that a merge kernel combines.
// Warp roles (384 threads): warp 0 issues the K loads, warp 2 the V loads
// (TMA); warp 1 owns TMEM and issues the MMAs and Q loads of query tile 0,
// warp 3 those of tile 1; warps 4..7 and 8..11 are the two softmax
// warpgroups (one thread per query row = TMEM lane).  For D = 128 warp 0
// issues both K and V into one ring.  TMEM holds S_q (128 fp32 columns) and
// O_q (D columns) for both tiles, and for D = 64 also P_q (packed bf16, 64
// columns); for D = 128 P_q is in shared memory.  S_q takes the next key tile's QK as soon as the
// softmax has read it, so the tensor core computes S_q(j+1) while the
// softmax of tile j runs, and PV_q(j) follows once P_q(j) is written; the
// softmax waits for PV_q(j) before it rescales O_q or writes P_q(j+1).
#include <atomic>
#include <mutex>

#include "lg_internal.h"
#include "lg_ptx.cuh"

namespace lg {
namespace {

constexpr int kThreads = 384;
// Register split between the warpgroups (setmaxnreg): the producer/MMA
// warpgroup gives registers to the two softmax warpgroups.  The launch holds
// kThreads x (registers per thread at launch); the split must fit in it.
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 216;
constexpr int kRegsLaunchMin = (128 * kRegsControl + 256 * kRegsSoftmax + kThreads - 1) / kThreads;
constexpr float kRescaleThreshold = 8.0f;  // log2 units; O is rescaled only when the max grows more
constexpr int kUnitSlots = 4;              // ring of claimed unit indices
constexpr int kTailRounds = 2;             // rounds of units claimed dynamically at the end
constexpr float kLn2 = 0.6931471805599453f;
// Bound of the drain waits, which hold a CTA until the TMA loads and MMAs it
// has already issued complete (always finite) before TMEM and shared memory
// are released: fixed, about two seconds, and independent of the cap of the
// work waits (which a caller may shorten).
constexpr long long kDrainCap = 4000000000LL;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTileM * D * 2;      // 128 rows x D bf16
  // Where P goes, so that QK_q of the next key tile can overwrite S_q as soon
  // as the softmax has read it (S, P and O of two query tiles do not fit the
  // 512 TMEM columns twice over).  D = 64: P_q in its own 64 TMEM columns.
  // D = 128: P_q in shared memory, one 32 KB buffer per query tile; K and V
  // then share one ring of three tiles, loaded in the order the MMAs take
  // them (K(0), then K(j) and V(j - 1) for each later j, then V(last)), and
  // the epilogue stages O in the query tile's own P buffer.
  static constexpr bool kSplitP = (D == 64);
  static constexpr bool kPSmem = (D == 128);
  static constexpr int kKStages = kPSmem ? 3 : 4;        // D = 128: the shared K/V ring
  static constexpr int kVStages = kPSmem ? 0 : 4;
  static constexpr int kOffQ = 0;                        // two query tiles
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  // D = 64: output staging, 4 KB per softmax warp; D = 128: P_0 and P_1.
  static constexpr int kOffStage = kOffV + kVStages * kTileBytes;
  static constexpr int kPBytes = kTileM * kTileN * 2;
  static constexpr int kOffMisc = kOffStage + (kPSmem ? 2 * kPBytes : 8 * 4096);
  static constexpr int kMiscBytes = 1024;
  static constexpr int kSmem = kOffMisc + kMiscBytes + 1024;  // +1024: base alignment slack
  // Readers of a unit slot: both issuing warps, the eight softmax warps and
  // (two rings) the V producer.
  static constexpr int kUnitReaders = kPSmem ? 10 : 11;
  // TMEM columns: S_q at 128 q; D = 64: P_q at 256 + 64 q, O_q at 384 + 64 q;
  // D = 128: O_q at 256 + 128 q.
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColP = 256;
  static constexpr uint32_t kPStride = 64;
  static constexpr uint32_t kColO = kSplitP ? 384 : 256;
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

// Rows one strided TMA box delivers for a dilation d (box height R*d <= 256).
__host__ __device__ __forceinline__ int rows_per_load(int d) {
  return d <= 2 ? 128 : (d <= 4 ? 64 : 32);
}

struct Unit {
  int grow;          // 1: global-row unit, 0: band unit
  int bh;
  int slot, d, c;    // band: dilation slot, stride, residue class
  int t0, n_c;       // band: first query step of tile 0, class length
  int band_lo;       // band: first key step of the tiles
  int n_band;        // band: band key tiles
  int kt0;           // grow: first key tile of the split
  int grow0;         // grow: first global row of the tile
  int n_tiles;
  int first[2], last[2];  // band: range of band tiles each query tile needs (first > last: none)
  int active[2];
  int seg;           // band, segment mode: class steps of a segment block (0: window mode)
};

// Unit u of a launch of n_units from its index (the arithmetic behind the
// unit table: a scan over heads and residue classes, with divisions; run once
// per unit per call).  The last n_tail_split band units are each split into
// two one-tile units, which come last (u = n_full + 2 i + h: rows t0 + 128 h
// of band unit n_full + i, worked by query tile 0), so that the last round of
// a launch can spread over more CTAs.
template <class P>
__device__ Unit decode_unit_slow(const P& p, int u, int n_units) {
  Unit w{};
  const int n_full = n_units - 2 * p.n_tail_split;
  int half = -1;
  if (u >= n_full) {
    half = (u - n_full) & 1;
    u = n_full + ((u - n_full) >> 1);
  }
  if constexpr (P::kPatterns) {
    // Several LongNet patterns: pattern k's units, then per batch and head as
    // for one pattern (one residue class per head, offset h mod r, in slot k).
    int k = 0;
    while (k + 1 < p.n_pat && p.pat_unit_start[k + 1] <= u) ++k;
    const int* hs = p.pat_head_unit_start[k];
    int rem = u - p.pat_unit_start[k];
    const int b = rem / hs[p.H];
    rem -= b * hs[p.H];
    int h = 0;
    while (h + 1 < p.H && hs[h + 1] <= rem) ++h;
    rem -= hs[h];
    const int pw = p.pat_w[k], pr = p.pat_r[k], s = h % pr;
    w.grow = 0;
    w.bh = b * p.H + h;
    w.slot = k;
    w.d = p.slot_dil[k];
    w.seg = p.pat_packed[k] ? seg_block(pw, pr, s) : pw / pr;
    w.c = p.pat_packed[k] ? 0 : s;
    w.n_c = p.pat_packed[k] ? seg_class_len(p.seg_n, pw, pr, s) : (p.seg_n - s + w.d - 1) / w.d;
    w.t0 = rem * 2 * kTileM;
  } else {
    // Two orders.  Global-row units first (the longest units start first), when
    // the launch's K and V fit in L2 anyway.  Otherwise, per (batch, head) block,
    // the head's band units with its global-row units interleaved in key order
    // (the n_gtiles units of key split s before band unit floor(nb s / n_splits)),
    // so that units reading the same K/V tiles run in the same round and share
    // them through L2 instead of reading them from HBM twice.
    const bool first = p.n_grow_units > 0 && !p.grow_interleave;
    if (first && u < p.n_grow_units) {
      w.grow = 1;
      const int split = u % p.n_splits;
      const int r = u / p.n_splits;
      w.grow0 = (r % p.n_gtiles) * kTileM;
      w.bh = r / p.n_gtiles;
      w.kt0 = split * p.grow_split;
      w.n_tiles = min(p.grow_split, p.n_key_tiles_grow - w.kt0);
      w.slot = 0; w.d = 1;
      w.active[0] = 1; w.active[1] = w.n_tiles > 1;
      return w;
    }
    if (first) u -= p.n_grow_units;
    const int gu = (p.n_grow_units > 0 && !first) ? p.n_gtiles * p.n_splits : 0;   // interleaved units per (b, h)
    const int per_batch = p.band_units_per_batch + p.H * gu;
    const int b = u / per_batch;
    int rem = u - b * per_batch;
    int h = 0;
    while (h + 1 < p.H && p.head_unit_start[h + 1] + (h + 1) * gu <= rem) ++h;
    rem -= p.head_unit_start[h] + h * gu;
    if (gu > 0) {
      const long long nb = p.head_unit_start[h + 1] - p.head_unit_start[h];
      int split = -1, gt = 0, band = rem - p.n_splits * p.n_gtiles;
      for (int sp = 0; sp < p.n_splits; ++sp) {
        const int st = static_cast<int>(nb * sp / p.n_splits) + sp * p.n_gtiles;
        if (rem < st) { band = rem - sp * p.n_gtiles; break; }
        if (rem < st + p.n_gtiles) { split = sp; gt = rem - st; break; }
      }
      if (split >= 0) {
        w.grow = 1;
        w.grow0 = gt * kTileM;
        w.bh = b * p.H + h;
        w.kt0 = split * p.grow_split;
        w.n_tiles = min(p.grow_split, p.n_key_tiles_grow - w.kt0);
        w.slot = 0; w.d = 1;
        w.active[0] = 1; w.active[1] = w.n_tiles > 1;
        return w;
      }
      rem = band;
    }
    w.grow = 0;
    w.bh = b * p.H + h;
    w.slot = p.head_slot[h];
    w.d = p.slot_dil[w.slot];
    w.seg = 0;
    if (p.seg_w > 0) {            // LongNet: one residue class per head (offset h mod r)
      const int s = h % p.seg_r;
      w.seg = p.seg_packed ? seg_block(p.seg_w, p.seg_r, s) : p.seg_w / p.seg_r;
      w.c = p.seg_packed ? 0 : s;
      w.n_c = p.seg_packed ? seg_class_len(p.seg_n, p.seg_w, p.seg_r, s) : (p.N - s + w.d - 1) / w.d;
      w.t0 = rem * 2 * kTileM;
    } else if (p.head_class[h] >= 0) {
      w.c = p.head_class[h];
      w.n_c = (p.N - w.c + w.d - 1) / w.d;
      w.t0 = rem * 2 * kTileM;
    } else {
      for (int c = 0; c < w.d; ++c) {
        const int n_c = (p.N - c + w.d - 1) / w.d;
        const int units = (n_c + 2 * kTileM - 1) / (2 * kTileM);
        if (rem < units) { w.c = c; w.n_c = n_c; w.t0 = rem * 2 * kTileM; break; }
        rem -= units;
      }
    }
  }
  const int span = half >= 0 ? 1 : 2;                 // query tiles of this unit
  if (half > 0) w.t0 += kTileM;
  if (w.n_c <= 0 || w.t0 >= w.n_c) { w.n_tiles = 0; return w; }
  const int t_last = min(w.t0 + span * kTileM - 1, w.n_c - 1);
  // key steps of a query step t: [t - w_left, t + w_right], or in segment
  // mode its block [B floor(t / B), B floor(t / B) + B - 1] (up to t if causal)
  const int B = w.seg;
  w.band_lo = B > 0 ? (w.t0 / B) * B : max(0, w.t0 - p.wl);
  const int band_hi = min(w.n_c - 1, B > 0 ? (p.seg_causal ? t_last : (t_last / B) * B + B - 1) : t_last + p.wr);
  w.n_band = (band_hi - w.band_lo + kTileN) / kTileN;
  const int n_gt = (p.n_glob + kTileN - 1) / kTileN;
  w.n_tiles = w.n_band + n_gt;
  for (int q = 0; q < 2; ++q) {
    const int a = w.t0 + q * kTileM;
    w.active[q] = q < span && a < w.n_c;
    if (!w.active[q]) { w.first[q] = 1; w.last[q] = 0; continue; }
    const int b_ = min(a + kTileM - 1, w.n_c - 1);
    const int klo = B > 0 ? (a / B) * B : max(0, a - p.wl);
    const int khi = min(w.n_c - 1, B > 0 ? (p.seg_causal ? b_ : (b_ / B) * B + B - 1) : b_ + p.wr);
    w.first[q] = (klo - w.band_lo) / kTileN;
    w.last[q] = (khi - w.band_lo) / kTileN;
  }
  return w;
}

// Unit records: 16 ints per unit, built once per launch by unit_table_kernel,
// so that a CTA reads a unit with four 16-byte loads.
template <class P>
__global__ void unit_table_kernel(const __grid_constant__ P p, int n_units) {
  grid_dep_launch();   // the tensor-core kernel may start its prologue
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += gridDim.x * blockDim.x) {
    const Unit w = decode_unit_slow(p, u, n_units);
    int4* rec = reinterpret_cast<int4*>(p.units) + 4 * static_cast<size_t>(u);
    const int flags = w.grow | (w.slot << 1) | (w.active[0] << 4) | (w.active[1] << 5) | (w.d << 8) | (w.c << 16);
    rec[0] = make_int4(w.bh, flags, w.t0, w.n_c);
    rec[1] = make_int4(w.band_lo, w.n_band, w.kt0, w.grow0);
    rec[2] = make_int4(w.n_tiles, w.first[0], w.first[1], w.last[0]);
    rec[3] = make_int4(w.last[1], w.grow ? 0 : w.seg, 0, 0);
  }
  grid_dep_wait();     // complete only after the call's earlier kernels
}

// Brings unit u's 64-byte record into this SM's L1 (shared by every warp of
// the CTA), so that the decode at the start of that unit does not wait for L2.
template <class P>
__device__ __forceinline__ void prefetch_unit(const P& p, int u) {
  if (u >= 0)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<const int4*>(p.units) + 4 * static_cast<size_t>(u)));
}

template <class P>
__device__ __forceinline__ Unit decode_unit(const P& p, int u) {
  const int4* rec = reinterpret_cast<const int4*>(p.units) + 4 * static_cast<size_t>(u);
  const int4 a = __ldg(rec), b = __ldg(rec + 1), c = __ldg(rec + 2), d = __ldg(rec + 3);
  Unit w;
  w.bh = a.x;
  w.grow = a.y & 1;
  w.slot = (a.y >> 1) & 7;
  w.active[0] = (a.y >> 4) & 1;
  w.active[1] = (a.y >> 5) & 1;
  w.d = (a.y >> 8) & 255;
  w.c = (a.y >> 16) & 255;
  w.t0 = a.z;
  w.n_c = a.w;
  w.band_lo = b.x;
  w.n_band = b.y;
  w.kt0 = b.z;
  w.grow0 = b.w;
  w.n_tiles = c.x;
  w.first[0] = c.y;
  w.first[1] = c.z;
  w.last[0] = c.w;
  w.last[1] = d.x;
  w.seg = d.y;
  return w;
}

// The tile list of one query tile in scalars (a runtime q indexing the
// Unit's arrays would move the whole Unit to local memory).
struct TileView {
  int grow, active, first, last, n_band, q;
  __device__ __forceinline__ bool uses(int j) const {
    const bool in_band = (j >= first) & (j <= last);
    const bool global_tile = j >= n_band;
    return grow ? (((j ^ q) & 1) == 0) : (active & (in_band | global_tile));
  }
};

__device__ __forceinline__ TileView tile_view(const Unit& w, int q) {
  TileView v;
  v.grow = w.grow; v.n_band = w.n_band; v.q = q;
  v.active = q ? w.active[1] : w.active[0];
  v.first = q ? w.first[1] : w.first[0];
  v.last = q ? w.last[1] : w.last[0];
  return v;
}

// Issues the TMA loads of one 128-row operand tile.  strided: the
// dilation-strided view of a slot; otherwise a plain view.
template <int D>
__device__ __forceinline__ void load_tile(const CUtensorMap* map, bool strided, int d, int y0, int bh,
                                          uint32_t dst, uint32_t bar) {
  const int R = strided ? rows_per_load(d) : kTileM;
#pragma unroll
  for (int blk = 0; blk < D / 64; ++blk) {
    for (int piece = 0; piece < kTileM / R; ++piece) {
      tma_load_3d(dst + blk * (kTileM * 128) + piece * R * 128, map, bar, blk * 64,
                  y0 + piece * R * (strided ? d : 1), bh);
    }
  }
}

// Bits of the columns [lo, hi] that fall in the 32-column word starting at `base`.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int base) {
  const int a = max(lo - base, 0), b = min(hi - base, 31);
  if (a > b) return 0u;
  const uint32_t upper = (b >= 31) ? 0xFFFFFFFFu : ((1u << (b + 1)) - 1u);
  return upper & ~((1u << a) - 1u);
}

// Cold paths of the softmax tile loop, out of line so that the loop's code stays compact.
// O_q *= f, 32 columns at a time (every lane of the warp calls it).
__device__ __noinline__ void rescale_o(uint32_t tO, float f, int n32) {
#pragma unroll 1
  for (int cc = 0; cc < n32; ++cc) {
    float o[32];
    tmem_ld32(tO + cc * 32, o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] *= f;
    tmem_st32(tO + cc * 32, o);
  }
}
// Columns [ca, cb) of a global tile starting at list index jj0 whose position is on the
// stride-d lattice of pos_q, as bits of four 32-column words.
__device__ __noinline__ uint4 lattice_bits(const int* gidx, int jj0, int ca, int cb, int pos_q, int d) {
  uint32_t b[4] = {0u, 0u, 0u, 0u};
#pragma unroll 1
  for (int c = ca; c < cb; ++c)
    if ((__ldg(gidx + jj0 + c) - pos_q) % d == 0) b[c >> 5] |= 1u << (c & 31);
  return make_uint4(b[0], b[1], b[2], b[3]);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Where key/value tile j of unit w comes from: the tensor map, whether it is
// the dilation-strided view, and the row coordinate.
template <class P>
__device__ __forceinline__ void tile_source(const P& p, const Unit& w, int j, bool is_k, int gt_src,
                                            const CUtensorMap*& m, bool& strided, int& y) {
  if (!w.grow) {
    if (j < w.n_band) {
      m = is_k ? &p.mapK[w.slot] : &p.mapV[w.slot]; strided = true;
      y = w.c + w.d * (w.band_lo + j * kTileN);
    } else {
      m = is_k ? &p.mapKg : &p.mapVg; strided = false;
      y = (j - w.n_band) * kTileN;
    }
  } else {
    const int kt = w.kt0 + j;
    if (p.etc && kt < gt_src) {
      m = is_k ? &p.mapKg : &p.mapVg; strided = false; y = kt * kTileN;
    } else {
      m = is_k ? &p.mapKgr : &p.mapVgr; strided = true;   // d = 1 view of the main sequence
      y = (kt - (p.etc ? gt_src : 0)) * kTileN;
    }
  }
}

template <int D, class P>
__global__ void __launch_bounds__(kThreads, 1) tc_attn_kernel(const __grid_constant__ P p, int n_units) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV;
  unsigned char* misc = smem + C::kOffMisc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  constexpr int KS = C::kKStages, VS = C::kVStages;
  constexpr int B_QFULL = 0, B_KFULL = 2, B_KEMPTY = B_KFULL + KS, B_VFULL = B_KEMPTY + KS,
                B_VEMPTY = B_VFULL + VS, B_SFULL = B_VEMPTY + VS, B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2,
                B_OFREE = B_ODONE + 2, B_FIN = B_OFREE + 2, B_SEMPTY = B_FIN + 2, B_PEMPTY = B_SEMPTY + 2,
                B_UFULL = B_PEMPTY + 2, B_UEMPTY = B_UFULL + kUnitSlots, NBARS = B_UEMPTY + kUnitSlots;
  static_assert(NBARS * 8 <= 512, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 516);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(misc + 528);  // claimed unit indices
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) {
      uint32_t count = 1;
      if (i == B_PFULL || i == B_PFULL + 1 || i == B_OFREE || i == B_OFREE + 1 || i == B_SEMPTY ||
          i == B_SEMPTY + 1)
        count = 128;
      // K/V stages are released by both MMA issuers (one arrival each; each
      // issuer waits on every stage it releases, so none falls two phases behind).
      if ((i >= B_KEMPTY && i < B_KEMPTY + KS) || (i >= B_VEMPTY && i < B_VEMPTY + VS)) count = 2;
      // A unit slot is read by each of its readers once.
      if (i >= B_UEMPTY && i < B_UEMPTY + kUnitSlots) count = C::kUnitReaders;
      mbar_init(bar(i), count);
    }
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
  // Everything above overlaps the previous kernel; the unit table, the unit
  // counter and the gathered global rows are read only after it completes.
  grid_dep_wait();
  grid_dep_launch();
  const long long cap = p.wait_cap;
  const int gt_src = (p.n_glob + kTileN - 1) / kTileN;

  // Work units (cost-ordered: global-row units first).  Turns k < k_static
  // take the fixed unit blockIdx.x + k * gridDim.x; the units of the last
  // rounds are claimed one at a time from a global counter, so CTAs that drew
  // short units take more of them and the CTAs end together.  The K producer
  // picks; the unit of a CTA's k-th turn goes to slot k % 4 of a ring in
  // shared memory (UFULL: written; UEMPTY: every reader has it).  A slot holds
  // -1 once the units are exhausted.  Every reader takes the slots in order,
  // so a parity wait on a slot always refers to its latest phase.  Waits on a
  // slot: all lanes of the calling warp (or the single thread).
  // (Several LongNet patterns: every unit is claimed, since their lengths
  // vary from one key tile to a whole segment block.)
  const int k_static = P::kPatterns ? 0 : max(0, n_units / static_cast<int>(gridDim.x) - kTailRounds);
  auto slot_wait = [&](int k) -> bool {
    return mbar_wait(bar(B_UFULL + (k % kUnitSlots)), (k / kUnitSlots) & 1, abort_flag, cap);
  };

  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.status, ST_TIMEOUT);
  };
  // Query tile q of unit w into Q slot q (global-row units: the same rows in both slots).
  auto load_q = [&](int q, const Unit& w) {
    const uint32_t dst = sQ + q * C::kTileBytes;
    mbar_arrive_expect_tx(bar(B_QFULL + q), C::kTileBytes);
    if (w.grow) load_tile<D>(&p.mapQg, false, 1, w.grow0, w.bh, dst, bar(B_QFULL + q));
    else load_tile<D>(&p.mapQ[w.slot], true, w.d, w.c + w.d * (w.t0 + q * kTileM), w.bh, dst, bar(B_QFULL + q));
  };

  if (warp < 4) {
  setmaxnreg_dec<kRegsControl>();
  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ K and V producers
    // Warp 0 loads the K ring, warp 2 the V ring, over all units of this CTA
    // (one global tile counter, so a ring never drains between units).  With
    // the shared K/V ring (D = 128) warp 0 loads both, warp 2 idles.
    if (lane == 0 && !(C::kPSmem && warp == 2)) {
      const bool is_k = (warp == 0);
      const int S = is_k ? KS : VS;
      const int b_full = is_k ? B_KFULL : B_VFULL, b_empty = is_k ? B_KEMPTY : B_VEMPTY;
      const uint32_t ring = is_k ? sK : sV;
      int g = 0, issued = 0;
      bool ok = true;
      // The K producer picks the units and publishes them; the V producer reads them.
      auto claim = [&](int k) -> int {
        if (k < k_static) return static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        const int c = k_static * static_cast<int>(gridDim.x) + atomicAdd(p.unit_counter, 1);
        return c < n_units ? c : -1;
      };
      auto publish = [&](int k, int v) -> bool {
        const int sl = k % kUnitSlots;
        if (k >= kUnitSlots && !mbar_wait(bar(B_UEMPTY + sl), ((k / kUnitSlots) - 1) & 1, abort_flag, cap))
          return false;
        unit_ring[sl] = v;
        mbar_arrive(bar(B_UFULL + sl));
        return true;
      };
      auto take = [&](int k, int& v) -> bool {
        if (!slot_wait(k)) return false;
        v = unit_ring[k % kUnitSlots];
        mbar_arrive(bar(B_UEMPTY + k % kUnitSlots));
        return true;
      };
      int u = -1;
      ok = is_k ? publish(0, u = claim(0)) : take(0, u);
      if (!ok) fail();
      for (int k = 0; ok && u >= 0; ++k) {
        int un = -1;
        if (is_k) {
          if (!publish(k + 1, un = claim(k + 1))) { fail(); ok = false; break; }
          prefetch_unit(p, un);   // every role decodes it at its next unit
        }
        const Unit w = decode_unit(p, u);
        // Tile j of the unit (K or V) into the next ring slot.
        auto put = [&](int j, bool kk) -> bool {
          const CUtensorMap* m;
          bool strided;
          int y;
          tile_source(p, w, j, kk, gt_src, m, strided, y);
          const int st = g % S;
          if (g >= S && !mbar_wait(bar(b_empty + st), ((g / S) - 1) & 1, abort_flag, cap)) return false;
          mbar_arrive_expect_tx(bar(b_full + st), C::kTileBytes);
          load_tile<D>(m, strided, strided ? w.d : 1, y, w.bh, ring + st * C::kTileBytes, bar(b_full + st));
          issued = ++g;
          return true;
        };
        // (p.withhold: a test of the timeout path; no load is issued, so the
        // consumers' first wait runs out with nothing in flight.)
        if (C::kPSmem) {
          // The shared ring, in the order the MMAs take the tiles: K(x), then V(x - 1).
          for (int x = 0; x <= w.n_tiles && !p.withhold; ++x) {
            if (x < w.n_tiles && !put(x, true)) { fail(); ok = false; break; }
            if (x >= 1 && !put(x - 1, false)) { fail(); ok = false; break; }
          }
        } else {
          for (int j = 0; j < w.n_tiles && !p.withhold; ++j) {
            if (!put(j, is_k)) { fail(); ok = false; break; }
          }
        }
        if (ok && !is_k && !take(k + 1, un)) { fail(); ok = false; }
        u = un;
      }
      // Drain: every load issued here has landed before the CTA exits (these
      // waits ignore the abort flag and are bounded by the cap alone).
      for (int x = max(0, issued - S); x < issued; ++x)
        mbar_wait(bar(b_full + x % S), (x / S) & 1, nullptr, kDrainCap);
    }
  } else {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the MMAs of query tile 0, warp 3 those of tile 1.  Each
    // issuing warp runs its loop converged (every lane waits, so the loop
    // state stays warp-uniform) and one elected lane issues every MMA, commit,
    // arrival and Q load (the same lane throughout: tcgen05 ordering and
    // commit tracking are per thread).  A tile's QK_q(j) goes first, as soon
    // as the softmax has read S_q of its previous tile, and the PV of that
    // previous tile follows once its P_q is written; the two issuers do not
    // wait for each other, so one tile's softmax overlaps the other tile's
    // MMAs.  Every ring phase is observed by both issuers in the order the
    // producer fills the ring (a parity wait is only sound once the barrier's
    // previous phase has been seen); a tile an issuer does not use is
    // released by it at once, a used one after its MMAs (commit).  The issuer
    // reloads its Q slot for the next unit as soon as its last QK of the unit
    // has completed, and a unit's first PV (which overwrites O) waits until
    // the softmax warpgroup has read the previous unit's O.
    // Every descriptor is precomputed: a K-major step adds 32 B (2 in 16-B
    // units) inside a 128-B row and 16 KB per 64-column block, an MN-major V
    // step adds 2 KB, a stage adds one tile; shared-memory addresses stay
    // below 256 KB, so the additions never carry out of the 14-bit address
    // field.
    constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, true);
    constexpr uint64_t kStage = C::kTileBytes >> 4;
    const int q = warp >> 1;
    const bool leader = elect_one();
    const uint64_t dQ = sdesc_sw128(sQ + q * C::kTileBytes, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(C::kPSmem ? sK : sV, kTileN * 128, 1024);
    const uint64_t dP = sdesc_sw128(sbase + C::kOffStage + q * C::kPBytes, 16, 1024);   // P_q in shared memory
    const uint32_t tS = tmem + C::kColS + q * 128;
    const uint32_t tP = tmem + C::kColP + q * C::kPStride;                             // P_q in TMEM
    const uint32_t tO = tmem + C::kColO + q * D;
    int g = 0, ks = 0, kph = 0;   // two rings: key tiles seen (all units), K stage of tile g and its phase parity
    int gr = 0;                   // shared ring: loads seen (all units)
    int ns = 0;                   // QKs issued
    int npv = 0;                  // PVs issued
    int nact = 0;                 // units in which this query tile was active
    int q_loads = 0, q_seen = 0;
    bool ok = true;
    auto wait_or_fail = [&](int b, int parity) -> bool {
      if (__all_sync(0xffffffffu, mbar_wait(bar(b), parity, abort_flag, cap))) return true;
      if (leader) fail();
      ok = false;
      return false;
    };
    // The unit of this CTA's k-th turn (all lanes wait on the slot; -1 after a failed wait).
    auto unit_in_slot = [&](int k) -> int {
      if (!wait_or_fail(B_UFULL + (k % kUnitSlots), (k / kUnitSlots) & 1)) return -1;
      const int v = unit_ring[k % kUnitSlots];
      __syncwarp();
      if (leader) mbar_arrive(bar(B_UEMPTY + k % kUnitSlots));   // this warp has read slot k
      return v;
    };
    int u = unit_in_slot(0);
    if (u >= 0 && !p.withhold) {   // withhold: no Q load and (no K tile arrives) no MMA
      if (leader) load_q(q, decode_unit(p, u));
      __syncwarp();
      ++q_loads;
    }
    for (int k = 0; ok && u >= 0; ++k) {
      // The next unit is published before this unit's first K tile is loaded.
      const int un = unit_in_slot(k + 1);
      if (!ok) break;
      const Unit w = decode_unit(p, u);
      const TileView tv = tile_view(w, q);
      int last = -1;
      for (int j = w.n_tiles - 1; j >= 0; --j)
        if (tv.uses(j)) { last = j; break; }
      bool first_pv = true, q_ready = false;
      // S_q = Q_q K^T with K in stage st; leader only.
      auto qk_mmas = [&](int st) {
        const uint64_t dk = dK0 + st * kStage;
        umma_bf16_ss(tS, dQ, dk, kIdQK, 0u);
#pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (kTileM * 128) + (kk & 3) * 32) >> 4);
          umma_bf16_ss(tS, dQ + o, dk + o, kIdQK, 1u);
        }
        umma_commit(bar(B_SFULL + q));
        umma_commit(bar(B_KEMPTY + st));
      };
      // O_q += P_q V with V in stage vs; leader only.  The commits: O_q
      // complete (last PV of the unit), the V stage free, P_q free (and O_q
      // idle for a rescale).
      auto pv_mmas = [&](int vs, bool unit_last) {
        const uint64_t dv = dV0 + vs * kStage;
        if constexpr (C::kPSmem) {
          // P from its buffer: K-major, 128-byte swizzle, the Q tile's layout
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (kTileM * 128) + (kk & 3) * 32) >> 4);
            umma_bf16_ss(tO, dP + o, dv + kk * 128, kIdPV, (first_pv && kk == 0) ? 0u : 1u);
          }
        } else {
          umma_bf16_ts(tO, tP, dv, kIdPV, first_pv ? 0u : 1u);
#pragma unroll
          for (int kk = 1; kk < kTileN / 16; ++kk) umma_bf16_ts(tO, tP + kk * 8, dv + kk * 128, kIdPV, 1u);
        }
        if (unit_last) umma_commit(bar(B_ODONE + q));
        umma_commit(bar(C::kPSmem ? B_KEMPTY + vs : B_VEMPTY + vs));
        umma_commit(bar(B_PEMPTY + q));
      };
      // QK_q of a tile: once the softmax has read the previous S_q and Q_q has landed.
      auto qk_step = [&](int st) -> bool {
        if (ns > 0 && !wait_or_fail(B_SEMPTY + q, (ns - 1) & 1)) return false;
        if (!q_ready) {
          if (!wait_or_fail(B_QFULL + q, q_seen & 1)) return false;
          ++q_seen;
          q_ready = true;
        }
        tc_fence_after();
        if (leader) qk_mmas(st);
        __syncwarp();
        ++ns;
        return true;
      };
      // PV_q of tile jp (its V in stage vs): once the O slot is free (first PV
      // of a unit) and P_q is written, which is usually the latest.
      auto pv_step = [&](int vs, int jp) -> bool {
        if (first_pv && nact > 0 && !wait_or_fail(B_OFREE + q, (nact - 1) & 1)) return false;
        if (!wait_or_fail(B_PFULL + q, npv & 1)) return false;
        tc_fence_after();
        if (leader) pv_mmas(vs, jp == last);
        __syncwarp();
        first_pv = false;
        ++npv;
        return true;
      };
      // The Q slot is free once QK_q of the unit's last tile has completed: load the next unit's tile.
      auto reload_q = [&]() -> bool {
        if (!wait_or_fail(B_SFULL + q, (ns - 1) & 1)) return false;
        if (leader) load_q(q, decode_unit(p, un));
        __syncwarp();
        ++q_loads;
        return true;
      };
      if constexpr (C::kPSmem) {
        // The shared ring, in the producer's order: K(x), then V(x - 1).
        for (int x = 0; x <= w.n_tiles; ++x) {
          if (x < w.n_tiles) {
            const int st = gr % KS;
            if (!wait_or_fail(B_KFULL + st, (gr / KS) & 1)) break;
            ++gr;
            if (tv.uses(x)) {
              if (!qk_step(st)) break;
            } else {
              if (leader) mbar_arrive(bar(B_KEMPTY + st));
              __syncwarp();
            }
          }
          if (x >= 1) {
            const int st = gr % KS;
            if (!wait_or_fail(B_KFULL + st, (gr / KS) & 1)) break;
            ++gr;
            if (tv.uses(x - 1)) {
              if (!pv_step(st, x - 1)) break;
            } else {
              if (leader) mbar_arrive(bar(B_KEMPTY + st));
              __syncwarp();
            }
          }
          if (x == last && un >= 0 && !reload_q()) break;
        }
      } else {
        // Two rings: QK_q(j), then the PV of the previous used tile (pend).
        static_assert((VS & (VS - 1)) == 0, "V ring depth must be a power of two");
        int pend = -1, pend_g = 0;
        for (int j = 0; j < w.n_tiles; ++j, ++g) {
          if (!wait_or_fail(B_KFULL + ks, kph)) break;
          if (!tv.uses(j)) {
            if (leader) mbar_arrive(bar(B_KEMPTY + ks));
            __syncwarp();
            const int vs = g & (VS - 1);
            if (!wait_or_fail(B_VFULL + vs, (g / VS) & 1)) break;
            if (leader) mbar_arrive(bar(B_VEMPTY + vs));
            __syncwarp();
            if (++ks == KS) { ks = 0; kph ^= 1; }
            continue;
          }
          if (!qk_step(ks)) break;
          if (pend >= 0) {
            const int vs = pend_g & (VS - 1);
            if (!wait_or_fail(B_VFULL + vs, (pend_g / VS) & 1) || !pv_step(vs, pend)) break;
          }
          pend = j;
          pend_g = g;
          if (++ks == KS) { ks = 0; kph ^= 1; }
          if (j == last && un >= 0 && !reload_q()) break;
        }
        if (ok && pend >= 0) {
          const int vs = pend_g & (VS - 1);
          if (wait_or_fail(B_VFULL + vs, (pend_g / VS) & 1)) pv_step(vs, pend);
        }
      }
      if (ok && last < 0) {
        // No key tile for this query tile: its Q load is consumed unused.
        if (wait_or_fail(B_QFULL + q, q_seen & 1)) {
          ++q_seen;
          if (un >= 0) {
            if (leader) load_q(q, decode_unit(p, un));
            __syncwarp();
            ++q_loads;
          }
        }
      }
      if (last >= 0) ++nact;
      u = un;
    }
    // Drain: a Q load issued for a unit never started has landed, and every
    // MMA issued here has completed before TMEM is released.
    if (q_loads > q_seen) mbar_wait(bar(B_QFULL + q), q_seen & 1, nullptr, kDrainCap);
    if (leader) umma_commit(bar(B_FIN + q));
    __syncwarp();
    mbar_wait(bar(B_FIN + q), 0, nullptr, kDrainCap);
  }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax + epilogue
    const int q = (warp - 4) >> 2;                      // query tile of this warpgroup
    const int r = threadIdx.x & 127;                    // row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS + q * 128;
    const uint32_t tP = tmem + lane_off + C::kColP + q * C::kPStride;
    const uint32_t tO = tmem + lane_off + C::kColO + q * D;
    const uint32_t sP = sbase + C::kOffStage + q * C::kPBytes;   // P_q in shared memory
    bool store_pending = false;                         // output stores of this warp may still read sP
    const float sl2 = p.scale_log2;
    int ns = 0;                                         // tiles processed (all units)
    int nact = 0;                                       // units in which this tile was active
    bool ok = true;
    // Every lane of a warp takes the same decision, so the warp-collective
    // tcgen05.ld/st and votes below always run converged.
    auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
      const bool got = mbar_wait(b, parity, abort_flag, cap);
      return __all_sync(0xffffffffu, got);
    };
    // The unit of this CTA's ut-th turn, read by every lane from slot ut % 4.
    auto unit_in_slot = [&](int ut, int& v) -> bool {
      if (!wait_all(bar(B_UFULL + ut % kUnitSlots), (ut / kUnitSlots) & 1)) {
        fail();
        ok = false;
        return false;
      }
      v = unit_ring[ut % kUnitSlots];
      return true;
    };
    int u = -1;
    unit_in_slot(0, u);
    for (int ut = 0; ok && u >= 0; ++ut) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_UEMPTY + ut % kUnitSlots));   // this warp has read slot ut
      const Unit w = decode_unit(p, u);
      const TileView tv = tile_view(w, q);
      const int T = w.n_tiles;
      const int t_q = w.t0 + q * kTileM + r;            // band: query step in the class
      const int pos_q = w.c + w.d * t_q;                // band: query position
      const bool row_valid = w.grow ? (w.grow0 + r < p.n_glob) : (t_q < w.n_c);
      // this row's key steps in its class: the window, or its segment block
      const int seg_b = w.seg > 0 ? (t_q / w.seg) * w.seg : 0;
      const int row_lo = w.seg > 0 ? seg_b : t_q - p.wl;
      const int row_hi = min(w.seg > 0 ? (p.seg_causal ? t_q : seg_b + w.seg - 1) : t_q + p.wr, w.n_c - 1);
      float m_run = -INFINITY, l_run = 0.f;             // m_run in log2 units of the scaled logits
      int n_unit = 0;
      // Global keys (Longformer) already inside this row's band are masked in
      // the global tiles, so they count once.  The global list is sorted, so
      // they have list indices in [g_a, g_b): the positions in [pos_q -
      // d*w_left, pos_q + d*w_right] (for d > 1 only those on the row's
      // stride lattice); gcount[x] = number of global positions below x.
      int g_a = 0, g_b = 0;
      if (!w.grow && !p.etc && p.n_glob > 0 && row_valid) {
        const long long a = static_cast<long long>(pos_q) - static_cast<long long>(w.d) * p.wl;
        const long long b = static_cast<long long>(pos_q) + static_cast<long long>(w.d) * p.wr + 1;
        g_a = __ldg(p.gcount + (a < 0 ? 0 : (a > p.N ? p.N : a)));
        g_b = __ldg(p.gcount + (b < 0 ? 0 : (b > p.N ? p.N : b)));
      }
      for (int j = 0; j < T; ++j) {
        if (!tv.uses(j)) continue;
      // Allowed columns of this tile as a 128-bit keep mask.
      int lo = 0, hi = kTileN - 1;
      int jj0 = -1;                                     // first global index of a Longformer global tile
      if (!w.grow) {
        if (j < w.n_band) {
          const int k0 = w.band_lo + j * kTileN;
          lo = row_lo - k0;
          hi = row_hi - k0;
        } else {
          const int g0 = (j - w.n_band) * kTileN;
          hi = min(kTileN, p.n_glob - g0) - 1;
          if (!p.etc) jj0 = g0;
        }
      } else {
        const int kt = w.kt0 + j;
        const int limit = (p.etc && kt < gt_src) ? p.n_glob - kt * kTileN
                                                 : p.N - (kt - (p.etc ? gt_src : 0)) * kTileN;
        hi = min(kTileN, limit) - 1;
      }
      // In-band global columns [ca, cb) of a Longformer global tile.
      const int ca = jj0 >= 0 ? max(g_a - jj0, 0) : 0, cb = jj0 >= 0 ? min(g_b - jj0, kTileN) : 0;
      // Most tiles need no mask in any row of the warp: decided from lo, hi and
      // [ca, cb) before any per-column work.
      const bool need_mask = __any_sync(0xffffffffu, (lo > 0) | (hi < kTileN - 1) | (ca < cb));
      uint32_t keep[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
      if (need_mask) {
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) keep[wd] = range_bits(lo, hi, 32 * wd);
        if (ca < cb) {
          if (w.d == 1) {
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) keep[wd] &= ~range_bits(ca, cb - 1, 32 * wd);
          } else {
            const uint4 lb = lattice_bits(p.gidx, jj0, ca, cb, pos_q, w.d);
            keep[0] &= ~lb.x;
            keep[1] &= ~lb.y;
            keep[2] &= ~lb.z;
            keep[3] &= ~lb.w;
          }
        }
      }

      if (!wait_all(bar(B_SFULL + q), ns & 1)) { fail(); ok = false; break; }
      tc_fence_after();
      float s[kTileN];
      tmem_ld128(tS, s);
      tc_fence_before();
      mbar_arrive(bar(B_SEMPTY + q));                   // S_q may take the next QK

      if (need_mask) {
        // Per 32-column word: nothing to do when every row of the warp keeps
        // it, a per-column select otherwise.
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          const uint32_t kw = keep[wd];
          if (!__all_sync(0xffffffffu, kw == 0xFFFFFFFFu)) {
#pragma unroll
            for (int c = 0; c < 32; ++c) s[32 * wd + c] = ((kw >> c) & 1u) ? s[32 * wd + c] : -INFINITY;
          }
        }
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmaxf(s[k], s[8 + k]);
#pragma unroll
      for (int col = 16; col < kTileN; col += 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[col + k], s[col + 8 + k]);
      }
      const float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      const float tmax2 = tmax * sl2;                   // log2 units (scale > 0 keeps the order)
      const float m_prev = m_run;
      float m_new = m_prev;
      if (tmax2 > m_prev + kRescaleThreshold) m_new = tmax2;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2_approx(m_prev - m_use);
      const bool need_rescale = (m_prev != -INFINITY) && (m_new != m_prev);
      uint32_t pk[kTileN / 2];
      uint64_t ps2[4];                                  // row sum in four packed pairs
#pragma unroll
      for (int k = 0; k < 4; ++k) ps2[k] = 0ull;
      const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(-m_use, -m_use);
#pragma unroll
      for (int i = 0; i < kTileN / 2; ++i) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sl2x2, negm2), x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        ps2[i & 3] = f2_add(ps2[i & 3], f2_pack(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      float a0, a1, b0, b1;
      f2_unpack(f2_add(ps2[0], ps2[1]), a0, a1);
      f2_unpack(f2_add(ps2[2], ps2[3]), b0, b1);
      const float psum = (a0 + a1) + (b0 + b1);
      l_run = l_run * corr + psum;
      m_run = m_new;
      // O_q is idle once PV_q of the previous tile has finished (its commit,
      // waited for here, also frees P_q), and PV_q of this tile waits for P_q.
      if (ns > 0) {
        if (!wait_all(bar(B_PEMPTY + q), (ns - 1) & 1)) { fail(); ok = false; break; }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, need_rescale)) rescale_o(tO, need_rescale ? corr : 1.f, D / 32);
      if constexpr (C::kPSmem) {
        // The previous unit's output stores read this warp's rows of the buffer.
        if (store_pending) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          store_pending = false;
        }
        // row r's 128 bf16 values: two 64-key blocks of 128-byte rows, the
        // 16-byte chunks XOR-swizzled by the row (the layout the MMA reads)
        const uint32_t prow = sP + r * 128;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int wv = 32 * blk + 4 * c;
            st_shared_v4(prow + blk * (kTileM * 128) + ((c ^ (r & 7)) << 4), pk[wv], pk[wv + 1], pk[wv + 2], pk[wv + 3]);
          }
        }
        fence_proxy_async_smem();
      } else {
        tmem_st64(tP, pk);
      }
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + q));
      ++ns;
      ++n_unit;
      }
      if (!ok) break;
      if (n_unit > 0) {
        if (!wait_all(bar(B_ODONE + q), nact & 1)) { fail(); ok = false; break; }
        tc_fence_after();
        ++nact;
        // The epilogue reads O 32 columns at a time in rolled loops: this code
        // runs once per unit, and kept small it evicts less of the tile loop
        // from the instruction cache.  O_q is released (OFREE) after its last
        // read; the next unit's first PV_q waits for that.
        if (!w.grow) {
          const float inv_l = row_valid ? 1.f / l_run : 0.f;
          // Each warp stages its 32 rows (positions c + d*t of one residue
          // class), 64 columns at a time, in shared memory (128-byte swizzle,
          // conflict-free) and writes them with one TMA store per 64 columns
          // through the slot's store map, whose element stride d puts row k of
          // the box at position row0 + d*k; rows past the end of the sequence
          // are clipped by the store.  D = 128: the 64-column halves go to
          // this warp's rows of the two 64-key blocks of its P buffer (free:
          // the unit's last PV has completed), so neither waits for a store.
          const int row0 = w.c + w.d * (w.t0 + q * kTileM + 32 * (warp & 3));
#pragma unroll 1
          for (int half = 0; half < D / 64; ++half) {
            const uint32_t stage = C::kPSmem ? sP + half * (kTileM * 128) + (warp & 3) * 4096
                                             : sbase + C::kOffStage + (warp - 4) * 4096;
            if (!C::kPSmem) {
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
              float o[32];
              tmem_ld32(tO + half * 64 + cc * 32, o);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int ci = cc * 4 + c;
                st_shared_v4(stage + lane * 128 + ((ci ^ (lane & 7)) << 4), pack_bf16x2(o[8 * c] * inv_l, o[8 * c + 1] * inv_l),
                             pack_bf16x2(o[8 * c + 2] * inv_l, o[8 * c + 3] * inv_l),
                             pack_bf16x2(o[8 * c + 4] * inv_l, o[8 * c + 5] * inv_l),
                             pack_bf16x2(o[8 * c + 6] * inv_l, o[8 * c + 7] * inv_l));
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&p.mapO[w.slot], stage, half * 64, row0, w.bh);
              bulk_commit_group();
            }
          }
          store_pending = true;
          tc_fence_before();
          mbar_arrive(bar(B_OFREE + q));
          if (row_valid) {
            const float lv = (m_run + __log2f(l_run)) * kLn2;
            if constexpr (P::kPatterns) p.pat_lse[w.slot][static_cast<size_t>(w.bh) * p.pat_rows[w.slot] + pos_q] = lv;
            else p.lse[static_cast<size_t>(w.bh) * p.N + pos_q] = lv;
          }
        } else {
          {
            // Every lane takes part in the warp-collective TMEM loads; only valid rows store.
            const int slot = (w.kt0 / p.grow_split) * 2 + q;
            const size_t prow = (static_cast<size_t>(w.bh) * p.n_glob + w.grow0 + r) * p.n_parts + slot;
            float4* dst = reinterpret_cast<float4*>(p.part_acc + prow * D);
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              float o[32];
              tmem_ld32(tO + cc * 32, o);
              if (row_valid) {
#pragma unroll
                for (int k = 0; k < 8; ++k) dst[8 * cc + k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
              }
              __syncwarp();   // reconverged before the next warp-collective TMEM load
            }
            if (row_valid) reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(m_run, l_run);
          }
          tc_fence_before();
          mbar_arrive(bar(B_OFREE + q));
        }
      } else if (w.grow && row_valid) {
        // A warpgroup with no key tile in this split leaves an empty partial.
        const int slot = (w.kt0 / p.grow_split) * 2 + q;
        const size_t prow = (static_cast<size_t>(w.bh) * p.n_glob + w.grow0 + r) * p.n_parts + slot;
        reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(-INFINITY, 0.f);
      }
      if (!unit_in_slot(ut + 1, u)) break;
    }
  }

  if (warp >= 4 && lane == 0) bulk_wait_all();   // output stores issued by this warp have completed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t tc_smem_bytes(int D) { return D == 64 ? Cfg<64>::kSmem : Cfg<128>::kSmem; }

// The register split only fits if the kernel launches with at least
// kRegsLaunchMin registers per thread; refuse to launch otherwise.
template <int D, class P>
cudaError_t prepare_kernel() {
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, tc_attn_kernel<D, P>);
  if (e != cudaSuccess) return e;
  if (a.numRegs < kRegsLaunchMin) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(tc_attn_kernel<D, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
}

// Persistent grid: one CTA per SM (shared memory allows no second one), each
// claiming units until the table is exhausted.
int grid_for(int n_units) {
  const int sms = device_sm_count();
  return n_units < sms ? n_units : sms;
}

namespace {
// The shared-memory attribute is a per-device setting: set it once for each
// device and kernel instance (head size, parameter block), under a lock (calls
// may come from several threads).
constexpr int kMaxDevices = 64;
std::mutex g_attr_mutex;
bool g_attr_done[kMaxDevices][4] = {};

// i: 0 / 1 for D = 64 / 128 with TcParams, 2 / 3 with TcParamsLn.
cudaError_t ensure_kernel_attributes(int i) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (g_attr_done[dev][i]) return cudaSuccess;
  switch (i) {
    case 0: e = prepare_kernel<64, TcParams>(); break;
    case 1: e = prepare_kernel<128, TcParams>(); break;
    case 2: e = prepare_kernel<64, TcParamsLn>(); break;
    default: e = prepare_kernel<128, TcParamsLn>(); break;
  }
  if (e == cudaSuccess) g_attr_done[dev][i] = true;
  return e;
}

template <class P>
cudaError_t launch_tc_impl(const P& p, int n_units, cudaStream_t s, bool chain_table) {
  if (n_units <= 0) return cudaSuccess;
  const int i = (p.D == 64 ? 0 : 1) + (P::kPatterns ? 2 : 0);
  cudaError_t ea = ensure_kernel_attributes(i);
  if (ea != cudaSuccess) return ea;
  cudaError_t e = launch_kernel(unit_table_kernel<P>, dim3((n_units + 255) / 256), dim3(256), 0, s, chain_table, p, n_units);
  if (e != cudaSuccess) return e;
  if (p.D == 64)
    return launch_kernel(tc_attn_kernel<64, P>, dim3(grid_for(n_units)), dim3(kThreads), Cfg<64>::kSmem, s, true, p, n_units);
  return launch_kernel(tc_attn_kernel<128, P>, dim3(grid_for(n_units)), dim3(kThreads), Cfg<128>::kSmem, s, true, p, n_units);
}
}  // namespace

cudaError_t launch_tc(const TcParams& p, int n_units, cudaStream_t s, bool chain_table) {
  return launch_tc_impl(p, n_units, s, chain_table);
}

cudaError_t launch_tc(const TcParamsLn& p, int n_units, cudaStream_t s, bool chain_table) {
  return launch_tc_impl(p, n_units, s, chain_table);
}

long long device_l2_bytes() {
  static std::atomic<long long> l2[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  long long v = l2[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int x = 0;
    v = (cudaDeviceGetAttribute(&x, cudaDevAttrL2CacheSize, dev) == cudaSuccess && x > 0) ? x : (128LL << 20);
    l2[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int device_sm_count() {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  int v = sms[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    sms[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int tc_rows_per_load(int d) { return rows_per_load(d); }

}  // namespace lg
