// bf16 window + dilation + global attention forward on the 5th-generation
// tensor cores (tcgen05 MMA with TMEM accumulators, TMA operand loads).
//
// Method: "Longformer: The Long-Document Transformer", section 3.4 ("Sliding
// Window Attention", "Dilated Sliding Window Attention", "Global Attention",
// causal mode from "Autoregressive Language Modeling Configuration"), and
// "ETC: Encoding Long and Structured Inputs in Transformers", section 3.4
// ("Global-Local Attention", "Softmax unification").
//
// One CTA handles one work unit: 128 query rows against a list of 128-key
// tiles.
//  * Band unit: the query rows t0..t0+127 of one dilation residue class
//    c (positions c + d*t).  Inside a class the dilated window is the
//    contiguous step range [t - w_left, t + w_right], so the key tiles are the
//    contiguous class rows that intersect it; the strided rows are fetched by
//    TMA with an element stride of d along the row dimension (the dilation is
//    folded into the TMA coordinates).  The global-key tiles follow; a global
//    key that is already in a row's band is masked there (counted once).
//  * Global-row unit: 128 global queries against one split of all keys.  It
//    writes partial softmax statistics that a merge kernel combines.
// Warp roles (256 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (one thread), warps 4..7 run the online softmax: one thread
// per query row, fp32 row max and row sum, exp2 of log2-scaled logits.
// S = Q K^T lands in TMEM (two 128-column buffers), P is written to shared
// memory as bf16 in the 128-byte swizzled K-major layout, and O += P V
// accumulates in TMEM (D columns).
#include "lg_internal.h"
#include "lg_ptx.cuh"

namespace lg {
namespace {

constexpr int kThreads = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units; O is rescaled only when the max grows more
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTileM * D * 2;      // 128 rows x D bf16
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr int kPBytes = kTileM * kTileN * 2;    // 128 x 128 bf16
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffP = kOffV + kStages * kTileBytes;
  static constexpr int kOffMisc = kOffP + kPBytes;
  static constexpr int kMiscBytes = 1024;
  static constexpr int kSmem = kOffMisc + kMiscBytes + 1024;  // +1024: base alignment slack
};

// Rows one strided TMA box delivers for a dilation d (box height R*d <= 256).
__host__ __device__ __forceinline__ int rows_per_load(int d) {
  return d <= 2 ? 128 : (d <= 4 ? 64 : 32);
}

struct Unit {
  int grow;          // 1: global-row unit, 0: band unit
  int bh;
  int slot, d, c;    // band: dilation slot, stride, residue class
  int t0, n_c;       // band: first query step, class length
  int band_lo;       // band: first key step of the tiles
  int n_band;        // band: band key tiles
  int n_gt;          // band: appended global-key tiles
  int kt0;           // grow: first key tile of the split
  int grow0;         // grow: first global row of the tile
  int n_tiles;
};

__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
  Unit w{};
  if (u < p.n_grow_units) {
    w.grow = 1;
    const int split = u % p.n_splits;
    const int r = u / p.n_splits;
    w.grow0 = (r % p.n_gtiles) * kTileM;
    w.bh = r / p.n_gtiles;
    w.kt0 = split * kSplitTiles;
    w.n_tiles = min(kSplitTiles, p.n_key_tiles_grow - w.kt0);
    w.slot = 0; w.d = 1;
    return w;
  }
  const int v = u - p.n_grow_units;
  const int b = v / p.band_units_per_batch;
  int rem = v % p.band_units_per_batch;
  int h = 0;
  while (h + 1 < p.H && p.head_unit_start[h + 1] <= rem) ++h;
  rem -= p.head_unit_start[h];
  w.grow = 0;
  w.bh = b * p.H + h;
  w.slot = p.head_slot[h];
  w.d = p.slot_dil[w.slot];
  for (int c = 0; c < w.d; ++c) {
    const int n_c = (p.N - c + w.d - 1) / w.d;
    const int tiles = (n_c + kTileM - 1) / kTileM;
    if (rem < tiles) { w.c = c; w.n_c = n_c; w.t0 = rem * kTileM; break; }
    rem -= tiles;
  }
  if (w.n_c <= 0) { w.n_tiles = 0; return w; }
  const int t_last = min(w.t0 + kTileM - 1, w.n_c - 1);
  w.band_lo = max(0, w.t0 - p.wl);
  const int band_hi = min(w.n_c - 1, t_last + p.wr);
  w.n_band = (band_hi - w.band_lo + kTileN) / kTileN;
  w.n_gt = (p.n_glob + kTileN - 1) / kTileN;
  w.n_tiles = w.n_band + w.n_gt;
  return w;
}

// Issues the TMA loads of one 128-row operand tile.  main == true: the
// dilation-strided view of the slot; otherwise the global-side view.
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1) tc_attn_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV,
                 sP = sbase + C::kOffP;
  unsigned char* misc = smem + C::kOffMisc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  // barrier indices
  constexpr int S = C::kStages;
  const int B_QFULL = 0, B_KFULL = 1, B_KEMPTY = 1 + S, B_VFULL = 1 + 2 * S, B_VEMPTY = 1 + 3 * S,
            B_SFULL = 1 + 4 * S, B_SFREE = 3 + 4 * S, B_PFULL = 5 + 4 * S, B_PVDONE = 6 + 4 * S,
            B_FIN = 7 + 4 * S, NBARS = 8 + 4 * S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) {
      uint32_t count = 1;
      if (i == B_SFREE || i == B_SFREE + 1 || i == B_PFULL) count = 128;
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
  const Unit w = decode_unit(p, blockIdx.x);
  const int T = w.n_tiles;
  const long long cap = p.wait_cap;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.status, ST_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued_k = 0, issued_v = 0;
      mbar_arrive_expect_tx(bar(B_QFULL), C::kTileBytes);
      if (w.grow) {
        load_tile<D>(&p.mapQg, false, 1, w.grow0, w.bh, sQ, bar(B_QFULL));
      } else {
        load_tile<D>(&p.mapQ[w.slot], true, w.d, w.c + w.d * w.t0, w.bh, sQ, bar(B_QFULL));
      }
      const int gt_src = (p.n_glob + kTileN - 1) / kTileN;
      for (int j = 0; j < T; ++j) {
        const int st = j % S;
        // which view and row coordinate holds key tile j
        const CUtensorMap *mk, *mv;
        bool strided;
        int y;
        if (!w.grow) {
          if (j < w.n_band) {
            mk = &p.mapK[w.slot]; mv = &p.mapV[w.slot]; strided = true;
            y = w.c + w.d * (w.band_lo + j * kTileN);
          } else {
            mk = &p.mapKg; mv = &p.mapVg; strided = false;
            y = (j - w.n_band) * kTileN;
          }
        } else {
          const int kt = w.kt0 + j;
          if (p.etc && kt < gt_src) {
            mk = &p.mapKg; mv = &p.mapVg; strided = false; y = kt * kTileN;
          } else {
            mk = &p.mapK[0]; mv = &p.mapV[0]; strided = true;
            y = (kt - (p.etc ? gt_src : 0)) * kTileN;
          }
        }
        if (j >= S && !mbar_wait(bar(B_KEMPTY + st), ((j / S) - 1) & 1, abort_flag, cap)) { fail(); break; }
        mbar_arrive_expect_tx(bar(B_KFULL + st), C::kTileBytes);
        load_tile<D>(mk, strided, strided ? w.d : 1, y, w.bh, sK + st * C::kTileBytes, bar(B_KFULL + st));
        issued_k = j + 1;
        if (j >= S && !mbar_wait(bar(B_VEMPTY + st), ((j / S) - 1) & 1, abort_flag, cap)) { fail(); break; }
        mbar_arrive_expect_tx(bar(B_VFULL + st), C::kTileBytes);
        load_tile<D>(mv, strided, strided ? w.d : 1, y, w.bh, sV + st * C::kTileBytes, bar(B_VFULL + st));
        issued_v = j + 1;
      }
      // Drain: every load issued here has landed before the CTA exits (these
      // waits ignore the abort flag and are bounded by the cap alone).
      mbar_wait(bar(B_QFULL), 0, nullptr, cap);
      for (int j = max(0, issued_k - S); j < issued_k; ++j)
        mbar_wait(bar(B_KFULL + j % S), (j / S) & 1, nullptr, cap);
      for (int j = max(0, issued_v - S); j < issued_v; ++j)
        mbar_wait(bar(B_VFULL + j % S), (j / S) & 1, nullptr, cap);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      const uint32_t tO = tmem + 256;
      bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, cap);
      if (!ok) fail();
      auto issue_pv = [&](int jj) -> bool {
        const int st = jj % S;
        if (!mbar_wait(bar(B_PFULL), jj & 1, abort_flag, cap)) return false;
        if (!mbar_wait(bar(B_VFULL + st), (jj / S) & 1, abort_flag, cap)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          const uint64_t a = sdesc_sw128(sP + (kk >> 2) * (kTileM * 128) + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(vbase + kk * 16 * 128, kTileN * 128, 1024);
          umma_bf16_ss(tO, a, b, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_PVDONE));
        umma_commit(bar(B_VEMPTY + st));
        return true;
      };
      for (int j = 0; j < T && ok; ++j) {
        const int st = j % S;
        const int sb = j & 1;
        if (!mbar_wait(bar(B_KFULL + st), (j / S) & 1, abort_flag, cap)) { fail(); ok = false; break; }
        if (j >= 2 && !mbar_wait(bar(B_SFREE + sb), ((j >> 1) - 1) & 1, abort_flag, cap)) { fail(); ok = false; break; }
        tc_fence_after();
        const uint32_t kbase = sK + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kTileM * 128) + (kk & 3) * 32;
          umma_bf16_ss(tmem + sb * 128, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                       idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_SFULL + sb));
        umma_commit(bar(B_KEMPTY + st));
        if (j >= 1 && !issue_pv(j - 1)) { fail(); ok = false; break; }
      }
      if (ok && T > 0 && !issue_pv(T - 1)) { fail(); ok = false; }
      // Every MMA issued here has completed before TMEM is released.
      umma_commit(bar(B_FIN));
      mbar_wait(bar(B_FIN), 0, nullptr, cap);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = threadIdx.x - 128;                    // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int t_q = w.t0 + r;                           // band: query step in the class
    const int pos_q = w.c + w.d * t_q;                  // band: query position
    const bool row_valid = w.grow ? (w.grow0 + r < p.n_glob) : (t_q < w.n_c);
    const int gt_src = (p.n_glob + kTileN - 1) / kTileN;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // Every lane of a warp takes the same decision, so the warp-collective
    // tcgen05.ld/st and votes below always run converged.
    auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
      const bool got = mbar_wait(b, parity, abort_flag, cap);
      return __all_sync(0xffffffffu, got);
    };
    for (int j = 0; j < T; ++j) {
      const int sb = j & 1;
      // Column window [lo, hi] of allowed keys for band tiles, and the tile kind.
      int lo = 0, hi = kTileN - 1;
      int kind = 0;  // 0: [lo, hi] range, 1: global-key tile with de-duplication (Longformer)
      int jj0 = 0;
      if (!w.grow) {
        if (j < w.n_band) {
          const int k0 = w.band_lo + j * kTileN;
          lo = t_q - p.wl - k0;
          hi = min(t_q + p.wr, w.n_c - 1) - k0;
        } else {
          jj0 = (j - w.n_band) * kTileN;
          hi = min(kTileN, p.n_glob - jj0) - 1;
          if (!p.etc) kind = 1;
        }
      } else {
        const int kt = w.kt0 + j;
        int limit;
        if (p.etc && kt < gt_src) limit = p.n_glob - kt * kTileN;
        else limit = p.N - (kt - (p.etc ? gt_src : 0)) * kTileN;
        hi = min(kTileN, limit) - 1;
      }
      if (!wait_all(bar(B_SFULL + sb), (j >> 1) & 1)) { fail(); ok = false; break; }
      tc_fence_after();
      float s[kTileN];
#pragma unroll
      for (int cc = 0; cc < kTileN / 32; ++cc) {
        float* dst = s + cc * 32;
        tmem_ld32(tmem + lane_off + sb * 128 + cc * 32, *reinterpret_cast<float(*)[32]>(dst));
      }
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + sb));

      float tmax = -INFINITY;
      if (kind == 0) {
#pragma unroll
        for (int col = 0; col < kTileN; ++col) {
          const bool ok_col = (col >= lo) && (col <= hi);
          s[col] = ok_col ? s[col] * p.scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, s[col]);
        }
      } else {
#pragma unroll
        for (int col = 0; col < kTileN; ++col) {
          const int gp = (col <= hi) ? __ldg(p.gidx + jj0 + col) : -1;
          bool ok_col = gp >= 0;
          if (ok_col) {
            const int diff = gp - pos_q;
            if (diff % w.d == 0) {
              const int tt = diff / w.d;
              if (tt >= -p.wl && tt <= p.wr) ok_col = false;  // already counted in the band
            }
          }
          s[col] = ok_col ? s[col] * p.scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, s[col]);
        }
      }
      const float m_prev = m_run;
      float m_new = m_prev;
      if (tmax > m_prev + kRescaleThreshold) m_new = tmax;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2_approx(m_prev - m_use);
      const bool need_rescale = (j > 0) && (m_prev != -INFINITY) && (m_new != m_prev);
      uint32_t pk[kTileN / 2];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < kTileN / 2; ++i) {
        const float p0 = ex2_approx(s[2 * i] - m_use);
        const float p1 = ex2_approx(s[2 * i + 1] - m_use);
        psum += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * corr + psum;
      m_run = m_new;
      if (j > 0) {
        if (!wait_all(bar(B_PVDONE), (j - 1) & 1)) { fail(); ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need_rescale)) {
          const float f = need_rescale ? corr : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            float o[32];
            tmem_ld32(tmem + lane_off + 256 + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tmem_st32(tmem + lane_off + 256 + cc * 32, o);
          }
        }
      }
      // P (bf16) into the 128-byte swizzled K-major tile: two 64-key blocks.
#pragma unroll
      for (int q = 0; q < kTileN / 8; ++q) {
        const uint32_t addr = sP + (q >> 3) * (kTileM * 128) + r * 128 + (((q & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]),
                     "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    if (ok && T > 0) {
      if (!wait_all(bar(B_PVDONE), (T - 1) & 1)) {
        fail();
      } else {
        tc_fence_after();
        if (!w.grow) {
          const float inv_l = 1.f / l_run;
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                (static_cast<size_t>(w.bh) * p.N + pos_q) * D;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            float o[32];
            tmem_ld32(tmem + lane_off + 256 + cc * 32, o);
            if (row_valid) {
              uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint4 val;
                val.x = pack_bf16x2(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l);
                val.y = pack_bf16x2(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l);
                val.z = pack_bf16x2(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l);
                val.w = pack_bf16x2(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l);
                dst[q] = val;
              }
            }
          }
          if (row_valid) p.lse[static_cast<size_t>(w.bh) * p.N + pos_q] = (m_run + __log2f(l_run)) * kLn2;
        } else {
          const int split = w.kt0 / kSplitTiles;
          const int grow = w.grow0 + r;
          const size_t prow = (static_cast<size_t>(w.bh) * p.n_glob + grow) * p.n_splits + split;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            float o[32];
            tmem_ld32(tmem + lane_off + 256 + cc * 32, o);
            if (row_valid) {
              float4* dst = reinterpret_cast<float4*>(p.part_acc + prow * D + cc * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q) dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            }
          }
          if (row_valid) reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(m_run, l_run);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t tc_smem_bytes(int D) { return D == 64 ? Cfg<64>::kSmem : Cfg<128>::kSmem; }

cudaError_t launch_tc(const TcParams& p, int n_units, cudaStream_t s) {
  if (n_units <= 0) return cudaSuccess;
  static bool attr_done[2] = {false, false};
  if (p.D == 64) {
    if (!attr_done[0]) {
      cudaError_t e = cudaFuncSetAttribute(tc_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<64>::kSmem);
      if (e != cudaSuccess) return e;
      attr_done[0] = true;
    }
    tc_attn_kernel<64><<<n_units, kThreads, Cfg<64>::kSmem, s>>>(p);
  } else {
    if (!attr_done[1]) {
      cudaError_t e = cudaFuncSetAttribute(tc_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<128>::kSmem);
      if (e != cudaSuccess) return e;
      attr_done[1] = true;
    }
    tc_attn_kernel<128><<<n_units, kThreads, Cfg<128>::kSmem, s>>>(p);
  }
  return cudaGetLastError();
}

int tc_rows_per_load(int d) { return rows_per_load(d); }

}  // namespace lg
