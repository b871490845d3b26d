/*
 * lg_attn.h -- C ABI of the window + dilation + global sparse self-attention
 * forward and backward passes for one NVIDIA GB300 GPU (sm_103a).
 *
 * What is computed (per batch b and head h, query i, key j, 0 <= i, j < N):
 *
 *   inband(i, j)  <=>  j = i + d_h * t  for an integer t with
 *                      -w_left <= t <= (causal ? 0 : w_right)
 *     "Longformer: The Long-Document Transformer", section 3.4, "Sliding
 *     Window Attention" (w/2 keys on each side plus the token itself) and
 *     "Dilated Sliding Window Attention" (keys i +- d*k for k <= w/2, same key
 *     count, span times d); causal mode from "Autoregressive Language
 *     Modeling Configuration" (only the keys to the left).  w_left / w_right
 *     count steps of the dilation; keys outside [0, N) are dropped.
 *
 *   allowed(i, j) <=>  inband(i, j) or i in G or j in G
 *     Longformer page, "Global Attention": a global token attends to every
 *     token and every token attends to it.  A global key that is also in the
 *     band counts once.  Causal mode restricts only the band.
 *
 *   LSE_i = ln sum_{j allowed} exp(s * <q_i, k_j>),
 *   O_i   = sum_{j allowed} exp(s * <q_i, k_j> - LSE_i) * v_j.
 *
 * The ETC call follows "ETC: Encoding Long and Structured Inputs in
 * Transformers", section 3.4, "Global-Local Attention": a separate global
 * input of G tokens; g2g, g2l and l2g are full, l2l is |i - j| <= radius
 * (clamped), and g2g+g2l / l2g+l2l each share one softmax.
 *
 * Conventions for every call:
 *  - Tensors q, k, v, out are contiguous row-major [B, H, N, D] of dtype dt,
 *    in device memory, 16-byte aligned.  lse is contiguous fp32 [B, H, N] in
 *    device memory.  Outputs have the input dtype (LG_F32 or LG_BF16); every
 *    softmax statistic and accumulation is fp32.
 *  - The caller owns every buffer, including the workspace; the library
 *    allocates no device memory.  Tensor-map descriptors are built on the host
 *    for each call and passed as kernel parameters.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *    none synchronises.  Argument errors are returned before anything is
 *    launched.  Errors found on the device (bad global indices, a bounded
 *    wait that ran out) are recorded in the workspace's status word and
 *    returned by lg_query_status.  Each call clears that word first.
 *  - Calls that share a workspace must not overlap on the device.  Calls with
 *    their own workspaces may come from several host threads at once
 *    (lg_profile_* and lg_attn_fwd_noalloc excepted, as stated there).
 */
#ifndef LG_ATTN_H
#define LG_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* lg_stream_t;

typedef enum {
  LG_OK = 0,
  LG_ERR_INVALID_ARG = 1,   /* a pointer, size or value is out of its documented range (ETC labels: found on the device) */
  LG_ERR_UNSUPPORTED = 2,   /* valid arguments this build does not run (e.g. bf16 with D not 64/128) */
  LG_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  LG_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out; outputs are undefined */
  LG_ERR_WORKSPACE = 5,     /* workspace NULL, misaligned or smaller than the *_workspace_size result */
  LG_ERR_GLOBAL_IDX = 6     /* global_idx not strictly increasing or outside [0, N) (found on the device) */
} lg_status;

typedef enum { LG_F32 = 0, LG_BF16 = 1 } lg_dtype;

/* Largest head count of one call, and largest per-head dilation of the bf16 path. */
#define LG_MAX_HEADS 128
#define LG_MAX_BF16_DILATION 8

/* Static string naming a status; never NULL. */
const char* lg_status_string(lg_status s);

/* Library version string, e.g. "0.1.0 sm_103a". */
const char* lg_version(void);

/*
 * Bytes of device workspace lg_attn_fwd needs for these sizes.  The workspace
 * holds the device status word and, for bf16, the gathered global-token rows,
 * a table of global-position counts (N + 1 ints), the partial softmax
 * statistics of the global-query rows and a table of work-unit records (64
 * bytes per unit, written by the call itself).  It must be 256-byte aligned.
 * Returns 0 if the sizes are invalid.
 */
size_t lg_attn_fwd_workspace_size(int B, int H, int N, int D, int n_global, lg_dtype dt);

/*
 * Longformer-style window + dilation + global attention, forward.
 *
 *  q, k, v     device, [B, H, N, D], dtype dt, read only.
 *  out         device, [B, H, N, D], dtype dt, written (every row).
 *  lse         device, fp32 [B, H, N], written: natural log of the softmax
 *              denominator of each row over the scaled logits.
 *  dt          LG_F32 (CUDA-core fp32 path, 1 <= D <= 128, D % 4 == 0) or
 *              LG_BF16 (tensor-core path, D in {64, 128}).
 *  w_left, w_right  window steps on each side, >= 0.  w_right is ignored
 *              when causal != 0.
 *  dilation    HOST pointer to H ints >= 1 (bf16: <= LG_MAX_BF16_DILATION);
 *              read during the call only.
 *  causal      0 or 1.
 *  global_idx  DEVICE pointer to n_global int32 positions, strictly
 *              increasing, in [0, N); may be NULL iff n_global == 0.  A bad
 *              list is reported as LG_ERR_GLOBAL_IDX by lg_query_status; no
 *              memory outside the tensors is touched in that case.
 *  n_global    0 <= n_global <= N.
 *  scale       logit scale s; a value <= 0 selects 1/sqrt(D).
 *  workspace   device, >= lg_attn_fwd_workspace_size(...) bytes.
 *  stream      CUDA stream the work is queued on.
 */
lg_status lg_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      lg_dtype dt, int B, int H, int N, int D,
                      int w_left, int w_right, const int32_t* dilation, int causal,
                      const int32_t* global_idx, int n_global, float scale,
                      void* workspace, size_t workspace_bytes, lg_stream_t stream);

/*
 * lg_attn_fwd with separate projections for global attention ("Longformer",
 * "Separate Linear Projections for Local vs. Global Attention": Q_s, K_s,
 * V_s for the sliding window, Q_g, K_g, V_g for global attention).
 *
 *  q, k, v     the local projections Q_s, K_s, V_s: [B, H, N, D] of every token.
 *  q_glob, k_glob, v_glob  the global projections Q_g, K_g, V_g: [B, H, N, D]
 *              of every token, same dtype and layout.
 * A global row i is softmax(s q_glob_i . k_glob_j over every j) applied to
 * v_glob.  Every other row attends to its band and to the global columns with
 * the local projections (q_i . k_j, v_j), as in lg_attn_fwd.  (The page does
 * not say which projection a local row uses for the global columns; the local
 * one is this library's reading.)  With q_glob = q, k_glob = k, v_glob = v the
 * result is lg_attn_fwd's.  Every other argument, the workspace size, the
 * checks and the errors are lg_attn_fwd's; the three extra pointers must be
 * non-NULL and 16-byte aligned.
 */
lg_status lg_attn_fwd_gproj(const void* q, const void* k, const void* v,
                            const void* q_glob, const void* k_glob, const void* v_glob,
                            void* out, float* lse, lg_dtype dt, int B, int H, int N, int D,
                            int w_left, int w_right, const int32_t* dilation, int causal,
                            const int32_t* global_idx, int n_global, float scale,
                            void* workspace, size_t workspace_bytes, lg_stream_t stream);

/*
 * lg_attn_fwd without a caller-supplied workspace.  (Not a step of the
 * method: the paper has no counterpart; this exists for integration.)
 *
 * For callers that cannot allocate device memory while they run, e.g. code
 * inside a host framework that plans all device memory up front, or a process
 * whose GPU memory is already held by another allocator.  The scratch space
 * comes from one fixed array of LG_NOALLOC_SCRATCH_BYTES inside the library;
 * each GPU this is used on keeps that array until the process exits.
 *
 * Arguments are those of lg_attn_fwd minus the workspace.  The caller still
 * owns and passes inputs and outputs.  Returns LG_ERR_WORKSPACE, before any
 * CUDA call, when lg_attn_fwd_workspace_size(...) exceeds the fixed size
 * (for bf16 with global tokens the scratch grows with B*H*g*N/512 for
 * N <= 8192, B*H*g*N/1024 up to N = 32768 and B*H*g*N/2048 beyond).  The
 * first call on a device looks up the array's device address (once, with
 * that device current); make it before any stream capture.  All calls share
 * the one array: calls that overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller.  Device-side status
 * (lg_query_status) is not available through this entry point.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 */
#define LG_NOALLOC_SCRATCH_BYTES (16u << 20)
lg_status lg_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                              lg_dtype dt, int B, int H, int N, int D,
                              int w_left, int w_right, const int32_t* dilation, int causal,
                              const int32_t* global_idx, int n_global, float scale, lg_stream_t stream);

/*
 * lg_attn_fwd on inputs and outputs in host memory, with the host<->device
 * copies overlapped with the computation.  (Not a step of the method: the
 * paper has no counterpart; this serves callers whose tensors live in host
 * memory.)
 *
 * The (batch, head) slices are processed in n_groups groups of consecutive
 * slices (more if a group would exceed LG_MAX_HEADS slices).  Group c's q, k,
 * v are copied to q_d, k_d, v_d on a copy stream, its attention runs on
 * `stream` (one lg_attn_fwd call on that group, viewed as B = 1), and its
 * out and lse are copied back on a second copy stream, so copies of one
 * group overlap the kernels of another.
 *
 *  q_h, k_h, v_h  HOST, [B, H, N, D], dtype dt, read only; should be
 *                 page-locked (pageable memory works, without overlap).
 *  out_h, lse_h   HOST, [B, H, N, D] and fp32 [B, H, N], written.
 *  q_d .. lse_d   DEVICE buffers of the same shapes, owned by the caller,
 *                 used as staging; their contents on return are unspecified.
 *  global_idx     DEVICE pointer, as for lg_attn_fwd.
 *  n_groups       >= 1; 1 means no overlap.
 *  workspace      device, >= lg_attn_fwd_workspace_size(B, H, N, D, ...)
 *                 bytes (the groups use it one after another).
 *  Other arguments as for lg_attn_fwd.
 *
 * Asynchronous: returns once everything is queued; `stream` completes after
 * the last copy back.  The library creates two CUDA streams per device on
 * first use and keeps them.  Argument errors return before anything is
 * queued; an error returned after that leaves out_h and lse_h unspecified.
 * lg_query_status on the workspace reports the last group's device status (a
 * bad global list is found by every group).
 */
lg_status lg_attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* out_h, float* lse_h,
                           void* q_d, void* k_d, void* v_d, void* out_d, float* lse_d,
                           lg_dtype dt, int B, int H, int N, int D,
                           int w_left, int w_right, const int32_t* dilation, int causal,
                           const int32_t* global_idx, int n_global, float scale,
                           void* workspace, size_t workspace_bytes, int n_groups, lg_stream_t stream);

/* Bytes of device workspace lg_etc_attn_fwd needs; 0 if the sizes are invalid. */
size_t lg_etc_attn_fwd_workspace_size(int B, int H, int L, int G, int D, lg_dtype dt);

/*
 * ETC-style global-local attention, forward.
 *
 *  q_l, k_l, v_l   device, long input [B, H, L, D], dtype dt.
 *  q_g, k_g, v_g   device, global input [B, H, G, D], dtype dt.
 *  out_l, out_g    device, [B, H, L, D] and [B, H, G, D], dtype dt, written.
 *  lse_l, lse_g    device, fp32 [B, H, L] and [B, H, G], written.
 *  radius          local radius r >= 0: long query i sees long keys with
 *                  |i - j| <= r plus all G global keys, in one softmax;
 *                  global query sees all G + L keys, in one softmax.
 *  L >= 1, G >= 1; dt, D, scale, workspace, stream as for lg_attn_fwd.
 */
lg_status lg_etc_attn_fwd(const void* q_l, const void* k_l, const void* v_l,
                          const void* q_g, const void* k_g, const void* v_g,
                          void* out_l, void* out_g, float* lse_l, float* lse_g,
                          lg_dtype dt, int B, int H, int L, int G, int D, int radius, float scale,
                          void* workspace, size_t workspace_bytes, lg_stream_t stream);

/*
 * Backward pass.  The gradients of the forward's function with respect to q,
 * k and v, given dO = dLoss/dout (the gradient of the LSE output is taken as
 * zero): the chain rule of the same masked softmax, with P recomputed from
 * the forward's saved out and lse instead of a second softmax pass,
 *   P_ij = exp(s <q_i, k_j> - LSE_i) on the allowed pairs, 0 elsewhere,
 *   dV = P^T dO,  Delta_i = <dO_i, out_i>,  dS_ij = P_ij (<dO_i, v_j> - Delta_i),
 *   dQ = s dS K,  dK = s dS^T Q.
 * The pages train with this attention and take these gradients through it
 * ("LONGNET: Scaling Transformers to 1,000,000,000 Tokens", section 3.4,
 * "Distributed Training Algorithm": the gradients of the keys and values;
 * "Longformer", "Autoregressive Language Modeling Configuration": the
 * activations recomputed in the backward pass).
 *
 * Bytes of device workspace lg_attn_bwd needs (256-byte aligned); 0 if the
 * sizes are invalid.  It holds the status word, Delta and LSE per row, the
 * gathered global rows and the partial sums of the global rows and keys.
 */
size_t lg_attn_bwd_workspace_size(int B, int H, int N, int D, int n_global, lg_dtype dt);

/*
 *  q, k, v, out, lse   the forward's inputs and outputs (as for lg_attn_fwd).
 *  dout         device, [B, H, N, D], dtype dt: the gradient of out.
 *  dq, dk, dv   device, [B, H, N, D], dtype dt, written (every row).
 *  Every other argument, the layouts, the checks and the errors are those of
 *  lg_attn_fwd, with this call's workspace size.  bf16: tensor cores, fp32
 *  accumulation, outputs rounded to bf16; fp32: CUDA cores (dk and dv are
 *  accumulated with atomic additions, so their low bits may differ between
 *  calls).  Asynchronous on `stream`.
 */
lg_status lg_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv,
                      lg_dtype dt, int B, int H, int N, int D,
                      int w_left, int w_right, const int32_t* dilation, int causal,
                      const int32_t* global_idx, int n_global, float scale,
                      void* workspace, size_t workspace_bytes, lg_stream_t stream);

/* Bytes of device workspace lg_etc_attn_bwd needs; 0 if the sizes are invalid. */
size_t lg_etc_attn_bwd_workspace_size(int B, int H, int L, int G, int D, lg_dtype dt);

/*
 * Backward of lg_etc_attn_fwd: gradients of the long input (dq_l, dk_l, dv_l,
 * [B, H, L, D]) and of the global input (dq_g, dk_g, dv_g, [B, H, G, D]),
 * given the forward's outputs and lse and the gradients dout_l, dout_g of
 * out_l, out_g.  Layouts, checks and errors as for lg_etc_attn_fwd.
 */
lg_status lg_etc_attn_bwd(const void* q_l, const void* k_l, const void* v_l,
                          const void* q_g, const void* k_g, const void* v_g,
                          const void* out_l, const void* out_g, const float* lse_l, const float* lse_g,
                          const void* dout_l, const void* dout_g,
                          void* dq_l, void* dk_l, void* dv_l, void* dq_g, void* dk_g, void* dv_g,
                          lg_dtype dt, int B, int H, int L, int G, int D, int radius, float scale,
                          void* workspace, size_t workspace_bytes, lg_stream_t stream);

/*
 * ETC global-local attention with relative-position labels and per-instance
 * masks ("ETC: Encoding Long and Structured Inputs in Transformers", section
 * 3.4, "Relative Position Encoding" and "Global-Local Attention"): the four
 * pieces' logits are
 *   e_ij = s q_i . (k_j + a^K_{h, label_ij}) - C (1 - M_ij),  C = 10000,
 * with one softmax over g2g + g2l for a global query and one over l2g + l2l
 * for a long query; l2l only for |i - j| <= radius (clamped to [0, L)).
 * Each edge carries a code byte: label_ij in bits 0..6, 1 - M_ij in bit 7
 * (so 0 = label 0, allowed; 128 = label 0, blocked).  A row whose every edge
 * is blocked keeps the weights it would have with none blocked (C is common
 * to its logits) and an LSE lower by C, as the formula gives.
 *
 *  q_l, k_l, v_l, out_l  device [B, H, L, D];  q_g, k_g, v_g, out_g  device
 *              [B, H, G, D]; bf16, D in {64, 128}; lse_l [B, H, L], lse_g
 *              [B, H, G] fp32.  G >= 1.
 *  rel_k       device [H, n_labels, D] bf16 (a^K per head and label), or NULL
 *              with n_labels = 0 (no relative term; labels ignored).
 *  n_labels    0..64 for D = 64, 0..40 for D = 128 (LG_ERR_UNSUPPORTED
 *              above).  A label >= n_labels on an edge is reported by
 *              lg_query_status as LG_ERR_INVALID_ARG (found on the device).
 *  code_l2l    device uint8 [B, L, 2*radius + 1]: entry [b, i, t + radius] is
 *              the code of long key j = i + t (entries with j outside [0, L)
 *              are ignored);  code_l2g [B, L, G];  code_g2l [B, G, L];
 *              code_g2g [B, G, G].  Any of them may be NULL: code 0 on every
 *              edge of that piece.  Read during the call only.
 *  workspace   >= lg_etc_struct_attn_fwd_workspace_size(...) bytes, 256-byte
 *              aligned: the status word and the codes laid out per (query
 *              tile, key tile) block (q . a^K is formed in tensor memory).
 * fp32 returns LG_ERR_UNSUPPORTED.  Other arguments, errors and asynchrony as
 * for lg_etc_attn_fwd.
 */
size_t lg_etc_struct_attn_fwd_workspace_size(int B, int H, int L, int G, int D, int radius, int n_labels,
                                             lg_dtype dt);
lg_status lg_etc_struct_attn_fwd(const void* q_l, const void* k_l, const void* v_l,
                                 const void* q_g, const void* k_g, const void* v_g,
                                 void* out_l, void* out_g, float* lse_l, float* lse_g,
                                 const void* rel_k, int n_labels,
                                 const uint8_t* code_l2l, const uint8_t* code_l2g,
                                 const uint8_t* code_g2l, const uint8_t* code_g2g,
                                 lg_dtype dt, int B, int H, int L, int G, int D, int radius, float scale,
                                 void* workspace, size_t workspace_bytes, lg_stream_t stream);

/*
 * LongNet mixture of dilated attentions ("LONGNET: Scaling Transformers to
 * 1,000,000,000 Tokens", section 3.4, "Dilated Attention: Core Mechanism",
 * "Mixture of Dilated Attentions", "Multi-Head Dilated Attention: Offset
 * Mechanism").  Pattern k (segment length seg_w[k], dilation rate seg_r[k])
 * on head h keeps the rows i*w + s, i*w + s + r, ... below (i+1)*w (s = h mod
 * r) of each segment [i*w, (i+1)*w) and runs softmax attention among the kept
 * rows of the segment (causal: a kept row sees the kept rows at or before
 * it).  The patterns of a row are mixed by their softmax denominators: LSE =
 * ln sum_k exp(LSE_k) over the patterns that keep the row, O = sum_k
 * exp(LSE_k - LSE) O_k; a row no pattern keeps gets O = 0 and LSE = -inf.
 *
 *  q, k, v, out  device, [B, H, N, D], bf16, D in {64, 128}; lse fp32 [B, H, N]
 *                (LG_ERR_UNSUPPORTED for fp32 or another D).
 *  n_patterns    1..16; seg_w, seg_r: HOST arrays of n_patterns ints >= 1
 *                (any r; r need not divide w).
 *  workspace     >= lg_longnet_attn_fwd_workspace_size(...) bytes, 256-byte
 *                aligned: one output and LSE per pattern, the packed copies
 *                of q, k, v for patterns read through a gather, and the
 *                work-unit table.
 * Other arguments, errors and asynchrony as for lg_attn_fwd.  0 from the
 * size query means invalid or unsupported arguments.
 */
size_t lg_longnet_attn_fwd_workspace_size(int B, int H, int N, int D, int n_patterns, const int32_t* seg_w,
                                          const int32_t* seg_r, lg_dtype dt);
lg_status lg_longnet_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                              lg_dtype dt, int B, int H, int N, int D,
                              int n_patterns, const int32_t* seg_w, const int32_t* seg_r, int causal,
                              float scale, void* workspace, size_t workspace_bytes, lg_stream_t stream);

/* Query-key pairs head `head` computes over all patterns (a pair two
 * patterns keep counts twice): the useful work of lg_longnet_attn_fwd is
 * 4 * D times the sum over batches and heads.  -1 on invalid arguments. */
int64_t lg_longnet_count_pairs(int N, int n_patterns, const int32_t* seg_w, const int32_t* seg_r, int causal,
                               int head);

/*
 * Synchronises `stream`, then returns the device status recorded in
 * `workspace` by the last call that used it (LG_OK if none) and clears it.
 * Returns LG_ERR_CUDA if the synchronisation or the read fails.
 */
lg_status lg_query_status(const void* workspace, lg_stream_t stream);

/*
 * Number of allowed (query, key) pairs of ONE head of lg_attn_fwd (host
 * computation; global_idx_host is a HOST array, sorted and unique).  The
 * useful work of a call is 4 * D * (sum over heads and batches) FLOPs:
 * one multiply-add of q.k and one of p*v per pair and dimension.
 * Returns -1 on invalid arguments.
 */
int64_t lg_count_pairs(int N, int w_left, int w_right, int dilation, int causal,
                       const int32_t* global_idx_host, int n_global);

/* Allowed pairs of ONE head of lg_etc_attn_fwd; -1 on invalid arguments. */
int64_t lg_etc_count_pairs(int L, int G, int radius);

/*
 * Testing aid for the device-side timeout path.  (Not a step of the method:
 * the paper has no counterpart.)
 *
 * Every wait of the tensor-core kernel is bounded: when a wait for a tile, a
 * score block or a work unit runs out, the kernel records a timeout in the
 * workspace's status word, every role stops taking new work, waits (with a
 * fixed bound of about two seconds that nothing here shortens) until the TMA
 * loads and MMAs it has already issued have completed, releases its tensor
 * memory and returns; lg_query_status then reports LG_ERR_TIMEOUT and the
 * outputs are undefined.  This call makes that path testable without a fault:
 *
 *  withhold         1: later bf16 calls issue no TMA load and no MMA in the
 *                   tensor-core kernel, so its first wait for a tile runs out
 *                   with nothing in flight; 0: normal operation.
 *  wait_cap_cycles  cap of the work waits in SM clock cycles; <= 0 restores
 *                   the default (about one second).
 *
 * Process-wide, applies to calls made after it returns; not for concurrent
 * use with other calls.  Returns LG_ERR_INVALID_ARG if withhold is not 0 or 1.
 */
lg_status lg_debug_timeout_test(int withhold, long long wait_cap_cycles);

/*
 * Kernel timing of the dominant attention kernel.  After lg_profile_begin,
 * each launch of that kernel is bracketed by CUDA events on its stream;
 * lg_profile_end synchronises those events and returns the summed elapsed
 * milliseconds and the number of launches, then stops recording.  Not for
 * use during stream capture; not thread safe.
 */
lg_status lg_profile_begin(void);
lg_status lg_profile_end(float* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* LG_ATTN_H */
