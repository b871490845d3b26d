// lg_attn_fwd_host: the Longformer-style forward pass on inputs and outputs
// in host memory, with the copies overlapped with the computation.
//
// The heads are independent, so the (batch, head) slices are processed in
// groups: while the kernels of group c run on the caller's stream, the q/k/v
// of group c + 1 are copied in on one stream and the out/lse of group c - 1
// are copied back on another.  Each group is one lg_attn_fwd call on a
// contiguous range of slices (viewed as B = 1 with that many heads).  Two
// non-blocking streams per device are created on first use and kept;
// events are created per call and released when their work has completed.
#include <algorithm>
#include <mutex>
#include <vector>

#include "lg_internal.h"

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_stream_mutex;
cudaStream_t g_in[kMaxDevices] = {};
cudaStream_t g_out[kMaxDevices] = {};

lg_status copy_streams(cudaStream_t* in, cudaStream_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_stream_mutex);
  if (g_in[dev] == nullptr) {
    if (cudaStreamCreateWithFlags(&g_in[dev], cudaStreamNonBlocking) != cudaSuccess) return LG_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&g_out[dev], cudaStreamNonBlocking) != cudaSuccess) return LG_ERR_CUDA;
  }
  *in = g_in[dev];
  *out = g_out[dev];
  return LG_OK;
}

struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);  // released once the recorded work completes
  }
  cudaError_t make(cudaEvent_t* e) {
    cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
    if (r == cudaSuccess) ev.push_back(*e);
    return r;
  }
};

}  // namespace

extern "C" lg_status lg_attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* out_h,
                                      float* lse_h, void* q_d, void* k_d, void* v_d, void* out_d, float* lse_d,
                                      lg_dtype dt, int B, int H, int N, int D, int w_left, int w_right,
                                      const int32_t* dilation, int causal, const int32_t* global_idx,
                                      int n_global, float scale, void* workspace, size_t workspace_bytes,
                                      int n_groups, lg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // The whole problem's checks before anything is queued: the host pointers,
  // the group count, and every check lg_attn_fwd makes (on the device staging
  // buffers, which share the host tensors' shapes).
  if (!q_h || !k_h || !v_h || !out_h || !lse_h || n_groups < 1) return LG_ERR_INVALID_ARG;
  lg_status st = lg::validate_fwd(q_d, k_d, v_d, out_d, lse_d, dt, B, H, N, D, w_left, w_right, dilation, causal,
                                  global_idx, n_global, workspace, workspace_bytes, false);
  if (st != LG_OK) return st;

  const long long BH = static_cast<long long>(B) * H;
  long long groups = std::min<long long>(n_groups, BH);
  groups = std::max<long long>(groups, (BH + LG_MAX_HEADS - 1) / LG_MAX_HEADS);  // at most LG_MAX_HEADS slices per call
  const size_t esz = dt == LG_BF16 ? 2 : 4;
  const size_t slice = static_cast<size_t>(N) * D * esz;  // bytes of one (b, h) slice of q, k, v or out
  const size_t lse_slice = static_cast<size_t>(N) * sizeof(float);

  cudaStream_t s_in, s_out;
  st = copy_streams(&s_in, &s_out);
  if (st != LG_OK) return st;
  Events evs;
  cudaEvent_t start;
  // The copies in may not overtake earlier work of the caller's stream on the device buffers.
  if (evs.make(&start) != cudaSuccess || cudaEventRecord(start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(s_in, start, 0) != cudaSuccess || cudaStreamWaitEvent(s_out, start, 0) != cudaSuccess)
    return LG_ERR_CUDA;

  std::vector<int32_t> dil;
  for (long long c = 0; c < groups && st == LG_OK; ++c) {
    const long long bh0 = c * BH / groups, bh1 = (c + 1) * BH / groups;
    const int nh = static_cast<int>(bh1 - bh0);
    const size_t off = static_cast<size_t>(bh0) * slice, bytes = static_cast<size_t>(nh) * slice;
    const size_t loff = static_cast<size_t>(bh0) * lse_slice, lbytes = static_cast<size_t>(nh) * lse_slice;
    cudaEvent_t in_done, comp_done;
    if (evs.make(&in_done) != cudaSuccess || evs.make(&comp_done) != cudaSuccess) { st = LG_ERR_CUDA; break; }
    if (cudaMemcpyAsync(static_cast<char*>(q_d) + off, static_cast<const char*>(q_h) + off, bytes,
                        cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(k_d) + off, static_cast<const char*>(k_h) + off, bytes,
                        cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(v_d) + off, static_cast<const char*>(v_h) + off, bytes,
                        cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaEventRecord(in_done, s_in) != cudaSuccess || cudaStreamWaitEvent(stream, in_done, 0) != cudaSuccess) {
      st = LG_ERR_CUDA;
      break;
    }
    dil.resize(nh);
    for (int i = 0; i < nh; ++i) dil[i] = dilation[(bh0 + i) % H];
    st = lg_attn_fwd(static_cast<const char*>(q_d) + off, static_cast<const char*>(k_d) + off,
                     static_cast<const char*>(v_d) + off, static_cast<char*>(out_d) + off,
                     reinterpret_cast<float*>(reinterpret_cast<char*>(lse_d) + loff), dt, 1, nh, N, D, w_left, w_right,
                     dil.data(), causal, global_idx, n_global, scale, workspace, workspace_bytes, stream_);
    if (st != LG_OK) break;
    if (cudaEventRecord(comp_done, stream) != cudaSuccess || cudaStreamWaitEvent(s_out, comp_done, 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(out_h) + off, static_cast<const char*>(out_d) + off, bytes,
                        cudaMemcpyDeviceToHost, s_out) != cudaSuccess ||
        cudaMemcpyAsync(reinterpret_cast<char*>(lse_h) + loff, reinterpret_cast<const char*>(lse_d) + loff, lbytes,
                        cudaMemcpyDeviceToHost, s_out) != cudaSuccess)
      st = LG_ERR_CUDA;
  }
  // On every path from here, success or not, the caller's stream completes
  // only after everything queued on the two copy streams, so a caller that
  // synchronises `stream` after an error may free its buffers safely.
  cudaEvent_t all_in, all_out;
  if (evs.make(&all_in) != cudaSuccess || evs.make(&all_out) != cudaSuccess ||
      cudaEventRecord(all_in, s_in) != cudaSuccess || cudaEventRecord(all_out, s_out) != cudaSuccess ||
      cudaStreamWaitEvent(stream, all_in, 0) != cudaSuccess || cudaStreamWaitEvent(stream, all_out, 0) != cudaSuccess)
    return LG_ERR_CUDA;
  return st;
}
