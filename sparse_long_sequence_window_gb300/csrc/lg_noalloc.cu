// lg_attn_fwd_noalloc: the Longformer-style forward pass for callers that
// cannot allocate device memory themselves.
//
// Who needs it: code that runs inside a host framework that plans all device
// memory ahead of time and forbids allocation while it executes (plugin
// interfaces of inference runtimes, for example), and processes in which
// another allocator already holds nearly all of the GPU's memory, so that a
// fresh cudaMalloc for the workspace would fail or fragment it.  Such callers
// still own their inputs and outputs; only the scratch space is provided here.
//
// How: the scratch lives in one file-scope __device__ array of a fixed size
// (LG_NOALLOC_SCRATCH_BYTES).  Every GPU on which this entry point is used
// keeps that array until the process exits.  Host code cannot use the array's
// name as a device address, so on the first call on each device (with that
// device current) its address is looked up with cudaGetSymbolAddress and
// cached; make that first call before any stream capture.  Nothing here calls
// cudaMalloc, cudaFree or an allocating library routine.
#include <mutex>

#include "lg_internal.h"

namespace {

constexpr size_t kScratchBytes = LG_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char lg_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
lg_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, lg_noalloc_scratch) != cudaSuccess || p == nullptr) return LG_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LG_OK;
}

}  // namespace

extern "C" lg_status lg_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                                         lg_dtype dt, int B, int H, int N, int D, int w_left, int w_right,
                                         const int32_t* dilation, int causal, const int32_t* global_idx,
                                         int n_global, float scale, lg_stream_t stream) {
  // Size check first, on the host only: problems whose scratch does not fit
  // the fixed array are refused before any CUDA call.
  const size_t need = lg_attn_fwd_workspace_size(B, H, N, D, n_global, dt);
  if (need == 0) return LG_ERR_INVALID_ARG;
  if (need > kScratchBytes) return LG_ERR_WORKSPACE;
  void* scratch = nullptr;
  lg_status st = scratch_for_current_device(&scratch);
  if (st != LG_OK) return st;
  // The regular call clears the status area at the head of the scratch and
  // fully rewrites everything else it reads, so stale contents from an earlier
  // call do not matter.
  return lg_attn_fwd(q, k, v, out, lse, dt, B, H, N, D, w_left, w_right, dilation, causal, global_idx, n_global,
                     scale, scratch, kScratchBytes, stream);
}
