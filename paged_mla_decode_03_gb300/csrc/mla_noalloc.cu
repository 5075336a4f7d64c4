// Allocation-free entry point: mla_decode_run_static_workspace.
//
// Some callers cannot hand the library a scratch buffer: code that enqueues
// decodes while a CUDA graph is being captured (cudaMalloc is not allowed
// there), runtimes that own every byte of device memory through their own
// pool and expose no allocator to plug-ins, or C callers without any device
// allocator at all.  This entry point serves them: its scratch lives in a
// fixed-size array in the library's own device memory (a file-scope
// __device__ array that every GPU which loads the library keeps until the
// process exits), so the call itself allocates nothing.
//
// Limits and sharing: the plan's workspace must fit in
// MLA_STATIC_WORKSPACE_BYTES.  Every call on a device uses the same array,
// so two calls that can overlap on the GPU (different streams, or the same
// graph replayed concurrently) race with each other; callers must order them.
// No zeroing is needed between calls: each run re-initialises every
// workspace byte it reads.
#include <mutex>

#include "../../include/mla_decode.h"

namespace {

__device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_address[kMaxDevices] = {};

// Device address of the static workspace on the current device (the host
// symbol is only a stand-in; cudaGetSymbolAddress must run with the device
// current).  Outside stream capture it is resolved on every call, so a
// device reset, which reloads the module and may move the array, is picked
// up; during capture the address cached by the last call outside capture is
// used, which is why the first call on a device must precede any capture.
int static_workspace_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cs == cudaStreamCaptureStatusNone) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr)
      return MLA_ERR_CUDA;
    g_address[dev] = ptr;
  } else if (!g_address[dev]) {
    return MLA_ERR_CUDA;  // never called outside capture on this device
  }
  *out = g_address[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_run_static_workspace(const mla_plan_t* plan, const void* query,
                                               const void* kv_cache, const int32_t* block_tables,
                                               const int32_t* seq_lens, const int32_t* qo_indptr,
                                               int64_t total_q, float bmm1_scale,
                                               float bmm2_scale, void* out, float* lse,
                                               void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  if (mla_decode_workspace_size(plan) > (size_t)MLA_STATIC_WORKSPACE_BYTES)
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  const int rc = static_workspace_address(static_cast<cudaStream_t>(stream), &ws);
  if (rc != MLA_OK) return rc;
  return mla_decode_run(plan, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q,
                        bmm1_scale, bmm2_scale, out, lse, ws, (size_t)MLA_STATIC_WORKSPACE_BYTES,
                        stream);
}
