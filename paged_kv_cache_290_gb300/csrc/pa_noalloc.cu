// pa_attention_static_scratch: paged attention for callers that cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc at all: plugins run by a host program
// that owns every byte of device memory through its own pool and gives them none, or code on a
// serving path where an allocation is not allowed because cudaMalloc may block or synchronise
// and cudaFree synchronises the whole device.  pa_attention needs a caller-provided workspace
// for its split-context partials; this entry point supplies that workspace from a fixed array
// in the library's own device memory instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ object: every GPU that loads the library holds its
// kStaticScratchBytes until the process exits.  All calls on a device share it and it keeps the
// last call's contents.  Nothing in it needs to start at zero: every partial slot the merge
// reads is written earlier in the same call.  Calls that overlap on the GPU (other streams, other host
// threads) race on it, so they must be ordered by the caller.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "pa.h"
#include "pa_kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// One-time set-up per device, with that device current: the host-side name of the array is a
// host stand-in, not a device address, so the device address is looked up here and cached.
int static_scratch_address(void** out, std::string* msg) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *msg = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return PA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *msg = "device ordinal out of range";
    return PA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      *msg = std::string("cudaGetSymbolAddress(static scratch): ") + cudaGetErrorString(e);
      return PA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_attention_static_scratch(const pa_tensor* q, const pa_tensor* k_cache,
                                const pa_tensor* v_cache, const pa_tensor* block_tables,
                                const pa_tensor* seq_lens, const pa_tensor* query_start_loc,
                                float scale, const pa_tensor* out, const pa_batch_hint* hint,
                                void* stream) {
  if (q && q->ndim == 3 && hint && hint->max_seq_len >= 0) {
    const size_t need =
        pa_attention_workspace_size(q->shape[0], q->shape[1], q->shape[2], hint->max_seq_len);
    if (need > kStaticScratchBytes) {
      return pa::set_last_error(
          PA_ERR_WORKSPACE, "batch needs " + std::to_string(need) +
                                " bytes of split-context scratch; the static array holds " +
                                std::to_string(kStaticScratchBytes) +
                                " (use pa_attention with a caller-provided workspace)");
    }
  }
  void* scratch = nullptr;
  std::string msg;
  int rc = static_scratch_address(&scratch, &msg);
  if (rc != PA_OK) return pa::set_last_error(rc, msg);
  return pa_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out,
                      hint, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
