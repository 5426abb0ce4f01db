// Allocation-free variant of the sparse draft attention entry point.
//
// Some callers cannot call cudaMalloc: runtimes and plugin hosts that own all
// device memory through their own pool and do not let a library allocate
// (cudaMalloc may synchronize the device and fragments their pool), and code
// that must not allocate on its hot path at all.  This entry point takes the
// same inputs and outputs as sspec_sparse_draft_attn but needs no workspace:
// its scratch is a fixed array in this library's device memory.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.cuh"

namespace {

// Scratch shared by every call on a device; every GPU that loads the library
// holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (in host code the array's name is only a host-side stand-in).
void* scratch_address(int* rc) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *rc = SSPEC_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      *rc = SSPEC_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *rc = SSPEC_OK;
  return addr[dev];
}

}  // namespace

extern "C" int sspec_sparse_draft_attn_noalloc(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch,
                                               const void* q, const int32_t* seq_lens, const int32_t* sel_lens,
                                               const int32_t* idx, const int64_t* idx_off, const int32_t* nsel,
                                               void* out, float* lse, int64_t total_tokens, int32_t* dev_error,
                                               sspec_stream_t stream) {
  if (!shape || total_tokens < 0 || batch < 0) return SSPEC_ERR_INVALID_ARG;
  const size_t need = sspec_workspace_size(shape, batch, 1, total_tokens);
  if (need == 0) return SSPEC_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return SSPEC_ERR_WORKSPACE_TOO_SMALL;   // beyond the 32 MiB scratch
  int rc = SSPEC_OK;
  void* scratch = scratch_address(&rc);
  if (rc != SSPEC_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the scratch keeps the previous call's contents: clear the error word and the
  // counters that must start at zero
  if (cudaMemsetAsync(scratch, 0, sspec::ws_region_offset(batch, shape->num_kv_heads), s) != cudaSuccess)
    return SSPEC_ERR_CUDA;
  rc = sspec_sparse_draft_attn(shape, kv, batch, q, seq_lens, sel_lens, idx, idx_off, nsel, out, lse, scratch,
                               kNoAllocScratchBytes, stream);
  if (rc == SSPEC_OK && dev_error &&
      cudaMemcpyAsync(dev_error, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return SSPEC_ERR_CUDA;
  return rc;
}
