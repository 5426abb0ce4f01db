// Allocation-free variant of the sparse draft attention entry point.
//
// Some callers cannot call cudaMalloc: runtimes and plugin hosts that own all
// device memory through their own pool and do not let a library allocate
// (cudaMalloc may synchronize the device and fragments their pool), and code
// that must not allocate on its hot path at all.  This entry point takes the
// same inputs and outputs as sspec_sparse_draft_attn but needs no workspace:
// its scratch is a fixed array in this library's device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.cuh"

namespace {

// Scratch shared by every call on a device; every GPU that loads the library
// holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Device address of g_noalloc_scratch in the current CUDA context (in host code the
// array's name is only a host-side stand-in).  The address is looked up once per
// context and cached under the context's id, which CUDA never reuses within a
// process: after cudaDeviceReset, or in another context on the same device, the
// library's module is loaded again, possibly elsewhere, and gets its own lookup.
void* scratch_address(int* rc) {
  static std::mutex mu;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  constexpr int kSlots = 64;
  static unsigned long long ids[kSlots] = {0};
  static void* addrs[kSlots] = {nullptr};
  static int used = 0;
  *rc = SSPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!get_current || !get_id) {
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", reinterpret_cast<void**>(&get_current), 12000,
                                         cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", reinterpret_cast<void**>(&get_id), 12000, cudaEnableDefault,
                                         &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess) {
      get_current = nullptr;
      get_id = nullptr;
      cudaGetLastError();
      return nullptr;
    }
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return nullptr;
  if (!ctx) {
    // no context is current yet: make the current device's primary context current
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return nullptr;
  for (int i = 0; i < used; ++i)
    if (ids[i] == id) {
      *rc = SSPEC_OK;
      return addrs[i];
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return nullptr;
  }
  const int slot = used < kSlots ? used++ : int(id % kSlots);   // beyond 64 contexts: overwrite a slot
  ids[slot] = id;
  addrs[slot] = p;
  *rc = SSPEC_OK;
  return p;
}

// Clears, on the call's stream, the part of the scratch the draft attention needs at
// zero: the header (error word, queue counters) and the per (request, kv head)
// arrival counters.  Runs after the call's host checks, so a rejected call enqueues
// nothing.
struct ClearCtx {
  void* scratch;
  size_t bytes;
};
int clear_scratch(void* c, cudaStream_t s) {
  const ClearCtx* cc = static_cast<const ClearCtx*>(c);
  if (cudaMemsetAsync(cc->scratch, 0, cc->bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return SSPEC_ERR_CUDA;
  }
  return SSPEC_OK;
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
  ClearCtx cc{scratch, sspec::kWsHeaderBytes + sspec::ws_counter_bytes(batch, shape->num_kv_heads)};
  rc = sspec::sparse_draft_attn(shape, kv, batch, q, seq_lens, sel_lens, idx, idx_off, nsel, out, lse, scratch,
                                kNoAllocScratchBytes, stream, sspec::PreLaunch{clear_scratch, &cc});
  if (rc == SSPEC_OK && batch > 0 && dev_error &&
      cudaMemcpyAsync(dev_error, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SSPEC_ERR_CUDA;
  }
  return rc;
}
