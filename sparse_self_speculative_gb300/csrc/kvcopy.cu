// KV-cache offload to host memory and reload, and the FIFO chunk planner that
// orders them (talk notes, section "Dynamic KV-cache management", paper
// Sec. 4.4: GPU memory is filled with KV cache instead of predicting output
// lengths; the cache of requests that no longer fit goes to host memory
// asynchronously, chunk by chunk, and comes back in FIFO order).
//
// On GB300 the host memory of the Grace CPU is reachable from the GPU over
// NVLink-C2C, so a kernel reads the scattered pages of the paged cache and
// writes them straight into page-locked host memory (and the reverse): one pass
// over the bytes, no staging buffer and no per-page copy calls.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <deque>
#include <new>

#include "internal.cuh"

namespace sspec {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kBlockWords = kPage * kHeadDim * 2 / 16;   // 16-byte words in one (page, head) block: 256
constexpr int kCopyUnroll = 8;                           // blocks a CTA moves per round: 8 x 16 B in flight a thread
constexpr int kCopyCtasPerSm = 4;                        // resident at <= 64 registers: 128 KB of loads in flight per SM
static_assert(kBlockWords == kCopyThreads, "one 16-byte word of each block per thread");

// Block u of the transfer, u < 2 * n_pages * hkv: cache c = u / (n_pages * hkv)
// (0 = K, 1 = V), then list entry i and head h of e = u mod (n_pages * hkv) =
// i * hkv + h.  The device block is page pages[i], head h; the host block is the
// e-th 4 KiB block of that cache's host buffer.  TO_HOST copies device -> host.
template <bool TO_HOST>
__global__ void __launch_bounds__(kCopyThreads, kCopyCtasPerSm)
    kv_copy_kernel(uint4* dev_k, uint4* dev_v, int num_pages, int hkv, const int32_t* __restrict__ pages,
                   int n_pages, uint4* host_k, uint4* host_v, int32_t* err) {
  const long long per_cache = (long long)n_pages * hkv;
  const long long total = 2 * per_cache;
  const int tid = threadIdx.x;
  for (long long base = (long long)blockIdx.x * kCopyUnroll; base < total;
       base += (long long)gridDim.x * kCopyUnroll) {
    uint4 v[kCopyUnroll];
    uint4* dst[kCopyUnroll];
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j) {
      const long long u = base + j;
      dst[j] = nullptr;
      if (u >= total) continue;
      const int c = u >= per_cache ? 1 : 0;
      const long long e = u - c * per_cache;
      const int i = int(e / hkv), h = int(e - (long long)i * hkv);
      const int pg = __ldg(pages + i);
      if (pg < 0 || pg >= num_pages) {
        if (tid == 0 && err) atomicOr(err, SSPEC_DEVERR_PAGE_OOB);
        continue;
      }
      uint4* dptr = (c ? dev_v : dev_k) + ((size_t)pg * hkv + h) * kBlockWords + tid;
      uint4* hptr = (c ? host_v : host_k) + (size_t)e * kBlockWords + tid;
      dst[j] = TO_HOST ? hptr : dptr;
      v[j] = __ldcs(TO_HOST ? dptr : hptr);
    }
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j)
      if (dst[j]) __stcs(dst[j], v[j]);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device address of a host buffer, which must be page-locked (or managed):
// pageable memory is rejected rather than faulted on.
int host_buffer_address(const void* p, void** dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return SSPEC_ERR_CUDA;
  }
  if (a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeManaged) return SSPEC_ERR_INVALID_ARG;
  *dev = a.devicePointer ? a.devicePointer : const_cast<void*>(p);
  return SSPEC_OK;
}

template <bool TO_HOST>
int kv_transfer(const sspec_shape* shape, void* k_cache, void* v_cache, int32_t num_pages, const int32_t* pages,
                int32_t n_pages, const void* host_k, const void* host_v, size_t host_bytes, int32_t* dev_error,
                sspec_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != SSPEC_OK) return rc;
  if (n_pages < 0 || num_pages < 1) return SSPEC_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || !host_k || !host_v || (n_pages > 0 && !pages)) return SSPEC_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(host_k) || !aligned16(host_v))
    return SSPEC_ERR_INVALID_ARG;
  // the kernel moves n_pages whole pages of each cache: both host buffers must hold them
  const size_t page_bytes = size_t(shape->num_kv_heads) * kPage * kHeadDim * 2;
  if (size_t(n_pages) * page_bytes > host_bytes) return SSPEC_ERR_INVALID_ARG;
  if (n_pages == 0) return SSPEC_OK;
  void* hk = nullptr;
  void* hv = nullptr;
  if ((rc = host_buffer_address(host_k, &hk)) != SSPEC_OK) return rc;
  if ((rc = host_buffer_address(host_v, &hv)) != SSPEC_OK) return rc;
  const int hkv = shape->num_kv_heads;
  const long long total = 2LL * n_pages * hkv;
  const long long want = (total + kCopyUnroll - 1) / kCopyUnroll;
  const int grid = int(std::min<long long>(want, (long long)device_sm_count() * kCopyCtasPerSm));
  kv_copy_kernel<TO_HOST><<<grid, kCopyThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_pages, hkv, pages, n_pages,
      static_cast<uint4*>(hk), static_cast<uint4*>(hv), dev_error);
  return cudaGetLastError() == cudaSuccess ? SSPEC_OK : SSPEC_ERR_CUDA;
}

}  // namespace
}  // namespace sspec

// FIFO of whole requests handed out as chunks of pages, oldest request first.
struct sspec_kv_fifo {
  struct Entry {
    int32_t request;
    int32_t n_pages;
    int32_t next;   // first page not yet handed out
  };
  std::deque<Entry> queue;
  int64_t pending = 0;
};

extern "C" {

int sspec_kv_offload(const sspec_shape* shape, const void* k_cache, const void* v_cache, int32_t num_pages,
                     const int32_t* pages, int32_t n_pages, void* host_k, void* host_v, size_t host_bytes,
                     int32_t* dev_error, sspec_stream_t stream) {
  return sspec::kv_transfer<true>(shape, const_cast<void*>(k_cache), const_cast<void*>(v_cache), num_pages,
                                  pages, n_pages, host_k, host_v, host_bytes, dev_error, stream);
}

int sspec_kv_reload(const sspec_shape* shape, void* k_cache, void* v_cache, int32_t num_pages,
                    const int32_t* pages, int32_t n_pages, const void* host_k, const void* host_v,
                    size_t host_bytes, int32_t* dev_error, sspec_stream_t stream) {
  return sspec::kv_transfer<false>(shape, k_cache, v_cache, num_pages, pages, n_pages, host_k, host_v, host_bytes,
                                   dev_error, stream);
}

sspec_kv_fifo* sspec_kv_fifo_create(void) { return new (std::nothrow) sspec_kv_fifo(); }

void sspec_kv_fifo_destroy(sspec_kv_fifo* fifo) { delete fifo; }

int sspec_kv_fifo_push(sspec_kv_fifo* fifo, int32_t request, int32_t n_pages) {
  if (!fifo || n_pages < 1) return SSPEC_ERR_INVALID_ARG;
  try {
    fifo->queue.push_back({request, n_pages, 0});
  } catch (...) {
    return SSPEC_ERR_INVALID_ARG;
  }
  fifo->pending += n_pages;
  return SSPEC_OK;
}

int sspec_kv_fifo_next(sspec_kv_fifo* fifo, int32_t max_pages, int32_t* request, int32_t* first_page,
                       int32_t* count) {
  if (!fifo || max_pages < 1 || !request || !first_page || !count) return SSPEC_ERR_INVALID_ARG;
  if (fifo->queue.empty()) return 0;
  sspec_kv_fifo::Entry& e = fifo->queue.front();
  const int32_t c = std::min(max_pages, e.n_pages - e.next);
  *request = e.request;
  *first_page = e.next;
  *count = c;
  e.next += c;
  fifo->pending -= c;
  if (e.next == e.n_pages) fifo->queue.pop_front();
  return 1;
}

int64_t sspec_kv_fifo_pending(const sspec_kv_fifo* fifo) { return fifo ? fifo->pending : 0; }

}  // extern "C"
