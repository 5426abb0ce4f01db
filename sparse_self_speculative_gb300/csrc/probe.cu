// A read-only streaming probe of device memory: the HBM read rate this GPU reaches
// on a plain sequential read, timed beside the attention launches so that their K/V
// rate can be set against a read-only peak as well as against a copy's (a copy also
// writes, and a read stream can go faster than one).  Not part of the method: the
// probe reads a buffer once and XOR-folds its 32-bit words into one word, which
// keeps the loads from being dropped and lets a test check that every byte was read.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.cuh"

namespace sspec {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeUnroll = 8;       // 16-byte loads in flight a thread
constexpr int kProbeCtasPerSm = 8;    // 2,048 threads an SM: 256 KB of loads in flight per SM

// Round t of a CTA covers the 16-byte words [base, base + kProbeThreads * kProbeUnroll)
// with base = (t * gridDim.x + blockIdx.x) * kProbeThreads * kProbeUnroll; load j of a
// thread is word base + j * kProbeThreads + threadIdx.x, so each warp load reads 512
// contiguous bytes and a CTA's round one contiguous 32 KB run.
__global__ void __launch_bounds__(kProbeThreads, kProbeCtasPerSm)
    hbm_read_probe_kernel(const uint4* __restrict__ buf, long long n16, uint32_t* sink) {
  constexpr long long kRound = (long long)kProbeThreads * kProbeUnroll;
  uint32_t acc = 0;
  for (long long base = (long long)blockIdx.x * kRound; base < n16; base += (long long)gridDim.x * kRound) {
    uint4 v[kProbeUnroll];
#pragma unroll
    for (int j = 0; j < kProbeUnroll; ++j) {
      const long long i = base + (long long)j * kProbeThreads + threadIdx.x;
      v[j] = i < n16 ? __ldcs(buf + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kProbeUnroll; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace
}  // namespace sspec

extern "C" int sspec_hbm_read_probe(const void* buf, size_t bytes, uint32_t* sink, sspec_stream_t stream) {
  using namespace sspec;
  if (!buf || !sink || bytes == 0 || (bytes & 15u) != 0 || (reinterpret_cast<uintptr_t>(buf) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(sink) & 3u) != 0)
    return SSPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return SSPEC_ERR_CUDA;
  }
  const long long n16 = (long long)(bytes / 16);
  const long long rounds = (n16 + kProbeThreads * kProbeUnroll - 1) / (kProbeThreads * kProbeUnroll);
  const int grid = int(rounds < (long long)sms * kProbeCtasPerSm ? rounds : (long long)sms * kProbeCtasPerSm);
  if (cudaMemsetAsync(sink, 0, sizeof(uint32_t), s) != cudaSuccess) {
    cudaGetLastError();
    return SSPEC_ERR_CUDA;
  }
  hbm_read_probe_kernel<<<grid, kProbeThreads, 0, s>>>(static_cast<const uint4*>(buf), n16, sink);
  if (cudaGetLastError() != cudaSuccess) return SSPEC_ERR_CUDA;
  return SSPEC_OK;
}
