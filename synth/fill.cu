// Device copy of the seeded input generator of synth/__init__.py: it writes
// the same bf16 bits as the host functions, element for element, so large
// paged caches can be filled in HBM without a host round trip.  No arithmetic
// of the attention method lives here.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr unsigned long long kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// output n of the splitmix64 stream seeded with `seed`
__device__ __forceinline__ unsigned long long splitmix64_at(unsigned long long seed, unsigned long long n) {
  return mix64(seed + (n + 1ull) * kGamma);
}

// Irwin-Hall(12) variate of element `c` as bf16 bits (round to nearest even)
__device__ __forceinline__ uint16_t normal_bf16(unsigned long long key, unsigned long long c) {
  long long total = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const unsigned long long w = splitmix64_at(key, 3ull * c + i);
#pragma unroll
    for (int m = 0; m < 4; ++m) total += (long long)((w >> (16 * m)) & 0xFFFFull);
  }
  const float z = __fmul_rn((float)(total - 393210), 1.0f / 65536.0f);
  const uint32_t bits = __float_as_uint(z);
  const uint32_t lsb = (bits >> 16) & 1u;
  return (uint16_t)((bits + 0x7FFFu + lsb) >> 16);
}

__device__ __forceinline__ uint16_t times4(uint16_t b) {
  return (b & 0x7FFFu) ? (uint16_t)(b + (2u << 7)) : b;
}

__global__ void fill_kv_kernel(uint16_t* cache, long long groups, int hkv, const int32_t* page_req,
                               const int32_t* page_idx, const int32_t* seq_lens, const long long* tok_base,
                               const uint8_t* plant, unsigned long long key) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < groups;
       e += (long long)gridDim.x * blockDim.x) {
    const int d0 = int(e % 16) * 8;
    const int slot = int((e / 16) % 16);
    const int h = int((e / 256) % hkv);
    const long long pg = e / (256ll * hkv);
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int r = page_req[pg];
    if (r >= 0) {
      const long long t = (long long)page_idx[pg] * 16 + slot;
      if (t < seq_lens[r]) {
        const bool big = plant && plant[(tok_base[r] + t) * hkv + h];
        const unsigned long long c0 = ((((unsigned long long)r << 20) + (unsigned long long)t) * 64ull + h) * 128ull;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint16_t b = normal_bf16(key, c0 + d0 + i);
          v[i] = big ? times4(b) : b;
        }
      }
    }
    uint4 pk;
    pk.x = v[0] | (uint32_t(v[1]) << 16);
    pk.y = v[2] | (uint32_t(v[3]) << 16);
    pk.z = v[4] | (uint32_t(v[5]) << 16);
    pk.w = v[6] | (uint32_t(v[7]) << 16);
    reinterpret_cast<uint4*>(cache)[e] = pk;
  }
}

}  // namespace

extern "C" int synth_fill_kv(void* cache, long long num_pages, int hkv, const int32_t* page_req,
                             const int32_t* page_idx, const int32_t* seq_lens, const long long* tok_base,
                             const uint8_t* plant, unsigned long long key, void* stream) {
  const long long groups = num_pages * hkv * 16 * 16;
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (groups + 255) / 256;
  const int grid = (int)(want < (long long)sms * 16 ? want : (long long)sms * 16);
  fill_kv_kernel<<<grid > 0 ? grid : 1, 256, 0, (cudaStream_t)stream>>>(
      (uint16_t*)cache, groups, hkv, page_req, page_idx, seq_lens, tok_base, plant, key);
  return (int)cudaGetLastError();
}
