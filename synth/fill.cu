// fill.cu -- device version of the seeded synthetic-gradient generator.
//
// Same definition as the host (numpy) version in this module's __init__.py:
// SplitMix64 outputs (Steele, Lea & Flood, OOPSLA 2014) indexed by counter,
// the sum-of-twelve-uniforms normal approximation or a uniform integer in
// [-1000, 1000], then single IEEE roundings (binary64 multiply, binary64 ->
// binary32, binary32 -> binary16).  Integer operations and correctly rounded
// conversions only, so host and device produce identical bits.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_kernel(void* dst, uint64_t n, uint64_t start, uint64_t key, int kind, double sigma,
                            int dtype) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    const uint64_t i = start + j;
    float x;
    if (kind == 0) {
      const uint64_t w = mix(key + (3 * i + 1) * kGamma);
      x = (float)((int64_t)((w >> 11) % 2001ull) - 1000);
    } else {
      int64_t s = 0;
      for (int q = 0; q < 3; ++q) {
        const uint64_t w = mix(key + (3 * i + q + 1) * kGamma);
        s += (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) + (int64_t)((w >> 32) & 0xFFFF) +
             (int64_t)(w >> 48);
      }
      const double z = __dmul_rn((double)(s - 393210), 1.0 / 65536.0);  // exact
      x = __double2float_rn(__dmul_rn(z, sigma));
    }
    if (dtype == 1) {
      ((__half*)dst)[j] = __float2half_rn(x);
    } else {
      ((float*)dst)[j] = x;
    }
  }
}

}  // namespace

extern "C" int synth_fill(void* dst, uint64_t n, uint64_t start, uint64_t seed, int rank, int kind,
                          double sigma, int dtype, void* stream) {
  if (n == 0) return 0;
  const uint64_t key = [&] {
    uint64_t z = seed + (uint64_t)(rank + 1) * kGamma;
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }();
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (n + 255) / 256;
  const uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(dst, n, start, key, kind, sigma, dtype);
  return (int)cudaGetLastError();
}
