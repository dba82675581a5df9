// Device twin of synth/gen.py: fills a buffer with the seeded bf16 stream of
// one emulated rank's tensor, bit-identical to the host generator.  Input
// generation only; it holds none of the reduce-scatter / all-gather arithmetic
// and libtide never links it.
//
// Stream: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014); element i of a stream keyed k is
// mix64(k + (i + 1) * GAMMA).  Value maps and bf16 rounding as in gen.py.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kMix1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kMix2 = 0x94D049BB133111EBull;
constexpr uint64_t kOutlierSalt = 0x5851F42D4C957F2Dull;
constexpr int64_t kOutlierThreshold = 1677721;  // floor(0.1 * 2^24)

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * kMix1;
  z = (z ^ (z >> 27)) * kMix2;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t to_bf16_rne(float f) {
  const uint32_t b = __float_as_uint(f);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ uint16_t value(uint64_t key, uint64_t i, int dist, float scale, float outlier_factor) {
  const uint64_t bits = mix64(key + (i + 1) * kGamma);
  float f;
  if (dist == 0) {  // uniform [-1, 1)
    const int32_t u = (int32_t)(bits >> 40) - (1 << 23);
    f = __fmul_rn(__int2float_rn(u), 1.0f / 8388608.0f);
  } else if (dist == 1 || dist == 2) {  // Irwin-Hall(4) approximately normal
    const int32_t t = (int32_t)((bits & 0xFFFF) + ((bits >> 16) & 0xFFFF) + ((bits >> 32) & 0xFFFF) + (bits >> 48)) -
                      2 * 65535;
    f = __fmul_rn(__int2float_rn(t), scale);
    if (dist == 2) {
      const uint64_t o = mix64((key ^ kOutlierSalt) + (i + 1) * kGamma) >> 40;
      if ((int64_t)o < kOutlierThreshold) f = __fmul_rn(f, outlier_factor);
    }
  } else {  // integers in [-128, 128]
    f = (float)((int32_t)((bits >> 32) % 257ull) - 128);
  }
  return to_bf16_rne(f);
}

__global__ void fill_kernel(uint16_t* dst, int64_t n, uint64_t key, int dist, float scale, float outlier_factor,
                            uint64_t idx0) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    dst[j] = value(key, idx0 + (uint64_t)j, dist, scale, outlier_factor);
}

}  // namespace

extern "C" {

// Fill dst[0..n) with elements idx0 .. idx0+n-1 of the stream `key`.
// dist: 0 uniform, 1 normal, 2 normal with x100 outliers, 3 integers.
// scale_bits: fp32 bit pattern of the normal scale (host-computed).
// Returns the cudaError_t of the launch (0 on success).
int synth_fill_bf16(void* dst, int64_t n, uint64_t key, int32_t dist, uint32_t scale_bits, uint64_t idx0,
                    void* stream) {
  if (n <= 0) return 0;
  if (!dst || dist < 0 || dist > 3) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return (int)err;
  const int threads = 256;
  const int64_t want = (n + threads - 1) / threads;
  const int grid = (int)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
  float scale;
  std::memcpy(&scale, &scale_bits, sizeof(scale));
  fill_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>((uint16_t*)dst, n, key, dist, scale, 100.0f, idx0);
  return (int)cudaGetLastError();
}
}
