// Device twin of the seeded synthetic-input generator in synth/__init__.py.
// Draws numbers only; it holds no arithmetic of the MoE method.
//
// splitmix64 stream (Steele, Lea and Flood, OOPSLA 2014) keyed per tensor, two
// outputs per element, Box--Muller (1958) in float64, float32 round-to-nearest,
// then bfloat16 round-to-nearest-even on the float32 bits.  Bit-identical to the
// host generator up to last-bit libm differences (see the Python module).
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kTagMul = 0xD1B54A32D192ED03ull;
constexpr double kTwoPi = 6.283185307179586;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ inline uint16_t f32_to_bf16_rne(float v) {
  uint32_t b = __float_as_uint(v);
  b = b + 0x7FFFu + ((b >> 16) & 1u);
  return static_cast<uint16_t>(b >> 16);
}

__global__ void normal_bf16_kernel(uint16_t* __restrict__ dst, uint64_t n, uint64_t start,
                                   uint64_t key, double sigma) {
  uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t j = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n; j += stride) {
    uint64_t i = start + j;
    uint64_t z1 = mix64(key + (2 * i + 1) * kGolden);
    uint64_t z2 = mix64(key + (2 * i + 2) * kGolden);
    double u1 = (static_cast<double>(z1 >> 11) + 1.0) * 0x1.0p-53;
    double u2 = static_cast<double>(z2 >> 11) * 0x1.0p-53;
    double nrm = sqrt(-2.0 * log(u1)) * cos(kTwoPi * u2);
    float v = __double2float_rn(sigma * nrm);
    dst[j] = f32_to_bf16_rne(v);
  }
}

}  // namespace

extern "C" int synth_normal_bf16(uint16_t* dst, uint64_t n, uint64_t start, uint64_t seed,
                                 uint32_t tag, double sigma, void* stream) {
  if (n == 0) return 0;
  uint64_t key = mix64(mix64(seed + kGolden) ^ (static_cast<uint64_t>(tag) * kTagMul));
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (n + 255) / 256;
  uint64_t cap = static_cast<uint64_t>(sms) * 16;
  if (blocks > cap) blocks = cap;
  normal_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      dst, n, start, key, sigma);
  return static_cast<int>(cudaGetLastError());
}
