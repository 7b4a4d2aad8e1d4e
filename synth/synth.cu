// CUDA implementation of the seeded input generator defined in synth/__init__.py
// (SplitMix64 counters -> Irwin-Hall(12) normal -> float32 * std -> optional
// bf16). Every step is integer arithmetic or one correctly rounded IEEE
// operation, so the output bits equal the NumPy implementation's. This file
// holds no optimizer arithmetic; it only fills device buffers with inputs.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t splitmix64_host(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float draw(uint64_t key, uint64_t i, float stdv) {
  const uint64_t base = key + 6ull * i;
  uint64_t s = 0;
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    const uint64_t w = splitmix64(base + k);
    s += (w & 0xFFFFFFFFull) + (w >> 32);
  }
  const double d = static_cast<double>(static_cast<int64_t>(s) - (int64_t(6) << 32)) * 0x1p-32;
  return __fmul_rn(__double2float_rn(d), stdv);
}

__global__ void fill_kernel(void* out, int dtype, int64_t count, uint64_t key, int64_t offset,
                            float stdv) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count;
       i += int64_t(gridDim.x) * blockDim.x) {
    const float x = draw(key, static_cast<uint64_t>(offset + i), stdv);
    if (dtype == 0)
      static_cast<float*>(out)[i] = x;
    else
      static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(x);
  }
}

}  // namespace

extern "C" {

// Fills `count` elements of `out` (device; dtype 0 = fp32, 1 = bf16) with the
// draws for flat indices offset .. offset+count-1 of (seed, tensor_id),
// scaled by `stdv`. Returns 0 or the cudaError_t of the launch.
int synth_normal_fill(void* out, int dtype, int64_t count, uint64_t seed, uint64_t tensor_id,
                      int64_t offset, float stdv, void* stream) {
  if (count <= 0) return 0;
  if (!out || (dtype != 0 && dtype != 1)) return static_cast<int>(cudaErrorInvalidValue);
  const uint64_t key = splitmix64_host(seed ^ splitmix64_host(tensor_id));
  const int64_t blocks64 = (count + 255) / 256;
  const int grid = static_cast<int>(blocks64 < 8192 ? blocks64 : 8192);
  fill_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(out, dtype, count, key, offset,
                                                                    stdv);
  return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
