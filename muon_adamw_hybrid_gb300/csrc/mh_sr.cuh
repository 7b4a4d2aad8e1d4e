// Stochastic rounding of fp32 values to bf16 (dew.training.optim,
// "stochastic_round_bf16"; "bf16_moments"): 16 uniform bits are added below
// the kept mantissa of the fp32 pattern and the low half is dropped, so a value
// rounds up with the probability of its distance to the lower bf16 neighbour.
// NaN stays NaN (the quiet NaN of its sign).
//
// The noise is a counter-based hash, a pure function of (seed, stream, flat
// index), built from the 32-bit finaliser of MurmurHash3 (fmix32):
//   key       = fmix32(fmix32(fmix32(stream) ^ seed_lo) ^ seed_hi)
//   noise(i)  = low (i even) or high (i odd) 16 bits of fmix32(key + floor(i/2))
// all mod 2^32, with stream = 4 * (tensor index in the call) + moment (0: Muon
// momentum or AdamW first moment, 1: AdamW second moment, 2: the parameter).
// One 32-bit hash serves two consecutive elements: a handful of integer
// operations per value, so the bf16-state passes stay HBM-bound.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace mh {

enum : int { SR_FIRST = 0, SR_SECOND = 1, SR_PARAM = 2 };

__host__ __device__ __forceinline__ uint32_t sr_fmix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x85EBCA6Bu;
  x ^= x >> 13;
  x *= 0xC2B2AE35u;
  x ^= x >> 16;
  return x;
}

__host__ __device__ __forceinline__ uint32_t sr_key(uint64_t seed, uint64_t stream) {
  return sr_fmix32(sr_fmix32(sr_fmix32(static_cast<uint32_t>(stream)) ^
                             static_cast<uint32_t>(seed)) ^
                   static_cast<uint32_t>(seed >> 32));
}

__host__ __device__ __forceinline__ uint64_t sr_stream(int64_t tensor_index, int moment) {
  return 4ull * static_cast<uint64_t>(tensor_index) + static_cast<uint64_t>(moment);
}

// fp32 pattern whose high half is x's stochastically rounded bf16 pattern.
__device__ __forceinline__ uint32_t sr_word(float x, uint32_t noise16) {
  const uint32_t u = __float_as_uint(x);
  const bool nan = (u & 0x7FFFFFFFu) > 0x7F800000u;
  return nan ? ((u & 0x80000000u) | 0x7FC00000u) : u + noise16;
}

__device__ __forceinline__ uint32_t sr_noise(uint32_t key, uint64_t index) {
  const uint32_t h = sr_fmix32(key + static_cast<uint32_t>(index >> 1));
  return (index & 1) ? (h >> 16) : (h & 0xFFFFu);
}

// Rounds x[0..N) (flat indices index0 .. index0+N-1, N even) into N/2 packed
// bf16 pairs (element 2k in the low half of word k).
template <int N>
__device__ __forceinline__ void sr_round_pairs(const float (&x)[N], uint32_t key, uint64_t index0,
                                               uint32_t (&out)[N / 2]) {
  static_assert(N % 2 == 0, "pairs of elements");
  if ((index0 & 1) == 0) {
    const uint32_t base = key + static_cast<uint32_t>(index0 >> 1);
#pragma unroll
    for (int q = 0; q < N / 2; ++q) {
      const uint32_t h = sr_fmix32(base + q);
      out[q] = __byte_perm(sr_word(x[2 * q], h & 0xFFFFu), sr_word(x[2 * q + 1], h >> 16),
                           0x7632);
    }
  } else {
#pragma unroll
    for (int q = 0; q < N / 2; ++q)
      out[q] = __byte_perm(sr_word(x[2 * q], sr_noise(key, index0 + 2 * q)),
                           sr_word(x[2 * q + 1], sr_noise(key, index0 + 2 * q + 1)), 0x7632);
  }
}

// Stores x[0..nvalid) (nvalid <= N) as stochastically rounded bf16 at dst.
// vec: dst is aligned to the vector (8 bytes for N = 4, 16 bytes for N a
// multiple of 8) and nvalid == N.
template <int N>
__device__ __forceinline__ void store_bf16_sr(__nv_bfloat16* dst, int nvalid, bool vec,
                                              const float (&x)[N], uint32_t key,
                                              uint64_t index0) {
  uint32_t w[N / 2];
  sr_round_pairs<N>(x, key, index0, w);
  if (vec && nvalid == N) {
    if constexpr (N == 4) {
      __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w[0], w[1]));
      return;
    } else {
      static_assert(N % 8 == 0, "vector stores take 8 bf16 values at a time");
#pragma unroll
      for (int q = 0; q < N / 8; ++q)
        __stcs(reinterpret_cast<uint4*>(dst) + q,
               make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
      return;
    }
  }
  uint16_t* d = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (k < nvalid) d[k] = static_cast<uint16_t>((k & 1) ? (w[k / 2] >> 16) : (w[k / 2] & 0xFFFFu));
}

// One stochastically rounded bf16 pattern (tails and unaligned tensors).
__device__ __forceinline__ uint16_t sr_bits(float x, uint32_t key, uint64_t index) {
  return static_cast<uint16_t>(sr_word(x, sr_noise(key, index)) >> 16);
}

}  // namespace mh
