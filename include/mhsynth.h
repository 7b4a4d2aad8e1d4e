/*
 * mhsynth.h -- seeded synthetic input generator (test and benchmark inputs).
 *
 * Not part of the optimizer: it fills device buffers with the same numbers the
 * NumPy generator in synth/__init__.py produces on the host, bit for bit, so
 * that the CPU oracle and the GPU path can be given identical inputs without
 * either one producing data for the other.
 *
 * Definition: key = splitmix64(seed ^ splitmix64(tensor_id)); element i sums
 * the twelve 32-bit halves of splitmix64(key + 6 i + k), k = 0..5, into S;
 * x = float32((S - 6 * 2^32) * 2^-32) * std (Irwin-Hall(12) normal), then
 * optionally rounded to bf16 (nearest, ties to even).
 */
#ifndef MHSYNTH_H
#define MHSYNTH_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif
/* out: device buffer of `count` elements, dtype 0 = fp32, 1 = bf16. stream:
 * cudaStream_t as void*. Returns 0, or a cudaError_t value on failure. */
int synth_normal_fill(void* out, int dtype, int64_t count, uint64_t seed, uint64_t tensor_id,
                      int64_t offset, float stdv, void* stream);
#ifdef __cplusplus
}
#endif
#endif
