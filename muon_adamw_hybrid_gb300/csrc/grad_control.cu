// Gradient control ahead of both halves of the hybrid step: the global norm of
// the unscaled gradients, the clip factor and the overflow skip.
//
// kimi-k3 "Optimization", "Keep the arithmetic and gradients under control":
// the trainer measures one global gradient norm before the optimizer step,
// clips it when max_grad_norm > 0 (0: observed only), and an FP16 overflow
// skips the whole hybrid update. dew.training.optim "build_optimizer": the
// clip reads every gradient of every parameter group together.
//
// Pass 1 (grad_sumsq_kernel, HBM-bound: every gradient element is read once)
// writes one fp64 partial per 65536-element chunk; a chunk holding an inf or
// NaN writes NaN. Pass 2 (grad_finalize_kernel, one block) sums the partials
// in a fixed order and writes the decision to device memory, where the step
// kernels read it: no host round trip, bitwise reproducible.
#include <cmath>

#include "mh_internal.h"
#include "muonhybrid.h"

namespace mh {

static_assert(sizeof(GradParams) <= 32000, "GradParams exceeds the kernel parameter space");

namespace {

constexpr int kGradThreads = 256;
constexpr int kGradPerThread = 8;
constexpr int kGradUnroll = 4;

__device__ __forceinline__ void load_grad8(const GradJob& J, int64_t i, int64_t end, float (&g)[8]) {
  if (i >= end) {
#pragma unroll
    for (int k = 0; k < 8; ++k) g[k] = 0.0f;
    return;
  }
  if (J.vec && i + 8 <= end) {
    if (J.gdt == MH_F32) {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(J.grad) + i);
      const float4 a = __ldcs(p), b = __ldcs(p + 1);
      g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
      g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
    } else {
      const uint4 u = __ldcs(reinterpret_cast<const uint4*>(static_cast<const bf16*>(J.grad) + i));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        g[2 * k] = f.x;
        g[2 * k + 1] = f.y;
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int64_t e = i + k;
    g[k] = e < end ? (J.gdt == MH_F32 ? static_cast<const float*>(J.grad)[e]
                                      : __bfloat162float(static_cast<const bf16*>(J.grad)[e]))
                   : 0.0f;
  }
}

// Sum of the squares of 8 unscaled gradients (fp32); flags inf / NaN.
__device__ __forceinline__ float sumsq8(const float (&g)[8], float inv_scale, bool& bad) {
  float s8 = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float x = g[k] * inv_scale;
    bad |= !isfinite(x);
    s8 = fmaf(x, x, s8);
  }
  return s8;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kGradThreads) grad_sumsq_kernel(const __grid_constant__ GradParams p) {
  __shared__ double sWarp[kGradThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t c = blockIdx.x; c < p.nchunks; c += gridDim.x) {
    const int64_t chunk = p.chunk_first + c;
    int lo = 0, hi = p.njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.jobs[mid].chunk_begin <= chunk) lo = mid; else hi = mid - 1;
    }
    const GradJob& J = p.jobs[lo];
    const int64_t start = (chunk - J.chunk_begin) * kGradChunk;
    const int64_t end = min(start + kGradChunk, J.numel);
    // fp32 within this thread's share of the chunk (at most 256 squares),
    // fp64 from there on; four 16-byte loads in flight per thread before any
    // is consumed.
    float acc = 0.0f;
    bool bad = false;
    constexpr int kStep = kGradPerThread * kGradThreads;  // elements per block-wide load
    for (int64_t i = start + kGradPerThread * static_cast<int64_t>(threadIdx.x); i < end;
         i += kGradUnroll * kStep) {
      if (J.vec && i + (kGradUnroll - 1) * kStep + 8 <= end) {
        // Interior: all loads issued back to back, then the arithmetic.
        if (J.gdt == MH_F32) {
          const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(J.grad) + i);
          float4 r[kGradUnroll][2];
#pragma unroll
          for (int u = 0; u < kGradUnroll; ++u) {
            r[u][0] = __ldcs(src + u * (kStep / 4));
            r[u][1] = __ldcs(src + u * (kStep / 4) + 1);
          }
#pragma unroll
          for (int u = 0; u < kGradUnroll; ++u) {
            const float g[8] = {r[u][0].x, r[u][0].y, r[u][0].z, r[u][0].w,
                                r[u][1].x, r[u][1].y, r[u][1].z, r[u][1].w};
            acc += sumsq8(g, p.inv_scale, bad);
          }
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(static_cast<const bf16*>(J.grad) + i);
          uint4 r[kGradUnroll];
#pragma unroll
          for (int u = 0; u < kGradUnroll; ++u) r[u] = __ldcs(src + u * (kStep / 8));
#pragma unroll
          for (int u = 0; u < kGradUnroll; ++u) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r[u]);
            float g[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = __bfloat1622float2(h[k]);
              g[2 * k] = f.x;
              g[2 * k + 1] = f.y;
            }
            acc += sumsq8(g, p.inv_scale, bad);
          }
        }
      } else {
        // Tail of a tensor, or a misaligned one: bounds-checked loads.
#pragma unroll 1
        for (int u = 0; u < kGradUnroll; ++u) {
          float g[8];
          load_grad8(J, i + u * kStep, end, g);
          acc += sumsq8(g, p.inv_scale, bad);
        }
      }
    }
    const int any_bad = __syncthreads_or(bad ? 1 : 0);
    const double w = warp_sum_d(static_cast<double>(acc));
    if (lane == 0) sWarp[warp] = w;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
#pragma unroll
      for (int k = 0; k < kGradThreads / 32; ++k) t += sWarp[k];
      p.partial[chunk] = any_bad ? nan("") : t;
    }
    __syncthreads();  // sWarp is reused by the next chunk
  }
}

constexpr int kFinThreads = 1024;

__global__ void __launch_bounds__(kFinThreads) grad_finalize_kernel(const __grid_constant__ GradFinParams p) {
  __shared__ double sWarp[kFinThreads / 32];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < p.nchunks; i += kFinThreads) acc += p.partial[i];
  acc = warp_sum_d(acc);
  if ((threadIdx.x & 31) == 0) sWarp[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int k = 0; k < kFinThreads / 32; ++k) total += sWarp[k];
    const bool skip = isnan(total);
    const double norm = skip ? nan("") : sqrt(total);
    double mult = 0.0;
    if (!skip) {
      double coef = 1.0;
      if (p.max_norm > 0.0) coef = fmin(1.0, p.max_norm / (norm + p.clip_eps));
      mult = p.inv_scale * coef;
    }
    *p.norm = norm;
    *p.mult = static_cast<float>(mult);
    *p.skip = skip ? 1 : 0;
    if (p.step != nullptr && !skip) *p.step += 1;
  }
}

}  // namespace

cudaError_t launch_grad_sumsq(const GradParams& p, int num_sms, cudaStream_t s) {
  if (p.nchunks <= 0) return cudaSuccess;
  const int64_t want = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(p.nchunks < want ? p.nchunks : want);
  grad_sumsq_kernel<<<grid, kGradThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_grad_finalize(const GradFinParams& p, cudaStream_t s) {
  grad_finalize_kernel<<<1, kFinThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mh
