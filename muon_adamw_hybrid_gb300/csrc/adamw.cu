// Fused multi-tensor AdamW step (the AdamW half of the hybrid optimizer).
//
// The pages name AdamW without printing it (dew.training.optim "OPTIMIZER_MAP":
// optax.adamw; Speedtronic "v2 optimizers", "CPU/CUDA/MPS behavior": PyTorch's
// fused AdamW). This is the standard decoupled form with bias correction:
//   m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2
//   W <- W (1 - lr wd) - lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)
//
// HBM-bound: every element is read once and written once (W, m, v) and the
// gradient is read once. One work item is a 16K-element chunk of one tensor;
// a persistent grid walks the chunks of all tensors of the launch, and each
// thread moves 8 elements per iteration with 16-byte loads and stores.
#include "mh_internal.h"
#include "muonhybrid.h"

namespace mh {

static_assert(sizeof(AdamParams) <= 32000, "AdamParams exceeds the kernel parameter space");

namespace {

struct F8 {
  float v[8];
};

__device__ __forceinline__ F8 load8(const void* base, int dt, int64_t i) {
  F8 r;
  if (dt == MH_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    float4 a = __ldcs(p), b = __ldcs(p + 1);
    r.v[0] = a.x; r.v[1] = a.y; r.v[2] = a.z; r.v[3] = a.w;
    r.v[4] = b.x; r.v[5] = b.y; r.v[6] = b.z; r.v[7] = b.w;
  } else {
    uint4 u = __ldcs(reinterpret_cast<const uint4*>(static_cast<const bf16*>(base) + i));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 f = __bfloat1622float2(h[k]);
      r.v[2 * k] = f.x;
      r.v[2 * k + 1] = f.y;
    }
  }
  return r;
}

__device__ __forceinline__ void store8(void* base, int dt, int64_t i, const F8& x) {
  if (dt == MH_F32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + i);
    __stcs(p, make_float4(x.v[0], x.v[1], x.v[2], x.v[3]));
    __stcs(p + 1, make_float4(x.v[4], x.v[5], x.v[6], x.v[7]));
  } else {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(x.v[2 * k], x.v[2 * k + 1]);
    __stcs(reinterpret_cast<uint4*>(static_cast<bf16*>(base) + i), u);
  }
}

__device__ __forceinline__ float load1(const void* base, int dt, int64_t i) {
  return dt == MH_F32 ? static_cast<const float*>(base)[i]
                      : __bfloat162float(static_cast<const bf16*>(base)[i]);
}

__device__ __forceinline__ void store1(void* base, int dt, int64_t i, float x) {
  if (dt == MH_F32)
    static_cast<float*>(base)[i] = x;
  else
    static_cast<bf16*>(base)[i] = __float2bfloat16_rn(x);
}

struct AdamConsts {
  float b1, omb1, b2, omb2, eps, inv_bc1, inv_sqrt_bc2;
};

// One element of AdamW in fp32.
__device__ __forceinline__ void adam_elem(float& w, float g, float& m, float& v, float lr,
                                          float decay, const AdamConsts& k) {
  m = k.b1 * m + k.omb1 * g;
  v = k.b2 * v + k.omb2 * (g * g);
  const float denom = sqrtf(v) * k.inv_sqrt_bc2 + k.eps;
  w = w * decay - (lr * k.inv_bc1) * (m / denom);
}

__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamParams p) {
  __shared__ float s_bc[2];
  if (step_skipped(p.skip)) return;
  const float gmul = p.grad_mult != nullptr ? *p.grad_mult : 1.0f;
  AdamConsts k;
  k.b1 = p.beta1;
  k.omb1 = 1.0f - p.beta1;
  k.b2 = p.beta2;
  k.omb2 = 1.0f - p.beta2;
  k.eps = p.eps;
  k.inv_bc1 = p.inv_bc1;
  k.inv_sqrt_bc2 = p.inv_sqrt_bc2;
  if (p.step != nullptr) {
    // Bias corrections from the device step count (advanced by the gradient
    // control only on applied steps), once per block, in double like the
    // host path.
    if (threadIdx.x == 0) {
      const double t = static_cast<double>(*p.step < 1 ? 1 : *p.step);
      s_bc[0] = static_cast<float>(1.0 / (1.0 - pow(static_cast<double>(p.beta1), t)));
      s_bc[1] = static_cast<float>(1.0 / sqrt(1.0 - pow(static_cast<double>(p.beta2), t)));
    }
    __syncthreads();
    k.inv_bc1 = s_bc[0];
    k.inv_sqrt_bc2 = s_bc[1];
  }

  for (int64_t chunk = blockIdx.x; chunk < p.total_chunks; chunk += gridDim.x) {
    int lo = 0, hi = p.njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.jobs[mid].chunk_begin <= chunk) lo = mid; else hi = mid - 1;
    }
    const AdamJob& J = p.jobs[lo];
    const int64_t start = (chunk - J.chunk_begin) * kAdamChunk;
    const int64_t end = min(start + kAdamChunk, J.numel);
    const float lr = J.lr;
    const float decay = 1.0f - J.lr * J.wd;
    if (J.vec) {
      for (int64_t i = start + 8 * static_cast<int64_t>(threadIdx.x); i < end; i += 8 * 256) {
        if (i + 8 <= end) {
          F8 w = load8(J.param, J.pdt, i);
          F8 g = load8(J.grad, J.gdt, i);
#pragma unroll
          for (int e = 0; e < 8; ++e) g.v[e] *= gmul;
          F8 m = load8(J.m, MH_F32, i);
          F8 v = load8(J.v, MH_F32, i);
#pragma unroll
          for (int e = 0; e < 8; ++e) adam_elem(w.v[e], g.v[e], m.v[e], v.v[e], lr, decay, k);
          store8(J.param, J.pdt, i, w);
          store8(J.m, MH_F32, i, m);
          store8(J.v, MH_F32, i, v);
        } else {
          for (int64_t e = i; e < end; ++e) {
            float w = load1(J.param, J.pdt, e), m = J.m[e], v = J.v[e];
            adam_elem(w, load1(J.grad, J.gdt, e) * gmul, m, v, lr, decay, k);
            store1(J.param, J.pdt, e, w);
            J.m[e] = m;
            J.v[e] = v;
          }
        }
      }
    } else {
      for (int64_t e = start + threadIdx.x; e < end; e += 256) {
        float w = load1(J.param, J.pdt, e), m = J.m[e], v = J.v[e];
        adam_elem(w, load1(J.grad, J.gdt, e) * gmul, m, v, lr, decay, k);
        store1(J.param, J.pdt, e, w);
        J.m[e] = m;
        J.v[e] = v;
      }
    }
  }
}

}  // namespace

cudaError_t launch_adamw(const AdamParams& p, int num_sms, cudaStream_t s) {
  if (p.total_chunks <= 0) return cudaSuccess;
  const int64_t want = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(p.total_chunks < want ? p.total_chunks : want);
  adamw_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mh
