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
#include "mh_sr.cuh"
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

// Stores 8 values at element i (16-byte aligned): fp32, nearest-even bf16,
// or stochastically rounded bf16 with the given key.
__device__ __forceinline__ void store8_state(void* base, int dt, bool sr, int64_t i, int nvalid,
                                             bool vec, const F8& x, uint32_t key) {
  if (dt == MH_BF16 && sr)
    store_bf16_sr<8>(static_cast<bf16*>(base) + i, nvalid, vec, x.v, key, static_cast<uint64_t>(i));
  else
    store8(base, dt, i, x);
}

__device__ __forceinline__ void store1_state(void* base, int dt, bool sr, int64_t e, float x,
                                             uint32_t key) {
  if (dt == MH_BF16 && sr)
    static_cast<uint16_t*>(base)[e] = sr_bits(x, key, static_cast<uint64_t>(e));
  else
    store1(base, dt, e, x);
}

// One element of AdamW with any mix of dtypes (tails and unaligned tensors).
__device__ __forceinline__ void adam_one(const AdamJob& J, int64_t e, float gmul, float lr,
                                         float decay, const AdamConsts& k, bool psr, bool ssr,
                                         uint32_t kp, uint32_t km, uint32_t kv) {
  float w = load1(J.param, J.pdt, e), m = load1(J.m, J.sdt, e), v = load1(J.v, J.sdt, e);
  adam_elem(w, load1(J.grad, J.gdt, e) * gmul, m, v, lr, decay, k);
  store1_state(J.param, J.pdt, psr, e, w, kp);
  store1_state(J.m, J.sdt, ssr, e, m, km);
  store1_state(J.v, J.sdt, ssr, e, v, kv);
}

// Raw 16-byte loads of 8 elements, unpacked only when consumed.
template <int DT>
struct Raw8 {
  uint4 v[DT == MH_F32 ? 2 : 1];
};

template <int DT>
__device__ __forceinline__ void raw_load8(Raw8<DT>& r, const void* base, int64_t i) {
  const uint4* s = DT == MH_F32
                       ? reinterpret_cast<const uint4*>(static_cast<const float*>(base) + i)
                       : reinterpret_cast<const uint4*>(static_cast<const bf16*>(base) + i);
#pragma unroll
  for (int q = 0; q < (DT == MH_F32 ? 2 : 1); ++q) r.v[q] = __ldcs(s + q);
}

template <int DT>
__device__ __forceinline__ F8 raw_unpack8(const Raw8<DT>& r) {
  F8 o;
  if constexpr (DT == MH_F32) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      o.v[4 * q + 0] = __uint_as_float(r.v[q].x);
      o.v[4 * q + 1] = __uint_as_float(r.v[q].y);
      o.v[4 * q + 2] = __uint_as_float(r.v[q].z);
      o.v[4 * q + 3] = __uint_as_float(r.v[q].w);
    }
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r.v[0]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      o.v[2 * k] = f.x;
      o.v[2 * k + 1] = f.y;
    }
  }
  return o;
}

// A full, 16-byte aligned 16K-element chunk: two groups of 8 elements per
// thread are loaded before either is consumed.
template <int PDT, int GDT, int SDT>
__device__ __forceinline__ void adam_chunk_fast(const AdamJob& J, int64_t start, float gmul,
                                                float lr, float decay, const AdamConsts& k,
                                                bool psr, uint32_t kp, uint32_t km, uint32_t kv) {
  constexpr int kStep = 8 * 256;
  constexpr int kIn = 2;
#pragma unroll 1
  for (int64_t i0 = start + 8 * static_cast<int64_t>(threadIdx.x); i0 < start + kAdamChunk;
       i0 += kIn * kStep) {
    Raw8<PDT> rw[kIn];
    Raw8<GDT> rg[kIn];
    Raw8<SDT> rm[kIn], rv[kIn];
#pragma unroll
    for (int u = 0; u < kIn; ++u) {
      const int64_t i = i0 + u * kStep;
      raw_load8<PDT>(rw[u], J.param, i);
      raw_load8<GDT>(rg[u], J.grad, i);
      raw_load8<SDT>(rm[u], J.m, i);
      raw_load8<SDT>(rv[u], J.v, i);
    }
#pragma unroll
    for (int u = 0; u < kIn; ++u) {
      const int64_t i = i0 + u * kStep;
      F8 w = raw_unpack8<PDT>(rw[u]), g = raw_unpack8<GDT>(rg[u]);
      F8 m = raw_unpack8<SDT>(rm[u]), v = raw_unpack8<SDT>(rv[u]);
#pragma unroll
      for (int e = 0; e < 8; ++e) adam_elem(w.v[e], g.v[e] * gmul, m.v[e], v.v[e], lr, decay, k);
      store8_state(J.param, PDT, psr, i, 8, true, w, kp);
      store8_state(J.m, SDT, SDT == MH_BF16, i, 8, true, m, km);
      store8_state(J.v, SDT, SDT == MH_BF16, i, 8, true, v, kv);
    }
  }
}

template <bool kB16, int PDT, int GDT>
__device__ __forceinline__ void adam_chunk_fast_s(const AdamJob& J, int64_t start, float gmul,
                                                  float lr, float decay, const AdamConsts& k,
                                                  bool psr, uint32_t kp, uint32_t km,
                                                  uint32_t kv) {
  if (kB16 || J.sdt == MH_BF16)
    adam_chunk_fast<PDT, GDT, MH_BF16>(J, start, gmul, lr, decay, k, psr, kp, km, kv);
  else
    adam_chunk_fast<PDT, GDT, MH_F32>(J, start, gmul, lr, decay, k, psr, kp, km, kv);
}

// kB16: every job keeps bf16 moments. That path is bound by the rounding
// arithmetic rather than by bytes in flight; the instantiation carries only
// its fast paths and runs three blocks per SM to hide more of it.
template <bool kB16>
__global__ void __launch_bounds__(256, kB16 ? 3 : 2)
    adamw_kernel(const __grid_constant__ AdamParams p) {
  __shared__ float s_bc[2];
  __shared__ uint64_t s_seed;
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
    // host path; the same count seeds the stochastic rounding.
    if (threadIdx.x == 0) {
      const int64_t t_dev = *p.step < 1 ? 1 : *p.step;
      const double t = static_cast<double>(t_dev);
      s_bc[0] = static_cast<float>(1.0 / (1.0 - pow(static_cast<double>(p.beta1), t)));
      s_bc[1] = static_cast<float>(1.0 / sqrt(1.0 - pow(static_cast<double>(p.beta2), t)));
      s_seed = static_cast<uint64_t>(t_dev);
    }
    __syncthreads();
    k.inv_bc1 = s_bc[0];
    k.inv_sqrt_bc2 = s_bc[1];
  }
  const uint64_t seed = p.step != nullptr ? s_seed : p.sr_seed;

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
    const int sdt = J.sdt;
    const bool ssr = sdt == MH_BF16;             // bf16 moments are always rounded stochastically
    const bool psr = J.psr != 0 && J.pdt == MH_BF16;
    const uint32_t km = ssr ? sr_key(seed, sr_stream(J.tindex, SR_FIRST)) : 0;
    const uint32_t kv = ssr ? sr_key(seed, sr_stream(J.tindex, SR_SECOND)) : 0;
    const uint32_t kp = psr ? sr_key(seed, sr_stream(J.tindex, SR_PARAM)) : 0;
    if (J.vec && end - start == kAdamChunk) {
      if (J.pdt == MH_BF16 && J.gdt == MH_BF16)
        adam_chunk_fast_s<kB16, MH_BF16, MH_BF16>(J, start, gmul, lr, decay, k, psr, kp, km, kv);
      else if (J.pdt == MH_BF16)
        adam_chunk_fast_s<kB16, MH_BF16, MH_F32>(J, start, gmul, lr, decay, k, psr, kp, km, kv);
      else if (J.gdt == MH_BF16)
        adam_chunk_fast_s<kB16, MH_F32, MH_BF16>(J, start, gmul, lr, decay, k, psr, kp, km, kv);
      else
        adam_chunk_fast_s<kB16, MH_F32, MH_F32>(J, start, gmul, lr, decay, k, psr, kp, km, kv);
    } else if (J.vec) {
      for (int64_t i = start + 8 * static_cast<int64_t>(threadIdx.x); i < end; i += 8 * 256) {
        if (i + 8 <= end) {
          F8 w = load8(J.param, J.pdt, i);
          F8 g = load8(J.grad, J.gdt, i);
          F8 m = load8(J.m, sdt, i);
          F8 v = load8(J.v, sdt, i);
#pragma unroll
          for (int e = 0; e < 8; ++e) g.v[e] *= gmul;
#pragma unroll
          for (int e = 0; e < 8; ++e) adam_elem(w.v[e], g.v[e], m.v[e], v.v[e], lr, decay, k);
          store8_state(J.param, J.pdt, psr, i, 8, true, w, kp);
          store8_state(J.m, sdt, ssr, i, 8, true, m, km);
          store8_state(J.v, sdt, ssr, i, 8, true, v, kv);
        } else {
          for (int64_t e = i; e < end; ++e)
            adam_one(J, e, gmul, lr, decay, k, psr, ssr, kp, km, kv);
        }
      }
    } else {
      for (int64_t e = start + threadIdx.x; e < end; e += 256)
        adam_one(J, e, gmul, lr, decay, k, psr, ssr, kp, km, kv);
    }
  }
}

}  // namespace

cudaError_t launch_adamw(const AdamParams& p, int num_sms, cudaStream_t s) {
  if (p.total_chunks <= 0) return cudaSuccess;
  bool all_b16 = p.njobs > 0;
  for (int j = 0; j < p.njobs; ++j) all_b16 = all_b16 && p.jobs[j].sdt == MH_BF16;
  // One wave of resident blocks: two per SM (108 registers), three for the
  // bf16-moment instantiation.
  const int64_t want = static_cast<int64_t>(num_sms) * (all_b16 ? 3 : 2);
  const int grid = static_cast<int>(p.total_chunks < want ? p.total_chunks : want);
  if (all_b16)
    adamw_kernel<true><<<grid, 256, 0, s>>>(p);
  else
    adamw_kernel<false><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mh
