// QK-Clip rescale after the optimizer update (kimi-k3 "Optimization",
// "QK-Clip watches a different failure mode"; dew.training.optim
// "scale_by_qk_clip", Kimi K2's MuonClip): for every head h whose observed
// maximum query-key score s_h exceeds tau, selected rows of its query and key
// projections are multiplied by gamma_h^exponent, gamma_h = min(1, tau/s_h);
// rows of heads at or below tau are not touched (not even rewritten).
//
// One warp per scaled row, 8 elements per lane per access; the per-head
// factor is read from device memory, so the call needs no host round trip.
#include <cmath>

#include "mh_internal.h"
#include "muonhybrid.h"

namespace mh {

static_assert(sizeof(QkClipParams) <= 32000, "QkClipParams exceeds the kernel parameter space");

namespace {

__device__ __forceinline__ void scale_row(void* base, int dt, int64_t off, int64_t cols, bool vec,
                                          float f) {
  const int lane = threadIdx.x & 31;
  if (dt == MH_F32) {
    float* p = static_cast<float*>(base) + off;
    if (vec) {
      for (int64_t c = 4 * lane; c + 4 <= cols; c += 128) {
        float4 v = *reinterpret_cast<float4*>(p + c);
        v.x *= f; v.y *= f; v.z *= f; v.w *= f;
        *reinterpret_cast<float4*>(p + c) = v;
      }
    } else {
      for (int64_t c = lane; c < cols; c += 32) p[c] *= f;
    }
  } else {
    bf16* p = static_cast<bf16*>(base) + off;
    if (vec) {
      for (int64_t c = 8 * lane; c + 8 <= cols; c += 256) {
        uint4 u = *reinterpret_cast<uint4*>(p + c);
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x = __bfloat1622float2(h[k]);
          h[k] = __floats2bfloat162_rn(x.x * f, x.y * f);
        }
        *reinterpret_cast<uint4*>(p + c) = u;
      }
    } else {
      for (int64_t c = lane; c < cols; c += 32)
        p[c] = __float2bfloat16_rn(__bfloat162float(p[c]) * f);
    }
  }
}

__global__ void __launch_bounds__(256) qk_clip_kernel(const __grid_constant__ QkClipParams p) {
  if (step_skipped(p.skip)) return;  // nothing is clipped after a skipped step
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < p.total_rows; row += warps) {
    int lo = 0, hi = p.nentries - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.entries[mid].row_begin <= row) lo = mid; else hi = mid - 1;
    }
    const QkClipEntry& E = p.entries[lo];
    const int64_t local = row - E.row_begin;
    const int64_t h = local / E.scaled_rows;
    const int64_t r = h * E.head_stride + E.row_offset + (local - h * E.scaled_rows);
    const float s = p.s_max[E.head_index0 + h];
    if (!(s > p.tau)) continue;  // warp-uniform; NaN scores are left alone
    const float f = powf(p.tau / s, E.exponent);
    scale_row(E.param, E.dt, r * E.cols, E.cols, E.vec != 0 && (E.cols % 8) == 0, f);
  }
}

}  // namespace

cudaError_t launch_qk_clip(const QkClipParams& p, int num_sms, cudaStream_t s) {
  if (p.total_rows <= 0) return cudaSuccess;
  const int64_t want_blocks = (p.total_rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(want_blocks < cap ? want_blocks : cap);
  qk_clip_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mh
