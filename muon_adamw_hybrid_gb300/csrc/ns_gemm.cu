// Grouped Newton-Schulz GEMM stage on sm_103a tensor cores (tcgen05 + TMEM,
// operands staged by TMA with 128-byte swizzle).
//
// One quintic step (Speedtronic "v2 optimizers", "Newton-Schulz"; flaxchat
// "Optimizer", "Muon Algorithm" step 2) is three launches of this kernel:
//
//   GEMM_GRAM   A = X X^T             (m x m; only tiles touching the upper
//                                      triangle are computed, each element
//                                      c >= r is stored and mirrored to (c, r))
//   GEMM_POLY   P = b A + c A A       (A symmetric, so A A = A A^T: both
//                                      operands are K-major rows of A; same
//                                      triangle scheme; b A read in the epilogue)
//   GEMM_APPLY  X' = a X + P X        (B operand = X read MN-major)
//
// On the first step the Frobenius normalisation 1/(||Q||_F + eps) is folded in:
// the gram epilogue scales by s^2 and the apply epilogue by s, so the
// prologue never has to re-read Q to normalise it.
//
// Layout: every view of every shape class is one problem; a persistent CTA
// (one per SM) walks a static list of 128 x 256 output tiles spanning all
// classes. Warp roles: warp 0 issues TMA loads into a 4-stage ring, warp 1
// issues tcgen05.mma (M=128, N=256, K=16) into one of two TMEM accumulators,
// warp 2 owns the TMEM allocation, warps 4-7 drain an accumulator with
// tcgen05.ld, apply the stage's epilogue in fp32 and store bf16, while the
// MMA warp already fills the other accumulator.
//
// Every mbarrier wait is bounded; on timeout the CTA records a status code in
// the workspace, drains what it has in flight, frees TMEM and exits.
#include "mh_internal.h"
#include "mh_ptx.cuh"

namespace mh {
namespace {

constexpr uint32_t kStageABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kStageBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kTmemCols = 2 * kBN;           // two fp32 accumulators
constexpr uint32_t kApplyChunkBytes = kBK * 64 * 2;  // one 64-col MN-major box: 8 KB

struct TileCoord {
  int cls, view, tm, tn;
};

__device__ __forceinline__ TileCoord map_tile(const GemmParams& p, int64_t t) {
  int c = 0;
  while (c + 1 < p.num_classes && t >= p.cls[c + 1].tile_begin) ++c;
  const GemmClass& C = p.cls[c];
  const int64_t local = t - C.tile_begin;
  TileCoord tc;
  tc.cls = c;
  tc.view = static_cast<int>(local / C.tiles_per_view);
  int w = static_cast<int>(local - static_cast<int64_t>(tc.view) * C.tiles_per_view);
  if (p.kind == GEMM_APPLY) {
    tc.tm = w % C.tiles_m;
    tc.tn = w / C.tiles_m;
  } else {
    // Row tm of 128 holds the 256-wide column tiles tn >= tm/2 (those that
    // reach the diagonal or lie above it).
    int tm = 0;
    while (true) {
      const int cnt = C.tiles_n - (tm >> 1);
      if (w < cnt) break;
      w -= cnt;
      ++tm;
    }
    tc.tm = tm;
    tc.tn = (tm >> 1) + w;
  }
  return tc;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void load_bf16x32(const bf16* src, float (&x)[32]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = s[q];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      x[q * 8 + 2 * k] = f.x;
      x[q * 8 + 2 * k + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void store_bf16x32(bf16* dst, const float (&x)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(x[q * 8 + 0], x[q * 8 + 1]);
    u.y = pack_bf16x2(x[q * 8 + 2], x[q * 8 + 3]);
    u.z = pack_bf16x2(x[q * 8 + 4], x[q * 8 + 5]);
    u.w = pack_bf16x2(x[q * 8 + 6], x[q * 8 + 7]);
    d[q] = u;
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kStageBBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int c = 0; c < p.num_classes; ++c) {
      prefetch_tmap(&p.cls[c].tmA);
      prefetch_tmap(&p.cls[c].tmB);
    }
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool apply = p.kind == GEMM_APPLY;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t inflight = 0;             // stages with a load issued
      uint32_t inflight_par = 0;         // parity of that load's phase
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
        const TileCoord tc = map_tile(p, t);
        const GemmClass& C = p.cls[tc.cls];
        const int nk = (C.K + kBK - 1) / kBK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_TMA)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kStageABytes + kStageBBytes);
          tma_load_3d(sA + stage * kStageABytes, &C.tmA, &full[stage], kb * kBK, tc.tm * kBM,
                      tc.view);
          uint8_t* b_dst = sB + stage * kStageBBytes;
          if (apply) {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j)
              tma_load_3d(b_dst + j * kApplyChunkBytes, &C.tmB, &full[stage], tc.tn * kBN + j * 64,
                          kb * kBK, tc.view);
          } else {
            tma_load_3d(b_dst, &C.tmB, &full[stage], kb * kBK, tc.tn * kBN, tc.view);
          }
          inflight |= 1u << stage;
          inflight_par = (inflight_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Let every issued copy land before the CTA's shared memory goes away.
        for (int s = 0; s < kStages; ++s)
          if (inflight & (1u << s)) mbar_wait_drain(&full[s], (inflight_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, kBN, 0, apply ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int64_t t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
        const TileCoord tc = map_tile(p, t);
        const GemmClass& C = p.cls[tc.cls];
        const int nk = (C.K + kBK - 1) / kBK;
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, p.status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(sA + stage * kStageABytes);
          const uint32_t b0 = smem_addr(sB + stage * kStageBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // K-major A: 16 bf16 of k = 32 bytes inside the 128-byte swizzle row.
            const uint64_t ad = smem_desc_sw128(a0 + k * 32, 16, 1024);
            // K-major B likewise; MN-major B: 16 k-rows = two 1024-byte atoms,
            // 64-col chunks 8 KB apart.
            const uint64_t bd = apply ? smem_desc_sw128(b0 + k * 2048, kApplyChunkBytes, 1024)
                                      : smem_desc_sw128(b0 + k * 32, 16, 1024);
            tc_mma_f16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok && issued) {
        tc_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int ew = warp - 4;  // TMEM lanes 32*ew .. 32*ew+31
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const TileCoord tc = map_tile(p, t);
      const GemmClass& C = p.cls[tc.cls];
      if (!mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, p.status, DEV_TIMEOUT_EPI)) break;
      tc_fence_after();

      const int r = tc.tm * kBM + ew * 32 + lane;
      const int n_out = apply ? C.n : C.m;
      float sc = 1.0f;
      if (p.first_iter) {
        const float s = 1.0f / (sqrtf(static_cast<float>(C.sumsq[tc.view])) + p.eps);
        sc = apply ? s : s * s;
      }
      bf16* out = C.out + static_cast<int64_t>(tc.view) * C.out_view_stride;
      const bf16* aux = C.aux + static_cast<int64_t>(tc.view) * C.aux_view_stride;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                             static_cast<uint32_t>(acc * kBN);

#pragma unroll 1
      for (int cc = 0; cc < kBN / 32; ++cc) {
        const int c0 = tc.tn * kBN + cc * 32;
        if (c0 >= n_out) break;  // warp-uniform
        uint32_t raw[32];
        tmem_ld_32x32b_x32(t_row + cc * 32, raw);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
        const bool row_ok = r < C.m;
        const bool full_cols = c0 + 32 <= n_out;

        if (apply) {
          if (row_ok) {
            const int64_t off = static_cast<int64_t>(r) * C.ld_out + c0;
            const int64_t aoff = static_cast<int64_t>(r) * C.ld_aux + c0;
            if (full_cols) {
              float x[32];
              load_bf16x32(aux + aoff, x);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = sc * (p.a * x[j] + v[j]);
              store_bf16x32(out + off, v);
            } else {
              for (int j = 0; j < n_out - c0; ++j)
                out[off + j] = __float2bfloat16_rn(sc * (p.a * __bfloat162float(aux[aoff + j]) + v[j]));
            }
          }
        } else {
          // Symmetric output: element (r, c) with c >= r is stored at (r, c)
          // and, when c > r, mirrored to (c, r).
          if (p.kind == GEMM_POLY) {
            if (row_ok) {
              const int64_t aoff = static_cast<int64_t>(r) * C.ld_aux + c0;
              if (full_cols) {
                float x[32];
                load_bf16x32(aux + aoff, x);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = p.b * x[j] + p.c * v[j];
              } else {
                for (int j = 0; j < 32; ++j)
                  if (c0 + j < n_out) v[j] = p.b * __bfloat162float(aux[aoff + j]) + p.c * v[j];
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= sc;
          }
          if (row_ok) {
            const int64_t off = static_cast<int64_t>(r) * C.ld_out + c0;
            if (full_cols && c0 >= r) {
              store_bf16x32(out + off, v);
            } else {
              for (int j = 0; j < 32; ++j) {
                const int c = c0 + j;
                if (c < n_out && c >= r) out[off + j] = __float2bfloat16_rn(v[j]);
              }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int c = c0 + j;
              if (c < n_out && c > r)
                out[static_cast<int64_t>(c) * C.ld_out + r] = __float2bfloat16_rn(v[j]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

size_t gemm_smem_bytes() {
  return 1024 + kStages * (kStageABytes + kStageBBytes) + (2 * kStages + 5) * sizeof(uint64_t) + 16;
}

cudaError_t launch_ns_gemm(const GemmParams& p, int grid, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const size_t smem = gemm_smem_bytes();
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(ns_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int g = static_cast<int>(p.total_tiles < grid ? p.total_tiles : grid);
  ns_gemm_kernel<<<g, kGemmThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mh
