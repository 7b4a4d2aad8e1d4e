// Elementwise passes of the Muon update, all HBM-bound and tiled over the
// stored (rows x cols) layout of each view in 32 x 256 tiles (the prologue of
// views whose columns are a multiple of 8 streams contiguous 8192-element
// chunks instead). The prologue deals tiles to the blocks of its persistent
// grid round robin, so that all blocks stream neighbouring chunks (6.5 TB/s
// on the 7B set; contiguous ranges per block ran at 6.2). The passes after the
// Newton-Schulz stages give each block one contiguous range, since their
// tensors are small and a block changing job record on nearly every tile cost
// more than the scattered access (MoE set apply: 2.5 -> 3.9 TB/s).
//
//   EW_PROLOGUE  B <- mu B + (1-mu) G;  Q = lerp(G, B, mu) (or B);
//                writes B (fp32 or bf16) and bf16(Q) into the Newton-Schulz
//                buffer (every view in its stored layout; the GEMMs read tall
//                views transposed), and per-warp partials of ||Q||_F^2 from
//                fp32 Q.
//                Speedtronic "v2 optimizers", "Muon update" / "Newton-Schulz";
//                flaxchat "Optimizer", "Muon Algorithm" step 1.
//   EW_ROWSQ     per stored row and column tile: sum_j U_ij^2 (NorMuon
//                statistics, Muon+ rows), as partials summed later in order.
//   EW_COLSQ     per stored col and row tile: sum_i (f_i U_ij)^2 (Muon+
//                columns), likewise.
//   EW_APPLY     W <- (1 - lr wd) W - lr s U, or a cautious form, with
//                U_ij = f_i h_j X_ij, f from NorMuon and Muon+ rows, h from
//                Muon+ columns. Speedtronic "Muon update",
//                "Muon+", "Cautious updates"; flaxchat step 4.
//   EW_COPYOUT   Newton-Schulz-only output U in the caller's dtype.
//
// Plus the per-view row finalisation (NorMuon state update, norm restore,
// Muon+ row factor; flaxchat step 3, Speedtronic "Muon+").
#include <atomic>
#include <cstring>
#include <unordered_map>
#include "mh_internal.h"
#include "mh_ptx.cuh"
#include "mh_sr.cuh"
#include "muonhybrid.h"

namespace mh {

// Kernel parameters live in the 32 KB (32764-byte) parameter space.
static_assert(sizeof(EwParams) <= 32000, "EwParams exceeds the kernel parameter space");
static_assert(sizeof(RowFinParams) <= 32000, "RowFinParams exceeds the kernel parameter space");
static_assert(sizeof(ColFinParams) <= 32000, "ColFinParams exceeds the kernel parameter space");
static_assert(sizeof(NormParams) <= 32000, "NormParams exceeds the kernel parameter space");
static_assert(sizeof(ActiveParams) <= 32000, "ActiveParams exceeds the kernel parameter space");

namespace {


__device__ __forceinline__ int find_job(const EwParams& p, int64_t tile) {
  int lo = 0, hi = p.njobs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.jobs[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct TileInfo {
  int job;
  int64_t v, r0, c0;
};

// Issues this thread's loads of its 4 x 8 block of U (rows r0+4*warp+i, cols
// c0+8*lane+k) from the Newton-Schulz output buffer, which holds every view in
// its stored layout (row pitch ldx, a multiple of 8: every row load is
// 16-byte aligned). All four loads are issued before any is used.
__device__ __forceinline__ void load_u_raw(const EwJob& J, const TileInfo& t, uint4 (&raw)[4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bf16* xv = J.xf + t.v * J.x_view_stride;
  const int64_t col = t.c0 + lane * 8;
  const int64_t nv = J.cols - col;
  const int nvalid = nv >= 8 ? 8 : (nv > 0 ? static_cast<int>(nv) : 0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = t.r0 + warp * 4 + i;
    raw[i] = make_uint4(0u, 0u, 0u, 0u);
    if (row < J.rows && nvalid == 8)
      raw[i] = __ldcs(reinterpret_cast<const uint4*>(xv + row * J.ldx + col));
  }
}

// Unpacks the block issued by load_u_raw (ragged last columns are read here),
// times `scale`.
__device__ __forceinline__ void unpack_u_block(const EwJob& J, const TileInfo& t,
                                               const uint4 (&raw)[4], float u[4][8],
                                               float scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bf16* xv = J.xf + t.v * J.x_view_stride;
  const int64_t col = t.c0 + lane * 8;
  const int64_t nv = J.cols - col;
  const int nvalid = nv >= 8 ? 8 : (nv > 0 ? static_cast<int>(nv) : 0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t wd[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      u[i][2 * k] = __uint_as_float(wd[k] << 16);
      u[i][2 * k + 1] = __uint_as_float(wd[k] & 0xFFFF0000u);
    }
    const int64_t row = t.r0 + warp * 4 + i;
    if (row < J.rows && nvalid > 0 && nvalid < 8) {  // ragged last columns
      const bf16* src = xv + row * J.ldx + col;
#pragma unroll
      for (int k = 0; k < 8; ++k) u[i][k] = k < nvalid ? __bfloat162float(src[k]) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) u[i][k] *= scale;
  }
}

// Tile -> (view, first row, first col) within the job record held in shared
// memory. 32-bit arithmetic: the host rejects tensors with 2^31 or more tiles,
// and a 64-bit division per tile is dozens of instructions in every thread.
__device__ __forceinline__ TileInfo tile_info_in(const EwJob& J, int job, int64_t tile) {
  TileInfo t;
  t.job = job;
  const uint32_t local = static_cast<uint32_t>(tile - J.tile_begin);
  const uint32_t tc = static_cast<uint32_t>(J.tiles_c);
  const uint32_t per_view = static_cast<uint32_t>(J.tiles_r) * tc;
  const uint32_t v = local / per_view;
  const uint32_t w = local - v * per_view;
  const uint32_t tr = w / tc;
  t.v = v;
  t.r0 = static_cast<int64_t>(tr) * kEwTileR;
  t.c0 = static_cast<int64_t>(w - tr * tc) * kEwTileC;
  return t;
}

// This block's contiguous share [begin, end) of `total` tiles: consecutive
// tiles mostly belong to one tensor, so the job record changes rarely.
__device__ __forceinline__ void block_tile_range(int64_t total, int64_t& begin, int64_t& end) {
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  begin = min(total, static_cast<int64_t>(blockIdx.x) * per);
  end = min(total, begin + per);
}

__device__ __forceinline__ void load8(const void* base, int dt, int64_t off, int nvalid, bool vec,
                                      float (&o)[8]) {
  if (vec && nvalid == 8) {
    if (dt == MH_F32) {
      const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
      const float4 a = __ldcs(s), b = __ldcs(s + 1);
      o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
      o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    } else {
      const uint4 t = __ldcs(reinterpret_cast<const uint4*>(static_cast<const bf16*>(base) + off));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&t);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        o[2 * k] = f.x;
        o[2 * k + 1] = f.y;
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k < nvalid)
      o[k] = dt == MH_F32 ? static_cast<const float*>(base)[off + k]
                          : __bfloat162float(static_cast<const bf16*>(base)[off + k]);
    else
      o[k] = 0.0f;
  }
}

__device__ __forceinline__ void store8(void* base, int dt, int64_t off, int nvalid, bool vec,
                                       const float (&x)[8]) {
  if (vec && nvalid == 8) {
    if (dt == MH_F32) {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
      __stcs(d, make_float4(x[0], x[1], x[2], x[3]));
      __stcs(d + 1, make_float4(x[4], x[5], x[6], x[7]));
    } else {
      uint4 t;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&t);
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
      __stcs(reinterpret_cast<uint4*>(static_cast<bf16*>(base) + off), t);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k < nvalid) {
      if (dt == MH_F32)
        static_cast<float*>(base)[off + k] = x[k];
      else
        static_cast<bf16*>(base)[off + k] = __float2bfloat16_rn(x[k]);
    }
  }
}

// Writes 8 (or nvalid) momentum values at flat element `off` of the tensor:
// fp32, or bf16 stochastically rounded (dew "bf16_moments").
__device__ __forceinline__ void store_mom8(const EwJob& J, int64_t off, int nvalid,
                                           const float (&b)[8]) {
  if (J.mom_dtype == MH_BF16)
    store_bf16_sr<8>(static_cast<bf16*>(J.mom) + off, nvalid, J.mom_vec, b, J.mom_key,
                     static_cast<uint64_t>(off));
  else
    store8(J.mom, MH_F32, off, nvalid, J.mom_vec, b);
}

// Raw 16-byte loads of 8 consecutive elements (bf16: one uint4; fp32: two),
// kept packed until they are needed so that many can be in flight per thread.
template <int DT>
struct Raw8 {
  uint4 v[DT == MH_F32 ? 2 : 1];
};

template <int DT>
__device__ __forceinline__ void raw_load8(Raw8<DT>& r, const void* base, int64_t off) {
  const uint4* s = DT == MH_F32
                       ? reinterpret_cast<const uint4*>(static_cast<const float*>(base) + off)
                       : reinterpret_cast<const uint4*>(static_cast<const bf16*>(base) + off);
#pragma unroll
  for (int q = 0; q < (DT == MH_F32 ? 2 : 1); ++q) r.v[q] = __ldcs(s + q);
}

template <int DT>
__device__ __forceinline__ void raw_unpack8(const Raw8<DT>& r, float (&o)[8]) {
  if constexpr (DT == MH_F32) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      o[4 * q + 0] = __uint_as_float(r.v[q].x);
      o[4 * q + 1] = __uint_as_float(r.v[q].y);
      o[4 * q + 2] = __uint_as_float(r.v[q].z);
      o[4 * q + 3] = __uint_as_float(r.v[q].w);
    }
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r.v[0]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      o[2 * k] = f.x;
      o[2 * k + 1] = f.y;
    }
  }
}

// One full interior chunk of the flat prologue (momentum on, 16-byte aligned
// gradient and momentum): every load of the chunk is issued before any is
// consumed, four groups of 8 elements per thread. Returns the thread's share
// of ||Q||^2. e0: first element of this thread's first group in the tensor;
// xd: the matching position in X.
template <int GDT, int MDT>
__device__ __forceinline__ float prologue_chunk_fast(const EwJob& J, const EwParams& p, float gmul,
                                                     int64_t e0, bf16* xd) {
  constexpr int kIt = kProChunk / (8 * kEwThreads);
  constexpr int kStep = 8 * kEwThreads;
  Raw8<GDT> gr[kIt];
  Raw8<MDT> br[kIt];
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    raw_load8<GDT>(gr[it], J.src, e0 + it * kStep);
    raw_load8<MDT>(br[it], J.mom, e0 + it * kStep);
  }
  float ss = 0.0f;
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    float g[8], b[8], q[8];
    raw_unpack8<GDT>(gr[it], g);
    raw_unpack8<MDT>(br[it], b);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      g[k] *= gmul;
      b[k] = p.mu * b[k] + (1.0f - p.mu) * g[k];
      q[k] = p.nesterov ? g[k] + p.mu * (b[k] - g[k]) : b[k];
      ss += q[k] * q[k];
    }
    if constexpr (MDT == MH_BF16)
      store_bf16_sr<8>(static_cast<bf16*>(J.mom) + e0 + it * kStep, 8, true, b, J.mom_key,
                       static_cast<uint64_t>(e0 + it * kStep));
    else
      store8(J.mom, MH_F32, e0 + it * kStep, 8, true, b);
    store8(xd + it * kStep, MH_BF16, 0, 8, true, q);
  }
  return ss;
}

// Prologue of views whose X layout equals their stored layout (cols a
// multiple of 8): a plain contiguous stream, like AdamW. One work item is a
// kProChunk-element chunk of one view; each thread handles 8 consecutive
// elements per step, the block 2048 per step, four steps per chunk. One
// ||Q||_F^2 partial per warp and chunk.
// kB16: every job keeps bf16 momentum. Its chunks move 8 B per element
// instead of 12, so a thread has fewer bytes in flight; the instantiation
// carries only the bf16-momentum fast paths and runs three blocks per SM.
template <bool kB16>
__global__ void __launch_bounds__(kEwThreads, kB16 ? 3 : 2)
    prologue_flat_kernel(const __grid_constant__ EwParams p) {
  __shared__ __align__(16) EwJob sJ;
  if (step_skipped(p.skip)) return;
  const float gmul = p.grad_mult != nullptr ? *p.grad_mult : 1.0f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cur_job = -1;
  for (int64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
    const int jb = find_job(p, tile);
    if (jb != cur_job) {  // block-uniform
      __syncthreads();
      constexpr int kWords = sizeof(EwJob) / 4;
      if (threadIdx.x < kWords)
        reinterpret_cast<uint32_t*>(&sJ)[threadIdx.x] =
            reinterpret_cast<const uint32_t*>(&p.jobs[jb])[threadIdx.x];
      __syncthreads();
      cur_job = jb;
    }
    const EwJob& J = sJ;
    const uint32_t local = static_cast<uint32_t>(tile - J.tile_begin);
    const uint32_t per_view = static_cast<uint32_t>(J.tiles_c);
    const uint32_t v32 = local / per_view;
    const int64_t v = v32;
    const int64_t w = local - v32 * per_view;
    const int64_t view_elem0 = v * J.rows * J.cols;
    const int64_t vsz = J.rows * J.cols;
    const int64_t base = w * kProChunk;
    const bool inactive = J.active != nullptr && J.active[v] == 0;  // block-uniform
    if (J.vrec != nullptr && threadIdx.x == 0 && w == 0) {
      ViewRec rec;
      rec.param = J.dst;
      rec.grad = J.src;
      rec.elem0 = view_elem0;
      rec.rows = J.rows;
      rec.cols = J.cols;
      rec.lr = J.lr;
      rec.wd = J.wd;
      rec.shape_scale = J.shape_scale;
      rec.pdt = J.dst_dtype;
      rec.gdt = J.src_dtype;
      rec.tall = 0;
      rec.vec = (J.dst_vec && J.src_vec && (J.cols % 8) == 0) ? 1 : 0;
      rec.psr = J.param_sr;
      rec.psr_key = J.param_key;
      rec.inactive = inactive ? 1 : 0;
      rec.stat_tiles_c = J.stat_tiles_c;
      rec.rowpart = J.rowpart != nullptr ? J.rowpart + v * J.stat_tiles_c * J.rows : nullptr;
      J.vrec[v] = rec;
    }
    bf16* xv = J.x0 + v * J.x_view_stride;
    float ss = 0.0f;
    if (inactive) {
      // Zero gradient under the inactive-expert rule: momentum untouched,
      // X = 0 (so U = 0), no norm contribution.
      const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int i = 0; i < kProChunk / (8 * kEwThreads); ++i) {
        const int64_t off = base + i * (8 * kEwThreads) + warp * 256 + lane * 8;
        const int64_t rem = vsz - off;
        const int nv = rem >= 8 ? 8 : (rem > 0 ? static_cast<int>(rem) : 0);
        if (nv > 0) store8(xv, MH_BF16, off, nv, true, z);
      }
      if (lane == 0) J.tile_ss[static_cast<int64_t>(local) * (kEwThreads / 32) + warp] = 0.0f;
      continue;
    }
    if (p.use_momentum && J.src_vec && J.mom_vec && base + kProChunk <= vsz) {
      const int64_t e0 = view_elem0 + base + 8 * static_cast<int64_t>(threadIdx.x);
      bf16* xd = xv + base + 8 * static_cast<int64_t>(threadIdx.x);
      if constexpr (kB16) {
        ss = J.src_dtype == MH_BF16 ? prologue_chunk_fast<MH_BF16, MH_BF16>(J, p, gmul, e0, xd)
                                    : prologue_chunk_fast<MH_F32, MH_BF16>(J, p, gmul, e0, xd);
      } else if (J.src_dtype == MH_BF16) {
        ss = J.mom_dtype == MH_BF16 ? prologue_chunk_fast<MH_BF16, MH_BF16>(J, p, gmul, e0, xd)
                                    : prologue_chunk_fast<MH_BF16, MH_F32>(J, p, gmul, e0, xd);
      } else {
        ss = J.mom_dtype == MH_BF16 ? prologue_chunk_fast<MH_F32, MH_BF16>(J, p, gmul, e0, xd)
                                    : prologue_chunk_fast<MH_F32, MH_F32>(J, p, gmul, e0, xd);
      }
      ss = warp_sum(ss);
      if (lane == 0) J.tile_ss[static_cast<int64_t>(local) * (kEwThreads / 32) + warp] = ss;
      continue;
    }
#pragma unroll 1
    for (int i = 0; i < kProChunk / (8 * kEwThreads); ++i) {
      const int64_t off = base + i * (8 * kEwThreads) + warp * 256 + lane * 8;
      const int64_t rem = vsz - off;
      const int nv = rem >= 8 ? 8 : (rem > 0 ? static_cast<int>(rem) : 0);
      if (nv == 0) continue;
      float g[8], q[8];
      load8(J.src, J.src_dtype, view_elem0 + off, nv, J.src_vec, g);
#pragma unroll
      for (int k = 0; k < 8; ++k) g[k] *= gmul;
      if (p.use_momentum) {
        float b[8];
        load8(J.mom, J.mom_dtype, view_elem0 + off, nv, J.mom_vec, b);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          b[k] = p.mu * b[k] + (1.0f - p.mu) * g[k];
          q[k] = p.nesterov ? g[k] + p.mu * (b[k] - g[k]) : b[k];
        }
        store_mom8(J, view_elem0 + off, nv, b);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = g[k];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) ss += q[k] * q[k];  // q[k] == 0 beyond nv
      store8(xv, MH_BF16, off, nv, true, q);
    }
    ss = warp_sum(ss);
    if (lane == 0) J.tile_ss[static_cast<int64_t>(local) * (kEwThreads / 32) + warp] = ss;
  }
}

// Momentum, Nesterov lerp, ||Q||_F^2 partials and bf16(Q) for views whose X
// row pitch differs from their cols (cols not a multiple of 8), over 32 x 256
// tiles (each thread: 4 rows x 8 columns, all loads issued before any
// store). Tile indices use 32-bit arithmetic (the host rejects tensors with
// 2^31 or more tiles).
__global__ void __launch_bounds__(kEwThreads) prologue_kernel(const __grid_constant__ EwParams p) {
  __shared__ __align__(16) EwJob sJ;
  if (step_skipped(p.skip)) return;
  const float gmul = p.grad_mult != nullptr ? *p.grad_mult : 1.0f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cur_job = -1;

  for (int64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
    const int jb = find_job(p, tile);
    if (jb != cur_job) {  // block-uniform
      __syncthreads();
      constexpr int kWords = sizeof(EwJob) / 4;
      if (threadIdx.x < kWords)
        reinterpret_cast<uint32_t*>(&sJ)[threadIdx.x] =
            reinterpret_cast<const uint32_t*>(&p.jobs[jb])[threadIdx.x];
      __syncthreads();
      cur_job = jb;
    }
    const EwJob& J = sJ;
    const uint32_t local = static_cast<uint32_t>(tile - J.tile_begin);
    const uint32_t tc_n = static_cast<uint32_t>(J.tiles_c);
    const uint32_t per_view = static_cast<uint32_t>(J.tiles_r) * tc_n;
    const uint32_t v32 = local / per_view;
    const uint32_t w = local - v32 * per_view;
    const int64_t v = v32;
    const int64_t view_elem0 = v * J.rows * J.cols;

    const uint32_t trow = w / tc_n;
    const int64_t r0 = static_cast<int64_t>(trow) * kEwTileR;
    const int64_t c0 = static_cast<int64_t>(w - trow * tc_n) * kProTileC;
    const int64_t col = c0 + lane * 8;
    const int64_t ncol = J.cols - col;
    const int nvalid = ncol >= 8 ? 8 : (ncol > 0 ? static_cast<int>(ncol) : 0);

    const bool inactive = J.active != nullptr && J.active[v] == 0;  // block-uniform
    if (J.vrec != nullptr && threadIdx.x == 0 && r0 == 0 && c0 == 0) {
      ViewRec rec;
      rec.param = J.dst;
      rec.grad = J.src;
      rec.elem0 = view_elem0;
      rec.rows = J.rows;
      rec.cols = J.cols;
      rec.lr = J.lr;
      rec.wd = J.wd;
      rec.shape_scale = J.shape_scale;
      rec.pdt = J.dst_dtype;
      rec.gdt = J.src_dtype;
      rec.tall = 0;
      rec.vec = (J.dst_vec && J.src_vec && (J.cols % 8) == 0) ? 1 : 0;
      rec.psr = J.param_sr;
      rec.psr_key = J.param_key;
      rec.inactive = inactive ? 1 : 0;
      rec.stat_tiles_c = J.stat_tiles_c;
      rec.rowpart = J.rowpart != nullptr ? J.rowpart + v * J.stat_tiles_c * J.rows : nullptr;
      J.vrec[v] = rec;
    }

    bf16* xv = J.x0 + v * J.x_view_stride;
    float g[4][8], b[4][8];
    bool ok[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + warp * 4 + i;
      ok[i] = row < J.rows && nvalid > 0;
      if (inactive) {
        // Zero gradient under the inactive-expert rule: X = 0, state untouched.
        if (ok[i]) {
          const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          store8(xv + row * J.ldx, MH_BF16, col, nvalid, true, z);
        }
        ok[i] = false;
        continue;
      }
      if (ok[i]) {
        const int64_t off = view_elem0 + row * J.cols + col;
        load8(J.src, J.src_dtype, off, nvalid, J.src_vec, g[i]);
#pragma unroll
        for (int k = 0; k < 8; ++k) g[i][k] *= gmul;
        if (p.use_momentum) load8(J.mom, J.mom_dtype, off, nvalid, J.mom_vec, b[i]);
      }
    }
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!ok[i]) continue;
      const int lr = warp * 4 + i;
      const int64_t row = r0 + lr;
      const int64_t off = view_elem0 + row * J.cols + col;
      float q[8];
      if (p.use_momentum) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          b[i][k] = p.mu * b[i][k] + (1.0f - p.mu) * g[i][k];
          q[k] = p.nesterov ? g[i][k] + p.mu * (b[i][k] - g[i][k]) : b[i][k];
        }
        store_mom8(J, off, nvalid, b[i]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = g[i][k];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) ss += q[k] * q[k];  // q[k] == 0 beyond nvalid
      store8(xv + row * J.ldx, MH_BF16, col, nvalid, true, q);
    }
    // ||Q||_F^2 of this warp's 4 x 256 block: one partial per warp, summed in
    // a fixed order by the view-norm kernel, so wide tiles need no block-wide
    // barrier.
    ss = warp_sum(ss);
    if (lane == 0) J.tile_ss[static_cast<int64_t>(local) * (kEwThreads / 32) + warp] = ss;
  }
}

template <int KIND>
__global__ void __launch_bounds__(kEwThreads, 2) ew_kernel(const __grid_constant__ EwParams p) {
  __shared__ float sRed[kEwThreads / 32][kEwTileC];
  // The tile's job record, copied once per tile from the parameter space:
  // indexing a large parameter table per access would keep missing the small
  // constant cache.
  __shared__ __align__(16) EwJob sJ;
  if (step_skipped(p.skip)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cur_job = -1;
  int64_t job_end = 0;
  int64_t tile_begin, tile_end;
  block_tile_range(p.total_tiles, tile_begin, tile_end);

  for (int64_t tile = tile_begin; tile < tile_end; ++tile) {
    if (cur_job < 0 || tile >= job_end) {  // block-uniform
      const int jb = find_job(p, tile);
      __syncthreads();
      constexpr int kWords = sizeof(EwJob) / 4;
      static_assert(sizeof(EwJob) % 4 == 0, "EwJob must be a whole number of words");
      if (threadIdx.x < kWords)
        reinterpret_cast<uint32_t*>(&sJ)[threadIdx.x] =
            reinterpret_cast<const uint32_t*>(&p.jobs[jb])[threadIdx.x];
      __syncthreads();
      cur_job = jb;
      job_end = sJ.tile_begin + sJ.views * sJ.tiles_r * sJ.tiles_c;
    }
    const EwJob& J = sJ;
    const TileInfo t = tile_info_in(J, cur_job, tile);
    const int64_t view_elem0 = t.v * J.rows * J.cols;
    const int64_t col = t.c0 + lane * 8;
    const int64_t ncol = J.cols - col;
    const int nvalid = ncol >= 8 ? 8 : (ncol > 0 ? static_cast<int>(ncol) : 0);

    // The U block's loads are issued here; the apply issues its parameter
    // loads before unpacking them, so both are in flight together.
    uint4 uraw[4];
    load_u_raw(J, t, uraw);
    float u[4][8];
    // Without Newton-Schulz steps U is the normalised momentum: the buffer
    // holds bf16(Q) and every pass scales it by 1/(||Q|| norm_scale + eps).
    const float uscale = p.u_scale_from_sumsq
                             ? ns_inv_norm(J.sumsq[t.v], p.ns_norm_scale, p.ns_eps)
                             : 1.0f;
    if constexpr (KIND != EW_APPLY) unpack_u_block(J, t, uraw, u, uscale);

    if constexpr (KIND == EW_ROWSQ) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) s += u[i][k] * u[i][k];
        s = warp_sum(s);
        const int64_t row = t.r0 + warp * 4 + i;
        if (lane == 0 && row < J.rows)
          J.rowpart[(t.v * J.tiles_c + t.c0 / kEwTileC) * J.rows + row] = s;
      }
    } else if constexpr (KIND == EW_COLSQ) {
      float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = t.r0 + warp * 4 + i;
        const float f = row < J.rows ? J.rowfac[t.v * J.rows + row] : 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float x = f * u[i][k];
          cs[k] += x * x;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) sRed[warp][lane * 8 + k] = cs[k];
      __syncthreads();
      {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kEwThreads / 32; ++w) s += sRed[w][threadIdx.x];
        const int64_t c = t.c0 + threadIdx.x;
        if (c < J.cols) J.colpart[(t.v * J.tiles_r + t.r0 / kEwTileR) * J.cols + c] = s;
      }
      __syncthreads();
    } else {
      // EW_APPLY / EW_COPYOUT: final update direction U_ij.
      // 16-byte access needs 8-element rows for bf16 and 4-element rows for fp32.
      const bool dvec = J.dst_vec && (J.dst_dtype == MH_F32 || (J.cols % 8) == 0);
      const bool svec = J.src_vec && (J.src_dtype == MH_F32 || (J.cols % 8) == 0);
      const bool active = J.active == nullptr || J.active[t.v] != 0;
      float w[4][8];
      float fr[4];
      // Every load of the block (U, parameters, row and column factors) is in
      // flight before any is used: the stores below may alias the parameter
      // loads, so nothing may be loaded between stores. A vector bf16
      // parameter is loaded raw and unpacked after U.
      // (The cautious-update instantiation also holds the gradient block and
      // has no registers to spare for the raw parameter block.)
      const bool wraw = KIND == EW_APPLY && dvec && J.dst_dtype == MH_BF16 && nvalid == 8 &&
                        active;
      uint4 wr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = t.r0 + warp * 4 + i;
        fr[i] = p.use_rowfac && row < J.rows ? J.rowfac[t.v * J.rows + row] : 1.0f;
        wr[i] = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (KIND == EW_APPLY || KIND == EW_APPLY_CU) {
          if (row < J.rows && nvalid > 0 && active) {
            const int64_t off = view_elem0 + row * J.cols + col;
            if (wraw)
              wr[i] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const bf16*>(J.dst) + off));
            else
              load8(J.dst, J.dst_dtype, off, nvalid, dvec, w[i]);
          }
        }
      }
      float h[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
      if (p.use_colfac) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < nvalid) h[k] = J.colfac[t.v * J.cols + col + k];
      }
      if constexpr (KIND == EW_APPLY) {
        unpack_u_block(J, t, uraw, u, uscale);
        if (wraw) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t wd[4] = {wr[i].x, wr[i].y, wr[i].z, wr[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              w[i][2 * k] = __uint_as_float(wd[k] << 16);
              w[i][2 * k + 1] = __uint_as_float(wd[k] & 0xFFFF0000u);
            }
          }
        }
      }
      // The cautious-update mask needs the gradient: a separate instantiation
      // keeps its 32 registers out of the common path.
      float gr[KIND == EW_APPLY_CU ? 4 : 1][8];
      if constexpr (KIND == EW_APPLY_CU) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t row = t.r0 + warp * 4 + i;
          if (row < J.rows && nvalid > 0 && active)
            load8(J.src, J.src_dtype, view_elem0 + row * J.cols + col, nvalid, svec, gr[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = t.r0 + warp * 4 + i;
        if (row >= J.rows || nvalid == 0) continue;
        const float f = fr[i];
        float uu[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) uu[k] = u[i][k] * f * h[k];
        const int64_t off = view_elem0 + row * J.cols + col;
        if constexpr (KIND == EW_COPYOUT) {
          const bool ovec = J.dst_vec && (J.dst_dtype == MH_F32 || (J.cols % 8) == 0);
          store8(J.dst, J.dst_dtype, off, nvalid, ovec, uu);
        } else if (active) {
          const float lr = J.lr, wd = J.wd, s = J.shape_scale;
          float* wi = w[i];
          if constexpr (KIND == EW_APPLY_CU) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float delta = lr * wd * wi[k] + (lr * s) * uu[k];
              if (delta * gr[i][k] > 0.0f) wi[k] = wi[k] - delta;
            }
          } else if (p.cautious == MH_CAUTIOUS_WD) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float g = s * uu[k];
              const float mask = (g * wi[k] >= 0.0f) ? 1.0f : 0.0f;
              wi[k] = wi[k] - lr * (g + wd * wi[k] * mask);
            }
          } else {
            const float decay = 1.0f - lr * wd;
#pragma unroll
            for (int k = 0; k < 8; ++k) wi[k] = decay * wi[k] - (lr * s) * uu[k];
          }
          if (J.param_sr && J.dst_dtype == MH_BF16)
            store_bf16_sr<8>(static_cast<bf16*>(J.dst) + off, nvalid, dvec, w[i], J.param_key,
                             static_cast<uint64_t>(off));
          else
            store8(J.dst, J.dst_dtype, off, nvalid, dvec, w[i]);
        }
      }
    }
  }
}

// ---- streaming passes -------------------------------------------------------
// The NorMuon / Muon+ apply (plain, cautious weight decay, or cautious update,
// which also reads the gradient) and the Muon+ column statistics read every
// element once and (apply) write the parameter once, so they are bound by
// HBM. Each block (one
// per SM) runs one producer warp and sixteen consumer warps over its range of
// 32 x 256 tiles through a ring of shared-memory stages:
//   producer  waits for a free stage, writes the stage's descriptor (and, at a
//             tensor boundary, the job record), then issues one TMA box of U
//             (from the Newton-Schulz buffer), one of the parameter and, for
//             the cautious update, one of the gradient, each 32 x 256 with
//             zero fill past the tensor's edges, and cp.async
//             copies of the tile's row and column factors. The stage's full
//             barrier completes when all have landed: 32 plain arrivals (each
//             lane's own writes), 32 cp.async arrivals and the boxes' bytes.
//             The job's fields and the tile coordinates stay in registers
//             (stepped tile by tile), so a tile costs the producer a few
//             instructions. (One box per operand: 32 row-sized bulk copies
//             per tile cost the copy engine about as much time per tile as
//             the HBM does.)
//   consumers groups of warps take turns with the tiles (apply: two groups of
//             eight warps, 4 rows each; statistics: four groups of four warps,
//             8 rows each). A group waits for the full barrier, computes the
//             tile from shared memory (each lane 8 columns: a warp reads 512
//             consecutive bytes per row, so no bank conflicts), stores the
//             parameter (apply) and releases the stage (one arrival per
//             warp). The
//             statistics write each warp's column partials to one of the
//             group's four reduction buffers and arrive on its mbarrier; the
//             cross-warp sum of the group's previous tile is taken after this
//             tile's partials are written, so a warp seldom waits for the
//             others. Several tiles in the consumers at once share out each
//             tile's fixed chain of waits and shared-memory round trips.
// Nothing a consumer waits for is a dependent global load. The apply's step
// scalars ride on the column factors (decrement lr s U f h, decay 1 - lr wd in
// one fma), which keeps its instruction count per element near ten: with the
// sixteen warps it is otherwise bound by instruction issue, not by HBM.
// Every wait is bounded by the launch's wait limit; on a
// timeout the block records DEV_TIMEOUT_STREAM in the status word, lets every
// copy it issued land and returns. A parameter whose rows are not whole
// aligned 16-byte groups (bf16 with cols % 8 != 0, unaligned storage, an fp32
// parameter in the bf16 layout) is read directly when the tile is processed,
// as ew_kernel does.

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, bool valid) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(sa), "l"(gmem),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Sixteen consumer warps and the producer warp: four warps per scheduler keep
// the per-element latency of the apply hidden. The apply splits them into two
// groups of eight (4 rows of a 32-row tile each); the column statistics, with
// little work per element and a fixed chain per tile, into four groups of
// four (8 rows each).
constexpr int kStreamConsumerWarps = 16;
constexpr int kStreamThreads = (kStreamConsumerWarps + 1) * 32;
template <int KIND>
struct StreamGroups {
  static constexpr int kGroups = KIND == EW_COLSQ ? 4 : 2;
  static constexpr int kWarps = kStreamConsumerWarps / kGroups;  // per group
  static constexpr int kRows = kEwTileR / kWarps;                // per warp
  static_assert(kRows % 4 == 0, "row factors are read four at a time");
};

// Stage layout of ew_stream_kernel<KIND, WB> (bytes from the stage's start).
// WB: parameter bytes per 8 elements (16: bf16, 32: fp32, 0: no parameter).
template <int KIND, int WB>
struct StreamLayout {
  static constexpr bool kApply = KIND == EW_APPLY || KIND == EW_APPLY_CU;
  static constexpr bool kGrad = KIND == EW_APPLY_CU;    // bf16 gradient box
  static constexpr int kURow = kEwTileC * 2;            // 512 B of bf16 U per row
  static constexpr int kWRow = kEwTileC / 8 * WB;       // parameter bytes per row
  static constexpr int kU = 0;
  static constexpr int kW = kU + kEwTileR * kURow;
  static constexpr int kG = kW + kEwTileR * kWRow;      // gradient (cautious update)
  static constexpr int kC = kG + (kGrad ? kEwTileR * kURow : 0);  // column factors (apply)
  static constexpr int kR = kC + (kApply ? kEwTileC * 4 : 0);  // row factors
  static constexpr int kD = kR + kEwTileR * 4;          // descriptor: 4 x int32
  static constexpr int kStage = (kD + 16 + 127) / 128 * 128;
  // Column statistics: per consumer group four [warp][256] float reduction
  // buffers after the stages (sixteen warps' rows in all).
  static constexpr int kRedBufs = kApply ? 0 : 4;
  static constexpr int kRedBytes = kRedBufs * kStreamConsumerWarps * kEwTileC * 4;
  static constexpr int kBudget = 204800 - kRedBytes;
  static constexpr int kStages = kBudget / kStage > 8 ? 8 : kBudget / kStage;
  static constexpr size_t kRed = static_cast<size_t>(kStages) * kStage;
  static constexpr size_t kSmem = kRed + kRedBytes;
  static_assert(kStages >= 3, "stage layout too large");
};

template <int KIND, int WB>
__host__ __device__ constexpr size_t stream_smem_bytes() {
  return StreamLayout<KIND, WB>::kSmem + 128;  // + alignment slack
}

// Whether the parameter of a job is loaded as TMA boxes: 16-byte aligned
// storage whose rows are whole 16-byte groups, of a dtype the layout holds.
template <int WB>
__device__ __forceinline__ bool stream_w_staged(const EwJob& J) {
  const bool vec = J.dst_vec && (J.dst_dtype == MH_F32 || (J.cols % 8) == 0);
  return vec && (J.dst_dtype == MH_BF16 ? WB >= 16 : WB >= 32);
}

// Whether the gradient of a job is loaded as TMA boxes (cautious update): a
// bf16 gradient in 16-byte aligned storage whose rows are whole 16-byte
// groups. Others are read directly when the tile is processed.
__device__ __host__ __forceinline__ bool stream_g_staged(const EwJob& J) {
  return J.src_vec && J.src_dtype == MH_BF16 && (J.cols % 8) == 0;
}

__device__ __forceinline__ int64_t job_end_tile(const EwJob& J) {
  return J.tile_begin + J.views * J.tiles_r * J.tiles_c;
}

// Launch parameters of the streaming passes: the elementwise parameters and,
// per job, tensor maps of its U view stack and of its parameter (the latter
// encoded only where stream_w_staged holds). A cautious-update launch carries
// at most kStreamCuJobs jobs and keeps job j's gradient map (where
// stream_g_staged holds) in tmU[kStreamCuJobs + j]: three maps per job for 64
// jobs would exceed the kernel parameter space.
constexpr int kStreamCuJobs = kMaxJobs / 2;
struct StreamParams {
  CUtensorMap tmU[kMaxJobs];
  CUtensorMap tmW[kMaxJobs];
  EwParams ew;
};

template <int KIND, int WB>
__global__ void __launch_bounds__(kStreamThreads, 1)
    ew_stream_kernel(const __grid_constant__ StreamParams sp) {
  using L = StreamLayout<KIND, WB>;
  using G = StreamGroups<KIND>;
  constexpr int kS = L::kStages;
  const EwParams& p = sp.ew;
  extern __shared__ uint8_t stream_smem_raw[];
  // TMA destinations: 128-byte aligned stage bases (the launch adds the slack).
  uint8_t* stream_smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(stream_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  __shared__ __align__(16) EwJob sJ[kS];
  __shared__ __align__(8) uint64_t full[kS], empty[kS], red_bar[G::kGroups][4];
  __shared__ int abort_flag;
  if (step_skipped(p.skip)) return;
  int64_t tile_begin, tile_end;
  block_tile_range(p.total_tiles, tile_begin, tile_end);
  const int64_t ntiles = tile_end - tile_begin;
  if (ntiles <= 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(&full[s], 64);
      mbar_init(&empty[s], G::kWarps);
    }
    for (int g = 0; g < G::kGroups; ++g)
      for (int b = 0; b < 4; ++b) mbar_init(&red_bar[g][b], G::kWarps);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_v = &abort_flag;

  if (warp == kStreamConsumerWarps) {
    // ---- producer warp ----
    constexpr int kWords = sizeof(EwJob) / 4;
    static_assert(sizeof(EwJob) % 4 == 0, "EwJob must be a whole number of words");
    int pj = -1, pseq = -1, slot = 0;
    int64_t pend = tile_begin;  // forces a job record for the first tile
    // The job's fields and the tile's coordinates live in registers: they are
    // reloaded at a tensor boundary and stepped tile by tile, so a tile costs
    // no shared-memory round trips and no divisions.
    int64_t rows = 0, cols = 0;
    int32_t tiles_r = 0, tiles_c = 0;
    const float* rowfac = nullptr;
    const float* colfac = nullptr;
    const int32_t* active = nullptr;
    uint32_t wbytes = 0, gbytes = 0;
    int32_t v = 0, tr = 0, tc = 0;
    bool new_view = true;
    const float* rf_view = nullptr;
    const float* cf_view = nullptr;
    bool act = true;
    int64_t issued = 0;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t i = 0; i < ntiles; ++i) {
      if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_v, p.status, DEV_TIMEOUT_STREAM,
                             p.wait_limit))
        break;
      const int64_t tile = tile_begin + i;
      if (tile >= pend) {  // warp-uniform: the next tensor takes the oldest job slot
        pj = find_job(p, tile);
        ++pseq;
        slot = pseq % kS;
        for (int w = lane; w < kWords; w += 32)
          reinterpret_cast<uint32_t*>(&sJ[slot])[w] =
              reinterpret_cast<const uint32_t*>(&p.jobs[pj])[w];
        __syncwarp();
        const EwJob& J = sJ[slot];
        pend = job_end_tile(J);
        rows = J.rows;
        cols = J.cols;
        tiles_r = J.tiles_r;
        tiles_c = J.tiles_c;
        rowfac = J.rowfac;
        colfac = J.colfac;
        active = J.active;
        // A box always completes its full size in bytes, zero-filled or not.
        wbytes = (WB > 0 && stream_w_staged<WB>(J))
                     ? kEwTileR * kEwTileC * (J.dst_dtype == MH_F32 ? 4u : 2u)
                     : 0u;
        gbytes = (L::kGrad && stream_g_staged(J)) ? kEwTileR * L::kURow : 0u;
        const TileInfo t = tile_info_in(J, pj, tile);
        v = static_cast<int32_t>(t.v);
        tr = static_cast<int32_t>(t.r0 / kEwTileR);
        tc = static_cast<int32_t>(t.c0 / kEwTileC);
        new_view = true;
      }
      if (new_view) {
        if (KIND == EW_COLSQ || p.use_rowfac) rf_view = rowfac + v * rows;
        if (L::kApply && p.use_colfac) cf_view = colfac + v * cols;
        // The active flag: one dependent load per view.
        if constexpr (L::kApply) act = active == nullptr || active[v] != 0;
        new_view = false;
      }
      const int32_t r0 = tr * kEwTileR, c0 = tc * kEwTileC;
      uint8_t* st = stream_smem + static_cast<size_t>(stage) * L::kStage;
      if (lane == 0) {
        *reinterpret_cast<int4*>(st + L::kD) = make_int4(slot, v, r0, c0 | (act ? 0 : (1 << 30)));
        if (act) {
          mbar_expect_tx(&full[stage], kEwTileR * L::kURow + wbytes + gbytes);
          tma_load_3d(st + L::kU, &sp.tmU[pj], &full[stage], c0, r0, v);
          if (wbytes) tma_load_3d(st + L::kW, &sp.tmW[pj], &full[stage], c0, r0, v);
          if (gbytes) tma_load_3d(st + L::kG, &sp.tmU[kStreamCuJobs + pj], &full[stage], c0, r0, v);
        }
      }
      if (act) {
        if (KIND == EW_COLSQ || p.use_rowfac) {
          const bool row_ok = r0 + lane < rows;
          cp_async4(st + L::kR + lane * 4, row_ok ? rf_view + r0 + lane : rowfac, row_ok);
        }
        if constexpr (L::kApply) {
          if (p.use_colfac) {
            const int64_t col = c0 + lane * 8;
            const float* cf = cf_view + col;
            uint8_t* d = st + L::kC + lane * 32;
            if (cols - col >= 8 && (reinterpret_cast<uintptr_t>(cf) & 15) == 0) {
              cp_async16(d, cf, true);
              cp_async16(d + 16, cf + 4, true);
            } else {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const bool ok = cols - col > q;
                cp_async4(d + 4 * q, ok ? cf + q : colfac, ok);
              }
            }
          }
        }
      }
      cp_async_mbar_arrive(&full[stage]);
      mbar_arrive(&full[stage]);
      ++issued;
      if (++stage == kS) { stage = 0; phase ^= 1u; }
      if (++tc == tiles_c) {
        tc = 0;
        if (++tr == tiles_r) {
          tr = 0;
          ++v;
          new_view = true;
        }
      }
    }
    // Let every copy this warp issued land before the block can leave: the
    // consumers normally wait for all of them; after an abort nobody does.
    cp_async_wait_all();
    for (int64_t j = issued > kS ? issued - kS : 0; j < issued; ++j)
      mbar_wait_drain(&full[j % kS], static_cast<uint32_t>((j / kS) & 1));
    return;
  }

  // ---- consumer warps ----
  // Group g takes tiles g, g + kGroups, ...; its k-th tile is g + k kGroups.
  constexpr int kR = G::kRows;
  const int grp = warp / G::kWarps, gw = warp % G::kWarps;
  const int gtid = threadIdx.x - grp * G::kWarps * 32;  // thread within the group
  float (*const red_base)[kEwTileC] =
      reinterpret_cast<float (*)[kEwTileC]>(stream_smem + L::kRed) + grp * 4 * G::kWarps;
  // Column statistics: the group's previous tile's output (colpart row
  // segment, valid cols), kept in registers: its job slot may be reused once
  // the stage is released.
  float* prev_out = nullptr;
  int64_t prev_ncol = 0;
  // Cross-warp sum of the group's k-th tile: each column summed over the
  // group's warps' partials in a fixed order.
  auto finish = [&](int64_t k, float* out, int64_t ncol) -> bool {
    if (!mbar_wait_bounded(&red_bar[grp][k & 3], static_cast<uint32_t>((k >> 2) & 1), abort_v,
                           p.status, DEV_TIMEOUT_STREAM, p.wait_limit))
      return false;
    const float (*red)[kEwTileC] = red_base + (k & 3) * G::kWarps;
#pragma unroll
    for (int c = gtid; c < kEwTileC; c += G::kWarps * 32) {
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < G::kWarps; ++w) sum += red[w][c];
      if (c < ncol) out[c] = sum;
    }
    return true;
  };
  int64_t k = 0;
  for (int64_t i = grp; i < ntiles; i += G::kGroups, ++k) {
    const int stage = static_cast<int>(i % kS);
    const uint32_t phase = static_cast<uint32_t>((i / kS) & 1);
    float* cur_out = nullptr;
    int64_t cur_ncol = 0;
    if (!mbar_wait_bounded(&full[stage], phase, abort_v, p.status, DEV_TIMEOUT_STREAM,
                           p.wait_limit))
      return;  // aborted: nothing further is written
    const uint8_t* st = stream_smem + static_cast<size_t>(stage) * L::kStage;
    const int4 d = *reinterpret_cast<const int4*>(st + L::kD);
    const EwJob& J = sJ[d.x];
    TileInfo t;
    t.job = 0;
    t.v = d.y;
    t.r0 = d.z;
    t.c0 = d.w & ((1 << 30) - 1);
    const bool act = (d.w >> 30) == 0;
    if (act) {
      const int64_t col = t.c0 + lane * 8;
      const int64_t ncol = J.cols - col;
      const int nvalid = ncol >= 8 ? 8 : (ncol > 0 ? static_cast<int>(ncol) : 0);
      // U's scale (1 unless U is the normalised momentum itself) is folded
      // into the per-row factor.
      const float uscale = p.u_scale_from_sumsq
                               ? ns_inv_norm(J.sumsq[t.v], p.ns_norm_scale, p.ns_eps)
                               : 1.0f;
      const int64_t row0 = t.r0 + gw * kR;
      float u[kR][8];
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        const uint4 raw =
            *reinterpret_cast<const uint4*>(st + L::kU + (gw * kR + r) * L::kURow + lane * 16);
        const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          u[r][2 * q] = __uint_as_float(wd[q] << 16);
          u[r][2 * q + 1] = __uint_as_float(wd[q] & 0xFFFF0000u);
        }
      }
      // Columns past the last and rows past the last are zero in the box;
      // they are still selected away in the rare ragged tile.
      if (nvalid < 8 || row0 + kR - 1 >= J.rows) {
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const bool row_ok = row0 + r < J.rows;
#pragma unroll
          for (int q = 0; q < 8; ++q) u[r][q] = (row_ok && q < nvalid) ? u[r][q] : 0.0f;
        }
      }
      float fr[kR];
#pragma unroll
      for (int r = 0; r < kR; ++r) fr[r] = 1.0f;
      if (KIND == EW_COLSQ || p.use_rowfac) {
#pragma unroll
        for (int r = 0; r < kR; r += 4) {
          const float4 f4 = *reinterpret_cast<const float4*>(st + L::kR + (gw * kR + r) * 4);
          fr[r] = f4.x; fr[r + 1] = f4.y; fr[r + 2] = f4.z; fr[r + 3] = f4.w;
        }
      }
      if constexpr (KIND == EW_COLSQ) {
        float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const float f = fr[r] * uscale;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float x = f * u[r][q];
            cs[q] += x * x;
          }
        }
        float (*red)[kEwTileC] = red_base + (k & 3) * G::kWarps;
        *reinterpret_cast<float4*>(&red[gw][lane * 8]) = make_float4(cs[0], cs[1], cs[2], cs[3]);
        *reinterpret_cast<float4*>(&red[gw][lane * 8 + 4]) = make_float4(cs[4], cs[5], cs[6], cs[7]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_bar[grp][k & 3]);
        cur_out = J.colpart + (t.v * J.tiles_r + t.r0 / kEwTileR) * J.cols + t.c0;
        cur_ncol = J.cols - t.c0;
      } else {
        const bool dvec = J.dst_vec && (J.dst_dtype == MH_F32 || (J.cols % 8) == 0);
        const bool wst = stream_w_staged<WB>(J);
        const int wrow = kEwTileC * (J.dst_dtype == MH_F32 ? 4 : 2);  // box row pitch
        // The step's scalars ride on the column factors: ga = lr s U_ij f_i h_j
        // is the decrement, keep = 1 - lr wd the decay.
        const float lrs = J.lr * J.shape_scale * uscale;
        const float keep = 1.0f - J.lr * J.wd;
        float hs[8];
        if (p.use_colfac) {
          const float4 a = *reinterpret_cast<const float4*>(st + L::kC + lane * 32);
          const float4 b = *reinterpret_cast<const float4*>(st + L::kC + lane * 32 + 16);
          hs[0] = a.x * lrs; hs[1] = a.y * lrs; hs[2] = a.z * lrs; hs[3] = a.w * lrs;
          hs[4] = b.x * lrs; hs[5] = b.y * lrs; hs[6] = b.z * lrs; hs[7] = b.w * lrs;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) hs[q] = lrs;
        }
        const bool cautious_wd = p.cautious == MH_CAUTIOUS_WD;
        const bool gst = L::kGrad && stream_g_staged(J);
        const bool svec = J.src_vec && (J.src_dtype == MH_F32 || (J.cols % 8) == 0);
        const float lrwd = J.lr * J.wd;
        const int64_t view_elem0 = t.v * J.rows * J.cols;
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const int64_t row = row0 + r;
          if (row >= J.rows || nvalid == 0) continue;
          const int64_t off = view_elem0 + row * J.cols + col;
          float w[8];
          if (wst) {
            const uint8_t* ws = st + L::kW + (gw * kR + r) * wrow;
            if (J.dst_dtype == MH_BF16) {
              const uint4 wr = *reinterpret_cast<const uint4*>(ws + lane * 16);
              const uint32_t wd4[4] = {wr.x, wr.y, wr.z, wr.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                w[2 * q] = __uint_as_float(wd4[q] << 16);
                w[2 * q + 1] = __uint_as_float(wd4[q] & 0xFFFF0000u);
              }
            } else {
              const float4 a = *reinterpret_cast<const float4*>(ws + lane * 32);
              const float4 b = *reinterpret_cast<const float4*>(ws + lane * 32 + 16);
              w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
              w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
            }
          } else {
            load8(J.dst, J.dst_dtype, off, nvalid, dvec, w);
          }
          const float f = fr[r];
          if constexpr (L::kGrad) {
            // Cautious update: the whole step delta = lr wd W + lr s U f h
            // applies only where it agrees in sign with the gradient.
            float g[8];
            if (gst) {
              const uint4 gr = *reinterpret_cast<const uint4*>(
                  st + L::kG + (gw * kR + r) * L::kURow + lane * 16);
              const uint32_t g4[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                g[2 * q] = __uint_as_float(g4[q] << 16);
                g[2 * q + 1] = __uint_as_float(g4[q] & 0xFFFF0000u);
              }
            } else {
              load8(J.src, J.src_dtype, off, nvalid, svec, g);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float delta = fmaf(lrwd, w[q], u[r][q] * f * hs[q]);
              if (delta * g[q] > 0.0f) w[q] = w[q] - delta;
            }
          } else if (cautious_wd) {
            // Weight decay only where the update and the weight agree in sign
            // (lr s f h >= 0, so ga has the sign of the update direction).
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float ga = u[r][q] * f * hs[q];
              w[q] = fmaf(w[q], ga * w[q] >= 0.0f ? keep : 1.0f, -ga);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) w[q] = fmaf(w[q], keep, -(u[r][q] * f * hs[q]));
          }
          if (J.param_sr && J.dst_dtype == MH_BF16)
            store_bf16_sr<8>(static_cast<bf16*>(J.dst) + off, nvalid, dvec, w, J.param_key,
                             static_cast<uint64_t>(off));
          else
            store8(J.dst, J.dst_dtype, off, nvalid, dvec, w);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if constexpr (KIND == EW_COLSQ) {
      // Buffer (k - 1) & 3 is rewritten by the group's tile k + 3 only after
      // every warp of the group has arrived for tile k + 1, which each does
      // after this sum.
      if (k > 0 && !finish(k - 1, prev_out, prev_ncol)) return;
      prev_out = cur_out;
      prev_ncol = cur_ncol;
    }
  }
  if constexpr (KIND == EW_COLSQ) {
    if (k > 0) finish(k - 1, prev_out, prev_ncol);
  }
}

// Inactive-expert rule: marks each view of a flagged tensor that has a
// nonzero gradient entry. Chunks of views already marked are skipped, so an
// active view usually costs one chunk; a silent view is read once in full.
__global__ void __launch_bounds__(256) view_active_kernel(const __grid_constant__ ActiveParams p) {
  for (int64_t c = blockIdx.x; c < p.total_chunks; c += gridDim.x) {
    int lo = 0, hi = p.njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.jobs[mid].chunk_begin <= c) lo = mid; else hi = mid - 1;
    }
    const ActiveJob& J = p.jobs[lo];
    const int64_t chunks_per_view = (J.view_elems + kActiveChunk - 1) / kActiveChunk;
    const int64_t local = c - J.chunk_begin;
    const int64_t v = local / chunks_per_view;
    if (*reinterpret_cast<volatile const int32_t*>(J.active + v) != 0) continue;  // block-uniform
    const int64_t start = v * J.view_elems + (local - v * chunks_per_view) * kActiveChunk;
    const int64_t end = min(start + kActiveChunk, (v + 1) * J.view_elems);
    bool nz = false;
    for (int64_t i = start + 8 * static_cast<int64_t>(threadIdx.x); i < end; i += 8 * 256) {
      float g[8];
      const int64_t rem = end - i;
      load8(J.grad, J.gdt, i, rem >= 8 ? 8 : static_cast<int>(rem), J.vec != 0, g);
#pragma unroll
      for (int k = 0; k < 8; ++k) nz |= g[k] != 0.0f;  // NaN counts as nonzero
    }
    if (__syncthreads_or(nz ? 1 : 0) && threadIdx.x == 0) J.active[v] = 1;
  }
}

__global__ void __launch_bounds__(256) row_finalize_kernel(const __grid_constant__ RowFinParams p) {
  __shared__ double red[2][8];
  __shared__ float s_kappa;
  if (step_skipped(p.skip)) return;
  for (int64_t vv = blockIdx.x; vv < p.total_views; vv += gridDim.x) {
    int lo = 0, hi = p.njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.jobs[mid].view_begin <= vv) lo = mid; else hi = mid - 1;
    }
    const RowFinJob& J = p.jobs[lo];
    const int64_t v = vv - J.view_begin;
    if (J.active != nullptr && J.active[v] == 0) continue;  // NorMuon state untouched
    float* part = J.rowpart + v * J.tiles_c * J.rows;
    float* fac = J.rowfac + v * J.rows;
    double tot = 0.0, tot2 = 0.0;
    for (int64_t i = threadIdx.x; i < J.rows; i += blockDim.x) {
      float q = 0.0f;
      for (int64_t tc = 0; tc < J.tiles_c; ++tc) q += part[tc * J.rows + i];
      float f = 1.0f;
      if (p.normuon) {
        float* sm = J.sm + v * J.rows;
        const float mean = q / static_cast<float>(J.cols);
        const float smn = sm[i] + (1.0f - p.beta2) * (mean - sm[i]);
        sm[i] = smn;
        f = 1.0f / sqrtf(fmaxf(smn, p.normuon_eps));
      }
      // fac holds f for now; the row sum q is needed again below, so keep it
      // in the first tile's partial slot (this view's partials are not read
      // by anyone else).
      fac[i] = f;
      part[i] = q;
      tot += static_cast<double>(q);
      tot2 += static_cast<double>(f) * static_cast<double>(f) * static_cast<double>(q);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      tot2 += __shfl_xor_sync(0xffffffffu, tot2, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
      red[0][warp] = tot;
      red[1][warp] = tot2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      double a = 0.0, b = 0.0;
      for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        a += red[0][w];
        b += red[1][w];
      }
      float kappa = 1.0f;
      if (p.normuon) kappa = static_cast<float>(sqrt(a) / fmax(sqrt(b), 1e-10));
      s_kappa = kappa;
    }
    __syncthreads();
    const float kappa = s_kappa;
    for (int64_t i = threadIdx.x; i < J.rows; i += blockDim.x) {
      float F = kappa * fac[i];
      if (p.muon_plus) F = F / sqrtf(F * F * part[i] + p.plus_eps);
      fac[i] = F;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) col_finalize_kernel(const __grid_constant__ ColFinParams p) {
  if (step_skipped(p.skip)) return;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < p.total;
       e += int64_t(gridDim.x) * blockDim.x) {
    int lo = 0, hi = p.njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.jobs[mid].elem_begin <= e) lo = mid; else hi = mid - 1;
    }
    const ColFinJob& J = p.jobs[lo];
    const int64_t local = e - J.elem_begin;
    const int64_t v = local / J.cols, c = local - v * J.cols;
    const float* part = J.colpart + v * J.tiles_r * J.cols + c;
    float s = 0.0f;
    for (int64_t tr = 0; tr < J.tiles_r; ++tr) s += part[tr * J.cols];
    J.colfac[local] = 1.0f / sqrtf(s + p.plus_eps);
  }
}

// One block per view: ||Q||_F^2 = the sum of the view's per-warp partials,
// each thread summing a fixed stride of them, then a fixed-order tree.
__global__ void __launch_bounds__(256) view_norm_kernel(const __grid_constant__ NormParams p) {
  __shared__ double red[256];
  if (step_skipped(p.skip)) return;
  for (int64_t vv = blockIdx.x; vv < p.total_views; vv += gridDim.x) {
    int lo = 0, hi = p.njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.jobs[mid].view_begin <= vv) lo = mid; else hi = mid - 1;
    }
    const NormJob& J = p.jobs[lo];
    const int64_t v = vv - J.view_begin;
    const int64_t n = J.tiles_per_view * (kEwThreads / 32);
    const float* part = J.tile_ss + v * n;
    double s = 0.0;
    for (int64_t k = threadIdx.x; k < n; k += 256) s += static_cast<double>(part[k]);
    red[threadIdx.x] = s;
    __syncthreads();
#pragma unroll
    for (int w = 128; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
      __syncthreads();
    }
    if (threadIdx.x == 0) J.sumsq[v] = red[0];
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_col_finalize(const ColFinParams& p, int num_sms, cudaStream_t s) {
  if (p.total <= 0) return cudaSuccess;
  const int64_t blocks = (p.total + 255) / 256;
  const int64_t want = static_cast<int64_t>(num_sms) * 8;
  col_finalize_kernel<<<static_cast<int>(blocks < want ? blocks : want), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_view_norm(const NormParams& p, cudaStream_t s) {
  if (p.total_views <= 0) return cudaSuccess;
  const int64_t blocks = p.total_views;
  view_norm_kernel<<<static_cast<int>(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(p);
  return cudaGetLastError();
}

// Resident blocks per SM of each elementwise kernel (queried once per kind),
// so that the persistent grids are exactly one wave. Calls from several host
// threads may race to fill an entry; they all store the same value.
int blocks_per_sm(EwKind kind, const void* kernel) {
  static std::atomic<int> cached[kEwKinds] = {};
  int b = cached[kind].load(std::memory_order_relaxed);
  if (b == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kEwThreads, 0) != cudaSuccess ||
        b <= 0) {
      (void)cudaGetLastError();
      b = 2;
    }
    cached[kind].store(b, std::memory_order_relaxed);
  }
  return b;
}

// Tensor maps of the streaming passes, per host thread: a map depends only on
// the base address, the dtype, the extents and the row pitch, so a step that
// is called again on the same tensors encodes nothing.
struct StreamMapKey {
  const void* base;
  int64_t inner, rows, views, ld;
  bool f32;
  bool operator==(const StreamMapKey& o) const {
    return base == o.base && inner == o.inner && rows == o.rows && views == o.views &&
           ld == o.ld && f32 == o.f32;
  }
};
struct StreamMapKeyHash {
  size_t operator()(const StreamMapKey& k) const {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    for (int64_t v : {k.inner, k.rows, k.views, k.ld, static_cast<int64_t>(k.f32)})
      h = (h ^ static_cast<uint64_t>(v)) * 0x100000001B3ull;
    return static_cast<size_t>(h ^ (h >> 29));
  }
};

static bool cached_stream_map(CUtensorMap* tm, const void* base, bool f32, int64_t inner,
                              int64_t rows, int64_t views, int64_t ld) {
  static thread_local std::unordered_map<StreamMapKey, CUtensorMap, StreamMapKeyHash> cache;
  const StreamMapKey key{base, inner, rows, views, ld, f32};
  auto it = cache.find(key);
  if (it != cache.end()) {
    std::memcpy(tm, &it->second, sizeof(CUtensorMap));
    return true;
  }
  if (!encode_stream_map(tm, base, f32, inner, rows, views, ld)) return false;
  if (cache.size() >= 4096) cache.clear();  // bounded: tensors come and go
  cache.emplace(key, *tm);
  return true;
}

cudaError_t launch_elementwise(EwKind kind, const EwParams& p, int num_sms, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  if (kind == EW_APPLY && p.cautious == MH_CAUTIOUS_UPDATE) kind = EW_APPLY_CU;
  if (kind == EW_PROLOGUE_FLAT && p.use_momentum) {
    bool all_b16 = p.njobs > 0;
    for (int j = 0; j < p.njobs; ++j) all_b16 = all_b16 && p.jobs[j].mom_dtype == MH_BF16;
    if (all_b16) kind = EW_PROLOGUE_FLAT_B16;
  }
  const void* fn = nullptr;
  switch (kind) {
    case EW_PROLOGUE: fn = reinterpret_cast<const void*>(prologue_kernel); break;
    case EW_PROLOGUE_FLAT: fn = reinterpret_cast<const void*>(prologue_flat_kernel<false>); break;
    case EW_PROLOGUE_FLAT_B16:
      fn = reinterpret_cast<const void*>(prologue_flat_kernel<true>);
      break;
    case EW_ROWSQ: fn = reinterpret_cast<const void*>(ew_kernel<EW_ROWSQ>); break;
    case EW_COLSQ: fn = reinterpret_cast<const void*>(ew_kernel<EW_COLSQ>); break;
    case EW_APPLY: fn = reinterpret_cast<const void*>(ew_kernel<EW_APPLY>); break;
    case EW_APPLY_CU: fn = reinterpret_cast<const void*>(ew_kernel<EW_APPLY_CU>); break;
    case EW_COPYOUT: fn = reinterpret_cast<const void*>(ew_kernel<EW_COPYOUT>); break;
  }
  // The register-staged kernels, on the whole launch or on a part of it.
  auto launch_staged = [&](const EwParams& q) -> cudaError_t {
    const int per_sm = blocks_per_sm(kind, fn);
    const int64_t want = static_cast<int64_t>(num_sms) * per_sm;
    const int grid = static_cast<int>(q.total_tiles < want ? q.total_tiles : want);
    if (grid <= 0) return cudaSuccess;
    switch (kind) {
      case EW_PROLOGUE: prologue_kernel<<<grid, kEwThreads, 0, s>>>(q); break;
      case EW_PROLOGUE_FLAT: prologue_flat_kernel<false><<<grid, kEwThreads, 0, s>>>(q); break;
      case EW_PROLOGUE_FLAT_B16: prologue_flat_kernel<true><<<grid, kEwThreads, 0, s>>>(q); break;
      case EW_ROWSQ: ew_kernel<EW_ROWSQ><<<grid, kEwThreads, 0, s>>>(q); break;
      case EW_COLSQ: ew_kernel<EW_COLSQ><<<grid, kEwThreads, 0, s>>>(q); break;
      case EW_APPLY: ew_kernel<EW_APPLY><<<grid, kEwThreads, 0, s>>>(q); break;
      case EW_APPLY_CU: ew_kernel<EW_APPLY_CU><<<grid, kEwThreads, 0, s>>>(q); break;
      case EW_COPYOUT: ew_kernel<EW_COPYOUT><<<grid, kEwThreads, 0, s>>>(q); break;
    }
    return cudaGetLastError();
  };
  // The apply (every cautious form) and the Muon+ column statistics take the
  // streaming kernel when the launch has a status word for its bounded waits:
  // one block per SM, the stage layout sized for the parameter dtypes of the
  // launch. The cautious update, with a gradient map per job as well, runs in
  // parts of at most kStreamCuJobs jobs.
  if ((kind == EW_APPLY || kind == EW_APPLY_CU || kind == EW_COLSQ) && p.status != nullptr) {
    bool any_f32 = false;
    for (int j = 0; j < p.njobs; ++j) any_f32 = any_f32 || p.jobs[j].dst_dtype == MH_F32;
    const void* ks[5] = {reinterpret_cast<const void*>(ew_stream_kernel<EW_COLSQ, 0>),
                         reinterpret_cast<const void*>(ew_stream_kernel<EW_APPLY, 16>),
                         reinterpret_cast<const void*>(ew_stream_kernel<EW_APPLY, 32>),
                         reinterpret_cast<const void*>(ew_stream_kernel<EW_APPLY_CU, 16>),
                         reinterpret_cast<const void*>(ew_stream_kernel<EW_APPLY_CU, 32>)};
    const size_t sz[5] = {stream_smem_bytes<EW_COLSQ, 0>(), stream_smem_bytes<EW_APPLY, 16>(),
                          stream_smem_bytes<EW_APPLY, 32>(), stream_smem_bytes<EW_APPLY_CU, 16>(),
                          stream_smem_bytes<EW_APPLY_CU, 32>()};
    const bool cu = kind == EW_APPLY_CU;
    const int which = kind == EW_COLSQ ? 0 : (cu ? 3 : 1) + (any_f32 ? 1 : 0);
    static thread_local int configured = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured != dev) {
      for (int k = 0; k < 5; ++k) {
        e = cudaFuncSetAttribute(ks[k], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sz[k]));
        if (e != cudaSuccess) return e;
      }
      configured = dev;
    }
    static thread_local StreamParams sp;
    const int per = cu ? kStreamCuJobs : kMaxJobs;
    for (int j0 = 0; j0 < p.njobs; j0 += per) {
      const int j1 = p.njobs - j0 < per ? p.njobs : j0 + per;
      // This part's jobs, their tile indices counted from its first tile.
      sp.ew = p;
      if (j0 > 0 || j1 < p.njobs) {
        const int64_t base = p.jobs[j0].tile_begin;
        const int64_t end = j1 < p.njobs ? p.jobs[j1].tile_begin : p.total_tiles;
        for (int k = 0; k < j1 - j0; ++k) {
          sp.ew.jobs[k] = p.jobs[j0 + k];
          sp.ew.jobs[k].tile_begin -= base;
        }
        sp.ew.njobs = j1 - j0;
        sp.ew.total_tiles = end - base;
      }
      const EwParams& q = sp.ew;
      if (q.total_tiles <= 0) continue;
      // Per job: the U view stack (row pitch ldx, zero fill past cols and
      // rows) and, where the apply stages them, the parameter and the
      // gradient.
      bool maps_ok = true;
      for (int k = 0; k < q.njobs && maps_ok; ++k) {
        const EwJob& J = q.jobs[k];
        maps_ok = cached_stream_map(&sp.tmU[k], J.xf, false, J.cols, J.rows, J.views, J.ldx);
        const bool wst = J.dst_vec && (J.dst_dtype == MH_F32 || (J.cols % 8) == 0);
        if (maps_ok && kind != EW_COLSQ && wst)
          maps_ok = cached_stream_map(&sp.tmW[k], J.dst, J.dst_dtype == MH_F32, J.cols, J.rows,
                                      J.views, J.cols);
        if (maps_ok && cu && stream_g_staged(J))
          maps_ok = cached_stream_map(&sp.tmU[kStreamCuJobs + k], J.src, false, J.cols, J.rows,
                                      J.views, J.cols);
      }
      if (!maps_ok) {
        if ((e = launch_staged(q)) != cudaSuccess) return e;
        continue;
      }
      const int grid = static_cast<int>(q.total_tiles < num_sms ? q.total_tiles : num_sms);
      void* args[] = {&sp};
      e = cudaLaunchKernel(ks[which], dim3(grid), dim3(kStreamThreads), args, sz[which], s);
      if (e != cudaSuccess) return e;
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  return launch_staged(p);
}

cudaError_t launch_view_active(const ActiveParams& p, int num_sms, cudaStream_t s) {
  if (p.total_chunks <= 0) return cudaSuccess;
  const int64_t want = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(p.total_chunks < want ? p.total_chunks : want);
  view_active_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_row_finalize(const RowFinParams& p, cudaStream_t s) {
  if (p.total_views <= 0) return cudaSuccess;
  const int grid = static_cast<int>(p.total_views < 4096 ? p.total_views : 4096);
  row_finalize_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mh
