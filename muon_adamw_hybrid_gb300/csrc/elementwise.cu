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
#include "mh_internal.h"
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
  const int per_sm = blocks_per_sm(kind, fn);
  const int64_t want = static_cast<int64_t>(num_sms) * per_sm;
  const int grid = static_cast<int>(p.total_tiles < want ? p.total_tiles : want);
  switch (kind) {
    case EW_PROLOGUE: prologue_kernel<<<grid, kEwThreads, 0, s>>>(p); break;
    case EW_PROLOGUE_FLAT: prologue_flat_kernel<false><<<grid, kEwThreads, 0, s>>>(p); break;
    case EW_PROLOGUE_FLAT_B16: prologue_flat_kernel<true><<<grid, kEwThreads, 0, s>>>(p); break;
    case EW_ROWSQ: ew_kernel<EW_ROWSQ><<<grid, kEwThreads, 0, s>>>(p); break;
    case EW_COLSQ: ew_kernel<EW_COLSQ><<<grid, kEwThreads, 0, s>>>(p); break;
    case EW_APPLY: ew_kernel<EW_APPLY><<<grid, kEwThreads, 0, s>>>(p); break;
    case EW_APPLY_CU: ew_kernel<EW_APPLY_CU><<<grid, kEwThreads, 0, s>>>(p); break;
    case EW_COPYOUT: ew_kernel<EW_COPYOUT><<<grid, kEwThreads, 0, s>>>(p); break;
  }
  return cudaGetLastError();
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
