// Grouped Newton-Schulz GEMM stage on sm_103a tensor cores (tcgen05 + TMEM,
// operands staged by TMA with 128-byte swizzle, CTA pairs sharing operands by
// TMA multicast).
//
// One quintic step (Speedtronic "v2 optimizers", "Newton-Schulz"; flaxchat
// "Optimizer", "Muon Algorithm" step 2) is three launches of this kernel:
//
//   GEMM_GRAM   A = X X^T             (m x m; only the upper block triangle is
//                                      computed: a 32 x 32 chunk above the
//                                      diagonal is stored and mirrored, one on
//                                      it stored whole)
//   GEMM_POLY   P = b A + c A A       (A symmetric, so A A = A A^T: both
//                                      operands are K-major rows of A; same
//                                      triangle scheme; b A read in the epilogue)
//   GEMM_APPLY  X' = a X + P X        (B operand = X read MN-major)
//
// A tall view (rows > cols) keeps its Newton-Schulz matrix in the stored
// layout T = X^T (n x m); for such shape classes the gram reads T with
// MN-major A and B operands (A = T^T T) and the apply computes T' = a T + T P
// with K-major operands (P is symmetric), so no pass ever transposes data.
//
// On the first step the Frobenius normalisation 1/(||Q||_F + eps) is folded in:
// the gram epilogue scales by s^2 and the apply epilogue by s, so the
// prologue never has to re-read Q to normalise it.
//
// Work unit: a 256 x 256 output block computed by a cluster of two CTAs, CTA
// rank k taking rows 128k..128k+127 (one tcgen05.mma M=128 N=256 K=16 per
// 16 of k). Both CTAs need the same 256 B-rows per k-step: each loads half of
// them and multicasts it to both, so every CTA fetches 32 KB per 64-deep k
// step from L2 instead of 48 KB. A CTA frees a pipeline stage only when the
// MMAs of both CTAs have read it (the MMA completion is multicast to both
// "empty" barriers).
//
// One launch per stage covers every shape class of the call, whatever its
// operand major-ness (see GemmMode): each role picks a k-loop specialised on
// the tile's mode once per tile, so nothing is re-read inside the k-loop.
//
// Blocks are handed out dynamically: CTA 0 of each pair claims the next block
// index from a counter in the workspace and publishes it to both CTAs through
// a small shared-memory ring, so every pair works on the block after the
// last one claimed. All pairs therefore stay within about one wave of
// consecutive blocks, which share the m x m operand (apply) or the row blocks
// of X (gram, poly) in L2; a static deal let fast and slow pairs drift apart
// by many blocks, and their operands no longer fitted in L2 together.
//
// Warp roles per CTA: warp 0 issues TMA loads into a 4-stage ring, warp 1
// issues tcgen05.mma into one of two TMEM accumulators, warp 2 owns the TMEM
// allocation, warps 4-7 drain an accumulator with tcgen05.ld (one row per
// lane, 32 columns at a time), apply the stage's epilogue in fp32 and, while
// the MMA warp fills the other accumulator, write each bf16 chunk (and its
// transpose, for the mirrored half of a symmetric output) into swizzled
// shared-memory boxes that one lane stores with TMA. The fused parameter
// update of the last apply stage reads and writes the parameters directly.
//
// Every mbarrier wait is bounded (the launch's wait limit); on timeout the CTA
// records a status code in the workspace, raises the abort flag of both CTAs
// of its pair, drains what it has in flight (with the fixed, long drain
// limit), frees TMEM and exits.
#include <map>
#include <mutex>

#include "mh_internal.h"
#include "mh_ptx.cuh"
#include "mh_sr.cuh"
#include "muonhybrid.h"

namespace mh {

static_assert(sizeof(GemmParams) <= 32000, "GemmParams exceeds the kernel parameter space");

namespace {

constexpr uint32_t kStageABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kStageBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kHalfBBytes = kStageBBytes / 2;
constexpr uint32_t kTmemCols = 2 * kBN;           // two fp32 accumulators
constexpr uint32_t kApplyChunkBytes = kBK * 64 * 2;  // one 64-col MN-major box: 8 KB
// Epilogue staging: each epilogue warp owns two buffers, each holding a 32 x 32
// bf16 box of the chunk (rows r0.., cols c0..) and one of its transpose (the
// mirrored block of a symmetric output), laid out as the 64-byte-swizzled
// boxes the output tensor map stores.
constexpr uint32_t kOutBoxBytes = 32 * 32 * 2;                 // 2 KB
constexpr uint32_t kOutWarpBytes = 2 * 2 * kOutBoxBytes;        // 8 KB per epilogue warp
constexpr uint16_t kPairMask = 0x3;

struct TileCoord {
  int cls, view, tm, tn;
};

// Maps a pair-tile index to (class, view, 256-row block pm, 256-col block tn)
// and returns this CTA's 128-row tile tm = 2 pm + rank.
__device__ __forceinline__ TileCoord map_tile(const GemmParams& p, int64_t t, uint32_t rank) {
  int c = 0;
  while (c + 1 < p.num_classes && t >= p.cls[c + 1].tile_begin) ++c;
  const GemmClass& C = p.cls[c];
  const int64_t local = t - C.tile_begin;
  TileCoord tc;
  tc.cls = c;
  tc.view = static_cast<int>(local / C.tiles_per_view);
  int w = static_cast<int>(local - static_cast<int64_t>(tc.view) * C.tiles_per_view);
  int pm;
  if (p.kind == GEMM_APPLY) {
    // Consecutive tiles walk the m x m operand P (which stays in L2) and share
    // one block of X: for X = m x n the row blocks of the output, for a tall
    // view's T = n x m (mode KK) its column blocks.
    if (C.mode == GEMM_MODE_KK) {
      tc.tn = w % C.tiles_n;
      pm = w / C.tiles_n;
    } else {
      pm = w % C.tiles_m;
      tc.tn = w / C.tiles_m;
    }
  } else {
    // Row block pm holds the column blocks tn >= pm (upper block triangle).
    pm = 0;
    while (true) {
      const int cnt = C.tiles_n - pm;
      if (w < cnt) break;
      w -= cnt;
      ++pm;
    }
    tc.tn = pm + w;
  }
  tc.tm = 2 * pm + static_cast<int>(rank);
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

// 32 bf16 of row r from column c0 of a (row pitch ld) into four 16-byte
// registers, when the row exists and all 32 columns are inside n_cols
// (ragged chunks are read element by element where they are used).
__device__ __forceinline__ void prefetch_aux32(const bf16* a, int64_t ld, int r, int c0,
                                               int n_rows, int n_cols, bool use,
                                               uint4 (&dst)[4]) {
  if (use && r < n_rows && c0 + 32 <= n_cols) {
    const uint4* s = reinterpret_cast<const uint4*>(a + static_cast<int64_t>(r) * ld + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = s[q];
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ void unpack_bf16x32(const uint4 (&u)[4], float (&x)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[q * 8 + 2 * k] = __uint_as_float(w[k] << 16);
      x[q * 8 + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
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

__device__ __forceinline__ void load_f32x32(const void* base, int dt, int64_t off, int nvalid,
                                            bool vec, float (&x)[32]) {
  if (vec) {
    if (dt == MH_F32) {
      const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 t = s[q];
        x[4 * q] = t.x; x[4 * q + 1] = t.y; x[4 * q + 2] = t.z; x[4 * q + 3] = t.w;
      }
    } else {
      load_bf16x32(static_cast<const bf16*>(base) + off, x);
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < nvalid)
      x[j] = dt == MH_F32 ? static_cast<const float*>(base)[off + j]
                          : __bfloat162float(static_cast<const bf16*>(base)[off + j]);
    else
      x[j] = 0.0f;
  }
}

__device__ __forceinline__ void store_f32x32(void* base, int dt, int64_t off, int nvalid, bool vec,
                                             const float (&x)[32]) {
  if (vec) {
    if (dt == MH_F32) {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        d[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    } else {
      store_bf16x32(static_cast<bf16*>(base) + off, x);
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < nvalid) {
      if (dt == MH_F32)
        static_cast<float*>(base)[off + j] = x[j];
      else
        static_cast<bf16*>(base)[off + j] = __float2bfloat16_rn(x[j]);
    }
  }
}

// The parameter update of Speedtronic "Muon update" (decoupled decay and
// max(1, rows/cols)^0.5 scale), or one of the cautious forms (flaxchat step
// 4; Speedtronic "Cautious updates"), on 32 consecutive elements of one
// stored row starting at element `off`; u holds the Newton-Schulz output.
// `wpre`: the 32 bf16 parameters at `off`, already loaded (full vector
// chunks of a bf16 parameter), or null to load them here.
__device__ __forceinline__ void update_w32(const ViewRec& R, int64_t off, int nvalid,
                                           const float (&u)[32], int cautious,
                                           const uint4 (*wpre)[4]) {
  if (R.inactive) return;  // zero gradient under the inactive-expert rule
  const bool vec = R.vec && nvalid == 32;
  float w[32];
  if (wpre)
    unpack_bf16x32(*wpre, w);
  else
    load_f32x32(R.param, R.pdt, off, nvalid, vec, w);
  const float lr = R.lr, wd = R.wd, sc = R.shape_scale;
  if (cautious == MH_CAUTIOUS_OFF) {
    const float decay = 1.0f - lr * wd;
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = decay * w[j] - (lr * sc) * u[j];
  } else if (cautious == MH_CAUTIOUS_WD) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float g = sc * u[j];
      const float mask = (g * w[j] >= 0.0f) ? 1.0f : 0.0f;
      w[j] = w[j] - lr * (g + wd * w[j] * mask);
    }
  } else {
    float gr[32];
    load_f32x32(R.grad, R.gdt, off, nvalid, vec, gr);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float delta = lr * wd * w[j] + (lr * sc) * u[j];
      if (delta * gr[j] > 0.0f) w[j] = w[j] - delta;
    }
  }
  if (R.psr && R.pdt == MH_BF16)
    store_bf16_sr<32>(static_cast<bf16*>(R.param) + off, nvalid, vec, w, R.psr_key,
                      static_cast<uint64_t>(off));
  else
    store_f32x32(R.param, R.pdt, off, nvalid, vec, w);
}

// Raises the abort flag of both CTAs of the pair.
__device__ __forceinline__ void abort_pair(volatile int* abort_flag) {
  *abort_flag = 1;
  st_cluster_s32(abort_flag, 0, 1);
  st_cluster_s32(abort_flag, 1, 1);
}

// The TMA loads of k-blocks kb0 .. kb1-1 of one tile in operand mode MODE.
// Returns false when the launch aborts.
template <int MODE>
__device__ __forceinline__ bool load_tile(const GemmParams& p, const GemmClass& C,
                                          const TileCoord& tc, uint32_t rank, int kb0, int kb1,
                                          uint8_t* sA, uint8_t* sB, uint64_t* full,
                                          uint64_t* empty, int& stage, uint32_t& phase,
                                          uint32_t& inflight, uint32_t& inflight_par,
                                          volatile int* abort_flag) {
  constexpr bool a_mn = MODE == GEMM_MODE_MM;
  constexpr bool b_mn = MODE != GEMM_MODE_KK;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_TMA,
                           p.wait_limit))
      return false;
    mbar_arrive_expect_tx(&full[stage], kStageABytes + kStageBBytes);
    uint8_t* a_dst = sA + stage * kStageABytes;
    if constexpr (a_mn) {
      // 128 columns of T as two MN-major 64-column chunks.
#pragma unroll
      for (int j = 0; j < 2; ++j)
        tma_load_3d(a_dst + j * kApplyChunkBytes, &C.tmA, &full[stage], tc.tm * kBM + j * 64,
                    kb * kBK, tc.view);
    } else {
      tma_load_3d(a_dst, &C.tmA, &full[stage], kb * kBK, tc.tm * kBM, tc.view);
    }
    uint8_t* b_dst = sB + stage * kStageBBytes;
    if constexpr (b_mn) {
      // This CTA's two 64-column chunks of the 256-column B block.
#pragma unroll
      for (int j = 2 * static_cast<int>(rank); j < 2 * static_cast<int>(rank) + 2; ++j)
        tma_load_3d_mc(b_dst + j * kApplyChunkBytes, &C.tmB, &full[stage], tc.tn * kBN + j * 64,
                       kb * kBK, tc.view, kPairMask);
    } else {
      // This CTA's 128 of the 256 B rows.
      tma_load_3d_mc(b_dst + rank * kHalfBBytes, &C.tmB, &full[stage], kb * kBK,
                     tc.tn * kBN + static_cast<int>(rank) * kBM, tc.view, kPairMask);
    }
    inflight |= 1u << stage;
    inflight_par = (inflight_par & ~(1u << stage)) | (phase << stage);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// The MMAs of k-blocks kb0 .. kb1-1 of one tile in operand mode MODE into the
// accumulator at d_tmem (k-block 0 overwrites it). Returns false when the
// launch aborts.
template <int MODE>
__device__ __forceinline__ bool mma_tile(const GemmParams& p, int kb0, int kb1, uint32_t d_tmem,
                                         uint8_t* sA, uint8_t* sB, uint64_t* full,
                                         uint64_t* empty, int& stage, uint32_t& phase,
                                         bool& issued, volatile int* abort_flag) {
  constexpr bool a_mn = MODE == GEMM_MODE_MM;
  constexpr bool b_mn = MODE != GEMM_MODE_KK;
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, a_mn ? 1 : 0, b_mn ? 1 : 0);
  // K-major: 16 bf16 of k = 32 bytes inside the 128-byte swizzle row.
  // MN-major: 16 k-rows = two 1024-byte atoms, 64-column chunks 8 KB apart.
  constexpr uint32_t a_kstep = a_mn ? 2048u : 32u, a_lbo = a_mn ? kApplyChunkBytes : 16u;
  constexpr uint32_t b_kstep = b_mn ? 2048u : 32u, b_lbo = b_mn ? kApplyChunkBytes : 16u;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, p.status, DEV_TIMEOUT_MMA,
                           p.wait_limit))
      return false;
    tc_fence_after();
    const uint32_t a0 = smem_addr(sA + stage * kStageABytes);
    const uint32_t b0 = smem_addr(sB + stage * kStageBBytes);
#pragma unroll
    for (int k = 0; k < kBK / 16; ++k) {
      const uint64_t ad = smem_desc_sw128(a0 + k * a_kstep, a_lbo, 1024);
      const uint64_t bd = smem_desc_sw128(b0 + k * b_kstep, b_lbo, 1024);
      tc_mma_f16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
    }
    issued = true;
    tc_commit_mc(&empty[stage], kPairMask);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

constexpr int kModeKK = 1 << GEMM_MODE_KK, kModeKM = 1 << GEMM_MODE_KM, kModeMM = 1 << GEMM_MODE_MM;

// The loads of one tile in a kernel specialised on the set MODES of operand
// modes its launch contains: a single mode needs no dispatch at all.
template <int MODES>
__device__ __forceinline__ bool load_tile_of(const GemmParams& p, const GemmClass& C,
                                             const TileCoord& tc, uint32_t rank, int kb0, int kb1,
                                             uint8_t* sA, uint8_t* sB, uint64_t* full,
                                             uint64_t* empty, int& stage, uint32_t& phase,
                                             uint32_t& inflight, uint32_t& inflight_par,
                                             volatile int* abort_flag) {
  if constexpr ((MODES & kModeKK) != 0)
    if (MODES == kModeKK || C.mode == GEMM_MODE_KK)
      return load_tile<GEMM_MODE_KK>(p, C, tc, rank, kb0, kb1, sA, sB, full, empty, stage,
                                     phase, inflight, inflight_par, abort_flag);
  if constexpr ((MODES & kModeKM) != 0)
    if (MODES == kModeKM || C.mode == GEMM_MODE_KM || (MODES & kModeMM) == 0)
      return load_tile<GEMM_MODE_KM>(p, C, tc, rank, kb0, kb1, sA, sB, full, empty, stage,
                                     phase, inflight, inflight_par, abort_flag);
  if constexpr ((MODES & kModeMM) != 0)
    return load_tile<GEMM_MODE_MM>(p, C, tc, rank, kb0, kb1, sA, sB, full, empty, stage, phase,
                                   inflight, inflight_par, abort_flag);
  return false;
}

template <int MODES>
__device__ __forceinline__ bool mma_tile_of(const GemmParams& p, int mode, int kb0, int kb1,
                                            uint32_t d_tmem, uint8_t* sA, uint8_t* sB,
                                            uint64_t* full, uint64_t* empty, int& stage,
                                            uint32_t& phase, bool& issued,
                                            volatile int* abort_flag) {
  if constexpr ((MODES & kModeKK) != 0)
    if (MODES == kModeKK || mode == GEMM_MODE_KK)
      return mma_tile<GEMM_MODE_KK>(p, kb0, kb1, d_tmem, sA, sB, full, empty, stage, phase,
                                    issued, abort_flag);
  if constexpr ((MODES & kModeKM) != 0)
    if (MODES == kModeKM || mode == GEMM_MODE_KM || (MODES & kModeMM) == 0)
      return mma_tile<GEMM_MODE_KM>(p, kb0, kb1, d_tmem, sA, sB, full, empty, stage, phase,
                                    issued, abort_flag);
  if constexpr ((MODES & kModeMM) != 0)
    return mma_tile<GEMM_MODE_MM>(p, kb0, kb1, d_tmem, sA, sB, full, empty, stage, phase,
                                  issued, abort_flag);
  return false;
}

// The pair's shared tile sequence. Entries 0 and 1 are static, the pair's
// own index p and p + npairs: every pair starts without waiting for a claim,
// a launch of at most two rounds of blocks claims nothing, and the first
// claim has a whole block's time to return. From entry 2 on, CTA 0's
// producer claims block indices from the launch's counter (offset by
// 2 npairs).
//
// Entry i >= 1 travels at ring position i - 1 (slot (i - 1) mod kTileRing)
// through two rings. The pair ring carries it from CTA 0's producer to CTA
// 1's producer only (cluster scope, one consumer). Each CTA's producer then
// publishes it on its own CTA's local ring, which that CTA's MMA issuer and
// four epilogue warps read (CTA scope, kLocalConsumers arrivals per entry),
// so the roles on the critical path never wait on the other CTA.
constexpr uint32_t kLocalConsumers = 5;

struct Rings {
  uint64_t* pair_full;   // in CTA 1: CTA 0 arrives once per entry
  uint64_t* pair_empty;  // in CTA 0: CTA 1's producer arrives once per entry
  uint32_t* pair_slots;  // in CTA 1, written by CTA 0
  uint64_t* local_full;  // this CTA's producer arrives once per entry
  uint64_t* local_empty; // this CTA's MMA issuer and epilogue warps arrive
  uint32_t* local_slots;
};

// CTA 0: hands the tile index t at ring position i to CTA 1's producer.
// Returns false when the launch aborts.
__device__ __forceinline__ bool pair_publish(const GemmParams& p, const Rings& R, uint32_t i,
                                             uint32_t t, volatile int* abort_flag) {
  const uint32_t s = i % kTileRing;
  const uint32_t par = (i / kTileRing) & 1u;
  if (!mbar_wait_bounded<true>(&R.pair_empty[s], par ^ 1u, abort_flag, p.status,
                               DEV_TIMEOUT_TMA, p.wait_limit))
    return false;
  // The index travels as an asynchronous store whose completion counts on
  // CTA 1's barrier, so no release (which would wait for this thread's TMA
  // loads in flight) is needed to order it before the arrive.
  mbar_arrive_expect_tx_relaxed(&R.pair_full[s], 1, 4);
  st_async_u32(&R.pair_slots[s], 1, t, &R.pair_full[s]);
  return true;
}

// CTA 1: the tile index at ring position i from CTA 0, then the slot is
// released; -1 when the launch aborts. The slot is read with acquire
// semantics, so the relaxed release arrive cannot be performed before it.
__device__ __forceinline__ int64_t pair_read(const GemmParams& p, const Rings& R, uint32_t i,
                                             volatile int* abort_flag) {
  const uint32_t s = i % kTileRing;
  const uint32_t par = (i / kTileRing) & 1u;
  if (!mbar_wait_bounded<true>(&R.pair_full[s], par, abort_flag, p.status, DEV_TIMEOUT_TMA,
                               p.wait_limit))
    return -1;
  const uint32_t t = ld_acquire_cluster_u32(&R.pair_slots[s]);
  mbar_arrive_cluster_relaxed(&R.pair_empty[s], 0);
  return static_cast<int64_t>(t);
}

// A CTA's producer: publishes the tile index t at ring position i to its
// own CTA's MMA issuer and epilogue warps. Returns false when the launch
// aborts.
__device__ __forceinline__ bool local_publish(const GemmParams& p, const Rings& R, uint32_t i,
                                              uint32_t t, volatile int* abort_flag) {
  const uint32_t s = i % kTileRing;
  const uint32_t par = (i / kTileRing) & 1u;
  if (!mbar_wait_bounded(&R.local_empty[s], par ^ 1u, abort_flag, p.status, DEV_TIMEOUT_TMA,
                         p.wait_limit))
    return false;
  // As in pair_publish, to this CTA's own ring.
  const uint32_t self = cluster_ctarank();
  mbar_arrive_expect_tx_relaxed(&R.local_full[s], self, 4);
  st_async_u32(&R.local_slots[s], self, t, &R.local_full[s]);
  return true;
}

// The tile index at ring position i of this CTA's local ring, read by one
// thread, which then releases the slot; -1 when the launch aborts. The read
// has acquire semantics and the release arrive is relaxed: the reader's own
// writes (an epilogue's parameter stores) need not wait for it.
__device__ __forceinline__ int64_t local_read(const GemmParams& p, const Rings& R, uint32_t i,
                                              volatile int* abort_flag, int code) {
  const uint32_t s = i % kTileRing;
  const uint32_t par = (i / kTileRing) & 1u;
  if (!mbar_wait_bounded(&R.local_full[s], par, abort_flag, p.status, code, p.wait_limit))
    return -1;
  const uint32_t t = ld_acquire_cta_u32(&R.local_slots[s]);
  mbar_arrive_relaxed(&R.local_empty[s]);
  return static_cast<int64_t>(t);
}

template <int MODES>
__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageABytes;
  uint8_t* sO = sB + kStages * kStageBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sO + 4 * kOutWarpBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  Rings R;
  R.pair_full = drain + 1;
  R.pair_empty = R.pair_full + kTileRing;
  R.local_full = R.pair_empty + kTileRing;
  R.local_empty = R.local_full + kTileRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(R.local_empty + kTileRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  R.pair_slots = tmem_slot + 2;
  R.local_slots = R.pair_slots + kTileRing;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t total = static_cast<uint32_t>(p.total_tiles);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);  // released by the MMAs of both CTAs
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kTileRing; ++s) {
      mbar_init(&R.pair_full[s], 1);
      mbar_init(&R.pair_empty[s], 1);
      mbar_init(&R.local_full[s], 1);
      mbar_init(&R.local_empty[s], kLocalConsumers);
    }
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
  cluster_sync();  // barrier inits of both CTAs visible before any remote traffic
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool apply = p.kind == GEMM_APPLY;

  // The kernel is launched as a programmatic dependent of the previous one
  // on the stream: the setup above (barriers, tensor-map prefetch, TMEM,
  // cluster barrier) touches only shared memory, TMEM and the parameter
  // block, so it overlaps that kernel's tail. Nothing it writes is read
  // before this wait. Then the next stage's grid may launch, so its CTAs are
  // resident by the time this grid finishes.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The launch after the next one claims from this counter: every launch
  // before it has completed by then, this one included.
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.next_counter = 0u;

  if (step_skipped(p.skip)) {
    // A skipped step (gradient control): every thread of both CTAs reads the
    // same flag, no role runs, and the teardown below still pairs the
    // cluster barrier and frees TMEM.
  } else if (warp == 0) {
    // ---------------- TMA producer (CTA 0: also claims the tiles) ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t inflight = 0;     // stages with a load issued
      uint32_t inflight_par = 0; // parity of that load's phase
      bool ok = true;
      // Entry i of the tile sequence is t. CTA 0 publishes entry i + 1 on
      // both rings before tile i's first load (it is static, or was claimed
      // during tile i - 1) and claims the index of entry i + 2, which it
      // needs a whole tile later. CTA 1's producer reads entry i + 1 once
      // tile i's loads are issued and publishes it on its own local ring. So
      // every read finds an entry published a tile earlier, and CTA 1's loads
      // never wait for CTA 0.
      const uint32_t npairs = gridDim.x >> 1;
      uint32_t i = 0;
      int64_t t = blockIdx.x >> 1;
      uint32_t next = (blockIdx.x >> 1) + npairs;  // CTA 0: entry i + 1
      auto claim = [&]() { return 2u * npairs + atomicAdd(p.tile_counter, 1u); };
      while (ok && t < total) {
        if (rank == 0) {
          ok = pair_publish(p, R, i, next, abort_flag) &&
               local_publish(p, R, i, next, abort_flag);
          if (!ok) break;
        }
        const int64_t t_pub = next;
        if (rank == 0 && next < total) next = claim();
        const TileCoord tc = map_tile(p, t, rank);
        const GemmClass& C = p.cls[tc.cls];
        const int nk = (C.K + kBK - 1) / kBK;
        ok = load_tile_of<MODES>(p, C, tc, rank, 0, nk, sA, sB, full, empty, stage, phase,
                                 inflight, inflight_par, abort_flag);
        if (!ok) break;
        int64_t t_next = t_pub;
        if (rank != 0) {
          t_next = pair_read(p, R, i, abort_flag);
          ok = t_next >= 0 && local_publish(p, R, i, static_cast<uint32_t>(t_next), abort_flag);
          if (!ok) break;
        }
        t = t_next;
        ++i;
      }
      if (ok) {
        // Wait until both CTAs' MMAs have released every stage this CTA
        // filled: after this, no arrive from the peer can still be on its way
        // to this CTA's barriers.
        for (int k = 0; k < kStages; ++k) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_TMA,
                                 p.wait_limit)) {
            ok = false;
            break;
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        abort_pair(abort_flag);
        // Let every copy into this CTA's shared memory land before it exits.
        for (int s = 0; s < kStages; ++s)
          if (inflight & (1u << s)) mbar_wait_drain(&full[s], (inflight_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      int64_t t = blockIdx.x >> 1;
      for (uint32_t i = 0;; ++i) {
        if (t < 0) {
          ok = false;
          break;
        }
        if (t >= total) break;
        const TileCoord tc = map_tile(p, t, rank);
        const GemmClass& C = p.cls[tc.cls];
        const int nk = (C.K + kBK - 1) / kBK;
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_MMA,
                               p.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        ok = mma_tile_of<MODES>(p, C.mode, 0, nk, d_tmem, sA, sB, full, empty, stage, phase,
                                issued, abort_flag);
        if (!ok) break;
        tc_commit(&tfull[acc]);
        // Entry i + 1 was published before this tile's loads.
        const int64_t t_next = local_read(p, R, i, abort_flag, DEV_TIMEOUT_MMA);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        t = t_next;
      }
      if (!ok) abort_pair(abort_flag);
      if (!ok && issued) {
        tc_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int ew = warp - 4;  // TMEM lanes 32*ew .. 32*ew+31
    uint8_t* obuf = sO + ew * kOutWarpBytes;
    uint32_t staged = 0;  // chunks this warp has handed to TMA stores (buffer = parity)
    int acc = 0;
    uint32_t acc_phase = 0;
    // Lane 0 reads each entry and releases its slot; the others take it from
    // lane 0, so the whole warp agrees on the tile (or on an abort). Entry
    // i + 1 (ring position i) is read once tile i's accumulator is full.
    auto read_entry = [&](uint32_t idx) -> int64_t {
      long long tl = 0;
      if (lane == 0)
        tl = local_read(p, R, idx, abort_flag, DEV_TIMEOUT_EPI);
      return __shfl_sync(0xffffffffu, tl, 0);
    };
    int64_t t = blockIdx.x >> 1;
    for (uint32_t i = 0;; ++i) {
      if (t < 0) {
        if (lane == 0) abort_pair(abort_flag);
        break;
      }
      if (t >= total) break;
      const TileCoord tc = map_tile(p, t, rank);
      const GemmClass& C = p.cls[tc.cls];
      const int r0 = tc.tm * kBM + ew * 32;  // first row of this warp
      const int r = r0 + lane;
      const int rows_out = apply ? C.out_rows : C.m;
      const int n_out = apply ? C.out_cols : C.m;
      const bf16* aux = C.aux + static_cast<int64_t>(tc.view) * C.aux_view_stride;
      // The epilogue's second operand (a X for apply, b A for poly) is an input
      // of this launch: the first 32 columns of this lane's row are fetched
      // before the accumulator is ready, and each later chunk one step ahead,
      // so no chunk waits for a load it has just issued.
      const bool use_aux = apply || p.kind == GEMM_POLY;
      uint4 pf[4];
      prefetch_aux32(aux, C.ld_aux, r, tc.tn * kBN, rows_out, n_out, use_aux, pf);
      // The fused update reads a bf16 parameter the same way, one chunk ahead.
      // The record's view is stored exactly like this tile's output (tall views
      // are kept in their stored layout), so row r / columns c0.. of the
      // output are row r / columns c0.. of the parameter.
      const bool fin = apply && p.final_update;
      ViewRec R;
      if (fin) R = C.vrec[tc.view];
      const bool w_pf = fin && R.vec && R.pdt == MH_BF16 && !R.inactive;
      const bf16* wbase = w_pf ? static_cast<const bf16*>(R.param) + R.elem0 : nullptr;
      uint4 pw[4];
      prefetch_aux32(wbase, fin ? R.cols : 0, r, tc.tn * kBN, rows_out, n_out, w_pf, pw);
      // Every lane waits for the accumulator; the warp goes on only if all
      // of them saw it full, so a timeout never splits the warp before the
      // warp-wide TMEM loads.
      const bool full_ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, p.status,
                                             DEV_TIMEOUT_EPI, p.wait_limit);
      if (!__all_sync(0xffffffffu, full_ok)) {
        if (lane == 0) abort_pair(abort_flag);
        break;
      }
      tc_fence_after();
      const int64_t t_next = read_entry(i);

      float sc = 1.0f;
      if (p.first_iter) {
        const float s = ns_inv_norm(C.sumsq[tc.view], p.norm_scale, p.eps);
        sc = apply ? s : s * s;
      }
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                             static_cast<uint32_t>(acc * kBN);
      // Last apply under NorMuon / Muon+: this lane's row sum of U^2 over the
      // tile's columns, of the values as stored (bf16).
      float rsq = 0.0f;

#pragma unroll 1
      for (int cc = 0; cc < kBN / 32; ++cc) {
        const int c0 = tc.tn * kBN + cc * 32;
        if (c0 >= n_out) break;  // warp-uniform
        uint4 cur[4], curw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          cur[q] = pf[q];
          curw[q] = pw[q];
        }
        if (cc + 1 < kBN / 32) {
          prefetch_aux32(aux, C.ld_aux, r, c0 + 32, rows_out, n_out, use_aux, pf);
          prefetch_aux32(wbase, fin ? R.cols : 0, r, c0 + 32, rows_out, n_out, w_pf, pw);
        }
        uint32_t raw[32];
        tmem_ld_32x32b_x32(t_row + cc * 32, raw);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
        const bool row_ok = r < rows_out;
        const bool full_cols = c0 + 32 <= n_out;

        if (apply && p.final_update) {
          // Last Newton-Schulz step: U = sc (a X + P X) goes straight into
          // the parameter update; X' is not stored.
          float u[32];
          if (row_ok) {
            const int64_t aoff = static_cast<int64_t>(r) * C.ld_aux + c0;
            if (full_cols) {
              float x[32];
              unpack_bf16x32(cur, x);
#pragma unroll
              for (int j = 0; j < 32; ++j) u[j] = sc * (p.a * x[j] + v[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                u[j] = c0 + j < n_out ? sc * (p.a * __bfloat162float(aux[aoff + j]) + v[j]) : 0.0f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) u[j] = 0.0f;
          }
          if (row_ok) {
            const int nvalid = n_out - c0 < 32 ? n_out - c0 : 32;
            update_w32(R, R.elem0 + static_cast<int64_t>(r) * R.cols + c0, nvalid, u,
                       p.cautious, w_pf && full_cols ? &curw : nullptr);
          }
          continue;
        }
        if (apply) {
          if (row_ok) {
            if (full_cols) {
              float x[32];
              unpack_bf16x32(cur, x);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = sc * (p.a * x[j] + v[j]);
            } else {
              const int64_t aoff = static_cast<int64_t>(r) * C.ld_aux + c0;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c0 + j < n_out) v[j] = sc * (p.a * __bfloat162float(aux[aoff + j]) + v[j]);
            }
            if (p.row_sums) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float q = __bfloat162float(__float2bfloat16_rn(v[j]));
                if (c0 + j < n_out) rsq += q * q;
              }
            }
          }
        } else if (p.kind == GEMM_POLY) {
          if (row_ok) {
            const int64_t aoff = static_cast<int64_t>(r) * C.ld_aux + c0;
            if (full_cols) {
              float x[32];
              unpack_bf16x32(cur, x);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = p.b * x[j] + p.c * v[j];
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c0 + j < n_out) v[j] = p.b * __bfloat162float(aux[aoff + j]) + p.c * v[j];
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= sc;
        }

        // Store through shared memory and TMA (rows and columns outside the
        // output are dropped by the tensor map). A symmetric output (gram,
        // poly) holds the upper block triangle only: the chunk on the diagonal
        // (c0 == r0) is stored whole, a chunk above it (c0 > r0) is stored and
        // mirrored to rows c0.., columns r0..; chunks below it are the mirror
        // images of chunks stored by the warp that owns rows c0...
        const bool direct = apply || c0 >= r0;
        const bool mirror = !apply && c0 > r0;
        if (!direct || r0 >= rows_out) continue;  // warp-uniform
        uint8_t* bd = obuf + (staged & 1u) * (2 * kOutBoxBytes);
        uint8_t* bm = bd + kOutBoxBytes;
        // The stores issued from this buffer two chunks ago have read it.
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        {
          // Row `lane` of the box: 16-byte piece q goes to slot q ^ ((lane >> 1) & 3).
          const uint32_t swz = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            u.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
            u.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
            u.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
            u.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
            *reinterpret_cast<uint4*>(bd + lane * 64 + ((static_cast<uint32_t>(q) ^ swz) << 4)) = u;
          }
        }
        if (mirror) {
          // Element (r0 + lane, c0 + j) is row j, column lane of the mirror box.
          const uint32_t piece = static_cast<uint32_t>(lane) >> 3;
          const uint32_t within = (static_cast<uint32_t>(lane) & 7u) << 1;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t slot = piece ^ ((static_cast<uint32_t>(j) >> 1) & 3u);
            *reinterpret_cast<bf16*>(bm + j * 64 + (slot << 4) + within) =
                __float2bfloat16_rn(v[j]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&C.tmOut, bd, c0, r0, tc.view);
          if (mirror) tma_store_3d(&C.tmOut, bm, r0, c0, tc.view);
          bulk_commit();
        }
        ++staged;
      }
      if (p.row_sums && r < rows_out) {
        float* rp = C.vrec[tc.view].rowpart;
        if (rp != nullptr) rp[static_cast<int64_t>(tc.tn) * rows_out + r] = rsq;
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
      t = t_next;
    }
    // Every TMA store of this warp has landed before the kernel ends.
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // Neither CTA of the pair leaves while the other may still multicast into
  // its shared memory or arrive on its barriers.
  tc_fence_before();
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

size_t gemm_smem_bytes() {
  // 1 KB alignment slack, operand ring, epilogue staging, mbarriers (stage
  // full/empty, two accumulators full/empty, drain, pair and local tile
  // rings full/empty), then the TMEM address, the abort flag and the two
  // rings' slots.
  return 1024 + kStages * (kStageABytes + kStageBBytes) + 4 * kOutWarpBytes +
         (2 * kStages + 5 + 4 * kTileRing) * sizeof(uint64_t) + 2 * sizeof(uint32_t) +
         2 * kTileRing * sizeof(uint32_t);
}
static_assert(1024 + kStages * (kStageABytes + kStageBBytes) + 4 * kOutWarpBytes +
                  (2 * kStages + 5 + 4 * kTileRing) * 8 + 8 + 8 * kTileRing <= 232448,
              "GEMM shared memory exceeds the 227 KB a CTA may use");

// Maximum number of co-resident CTA pairs on the current device (GPCs with an
// odd number of free SMs leave one SM out), cached per device.
int gemm_max_pairs(int dev, int num_sms) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, ns_gemm_kernel<kModeKK>, &cfg) != cudaSuccess ||
      clusters <= 0) {
    (void)cudaGetLastError();
    clusters = num_sms / 2;
  }
  cache[dev] = clusters;
  return clusters;
}

cudaError_t launch_ns_gemm(const GemmParams& p, int num_sms, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  int modes = 0;
  for (int c = 0; c < p.num_classes; ++c) {
    if (p.cls[c].mode < 0 || p.cls[c].mode >= kGemmModes) return cudaErrorInvalidValue;
    modes |= 1 << p.cls[c].mode;
  }
  if (p.tile_counter == nullptr || p.next_counter == nullptr) return cudaErrorInvalidValue;
  // One instantiation per set of operand modes a stage can contain: gram
  // {KK, MM}, poly {KK}, apply {KK, KM}, each mode alone or with the other.
  using Kernel = void (*)(GemmParams);
  static constexpr Kernel kKernels[8] = {
      nullptr, ns_gemm_kernel<kModeKK>, ns_gemm_kernel<kModeKM>, ns_gemm_kernel<kModeKK | kModeKM>,
      ns_gemm_kernel<kModeMM>, ns_gemm_kernel<kModeKK | kModeMM>, nullptr, nullptr};
  const Kernel kernel = kKernels[modes];
  if (kernel == nullptr) return cudaErrorInvalidValue;
  const size_t smem = gemm_smem_bytes();
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    for (Kernel k : kKernels) {
      if (k == nullptr) continue;
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    configured_device = dev;
  }
  const int64_t max_pairs = gemm_max_pairs(dev, num_sms);
  const int64_t pairs = p.total_tiles < max_pairs ? p.total_tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mh
