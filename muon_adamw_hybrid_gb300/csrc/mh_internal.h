// Internal host/device interface of libmuonhybrid: the launch records the host
// planner fills and the kernels read from their parameter space. Not part of
// the public ABI (see include/muonhybrid.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mh {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// Elementwise passes (prologue, NorMuon/Muon+ statistics, apply, copy-out).
// One record per tensor; all views of a tensor share one shape and therefore
// one Newton-Schulz shape class, and occupy consecutive class slots.
// ---------------------------------------------------------------------------
constexpr int kEwTileR = 32;   // tile rows (stored orientation)
constexpr int kEwTileC = 256;  // tile cols (stored orientation): 8 per lane
constexpr int kProTileC = 256; // prologue tile cols: 8 per lane
constexpr int kProChunk = 8192;  // prologue chunk of a flat (wide) view: 32 per thread
constexpr int kEwThreads = 256;
constexpr int kMaxJobs = 64;   // tensors per elementwise launch (param space)

// Per-view record written by the prologue and read by the final Newton-Schulz
// apply when it applies the parameter update itself (no NorMuon / Muon+).
struct ViewRec {
  void* param;          // tensor base
  const void* grad;     // tensor base
  int64_t elem0;        // first element of this view
  int64_t rows, cols;   // stored view
  float lr, wd, shape_scale;
  int32_t pdt, gdt;
  int32_t tall;
  int32_t vec;          // param and grad 16-byte aligned and cols % 8 == 0
  int32_t psr;          // bf16 parameter written stochastically rounded
  uint32_t psr_key;     // its rounding key
  int32_t inactive;     // zero gradient under the inactive-expert rule: leave it alone
  int32_t stat_tiles_c; // 256-column tiles of the row statistics
  float* rowpart;       // [stat_tiles_c][rows] partial row sums of U^2 of this view, or
                        // null; written by the last Newton-Schulz apply stage
};

struct EwJob {
  const void* src;       // prologue: gradient (Muon) or input x (NS only)
  void* mom;             // Muon momentum (mom_dtype), null for NS only
  void* dst;             // apply: parameter; copy-out: NS output
  float* sm;             // NorMuon second moment (views*rows)
  float* tile_ss;        // per prologue tile and warp: partial ||Q||^2 (this tensor's first)
  float* rowpart;        // [views][tiles_c][rows] partial row sums of U^2
  float* colpart;        // [views][tiles_r][cols] partial col sums of (f U)^2
  float* rowfac;         // [views][rows] final row factor
  float* colfac;         // [views][cols] final col factor
  bf16* x0;              // NS input buffer: first view of this tensor
  const bf16* xf;        // NS output buffer: first view of this tensor
  const double* sumsq;   // per view ||Q||_F^2 (first view of this tensor)
  ViewRec* vrec;         // per view record (first view of this tensor), or null
  int64_t rows, cols, views;
  int64_t ldx;           // leading dimension of the X buffers (elements)
  int64_t x_view_stride; // elements between views in the X buffers
  int64_t tile_begin;    // first global tile index of this tensor
  int32_t tiles_r, tiles_c;
  int32_t stat_tiles_c;  // 256-column tiles of the row statistics (tiles_c of the stats passes)
  int32_t tall;          // unused by the kernels (X is always in stored layout)
  int32_t flat;          // prologue: wide view stored like X (cols % 8 == 0): streamed
                         // as contiguous kProChunk-element chunks, tiles_r = 1
  int32_t src_dtype, dst_dtype;
  int32_t src_vec, dst_vec, mom_vec;  // 16-byte aligned and cols % 4 == 0
  float lr, wd, shape_scale;
  int32_t mom_dtype;     // momentum: MH_F32, or MH_BF16 stored stochastically rounded
  int32_t param_sr;      // bf16 parameter written stochastically rounded
  uint32_t mom_key, param_key;  // rounding keys (momentum, parameter streams)
  const int32_t* active;  // per view: 1 if its gradient has a nonzero entry; null: all active
};

struct EwParams {
  EwJob jobs[kMaxJobs];
  int32_t njobs;
  int64_t total_tiles;
  // hyperparameters
  float mu;
  int32_t nesterov;
  int32_t use_momentum;  // 0: NS only (Q = x)
  int32_t cautious;
  int32_t use_rowfac, use_colfac;
  float ns_eps;
  float ns_norm_scale;         // X0 = Q / (||Q|| * ns_norm_scale + ns_eps)
  int32_t u_scale_from_sumsq;  // ns_steps == 0: U = X0
  const float* grad_mult;      // device: gradients are read as g * (*grad_mult), or null
  const int32_t* skip;         // device: *skip != 0 -> the kernel returns at once, or null
  int* status;                 // device status word for bounded-wait timeouts, or null:
                               // the streaming apply / column-statistics kernel runs only
                               // with one (its waits report through it)
  long long wait_limit;        // cycles a bounded wait may take before the launch aborts
};

// 1 / (||Q|| * norm_scale + eps), or 0 for a zero matrix with eps 0.
__host__ __device__ __forceinline__ float ns_inv_norm(double sumsq, float norm_scale, float eps) {
  const float den = sqrtf(static_cast<float>(sumsq)) * norm_scale + eps;
  return den > 0.0f ? 1.0f / den : 0.0f;
}

// True when a gradient-control block asks the step to write nothing.
__device__ __forceinline__ bool step_skipped(const int32_t* skip) {
  return skip != nullptr && *skip != 0;
}

enum EwKind {
  EW_PROLOGUE = 0,       // transposing 32 x 256 tiles (tall views, ragged wide views)
  EW_ROWSQ = 1,
  EW_COLSQ = 2,
  EW_APPLY = 3,
  EW_COPYOUT = 4,
  EW_PROLOGUE_FLAT = 5,  // contiguous chunks (wide views with cols % 8 == 0)
  EW_APPLY_CU = 6,       // EW_APPLY with the cautious-update mask (reads the gradient);
                         // chosen by launch_elementwise, never planned on its own
  EW_PROLOGUE_FLAT_B16 = 7  // EW_PROLOGUE_FLAT when every job keeps bf16 momentum: a leaner
                            // instantiation at three blocks per SM; chosen by launch_elementwise
};
constexpr int kEwKinds = 8;

// Row finalisation (NorMuon state, NorMuon norm restore, Muon+ row factor):
// one CTA per view. Every reduction sums per-tile partials in a fixed order,
// so a step is bitwise reproducible.
struct RowFinJob {
  float* sm;
  float* rowpart;        // [views][tiles_c][rows]; slot tc = 0 reused for row sums
  float* rowfac;
  int64_t rows, cols, views, tiles_c;
  int64_t view_begin;  // prefix over views
  const int32_t* active;  // per view, or null (see EwJob)
};
constexpr int kMaxRowFinJobs = 96;
struct RowFinParams {
  RowFinJob jobs[kMaxRowFinJobs];
  int32_t njobs;
  int64_t total_views;
  int32_t normuon, muon_plus;
  float beta2, plus_eps;
  float normuon_eps;     // floor of the NorMuon second moment inside the rsqrt
  const int32_t* skip;   // gradient control: return at once when set, or null
};

// Column finalisation (Muon+ column factor 1/sqrt(sum + eps)), one thread per
// (view, column).
struct ColFinJob {
  const float* colpart;  // [views][tiles_r][cols]
  float* colfac;         // [views][cols]
  int64_t cols, views, tiles_r;
  int64_t elem_begin;    // prefix over views*cols
};
constexpr int kMaxColFinJobs = 96;
struct ColFinParams {
  ColFinJob jobs[kMaxColFinJobs];
  int32_t njobs;
  int64_t total;
  float plus_eps;
  const int32_t* skip;
};

// Per-view ||Q||_F^2 from the prologue's per-tile partials, one warp per view.
struct NormJob {
  const float* tile_ss;   // this tensor's first per-warp partial
  double* sumsq;          // this tensor's first view
  int64_t tiles_per_view, views;
  int64_t view_begin;
};
constexpr int kMaxNormJobs = 96;
struct NormParams {
  NormJob jobs[kMaxNormJobs];
  int32_t njobs;
  int64_t total_views;
  const int32_t* skip;
};

// Inactive-expert rule: per view of a flagged tensor, whether its gradient
// has any nonzero entry (chunks of a view already known active are skipped).
constexpr int kMaxActiveJobs = 256;
constexpr int64_t kActiveChunk = 8192;
struct ActiveJob {
  const void* grad;
  int32_t* active;       // this tensor's first view
  int64_t view_elems, views;
  int64_t chunk_begin;   // global chunk index of this tensor's first chunk
  int32_t gdt;
  int32_t vec;           // 16-byte aligned and view_elems % 8 == 0
};
struct ActiveParams {
  ActiveJob jobs[kMaxActiveJobs];
  int32_t njobs;
  int64_t total_chunks;
};
cudaError_t launch_view_active(const ActiveParams& p, int num_sms, cudaStream_t s);

cudaError_t launch_elementwise(EwKind kind, const EwParams& p, int num_sms, cudaStream_t s);

// Tensor map over `views` stacked (rows x inner) matrices of row pitch `ld`
// elements (bf16, or fp32 when `f32`), box 256 x 32 x 1, no swizzle, zero
// fill: the tiles of the streaming elementwise passes. False if the driver
// cannot encode it (the caller then takes the register-staged kernel).
bool encode_stream_map(CUtensorMap* tm, const void* base, bool f32, int64_t inner, int64_t rows,
                       int64_t views, int64_t ld);
cudaError_t launch_row_finalize(const RowFinParams& p, cudaStream_t s);
cudaError_t launch_col_finalize(const ColFinParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_view_norm(const NormParams& p, cudaStream_t s);

// ---------------------------------------------------------------------------
// Grouped Newton-Schulz GEMM stage: one persistent launch covers every view
// of up to kMaxClasses shape classes.
// ---------------------------------------------------------------------------
constexpr int kBM = 128;  // tile rows (TMEM lanes)
constexpr int kBN = 256;  // tile cols (MMA N)
constexpr int kBK = 64;   // k per stage: one 128-byte swizzle atom of bf16
constexpr int kStages = 4;
constexpr int kMaxClasses = 8;
constexpr int kGemmThreads = 256;

enum GemmKind { GEMM_GRAM = 0, GEMM_POLY = 1, GEMM_APPLY = 2 };

// Operand major-ness of one shape class in one stage (A, B): K-major (K) or
// MN-major (M). The gram of a tall view reads both operands as MN-major
// chunks of T; the apply reads X MN-major as B, except for tall views (T P:
// both K-major); every other stage is K-major. One launch per stage covers
// classes of every mode: the kernel selects a mode-specialised k-loop once
// per tile.
enum GemmMode { GEMM_MODE_KK = 0, GEMM_MODE_KM = 1, GEMM_MODE_MM = 2 };
constexpr int kGemmModes = 3;
inline int gemm_mode(int kind, bool tstore) {
  if (kind == GEMM_GRAM) return tstore ? GEMM_MODE_MM : GEMM_MODE_KK;
  if (kind == GEMM_APPLY) return tstore ? GEMM_MODE_KK : GEMM_MODE_KM;
  return GEMM_MODE_KK;
}

struct GemmClass {
  CUtensorMap tmA;         // operand A: rows of X (gram), A (poly), P or T (apply);
                           //   K-major box 64 x 128, or MN-major 64 x 64 chunks of T (gram, tstore)
  CUtensorMap tmB;         // operand B: 128 of the 256 B rows per CTA of a pair: X (gram),
                           //   A (poly), P (apply, tstore) K-major; X (apply) or T
                           //   (gram, tstore) as MN-major 64 x 64 chunks
  CUtensorMap tmOut;       // output (A, P or X'): 32 x 32 boxes, 64-byte swizzle, stored
                           //   by the epilogue from shared memory
  bf16* out;               // output base (first view of the class)
  const bf16* aux;         // poly: A (b*A term); apply: X (a*X term)
  const double* sumsq;     // per view sum of squares of Q (first iteration only)
  const ViewRec* vrec;     // per view records (final update only)
  int64_t out_view_stride, aux_view_stride;  // elements
  int64_t ld_out, ld_aux;                     // elements
  int32_t m, n;            // Newton-Schulz orientation (m <= n)
  int32_t tstore;          // X is kept in its stored (n x m) layout T = X^T: the gram
                           // reads T with MN-major operands (A = T^T T) and the apply
                           // computes T' = a T + T P
  int32_t out_rows, out_cols;  // apply output (m x n, or n x m when tstore)
  int32_t views;
  int32_t tiles_m, tiles_n, tiles_per_view;  // in 256 x 256 pair blocks
  int32_t K;               // contraction length
  int32_t mode;            // GemmMode of this class in this stage
  int64_t tile_begin;      // first global pair-block index of this class
};

// Work distribution: CTA 0 of each pair claims the next 256 x 256 block from
// a per-launch counter in the workspace header and hands its index to both
// CTAs' roles through a ring of kTileRing shared-memory slots. The header
// holds kTileCounters counters; launch k of a call claims from counter
// k mod kTileCounters and zeroes counter k + 2 for a later launch (a launch
// reads global memory only after the launch before it has completed, so the
// reset lands before that launch's first claim).
constexpr int kTileRing = 4;
constexpr int kTileCounters = 32;
constexpr int kTileCounterOffset = 64;  // bytes into the workspace header

struct GemmParams {
  GemmClass cls[kMaxClasses];
  int32_t num_classes;
  int32_t kind;            // GemmKind
  int32_t first_iter;      // fold the Frobenius normalisation in
  int32_t final_update;    // apply: update the parameters instead of writing X'
  int32_t row_sums;        // last apply: also write each view's partial row sums of U^2
  int32_t cautious;        // MH_CAUTIOUS_* for the final update
  int64_t total_tiles;
  float a, b, c, eps;
  float norm_scale;        // first iteration: X0 = Q / (||Q|| * norm_scale + eps)
  int* status;             // device status word (bounded-wait timeouts)
  const int32_t* skip;     // gradient control: every thread returns at once when set
  uint32_t* tile_counter;  // this launch's block counter (zero at launch)
  uint32_t* next_counter;  // the counter of the launch after the next one: zeroed here
  long long wait_limit;    // cycles a bounded wait may take before the launch aborts
};

// Cycles a bounded wait in a GEMM stage may take before the launch gives up
// (mh_set_wait_limit; default kWaitLimitCycles).
long long gemm_wait_limit();

size_t gemm_smem_bytes();
// Launches one persistent grid of CTA pairs (clusters of two), at most one
// pair per two SMs that can hold a cluster.
cudaError_t launch_ns_gemm(const GemmParams& p, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------
// AdamW
// ---------------------------------------------------------------------------
constexpr int kMaxAdamJobs = 160;
constexpr int64_t kAdamChunk = 16384;  // elements per work item

struct AdamJob {
  void* param;
  const void* grad;
  void* m;               // first moment, sdt
  void* v;               // second moment, sdt
  int64_t numel;
  int64_t chunk_begin;
  int32_t pdt, gdt;
  int32_t vec;  // all four pointers 16-byte aligned
  float lr, wd;  // lr already multiplied by lr_mult
  int32_t sdt;   // moments: MH_F32, or MH_BF16 stored stochastically rounded
  int32_t psr;   // bf16 parameter written stochastically rounded
  int64_t tindex;  // index of the tensor in the call (its rounding streams)
};

struct AdamParams {
  AdamJob jobs[kMaxAdamJobs];
  int32_t njobs;
  int64_t total_chunks;
  float beta1, beta2, eps;
  float inv_bc1, inv_sqrt_bc2;  // 1/(1-b1^t), 1/sqrt(1-b2^t), when step is null
  const float* grad_mult;       // device: gradients read as g * (*grad_mult), or null
  const int32_t* skip;          // device: write nothing when set, or null
  const int64_t* step;          // device: bias-correction count t, or null (use the above)
  uint64_t sr_seed;             // stochastic-rounding seed when step is null (the host step)
};

cudaError_t launch_adamw(const AdamParams& p, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------
// Gradient control: global norm of the unscaled gradients, clip factor and
// overflow skip (one pass over every gradient, then a one-block finalise).
// ---------------------------------------------------------------------------
constexpr int kMaxGradJobs = 512;
constexpr int64_t kGradChunk = 65536;  // elements per partial sum

struct GradJob {
  const void* grad;
  int64_t numel;
  int64_t chunk_begin;   // global index of this tensor's first chunk
  int32_t gdt;
  int32_t vec;           // 16-byte aligned
};

struct GradParams {
  GradJob jobs[kMaxGradJobs];
  int32_t njobs;
  int64_t chunk_first;   // first global chunk of this launch
  int64_t nchunks;       // chunks in this launch
  float inv_scale;
  double* partial;       // [all chunks] sum of u^2, NaN if the chunk holds inf/NaN
};

struct GradFinParams {
  const double* partial;
  int64_t nchunks;
  double inv_scale, max_norm, clip_eps;
  float* mult;
  int32_t* skip;
  double* norm;
  int64_t* step;
};

cudaError_t launch_grad_sumsq(const GradParams& p, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------
// QK-Clip: rows of query / key projections of heads past tau scaled by
// min(1, tau / s_h)^exponent.
// ---------------------------------------------------------------------------
constexpr int kMaxQkClipEntries = 256;
struct QkClipEntry {
  void* param;
  int64_t cols;
  int64_t head_stride, row_offset, scaled_rows;
  int64_t row_begin;     // prefix over entries of heads * scaled_rows
  int32_t head_index0;
  int32_t dt;
  int32_t vec;           // 16-byte aligned
  float exponent;
};
struct QkClipParams {
  QkClipEntry entries[kMaxQkClipEntries];
  int32_t nentries;
  int64_t total_rows;
  const float* s_max;    // device, per head
  float tau;
  const int32_t* skip;   // gradient control: clip nothing after a skipped step
};
cudaError_t launch_qk_clip(const QkClipParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_grad_finalize(const GradFinParams& p, cudaStream_t s);

// Sets the calling thread's message returned by mh_last_error().
void set_last_error(const char* msg);

}  // namespace mh
