/*
 * muonhybrid.h -- C ABI of the GB300 (sm_103a) hybrid Muon + AdamW optimizer step.
 *
 * What it computes (sources are the pages' titles and sections):
 *
 *   Muon, for every routed 2-D matrix and every declared matrix view
 *   (Speedtronic docs "v2 optimizers", sections "Newton-Schulz", "Muon update",
 *   "Muon+", "Cautious updates"; flaxchat "Optimizer", "Muon Algorithm";
 *   kimi-k3 "Optimization", "A tensor's storage shape can be misleading"):
 *
 *       B <- mu*B + (1-mu)*G                       momentum (fp32, or bf16 rounded
 *                                                  stochastically)
 *       Q <- lerp(G, B, mu) = G + mu*(B - G)        Nesterov form (else Q = B)
 *       X <- T / (||T||_F * norm_scale + eps),  T = Q^T if rows > cols else Q
 *       repeat ns_steps:  A = X X^T;  X <- a X + (b A + c A^2) X
 *                         (one (a, b, c) for every iteration, or a schedule)
 *       U <- X^T if rows > cols else X
 *       [NorMuon per-row second moment]  [Muon+ row_col]
 *       W <- (1 - lr*wd) W - lr * s * U   (or a cautious form), s = max(1, rows/cols)^0.5
 *                                          (or the Moonlight factor: MH_SHAPE_*)
 *
 *   AdamW for everything else (dew.training.optim "OPTIMIZER_MAP" names
 *   optax.adamw; Speedtronic "CPU/CUDA/MPS behavior" names PyTorch's fused
 *   AdamW): standard decoupled AdamW with bias correction.
 *
 * Conventions shared by every entry point:
 *   - All pointers to tensors are DEVICE pointers into memory the caller owns
 *     (parameters, gradients, optimizer state, workspace). The library never
 *     allocates device memory in these calls and keeps no pointer after the
 *     call returns. A pointer may also be host memory that the device reads
 *     at the same address (page-locked and mapped, or coherent system memory
 *     on a Grace-Blackwell system): the kernels then stream it over the
 *     host link, with no separate copy. mh_pointer_device_accessible tells
 *     whether a pointer qualifies.
 *   - Tensors are contiguous and row-major. A Muon tensor with views = k is
 *     k independent rows x cols matrices stored back to back, i.e. the array
 *     (k*rows, cols); its momentum buffer has the same layout.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued on it; nothing synchronises the host.
 *   - Arguments are checked on the host before anything is enqueued. A failed
 *     check returns a non-zero mh_status, enqueues nothing, and leaves a
 *     message for mh_last_error(). A CUDA launch error returns MH_ECUDA.
 *   - Supported dtypes are fp32 and bf16. Anything else (complex, sparse
 *     layouts, fp16, fp64) is rejected with MH_EDTYPE; the pages require a
 *     clear error for sparse and complex gradients.
 *   - Calls are thread-safe as long as concurrent calls use distinct
 *     workspaces; the error message is per host thread.
 */
#ifndef MUONHYBRID_H
#define MUONHYBRID_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MH_OK = 0,
  MH_EINVAL = 1,       /* null pointer, bad count, bad hyperparameter */
  MH_EDTYPE = 2,       /* unsupported dtype (complex/sparse/fp16/fp64...) */
  MH_ESHAPE = 3,       /* non-positive or too large dimension */
  MH_EWORKSPACE = 4,   /* workspace null, too small or misaligned */
  MH_ECUDA = 5,        /* a CUDA runtime call or launch failed */
  MH_EUNSUPPORTED = 6, /* valid request this build does not handle */
  MH_ETIMEOUT = 7      /* a device-side bounded wait gave up (see mh_workspace_status) */
} mh_status;

typedef enum { MH_F32 = 0, MH_BF16 = 1 } mh_dtype;

/* Cautious variants (both from the pages; 0 = off).
 *   MH_CAUTIOUS_WD     flaxchat "Muon Algorithm" step 4: the mask gates the
 *                      weight decay only and keeps entries with
 *                      update*param >= 0.
 *   MH_CAUTIOUS_UPDATE Speedtronic "Cautious updates": the mask gates the
 *                      whole observed update (decay included) and keeps
 *                      entries with update*gradient > 0. */
enum { MH_CAUTIOUS_OFF = 0, MH_CAUTIOUS_WD = 1, MH_CAUTIOUS_UPDATE = 2 };

/* Shape factor s of the update W <- (1 - lr wd) W - lr s U, from the rows
 * and cols of the stored view (mh_muon_hparams.shape_rule):
 *   MH_SHAPE_RATIO      Speedtronic "Muon update": s = max(1, rows/cols)^0.5.
 *   MH_SHAPE_MOONLIGHT  kimi-k3 "Why treat a matrix differently?" names the
 *                       Moonlight shape factor as its trainer's default but
 *                       its formula did not survive on the page; read as the
 *                       published Moonlight rule s = 0.2 sqrt(max(rows, cols)),
 *                       which gives a full-rank U with unit singular values an
 *                       RMS of 0.2. */
enum { MH_SHAPE_RATIO = 0, MH_SHAPE_MOONLIGHT = 1 };

/* One Muon-routed parameter (a 2-D matrix or a stack of `views` matrices). */
typedef struct {
  void* param;            /* (views*rows, cols), param_dtype, updated in place */
  const void* grad;       /* (views*rows, cols), grad_dtype, read only */
  void* momentum;         /* (views*rows, cols) momentum_dtype, updated in place */
  float* normuon_sm;      /* (views*rows) fp32 NorMuon second moment, updated in
                             place; required when hparams.normuon != 0, else
                             ignored (may be NULL). Zero-initialise it. */
  int32_t param_dtype;    /* mh_dtype */
  int32_t grad_dtype;     /* mh_dtype */
  int64_t views;          /* >= 1: independent matrices in the tensor */
  int64_t rows;           /* rows of one view (>= 1) */
  int64_t cols;           /* cols of one view (>= 1) */
  float lr_mult;          /* this tensor's lr = hparams.lr * lr_mult */
  float wd;               /* this tensor's decoupled weight decay */
  int32_t momentum_dtype; /* MH_F32 (0, default) or MH_BF16: bf16 state, updated in fp32
                             and written back stochastically rounded (below) */
  int32_t param_sr;       /* 1: a bf16 param is written stochastically rounded
                             instead of to nearest even (bf16 params only) */
  int32_t skip_zero_grad; /* 1: inactive-expert rule (kimi-k3 "Optimization", "One more
                             kind of state: which experts learn?"): a view whose
                             gradient is zero everywhere keeps its parameter,
                             momentum and NorMuon state unchanged. Costs one read
                             of the gradients of silent views (a chunk for others). */
} mh_muon_tensor;

/* Muon hyperparameters shared by one call. Defaults from the pages:
 * momentum 0.95 with Nesterov, ns_steps 5, (a,b,c) = (3.4445, -4.7750, 2.0315),
 * eps 1e-7 (Speedtronic "Newton-Schulz"). */
typedef struct {
  float lr;
  float momentum;     /* mu in [0, 1) */
  int32_t nesterov;   /* 1: Q = lerp(G, B, mu); 0: Q = B */
  float eps;          /* Frobenius-normalisation guard, >= 0 */
  int32_t ns_steps;   /* 0..16 quintic iterations */
  float a, b, c;      /* quintic coefficients */
  int32_t normuon;    /* 1: NorMuon per-row second moment (flaxchat step 3) */
  float beta2;        /* NorMuon EMA coefficient, in [0, 1) */
  int32_t muon_plus;  /* 1: Muon+ row_col normalisation (Speedtronic "Muon+") */
  float plus_eps;     /* Muon+ eps inside each square root, > 0 */
  int32_t cautious;   /* MH_CAUTIOUS_* */
  /* Gradient control written by mh_grad_prepare (both DEVICE pointers, read
   * by the kernels of this call, NULL = off): */
  const float* grad_mult;  /* every gradient element is read as g * (*grad_mult) */
  const int32_t* skip;     /* when *skip != 0 the call writes nothing at all */
  uint64_t sr_seed;        /* stochastic-rounding seed of this call, e.g. the step count */
  /* Polar Express form (flaxchat "Muon Algorithm" step 2): one (a, b, c) per
   * iteration and X = Q / (||Q||_F * norm_scale + eps), e.g. norm_scale 1.01
   * with eps 0. */
  const float* coeff_schedule;  /* HOST array of ns_steps x 3 floats (a, b, c of each
                                   iteration in order), or NULL: (a, b, c) above every time */
  float norm_scale;             /* > 0; 0 means 1 (the Speedtronic form) */
  /* Parameter-write fence: a cudaEvent_t, or NULL for none. The call makes its
   * stream wait for this event (cudaStreamWaitEvent) just before its first
   * kernel that writes a parameter -- the last Newton-Schulz apply stage, or
   * the separate apply when NorMuon or Muon+ is on -- and not before. Work
   * the caller ordered before recording the event on another stream (e.g. a
   * device-to-host copy of the previous step's parameters) thus runs
   * alongside this call's momentum, normalisation and Newton-Schulz kernels
   * and still finishes before any parameter changes; everything enqueued on
   * the stream after this call is ordered after the wait as well. The event
   * is only waited on, never recorded or destroyed by the library. */
  void* param_fence;
  /* Step phase (MH_STEP_*). A step may be split into two calls on the same
   * stream with the same tensors, hyperparameters (but for this field) and
   * workspace, the second enqueued after the first:
   *   MH_STEP_GRADIENTS clears the workspace status and runs every kernel
   *                     that reads the gradients (inactive-expert scan,
   *                     momentum / Nesterov prologue, Frobenius norms);
   *   MH_STEP_FINISH    runs the Newton-Schulz stages and the update, reading
   *                     only the momentum, the parameters and the workspace
   *                     (and the gradients again with MH_CAUTIOUS_UPDATE,
   *                     whose mask compares the update with the gradient).
   * Between the two the caller may enqueue work that must follow the last
   * gradient read: reuse of the gradient buffers, or a copy-out of the
   * previous step's parameters that should not compete with the gradient
   * reads for host memory. param_fence applies to MH_STEP_FINISH and
   * MH_STEP_ALL. */
  int32_t phase;
  /* NorMuon floor (flaxchat "Muon Algorithm" step 3): each row is scaled by
   * 1/sqrt(max(second moment, normuon_eps)). >= 0, finite; 0 means 1e-10.
   * (The Frobenius-norm restore that follows divides by the norm after the
   * row scaling, floored at 1e-10 against division by zero.) */
  float normuon_eps;
  /* Shape factor of the update (MH_SHAPE_*); 0 is the Speedtronic ratio rule. */
  int32_t shape_rule;
} mh_muon_hparams;

enum { MH_STEP_ALL = 0, MH_STEP_GRADIENTS = 1, MH_STEP_FINISH = 2 };

/* Bytes of device workspace mh_muon_step_batched needs for these tensors and
 * flags (256-byte aligned pointer required). Returns 0 and sets the error
 * message when the arguments are invalid. Host-only; touches no device. */
size_t mh_muon_workspace_bytes(const mh_muon_tensor* tensors, int32_t n,
                               const mh_muon_hparams* hp);

/* The batched Muon update over all `n` tensors and all their views, in one
 * stream-ordered sequence: a fused momentum/Nesterov/norm prologue, one
 * grouped tcgen05 GEMM launch per Newton-Schulz stage over every view of
 * every shape, and a fused NorMuon/Muon+/cautious/decay/apply epilogue.
 * Views whose rows*cols is zero are skipped; n = 0 is a no-op.
 * The workspace's previous contents do not matter. */
int mh_muon_step_batched(const mh_muon_tensor* tensors, int32_t n, const mh_muon_hparams* hp,
                         void* workspace, size_t workspace_bytes, void* stream);

/* One Newton-Schulz problem: U = NS(X) for each of `views` rows x cols
 * matrices (Speedtronic "Newton-Schulz": tall matrices are transposed
 * internally, normalised by ||X||_F + eps, iterated, transposed back; a zero
 * matrix stays zero). x and out may not overlap. */
typedef struct {
  const void* x;      /* (views*rows, cols) in in_dtype */
  void* out;          /* (views*rows, cols) in out_dtype */
  int32_t in_dtype;   /* mh_dtype */
  int32_t out_dtype;  /* mh_dtype */
  int64_t views, rows, cols;
} mh_ns_problem;

size_t mh_ns_workspace_bytes(const mh_ns_problem* problems, int32_t n);

/* Batched Newton-Schulz only, with bf16 operands and fp32 accumulation. */
int mh_newton_schulz_batched(const mh_ns_problem* problems, int32_t n, int32_t steps, float a,
                             float b, float c, float eps, void* workspace,
                             size_t workspace_bytes, void* stream);

/* mh_newton_schulz_batched with one (a, b, c) per iteration and the
 * normalisation X = X0 / (||X0||_F * norm_scale + eps) (flaxchat "Muon
 * Algorithm" step 2, Polar Express: norm_scale 1.01, eps 0): `coeffs` is a HOST
 * array of steps x 3 floats, read during the call. norm_scale > 0, eps >= 0;
 * a zero matrix stays zero. Same workspace as mh_newton_schulz_batched. */
int mh_newton_schulz_batched_ex(const mh_ns_problem* problems, int32_t n, int32_t steps,
                                const float* coeffs, float eps, float norm_scale,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Size of the fixed scratch array behind mh_newton_schulz_batched_noalloc. */
#define MH_NS_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/* mh_newton_schulz_batched for callers that cannot allocate device memory.
 * None of the pages describes this entry point; it exists for callers
 * that have no way to provide a workspace -- for example a plugin that its
 * host application gives only input and output buffers, or a program whose
 * device memory is already fully reserved by its own pool -- and so can
 * neither call cudaMalloc nor keep a scratch buffer between calls.
 * Same problems, arguments and results as mh_newton_schulz_batched, with the
 * workspace taken from a file-scope device array of
 * MH_NS_STATIC_SCRATCH_BYTES (64 MiB) inside the library instead of from
 * the caller; the call allocates nothing.
 *   - Requests whose mh_ns_workspace_bytes exceeds that size return
 *     MH_EWORKSPACE (with a message) before anything is enqueued.
 *   - Each GPU that loads the library holds its own array until exit.
 *   - All calls on one device share its array, which keeps the last call's
 *     contents (nothing stale is ever read: the status word is cleared and
 *     every other byte is written before use). Calls whose GPU work overlaps,
 *     e.g. on two unordered streams, race on the array: serialise them.
 *   - The first call on each device looks up the array's device address
 *     with that device current, and so does the first call after the
 *     device's context was destroyed (cudaDeviceReset); make that first call
 *     before any stream capture on the device. */
int mh_newton_schulz_batched_noalloc(const mh_ns_problem* problems, int32_t n, int32_t steps,
                                     float a, float b, float c, float eps, void* stream);

/* One AdamW-routed tensor, treated as a flat array of numel elements. */
typedef struct {
  void* param;            /* numel, param_dtype, updated in place */
  const void* grad;       /* numel, grad_dtype */
  void* exp_avg;          /* numel first moment (state_dtype), updated in place */
  void* exp_avg_sq;       /* numel second moment (state_dtype), updated in place */
  int32_t param_dtype;
  int32_t grad_dtype;
  int64_t numel;          /* >= 0 */
  float lr_mult;
  float wd;
  int32_t state_dtype;    /* MH_F32 (0, default) or MH_BF16 moments, stochastically rounded */
  int32_t param_sr;       /* 1: a bf16 param is written stochastically rounded */
} mh_adamw_tensor;

/* bf16 state (dew.training.optim "bf16_moments", "stochastic_round_bf16"):
 * the update reads the state widened to fp32, computes in fp32 exactly as for
 * fp32 state, and writes the new state rounded to bf16 up or down with the
 * probability of its distance to each: 16 noise bits are added below the kept
 * mantissa and the low half dropped. The noise of flat element i of a tensor
 * is the low (i even) or high (i odd) half of fmix32(key + floor(i/2)), with
 * key = fmix32(fmix32(fmix32(4*t + m) ^ seed_lo) ^ seed_hi): fmix32 the 32-bit
 * finaliser of MurmurHash3, all arithmetic mod 2^32, t the tensor's index in
 * the call, m = 0 for the momentum / first moment, 1 for the second moment, 2
 * for the parameter, seed_lo/hi the halves of the 64-bit seed. The seed is
 * hparams.sr_seed for Muon and the 1-based step count for AdamW. NaN stays
 * NaN. */

/* Fused multi-tensor AdamW step (step >= 1, the 1-based count used for bias
 * correction):
 *   m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2
 *   W <- W (1 - lr*wd) - lr * (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)
 * in fp32; bf16 parameters are rounded to nearest even on store, or
 * stochastically with param_sr, and bf16 moments stochastically (above). */
int mh_adamw_step(const mh_adamw_tensor* tensors, int32_t n, float lr, float beta1, float beta2,
                  float eps, int64_t step, void* stream);

/* ---- Gradient control ahead of both optimizer halves -------------------
 * kimi-k3 "Optimization", "Keep the arithmetic and gradients under control":
 * the global gradient norm is measured before the optimizer step; a positive
 * max_grad_norm clips it when needed, 0 disables clipping while the norm is
 * still observed; under FP16 a gradient scaler is used and an overflow skips
 * the whole hybrid update (Muon and AdamW). dew.training.optim
 * "build_optimizer": the clip reads every gradient of every group together.
 *
 * mh_grad_prepare reads every gradient once and leaves its decision in
 * device memory, so the step calls that follow (same stream) apply it
 * without a host round trip:
 *   u      = g * inv_loss_scale                     (unscaled gradient)
 *   norm   = sqrt(sum of u^2 over every element of every gradient)
 *   skip   = some u is inf or NaN
 *   mult   = skip ? 0 : inv_loss_scale * (max_norm > 0 ? min(1, max_norm / (norm + 1e-6)) : 1)
 *   step  += skip ? 0 : 1                           (when ctl->step != NULL)
 * The clip factor is PyTorch's clip_grad_norm_ definition. The sum of
 * squares is accumulated in fp32 within each thread's share of a
 * 65536-element chunk (at most 256 squares) and in fp64 across threads and
 * chunks, in a fixed order (bitwise reproducible). A finite
 * gradient whose square overflows fp32 (|u| > 1.8e19) gives norm = inf and
 * mult = 0, not a skip. */
typedef struct {
  const void* grad;   /* numel elements, grad_dtype, DEVICE */
  int32_t grad_dtype; /* mh_dtype */
  int64_t numel;      /* >= 0 */
} mh_grad_ref;

typedef struct {
  float* grad_mult;   /* DEVICE float: the factor above */
  int32_t* skip;      /* DEVICE int32: 1 when the step must be skipped, else 0 */
  double* norm;       /* DEVICE double: the global norm (NaN when skipping) */
  int64_t* step;      /* DEVICE int64 step count advanced on applied steps, or NULL */
} mh_grad_control;

/* Workspace bytes mh_grad_prepare needs (8 per 65536 gradient elements). */
size_t mh_grad_prepare_workspace_bytes(const mh_grad_ref* grads, int32_t n);

/* Computes the control block above for `n` gradients. inv_loss_scale > 0
 * and finite, max_norm >= 0. ctl->grad_mult, ctl->skip and ctl->norm must be
 * non-NULL. n = 0 gives norm 0, mult = inv_loss_scale, no skip. */
int mh_grad_prepare(const mh_grad_ref* grads, int32_t n, float inv_loss_scale, float max_norm,
                    const mh_grad_control* ctl, void* workspace, size_t workspace_bytes,
                    void* stream);

/* mh_adamw_step under a control block: gradients are read as g * (*grad_mult),
 * nothing is written when *skip != 0, and the bias-correction count t is read
 * on the device from *ctl->step (required, >= 1 once mh_grad_prepare has run). */
int mh_adamw_step_ctl(const mh_adamw_tensor* tensors, int32_t n, float lr, float beta1,
                      float beta2, float eps, const mh_grad_control* ctl, void* stream);

/* ---- QK-Clip after the update ---------------------------------------------
 * kimi-k3 "Optimization", "QK-Clip watches a different failure mode";
 * dew.training.optim "scale_by_qk_clip" (Kimi K2's MuonClip): each head h has
 * an observed maximum query-key score s_h (scaled by the square root of the
 * query-key dimension, maxed over microbatches by the caller). For s_h > tau,
 * selected rows of the head's query and key projections are multiplied by
 * gamma_h^exponent, gamma_h = tau / s_h; other heads are not touched. Give
 * query and key rows of a head exponents summing to 1 (0.5 each) so its
 * scores scale by gamma_h; an MLA rotary query whose key is shared takes 1.
 * One entry describes a weight stored (rows, cols) with one block of
 * head_stride rows per head, of which scaled_rows rows starting at
 * row_offset are scaled; several entries may name one weight (disjoint rows). */
typedef struct {
  void* param;            /* (rows, cols), param_dtype, DEVICE, scaled in place */
  int32_t param_dtype;    /* mh_dtype; bf16 is rounded to nearest even */
  int32_t heads;          /* heads in this entry */
  int64_t rows, cols;     /* stored shape; heads * head_stride <= rows */
  int64_t head_stride;    /* rows from one head's block to the next */
  int64_t row_offset;     /* first scaled row inside a block */
  int64_t scaled_rows;    /* rows scaled per head; row_offset + scaled_rows <= head_stride */
  int32_t head_index0;    /* s_max index of this entry's first head */
  float exponent;         /* >= 0 */
} mh_qk_clip_entry;

/* s_max: DEVICE float array (head_index0 + heads entries at least for every
 * entry). tau > 0. skip: the gradient-control flag (DEVICE, may be NULL):
 * nothing is clipped after a skipped step. */
int mh_qk_clip(const mh_qk_clip_entry* entries, int32_t n, const float* s_max, float tau,
               const int32_t* skip, void* stream);

/* Optional per-kernel timing. When enabled, every kernel the library launches
 * is bracketed by two CUDA events recorded on its own stream, and the
 * launch's algorithmic work is noted: bytes that must cross HBM at least
 * once for the elementwise kernels, and the nominal dense FLOPs of the
 * Newton-Schulz GEMM stages (2 m^2 n for X X^T and for P X, 2 m^3 for A A),
 * plus the FLOPs the tensor cores actually execute (fewer, since only the
 * upper triangle of the symmetric products is computed). Events are host
 * objects created on first use; no device memory is allocated. Disabled by
 * default; when disabled the calls above record nothing. Independently of
 * it, every launch sits inside an NVTX range named after its stage
 * (e.g. "ns_gemm.gram"), a no-op unless a profiling tool is attached. */
typedef struct {
  char name[32];          /* kernel family, e.g. "ns_gemm", "muon_prologue" */
  int64_t launches;       /* launches recorded since the last reset */
  double total_ms;        /* summed event time of those launches */
  double bytes;           /* summed algorithmic HBM bytes */
  double flops;           /* summed nominal FLOPs (GEMM stages) */
  double flops_executed;  /* summed tensor-core FLOPs actually issued */
} mh_kernel_stats;

int mh_profiler_enable(int32_t enable);
/* Drops every recorded launch. */
int mh_profiler_reset(void);
/* Waits for the recorded events and aggregates them per kernel family into
 * `out` (capacity `max`); `*count` receives the number of families. */
int mh_profiler_read(mh_kernel_stats* out, int32_t max, int32_t* count);

/* Reads the device status word the last Muon or Newton-Schulz call left in
 * `workspace`, synchronising `stream`. MH_OK, or MH_ETIMEOUT when a kernel's
 * bounded wait gave up (its outputs are then undefined). */
int mh_workspace_status(const void* workspace, void* stream);

/* Bounded waits of the Newton-Schulz GEMM stages and of the streaming
 * NorMuon / Muon+ apply and column-statistics passes of mh_muon_step_batched.
 * The pages have no counterpart: every wait of such a launch on its pipeline
 * (operand loads, MMAs, accumulators, the pair's shared block sequence, a
 * stage of the streaming ring) gives up after this many SM clock cycles; the
 * launch then records MH_ETIMEOUT in the workspace status word
 * (mh_workspace_status), lets whatever copies and MMAs it had issued land,
 * frees its tensor memory and returns, and the call's outputs are
 * undefined. The default, about one second at GB300 clocks, is far above
 * any legitimate wait. A smaller value makes the failure path observable in
 * a test without a fault or a hang.
 *   cycles: > 0 sets the limit for launches enqueued from now on, process
 *           wide; 0 restores the default; < 0 returns MH_EINVAL.
 * Launches already enqueued keep the limit they were given. */
int mh_set_wait_limit(int64_t cycles);
/* The current limit in cycles. */
int64_t mh_get_wait_limit(void);

/* *accessible = 1 when the current device can read and write `ptr` at that
 * very address: device memory, managed memory, or host memory that is
 * page-locked and mapped into the device's address space (0 otherwise, e.g.
 * pageable host memory or an unknown pointer). Host-only query. */
int mh_pointer_device_accessible(const void* ptr, int32_t* accessible);

/* Message for the last non-OK status on this host thread ("" if none). */
const char* mh_last_error(void);

/* Library version, e.g. "0.1.0". */
const char* mh_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MUONHYBRID_H */
