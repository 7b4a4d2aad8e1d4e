// Host side of libmuonhybrid: argument checks, the per-call plan (shape
// classes, workspace layout, tile lists, TMA tensor maps) and the
// stream-ordered launch sequence behind the three entry points of
// include/muonhybrid.h.
//
// Plan. Every view is a Newton-Schulz problem of size m x n (m = min(rows,
// cols), n = max(rows, cols)); for a tall view (rows > cols) the iteration
// runs on the transpose, as the Speedtronic "Newton-Schulz" section
// prescribes. No data is transposed: a tall view's X is kept in its stored
// (n x m) layout and the GEMM stages read it with transposed operands. Views
// with the same (m, n, tall) form a shape class whose buffers are stacked in
// the workspace, so one 3-D tensor map covers a whole class and one grouped
// launch per Newton-Schulz stage covers every class.
//
// Workspace (256-byte aligned base):
//   [0, 256)        header: device status word (bounded-wait timeouts) at 0,
//                   the GEMM stages' block counters at kTileCounterOffset
//   sumsq           double per view: ||Q||_F^2
//   tile_ss         float per prologue tile and warp: partial ||Q||_F^2
//   vrec            per view: parameter/gradient pointers, shape, lr, wd (the
//                   last Newton-Schulz apply updates parameters directly)
//   rowpart         float per (view, column tile, stored row)   (NorMuon / Muon+)
//   rowfac          float per (view, stored row)                 (NorMuon / Muon+)
//   colpart         float per (view, row tile, stored col)       (Muon+)
//   colfac          float per (view, stored col)                 (Muon+)
//   per class       X0, X1 (bf16, per view m x ldx, or n x ldx for tall views),
//                   A, P (bf16, m x lda)
// Every reduction is a sum of per-tile partials taken in a fixed order, so a
// step's results do not depend on scheduling.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "mh_internal.h"
#include "mh_ptx.cuh"
#include "mh_sr.cuh"
#include "muonhybrid.h"

namespace mh {
namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MH_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kMaxDim = int64_t(1) << 24;   // rows or cols of a view
constexpr int64_t kMaxNsDim = 32768;            // min(rows, cols) of a view
constexpr size_t kHeaderBytes = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(int32_t d) { return d == MH_F32 || d == MH_BF16; }

struct ClassInfo {
  int64_t m = 0, n = 0, ldx = 0, lda = 0, count = 0;
  bool tstore = false;       // X kept in the stored (n x m) layout of tall views
  int64_t xrows = 0;         // rows of one view's X buffer: m, or n when tstore
  size_t off_x[2] = {0, 0}, off_a = 0, off_p = 0;
};

struct TensorInfo {
  int idx = 0;          // index in the caller's array
  int64_t views = 0, rows = 0, cols = 0;
  int cls = 0;
  int64_t class_slot = 0;  // slot of the first view within its class
  int64_t view_slot = 0;   // global view index (sumsq)
  int64_t tile_off = 0;    // first prologue tile (tile_ss index)
  int64_t tiles_r = 0, tiles_c = 0;  // 32 x 256 tiles of the statistics/apply passes
  int64_t ptiles_c = 0;              // 32 x 256 tiles of the prologue
  bool flat = false;                 // prologue streams the view as contiguous chunks
  int64_t pro_tiles_per_view = 0;    // prologue work items per view
  int64_t rowpart_off = 0, rowfac_off = 0;  // elements
  int64_t colpart_off = 0, colfac_off = 0;  // elements
  bool tall = false;
};

struct Plan {
  std::vector<ClassInfo> classes;
  std::vector<TensorInfo> tensors;
  int64_t total_views = 0, total_tiles = 0;
  int64_t n_rowpart = 0, n_rowfac = 0, n_colpart = 0, n_colfac = 0;
  size_t off_active = 0;  // int32 per view (inactive-expert rule)
  size_t off_sumsq = 0, off_tile_ss = 0, off_vrec = 0, off_rowpart = 0, off_rowfac = 0,
         off_colpart = 0, off_colfac = 0;
  size_t bytes = 0;
};

struct Shape {
  int64_t views, rows, cols;
};

// Groups views by Newton-Schulz shape and lays out the workspace.
Plan make_plan(const std::vector<Shape>& shapes, bool need_rows, bool need_cols) {
  Plan P;
  std::map<std::pair<std::pair<int64_t, int64_t>, bool>, int> cls_of;
  for (size_t i = 0; i < shapes.size(); ++i) {
    const Shape& s = shapes[i];
    if (s.views == 0 || s.rows == 0 || s.cols == 0) continue;
    TensorInfo T;
    T.idx = static_cast<int>(i);
    T.views = s.views;
    T.rows = s.rows;
    T.cols = s.cols;
    T.tall = s.rows > s.cols;
    const int64_t m = T.tall ? s.cols : s.rows;
    const int64_t n = T.tall ? s.rows : s.cols;
    // Tall views keep X in their stored layout; the GEMMs read it transposed.
    auto key = std::make_pair(std::make_pair(m, n), T.tall);
    auto it = cls_of.find(key);
    if (it == cls_of.end()) {
      ClassInfo C;
      C.m = m;
      C.n = n;
      C.tstore = T.tall;
      C.xrows = T.tall ? n : m;
      C.ldx = ((T.tall ? m : n) + 7) / 8 * 8;
      C.lda = (m + 7) / 8 * 8;
      it = cls_of.emplace(key, static_cast<int>(P.classes.size())).first;
      P.classes.push_back(C);
    }
    T.cls = it->second;
    T.class_slot = P.classes[T.cls].count;
    P.classes[T.cls].count += s.views;
    P.tensors.push_back(T);
  }
  // Global view slots ordered by class, then by tensor within the class.
  int64_t slot = 0;
  std::vector<int64_t> class_first(P.classes.size(), 0);
  for (size_t c = 0; c < P.classes.size(); ++c) {
    class_first[c] = slot;
    slot += P.classes[c].count;
  }
  P.total_views = slot;
  for (TensorInfo& T : P.tensors) {
    T.view_slot = class_first[T.cls] + T.class_slot;
    T.tiles_r = ceil_div(T.rows, kEwTileR);
    T.tiles_c = ceil_div(T.cols, kEwTileC);
    T.ptiles_c = ceil_div(T.cols, kProTileC);
    // X holds every view in its stored layout; when the row pitch equals the
    // stored cols the prologue streams the view in contiguous chunks.
    T.flat = (T.cols % 8) == 0;
    T.pro_tiles_per_view = T.flat ? ceil_div(T.rows * T.cols, kProChunk) : T.tiles_r * T.ptiles_c;
    T.tile_off = P.total_tiles;
    P.total_tiles += T.views * T.pro_tiles_per_view;
    T.rowpart_off = P.n_rowpart;
    T.rowfac_off = P.n_rowfac;
    T.colpart_off = P.n_colpart;
    T.colfac_off = P.n_colfac;
    P.n_rowpart += T.views * T.tiles_c * T.rows;
    P.n_rowfac += T.views * T.rows;
    P.n_colpart += T.views * T.tiles_r * T.cols;
    P.n_colfac += T.views * T.cols;
  }
  size_t off = kHeaderBytes;
  P.off_sumsq = off;
  off = align_up(off + sizeof(double) * static_cast<size_t>(P.total_views), 256);
  P.off_tile_ss = off;
  off = align_up(off + sizeof(float) * (kEwThreads / 32) * static_cast<size_t>(P.total_tiles), 256);
  P.off_vrec = off;
  off = align_up(off + sizeof(ViewRec) * static_cast<size_t>(P.total_views), 256);
  P.off_active = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(P.total_views), 256);
  if (need_rows) {
    P.off_rowpart = off;
    off = align_up(off + sizeof(float) * static_cast<size_t>(P.n_rowpart), 256);
    P.off_rowfac = off;
    off = align_up(off + sizeof(float) * static_cast<size_t>(P.n_rowfac), 256);
  }
  if (need_cols) {
    P.off_colpart = off;
    off = align_up(off + sizeof(float) * static_cast<size_t>(P.n_colpart), 256);
    P.off_colfac = off;
    off = align_up(off + sizeof(float) * static_cast<size_t>(P.n_colfac), 256);
  }
  off = align_up(off, 1024);
  for (ClassInfo& C : P.classes) {
    const size_t xb = static_cast<size_t>(C.count) * C.xrows * C.ldx * sizeof(bf16);
    const size_t ab = static_cast<size_t>(C.count) * C.m * C.lda * sizeof(bf16);
    C.off_x[0] = off; off = align_up(off + xb, 1024);
    C.off_x[1] = off; off = align_up(off + xb, 1024);
    C.off_a = off; off = align_up(off + ab, 1024);
    C.off_p = off; off = align_up(off + ab, 1024);
  }
  P.bytes = off;
  return P;
}

int check_shape(int64_t views, int64_t rows, int64_t cols, int i, const char* what) {
  if (views < 0 || rows < 0 || cols < 0)
    return fail(MH_ESHAPE, "%s[%d]: negative shape (views=%lld rows=%lld cols=%lld)", what, i,
                (long long)views, (long long)rows, (long long)cols);
  if (rows > kMaxDim || cols > kMaxDim || views > kMaxDim)
    return fail(MH_ESHAPE, "%s[%d]: dimension above 2^24 (views=%lld rows=%lld cols=%lld)", what,
                i, (long long)views, (long long)rows, (long long)cols);
  if ((rows < cols ? rows : cols) > kMaxNsDim)
    return fail(MH_EUNSUPPORTED, "%s[%d]: min(rows, cols) = %lld exceeds %lld", what, i,
                (long long)(rows < cols ? rows : cols), (long long)kMaxNsDim);
  return MH_OK;
}

// ---- TMA tensor maps ---------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 map over a stacked class buffer: (inner, rows, views) with the
// given row pitch; box (64, box_rows, 1), 128-byte swizzle, zero fill.
// bf16 tensor map over `views` stacked (rows x inner) matrices of row pitch
// `ld` elements, box (box_inner x box_rows x 1).
int encode_tmap(CUtensorMap* tm, const void* base, int64_t inner, int64_t rows, int64_t views,
                int64_t ld, int box_inner, int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(MH_ECUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(views)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2,
                           static_cast<cuuint64_t>(ld) * 2 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MH_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return MH_OK;
}

// Operand loads: 64-element (128-byte) rows, 128-byte swizzle.
int make_tmap(CUtensorMap* tm, const void* base, int64_t inner, int64_t rows, int64_t views,
              int64_t ld, int box_rows) {
  return encode_tmap(tm, base, inner, rows, views, ld, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Epilogue stores: 32 x 32 boxes with 64-byte rows, 64-byte swizzle.
int make_tmap_out(CUtensorMap* tm, const void* base, int64_t inner, int64_t rows, int64_t views,
                  int64_t ld) {
  return encode_tmap(tm, base, inner, rows, views, ld, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

int device_sms(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) {
    *out = it->second;
    return MH_OK;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  cache[dev] = sms;
  *out = sms;
  return MH_OK;
}

// ---- optional per-kernel event timing ---------------------------------------------

struct ProfRecord {
  cudaEvent_t begin, end;
  const char* name;
  double bytes, flops, flops_exec;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<ProfRecord> records;
  std::vector<cudaEvent_t> pool;
};

Profiler& profiler() {
  static Profiler p;
  return p;
}

cudaEvent_t prof_event(Profiler& P) {
  if (!P.pool.empty()) {
    cudaEvent_t e = P.pool.back();
    P.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one launch with events on its stream when profiling is on.
// Around each launch: an NVTX range named after the stage (for nsys / ncu
// --nvtx filtering; a no-op unless a tool is attached) and, while the
// profiler is on, a pair of CUDA events on the launch stream.
class ProfScope {
 public:
  ProfScope(cudaStream_t s, const char* name, double bytes, double flops = 0.0,
            double flops_exec = 0.0)
      : s_(s) {
    nvtxRangePushA(name);
    Profiler& P = profiler();
    std::lock_guard<std::mutex> lock(P.mu);
    if (!P.on) return;
    rec_.begin = prof_event(P);
    rec_.end = prof_event(P);
    if (!rec_.begin || !rec_.end) return;
    rec_.name = name;
    rec_.bytes = bytes;
    rec_.flops = flops;
    rec_.flops_exec = flops_exec;
    active_ = cudaEventRecord(rec_.begin, s_) == cudaSuccess;
  }
  ~ProfScope() {
    nvtxRangePop();
    if (!active_) return;
    Profiler& P = profiler();
    std::lock_guard<std::mutex> lock(P.mu);
    if (cudaEventRecord(rec_.end, s_) == cudaSuccess) P.records.push_back(rec_);
  }

 private:
  cudaStream_t s_;
  ProfRecord rec_{};
  bool active_ = false;
};

// ---- Newton-Schulz stages --------------------------------------------------------

// Launches the 3 * steps grouped GEMM stages. When `final_update` is set, the
// last apply stage writes the parameter update (from the per-view records)
// instead of the last X.
// Newton-Schulz stages of every view: `steps` iterations, iteration `it`
// using (sched[3 it], sched[3 it + 1], sched[3 it + 2]) when a schedule is
// given, else (a, b, c).
int run_ns(const Plan& P, uint8_t* ws, int steps, float a, float b, float c, float eps, int sms,
           cudaStream_t stream, int* final_buf, bool final_update = false, int cautious = 0,
           const int32_t* skip = nullptr, const float* sched = nullptr,
           float norm_scale = 1.0f, cudaEvent_t fence = nullptr, bool row_sums = false) {
  int cur = 0;
  const int nclass = static_cast<int>(P.classes.size());
  double* sumsq = reinterpret_cast<double*>(ws + P.off_sumsq);
  int* status = reinterpret_cast<int*>(ws);
  // Global view slot of the first view of each class.
  std::vector<int64_t> class_first(nclass, 0);
  for (int k = 1; k < nclass; ++k) class_first[k] = class_first[k - 1] + P.classes[k - 1].count;
  // Block counters of the stage launches (see kTileRing): the first two
  // launches claim from counters zeroed here, every launch zeroes the one
  // two launches ahead.
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + kTileCounterOffset);
  static_assert(kTileCounterOffset + kTileCounters * sizeof(uint32_t) <= kHeaderBytes,
                "tile counters must fit in the workspace header");
  if (steps > 0) {
    const cudaError_t me = cudaMemsetAsync(counters, 0, 2 * sizeof(uint32_t), stream);
    if (me != cudaSuccess) return cuda_fail(me, "cudaMemsetAsync(tile counters)");
  }
  int launch = 0;
  const long long wait_limit = gemm_wait_limit();

  for (int it = 0; it < steps; ++it) {
    for (int kind = GEMM_GRAM; kind <= GEMM_APPLY; ++kind) {
      // One launch per stage over every class (more only beyond kMaxClasses
      // classes); each class carries its own operand mode.
      {
        std::vector<int> ids;
        for (int k = 0; k < nclass; ++k) ids.push_back(k);
        const int nids = static_cast<int>(ids.size());
        for (int c0 = 0; c0 < nids; c0 += kMaxClasses) {
          GemmParams gp;
          std::memset(&gp, 0, sizeof(gp));
          gp.kind = kind;
          gp.first_iter = it == 0 ? 1 : 0;
          gp.tile_counter = counters + launch % kTileCounters;
          gp.next_counter = counters + (launch + 2) % kTileCounters;
          gp.wait_limit = wait_limit;
          ++launch;
          gp.a = sched ? sched[3 * it] : a;
          gp.b = sched ? sched[3 * it + 1] : b;
          gp.c = sched ? sched[3 * it + 2] : c;
          gp.eps = eps;
          gp.norm_scale = norm_scale;
          gp.status = status;
          gp.skip = skip;
          const bool fused = final_update && kind == GEMM_APPLY && it == steps - 1;
          gp.final_update = fused ? 1 : 0;
          gp.row_sums = row_sums && kind == GEMM_APPLY && it == steps - 1 ? 1 : 0;
          if (fused && fence) {
            // First launch that writes parameters (stream order carries the
            // wait to every later launch).
            const cudaError_t fe = cudaStreamWaitEvent(stream, fence, 0);
            if (fe != cudaSuccess) return cuda_fail(fe, "cudaStreamWaitEvent(param_fence)");
            fence = nullptr;
          }
          gp.cautious = cautious;
          int64_t tiles = 0;
          int nc = 0;
          for (; c0 + nc < nids && nc < kMaxClasses; ++nc) {
            const int k = ids[c0 + nc];
            const ClassInfo& C = P.classes[k];
            GemmClass& G = gp.cls[nc];
            bf16* X = reinterpret_cast<bf16*>(ws + C.off_x[cur]);
            bf16* Xn = reinterpret_cast<bf16*>(ws + C.off_x[cur ^ 1]);
            bf16* A = reinterpret_cast<bf16*>(ws + C.off_a);
            bf16* Pm = reinterpret_cast<bf16*>(ws + C.off_p);
            G.m = static_cast<int32_t>(C.m);
            G.n = static_cast<int32_t>(C.n);
            G.tstore = C.tstore ? 1 : 0;
            G.mode = gemm_mode(kind, C.tstore);
            G.out_rows = static_cast<int32_t>(C.tstore ? C.n : C.m);
            G.out_cols = static_cast<int32_t>(C.tstore ? C.m : C.n);
            G.views = static_cast<int32_t>(C.count);
            G.sumsq = sumsq + class_first[k];
            G.vrec = reinterpret_cast<const ViewRec*>(ws + P.off_vrec) + class_first[k];
            // Work units are 256 x 256 blocks, one per CTA pair (2 x 128 rows).
            G.tiles_m = static_cast<int32_t>(ceil_div(C.m, 2 * kBM));
            int rc;
            if (kind == GEMM_GRAM || kind == GEMM_POLY) {
              // Upper block triangle: row block pm holds column blocks pm..T-1.
              G.tiles_n = static_cast<int32_t>(ceil_div(C.m, kBN));
              G.tiles_per_view = G.tiles_n * (G.tiles_n + 1) / 2;
              G.out = kind == GEMM_GRAM ? A : Pm;
              G.out_view_stride = C.m * C.lda;
              G.ld_out = C.lda;
              if (kind == GEMM_GRAM) {
                G.K = static_cast<int32_t>(C.n);
                G.aux = X;
                G.aux_view_stride = C.xrows * C.ldx;
                G.ld_aux = C.ldx;
                if (C.tstore) {
                  // T is n x m: both operands are 64 x 64 MN-major chunks of T.
                  if ((rc = make_tmap(&G.tmA, X, C.m, C.n, C.count, C.ldx, 64)) != MH_OK) return rc;
                } else {
                  if ((rc = make_tmap(&G.tmA, X, C.n, C.m, C.count, C.ldx, kBM)) != MH_OK) return rc;
                }
                G.tmB = G.tmA;  // each CTA of a pair loads 128 of the 256 B rows
              } else {
                G.K = static_cast<int32_t>(C.m);
                G.aux = A;
                G.aux_view_stride = C.m * C.lda;
                G.ld_aux = C.lda;
                if ((rc = make_tmap(&G.tmA, A, C.m, C.m, C.count, C.lda, kBM)) != MH_OK) return rc;
                G.tmB = G.tmA;
              }
              if ((rc = make_tmap_out(&G.tmOut, G.out, C.m, C.m, C.count, C.lda)) != MH_OK)
                return rc;
            } else {
              G.tiles_m = static_cast<int32_t>(ceil_div(G.out_rows, 2 * kBM));
              G.tiles_n = static_cast<int32_t>(ceil_div(G.out_cols, kBN));
              G.tiles_per_view = G.tiles_m * G.tiles_n;
              G.K = static_cast<int32_t>(C.m);
              G.out = Xn;
              G.out_view_stride = C.xrows * C.ldx;
              G.ld_out = C.ldx;
              G.aux = X;
              G.aux_view_stride = C.xrows * C.ldx;
              G.ld_aux = C.ldx;
              if (C.tstore) {
                // T' = a T + T P: rows of T and rows of P, both K-major.
                if ((rc = make_tmap(&G.tmA, X, C.m, C.n, C.count, C.ldx, kBM)) != MH_OK) return rc;
                if ((rc = make_tmap(&G.tmB, Pm, C.m, C.m, C.count, C.lda, kBM)) != MH_OK) return rc;
              } else {
                if ((rc = make_tmap(&G.tmA, Pm, C.m, C.m, C.count, C.lda, kBM)) != MH_OK) return rc;
                if ((rc = make_tmap(&G.tmB, X, C.n, C.m, C.count, C.ldx, 64)) != MH_OK) return rc;
              }
              if ((rc = make_tmap_out(&G.tmOut, Xn, G.out_cols, G.out_rows, C.count, C.ldx)) !=
                  MH_OK)
                return rc;
            }
            G.tile_begin = tiles;
            tiles += static_cast<int64_t>(G.tiles_per_view) * C.count;
          }
          gp.num_classes = nc;
          gp.total_tiles = tiles;
          if (tiles >= (int64_t(1) << 31))
            return fail(MH_EUNSUPPORTED, "too many GEMM tiles in one stage (%lld)", (long long)tiles);
          double flops = 0.0, fexec = 0.0, bytes = 0.0;
          for (int k = 0; k < nc; ++k) {
            const GemmClass& G = gp.cls[k];
            const double m = G.m, nn = G.n, v = G.views;
            flops += v * (kind == GEMM_POLY ? 2.0 * m * m * m : 2.0 * m * m * nn);
            const double kpad = std::ceil(G.K / double(kBK)) * kBK;
            fexec += double(G.tiles_per_view) * v * 2.0 * (2.0 * kBM) * kBN * kpad;
            // operands read once and the output written once (bf16)
            if (kind == GEMM_GRAM) bytes += v * 2.0 * (m * nn + m * m);
            else if (kind == GEMM_POLY) bytes += v * 2.0 * (m * m + m * m);
            else if (!fused) bytes += v * 2.0 * (m * m + 2.0 * m * nn);
            else bytes += v * (2.0 * (m * m + m * nn) + 2.0 * 2.0 * m * nn);  // + W read/write (bf16)
          }
          static const char* kNames[4] = {"ns_gemm.gram", "ns_gemm.poly", "ns_gemm.apply",
                                           "ns_gemm.apply_update"};
          ProfScope ps(stream, kNames[fused ? 3 : kind], bytes, flops, fexec);
          cudaError_t e = launch_ns_gemm(gp, sms, stream);
          if (e != cudaSuccess) return cuda_fail(e, "Newton-Schulz GEMM launch");
        }
      }
    }
    cur ^= 1;
  }
  *final_buf = cur;
  return MH_OK;
}

// ---- elementwise launches in batches of kMaxJobs tensors -------------------------

double dsize(int32_t dt) { return dt == MH_F32 ? 4.0 : 2.0; }

// Bytes each elementwise pass must move through HBM at least once.
double ew_bytes(EwKind kind, const EwParams& p, const EwJob& J) {
  const double e = double(J.rows) * J.cols * J.views;
  switch (kind) {
    case EW_PROLOGUE:
    case EW_PROLOGUE_FLAT:
    case EW_PROLOGUE_FLAT_B16:
      return e * (dsize(J.src_dtype) + (p.use_momentum ? 2.0 * dsize(J.mom_dtype) : 0.0) + 2.0);
    case EW_ROWSQ:
      return e * 2.0;
    case EW_COLSQ:
      return e * 2.0;
    case EW_APPLY:
    case EW_APPLY_CU:
      return e * (2.0 + 2.0 * dsize(J.dst_dtype) +
                  (p.cautious == MH_CAUTIOUS_UPDATE ? dsize(J.src_dtype) : 0.0));
    case EW_COPYOUT:
      return e * (2.0 + dsize(J.dst_dtype));
  }
  return 0.0;
}

const char* ew_name(EwKind kind, bool muon) {
  switch (kind) {
    case EW_PROLOGUE:
    case EW_PROLOGUE_FLAT:
    case EW_PROLOGUE_FLAT_B16: return muon ? "muon_prologue" : "ns_prologue";
    case EW_ROWSQ: return "muon_rowstats";
    case EW_COLSQ: return "muon_colstats";
    case EW_APPLY:
    case EW_APPLY_CU: return "muon_apply";
    case EW_COPYOUT: return "ns_copyout";
  }
  return "elementwise";
}

template <typename Fill, typename Sel>
int run_ew_sel(EwKind kind, const Plan& P, const EwParams& proto, Fill fill, int sms,
               cudaStream_t stream, Sel sel) {
  std::vector<size_t> idx;
  for (size_t t = 0; t < P.tensors.size(); ++t)
    if (sel(P.tensors[t])) idx.push_back(t);
  const size_t nt = idx.size();
  for (size_t t0 = 0; t0 < nt; t0 += kMaxJobs) {
    EwParams ep = proto;
    ep.njobs = 0;
    int64_t tiles = 0;
    for (size_t q = t0; q < nt && ep.njobs < kMaxJobs; ++q) {
      const TensorInfo& T = P.tensors[idx[q]];
      EwJob& J = ep.jobs[ep.njobs++];
      std::memset(&J, 0, sizeof(J));
      J.rows = T.rows;
      J.cols = T.cols;
      J.views = T.views;
      J.tall = 0;  // X of a tall view is kept in its stored layout
      J.tiles_r = static_cast<int32_t>(T.tiles_r);
      J.tiles_c = static_cast<int32_t>(T.tiles_c);
      if (kind == EW_PROLOGUE || kind == EW_PROLOGUE_FLAT) {
        J.flat = T.flat ? 1 : 0;
        J.tiles_r = T.flat ? 1 : static_cast<int32_t>(T.tiles_r);
        J.tiles_c = static_cast<int32_t>(T.flat ? T.pro_tiles_per_view : T.ptiles_c);
      }
      J.tile_begin = tiles;
      tiles += static_cast<int64_t>(J.tiles_r) * J.tiles_c * T.views;
      fill(T, J);
      if ((kind == EW_PROLOGUE || kind == EW_PROLOGUE_FLAT) && (T.cols % 8) != 0) {
        // the prologue moves 8 consecutive elements per access
        J.src_vec = J.dst_vec = J.mom_vec = 0;
      }
    }
    ep.total_tiles = tiles;
    double bytes = 0.0;
    for (int k = 0; k < ep.njobs; ++k) bytes += ew_bytes(kind, ep, ep.jobs[k]);
    ProfScope ps(stream, ew_name(kind, proto.use_momentum != 0), bytes);
    cudaError_t e = launch_elementwise(kind, ep, sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "elementwise launch");
  }
  return MH_OK;
}

template <typename Fill>
int run_ew(EwKind kind, const Plan& P, const EwParams& proto, Fill fill, int sms,
           cudaStream_t stream) {
  if (kind == EW_PROLOGUE) {
    // Wide views stored like X are streamed by their own kernel.
    int rc = run_ew_sel(EW_PROLOGUE_FLAT, P, proto, fill, sms, stream,
                        [](const TensorInfo& T) { return T.flat; });
    if (rc != MH_OK) return rc;
    return run_ew_sel(EW_PROLOGUE, P, proto, fill, sms, stream,
                      [](const TensorInfo& T) { return !T.flat; });
  }
  return run_ew_sel(kind, P, proto, fill, sms, stream, [](const TensorInfo&) { return true; });
}

int run_view_norm(const Plan& P, float* tile_ss, double* sumsq, cudaStream_t stream,
                  const int32_t* skip = nullptr) {
  for (size_t t0 = 0; t0 < P.tensors.size(); t0 += kMaxNormJobs) {
    NormParams np;
    std::memset(&np, 0, sizeof(np));
    np.skip = skip;
    int64_t views = 0;
    for (size_t t = t0; t < P.tensors.size() && np.njobs < kMaxNormJobs; ++t) {
      const TensorInfo& T = P.tensors[t];
      NormJob& J = np.jobs[np.njobs++];
      J.tile_ss = tile_ss + T.tile_off * (kEwThreads / 32);
      J.sumsq = sumsq + T.view_slot;
      J.tiles_per_view = T.pro_tiles_per_view;
      J.views = T.views;
      J.view_begin = views;
      views += T.views;
    }
    np.total_views = views;
    ProfScope ps(stream, "view_norm", 0.0);
    cudaError_t e = launch_view_norm(np, stream);
    if (e != cudaSuccess) return cuda_fail(e, "view norm launch");
  }
  return MH_OK;
}

// Inactive-expert rule: clears the per-view flags and marks the views of
// flagged tensors that have a nonzero gradient entry.
int run_view_active(const Plan& P, const mh_muon_tensor* tensors, int32_t* active, int sms,
                    cudaStream_t stream) {
  bool any = false;
  for (const TensorInfo& T : P.tensors) any = any || tensors[T.idx].skip_zero_grad;
  if (!any) return MH_OK;
  cudaError_t e = cudaMemsetAsync(active, 0, sizeof(int32_t) * P.total_views, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(active flags)");
  ActiveParams ap;
  std::memset(&ap, 0, sizeof(ap));
  int64_t chunks = 0;
  auto flush = [&]() -> int {
    ap.total_chunks = chunks;
    double bytes = 0.0;
    for (int k = 0; k < ap.njobs; ++k)
      bytes += double(ap.jobs[k].view_elems) * ap.jobs[k].views * dsize(ap.jobs[k].gdt);
    ProfScope ps(stream, "muon_active", bytes);
    cudaError_t err = launch_view_active(ap, sms, stream);
    ap.njobs = 0;
    chunks = 0;
    if (err != cudaSuccess) return cuda_fail(err, "inactive-expert scan launch");
    return MH_OK;
  };
  int rc;
  for (const TensorInfo& T : P.tensors) {
    const mh_muon_tensor& U = tensors[T.idx];
    if (!U.skip_zero_grad) continue;
    ActiveJob& J = ap.jobs[ap.njobs++];
    J.grad = U.grad;
    J.active = active + T.view_slot;
    J.view_elems = T.rows * T.cols;
    J.views = T.views;
    J.gdt = U.grad_dtype;
    J.vec = aligned16(U.grad) && (J.view_elems % 8) == 0;
    J.chunk_begin = chunks;
    chunks += T.views * ((J.view_elems + kActiveChunk - 1) / kActiveChunk);
    if (ap.njobs == kMaxActiveJobs && (rc = flush()) != MH_OK) return rc;
  }
  if (ap.njobs > 0 && (rc = flush()) != MH_OK) return rc;
  return MH_OK;
}

int check_muon_args(const mh_muon_tensor* t, int32_t n, const mh_muon_hparams* hp) {
  if (n < 0) return fail(MH_EINVAL, "n must be >= 0 (got %d)", n);
  if (n > 0 && !t) return fail(MH_EINVAL, "tensors is NULL");
  if (!hp) return fail(MH_EINVAL, "hparams is NULL");
  if (!std::isfinite(hp->lr)) return fail(MH_EINVAL, "lr must be finite");
  if (!(hp->momentum >= 0.0f && hp->momentum < 1.0f))
    return fail(MH_EINVAL, "momentum must be in [0, 1) (got %g)", hp->momentum);
  if (!(hp->eps >= 0.0f) || !std::isfinite(hp->eps)) return fail(MH_EINVAL, "eps must be >= 0");
  if (!(hp->norm_scale >= 0.0f) || !std::isfinite(hp->norm_scale))
    return fail(MH_EINVAL, "norm_scale must be finite and >= 0 (0 means 1)");
  if (hp->ns_steps < 0 || hp->ns_steps > 16)
    return fail(MH_EINVAL, "ns_steps must be in [0, 16] (got %d)", hp->ns_steps);
  if (!std::isfinite(hp->a) || !std::isfinite(hp->b) || !std::isfinite(hp->c))
    return fail(MH_EINVAL, "Newton-Schulz coefficients must be finite");
  if (hp->coeff_schedule)
    for (int k = 0; k < 3 * hp->ns_steps; ++k)
      if (!std::isfinite(hp->coeff_schedule[k]))
        return fail(MH_EINVAL, "coeff_schedule[%d] is not finite", k);
  if (hp->normuon && !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return fail(MH_EINVAL, "beta2 must be in [0, 1) (got %g)", hp->beta2);
  if (hp->muon_plus && !(hp->plus_eps > 0.0f))
    return fail(MH_EINVAL, "plus_eps must be > 0 with muon_plus");
  if (hp->cautious < MH_CAUTIOUS_OFF || hp->cautious > MH_CAUTIOUS_UPDATE)
    return fail(MH_EINVAL, "cautious must be 0, 1 or 2 (got %d)", hp->cautious);
  if (!(hp->normuon_eps >= 0.0f) || !std::isfinite(hp->normuon_eps))
    return fail(MH_EINVAL, "normuon_eps must be finite and >= 0 (0 means 1e-10)");
  if (hp->phase < MH_STEP_ALL || hp->phase > MH_STEP_FINISH)
    return fail(MH_EINVAL, "phase must be 0, 1 or 2 (got %d)", hp->phase);
  if (hp->shape_rule != MH_SHAPE_RATIO && hp->shape_rule != MH_SHAPE_MOONLIGHT)
    return fail(MH_EINVAL, "shape_rule must be 0 or 1 (got %d)", hp->shape_rule);
  for (int i = 0; i < n; ++i) {
    const mh_muon_tensor& T = t[i];
    int rc = check_shape(T.views, T.rows, T.cols, i, "tensors");
    if (rc != MH_OK) return rc;
    if (T.views * ceil_div(T.rows, kEwTileR) * ceil_div(T.cols, kEwTileC) >= (int64_t(1) << 31))
      return fail(MH_EUNSUPPORTED, "tensors[%d]: too many elements for one tensor", i);
    if (!valid_dtype(T.param_dtype) || !valid_dtype(T.grad_dtype) ||
        !valid_dtype(T.momentum_dtype))
      return fail(MH_EDTYPE,
                  "tensors[%d]: only fp32 and bf16 dense tensors are supported (sparse and complex "
                  "gradients are rejected)",
                  i);
    if (T.param_sr != 0 && T.param_sr != 1)
      return fail(MH_EINVAL, "tensors[%d]: param_sr must be 0 or 1", i);
    if (T.param_sr && T.param_dtype != MH_BF16)
      return fail(MH_EINVAL, "tensors[%d]: param_sr needs a bf16 parameter", i);
    if (T.skip_zero_grad != 0 && T.skip_zero_grad != 1)
      return fail(MH_EINVAL, "tensors[%d]: skip_zero_grad must be 0 or 1", i);
    if (T.views * T.rows * T.cols == 0) continue;
    if (!T.param || !T.grad || !T.momentum)
      return fail(MH_EINVAL, "tensors[%d]: param, grad and momentum must be non-NULL", i);
    if (hp->normuon && !T.normuon_sm)
      return fail(MH_EINVAL, "tensors[%d]: normuon_sm is required when normuon is on", i);
    if (!std::isfinite(T.lr_mult) || !std::isfinite(T.wd))
      return fail(MH_EINVAL, "tensors[%d]: lr_mult and wd must be finite", i);
  }
  return MH_OK;
}

Plan muon_plan(const mh_muon_tensor* t, int32_t n, const mh_muon_hparams* hp) {
  std::vector<Shape> shapes(n);
  for (int i = 0; i < n; ++i) shapes[i] = {t[i].views, t[i].rows, t[i].cols};
  const bool rows = hp->normuon || hp->muon_plus;
  return make_plan(shapes, rows, hp->muon_plus != 0);
}

int check_workspace(const Plan& P, const void* ws, size_t bytes) {
  if (!ws) return fail(MH_EWORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(MH_EWORKSPACE, "workspace must be 256-byte aligned");
  if (bytes < P.bytes)
    return fail(MH_EWORKSPACE, "workspace too small: %zu bytes given, %zu needed", bytes, P.bytes);
  return MH_OK;
}

}  // namespace

void set_last_error(const char* msg) { g_err = msg ? msg : ""; }

// Cycles a bounded wait in a GEMM stage may take (mh_set_wait_limit).
std::atomic<long long> g_wait_limit{kWaitLimitCycles};
long long gemm_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

bool encode_stream_map(CUtensorMap* tm, const void* base, bool f32, int64_t inner, int64_t rows,
                       int64_t views, int64_t ld) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(views)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * es,
                           static_cast<cuuint64_t>(ld) * es * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kEwTileC), static_cast<cuuint32_t>(kEwTileR), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mh

using namespace mh;

extern "C" {

const char* mh_last_error(void) { return g_err.c_str(); }

const char* mh_version(void) { return "0.1.0"; }

int mh_pointer_device_accessible(const void* ptr, int32_t* accessible) {
  if (!accessible) return fail(MH_EINVAL, "accessible is NULL");
  *accessible = 0;
  if (!ptr) return MH_OK;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // an unknown pointer is simply not accessible
    return MH_OK;
  }
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  switch (a.type) {
    case cudaMemoryTypeDevice:
      *accessible = a.device == dev ? 1 : 0;
      break;
    case cudaMemoryTypeManaged:
      *accessible = 1;
      break;
    case cudaMemoryTypeHost:
      *accessible = a.devicePointer == ptr ? 1 : 0;
      break;
    default:
      break;
  }
  return MH_OK;
}

size_t mh_muon_workspace_bytes(const mh_muon_tensor* tensors, int32_t n, const mh_muon_hparams* hp) {
  if (check_muon_args(tensors, n, hp) != MH_OK) return 0;
  return muon_plan(tensors, n, hp).bytes;
}

int mh_muon_step_batched(const mh_muon_tensor* tensors, int32_t n, const mh_muon_hparams* hp,
                         void* workspace, size_t workspace_bytes, void* stream_) {
  int rc = check_muon_args(tensors, n, hp);
  if (rc != MH_OK) return rc;
  const Plan P = muon_plan(tensors, n, hp);
  if (P.tensors.empty()) return MH_OK;
  if ((rc = check_workspace(P, workspace, workspace_bytes)) != MH_OK) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int sms = 0;
  if ((rc = device_sms(&sms)) != MH_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool grad_phase = hp->phase != MH_STEP_FINISH;
  const bool finish_phase = hp->phase != MH_STEP_GRADIENTS;

  cudaError_t e = cudaSuccess;
  if (grad_phase) {
    e = cudaMemsetAsync(ws, 0, kHeaderBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace status)");
  }

  double* sumsq = reinterpret_cast<double*>(ws + P.off_sumsq);
  float* tile_ss = reinterpret_cast<float*>(ws + P.off_tile_ss);
  float* rowpart = reinterpret_cast<float*>(ws + P.off_rowpart);
  float* rowfac = reinterpret_cast<float*>(ws + P.off_rowfac);
  float* colpart = reinterpret_cast<float*>(ws + P.off_colpart);
  float* colfac = reinterpret_cast<float*>(ws + P.off_colfac);
  ViewRec* vrec = reinterpret_cast<ViewRec*>(ws + P.off_vrec);
  int32_t* active = reinterpret_cast<int32_t*>(ws + P.off_active);
  if (grad_phase && (rc = run_view_active(P, tensors, active, sms, stream)) != MH_OK) return rc;
  const bool need_rows = hp->normuon || hp->muon_plus;
  // Without NorMuon / Muon+ the update needs nothing beyond U itself, so the
  // last Newton-Schulz apply stage writes the parameters directly.
  const bool fuse_update = !need_rows && hp->ns_steps >= 1;

  EwParams proto;
  std::memset(&proto, 0, sizeof(proto));
  proto.mu = hp->momentum;
  proto.nesterov = hp->nesterov ? 1 : 0;
  proto.use_momentum = 1;
  proto.cautious = hp->cautious;
  proto.use_rowfac = need_rows ? 1 : 0;
  proto.use_colfac = hp->muon_plus ? 1 : 0;
  proto.ns_eps = hp->eps;
  proto.ns_norm_scale = hp->norm_scale > 0.0f ? hp->norm_scale : 1.0f;
  proto.u_scale_from_sumsq = hp->ns_steps == 0 ? 1 : 0;
  proto.grad_mult = hp->grad_mult;
  proto.skip = hp->skip;
  proto.status = reinterpret_cast<int*>(ws);
  proto.wait_limit = gemm_wait_limit();

  int final_buf = 0;
  auto fill_common = [&](const TensorInfo& T, EwJob& J, int xbuf) {
    const mh_muon_tensor& U = tensors[T.idx];
    const ClassInfo& C = P.classes[T.cls];
    J.src = U.grad;
    J.mom = U.momentum;
    J.mom_dtype = U.momentum_dtype;
    J.param_sr = U.param_sr;
    J.mom_key = sr_key(hp->sr_seed, sr_stream(T.idx, SR_FIRST));
    J.param_key = sr_key(hp->sr_seed, sr_stream(T.idx, SR_PARAM));
    J.active = U.skip_zero_grad ? active + T.view_slot : nullptr;
    J.dst = U.param;
    J.sm = U.normuon_sm;
    J.src_dtype = U.grad_dtype;
    J.dst_dtype = U.param_dtype;
    const bool cols4 = (T.cols % 4) == 0;
    J.src_vec = cols4 && aligned16(U.grad);
    J.dst_vec = cols4 && aligned16(U.param);
    J.mom_vec = cols4 && aligned16(U.momentum);
    J.ldx = C.ldx;
    J.x_view_stride = C.xrows * C.ldx;
    J.stat_tiles_c = static_cast<int32_t>(T.tiles_c);
    bf16* xb = reinterpret_cast<bf16*>(ws + C.off_x[xbuf]) + T.class_slot * C.xrows * C.ldx;
    J.x0 = xb;
    J.xf = xb;
    J.sumsq = sumsq + T.view_slot;
    J.tile_ss = tile_ss + T.tile_off * (kEwThreads / 32);
    J.vrec = vrec + T.view_slot;
    if (need_rows) {
      J.rowpart = rowpart + T.rowpart_off;
      J.rowfac = rowfac + T.rowfac_off;
    }
    if (hp->muon_plus) {
      J.colpart = colpart + T.colpart_off;
      J.colfac = colfac + T.colfac_off;
    }
    J.lr = hp->lr * U.lr_mult;
    J.wd = U.wd;
    J.shape_scale = static_cast<float>(
        hp->shape_rule == MH_SHAPE_MOONLIGHT
            ? 0.2 * std::sqrt(static_cast<double>(std::max(T.rows, T.cols)))
            : std::sqrt(std::max(1.0, double(T.rows) / double(T.cols))));
  };

  if (grad_phase) {
    rc = run_ew(EW_PROLOGUE, P, proto,
                [&](const TensorInfo& T, EwJob& J) { fill_common(T, J, 0); }, sms, stream);
    if (rc != MH_OK) return rc;
    if ((rc = run_view_norm(P, tile_ss, sumsq, stream, hp->skip)) != MH_OK) return rc;
  }
  if (!finish_phase) return MH_OK;
  cudaEvent_t fence = static_cast<cudaEvent_t>(hp->param_fence);
  // Under NorMuon / Muon+ the last apply stage also writes the row partials
  // of U^2, so no separate statistics pass re-reads U.
  const bool gemm_row_sums = need_rows && hp->ns_steps >= 1;
  rc = run_ns(P, ws, hp->ns_steps, hp->a, hp->b, hp->c, hp->eps, sms, stream, &final_buf,
              fuse_update, hp->cautious, hp->skip, hp->coeff_schedule, proto.ns_norm_scale,
              fuse_update ? fence : nullptr, gemm_row_sums);
  if (rc != MH_OK) return rc;
  if (fuse_update) return MH_OK;
  auto fill_final = [&](const TensorInfo& T, EwJob& J) { fill_common(T, J, final_buf); };
  if (need_rows) {
    if (!gemm_row_sums) {
      rc = run_ew(EW_ROWSQ, P, proto, fill_final, sms, stream);
      if (rc != MH_OK) return rc;
    }
    for (size_t t0 = 0; t0 < P.tensors.size(); t0 += kMaxRowFinJobs) {
      RowFinParams rp;
      std::memset(&rp, 0, sizeof(rp));
      rp.normuon = hp->normuon ? 1 : 0;
      rp.muon_plus = hp->muon_plus ? 1 : 0;
      rp.beta2 = hp->beta2;
      rp.normuon_eps = hp->normuon_eps > 0.0f ? hp->normuon_eps : 1e-10f;
      rp.plus_eps = hp->plus_eps;
      rp.skip = hp->skip;
      int64_t views = 0;
      for (size_t t = t0; t < P.tensors.size() && rp.njobs < kMaxRowFinJobs; ++t) {
        const TensorInfo& T = P.tensors[t];
        RowFinJob& J = rp.jobs[rp.njobs++];
        J.sm = tensors[T.idx].normuon_sm;
        J.rowpart = rowpart + T.rowpart_off;
        J.rowfac = rowfac + T.rowfac_off;
        J.rows = T.rows;
        J.cols = T.cols;
        J.views = T.views;
        J.tiles_c = T.tiles_c;
        J.view_begin = views;
        J.active = tensors[T.idx].skip_zero_grad ? active + T.view_slot : nullptr;
        views += T.views;
      }
      rp.total_views = views;
      ProfScope ps(stream, "muon_rowfinal", 0.0);
      e = launch_row_finalize(rp, stream);
      if (e != cudaSuccess) return cuda_fail(e, "row finalisation launch");
    }
    if (hp->muon_plus) {
      rc = run_ew(EW_COLSQ, P, proto, fill_final, sms, stream);
      if (rc != MH_OK) return rc;
      for (size_t t0 = 0; t0 < P.tensors.size(); t0 += kMaxColFinJobs) {
        ColFinParams cp;
        std::memset(&cp, 0, sizeof(cp));
        cp.plus_eps = hp->plus_eps;
        cp.skip = hp->skip;
        int64_t total = 0;
        for (size_t t = t0; t < P.tensors.size() && cp.njobs < kMaxColFinJobs; ++t) {
          const TensorInfo& T = P.tensors[t];
          ColFinJob& J = cp.jobs[cp.njobs++];
          J.colpart = colpart + T.colpart_off;
          J.colfac = colfac + T.colfac_off;
          J.cols = T.cols;
          J.views = T.views;
          J.tiles_r = T.tiles_r;
          J.elem_begin = total;
          total += T.views * T.cols;
        }
        cp.total = total;
        ProfScope ps(stream, "muon_colfinal", 0.0);
        e = launch_col_finalize(cp, sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "column finalisation launch");
      }
    }
  }
  if (fence) {
    e = cudaStreamWaitEvent(stream, fence, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(param_fence)");
  }
  return run_ew(EW_APPLY, P, proto, fill_final, sms, stream);
}

size_t mh_ns_workspace_bytes(const mh_ns_problem* problems, int32_t n) {
  if (n < 0 || (n > 0 && !problems)) {
    fail(MH_EINVAL, "bad problem list");
    return 0;
  }
  std::vector<Shape> shapes(n);
  for (int i = 0; i < n; ++i) {
    if (check_shape(problems[i].views, problems[i].rows, problems[i].cols, i, "problems") != MH_OK)
      return 0;
    shapes[i] = {problems[i].views, problems[i].rows, problems[i].cols};
  }
  return make_plan(shapes, false, false).bytes;
}

// Newton-Schulz only; `sched` (host, steps x 3) overrides (a, b, c) when
// non-null.
static int ns_impl(const mh_ns_problem* problems, int32_t n, int32_t steps, float a, float b,
                   float c, const float* sched, float eps, float norm_scale, void* workspace,
                   size_t workspace_bytes, void* stream_) {
  if (n < 0) return fail(MH_EINVAL, "n must be >= 0 (got %d)", n);
  if (n > 0 && !problems) return fail(MH_EINVAL, "problems is NULL");
  if (steps < 0 || steps > 16) return fail(MH_EINVAL, "steps must be in [0, 16] (got %d)", steps);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(MH_EINVAL, "eps must be >= 0");
  if (!(norm_scale > 0.0f) || !std::isfinite(norm_scale))
    return fail(MH_EINVAL, "norm_scale must be finite and > 0");
  if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c))
    return fail(MH_EINVAL, "Newton-Schulz coefficients must be finite");
  if (sched)
    for (int k = 0; k < 3 * steps; ++k)
      if (!std::isfinite(sched[k])) return fail(MH_EINVAL, "coeffs[%d] is not finite", k);
  std::vector<Shape> shapes(n);
  for (int i = 0; i < n; ++i) {
    const mh_ns_problem& p = problems[i];
    int rc = check_shape(p.views, p.rows, p.cols, i, "problems");
    if (rc != MH_OK) return rc;
    if (p.views * ceil_div(p.rows, kEwTileR) * ceil_div(p.cols, kEwTileC) >= (int64_t(1) << 31))
      return fail(MH_EUNSUPPORTED, "problems[%d]: too many elements for one problem", i);
    if (!valid_dtype(p.in_dtype) || !valid_dtype(p.out_dtype))
      return fail(MH_EDTYPE, "problems[%d]: only fp32 and bf16 dense matrices are supported", i);
    if (p.views * p.rows * p.cols > 0 && (!p.x || !p.out))
      return fail(MH_EINVAL, "problems[%d]: x and out must be non-NULL", i);
    shapes[i] = {p.views, p.rows, p.cols};
  }
  const Plan P = make_plan(shapes, false, false);
  if (P.tensors.empty()) return MH_OK;
  int rc = check_workspace(P, workspace, workspace_bytes);
  if (rc != MH_OK) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int sms = 0;
  if ((rc = device_sms(&sms)) != MH_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeaderBytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace status)");
  double* sumsq = reinterpret_cast<double*>(ws + P.off_sumsq);
  float* tile_ss = reinterpret_cast<float*>(ws + P.off_tile_ss);

  EwParams proto;
  std::memset(&proto, 0, sizeof(proto));
  proto.use_momentum = 0;
  proto.ns_eps = eps;
  proto.ns_norm_scale = norm_scale;
  proto.u_scale_from_sumsq = steps == 0 ? 1 : 0;
  int final_buf = 0;
  auto fill = [&](const TensorInfo& T, EwJob& J, int xbuf) {
    const mh_ns_problem& p = problems[T.idx];
    const ClassInfo& C = P.classes[T.cls];
    J.src = p.x;
    J.dst = p.out;
    J.src_dtype = p.in_dtype;
    J.dst_dtype = p.out_dtype;
    const bool cols4 = (T.cols % 4) == 0;
    J.src_vec = cols4 && aligned16(p.x);
    J.dst_vec = cols4 && aligned16(p.out);
    J.ldx = C.ldx;
    J.x_view_stride = C.xrows * C.ldx;
    J.stat_tiles_c = static_cast<int32_t>(T.tiles_c);
    bf16* xb = reinterpret_cast<bf16*>(ws + C.off_x[xbuf]) + T.class_slot * C.xrows * C.ldx;
    J.x0 = xb;
    J.xf = xb;
    J.sumsq = sumsq + T.view_slot;
    J.tile_ss = tile_ss + T.tile_off * (kEwThreads / 32);
  };
  rc = run_ew(EW_PROLOGUE, P, proto, [&](const TensorInfo& T, EwJob& J) { fill(T, J, 0); }, sms,
              stream);
  if (rc != MH_OK) return rc;
  if ((rc = run_view_norm(P, tile_ss, sumsq, stream)) != MH_OK) return rc;
  rc = run_ns(P, ws, steps, a, b, c, eps, sms, stream, &final_buf, false, 0, nullptr, sched,
              norm_scale);
  if (rc != MH_OK) return rc;
  return run_ew(EW_COPYOUT, P, proto,
                [&](const TensorInfo& T, EwJob& J) { fill(T, J, final_buf); }, sms, stream);
}

int mh_newton_schulz_batched(const mh_ns_problem* problems, int32_t n, int32_t steps, float a,
                             float b, float c, float eps, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!(eps > 0.0f)) return fail(MH_EINVAL, "eps must be > 0");
  return ns_impl(problems, n, steps, a, b, c, nullptr, eps, 1.0f, workspace, workspace_bytes,
                 stream);
}

int mh_newton_schulz_batched_ex(const mh_ns_problem* problems, int32_t n, int32_t steps,
                                const float* coeffs, float eps, float norm_scale,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (steps > 0 && !coeffs) return fail(MH_EINVAL, "coeffs is NULL");
  return ns_impl(problems, n, steps, 0.0f, 0.0f, 0.0f, coeffs, eps, norm_scale, workspace,
                 workspace_bytes, stream);
}

// AdamW over `n` tensors; with a control block the gradient factor, the skip
// flag and the step count are read on the device.
static int adamw_impl(const mh_adamw_tensor* tensors, int32_t n, float lr, float beta1,
                      float beta2, float eps, int64_t step, const mh_grad_control* ctl,
                      void* stream_) {
  if (n < 0) return fail(MH_EINVAL, "n must be >= 0 (got %d)", n);
  if (n > 0 && !tensors) return fail(MH_EINVAL, "tensors is NULL");
  if (ctl == nullptr && step < 1)
    return fail(MH_EINVAL, "step must be >= 1 (got %lld)", (long long)step);
  if (ctl != nullptr && (!ctl->grad_mult || !ctl->skip || !ctl->step))
    return fail(MH_EINVAL, "the control block needs grad_mult, skip and step");
  if (!std::isfinite(lr)) return fail(MH_EINVAL, "lr must be finite");
  if (!(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f))
    return fail(MH_EINVAL, "betas must be in [0, 1) (got %g, %g)", beta1, beta2);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(MH_EINVAL, "eps must be >= 0");
  for (int i = 0; i < n; ++i) {
    const mh_adamw_tensor& T = tensors[i];
    if (T.numel < 0) return fail(MH_ESHAPE, "tensors[%d]: numel must be >= 0", i);
    if (!valid_dtype(T.param_dtype) || !valid_dtype(T.grad_dtype) ||
        !valid_dtype(T.state_dtype))
      return fail(MH_EDTYPE,
                  "tensors[%d]: only fp32 and bf16 dense tensors are supported (sparse and complex "
                  "gradients are rejected)",
                  i);
    if (T.param_sr != 0 && T.param_sr != 1)
      return fail(MH_EINVAL, "tensors[%d]: param_sr must be 0 or 1", i);
    if (T.param_sr && T.param_dtype != MH_BF16)
      return fail(MH_EINVAL, "tensors[%d]: param_sr needs a bf16 parameter", i);
    if (T.numel > 0 && (!T.param || !T.grad || !T.exp_avg || !T.exp_avg_sq))
      return fail(MH_EINVAL, "tensors[%d]: param, grad, exp_avg and exp_avg_sq must be non-NULL", i);
    if (!std::isfinite(T.lr_mult) || !std::isfinite(T.wd))
      return fail(MH_EINVAL, "tensors[%d]: lr_mult and wd must be finite", i);
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  bool any = false;
  for (int i = 0; i < n; ++i) any = any || tensors[i].numel > 0;
  if (!any) return MH_OK;
  int sms = 0;
  int rc = device_sms(&sms);
  if (rc != MH_OK) return rc;
  AdamParams ap;
  std::memset(&ap, 0, sizeof(ap));
  ap.beta1 = beta1;
  ap.beta2 = beta2;
  ap.eps = eps;
  if (ctl != nullptr) {
    ap.grad_mult = ctl->grad_mult;
    ap.skip = ctl->skip;
    ap.step = ctl->step;
  } else {
    const double bc1 = 1.0 - std::pow(double(beta1), double(step));
    const double bc2 = 1.0 - std::pow(double(beta2), double(step));
    ap.inv_bc1 = static_cast<float>(1.0 / bc1);
    ap.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
    ap.sr_seed = static_cast<uint64_t>(step);
  }
  int64_t chunks = 0;
  auto flush = [&]() -> int {
    ap.total_chunks = chunks;
    double bytes = 0.0;
    for (int k = 0; k < ap.njobs; ++k)
      bytes += double(ap.jobs[k].numel) * (2.0 * dsize(ap.jobs[k].pdt) + dsize(ap.jobs[k].gdt) +
                                           4.0 * dsize(ap.jobs[k].sdt));
    ProfScope ps(stream, "adamw", bytes);
    cudaError_t e = launch_adamw(ap, sms, stream);
    ap.njobs = 0;
    chunks = 0;
    if (e != cudaSuccess) return cuda_fail(e, "AdamW launch");
    return MH_OK;
  };
  for (int i = 0; i < n; ++i) {
    const mh_adamw_tensor& T = tensors[i];
    if (T.numel == 0) continue;
    AdamJob& J = ap.jobs[ap.njobs++];
    J.param = T.param;
    J.grad = T.grad;
    J.m = T.exp_avg;
    J.v = T.exp_avg_sq;
    J.numel = T.numel;
    J.pdt = T.param_dtype;
    J.gdt = T.grad_dtype;
    J.vec = aligned16(T.param) && aligned16(T.grad) && aligned16(T.exp_avg) &&
            aligned16(T.exp_avg_sq);
    J.lr = lr * T.lr_mult;
    J.wd = T.wd;
    J.sdt = T.state_dtype;
    J.psr = T.param_sr;
    J.tindex = i;
    J.chunk_begin = chunks;
    chunks += (T.numel + kAdamChunk - 1) / kAdamChunk;
    if (ap.njobs == kMaxAdamJobs && (rc = flush()) != MH_OK) return rc;
  }
  if (ap.njobs > 0 && (rc = flush()) != MH_OK) return rc;
  return MH_OK;
}

int mh_adamw_step(const mh_adamw_tensor* tensors, int32_t n, float lr, float beta1, float beta2,
                  float eps, int64_t step, void* stream) {
  return adamw_impl(tensors, n, lr, beta1, beta2, eps, step, nullptr, stream);
}

int mh_adamw_step_ctl(const mh_adamw_tensor* tensors, int32_t n, float lr, float beta1,
                      float beta2, float eps, const mh_grad_control* ctl, void* stream) {
  if (!ctl) return fail(MH_EINVAL, "ctl is NULL");
  return adamw_impl(tensors, n, lr, beta1, beta2, eps, 0, ctl, stream);
}

// ---- QK-Clip ---------------------------------------------------------------------

int mh_qk_clip(const mh_qk_clip_entry* entries, int32_t n, const float* s_max, float tau,
               const int32_t* skip, void* stream_) {
  if (n < 0) return fail(MH_EINVAL, "n must be >= 0 (got %d)", n);
  if (n > 0 && (!entries || !s_max)) return fail(MH_EINVAL, "entries and s_max must be non-NULL");
  if (!(tau > 0.0f) || !std::isfinite(tau)) return fail(MH_EINVAL, "tau must be finite and > 0");
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    const mh_qk_clip_entry& E = entries[i];
    if (!valid_dtype(E.param_dtype)) return fail(MH_EDTYPE, "entries[%d]: fp32 or bf16 only", i);
    if (E.heads < 0 || E.rows < 0 || E.cols < 0 || E.head_stride < 0 || E.row_offset < 0 ||
        E.scaled_rows < 0 || E.head_index0 < 0)
      return fail(MH_ESHAPE, "entries[%d]: negative size or index", i);
    if (int64_t(E.heads) * E.head_stride > E.rows || E.row_offset + E.scaled_rows > E.head_stride)
      return fail(MH_ESHAPE, "entries[%d]: head blocks do not fit the weight", i);
    if (!(E.exponent >= 0.0f) || !std::isfinite(E.exponent))
      return fail(MH_EINVAL, "entries[%d]: exponent must be finite and >= 0", i);
    if (E.heads > 0 && E.scaled_rows > 0 && E.cols > 0 && !E.param)
      return fail(MH_EINVAL, "entries[%d]: param is NULL", i);
    total += int64_t(E.heads) * E.scaled_rows;
  }
  if (total == 0) return MH_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int sms = 0;
  int rc = device_sms(&sms);
  if (rc != MH_OK) return rc;
  QkClipParams qp;
  std::memset(&qp, 0, sizeof(qp));
  qp.s_max = s_max;
  qp.tau = tau;
  qp.skip = skip;
  int64_t rows = 0;
  auto flush = [&]() -> int {
    qp.total_rows = rows;
    ProfScope ps(stream, "qk_clip", 0.0);
    cudaError_t e = launch_qk_clip(qp, sms, stream);
    qp.nentries = 0;
    rows = 0;
    if (e != cudaSuccess) return cuda_fail(e, "QK-Clip launch");
    return MH_OK;
  };
  for (int i = 0; i < n; ++i) {
    const mh_qk_clip_entry& E = entries[i];
    if (E.heads == 0 || E.scaled_rows == 0 || E.cols == 0) continue;
    QkClipEntry& Q = qp.entries[qp.nentries++];
    Q.param = E.param;
    Q.cols = E.cols;
    Q.head_stride = E.head_stride;
    Q.row_offset = E.row_offset;
    Q.scaled_rows = E.scaled_rows;
    Q.head_index0 = E.head_index0;
    Q.dt = E.param_dtype;
    Q.vec = aligned16(E.param) ? 1 : 0;
    Q.exponent = E.exponent;
    Q.row_begin = rows;
    rows += int64_t(E.heads) * E.scaled_rows;
    if (qp.nentries == kMaxQkClipEntries && (rc = flush()) != MH_OK) return rc;
  }
  if (qp.nentries > 0 && (rc = flush()) != MH_OK) return rc;
  return MH_OK;
}

// ---- gradient control --------------------------------------------------------

static int check_grads(const mh_grad_ref* grads, int32_t n, int64_t* chunks) {
  if (n < 0) return fail(MH_EINVAL, "n must be >= 0 (got %d)", n);
  if (n > 0 && !grads) return fail(MH_EINVAL, "grads is NULL");
  int64_t c = 0;
  for (int i = 0; i < n; ++i) {
    const mh_grad_ref& G = grads[i];
    if (G.numel < 0) return fail(MH_ESHAPE, "grads[%d]: numel must be >= 0", i);
    if (!valid_dtype(G.grad_dtype))
      return fail(MH_EDTYPE, "grads[%d]: only fp32 and bf16 dense gradients are supported", i);
    if (G.numel > 0 && !G.grad) return fail(MH_EINVAL, "grads[%d]: grad is NULL", i);
    c += (G.numel + kGradChunk - 1) / kGradChunk;
  }
  *chunks = c;
  return MH_OK;
}

size_t mh_grad_prepare_workspace_bytes(const mh_grad_ref* grads, int32_t n) {
  int64_t chunks = 0;
  if (check_grads(grads, n, &chunks) != MH_OK) return 0;
  return static_cast<size_t>(std::max<int64_t>(chunks, 1)) * sizeof(double);
}

int mh_grad_prepare(const mh_grad_ref* grads, int32_t n, float inv_loss_scale, float max_norm,
                    const mh_grad_control* ctl, void* workspace, size_t workspace_bytes,
                    void* stream_) {
  int64_t chunks = 0;
  int rc = check_grads(grads, n, &chunks);
  if (rc != MH_OK) return rc;
  if (!(inv_loss_scale > 0.0f) || !std::isfinite(inv_loss_scale))
    return fail(MH_EINVAL, "inv_loss_scale must be finite and > 0 (got %g)", inv_loss_scale);
  if (!(max_norm >= 0.0f) || !std::isfinite(max_norm))
    return fail(MH_EINVAL, "max_norm must be finite and >= 0 (got %g)", max_norm);
  if (!ctl || !ctl->grad_mult || !ctl->skip || !ctl->norm)
    return fail(MH_EINVAL, "ctl, ctl->grad_mult, ctl->skip and ctl->norm must be non-NULL");
  const size_t need = static_cast<size_t>(std::max<int64_t>(chunks, 1)) * sizeof(double);
  if (!workspace || workspace_bytes < need)
    return fail(MH_EWORKSPACE, "workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) % 8 != 0)
    return fail(MH_EWORKSPACE, "workspace must be 8-byte aligned");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int sms = 0;
  if ((rc = device_sms(&sms)) != MH_OK) return rc;
  double* partial = static_cast<double*>(workspace);

  GradParams gp;
  std::memset(&gp, 0, sizeof(gp));
  gp.inv_scale = inv_loss_scale;
  gp.partial = partial;
  int64_t next = 0;  // global chunk index of the next tensor
  auto flush = [&]() -> int {
    gp.nchunks = next - gp.chunk_first;
    double bytes = 0.0;
    for (int k = 0; k < gp.njobs; ++k) bytes += double(gp.jobs[k].numel) * dsize(gp.jobs[k].gdt);
    ProfScope ps(stream, "grad_norm", bytes);
    cudaError_t e = launch_grad_sumsq(gp, sms, stream);
    gp.njobs = 0;
    gp.chunk_first = next;
    if (e != cudaSuccess) return cuda_fail(e, "gradient norm launch");
    return MH_OK;
  };
  for (int i = 0; i < n; ++i) {
    const mh_grad_ref& G = grads[i];
    if (G.numel == 0) continue;
    GradJob& J = gp.jobs[gp.njobs++];
    J.grad = G.grad;
    J.numel = G.numel;
    J.gdt = G.grad_dtype;
    J.vec = aligned16(G.grad) ? 1 : 0;
    J.chunk_begin = next;
    next += (G.numel + kGradChunk - 1) / kGradChunk;
    if (gp.njobs == kMaxGradJobs && (rc = flush()) != MH_OK) return rc;
  }
  if (gp.njobs > 0 && (rc = flush()) != MH_OK) return rc;

  GradFinParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.partial = partial;
  fp.nchunks = next;
  fp.inv_scale = inv_loss_scale;
  fp.max_norm = max_norm;
  fp.clip_eps = 1e-6;
  fp.mult = ctl->grad_mult;
  fp.skip = ctl->skip;
  fp.norm = ctl->norm;
  fp.step = ctl->step;
  ProfScope ps(stream, "grad_finalize", 0.0);
  cudaError_t e = launch_grad_finalize(fp, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gradient norm finalisation launch");
  return MH_OK;
}

int mh_profiler_enable(int32_t enable) {
  Profiler& P = profiler();
  std::lock_guard<std::mutex> lock(P.mu);
  P.on = enable != 0;
  return MH_OK;
}

int mh_profiler_reset(void) {
  Profiler& P = profiler();
  std::lock_guard<std::mutex> lock(P.mu);
  for (ProfRecord& r : P.records) {
    cudaEventSynchronize(r.end);
    P.pool.push_back(r.begin);
    P.pool.push_back(r.end);
  }
  P.records.clear();
  return MH_OK;
}

int mh_profiler_read(mh_kernel_stats* out, int32_t max, int32_t* count) {
  if (!count || (max > 0 && !out)) return fail(MH_EINVAL, "bad output arguments");
  Profiler& P = profiler();
  std::lock_guard<std::mutex> lock(P.mu);
  std::vector<mh_kernel_stats> agg;
  int rc = MH_OK;
  for (ProfRecord& r : P.records) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(r.end);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.begin, r.end);
    if (e != cudaSuccess) rc = cuda_fail(e, "profiler event");
    size_t k = 0;
    while (k < agg.size() && std::strcmp(agg[k].name, r.name) != 0) ++k;
    if (k == agg.size()) {
      mh_kernel_stats z;
      std::memset(&z, 0, sizeof(z));
      std::snprintf(z.name, sizeof(z.name), "%s", r.name);
      agg.push_back(z);
    }
    agg[k].launches += 1;
    agg[k].total_ms += ms;
    agg[k].bytes += r.bytes;
    agg[k].flops += r.flops;
    agg[k].flops_executed += r.flops_exec;
    P.pool.push_back(r.begin);
    P.pool.push_back(r.end);
  }
  P.records.clear();
  *count = static_cast<int32_t>(agg.size());
  for (int32_t k = 0; k < max && k < static_cast<int32_t>(agg.size()); ++k) out[k] = agg[k];
  return rc;
}

int mh_set_wait_limit(int64_t cycles) {
  if (cycles < 0) return fail(MH_EINVAL, "wait limit must be >= 0 (0 restores the default)");
  g_wait_limit.store(cycles == 0 ? kWaitLimitCycles : static_cast<long long>(cycles),
                     std::memory_order_relaxed);
  return MH_OK;
}

int64_t mh_get_wait_limit(void) { return gemm_wait_limit(); }

int mh_workspace_status(const void* workspace, void* stream_) {
  if (!workspace) return fail(MH_EWORKSPACE, "workspace is NULL");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int status = 0;
  cudaError_t e = cudaMemcpyAsync(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(status)");
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (status != 0)
    return fail(MH_ETIMEOUT, "a device-side bounded wait gave up (code %d)", status);
  return MH_OK;
}

}  // extern "C"
