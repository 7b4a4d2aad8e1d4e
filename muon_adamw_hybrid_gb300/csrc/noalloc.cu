// Batched Newton-Schulz for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace buffer: a plugin that a
// host application hands only its input and output buffers, or a program
// whose device memory is already fully reserved by its own pool allocator,
// cannot call cudaMalloc (or any allocating library routine) and cannot hold
// a separate scratch buffer across calls. This entry point serves them: its
// scratch space is a fixed array compiled into the library, so the call
// itself allocates nothing. The caller still passes the inputs and outputs.
//
// Limits and sharing rules:
//   - The array holds kStaticScratchBytes (64 MiB). Problems whose workspace
//     (mh_ns_workspace_bytes) would exceed it are rejected with
//     MH_EWORKSPACE before any work is enqueued. For scale: one 2048 x 2048
//     matrix needs 32 MiB, one 1024 x 4096 matrix 20 MiB.
//   - Every GPU that loads the library holds its own copy of the array until
//     the process exits.
//   - All calls on a device share that device's array and it keeps the last
//     call's contents. Calls whose work overlaps on the GPU (for example on
//     two streams without ordering between them) race on it and give wrong
//     results: order them on one stream or with events.
//   - The first call on each device (and again after the device's context
//     was destroyed, e.g. by cudaDeviceReset) looks up the array's device
//     address with that device current (cudaGetSymbolAddress). Make that
//     first call before starting any stream capture on the device.
#include <cstdio>
#include <map>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "mh_internal.h"
#include "muonhybrid.h"

namespace {

constexpr size_t kStaticScratchBytes = MH_NS_STATIC_SCRATCH_BYTES;

// The scratch space itself. Host code must not use this name as a device
// address: on the host it denotes a stand-in object, so the real address is
// looked up per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_ns_scratch[kStaticScratchBytes];

// The driver's context calls, looked up once through the runtime (the
// library links only the runtime).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

bool context_id(unsigned long long* id) {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
         get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_ns_scratch in the current device's context. It is
// looked up once per device and context: the cache is keyed by the
// context's unique id, so a context created after cudaDeviceReset (where the
// array may sit elsewhere) gets a fresh lookup. Returns nullptr and sets the
// error message on failure.
void* scratch_for_current_device() {
  static std::mutex mu;
  static std::map<std::pair<int, unsigned long long>, void*> addr;
  int dev = 0;
  char msg[256];
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    std::snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    mh::set_last_error(msg);
    return nullptr;
  }
  unsigned long long ctx = 0;
  std::lock_guard<std::mutex> lock(mu);
  // No context yet (the process's first CUDA call): the lookup below
  // creates the primary context, and the address is cached under its id.
  if (context_id(&ctx)) {
    auto it = addr.find(std::make_pair(dev, ctx));
    if (it != addr.end()) return it->second;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_ns_scratch);
  if (e != cudaSuccess || p == nullptr) {
    std::snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(scratch) on device %d: %s", dev,
                  cudaGetErrorString(e));
    mh::set_last_error(msg);
    return nullptr;
  }
  // Without a context id the address is looked up again on the next call.
  if (context_id(&ctx)) addr[std::make_pair(dev, ctx)] = p;
  return p;
}

}  // namespace

extern "C" int mh_newton_schulz_batched_noalloc(const mh_ns_problem* problems, int32_t n,
                                                int32_t steps, float a, float b, float c,
                                                float eps, void* stream) {
  // Size check first: it needs no device and rejects oversized requests
  // before anything is enqueued.
  const size_t need = mh_ns_workspace_bytes(problems, n);
  if (need == 0 && n > 0) return MH_EINVAL;  // invalid problem list; message already set
  if (need > kStaticScratchBytes) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "these problems need %zu bytes of scratch; the allocation-free entry point "
                  "holds at most %zu bytes (use mh_newton_schulz_batched with a workspace)",
                  need, kStaticScratchBytes);
    mh::set_last_error(msg);
    return MH_EWORKSPACE;
  }
  void* ws = scratch_for_current_device();
  if (ws == nullptr) return MH_ECUDA;
  // The regular entry point clears the status word at the start of each call
  // and overwrites every other part of the workspace before reading it, so
  // nothing left in the array by an earlier call is ever used.
  return mh_newton_schulz_batched(problems, n, steps, a, b, c, eps, ws, kStaticScratchBytes,
                                  stream);
}
