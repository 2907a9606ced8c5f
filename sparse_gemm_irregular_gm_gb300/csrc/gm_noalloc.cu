// gm_noalloc.cu -- exclusive prefix sum over int64 that allocates no memory.
//
// Who needs it: code that may not call cudaMalloc or any allocator while it
// runs -- for example work recorded into a CUDA graph (allocation calls are not
// allowed during stream capture), host callbacks and real-time loops that must
// not block on the allocator, or a host application whose framework owns all
// device memory and forbids other libraries from taking more. Such callers pass
// their input and output buffers and get the scan that C.rowPtr uses, with its
// per-block partial sums kept in a fixed array of this library.
//
// The scratch is a file-scope __device__ array (g_scan_scratch): every device
// that loads the library holds it until the process exits. Host code never
// dereferences its name (on the host it is only a stand-in); the device address
// is looked up with cudaGetSymbolAddress and handed to the kernels. The address
// belongs to one CUDA context: it is cached per device together with the id of
// the context it was taken in, and looked up again when the device's current
// context is another one (after cudaDeviceReset, say, the module is loaded anew
// and the old address is gone). All calls share the array, so calls whose work
// overlaps on the GPU (other streams, other threads) race and must be
// serialised by the caller. Each call writes every scratch entry it later reads,
// so nothing needs clearing between calls; the array keeps whatever the last
// call left there.
#include <cuda.h>

#include <mutex>

#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

// Up to 65536 partial sums of 2048 elements, plus the second level's 32.
constexpr int64_t kNoAllocScratchElems = 65536 + 64;
constexpr int64_t kNoAllocMaxN = int64_t(65536) * 2048;  // 134,217,728 elements

static __device__ __align__(256) int64_t g_scan_scratch[kNoAllocScratchElems];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // context the address was taken in (0: none yet)
  int64_t* addr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the current thread's CUDA context (0 when there is none or the driver
// cannot say). The driver entry points come through the runtime, so the library
// needs no link against the driver library.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    looked_up = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
  }
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_scan_scratch in the current device's current context,
// looked up when the device or its context is new to this table.
gm_status scratch_for_current_device(int64_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const unsigned long long id = current_context_id();
  ScratchAddr& c = g_scratch[dev];
  if (!c.addr || id == 0 || c.ctx_id != id) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_scan_scratch);  // also makes the device's primary context current
    if (e != cudaSuccess || !ptr) {
      cudaGetLastError();
      return GM_ERR_CUDA;
    }
    c.addr = static_cast<int64_t*>(ptr);
    c.ctx_id = current_context_id();  // the context the lookup used (0: look up on every call)
  }
  *out = c.addr;
  return GM_OK;
}

}  // namespace

}  // namespace gm

extern "C" gm_status gm_prefix_sum_noalloc(const int64_t* in, int64_t* out, int64_t n, int64_t* total,
                                           void* stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return GM_ERR_INVALID_ARG;
  if (n > gm::kNoAllocMaxN) return GM_ERR_WORKSPACE;
  // An error left pending by earlier work belongs to that work: report it
  // without clearing it and queue nothing, so that a failure of this call's own
  // launches below is never confused with it.
  if (cudaPeekAtLastError() != cudaSuccess) return GM_ERR_CUDA;
  int64_t* scratch = nullptr;
  const gm_status st = gm::scratch_for_current_device(&scratch);
  if (st != GM_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!gm::scan_exclusive_i64_scratch(in, out, n, total, scratch, gm::kNoAllocScratchElems, s))
    return GM_ERR_WORKSPACE;
  if (cudaGetLastError() != cudaSuccess) return GM_ERR_CUDA;  // a launch of this call failed
  return GM_OK;
}
