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
// is looked up once per device with cudaGetSymbolAddress and handed to the
// kernels. All calls share the array, so calls whose work overlaps on the GPU
// (other streams, other threads) race and must be serialised by the caller.
// Each call writes every scratch entry it later reads, so nothing needs clearing
// between calls; the array keeps whatever the last call left there.
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
int64_t* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scan_scratch on the current device (looked up once per device).
gm_status scratch_for_current_device(int64_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_scan_scratch);
    if (e != cudaSuccess || !ptr) {
      cudaGetLastError();
      return GM_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<int64_t*>(ptr);
  }
  *out = g_scratch_addr[dev];
  return GM_OK;
}

}  // namespace

}  // namespace gm

extern "C" gm_status gm_prefix_sum_noalloc(const int64_t* in, int64_t* out, int64_t n, int64_t* total,
                                           void* stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return GM_ERR_INVALID_ARG;
  if (n > gm::kNoAllocMaxN) return GM_ERR_WORKSPACE;
  int64_t* scratch = nullptr;
  const gm_status st = gm::scratch_for_current_device(&scratch);
  if (st != GM_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!gm::scan_exclusive_i64_scratch(in, out, n, total, scratch, gm::kNoAllocScratchElems, s))
    return GM_ERR_WORKSPACE;
  const cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GM_ERR_CUDA;
  }
  return GM_OK;
}
