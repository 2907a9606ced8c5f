// gm_device.cuh -- small device helpers: warp and block scans, grid sizing.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gm {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Runs of equal keys in consecutive lanes. run_heads() returns the ballot of the
// lanes that start a run; keys equal but not adjacent form separate runs (each
// run then makes its own update, which stays correct).
template <class K>
__device__ __forceinline__ unsigned run_heads(K key) {
  const int lane = threadIdx.x & 31;
  const K prev = __shfl_up_sync(kFull, key, 1);
  return __ballot_sync(kFull, lane == 0 || prev != key);
}
// First lane of the run holding this lane.
__device__ __forceinline__ int run_head_lane(unsigned heads) {
  const int lane = threadIdx.x & 31;
  const unsigned le = lane == 31 ? kFull : ((2u << lane) - 1u);
  return 31 - __clz(heads & le);
}
// Length of the run starting at this lane (meaningful on head lanes).
__device__ __forceinline__ int run_length(unsigned heads) {
  const int lane = threadIdx.x & 31;
  const unsigned after = lane == 31 ? 0u : (heads & ~((2u << lane) - 1u));
  return (after ? __ffs(after) - 1 : 32) - lane;
}

template <class T>
__device__ __forceinline__ T warp_inclusive_scan(T x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T y = __shfl_up_sync(kFull, x, d);
    if (lane >= d) x += y;
  }
  return x;
}

template <class T>
__device__ __forceinline__ T warp_reduce_sum(T x) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) x += __shfl_xor_sync(kFull, x, d);
  return x;
}

// Exclusive block-wide scan of one value per thread. `warp_sums` must hold 33
// elements (blockDim.x <= 1024). Returns the exclusive prefix; *total gets the block sum.
// Contains two __syncthreads(); every thread of the block must call it.
template <class T>
__device__ __forceinline__ T block_exclusive_scan(T x, T* warp_sums, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  T inc = warp_inclusive_scan(x);
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nwarps ? warp_sums[lane] : T(0);
    T wi = warp_inclusive_scan(w);
    if (lane < nwarps) warp_sums[lane] = wi - w;
    if (lane == nwarps - 1) warp_sums[32] = wi;
  }
  __syncthreads();
  T res = warp_sums[warp] + inc - x;
  if (total) *total = warp_sums[32];
  return res;
}

inline unsigned grid_for(int64_t n, int block, int64_t max_blocks = 152 * 64) {
  int64_t g = (n + block - 1) / block;
  if (g < 1) g = 1;
  if (g > max_blocks) g = max_blocks;
  return static_cast<unsigned>(g);
}

}  // namespace gm
