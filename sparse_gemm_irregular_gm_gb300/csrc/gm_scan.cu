// gm_scan.cu -- device-wide prefix sums (gMAGNUS Algorithm 3: PrefixSum of
// C-hat.rowPtr, C-hat_reord.rowPtr and C.rowPtr).
//
// Reduce-then-scan in three launches: per-tile sums, a scan of the tile sums
// (recursively), then the per-tile scan with its offset. No block waits on
// another block, so nothing can spin.
#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int64_t kScanTile = kScanThreads * kScanItems;

__global__ void __launch_bounds__(kScanThreads) k_tile_sums(const int64_t* __restrict__ in, int64_t n,
                                                          int64_t* __restrict__ sums) {
  __shared__ int64_t ws[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile;
  int64_t acc = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    int64_t i = base + k * kScanThreads + threadIdx.x;
    if (i < n) acc += in[i];
  }
  int64_t tot;
  block_exclusive_scan(acc, ws, &tot);
  if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kScanThreads) k_tile_scan(const int64_t* in, int64_t n, int64_t* out,
                                                          const int64_t* __restrict__ offs,
                                                          int64_t* __restrict__ d_total) {
  __shared__ int64_t ws[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanItems;
  int64_t v[kScanItems];
  int64_t acc = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    int64_t i = base + k;
    v[k] = i < n ? in[i] : 0;
    acc += v[k];
  }
  int64_t tot;
  int64_t pre = block_exclusive_scan(acc, ws, &tot) + (offs ? offs[blockIdx.x] : 0);
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    int64_t i = base + k;
    if (i < n) out[i] = pre;
    pre += v[k];
  }
  if (d_total && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) *d_total = (offs ? offs[blockIdx.x] : 0) + tot;
}

__global__ void k_segmented_offsets(const int64_t* val, int64_t* off, const int64_t* __restrict__ base,
                                    int64_t n_parents, int v, int64_t* __restrict__ sums) {
  // One warp per parent: v <= 1 << 16 children scanned 32 at a time.
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t p = warp; p < n_parents; p += nw) {
    int64_t run = base ? base[p] : 0;
    const int64_t start = run;
    for (int c0 = 0; c0 < v; c0 += 32) {
      const int c = c0 + lane;
      int64_t x = c < v ? val[p * v + c] : 0;
      int64_t inc = warp_inclusive_scan(x);
      if (c < v) off[p * v + c] = run + inc - x;
      run += __shfl_sync(kFull, inc, 31);
    }
    if (sums && lane == 0) sums[p] = run - start;
  }
}

__global__ void k_sum_children(const int64_t* __restrict__ src, const int64_t* __restrict__ slot,
                               int64_t* __restrict__ dst, int64_t n_parents, int v) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t p = warp; p < n_parents; p += nw) {
    int64_t acc = 0;
    for (int c = lane; c < v; c += 32) acc += src[p * v + c];
    acc = warp_reduce_sum(acc);
    if (lane == 0) dst[slot[p]] = acc;
  }
}

}  // namespace

bool scan_exclusive_i64(const int64_t* in, int64_t* out, int64_t n, int64_t* d_total, cudaStream_t s) {
  if (n <= 0) {
    if (d_total) cudaMemsetAsync(d_total, 0, sizeof(int64_t), s);
    return true;
  }
  const int64_t tiles = (n + kScanTile - 1) / kScanTile;
  if (tiles == 1) {
    (k_tile_scan<<<1, kScanThreads, 0, s>>>(in, n, out, nullptr, d_total), note_launch());
    return true;
  }
  DevBuf<int64_t> sums;
  if (!sums.alloc(tiles, s)) return false;
  (k_tile_sums<<<static_cast<unsigned>(tiles), kScanThreads, 0, s>>>(in, n, sums.p), note_launch());
  if (!scan_exclusive_i64(sums.p, sums.p, tiles, nullptr, s)) return false;
  (k_tile_scan<<<static_cast<unsigned>(tiles), kScanThreads, 0, s>>>(in, n, out, sums.p, d_total), note_launch());
  return true;
}

int64_t scan_scratch_elems(int64_t n) {
  int64_t need = 0;
  while (n > kScanTile) {
    n = (n + kScanTile - 1) / kScanTile;
    need += n;
  }
  return need;
}

bool scan_exclusive_i64_scratch(const int64_t* in, int64_t* out, int64_t n, int64_t* d_total, int64_t* scratch,
                                int64_t scratch_elems, cudaStream_t s) {
  if (n <= 0) {
    if (d_total) cudaMemsetAsync(d_total, 0, sizeof(int64_t), s);
    return true;
  }
  const int64_t tiles = (n + kScanTile - 1) / kScanTile;
  if (tiles == 1) {
    (k_tile_scan<<<1, kScanThreads, 0, s>>>(in, n, out, nullptr, d_total), note_launch());
    return true;
  }
  if (scratch_elems < tiles) return false;
  (k_tile_sums<<<static_cast<unsigned>(tiles), kScanThreads, 0, s>>>(in, n, scratch), note_launch());
  if (!scan_exclusive_i64_scratch(scratch, scratch, tiles, nullptr, scratch + tiles, scratch_elems - tiles, s))
    return false;
  (k_tile_scan<<<static_cast<unsigned>(tiles), kScanThreads, 0, s>>>(in, n, out, scratch, d_total), note_launch());
  return true;
}

void segmented_offsets(const int64_t* val, int64_t* off, const int64_t* base, int64_t n_parents, int v,
                       int64_t* sums, cudaStream_t s) {
  if (n_parents <= 0) return;
  (k_segmented_offsets<<<grid_for(n_parents * 32, 256), 256, 0, s>>>(val, off, base, n_parents, v, sums), note_launch());
}

void sum_children(const int64_t* src, const int64_t* parent_slot, int64_t* dst, int64_t n_parents, int v,
                  cudaStream_t s) {
  if (n_parents <= 0) return;
  (k_sum_children<<<grid_for(n_parents * 32, 256), 256, 0, s>>>(src, parent_slot, dst, n_parents, v), note_launch());
}

}  // namespace gm
