// gm_analyze.cu -- setup phase of gMAGNUS (Algorithm 3 lines 3-4, Sec. III-A):
// input validation, per-row intermediate-product counts (InterOffsets) and the
// order-preserving partition of rows into size bins (ThreshPartition, extended
// with the binning of light rows by size described in Sec. III-E).
#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

__global__ void k_validate_rowptr(const int64_t* __restrict__ rp, int64_t n_rows, int64_t nnz, int bad_bit,
                                  int* status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i <= n_rows; i += stride) {
    const int64_t r = rp[i];
    if (i == 0 && r != 0) bad = true;
    if (i == n_rows && r != nnz) bad = true;
    if (i < n_rows && rp[i + 1] < r) bad = true;
    if (r < 0 || r > nnz) bad = true;
  }
  if (__any_sync(kFull, bad) && (threadIdx.x & 31) == 0) atomicOr(status, bad_bit);
}

__global__ void k_validate_cols(const int32_t* __restrict__ col, int64_t nnz, int64_t n_cols, int bad_bit,
                                int* status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nnz; i += stride) {
    const int64_t c = col[i];
    if (c < 0 || c >= n_cols) bad = true;
  }
  if (__any_sync(kFull, bad) && (threadIdx.x & 31) == 0) atomicOr(status, bad_bit);
}

// *flags |= 1 when some row has a column greater than the next one in that row,
// |= 2 when some row holds a column twice in a row (one warp per row, lanes
// compare neighbouring entries).
__global__ void k_rows_sorted(const int64_t* __restrict__ rp, const int32_t* __restrict__ col, int64_t n_rows,
                              int* flags) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  bool down = false, same = false;
  for (int64_t r = warp; r < n_rows; r += nw)
    for (int64_t q = rp[r] + lane; q + 1 < rp[r + 1]; q += 32) {
      down |= col[q] > col[q + 1];
      same |= col[q] == col[q + 1];
    }
  const int f = (__any_sync(kFull, down) ? 1 : 0) | (__any_sync(kFull, same) ? 2 : 0);
  if (f && lane == 0) atomicOr(flags, f);
}

__device__ __forceinline__ uint8_t bin_of(int64_t size, const BinSpec& spec) {
  if (size == 0) return 0;
  int b = 1;
  while (b < spec.nbins - 1 && size > spec.ub[b]) ++b;
  return static_cast<uint8_t>(b);
}

// One warp per row: lanes read A's entries of the row (coalesced) and gather
// the length of the B row each one selects.
__global__ void k_ip_count(const int64_t* __restrict__ a_rp, const int32_t* __restrict__ a_col, int64_t n_rows,
                           const int64_t* __restrict__ b_rp, int64_t* __restrict__ u, uint8_t* __restrict__ bin,
                           BinSpec spec) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t i = warp; i < n_rows; i += nw) {
    const int64_t lo = a_rp[i], hi = a_rp[i + 1];
    int64_t acc = 0;
    for (int64_t p = lo + lane; p < hi; p += 32) {
      const int k = a_col[p];
      acc += b_rp[k + 1] - b_rp[k];
    }
    acc = warp_reduce_sum(acc);
    if (lane == 0) {
      u[i] = acc;
      bin[i] = bin_of(acc, spec);
    }
  }
}

__global__ void k_bin_sizes(const int64_t* __restrict__ size, int64_t n, uint8_t* __restrict__ bin, BinSpec spec) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    bin[i] = bin_of(size[i], spec);
}

constexpr int kPartThreads = 1024;
constexpr int kPartRounds = 4;
constexpr int64_t kPartTile = kPartThreads * kPartRounds;

// Per-tile bin counts: counts[b * n_tiles + tile].
__global__ void __launch_bounds__(kPartThreads) k_part_count(const uint8_t* __restrict__ bin, int64_t n,
                                                             int nbins, int64_t n_tiles,
                                                             int64_t* __restrict__ counts) {
  __shared__ int cnt[kMaxBins];
  if (threadIdx.x < kMaxBins) cnt[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kPartTile;
  for (int r = 0; r < kPartRounds; ++r) {
    const int64_t i = base + r * kPartThreads + threadIdx.x;
    const int b = i < n ? bin[i] : -1;
    const unsigned peers = __match_any_sync(kFull, b);
    if (b >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&cnt[b], __popc(peers));
  }
  __syncthreads();
  if (threadIdx.x < nbins) counts[static_cast<int64_t>(threadIdx.x) * n_tiles + blockIdx.x] = cnt[threadIdx.x];
}

// Stable scatter: position = tile offset of the bin + rank among earlier items of
// the same bin within the tile (round, warp, lane order = index order).
__global__ void __launch_bounds__(kPartThreads) k_part_scatter(const uint8_t* __restrict__ bin, int64_t n,
                                                               int nbins, int64_t n_tiles,
                                                               const int64_t* __restrict__ offs,
                                                               int32_t* __restrict__ out_idx) {
  __shared__ int wcnt[32][kMaxBins];
  __shared__ int rtot[kMaxBins];
  __shared__ int64_t run[kMaxBins];
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x < nbins) run[threadIdx.x] = offs[static_cast<int64_t>(threadIdx.x) * n_tiles + blockIdx.x];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kPartTile;
  for (int r = 0; r < kPartRounds; ++r) {
    for (int k = threadIdx.x; k < 32 * kMaxBins; k += kPartThreads) (&wcnt[0][0])[k] = 0;
    __syncthreads();
    const int64_t i = base + r * kPartThreads + threadIdx.x;
    const int b = i < n ? bin[i] : -1;
    const unsigned peers = __match_any_sync(kFull, b);
    const int rank = __popc(peers & lanemask_lt());
    if (b >= 0 && rank == 0) wcnt[warp][b] = __popc(peers);
    __syncthreads();
    if (threadIdx.x < nbins) {  // exclusive scan over warps, one thread per bin
      int acc = 0;
      for (int w = 0; w < 32; ++w) {
        const int c = wcnt[w][threadIdx.x];
        wcnt[w][threadIdx.x] = acc;
        acc += c;
      }
      rtot[threadIdx.x] = acc;
    }
    __syncthreads();
    if (b >= 0) out_idx[run[b] + wcnt[warp][b] + rank] = static_cast<int32_t>(i);
    __syncthreads();
    if (threadIdx.x < nbins) run[threadIdx.x] += rtot[threadIdx.x];
  }
}

__global__ void k_bin_starts(const int64_t* __restrict__ offs, int nbins, int64_t n_tiles, int64_t n,
                             int64_t* __restrict__ starts) {
  const int b = threadIdx.x;
  if (b < nbins) starts[b] = offs[static_cast<int64_t>(b) * n_tiles];
  if (b == nbins) starts[b] = n;
}

__global__ void k_gather_i64(const int64_t* __restrict__ src, const int32_t* __restrict__ idx, int64_t n,
                             int64_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = src[idx[i]];
}
__global__ void k_gather_i64_i64(const int64_t* __restrict__ src, const int64_t* __restrict__ idx, int64_t n,
                                 int64_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = src[idx[i]];
}
__global__ void k_scatter_i64(const int64_t* __restrict__ src, const int32_t* __restrict__ idx, int64_t n,
                              int64_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[idx[i]] = src[i];
}
__global__ void k_iota_i64(int64_t* __restrict__ dst, int64_t n, int64_t start) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = start + i;
}
__global__ void k_fill_i64(int64_t* __restrict__ dst, int64_t n, int64_t v) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = v;
}

// out[i] = in[i] widened to 64 bits.
__global__ void k_widen_i32(const int32_t* __restrict__ in, int64_t* __restrict__ out, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) out[i] = in[i];
}

// out[i] = in[i] narrowed to 32 bits when it lies in [0, bound), else -1 (which
// the index validation that follows reports; bound <= 2^31).
__global__ void k_narrow_i64(const int64_t* __restrict__ in, int32_t* __restrict__ out, int64_t n, int64_t bound) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t v = in[i];
    out[i] = v >= 0 && v < bound ? static_cast<int32_t>(v) : -1;
  }
}

}  // namespace

void launch_widen_i32(const int32_t* in, int64_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return;
  (k_widen_i32<<<grid_for(n, 256), 256, 0, s>>>(in, out, n), note_launch());
}

void launch_narrow_i64(const int64_t* in, int32_t* out, int64_t n, int64_t bound, cudaStream_t s) {
  if (n <= 0) return;
  (k_narrow_i64<<<grid_for(n, 256), 256, 0, s>>>(in, out, n, bound), note_launch());
}

void launch_validate_rowptr(const int64_t* rp, int64_t n_rows, int64_t nnz, int bad_bit, int* status,
                            cudaStream_t s) {
  (k_validate_rowptr<<<grid_for(n_rows + 1, 256), 256, 0, s>>>(rp, n_rows, nnz, bad_bit, status), note_launch());
}

void launch_validate_cols(const int32_t* col, int64_t nnz, int64_t n_cols, int bad_bit, int* status,
                          cudaStream_t s) {
  if (nnz <= 0) return;
  (k_validate_cols<<<grid_for(nnz, 256), 256, 0, s>>>(col, nnz, n_cols, bad_bit, status), note_launch());
}

void launch_check_sorted(const int64_t* rp, const int32_t* col, int64_t n_rows, int* flags, cudaStream_t s) {
  if (n_rows <= 0) return;
  (k_rows_sorted<<<grid_for(n_rows * 32, 256), 256, 0, s>>>(rp, col, n_rows, flags), note_launch());
}

void launch_ip_count(const int64_t* a_rp, const int32_t* a_col, int64_t n_rows, const int64_t* b_rp,
                     int64_t* u, uint8_t* bin, BinSpec spec, cudaStream_t s) {
  if (n_rows <= 0) return;
  (k_ip_count<<<grid_for(n_rows * 32, 256), 256, 0, s>>>(a_rp, a_col, n_rows, b_rp, u, bin, spec), note_launch());
}

void launch_bin_sizes(const int64_t* size, int64_t n, uint8_t* bin, BinSpec spec, cudaStream_t s) {
  if (n <= 0) return;
  (k_bin_sizes<<<grid_for(n, 256), 256, 0, s>>>(size, n, bin, spec), note_launch());
}

bool partition_by_bin(const uint8_t* bin, int64_t n, int nbins, int32_t* out_idx, int64_t* d_bin_start,
                      cudaStream_t s) {
  if (n <= 0) {
    cudaMemsetAsync(d_bin_start, 0, (nbins + 1) * sizeof(int64_t), s);
    return true;
  }
  const int64_t tiles = (n + kPartTile - 1) / kPartTile;
  DevBuf<int64_t> counts;
  if (!counts.alloc(static_cast<size_t>(tiles) * nbins, s)) return false;
  (k_part_count<<<static_cast<unsigned>(tiles), kPartThreads, 0, s>>>(bin, n, nbins, tiles, counts.p), note_launch());
  if (!scan_exclusive_i64(counts.p, counts.p, tiles * nbins, nullptr, s)) return false;
  (k_part_scatter<<<static_cast<unsigned>(tiles), kPartThreads, 0, s>>>(bin, n, nbins, tiles, counts.p, out_idx), note_launch());
  (k_bin_starts<<<1, 32, 0, s>>>(counts.p, nbins, tiles, n, d_bin_start), note_launch());
  return true;
}

void launch_gather_i64(const int64_t* src, const int32_t* idx, int64_t n, int64_t* dst, cudaStream_t s) {
  if (n <= 0) return;
  (k_gather_i64<<<grid_for(n, 256), 256, 0, s>>>(src, idx, n, dst), note_launch());
}
void launch_gather_i64_i64(const int64_t* src, const int64_t* idx, int64_t n, int64_t* dst, cudaStream_t s) {
  if (n <= 0) return;
  (k_gather_i64_i64<<<grid_for(n, 256), 256, 0, s>>>(src, idx, n, dst), note_launch());
}
void launch_scatter_i64(const int64_t* src, const int32_t* idx, int64_t n, int64_t* dst, cudaStream_t s) {
  if (n <= 0) return;
  (k_scatter_i64<<<grid_for(n, 256), 256, 0, s>>>(src, idx, n, dst), note_launch());
}
void launch_iota_i64(int64_t* dst, int64_t n, int64_t start, cudaStream_t s) {
  if (n <= 0) return;
  (k_iota_i64<<<grid_for(n, 256), 256, 0, s>>>(dst, n, start), note_launch());
}
void launch_fill_i64(int64_t* dst, int64_t n, int64_t value, cudaStream_t s) {
  if (n <= 0) return;
  (k_fill_i64<<<grid_for(n, 256), 256, 0, s>>>(dst, n, value), note_launch());
}

}  // namespace gm
