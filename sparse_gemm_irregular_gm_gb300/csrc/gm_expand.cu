// gm_expand.cu -- heavy-row expansion of gMAGNUS (Algorithm 3 lines 7-8).
//
// * Masked CSR -> CSC of A[x_heavy, :] by a counting sort over columns (the
//   pages use a key-value sort; a counting sort is that sort for integer keys).
//   B-tilde, the rows of B selected by the non-empty columns of A-tilde, is not
//   copied: slice k reads row k of B in place through B.rowPtr.
// * OuterProduct (Sec. III-B, Algorithm 4): the flattened index space of all
//   slices A-tilde[:,k] (x) B[k,:] is cut statically into work groups of E
//   elements. A work group reserves, per A-tilde entry it touches, a contiguous
//   range of that entry's C-hat row with one atomic add on the row's cursor, then
//   writes consecutive B-row elements to consecutive C-hat positions.
#include <algorithm>

#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

__global__ void k_col_count(TransposeArgs a, unsigned long long* __restrict__ cnt) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t h = warp; h < a.n_batch; h += nw) {
    const int64_t r = a.heavy_rows[h];
    for (int64_t p = a.a_rp[r] + lane; p < a.a_rp[r + 1]; p += 32) atomicAdd(&cnt[a.a_col[p]], 1ull);
  }
}

template <typename V>
__global__ void k_csc_fill(TransposeArgs a, unsigned long long* __restrict__ cursor, int32_t* __restrict__ t_row,
                           V* __restrict__ t_val) {
  const V* __restrict__ a_val = static_cast<const V*>(a.a_val);
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t h = warp; h < a.n_batch; h += nw) {
    const int64_t r = a.heavy_rows[h];
    for (int64_t p = a.a_rp[r] + lane; p < a.a_rp[r + 1]; p += 32) {
      const unsigned long long pos = atomicAdd(&cursor[a.a_col[p]], 1ull);
      t_row[pos] = static_cast<int32_t>(h);
      t_val[pos] = a_val[p];
    }
  }
}

__global__ void k_slice_sizes(const int64_t* __restrict__ col_ptr, const int64_t* __restrict__ b_rp, int64_t n,
                              int64_t* __restrict__ size) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n; k += stride)
    size[k] = (col_ptr[k + 1] - col_ptr[k]) * (b_rp[k + 1] - b_rp[k]);
}

// wg[g] = the slice holding flattened position g * E: the largest s with
// off[s] <= g * E (a non-empty slice; off has n_slices + 1 entries). One thread
// per work group, binary search.
__global__ void k_wg_slice(const int64_t* __restrict__ off, int64_t n_slices, int64_t E, int64_t n_wg,
                           int32_t* __restrict__ wg) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < n_wg; g += stride) {
    const int64_t x = g * E;
    int64_t lo = 0, hi = n_slices - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (off[mid] <= x) lo = mid; else hi = mid - 1;
    }
    wg[g] = static_cast<int32_t>(lo);
  }
}

__global__ void k_copy_u64(const int64_t* __restrict__ src, unsigned long long* __restrict__ dst, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = static_cast<unsigned long long>(src[i]);
}

constexpr int kOpThreads = 512;
constexpr int kOpCap = 512;  // A-tilde entries handled per round (one per thread)

// largest s in [lo, hi] with arr[s] <= x (arr non-decreasing, arr[lo] <= x)
__device__ __forceinline__ int64_t upper_floor(const int64_t* __restrict__ arr, int64_t lo, int64_t hi, int64_t x) {
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (arr[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename V, bool VAL, bool HISTO>
__global__ void __launch_bounds__(kOpThreads) k_outer(OuterArgs a) {
  const V* __restrict__ t_val = static_cast<const V*>(a.t_val);
  const V* __restrict__ b_val = static_cast<const V*>(a.b_val);
  V* __restrict__ out_val = static_cast<V*>(a.out_val);
  __shared__ int32_t s_lo[kOpCap];      // local flattened start of each entry's portion
  __shared__ int64_t s_dst[kOpCap];     // C-hat index of local position p: s_dst + p
  __shared__ int64_t s_b[kOpCap];       // B index of local position p: s_b + p
  __shared__ V s_a[kOpCap];
  __shared__ int32_t s_row[kOpCap];
  __shared__ int s_end;
  const int64_t S = static_cast<int64_t>(blockIdx.x) * a.E;
  const int64_t end = min(S + a.E, a.total);
  const int64_t s0 = a.wg_first[blockIdx.x];
  // slice of the last element: largest s with slice_off[s] <= end-1
  const int64_t s1 = upper_floor(a.slice_off, s0, a.n_slices - 1, end - 1);
  const int64_t lb0 = a.b_rp[s0 + 1] - a.b_rp[s0];
  const int64_t lb1 = a.b_rp[s1 + 1] - a.b_rp[s1];
  const int64_t a0 = a.col_ptr[s0] + (S - a.slice_off[s0]) / lb0;
  const int64_t a1 = a.col_ptr[s1] + (end - 1 - a.slice_off[s1]) / lb1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int64_t rs = a0; rs <= a1; rs += kOpCap) {
    const int nr = static_cast<int>(min(static_cast<int64_t>(kOpCap), a1 - rs + 1));
    if (threadIdx.x == 0) s_end = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < nr; j += blockDim.x) {
      const int64_t e = rs + j;
      const int64_t s = upper_floor(a.col_ptr, s0, s1, e);
      const int64_t lb = a.b_rp[s + 1] - a.b_rp[s];
      const int64_t seg = a.slice_off[s] + (e - a.col_ptr[s]) * lb;
      const int64_t lo = max(S, seg), hi = min(end, seg + lb);
      const int64_t cnt = hi > lo ? hi - lo : 0;
      const int lo_loc = static_cast<int>(min(max(lo, S), end) - S);
      s_lo[j] = lo_loc;
      if (cnt > 0) {
        const int32_t row = a.t_row[e];
        const unsigned long long d = atomicAdd(&a.cursor[row], static_cast<unsigned long long>(cnt));
        s_dst[j] = static_cast<int64_t>(d) - lo_loc;
        s_b[j] = a.b_rp[s] + (lo - seg) - lo_loc;
        s_a[j] = VAL ? t_val[e] : V(0);
        s_row[j] = row;
        atomicMax(&s_end, static_cast<int>(hi - S));
      }
    }
    __syncthreads();
    const int p_beg = s_lo[0], p_end = s_end;
    int j = 0;
    for (int base = p_beg + warp * 32; base < p_end; base += nwarps * 32) {
      const int p = base + lane;
      const bool ok = p < p_end;
      // largest j with s_lo[j] <= p; entries only move forward with p. Fast path:
      // the lane is still inside the warp's current entry.
      int lo_j = j;
      if (lo_j + 1 < nr && s_lo[lo_j + 1] <= p) {
        int hi_j = nr - 1;
        while (lo_j < hi_j) {
          const int mid = (lo_j + hi_j + 1) >> 1;
          if (s_lo[mid] <= p) lo_j = mid; else hi_j = mid - 1;
        }
      }
      const int jj = lo_j;
      j = __shfl_sync(kFull, jj, 0);
      int32_t col = 0;
      if (ok) {
        const int64_t bi = s_b[jj] + p;
        col = a.b_col[bi];
        const int64_t d = s_dst[jj] + p;
        a.out_col[d] = col;
        if (VAL) out_val[d] = s_a[jj] * b_val[bi];
      }
      if (HISTO) {
        const unsigned long long key =
            ok ? static_cast<unsigned long long>(s_row[jj]) * a.v + (static_cast<uint32_t>(col) >> a.shift)
               : ~0ull;
        const unsigned heads = run_heads(key);
        if (ok && ((heads >> lane) & 1u))
          atomicAdd(&a.histo[key], static_cast<unsigned long long>(run_length(heads)));
      }
    }
    __syncthreads();
  }
}

}  // namespace

bool masked_transpose(const TransposeArgs& a, int64_t nnz_batch, int64_t* col_ptr, int32_t* t_row,
                      void* t_val, cudaStream_t s) {
  DevBuf<unsigned long long> cnt;
  if (!cnt.alloc(a.n_cols + 1, s)) return false;
  cudaMemsetAsync(cnt.p, 0, (a.n_cols + 1) * sizeof(unsigned long long), s);
  if (a.n_batch > 0) (k_col_count<<<grid_for(a.n_batch * 32, 256), 256, 0, s>>>(a, cnt.p), note_launch());
  // counts -> exclusive offsets; the extra last slot (zero) receives the total
  if (!scan_exclusive_i64(reinterpret_cast<int64_t*>(cnt.p), col_ptr, a.n_cols + 1, nullptr, s)) return false;
  (k_copy_u64<<<grid_for(a.n_cols + 1, 256), 256, 0, s>>>(col_ptr, cnt.p, a.n_cols + 1), note_launch());
  if (a.n_batch > 0 && nnz_batch > 0) {
    const unsigned g = grid_for(a.n_batch * 32, 256);
    if (a.f32) (k_csc_fill<float><<<g, 256, 0, s>>>(a, cnt.p, t_row, static_cast<float*>(t_val)), note_launch());
    else (k_csc_fill<double><<<g, 256, 0, s>>>(a, cnt.p, t_row, static_cast<double*>(t_val)), note_launch());
  }
  return true;
}

bool slice_offsets(const int64_t* col_ptr, const int64_t* b_rp, int64_t n_cols, int64_t* slice_off,
                   cudaStream_t s) {
  cudaMemsetAsync(slice_off + n_cols, 0, sizeof(int64_t), s);
  if (n_cols > 0) (k_slice_sizes<<<grid_for(n_cols, 256), 256, 0, s>>>(col_ptr, b_rp, n_cols, slice_off), note_launch());
  return scan_exclusive_i64(slice_off, slice_off, n_cols + 1, nullptr, s);
}

void launch_wg_slice(const int64_t* slice_off, int64_t n_slices, int64_t total, int64_t E, int32_t* wg_first,
                     cudaStream_t s) {
  const int64_t n_wg = (total + E - 1) / E;
  if (n_slices <= 0 || n_wg <= 0) return;
  (k_wg_slice<<<grid_for(n_wg, 256), 256, 0, s>>>(slice_off, n_slices, E, n_wg, wg_first), note_launch());
}

void launch_outer_product(const OuterArgs& a, cudaStream_t s) {
  if (a.total <= 0) return;
  const int64_t n_wg = (a.total + a.E - 1) / a.E;
  const unsigned g = static_cast<unsigned>(n_wg);
  if (a.out_val && a.f32) {
    if (a.histo) (k_outer<float, true, true><<<g, kOpThreads, 0, s>>>(a), note_launch());
    else (k_outer<float, true, false><<<g, kOpThreads, 0, s>>>(a), note_launch());
  } else if (a.out_val) {
    if (a.histo) (k_outer<double, true, true><<<g, kOpThreads, 0, s>>>(a), note_launch());
    else (k_outer<double, true, false><<<g, kOpThreads, 0, s>>>(a), note_launch());
  } else {
    if (a.histo) (k_outer<double, false, true><<<g, kOpThreads, 0, s>>>(a), note_launch());
    else (k_outer<double, false, false><<<g, kOpThreads, 0, s>>>(a), note_launch());
  }
}

}  // namespace gm
