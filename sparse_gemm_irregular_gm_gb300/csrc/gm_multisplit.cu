// gm_multisplit.cu -- Histogram and Multisplit of gMAGNUS (Sec. III-C, Algorithm 5).
//
// A static partition of the level's input (rows of C-hat, or heavy chunks of the
// previous level) gives each work group E consecutive elements, which span at
// most n_group_rows rows because every input row holds more than tau elements.
// Chunk of an element: local_row * v + (col >> shift) (GetChunk; v and the chunk
// width 1 << shift are powers of two, so the division is a shift).
//
// Multisplit per work group: elements are loaded once into registers, counted in
// a shared histogram with warp-aggregated atomics (__match_any_sync), the block
// reserves each non-empty chunk's global range with one atomic add, an in-block
// prefix sum gives local offsets, elements are permuted into shared buffers and
// then written out chunk-run by chunk-run (consecutive threads -> consecutive
// addresses) with the column shifted into the chunk's local range.
#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

constexpr int kMsThreads = 512;

__global__ void k_wg_row(const int64_t* __restrict__ rp, int64_t n_rows, int64_t E, int32_t* __restrict__ wg) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t base = rp[0];
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < n_rows; r += stride) {
    const int64_t lo = rp[r] - base, hi = rp[r + 1] - base;
    for (int64_t g = (lo + E - 1) / E; g * E < hi; ++g) wg[g] = static_cast<int32_t>(r);
  }
}

// smallest j in [0, n) with e < row_end[j]; n when none (row_end non-decreasing)
__device__ __forceinline__ int local_row(const int* __restrict__ row_end, int n, int e) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (e < row_end[mid]) hi = mid; else lo = mid + 1;
  }
  return lo;
}

struct Layout {
  int64_t* gpos;
  int* hist;
  int* loff;
  int* row_end;
  int32_t* col_buf;
  double* val_buf;
};

__device__ __forceinline__ Layout carve(unsigned char* smem, int nk, int ngr, int E, bool with_buf) {
  Layout L;
  L.gpos = reinterpret_cast<int64_t*>(smem);
  L.hist = reinterpret_cast<int*>(L.gpos + nk);
  L.loff = L.hist + nk;
  L.row_end = L.loff + nk;
  unsigned char* p = reinterpret_cast<unsigned char*>(L.row_end + ngr);
  p = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15));
  L.col_buf = with_buf ? reinterpret_cast<int32_t*>(p) : nullptr;
  L.val_buf = with_buf ? reinterpret_cast<double*>(p + ((static_cast<size_t>(E) * 4 + 15) & ~size_t(15))) : nullptr;
  return L;
}

__device__ __forceinline__ void setup_rows(const SplitArgs& a, const Layout& L, int64_t r0, int64_t S, int n,
                                           int nk) {
  for (int k = threadIdx.x; k < nk; k += blockDim.x) L.hist[k] = 0;
  for (int j = threadIdx.x; j < a.n_group_rows; j += blockDim.x) {
    const int64_t r = r0 + j;
    int64_t e = n;
    if (r < a.n_parents) e = min(max(a.in_rp[r + 1] - a.base - S, int64_t(0)), static_cast<int64_t>(n));
    L.row_end[j] = static_cast<int>(e);
  }
}

template <bool VAL, int ITEMS, bool SPLIT>
__global__ void __launch_bounds__(kMsThreads, 3) k_split(SplitArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int T = blockDim.x;
  const int E = T * ITEMS;
  const int nk = a.n_group_rows * a.v;
  const Layout L = carve(smem, nk, a.n_group_rows, E, SPLIT);
  const int64_t S = static_cast<int64_t>(blockIdx.x) * E;
  const int n = static_cast<int>(min(static_cast<int64_t>(E), a.total - S));
  const int64_t r0 = a.wg_first[blockIdx.x];
  setup_rows(a, L, r0, S, n, nk);
  __syncthreads();

  int key[ITEMS];
  int32_t col[ITEMS];
  bool bad = false;
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const int e = k * T + threadIdx.x;
    key[k] = -1;
    col[k] = 0;
    if (e < n) {
      col[k] = a.in_col[a.base + S + e];
      const int j = local_row(L.row_end, a.n_group_rows, e);
      if (j < a.n_group_rows) key[k] = j * a.v + (static_cast<uint32_t>(col[k]) >> a.shift);
      else bad = true;
    }
  }
  if (bad) atomicOr(a.status, kStGroupRows);
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const unsigned heads = run_heads(key[k]);
    if (key[k] >= 0 && ((heads >> (threadIdx.x & 31)) & 1u)) atomicAdd(&L.hist[key[k]], run_length(heads));
  }
  __syncthreads();

  if (!SPLIT) {
    for (int k = threadIdx.x; k < nk; k += T) {
      const int c = L.hist[k];
      if (c > 0) {
        const int64_t child = (r0 + k / a.v) * a.v + (k % a.v);
        atomicAdd(&a.counts[child], static_cast<unsigned long long>(c));
      }
    }
    return;
  }

  // Local prefix sum over the nk chunk counters (each thread a contiguous run)
  // and one global reservation per non-empty chunk.
  {
    __shared__ int ws[33];
    const int per = (nk + T - 1) / T;
    const int k0 = threadIdx.x * per;
    int acc = 0;
    for (int k = k0; k < min(nk, k0 + per); ++k) acc += L.hist[k];
    int tot;
    int pre = block_exclusive_scan(acc, ws, &tot);
    for (int k = k0; k < min(nk, k0 + per); ++k) {
      const int c = L.hist[k];
      L.loff[k] = pre;
      if (c > 0) {
        const int64_t child = (r0 + k / a.v) * a.v + (k % a.v);
        const int64_t m = a.inv ? a.inv[child] : child;
        L.gpos[k] = static_cast<int64_t>(atomicAdd(&a.cursor[m], static_cast<unsigned long long>(c)));
      }
      pre += c;
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < nk; k += T) L.hist[k] = L.loff[k];  // running local cursor
  __syncthreads();

  // Permute in shared memory: slots first, then the values read once (all loads
  // of a thread in flight together) straight into their permuted slots.
  const int lane = threadIdx.x & 31;
  int pos[ITEMS];
#pragma unroll
  for (int k = 0; k < ITEMS; ++k) {
    const unsigned heads = run_heads(key[k]);
    const int leader = run_head_lane(heads);
    int b = 0;
    if (key[k] >= 0 && lane == leader) b = atomicAdd(&L.hist[key[k]], run_length(heads));
    b = __shfl_sync(kFull, b, leader);
    pos[k] = b + (lane - leader);
    if (key[k] >= 0) L.col_buf[pos[k]] = col[k];
  }
  if (VAL) {
    double v[ITEMS];
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) v[k] = key[k] >= 0 ? a.in_val[a.base + S + k * T + threadIdx.x] : 0.0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k)
      if (key[k] >= 0) L.val_buf[pos[k]] = v[k];
  }
  __syncthreads();

  // Coalesced write-out: permuted position i keeps the row boundaries of the input.
  const int32_t mask = static_cast<int32_t>((1u << a.shift) - 1u);
  for (int i = threadIdx.x; i < n; i += T) {
    const int32_t c = L.col_buf[i];
    const int j = local_row(L.row_end, a.n_group_rows, i);
    if (j >= a.n_group_rows) continue;
    const int kk = j * a.v + (static_cast<uint32_t>(c) >> a.shift);
    const int64_t dest = L.gpos[kk] + (i - L.loff[kk]);
    a.out_col[dest] = c & mask;
    if (VAL) a.out_val[dest] = L.val_buf[i];
  }
}

size_t split_smem_bytes(int v, int ngr, int E, bool with_buf, bool with_val) {
  const size_t nk = static_cast<size_t>(v) * ngr;
  size_t b = nk * (8 + 4 + 4) + static_cast<size_t>(ngr) * 4 + 16;
  if (with_buf) b += ((static_cast<size_t>(E) * 4 + 15) & ~size_t(15)) + (with_val ? static_cast<size_t>(E) * 8 : 0);
  return b;
}

template <bool VAL, int ITEMS, bool SPLIT>
void launch_split_t(const SplitArgs& a, cudaStream_t s) {
  const int E = kMsThreads * ITEMS;
  const size_t smem = split_smem_bytes(a.v, a.n_group_rows, E, SPLIT, VAL);
  auto fn = k_split<VAL, ITEMS, SPLIT>;
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int64_t n_wg = (a.total + E - 1) / E;
  (fn<<<static_cast<unsigned>(n_wg), kMsThreads, smem, s>>>(a), note_launch());
}

template <bool SPLIT>
void launch_split(const SplitArgs& a, cudaStream_t s) {
  if (a.total <= 0) return;
  const bool val = a.in_val != nullptr && SPLIT;
  switch (a.E / kMsThreads) {
    case 8: val ? launch_split_t<true, 8, SPLIT>(a, s) : launch_split_t<false, 8, SPLIT>(a, s); break;
    case 4: val ? launch_split_t<true, 4, SPLIT>(a, s) : launch_split_t<false, 4, SPLIT>(a, s); break;
    default: val ? launch_split_t<true, 1, SPLIT>(a, s) : launch_split_t<false, 1, SPLIT>(a, s); break;
  }
}

}  // namespace

void launch_wg_row(const int64_t* rp, int64_t n_rows, int64_t E, int32_t* wg_first, cudaStream_t s) {
  if (n_rows <= 0) return;
  (k_wg_row<<<grid_for(n_rows, 256), 256, 0, s>>>(rp, n_rows, E, wg_first), note_launch());
}

void launch_histogram(const SplitArgs& a, cudaStream_t s) { launch_split<false>(a, s); }
void launch_multisplit(const SplitArgs& a, cudaStream_t s) { launch_split<true>(a, s); }

// Largest work-group size E (512 threads x {8, 4, 1} elements) whose shared
// arrays fit `smem_max` bytes for v chunks, given that every input row holds more
// than tau elements; 0 when none fits. *ngr_out receives n_group_rows.
int64_t multisplit_pick_E(int v, int64_t tau, bool with_val, int64_t smem_max, int* ngr_out) {
  for (int items : {8, 4, 1}) {
    const int64_t E = static_cast<int64_t>(kMsThreads) * items;
    const int64_t ngr = (E - 1 + tau) / (tau + 1) + 1;
    if (ngr > (1 << 20)) continue;
    const size_t need = split_smem_bytes(v, static_cast<int>(ngr), static_cast<int>(E), true, with_val);
    if (need <= static_cast<size_t>(smem_max)) {
      *ngr_out = static_cast<int>(ngr);
      return E;
    }
  }
  return 0;
}

}  // namespace gm
