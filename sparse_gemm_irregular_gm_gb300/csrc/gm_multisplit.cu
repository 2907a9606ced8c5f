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
#include <algorithm>

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
  void* val_buf;              // E values (8 bytes a slot: room for float or double)
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
  L.val_buf = with_buf ? static_cast<void*>(p + ((static_cast<size_t>(E) * 4 + 15) & ~size_t(15))) : nullptr;
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

template <typename V, bool VAL, int ITEMS, bool SPLIT>
__global__ void __launch_bounds__(kMsThreads, 3) k_split(SplitArgs a) {
  const V* __restrict__ in_val = static_cast<const V*>(a.in_val);
  V* __restrict__ out_val = static_cast<V*>(a.out_val);
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
    V v[ITEMS];
    V* const vbuf = static_cast<V*>(L.val_buf);
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) v[k] = key[k] >= 0 ? in_val[a.base + S + k * T + threadIdx.x] : V(0);
#pragma unroll
    for (int k = 0; k < ITEMS; ++k)
      if (key[k] >= 0) vbuf[pos[k]] = v[k];
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
    if (VAL) out_val[dest] = static_cast<const V*>(L.val_buf)[i];
  }
}

size_t split_smem_bytes(int v, int ngr, int E, bool with_buf, bool with_val) {
  const size_t nk = static_cast<size_t>(v) * ngr;
  size_t b = nk * (8 + 4 + 4) + static_cast<size_t>(ngr) * 4 + 16;
  if (with_buf) b += ((static_cast<size_t>(E) * 4 + 15) & ~size_t(15)) + (with_val ? static_cast<size_t>(E) * 8 : 0);
  return b;
}

template <typename V, bool VAL, int ITEMS, bool SPLIT>
void launch_split_t(const SplitArgs& a, cudaStream_t s) {
  const int E = kMsThreads * ITEMS;
  const size_t smem = split_smem_bytes(a.v, a.n_group_rows, E, SPLIT, VAL);
  auto fn = k_split<V, VAL, ITEMS, SPLIT>;
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int64_t n_wg = (a.total + E - 1) / E;
  (fn<<<static_cast<unsigned>(n_wg), kMsThreads, smem, s>>>(a), note_launch());
}

template <bool SPLIT>
void launch_split(const SplitArgs& a, cudaStream_t s) {
  if (a.total <= 0) return;
  const bool val = a.in_val != nullptr && SPLIT;
  switch (a.E / kMsThreads) {
    case 8:
      if (!val) launch_split_t<double, false, 8, SPLIT>(a, s);
      else if (a.f32) launch_split_t<float, true, 8, SPLIT>(a, s);
      else launch_split_t<double, true, 8, SPLIT>(a, s);
      break;
    case 4:
      if (!val) launch_split_t<double, false, 4, SPLIT>(a, s);
      else if (a.f32) launch_split_t<float, true, 4, SPLIT>(a, s);
      else launch_split_t<double, true, 4, SPLIT>(a, s);
      break;
    default:
      if (!val) launch_split_t<double, false, 1, SPLIT>(a, s);
      else if (a.f32) launch_split_t<float, true, 1, SPLIT>(a, s);
      else launch_split_t<double, true, 1, SPLIT>(a, s);
      break;
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

namespace gm {

namespace {

constexpr int kExThreads = 512;
constexpr int kExItems = kExpandE / kExThreads;  // 8

template <typename V>
__global__ void k_gather_entries(const int32_t* __restrict__ rows, int64_t nb, const int64_t* __restrict__ anz,
                                 const int64_t* __restrict__ a_rp, const int32_t* __restrict__ a_col,
                                 const V* __restrict__ a_val, const int64_t* __restrict__ b_rp,
                                 int64_t* __restrict__ e_b, V* __restrict__ e_a, int32_t* __restrict__ e_row,
                                 int64_t* __restrict__ e_len, int32_t* __restrict__ e_k) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t h = warp; h < nb; h += nw) {
    const int64_t r = rows[h];
    const int64_t base = anz[h] - anz[0];
    for (int64_t p = a_rp[r] + lane; p < a_rp[r + 1]; p += 32) {
      const int64_t i = base + (p - a_rp[r]);
      const int k = a_col[p];
      if (e_k) e_k[i] = k;
      if (e_a) e_a[i] = a_val[p];
      if (e_row) e_row[i] = static_cast<int32_t>(h);
      if (e_b || e_len) {  // null for the chunk-major expansion
        const int64_t b0 = b_rp[k];
        if (e_b) e_b[i] = b0;
        if (e_len) e_len[i] = b_rp[k + 1] - b0;
      }
    }
  }
}

// largest j in [lo, hi] with arr[j] <= x (arr non-decreasing, arr[lo] <= x)
__device__ __forceinline__ int64_t floor_index(const int64_t* __restrict__ arr, int64_t lo, int64_t hi, int64_t x) {
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (arr[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// bounds = sorted union of {g * E} and {e_off[m * CAP]}, then total.
__global__ void k_expand_bounds(const int64_t* __restrict__ e_off, int64_t n_e, int64_t total, int64_t n1,
                                int64_t n2, int64_t* __restrict__ bounds) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n1 + n2; t += stride) {
    if (t < n1) {  // element boundary x = t * E: its rank counts the entry boundaries below x
      const int64_t x = t * kExpandE;
      int64_t lo = 0, hi = n2;  // number of m with e_off[m * CAP] < x
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (e_off[mid * kExpandCap] < x) lo = mid + 1; else hi = mid;
      }
      bounds[t + lo] = x;
    } else {       // entry boundary y = e_off[m * CAP]: its rank counts the element boundaries <= y
      const int64_t m = t - n1;
      const int64_t y = e_off[m * kExpandCap];
      const int64_t c = min(n1, y / kExpandE + 1);
      bounds[m + c] = y;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) bounds[n1 + n2] = total;
}

// Per work group: the entry holding its first product, how many entries it
// touches and the batch row of the first one (what every thread of the group
// needs first, found here once instead of by a search inside the group).
__global__ void k_expand_wg_info(const int64_t* __restrict__ e_off, const int32_t* __restrict__ e_row, int64_t n_e,
                                 const int64_t* __restrict__ bounds, int64_t n_wg, int4* __restrict__ info) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < n_wg; g += stride) {
    const int64_t x = bounds[g], end = bounds[g + 1];
    const int64_t j0 = x >= e_off[n_e] ? n_e - 1 : floor_index(e_off, 0, n_e - 1, x);
    int64_t ne = 0;
    if (end > x) ne = floor_index(e_off, j0, min(n_e - 1, j0 + kExpandCap + 1), end - 1) - j0 + 1;
    info[g] = make_int4(static_cast<int>(j0), static_cast<int>(ne), e_row[j0], 0);
  }
}

constexpr uint32_t kNoKey = 0xFFFFFFFFu;

// One work group: products [S, end) of the batch in row order (at most
// kExpandE of them, from at most kExpandCap + 2 A entries). Each thread
// generates kExItems products (position k * T + tid), loading the B column and
// value of all of them before the first is used; chunk keys are counted, the
// chunks' global ranges reserved, and the products permuted through shared
// memory so that each chunk's run is written contiguously. A product is carried
// as one word: its key (local row * v + chunk) in the high 16 bits and its
// column inside the chunk in the low 16 bits.
template <typename V, bool VAL>
__global__ void __launch_bounds__(kExThreads, 3) k_expand_split(ExpandArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int T = kExThreads;
  const int nk = a.n_group_rows * a.v;
  const Layout L = carve(smem, nk, a.n_group_rows, kExpandE, true);
  uint32_t* const pk_buf = reinterpret_cast<uint32_t*>(L.col_buf);
  V* const vbuf = static_cast<V*>(L.val_buf);
  const V* __restrict__ e_a = static_cast<const V*>(a.e_a);
  const V* __restrict__ b_val = static_cast<const V*>(a.b_val);
  V* __restrict__ out_val = static_cast<V*>(a.out_val);
  // entry table after the multisplit layout (whose value buffer has 8 bytes a slot)
  unsigned char* tail = static_cast<unsigned char*>(L.val_buf) + static_cast<size_t>(kExpandE) * 8;
  int64_t* s_b = reinterpret_cast<int64_t*>(tail);                    // kExpandCap + 2
  V* s_a = reinterpret_cast<V*>(s_b + kExpandCap + 2);                // kExpandCap + 2
  int* s_lo = reinterpret_cast<int*>(s_a + kExpandCap + 2);           // kExpandCap + 2
  __shared__ int s_total;

  const int64_t g = blockIdx.x;
  const int64_t S = a.bounds[g];
  const int64_t end = a.bounds[g + 1];
  const int4 info = a.wg_info[g];
  const int n = static_cast<int>(end - S);
  if (n <= 0) return;
  const int64_t j0 = info.x;
  const int ne = info.y;
  const int64_t r0 = info.z;
  if (ne < 1 || ne > kExpandCap + 2) {  // bounds guarantee otherwise; never index past the table
    if (threadIdx.x == 0) atomicOr(a.status, kStInternal);
    return;
  }
  for (int i = threadIdx.x; i < ne; i += T) {
    const int64_t j = j0 + i;
    const int64_t off = a.e_off[j];
    const int64_t lo = max(S, off);
    const int lo_loc = static_cast<int>(min(lo, end) - S);
    s_lo[i] = lo_loc;
    s_b[i] = a.e_b[j] + (lo - off) - lo_loc;  // B index of local position p: s_b + p
    s_a[i] = VAL ? e_a[j] : V(0);
  }
  int* const s_ent = reinterpret_cast<int*>(L.col_buf);  // entry of each position (until the permute)
  for (int q = threadIdx.x; q < kExpandE; q += T) s_ent[q] = -1;
  for (int k = threadIdx.x; k < nk; k += T) L.hist[k] = 0;
  for (int jr = threadIdx.x; jr < a.n_group_rows; jr += T) {
    const int64_t r = r0 + jr;
    int64_t e = n;
    if (r < a.n_parents) e = min(max(a.in_rp[r + 1] - S, int64_t(0)), static_cast<int64_t>(n));
    L.row_end[jr] = static_cast<int>(e);
  }
  __syncthreads();
  // entry of each product = the last non-empty entry starting at or before it:
  // mark each non-empty entry at its first position, then a block-wide max scan
  for (int i = threadIdx.x; i < ne; i += T) {
    const int lo = s_lo[i];
    if (i + 1 == ne || s_lo[i + 1] > lo) s_ent[lo] = i;
  }
  __syncthreads();
  {
    __shared__ int s_wmax[kExThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int4* const q4 = reinterpret_cast<int4*>(s_ent + threadIdx.x * kExItems);
    int4 u0 = q4[0], u1 = q4[1];
    u0.y = max(u0.y, u0.x); u0.z = max(u0.z, u0.y); u0.w = max(u0.w, u0.z);
    u1.x = max(u1.x, u0.w); u1.y = max(u1.y, u1.x); u1.z = max(u1.z, u1.y); u1.w = max(u1.w, u1.z);
    int inc = u1.w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, d);
      if (lane >= d) inc = max(inc, y);
    }
    if (lane == 31) s_wmax[warp] = inc;
    int carry = __shfl_up_sync(kFull, inc, 1);
    if (lane == 0) carry = -1;
    __syncthreads();
    for (int w = 0; w < warp; ++w) carry = max(carry, s_wmax[w]);
    u0.x = max(u0.x, carry); u0.y = max(u0.y, carry); u0.z = max(u0.z, carry); u0.w = max(u0.w, carry);
    u1.x = max(u1.x, carry); u1.y = max(u1.y, carry); u1.z = max(u1.z, carry); u1.w = max(u1.w, carry);
    q4[0] = u0;
    q4[1] = u1;
  }
  __syncthreads();
  // all B loads of the thread in flight together
  int32_t col[kExItems];
  V vv[kExItems];
#pragma unroll
  for (int k = 0; k < kExItems; ++k) {
    const int p = k * T + threadIdx.x;
    const int64_t bi = s_b[max(s_ent[p], 0)] + p;
    col[k] = p < n ? a.b_col[bi] : 0;
    if (VAL) vv[k] = p < n ? b_val[bi] : V(0);
  }
  uint32_t pk[kExItems];
  bool bad = false;
  const uint32_t mask = (1u << a.shift) - 1u;
#pragma unroll
  for (int k = 0; k < kExItems; ++k) {
    const int p = k * T + threadIdx.x;
    pk[k] = kNoKey;
    if (p < n) {
      const int jr = local_row(L.row_end, a.n_group_rows, p);
      if (jr < a.n_group_rows) {
        const uint32_t key = static_cast<uint32_t>(jr * a.v) + (static_cast<uint32_t>(col[k]) >> a.shift);
        pk[k] = (key << 16) | (static_cast<uint32_t>(col[k]) & mask);
      } else {
        bad = true;
      }
    }
    if (VAL) vv[k] *= s_a[max(s_ent[p], 0)];
  }
  if (bad) atomicOr(a.status, kStGroupRows);
#pragma unroll
  for (int k = 0; k < kExItems; ++k) {
    const int key = pk[k] == kNoKey ? -1 : static_cast<int>(pk[k] >> 16);
    const unsigned heads = run_heads(key);
    if (key >= 0 && ((heads >> (threadIdx.x & 31)) & 1u)) atomicAdd(&L.hist[key], run_length(heads));
  }
  __syncthreads();
  {
    __shared__ int ws[33];
    const int per = (nk + T - 1) / T;
    const int k0 = threadIdx.x * per;
    int acc = 0;
    for (int k = k0; k < min(nk, k0 + per); ++k) acc += L.hist[k];
    int pre = block_exclusive_scan(acc, ws, static_cast<int*>(nullptr));
    for (int k = k0; k < min(nk, k0 + per); ++k) {
      const int c = L.hist[k];
      L.loff[k] = pre;
      if (c > 0) {
        const int64_t child = (r0 + k / a.v) * a.v + (k % a.v);
        L.gpos[k] = static_cast<int64_t>(atomicAdd(&a.cursor[child], static_cast<unsigned long long>(c)));
      }
      pre += c;
    }
    if (k0 < nk && k0 + per >= nk) s_total = pre;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < nk; k += T) L.hist[k] = L.loff[k];
  __syncthreads();
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < kExItems; ++k) {
    const int key = pk[k] == kNoKey ? -1 : static_cast<int>(pk[k] >> 16);
    const unsigned heads = run_heads(key);
    const int leader = run_head_lane(heads);
    int b = 0;
    if (key >= 0 && lane == leader) b = atomicAdd(&L.hist[key], run_length(heads));
    b = __shfl_sync(kFull, b, leader);
    if (key >= 0) {
      const int pos = b + (lane - leader);
      pk_buf[pos] = pk[k];
      if (VAL) vbuf[pos] = vv[k];
    }
  }
  __syncthreads();
  const int placed = s_total;
  for (int i = threadIdx.x; i < placed; i += T) {
    const uint32_t q = pk_buf[i];
    const int kk = static_cast<int>(q >> 16);
    const int64_t dest = L.gpos[kk] + (i - L.loff[kk]);
    a.out_col[dest] = static_cast<int32_t>(q & 0xFFFFu);
    if (VAL) out_val[dest] = vbuf[i];
  }
}

size_t expand_smem_bytes(int v, int ngr) {
  return split_smem_bytes(v, ngr, kExpandE, true, true) + static_cast<size_t>(kExpandCap + 2) * 20 + 64;
}

}  // namespace

int expand_group_rows(int64_t tau) { return static_cast<int>((kExpandE - 1 + tau) / (tau + 1) + 1); }

bool expand_fits(int v, int64_t w, int64_t tau, size_t smem) {
  const int64_t nk = static_cast<int64_t>(expand_group_rows(tau)) * v;
  return v >= 1 && w >= 1 && w <= 65536 && nk < 65535 && expand_smem_bytes(v, expand_group_rows(tau)) + 1024 <= smem;
}

void launch_gather_entries(const int32_t* heavy_rows, int64_t nb, const int64_t* anz_batch, const int64_t* a_rp,
                           const int32_t* a_col, const void* a_val, bool f32, const int64_t* b_rp, int64_t* e_b,
                           void* e_a, int32_t* e_row, int64_t* e_len, cudaStream_t s, int32_t* e_k) {
  if (nb <= 0) return;
  const unsigned g = grid_for(nb * 32, 256);
  if (f32)
    (k_gather_entries<float><<<g, 256, 0, s>>>(heavy_rows, nb, anz_batch, a_rp, a_col, static_cast<const float*>(a_val),
                                               b_rp, e_b, static_cast<float*>(e_a), e_row, e_len, e_k), note_launch());
  else
    (k_gather_entries<double><<<g, 256, 0, s>>>(heavy_rows, nb, anz_batch, a_rp, a_col,
                                                static_cast<const double*>(a_val), b_rp, e_b,
                                                static_cast<double*>(e_a), e_row, e_len, e_k), note_launch());
}

int64_t expand_num_wg(int64_t total, int64_t n_e) {
  return (total + kExpandE - 1) / kExpandE + (n_e + kExpandCap - 1) / kExpandCap;
}

void launch_expand_bounds(const int64_t* e_off, const int32_t* e_row, int64_t n_e, int64_t total, int64_t* bounds,
                          int4* wg_info, cudaStream_t s) {
  const int64_t n1 = (total + kExpandE - 1) / kExpandE, n2 = (n_e + kExpandCap - 1) / kExpandCap;
  (k_expand_bounds<<<grid_for(n1 + n2, 256), 256, 0, s>>>(e_off, n_e, total, n1, n2, bounds), note_launch());
  (k_expand_wg_info<<<grid_for(n1 + n2, 256), 256, 0, s>>>(e_off, e_row, n_e, bounds, n1 + n2, wg_info),
   note_launch());
}

void launch_expand_split(const ExpandArgs& a, cudaStream_t s) {
  if (a.n_wg <= 0) return;
  const size_t smem = expand_smem_bytes(a.v, a.n_group_rows);
  const unsigned g = static_cast<unsigned>(a.n_wg);
  if (a.out_val && a.f32) {
    cudaFuncSetAttribute(k_expand_split<float, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    (k_expand_split<float, true><<<g, kExThreads, smem, s>>>(a), note_launch());
  } else if (a.out_val) {
    cudaFuncSetAttribute(k_expand_split<double, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    (k_expand_split<double, true><<<g, kExThreads, smem, s>>>(a), note_launch());
  } else {
    cudaFuncSetAttribute(k_expand_split<double, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    (k_expand_split<double, false><<<g, kExThreads, smem, s>>>(a), note_launch());
  }
}

namespace {

// Row-order expansion into the level-0 chunks with long contiguous writes (B
// rows sorted, per-B-row chunk starts in a.bcp). The batch's heavy products, in
// row order, are cut into units of a.U; one block takes a unit at a time:
//  1. each warp takes an equal consecutive share of the unit's products (the
//     entries at its ends only in part) and counts, from the chunk starts of
//     each entry's B row, how many of them fall in every (row, chunk) -- lane l
//     holds chunks l and l + 32;
//  2. every (row, chunk) of the unit is reserved with one atomic add, and each
//     warp gets its own consecutive part of that range;
//  3. the warps walk their entries again and write the products: a run of one
//     entry in one chunk goes to the warp's cursor for that chunk.
// So each chunk of a row receives one contiguous block per unit (about
// U / 64 elements) instead of one short run per A entry.
constexpr int kRrWarps = 8;
constexpr int kRrRows = 8;   // rows a unit may touch (a.U keeps it below this)
constexpr int kRrU = 4;

// B's rows are re-read by every A entry that selects them. With KEEP their loads
// carry an L2 evict-last policy, so that the stream of chunk elements written
// meanwhile (evict-first stores) pushes them out of L2 less often (at scale 20
// this took the expansion from 81.3 to 80.2 ms).
__device__ __forceinline__ uint64_t l2_keep_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
template <bool KEEP>
__device__ __forceinline__ uint32_t ld_b(const int32_t* p, uint64_t pol) {
  if (!KEEP) return static_cast<uint32_t>(*p);
  uint32_t x;
  asm volatile("ld.global.nc.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(x) : "l"(p), "l"(pol));
  return x;
}
template <bool KEEP>
__device__ __forceinline__ double ld_b(const double* p, uint64_t pol) {
  if (!KEEP) return *p;
  double x;
  asm volatile("ld.global.nc.L2::cache_hint.f64 %0, [%1], %2;" : "=d"(x) : "l"(p), "l"(pol));
  return x;
}
template <bool KEEP>
__device__ __forceinline__ float ld_b(const float* p, uint64_t pol) {
  if (!KEEP) return *p;
  float x;
  asm volatile("ld.global.nc.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(x) : "l"(p), "l"(pol));
  return x;
}

template <typename V, typename CT, bool VAL, bool KEEP = false>
__global__ void __launch_bounds__(kRrWarps * 32, 5) k_expand_rows(RowRunArgs a) {
  const V* __restrict__ e_a = static_cast<const V*>(a.e_a);
  V* __restrict__ out_val = static_cast<V*>(a.out_val);
  CT* __restrict__ out_col = static_cast<CT*>(a.out_col);
  __shared__ int s_cnt[kRrWarps][kRrRows][64];  // counts, then each warp's offset inside the reservation
  __shared__ int64_t s_rbase[kRrRows][64];       // reservation of each (row, chunk) of the unit
  __shared__ int64_t s_base[kRrWarps][64];
  __shared__ int64_t s_unit;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t mask = (1u << a.shift) - 1u;
  const int v = a.v, vp1 = a.v + 1;
  const uint64_t pol = KEEP ? l2_keep_policy() : 0;
  while (true) {
    if (threadIdx.x == 0) s_unit = static_cast<int64_t>(atomicAdd(a.unit_counter, 1u));
    for (int i = threadIdx.x; i < kRrWarps * kRrRows * 64; i += blockDim.x) (&s_cnt[0][0][0])[i] = 0;
    __syncthreads();
    const int64_t g = s_unit;
    if (g >= a.n_units) break;
    const int64_t P0 = g * a.U, P1 = min(P0 + a.U, a.total);
    const int64_t e_lo = a.unit_first[g];
    const int64_t e_hi = g + 1 < a.n_units ? a.unit_first[g + 1] : a.n_e - 1;
    const int32_t row0 = a.e_row[e_lo];
    // this warp's equal share [W0, W1) of the unit's products, from the entry holding W0
    const int64_t share = (P1 - P0 + kRrWarps - 1) / kRrWarps;
    const int64_t W0 = min(P1, P0 + w * share), W1 = min(P1, W0 + share);
    int64_t ew = e_lo;
    {
      int64_t hi = e_hi;
      while (ew < hi) {
        const int64_t mid = (ew + hi + 1) >> 1;
        if (a.e_off[mid] <= W0) ew = mid; else hi = mid - 1;
      }
    }
    // 1. counts per (row, chunk) of this warp's share
    for (int64_t e = ew; e < a.n_e && W0 < W1; ++e) {
      const int64_t o0 = a.e_off[e];
      if (o0 >= W1) break;
      const int64_t o1 = a.e_off[e + 1];
      if (o1 <= max(o0, W0)) continue;
      const int64_t q0 = max(W0, o0) - o0, q1 = min(W1, o1) - o0;
      const int slot = a.e_row[e] - row0;
      if (slot < 0 || slot >= kRrRows) {
        if (lane == 0) atomicOr(a.status, kStGroupRows);
        continue;
      }
      const int32_t* const t = a.bcp + static_cast<int64_t>(a.e_k[e]) * vp1;
      for (int c = lane; c < v; c += 32)
        s_cnt[w][slot][c] += static_cast<int>(max(int64_t(0), min(q1, static_cast<int64_t>(t[c + 1])) -
                                                                  max(q0, static_cast<int64_t>(t[c]))));
    }
    __syncthreads();
    // 2. one reservation per (row, chunk); consecutive parts per warp
    for (int i = threadIdx.x; i < kRrRows * v; i += blockDim.x) {
      const int slot = i / v, c = i - slot * v;
      int tot = 0;
#pragma unroll
      for (int ww = 0; ww < kRrWarps; ++ww) tot += s_cnt[ww][slot][c];
      if (tot > 0) {
        s_rbase[slot][c] = static_cast<int64_t>(atomicAdd(&a.cursor[static_cast<int64_t>(row0 + slot) * v + c],
                                                          static_cast<unsigned long long>(tot)));
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < kRrWarps; ++ww) {
          const int x = s_cnt[ww][slot][c];
          s_cnt[ww][slot][c] = run;
          run += x;
        }
      }
    }
    __syncthreads();
    // 3. products, run by run, at the warp's cursors
    for (int64_t e = ew; e < a.n_e && W0 < W1; ++e) {
      const int64_t o0 = a.e_off[e];
      if (o0 >= W1) break;
      const int64_t o1 = a.e_off[e + 1];
      if (o1 <= max(o0, W0)) continue;
      const int slot = a.e_row[e] - row0;
      if (slot < 0 || slot >= kRrRows) continue;
      const int q0 = static_cast<int>(max(W0, o0) - o0), q1 = static_cast<int>(min(W1, o1) - o0);
      const int32_t* const t = a.bcp + static_cast<int64_t>(a.e_k[e]) * vp1;
      const int32_t* const bc = a.b_col + a.e_b[e];
      const V* const bvp = static_cast<const V*>(a.b_val) + a.e_b[e];
      const V av = VAL ? e_a[e] : V(0);
      __syncwarp();
      for (int c = lane; c < v; c += 32) {
        const int x0 = max(q0, t[c]), x1 = min(q1, t[c + 1]);
        if (x1 > x0) {
          s_base[w][c] = s_rbase[slot][c] + s_cnt[w][slot][c] - x0;
          s_cnt[w][slot][c] += x1 - x0;
        }
      }
      __syncwarp();
      uint32_t ncol[kRrU];
      V nbv[kRrU];
#pragma unroll
      for (int u = 0; u < kRrU; ++u) {
        const int q = q0 + u * 32 + lane;
        ncol[u] = q < q1 ? ld_b<KEEP>(bc + q, pol) : 0u;
        nbv[u] = (VAL && q < q1) ? ld_b<KEEP>(bvp + q, pol) : V(0);
      }
      for (int qb = q0; qb < q1; qb += 32 * kRrU) {
        uint32_t col[kRrU];
        V bv[kRrU];
#pragma unroll
        for (int u = 0; u < kRrU; ++u) {
          col[u] = ncol[u];
          bv[u] = nbv[u];
        }
        if (qb + 32 * kRrU < q1) {  // the next step's loads in flight while this one is stored
#pragma unroll
          for (int u = 0; u < kRrU; ++u) {
            const int q = qb + 32 * kRrU + u * 32 + lane;
            ncol[u] = q < q1 ? ld_b<KEEP>(bc + q, pol) : 0u;
            nbv[u] = (VAL && q < q1) ? ld_b<KEEP>(bvp + q, pol) : V(0);
          }
        }
#pragma unroll
        for (int u = 0; u < kRrU; ++u) {
          const int q = qb + u * 32 + lane;
          if (q < q1) {
            const int64_t dst = s_base[w][col[u] >> a.shift] + q;
#ifdef GM_BOUNDS_CHECK
            if (a.chunk_rp) {  // inside the (row, chunk) range the symbolic pass counted
              const int64_t ch = static_cast<int64_t>(row0 + slot) * v + (col[u] >> a.shift);
              if (!GM_CHECKED(dst >= a.chunk_rp[ch] && dst < a.chunk_rp[ch + 1], a.status)) continue;
            }
#endif
            // written once, read once by the accumulators: streaming stores, so that
            // they do not push B and the cursors out of L2
            __stcs(out_col + dst, static_cast<CT>(col[u] & mask));
            if (VAL) __stcs(out_val + dst, av * bv[u]);
          }
        }
      }
    }
    __syncthreads();
  }
}

// first[g] = the entry holding position g * U: the largest e with e_off[e] <= g * U.
__global__ void k_unit_first(const int64_t* __restrict__ e_off, int64_t n_e, int64_t U, int64_t n_units,
                             int64_t* __restrict__ first) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < n_units; g += stride) {
    const int64_t x = g * U;
    int64_t lo = 0, hi = n_e - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (e_off[mid] <= x) lo = mid; else hi = mid - 1;
    }
    first[g] = lo;
  }
}

// ---- chunk-major expansion -------------------------------------------------
// B is copied once per numeric pass into chunk-major order: the entries of every
// B row that fall into level-0 chunk c, for c = 0, 1, ..., with chunk-local
// columns. bct[c * (nB + 1) + k] is where row k's part of chunk c starts in the
// copy (bct[c * (nB + 1) + nB] is the end of chunk c). The expansion then takes
// the (heavy row, chunk) pairs chunk by chunk, so the part of B it reads (one
// chunk's copy and its starts, a few MB) stays in L2, and each pair's products
// are written as one contiguous run into the chunk's region.

// cnt[c * (nB + 1) + k]: entries of B row k in chunk c (0 for k == nB). A thread
// per row reads the row's v + 1 starts in order; for each c the threads of a
// warp write consecutive k.
__global__ void k_bc_counts(const int32_t* __restrict__ bcp, int64_t nB, int v, int64_t* __restrict__ cnt) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k <= nB; k += stride) {
    const int32_t* t = bcp + k * (v + 1);
    int32_t prev = k < nB ? t[0] : 0;
    for (int c = 0; c < v; ++c) {
      const int32_t next = k < nB ? t[c + 1] : 0;
      cnt[static_cast<int64_t>(c) * (nB + 1) + k] = next - prev;
      prev = next;
    }
  }
}

// One warp per B row (rows sorted by column): entry j of row k, in chunk c,
// goes to bct[c * (nB + 1) + k] + j - (row k's entries below chunk c).
template <typename V, typename CT>
__global__ void k_bc_fill(const int64_t* __restrict__ b_rp, const int32_t* __restrict__ b_col,
                          const V* __restrict__ b_val, int64_t nB, const int32_t* __restrict__ bcp, int v, int shift,
                          const int64_t* __restrict__ bct, CT* __restrict__ bc_col, V* __restrict__ bc_val) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const uint32_t mask = (1u << shift) - 1u;
  for (int64_t k = warp; k < nB; k += nw) {
    const int64_t rs = b_rp[k], len = b_rp[k + 1] - rs;
    const int32_t* t = bcp + k * (v + 1);
    for (int64_t j = lane; j < len; j += 32) {
      const uint32_t col = static_cast<uint32_t>(b_col[rs + j]);
      const int c = static_cast<int>(col >> shift);
      const int64_t pos = bct[static_cast<int64_t>(c) * (nB + 1) + k] + (j - t[c]);
      bc_col[pos] = static_cast<CT>(col & mask);
      if (bc_val) bc_val[pos] = b_val[rs + j];
    }
  }
}

constexpr int kCmWarps = 8;
constexpr int kCmU = 4;  // products a lane has in flight (8 measured slower: 71.8 against 61.4 ms)

// One warp per (heavy row h, chunk c) pair, taken chunk-major from a counter one
// pair at a time (warps that took several consecutive pairs each wrote slower:
// 79 against 60 ms for the C = A·A product of an R-MAT scale-20 matrix).
// The warp walks the row's A entries 32 at a time: lane l looks up entry l's
// part of chunk c (start and length in the chunk-major copy of B), a warp scan
// gives each part its offset in the pair's run, and the lanes then write the
// run's products at consecutive positions (lane l the products l, l + 32, ...),
// multiplying by the entry's A value.
template <typename V, typename CT, bool VAL>
__global__ void __launch_bounds__(kCmWarps * 32) k_expand_cm(ChunkMajorArgs a) {
  const V* __restrict__ e_a = static_cast<const V*>(a.e_a);
  const CT* __restrict__ bc_col = static_cast<const CT*>(a.bc_col);
  const V* __restrict__ bc_val = static_cast<const V*>(a.bc_val);
  CT* __restrict__ out_col = static_cast<CT*>(a.out_col);
  V* __restrict__ out_val = static_cast<V*>(a.out_val);
  // the group's parts with at least one product, in order: their start in the
  // copy of B, their A value and their offset in the run
  __shared__ int64_t s_src[kCmWarps][32];
  __shared__ V s_av[kCmWarps][32];
  __shared__ int s_ex[kCmWarps][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned le_mask = lane == 31 ? kFull : ((2u << lane) - 1u);  // lanes 0..lane
  const int64_t n_items = a.nb * a.v;
  const int64_t e_base = a.anz[0];
  while (true) {
    unsigned long long t = 0;
    if (lane == 0) t = atomicAdd(a.counter, 1ull);
    const int64_t g = static_cast<int64_t>(__shfl_sync(kFull, t, 0));
    if (g >= n_items) break;
    const int64_t c = g / a.nb, h = g - c * a.nb;
    const int64_t e0 = a.anz[h] - e_base, e1 = a.anz[h + 1] - e_base;
    const int64_t child = h * a.v + c;
    int64_t dst = a.rrp[child];
    const int64_t* __restrict__ bc = a.bct + c * a.nB1;
    for (int64_t eb = e0; eb < e1; eb += 32) {
      const int64_t e = eb + lane;
      int64_t src = 0;
      int len = 0;
      V av = V(0);
      if (e < e1) {
        const int k = a.e_k[e];
        src = bc[k];
        len = static_cast<int>(bc[k + 1] - src);
        if (VAL) av = e_a[e];
      }
      const int incl = warp_inclusive_scan(len);
      const int tot = __shfl_sync(kFull, incl, 31);
      const int ex = incl - len;
      const unsigned ne = __ballot_sync(kFull, len > 0);
      if (len > 0) {  // compacted: rank among the non-empty parts
        const int r = __popc(ne & lanemask_lt());
        s_src[w][r] = src;
        if (VAL) s_av[w][r] = av;
        s_ex[w][r] = ex;
      }
      __syncwarp();
#ifdef GM_BOUNDS_CHECK
      if (lane == 0) GM_CHECKED(dst + tot <= a.rrp[child + 1], a.status);
#endif
      // Position q of the run belongs to the last non-empty part starting at or
      // before q. Per window of 32 positions: the parts starting before it are
      // counted by a ballot, those starting inside it form a bit mask (an OR
      // over the lanes), and a lane's part is the count up to its position.
      for (int p0 = 0; p0 < tot; p0 += 32 * kCmU) {
        int64_t from[kCmU];
        V f[kCmU];
#pragma unroll
        for (int u = 0; u < kCmU; ++u) {
          const int ws = p0 + u * 32;
          const unsigned starts = __reduce_or_sync(kFull, (len > 0 && ex >= ws && ex < ws + 32) ? 1u << (ex - ws) : 0u);
          const int before = __popc(__ballot_sync(kFull, len > 0 && ex < ws));
          const int r = before + __popc(starts & le_mask) - 1;
          from[u] = -1;
          if (ws + lane < tot) {
            from[u] = s_src[w][r] + (ws + lane - s_ex[w][r]);
            if (VAL) f[u] = s_av[w][r];
          }
        }
        CT cc[kCmU];
        V bv[kCmU];
#pragma unroll
        for (int u = 0; u < kCmU; ++u) {
          if (from[u] >= 0) {
            cc[u] = bc_col[from[u]];
            if (VAL) bv[u] = bc_val[from[u]];
          }
        }
#pragma unroll
        for (int u = 0; u < kCmU; ++u) {
          if (from[u] >= 0) {
            const int64_t o = dst + p0 + u * 32 + lane;
#ifdef GM_BOUNDS_CHECK
            if (!GM_CHECKED(o < a.rrp[child + 1], a.status)) continue;
#endif
            // written once, read once by the accumulators: streaming stores
            __stcs(out_col + o, cc[u]);
            if (VAL) __stcs(out_val + o, f[u] * bv[u]);
          }
        }
      }
      dst += tot;
      __syncwarp();
    }
  }
}

}  // namespace

int64_t row_runs_unit(int64_t tau) { return std::min<int64_t>(32768, (kRrRows - 2) * (tau + 1)); }

void launch_row_runs(const RowRunArgs& a, int num_sms, cudaStream_t s) {
  if (a.total <= 0 || a.n_e <= 0) return;
  (k_unit_first<<<grid_for(a.n_units, 256), 256, 0, s>>>(a.e_off, a.n_e, a.U, a.n_units, a.unit_first),
   note_launch());
  cudaMemsetAsync(a.unit_counter, 0, sizeof(unsigned), s);
  const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(a.n_units, static_cast<int64_t>(num_sms) * 6));
  if (a.out_val && a.f32 && a.col16)
    (k_expand_rows<float, uint16_t, true, true><<<blocks, kRrWarps * 32, 0, s>>>(a), note_launch());
  else if (a.out_val && a.f32) (k_expand_rows<float, int32_t, true, true><<<blocks, kRrWarps * 32, 0, s>>>(a), note_launch());
  else if (a.out_val && a.col16)
    (k_expand_rows<double, uint16_t, true, true><<<blocks, kRrWarps * 32, 0, s>>>(a), note_launch());
  else if (a.out_val) (k_expand_rows<double, int32_t, true, true><<<blocks, kRrWarps * 32, 0, s>>>(a), note_launch());
  else (k_expand_rows<double, int32_t, false><<<blocks, kRrWarps * 32, 0, s>>>(a), note_launch());
}

int64_t bchunk_starts_len(int64_t b_rows, int v) { return static_cast<int64_t>(v) * (b_rows + 1); }

bool build_bchunks(const int64_t* b_rp, const int32_t* b_col, const void* b_val, bool f32, int64_t b_rows,
                   const int32_t* bcp, int v, int shift, bool col16, int64_t* bct, void* bc_col, void* bc_val,
                   cudaStream_t s) {
  const int64_t n = bchunk_starts_len(b_rows, v);
  (k_bc_counts<<<grid_for(b_rows + 1, 256), 256, 0, s>>>(bcp, b_rows, v, bct), note_launch());
  if (!scan_exclusive_i64(bct, bct, n, nullptr, s)) return false;
  const unsigned g = grid_for(std::max<int64_t>(b_rows, 1) * 32, 256);
  if (f32 && col16)
    (k_bc_fill<float, uint16_t><<<g, 256, 0, s>>>(b_rp, b_col, static_cast<const float*>(b_val), b_rows, bcp, v, shift,
                                                  bct, static_cast<uint16_t*>(bc_col), static_cast<float*>(bc_val)), note_launch());
  else if (f32)
    (k_bc_fill<float, int32_t><<<g, 256, 0, s>>>(b_rp, b_col, static_cast<const float*>(b_val), b_rows, bcp, v, shift,
                                                 bct, static_cast<int32_t*>(bc_col), static_cast<float*>(bc_val)), note_launch());
  else if (col16)
    (k_bc_fill<double, uint16_t><<<g, 256, 0, s>>>(b_rp, b_col, static_cast<const double*>(b_val), b_rows, bcp, v,
                                                   shift, bct, static_cast<uint16_t*>(bc_col),
                                                   static_cast<double*>(bc_val)), note_launch());
  else
    (k_bc_fill<double, int32_t><<<g, 256, 0, s>>>(b_rp, b_col, static_cast<const double*>(b_val), b_rows, bcp, v,
                                                  shift, bct, static_cast<int32_t*>(bc_col),
                                                  static_cast<double*>(bc_val)), note_launch());
  return true;
}

void launch_expand_cm(const ChunkMajorArgs& a, int num_sms, cudaStream_t s) {
  if (a.nb <= 0) return;
  cudaMemsetAsync(a.counter, 0, sizeof(unsigned long long), s);
  const unsigned blocks = static_cast<unsigned>(
      std::min<int64_t>((a.nb * a.v + kCmWarps - 1) / kCmWarps, static_cast<int64_t>(num_sms) * 8));
  const unsigned T = kCmWarps * 32;
  if (a.out_val && a.f32 && a.col16) (k_expand_cm<float, uint16_t, true><<<blocks, T, 0, s>>>(a), note_launch());
  else if (a.out_val && a.f32) (k_expand_cm<float, int32_t, true><<<blocks, T, 0, s>>>(a), note_launch());
  else if (a.out_val && a.col16) (k_expand_cm<double, uint16_t, true><<<blocks, T, 0, s>>>(a), note_launch());
  else if (a.out_val) (k_expand_cm<double, int32_t, true><<<blocks, T, 0, s>>>(a), note_launch());
  else if (a.col16) (k_expand_cm<double, uint16_t, false><<<blocks, T, 0, s>>>(a), note_launch());
  else (k_expand_cm<double, int32_t, false><<<blocks, T, 0, s>>>(a), note_launch());
}

}  // namespace gm
