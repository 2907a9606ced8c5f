// gm_accum.cu -- local-memory accumulators of gMAGNUS (Sec. III-E, Algorithm 3
// lines 21-22 and 26-27). Nothing here falls back to global-memory accumulation.
//
// * Light rows (u(i) <= tau): rows are binned by u(i) and each bin gets a work
//   group size (the binning of Sec. III-E). Rows with u <= 256 use one warp and a
//   per-warp shared array: the products are sorted by column (bitonic network)
//   and equal columns are merged. Larger rows use one block and a shared hash
//   table of >= 2u slots (load factor alpha = 2, linear probing; the column is
//   scrambled by a multiplicative hash before the modulo), then a bitonic sort of
//   the occupied slots (Sec. III-E).
// * Chunks of C-hat_reord narrower than the dense width: a shared bitmap of the
//   chunk's columns gives nnz (symbolic) and, by a prefix sum over the bitmap
//   words, the rank of every column, so values are summed straight into their
//   sorted output slot (the dense accumulator with the bitmap prefix sum of
//   Sec. III-E, indexed by rank instead of by column).
// * Light chunks of a wider level: the block hash accumulator with list input.
#include <algorithm>
#include <climits>

#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

constexpr int32_t kEmpty = -1;

// ---- light rows: one warp per row, sort-based ---------------------------------

template <typename V, bool SYM, int CAPW, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) k_light_warp(LightArgs a) {
  const V* __restrict__ a_val = static_cast<const V*>(a.a_val);
  const V* __restrict__ b_val = static_cast<const V*>(a.b_val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  __shared__ int32_t s_key[WARPS][CAPW];
  __shared__ V s_val[SYM ? 1 : WARPS][SYM ? 1 : CAPW];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int32_t* key = s_key[w];
  V* val = SYM ? nullptr : s_val[w];
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * WARPS + w; item < a.n_items;
       item += static_cast<int64_t>(gridDim.x) * WARPS) {
    const int64_t r = a.rows[item];
    const int64_t lo = a.a_rp[r], hi = a.a_rp[r + 1];
    int pos = 0;
    for (int64_t p0 = lo; p0 < hi; p0 += 32) {
      const int64_t p = p0 + lane;
      int len = 0;
      int64_t bs = 0;
      V av = 0.0;
      if (p < hi) {
        const int k = a.a_col[p];
        bs = a.b_rp[k];
        len = static_cast<int>(a.b_rp[k + 1] - bs);
        if (!SYM) av = a_val[p];
      }
      const int inc = warp_inclusive_scan(len);
      const int off = pos + inc - len;
      for (int q = 0; q < len; ++q) {
        if (off + q < CAPW) {
          key[off + q] = a.b_col[bs + q];
          if (!SYM) val[off + q] = av * b_val[bs + q];
        }
      }
      pos += __shfl_sync(kFull, inc, 31);
    }
    const int n = pos;
    if (n > CAPW && lane == 0) atomicOr(a.status, kStInternal);
    for (int i = n + lane; i < CAPW; i += 32) key[i] = INT_MAX;
    __syncwarp();
    for (int k = 2; k <= CAPW; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = lane; i < CAPW; i += 32) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const int32_t ki = key[i], kj = key[ixj];
            const bool up = (i & k) == 0;
            if ((ki > kj) == up) {
              key[i] = kj;
              key[ixj] = ki;
              if (!SYM) {
                const V t = val[i];
                val[i] = val[ixj];
                val[ixj] = t;
              }
            }
          }
        }
        __syncwarp();
      }
    }
    const int nn = min(n, CAPW);
    int run = 0;
    const int64_t out = SYM ? 0 : a.c_rp[r];
    for (int i0 = 0; i0 < nn; i0 += 32) {
      const int i = i0 + lane;
      const bool head = i < nn && (i == 0 || key[i] != key[i - 1]);
      const unsigned hb = __ballot_sync(kFull, head);
      if (!SYM && head) {
        V s = 0.0;
        const int32_t c = key[i];
        for (int t = i; t < nn && key[t] == c; ++t) s += val[t];
        const int rank = run + __popc(hb & lanemask_lt());
        if (GM_CHECKED(out + rank < a.c_nnz, a.status)) {
          a.c_col[out + rank] = c;
          c_val[out + rank] = s;
        }
      }
      run += __popc(hb);
    }
    if (SYM && lane == 0) a.c_rp[r] = run;
    __syncwarp();
  }
}

// ---- block hash accumulator (light rows and light chunks) ---------------------

// Home slot of column c: the column is scrambled by a multiplicative (Fibonacci)
// hash before the reduction to [0, cap). Plain c mod cap clusters badly on
// power-law columns, whose low bits are far from uniform.
template <bool POW2>
__device__ __forceinline__ int slot_of(uint32_t c, int cap) {
  const uint32_t h = c * 0x9E3779B1u;
  return POW2 ? static_cast<int>(h >> (__clz(cap) + 1))
              : static_cast<int>((static_cast<uint64_t>(h) * static_cast<uint32_t>(cap)) >> 32);
}

// Insert column c; returns the slot and sets *fresh when the key was new.
template <bool POW2>
__device__ __forceinline__ int hash_insert(int32_t* keys, int cap, int32_t c, bool* fresh, bool* full) {
  int s = slot_of<POW2>(static_cast<uint32_t>(c), cap);
  for (int t = 0; t < cap; ++t) {
    const int32_t old = atomicCAS(&keys[s], kEmpty, c);
    if (old == kEmpty) {
      *fresh = true;
      return s;
    }
    if (old == c) return s;
    s = (s + 1 == cap) ? 0 : s + 1;
  }
  *full = true;
  return -1;
}

// After accumulation: move the occupied slots to the front (order kept), sort
// them by column and write nnz entries at out. keys/vals hold cap slots.
template <typename V>
__device__ void compact_sort_write(int32_t* keys, V* vals, int cap, int nnz, int32_t* c_col, V* c_val,
                                   int64_t out, int64_t col_base, int64_t c_nnz, int* status) {
  __shared__ int ws[33];
  int run = 0;
  for (int base = 0; base < cap; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int32_t k = i < cap ? keys[i] : kEmpty;
    const V v = i < cap ? vals[i] : 0.0;
    const int flag = k != kEmpty;
    int tot;
    const int pre = block_exclusive_scan(flag, ws, &tot);
    __syncthreads();
    if (flag) {
      keys[run + pre] = k;
      vals[run + pre] = v;
    }
    run += tot;
    __syncthreads();
  }
  int P = 1;
  while (P < nnz) P <<= 1;
  for (int i = nnz + threadIdx.x; i < P; i += blockDim.x) keys[i] = INT_MAX;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int32_t ki = keys[i], kj = keys[ixj];
          const bool up = (i & k) == 0;
          if ((ki > kj) == up) {
            keys[i] = kj;
            keys[ixj] = ki;
            const V t = vals[i];
            vals[i] = vals[ixj];
            vals[ixj] = t;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < nnz; i += blockDim.x) {
    if (GM_CHECKED(out + i < c_nnz, status)) {
      c_col[out + i] = static_cast<int32_t>(col_base + keys[i]);
      c_val[out + i] = vals[i];
    }
  }
}

template <typename V, bool SYM, bool POW2>
__global__ void k_light_hash(LightArgs a, int cap) {
  const V* __restrict__ a_val = static_cast<const V*>(a.a_val);
  const V* __restrict__ b_val = static_cast<const V*>(a.b_val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  extern __shared__ __align__(16) unsigned char smem[];
  V* vals = reinterpret_cast<V*>(smem);
  int32_t* keys = reinterpret_cast<int32_t*>(smem + (SYM ? 0 : static_cast<size_t>(cap) * sizeof(V)));
  __shared__ int ws[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const int64_t r = a.rows[item];
    for (int i = threadIdx.x; i < cap; i += blockDim.x) {
      keys[i] = kEmpty;
      if (!SYM) vals[i] = 0.0;
    }
    __syncthreads();
    int fresh_count = 0;
    bool full = false;
    for (int64_t p = a.a_rp[r] + warp; p < a.a_rp[r + 1]; p += nwarps) {
      const int k = a.a_col[p];
      const V av = SYM ? 0.0 : a_val[p];
      for (int64_t q = a.b_rp[k] + lane; q < a.b_rp[k + 1]; q += 32) {
        bool fresh = false;
        const int s = hash_insert<POW2>(keys, cap, a.b_col[q], &fresh, &full);
        fresh_count += fresh;
        if (!SYM && s >= 0) atomicAdd(&vals[s], av * b_val[q]);
      }
    }
    if (full) atomicOr(a.status, kStHashFull);
    __syncthreads();
    if (SYM) {
      int tot;
      block_exclusive_scan(fresh_count, ws, &tot);
      if (threadIdx.x == 0) a.c_rp[r] = tot;
    } else {
      const int64_t out = a.c_rp[r];
      const int nnz = static_cast<int>(a.c_rp[r + 1] - out);
      compact_sort_write(keys, vals, cap, nnz, a.c_col, c_val, out, 0, a.c_nnz, a.status);
    }
    __syncthreads();
  }
}

}  // namespace

namespace {

__device__ __forceinline__ int64_t leaf_col_base(const ListArgs& a, int64_t child_local) {
  const int64_t parent = child_local / a.v;
  const int64_t base = a.parent_colbase ? a.parent_colbase[parent] : 0;
  return base + (child_local % a.v) * a.width;
}

// Chunk of width <= dense width: bitmap of its columns, prefix sum over the
// bitmap words, values summed into their rank (= sorted output position).
template <typename V, typename CT, bool SYM>
__global__ void k_leaf_bitmap(ListArgs a, int nwords, int cap_vals) {
  const CT* __restrict__ in_col = static_cast<const CT*>(a.col);

  const V* __restrict__ in_val = static_cast<const V*>(a.val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  extern __shared__ __align__(16) unsigned char smem[];
  V* vals = reinterpret_cast<V*>(smem);                                                  // cap_vals
  uint32_t* bm = reinterpret_cast<uint32_t*>(smem + (SYM ? 0 : (static_cast<size_t>(cap_vals) * sizeof(V) + 15) & ~size_t(15)));  // nwords
  int* pre = reinterpret_cast<int*>(bm + nwords);                                                    // nwords
  __shared__ int ws[33];
  const int T = blockDim.x;
  const int per = (nwords + T - 1) / T;
  const int w0 = threadIdx.x * per, w1 = min(nwords, w0 + per);
  for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const int64_t m = a.items[item];
    const int64_t lo = a.rp[m], hi = a.rp[m + 1];
    const int64_t child_local = a.child_of ? a.child_of[m] : m;
    for (int w = threadIdx.x; w < nwords; w += T) bm[w] = 0u;
    __syncthreads();
    for (int64_t e0 = lo + threadIdx.x; e0 < hi; e0 += 4 * T) {  // 4 loads in flight per thread
      uint32_t c[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) c[u] = e0 + u * T < hi ? static_cast<uint32_t>(in_col[e0 + u * T]) : ~0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c[u] != ~0u) atomicOr(&bm[c[u] >> 5], 1u << (c[u] & 31));
    }
    __syncthreads();
    int acc = 0;
    for (int w = w0; w < w1; ++w) acc += __popc(bm[w]);
    int nnz;
    int run = block_exclusive_scan(acc, ws, &nnz);
    if (SYM) {
      if (threadIdx.x == 0) a.nnz_out[a.child_base + child_local] = nnz;
      __syncthreads();
      continue;
    }
    if (nnz > cap_vals) {
      if (threadIdx.x == 0) atomicOr(a.status, kStInternal);
      __syncthreads();
      continue;
    }
    for (int w = w0; w < w1; ++w) {
      pre[w] = run;
      run += __popc(bm[w]);
    }
    for (int r = threadIdx.x; r < nnz; r += T) vals[r] = 0.0;
    __syncthreads();
    for (int64_t e0 = lo + threadIdx.x; e0 < hi; e0 += 4 * T) {
      uint32_t c[4];
      V v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = e0 + u * T < hi;
        c[u] = in ? static_cast<uint32_t>(in_col[e0 + u * T]) : ~0u;
        v[u] = in ? in_val[e0 + u * T] : 0.0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c[u] == ~0u) continue;
        const int w = c[u] >> 5;
        const int r = pre[w] + __popc(bm[w] & ((1u << (c[u] & 31)) - 1u));
        atomicAdd(&vals[r], v[u]);
      }
    }
    __syncthreads();
    // columns come back from the bitmap: words round-robin over threads, so the
    // lanes of a warp write adjacent output ranges
    const int64_t out = a.off_in[a.child_base + child_local];
    const int64_t cb = leaf_col_base(a, child_local);
    for (int w = threadIdx.x; w < nwords; w += T) {
      uint32_t bits = bm[w];
      int pos = pre[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (GM_CHECKED(out + pos < a.c_nnz, a.status)) {
          a.c_col[out + pos] = static_cast<int32_t>(cb + w * 32 + b);
          c_val[out + pos] = vals[pos];
        }
        ++pos;
      }
    }
    __syncthreads();
  }
}

// Small chunk of width <= dense width, elements held in registers (n <= T * ITEMS).
// Symbolic: bitmap popcount. Numeric without floating-point atomics: the bitmap
// prefix gives each element its rank r (sorted output slot); an int32 atomic on
// cnt[r] gives its arrival index j; a prefix sum over cnt turns counts into
// segment starts; values are placed at seg[r] + j and each output entry sums its
// own segment.
template <typename V, typename CT, bool SYM, int T, int ITEMS>
__global__ void __launch_bounds__(T) k_leaf_small(ListArgs a, int nwords) {
  const CT* __restrict__ in_col = static_cast<const CT*>(a.col);

  const V* __restrict__ in_val = static_cast<const V*>(a.val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  constexpr int CAP = T * ITEMS;
  extern __shared__ __align__(16) unsigned char smem[];
  V* vbuf = reinterpret_cast<V*>(smem);                              // CAP
  int32_t* cols = reinterpret_cast<int32_t*>(vbuf + (SYM ? 0 : CAP));           // CAP
  int* seg = reinterpret_cast<int*>(cols + (SYM ? 0 : CAP));                     // CAP + 1
  uint32_t* bm = reinterpret_cast<uint32_t*>(seg + (SYM ? 0 : CAP + 1));         // nwords
  int* pre = reinterpret_cast<int*>(bm + nwords);                                // nwords
  __shared__ int ws[33];
  const int per = (nwords + T - 1) / T;
  const int w0 = threadIdx.x * per, w1 = min(nwords, w0 + per);
  for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const int64_t m = a.items[item];
    const int64_t lo = a.rp[m], hi = a.rp[m + 1];
    const int64_t child_local = a.child_of ? a.child_of[m] : m;
    int key[ITEMS];   // column, later rank
    int arr[ITEMS];   // arrival index within the rank
    V val[ITEMS];
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      const int64_t e = lo + k * T + threadIdx.x;
      key[k] = -1;
      val[k] = 0.0;
      if (e < hi) {
        key[k] = in_col[e];
        if (!SYM) val[k] = in_val[e];
      }
    }
    for (int w = threadIdx.x; w < nwords; w += T) bm[w] = 0u;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < ITEMS; ++k)
      if (key[k] >= 0) atomicOr(&bm[key[k] >> 5], 1u << (key[k] & 31));
    __syncthreads();
    int acc = 0;
    for (int w = w0; w < w1; ++w) acc += __popc(bm[w]);
    int nnz;
    int run = block_exclusive_scan(acc, ws, &nnz);
    if (SYM) {
      if (threadIdx.x == 0) a.nnz_out[a.child_base + child_local] = nnz;
      __syncthreads();
      continue;
    }
    for (int w = w0; w < w1; ++w) {
      pre[w] = run;
      uint32_t bits = bm[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        cols[run++] = w * 32 + b;
      }
    }
    for (int r = threadIdx.x; r <= nnz; r += T) seg[r] = 0;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      if (key[k] >= 0) {
        const int w = key[k] >> 5;
        key[k] = pre[w] + __popc(bm[w] & ((1u << (key[k] & 31)) - 1u));
        arr[k] = atomicAdd(&seg[key[k]], 1);
      }
    }
    __syncthreads();
    {  // counts -> segment starts (exclusive), contiguous run per thread
      const int per_r = (nnz + T) / T;
      const int r0 = threadIdx.x * per_r, r1 = min(nnz + 1, r0 + per_r);
      int c = 0;
      for (int r = r0; r < r1; ++r) c += seg[r];
      int base = block_exclusive_scan(c, ws, static_cast<int*>(nullptr));
      for (int r = r0; r < r1; ++r) {
        const int x = seg[r];
        seg[r] = base;
        base += x;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < ITEMS; ++k)
      if (key[k] >= 0) vbuf[seg[key[k]] + arr[k]] = val[k];
    __syncthreads();
    const int64_t out = a.off_in[a.child_base + child_local];
    const int64_t cb = leaf_col_base(a, child_local);
    for (int r = threadIdx.x; r < nnz; r += T) {
      V sum = 0.0;
      for (int q = seg[r]; q < seg[r + 1]; ++q) sum += vbuf[q];
      if (GM_CHECKED(out + r < a.c_nnz, a.status)) {
        a.c_col[out + r] = static_cast<int32_t>(cb + cols[r]);
        c_val[out + r] = sum;
      }
    }
    __syncthreads();
  }
}

// Numeric chunk of at most vcap elements, one warp per chunk with no block
// barrier, so many chunks are in flight per SM. Elements come through registers
// 32 * ITEMS at a time (a chunk of one such tile is read once; a longer one has
// its columns read twice, the second time from L2). The warp's private bitmap of
// the chunk's columns is counted in 16-byte pieces (consecutive lanes,
// consecutive pieces) into a word prefix, which gives every column its rank;
// values are added into their rank's slot (chunks this small rarely repeat a
// column, so the atomics seldom meet), and the chunk is written in column order
// by words.
template <typename V, typename CT, int ITEMS, int WARPS>
__global__ void __launch_bounds__(32 * WARPS, (ITEMS >= 16 ? 160 : 256) / WARPS) k_leaf_warpbm(ListArgs a, int nwp, int vcap) {
  const CT* __restrict__ in_col = static_cast<const CT*>(a.col);

  const V* __restrict__ in_val = static_cast<const V*>(a.val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int CAPW = 32 * ITEMS;
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  unsigned char* mine = smem + static_cast<size_t>(wib) * (static_cast<size_t>(nwp) * 8 + ((static_cast<size_t>(vcap) * sizeof(V) + 15) & ~size_t(15)));
  uint32_t* bm = reinterpret_cast<uint32_t*>(mine);                 // nwp (a multiple of 128)
  int* pre = reinterpret_cast<int*>(bm + nwp);                      // nwp
  V* vals = reinterpret_cast<V*>(pre + nwp);              // vcap
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * WARPS + wib;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * WARPS;
  for (int64_t item = gw; item < a.n_items; item += nw) {
    const int64_t m = a.items[item];
    const int64_t lo = a.rp[m];
    const int n = static_cast<int>(min(a.rp[m + 1] - lo, static_cast<int64_t>(vcap)));
    const int64_t child_local = a.child_of ? a.child_of[m] : m;
    const int64_t out = a.off_in[a.child_base + child_local];
    const int64_t cb = leaf_col_base(a, child_local);
    int key[ITEMS];
    V val[ITEMS];
    for (int w = lane * 4; w < nwp; w += 128) *reinterpret_cast<uint4*>(bm + w) = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    for (int t0 = 0; t0 < n; t0 += CAPW) {  // columns: set the bits
#pragma unroll
      for (int k = 0; k < ITEMS; ++k) {
        const int e = t0 + k * 32 + lane;
        key[k] = e < n ? in_col[lo + e] : -1;
        if (n <= CAPW) val[k] = e < n ? in_val[lo + e] : 0.0;
      }
#pragma unroll
      for (int k = 0; k < ITEMS; ++k)
        if (key[k] >= 0) atomicOr(&bm[key[k] >> 5], 1u << (key[k] & 31));
    }
    __syncwarp();
    int base = 0;
    for (int w = lane * 4; w < nwp; w += 128) {  // word prefix, 4 words a lane per round
      const uint4 q = *reinterpret_cast<const uint4*>(bm + w);
      const int c0 = __popc(q.x), c1 = __popc(q.y), c2 = __popc(q.z), c3 = __popc(q.w);
      const int c = c0 + c1 + c2 + c3;
      const int inc = warp_inclusive_scan(c);
      const int p0 = base + inc - c;
      *reinterpret_cast<int4*>(pre + w) = make_int4(p0, p0 + c0, p0 + c0 + c1, p0 + c0 + c1 + c2);
      base += __shfl_sync(kFull, inc, 31);
    }
    const int nnz = base;
    if (a.expect_nnz) GM_CHECKED(nnz == a.expect_nnz[a.child_base + child_local], a.status);
    for (int i = lane; i < nnz; i += 32) vals[i] = 0.0;
    __syncwarp();
    for (int t0 = 0; t0 < n; t0 += CAPW) {  // values into their rank's slot
      if (n > CAPW) {
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
          const int e = t0 + k * 32 + lane;
          key[k] = e < n ? in_col[lo + e] : -1;
          val[k] = e < n ? in_val[lo + e] : 0.0;
        }
      }
#pragma unroll
      for (int k = 0; k < ITEMS; ++k) {
        if (key[k] >= 0) {
          const int w = key[k] >> 5;
          atomicAdd(&vals[pre[w] + __popc(bm[w] & ((1u << (key[k] & 31)) - 1u))], val[k]);
        }
      }
    }
    __syncwarp();
    for (int w = lane; w < nwp; w += 32) {  // words round-robin over lanes
      uint32_t bits = bm[w];
      int pos = pre[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (GM_CHECKED(out + pos < a.c_nnz, a.status)) {
          a.c_col[out + pos] = static_cast<int32_t>(cb + w * 32 + b);
          c_val[out + pos] = vals[pos];
        }
        ++pos;
      }
    }
    __syncwarp();
  }
}

// The same accumulator for chunks of up to vcap output columns with T threads per
// chunk: elements in tiles of T * ITEMS through registers, bitmap word prefix by
// a block scan over 16-byte pieces, values added into their rank's slot; the
// column of every rank is then taken from the bitmap into shared memory, so
// that the chunk's row of C is written with consecutive threads on consecutive
// entries. CR holds a column inside the chunk (uint16_t up to 65536 columns).
template <typename V, typename CT, int ITEMS, int T, typename CR>
__global__ void __launch_bounds__(T) k_leaf_blkbm(ListArgs a, int nwp, int vcap, int ecap) {
  const CT* __restrict__ in_col = static_cast<const CT*>(a.col);

  const V* __restrict__ in_val = static_cast<const V*>(a.val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int CAPB = T * ITEMS;
  uint32_t* bm = reinterpret_cast<uint32_t*>(smem);                 // nwp (a multiple of 512)
  int* pre = reinterpret_cast<int*>(bm + nwp);                      // nwp
  V* vals = reinterpret_cast<V*>(pre + nwp);              // vcap
  __shared__ int ws[33];
  for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const int64_t m = a.items[item];
    const int64_t lo = a.rp[m];
    const int n = static_cast<int>(min(a.rp[m + 1] - lo, static_cast<int64_t>(ecap)));
    const int64_t child_local = a.child_of ? a.child_of[m] : m;
    const int64_t out = a.off_in[a.child_base + child_local];
    const int64_t cb = leaf_col_base(a, child_local);
    int key[ITEMS];
    V val[ITEMS];
    // the chunk's column bitmap: kept by the symbolic pass (then no marks), or built
    const int32_t slot = a.bm_slot ? a.bm_slot[a.child_base + child_local] : -1;
    if (slot >= 0) {
      const uint4* kept = reinterpret_cast<const uint4*>(a.bm_store + static_cast<int64_t>(slot) * nwp);
      for (int w = threadIdx.x; w < nwp / 4; w += T) reinterpret_cast<uint4*>(bm)[w] = kept[w];
    } else {
      for (int w = threadIdx.x * 4; w < nwp; w += 4 * T) *reinterpret_cast<uint4*>(bm + w) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    for (int t0 = 0; slot < 0 && t0 < n; t0 += CAPB) {  // columns: set the bits
#pragma unroll
      for (int k = 0; k < ITEMS; ++k) {
        const int e = t0 + k * T + threadIdx.x;
        key[k] = e < n ? in_col[lo + e] : -1;
        if (n <= CAPB) val[k] = e < n ? in_val[lo + e] : 0.0;
      }
#pragma unroll
      for (int k = 0; k < ITEMS; ++k)
        if (key[k] >= 0) atomicOr(&bm[key[k] >> 5], 1u << (key[k] & 31));
    }
    __syncthreads();
    int base = 0;
    for (int w0 = 0; w0 < nwp; w0 += 4 * T) {  // word prefix, 4 words a thread per round
      const int w = w0 + threadIdx.x * 4;
      const uint4 q = w < nwp ? *reinterpret_cast<const uint4*>(bm + w) : make_uint4(0u, 0u, 0u, 0u);
      const int c0 = __popc(q.x), c1 = __popc(q.y), c2 = __popc(q.z), c3 = __popc(q.w);
      int tot;
      const int p0 = base + block_exclusive_scan(c0 + c1 + c2 + c3, ws, &tot);
      if (w < nwp) *reinterpret_cast<int4*>(pre + w) = make_int4(p0, p0 + c0, p0 + c0 + c1, p0 + c0 + c1 + c2);
      base += tot;
      __syncthreads();
    }
    const int nnz = base;
    if (a.expect_nnz && threadIdx.x == 0) GM_CHECKED(nnz == a.expect_nnz[a.child_base + child_local], a.status);
    if (nnz > vcap) {  // uniform: the chunk's class promised at most vcap columns
      if (threadIdx.x == 0) atomicOr(a.status, kStInternal);
      __syncthreads();
      continue;
    }
    for (int i = threadIdx.x; i < nnz; i += T) vals[i] = 0.0;
    __syncthreads();
    for (int t0 = 0; t0 < n; t0 += CAPB) {  // values into their rank's slot
      if (n > CAPB || slot >= 0) {
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
          const int e = t0 + k * T + threadIdx.x;
          key[k] = e < n ? in_col[lo + e] : -1;
          val[k] = e < n ? in_val[lo + e] : 0.0;
        }
      }
#pragma unroll
      for (int k = 0; k < ITEMS; ++k) {
        if (key[k] >= 0) {
          const int w = key[k] >> 5;
          atomicAdd(&vals[pre[w] + __popc(bm[w] & ((1u << (key[k] & 31)) - 1u))], val[k]);
        }
      }
    }
    __syncthreads();
    {  // columns of every rank into shared memory, then coalesced rows of C
      CR* colr = reinterpret_cast<CR*>(vals + vcap);
      for (int w = threadIdx.x; w < nwp; w += T) {
        uint32_t bits = bm[w];
        int pos = pre[w];
        while (bits) {
          const int b = __ffs(bits) - 1;
          bits &= bits - 1;
          colr[pos++] = static_cast<CR>(w * 32 + b);
        }
      }
      __syncthreads();
      for (int r = threadIdx.x; r < nnz; r += T) {
        if (GM_CHECKED(out + r < a.c_nnz, a.status)) {
          a.c_col[out + r] = static_cast<int32_t>(cb + colr[r]);
          c_val[out + r] = vals[r];
        }
      }
    }
    __syncthreads();
  }
}

// Tiny chunk (at most CAPW elements): one warp loads it into shared memory,
// sorts (column, value) pairs with a bitonic network, merges equal columns and
// writes the chunk in column order. No bitmap, no block barrier.
template <typename V, typename CT, int CAPW, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) k_leaf_warp(ListArgs a) {
  const CT* __restrict__ in_col = static_cast<const CT*>(a.col);

  const V* __restrict__ in_val = static_cast<const V*>(a.val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  __shared__ int32_t s_key[WARPS][CAPW];
  __shared__ V s_val[WARPS][CAPW];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int32_t* key = s_key[w];
  V* val = s_val[w];
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * WARPS + w; item < a.n_items;
       item += static_cast<int64_t>(gridDim.x) * WARPS) {
    const int64_t m = a.items[item];
    const int64_t lo = a.rp[m];
    const int n = static_cast<int>(min(a.rp[m + 1] - lo, static_cast<int64_t>(CAPW)));
    const int64_t child_local = a.child_of ? a.child_of[m] : m;
    for (int i = lane; i < CAPW; i += 32) {
      key[i] = i < n ? in_col[lo + i] : INT_MAX;
      val[i] = i < n ? in_val[lo + i] : 0.0;
    }
    __syncwarp();
    for (int k = 2; k <= CAPW; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = lane; i < CAPW; i += 32) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const int32_t ki = key[i], kj = key[ixj];
            if ((ki > kj) == ((i & k) == 0)) {
              key[i] = kj;
              key[ixj] = ki;
              const V t = val[i];
              val[i] = val[ixj];
              val[ixj] = t;
            }
          }
        }
        __syncwarp();
      }
    }
    const int64_t out = a.off_in[a.child_base + child_local];
    const int64_t cb = leaf_col_base(a, child_local);
    int run = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      const bool head = i < n && (i == 0 || key[i] != key[i - 1]);
      const unsigned hb = __ballot_sync(kFull, head);
      if (head) {
        V sum = 0.0;
        const int32_t c = key[i];
        for (int t = i; t < n && key[t] == c; ++t) sum += val[t];
        const int r = run + __popc(hb & lanemask_lt());
        if (GM_CHECKED(out + r < a.c_nnz, a.status)) {
          a.c_col[out + r] = static_cast<int32_t>(cb + c);
          c_val[out + r] = sum;
        }
      }
      run += __popc(hb);
    }
    __syncwarp();
  }
}

// Light chunk of a level wider than the dense width: block hash accumulator.
template <typename V, bool SYM, bool POW2>
__global__ void k_leaf_hash(ListArgs a, int cap) {
  const V* __restrict__ in_val = static_cast<const V*>(a.val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  extern __shared__ __align__(16) unsigned char smem[];
  V* vals = reinterpret_cast<V*>(smem);
  int32_t* keys = reinterpret_cast<int32_t*>(smem + (SYM ? 0 : static_cast<size_t>(cap) * sizeof(V)));
  __shared__ int ws[33];
  for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const int64_t m = a.items[item];
    const int64_t child_local = a.child_of ? a.child_of[m] : m;
    for (int i = threadIdx.x; i < cap; i += blockDim.x) {
      keys[i] = kEmpty;
      if (!SYM) vals[i] = 0.0;
    }
    __syncthreads();
    int fresh_count = 0;
    bool full = false;
    for (int64_t e = a.rp[m] + threadIdx.x; e < a.rp[m + 1]; e += blockDim.x) {
      bool fresh = false;
      const int s = hash_insert<POW2>(keys, cap, static_cast<const int32_t*>(a.col)[e], &fresh, &full);
      fresh_count += fresh;
      if (!SYM && s >= 0) atomicAdd(&vals[s], in_val[e]);
    }
    if (full) atomicOr(a.status, kStHashFull);
    int nnz;
    block_exclusive_scan(fresh_count, ws, &nnz);
    if (SYM) {
      if (threadIdx.x == 0) a.nnz_out[a.child_base + child_local] = nnz;
    } else {
      compact_sort_write(keys, vals, cap, nnz, a.c_col, c_val, a.off_in[a.child_base + child_local],
                         leaf_col_base(a, child_local), a.c_nnz, a.status);
    }
    __syncthreads();
  }
}

// Always opt in: the kernels' static shared arrays add to the dynamic size.
template <class K>
void set_smem(K fn, size_t smem) {
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

unsigned item_grid(int64_t n_items, int per_sm) {
  int64_t g = n_items;
  const int64_t cap = 152LL * per_sm * 4;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

int hash_threads(int cap) { return cap <= 1024 ? 128 : cap <= 2048 ? 256 : cap <= 4096 ? 512 : 1024; }

}  // namespace

int64_t light_bin_ub(int b) { return int64_t(16) << b; }  // bins 1..9: 32 .. 8192

int light_bin_cap(int b, int64_t tau, int64_t smem_max, int vb) {
  if (b <= kLightWarpBins) return static_cast<int>(light_bin_ub(b));
  if (b <= 9) return static_cast<int>(2 * light_bin_ub(b));
  return static_cast<int>(std::min<int64_t>(2 * tau, (smem_max - 1024) / (4 + vb)));
}

namespace {

template <typename V>
void launch_light_rows_t(const LightArgs& a, int cap, bool symbolic, cudaStream_t s) {
  constexpr size_t vb = sizeof(V);
  if (cap <= 256) {
    constexpr int W = 8;
    const unsigned g = static_cast<unsigned>(std::min<int64_t>((a.n_items + W - 1) / W, 152LL * 64));
    switch (cap) {
      case 32: symbolic ? (k_light_warp<V, true, 32, W><<<g, W * 32, 0, s>>>(a), note_launch()) : (k_light_warp<V, false, 32, W><<<g, W * 32, 0, s>>>(a), note_launch()); break;
      case 64: symbolic ? (k_light_warp<V, true, 64, W><<<g, W * 32, 0, s>>>(a), note_launch()) : (k_light_warp<V, false, 64, W><<<g, W * 32, 0, s>>>(a), note_launch()); break;
      case 128: symbolic ? (k_light_warp<V, true, 128, W><<<g, W * 32, 0, s>>>(a), note_launch()) : (k_light_warp<V, false, 128, W><<<g, W * 32, 0, s>>>(a), note_launch()); break;
      default: symbolic ? (k_light_warp<V, true, 256, W><<<g, W * 32, 0, s>>>(a), note_launch()) : (k_light_warp<V, false, 256, W><<<g, W * 32, 0, s>>>(a), note_launch()); break;
    }
    return;
  }
  const bool pow2 = (cap & (cap - 1)) == 0;
  const size_t smem = static_cast<size_t>(cap) * (symbolic ? 4 : 4 + vb);
  const int T = hash_threads(cap);
  const unsigned g = item_grid(a.n_items, 2);
  if (symbolic) {
    auto fn = pow2 ? k_light_hash<V, true, true> : k_light_hash<V, true, false>;
    set_smem(fn, smem);
    (fn<<<g, T, smem, s>>>(a, cap), note_launch());
  } else {
    auto fn = pow2 ? k_light_hash<V, false, true> : k_light_hash<V, false, false>;
    set_smem(fn, smem);
    (fn<<<g, T, smem, s>>>(a, cap), note_launch());
  }
}

template <typename V, typename CT>
void launch_leaf_small_t(const ListArgs& a, int max_elems, bool symbolic, cudaStream_t s) {
  const int nwords = static_cast<int>((a.width + 31) / 32);
  const unsigned g = item_grid(a.n_items, 8);
  if (max_elems <= 1024) {
    const size_t smem = static_cast<size_t>(leaf_small_smem(a.width, 1024, symbolic, sizeof(V)));
    auto fn = symbolic ? k_leaf_small<V, CT, true, 128, 8> : k_leaf_small<V, CT, false, 128, 8>;
    set_smem(fn, smem);
    (fn<<<g, 128, smem, s>>>(a, nwords), note_launch());
  } else {
    const size_t smem = static_cast<size_t>(leaf_small_smem(a.width, 4096, symbolic, sizeof(V)));
    auto fn = symbolic ? k_leaf_small<V, CT, true, 256, 16> : k_leaf_small<V, CT, false, 256, 16>;
    set_smem(fn, smem);
    (fn<<<g, 256, smem, s>>>(a, nwords), note_launch());
  }
}

template <typename V, typename CT>
void launch_leaf_warpbm_t(const ListArgs& a, int max_elems, int nwp, int W, size_t smem, cudaStream_t s) {
  const unsigned g = static_cast<unsigned>(std::min<int64_t>((a.n_items + W - 1) / W, 152LL * 64));
  if (max_elems <= 128) {
    set_smem(k_leaf_warpbm<V, CT, 4, 4>, smem);
    (k_leaf_warpbm<V, CT, 4, 4><<<g, 128, smem, s>>>(a, nwp, max_elems), note_launch());
  } else if (W == 4) {
    set_smem(k_leaf_warpbm<V, CT, 16, 4>, smem);
    (k_leaf_warpbm<V, CT, 16, 4><<<g, 128, smem, s>>>(a, nwp, max_elems), note_launch());
  } else {
    set_smem(k_leaf_warpbm<V, CT, 16, 1>, smem);
    (k_leaf_warpbm<V, CT, 16, 1><<<g, 32, smem, s>>>(a, nwp, max_elems), note_launch());
  }
}

// smem: bitmap and prefix (nwp words each), the value array and the column of
// every rank (max_nnz entries each).
template <typename V, typename CT, typename CR>
void launch_leaf_blkbm_c(const ListArgs& a, int max_nnz, int max_elems, int nwp, size_t smem, cudaStream_t s) {
  const unsigned g = static_cast<unsigned>(std::min<int64_t>(a.n_items, 152LL * 32));
  // threads per chunk grow with the value array; float chunks of up to 8192
  // columns take more threads than double ones (measured: the C = A·A product
  // of an R-MAT scale-20 matrix is fastest with 256 / 256 threads for doubles
  // and 256 / 512 for floats)
  if (max_nnz <= 4096) {
    set_smem(k_leaf_blkbm<V, CT, 8, 256, CR>, smem);
    (k_leaf_blkbm<V, CT, 8, 256, CR><<<g, 256, smem, s>>>(a, nwp, max_nnz, max_elems), note_launch());
  } else if (max_nnz <= 8192 && sizeof(V) == 4) {
    set_smem(k_leaf_blkbm<V, CT, 8, 512, CR>, smem);
    (k_leaf_blkbm<V, CT, 8, 512, CR><<<g, 512, smem, s>>>(a, nwp, max_nnz, max_elems), note_launch());
  } else if (max_nnz <= 8192) {
    set_smem(k_leaf_blkbm<V, CT, 8, 256, CR>, smem);
    (k_leaf_blkbm<V, CT, 8, 256, CR><<<g, 256, smem, s>>>(a, nwp, max_nnz, max_elems), note_launch());
  } else {
    set_smem(k_leaf_blkbm<V, CT, 8, 1024, CR>, smem);
    (k_leaf_blkbm<V, CT, 8, 1024, CR><<<g, 1024, smem, s>>>(a, nwp, max_nnz, max_elems), note_launch());
  }
}
template <typename V, typename CT>
void launch_leaf_blkbm_t(const ListArgs& a, int max_nnz, int max_elems, int nwp, size_t smem, cudaStream_t s) {
  if (a.width <= 65536) launch_leaf_blkbm_c<V, CT, uint16_t>(a, max_nnz, max_elems, nwp, smem, s);
  else launch_leaf_blkbm_c<V, CT, uint32_t>(a, max_nnz, max_elems, nwp, smem, s);
}

template <typename V, typename CT>
void launch_leaf_bitmap_t(const ListArgs& a, int cap_vals, bool symbolic, cudaStream_t s) {
  const int nwords = static_cast<int>((a.width + 31) / 32);
  const size_t smem = static_cast<size_t>(leaf_bitmap_smem(a.width, cap_vals, symbolic, sizeof(V)));
  const int T = symbolic ? 256 : (cap_vals <= 1024 ? 256 : cap_vals <= 8192 ? 512 : 1024);
  const unsigned g = item_grid(a.n_items, 4);
  auto fn = symbolic ? k_leaf_bitmap<V, CT, true> : k_leaf_bitmap<V, CT, false>;
  set_smem(fn, smem);
  (fn<<<g, T, smem, s>>>(a, nwords, cap_vals), note_launch());
}

template <typename V>
void launch_leaf_hash_t(const ListArgs& a, int cap, bool symbolic, cudaStream_t s) {
  const bool pow2 = (cap & (cap - 1)) == 0;
  const size_t smem = static_cast<size_t>(cap) * (symbolic ? 4 : 4 + sizeof(V));
  const int T = hash_threads(cap);
  const unsigned g = item_grid(a.n_items, 2);
  if (symbolic) {
    auto fn = pow2 ? k_leaf_hash<V, true, true> : k_leaf_hash<V, true, false>;
    set_smem(fn, smem);
    (fn<<<g, T, smem, s>>>(a, cap), note_launch());
  } else {
    auto fn = pow2 ? k_leaf_hash<V, false, true> : k_leaf_hash<V, false, false>;
    set_smem(fn, smem);
    (fn<<<g, T, smem, s>>>(a, cap), note_launch());
  }
}

}  // namespace

void launch_light_rows(const LightArgs& a, int cap, bool symbolic, cudaStream_t s) {
  if (a.n_items <= 0) return;
  if (a.f32) launch_light_rows_t<float>(a, cap, symbolic, s);
  else launch_light_rows_t<double>(a, cap, symbolic, s);
}

int leaf_bitmap_smem(int64_t width, int cap_vals, bool symbolic, int vb) {
  const int64_t nwords = (width + 31) / 32;
  return static_cast<int>(nwords * 8 + (symbolic ? 0 : (static_cast<int64_t>(cap_vals) * vb + 15) & ~int64_t(15)));
}

int leaf_small_smem(int64_t width, int cap, bool symbolic, int vb) {
  const int64_t nwords = (width + 31) / 32;
  return static_cast<int>(nwords * 8 + (symbolic ? 0 : static_cast<int64_t>(cap) * (vb + 8) + 4));
}

void launch_leaf_small(const ListArgs& a, int max_elems, bool symbolic, cudaStream_t s) {
  if (a.n_items <= 0) return;
  if (a.f32 && a.col16) launch_leaf_small_t<float, uint16_t>(a, max_elems, symbolic, s);
  else if (a.f32) launch_leaf_small_t<float, int32_t>(a, max_elems, symbolic, s);
  else if (a.col16) launch_leaf_small_t<double, uint16_t>(a, max_elems, symbolic, s);
  else launch_leaf_small_t<double, int32_t>(a, max_elems, symbolic, s);
}

int64_t leaf_warpbm_words(int64_t width) { return ((width + 31) / 32 + 127) & ~int64_t(127); }

// Warps per block for chunks of at most max_elems elements (the value array of
// every warp is sized by max_elems).
static int warpbm_warps(int max_elems) { return max_elems <= 1024 ? 4 : 1; }

static int64_t warpbm_region(int64_t nwp, int max_elems, int vb) {
  return nwp * 8 + ((static_cast<int64_t>(max_elems) * vb + 15) & ~int64_t(15));
}

bool leaf_warpbm_fits(int64_t width, int max_elems, int64_t smem_max, int vb) {
  const int64_t per_warp = warpbm_region(leaf_warpbm_words(width), max_elems, vb);
  return max_elems <= 4096 && warpbm_warps(max_elems) * per_warp + 1024 <= smem_max;
}

void launch_leaf_warpbm(const ListArgs& a, int max_elems, cudaStream_t s) {
  if (a.n_items <= 0) return;
  const int nwp = static_cast<int>(leaf_warpbm_words(a.width));
  const int W = warpbm_warps(max_elems);
  const size_t smem = static_cast<size_t>(W * warpbm_region(nwp, max_elems, a.f32 ? 4 : 8));
  if (a.f32 && a.col16) launch_leaf_warpbm_t<float, uint16_t>(a, max_elems, nwp, W, smem, s);
  else if (a.f32) launch_leaf_warpbm_t<float, int32_t>(a, max_elems, nwp, W, smem, s);
  else if (a.col16) launch_leaf_warpbm_t<double, uint16_t>(a, max_elems, nwp, W, smem, s);
  else launch_leaf_warpbm_t<double, int32_t>(a, max_elems, nwp, W, smem, s);
}

int64_t leaf_blkbm_words(int64_t width) { return ((width + 31) / 32 + 511) & ~int64_t(511); }

static int blkbm_col_bytes(int64_t width) { return width <= 65536 ? 2 : 4; }

bool leaf_blkbm_fits(int64_t width, int max_nnz, int64_t smem_max, int vb) {
  return leaf_blkbm_words(width) * 8 + static_cast<int64_t>(max_nnz) * (vb + blkbm_col_bytes(width)) + 1024 <=
         smem_max;
}

void launch_leaf_blkbm(const ListArgs& a, int max_nnz, int max_elems, cudaStream_t s) {
  if (a.n_items <= 0) return;
  const int nwp = static_cast<int>(leaf_blkbm_words(a.width));
  const size_t smem =
      static_cast<size_t>(nwp) * 8 + static_cast<size_t>(max_nnz) * ((a.f32 ? 4 : 8) + blkbm_col_bytes(a.width));
  if (a.f32 && a.col16) launch_leaf_blkbm_t<float, uint16_t>(a, max_nnz, max_elems, nwp, smem, s);
  else if (a.f32) launch_leaf_blkbm_t<float, int32_t>(a, max_nnz, max_elems, nwp, smem, s);
  else if (a.col16) launch_leaf_blkbm_t<double, uint16_t>(a, max_nnz, max_elems, nwp, smem, s);
  else launch_leaf_blkbm_t<double, int32_t>(a, max_nnz, max_elems, nwp, smem, s);
}

void launch_leaf_warp(const ListArgs& a, cudaStream_t s) {
  if (a.n_items <= 0) return;
  constexpr int W = 8;
  const unsigned g = static_cast<unsigned>(std::min<int64_t>((a.n_items + W - 1) / W, 152LL * 64));
  if (a.f32 && a.col16) (k_leaf_warp<float, uint16_t, 128, W><<<g, W * 32, 0, s>>>(a), note_launch());
  else if (a.f32) (k_leaf_warp<float, int32_t, 128, W><<<g, W * 32, 0, s>>>(a), note_launch());
  else if (a.col16) (k_leaf_warp<double, uint16_t, 128, W><<<g, W * 32, 0, s>>>(a), note_launch());
  else (k_leaf_warp<double, int32_t, 128, W><<<g, W * 32, 0, s>>>(a), note_launch());
}

void launch_leaf_bitmap(const ListArgs& a, int cap_vals, bool symbolic, cudaStream_t s) {
  if (a.n_items <= 0) return;
  if (a.f32 && a.col16) launch_leaf_bitmap_t<float, uint16_t>(a, cap_vals, symbolic, s);
  else if (a.f32) launch_leaf_bitmap_t<float, int32_t>(a, cap_vals, symbolic, s);
  else if (a.col16) launch_leaf_bitmap_t<double, uint16_t>(a, cap_vals, symbolic, s);
  else launch_leaf_bitmap_t<double, int32_t>(a, cap_vals, symbolic, s);
}

void launch_leaf_hash(const ListArgs& a, int cap, bool symbolic, cudaStream_t s) {
  if (a.n_items <= 0) return;
  if (a.f32) launch_leaf_hash_t<float>(a, cap, symbolic, s);
  else launch_leaf_hash_t<double>(a, cap, symbolic, s);
}

}  // namespace gm
