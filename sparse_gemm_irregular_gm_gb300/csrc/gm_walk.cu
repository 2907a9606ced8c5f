// gm_walk.cu -- heavy rows' level-0 chunks accumulated straight from B.
//
// gMAGNUS (Sec. III-B to III-E, Algorithm 3) writes the heavy rows' intermediate
// products (C-hat), reorders them into column-range chunks with the multisplit
// and accumulates every chunk in shared memory. When each row of B is sorted by
// column, the part of B row k that falls into chunk c is one contiguous range,
// [bcp[k][c], bcp[k][c + 1]) from the per-B-row chunk starts, so chunk c of heavy
// row i can be summed directly: every stored A[i,k] times the range of B row k
// inside chunk c. The sum and its grouping into chunks are the method's; the
// intermediate products are never written or read back.
//
// The symbolic pass leaves every heavy row's whole-row bitmap in HBM. A chunk's
// bitmap words and their word prefix give each column its rank, i.e. its slot
// in the chunk's sorted output. Items (heavy row, chunk) are handed out in
// chunk-major order, so while all heavy rows walk chunk c only B's slice of
// chunk c is being read and it stays in L2.
//
// Warp items (at most CAP columns): one warp per item; the ranges of 32 A
// entries are laid end to end and walked 32 products a step, a product added
// with a plain fused multiply-add unless another lane holds the same rank in
// that step. Block items (more columns): a block per item, every add atomic;
// ranges of at least kLongRange entries are split evenly over the block's warps.
// Values are double only: the planner does not offer this pipeline for float.
#include <algorithm>
#include <climits>

#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

constexpr uint32_t kNone = 0xFFFFFFFFu;

__device__ __forceinline__ int rank_of(const uint32_t* bm, const int* pre, uint32_t c) {
  const int w = static_cast<int>(c >> 5);
  return pre[w] + __popc(bm[w] & ((1u << (c & 31)) - 1u));
}

// Item j (chunk-major): chunk c = j / nh of heavy row h = j % nh.
__device__ __forceinline__ void item_of(const WalkArgs& a, int64_t j, int& c, int64_t& h) {
  c = static_cast<int>(j / a.nh);
  h = j - static_cast<int64_t>(c) * a.nh;
}

constexpr int kLongRange = 512;  // block items: ranges this long are split over all warps
constexpr int kMaxLong = 128;    // such ranges kept per item (more are walked by their warp)

struct LongRanges {
  int n;
  int64_t s[kMaxLong], e[kMaxLong];
  double a[kMaxLong];
};

// The warp adds av * B[q] for q in [s, e) (columns inside this chunk), 4 loads
// of 32 entries in flight.
template <bool ATOMIC>
__device__ __forceinline__ void add_range(const WalkArgs& a, int64_t s, int64_t e, double av, uint32_t mask,
                                          const uint32_t* bm, const int* pre, double* vals, int lane) {
  for (int64_t q0 = s; q0 < e; q0 += 128) {
    uint32_t cc[4];
    double bv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t q = q0 + u * 32 + lane;
      cc[u] = q < e ? (static_cast<uint32_t>(a.b_col[q]) & mask) : kNone;
      bv[u] = q < e ? static_cast<const double*>(a.b_val)[q] : 0.0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (cc[u] != kNone) {
        const int r = rank_of(bm, pre, cc[u]);
        if (ATOMIC) atomicAdd(&vals[r], av * bv[u]);
        else vals[r] = fma(av, bv[u], vals[r]);
      }
    }
  }
}

// Chunk c of heavy row h: its bitmap words into bm and their exclusive word
// prefix into pre, 4 words a lane per round of 128 words (consecutive lanes,
// consecutive 16-byte pieces). Returns the chunk's nnz.
__device__ __forceinline__ int warp_load_bitmap(const WalkArgs& a, int64_t h, int c, uint32_t* bm, int* pre,
                                                int lane) {
  const int64_t first = static_cast<int64_t>(c) * a.nwc;
  const uint32_t* src = a.bits + h * a.nwr + first;
  const int64_t lim = a.nwr - first;  // words of the row's bitmap from the chunk's first word on
  int base = 0;
  for (int w0 = 0; w0 < a.nwc; w0 += 128) {
    const int w = w0 + lane * 4;
    const uint4 q = (w < a.nwc && w < lim) ? __ldg(reinterpret_cast<const uint4*>(src + w)) : make_uint4(0u, 0u, 0u, 0u);
    const int c0 = __popc(q.x), c1 = __popc(q.y), c2 = __popc(q.z), c3 = __popc(q.w);
    const int cnt = c0 + c1 + c2 + c3;
    const int inc = warp_inclusive_scan(cnt);
    const int p0 = base + inc - cnt;
    if (w < a.nwc) {
      *reinterpret_cast<uint4*>(bm + w) = q;
      *reinterpret_cast<int4*>(pre + w) = make_int4(p0, p0 + c0, p0 + c0 + c1, p0 + c0 + c1 + c2);
    }
    base += __shfl_sync(kFull, inc, 31);
  }
  return base;
}

// B range of A entry p (< hi) of the row inside chunk c: [s, s + len), and the A value.
__device__ __forceinline__ void range_of(const WalkArgs& a, int64_t p, int64_t hi, int c, int64_t& s, int& len,
                                         double& av) {
  s = 0;
  len = 0;
  av = 0.0;
  if (p < hi) {
    const int k = a.a_col[p];
    av = static_cast<const double*>(a.a_val)[p];
    const int32_t* t = a.bcp + static_cast<int64_t>(k) * (a.v + 1) + c;
    const int32_t t0 = t[0];
    s = a.b_rp[k] + t0;
    len = t[1] - t0;
  }
}

// Adds A[row, :] * B[:, chunk c] into vals[rank]. This warp takes the row's A
// entries in batches of 32 (batch sub, sub + nsub, ...), looking up the next
// batch's B ranges while it adds the current one. The batch's ranges are laid
// end to end (a warp scan of their lengths) and walked 32 * kSteps products at
// a time: lane l takes product g = g0 + l, finds its range by a binary search
// over the scan and loads the B entry, so short ranges keep every lane busy and
// kSteps loads are in flight. A product whose rank no other lane holds in the
// same step is added with a plain fused multiply-add, the others with atomic
// adds; with ATOMIC (other warps add to vals too) every add is atomic. With a
// shared list `longs` (block items), ranges of at least kLongRange entries are
// left there for the whole block.
constexpr int kSteps = 4;

template <bool ATOMIC>
__device__ __forceinline__ void walk_row(const WalkArgs& a, int64_t row, int c, const uint32_t* bm, const int* pre,
                                         double* vals, int lane, int sub, int nsub, LongRanges* longs) {
  const int64_t lo = a.a_rp[row], hi = a.a_rp[row + 1];
  const uint32_t mask = (1u << a.shift) - 1u;
  const int64_t step = static_cast<int64_t>(nsub) * 32;
  int64_t p0 = lo + static_cast<int64_t>(sub) * 32;
  int64_t ns;
  int nl;
  double na;
  range_of(a, p0 + lane, hi, c, ns, nl, na);
  for (; p0 < hi; p0 += step) {
    const int64_t s = ns;
    int len = nl;
    const double av = na;
    range_of(a, p0 + step + lane, hi, c, ns, nl, na);
    if (longs && len >= kLongRange) {
      const int slot = atomicAdd(&longs->n, 1);
      if (slot < kMaxLong) {
        longs->s[slot] = s;
        longs->e[slot] = s + len;
        longs->a[slot] = av;
        len = 0;
      }
    }
    const int incl = warp_inclusive_scan(len);
    const int total = __shfl_sync(kFull, incl, 31);
    const int excl = incl - len;
    for (int g0 = 0; g0 < total; g0 += 32 * kSteps) {
      uint32_t cc[kSteps];
      double bv[kSteps], aa[kSteps];
#pragma unroll
      for (int u = 0; u < kSteps; ++u) {
        const int g = g0 + u * 32 + lane;
        int j = 0;  // first lane whose range ends after g
#pragma unroll
        for (int b = 16; b; b >>= 1) {
          const int t = __shfl_sync(kFull, incl, j + b - 1);
          if (t <= g) j += b;
        }
        j = min(j, 31);
        const int64_t sj = __shfl_sync(kFull, s, j);
        const int ej = __shfl_sync(kFull, excl, j);
        aa[u] = __shfl_sync(kFull, av, j);
        const bool ok = g < total;
        const int64_t q = sj + (g - ej);
        cc[u] = ok ? (static_cast<uint32_t>(a.b_col[q]) & mask) : kNone;
        bv[u] = ok ? static_cast<const double*>(a.b_val)[q] : 0.0;
      }
#pragma unroll
      for (int u = 0; u < kSteps; ++u) {
        const int r = cc[u] != kNone ? rank_of(bm, pre, cc[u]) : -1 - lane;
        if (ATOMIC) {
          if (r >= 0) atomicAdd(&vals[r], aa[u] * bv[u]);
        } else {
          const unsigned peers = __match_any_sync(kFull, r);
          if (r >= 0) {
            if (peers == (1u << lane)) vals[r] = fma(aa[u], bv[u], vals[r]);
            else atomicAdd(&vals[r], aa[u] * bv[u]);
          }
          __syncwarp();
        }
      }
    }
  }
}

// Writes the chunk in column order: words round-robin over the threads t of T.
__device__ __forceinline__ void write_chunk(const WalkArgs& a, int64_t out, int c, const uint32_t* bm, const int* pre,
                                            const double* vals, int t, int T) {
  const int32_t cbase = static_cast<int32_t>(static_cast<int64_t>(c) << a.shift);
  for (int w = t; w < a.nwc; w += T) {
    uint32_t bits = bm[w];
    int pos = pre[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      a.c_col[out + pos] = cbase + w * 32 + b;
      static_cast<double*>(a.c_val)[out + pos] = vals[pos];
      ++pos;
    }
  }
}

template <int CAP, int WARPS>
__global__ void __launch_bounds__(32 * WARPS) k_walk_warp(WalkArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  unsigned char* mine = smem + static_cast<size_t>(wib) * (static_cast<size_t>(a.nwc) * 8 + CAP * 8);
  uint32_t* bm = reinterpret_cast<uint32_t*>(mine);
  int* pre = reinterpret_cast<int*>(bm + a.nwc);
  double* vals = reinterpret_cast<double*>(pre + a.nwc);
  while (true) {
    unsigned it = 0;
    if (lane == 0) it = atomicAdd(a.counter, 1u);
    it = __shfl_sync(kFull, it, 0);
    if (it >= a.n_items) break;
    const int64_t j = a.items[it];
    int c;
    int64_t h;
    item_of(a, j, c, h);
    const int nnz = warp_load_bitmap(a, h, c, bm, pre, lane);
    if (nnz > CAP) {  // uniform: the item's class promised at most CAP columns
      if (lane == 0) atomicOr(a.status, kStInternal);
      continue;
    }
    for (int i = lane; i < nnz; i += 32) vals[i] = 0.0;
    __syncwarp();
    walk_row<false>(a, a.heavy_rows[h], c, bm, pre, vals, lane, 0, 1, nullptr);
    __syncwarp();
    write_chunk(a, a.off[h * a.v + c], c, bm, pre, vals, lane, 32);
    __syncwarp();
  }
}

template <int T>
__global__ void __launch_bounds__(T, 1024 / T) k_walk_block(WalkArgs a, int cap) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* bm = reinterpret_cast<uint32_t*>(smem);
  int* pre = reinterpret_cast<int*>(bm + a.nwc);
  double* vals = reinterpret_cast<double*>(pre + a.nwc);
  __shared__ int ws[33];
  __shared__ unsigned s_it;
  __shared__ LongRanges longs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = T / 32;
  const uint32_t mask = (1u << a.shift) - 1u;
  while (true) {
    if (threadIdx.x == 0) {
      s_it = atomicAdd(a.counter, 1u);
      longs.n = 0;
    }
    __syncthreads();
    const unsigned it = s_it;
    if (it >= a.n_items) break;
    const int64_t j = a.items[it];
    int c;
    int64_t h;
    item_of(a, j, c, h);
    const int64_t first = static_cast<int64_t>(c) * a.nwc;
    const uint32_t* src = a.bits + h * a.nwr + first;
    const int64_t lim = a.nwr - first;
    int base = 0;
    for (int w0 = 0; w0 < a.nwc; w0 += 4 * T) {  // bitmap words and their prefix, 4 words a thread per round
      const int w = w0 + threadIdx.x * 4;
      const uint4 q =
          (w < a.nwc && w < lim) ? __ldg(reinterpret_cast<const uint4*>(src + w)) : make_uint4(0u, 0u, 0u, 0u);
      const int c0 = __popc(q.x), c1 = __popc(q.y), c2 = __popc(q.z), c3 = __popc(q.w);
      int tot;
      const int p0 = base + block_exclusive_scan(c0 + c1 + c2 + c3, ws, &tot);
      if (w < a.nwc) {
        *reinterpret_cast<uint4*>(bm + w) = q;
        *reinterpret_cast<int4*>(pre + w) = make_int4(p0, p0 + c0, p0 + c0 + c1, p0 + c0 + c1 + c2);
      }
      base += tot;
      __syncthreads();
    }
    const int nnz = base;
    if (nnz > cap) {  // uniform
      if (threadIdx.x == 0) atomicOr(a.status, kStInternal);
      __syncthreads();
      continue;
    }
    for (int i = threadIdx.x; i < nnz; i += T) vals[i] = 0.0;
    __syncthreads();
    walk_row<true>(a, a.heavy_rows[h], c, bm, pre, vals, lane, warp, NW, &longs);
    __syncthreads();
    const int nlong = min(longs.n, kMaxLong);
    for (int i = 0; i < nlong; ++i) {  // long ranges: an equal share for every warp
      const int64_t s0 = longs.s[i], len = longs.e[i] - s0;
      add_range<true>(a, s0 + len * warp / NW, s0 + len * (warp + 1) / NW, longs.a[i], mask, bm, pre, vals, lane);
    }
    __syncthreads();
    write_chunk(a, a.off[h * a.v + c], c, bm, pre, vals, threadIdx.x, T);
    __syncthreads();
  }
}

// Class of item j (chunk-major) by the nnz of its chunk: 0 empty, then
// warp items of <= 256, <= 1024, <= 2048 columns, block items of <= 8192 and more.
__global__ void k_walk_class(const int64_t* __restrict__ cnnz, int64_t nh, int v, uint8_t* __restrict__ cls) {
  const int64_t n = nh * v;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n; j += stride) {
    const int64_t c = j / nh, h = j - c * nh;
    const int64_t z = cnnz[h * v + c];
    cls[j] = z == 0 ? 0 : z <= 256 ? 1 : z <= 1024 ? 2 : z <= 2048 ? 3 : z <= 8192 ? 4 : 5;
  }
}

template <class K>
void opt_in(K fn, size_t smem) {
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

unsigned walk_grid(int64_t n_items, int num_sms, int per_sm) {
  const int64_t g = std::min<int64_t>(n_items, static_cast<int64_t>(num_sms) * std::max(per_sm, 1));
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

}  // namespace

int64_t walk_class_cap(int cls, int64_t width) {
  const int64_t cap = cls == 1 ? 256 : cls == 2 ? 1024 : cls == 3 ? 2048 : cls == 4 ? 8192 : width;
  return std::min<int64_t>(cap, width);
}

// Dynamic shared memory of a class's block. A warp item's region is laid out
// for the kernel's full CAP (256, 1024, 2048) whatever the width.
int64_t walk_smem(int cls, int64_t width) {
  const int64_t nwc = width / 32;
  if (cls == 1) return 4 * (nwc * 8 + 256 * 8);   // 4 warps a block
  if (cls == 2) return 4 * (nwc * 8 + 1024 * 8);  // 4 warps a block
  if (cls == 3) return 2 * (nwc * 8 + 2048 * 8);  // 2 warps a block
  return nwc * 8 + walk_class_cap(cls, width) * 8;
}

bool walk_fits(int64_t width, int64_t smem_max) {
  if (width < 128 || (width & (width - 1)) != 0) return false;
  for (int cls = 1; cls <= 5; ++cls)
    if (walk_smem(cls, width) + static_cast<int64_t>(sizeof(LongRanges)) + 1024 > smem_max) return false;
  return true;
}

void launch_walk_class(const int64_t* cnnz, int64_t nh, int v, uint8_t* cls, cudaStream_t s) {
  if (nh <= 0) return;
  (k_walk_class<<<grid_for(nh * v, 256), 256, 0, s>>>(cnnz, nh, v, cls), note_launch());
}

void launch_walk(const WalkArgs& a, int cls, int num_sms, int64_t smem_max, cudaStream_t s) {
  if (a.n_items <= 0) return;
  cudaMemsetAsync(a.counter, 0, sizeof(unsigned), s);
  const int64_t width = static_cast<int64_t>(a.nwc) * 32;
  const size_t smem = static_cast<size_t>(walk_smem(cls, width));
  const int per_sm = static_cast<int>(smem_max / static_cast<int64_t>(smem + sizeof(LongRanges) + 1024));
  switch (cls) {
    case 1:
      opt_in(k_walk_warp<256, 4>, smem);
      (k_walk_warp<256, 4><<<walk_grid(a.n_items, num_sms, std::min(per_sm, 16)), 128, smem, s>>>(a), note_launch());
      break;
    case 2:
      opt_in(k_walk_warp<1024, 4>, smem);
      (k_walk_warp<1024, 4><<<walk_grid(a.n_items, num_sms, std::min(per_sm, 16)), 128, smem, s>>>(a), note_launch());
      break;
    case 3:
      opt_in(k_walk_warp<2048, 2>, smem);
      (k_walk_warp<2048, 2><<<walk_grid(a.n_items, num_sms, std::min(per_sm, 32)), 64, smem, s>>>(a), note_launch());
      break;
    case 4:
      opt_in(k_walk_block<512>, smem);
      (k_walk_block<512><<<walk_grid(a.n_items, num_sms, std::min(per_sm, 4)), 512, smem, s>>>(
           a, static_cast<int>(walk_class_cap(4, width))), note_launch());
      break;
    default:
      opt_in(k_walk_block<1024>, smem);
      (k_walk_block<1024><<<walk_grid(a.n_items, num_sms, std::min(per_sm, 2)), 1024, smem, s>>>(
           a, static_cast<int>(walk_class_cap(5, width))), note_launch());
      break;
  }
}

}  // namespace gm
