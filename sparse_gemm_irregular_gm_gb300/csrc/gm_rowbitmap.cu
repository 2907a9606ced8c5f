// gm_rowbitmap.cu -- whole-row shared-memory bitmaps (gMAGNUS Sec. III-E: any
// local-memory accumulator may serve; here the dense accumulator keeps one bit
// per column of C, so a row of up to 8 * s_LM columns fits one block).
//
// * Symbolic: a row's products set bits; the nnz of any column range (a level-0
//   chunk of width w, or the whole row) is a popcount over the range. Used for
//   the heavy rows when the hierarchy has at most one level, so the symbolic pass
//   needs neither the outer product nor the multisplit.
// * Light rows (symbolic and numeric): the row's products are spread evenly over
//   the block and held in registers; in the numeric pass prefix sums over groups
//   of 8 bitmap words give every column its rank, i.e. its slot in the sorted
//   row; products are summed into that slot and the row is written in column
//   order with no sort.
//
// Rows are taken from a global work counter (dynamic scheduling; no waiting).
#include <algorithm>

#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

constexpr int kRbThreads = 1024;

__device__ __forceinline__ void zero_words(uint32_t* bm, int nwords) {
  uint4* b4 = reinterpret_cast<uint4*>(bm);
  const int n4 = nwords >> 2;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) b4[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = (n4 << 2) + threadIdx.x; i < nwords; i += blockDim.x) bm[i] = 0u;
}

// Sets the bits of the B columns col[s0, s1) with a group of G threads (thread i
// of the group): up to 3 leading columns one by one until 16-byte alignment,
// then 4 columns per 16-byte load with 4 loads in flight per thread, then the
// trailing columns.
__device__ __forceinline__ void mark_segment(const int32_t* __restrict__ col, int64_t s0, int64_t s1, uint32_t* bm,
                                             int i, int G) {
  const uintptr_t addr = reinterpret_cast<uintptr_t>(col + s0);
  const int64_t head = min(static_cast<int64_t>(((16 - (addr & 15)) & 15) >> 2), s1 - s0);
  if (i < head) {
    const uint32_t c = static_cast<uint32_t>(col[s0 + i]);
    atomicOr(&bm[c >> 5], 1u << (c & 31));
  }
  const int64_t a0 = s0 + head;
  const int64_t n4 = (s1 - a0) >> 2;
  const int4* v = reinterpret_cast<const int4*>(col + a0);
  for (int64_t j = i; j < n4; j += 4 * static_cast<int64_t>(G)) {
    int4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = j + u * G < n4 ? v[j + u * G] : make_int4(-1, -1, -1, -1);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (x[u].x < 0) continue;
      const uint32_t c[4] = {static_cast<uint32_t>(x[u].x), static_cast<uint32_t>(x[u].y),
                             static_cast<uint32_t>(x[u].z), static_cast<uint32_t>(x[u].w)};
#pragma unroll
      for (int t = 0; t < 4; ++t) atomicOr(&bm[c[t] >> 5], 1u << (c[t] & 31));
    }
  }
  const int64_t t0 = a0 + (n4 << 2);
  if (i < s1 - t0) {
    const uint32_t c = static_cast<uint32_t>(col[t0 + i]);
    atomicOr(&bm[c >> 5], 1u << (c & 31));
  }
}

// Sets the bit of every product column of row r. Warp w takes the A entries w,
// w + nwarps, ... (every warp busy even on rows with few entries); their
// metadata is loaded 32 entries at a time, then the warp marks each entry's B
// row; B rows longer than kLongRow are marked afterwards by the whole block.
constexpr int kLongRow = 4096;
constexpr int kMaxLong = 64;     // deferred long rows kept per row (more are marked by their warp)

struct LongRows {
  int n;
  int64_t s0[kMaxLong], s1[kMaxLong];
};

__device__ __forceinline__ void mark_row(const RowBitmapArgs& a, int64_t r, uint32_t* bm, LongRows& longs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int64_t lo = a.a_rp[r], hi = a.a_rp[r + 1];
  if (threadIdx.x == 0) longs.n = 0;
  __syncthreads();
  for (int64_t g = lo + warp; g < hi; g += static_cast<int64_t>(nwarps) * 32) {
    const int64_t p = g + static_cast<int64_t>(lane) * nwarps;
    int64_t bs = 0, be = 0;
    if (p < hi) {
      const int k = a.a_col[p];
      bs = a.b_rp[k];
      be = a.b_rp[k + 1];
    }
    if (be - bs > kLongRow) {  // long rows go to the shared list when there is room
      const int slot = atomicAdd(&longs.n, 1);
      if (slot < kMaxLong) {
        longs.s0[slot] = bs;
        longs.s1[slot] = be;
        be = bs;
      }
    }
    const unsigned live = __ballot_sync(kFull, be > bs);
    for (unsigned m = live; m; m &= m - 1) {
      const int j = __ffs(m) - 1;
      mark_segment(a.b_col, __shfl_sync(kFull, bs, j), __shfl_sync(kFull, be, j), bm, lane, 32);
    }
  }
  __syncthreads();
  const int nl = min(longs.n, kMaxLong);
  for (int i = 0; i < nl; ++i) mark_segment(a.b_col, longs.s0[i], longs.s1[i], bm, threadIdx.x, blockDim.x);
}

// Number of set bits in [lo, hi).
__device__ __forceinline__ int count_range(const uint32_t* bm, int64_t lo, int64_t hi) {
  int n = 0;
  while (lo < hi) {
    const int64_t w = lo >> 5;
    const int b0 = static_cast<int>(lo & 31);
    const int64_t wend = (w + 1) << 5;
    const int b1 = hi < wend ? static_cast<int>(hi & 31) : 32;
    uint32_t m = bm[w] >> b0;
    if (b1 - b0 < 32) m &= (1u << (b1 - b0)) - 1u;
    n += __popc(m);
    lo = (w << 5) + b1;
  }
  return n;
}

__global__ void __launch_bounds__(kRbThreads) k_rowbm_symbolic(RowBitmapArgs a, int nwords) {
  extern __shared__ __align__(16) uint32_t bm[];
  __shared__ int64_t s_item;
  __shared__ LongRows longs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int64_t nbits = static_cast<int64_t>(nwords) * 32;
  while (true) {
    if (threadIdx.x == 0) s_item = atomicAdd(a.work_counter, 1u);
    __syncthreads();
    const int64_t item = s_item;
    if (item >= a.n_items) break;
    const int64_t r = a.rows[item];
    zero_words(bm, nwords);
    __syncthreads();
    mark_row(a, r, bm, longs);
    __syncthreads();
    if (a.v == 1 && a.width >= nbits) {  // whole row
      int n = 0;
      for (int w = threadIdx.x; w < nwords; w += blockDim.x) n += __popc(bm[w]);
      n = warp_reduce_sum(n);
      __shared__ int part[32];
      if (lane == 0) part[warp] = n;
      __syncthreads();
      if (warp == 0) {
        int t = lane < nwarps ? part[lane] : 0;
        t = warp_reduce_sum(t);
        if (lane == 0) {
          if (a.nnz_out) a.nnz_out[a.item_base + item] = t;
          else a.c_rp[r] = t;
        }
      }
    } else {  // one warp per chunk of width w
      for (int c = warp; c < a.v; c += nwarps) {
        const int64_t lo = static_cast<int64_t>(c) * a.width;
        const int64_t hi = min(lo + a.width, nbits);
        const int64_t span = (hi - lo + 31) / 32;
        int n = 0;
        for (int64_t j = lane; j < span; j += 32) n += count_range(bm, lo + j * 32, min(hi, lo + j * 32 + 32));
        n = warp_reduce_sum(n);
        const int64_t child = (a.item_base + item) * a.v + c;
        if (lane == 0) a.nnz_out[child] = n;
        if (a.bm_slot) {  // keep the chunk's words for the numeric pass (width a multiple of 32)
          const int32_t slot = a.bm_slot[child];
          if (slot >= 0) {
            uint32_t* dst = a.bm_store + static_cast<int64_t>(slot) * a.store_words;
            const uint32_t* src = bm + (lo >> 5);
            for (int j = lane; j < a.store_words; j += 32) dst[j] = j < span ? src[j] : 0u;
          }
        }
      }
    }
    __syncthreads();
  }
}

constexpr int kGroupWords = 8;  // rank prefix kept per 8 bitmap words (256 columns)
__host__ __device__ constexpr int64_t light_a16(int64_t b) { return (b + 15) & ~int64_t(15); }
constexpr int kRlItems = 10;    // products per thread in k_rowbm_light: rows of up to 10240 products
constexpr int kRlItemsWide = 16; // ... for the symbolic pass and float values: up to 16384 products
constexpr uint32_t kNoCol = 0xFFFFFFFFu;
constexpr int64_t kLightSymRegion = 65536;  // entry-table bytes of the symbolic light kernel

// Rank of column c (number of set bits below it) from the 8-word group prefix:
// the 16-byte half of the group holding c, plus the first half's count when c
// lies in the second.
__device__ __forceinline__ int bitmap_rank(const uint32_t* bm, const uint16_t* gpre, uint32_t c) {
  const int w = c >> 5, g = w >> 3, wi = w & 7, j = wi & 3;
  const uint4* g4 = reinterpret_cast<const uint4*>(bm + g * kGroupWords);
  int r = gpre[g];
  if (wi >= 4) {
    const uint4 q0 = g4[0];
    r += __popc(q0.x) + __popc(q0.y) + __popc(q0.z) + __popc(q0.w);
  }
  const uint4 q = g4[wi >> 2];
  r += (j > 0 ? __popc(q.x) : 0) + (j > 1 ? __popc(q.y) : 0) + (j > 2 ? __popc(q.z) : 0);
  const uint32_t word = j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
  return r + __popc(word & ((1u << (c & 31)) - 1u));
}

// Writes, in increasing order, the index of every group whose bit is set in the
// group summary gsum (nsw words) to glist and returns their number. Every thread
// of the block must call it; it ends with a barrier.
__device__ __forceinline__ int list_groups(const uint32_t* gsum, int nsw, uint16_t* glist, int* ws) {
  int ng = 0;
  for (int s0 = 0; s0 < nsw; s0 += blockDim.x) {
    const int sw = s0 + threadIdx.x;
    uint32_t w = sw < nsw ? gsum[sw] : 0u;
    int tot;
    int off = ng + block_exclusive_scan(__popc(w), ws, &tot);
    while (w) {
      const int b = __ffs(w) - 1;
      w &= w - 1;
      glist[off++] = static_cast<uint16_t>((sw << 5) + b);
    }
    ng += tot;
    __syncthreads();
  }
  return ng;
}

__device__ __forceinline__ int group_popc(const uint32_t* bm, int g) {
  const uint4* g4 = reinterpret_cast<const uint4*>(bm + g * kGroupWords);
  const uint4 q0 = g4[0], q1 = g4[1];
  return __popc(q0.x) + __popc(q0.y) + __popc(q0.z) + __popc(q0.w) + __popc(q1.x) + __popc(q1.y) + __popc(q1.z) +
         __popc(q1.w);
}

__device__ __forceinline__ void zero_group(uint32_t* bm, int g) {
  uint4* g4 = reinterpret_cast<uint4*>(bm + g * kGroupWords);
  g4[0] = make_uint4(0u, 0u, 0u, 0u);
  g4[1] = make_uint4(0u, 0u, 0u, 0u);
}

// Light rows (u <= kRbThreads * kRlItems) with a whole-row bitmap, every product
// held in registers: thread t takes products t, t + T, ... of the row in row
// order, so the block's work is balanced whatever the lengths of the B rows.
// The row's A entries are staged in shared memory (B row start, A value, and a
// prefix of the B row lengths, te_cap entries at a time), and each warp writes
// the index of its entries into every product position they cover, so a
// product reads its entry in one load. All B loads of a thread are issued
// before the first is used. The products' columns set the bitmap; then
//  * symbolic: the row's nnz is the bitmap's popcount (written to c_rp[row]),
//    and the words are cleared as they are counted;
//  * numeric: the first bit set in a word also sets its group's bit (8 words,
//    256 columns) in a summary, and only the groups listed from the summary are
//    visited afterwards (a light row touches a few thousand of the row's groups
//    at most): prefix sums over them give every column its rank, the values are
//    summed into their rank in shared memory (the entry table's space is
//    reused), the row is written in column order and the listed groups are
//    cleared. The bitmap is zeroed once per block, not once per row.
template <typename V, bool SYM, int kRlItems>
__global__ void __launch_bounds__(kRbThreads, 1)
    k_rowbm_light(RowBitmapArgs a, int nwords, int wwords, int cap, int te_cap, int region_bytes) {
  const V* __restrict__ a_val = static_cast<const V*>(a.a_val);
  const V* __restrict__ b_val = static_cast<const V*>(a.b_val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);

  extern __shared__ __align__(16) unsigned char smem[];
  int64_t* s_bs = reinterpret_cast<int64_t*>(smem);                       // te_cap
  V* s_av = reinterpret_cast<V*>(s_bs + te_cap);                // te_cap (numeric)
  int* s_pre = reinterpret_cast<int*>(SYM ? static_cast<void*>(s_bs + te_cap) : static_cast<void*>(s_av + te_cap));
  uint16_t* s_ent = reinterpret_cast<uint16_t*>(s_pre + te_cap);          // cap: entry of each product position
  V* vals = reinterpret_cast<V*>(smem);                         // numeric, after the products are loaded
  const int ngroups = (nwords + kGroupWords - 1) / kGroupWords;           // symbolic: the whole row
  const int nbw = SYM ? ngroups * kGroupWords : wwords;                   // bitmap words (whole groups)
  const int nbg = nbw / kGroupWords, nsw = (nbg + 31) / 32;               // groups, summary words
  uint32_t* bm = reinterpret_cast<uint32_t*>(smem + region_bytes);
  unsigned char* tail = reinterpret_cast<unsigned char*>(bm + nbw);
  // numeric only: nbg group prefixes, the nsw-word group summary, the list of up to nbg groups
  uint16_t* gpre = reinterpret_cast<uint16_t*>(tail);
  uint32_t* gsum = reinterpret_cast<uint32_t*>(tail + light_a16(static_cast<int64_t>(nbg) * 2));
  uint16_t* glist = reinterpret_cast<uint16_t*>(reinterpret_cast<unsigned char*>(gsum) +
                                                light_a16(static_cast<int64_t>(nsw) * 4));
  __shared__ int64_t s_item;
  __shared__ int ws[33];
  constexpr int T = kRbThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  zero_words(bm, nbw);  // rows leave the bitmap and the summary clear
  if (!SYM)
    for (int i = threadIdx.x; i < nsw; i += T) gsum[i] = 0u;
  while (true) {
    if (threadIdx.x == 0) s_item = atomicAdd(a.work_counter, 1u);
    __syncthreads();
    const int64_t item = s_item;
    if (item >= a.n_items) break;
    const int64_t r = a.rows[item];
    const int64_t lo = a.a_rp[r], ne = a.a_rp[r + 1] - lo;
    uint32_t col[kRlItems];
    V val[kRlItems];
#pragma unroll
    for (int k = 0; k < kRlItems; ++k) {
      col[k] = kNoCol;
      val[k] = 0.0;
    }
    int64_t P0 = 0;  // products of the earlier entry tiles
    for (int64_t e0 = 0; e0 < ne; e0 += te_cap) {
      const int nt = static_cast<int>(min(static_cast<int64_t>(te_cap), ne - e0));
      __syncthreads();  // the previous tile's table is no longer read
      for (int i = threadIdx.x; i < nt; i += T) {
        const int64_t p = lo + e0 + i;
        const int kb = a.a_col[p];
        const int64_t bs = a.b_rp[kb];
        s_bs[i] = bs;
        s_pre[i] = static_cast<int>(a.b_rp[kb + 1] - bs);
        if (!SYM) s_av[i] = a_val[p];
      }
      __syncthreads();
      int tot;
      {
        const int per = (nt + T - 1) / T;
        const int i0 = threadIdx.x * per, i1 = min(nt, i0 + per);
        int acc = 0;
        for (int i = i0; i < i1; ++i) acc += s_pre[i];
        int run = block_exclusive_scan(acc, ws, &tot);
        for (int i = i0; i < i1; ++i) {
          const int x = s_pre[i];
          s_pre[i] = run;
          run += x;
        }
      }
      __syncthreads();
      {  // position -> entry map of this tile (positions beyond the registers or the map are never read)
        const int npos = min(tot, min(cap, static_cast<int>(static_cast<int64_t>(T) * kRlItems - min(P0, static_cast<int64_t>(T) * kRlItems))));
        for (int i = warp; i < nt; i += T / 32) {
          const int st = s_pre[i];
          const int en = min(i + 1 < nt ? s_pre[i + 1] : tot, npos);
          for (int q = st + lane; q < en; q += 32) s_ent[q] = static_cast<uint16_t>(i);
        }
        if (tot > cap && threadIdx.x == 0) atomicOr(a.status, kStInternal);
      }
      __syncthreads();
      // register slots this tile fills (the same for every thread): the symbolic
      // pass skips the others (in the numeric pass the branches cost registers)
      const int k0 = static_cast<int>(min(static_cast<int64_t>(kRlItems), P0 / T));
      const int k1 = static_cast<int>(min(static_cast<int64_t>(kRlItems), (P0 + tot + T - 1) / T));
      int ent[kRlItems];
#pragma unroll
      for (int k = 0; k < kRlItems; ++k) {
        ent[k] = -1;
        if (SYM && (k < k0 || k >= k1)) continue;
        const int64_t rel = static_cast<int64_t>(k) * T + threadIdx.x - P0;
        if (rel >= 0 && rel < tot && rel < cap) {
          const int lo_i = s_ent[rel];
          ent[k] = lo_i;
          const int64_t bi = s_bs[lo_i] + (rel - s_pre[lo_i]);
          col[k] = static_cast<uint32_t>(a.b_col[bi]);
          if (!SYM) val[k] = b_val[bi];
        }
      }
#pragma unroll
      for (int k = 0; k < kRlItems; ++k) {
        if ((!SYM || (k >= k0 && k < k1)) && ent[k] >= 0) {
          if (!SYM) val[k] *= s_av[ent[k]];
          if (SYM) atomicOr(&bm[col[k] >> 5], 1u << (col[k] & 31));
        }
      }
      P0 += tot;
    }
    __syncthreads();
    if (P0 > static_cast<int64_t>(T) * kRlItems) {  // more products than the registers hold
      if (threadIdx.x == 0) atomicOr(a.status, kStInternal);
      continue;  // uniform: every thread saw the same P0
    }
    if (SYM) {  // popcount and clear of the whole row (cheaper here than a group summary)
      int n = 0;
      uint4* b4 = reinterpret_cast<uint4*>(bm);
      for (int i = threadIdx.x; i < nbw / 4; i += T) {
        const uint4 q = b4[i];
        n += __popc(q.x) + __popc(q.y) + __popc(q.z) + __popc(q.w);
        b4[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      n = warp_reduce_sum(n);
      if (lane == 0) ws[warp] = n;
      __syncthreads();
      if (warp == 0) {
        int t = lane < T / 32 ? ws[lane] : 0;
        t = warp_reduce_sum(t);
        if (lane == 0) a.c_rp[r] = t;
      }
      __syncthreads();
      continue;
    }
    // Numeric: the columns are taken window by window (wwords bitmap words each);
    // per window: bits, group ranks (conflict-free group counts), the products'
    // values added into their rank's slot, then the window's part of the row
    // written in column order.
    V* const vals = reinterpret_cast<V*>(smem);                       // cap
    const int64_t out = a.c_rp[r];
    int done = 0;
    for (int64_t base = 0; base < static_cast<int64_t>(nwords) * 32; base += static_cast<int64_t>(wwords) * 32) {
      uint32_t cw[kRlItems];  // column inside the window, kNoCol outside
#pragma unroll
      for (int k = 0; k < kRlItems; ++k) {
        const int64_t c = static_cast<int64_t>(col[k]) - base;
        cw[k] = (col[k] != kNoCol && c >= 0 && c < static_cast<int64_t>(wwords) * 32) ? static_cast<uint32_t>(c) : kNoCol;
        if (cw[k] != kNoCol && atomicOr(&bm[cw[k] >> 5], 1u << (cw[k] & 31)) == 0u)
          atomicOr(&gsum[cw[k] >> 13], 1u << ((cw[k] >> 8) & 31));  // the word's first bit marks its group
      }
      __syncthreads();
      // the window's groups in column order; counts of consecutive listed groups
      // per thread, scanned into group prefixes
      const int ng = list_groups(gsum, nsw, glist, ws);
      const int per = (ng + T - 1) / T;
      const int j0 = min(ng, static_cast<int>(threadIdx.x) * per), j1 = min(ng, j0 + per);
      int acc = 0;
      for (int j = j0; j < j1; ++j) {
        const int g = glist[j];
        const int c = group_popc(bm, g);
        gpre[g] = static_cast<uint16_t>(c);
        acc += c;
      }
      int nnz;
      int run = block_exclusive_scan(acc, ws, &nnz);
      for (int j = j0; j < j1; ++j) {
        const int g = glist[j];
        const int x = gpre[g];
        gpre[g] = static_cast<uint16_t>(run);
        run += x;
      }
      if (done + nnz > cap) {  // uniform: the bin promised at most cap products
        if (threadIdx.x == 0) atomicOr(a.status, kStInternal);
        break;
      }
      for (int i = threadIdx.x; i < nnz; i += T) vals[i] = 0.0;
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kRlItems; ++k)
        if (cw[k] != kNoCol) atomicAdd(&vals[bitmap_rank(bm, gpre, cw[k])], val[k]);
      __syncthreads();
      for (int j = threadIdx.x; j < ng; j += T) {  // listed groups round-robin: adjacent output per warp
        const int g = glist[j];
        const uint4* g4 = reinterpret_cast<const uint4*>(bm + g * kGroupWords);
        const uint4 q0 = g4[0], q1 = g4[1];
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        int pos = gpre[g];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          uint32_t bits = words[x];
          while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1;
            if (GM_CHECKED(out + done + pos < a.c_nnz, a.status)) {
              a.c_col[out + done + pos] = static_cast<int32_t>(base + (g * kGroupWords + x) * 32 + b);
              c_val[out + done + pos] = vals[pos];
            }
            ++pos;
          }
        }
        zero_group(bm, g);
      }
      for (int i = threadIdx.x; i < nsw; i += T) gsum[i] = 0u;
      done += nnz;
      __syncthreads();
    }
  }
}

// Numeric region: the row's values by rank (8 * cap); while a row's products
// are loaded it holds the entry table and the position map.
// After the numeric bitmap: 16-bit group prefixes, the group summary and the
// 16-bit list of the groups it marks, each on a 16-byte boundary.
int64_t light_tail_bytes(int64_t words, bool symbolic) {
  const int64_t g = words / kGroupWords;
  return symbolic ? 0 : light_a16(g * 2) + light_a16((g + 31) / 32 * 4) + light_a16(g * 2);
}
int64_t light_region_bytes(int cap, bool symbolic) {
  return symbolic ? kLightSymRegion : ((static_cast<int64_t>(cap) * 8 + 16 + 15) & ~int64_t(15));
}

// Bitmap words per column window of the numeric kernel: the whole row when it
// fits beside the region, else halved (a multiple of 8 words); 0 when none fits.
int64_t light_window_words(int64_t c_m, int cap, int64_t smem_max) {
  const int64_t nwords = (c_m + 31) / 32;
  int64_t w = (nwords + kGroupWords - 1) / kGroupWords * kGroupWords;
  while (w >= kGroupWords) {
    if (light_region_bytes(cap, false) + w * 4 + light_tail_bytes(w, false) + 4096 <= smem_max) return w;
    w = (w / 2 + kGroupWords - 1) / kGroupWords * kGroupWords;
    if (w == kGroupWords && light_region_bytes(cap, false) + w * 4 + light_tail_bytes(w, false) + 4096 > smem_max)
      return 0;
  }
  return 0;
}

}  // namespace

int64_t rowbm_symbolic_smem(int64_t c_m) { return ((c_m + 127) / 128) * 16; }

int64_t rowbm_light_smem(int64_t c_m, int cap, bool symbolic, int64_t smem_max) {
  if (symbolic) {
    const int64_t nwords = (c_m + 31) / 32;
    const int64_t ngroups = (nwords + kGroupWords - 1) / kGroupWords;
    return light_region_bytes(cap, true) + ngroups * kGroupWords * 4 + light_tail_bytes(ngroups * kGroupWords, true);
  }
  const int64_t w = light_window_words(c_m, cap, smem_max);
  return light_region_bytes(cap, false) + w * 4 + light_tail_bytes(w, false);
}

bool rowbm_light_fits(int64_t c_m, int cap, bool symbolic, int64_t smem_max, int vb) {
  const int items = (symbolic || vb == 4) ? kRlItemsWide : kRlItems;
  if (cap < 1 || cap > kRbThreads * items || c_m > (int64_t(1) << 31)) return false;
  const int64_t te = (light_region_bytes(cap, symbolic) - 2 * static_cast<int64_t>(cap) - 16) / (symbolic ? 12 : 20);
  if (te < 64) return false;
  if (!symbolic && light_window_words(c_m, cap, smem_max) < kGroupWords) return false;
  return rowbm_light_smem(c_m, cap, symbolic, smem_max) + 4096 <= smem_max;
}

void launch_rowbm_light(const RowBitmapArgs& a, bool symbolic, int cap, int num_sms, int64_t smem_max, cudaStream_t s) {
  if (a.n_items <= 0) return;
  cudaMemsetAsync(a.work_counter, 0, sizeof(unsigned int), s);
  const int nwords = static_cast<int>((a.c_m + 31) / 32);
  const int64_t region = light_region_bytes(cap, symbolic);
  const int te_cap = static_cast<int>((region - 2 * static_cast<int64_t>(cap) - 16) / (symbolic ? 12 : 20));
  const int wwords = symbolic ? 0 : static_cast<int>(light_window_words(a.c_m, cap, smem_max));
  const size_t smem = static_cast<size_t>(rowbm_light_smem(a.c_m, cap, symbolic, smem_max));
  const int64_t blocks = std::min<int64_t>(a.n_items, num_sms);
  // products a thread holds: the fewest that cover the bin's cap, so that the
  // unrolled per-product loops carry no empty slots (more than kRlItems only for
  // symbolic passes and float values)
  const int items = cap <= kRbThreads ? 1 : cap <= 2 * kRbThreads ? 2 : cap <= 4 * kRbThreads ? 4
                    : cap <= 8 * kRbThreads ? 8 : cap <= kRlItems * kRbThreads ? kRlItems : kRlItemsWide;
  auto pick = [items](auto f1, auto f2, auto f4, auto f8, auto f10, auto f16) {
    return items == 1 ? f1 : items == 2 ? f2 : items == 4 ? f4 : items == 8 ? f8 : items == kRlItems ? f10 : f16;
  };
  auto fn = symbolic ? pick(k_rowbm_light<double, true, 2>, k_rowbm_light<double, true, 2>,
                            k_rowbm_light<double, true, 4>, k_rowbm_light<double, true, 8>,
                            k_rowbm_light<double, true, kRlItems>, k_rowbm_light<double, true, kRlItemsWide>)
            : a.f32  ? pick(k_rowbm_light<float, false, 1>, k_rowbm_light<float, false, 2>,
                            k_rowbm_light<float, false, 4>, k_rowbm_light<float, false, 8>,
                            k_rowbm_light<float, false, kRlItems>, k_rowbm_light<float, false, kRlItemsWide>)
                     : pick(k_rowbm_light<double, false, 1>, k_rowbm_light<double, false, 2>,
                            k_rowbm_light<double, false, 4>, k_rowbm_light<double, false, 8>,
                            k_rowbm_light<double, false, kRlItems>, k_rowbm_light<double, false, kRlItems>);
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  (fn<<<static_cast<unsigned>(blocks), kRbThreads, smem, s>>>(a, nwords, wwords, cap, te_cap,
                                                               static_cast<int>(region)), note_launch());
}

void launch_rowbm(const RowBitmapArgs& a, int num_sms, int64_t smem_max, cudaStream_t s) {
  if (a.n_items <= 0) return;
  cudaMemsetAsync(a.work_counter, 0, sizeof(unsigned int), s);
  const int64_t nwords4 = rowbm_words(a.c_m);  // whole uint4 stores
  const size_t smem = static_cast<size_t>(rowbm_symbolic_smem(a.c_m));
  const int per_sm = std::max<int>(1, static_cast<int>(smem_max / static_cast<int64_t>(smem + 1024)));
  const int64_t blocks = std::min<int64_t>(a.n_items, static_cast<int64_t>(num_sms) * std::min(per_sm, 2));
  cudaFuncSetAttribute(k_rowbm_symbolic, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  (k_rowbm_symbolic<<<static_cast<unsigned>(blocks), kRbThreads, smem, s>>>(a, static_cast<int>(nwords4)),
   note_launch());
}

}  // namespace gm

namespace gm {

namespace {

// bcp[k * (v + 1) + c] = number of stored B[k, j] with j >> shift < c, for c in
// [0, v] (one warp per B row: shared per-warp histogram, then a warp scan). In a
// row sorted by column, chunk c of the row is the index range [bcp[c], bcp[c+1]).
__global__ void k_b_chunk_prefix(const int64_t* __restrict__ b_rp, const int32_t* __restrict__ b_col, int64_t n_rows,
                                 int v, int shift, int32_t* __restrict__ bcp) {
  extern __shared__ int sh[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int* h = sh + w * v;
  const int per = (v + 31) / 32;  // chunks per lane, contiguous
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * nw + w; k < n_rows; k += static_cast<int64_t>(gridDim.x) * nw) {
    for (int c = lane; c < v; c += 32) h[c] = 0;
    __syncwarp();
    for (int64_t q = b_rp[k] + lane; q < b_rp[k + 1]; q += 32)
      atomicAdd(&h[static_cast<uint32_t>(b_col[q]) >> shift], 1);
    __syncwarp();
    int sum = 0;
    for (int c = lane * per; c < min(v, lane * per + per); ++c) sum += h[c];
    int run = warp_inclusive_scan(sum) - sum;
    int32_t* const out = bcp + k * (v + 1);
    for (int c = lane * per; c < min(v, lane * per + per); ++c) {
      out[c] = run;
      run += h[c];
    }
    if (lane == 31) out[v] = run;
    __syncwarp();
  }
}

// cnt[h * v + c] += elements of chunk c of heavy row h: the heavy rows' A entries,
// concatenated (anz = prefix of their lengths), are cut into segments of 256 per
// warp; each entry adds the chunk counts of the B row it selects, and a warp
// flushes its sums with one atomic per chunk whenever its segment leaves a row.
constexpr int kSegEntries = 256;

__global__ void k_heavy_chunk_counts(const int32_t* __restrict__ rows, int64_t n, const int64_t* __restrict__ anz,
                                     const int64_t* __restrict__ a_rp, const int32_t* __restrict__ a_col,
                                     const int32_t* __restrict__ bcp, int v, unsigned long long* __restrict__ cnt) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = anz[n];
  const int nc = (v + 31) / 32;  // <= 8 chunks per lane
  for (int64_t seg = warp; seg * kSegEntries < total; seg += nw) {
    const int64_t e0 = seg * kSegEntries, e1 = min(e0 + kSegEntries, total);
    int64_t lo = 0, hi = n - 1;  // heavy row holding entry e0
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (anz[mid] <= e0) lo = mid; else hi = mid - 1;
    }
    int64_t h = lo;
    int64_t row_end = anz[h + 1];
    int64_t pbase = a_rp[rows[h]] - anz[h];
    int acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int64_t e = e0; e < e1; ++e) {
      while (e >= row_end) {
        for (int i = 0; i < nc; ++i) {
          const int c = i * 32 + lane;
          if (c < v && acc[i]) atomicAdd(&cnt[h * v + c], static_cast<unsigned long long>(acc[i]));
          acc[i] = 0;
        }
        ++h;
        row_end = anz[h + 1];
        pbase = a_rp[rows[h]] - anz[h];
      }
      const int32_t* const t = bcp + static_cast<int64_t>(a_col[pbase + e]) * (v + 1);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = i * 32 + lane;
        if (i < nc && c < v) acc[i] += t[c + 1] - t[c];
      }
    }
    for (int i = 0; i < nc; ++i) {
      const int c = i * 32 + lane;
      if (c < v && acc[i]) atomicAdd(&cnt[h * v + c], static_cast<unsigned long long>(acc[i]));
    }
  }
}

}  // namespace

void build_chunk_starts(const int64_t* b_rp, const int32_t* b_col, int64_t b_rows, int v, int shift, int32_t* bcp,
                        cudaStream_t s) {
  const int warps = 8;
  if (b_rows > 0)
    (k_b_chunk_prefix<<<grid_for(b_rows * 32, warps * 32), warps * 32, warps * v * sizeof(int), s>>>(
         b_rp, b_col, b_rows, v, shift, bcp), note_launch());
}

bool heavy_chunk_counts(const int32_t* heavy_rows, int64_t n_heavy, const int64_t* anz, const int64_t* a_rp,
                        const int32_t* a_col, const int64_t* b_rp, const int32_t* b_col, int64_t b_rows, int v,
                        int shift, int32_t* bcp, int64_t* cnt, cudaStream_t s) {
  if (v > 256) return false;
  if (b_rp) build_chunk_starts(b_rp, b_col, b_rows, v, shift, bcp, s);
  if (n_heavy <= 0 || cnt == nullptr) return true;
  cudaMemsetAsync(cnt, 0, static_cast<size_t>(n_heavy) * v * sizeof(int64_t), s);
  (k_heavy_chunk_counts<<<152 * 16, 256, 0, s>>>(heavy_rows, n_heavy, anz, a_rp, a_col, bcp, v,
                                                 reinterpret_cast<unsigned long long*>(cnt)), note_launch());
  return true;
}

}  // namespace gm
