// gm_stream.cu -- streamed numeric accumulation of large chunks (gMAGNUS
// Sec. III-E, the dense accumulator; Sec. III-C stages a chunk's tiles in local
// memory, here they arrive by bulk asynchronous copies).
//
// One block per SM, warp-specialised:
//  * the producer warp (one elected lane) takes chunks from a work counter and
//    streams each chunk's elements, in tiles of kTile, into a ring of kStages
//    shared-memory stages with cp.async.bulk (global -> shared, completion
//    counted in bytes on the stage's "full" mbarrier). A tile's copy starts at
//    the 16-byte boundary at or below its first element and ends at the one at
//    or above its last, so the element arrays must stay readable up to 16 bytes
//    past their end; the stage header tells the consumers how many elements to
//    skip at the front.
//  * the consumer warps wait for a stage, add every element into a dense value
//    array of the chunk's width (shared fp64 / fp32 atomics) and mark its column
//    with a plain byte store (lanes holding a sorted run of columns would all
//    meet on one word of a bitmap), then release the stage ("empty" mbarrier,
//    one arrival a warp). After a chunk's last tile they pack the marks into
//    bitmap words, scan them, write the chunk's row of C in column order and
//    clear what they used.
// Each element is read once from HBM (10 bytes with 16-bit chunk columns and
// double values), and the copies of the next tiles overlap the adds of the
// current one. Every wait is bounded in time; a wait that gives up sets
// kStWaitTimeout in the status word and the block stops (the producer first
// waits, also bounded, for its copies in flight).
#include <algorithm>

#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

namespace {

constexpr int kTile = 2048;            // elements a stage holds
constexpr int kStages = 3;
constexpr int kConsumers = 512;        // consumer threads (16 warps); the producer warp comes after them
constexpr int kConsumerWarps = kConsumers / 32;
constexpr uint64_t kWaitNs = 2000000000ull;  // a wait gives up after 2 s

__host__ __device__ constexpr int round16(int x) { return (x + 15) & ~15; }
template <typename CT>
__host__ __device__ constexpr int col_stage_bytes() { return round16(kTile * static_cast<int>(sizeof(CT)) + 16); }
template <typename V>
__host__ __device__ constexpr int val_stage_bytes() { return round16(kTile * static_cast<int>(sizeof(V)) + 16); }

struct StageHdr {
  int64_t item;   // index into the class's item list; -1: no more chunks
  int n;          // elements in the tile
  int c_skip;     // elements before the tile's first one in the copied column bytes
  int v_skip;     // the same for the values
  int last;       // the chunk's last tile
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// The producer's arrival on a "full" barrier, announcing the bytes its copies will deliver.
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Waits until the barrier's phase of the given parity has completed; false when
// kWaitNs passed first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = now_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (now_ns() - t0 > kWaitNs) return false;
  }
}
// Bulk copy of `bytes` (a multiple of 16) from global to shared memory, both
// 16-byte aligned; completion is counted on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Barrier of the consumer warps on an mbarrier (one arrival a warp), bounded in
// time like every wait here: false when it gave up. phase counts the uses.
__device__ __forceinline__ bool consumers_sync(uint64_t* bar, uint32_t& phase) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase & 1u);
  ++phase;
  __syncwarp();
  return ok;
}

// Exclusive scan over the consumer threads; *total gets the sum. False when a
// barrier gave up.
__device__ __forceinline__ bool consumer_scan(int x, int* ws, uint64_t* bar, uint32_t& phase, int* pre, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int inc = warp_inclusive_scan(x);
  if (lane == 31) ws[warp] = inc;
  if (!consumers_sync(bar, phase)) return false;
  if (warp == 0) {
    const int w = lane < kConsumerWarps ? ws[lane] : 0;
    const int wi = warp_inclusive_scan(w);
    if (lane < kConsumerWarps) ws[lane] = wi - w;
    if (lane == kConsumerWarps - 1) ws[32] = wi;
  }
  if (!consumers_sync(bar, phase)) return false;
  *total = ws[32];
  *pre = ws[warp] + inc - x;
  return true;
}

constexpr int kMaxWordsPerThread = 4;  // bitmap words a consumer thread packs (chunks up to 65536 columns)

// The 32 marks (bytes, 0 or 1) of columns 32w .. 32w + 31 as one bitmap word:
// multiplying the 4 marks of a 32-bit word by 0x01020408 gathers them into bits
// 24..27 (no two partial products share a bit, so nothing carries).
__device__ __forceinline__ uint32_t pack_marks(const uint8_t* m) {
  const uint4* m4 = reinterpret_cast<const uint4*>(m);
  const uint4 q0 = m4[0], q1 = m4[1];
  const uint32_t x[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) bits |= (((x[i] & 0x01010101u) * 0x01020408u) >> 24 & 0xFu) << (4 * i);
  return bits;
}

__device__ __forceinline__ int64_t chunk_col_base(const ListArgs& a, int64_t child_local) {
  const int64_t parent = child_local / a.v;
  const int64_t base = a.parent_colbase ? a.parent_colbase[parent] : 0;
  return base + (child_local % a.v) * a.width;
}

template <typename V, typename CT>
__global__ void __launch_bounds__(kConsumers + 32, 1) k_leaf_stream(ListArgs a, int nwords) {
  const CT* __restrict__ in_col = static_cast<const CT*>(a.col);
  const V* __restrict__ in_val = static_cast<const V*>(a.val);
  V* __restrict__ c_val = static_cast<V*>(a.c_val);
  constexpr int kColBytes = col_stage_bytes<CT>();
  constexpr int kStageBytes = kColBytes + val_stage_bytes<V>();

  extern __shared__ __align__(128) unsigned char smem[];
  const int width = nwords * 32;
  V* vals = reinterpret_cast<V*>(smem);                                // width
  uint8_t* touched = reinterpret_cast<uint8_t*>(vals + width);         // width: 1 where a column was met
  unsigned char* stages = touched + width;                             // kStages * kStageBytes, 16-aligned
  __shared__ StageHdr hdr[kStages];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], cbar;
  __shared__ int ws[33];
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  for (int i = tid; i < width; i += blockDim.x) vals[i] = V(0);
  for (int i = tid; i < width / 16; i += blockDim.x) reinterpret_cast<uint4*>(touched)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&cbar, kConsumerWarps);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (tid >= kConsumers) {  // ---- producer warp
    if (tid != kConsumers) return;
    int64_t k = 0;  // tiles issued
    bool ok = true;
    // Waits (bounded) until the copies of the last tiles issued have landed. A
    // parity wait only tells the current phase from the one before it, so this
    // runs before the stop marker arrives on a stage (which advances its phase).
    auto drain = [&]() {
      bool landed = true;
      for (int64_t j = k > kStages ? k - kStages : 0; j < k; ++j)
        landed &= mbar_wait(&full[j % kStages], static_cast<uint32_t>((j / kStages) & 1));
      if (!landed) atomicOr(a.status, kStWaitTimeout);
    };
    for (bool more = true; more && ok;) {
      const int64_t item = static_cast<int64_t>(atomicAdd(a.counter, 1u));
      more = item < a.n_items;
      int64_t lo = 0, n = 0;
      if (more) {
        const int64_t m = a.items[item];
        lo = a.rp[m];
        n = a.rp[m + 1] - lo;
      }
      const int64_t tiles = more && n > kTile ? (n + kTile - 1) / kTile : 1;
      for (int64_t t = 0; t < tiles; ++t, ++k) {
        const int st = static_cast<int>(k % kStages);
        const int64_t round = k / kStages;
        if (round > 0 && !mbar_wait(&empty[st], static_cast<uint32_t>((round - 1) & 1))) {
          ok = false;
          break;
        }
        StageHdr h{};
        if (!more) {  // no more chunks: an empty stage tells the consumers to stop
          drain();
          h.item = -1;
          hdr[st] = h;
          mbar_arrive(&full[st]);
          break;
        }
        const int64_t e0 = lo + t * kTile;
        const int nt = static_cast<int>(n - t * kTile < kTile ? n - t * kTile : kTile);
        const uintptr_t c0 = reinterpret_cast<uintptr_t>(in_col + e0), c1 = reinterpret_cast<uintptr_t>(in_col + e0 + nt);
        const uintptr_t v0 = reinterpret_cast<uintptr_t>(in_val + e0), v1 = reinterpret_cast<uintptr_t>(in_val + e0 + nt);
        const uintptr_t ca = c0 & ~uintptr_t(15), va = v0 & ~uintptr_t(15);
        const uintptr_t cr = ((c1 - ca) + 15) & ~uintptr_t(15), vr = ((v1 - va) + 15) & ~uintptr_t(15);
        const uint32_t cb = static_cast<uint32_t>(cr < 16 ? 16 : cr), vb = static_cast<uint32_t>(vr < 16 ? 16 : vr);
        h.item = item;
        h.n = nt;
        h.c_skip = static_cast<int>((c0 - ca) / sizeof(CT));
        h.v_skip = static_cast<int>((v0 - va) / sizeof(V));
        h.last = t + 1 == tiles;
        hdr[st] = h;
        unsigned char* dst = stages + static_cast<size_t>(st) * kStageBytes;
        mbar_arrive_tx(&full[st], cb + vb);
        bulk_copy_g2s(dst, reinterpret_cast<const void*>(ca), cb, &full[st]);
        bulk_copy_g2s(dst + kColBytes, reinterpret_cast<const void*>(va), vb, &full[st]);
      }
    }
    if (!ok) {  // the consumers stopped taking tiles: let the copies in flight land before leaving
      atomicOr(a.status, kStWaitTimeout);
      s_abort = 1;
      drain();
    }
    return;
  }

  // ---- consumer warps
  const int lane = tid & 31;
  uint32_t cphase = 0;
  int64_t k = 0;
  bool ok = true;
  while (ok) {
    const int st = static_cast<int>(k % kStages);
    if (!mbar_wait(&full[st], static_cast<uint32_t>((k / kStages) & 1)) || s_abort) {
      ok = false;
      break;
    }
    const StageHdr h = hdr[st];
    if (h.item < 0) break;
    const unsigned char* src = stages + static_cast<size_t>(st) * kStageBytes;
    const CT* cs = reinterpret_cast<const CT*>(src) + h.c_skip;
    const V* vs = reinterpret_cast<const V*>(src + kColBytes) + h.v_skip;
#pragma unroll 4
    for (int i = tid; i < h.n; i += kConsumers) {
      const uint32_t c = static_cast<uint32_t>(cs[i]);
      if (!GM_CHECKED(c < static_cast<uint32_t>(width), a.status)) continue;
      touched[c] = 1;
      atomicAdd(&vals[c], vs[i]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    ++k;
    if (!h.last) continue;
    // the chunk is complete: its row of C in column order
    if (!consumers_sync(&cbar, cphase)) {
      ok = false;
      break;
    }
    const int64_t m = a.items[h.item];
    const int64_t child_local = a.child_of ? a.child_of[m] : m;
    const int64_t out = a.off_in[a.child_base + child_local];
    const int64_t cbase = chunk_col_base(a, child_local);
    const int per = nwords / kConsumers;  // words a thread, consecutive (nwords is a multiple of kConsumers)
    const int w0 = tid * per;
    uint32_t words[kMaxWordsPerThread];
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kMaxWordsPerThread; ++j) {
      words[j] = j < per ? pack_marks(touched + (w0 + j) * 32) : 0u;
      cnt += __popc(words[j]);
    }
    int pos = 0, total = 0;
    if (!consumer_scan(cnt, ws, &cbar, cphase, &pos, &total)) {
      ok = false;
      break;
    }
    if (a.expect_nnz && tid == 0) GM_CHECKED(total == a.expect_nnz[a.child_base + child_local], a.status);
#pragma unroll
    for (int j = 0; j < kMaxWordsPerThread; ++j) {
      if (j >= per) break;
      const int w = w0 + j;
      uint32_t bits = words[j];
      while (bits) {
        const int col = w * 32 + __ffs(bits) - 1;
        bits &= bits - 1;
        if (GM_CHECKED(out + pos < a.c_nnz, a.status)) {
          a.c_col[out + pos] = static_cast<int32_t>(cbase + col);
          c_val[out + pos] = vals[col];
        }
        vals[col] = V(0);
        ++pos;
      }
      uint4* t4 = reinterpret_cast<uint4*>(touched + w * 32);
      t4[0] = make_uint4(0u, 0u, 0u, 0u);
      t4[1] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (!consumers_sync(&cbar, cphase)) {
      ok = false;
      break;
    }
  }
  if (!ok && lane == 0) atomicOr(a.status, kStWaitTimeout);
}

template <typename V, typename CT>
size_t stream_smem(int nwords) {
  return static_cast<size_t>(nwords) * 32 * sizeof(V) + static_cast<size_t>(nwords) * 32 +
         static_cast<size_t>(kStages) * (col_stage_bytes<CT>() + val_stage_bytes<V>());
}

int stream_words(int64_t width) {
  return static_cast<int>(((width + 31) / 32 + kConsumers - 1) / kConsumers * kConsumers);
}

template <typename V, typename CT>
void launch_stream_t(const ListArgs& a, int num_sms, cudaStream_t s) {
  const int nwords = stream_words(a.width);
  const size_t smem = stream_smem<V, CT>(nwords);
  cudaFuncSetAttribute(k_leaf_stream<V, CT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  cudaMemsetAsync(a.counter, 0, sizeof(unsigned int), s);
  const unsigned g = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(a.n_items, num_sms)));
  (k_leaf_stream<V, CT><<<g, kConsumers + 32, smem, s>>>(a, nwords), note_launch());
}

}  // namespace

bool leaf_stream_fits(int64_t width, bool col16, int64_t smem_max, int vb) {
  if (width > 65536) return false;
  const int nwords = stream_words(width);
  size_t need;
  if (vb == 4) need = col16 ? stream_smem<float, uint16_t>(nwords) : stream_smem<float, int32_t>(nwords);
  else need = col16 ? stream_smem<double, uint16_t>(nwords) : stream_smem<double, int32_t>(nwords);
  return static_cast<int64_t>(need) + 2048 <= smem_max;  // + the static arrays
}

void launch_leaf_stream(const ListArgs& a, int num_sms, cudaStream_t s) {
  if (a.n_items <= 0) return;
  if (a.f32 && a.col16) launch_stream_t<float, uint16_t>(a, num_sms, s);
  else if (a.f32) launch_stream_t<float, int32_t>(a, num_sms, s);
  else if (a.col16) launch_stream_t<double, uint16_t>(a, num_sms, s);
  else launch_stream_t<double, int32_t>(a, num_sms, s);
}

}  // namespace gm
