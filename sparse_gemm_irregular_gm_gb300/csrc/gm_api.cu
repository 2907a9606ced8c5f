// gm_api.cu -- the C ABI (include/gm_spgemm.h) and the host driver of gMAGNUS
// Algorithm 3: setup, heavy-row batches through outer product and hierarchical
// multisplit, light rows through the binned shared-memory accumulators, and the
// prefix sums that place every row and chunk of C.
#include <algorithm>
#include <climits>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "gm_device.cuh"
#include "gm_internal.h"

namespace gm {

// ---- workspace allocation ------------------------------------------------------

static gm_alloc_fn g_alloc = nullptr;
static gm_free_fn g_free = nullptr;
static gm_avail_fn g_avail = nullptr;
static void* g_ctx = nullptr;
static std::atomic<int64_t> g_ws_now{0}, g_ws_peak{0};
static std::atomic<int64_t> g_launches{0};

static std::atomic<int> g_launch_err{0};

// Counts the launch and records a failed launch (checked at the next sync point).
void note_launch(int n) {
  g_launches += n;
  const cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) g_launch_err = static_cast<int>(e);
}
int64_t launch_count() { return g_launches.load(); }

static bool env_log_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("GM_SPGEMM_LOG");
    return e && e[0] == '1';
  }();
  return on;
}

void* ws_alloc(size_t bytes, cudaStream_t s) {
  if (bytes == 0) return nullptr;
  void* p = nullptr;
  if (g_alloc) {
    p = g_alloc(g_ctx, bytes, s);
  } else if (cudaMallocAsync(&p, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    p = nullptr;
  }
  if (!p && env_log_enabled())
    std::fprintf(stderr, "[gm_spgemm] workspace allocation of %.3f GB failed (%.3f GB held)\n", bytes / 1e9,
                 g_ws_now.load() / 1e9);
  if (p) {
    const int64_t now = g_ws_now += static_cast<int64_t>(bytes);
    int64_t pk = g_ws_peak.load();
    while (now > pk && !g_ws_peak.compare_exchange_weak(pk, now)) {
    }
  }
  return p;
}

void ws_free(void* p, size_t bytes, cudaStream_t s) {
  if (!p) return;
  g_ws_now -= static_cast<int64_t>(bytes);
  if (g_free) g_free(g_ctx, p, bytes, s);
  else cudaFreeAsync(p, s);
}

// ---- small helper kernels --------------------------------------------------------

namespace {

__global__ void k_sub_to_u64(const int64_t* __restrict__ src, int64_t n, int64_t base,
                             unsigned long long* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = static_cast<unsigned long long>(src[i] - base);
}
__global__ void k_sub_i64(const int64_t* __restrict__ src, int64_t n, int64_t base, int64_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = src[i] - base;
}
__global__ void k_i32_to_i64(const int32_t* __restrict__ src, int64_t n, int64_t add, int64_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = static_cast<int64_t>(src[i]) + add;
}
// heavy children first: bin 0 when count > tau, else bin 1
__global__ void k_heavy_bin(const unsigned long long* __restrict__ cnt, int64_t n, int64_t tau,
                            uint8_t* __restrict__ bin) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    bin[i] = cnt[i] > static_cast<unsigned long long>(tau) ? 0 : 1;
}
// mapped counts: out[m] = cnt[perm[m]] (perm null: identity)
__global__ void k_mapped_counts(const unsigned long long* __restrict__ cnt, const int32_t* __restrict__ perm,
                                int64_t n, int64_t* __restrict__ out, int64_t* __restrict__ inv) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t m = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; m < n; m += stride) {
    const int64_t c = perm ? perm[m] : m;
    out[m] = static_cast<int64_t>(cnt[c]);
    if (inv) inv[c] = m;
  }
}
// cursor of child c = the start of the mapped row it became: rrp[inv[c]]
__global__ void k_child_cursor(const int64_t* __restrict__ rrp, const int64_t* __restrict__ inv, int64_t n,
                               unsigned long long* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < n; c += stride)
    out[c] = static_cast<unsigned long long>(rrp[inv[c]]);
}
// column base of each new parent: base_prev[g / v] + (g % v) * w, g = global child id at the previous level
__global__ void k_child_colbase(const int64_t* __restrict__ ids, int64_t n, const int64_t* __restrict__ base_prev,
                                int64_t v, int64_t w, int64_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t g = ids[i];
    out[i] = (base_prev ? base_prev[g / v] : 0) + (g % v) * w;
  }
}
__global__ void k_i32_gather_to_i64(const int32_t* __restrict__ perm, int64_t n, int64_t add,
                                    int64_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = perm[i] + add;
}

// Size class of a last-level chunk for the numeric accumulators: 0 empty; by
// elements 1 (<= 128), 2 (<= 512), 7 (<= 1024): one warp a chunk; 8 (<= 2048),
// 3 (<= 4096): one block; more elements, by columns: 4 (<= 4096), 5 (<= 8192)
// one block, 6 (more) one block with a value array of the chunk's width, or with
// double values the streamed accumulator.
__global__ void k_leaf_class(const int64_t* __restrict__ mcount, const int64_t* __restrict__ nnz, int64_t n,
                             int64_t nnz_base, uint8_t* __restrict__ cls) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t c = mcount[i];
    uint8_t k = 0;
    if (c > 0) {
      if (c <= 128) k = 1;
      else if (c <= 512) k = 2;
      else if (c <= 1024) k = 7;
      else if (c <= 2048) k = 8;
      else if (c <= 4096) k = 3;
      else {
        const int64_t z = nnz[nnz_base + i];
        k = z <= 4096 ? 4 : z <= 8192 ? 5 : 6;
      }
    }
    cls[i] = k;
  }
}

// f[i] = 1 when chunk i has more than min_elems elements (its bitmap is kept)
__global__ void k_keep_flags(const int64_t* __restrict__ cnt, int64_t n, int64_t min_elems, int64_t* __restrict__ f) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    f[i] = cnt[i] > min_elems ? 1 : 0;
}
__global__ void k_keep_slots(const int64_t* __restrict__ cnt, const int64_t* __restrict__ pre, int64_t n,
                             int64_t min_elems, int32_t* __restrict__ slot) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    slot[i] = cnt[i] > min_elems ? static_cast<int32_t>(pre[i]) : -1;
}

}  // namespace

static void sub_to_u64(const int64_t* src, int64_t n, int64_t base, unsigned long long* dst, cudaStream_t s) {
  if (n > 0) (k_sub_to_u64<<<grid_for(n, 256), 256, 0, s>>>(src, n, base, dst), note_launch());
}
static void sub_i64(const int64_t* src, int64_t n, int64_t base, int64_t* dst, cudaStream_t s) {
  if (n > 0) (k_sub_i64<<<grid_for(n, 256), 256, 0, s>>>(src, n, base, dst), note_launch());
}
static void i32_to_i64(const int32_t* src, int64_t n, int64_t add, int64_t* dst, cudaStream_t s) {
  if (n > 0) (k_i32_to_i64<<<grid_for(n, 256), 256, 0, s>>>(src, n, add, dst), note_launch());
}

// ---- parameters (Sec. III-D) -----------------------------------------------------

static int64_t floor_pow2(int64_t x) {
  int64_t p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}
static int64_t next_pow2(int64_t x) {
  int64_t p = 1;
  while (p < x) p *= 2;
  return p;
}
static int ilog2(int64_t x) {
  int l = 0;
  while ((int64_t(1) << l) < x) ++l;
  return l;
}
static bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

constexpr int64_t kSizeCol = 4, kSizeRowPtr = 8, kSizeHisto = 4, kSizeBitmap = 1, kSubGroups = 32;

// s_C.val of Sec. III-D: bytes of one value of the configured type (0 for an unknown type).
static int64_t value_bytes(const gm_config* cfg) {
  const int32_t t = cfg ? cfg->value_type : GM_VALUE_F64;
  return t == GM_VALUE_F64 ? 8 : t == GM_VALUE_F32 ? 4 : 0;
}
constexpr int64_t kDefaultSmem = 232448;  // opt-in shared memory per block on sm_103a

// GetMagnusParams: Eq. (4) tau, n_denseNumeric, Eq. (5)-(6) n_chunksMax, Eq. (7) levels.
static gm_status compute_params(int64_t c_m, const gm_config* cfg, int64_t smem_dev, gm_params* out) {
  if (!out || c_m < 1) return GM_ERR_INVALID_ARG;
  gm_params p;
  std::memset(&p, 0, sizeof(p));
  const int64_t kSizeVal = value_bytes(cfg);
  if (kSizeVal == 0) return GM_ERR_INVALID_ARG;
  p.s_lm = (cfg && cfg->smem_budget_bytes) ? cfg->smem_budget_bytes : smem_dev;
  if (p.s_lm < 1024 || p.s_lm > smem_dev) return GM_ERR_INVALID_ARG;
  const int64_t tau_eq4 = p.s_lm / (2 * (kSizeCol + kSizeVal));
  p.tau = (cfg && cfg->tau) ? cfg->tau : tau_eq4;
  if (p.tau < 1 || p.tau > tau_eq4) return GM_ERR_INVALID_ARG;
  const int64_t n_dense = p.s_lm / (kSizeVal + kSizeBitmap);
  p.dense_width = (cfg && cfg->dense_width) ? cfg->dense_width : floor_pow2(n_dense);
  // the widest chunk's values and its bitmap with word prefix must fit one block
  if (!is_pow2(p.dense_width) || p.dense_width * kSizeVal + p.dense_width / 4 + 1024 > smem_dev)
    return GM_ERR_INVALID_ARG;
  p.n_chunks_required = next_pow2((c_m + p.dense_width - 1) / p.dense_width);
  const int64_t n_min = p.s_lm / (2 * (kSizeCol + kSizeVal));
  const int64_t n_gr = (n_min - 1 + p.tau - 1) / p.tau + 1;
  const int64_t ncm_raw = (p.s_lm - n_min * (kSizeCol + kSizeVal) - kSizeHisto) /
                          (n_gr * kSubGroups * kSizeHisto + kSizeRowPtr * n_gr);
  if (cfg && cfg->n_chunks_max) {
    if (!is_pow2(cfg->n_chunks_max) || cfg->n_chunks_max < 2) return GM_ERR_INVALID_ARG;
    p.n_chunks_max = cfg->n_chunks_max;
  } else {
    if (ncm_raw < 1) return GM_ERR_INVALID_ARG;
    p.n_chunks_max = floor_pow2(ncm_raw);
  }
  const int64_t req = p.n_chunks_required;
  if (req > 1 && p.n_chunks_max < 2) return GM_ERR_INVALID_ARG;  // levels needed but none can split
  if (req == 1) {
    p.n_levels = 0;
  } else if (req <= p.n_chunks_max) {
    p.n_levels = 1;
    p.v_chunks[0] = req;
  } else {
    const int lr = ilog2(req), lm = ilog2(p.n_chunks_max);
    p.n_levels = (lr + lm - 1) / lm;
    if (p.n_levels > GM_MAX_LEVELS) return GM_ERR_INDEX_OVERFLOW;
    int64_t prod = 1;
    for (int64_t i = 0; i + 1 < p.n_levels; ++i) {
      p.v_chunks[i] = p.n_chunks_max;
      prod *= p.n_chunks_max;
    }
    p.v_chunks[p.n_levels - 1] = req / prod;
  }
  int64_t w = p.dense_width * req;
  for (int64_t i = 0; i < p.n_levels; ++i) {
    w /= p.v_chunks[i];
    p.widths[i] = w;
  }
  if (p.dense_width * req > (int64_t(1) << 32)) return GM_ERR_INDEX_OVERFLOW;
  *out = p;
  return GM_OK;
}

}  // namespace gm

namespace gm {

namespace {
__global__ void k_row_len(const int64_t* __restrict__ rp, const int32_t* __restrict__ idx, int64_t n,
                          int64_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t r = idx[i];
    out[i] = rp[r + 1] - rp[r];
  }
}
}  // namespace

// Device array that keeps its contents when it grows.
struct GrowBuf {
  int64_t* p = nullptr;
  size_t cap = 0;
  cudaStream_t s = nullptr;
  bool ensure(size_t need, size_t keep, cudaStream_t stream) {
    s = stream;
    if (need <= cap) return true;
    size_t nc = std::max(need, cap * 2);
    int64_t* q = static_cast<int64_t*>(ws_alloc(nc * sizeof(int64_t), stream));
    if (!q) return false;
    if (p && keep) cudaMemcpyAsync(q, p, keep * sizeof(int64_t), cudaMemcpyDeviceToDevice, stream);
    if (p) ws_free(p, cap * sizeof(int64_t), stream);
    p = q;
    cap = nc;
    return true;
  }
  void release() {
    if (p) ws_free(p, cap * sizeof(int64_t), s);
    p = nullptr;
    cap = 0;
  }
  ~GrowBuf() { release(); }
};

struct StageEv {
  int stage;
  cudaEvent_t a, b;      // with GM_FLAG_TIMING only
  cudaStream_t on;       // the stream the stage's work runs on
  nvtxRangeId_t range;   // NVTX range of the stage's host calls (0 once ended)
};

// NVTX names of the stages (gm_stage order) and of the public calls; a profiler
// shows where each stage's work was issued, with or without GM_FLAG_TIMING.
const char* const kStageNvtx[GM_NUM_STAGES] = {
    "gm:analyze",   "gm:transpose",     "gm:outer",      "gm:histogram",     "gm:multisplit", "gm:sym_heavy",
    "gm:sym_light", "gm:scan",          "gm:num_heavy",  "gm:num_light",     "gm:other",      "gm:transpose_sym",
    "gm:outer_sym", "gm:histogram_sym", "gm:multisplit_sym", "gm:unused"};

struct NvtxCall {  // one range around a public call, ended on every return path
  explicit NvtxCall(const char* name) { nvtxRangePushA(name); }
  ~NvtxCall() { nvtxRangePop(); }
  NvtxCall(const NvtxCall&) = delete;
  NvtxCall& operator=(const NvtxCall&) = delete;
};

struct LevelDbg {
  DevBuf<int64_t> rp;
  DevBuf<int32_t> col;
  DevBuf<unsigned char> val;  // bytes of the plan's value type
  DevBuf<int64_t> child;
  int64_t rows = 0, nnz = 0;
};

// Row bins of the analysis: 0 empty, 1..10 light (u <= tau), 11 heavy.
constexpr int kRowBins = 12;
constexpr int kHeavyBin = 11;

}  // namespace gm

namespace gm {
// A CSR operand as the path reads it: int64 row pointers, int32 columns (the
// caller's arrays, or the plan's converted copies for other index types).
struct CsrDev {
  int64_t n_rows = 0, n_cols = 0, nnz = 0;
  const int64_t* row_ptr = nullptr;
  const int32_t* col_idx = nullptr;
  const void* vals = nullptr;
};
}  // namespace gm

struct gm_plan {
  gm::CsrDev A{}, B{};
  gm_config cfg{};
  cudaStream_t s = nullptr;
  int device = 0;
  int64_t smem_dev = 0;
  int num_sms = 1;
  int64_t c_m = 1;
  bool sym_rowbm = false;  // heavy symbolic through whole-row bitmaps
  bool rowwise = false;    // numeric heavy path: row-order expansion fused with the multisplit
  bool b_sorted = false;   // every row of B has non-decreasing columns (runs per chunk are contiguous)
  int32_t b_unsorted_h = 0;  // 1: some B row decreases, 2: some B row repeats a column
  bool b_strict = false;   // every row of B has strictly increasing columns
  bool f32 = false;        // values are float (GM_VALUE_F32), else double
  int vb = 8;              // bytes of a value
  int arena_cb = 4;        // bytes of a column in the element arenas (2: chunk-local uint16)
  bool rowexp0 = false;    // two or more levels: level 0 by the row-order expansion, no C-hat
  int32_t index_type = 0;  // GM_INDEX_* flags of the caller's arrays
  gm::DevBuf<int64_t> a_rp64, b_rp64, c_rp64;  // int32 row pointers widened (C: until numeric)
  gm::DevBuf<int64_t> a_rps;                   // row pointers of a row range of A, rebased to 0
  gm::DevBuf<int32_t> a_col32, b_col32;        // int64 columns narrowed
  gm_params P{};
  int L = 0;
  int state = 0;  // 1 analyzed, 2 symbolic done, 3 numeric done, 4 C.nnz does not fit int32 row pointers
  int pipeline = GM_PIPE_FUSED_HISTO;
  bool timing = false, log = false, keep = false;
  gm::DevBuf<int> status;
  gm::DevBuf<unsigned int> work_counter;
  gm::DevBuf<int64_t> u;
  gm::DevBuf<uint8_t> bin;
  gm::DevBuf<int32_t> rows_by_bin;
  gm::DevBuf<int64_t> bin_start_d;
  int64_t bin_start[gm::kMaxBins + 1] = {};
  int64_t n_heavy = 0, n_light = 0, n_empty = 0, ip_total = 0, ip_heavy = 0;
  gm::DevBuf<int64_t> chat_rp;      // C-hat.rowPtr over all heavy rows (n_heavy + 1)
  gm::DevBuf<int64_t> heavy_ids64;  // x_heavy as int64
  gm::DevBuf<int64_t> anz;          // prefix of nnz(A[x_heavy[h], :]) (n_heavy + 1)
  gm::DevBuf<int64_t> cnt0;         // row-order pipeline: elements of each level-0 chunk (n_heavy * v0)
  gm::DevBuf<int32_t> bcp;          // row-order pipeline: per-B-row level-0 chunk starts (B.n_rows * (v0 + 1))
  gm::DevBuf<int32_t> bm_slot;      // chunk-direct: [heavy row * v0 + chunk] slot of a kept bitmap, -1: none
  gm::DevBuf<uint32_t> bm_store;    // ... the column bitmaps of the larger chunks, symbolic to numeric
  gm::DevBuf<int64_t> bct;          // numeric, chunk-direct: chunk-major starts of B's copy
  gm::DevBuf<uint8_t> bc_col, bc_val;  // ... and the chunk-major copy of B (live during numeric)
  std::vector<int64_t> h_chat_rp;   // host copy of chat_rp
  std::vector<int64_t> h_anz;       // prefix of nnz(A[x_heavy[h], :])
  gm::GrowBuf nnz[GM_MAX_LEVELS];        // per level, per child: nnz (symbolic) then output offset
  gm::GrowBuf heavy_list[GM_MAX_LEVELS]; // per level: global ids of heavy children (parents of the next level)
  gm::GrowBuf pbase[GM_MAX_LEVELS];      // per level >= 1: column base of each parent
  gm::DevBuf<int64_t> leaf_nnz;          // nnz of each last-level chunk (kept for sizing numeric work)
  int64_t n_par[GM_MAX_LEVELS + 1] = {};
  int64_t c_nnz = -1;
  int64_t* c_rp = nullptr;
  int64_t n_batches = 0, n_leaves = 0, ws_peak = 0, launches = 0;
  int cuda_error = 0, dev_status = 0;
  float stage_ms[GM_NUM_STAGES] = {};
  std::vector<gm::StageEv> evs;
  // intermediates kept for gm_spgemm_debug_copy
  // Two element buffers (columns, values) reused by every batch and level of a
  // pass: C-hat in buffer 0, level i writes buffer (i + 1) % 2. One allocation
  // (arena_block) holds all four, so a caching allocator sees one fixed size.
  gm::DevBuf<unsigned char> arena_block;
  struct {
    int32_t* p = nullptr;
    size_t n = 0;
  } arena_col[2];
  struct {
    void* p = nullptr;  // n values of the plan's value type
    size_t n = 0;
  } arena_val[2];
  gm::DevBuf<int32_t> dbg_chat_col;
  gm::DevBuf<unsigned char> dbg_chat_val;
  gm::DevBuf<int64_t> dbg_chat_rp;
  std::vector<std::unique_ptr<gm::LevelDbg>> dbg_levels;
  bool dbg_ok = false;

  // GM_FLAG_OVERLAP: the light rows run on a second stream with their own
  // status word and work counter, forked from and joined into the plan's stream
  bool overlap = false;
  cudaStream_t s2 = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  gm::DevBuf<int> status2;
  gm::DevBuf<unsigned int> work_counter2;

  int stage_begin(int stage, cudaStream_t on = nullptr) {
    gm::StageEv e{stage, nullptr, nullptr, on ? on : s, nvtxRangeStartA(gm::kStageNvtx[stage])};
    if (timing) {
      cudaEventCreate(&e.a);
      cudaEventCreate(&e.b);
      cudaEventRecord(e.a, e.on);
    }
    evs.push_back(e);
    return static_cast<int>(evs.size()) - 1;
  }
  void stage_end(int idx) {
    if (idx < 0) return;
    gm::StageEv& e = evs[idx];
    if (e.b) cudaEventRecord(e.b, e.on);
    if (e.range) nvtxRangeEnd(e.range);
    e.range = 0;
  }
  // Adds the recorded stage times (GM_FLAG_TIMING: after the plan's streams are
  // done) and ends any range an early return left open.
  void collect_times() {
    bool events = false;
    for (auto& e : evs) {
      if (e.range) nvtxRangeEnd(e.range);
      if (!e.a) continue;
      events = true;
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, e.a, e.b) == cudaSuccess) stage_ms[e.stage] += ms;
      cudaEventDestroy(e.a);
      cudaEventDestroy(e.b);
    }
    evs.clear();
    if (events) cudaGetLastError();  // an event never recorded (a stage an error cut short)
  }
  ~gm_plan() {
    if (s2) cudaStreamSynchronize(s2);
    if (!evs.empty()) {
      if (timing) cudaStreamSynchronize(s);  // the events must be complete before they are destroyed
      collect_times();
    }
    if (ev_fork) cudaEventDestroy(ev_fork);
    if (ev_join) cudaEventDestroy(ev_join);
    if (s2) cudaStreamDestroy(s2);
  }
};

namespace gm {

static gm_status cuda_status(gm_plan* p, cudaError_t e) {
  if (e == cudaSuccess) return GM_OK;
  if (p) p->cuda_error = static_cast<int>(e);
  if (e == cudaErrorMemoryAllocation) return GM_ERR_OOM;
  return GM_ERR_CUDA;
}

// Small device-to-host reads (counts, totals, row pointers of the heavy rows)
// go through a pinned, device-mapped staging buffer written by a kernel, not
// through a copy engine: a caller that copies large results to the host on
// other streams (C of one part while the next part is computed) keeps the copy
// engines busy, and a readback queued behind such a copy would stall the plan.
// One buffer for the process, taken under a lock; reads larger than it, or when
// it cannot be had, use cudaMemcpyAsync.
namespace {
constexpr size_t kStageBytes = size_t(64) << 20;
std::mutex g_stage_mu;
unsigned char* g_stage_host = nullptr;
unsigned char* g_stage_dev = nullptr;
bool g_stage_failed = false;

__global__ void k_stage_copy(const unsigned char* __restrict__ src, unsigned char* __restrict__ dst, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}
}  // namespace

// Copies bytes from device memory to host memory after the work queued on s, and
// waits for it.
static cudaError_t read_to_host(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  std::unique_lock<std::mutex> lk(g_stage_mu);
  if (!g_stage_host && !g_stage_failed) {
    void* h = nullptr;
    void* d = nullptr;
    if (cudaHostAlloc(&h, kStageBytes, cudaHostAllocMapped | cudaHostAllocPortable) == cudaSuccess &&
        cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess) {
      g_stage_host = static_cast<unsigned char*>(h);
      g_stage_dev = static_cast<unsigned char*>(d);
    } else {
      if (h) cudaFreeHost(h);
      cudaGetLastError();
      g_stage_failed = true;
    }
  }
  if (!g_stage_host || bytes > kStageBytes) {
    lk.unlock();
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
  }
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((bytes + threads - 1) / threads, 1024));
  (k_stage_copy<<<blocks, threads, 0, s>>>(static_cast<const unsigned char*>(src), g_stage_dev, bytes), note_launch());
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) std::memcpy(dst, g_stage_host, bytes);
  return e;
}

// Synchronise the plan's stream and turn CUDA errors and device status bits into a status.
static gm_status sync_check(gm_plan* p) {
  cudaError_t e = cudaStreamSynchronize(p->s);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess && g_launch_err.load() != 0) e = static_cast<cudaError_t>(g_launch_err.exchange(0));
  if (e != cudaSuccess) return cuda_status(p, e);
  int st = 0;
  e = read_to_host(&st, p->status.p, sizeof(int), p->s);
  if (e != cudaSuccess) return cuda_status(p, e);
  if (p->overlap && p->status2.p) {  // the light stream's word (its work is joined into p->s)
    int st2 = 0;
    e = read_to_host(&st2, p->status2.p, sizeof(int), p->s);
    if (e != cudaSuccess) return cuda_status(p, e);
    st |= st2;
  }
  p->dev_status |= st;
  if (st & (kStBadARowPtr | kStBadBRowPtr | kStBadACol | kStBadBCol)) return GM_ERR_BAD_INDEX;
  if (st) return GM_ERR_INTERNAL;  // the library's own checks: never the input's or the driver's fault
  return GM_OK;
}

static bool env_log() {
  const char* e = std::getenv("GM_SPGEMM_LOG");
  return e && e[0] == '1';
}

static gm_status check_csr(const gm_csr* M, int32_t index_type) {
  if (!M || M->n_rows < 0 || M->n_cols < 0 || M->nnz < 0 || !M->row_ptr) return GM_ERR_INVALID_ARG;
  if (M->nnz > 0 && (!M->col_idx || !M->vals)) return GM_ERR_INVALID_ARG;
  if (M->n_rows >= (int64_t(1) << 31) || M->n_cols > (int64_t(1) << 31)) return GM_ERR_INDEX_OVERFLOW;
  if ((index_type & GM_INDEX_ROWPTR32) && M->nnz >= (int64_t(1) << 31)) return GM_ERR_INDEX_OVERFLOW;
  return GM_OK;
}

// The caller's index types (gm_config.index_type) turned into the int64 row
// pointers and int32 columns the path reads: converted copies owned by the plan,
// one per distinct array (A and B of A*A share theirs). Out-of-range int64
// columns become -1, which the validation in analyze_impl reports.
// Rows [r0, r1) of A only (the whole of A when r0 = 0 and r1 = A.n_rows): the
// caller's row pointers are validated whole first, then the range's pointers are
// copied and rebased to start at 0 and its columns and values addressed in
// place, from the range's first entry on.
static gm_status adapt_inputs(gm_plan* p, const gm_csr* A, const gm_csr* B, int64_t r0, int64_t r1) {
  const cudaStream_t s = p->s;
  const bool rp32 = (p->index_type & GM_INDEX_ROWPTR32) != 0;
  const bool col64 = (p->index_type & GM_INDEX_COL64) != 0;
  const bool sliced = r0 != 0 || r1 != A->n_rows;
  const bool shared_rp = B->row_ptr == A->row_ptr && B->n_rows == A->n_rows;
  // whole row pointers as int64
  const int64_t* a_rp = static_cast<const int64_t*>(A->row_ptr);
  const int64_t* b_rp = static_cast<const int64_t*>(B->row_ptr);
  if (rp32) {
    if (!p->a_rp64.alloc(A->n_rows + 1, s)) return GM_ERR_OOM;
    launch_widen_i32(static_cast<const int32_t*>(A->row_ptr), p->a_rp64.p, A->n_rows + 1, s);
    a_rp = p->a_rp64.p;
    if (shared_rp) {
      b_rp = a_rp;
    } else {
      if (!p->b_rp64.alloc(B->n_rows + 1, s)) return GM_ERR_OOM;
      launch_widen_i32(static_cast<const int32_t*>(B->row_ptr), p->b_rp64.p, B->n_rows + 1, s);
      b_rp = p->b_rp64.p;
    }
  }
  int64_t lo = 0, hi = A->nnz;
  const int64_t* a_rp_used = a_rp;
  if (sliced) {
    launch_validate_rowptr(a_rp, A->n_rows, A->nnz, kStBadARowPtr, p->status.p, s);
    const gm_status st = sync_check(p);
    if (st != GM_OK) return st;
    int64_t ends[2] = {0, 0};
    cudaError_t e = read_to_host(&ends[0], a_rp + r0, sizeof(int64_t), s);
    if (e == cudaSuccess) e = read_to_host(&ends[1], a_rp + r1, sizeof(int64_t), s);
    if (e != cudaSuccess) return cuda_status(p, e);
    lo = ends[0];
    hi = ends[1];
    if (!p->a_rps.alloc(r1 - r0 + 1, s)) return GM_ERR_OOM;
    sub_i64(a_rp + r0, r1 - r0 + 1, lo, p->a_rps.p, s);
    a_rp_used = p->a_rps.p;
  }
  p->A.n_rows = r1 - r0;
  p->A.n_cols = A->n_cols;
  p->A.nnz = hi - lo;
  p->A.row_ptr = a_rp_used;
  p->A.vals = static_cast<const unsigned char*>(A->vals) + lo * p->vb;
  p->B.n_rows = B->n_rows;
  p->B.n_cols = B->n_cols;
  p->B.nnz = B->nnz;
  p->B.row_ptr = b_rp;
  p->B.vals = B->vals;
  if (col64) {
    const int64_t* a_col = static_cast<const int64_t*>(A->col_idx) + lo;
    if (!p->a_col32.alloc(p->A.nnz, s)) return GM_ERR_OOM;
    launch_narrow_i64(a_col, p->a_col32.p, p->A.nnz, A->n_cols, s);
    p->A.col_idx = p->a_col32.p;
    if (!sliced && B->col_idx == A->col_idx && B->nnz == A->nnz && B->n_cols == A->n_cols) {
      p->B.col_idx = p->a_col32.p;
    } else {
      if (!p->b_col32.alloc(B->nnz, s)) return GM_ERR_OOM;
      launch_narrow_i64(static_cast<const int64_t*>(B->col_idx), p->b_col32.p, B->nnz, B->n_cols, s);
      p->B.col_idx = p->b_col32.p;
    }
  } else {
    p->A.col_idx = static_cast<const int32_t*>(A->col_idx) + lo;
    p->B.col_idx = static_cast<const int32_t*>(B->col_idx);
  }
  return GM_OK;
}

// Validation first: nothing after it may index with unchecked row pointers or columns.
static gm_status validate_inputs(gm_plan* p) {
  const cudaStream_t s = p->s;
  launch_validate_rowptr(p->A.row_ptr, p->A.n_rows, p->A.nnz, kStBadARowPtr, p->status.p, s);
  launch_validate_rowptr(p->B.row_ptr, p->B.n_rows, p->B.nnz, kStBadBRowPtr, p->status.p, s);
  launch_validate_cols(p->A.col_idx, p->A.nnz, p->A.n_cols, kStBadACol, p->status.p, s);
  launch_validate_cols(p->B.col_idx, p->B.nnz, p->B.n_cols, kStBadBCol, p->status.p, s);
  return sync_check(p);
}

namespace {
// bounds[q] for q in [0, n_parts]: 0, then for 0 < q < n_parts the row r where
// n_parts * S[r] comes closest to q * S[n] (S = exclusive prefix of the row
// products, S[n] their total): of the last r below that target and the first r
// reaching it, the nearer one, the lower on a tie; then n. Without products the
// rows are split evenly.
__global__ void k_row_split(const int64_t* __restrict__ S, int64_t n, int64_t n_parts, int64_t* __restrict__ bounds) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t T = S[n];
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q <= n_parts; q += stride) {
    int64_t r;
    if (q == 0) r = 0;
    else if (q == n_parts) r = n;
    else if (T == 0) r = static_cast<int64_t>(static_cast<__int128>(q) * n / n_parts);
    else {
      const __int128 want = static_cast<__int128>(q) * T;
      int64_t lo = 0, hi = n;  // S[n] * n_parts >= want always holds
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (static_cast<__int128>(n_parts) * S[mid] >= want) hi = mid; else lo = mid + 1;
      }
      r = lo;  // the first row reaching the target; lo > 0 since S[0] = 0 < want
      const __int128 above = static_cast<__int128>(n_parts) * S[lo] - want;
      const __int128 below = want - static_cast<__int128>(n_parts) * S[lo - 1];
      if (below <= above) r = lo - 1;
    }
    bounds[q] = r;
  }
}
template <typename T>
__global__ void k_add_base(T* __restrict__ x, int64_t n, int64_t base) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    x[i] = static_cast<T>(x[i] + base);
}
}  // namespace

// Row split for several GPUs: the products of every row, their prefix, and the
// split points (k_row_split).
static gm_status row_split_impl(gm_plan* p, int64_t n_parts, int64_t* bounds) {
  const cudaStream_t s = p->s;
  const int64_t n = p->A.n_rows;
  gm_status st = validate_inputs(p);
  if (st != GM_OK) return st;
  BinSpec spec{};
  spec.nbins = 2;
  spec.ub[0] = 0;
  spec.ub[1] = INT64_MAX;
  DevBuf<int64_t> u, S, out;
  DevBuf<uint8_t> bin;
  if (!u.alloc(std::max<int64_t>(n, 1), s) || !bin.alloc(std::max<int64_t>(n, 1), s) || !S.alloc(n + 1, s) ||
      !out.alloc(n_parts + 1, s))
    return GM_ERR_OOM;
  launch_ip_count(p->A.row_ptr, p->A.col_idx, n, p->B.row_ptr, u.p, bin.p, spec, s);
  if (n == 0) cudaMemsetAsync(S.p, 0, sizeof(int64_t), s);
  else if (!scan_exclusive_i64(u.p, S.p, n, S.p + n, s)) return GM_ERR_OOM;
  (k_row_split<<<grid_for(n_parts + 1, 256), 256, 0, s>>>(S.p, n, n_parts, out.p), note_launch());
  const cudaError_t e = read_to_host(bounds, out.p, (n_parts + 1) * sizeof(int64_t), s);
  if (e != cudaSuccess) return cuda_status(p, e);
  return sync_check(p);
}

static gm_status analyze_impl(gm_plan* p) {
  const cudaStream_t s = p->s;
  const int64_t n = p->A.n_rows;
  if (!p->work_counter.alloc(1, s)) return GM_ERR_OOM;
  const int t0 = p->stage_begin(GM_STAGE_ANALYZE);
  gm_status st = validate_inputs(p);
  if (st != GM_OK) return st;
  {  // is every B row sorted? (decides how heavy products are scattered into chunks)
    DevBuf<int> flag;
    if (!flag.alloc(1, s)) return GM_ERR_OOM;
    cudaMemsetAsync(flag.p, 0, sizeof(int), s);
    launch_check_sorted(p->B.row_ptr, p->B.col_idx, p->B.n_rows, flag.p, s);
    const cudaError_t e = read_to_host(&p->b_unsorted_h, flag.p, sizeof(int), s);
    if (e != cudaSuccess) return cuda_status(p, e);
    st = sync_check(p);
    if (st != GM_OK) return st;
    p->b_sorted = (p->b_unsorted_h & 1) == 0;
    p->b_strict = p->b_unsorted_h == 0;
  }

  BinSpec spec{};
  spec.nbins = kRowBins;
  spec.ub[0] = 0;
  for (int b = 1; b <= 9; ++b) spec.ub[b] = std::min<int64_t>(light_bin_ub(b), p->P.tau);
  spec.ub[10] = p->P.tau;
  spec.ub[kHeavyBin] = INT64_MAX;
  if (!p->u.alloc(n, s) || !p->bin.alloc(n, s) || !p->rows_by_bin.alloc(n, s) ||
      !p->bin_start_d.alloc(kRowBins + 1, s))
    return GM_ERR_OOM;
  launch_ip_count(p->A.row_ptr, p->A.col_idx, n, p->B.row_ptr, p->u.p, p->bin.p, spec, s);
  if (!partition_by_bin(p->bin.p, n, kRowBins, p->rows_by_bin.p, p->bin_start_d.p, s)) return GM_ERR_OOM;
  DevBuf<int64_t> tmp, tot;
  if (!tmp.alloc(std::max<int64_t>(n, 1), s) || !tot.alloc(2, s)) return GM_ERR_OOM;
  if (!scan_exclusive_i64(p->u.p, tmp.p, n, tot.p, s)) return GM_ERR_OOM;
  cudaError_t re = read_to_host(p->bin_start, p->bin_start_d.p, (kRowBins + 1) * sizeof(int64_t), s);
  if (re == cudaSuccess) re = read_to_host(&p->ip_total, tot.p, sizeof(int64_t), s);
  if (re != cudaSuccess) return cuda_status(p, re);
  st = sync_check(p);
  if (st != GM_OK) return st;
  p->n_empty = p->bin_start[1] - p->bin_start[0];
  p->n_heavy = p->bin_start[kRowBins] - p->bin_start[kHeavyBin];
  p->n_light = p->bin_start[kHeavyBin] - p->bin_start[1];

  // C-hat.rowPtr over the heavy rows and the nnz of their A rows (for batching).
  const int64_t nh = p->n_heavy;
  const int32_t* heavy = p->rows_by_bin.p + p->bin_start[kHeavyBin];
  if (!p->chat_rp.alloc(nh + 1, s) || !p->heavy_ids64.alloc(std::max<int64_t>(nh, 1), s)) return GM_ERR_OOM;
  DevBuf<int64_t>& anz = p->anz;
  if (!anz.alloc(nh + 1, s)) return GM_ERR_OOM;
  cudaMemsetAsync(p->chat_rp.p + nh, 0, sizeof(int64_t), s);
  cudaMemsetAsync(anz.p + nh, 0, sizeof(int64_t), s);
  launch_gather_i64(p->u.p, heavy, nh, p->chat_rp.p, s);
  if (nh > 0) (k_row_len<<<grid_for(nh, 256), 256, 0, s>>>(p->A.row_ptr, heavy, nh, anz.p), note_launch());
  if (!scan_exclusive_i64(p->chat_rp.p, p->chat_rp.p, nh + 1, nullptr, s)) return GM_ERR_OOM;
  if (!scan_exclusive_i64(anz.p, anz.p, nh + 1, nullptr, s)) return GM_ERR_OOM;
  i32_to_i64(heavy, nh, 0, p->heavy_ids64.p, s);
  p->h_chat_rp.resize(nh + 1);
  p->h_anz.resize(nh + 1);
  re = read_to_host(p->h_chat_rp.data(), p->chat_rp.p, (nh + 1) * sizeof(int64_t), s);
  if (re == cudaSuccess) re = read_to_host(p->h_anz.data(), anz.p, (nh + 1) * sizeof(int64_t), s);
  if (re != cudaSuccess) return cuda_status(p, re);
  p->stage_end(t0);
  st = sync_check(p);
  if (st != GM_OK) return st;
  p->ip_heavy = p->h_chat_rp[nh];
  p->n_par[0] = nh;
  return GM_OK;
}

}  // namespace gm

namespace gm {

namespace {
constexpr int64_t kOuterE = 8192;  // outer-product work-group elements (flattened space)

BinSpec bitmap_leaf_spec() {
  BinSpec s{};
  s.nbins = 4;
  s.ub[1] = 1024;
  s.ub[2] = 4096;
  s.ub[3] = INT64_MAX;
  return s;
}
int bitmap_leaf_cap(int b, int64_t width) {
  const int64_t c = b == 1 ? 1024 : b == 2 ? 4096 : width;
  return static_cast<int>(std::min<int64_t>(c, width));
}
BinSpec hash_leaf_spec() {
  BinSpec s{};
  s.nbins = 11;
  for (int b = 1; b <= 9; ++b) s.ub[b] = light_bin_ub(b);
  s.ub[10] = INT64_MAX;
  return s;
}
// Most elements (hence columns) of a light chunk in hash bin b: the bin's bound,
// tau for the top bin (a light chunk holds at most tau elements).
int light_chunk_cap(int b, int64_t tau) {
  return static_cast<int>(b <= 9 ? light_bin_ub(b) : tau);
}
int hash_leaf_cap(int b, int64_t tau, int64_t smem_max, int vb) {
  if (b <= 9) return static_cast<int>(std::max<int64_t>(64, 2 * light_bin_ub(b)));
  return light_bin_cap(10, tau, smem_max, vb);
}
}  // namespace

// Accumulates the chunks [lo, lo + n) (mapped rows of one level's output) whose
// element counts are mcount[lo ...]: bitmap accumulator when `dense`, hash
// otherwise, except numeric light chunks of more than 512 elements, which take
// the bitmap-rank block accumulator when a bitmap of the level's width fits.
static gm_status run_leaves(gm_plan* p, ListArgs la, const int64_t* mcount, int64_t lo, int64_t n, bool dense,
                            bool numeric) {
  if (n <= 0) return GM_OK;
  const cudaStream_t s = p->s;
  // numeric last-level chunks with known nnz: classes sized by nnz (k_leaf_class)
  const bool by_nnz = dense && numeric && p->leaf_nnz.p && la.child_of == nullptr;
  BinSpec spec = dense ? bitmap_leaf_spec() : hash_leaf_spec();
  if (by_nnz) spec.nbins = 9;
  const bool warp_ok = leaf_warpbm_fits(la.width, 1024, p->smem_dev, p->vb);
  const bool blk4k_ok = leaf_blkbm_fits(la.width, 4096, p->smem_dev, p->vb);
  // chunks of more than 8192 columns with double values: streamed through shared
  // memory by bulk copies (measured faster than the block accumulator there, slower
  // for smaller chunks and for float values)
  const bool stream_ok = !p->f32 && leaf_stream_fits(la.width, la.col16, p->smem_dev, p->vb);
  la.counter = p->work_counter.p;
  la.c_nnz = p->c_nnz;
  la.expect_nnz = by_nnz ? p->leaf_nnz.p : nullptr;
  DevBuf<uint8_t> bins;
  DevBuf<int32_t> idx;
  DevBuf<int64_t> starts_d, items;
  if (!bins.alloc(n, s) || !idx.alloc(n, s) || !starts_d.alloc(spec.nbins + 1, s) || !items.alloc(n, s))
    return GM_ERR_OOM;
  if (by_nnz)
    (k_leaf_class<<<grid_for(n, 256), 256, 0, s>>>(mcount + lo, p->leaf_nnz.p, n, la.child_base + lo, bins.p),
     note_launch());
  else
    launch_bin_sizes(mcount + lo, n, bins.p, spec, s);
  if (!partition_by_bin(bins.p, n, spec.nbins, idx.p, starts_d.p, s)) return GM_ERR_OOM;
  int64_t starts[kMaxBins + 1];
  cudaError_t e = read_to_host(starts, starts_d.p, (spec.nbins + 1) * sizeof(int64_t), s);
  if (e != cudaSuccess) return cuda_status(p, e);
  i32_to_i64(idx.p, n, lo, items.p, s);
  for (int b = 1; b < spec.nbins; ++b) {
    const int64_t cnt = starts[b + 1] - starts[b];
    if (cnt <= 0) continue;
    ListArgs a = la;
    a.items = items.p + starts[b];
    a.n_items = cnt;
    p->n_leaves += numeric ? 0 : cnt;
    if (by_nnz) {
      if (b == 1 && warp_ok) launch_leaf_warpbm(a, 128, s);
      else if (b == 1) launch_leaf_warp(a, s);
      else if (b == 2 && warp_ok) launch_leaf_warpbm(a, 512, s);
      else if (b == 7 && warp_ok) launch_leaf_warpbm(a, 1024, s);
      else if (b == 8 && blk4k_ok) launch_leaf_blkbm(a, 2048, 2048, s);
      else if (b == 3 && blk4k_ok) launch_leaf_blkbm(a, 4096, 4096, s);
      else if (b == 6 && stream_ok) launch_leaf_stream(a, p->num_sms, s);
      else if (b == 4 && blk4k_ok) launch_leaf_blkbm(a, 4096, INT_MAX, s);
      else if (b == 5 && leaf_blkbm_fits(la.width, 8192, p->smem_dev, p->vb)) launch_leaf_blkbm(a, 8192, INT_MAX, s);
      else if (b == 6 && leaf_blkbm_fits(la.width, static_cast<int>(la.width), p->smem_dev, p->vb))
        launch_leaf_blkbm(a, static_cast<int>(la.width), INT_MAX, s);
      else if (b == 2 || b == 7) launch_leaf_small(a, 1024, false, s);
      else if (b == 3 || b == 8) launch_leaf_small(a, 4096, false, s);
      else launch_leaf_bitmap(a, static_cast<int>(std::min<int64_t>(b == 4 ? 4096 : b == 5 ? 8192 : la.width, la.width)), false, s);
    } else if (dense && b <= 2) launch_leaf_small(a, b == 1 ? 1024 : 4096, !numeric, s);
    else if (dense) launch_leaf_bitmap(a, bitmap_leaf_cap(b, la.width), !numeric, s);
    else if (numeric && b >= 6 && leaf_blkbm_fits(la.width, light_chunk_cap(b, p->P.tau), p->smem_dev, p->vb))
      launch_leaf_blkbm(a, light_chunk_cap(b, p->P.tau), INT_MAX, s);  // wide light chunk of > 512 elements
    else launch_leaf_hash(a, hash_leaf_cap(b, p->P.tau, p->smem_dev, p->vb), !numeric, s);
  }
  e = cudaGetLastError();
  return cuda_status(p, e);
}

template <class T>
static void dbg_copy(DevBuf<T>& dst, const T* src, int64_t n, cudaStream_t s) {
  if (dst.alloc(std::max<int64_t>(n, 1), s) && n > 0)
    cudaMemcpyAsync(dst.p, src, n * sizeof(T), cudaMemcpyDeviceToDevice, s);
}

// Heavy rows [h0, h1), numeric pass of the row-order pipeline (one level): the
// batch's A entries are gathered in row order, their products expanded straight
// into the level-0 chunks (k_expand_split; C-hat is not written) whose sizes the
// symbolic pass counted, then every chunk is accumulated.
// Accumulates the level-0 chunks of heavy batch rows [h0, h1) (already filled,
// sizes mcount) into C: the numeric leaves of the one-level hierarchy.
static gm_status rowwise_leaves(gm_plan* p, int64_t nb, const int64_t* rrp, const int64_t* mcount, int64_t* par_base,
                                int32_t* c_col, void* c_val, bool col16) {
  const int v = static_cast<int>(p->P.v_chunks[0]);
  ListArgs la{};
  la.f32 = p->f32;
  la.status = p->status.p;
  la.c_col = c_col;
  la.c_val = c_val;
  la.rp = rrp;
  la.col = p->arena_col[0].p;
  la.col16 = col16;
  la.val = p->arena_val[0].p;
  la.child_base = par_base[0] * v;
  la.v = v;
  la.width = p->P.widths[0];
  la.nnz_out = p->nnz[0].p;
  la.off_in = p->nnz[0].p;
  la.bm_slot = p->bm_slot.p;
  la.bm_store = p->bm_store.p;
  const int t = p->stage_begin(GM_STAGE_NUM_HEAVY);
  const gm_status st = run_leaves(p, la, mcount, 0, nb * v, true, true);
  p->stage_end(t);
  par_base[0] += nb;
  if (st != GM_OK) return st;
  return cuda_status(p, cudaGetLastError());
}

// Writes the products of heavy rows [h0, h1) straight into their level-0 chunks
// (B rows sorted, per-B-row chunk starts in p->bcp, v0 <= 64): the batch rows'
// A entries are gathered in row order and k_expand_rows writes each product at
// its chunk's cursor, one contiguous block per (unit of products, row, chunk).
// cursor[c] (child c = batch row * v0 + chunk) is where chunk c's elements start
// in the caller's layout; columns are stored chunk-local (16 bits with col16).
static gm_status expand_into_chunks(gm_plan* p, int64_t h0, int64_t h1, unsigned long long* cursor, void* out_col,
                                    void* out_val, bool col16, bool numeric, const int64_t* chunk_rp = nullptr) {
  const cudaStream_t s = p->s;
  const int64_t nb = h1 - h0;
  const int64_t ip = p->h_chat_rp[h1] - p->h_chat_rp[h0];
  const int64_t ne = p->h_anz[h1] - p->h_anz[h0];
  const int32_t* heavy = p->rows_by_bin.p + p->bin_start[kHeavyBin] + h0;
  int t = p->stage_begin(numeric ? GM_STAGE_TRANSPOSE : GM_STAGE_TRANSPOSE_SYM);
  DevBuf<int32_t> e_row, e_k;
  DevBuf<double> e_a;
  DevBuf<int64_t> e_b, e_off, ufirst;
  const int64_t U = row_runs_unit(p->P.tau);
  const int64_t n_units = (ip + U - 1) / U;
  if (!e_b.alloc(ne, s) || !e_row.alloc(ne, s) || !e_a.alloc(ne, s) || !e_off.alloc(ne + 1, s) ||
      !e_k.alloc(ne, s) || !ufirst.alloc(std::max<int64_t>(n_units, 1), s))
    return GM_ERR_OOM;
  launch_gather_entries(heavy, nb, p->anz.p + h0, p->A.row_ptr, p->A.col_idx, p->A.vals, p->f32, p->B.row_ptr,
                        e_b.p, e_a.p, e_row.p, e_off.p, s, e_k.p);
  cudaMemsetAsync(e_off.p + ne, 0, sizeof(int64_t), s);
  if (!scan_exclusive_i64(e_off.p, e_off.p, ne + 1, nullptr, s)) return GM_ERR_OOM;
  p->stage_end(t);

  t = p->stage_begin(numeric ? GM_STAGE_MULTISPLIT : GM_STAGE_MULTISPLIT_SYM);
  RowRunArgs ra{};
  ra.f32 = p->f32;
  ra.e_k = e_k.p;
  ra.e_b = e_b.p;
  ra.e_a = out_val ? e_a.p : nullptr;
  ra.e_off = e_off.p;
  ra.e_row = e_row.p;
  ra.n_e = ne;
  ra.total = ip;
  ra.U = U;
  ra.n_units = n_units;
  ra.unit_first = ufirst.p;
  ra.b_col = p->B.col_idx;
  ra.b_val = p->B.vals;
  ra.bcp = p->bcp.p;
  ra.v = static_cast<int>(p->P.v_chunks[0]);
  ra.shift = ilog2(p->P.widths[0]);
  ra.cursor = cursor;
  ra.out_col = out_col;
  ra.col16 = col16;
  ra.out_val = out_val;
  ra.unit_counter = p->work_counter.p;
  ra.status = p->status.p;
  ra.chunk_rp = chunk_rp;
  launch_row_runs(ra, p->num_sms, s);
  p->stage_end(t);
  return cuda_status(p, cudaGetLastError());
}

// The products of heavy rows [h0, h1) into their level-0 chunks from the
// chunk-major copy of B (p->bct, p->bc_col, p->bc_val): the batch rows' A
// entries are gathered in row order, then k_expand_cm writes each (row, chunk)
// pair's products as one run at rrp[pair].
static gm_status expand_chunk_major(gm_plan* p, int64_t h0, int64_t h1, const int64_t* rrp, bool col16) {
  const cudaStream_t s = p->s;
  const int64_t nb = h1 - h0;
  const int64_t ne = p->h_anz[h1] - p->h_anz[h0];
  const int32_t* heavy = p->rows_by_bin.p + p->bin_start[kHeavyBin] + h0;
  int t = p->stage_begin(GM_STAGE_TRANSPOSE);
  DevBuf<int32_t> e_k;
  DevBuf<double> e_a;
  DevBuf<unsigned long long> counter;
  if (!e_a.alloc(ne, s) || !e_k.alloc(ne, s) || !counter.alloc(1, s)) return GM_ERR_OOM;
  launch_gather_entries(heavy, nb, p->anz.p + h0, p->A.row_ptr, p->A.col_idx, p->A.vals, p->f32, p->B.row_ptr,
                        nullptr, e_a.p, nullptr, nullptr, s, e_k.p);
  p->stage_end(t);
  t = p->stage_begin(GM_STAGE_MULTISPLIT);
  ChunkMajorArgs ca{};
  ca.nb = nb;
  ca.v = static_cast<int>(p->P.v_chunks[0]);
  ca.anz = p->anz.p + h0;
  ca.e_k = e_k.p;
  ca.e_a = e_a.p;
  ca.f32 = p->f32;
  ca.bct = p->bct.p;
  ca.nB1 = p->B.n_rows + 1;
  ca.bc_col = p->bc_col.p;
  ca.bc_val = p->bc_val.p;
  ca.rrp = rrp;
  ca.out_col = p->arena_col[0].p;
  ca.out_val = p->arena_val[0].p;
  ca.col16 = col16;
  ca.counter = counter.p;
  ca.status = p->status.p;
  launch_expand_cm(ca, p->num_sms, s);
  p->stage_end(t);
  return cuda_status(p, cudaGetLastError());
}

// Chunk-direct pipeline when B's rows are sorted (one level): the products go
// straight into the level-0 chunks, laid out child by child (chunk sizes from the
// symbolic pass); C-hat is never written.
static gm_status run_batch_runs(gm_plan* p, int64_t h0, int64_t h1, int64_t* par_base, int32_t* c_col,
                                void* c_val) {
  const cudaStream_t s = p->s;
  const int64_t nb = h1 - h0;
  const int64_t ip = p->h_chat_rp[h1] - p->h_chat_rp[h0];
  const int v = static_cast<int>(p->P.v_chunks[0]);
  const int64_t children = nb * v;
  if (p->arena_col[0].n < static_cast<size_t>(ip) || p->arena_val[0].n < static_cast<size_t>(ip))
    return GM_ERR_WORKSPACE;
  int t = p->stage_begin(GM_STAGE_HISTOGRAM);
  const int64_t* mcount = p->cnt0.p + h0 * v;  // chunk sizes from the symbolic pass
  DevBuf<int64_t> rrp;
  DevBuf<unsigned long long> cur;
  if (!rrp.alloc(children + 1, s) || !cur.alloc(children, s)) return GM_ERR_OOM;
  if (!scan_exclusive_i64(mcount, rrp.p, children, rrp.p + children, s)) return GM_ERR_OOM;
  sub_to_u64(rrp.p, children, 0, cur.p, s);
  p->stage_end(t);
  const bool col16 = p->arena_cb == 2;  // chunk-local columns in 16 bits: 10 (or 6) bytes a product
  const gm_status st = p->bct.p ? expand_chunk_major(p, h0, h1, rrp.p, col16)
                                : expand_into_chunks(p, h0, h1, cur.p, p->arena_col[0].p, p->arena_val[0].p, col16,
                                                     true, rrp.p);
  if (st != GM_OK) return st;
  cur.release();
  return rowwise_leaves(p, nb, rrp.p, mcount, par_base, c_col, c_val, col16);
}

static gm_status run_batch_rowwise(gm_plan* p, int64_t h0, int64_t h1, int64_t* par_base, int32_t* c_col,
                                   void* c_val) {
  const cudaStream_t s = p->s;
  const int64_t nb = h1 - h0;
  const int64_t ip = p->h_chat_rp[h1] - p->h_chat_rp[h0];
  const int64_t ne = p->h_anz[h1] - p->h_anz[h0];
  const int32_t* heavy = p->rows_by_bin.p + p->bin_start[kHeavyBin] + h0;
  const int v = static_cast<int>(p->P.v_chunks[0]);
  const int64_t children = nb * v;
  if (p->arena_col[0].n < static_cast<size_t>(ip)) return GM_ERR_WORKSPACE;

  if (p->b_sorted && p->P.v_chunks[0] <= 64) return run_batch_runs(p, h0, h1, par_base, c_col, c_val);
  if (ne >= INT32_MAX) return GM_ERR_INDEX_OVERFLOW;  // entries are indexed by int32 inside the kernels
  int t = p->stage_begin(GM_STAGE_TRANSPOSE);
  DevBuf<int32_t> e_row;
  DevBuf<int4> wg_info;
  DevBuf<double> e_a;
  DevBuf<int64_t> e_b, e_off, lrp, bounds;
  const int64_t n_wg = expand_num_wg(ip, ne);
  if (!e_b.alloc(ne, s) || !e_row.alloc(ne, s) || !e_a.alloc(ne, s) || !e_off.alloc(ne + 1, s) ||
      !lrp.alloc(nb + 1, s) || !bounds.alloc(n_wg + 1, s) || !wg_info.alloc(n_wg, s))
    return GM_ERR_OOM;
  launch_gather_entries(heavy, nb, p->anz.p + h0, p->A.row_ptr, p->A.col_idx, p->A.vals, p->f32, p->B.row_ptr, e_b.p, e_a.p,
                        e_row.p, e_off.p, s);
  cudaMemsetAsync(e_off.p + ne, 0, sizeof(int64_t), s);
  if (!scan_exclusive_i64(e_off.p, e_off.p, ne + 1, nullptr, s)) return GM_ERR_OOM;
  sub_i64(p->chat_rp.p + h0, nb + 1, p->h_chat_rp[h0], lrp.p, s);
  launch_expand_bounds(e_off.p, e_row.p, ne, ip, bounds.p, wg_info.p, s);
  p->stage_end(t);

  t = p->stage_begin(GM_STAGE_HISTOGRAM);
  const int64_t* mcount = p->cnt0.p + h0 * v;  // chunk sizes from the symbolic pass
  DevBuf<int64_t> rrp;
  DevBuf<unsigned long long> cur;
  if (!rrp.alloc(children + 1, s) || !cur.alloc(children, s)) return GM_ERR_OOM;
  if (!scan_exclusive_i64(mcount, rrp.p, children, rrp.p + children, s)) return GM_ERR_OOM;
  sub_to_u64(rrp.p, children, 0, cur.p, s);
  p->stage_end(t);

  t = p->stage_begin(GM_STAGE_MULTISPLIT);
  ExpandArgs ea{};
  ea.f32 = p->f32;
  ea.e_b = e_b.p;
  ea.e_a = e_a.p;
  ea.e_off = e_off.p;
  ea.e_row = e_row.p;
  ea.n_e = ne;
  ea.b_rp = p->B.row_ptr;
  ea.b_col = p->B.col_idx;
  ea.b_val = p->B.vals;
  ea.in_rp = lrp.p;
  ea.n_parents = nb;
  ea.bounds = bounds.p;
  ea.wg_info = wg_info.p;
  ea.n_wg = n_wg;
  ea.v = v;
  ea.shift = ilog2(p->P.widths[0]);
  ea.n_group_rows = expand_group_rows(p->P.tau);
  ea.status = p->status.p;
  ea.cursor = cur.p;
  ea.out_col = p->arena_col[0].p;
  ea.out_val = p->arena_val[0].p;
  launch_expand_split(ea, s);
  p->stage_end(t);
  e_b.release();
  e_a.release();
  e_row.release();
  e_off.release();
  cur.release();
  return rowwise_leaves(p, nb, rrp.p, mcount, par_base, c_col, c_val, false);
}

// Heavy rows [h0, h1): outer product, multisplit levels and chunk accumulation.
// Symbolic: leaf nnz into p->nnz[level], heavy children into p->heavy_list / p->pbase.
// Numeric: C entries at the offsets held in p->nnz[level].
static gm_status run_batch(gm_plan* p, int64_t h0, int64_t h1, bool numeric, int64_t* par_base, int32_t* c_col,
                           void* c_val) {
  const cudaStream_t s = p->s;
  const int64_t nb = h1 - h0;
  const int64_t ip = p->h_chat_rp[h1] - p->h_chat_rp[h0];
  const int64_t anz = p->h_anz[h1] - p->h_anz[h0];
  const bool with_val = numeric || p->keep;
  const int32_t* heavy = p->rows_by_bin.p + p->bin_start[kHeavyBin] + h0;
  const int64_t ncols = p->A.n_cols;
  const int L = p->L;
  gm_status st = GM_OK;

  const bool rowexp = p->rowexp0;  // level 0 written by the row-order expansion (no C-hat)
  int t = 0;
  int32_t* chat_col = p->arena_col[0].p;
  void* chat_val = with_val ? p->arena_val[0].p : nullptr;
  DevBuf<int64_t> lrp;
  DevBuf<unsigned long long> cnt0;
  const bool fused = L >= 1 && p->pipeline == GM_PIPE_FUSED_HISTO;
  if (rowexp) {  // level-0 chunk sizes of the batch from the per-B-row chunk starts
    t = p->stage_begin(numeric ? GM_STAGE_HISTOGRAM : GM_STAGE_HISTOGRAM_SYM);
    if (p->arena_col[1].n < static_cast<size_t>(ip) || (with_val && p->arena_val[1].n < static_cast<size_t>(ip)))
      return GM_ERR_WORKSPACE;
    DevBuf<int64_t> anz_b;  // the batch's A-entry prefix, rebased to 0
    if (!anz_b.alloc(nb + 1, s) || !cnt0.alloc(nb * p->P.v_chunks[0], s)) return GM_ERR_OOM;
    sub_i64(p->anz.p + h0, nb + 1, p->h_anz[h0], anz_b.p, s);
    if (!heavy_chunk_counts(heavy, nb, anz_b.p, p->A.row_ptr, p->A.col_idx, nullptr, p->B.col_idx, p->B.n_rows,
                            static_cast<int>(p->P.v_chunks[0]), ilog2(p->P.widths[0]), p->bcp.p,
                            reinterpret_cast<int64_t*>(cnt0.p), s))
      return GM_ERR_OOM;
    p->stage_end(t);
  } else {
  // 1. Masked CSR -> CSC of the batch rows and the slice offsets (Algorithm 3 line 7).
  t = p->stage_begin(numeric ? GM_STAGE_TRANSPOSE : GM_STAGE_TRANSPOSE_SYM);
  DevBuf<int64_t> col_ptr, slice_off;
  DevBuf<int32_t> t_row, wg_op;
  DevBuf<double> t_val;
  const int64_t n_wg_op = (ip + kOuterE - 1) / kOuterE;
  if (!col_ptr.alloc(ncols + 1, s) || !slice_off.alloc(ncols + 1, s) || !t_row.alloc(anz, s) ||
      !t_val.alloc(anz, s) || !wg_op.alloc(n_wg_op, s))
    return GM_ERR_OOM;
  TransposeArgs ta{heavy, nb, p->A.row_ptr, p->A.col_idx, p->A.vals, ncols, p->f32};
  if (!masked_transpose(ta, anz, col_ptr.p, t_row.p, t_val.p, s)) return GM_ERR_OOM;
  if (!slice_offsets(col_ptr.p, p->B.row_ptr, ncols, slice_off.p, s)) return GM_ERR_OOM;
  launch_wg_slice(slice_off.p, ncols, ip, kOuterE, wg_op.p, s);
  p->stage_end(t);

  // 2. Outer product into C-hat (Algorithm 4), optionally counting level-0 chunks.
  t = p->stage_begin(numeric ? GM_STAGE_OUTER : GM_STAGE_OUTER_SYM);
  if (p->arena_col[0].n < static_cast<size_t>(ip) || (with_val && p->arena_val[0].n < static_cast<size_t>(ip)))
    return GM_ERR_WORKSPACE;
  DevBuf<unsigned long long> cursor;
  if (!lrp.alloc(nb + 1, s) || !cursor.alloc(nb, s)) return GM_ERR_OOM;
  sub_i64(p->chat_rp.p + h0, nb + 1, p->h_chat_rp[h0], lrp.p, s);
  sub_to_u64(p->chat_rp.p + h0, nb, p->h_chat_rp[h0], cursor.p, s);
  if (L >= 1) {
    if (!cnt0.alloc(nb * p->P.v_chunks[0], s)) return GM_ERR_OOM;
    cudaMemsetAsync(cnt0.p, 0, cnt0.bytes(), s);
  }
  OuterArgs oa{};
  oa.f32 = p->f32;
  oa.slice_off = slice_off.p;
  oa.col_ptr = col_ptr.p;
  oa.t_row = t_row.p;
  oa.t_val = t_val.p;
  oa.b_rp = p->B.row_ptr;
  oa.b_col = p->B.col_idx;
  oa.b_val = p->B.vals;
  oa.n_slices = ncols;
  oa.total = ip;
  oa.E = kOuterE;
  oa.wg_first = wg_op.p;
  oa.cursor = cursor.p;
  oa.out_col = chat_col;
  oa.out_val = chat_val;
  oa.histo = fused ? cnt0.p : nullptr;
  oa.v = L >= 1 ? static_cast<int>(p->P.v_chunks[0]) : 1;
  oa.shift = L >= 1 ? ilog2(p->P.widths[0]) : 0;
  launch_outer_product(oa, s);
  p->stage_end(t);
  t_row.release();
  t_val.release();
  col_ptr.release();
  slice_off.release();
  wg_op.release();
  cursor.release();
  if (p->keep) {
    dbg_copy(p->dbg_chat_col, static_cast<const int32_t*>(chat_col), ip, s);
    if (with_val) dbg_copy(p->dbg_chat_val, static_cast<const unsigned char*>(chat_val), ip * p->vb, s);
    dbg_copy(p->dbg_chat_rp, lrp.p, nb + 1, s);
  }
  }  // C-hat

  ListArgs base_la{};
  base_la.f32 = p->f32;
  base_la.status = p->status.p;
  base_la.c_col = c_col;
  base_la.c_val = c_val;

  if (L == 0) {  // C.m <= dense width: the rows of C-hat are the chunks
    DevBuf<int64_t> rows_cnt;
    if (!rows_cnt.alloc(nb, s)) return GM_ERR_OOM;
    launch_gather_i64(p->u.p, heavy, nb, rows_cnt.p, s);
    ListArgs la = base_la;
    la.rp = lrp.p;
    la.col = chat_col;
    la.val = chat_val;
    la.child_base = par_base[0];
    la.v = 1;
    la.width = p->c_m;
    la.nnz_out = p->nnz[0].p;
    la.off_in = p->nnz[0].p;
    t = p->stage_begin(numeric ? GM_STAGE_NUM_HEAVY : GM_STAGE_SYM_HEAVY);
    st = run_leaves(p, la, rows_cnt.p, 0, nb, true, numeric);
    p->stage_end(t);
    par_base[0] += nb;
    return st;
  }

  // 3. Hierarchical multisplit (Algorithm 3 lines 10-20) and accumulation of the
  //    chunks that leave the hierarchy at each level.
  const int64_t* in_rp = lrp.p;
  const int32_t* in_col = chat_col;
  const void* in_val = chat_val;
  int64_t P_b = nb, in_total = ip;
  std::unique_ptr<DevBuf<int64_t>> prev_rp;
  for (int i = 0; i < L; ++i) {
    const bool last = i == L - 1;
    const int v = static_cast<int>(p->P.v_chunks[i]);
    const int shift = ilog2(p->P.widths[i]);
    const int64_t children = P_b * v;
    int ngr = 0;
    const int64_t E = multisplit_pick_E(v, p->P.tau, with_val, p->smem_dev - 1024, &ngr);
    if (E == 0) return GM_ERR_INVALID_ARG;

    t = p->stage_begin(numeric ? GM_STAGE_HISTOGRAM : GM_STAGE_HISTOGRAM_SYM);
    const bool expand_here = i == 0 && rowexp;  // level 0 comes from the expansion, not a multisplit
    DevBuf<int32_t> wg;
    if (!expand_here) {
      if (!wg.alloc((in_total + E - 1) / E, s)) return GM_ERR_OOM;
      launch_wg_row(in_rp, P_b, E, wg.p, s);
    }
    SplitArgs sa{};
    sa.f32 = p->f32;
    sa.in_rp = in_rp;
    sa.n_parents = P_b;
    sa.in_col = in_col;
    sa.in_val = in_val;
    sa.base = 0;
    sa.total = in_total;
    sa.v = v;
    sa.shift = shift;
    sa.E = E;
    sa.n_group_rows = ngr;
    sa.wg_first = wg.p;
    sa.status = p->status.p;
    DevBuf<unsigned long long> cnt_own;
    unsigned long long* cnt = cnt0.p;
    if (!(i == 0 && (fused || rowexp))) {
      if (!cnt_own.alloc(children, s)) return GM_ERR_OOM;
      cudaMemsetAsync(cnt_own.p, 0, cnt_own.bytes(), s);
      cnt = cnt_own.p;
      sa.counts = cnt;
      launch_histogram(sa, s);
    }
    // Heavy chunks first (ThreshPartition on the chunk sizes), order kept.
    DevBuf<int32_t> perm;
    DevBuf<int64_t> inv, perm64;
    int64_t nH = 0;
    if (!last) {
      DevBuf<uint8_t> hb;
      DevBuf<int64_t> st2;
      if (!hb.alloc(children, s) || !perm.alloc(children, s) || !st2.alloc(3, s) || !inv.alloc(children, s) ||
          !perm64.alloc(children, s))
        return GM_ERR_OOM;
      (k_heavy_bin<<<grid_for(children, 256), 256, 0, s>>>(cnt, children, p->P.tau, hb.p), note_launch());
      if (!partition_by_bin(hb.p, children, 2, perm.p, st2.p, s)) return GM_ERR_OOM;
      int64_t hst[3];
      cudaError_t e = read_to_host(hst, st2.p, sizeof(hst), s);
      if (e != cudaSuccess) return cuda_status(p, e);
      nH = hst[1] - hst[0];
      i32_to_i64(perm.p, children, 0, perm64.p, s);
    }
    DevBuf<int64_t> mcount;
    auto rrp = std::make_unique<DevBuf<int64_t>>();
    DevBuf<unsigned long long> cur;
    if (!mcount.alloc(children, s) || !rrp->alloc(children + 1, s) || !cur.alloc(children, s)) return GM_ERR_OOM;
    (k_mapped_counts<<<grid_for(children, 256), 256, 0, s>>>(cnt, last ? nullptr : perm.p, children, mcount.p,
                                                            last ? nullptr : inv.p), note_launch());
    if (!scan_exclusive_i64(mcount.p, rrp->p, children, rrp->p + children, s)) return GM_ERR_OOM;
    sub_to_u64(rrp->p, children, 0, cur.p, s);
    p->stage_end(t);

    t = p->stage_begin(numeric ? GM_STAGE_MULTISPLIT : GM_STAGE_MULTISPLIT_SYM);
    int32_t* const out_col = p->arena_col[(i + 1) % 2].p;
    void* const out_val = with_val ? p->arena_val[(i + 1) % 2].p : nullptr;
    sa.inv = last ? nullptr : inv.p;
    sa.cursor = cur.p;
    sa.out_col = out_col;
    sa.out_val = out_val;
    if (expand_here) {  // each child's products go to the start of the row it is mapped to
      p->stage_end(t);
      DevBuf<unsigned long long> ccur;
      if (!ccur.alloc(children, s)) return GM_ERR_OOM;
      (k_child_cursor<<<grid_for(children, 256), 256, 0, s>>>(rrp->p, inv.p, children, ccur.p), note_launch());
      st = expand_into_chunks(p, h0, h1, ccur.p, out_col, out_val, false, numeric);
      if (st != GM_OK) return st;
      t = p->stage_begin(numeric ? GM_STAGE_MULTISPLIT : GM_STAGE_MULTISPLIT_SYM);
    } else {
      launch_multisplit(sa, s);
    }
    p->stage_end(t);
    if (i == 0) cnt0.release();
    if (p->keep) {
      auto d = std::make_unique<LevelDbg>();
      dbg_copy(d->rp, rrp->p, children + 1, s);
      dbg_copy(d->col, static_cast<const int32_t*>(out_col), in_total, s);
      if (with_val) dbg_copy(d->val, static_cast<const unsigned char*>(out_val), in_total * p->vb, s);
      if (!d->child.alloc(children, s)) return GM_ERR_OOM;
      if (last) launch_iota_i64(d->child.p, children, 0, s);
      else cudaMemcpyAsync(d->child.p, perm64.p, children * sizeof(int64_t), cudaMemcpyDeviceToDevice, s);
      d->rows = children;
      d->nnz = in_total;
      p->dbg_levels.push_back(std::move(d));
    }

    // Chunks that leave the hierarchy here: all chunks of the last level (width
    // <= dense width, bitmap accumulator) or the light chunks of a wider level (hash).
    if (!numeric) {
      if (!p->nnz[i].ensure((par_base[i] + P_b) * v, par_base[i] * v, s)) return GM_ERR_OOM;
      cudaMemsetAsync(p->nnz[i].p + par_base[i] * v, 0, children * sizeof(int64_t), s);
    }
    ListArgs la = base_la;
    la.rp = rrp->p;
    la.col = out_col;
    la.val = out_val;
    la.child_of = last ? nullptr : perm64.p;
    la.child_base = par_base[i] * v;
    la.v = v;
    la.width = p->P.widths[i];
    la.parent_colbase = i == 0 ? nullptr : p->pbase[i].p + par_base[i];
    la.nnz_out = p->nnz[i].p;
    la.off_in = p->nnz[i].p;
    t = p->stage_begin(numeric ? GM_STAGE_NUM_HEAVY : GM_STAGE_SYM_HEAVY);
    st = last ? run_leaves(p, la, mcount.p, 0, children, true, numeric)
              : run_leaves(p, la, mcount.p, nH, children - nH, false, numeric);
    p->stage_end(t);
    if (st != GM_OK) return st;

    const int64_t P_old = P_b;
    if (!last && nH > 0) {
      int64_t next_total = 0;
      const cudaError_t re = read_to_host(&next_total, rrp->p + nH, sizeof(int64_t), s);
      if (re != cudaSuccess) return cuda_status(p, re);
      if (!numeric) {
        const int64_t at = par_base[i + 1];
        if (!p->heavy_list[i].ensure(at + nH, at, s) || !p->pbase[i + 1].ensure(at + nH, at, s)) return GM_ERR_OOM;
        (k_i32_gather_to_i64<<<grid_for(nH, 256), 256, 0, s>>>(perm.p, nH, par_base[i] * v, p->heavy_list[i].p + at), note_launch());
        (k_child_colbase<<<grid_for(nH, 256), 256, 0, s>>>(p->heavy_list[i].p + at, nH,
                                                          i == 0 ? nullptr : p->pbase[i].p, v, p->P.widths[i],
                                                          p->pbase[i + 1].p + at), note_launch());
      }
      cudaError_t e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return cuda_status(p, e);
      prev_rp = std::move(rrp);
      in_rp = prev_rp->p;
      in_col = out_col;
      in_val = out_val;
      P_b = nH;
      in_total = next_total;
    }
    par_base[i] += P_old;
    if (last || nH == 0) break;
  }
  return cuda_status(p, cudaGetLastError());
}

}  // namespace gm

namespace gm {

// Splits the heavy rows into consecutive batches whose workspace fits `cap`.
static gm_status plan_batches(gm_plan* p, int64_t bytes_per_ip, int64_t cap,
                              std::vector<std::pair<int64_t, int64_t>>& out) {
  const int64_t nh = p->n_heavy;
  const int64_t v0 = p->L >= 1 ? p->P.v_chunks[0] : 1;
  const int64_t fixed = (p->A.n_cols + 1) * 8 * 3 + (int64_t(4) << 20);
  auto bytes = [&](int64_t h0, int64_t h1) {
    const int64_t ip = p->h_chat_rp[h1] - p->h_chat_rp[h0];
    const int64_t anz = p->h_anz[h1] - p->h_anz[h0];
    return fixed + ip * bytes_per_ip + anz * 24 + (h1 - h0) * (32 + v0 * 72) + ip / 512 * 12;
  };
  out.clear();
  int64_t h0 = 0;
  while (h0 < nh) {
    if (bytes(h0, h0 + 1) > cap) return GM_ERR_WORKSPACE;
    // largest h1 with bytes(h0, h1) <= cap (bytes grows with h1)
    int64_t lo = h0 + 1, hi = nh;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) / 2;
      if (bytes(h0, mid) <= cap) lo = mid; else hi = mid - 1;
    }
    out.emplace_back(h0, lo);
    h0 = lo;
  }
  return GM_OK;
}

static int64_t workspace_cap(gm_plan* p);

// Element buffers for the largest batch of a pass (values only in the numeric pass
// or when intermediates are kept).
static gm_status alloc_arena(gm_plan* p, const std::vector<std::pair<int64_t, int64_t>>& batches, bool with_val,
                             int nbuf = 2) {
  int64_t mx = 0;
  for (auto& b : batches) mx = std::max(mx, p->h_chat_rp[b.second] - p->h_chat_rp[b.first]);
  if (p->log)
    std::fprintf(stderr, "[gm_spgemm] %zu batch(es), largest %lld products, arena %.2f GB\n", batches.size(),
                 (long long)mx, mx * (with_val ? 24.0 : 8.0) / 1e9);
  // 256 bytes past each array's end: the streamed accumulator's bulk copies end
  // at the 16-byte boundary at or above a chunk's last element
  const size_t col_b = ((static_cast<size_t>(mx) * p->arena_cb + 255) / 256) * 256 + 256;
  const size_t val_b = with_val ? ((static_cast<size_t>(mx) * p->vb + 255) / 256) * 256 + 256 : 0;
  if (!p->arena_block.alloc(nbuf * (col_b + val_b), p->s)) return GM_ERR_OOM;
  unsigned char* base = p->arena_block.p;
  for (int k = 0; k < 2; ++k) {
    p->arena_col[k] = {};
    p->arena_val[k] = {};
  }
  for (int k = 0; k < nbuf; ++k) {
    p->arena_val[k].p = with_val ? static_cast<void*>(base + k * val_b) : nullptr;
    p->arena_val[k].n = with_val ? mx : 0;
    p->arena_col[k].p = reinterpret_cast<int32_t*>(base + nbuf * val_b + k * col_b);
    p->arena_col[k].n = mx;
  }
  return GM_OK;
}

static void free_arena(gm_plan* p) {
  p->arena_block.release();
  for (int k = 0; k < 2; ++k) {
    p->arena_col[k] = {};
    p->arena_val[k] = {};
  }
}

// Plans batches under the workspace cap and allocates the arena; when the arena
// does not fit after all (a caching allocator's blocks can be fragmented), the
// cap is halved and the batches planned again, a few times.
static gm_status plan_and_alloc(gm_plan* p, int64_t bytes_per_ip, bool with_val,
                                std::vector<std::pair<int64_t, int64_t>>& batches, int nbuf = 2) {
  int64_t cap = workspace_cap(p);
  for (int attempt = 0; attempt < 6; ++attempt) {
    gm_status st = plan_batches(p, bytes_per_ip, cap, batches);
    // after a failed arena, a budget halved below one row's needs is still an allocation failure
    if (st != GM_OK) return attempt == 0 ? st : GM_ERR_OOM;
    st = alloc_arena(p, batches, with_val, nbuf);
    if (st == GM_OK) return GM_OK;
    free_arena(p);
    cudaStreamSynchronize(p->s);
    cudaGetLastError();
    cap /= 2;
    if (p->log) std::fprintf(stderr, "[gm_spgemm] arena did not fit; retrying with a cap of %.2f GB\n", cap / 1e9);
  }
  return GM_ERR_OOM;
}

static int64_t workspace_cap(gm_plan* p) {
  if (p->cfg.workspace_cap_bytes > 0) return p->cfg.workspace_cap_bytes;
  size_t free_b = 0, total_b = 0;
  cudaStreamSynchronize(p->s);
  if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) {
    cudaGetLastError();
    return int64_t(1) << 30;
  }
  int64_t avail = static_cast<int64_t>(free_b);
  if (g_avail) {
    const int64_t a = g_avail(g_ctx);
    if (a >= 0) avail = a;
  }
  const int64_t reserve = (int64_t(1) << 30) + static_cast<int64_t>(total_b) / 50;
  const int64_t cap = std::max<int64_t>(avail - reserve, int64_t(256) << 20);
  if (p->log)
    std::fprintf(stderr, "[gm_spgemm] free %.2f GB, available %.2f GB, workspace cap %.2f GB\n", free_b / 1e9,
                 avail / 1e9, cap / 1e9);
  return cap;
}

// Light rows, bin by bin, on stream `on` with the given work counter and status word.
static void launch_light(gm_plan* p, bool numeric, int32_t* c_col, void* c_val, cudaStream_t on,
                         unsigned int* counter, int* status) {
  for (int b = 1; b <= 10; ++b) {
    const int64_t cnt = p->bin_start[b + 1] - p->bin_start[b];
    if (cnt <= 0) continue;
    const int cap = b <= 9 ? static_cast<int>(light_bin_ub(b)) : static_cast<int>(p->P.tau);
    // the whole-row bitmap kernel for rows of more than 1024 products in both passes,
    // and in the numeric pass also for rows of 513-1024 products (measured: the hash
    // table and sort were faster for their symbolic pass, slower for the numeric one;
    // both give the same rows of C)
    if ((b >= 7 || (b == 6 && numeric)) && rowbm_light_fits(p->c_m, cap, false, p->smem_dev, p->vb) &&
        rowbm_light_fits(p->c_m, cap, true, p->smem_dev, p->vb)) {
      RowBitmapArgs ra{};
      ra.f32 = p->f32;
      ra.rows = p->rows_by_bin.p + p->bin_start[b];
      ra.n_items = cnt;
      ra.a_rp = p->A.row_ptr;
      ra.a_col = p->A.col_idx;
      ra.a_val = p->A.vals;
      ra.b_rp = p->B.row_ptr;
      ra.b_col = p->B.col_idx;
      ra.b_val = p->B.vals;
      ra.c_m = p->c_m;
      ra.c_rp = p->c_rp;
      ra.c_col = c_col;
      ra.c_val = c_val;
      ra.work_counter = counter;
      ra.status = status;
      ra.c_nnz = p->c_nnz;
      launch_rowbm_light(ra, !numeric, cap, p->num_sms, p->smem_dev, on);
      continue;
    }
    LightArgs la{};
    la.f32 = p->f32;
    la.rows = p->rows_by_bin.p + p->bin_start[b];
    la.n_items = cnt;
    la.a_rp = p->A.row_ptr;
    la.a_col = p->A.col_idx;
    la.a_val = p->A.vals;
    la.b_rp = p->B.row_ptr;
    la.b_col = p->B.col_idx;
    la.b_val = p->B.vals;
    la.c_rp = p->c_rp;
    la.c_col = c_col;
    la.c_val = c_val;
    la.status = status;
    la.c_nnz = p->c_nnz;
    launch_light_rows(la, light_bin_cap(b, p->P.tau, p->smem_dev, p->vb), !numeric, on);
  }
}

// The light rows of one pass: on the plan's stream, or (GM_FLAG_OVERLAP) on the
// second stream after everything queued so far on the plan's stream; join_light
// makes the plan's stream wait for them.
static void run_light(gm_plan* p, bool numeric, int32_t* c_col, void* c_val) {
  const int stage = numeric ? GM_STAGE_NUM_LIGHT : GM_STAGE_SYM_LIGHT;
  if (!p->overlap) {
    const int t = p->stage_begin(stage);
    launch_light(p, numeric, c_col, c_val, p->s, p->work_counter.p, p->status.p);
    p->stage_end(t);
    return;
  }
  cudaEventRecord(p->ev_fork, p->s);
  cudaStreamWaitEvent(p->s2, p->ev_fork, 0);
  const int t = p->stage_begin(stage, p->s2);
  launch_light(p, numeric, c_col, c_val, p->s2, p->work_counter2.p, p->status2.p);
  p->stage_end(t);
  cudaEventRecord(p->ev_join, p->s2);
}
static void join_light(gm_plan* p) {
  if (p->overlap) cudaStreamWaitEvent(p->s, p->ev_join, 0);
}

// Chunk-direct pipeline: the symbolic pass keeps the column bitmap of every
// level-0 chunk of more than 1024 elements (the chunks of the block accumulators
// and of the streamed one), so that the numeric pass loads it instead of marking
// the chunk's columns again. When the store cannot be allocated nothing is kept.
static gm_status keep_chunk_bitmaps(gm_plan* p, int64_t n, RowBitmapArgs& ra) {
  const cudaStream_t s = p->s;
  p->bm_slot.release();
  p->bm_store.release();
  const int64_t width = p->P.widths[0];
  if (width % 32 != 0 || n <= 0) return GM_OK;
  constexpr int64_t kKeepAbove = 1024;
  DevBuf<int64_t> pre;
  if (!pre.alloc(n + 1, s)) return GM_ERR_OOM;
  (k_keep_flags<<<grid_for(n, 256), 256, 0, s>>>(p->cnt0.p, n, kKeepAbove, pre.p), note_launch());
  if (!scan_exclusive_i64(pre.p, pre.p, n, pre.p + n, s)) return GM_ERR_OOM;
  int64_t kept = 0;
  const cudaError_t e = read_to_host(&kept, pre.p + n, sizeof(int64_t), s);
  if (e != cudaSuccess) return cuda_status(p, e);
  const int64_t words = leaf_blkbm_words(width);
  if (kept <= 0 || kept >= (int64_t(1) << 31)) return GM_OK;
  if (!p->bm_slot.alloc(n, s) || !p->bm_store.alloc(kept * words, s)) {
    if (p->log) std::fprintf(stderr, "[gm_spgemm] no room to keep %lld chunk bitmaps; marking them again\n", (long long)kept);
    p->bm_slot.release();
    p->bm_store.release();
    return GM_OK;
  }
  (k_keep_slots<<<grid_for(n, 256), 256, 0, s>>>(p->cnt0.p, pre.p, n, kKeepAbove, p->bm_slot.p), note_launch());
  ra.bm_slot = p->bm_slot.p;
  ra.bm_store = p->bm_store.p;
  ra.store_words = static_cast<int>(words);
  return GM_OK;
}

static gm_status symbolic_impl(gm_plan* p, int64_t* C_rp, int64_t* C_nnz) {
  const cudaStream_t s = p->s;
  const int64_t n = p->A.n_rows;
  p->c_rp = C_rp;
  cudaMemsetAsync(C_rp, 0, (n + 1) * sizeof(int64_t), s);
  run_light(p, false, nullptr, nullptr);
  int t = -1;
  const int L = p->L;
  const int64_t nh = p->n_heavy;
  if (nh > 0) {
    const int64_t v0 = L >= 1 ? p->P.v_chunks[0] : 1;
    if (!p->nnz[0].ensure(nh * v0, 0, s)) return GM_ERR_OOM;
    cudaMemsetAsync(p->nnz[0].p, 0, nh * v0 * sizeof(int64_t), s);
    if (p->sym_rowbm) {
      // whole-row bitmaps: chunk nnz without expanding C-hat (at most one level)
      RowBitmapArgs ra{};
      ra.f32 = p->f32;
      ra.rows = p->rows_by_bin.p + p->bin_start[kHeavyBin];
      ra.n_items = nh;
      ra.a_rp = p->A.row_ptr;
      ra.a_col = p->A.col_idx;
      ra.a_val = p->A.vals;
      ra.b_rp = p->B.row_ptr;
      ra.b_col = p->B.col_idx;
      ra.b_val = p->B.vals;
      ra.c_m = p->c_m;
      ra.v = static_cast<int>(v0);
      ra.width = L >= 1 ? p->P.widths[0] : (int64_t(1) << 40);
      ra.nnz_out = p->nnz[0].p;
      ra.item_base = 0;
      ra.c_rp = C_rp;
      ra.work_counter = p->work_counter.p;
      ra.status = p->status.p;
      const int ts = p->stage_begin(GM_STAGE_SYM_HEAVY);
      const int32_t* hrows = p->rows_by_bin.p + p->bin_start[kHeavyBin];
      const int shift0 = ilog2(p->P.widths[0]);
      if (p->rowwise) {  // per-B-row chunk starts, and the level-0 chunk sizes for the expansion
        if (!p->bcp.alloc(std::max<int64_t>(p->B.n_rows, 1) * (v0 + 1), s)) return GM_ERR_OOM;
        build_chunk_starts(p->B.row_ptr, p->B.col_idx, p->B.n_rows, static_cast<int>(v0), shift0, p->bcp.p, s);
        if (!p->cnt0.alloc(nh * v0, s)) return GM_ERR_OOM;
        if (!heavy_chunk_counts(hrows, nh, p->anz.p, p->A.row_ptr, p->A.col_idx, nullptr, p->B.col_idx,
                                p->B.n_rows, static_cast<int>(v0), shift0, p->bcp.p, p->cnt0.p, s))
          return GM_ERR_OOM;
        const gm_status kst = keep_chunk_bitmaps(p, nh * v0, ra);
        if (kst != GM_OK) return kst;
      }
      launch_rowbm(ra, p->num_sms, p->smem_dev, s);
      p->stage_end(ts);
      p->n_batches = 0;
      p->n_leaves += nh * v0;
      if (L >= 1) sum_children(p->nnz[0].p, p->heavy_ids64.p, C_rp, nh, static_cast<int>(v0), s);
      else launch_scatter_i64(p->nnz[0].p, p->rows_by_bin.p + p->bin_start[kHeavyBin], nh, C_rp, s);
      goto heavy_done;
    }
    std::vector<std::pair<int64_t, int64_t>> batches;
    gm_status st = plan_and_alloc(p, p->keep ? 24 : 8, p->keep, batches);
    if (st != GM_OK) return st;
    if (p->rowexp0) {  // per-B-row starts of the level-0 chunks, for both passes
      if (!p->bcp.alloc(std::max<int64_t>(p->B.n_rows, 1) * (v0 + 1), s)) return GM_ERR_OOM;
      build_chunk_starts(p->B.row_ptr, p->B.col_idx, p->B.n_rows, static_cast<int>(v0), ilog2(p->P.widths[0]),
                         p->bcp.p, s);
    }
    if (p->keep && batches.size() != 1) {  // intermediates are kept for a single batch only
      p->keep = false;
      free_arena(p);
      st = alloc_arena(p, batches, false);
      if (st != GM_OK) return st;
    }
    p->n_batches = static_cast<int64_t>(batches.size());
    int64_t par_base[GM_MAX_LEVELS + 1] = {};
    for (auto& bt : batches) {
      st = run_batch(p, bt.first, bt.second, false, par_base, nullptr, nullptr);
      if (st != GM_OK) return st;
    }
    free_arena(p);
    for (int i = 0; i <= L; ++i) p->n_par[i] = par_base[i];
    p->n_par[0] = nh;
    // bottom-up: a heavy chunk's nnz is the sum over its chunks at the next level
    for (int i = L - 2; i >= 0; --i)
      if (p->n_par[i + 1] > 0)
        sum_children(p->nnz[i + 1].p, p->heavy_list[i].p, p->nnz[i].p, p->n_par[i + 1],
                     static_cast<int>(p->P.v_chunks[i + 1]), s);
    if (L >= 1) sum_children(p->nnz[0].p, p->heavy_ids64.p, C_rp, nh, static_cast<int>(v0), s);
    else launch_scatter_i64(p->nnz[0].p, p->rows_by_bin.p + p->bin_start[kHeavyBin], nh, C_rp, s);
  }
heavy_done:
  if (nh > 0) {  // nnz of the last level's chunks, before they turn into offsets
    const int li = L >= 1 ? L - 1 : 0;
    const int64_t cnt = L >= 1 ? p->n_par[li] * p->P.v_chunks[li] : nh;
    if (cnt > 0 && p->leaf_nnz.alloc(cnt, s))
      cudaMemcpyAsync(p->leaf_nnz.p, p->nnz[li].p, cnt * sizeof(int64_t), cudaMemcpyDeviceToDevice, s);
  }
  join_light(p);  // the light rows' counts are in C_rp
  t = p->stage_begin(GM_STAGE_SCAN);
  if (!scan_exclusive_i64(C_rp, C_rp, n + 1, nullptr, s)) return GM_ERR_OOM;
  {
    const cudaError_t re = read_to_host(&p->c_nnz, C_rp + n, sizeof(int64_t), s);
    if (re != cudaSuccess) return cuda_status(p, re);
  }
  // top-down: output offset of every chunk = its parent's offset + nnz of earlier siblings
  if (nh > 0) {
    if (L >= 1) {
      DevBuf<int64_t> base;
      if (!base.alloc(nh, s)) return GM_ERR_OOM;
      launch_gather_i64_i64(C_rp, p->heavy_ids64.p, nh, base.p, s);
      segmented_offsets(p->nnz[0].p, p->nnz[0].p, base.p, nh, static_cast<int>(p->P.v_chunks[0]), nullptr, s);
      for (int i = 1; i < L; ++i) {
        const int64_t np = p->n_par[i];
        if (np <= 0) break;
        DevBuf<int64_t> b2;
        if (!b2.alloc(np, s)) return GM_ERR_OOM;
        launch_gather_i64_i64(p->nnz[i - 1].p, p->heavy_list[i - 1].p, np, b2.p, s);
        segmented_offsets(p->nnz[i].p, p->nnz[i].p, b2.p, np, static_cast<int>(p->P.v_chunks[i]), nullptr, s);
      }
    } else {
      launch_gather_i64_i64(C_rp, p->heavy_ids64.p, nh, p->nnz[0].p, s);
    }
  }
  p->stage_end(t);
  gm_status st = sync_check(p);
  if (st != GM_OK) return st;
  p->dbg_ok = p->keep;
  if (C_nnz) *C_nnz = p->c_nnz;
  return GM_OK;
}

static gm_status numeric_impl(gm_plan* p, int32_t* C_col, void* C_val) {
  run_light(p, true, C_col, C_val);
  if (p->n_heavy > 0) {
    const bool keep = p->keep;
    p->keep = false;
    std::vector<std::pair<int64_t, int64_t>> batches;
    // the chunk-direct expansion stores chunk-local columns in 16 bits
    p->arena_cb = p->rowwise && p->b_sorted && p->P.v_chunks[0] <= 64 && p->P.widths[0] <= 65536 ? 2 : 4;
    if (p->rowwise && p->b_sorted && p->P.v_chunks[0] <= 64) {
      // chunk-major copy of B for the expansion (when it does not fit, the row-order one runs)
      const int v0 = static_cast<int>(p->P.v_chunks[0]);
      const int t = p->stage_begin(GM_STAGE_TRANSPOSE);
      if (p->bct.alloc(bchunk_starts_len(p->B.n_rows, v0), p->s) &&
          p->bc_col.alloc(std::max<int64_t>(p->B.nnz, 1) * p->arena_cb, p->s) &&
          p->bc_val.alloc(std::max<int64_t>(p->B.nnz, 1) * p->vb, p->s) &&
          build_bchunks(p->B.row_ptr, p->B.col_idx, p->B.vals, p->f32, p->B.n_rows, p->bcp.p, v0,
                        ilog2(p->P.widths[0]), p->arena_cb == 2, p->bct.p, p->bc_col.p, p->bc_val.p, p->s)) {
      } else {
        if (p->log) std::fprintf(stderr, "[gm_spgemm] no room for the chunk-major copy of B; row-order expansion\n");
        p->bct.release();
        p->bc_col.release();
        p->bc_val.release();
      }
      p->stage_end(t);
    }
    gm_status st = p->rowwise ? plan_and_alloc(p, p->arena_cb + p->vb, true, batches, 1)
                              : plan_and_alloc(p, 24, true, batches);
    if (st != GM_OK) return st;
    p->n_batches = std::max<int64_t>(p->n_batches, static_cast<int64_t>(batches.size()));
    int64_t par_base[GM_MAX_LEVELS + 1] = {};
    for (auto& bt : batches) {
      st = p->rowwise ? run_batch_rowwise(p, bt.first, bt.second, par_base, C_col, C_val)
                      : run_batch(p, bt.first, bt.second, true, par_base, C_col, C_val);
      if (st != GM_OK) return st;
    }
    free_arena(p);
    p->bct.release();
    p->bc_col.release();
    p->bc_val.release();
    p->bm_slot.release();  // the kept bitmaps serve one numeric pass
    p->bm_store.release();
    p->keep = keep;
  }
  join_light(p);
  return sync_check(p);
}

static void log_plan(const gm_plan* p) {
  std::fprintf(stderr,
               "[gm_spgemm] C %lld x %lld  tau=%lld D=%lld chunks_req=%lld chunks_max=%lld levels=%lld  "
               "rows: heavy=%lld light=%lld empty=%lld  IP total=%lld heavy=%lld\n",
               (long long)p->A.n_rows, (long long)p->c_m, (long long)p->P.tau, (long long)p->P.dense_width,
               (long long)p->P.n_chunks_required, (long long)p->P.n_chunks_max, (long long)p->P.n_levels,
               (long long)p->n_heavy, (long long)p->n_light, (long long)p->n_empty, (long long)p->ip_total,
               (long long)p->ip_heavy);
}

}  // namespace gm

extern "C" {

void gm_set_allocator(gm_alloc_fn alloc_fn, gm_free_fn free_fn, gm_avail_fn avail_fn, void* ctx) {
  gm::g_alloc = alloc_fn;
  gm::g_free = free_fn;
  gm::g_avail = avail_fn;
  gm::g_ctx = ctx;
}

gm_status gm_spgemm_params(int64_t c_m, const gm_config* cfg, gm_params* out) {
  return gm::compute_params(c_m, cfg, gm::kDefaultSmem, out);
}

}  // extern "C"

namespace gm {
// Argument checks and the plan object (no device work yet): parameters, device
// properties, pipeline choice.
static gm_status plan_setup(const gm_csr* A, const gm_csr* B, const gm_config* cfg, void* stream,
                            std::unique_ptr<gm_plan>& p) {
  const int32_t index_type = cfg ? cfg->index_type : 0;
  if (index_type & ~(GM_INDEX_ROWPTR32 | GM_INDEX_COL64)) return GM_ERR_INVALID_ARG;
  if (cfg && (cfg->pipeline < GM_PIPE_AUTO || cfg->pipeline > GM_PIPE_ROWWISE)) return GM_ERR_INVALID_ARG;
  gm_status st = check_csr(A, index_type);
  if (st == GM_OK) st = check_csr(B, index_type);
  if (st != GM_OK) return st;
  if (A->n_cols != B->n_rows) return GM_ERR_DIM_MISMATCH;
  p.reset(new (std::nothrow) gm_plan);
  if (!p) return GM_ERR_OOM;
  if (cfg) p->cfg = *cfg;
  p->index_type = index_type;
  p->s = static_cast<cudaStream_t>(stream);
  p->pipeline = p->cfg.pipeline == GM_PIPE_UNFUSED ? GM_PIPE_UNFUSED : GM_PIPE_FUSED_HISTO;  // may become ROWWISE
  p->f32 = p->cfg.value_type == GM_VALUE_F32;
  p->vb = p->f32 ? 4 : 8;
  p->timing = (p->cfg.flags & GM_FLAG_TIMING) != 0;
  p->keep = (p->cfg.flags & GM_FLAG_KEEP_INTERMEDIATES) != 0;
  p->log = (p->cfg.flags & GM_FLAG_LOG) != 0 || env_log();
  cudaError_t e = cudaGetDevice(&p->device);
  int smem = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GM_ERR_CUDA;
  }
  p->smem_dev = smem;
  p->c_m = std::max<int64_t>(B->n_cols, 1);
  st = compute_params(p->c_m, &p->cfg, p->smem_dev, &p->P);
  if (st != GM_OK) return st;
  p->L = static_cast<int>(p->P.n_levels);
  p->sym_rowbm = p->L <= 1 && p->pipeline != GM_PIPE_UNFUSED && !p->keep &&
                 rowbm_symbolic_smem(p->c_m) + 4096 <= p->smem_dev;
  p->rowwise = p->sym_rowbm && p->L == 1 && p->P.v_chunks[0] <= 256 &&
               expand_fits(static_cast<int>(p->P.v_chunks[0]), p->P.widths[0], p->P.tau, p->smem_dev) &&
               (p->cfg.pipeline == GM_PIPE_AUTO || p->cfg.pipeline == GM_PIPE_ROWWISE);
  if (p->rowwise) p->pipeline = GM_PIPE_ROWWISE;
  if (!p->status.alloc(1, p->s)) return GM_ERR_OOM;
  cudaMemsetAsync(p->status.p, 0, sizeof(int), p->s);
  p->overlap = (p->cfg.flags & GM_FLAG_OVERLAP) != 0;
  if (p->overlap) {
    if (!p->status2.alloc(1, p->s) || !p->work_counter2.alloc(1, p->s)) return GM_ERR_OOM;
    cudaMemsetAsync(p->status2.p, 0, sizeof(int), p->s);
    if (cudaStreamCreateWithFlags(&p->s2, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return GM_ERR_CUDA;
    }
  }
  return GM_OK;
}
}  // namespace gm

extern "C" {

gm_status gm_spgemm_analyze(const gm_csr* A, const gm_csr* B, const gm_config* cfg, void* stream,
                            gm_plan** plan_out) {
  if (!A) return GM_ERR_INVALID_ARG;
  return gm_spgemm_analyze_rows(A, B, 0, A->n_rows, cfg, stream, plan_out);
}

gm_status gm_spgemm_analyze_rows(const gm_csr* A, const gm_csr* B, int64_t row_begin, int64_t row_end,
                                 const gm_config* cfg, void* stream, gm_plan** plan_out) {
  const gm::NvtxCall nvtx_call("gm_spgemm_analyze_rows");
  if (!plan_out) return GM_ERR_INVALID_ARG;
  *plan_out = nullptr;
  std::unique_ptr<gm_plan> p;
  gm_status st = gm::plan_setup(A, B, cfg, stream, p);
  if (st != GM_OK) return st;
  if (row_begin < 0 || row_end < row_begin || row_end > A->n_rows) return GM_ERR_INVALID_ARG;
  gm::g_ws_peak = gm::g_ws_now.load();
  const int64_t l0 = gm::launch_count();
  st = gm::adapt_inputs(p.get(), A, B, row_begin, row_end);
  if (st == GM_OK) st = gm::analyze_impl(p.get());
  p->launches += gm::launch_count() - l0;
  p->collect_times();
  if (st != GM_OK) {
    cudaStreamSynchronize(p->s);
    cudaGetLastError();
    return st;
  }
  // two or more levels, B's rows sorted: level 0 by the row-order expansion
  p->rowexp0 = !p->rowwise && p->L >= 2 && p->b_sorted && p->P.v_chunks[0] <= 64 &&
               p->cfg.pipeline == GM_PIPE_AUTO && !p->keep;
  if (p->rowexp0) p->pipeline = GM_PIPE_ROWWISE;
  p->state = 1;
  if (p->log) gm::log_plan(p.get());
  *plan_out = p.release();
  return GM_OK;
}

gm_status gm_spgemm_row_split(const gm_csr* A, const gm_csr* B, const gm_config* cfg, int64_t n_parts,
                              void* stream, int64_t* bounds) {
  const gm::NvtxCall nvtx_call("gm_spgemm_row_split");
  if (!bounds || n_parts < 1 || n_parts > (int64_t(1) << 20)) return GM_ERR_INVALID_ARG;
  std::unique_ptr<gm_plan> p;
  gm_status st = gm::plan_setup(A, B, cfg, stream, p);
  if (st != GM_OK) return st;
  st = gm::adapt_inputs(p.get(), A, B, 0, A->n_rows);
  if (st == GM_OK) st = gm::row_split_impl(p.get(), n_parts, bounds);
  if (st != GM_OK) {
    cudaStreamSynchronize(p->s);
    cudaGetLastError();
  }
  return st;
}

gm_status gm_row_ptr_shift(void* row_ptr, int64_t n, int64_t base, int32_t index_type, void* stream) {
  if (n < 0 || (n > 0 && !row_ptr) || base < 0) return GM_ERR_INVALID_ARG;
  if (index_type & ~(GM_INDEX_ROWPTR32 | GM_INDEX_COL64)) return GM_ERR_INVALID_ARG;
  if (n == 0 || base == 0) return GM_OK;
  if (cudaPeekAtLastError() != cudaSuccess) return GM_ERR_CUDA;  // an earlier error stays with its owner
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (index_type & GM_INDEX_ROWPTR32) {
    int32_t last = 0;  // the largest entry of a valid row-pointer array
    const cudaError_t e = gm::read_to_host(&last, static_cast<int32_t*>(row_ptr) + (n - 1), sizeof(int32_t), s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GM_ERR_CUDA;
    }
    if (base + static_cast<int64_t>(last) >= (int64_t(1) << 31)) return GM_ERR_INDEX_OVERFLOW;
    (gm::k_add_base<int32_t><<<gm::grid_for(n, 256), 256, 0, s>>>(static_cast<int32_t*>(row_ptr), n, base),
     gm::note_launch());
  } else {
    (gm::k_add_base<int64_t><<<gm::grid_for(n, 256), 256, 0, s>>>(static_cast<int64_t*>(row_ptr), n, base),
     gm::note_launch());
  }
  return cudaGetLastError() == cudaSuccess ? GM_OK : GM_ERR_CUDA;
}

gm_status gm_spgemm_symbolic(gm_plan* plan, void* C_row_ptr, int64_t* C_nnz) {
  const gm::NvtxCall nvtx_call("gm_spgemm_symbolic");
  if (!plan) return GM_ERR_INVALID_ARG;
  if (plan->state != 1) return GM_ERR_STATE;
  if (!C_row_ptr) return GM_ERR_INVALID_ARG;
  const int64_t l0 = gm::launch_count();
  const bool rp32 = (plan->index_type & GM_INDEX_ROWPTR32) != 0;
  gm_status st = GM_OK;
  if (rp32 && !plan->c_rp64.alloc(plan->A.n_rows + 1, plan->s)) st = GM_ERR_OOM;
  if (st == GM_OK)
    st = gm::symbolic_impl(plan, rp32 ? plan->c_rp64.p : static_cast<int64_t*>(C_row_ptr), C_nnz);
  if (plan->s2) cudaStreamSynchronize(plan->s2);  // no light work outlives the call, error or not
  if (st == GM_OK && rp32) {  // C.rowPtr narrowed into the caller's int32 array
    if (plan->c_nnz >= (int64_t(1) << 31)) {
      st = GM_ERR_INDEX_OVERFLOW;
      plan->state = 4;  // C cannot be given in this index type: no further calls
    } else {
      gm::launch_narrow_i64(plan->c_rp64.p, static_cast<int32_t*>(C_row_ptr), plan->A.n_rows + 1,
                            int64_t(1) << 31, plan->s);
      st = gm::sync_check(plan);
    }
  }
  plan->launches += gm::launch_count() - l0;
  if (plan->timing) cudaStreamSynchronize(plan->s);
  plan->collect_times();
  plan->ws_peak = std::max<int64_t>(plan->ws_peak, gm::g_ws_peak.load());
  if (st == GM_OK) plan->state = 2;
  return st;
}

gm_status gm_spgemm_numeric(gm_plan* plan, void* C_col_idx, void* C_vals) {
  const gm::NvtxCall nvtx_call("gm_spgemm_numeric");
  if (!plan) return GM_ERR_INVALID_ARG;
  if (plan->state != 2) return GM_ERR_STATE;
  if (plan->c_nnz > 0 && (!C_col_idx || !C_vals)) return GM_ERR_INVALID_ARG;
  const int64_t l0 = gm::launch_count();
  gm_status st = GM_OK;
  if (plan->index_type & GM_INDEX_COL64) {  // int32 columns in a plan buffer, then widened
    gm::DevBuf<int32_t> col32;
    if (!col32.alloc(plan->c_nnz, plan->s)) {
      st = GM_ERR_OOM;
    } else {
      st = gm::numeric_impl(plan, col32.p, C_vals);
      if (st == GM_OK) {
        gm::launch_widen_i32(col32.p, static_cast<int64_t*>(C_col_idx), plan->c_nnz, plan->s);
        st = gm::sync_check(plan);
      }
    }
  } else {
    st = gm::numeric_impl(plan, static_cast<int32_t*>(C_col_idx), C_vals);
  }
  if (plan->s2) cudaStreamSynchronize(plan->s2);  // no light work outlives the call, error or not
  if (st == GM_OK) plan->c_rp64.release();
  plan->launches += gm::launch_count() - l0;
  if (plan->timing) cudaStreamSynchronize(plan->s);
  plan->collect_times();
  plan->ws_peak = std::max<int64_t>(plan->ws_peak, gm::g_ws_peak.load());
  if (st == GM_OK) plan->state = 3;
  return st;
}

gm_status gm_spgemm_plan_info(const gm_plan* plan, gm_plan_info* out) {
  if (!plan || !out) return GM_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->params = plan->P;
  out->n_rows = plan->A.n_rows;
  out->n_cols = plan->B.n_cols;
  out->n_heavy_rows = plan->n_heavy;
  out->n_light_rows = plan->n_light;
  out->n_empty_rows = plan->n_empty;
  out->ip_total = plan->ip_total;
  out->ip_heavy = plan->ip_heavy;
  out->c_nnz = plan->c_nnz;
  out->chat_bytes = plan->ip_heavy * (4 + plan->vb);  // int32 column + value a product
  out->n_batches = plan->n_batches;
  out->workspace_peak_bytes = plan->ws_peak;
  out->n_leaves = plan->n_leaves;
  out->keeps_reordered = 0;
  out->pipeline = plan->pipeline;
  out->cuda_error = plan->cuda_error;
  out->device_status = plan->dev_status;
  for (int i = 0; i < GM_NUM_STAGES; ++i) out->stage_ms[i] = plan->stage_ms[i];
  out->kernel_launches = plan->launches;
  out->value_type = plan->f32 ? GM_VALUE_F32 : GM_VALUE_F64;
  out->chunk_col_bytes = plan->arena_cb;
  out->index_type = plan->index_type;
  return GM_OK;
}

void gm_spgemm_plan_destroy(gm_plan* plan) {
  if (!plan) return;
  cudaStreamSynchronize(plan->s);
  cudaGetLastError();
  delete plan;
}

const char* gm_status_string(gm_status s) {
  switch (s) {
    case GM_OK: return "GM_OK";
    case GM_ERR_INVALID_ARG: return "GM_ERR_INVALID_ARG: invalid argument";
    case GM_ERR_DIM_MISMATCH: return "GM_ERR_DIM_MISMATCH: A.n_cols != B.n_rows";
    case GM_ERR_INDEX_OVERFLOW: return "GM_ERR_INDEX_OVERFLOW: size exceeds the index types";
    case GM_ERR_OOM: return "GM_ERR_OOM: device allocation failed";
    case GM_ERR_WORKSPACE: return "GM_ERR_WORKSPACE: a heavy row needs more than the workspace cap";
    case GM_ERR_CUDA: return "GM_ERR_CUDA: a CUDA call failed";
    case GM_ERR_DEVICE_TIMEOUT: return "GM_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    case GM_ERR_STATE: return "GM_ERR_STATE: call out of order";
    case GM_ERR_BAD_INDEX: return "GM_ERR_BAD_INDEX: column index or row pointer out of range";
    case GM_ERR_INTERNAL: return "GM_ERR_INTERNAL: a device-side consistency check of the library failed";
  }
  return "unknown gm_status";
}

gm_status gm_spgemm_debug_copy(const gm_plan* plan, int view, int level, void* dst, int64_t bytes,
                               int64_t* out_bytes) {
  if (!plan) return GM_ERR_INVALID_ARG;
  if (plan->state < 1) return GM_ERR_STATE;
  const void* src = nullptr;
  int64_t size = 0;
  const int64_t nh = plan->n_heavy;
  const gm::LevelDbg* L = nullptr;
  if (view >= GM_DBG_CHAT_COL) {
    if (!plan->dbg_ok) return GM_ERR_STATE;
    if (view >= GM_DBG_REORD_ROWPTR) {
      if (level < 0 || level >= static_cast<int>(plan->dbg_levels.size())) return GM_ERR_INVALID_ARG;
      L = plan->dbg_levels[level].get();
    }
  }
  switch (view) {
    case GM_DBG_IP_COUNTS: src = plan->u.p; size = plan->A.n_rows * 8; break;
    case GM_DBG_HEAVY_ROWS: src = plan->rows_by_bin.p + plan->bin_start[gm::kHeavyBin]; size = nh * 4; break;
    case GM_DBG_LIGHT_ROWS: src = plan->rows_by_bin.p; size = plan->bin_start[gm::kHeavyBin] * 4; break;
    case GM_DBG_CHAT_ROWPTR: src = plan->chat_rp.p; size = (nh + 1) * 8; break;
    case GM_DBG_CHAT_COL: src = plan->dbg_chat_col.p; size = plan->ip_heavy * 4; break;
    case GM_DBG_CHAT_VAL: src = plan->dbg_chat_val.p; size = plan->ip_heavy * plan->vb; break;
    case GM_DBG_REORD_ROWPTR: src = L->rp.p; size = (L->rows + 1) * 8; break;
    case GM_DBG_REORD_COL: src = L->col.p; size = L->nnz * 4; break;
    case GM_DBG_REORD_VAL: src = L->val.p; size = L->nnz * plan->vb; break;
    case GM_DBG_REORD_CHILD: src = L->child.p; size = L->rows * 8; break;
    default: return GM_ERR_INVALID_ARG;
  }
  if (out_bytes) *out_bytes = size;
  if (!dst) return GM_OK;
  if (bytes != size) return GM_ERR_INVALID_ARG;
  if (size == 0) return GM_OK;
  if (!src) return GM_ERR_STATE;
  cudaStreamSynchronize(plan->s);
  const cudaError_t e = cudaMemcpy(dst, src, static_cast<size_t>(size), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? GM_OK : GM_ERR_CUDA;
}

}  // extern "C"
