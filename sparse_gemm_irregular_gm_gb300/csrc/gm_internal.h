// gm_internal.h -- declarations shared by the CUDA translation units of libgm_spgemm.
//
// Layout conventions (device memory):
//   * CSR inputs: row_ptr int64, col int32, val fp64.
//   * C-hat (intermediate matrix of the heavy rows, gMAGNUS Sec. III-A): CSR over
//     the rows of one heavy batch, int64 row pointers, int32 columns, fp64 values.
//   * C-hat_reord (one multisplit level, Sec. III-C): CSR over children
//     (parent * v + chunk) in "mapped" order (heavy children first), int32
//     chunk-local columns, fp64 values.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gm_spgemm.h"

namespace gm {

// ---- device status bits (written with atomicOr into a status word) ----------
enum : int {
  kStBadARowPtr = 1 << 0,
  kStBadBRowPtr = 1 << 1,
  kStBadACol = 1 << 2,
  kStBadBCol = 1 << 3,
  kStHashFull = 1 << 4,     // a probe sequence ran through the whole table
  kStGroupRows = 1 << 5,    // a multisplit work group met more rows than planned
  kStInternal = 1 << 6,     // an internal consistency check failed
  kStWaitTimeout = 1 << 7,  // a bounded wait inside a kernel gave up
  kStBounds = 1 << 8,       // GM_BOUNDS_CHECK builds: a cursor or slot outside its range
};

// GM_BOUNDS_CHECK builds check the index of every write of C and of the chunk
// elements before it is made: an index out of its range sets kStBounds in the
// status word and the write is skipped (never a trap). Other builds compile the
// checks away.
#ifdef GM_BOUNDS_CHECK
#define GM_CHECKED(cond, status) ((cond) || (atomicOr((status), ::gm::kStBounds), false))
#else
#define GM_CHECKED(cond, status) true
#endif

constexpr int kMaxBins = 16;

// Binning by size: bin 0 holds items of size 0; otherwise the first b >= 1 with
// size <= ub[b]. ub must be non-decreasing and ub[nbins-1] must cover every size.
struct BinSpec {
  int nbins;
  int64_t ub[kMaxBins];
};

// ---- kernel launch accounting ----------------------------------------------
// Every launch site calls note_launch(); plans report the count they caused.
void note_launch(int n = 1);
int64_t launch_count();

// ---- workspace ------------------------------------------------------------
// Stream-ordered device allocations routed through the caller's hooks (or
// cudaMallocAsync). Returns nullptr on failure.
void* ws_alloc(size_t bytes, cudaStream_t s);
void ws_free(void* p, size_t bytes, cudaStream_t s);

template <class T>
struct DevBuf {
  T* p = nullptr;
  size_t n = 0;
  cudaStream_t s = nullptr;
  bool alloc(size_t count, cudaStream_t stream) {
    release();
    s = stream;
    n = count;
    if (count == 0) return true;
    p = static_cast<T*>(ws_alloc(count * sizeof(T), stream));
    if (!p) n = 0;
    return p != nullptr;
  }
  void release() {
    if (p) ws_free(p, n * sizeof(T), s);
    p = nullptr;
    n = 0;
  }
  size_t bytes() const { return n * sizeof(T); }
  ~DevBuf() { release(); }
  DevBuf() = default;
  DevBuf(const DevBuf&) = delete;
  DevBuf& operator=(const DevBuf&) = delete;
};

// ---- scans (gm_scan.cu) -----------------------------------------------------
// out[i] = sum_{j<i} in[j] for i in [0, n); in == out allowed. When d_total is
// not null it receives sum of all n inputs. Returns false on allocation failure.
bool scan_exclusive_i64(const int64_t* in, int64_t* out, int64_t n, int64_t* d_total, cudaStream_t s);
// The same scan with caller-provided scratch (scratch_elems int64 entries; needs
// scan_scratch_elems(n)). Returns false when the scratch is too small.
int64_t scan_scratch_elems(int64_t n);
bool scan_exclusive_i64_scratch(const int64_t* in, int64_t* out, int64_t n, int64_t* d_total, int64_t* scratch,
                                int64_t scratch_elems, cudaStream_t s);
// Fixed-size segments: for each parent p, the v children p*v .. p*v+v-1 get
// off[p*v+c] = base[p] + sum_{c'<c} val[p*v+c'] (in place: val may equal off).
// Returns the per-parent sums in sums (nullable).
void segmented_offsets(const int64_t* val, int64_t* off, const int64_t* base, int64_t n_parents, int v,
                       int64_t* sums, cudaStream_t s);
// Sum of v consecutive children into their parent slot: dst[idx[p]] = sum_c src[p*v+c].
void sum_children(const int64_t* src, const int64_t* parent_slot, int64_t* dst, int64_t n_parents, int v,
                  cudaStream_t s);

// ---- analysis (gm_analyze.cu) ---------------------------------------------
// Index-type conversions at the interface: out[i] = in[i] (int32 -> int64), and
// int64 -> int32 with values outside [0, bound) written as -1.
void launch_widen_i32(const int32_t* in, int64_t* out, int64_t n, cudaStream_t s);
void launch_narrow_i64(const int64_t* in, int32_t* out, int64_t n, int64_t bound, cudaStream_t s);
void launch_validate_rowptr(const int64_t* rp, int64_t n_rows, int64_t nnz, int bad_bit, int* status,
                            cudaStream_t s);
void launch_validate_cols(const int32_t* col, int64_t nnz, int64_t n_cols, int bad_bit, int* status,
                          cudaStream_t s);
// *unsorted |= 1 when a row's columns are not non-decreasing (rows validated first).
// *flags |= 1 when some row of B has a column greater than the next one, |= 2
// when some row repeats a column.
void launch_check_sorted(const int64_t* rp, const int32_t* col, int64_t n_rows, int* flags, cudaStream_t s);
// u[i] = sum over stored A[i,k] of nnz(B[k,:]); bin[i] from spec.
void launch_ip_count(const int64_t* a_rp, const int32_t* a_col, int64_t n_rows, const int64_t* b_rp,
                     int64_t* u, uint8_t* bin, BinSpec spec, cudaStream_t s);
// bin[i] for sizes given in an int64 array (optionally gathered: size[idx[i]]).
void launch_bin_sizes(const int64_t* size, int64_t n, uint8_t* bin, BinSpec spec, cudaStream_t s);
// Stable partition of [0, n) by bin: out_idx holds the indices bin-major, ascending
// within a bin; d_bin_start[b] (nbins+1 entries) the start of each bin.
bool partition_by_bin(const uint8_t* bin, int64_t n, int nbins, int32_t* out_idx, int64_t* d_bin_start,
                      cudaStream_t s);
// dst[i] = src[idx[i]] for i in [0, n).
void launch_gather_i64(const int64_t* src, const int32_t* idx, int64_t n, int64_t* dst, cudaStream_t s);
void launch_gather_i64_i64(const int64_t* src, const int64_t* idx, int64_t n, int64_t* dst, cudaStream_t s);
// dst[idx[i]] = src[i].
void launch_scatter_i64(const int64_t* src, const int32_t* idx, int64_t n, int64_t* dst, cudaStream_t s);
void launch_iota_i64(int64_t* dst, int64_t n, int64_t start, cudaStream_t s);
void launch_fill_i64(int64_t* dst, int64_t n, int64_t value, cudaStream_t s);

// ---- expansion (gm_expand.cu) -----------------------------------------------
struct TransposeArgs {
  const int32_t* heavy_rows;  // original row id of each batch row
  int64_t n_batch;
  const int64_t* a_rp;
  const int32_t* a_col;
  const void* a_val;          // float or double (f32)
  int64_t n_cols;             // A.n_cols
  bool f32;
};
// Masked CSR -> CSC of A[heavy_rows, :] (counting sort by column):
// col_ptr[n_cols+1], t_row[nnz_batch] (batch-local row), t_val[nnz_batch].
bool masked_transpose(const TransposeArgs& a, int64_t nnz_batch, int64_t* col_ptr, int32_t* t_row,
                      void* t_val, cudaStream_t s);
// slice_off[k] = sum_{k'<k} (col_ptr[k'+1]-col_ptr[k']) * nnz(B[k',:]), k in [0, n_cols].
bool slice_offsets(const int64_t* col_ptr, const int64_t* b_rp, int64_t n_cols, int64_t* slice_off,
                   cudaStream_t s);
// wg_first[g] = the slice holding flattened position g*E (g in [0, ceil(total/E))).
void launch_wg_slice(const int64_t* slice_off, int64_t n_slices, int64_t total, int64_t E, int32_t* wg_first,
                     cudaStream_t s);

struct OuterArgs {
  const int64_t* slice_off;   // n_cols + 1
  const int64_t* col_ptr;     // n_cols + 1 (A-tilde CSC)
  const int32_t* t_row;       // A-tilde rows (batch-local C-hat rows)
  const void* t_val;          // values are float or double (f32)
  const int64_t* b_rp;
  const int32_t* b_col;
  const void* b_val;
  int64_t n_slices;
  int64_t total;              // C-hat.nnz of the batch
  int64_t E;                  // flattened elements per work group
  const int32_t* wg_first;
  unsigned long long* cursor; // write cursor per C-hat row (starts at C-hat.rowPtr)
  int32_t* out_col;
  void* out_val;              // null: columns only
  bool f32;
  // fused level-0 histogram (null when not fused)
  unsigned long long* histo;  // [rows * v]
  int v;
  int shift;                  // chunk = col >> shift
};
void launch_outer_product(const OuterArgs& a, cudaStream_t s);

// ---- multisplit (gm_multisplit.cu) ------------------------------------------
// wg_first[g] = the row holding position g*E.
void launch_wg_row(const int64_t* rp, int64_t n_rows, int64_t E, int32_t* wg_first, cudaStream_t s);

struct SplitArgs {
  const int64_t* in_rp;       // parent row pointers (batch-local, in_rp[0] may be > 0)
  int64_t n_parents;
  const int32_t* in_col;      // parent-local columns
  const void* in_val;         // null: columns only; float or double (f32)
  bool f32;
  int64_t base;               // in_rp[0]
  int64_t total;              // in_rp[n_parents] - in_rp[0]
  int v;                      // chunks per parent
  int shift;                  // chunk = col >> shift
  int64_t E;
  int n_group_rows;           // rows a work group may meet
  const int32_t* wg_first;
  int* status;
  // histogram output
  unsigned long long* counts; // [n_parents * v]
  // multisplit output
  const int64_t* inv;         // child -> mapped row (null: identity)
  unsigned long long* cursor; // write cursor per mapped row (starts at its row pointer)
  int32_t* out_col;
  void* out_val;
};
void launch_histogram(const SplitArgs& a, cudaStream_t s);
void launch_multisplit(const SplitArgs& a, cudaStream_t s);
// Largest work-group size E whose shared arrays fit smem_max bytes (0: none);
// *ngr_out gets the rows a work group may meet when input rows exceed tau elements.
int64_t multisplit_pick_E(int v, int64_t tau, bool with_val, int64_t smem_max, int* ngr_out);

// Row-order expansion fused with the first multisplit level (gm_multisplit.cu):
// the products of a batch of heavy rows are generated in row order (A entry by
// A entry, B row by B row) straight into their level-0 chunks; C-hat is never
// written. Entries of the batch are concatenated in row order.
struct ExpandArgs {
  const int64_t* e_b;         // B.rowPtr of the B row each entry selects (B.rowPtr[A.col])
  const void* e_a;            // A value of each entry (null: columns only); float or double (f32)
  bool f32;
  const int64_t* e_off;       // flattened start of each entry's products, n_e + 1
  const int32_t* e_row;       // batch-local row of each entry
  int64_t n_e;
  const int64_t* b_rp;
  const int32_t* b_col;
  const void* b_val;
  const int64_t* in_rp;       // batch row starts in the flattened space, n_parents + 1
  int64_t n_parents;
  const int64_t* bounds;      // work group g covers [bounds[g], bounds[g+1])
  const int4* wg_info;        // per work group: first entry, number of entries, its first batch row
  int64_t n_wg;
  int v;
  int shift;
  int n_group_rows;
  int* status;
  unsigned long long* cursor; // per chunk (row * v + c): write cursor from its row pointer
  int32_t* out_col;
  void* out_val;              // null: columns only
};
constexpr int kExpandE = 4096;    // elements per work group (at most)
constexpr int kExpandCap = 1024;  // entries starting inside a work group (at most)
// Builds the batch entry arrays (e_len into e_off, then the caller scans it).
void launch_gather_entries(const int32_t* heavy_rows, int64_t nb, const int64_t* anz_batch, const int64_t* a_rp,
                           const int32_t* a_col, const void* a_val, bool f32, const int64_t* b_rp, int64_t* e_b,
                           void* e_a, int32_t* e_row, int64_t* e_len, cudaStream_t s, int32_t* e_k = nullptr);

// Row-order expansion into level-0 chunks with one reservation per (unit, row,
// chunk) and contiguous writes per warp (B rows sorted; per-B-row chunk starts
// in bcp; v <= 64). Units are U consecutive products of the batch in row order.
struct RowRunArgs {
  const int32_t* e_k;         // B row of each entry
  const int64_t* e_b;         // B.rowPtr of that row
  const void* e_a;            // A value (null: columns only); float or double (f32)
  bool f32;
  const int64_t* e_off;       // flattened start of each entry's products, n_e + 1
  const int32_t* e_row;       // batch-local row of each entry
  int64_t n_e;
  int64_t total;              // products of the batch
  int64_t U;                  // products per unit (row_runs_unit)
  int64_t n_units;
  int64_t* unit_first;        // n_units scratch: first entry of each unit
  const int32_t* b_col;
  const void* b_val;
  const int32_t* bcp;
  int v;
  int shift;
  unsigned long long* cursor; // per chunk (row * v + c): write cursor
  void* out_col;              // chunk-local columns: int32, or uint16 with col16
  void* out_val;
  bool col16;
  unsigned* unit_counter;
  int* status;
  const int64_t* chunk_rp;    // GM_BOUNDS_CHECK: chunk c's elements lie in [chunk_rp[c], chunk_rp[c+1]) (null: unchecked)
};
// Chunk-major expansion (rows of B sorted, one level of at most 64 chunks).
struct ChunkMajorArgs {
  int64_t nb;                 // heavy rows of the batch
  int v;                      // level-0 chunks a row
  const int64_t* anz;         // prefix of the batch rows' A entries (nb + 1, absolute)
  const int32_t* e_k;         // B row of each gathered A entry (batch-relative, row order)
  const void* e_a;            // A value of each entry (null: columns only); float or double (f32)
  bool f32;
  const int64_t* bct;         // chunk-major starts (bchunk_starts_len entries)
  int64_t nB1;                // B.n_rows + 1
  const void* bc_col;         // chunk-major copy of B: chunk-local columns (uint16 with col16, else int32)
  const void* bc_val;         // and values
  const int64_t* rrp;         // region of (row, chunk) pair i = h * v + c: [rrp[i], rrp[i + 1])
  void* out_col;
  void* out_val;
  bool col16;
  unsigned long long* counter;
  int* status;
};
int64_t bchunk_starts_len(int64_t b_rows, int v);
// bct (bchunk_starts_len entries), bc_col and bc_val (B.nnz entries each) from the
// per-B-row chunk starts bcp; B's rows must be sorted by column.
bool build_bchunks(const int64_t* b_rp, const int32_t* b_col, const void* b_val, bool f32, int64_t b_rows,
                   const int32_t* bcp, int v, int shift, bool col16, int64_t* bct, void* bc_col, void* bc_val,
                   cudaStream_t s);
void launch_expand_cm(const ChunkMajorArgs& a, int num_sms, cudaStream_t s);
int64_t row_runs_unit(int64_t tau);
void launch_row_runs(const RowRunArgs& a, int num_sms, cudaStream_t s);
// Work-group bounds: multiples of kExpandE merged with the starts of every
// kExpandCap-th entry; bounds has n_wg + 1 entries, wg_info n_wg.
int64_t expand_num_wg(int64_t total, int64_t n_e);
void launch_expand_bounds(const int64_t* e_off, const int32_t* e_row, int64_t n_e, int64_t total, int64_t* bounds,
                          int4* wg_info, cudaStream_t s);
void launch_expand_split(const ExpandArgs& a, cudaStream_t s);
int expand_group_rows(int64_t tau);
// Whether k_expand_split can take v chunks per row of width w at this tau within
// smem bytes of shared memory (packed keys need n_group_rows * v < 65535, w <= 65536).
bool expand_fits(int v, int64_t w, int64_t tau, size_t smem);

// ---- accumulation (gm_accum.cu) ---------------------------------------------
struct LightArgs {
  const int32_t* rows;        // rows of this bin
  int64_t n_items;
  const int64_t* a_rp;
  const int32_t* a_col;
  const void* a_val;          // values are float or double (f32)
  const int64_t* b_rp;
  const int32_t* b_col;
  const void* b_val;
  int64_t* c_rp;              // symbolic: counts out at c_rp[row]; numeric: row offsets in
  int32_t* c_col;
  void* c_val;
  int* status;
  bool f32;
  int64_t c_nnz;              // GM_BOUNDS_CHECK: entries of C (numeric)
};
// Light rows of one bin: cap = table slots (>= 2 * max u in bin).
void launch_light_rows(const LightArgs& a, int bin_cap, bool symbolic, cudaStream_t s);

struct ListArgs {
  const int64_t* items;       // mapped C-hat_reord rows to accumulate
  int64_t n_items;
  const int64_t* rp;          // C-hat_reord row pointers (mapped order)
  const void* col;            // chunk-local columns: int32, or uint16 with col16
  const void* val;            // float or double (f32)
  bool col16;                 // columns stored in 16 bits (chunks at most 65536 wide)
  const int64_t* child_of;    // mapped row -> batch-local child id (null: identity)
  int64_t child_base;         // global child id of batch-local child 0
  int v;                      // chunks per parent (child = parent * v + chunk)
  int64_t width;              // chunk width
  const int64_t* parent_colbase; // batch-local parent -> global column base (null: 0)
  int64_t* nnz_out;           // symbolic: [global child] nnz
  const int64_t* off_in;      // numeric: [global child] output offset
  int32_t* c_col;
  void* c_val;
  int* status;
  bool f32;
  unsigned int* counter;      // dynamic chunk scheduling (launch_leaf_stream)
  int64_t c_nnz;              // GM_BOUNDS_CHECK: entries of C (numeric)
  const int64_t* expect_nnz;  // GM_BOUNDS_CHECK: the symbolic pass's nnz of each chunk (null: unchecked)
  // block accumulator: [global child] slot of the chunk's column bitmap kept by the
  // symbolic pass (-1: none), and the kept bitmaps (leaf_blkbm_words(width) words a slot)
  const int32_t* bm_slot;
  const uint32_t* bm_store;
};
// Chunks narrower than the dense width: shared-memory bitmap + rank accumulator.
void launch_leaf_bitmap(const ListArgs& a, int cap_vals, bool symbolic, cudaStream_t s);
// Light chunks of a wide level: shared-memory hash accumulator (cap slots).
void launch_leaf_hash(const ListArgs& a, int cap, bool symbolic, cudaStream_t s);
int leaf_bitmap_smem(int64_t width, int cap_vals, bool symbolic, int vb = 8);  // vb: bytes a value
// Chunks with at most max_elems (<= 4096) elements, held in registers; no
// floating-point atomics.
void launch_leaf_small(const ListArgs& a, int max_elems, bool symbolic, cudaStream_t s);
// Numeric chunks of at most 128 elements: one warp sorts and merges each.
void launch_leaf_warp(const ListArgs& a, cudaStream_t s);
// Numeric chunks of at most max_elems (<= 4096) elements: one warp per chunk with
// its own bitmap, rank prefix and value array in shared memory.
void launch_leaf_warpbm(const ListArgs& a, int max_elems, cudaStream_t s);
bool leaf_warpbm_fits(int64_t width, int max_elems, int64_t smem_max, int vb = 8);
// The same with 4 warps per chunk: chunks of at most max_elems elements (INT_MAX:
// any) and max_nnz output columns (the value array of the block).
void launch_leaf_blkbm(const ListArgs& a, int max_nnz, int max_elems, cudaStream_t s);
bool leaf_blkbm_fits(int64_t width, int max_nnz, int64_t smem_max, int vb = 8);
int64_t leaf_blkbm_words(int64_t width);
// Numeric chunks of any size, streamed: one producer warp copies each chunk's
// tiles into a shared-memory ring with bulk asynchronous copies, the consumer
// warps add them into a dense accumulator of the chunk's width. One block per
// SM; a.counter is reset by the launch. Needs a.width <= 65536 and the chunk
// element arrays readable 16 bytes past their last element.
bool leaf_stream_fits(int64_t width, bool col16, int64_t smem_max, int vb = 8);
void launch_leaf_stream(const ListArgs& a, int num_sms, cudaStream_t s);
int leaf_small_smem(int64_t width, int cap, bool symbolic, int vb = 8);

// ---- whole-row bitmaps (gm_rowbitmap.cu) -----------------------------------------
struct RowBitmapArgs {
  const int32_t* rows;        // rows of A to process (original ids)
  int64_t n_items;
  const int64_t* a_rp;
  const int32_t* a_col;
  const void* a_val;          // values are float or double (f32)
  const int64_t* b_rp;
  const int32_t* b_col;
  const void* b_val;
  int64_t c_m;                // columns of C
  int v;                      // symbolic: chunks per row (1 with width >= C.m: whole row)
  int64_t width;              // symbolic: chunk width
  int64_t* nnz_out;           // symbolic: [(item_base + item) * v + c]; whole row: null writes c_rp[row]
  int64_t item_base;
  int64_t* c_rp;              // whole-row symbolic: counts out; numeric: row offsets in
  int32_t* c_col;
  void* c_val;
  unsigned int* work_counter; // device counter for dynamic row scheduling
  int* status;
  bool f32;
  int64_t c_nnz;              // GM_BOUNDS_CHECK: entries of C (numeric)
  // symbolic, chunks: [global child] slot where the chunk's bitmap words are kept
  // for the numeric pass (-1: not kept), store_words words a slot
  const int32_t* bm_slot;
  uint32_t* bm_store;
  int store_words;
};
int64_t rowbm_symbolic_smem(int64_t c_m);
// Words of a whole-row bitmap of C.m columns (whole 16-byte pieces).
inline int64_t rowbm_words(int64_t c_m) { return ((c_m + 127) / 128) * 4; }
// Heavy rows: chunk nnz (v chunks of a.width) or whole-row nnz from a whole-row bitmap.
void launch_rowbm(const RowBitmapArgs& a, int num_sms, int64_t smem_max, cudaStream_t s);
// Light rows of at most cap products (symbolic: whole-row nnz into c_rp; numeric: the row of C).
// Numeric: columns in windows of a bitmap that fits beside the placed values and
// counters; int32 count-and-place by rank, no floating-point atomics.
int64_t rowbm_light_smem(int64_t c_m, int cap, bool symbolic, int64_t smem_max);
bool rowbm_light_fits(int64_t c_m, int cap, bool symbolic, int64_t smem_max, int vb = 8);
void launch_rowbm_light(const RowBitmapArgs& a, bool symbolic, int cap, int num_sms, int64_t smem_max, cudaStream_t s);

// bcp only (see heavy_chunk_counts), v <= 256.
void build_chunk_starts(const int64_t* b_rp, const int32_t* b_col, int64_t b_rows, int v, int shift, int32_t* bcp,
                        cudaStream_t s);
// cnt[h * v + c] = products of heavy row h whose column falls in level-0 chunk c
// (col >> shift == c), from per-B-row chunk counts, which are left in bcp
// (b_rows * (v + 1) entries: bcp[k * (v + 1) + c] = entries of B row k in chunks
// below c; for a row sorted by column, chunk c is its index range [bcp[c], bcp[c+1])).
// anz: prefix of the heavy rows' A-row lengths (n_heavy + 1). cnt null: bcp only;
// b_rp null: bcp is already built. False when v > 256.
bool heavy_chunk_counts(const int32_t* heavy_rows, int64_t n_heavy, const int64_t* anz, const int64_t* a_rp,
                        const int32_t* a_col, const int64_t* b_rp, const int32_t* b_col, int64_t b_rows, int v,
                        int shift, int32_t* bcp, int64_t* cnt, cudaStream_t s);

// Light-row bins: upper bounds on u and table capacity per bin.
constexpr int kLightWarpBins = 4;   // bins 1..4 use a warp per row
int64_t light_bin_ub(int b);        // b in [1, 10]
// Table slots for bin b; the top bin holds 2 * tau slots, fewer when they would
// not leave 1 KB of the block's shared memory (smem_max bytes) for static arrays.
int light_bin_cap(int b, int64_t tau, int64_t smem_max, int vb = 8);

}  // namespace gm
