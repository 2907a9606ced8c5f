/*
 * gm_spgemm.h -- C ABI of the GB300 gMAGNUS SpGEMM, C = A * B over CSR.
 *
 * Method: gMAGNUS, "Fast SpGEMM on GPUs for Irregular Matrices via Hierarchical
 * Multisplit" (Wolfson-Pou, Helal, Petrini). Algorithm 3 there states the problem
 * as "Input: A, B. Output: C" with every array in device memory (Sec. III-A), a
 * symbolic phase that yields C.rowPtr and C.nnz and a numeric phase that fills
 * C.col and C.val (Sec. II-B, Algorithm 1). This interface follows that split:
 *
 *   gm_spgemm_analyze   -- Algorithm 3 lines 2-5: parameters (Sec. III-D), per-row
 *                          intermediate-product counts, heavy/light partition.
 *   gm_spgemm_symbolic  -- lines 7-25: outer product, hierarchical multisplit,
 *                          symbolic accumulation, prefix sum of C.rowPtr.
 *   gm_spgemm_numeric   -- lines 26-28: numeric accumulation, C.col / C.val.
 *
 * Conventions common to every call
 *   - Matrices are CSR: row_ptr[n_rows+1] (row_ptr[0] = 0, non-decreasing,
 *     row_ptr[n_rows] = nnz), col_idx[nnz] in [0, n_cols), vals[nnz]. Row
 *     pointers are int64 and columns int32 unless gm_config.index_type says
 *     otherwise; values are of the type gm_config.value_type selects (double,
 *     the default, or float). A, B and C share these types. Rows need not be
 *     sorted and may repeat a column; repeated entries add.
 *   - Pointers documented "device" must be device (or managed) memory of the
 *     current CUDA device; "host" pointers are ordinary host memory.
 *   - Every call but gm_spgemm_plan_destroy, gm_set_allocator and
 *     gm_status_string returns a gm_status; nothing is thrown across the ABI. A call
 *     made out of order returns GM_ERR_STATE and leaves the plan unchanged.
 *   - Work is issued on the stream given to gm_spgemm_analyze (a cudaStream_t;
 *     NULL is the legacy default stream). Calls block the host only where a
 *     count must be known on the host (documented per call).
 *   - Results: C rows sorted by column; an entry exists when some stored A[i,k]
 *     meets a stored B[k,j], also when its value is zero (structure is symbolic).
 *     Sums are formed in the value type, in an unspecified order.
 */
#ifndef GM_SPGEMM_H
#define GM_SPGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gm_status {
  GM_OK = 0,
  GM_ERR_INVALID_ARG = 1,     /* null pointer, negative size, malformed CSR      */
  GM_ERR_DIM_MISMATCH = 2,    /* A.n_cols != B.n_rows                            */
  GM_ERR_INDEX_OVERFLOW = 3,  /* a size that does not fit the index types        */
  GM_ERR_OOM = 4,             /* device allocation failed                        */
  GM_ERR_WORKSPACE = 5,       /* one heavy row needs more than the workspace cap */
  GM_ERR_CUDA = 6,            /* a CUDA call failed; see gm_plan_info.cuda_error */
  GM_ERR_DEVICE_TIMEOUT = 7,  /* a bounded device-side wait gave up              */
  GM_ERR_STATE = 8,           /* call out of order (analyze, symbolic, numeric)  */
  GM_ERR_BAD_INDEX = 9,       /* a column index out of range, found on device    */
  GM_ERR_INTERNAL = 10        /* a device-side consistency check of the library
                                 failed (a bug in this library, not in the input or
                                 the driver); gm_plan_info.device_status holds the bits */
} gm_status;

/* A CSR matrix. The library only reads these arrays; they stay owned by the
 * caller and must remain valid and unchanged until gm_spgemm_numeric returns. */
typedef struct gm_csr {
  int64_t n_rows;
  int64_t n_cols;
  int64_t nnz;
  const void* row_ptr;    /* device, n_rows + 1 int64 (int32 with GM_INDEX_ROWPTR32) */
  const void* col_idx;    /* device, nnz int32 (int64 with GM_INDEX_COL64)           */
  const void* vals;       /* device, nnz values of gm_config.value_type (double by default) */
} gm_csr;

/* Value types for gm_config.value_type. The planner takes the value size into
 * Eqs. (4)-(6) (gMAGNUS Sec. III-D: s_C.val), so float values get a larger tau
 * and dense width than double ones. */
#define GM_VALUE_F64 0 /* double */
#define GM_VALUE_F32 1 /* float  */

/* Index types for gm_config.index_type, flags that may be combined; 0 means int64
 * row pointers and int32 columns. They set the element type of every row-pointer
 * array (A, B and C.rowPtr) and of every column array (A, B and C.col) at this
 * interface. Inside, the path keeps int64 row pointers and int32 columns: int32
 * row pointers are widened and int64 columns narrowed into copies the plan owns
 * (12 bytes per row and 4 per stored entry of A and B, once when A and B share
 * an array), and C's arrays are written through plan-owned buffers that are then
 * converted into the caller's. The planner's s_C.col stays 4 bytes, the width of
 * the columns held in shared memory. */
#define GM_INDEX_ROWPTR32 1 /* row pointers int32: nnz of A, B and C at most 2^31 - 1 */
#define GM_INDEX_COL64 2    /* columns int64, each in [0, n_cols) (n_cols <= 2^31 as always);
                               numeric needs 4 more bytes of workspace per entry of C */

/* Flags for gm_config.flags. */
#define GM_FLAG_TIMING 1             /* record per-stage device times (gm_plan_info.stage_ms) */
#define GM_FLAG_KEEP_INTERMEDIATES 2 /* keep C-hat / C-hat_reord of a single batch for gm_spgemm_debug_copy */
#define GM_FLAG_LOG 4                /* print the plan to stderr (also env GM_SPGEMM_LOG=1) */
#define GM_FLAG_OVERLAP 8            /* light rows on a second stream, concurrently with the heavy rows
                                        (gMAGNUS Algorithm 3 runs its light and heavy queues at once);
                                        the plan creates the stream and joins it into the plan's stream
                                        before C.rowPtr is scanned and before numeric returns */

/* Heavy-path pipelines for gm_config.pipeline. */
#define GM_PIPE_AUTO 0        /* GM_PIPE_ROWWISE when it applies, else GM_PIPE_FUSED_HISTO */
#define GM_PIPE_UNFUSED 1     /* outer product -> C-hat -> histogram -> multisplit (Algorithm 3 as printed) */
#define GM_PIPE_FUSED_HISTO 2 /* outer product counts the level-0 chunk histogram while it writes C-hat */
#define GM_PIPE_ROWWISE 3     /* heavy rows expanded in row order straight into their level-0 chunks
                                 (C-hat is not written); with one level the chunk sizes come from the
                                 symbolic pass, with more (GM_PIPE_AUTO, B rows sorted, at most 64
                                 level-0 chunks) the chunks then go through the multisplit levels */

/* Tuning and test overrides; zero selects the automatic value for every field.
 * Overrides change how the work is split, never the result. A NULL config is
 * the same as all zeros. */
typedef struct gm_config {
  int64_t smem_budget_bytes;   /* s_LM; 0 = the device's opt-in shared memory per block        */
  int64_t tau;                 /* heavy-row threshold; 0 = Eq. (4)                             */
  int64_t dense_width;         /* last-level chunk width (power of two); 0 = derived           */
  int64_t n_chunks_max;        /* chunks per multisplit level (power of two >= 2); 0 = Eq. (6) */
  int64_t workspace_cap_bytes; /* cap on heavy-path workspace; 0 = free memory minus a reserve  */
  int32_t pipeline;            /* GM_PIPE_*; another value is GM_ERR_INVALID_ARG               */
  int32_t flags;               /* GM_FLAG_*                                                    */
  int32_t value_type;          /* GM_VALUE_*: element type of A.vals, B.vals and C's values    */
  int32_t index_type;          /* GM_INDEX_* flags: row-pointer and column types of A, B and C */
} gm_config;

#define GM_MAX_LEVELS 16

/* Parameters of gMAGNUS Sec. III-D (GetMagnusParams). */
typedef struct gm_params {
  int64_t s_lm;                /* local-memory budget in bytes                          */
  int64_t tau;                 /* Eq. (4): heavy when intermediate products exceed tau   */
  int64_t dense_width;         /* n_denseNumeric floored to a power of two               */
  int64_t n_chunks_required;   /* ceil(C.m / dense_width) rounded up to a power of two   */
  int64_t n_chunks_max;        /* Eq. (5)/(6), floored to a power of two                 */
  int64_t n_levels;            /* Eq. (7); 0 when n_chunks_required == 1                 */
  int64_t v_chunks[GM_MAX_LEVELS]; /* chunks per row at each level                       */
  int64_t widths[GM_MAX_LEVELS];   /* column width of a chunk after each level           */
} gm_params;

#define GM_NUM_STAGES 16
/* Stage indices of gm_plan_info.stage_ms (device time, filled with GM_FLAG_TIMING).
 * The heavy-row expansion and multisplit run once in the symbolic pass (columns
 * only) and once in the numeric pass (columns and values); they are timed apart.
 * Whatever the flags, the host calls of each stage form an NVTX range named
 * "gm:" and the stage's name (gm:analyze, gm:num_heavy, ...), and every
 * analyze, row split, symbolic and numeric call an NVTX range with the call's
 * name, for profilers that record NVTX. */
enum {
  GM_STAGE_ANALYZE = 0,        /* counts, validation, partition, heavy row pointers */
  GM_STAGE_TRANSPOSE = 1,      /* masked CSR -> CSC of the heavy rows (numeric pass) */
  GM_STAGE_OUTER = 2,          /* outer product (numeric pass)                      */
  GM_STAGE_HISTOGRAM = 3,      /* chunk histograms, partitions, scans (numeric)      */
  GM_STAGE_MULTISPLIT = 4,     /* multisplit levels (numeric pass)                  */
  GM_STAGE_SYM_HEAVY = 5,      /* symbolic accumulation of chunks                    */
  GM_STAGE_SYM_LIGHT = 6,      /* symbolic accumulation of light rows                */
  GM_STAGE_SCAN = 7,           /* prefix sum of C.rowPtr and chunk offsets           */
  GM_STAGE_NUM_HEAVY = 8,      /* numeric accumulation of chunks                     */
  GM_STAGE_NUM_LIGHT = 9,      /* numeric accumulation of light rows                 */
  GM_STAGE_OTHER = 10,         /* everything else                                    */
  GM_STAGE_TRANSPOSE_SYM = 11, /* the same four stages in the symbolic pass          */
  GM_STAGE_OUTER_SYM = 12,
  GM_STAGE_HISTOGRAM_SYM = 13,
  GM_STAGE_MULTISPLIT_SYM = 14
};

typedef struct gm_plan_info {
  gm_params params;
  int64_t n_rows;              /* C.n                                   */
  int64_t n_cols;              /* C.m                                   */
  int64_t n_heavy_rows;
  int64_t n_light_rows;        /* rows with 0 < u(i) <= tau             */
  int64_t n_empty_rows;        /* rows with u(i) == 0                   */
  int64_t ip_total;            /* sum of u(i): intermediate products    */
  int64_t ip_heavy;            /* C-hat.nnz                             */
  int64_t c_nnz;               /* -1 before symbolic                    */
  int64_t chat_bytes;          /* C-hat size in bytes: an int32 column and a value a
                                  product (12 bytes with double values, 8 with float) */
  int64_t n_batches;           /* heavy-row batches under the workspace cap */
  int64_t workspace_peak_bytes;
  int64_t n_leaves;            /* chunks accumulated                    */
  int32_t keeps_reordered;     /* 1 when symbolic kept C-hat_reord for numeric */
  int32_t pipeline;            /* GM_PIPE_* in effect                   */
  int32_t cuda_error;          /* last cudaError_t seen, 0 if none      */
  int32_t device_status;       /* device-side error bits, 0 if none     */
  float stage_ms[GM_NUM_STAGES];
  int64_t kernel_launches;     /* kernels this plan has launched so far */
  int32_t value_type;          /* GM_VALUE_* of the plan                */
  int32_t chunk_col_bytes;     /* bytes of a stored chunk column in the numeric pass
                                  (2: chunk-local uint16, 4: int32)      */
  int32_t index_type;          /* GM_INDEX_* flags of the plan          */
} gm_plan_info;

typedef struct gm_plan gm_plan; /* opaque; owns every workspace buffer */

/* Device memory hooks for the plan's workspace. alloc returns NULL on failure.
 * Both run on the host, in stream order on `stream`. avail (nullable) returns the
 * bytes further allocations can still obtain (for sizing heavy-row batches; a
 * caching allocator counts its cached free blocks), or a negative value when
 * unknown, in which case cudaMemGetInfo is used. NULL alloc/free hooks select
 * cudaMallocAsync / cudaFreeAsync. Set before gm_spgemm_analyze; the hooks are
 * process-wide. */
typedef void* (*gm_alloc_fn)(void* ctx, size_t bytes, void* stream);
typedef void (*gm_free_fn)(void* ctx, void* ptr, size_t bytes, void* stream);
typedef int64_t (*gm_avail_fn)(void* ctx);
void gm_set_allocator(gm_alloc_fn alloc_fn, gm_free_fn free_fn, gm_avail_fn avail_fn, void* ctx);

/* Host only. Fills *out with the parameters gMAGNUS Sec. III-D derives for a
 * product with c_m columns (Eqs. (4)-(7)) for int32 columns, int64 row pointers
 * (the widths held in shared memory, whatever cfg->index_type) and the value type of cfg (8-byte double by default, 4-byte float), honouring
 * the overrides in cfg (nullable). cfg->smem_budget_bytes == 0 means 232448
 * bytes (227 KB, the opt-in shared memory per block of sm_103a). Errors:
 * GM_ERR_INVALID_ARG for c_m < 1, a null out, an unknown value type, or
 * overrides that are not powers of two / too small. */
gm_status gm_spgemm_params(int64_t c_m, const gm_config* cfg, gm_params* out);

/* Algorithm 3 lines 2-5. Validates A and B (sizes on the host, indices on the
 * device), derives the parameters, counts the intermediate products of every row
 * (u(i) = sum over stored A[i,k] of nnz(B[k,:]), Sec. III-A InterOffsets), splits
 * rows into heavy (u > tau) and light ones and computes C-hat.rowPtr.
 * A and B: host pointers to descriptors of device arrays (copied; the arrays are
 * not). cfg: nullable. stream: a cudaStream_t used for all later work of the plan.
 * Blocks until the row counts are on the host. On success *plan_out owns all
 * workspace; release it with gm_spgemm_plan_destroy.
 * Errors: GM_ERR_INVALID_ARG, GM_ERR_DIM_MISMATCH, GM_ERR_INDEX_OVERFLOW,
 * GM_ERR_BAD_INDEX (a column out of range, also an int64 column that does not
 * fit 32 bits, or a malformed row_ptr), GM_ERR_OOM, GM_ERR_CUDA. GM_ERR_INVALID_ARG
 * also for an unknown value type or index flag. *plan_out is NULL on error. */
gm_status gm_spgemm_analyze(const gm_csr* A, const gm_csr* B, const gm_config* cfg, void* stream,
                            gm_plan** plan_out);

/* gm_spgemm_analyze for the rows [row_begin, row_end) of A only: the plan computes
 * those rows of C = A * B (C.rowPtr then has row_end - row_begin + 1 entries and
 * starts at 0; gm_row_ptr_shift places it inside a larger C). A's row pointers
 * are validated whole first; the range's row pointers are copied and rebased by
 * the plan, its columns and values read in place. B is used whole. This is the
 * per-GPU part of a product split by rows over several GPUs (gm_spgemm_row_split);
 * the gMAGNUS paper runs on one GPU and has no such split.
 * Errors: those of gm_spgemm_analyze, and GM_ERR_INVALID_ARG unless
 * 0 <= row_begin <= row_end <= A.n_rows. */
gm_status gm_spgemm_analyze_rows(const gm_csr* A, const gm_csr* B, int64_t row_begin, int64_t row_end,
                                 const gm_config* cfg, void* stream, gm_plan** plan_out);

/* Split of A's rows into n_parts consecutive ranges with about equal work, for
 * running one product on n_parts GPUs (one process a GPU, each holding A and B):
 * the work of a row is its intermediate products u(i) (gMAGNUS Sec. III-A, the
 * quantity the method's cost follows); with S(r) the products of rows [0, r) and
 * T = S(A.n_rows), bounds[q] (host, n_parts + 1 entries) is 0 for q = 0, A.n_rows
 * for q = n_parts, and otherwise the row r at which n_parts * S(r) comes nearest
 * to q * T (of the last r below q * T and the first r reaching it, the nearer one,
 * the lower on a tie), so part q, rows [bounds[q], bounds[q+1]), holds T / n_parts
 * products give or take one row's. Without any products the rows are split
 * evenly (bounds[q] = q * A.n_rows / n_parts, rounded down). The paper runs on
 * one GPU and has no such split. A and B are validated as in gm_spgemm_analyze.
 * Blocks until bounds is written. Workspace: 17 bytes a row of A, taken through
 * the allocator hooks and returned before the call returns.
 * Errors: those of gm_spgemm_analyze; GM_ERR_INVALID_ARG also for bounds NULL or
 * n_parts outside [1, 2^20]. */
gm_status gm_spgemm_row_split(const gm_csr* A, const gm_csr* B, const gm_config* cfg, int64_t n_parts,
                              void* stream, int64_t* bounds);

/* Adds base to the n entries of a row-pointer array (device; int64, or int32 with
 * GM_INDEX_ROWPTR32 in index_type): places the C.rowPtr of one row range (which
 * starts at 0) inside the C of the whole product, whose entries before the range
 * number base. Stream-ordered on stream; with int32 row pointers the call first
 * reads the array's last entry (blocking) and returns GM_ERR_INDEX_OVERFLOW when
 * base plus it does not fit int32, changing nothing. The paper has no counterpart
 * (it runs on one GPU).
 * Errors: GM_ERR_INVALID_ARG (n < 0, base < 0, NULL row_ptr with n > 0, unknown
 * index flags), GM_ERR_INDEX_OVERFLOW, GM_ERR_CUDA (a launch failed, or a CUDA
 * error from earlier work was still pending: left pending, nothing queued). */
gm_status gm_row_ptr_shift(void* row_ptr, int64_t n, int64_t base, int32_t index_type, void* stream);

/* Algorithm 3 lines 7-25. Writes C.rowPtr (device, A.n_rows + 1 row pointers of
 * the plan's index type, caller allocated) and *C_nnz (host). Heavy rows go
 * through the outer product and the hierarchical multisplit in batches that fit
 * the workspace cap; light rows are counted with a shared-memory accumulator.
 * Blocks until C.rowPtr is written and C.nnz is on the host.
 * Errors: GM_ERR_STATE (not right after analyze), GM_ERR_INVALID_ARG,
 * GM_ERR_WORKSPACE (a single heavy row does not fit the cap), GM_ERR_OOM,
 * GM_ERR_CUDA, GM_ERR_DEVICE_TIMEOUT, GM_ERR_INTERNAL, GM_ERR_INDEX_OVERFLOW (GM_INDEX_ROWPTR32
 * and C.nnz above 2^31 - 1: *C_nnz holds C.nnz, C_row_ptr is not written and
 * the plan takes no further symbolic or numeric call). */
gm_status gm_spgemm_symbolic(gm_plan* plan, void* C_row_ptr, int64_t* C_nnz);

/* Algorithm 3 lines 26-28. Fills C.col (device, C_nnz columns of the plan's
 * index type) and C.val (device, C_nnz values of the plan's value type), both
 * caller allocated after gm_spgemm_symbolic; each row sorted by column. Returns
 * once the work is issued and has completed (stream synchronised).
 * Errors: GM_ERR_STATE (symbolic not done, or numeric already done),
 * GM_ERR_INVALID_ARG, GM_ERR_WORKSPACE, GM_ERR_OOM, GM_ERR_CUDA, GM_ERR_INTERNAL. */
gm_status gm_spgemm_numeric(gm_plan* plan, void* C_col_idx, void* C_vals);

/* Copies the plan's parameters, sizes and statistics (gMAGNUS Tables V/VI:
 * C-hat size, heavy IP and row fractions, chunks per level) into *out (host). */
gm_status gm_spgemm_plan_info(const gm_plan* plan, gm_plan_info* out);

/* Releases every buffer the plan owns (stream-ordered on the plan's stream). NULL is a no-op. */
void gm_spgemm_plan_destroy(gm_plan* plan);

/* A static, human-readable name of a status code. */
const char* gm_status_string(gm_status s);

/* Debug view of a plan's device arrays, copied to host memory `dst` of `bytes`
 * bytes (which must equal the array size reported through *out_bytes when dst is
 * NULL). Available after analyze (GM_DBG_IP_COUNTS, GM_DBG_HEAVY_ROWS,
 * GM_DBG_LIGHT_ROWS, GM_DBG_CHAT_ROWPTR) and, with GM_FLAG_KEEP_INTERMEDIATES and a
 * single heavy batch, after symbolic (C-hat and the C-hat_reord of each level).
 * `level` selects the multisplit level for the GM_DBG_REORD_* views.
 * Errors: GM_ERR_INVALID_ARG (unknown view or size), GM_ERR_STATE (not available). */
enum {
  GM_DBG_IP_COUNTS = 0,    /* int64[n_rows]   u(i)                          */
  GM_DBG_HEAVY_ROWS = 1,   /* int32[n_heavy]  x_heavy, ascending            */
  GM_DBG_LIGHT_ROWS = 2,   /* int32[n_light + n_empty] x_light, ascending   */
  GM_DBG_CHAT_ROWPTR = 3,  /* int64[n_heavy+1] C-hat.rowPtr                 */
  GM_DBG_CHAT_COL = 4,     /* int32[ip_heavy] C-hat.col                     */
  GM_DBG_CHAT_VAL = 5,     /* value type[ip_heavy] C-hat.val                */
  GM_DBG_REORD_ROWPTR = 6, /* int64[rows+1]   C-hat_reord.rowPtr at `level` */
  GM_DBG_REORD_COL = 7,    /* int32[...]      chunk-local columns           */
  GM_DBG_REORD_VAL = 8,    /* value type[...]                               */
  GM_DBG_REORD_CHILD = 9   /* int64[rows]     id (parent * v + chunk) of each C-hat_reord row */
};
gm_status gm_spgemm_debug_copy(const gm_plan* plan, int view, int level, void* dst, int64_t bytes,
                               int64_t* out_bytes);

/* Exclusive prefix sum that allocates nothing: out[i] = in[0] + ... + in[i-1] for
 * i < n, and *total = the sum of all n inputs when total is not NULL. This has no
 * counterpart in the gMAGNUS paper; it is the scan that places C.rowPtr, offered
 * to callers that cannot allocate device memory while they run (work being
 * captured into a CUDA graph, host callbacks or real-time loops that must not
 * block on an allocator, hosts whose framework owns all device memory).
 * in, out: device int64[n] (may be the same array); total: device int64 or NULL;
 * stream: a cudaStream_t (NULL = legacy default stream). The work is queued on
 * the stream; the call does not wait for it.
 * Scratch: a fixed array inside the library, 65,600 int64 (about 525 KB) on every
 * device that loads the library, held until the process exits. Largest n:
 * 134,217,728 (2^27); larger n returns GM_ERR_WORKSPACE and queues nothing.
 * The first call on a device looks the array's device address up, and so does
 * the first call after the device's context was replaced (cudaDeviceReset): make
 * that call before any stream capture. Every call shares the array: calls whose
 * work overlaps on the GPU race, so serialise them. Nothing needs clearing
 * between calls.
 * Errors: GM_ERR_INVALID_ARG (n < 0, or NULL in/out with n > 0), GM_ERR_WORKSPACE
 * (n too large), GM_ERR_CUDA (the device lookup or a launch of this call failed,
 * or a CUDA error from earlier work was still pending: that one is left pending
 * for its owner and nothing is queued). */
gm_status gm_prefix_sum_noalloc(const int64_t* in, int64_t* out, int64_t n, int64_t* total, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GM_SPGEMM_H */
