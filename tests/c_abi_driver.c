/* c_abi_driver.c -- C = A * B through the C ABI from a plain C program.
 *
 * Test infrastructure: reads A and B from binary CSR files, copies them to the
 * device with the CUDA runtime, calls gm_spgemm_analyze, gm_spgemm_symbolic and
 * gm_spgemm_numeric with a NULL config (the planner's defaults) on the legacy
 * default stream, and writes C to a binary CSR file.
 *
 * File layout (little endian): int64 n_rows, n_cols, nnz; int64 row_ptr[n_rows + 1];
 * int32 col[nnz]; double val[nnz].
 *
 * Usage: c_abi_driver A.bin B.bin C.bin [parts]. With parts > 1 the product is
 * computed the way one rank of a multi-GPU run computes its share, here one part
 * after another: gm_spgemm_row_split cuts A's rows into parts of about equal
 * products, each part runs gm_spgemm_analyze_rows, symbolic and numeric, and
 * gm_row_ptr_shift places its row pointers behind the entries of the parts
 * before it; the parts are put together on the host.
 * Exit status 0 on success, 2 when a library call fails (its gm_status_string is
 * printed), 1 on any other error.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "gm_spgemm.h"

typedef struct {
  int64_t n_rows, n_cols, nnz;
  int64_t* row_ptr;
  int32_t* col;
  double* val;
} host_csr;

static void* xmalloc(size_t bytes) {
  void* p = malloc(bytes ? bytes : 1);
  if (!p) {
    fprintf(stderr, "out of host memory\n");
    exit(1);
  }
  return p;
}

static int read_csr(const char* path, host_csr* m) {
  FILE* f = fopen(path, "rb");
  if (!f) return 0;
  int64_t h[3];
  int ok = fread(h, sizeof(int64_t), 3, f) == 3 && h[0] >= 0 && h[1] >= 0 && h[2] >= 0;
  if (ok) {
    m->n_rows = h[0];
    m->n_cols = h[1];
    m->nnz = h[2];
    m->row_ptr = xmalloc((size_t)(m->n_rows + 1) * sizeof(int64_t));
    m->col = xmalloc((size_t)m->nnz * sizeof(int32_t));
    m->val = xmalloc((size_t)m->nnz * sizeof(double));
    ok = fread(m->row_ptr, sizeof(int64_t), (size_t)(m->n_rows + 1), f) == (size_t)(m->n_rows + 1) &&
         fread(m->col, sizeof(int32_t), (size_t)m->nnz, f) == (size_t)m->nnz &&
         fread(m->val, sizeof(double), (size_t)m->nnz, f) == (size_t)m->nnz;
  }
  fclose(f);
  return ok;
}

static int write_csr(const char* path, const host_csr* m) {
  FILE* f = fopen(path, "wb");
  if (!f) return 0;
  const int64_t h[3] = {m->n_rows, m->n_cols, m->nnz};
  int ok = fwrite(h, sizeof(int64_t), 3, f) == 3 &&
           fwrite(m->row_ptr, sizeof(int64_t), (size_t)(m->n_rows + 1), f) == (size_t)(m->n_rows + 1) &&
           fwrite(m->col, sizeof(int32_t), (size_t)m->nnz, f) == (size_t)m->nnz &&
           fwrite(m->val, sizeof(double), (size_t)m->nnz, f) == (size_t)m->nnz;
  return fclose(f) == 0 && ok;
}

/* Device copies of a host CSR; the descriptor points at them. */
static int to_device(const host_csr* m, gm_csr* d) {
  void *rp = NULL, *col = NULL, *val = NULL;
  const size_t rp_b = (size_t)(m->n_rows + 1) * sizeof(int64_t);
  const size_t col_b = (size_t)m->nnz * sizeof(int32_t), val_b = (size_t)m->nnz * sizeof(double);
  if (cudaMalloc(&rp, rp_b) != cudaSuccess || cudaMemcpy(rp, m->row_ptr, rp_b, cudaMemcpyHostToDevice) != cudaSuccess)
    return 0;
  if (m->nnz > 0) {
    if (cudaMalloc(&col, col_b) != cudaSuccess || cudaMalloc(&val, val_b) != cudaSuccess) return 0;
    if (cudaMemcpy(col, m->col, col_b, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(val, m->val, val_b, cudaMemcpyHostToDevice) != cudaSuccess)
      return 0;
  }
  d->n_rows = m->n_rows;
  d->n_cols = m->n_cols;
  d->nnz = m->nnz;
  d->row_ptr = rp;
  d->col_idx = col;
  d->vals = val;
  return 1;
}

static int fail(const char* call, gm_status st) {
  fprintf(stderr, "%s: %s\n", call, gm_status_string(st));
  return 2;
}

/* Rows [r0, r1) of C = A * B through the ABI, their row pointers shifted by
 * base; the part's arrays are copied into C (row pointers r0 .. r1, entries from
 * base on). Returns 0, or the driver's exit status. */
static int run_part(const gm_csr* dA, const gm_csr* dB, int64_t r0, int64_t r1, int64_t base, host_csr* C,
                    int64_t* nnz_out, gm_plan_info* info) {
  gm_plan* plan = NULL;
  gm_status st = gm_spgemm_analyze_rows(dA, dB, r0, r1, NULL, NULL, &plan);
  if (st != GM_OK) return fail("gm_spgemm_analyze_rows", st);
  const int64_t rows = r1 - r0;
  void* c_rp = NULL;
  if (cudaMalloc(&c_rp, (size_t)(rows + 1) * sizeof(int64_t)) != cudaSuccess) return 1;
  int64_t nnz = -1;
  st = gm_spgemm_symbolic(plan, c_rp, &nnz);
  if (st != GM_OK) return fail("gm_spgemm_symbolic", st);
  void *c_col = NULL, *c_val = NULL;
  if (nnz > 0 && (cudaMalloc(&c_col, (size_t)nnz * sizeof(int32_t)) != cudaSuccess ||
                  cudaMalloc(&c_val, (size_t)nnz * sizeof(double)) != cudaSuccess))
    return 1;
  st = gm_spgemm_numeric(plan, c_col, c_val);
  if (st != GM_OK) return fail("gm_spgemm_numeric", st);
  st = gm_spgemm_plan_info(plan, info);
  if (st != GM_OK) return fail("gm_spgemm_plan_info", st);
  gm_spgemm_plan_destroy(plan);
  st = gm_row_ptr_shift(c_rp, rows + 1, base, 0, NULL);
  if (st != GM_OK) return fail("gm_row_ptr_shift", st);
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  C->col = realloc(C->col, (size_t)(base + nnz + 1) * sizeof(int32_t));
  C->val = realloc(C->val, (size_t)(base + nnz + 1) * sizeof(double));
  if (!C->col || !C->val) return 1;
  if (cudaMemcpy(C->row_ptr + r0, c_rp, (size_t)(rows + 1) * sizeof(int64_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return 1;
  if (nnz > 0 && (cudaMemcpy(C->col + base, c_col, (size_t)nnz * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess ||
                  cudaMemcpy(C->val + base, c_val, (size_t)nnz * sizeof(double), cudaMemcpyDeviceToHost) != cudaSuccess))
    return 1;
  cudaFree(c_rp);
  cudaFree(c_col);
  cudaFree(c_val);
  *nnz_out = nnz;
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 4 && argc != 5) {
    fprintf(stderr, "usage: %s A.bin B.bin C.bin [parts]\n", argv[0]);
    return 1;
  }
  const int64_t parts = argc == 5 ? atoll(argv[4]) : 1;
  host_csr A, B, C;
  if (!read_csr(argv[1], &A) || !read_csr(argv[2], &B)) {
    fprintf(stderr, "cannot read the input matrices\n");
    return 1;
  }
  gm_csr dA, dB;
  if (!to_device(&A, &dA) || !to_device(&B, &dB)) {
    fprintf(stderr, "device copies failed\n");
    return 1;
  }

  if (parts > 1) {  /* the product part by part, as the ranks of a row split compute it */
    int64_t* bounds = xmalloc((size_t)(parts + 1) * sizeof(int64_t));
    gm_status st = gm_spgemm_row_split(&dA, &dB, NULL, parts, NULL, bounds);
    if (st != GM_OK) return fail("gm_spgemm_row_split", st);
    C.n_rows = A.n_rows;
    C.n_cols = B.n_cols;
    C.row_ptr = xmalloc((size_t)(C.n_rows + 1) * sizeof(int64_t));
    C.col = xmalloc(sizeof(int32_t));
    C.val = xmalloc(sizeof(double));
    C.row_ptr[0] = 0;
    int64_t base = 0, heavy = 0;
    gm_plan_info info;
    for (int64_t q = 0; q < parts; ++q) {
      int64_t nnz = 0;
      const int rc = run_part(&dA, &dB, bounds[q], bounds[q + 1], base, &C, &nnz, &info);
      if (rc) return rc;
      base += nnz;
      heavy += info.n_heavy_rows;
    }
    C.nnz = base;
    if (!write_csr(argv[3], &C)) {
      fprintf(stderr, "cannot write C\n");
      return 1;
    }
    printf("nnz %lld heavy %lld parts %lld\n", (long long)base, (long long)heavy, (long long)parts);
    return 0;
  }

  gm_plan* plan = NULL;
  gm_status st = gm_spgemm_analyze(&dA, &dB, NULL, NULL, &plan);
  if (st != GM_OK) return fail("gm_spgemm_analyze", st);
  void* c_rp = NULL;
  if (cudaMalloc(&c_rp, (size_t)(A.n_rows + 1) * sizeof(int64_t)) != cudaSuccess) return 1;
  int64_t nnz = -1;
  st = gm_spgemm_symbolic(plan, c_rp, &nnz);
  if (st != GM_OK) return fail("gm_spgemm_symbolic", st);
  void *c_col = NULL, *c_val = NULL;
  if (nnz > 0 && (cudaMalloc(&c_col, (size_t)nnz * sizeof(int32_t)) != cudaSuccess ||
                  cudaMalloc(&c_val, (size_t)nnz * sizeof(double)) != cudaSuccess))
    return 1;
  st = gm_spgemm_numeric(plan, c_col, c_val);
  if (st != GM_OK) return fail("gm_spgemm_numeric", st);
  gm_plan_info info;
  st = gm_spgemm_plan_info(plan, &info);
  if (st != GM_OK) return fail("gm_spgemm_plan_info", st);
  gm_spgemm_plan_destroy(plan);

  C.n_rows = A.n_rows;
  C.n_cols = B.n_cols;
  C.nnz = nnz;
  C.row_ptr = xmalloc((size_t)(C.n_rows + 1) * sizeof(int64_t));
  C.col = xmalloc((size_t)nnz * sizeof(int32_t));
  C.val = xmalloc((size_t)nnz * sizeof(double));
  if (cudaMemcpy(C.row_ptr, c_rp, (size_t)(C.n_rows + 1) * sizeof(int64_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return 1;
  if (nnz > 0 && (cudaMemcpy(C.col, c_col, (size_t)nnz * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess ||
                  cudaMemcpy(C.val, c_val, (size_t)nnz * sizeof(double), cudaMemcpyDeviceToHost) != cudaSuccess))
    return 1;
  if (!write_csr(argv[3], &C)) {
    fprintf(stderr, "cannot write C\n");
    return 1;
  }
  printf("nnz %lld heavy %lld levels %lld pipeline %d\n", (long long)nnz, (long long)info.n_heavy_rows,
         (long long)info.params.n_levels, (int)info.pipeline);
  return 0;
}
