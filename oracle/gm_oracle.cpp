// gm_oracle.cpp -- CPU oracle for C = A*B over CSR (test infrastructure only).
//
// This file is the correctness reference for the GPU SpGEMM. It is deliberately
// plain and slow: row-wise Gustavson with one std::map accumulator per row.
// It shares no code with the CUDA library; only tests, the package smoke check
// and the benchmark's CPU-baseline leg may load it.
//
// What it follows (gMAGNUS, "Fast SpGEMM on GPUs for Irregular Matrices via
// Hierarchical Multisplit"):
//   * Sec. II-B, Eq. (1): C[i,:] = sum_j A[i,j] * B[j,:].
//   * Sec. II-B, Algorithm 1 (Gustavson): for every stored A[i,j], add A[i,j]*B[j,k]
//     into an accumulator keyed by column k, then emit the row sorted by column.
//   * Structure is symbolic: an entry (i,k) exists when some stored A[i,j] meets
//     a stored B[j,k], even if the values cancel or are zero (the symbolic phase
//     fixes C.rowPtr before any value is known, Sec. II-B).
//   * Per-row intermediate-product count u(i) = sum over stored A[i,j] of nnz(B[j,:])
//     (Sec. III-A, InterOffsets; SparseDitto, "SpGEMM", Eq. (1)).
// Alongside each value the oracle returns sum_j |A[i,j]*B[j,k]|, the scale of the
// fp64 tolerance used when comparing against a reordered summation.
//
// Build: g++ -O2 -std=c++17 -fopenmp -shared -fPIC gm_oracle.cpp -o libgm_oracle.so

#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <utility>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

struct Acc {
  double sum = 0.0;  // sum of products in the order Algorithm 1 visits them
  double abs = 0.0;  // sum of |products|
};

struct RowOut {
  std::vector<int32_t> col;
  std::vector<double> val;
  std::vector<double> abs;
};

}  // namespace

struct gm_oracle_result {
  std::vector<RowOut> rows;
  int64_t nnz = 0;
};

extern "C" {

// u[i] = sum_{p in A[i,:]} (B.rowPtr[A.col[p]+1] - B.rowPtr[A.col[p]]).
// Returns 0, or -1 when a column index of A is outside [0, b_rows).
int gm_oracle_ip_counts(int64_t a_rows, const int64_t* a_rp, const int32_t* a_col,
                        int64_t b_rows, const int64_t* b_rp, int64_t* u_out) {
  int bad = 0;
  for (int64_t i = 0; i < a_rows; ++i) {
    int64_t u = 0;
    for (int64_t p = a_rp[i]; p < a_rp[i + 1]; ++p) {
      int64_t k = a_col[p];
      if (k < 0 || k >= b_rows) { bad = 1; continue; }
      u += b_rp[k + 1] - b_rp[k];
    }
    u_out[i] = u;
  }
  return bad ? -1 : 0;
}

// Gustavson (Algorithm 1) on the selected rows of A (all rows when rows == nullptr).
// Returns nullptr when an index is out of range.
gm_oracle_result* gm_oracle_spgemm_rows(int64_t a_rows, int64_t a_cols, const int64_t* a_rp,
                                        const int32_t* a_col, const double* a_val,
                                        int64_t b_rows, int64_t b_cols, const int64_t* b_rp,
                                        const int32_t* b_col, const double* b_val,
                                        const int64_t* rows, int64_t n_sel, int n_threads) {
  if (a_cols != b_rows) return nullptr;
  const int64_t n_out = rows ? n_sel : a_rows;
  for (int64_t s = 0; s < n_out; ++s) {
    int64_t i = rows ? rows[s] : s;
    if (i < 0 || i >= a_rows) return nullptr;
  }
  auto* res = new gm_oracle_result;
  res->rows.resize(n_out);
  int bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
#endif
  for (int64_t s = 0; s < n_out; ++s) {
    const int64_t i = rows ? rows[s] : s;
    std::map<int32_t, Acc> acc;
    for (int64_t p = a_rp[i]; p < a_rp[i + 1]; ++p) {
      const int64_t j = a_col[p];
      if (j < 0 || j >= b_rows) { bad = 1; continue; }
      const double a = a_val[p];
      for (int64_t q = b_rp[j]; q < b_rp[j + 1]; ++q) {
        const int32_t k = b_col[q];
        if (k < 0 || k >= b_cols) { bad = 1; continue; }
        const double prod = a * b_val[q];
        Acc& e = acc[k];
        e.sum += prod;
        e.abs += std::fabs(prod);
      }
    }
    RowOut& out = res->rows[s];
    out.col.reserve(acc.size());
    out.val.reserve(acc.size());
    out.abs.reserve(acc.size());
    for (const auto& kv : acc) {  // std::map iterates in ascending column order
      out.col.push_back(kv.first);
      out.val.push_back(kv.second.sum);
      out.abs.push_back(kv.second.abs);
    }
  }
  if (bad) {
    delete res;
    return nullptr;
  }
  for (const auto& r : res->rows) res->nnz += static_cast<int64_t>(r.col.size());
  return res;
}

int64_t gm_oracle_result_rows(const gm_oracle_result* r) { return static_cast<int64_t>(r->rows.size()); }
int64_t gm_oracle_result_nnz(const gm_oracle_result* r) { return r->nnz; }

// Copies the result out: row_ptr[n_rows+1], col[nnz], val[nnz], abs_scale[nnz] (nullable).
void gm_oracle_result_copy(const gm_oracle_result* r, int64_t* row_ptr, int32_t* col, double* val,
                           double* abs_scale) {
  int64_t pos = 0;
  row_ptr[0] = 0;
  for (size_t s = 0; s < r->rows.size(); ++s) {
    const RowOut& o = r->rows[s];
    const size_t n = o.col.size();
    if (n) {
      std::memcpy(col + pos, o.col.data(), n * sizeof(int32_t));
      std::memcpy(val + pos, o.val.data(), n * sizeof(double));
      if (abs_scale) std::memcpy(abs_scale + pos, o.abs.data(), n * sizeof(double));
    }
    pos += static_cast<int64_t>(n);
    row_ptr[s + 1] = pos;
  }
}

void gm_oracle_result_free(gm_oracle_result* r) { delete r; }

int gm_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
