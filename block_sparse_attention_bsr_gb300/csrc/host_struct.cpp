// Host-side BSR structure helpers: validation and the BSC transpose.
//
// The column-first (BSC) view is what the dK/dV walk traverses
// ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG [0.5.1]: the dK/dV kernel walks
// block columns over a BSC view built on the host, so no atomic scatter is
// needed).  It is a counting sort of the stored (row, column) pairs by column;
// scanning rows in ascending order keeps the rows of one column ascending.

#include "internal.h"

#include <vector>

extern "C" bsr_status bsr_validate(const int32_t* row_ptr_h, const int32_t* col_idx_h,
                                   int32_t n_brows, int32_t n_bcols) {
  if (!row_ptr_h) return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_validate: row_ptr is null");
  if (n_brows < 0 || n_bcols < 0)
    return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_validate: negative n_brows (%d) or n_bcols (%d)", n_brows, n_bcols);
  if (row_ptr_h[0] != 0) return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_validate: row_ptr[0] = %d, expected 0", row_ptr_h[0]);
  for (int32_t m = 0; m < n_brows; ++m) {
    if (row_ptr_h[m + 1] < row_ptr_h[m])
      return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_validate: row_ptr decreases at block row %d (%d -> %d)", m,
                       row_ptr_h[m], row_ptr_h[m + 1]);
  }
  const int64_t nnzb = row_ptr_h[n_brows];
  if (nnzb > 0 && !col_idx_h) return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_validate: col_idx is null");
  if (nnzb > (int64_t)n_brows * (int64_t)n_bcols)
    return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_validate: %lld stored blocks exceed the %d x %d grid", (long long)nnzb,
                     n_brows, n_bcols);
  for (int32_t m = 0; m < n_brows; ++m) {
    int32_t prev = -1;
    for (int32_t j = row_ptr_h[m]; j < row_ptr_h[m + 1]; ++j) {
      const int32_t n = col_idx_h[j];
      if (n < 0 || n >= n_bcols)
        return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_validate: col_idx[%d] = %d outside [0, %d)", j, n, n_bcols);
      if (n <= prev)
        return bsr::fail(BSR_ERR_INVALID_ARG,
                         "bsr_validate: block row %d columns not strictly ascending (%d after %d)", m, n, prev);
      prev = n;
    }
  }
  return BSR_OK;
}

extern "C" bsr_status bsr_build_bsc(const int32_t* row_ptr_h, const int32_t* col_idx_h,
                                    int32_t n_brows, int32_t n_bcols,
                                    int32_t* col_ptr_h, int32_t* row_idx_h) {
  bsr_status st = bsr_validate(row_ptr_h, col_idx_h, n_brows, n_bcols);
  if (st != BSR_OK) return st;
  const int32_t nnzb = row_ptr_h[n_brows];
  if (!col_ptr_h || (nnzb > 0 && !row_idx_h))
    return bsr::fail(BSR_ERR_INVALID_ARG, "bsr_build_bsc: null output array");
  std::vector<int32_t> count(n_bcols + 1, 0);
  for (int32_t j = 0; j < nnzb; ++j) count[col_idx_h[j] + 1]++;
  for (int32_t n = 0; n < n_bcols; ++n) count[n + 1] += count[n];
  for (int32_t n = 0; n <= n_bcols; ++n) col_ptr_h[n] = count[n];
  std::vector<int32_t> fill(count.begin(), count.end() - 1);
  for (int32_t m = 0; m < n_brows; ++m)
    for (int32_t j = row_ptr_h[m]; j < row_ptr_h[m + 1]; ++j) row_idx_h[fill[col_idx_h[j]]++] = m;
  return BSR_OK;
}
