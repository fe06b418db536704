// format.h -- host-side construction of the BCSR and WCSR formats from CSR.
#pragma once

#include <stdint.h>

#include <string>
#include <vector>

namespace spmm {

// Checks row_ptr[0] == 0, non-decreasing row_ptr, columns in [0, k) and
// strictly ascending per row.  Returns an empty string when valid, else a
// description of the first violation.
std::string check_csr(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx);

struct HostFormat {
  std::vector<int64_t> ptr;    // block_row_ptr / window_row_ptr
  std::vector<int32_t> idx;    // block_col_idx / window_col_idx
  std::vector<uint16_t> vals;  // blocks / values
  int64_t n_units = 0;         // stored blocks / padded column positions
};

// BCSR ("AsyncSparse", Section II-C, Fig. 2).  vals == nullptr skips values.
void build_bcsr(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx, const uint16_t *vals,
                int b_row, int b_col, HostFormat &out);

// WCSR ("AsyncSparse", Section II-C, Fig. 2); values row-major [h][P_total].
void build_wcsr(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx, const uint16_t *vals,
                int h, int pad, HostFormat &out);

}  // namespace spmm
