// format.cpp -- CSR -> BCSR and CSR -> WCSR on the host.
//
// "AsyncSparse", Section II-C and Fig. 2.  BCSR keeps every b_row x b_col
// block that holds a CSR entry, dense and row-major, in ascending block-column
// order per block row.  WCSR keeps, per window of h rows, the ascending union
// of the rows' columns padded with -1 to a multiple of `pad`, and packs the
// values into one row-major [h][P_total] array.  Partial last block rows,
// block columns and windows are zero-padded.
#include "format.h"

#include <algorithm>
#include <cstring>

namespace spmm {

std::string check_csr(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx) {
  if (m < 0 || k < 0) return "negative dimension";
  if (row_ptr[0] != 0) return "row_ptr[0] != 0";
  for (int64_t i = 0; i < m; ++i) {
    const int64_t b = row_ptr[i], e = row_ptr[i + 1];
    if (e < b) return "row_ptr decreases at row " + std::to_string(i);
    int64_t prev = -1;
    for (int64_t t = b; t < e; ++t) {
      const int64_t c = col_idx[t];
      if (c < 0 || c >= k) return "column out of range in row " + std::to_string(i);
      if (c <= prev) return "columns not strictly ascending in row " + std::to_string(i);
      prev = c;
    }
  }
  return std::string();
}

void build_bcsr(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx, const uint16_t *vals,
                int b_row, int b_col, HostFormat &out) {
  const int64_t nbr = (m + b_row - 1) / b_row;
  const int64_t nbc = (k + b_col - 1) / b_col;
  const int64_t bs = static_cast<int64_t>(b_row) * b_col;
  out.ptr.assign(nbr + 1, 0);
  out.idx.clear();
  out.vals.clear();
  // seen[c] == R + 1 marks block column c as touched in block row R;
  // where[c] is its index among the stored blocks.
  std::vector<int64_t> seen(static_cast<size_t>(nbc), 0);
  std::vector<int64_t> where(static_cast<size_t>(nbc), 0);
  std::vector<int32_t> cols;
  for (int64_t R = 0; R < nbr; ++R) {
    const int64_t r0 = R * b_row, r1 = std::min<int64_t>(m, r0 + b_row);
    cols.clear();
    for (int64_t t = row_ptr[r0]; t < row_ptr[r1]; ++t) {
      const int32_t c = col_idx[t] / b_col;
      if (seen[c] != R + 1) {
        seen[c] = R + 1;
        cols.push_back(c);
      }
    }
    std::sort(cols.begin(), cols.end());
    const int64_t base = static_cast<int64_t>(out.idx.size());
    for (size_t j = 0; j < cols.size(); ++j) {
      where[cols[j]] = base + static_cast<int64_t>(j);
      out.idx.push_back(cols[j]);
    }
    out.ptr[R + 1] = static_cast<int64_t>(out.idx.size());
    if (vals) {
      out.vals.resize(out.idx.size() * bs, 0);
      for (int64_t i = r0; i < r1; ++i)
        for (int64_t t = row_ptr[i]; t < row_ptr[i + 1]; ++t) {
          const int64_t c = col_idx[t];
          const int64_t blk = where[c / b_col];
          out.vals[blk * bs + (i - r0) * b_col + (c % b_col)] = vals[t];
        }
    }
  }
  out.n_units = static_cast<int64_t>(out.idx.size());
}

void build_wcsr(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx, const uint16_t *vals,
                int h, int pad, HostFormat &out) {
  const int64_t nw = (m + h - 1) / h;
  out.ptr.assign(nw + 1, 0);
  out.idx.clear();
  out.vals.clear();
  std::vector<int64_t> seen(static_cast<size_t>(k), 0);
  std::vector<int32_t> cols;
  // Pass 1: column unions and their padded lengths.
  for (int64_t w = 0; w < nw; ++w) {
    const int64_t r0 = w * h, r1 = std::min<int64_t>(m, r0 + h);
    cols.clear();
    for (int64_t t = row_ptr[r0]; t < row_ptr[r1]; ++t) {
      const int32_t c = col_idx[t];
      if (seen[c] != w + 1) {
        seen[c] = w + 1;
        cols.push_back(c);
      }
    }
    std::sort(cols.begin(), cols.end());
    const int64_t padded = (static_cast<int64_t>(cols.size()) + pad - 1) / pad * pad;
    out.idx.insert(out.idx.end(), cols.begin(), cols.end());
    out.idx.insert(out.idx.end(), static_cast<size_t>(padded - static_cast<int64_t>(cols.size())), -1);
    out.ptr[w + 1] = static_cast<int64_t>(out.idx.size());
  }
  out.n_units = static_cast<int64_t>(out.idx.size());
  if (!vals) return;
  // Pass 2: scatter values; slot[c] is column c's packed position in the
  // current window.
  const int64_t P = out.n_units;
  out.vals.assign(static_cast<size_t>(P * h), 0);
  std::vector<int64_t> slot(static_cast<size_t>(k), 0);
  for (int64_t w = 0; w < nw; ++w) {
    for (int64_t p = out.ptr[w]; p < out.ptr[w + 1]; ++p)
      if (out.idx[p] >= 0) slot[out.idx[p]] = p;
    const int64_t r0 = w * h, r1 = std::min<int64_t>(m, r0 + h);
    for (int64_t i = r0; i < r1; ++i)
      for (int64_t t = row_ptr[i]; t < row_ptr[i + 1]; ++t)
        out.vals[(i - r0) * P + slot[col_idx[t]]] = vals[t];
  }
}

}  // namespace spmm
