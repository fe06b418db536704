// spmm_api.cu -- the C ABI (include/spmm.h): handle life cycle, validation,
// upload, TMA descriptor encoding, WCSR task decomposition and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/spmm.h"
#include "format.h"
#include "internal.h"
#include "ptx.cuh"

using spmm::HostFormat;

namespace {

thread_local std::string g_last_error;

spmm_status fail(spmm_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

spmm_status cuda_fail(cudaError_t e, const char *what) {
  return fail(e == cudaErrorMemoryAllocation ? SPMM_ERR_OOM : SPMM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CUDA_TRY(call, what)                      \
  do {                                            \
    cudaError_t e_ = (call);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;  // 4 s per mbarrier wait

// ---------------------------------------------------------------- driver entry
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D row-major tensor of 16-bit elements: `rows` x `cols`, row pitch
// `pitch_elems`; boxes of box_rows x box_cols (box_cols * 2 <= 128 bytes),
// 128-byte swizzle, out-of-bounds elements read as zero.
spmm_status encode_2d(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols,
                      uint64_t pitch_elems, uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(SPMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return SPMM_OK;
}

// C as the destination of TMA stores: `rows` x `cols` row-major elements of
// bf16 or fp32.  Narrow (N <= 128) tiles store 16-row x 128-byte boxes with the
// 128-byte swizzle, wide ones 32-row x 64-byte boxes with the 64-byte swizzle
// (see bcsr_wide_tiles).
spmm_status encode_c(CUtensorMap *map, void *base, bool bf16, uint64_t rows, uint64_t cols, bool wide) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(SPMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const uint64_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>((wide ? 64 : 128) / esz), wide ? 32u : 16u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  wide ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPMM_ERR_CUDA, "cuTensorMapEncodeTiled (C) failed (%d)", static_cast<int>(r));
  return SPMM_OK;
}

// X of the linear-layer product as a TMA source: N rows x k columns of
// 16-bit elements, 256-row x 64-column boxes, 128-byte swizzle.
spmm_status encode_x(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols) {
  return encode_2d(map, base, bf16, rows, cols, cols, 256, 64);
}

// Y of the linear-layer product as a TMA destination: N rows x m columns of
// bf16 or fp32, 32-row x 128-byte boxes, 128-byte swizzle.
spmm_status encode_y(CUtensorMap *map, void *base, bool bf16, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(SPMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const uint64_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), 32u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPMM_ERR_CUDA, "cuTensorMapEncodeTiled (Y) failed (%d)", static_cast<int>(r));
  return SPMM_OK;
}

}  // namespace

struct spmm_handle_s {
  int format = 0;
  int64_t m = 0, k = 0, nnz = 0;
  int b_row = 0, b_col = 0;
  spmm_dtype in_t = SPMM_BF16, out_t = SPMM_F32;
  int device = 0;
  int num_sms = 0;
  bool sm103 = false;
  int64_t n_groups = 0, n_units = 0, stored = 0;

  int64_t *d_ptr = nullptr;
  int32_t *d_idx = nullptr;
  uint16_t *d_vals = nullptr;
  size_t vals_bytes = 0;
  CUtensorMap tm_vals;  // BCSR: the blocks array as [n_blocks*64 rows, 64 cols] for TMA

  const void *b_cached = nullptr;
  int64_t n_cached = -1;
  CUtensorMap tm_B;
  void *c_cached = nullptr;
  int64_t nc_cached = -1;
  CUtensorMap tm_C;
  // the linear-layer product's X and Y
  const void *x_cached = nullptr;
  int64_t nx_cached = -1;
  CUtensorMap tm_X;
  void *y_cached = nullptr;
  int64_t ny_cached = -1;
  CUtensorMap tm_Y;

  // Work decomposition.  WCSR: stages of <= 64 packed columns.  BCSR: the
  // prefix sums of max(1, blocks) per block row (the split schedule's stage
  // list).  Both: the partial-sum workspace of groups cut between persistent
  // CTAs (BCSR: allocated only when the split schedule can be chosen).
  int32_t max_ctas = 0;  // 0: the kernels' default CTAs per SM
  int32_t schedule = SPMM_SCHEDULE_AUTO;
  int64_t n_stages = 0;
  int64_t *d_stage_row_ptr = nullptr;
  uint8_t *d_stage_pack = nullptr;
  float *d_ws = nullptr;
  spmm::PartialRec *d_partials = nullptr;
  int64_t ws_slots = 0;
  std::vector<int32_t> stage_first;  // host copy of the stage list's first-stage flags (for statistics)

  uint32_t *d_status = nullptr;
  uint64_t wait_limit_ns = kDefaultWaitLimitNs;

  void *d_bstage = nullptr;
  size_t bstage_bytes = 0;
  void *d_cstage = nullptr;
  size_t cstage_bytes = 0;
};

namespace {

size_t elem_size(spmm_dtype t) { return t == SPMM_F32 ? 4 : 2; }

spmm_status check_common(spmm_handle *out, int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                         const void *vals, spmm_dtype in_t, spmm_dtype out_t, int a, int b) {
  if (out) *out = nullptr;
  if (!out) return fail(SPMM_ERR_INVALID_ARG, "out is NULL");
  if (m < 0 || k < 0 || m >= (1ll << 31) || k >= (1ll << 31)) return fail(SPMM_ERR_INVALID_ARG, "m, k must be in [0, 2^31)");
  if (!row_ptr) return fail(SPMM_ERR_INVALID_ARG, "row_ptr is NULL");
  const int64_t nnz = row_ptr[m];
  if (nnz > 0 && (!col_idx || !vals)) return fail(SPMM_ERR_INVALID_ARG, "col_idx or vals is NULL");
  if (in_t != SPMM_F16 && in_t != SPMM_BF16) return fail(SPMM_ERR_INVALID_ARG, "in_t must be F16 or BF16");
  if (out_t != SPMM_F32 && out_t != SPMM_BF16) return fail(SPMM_ERR_INVALID_ARG, "out_t must be F32 or BF16");
  if (a < 1 || a > 256 || b < 1 || b > 256) return fail(SPMM_ERR_INVALID_ARG, "block / window parameters must be in [1, 256]");
  std::string why = spmm::check_csr(m, k, row_ptr, col_idx);
  if (!why.empty()) return fail(SPMM_ERR_INVALID_ARG, "invalid CSR: %s", why.c_str());
  return SPMM_OK;
}

void free_handle(spmm_handle h) {
  if (!h) return;
  cudaFree(h->d_ptr);
  cudaFree(h->d_idx);
  cudaFree(h->d_vals);
  cudaFree(h->d_stage_pack);
  cudaFree(h->d_stage_row_ptr);
  cudaFree(h->d_partials);
  cudaFree(h->d_ws);
  cudaFree(h->d_status);
  cudaFree(h->d_bstage);
  cudaFree(h->d_cstage);
  delete h;
}

spmm_status upload_common(spmm_handle h, const HostFormat &f) {
  CUDA_TRY(cudaGetDevice(&h->device), "cudaGetDevice");
  cudaDeviceProp prop;
  CUDA_TRY(cudaGetDeviceProperties(&prop, h->device), "cudaGetDeviceProperties");
  h->num_sms = prop.multiProcessorCount;
  h->sm103 = prop.major == 10 && prop.minor == 3;
  CUDA_TRY(cudaMalloc(&h->d_ptr, f.ptr.size() * sizeof(int64_t)), "cudaMalloc(ptr)");
  CUDA_TRY(cudaMemcpy(h->d_ptr, f.ptr.data(), f.ptr.size() * sizeof(int64_t), cudaMemcpyHostToDevice), "upload ptr");
  const size_t ni = std::max<size_t>(f.idx.size(), 1);
  CUDA_TRY(cudaMalloc(&h->d_idx, ni * sizeof(int32_t)), "cudaMalloc(idx)");
  if (!f.idx.empty())
    CUDA_TRY(cudaMemcpy(h->d_idx, f.idx.data(), f.idx.size() * sizeof(int32_t), cudaMemcpyHostToDevice), "upload idx");
  // At least one zero 64 x 64 tile so a tensor map can always be encoded.
  h->vals_bytes = std::max<size_t>(f.vals.size() * 2, 64 * 64 * 2);
  CUDA_TRY(cudaMalloc(&h->d_vals, h->vals_bytes), "cudaMalloc(values)");
  CUDA_TRY(cudaMemset(h->d_vals, 0, h->vals_bytes), "cudaMemset(values)");
  if (!f.vals.empty())
    CUDA_TRY(cudaMemcpy(h->d_vals, f.vals.data(), f.vals.size() * 2, cudaMemcpyHostToDevice), "upload values");
  CUDA_TRY(cudaMalloc(&h->d_status, sizeof(uint32_t)), "cudaMalloc(status)");
  CUDA_TRY(cudaMemset(h->d_status, 0, sizeof(uint32_t)), "cudaMemset(status)");
  return SPMM_OK;
}

// The WCSR stage list: each window cut into stages of at most 64 packed
// columns, in window order; a window without columns gets one empty stage.
// The kernel reads each stage as one record (its H x 64 value tile, column
// indices and descriptor; see wcsr_pack_bytes, H = the window height).  In
// those records a window of ns >= 2 stages deals its padded column list
// round-robin over its stages (stage j takes positions j, j + ns, j + 2 ns,
// ...; positions past P_w are padding), so each stage's rows of B span the
// whole window: packed columns are sorted, and windows processed at the same
// time by different CTAs would otherwise all gather from the same band of B
// rows and the same L2 slices.  The product is the same sum in another order.
// A stage's column count is rounded up to the MMA's 16-deep k step with
// padding positions (a column padding of 8 leaves odd multiples of 8).
spmm_status build_stages(spmm_handle h, const std::vector<int64_t> &wptr, const std::vector<int32_t> &widx,
                         const std::vector<uint16_t> &wvals) {
  std::vector<spmm::WcsrStage> st;
  std::vector<uint8_t> pack;
  const int64_t nw = h->n_groups;
  const int64_t P = h->n_units;
  const int H = h->b_row;
  const size_t rec = static_cast<size_t>(spmm::wcsr_pack_bytes(H));
  // stage s's record at s * rec
  auto new_stage = [&](int32_t p_begin, int32_t window, int32_t ncols, int32_t flags) -> size_t {
    const size_t s = st.size();
    st.push_back({p_begin, window, ncols, flags});
    pack.resize(pack.size() + rec, 0);
    int32_t *idx = reinterpret_cast<int32_t *>(&pack[s * rec + spmm::wcsr_pack_idx_off(H)]);
    for (int c = 0; c < 64; ++c) idx[c] = c < ncols ? -1 : -2;
    const int32_t desc[4] = {ncols, flags, window, 0};
    std::memcpy(&pack[s * rec + spmm::wcsr_pack_desc_off(H)], desc, sizeof desc);
    return s;
  };
  auto put_val = [&](size_t s, int r, int c, uint16_t v) {
    // row r at r * 128 bytes, 16-byte unit u stored at unit u ^ (r % 8)
    uint16_t *tile = reinterpret_cast<uint16_t *>(&pack[s * rec]);
    tile[r * 64 + (((c >> 3) ^ (r & 7)) << 3) + (c & 7)] = v;
  };
  auto put_idx = [&](size_t s, int c, int32_t col) {
    std::memcpy(&pack[s * rec + spmm::wcsr_pack_idx_off(H) + 4 * c], &col, 4);
  };
  for (int64_t w = 0; w < nw; ++w) {
    const int64_t b = wptr[w], e = wptr[w + 1], pw = e - b;
    if (pw == 0) {
      new_stage(static_cast<int32_t>(b), static_cast<int32_t>(w), 0, spmm::kStageFirst | spmm::kStageLast);
      continue;
    }
    const int64_t ns = (pw + 63) / 64;
    for (int64_t j = 0; j < ns; ++j) {
      const int32_t flags = (j == 0 ? spmm::kStageFirst : 0) | (j == ns - 1 ? spmm::kStageLast : 0);
      const int32_t ncols = ns == 1 ? static_cast<int32_t>((pw + 15) / 16 * 16) : 64;
      const size_t s = new_stage(static_cast<int32_t>(b + 64 * j), static_cast<int32_t>(w), ncols, flags);
      for (int c = 0; c < ncols; ++c) {
        const int64_t q = ns == 1 ? c : j + ns * c;  // position within the window
        if (q >= pw) continue;                       // padding: zero values, no B row
        put_idx(s, c, widx[b + q]);
        for (int r = 0; r < H; ++r) put_val(s, r, c, wvals[r * P + b + q]);
      }
    }
  }
  h->n_stages = static_cast<int64_t>(st.size());
  h->stage_first.resize(st.size());
  for (size_t i = 0; i < st.size(); ++i) h->stage_first[i] = st[i].flags & spmm::kStageFirst;
  CUDA_TRY(cudaMalloc(&h->d_stage_pack, std::max<size_t>(pack.size(), rec)), "cudaMalloc(stage records)");
  if (!pack.empty())
    CUDA_TRY(cudaMemcpy(h->d_stage_pack, pack.data(), pack.size(), cudaMemcpyHostToDevice), "upload stage records");
  // Two partial slots per CTA, sized for the largest grid.
  h->ws_slots = 2 * static_cast<int64_t>(spmm::kWcsrMaxCtasPerSm) * std::max(h->num_sms, 1);
  const int64_t slot_floats = H == 64 ? spmm::kWcsr64SlotFloats : spmm::kWcsrSlotFloats;
  CUDA_TRY(cudaMalloc(&h->d_ws, h->ws_slots * slot_floats * sizeof(float)), "cudaMalloc(workspace)");
  CUDA_TRY(cudaMalloc(&h->d_partials, h->ws_slots * sizeof(spmm::PartialRec)), "cudaMalloc(partials)");
  return SPMM_OK;
}

// BCSR split schedule: the stage list's prefix sums per block row
// (max(1, blocks): a block row without blocks is one stage) and, when the
// problem has few enough block rows that some N can select the schedule, its
// partial-sum workspace.
spmm_status build_bcsr_split(spmm_handle h, const std::vector<int64_t> &bptr) {
  const int64_t nbr = h->n_groups;
  std::vector<int64_t> srp(nbr + 1, 0);
  for (int64_t r = 0; r < nbr; ++r) srp[r + 1] = srp[r] + std::max<int64_t>(1, bptr[r + 1] - bptr[r]);
  h->n_stages = srp[nbr];
  CUDA_TRY(cudaMalloc(&h->d_stage_row_ptr, srp.size() * sizeof(int64_t)), "cudaMalloc(stage row pointers)");
  CUDA_TRY(cudaMemcpy(h->d_stage_row_ptr, srp.data(), srp.size() * sizeof(int64_t), cudaMemcpyHostToDevice),
           "upload stage row pointers");
  if (nbr < static_cast<int64_t>(spmm::kBcsrSplitBelowTilesPerSm) * std::max(h->num_sms, 1)) {
    h->ws_slots = 2 * static_cast<int64_t>(spmm::kBcsrSplitCtasPerSm) * std::max(h->num_sms, 1);
    CUDA_TRY(cudaMalloc(&h->d_ws, h->ws_slots * spmm::kBcsrSlotFloats * sizeof(float)), "cudaMalloc(workspace)");
    CUDA_TRY(cudaMalloc(&h->d_partials, h->ws_slots * sizeof(spmm::PartialRec)), "cudaMalloc(partials)");
  }
  return SPMM_OK;
}

// BCSR grid of the split schedule at dense width N, or 0 for the tile
// schedule (whole tiles per CTA).  SPMM_SCHEDULE_AUTO takes the split schedule
// when fewer than half the SMs would get a tile and the tiles average at
// least 8 stages: there the tile schedule leaves most SMs idle while a few
// walk long block rows, and spreading the stages outweighs the second pass.
// The grid is up to kBcsrSplitCtasPerSm CTAs per SM with at least
// kBcsrSplitMinStages stages each (and at most the spmm_set_max_ctas cap).
int32_t bcsr_split_grid(spmm_handle h, int64_t N) {
  if (!h->d_ws || h->schedule == SPMM_SCHEDULE_TILES) return 0;
  const int64_t col_tiles = (N + spmm::bcsr_tile_cols(N) - 1) / spmm::bcsr_tile_cols(N);
  const int64_t sms = std::max(h->num_sms, 1);
  const int64_t tiles = h->n_groups * col_tiles;
  if (tiles >= spmm::kBcsrSplitBelowTilesPerSm * sms) return 0;
  if (h->schedule == SPMM_SCHEDULE_AUTO && (2 * tiles > sms || h->n_stages < 8 * h->n_groups)) return 0;
  const int64_t stages = h->n_stages * col_tiles;
  int64_t g = std::min<int64_t>(spmm::kBcsrSplitCtasPerSm * sms,
                                (stages + spmm::kBcsrSplitMinStages - 1) / spmm::kBcsrSplitMinStages);
  if (h->max_ctas > 0) g = std::min<int64_t>(g, h->max_ctas);
  return static_cast<int32_t>(std::max<int64_t>(1, g));
}

// Persistent grid of the WCSR kernel for N columns.
int32_t wcsr_grid(spmm_handle h, int64_t N) {
  const int64_t bn = h->b_row == 64 ? 256 : spmm::wcsr_tile_cols(N);
  const int64_t items = h->n_stages * ((N + bn - 1) / bn);
  const int64_t most = static_cast<int64_t>(spmm::kWcsrMaxCtasPerSm) * h->num_sms;
  const int per_sm = h->b_row == 64 ? spmm::wcsr64_ctas_per_sm() : spmm::wcsr_ctas_per_sm(N);
  int64_t g = h->max_ctas > 0 ? std::min<int64_t>(h->max_ctas, most) : static_cast<int64_t>(per_sm) * h->num_sms;
  return static_cast<int32_t>(std::max<int64_t>(0, std::min(g, items)));
}

spmm_status check_run_args(spmm_handle h, const void *B, void *C, int64_t N) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  if (N <= 0 || N >= (1ll << 31)) return fail(SPMM_ERR_INVALID_ARG, "N must be in (0, 2^31)");
  if (!B || !C) return fail(SPMM_ERR_INVALID_ARG, "B or C is NULL");
  if (N % 8 != 0) return fail(SPMM_ERR_UNSUPPORTED, "N must be a multiple of 8 (16-byte rows of B)");
  if (N > 65535ll * 128) return fail(SPMM_ERR_UNSUPPORTED, "N above 65535 * 128 exceeds the launch grid");
  if ((reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15)
    return fail(SPMM_ERR_UNSUPPORTED, "B and C must be 16-byte aligned");
  if (!h->sm103) return fail(SPMM_ERR_UNSUPPORTED, "the kernels need an sm_103 (GB300) device");
  return SPMM_OK;
}

spmm_status run_device(spmm_handle h, const void *B, void *C, int64_t N, cudaStream_t s) {
  if (h->m == 0) return SPMM_OK;
  const bool in_bf16 = h->in_t == SPMM_BF16;
  const bool out_bf16 = h->out_t == SPMM_BF16;
  if (h->format == SPMM_FORMAT_BCSR) {
    if (h->b_row != 64 || h->b_col != 64) return fail(SPMM_ERR_UNSUPPORTED, "the BCSR kernel takes 64 x 64 blocks");
    if (h->b_cached != B || h->n_cached != N) {
      spmm_status st = encode_2d(&h->tm_B, B, in_bf16, static_cast<uint64_t>(std::max<int64_t>(h->k, 1)),
                                 static_cast<uint64_t>(N), static_cast<uint64_t>(N), 64, 64);
      if (st != SPMM_OK) return st;
      h->b_cached = B;
      h->n_cached = N;
    }
    if (h->c_cached != C || h->nc_cached != N) {
      spmm_status st = encode_c(&h->tm_C, C, out_bf16, static_cast<uint64_t>(h->m), static_cast<uint64_t>(N),
                                spmm::bcsr_wide_tiles(N));
      if (st != SPMM_OK) return st;
      h->c_cached = C;
      h->nc_cached = N;
    }
    spmm::BcsrParams p;
    p.block_row_ptr = h->d_ptr;
    p.block_col_idx = h->d_idx;
    p.blocks = h->d_vals;
    p.stage_row_ptr = h->d_stage_row_ptr;
    p.workspace = h->d_ws;
    p.partials = h->d_partials;
    p.split_grid = bcsr_split_grid(h, N);
    p.split_stages = h->n_stages;
    p.n_blocks = h->n_units;
    p.B = B;
    p.C = C;
    p.ldc = N;
    p.M = static_cast<int32_t>(h->m);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(h->k);
    p.n_block_rows = static_cast<int32_t>(h->n_groups);
    p.max_ctas = h->max_ctas;
    p.num_sms = std::max(h->num_sms, 1);
    p.status = h->d_status;
    p.wait_limit_ns = h->wait_limit_ns;
    cudaError_t e = spmm::launch_bcsr(h->tm_vals, h->tm_B, h->tm_C, p, in_bf16, out_bf16, s);
    if (e != cudaSuccess) return cuda_fail(e, "BCSR kernel launch");
    return SPMM_OK;
  }
  // WCSR
  const bool w64 = h->b_row == 64;
  if (!((h->b_row == 16 && h->b_col % 16 == 0) || (w64 && h->b_col % 8 == 0)))
    return fail(SPMM_ERR_UNSUPPORTED,
                "the WCSR kernels take window height 16 with column padding a multiple of 16, or window height 64 "
                "with column padding a multiple of 8");
  if (w64 && (h->c_cached != C || h->nc_cached != N)) {
    spmm_status st = encode_c(&h->tm_C, C, out_bf16, static_cast<uint64_t>(h->m), static_cast<uint64_t>(N), true);
    if (st != SPMM_OK) return st;
    h->c_cached = C;
    h->nc_cached = N;
  }
  spmm::WcsrParams p;
  p.stages = nullptr;
  p.stage_pack = h->d_stage_pack;
  p.values = h->d_vals;
  p.window_col_idx = h->d_idx;
  p.n_stages_dev = nullptr;
  p.P_total = h->n_units;
  p.B = B;
  p.C = C;
  p.workspace = h->d_ws;
  p.partials = h->d_partials;
  p.n_stages = h->n_stages;
  p.M = static_cast<int32_t>(h->m);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(h->k);
  p.grid = wcsr_grid(h, N);
  p.dynamic = 0;
  if (!w64 && h->schedule == SPMM_SCHEDULE_DYNAMIC && p.grid > 0) {
    // one CTA per chunk, about kWcsrDynChunksPerCta chunks per CTA that fits,
    // each of at least kWcsrDynMinChunkItems work items
    const int64_t items = h->n_stages * ((N + spmm::wcsr_tile_cols(N) - 1) / spmm::wcsr_tile_cols(N));
    const int64_t chunks = std::min<int64_t>({static_cast<int64_t>(spmm::kWcsrDynChunksPerCta) * p.grid,
                                              items / spmm::kWcsrDynMinChunkItems, h->ws_slots / 2});
    if (chunks > p.grid) {
      p.grid = static_cast<int32_t>(chunks);
      p.dynamic = 1;
    }
  }
  p.status = h->d_status;
  p.wait_limit_ns = h->wait_limit_ns;
  cudaError_t e = w64 ? spmm::launch_wcsr64(h->tm_C, p, in_bf16, out_bf16, s) : spmm::launch_wcsr(p, in_bf16, out_bf16, s);
  if (e != cudaSuccess) return cuda_fail(e, "WCSR kernel launch");
  return SPMM_OK;
}

}  // namespace

extern "C" {

const char *spmm_status_str(spmm_status s) {
  switch (s) {
    case SPMM_OK: return "SPMM_OK";
    case SPMM_ERR_INVALID_ARG: return "SPMM_ERR_INVALID_ARG";
    case SPMM_ERR_UNSUPPORTED: return "SPMM_ERR_UNSUPPORTED";
    case SPMM_ERR_CUDA: return "SPMM_ERR_CUDA";
    case SPMM_ERR_OOM: return "SPMM_ERR_OOM";
    case SPMM_ERR_TIMEOUT: return "SPMM_ERR_TIMEOUT";
    case SPMM_ERR_DEVICE_CHECK: return "SPMM_ERR_DEVICE_CHECK";
  }
  return "unknown spmm_status";
}

const char *spmm_last_error(void) { return g_last_error.c_str(); }

spmm_status spmm_bcsr_convert(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx, const void *vals,
                              int b_row, int b_col, int64_t *n_blocks, int64_t *block_row_ptr, int32_t *block_col_idx,
                              uint16_t *blocks) {
  spmm_handle dummy;
  spmm_status st = check_common(&dummy, m, k, row_ptr, col_idx, vals, SPMM_BF16, SPMM_F32, b_row, b_col);
  if (st != SPMM_OK) return st;
  if (!n_blocks) return fail(SPMM_ERR_INVALID_ARG, "n_blocks is NULL");
  HostFormat f;
  spmm::build_bcsr(m, k, row_ptr, col_idx, block_col_idx && blocks ? static_cast<const uint16_t *>(vals) : nullptr,
                   b_row, b_col, f);
  *n_blocks = f.n_units;
  if (!block_col_idx) return SPMM_OK;
  if (block_row_ptr) std::memcpy(block_row_ptr, f.ptr.data(), f.ptr.size() * sizeof(int64_t));
  if (!f.idx.empty()) std::memcpy(block_col_idx, f.idx.data(), f.idx.size() * sizeof(int32_t));
  if (blocks && !f.vals.empty()) std::memcpy(blocks, f.vals.data(), f.vals.size() * 2);
  return SPMM_OK;
}

spmm_status spmm_wcsr_convert(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx, const void *vals,
                              int window_h, int col_pad, int64_t *p_total, int64_t *window_row_ptr,
                              int32_t *window_col_idx, uint16_t *values) {
  spmm_handle dummy;
  spmm_status st = check_common(&dummy, m, k, row_ptr, col_idx, vals, SPMM_BF16, SPMM_F32, window_h, col_pad);
  if (st != SPMM_OK) return st;
  if (!p_total) return fail(SPMM_ERR_INVALID_ARG, "p_total is NULL");
  HostFormat f;
  spmm::build_wcsr(m, k, row_ptr, col_idx, window_col_idx && values ? static_cast<const uint16_t *>(vals) : nullptr,
                   window_h, col_pad, f);
  *p_total = f.n_units;
  if (!window_col_idx) return SPMM_OK;
  if (window_row_ptr) std::memcpy(window_row_ptr, f.ptr.data(), f.ptr.size() * sizeof(int64_t));
  if (!f.idx.empty()) std::memcpy(window_col_idx, f.idx.data(), f.idx.size() * sizeof(int32_t));
  if (values && !f.vals.empty()) std::memcpy(values, f.vals.data(), f.vals.size() * 2);
  return SPMM_OK;
}

spmm_status spmm_bcsr_create(spmm_handle *out, int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                             const void *vals, spmm_dtype in_t, spmm_dtype out_t, int b_row, int b_col) {
  spmm_status st = check_common(out, m, k, row_ptr, col_idx, vals, in_t, out_t, b_row, b_col);
  if (st != SPMM_OK) return st;
  HostFormat f;
  spmm::build_bcsr(m, k, row_ptr, col_idx, static_cast<const uint16_t *>(vals), b_row, b_col, f);
  if (f.n_units * b_row >= (1ll << 31)) return fail(SPMM_ERR_UNSUPPORTED, "too many stored blocks");
  spmm_handle h = new spmm_handle_s;
  h->format = SPMM_FORMAT_BCSR;
  h->m = m;
  h->k = k;
  h->nnz = row_ptr[m];
  h->b_row = b_row;
  h->b_col = b_col;
  h->in_t = in_t;
  h->out_t = out_t;
  h->n_groups = static_cast<int64_t>(f.ptr.size()) - 1;
  h->n_units = f.n_units;
  h->stored = f.n_units * b_row * b_col;
  st = upload_common(h, f);
  if (st == SPMM_OK) st = build_bcsr_split(h, f.ptr);
  if (st == SPMM_OK && b_row == 64 && b_col == 64)
    st = encode_2d(&h->tm_vals, h->d_vals, in_t == SPMM_BF16, static_cast<uint64_t>(std::max<int64_t>(f.n_units, 1) * 64),
                   64, 64, 64, 64);
  if (st != SPMM_OK) {
    free_handle(h);
    return st;
  }
  *out = h;
  return SPMM_OK;
}

spmm_status spmm_wcsr_create(spmm_handle *out, int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                             const void *vals, spmm_dtype in_t, spmm_dtype out_t, int window_h, int col_pad) {
  spmm_status st = check_common(out, m, k, row_ptr, col_idx, vals, in_t, out_t, window_h, col_pad);
  if (st != SPMM_OK) return st;
  HostFormat f;
  spmm::build_wcsr(m, k, row_ptr, col_idx, static_cast<const uint16_t *>(vals), window_h, col_pad, f);
  if (f.n_units >= (1ll << 31)) return fail(SPMM_ERR_UNSUPPORTED, "too many packed columns");
  spmm_handle h = new spmm_handle_s;
  h->format = SPMM_FORMAT_WCSR;
  h->m = m;
  h->k = k;
  h->nnz = row_ptr[m];
  h->b_row = window_h;
  h->b_col = col_pad;
  h->in_t = in_t;
  h->out_t = out_t;
  h->n_groups = static_cast<int64_t>(f.ptr.size()) - 1;
  h->n_units = f.n_units;
  h->stored = f.n_units * window_h;
  st = upload_common(h, f);
  if (st == SPMM_OK && (window_h == 16 || window_h == 64)) st = build_stages(h, f.ptr, f.idx, f.vals);
  if (st != SPMM_OK) {
    free_handle(h);
    return st;
  }
  *out = h;
  return SPMM_OK;
}

spmm_status spmm_set_max_ctas(spmm_handle h, int32_t ctas) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  if (ctas < 0) return fail(SPMM_ERR_INVALID_ARG, "ctas must be >= 0");
  h->max_ctas = ctas;
  return SPMM_OK;
}

spmm_status spmm_set_schedule(spmm_handle h, int32_t schedule) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  if (schedule != SPMM_SCHEDULE_AUTO && schedule != SPMM_SCHEDULE_TILES && schedule != SPMM_SCHEDULE_SPLIT &&
      schedule != SPMM_SCHEDULE_DYNAMIC)
    return fail(SPMM_ERR_INVALID_ARG, "unknown schedule %d", schedule);
  if (schedule == SPMM_SCHEDULE_DYNAMIC) {
    if (h->format != SPMM_FORMAT_WCSR || h->b_row != 16)
      return fail(SPMM_ERR_UNSUPPORTED, "the dynamic schedule takes WCSR handles with window height 16");
    // two partial slots per chunk, for the most chunks any N can give
    const int64_t slots = 2ll * spmm::kWcsrDynChunksPerCta * spmm::kWcsrMaxCtasPerSm * std::max(h->num_sms, 1);
    if (slots > h->ws_slots) {
      float *ws = nullptr;
      spmm::PartialRec *rec = nullptr;
      if (cudaMalloc(&ws, slots * spmm::kWcsrSlotFloats * sizeof(float)) != cudaSuccess ||
          cudaMalloc(&rec, slots * sizeof(spmm::PartialRec)) != cudaSuccess) {
        cudaFree(ws);
        cudaGetLastError();
        return fail(SPMM_ERR_OOM, "cudaMalloc(dynamic-schedule workspace) failed");
      }
      cudaFree(h->d_ws);
      cudaFree(h->d_partials);
      h->d_ws = ws;
      h->d_partials = rec;
      h->ws_slots = slots;
    }
  }
  h->schedule = schedule;
  return SPMM_OK;
}

spmm_status spmm_wcsr_run_noalloc(const int64_t *window_row_ptr, const int32_t *window_col_idx, const void *values,
                                  int64_t m, int64_t k, int64_t p_total, spmm_dtype in_t, spmm_dtype out_t,
                                  const void *B, void *C, int64_t N, void *stream) {
  if (!window_row_ptr || !B || !C || (p_total > 0 && (!window_col_idx || !values)))
    return fail(SPMM_ERR_INVALID_ARG, "a device pointer is NULL");
  if (m < 0 || k < 0 || m >= (1ll << 31) || k >= (1ll << 31) || p_total < 0 || p_total >= (1ll << 31))
    return fail(SPMM_ERR_INVALID_ARG, "m, k, p_total must be in [0, 2^31)");
  if (in_t != SPMM_F16 && in_t != SPMM_BF16) return fail(SPMM_ERR_INVALID_ARG, "in_t must be F16 or BF16");
  if (out_t != SPMM_F32 && out_t != SPMM_BF16) return fail(SPMM_ERR_INVALID_ARG, "out_t must be F32 or BF16");
  if (N <= 0 || N >= (1ll << 31)) return fail(SPMM_ERR_INVALID_ARG, "N must be in (0, 2^31)");
  if (N % 8 != 0) return fail(SPMM_ERR_UNSUPPORTED, "N must be a multiple of 8 (16-byte rows of B)");
  if (N > 65535ll * 128) return fail(SPMM_ERR_UNSUPPORTED, "N above 65535 * 128 exceeds the launch grid");
  if (p_total % 16 != 0) return fail(SPMM_ERR_UNSUPPORTED, "p_total must be a multiple of 16 (column padding)");
  if ((reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C) | reinterpret_cast<uintptr_t>(values)) & 15)
    return fail(SPMM_ERR_UNSUPPORTED, "B, C and values must be 16-byte aligned");
  const int64_t n_windows = (m + 15) / 16;
  const int64_t max_stages = n_windows + p_total / 64;  // each window: ceil(P_w/64) <= P_w/64 + 1 stages
  if (max_stages > spmm::kNoallocMaxStages)
    return fail(SPMM_ERR_UNSUPPORTED,
                "problem needs up to %lld stages; the static scratch of spmm_wcsr_run_noalloc holds %lld "
                "(ceil(m/16) + p_total/64 must not exceed it)",
                static_cast<long long>(max_stages), static_cast<long long>(spmm::kNoallocMaxStages));
  if (m == 0) return SPMM_OK;
  int dev = 0, sms = 0, major = 0, minor = 0;
  CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "device attribute");
  CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "device attribute");
  CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "device attribute");
  if (major != 10 || minor != 3) return fail(SPMM_ERR_UNSUPPORTED, "the kernels need an sm_103 (GB300) device");
  spmm::WcsrParams p;
  std::memset(&p, 0, sizeof p);
  p.values = values;
  p.window_col_idx = window_col_idx;
  p.B = B;
  p.C = C;
  p.P_total = p_total;
  p.M = static_cast<int32_t>(m);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(k);
  p.wait_limit_ns = kDefaultWaitLimitNs;
  cudaError_t e = spmm::launch_wcsr_noalloc(p, window_row_ptr, n_windows, sms, in_t == SPMM_BF16,
                                            out_t == SPMM_BF16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "no-allocation WCSR launch");
  return SPMM_OK;
}

spmm_status spmm_run(spmm_handle h, const void *B, void *C, int64_t N, void *stream) {
  spmm_status st = check_run_args(h, B, C, N);
  if (st != SPMM_OK) return st;
  return run_device(h, B, C, N, static_cast<cudaStream_t>(stream));
}

spmm_status spmm_run_linear(spmm_handle h, const void *X, void *Y, int64_t N, void *stream) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  if (h->format != SPMM_FORMAT_BCSR) return fail(SPMM_ERR_UNSUPPORTED, "spmm_run_linear takes a BCSR handle");
  if (N <= 0 || N >= (1ll << 31)) return fail(SPMM_ERR_INVALID_ARG, "N must be in (0, 2^31)");
  if (!X || !Y) return fail(SPMM_ERR_INVALID_ARG, "X or Y is NULL");
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Y)) & 15)
    return fail(SPMM_ERR_UNSUPPORTED, "X and Y must be 16-byte aligned");
  spmm_status st = SPMM_OK;
  if (h->b_row != 64 || h->b_col != 64) return fail(SPMM_ERR_UNSUPPORTED, "the BCSR kernel takes 64 x 64 blocks");
  const bool in_bf16 = h->in_t == SPMM_BF16;
  const bool out_bf16 = h->out_t == SPMM_BF16;
  if (h->k % 8 != 0) return fail(SPMM_ERR_UNSUPPORTED, "k must be a multiple of 8 (16-byte rows of X)");
  if (h->m % (out_bf16 ? 8 : 4) != 0) return fail(SPMM_ERR_UNSUPPORTED, "m must make 16-byte rows of Y");
  if (!h->sm103) return fail(SPMM_ERR_UNSUPPORTED, "the kernels need an sm_103 (GB300) device");
  if (h->m == 0) return SPMM_OK;
  if (h->x_cached != X || h->nx_cached != N) {
    st = encode_x(&h->tm_X, X, in_bf16, static_cast<uint64_t>(N), static_cast<uint64_t>(std::max<int64_t>(h->k, 8)));
    if (st != SPMM_OK) return st;
    h->x_cached = X;
    h->nx_cached = N;
  }
  if (h->y_cached != Y || h->ny_cached != N) {
    st = encode_y(&h->tm_Y, Y, out_bf16, static_cast<uint64_t>(N), static_cast<uint64_t>(h->m));
    if (st != SPMM_OK) return st;
    h->y_cached = Y;
    h->ny_cached = N;
  }
  spmm::BcsrParams p;
  std::memset(&p, 0, sizeof p);
  p.block_row_ptr = h->d_ptr;
  p.block_col_idx = h->d_idx;
  p.blocks = h->d_vals;
  p.B = X;
  p.C = Y;
  p.ldc = h->m;
  p.M = static_cast<int32_t>(h->m);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(h->k);
  p.n_block_rows = static_cast<int32_t>(h->n_groups);
  p.max_ctas = h->max_ctas;
  p.num_sms = std::max(h->num_sms, 1);
  p.status = h->d_status;
  p.wait_limit_ns = h->wait_limit_ns;
  cudaError_t e = spmm::launch_bcsr_linear(h->tm_vals, h->tm_X, h->tm_Y, p, in_bf16, out_bf16,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "BCSR linear kernel launch");
  return SPMM_OK;
}

spmm_status spmm_check(spmm_handle h, void *stream) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  CUDA_TRY(cudaMemcpyAsync(&word, h->d_status, sizeof word, cudaMemcpyDeviceToHost, s), "read status");
  CUDA_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  if (word) {
    CUDA_TRY(cudaMemsetAsync(h->d_status, 0, sizeof(uint32_t), s), "clear status");
    CUDA_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    if (word & spmm::kDevTimeout) return fail(SPMM_ERR_TIMEOUT, "a kernel's bounded wait ran out");
    return fail(SPMM_ERR_DEVICE_CHECK, "a kernel's index check failed (status 0x%x)", word);
  }
  return SPMM_OK;
}

spmm_status spmm_run_host(spmm_handle h, const void *B_host, void *C_host, int64_t N, void *stream) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  if (!B_host || !C_host) return fail(SPMM_ERR_INVALID_ARG, "B or C is NULL");
  if (N <= 0) return fail(SPMM_ERR_INVALID_ARG, "N must be positive");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bb = static_cast<size_t>(h->k) * N * elem_size(h->in_t);
  const size_t cb = static_cast<size_t>(h->m) * N * elem_size(h->out_t);
  if (!h->d_bstage || bb > h->bstage_bytes) {
    cudaFree(h->d_bstage);
    h->d_bstage = nullptr;
    h->bstage_bytes = 0;
    CUDA_TRY(cudaMalloc(&h->d_bstage, std::max<size_t>(bb, 16)), "cudaMalloc(B staging)");
    h->bstage_bytes = std::max<size_t>(bb, 16);
  }
  if (!h->d_cstage || cb > h->cstage_bytes) {
    cudaFree(h->d_cstage);
    h->d_cstage = nullptr;
    h->cstage_bytes = 0;
    CUDA_TRY(cudaMalloc(&h->d_cstage, std::max<size_t>(cb, 16)), "cudaMalloc(C staging)");
    h->cstage_bytes = std::max<size_t>(cb, 16);
  }
  void *dB = h->d_bstage;
  void *dC = h->d_cstage;
  spmm_status st = check_run_args(h, dB, dC, N);
  if (st != SPMM_OK) return st;
  if (bb) CUDA_TRY(cudaMemcpyAsync(dB, B_host, bb, cudaMemcpyHostToDevice, s), "copy B to device");
  st = run_device(h, dB, dC, N, s);
  if (st != SPMM_OK) return st;
  if (cb) CUDA_TRY(cudaMemcpyAsync(C_host, dC, cb, cudaMemcpyDeviceToHost, s), "copy C to host");
  return spmm_check(h, stream);
}

spmm_status spmm_destroy(spmm_handle h) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_handle(h);
  return SPMM_OK;
}

spmm_status spmm_format_info(spmm_handle h, spmm_info *info) {
  if (!h || !info) return fail(SPMM_ERR_INVALID_ARG, "handle or info is NULL");
  std::memset(info, 0, sizeof *info);
  info->format = h->format;
  info->b_row = h->b_row;
  info->b_col = h->b_col;
  info->m = h->m;
  info->k = h->k;
  info->nnz = h->nnz;
  info->n_groups = h->n_groups;
  info->n_units = h->n_units;
  info->stored = h->stored;
  info->padding = h->stored - h->nnz;
  info->idx_bytes = (h->n_groups + 1) * 8 + h->n_units * 4;
  info->val_bytes = h->stored * 2;
  if (h->format == SPMM_FORMAT_WCSR) {
    info->n_tasks = h->n_stages;
    info->split_cols = 64;
    // windows cut by a CTA boundary when the product has one column tile
    const int64_t g = wcsr_grid(h, 8);
    int64_t cut = 0;
    for (int64_t c = 1; c < g; ++c) {
      const int64_t f = h->n_stages * c / g;
      if (!h->stage_first[f]) ++cut;
    }
    info->n_split_windows = cut;
  } else {
    info->n_tasks = h->n_groups;
  }
  return SPMM_OK;
}

spmm_status spmm_export_format(spmm_handle h, int64_t *ptr_out, int32_t *idx_out, uint16_t *vals_out) {
  if (!h) return fail(SPMM_ERR_INVALID_ARG, "handle is NULL");
  CUDA_TRY(cudaSetDevice(h->device), "cudaSetDevice");
  CUDA_TRY(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  if (ptr_out)
    CUDA_TRY(cudaMemcpy(ptr_out, h->d_ptr, (h->n_groups + 1) * sizeof(int64_t), cudaMemcpyDeviceToHost), "download ptr");
  if (idx_out && h->n_units)
    CUDA_TRY(cudaMemcpy(idx_out, h->d_idx, h->n_units * sizeof(int32_t), cudaMemcpyDeviceToHost), "download idx");
  if (vals_out && h->stored)
    CUDA_TRY(cudaMemcpy(vals_out, h->d_vals, h->stored * 2, cudaMemcpyDeviceToHost), "download values");
  return SPMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- self test
namespace spmm {
namespace {
__global__ void wait_selftest_kernel(uint32_t *status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  // Nothing arrives: the phase never completes and the bounded wait gives up.
  if (!mbar_wait(b, 0, limit_ns)) atomicOr(status, kDevTimeout);
}
}  // namespace

cudaError_t launch_wait_selftest(uint32_t *status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 1, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}
}  // namespace spmm

extern "C" spmm_status spmm_selftest_wait_timeout(int64_t timeout_ns, void *stream, int32_t *dev_status) {
  if (!dev_status) return fail(SPMM_ERR_INVALID_ARG, "dev_status is NULL");
  if (timeout_ns < 1000 || timeout_ns > 10000000000ll) return fail(SPMM_ERR_INVALID_ARG, "timeout_ns out of range");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t *d = nullptr;
  CUDA_TRY(cudaMalloc(&d, sizeof(uint32_t)), "cudaMalloc(status)");
  uint32_t word = 0;
  cudaError_t e = cudaMemsetAsync(d, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = spmm::launch_wait_selftest(d, static_cast<uint64_t>(timeout_ns), s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&word, d, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  cudaFree(d);
  if (e != cudaSuccess) return cuda_fail(e, "wait self test");
  *dev_status = (word & spmm::kDevTimeout) ? SPMM_ERR_TIMEOUT : SPMM_OK;
  return SPMM_OK;
}

// ---------------------------------------------------------------- L2 read probe
namespace spmm {
namespace {
// Every thread streams 16-byte loads that bypass L1 (ld.global.cg) with four
// in flight, over `passes` back-to-back sweeps of the buffer taken as one
// sequence (so a small buffer still gives every thread a long stream); the
// XOR of the data decides a store nobody expects, so the loads cannot be
// dropped.
__global__ void __launch_bounds__(512) l2_read_kernel(const uint4 *__restrict__ buf, int64_t n16, int32_t passes,
                                                      uint4 *sink) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t total = n16 * passes;
  const int64_t step = stride % n16;  // index advance per stride, wrapped
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t j = i % n16;
  auto next = [&](int64_t x) {
    x += step;
    return x >= n16 ? x - n16 : x;
  };
  uint32_t acc = 0;
  for (; i + 3 * stride < total; i += 4 * stride) {
    const int64_t j1 = next(j), j2 = next(j1), j3 = next(j2);
    const uint4 a = __ldcg(buf + j), b = __ldcg(buf + j1), c = __ldcg(buf + j2), d = __ldcg(buf + j3);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    j = next(j3);
  }
  for (; i < total; i += stride) {
    const uint4 a = __ldcg(buf + j);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
    j = next(j);
  }
  if (acc == 0x9E3779B9u && threadIdx.x == blockDim.x - 1) sink[0] = make_uint4(acc, blockIdx.x, 0, 0);
}
}  // namespace
}  // namespace spmm

extern "C" spmm_status spmm_wcsr_noalloc_check(void *stream) {
  uint32_t word = 0;
  cudaError_t e = spmm::wcsr_noalloc_take_status(&word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reading the no-allocation status word");
  if (word & spmm::kDevIndex)
    return fail(SPMM_ERR_DEVICE_CHECK, "window_row_ptr failed the device check; no work was listed");
  if (word & spmm::kDevTimeout) return fail(SPMM_ERR_TIMEOUT, "a bounded wait ran out in the WCSR kernel");
  return SPMM_OK;
}

extern "C" spmm_status spmm_probe_l2_read(const void *buf, int64_t bytes, int32_t passes, void *sink,
                                          void *stream) {
  if (!buf || !sink) return fail(SPMM_ERR_INVALID_ARG, "buf or sink is NULL");
  if (bytes <= 0 || bytes % 16 != 0) return fail(SPMM_ERR_INVALID_ARG, "bytes must be positive and a multiple of 16");
  if (passes < 1) return fail(SPMM_ERR_INVALID_ARG, "passes < 1");
  if ((reinterpret_cast<uintptr_t>(buf) | reinterpret_cast<uintptr_t>(sink)) % 16 != 0)
    return fail(SPMM_ERR_INVALID_ARG, "buf and sink must be 16-byte aligned");
  int dev = 0, sms = 0;
  CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
  spmm::l2_read_kernel<<<4 * sms, 512, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(buf), bytes / 16, passes, static_cast<uint4 *>(sink));
  CUDA_TRY(cudaGetLastError(), "L2 read probe launch");
  return SPMM_OK;
}
