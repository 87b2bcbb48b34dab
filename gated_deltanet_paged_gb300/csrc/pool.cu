// pool.cu -- whole-row utilities on a state pool: bit-exact row copies and
// zeroed rows.
//
// "gdn-prefix-cache" (the gaudi-cookbook fix write-up), §The fix: the state a
// cached block needs is kept as a checkpoint in that block's page and moved as
// bit-exact row copies -- after a step whose tokens end on a block boundary
// the request's own row is copied into the block, and before a step that
// starts from a hit the block is copied back; new blocks and rows are zeroed,
// so that no non-finite value outlives the step that produced it.  On the
// paged pool of this library the same two moves are a copy of row src to row
// dst (a copy-on-write fork of a shared page) and a zero fill of a new page.
//
// Both kernels treat a row as row_bytes of opaque data (any element type),
// moved in 16-byte pieces with streaming loads and stores: HBM-bound.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kPiecesPerThread = 8;                            // 16-byte pieces
constexpr int64_t kSliceBytes = kThreads * kPiecesPerThread * 16;  // one CTA's share of a row: 32 KB

struct RowArgs {
  uint8_t* pool;
  int64_t row_bytes;
  int64_t stride_bytes;
  const int32_t* src_rows;  // copy: source rows; zero: nullptr
  const int32_t* dst_rows;
  int32_t n;
  int32_t num_rows;
  int32_t* err_word;
};

// blockIdx.y: the pair; blockIdx.x: a 32 KB slice of the row.
__global__ void __launch_bounds__(kThreads) rows_kernel(const RowArgs a) {
  const int i = blockIdx.y;
  const int32_t dst = a.dst_rows[i];
  const int32_t src = a.src_rows ? a.src_rows[i] : 0;
  if (dst < 0 || (a.src_rows && src < 0)) return;  // -1 skips the pair
  if (dst >= a.num_rows || (a.src_rows && src >= a.num_rows)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) gdn::record_error(a.err_word, GDN_DEVERR_PAGE_ID, i);
    return;
  }
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSliceBytes;
  uint4* d = reinterpret_cast<uint4*>(a.pool + dst * a.stride_bytes + begin);
  const int64_t pieces = min(kSliceBytes, a.row_bytes - begin) / 16;
  if (a.src_rows) {
    const uint4* s = reinterpret_cast<const uint4*>(a.pool + src * a.stride_bytes + begin);
    uint4 x[kPiecesPerThread];
#pragma unroll
    for (int k = 0; k < kPiecesPerThread; ++k) {
      const int64_t p = threadIdx.x + static_cast<int64_t>(k) * kThreads;
      if (p < pieces) x[k] = __ldcs(s + p);
    }
#pragma unroll
    for (int k = 0; k < kPiecesPerThread; ++k) {
      const int64_t p = threadIdx.x + static_cast<int64_t>(k) * kThreads;
      if (p < pieces) __stcs(d + p, x[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPiecesPerThread; ++k) {
      const int64_t p = threadIdx.x + static_cast<int64_t>(k) * kThreads;
      if (p < pieces) __stcs(d + p, make_uint4(0u, 0u, 0u, 0u));
    }
  }
}

int launch_rows(void* pool, int64_t row_bytes, int64_t stride_bytes, const int32_t* src_rows,
                const int32_t* dst_rows, int32_t n, int32_t num_rows, int32_t* err_word, void* stream) {
  if (n < 0 || num_rows < 1 || row_bytes <= 0 || row_bytes % 16 != 0 || stride_bytes < row_bytes ||
      stride_bytes % 16 != 0)
    return GDN_ERR_INVALID_ARGUMENT;
  if (n == 0) return GDN_OK;
  if (!pool || !dst_rows || !gdn_host::aligned16(pool)) return GDN_ERR_INVALID_ARGUMENT;
  const int64_t slices = (row_bytes + kSliceBytes - 1) / kSliceBytes;
  if (slices > 0x7FFFFFFF || n > 65535) return GDN_ERR_UNSUPPORTED;
  int rc = gdn_host::check_device(nullptr);
  if (rc != GDN_OK) return rc;
  RowArgs a{static_cast<uint8_t*>(pool), row_bytes, stride_bytes, src_rows, dst_rows, n, num_rows, err_word};
  rows_kernel<<<dim3(static_cast<unsigned>(slices), static_cast<unsigned>(n)), kThreads, 0,
                static_cast<cudaStream_t>(stream)>>>(a);
  return gdn_host::launch_status();
}

}  // namespace

extern "C" int gdn_pool_copy_rows(void* pool, int64_t row_bytes, int64_t pool_row_stride_bytes,
                                  const int32_t* src_rows, const int32_t* dst_rows, int32_t n, int32_t num_rows,
                                  int32_t* err_word, void* stream) {
  if (n > 0 && !src_rows) return GDN_ERR_INVALID_ARGUMENT;
  return launch_rows(pool, row_bytes, pool_row_stride_bytes, src_rows, dst_rows, n, num_rows, err_word, stream);
}

extern "C" int gdn_pool_zero_rows(void* pool, int64_t row_bytes, int64_t pool_row_stride_bytes, const int32_t* rows,
                                  int32_t n, int32_t num_rows, int32_t* err_word, void* stream) {
  return launch_rows(pool, row_bytes, pool_row_stride_bytes, nullptr, rows, n, num_rows, err_word, stream);
}
