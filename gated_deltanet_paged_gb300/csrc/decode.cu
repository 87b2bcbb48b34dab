// decode.cu -- single-token paged GDN decode ("flashinfer.gdn_paged",
// gated_delta_rule_decode_paged and the decode paragraph).
//
// For every (sequence b, head h) the 128 x 128 state (fp32, or bf16 in a bf16
// pool: carried in fp32 and rounded to the nearest bf16 on the way out) is read
// once from its read row, updated and written once to its write row:
//     S' = e S + beta (v - e S k) k^T,   o = scale S' q = scale (e S q + d (k.q))
// with e = exp(g) and d = beta (v - e S k) per state row.  The kernel is a
// streaming read-update-write bound by HBM bandwidth: each warp owns 16 rows,
// each lane one float4 of every row (16-byte coalesced, evict-first loads and
// streaming stores, all 16 loads in flight before any arithmetic); the 32 dot
// products a warp needs (S k and S q of its 16 rows) are reduced together by
// a transpose reduction (31 shuffles instead of 160).
#include <math.h>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 16;
static_assert(kThreads / 32 * kRowsPerWarp == gdn::kDimV, "one CTA covers one 128-row state");

struct DecodeArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  __nv_bfloat16* o;
  void* pool;  // float or __nv_bfloat16 elements (the kernel's template argument)
  int64_t row_stride;
  int32_t H;
  int32_t num_pages;
  int32_t page_size;
  float scale;
  const int32_t* in_rows;  // explicit rows (slots) or nullptr: derive from the page table
  const int32_t* out_rows;
  const int32_t* indptr;
  const int32_t* pages;
  const int32_t* last_len;
  int32_t* err_word;
};

// After the call lane l holds the warp-wide sum of x[l].
__device__ __forceinline__ float transpose_reduce32(float (&x)[32], int lane) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = upper ? x[i] : x[i + m];
      const float keep = upper ? x[i + m] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  return x[0];
}

__device__ __forceinline__ void bf16x4(const __nv_bfloat16* p, float (&f)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = gdn::unpack_bf162(u.x), b = gdn::unpack_bf162(u.y);
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

// Four consecutive state values of one row: 16 bytes of fp32 or 8 of bf16.
__device__ __forceinline__ float4 load4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
  const float2 a = gdn::unpack_bf162(u.x), b = gdn::unpack_bf162(u.y);
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float* p, float4 x) { __stcs(reinterpret_cast<float4*>(p), x); }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 x) {
  __stcs(reinterpret_cast<uint2*>(p), make_uint2(gdn::pack_bf162(x.x, x.y), gdn::pack_bf162(x.z, x.w)));
}

template <typename St>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs a) {
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int in_row, out_row;
  bool bad = false;
  int kind = 0;
  if (a.in_rows) {
    in_row = a.in_rows[b];
    out_row = a.out_rows[b];
  } else {
    const int32_t i0 = a.indptr[b], i1 = a.indptr[b + 1];
    const int32_t lpl = a.last_len[b];
    if (i1 - i0 < 1) {
      if (threadIdx.x == 0) gdn::record_error(a.err_word, GDN_DEVERR_PAGE_TABLE, b);
      return;
    }
    out_row = a.pages[i1 - 1];
    in_row = (lpl == 1) ? (i1 - i0 >= 2 ? a.pages[i1 - 2] : -1) : out_row;
    if (a.err_word) {
      if (lpl < 1 || lpl > a.page_size) bad = true, kind = GDN_DEVERR_PAGE_TABLE;
      else if (in_row < 0) bad = true, kind = GDN_DEVERR_NO_PREV_TOKEN;
    }
  }
  if (a.err_word && !bad && (in_row < -1 || in_row >= a.num_pages || out_row < -1 || out_row >= a.num_pages))
    bad = true, kind = GDN_DEVERR_PAGE_ID;
  if (bad) {
    if (threadIdx.x == 0) gdn::record_error(a.err_word, kind, b);
    return;
  }

  const int r0 = warp * kRowsPerWarp;
  const int64_t head_off = static_cast<int64_t>(h) * gdn::kDimV * gdn::kDimK;

  St* const pool = static_cast<St*>(a.pool);
  float4 s[kRowsPerWarp];
  if (in_row >= 0) {
    const St* src = pool + in_row * a.row_stride + head_off + r0 * gdn::kDimK + 4 * lane;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) s[i] = load4(src + i * gdn::kDimK);
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  float kk[4], qq[4];
  bf16x4(a.k + static_cast<int64_t>(bh) * gdn::kDimK + 4 * lane, kk);
  bf16x4(a.q + static_cast<int64_t>(bh) * gdn::kDimK + 4 * lane, qq);
  float kq = kk[0] * qq[0] + kk[1] * qq[1] + kk[2] * qq[2] + kk[3] * qq[3];
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, m);
  const float e = expf(a.g[bh]);
  const float be = a.beta[bh];
  const float myv = __bfloat162float(a.v[static_cast<int64_t>(bh) * gdn::kDimV + r0 + (lane >> 1)]);

  float x[32];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    x[2 * i] = s[i].x * kk[0] + s[i].y * kk[1] + s[i].z * kk[2] + s[i].w * kk[3];
    x[2 * i + 1] = s[i].x * qq[0] + s[i].y * qq[1] + s[i].z * qq[2] + s[i].w * qq[3];
  }
  // lane 2i: (S k) of row r0+i; lane 2i+1: (S q) of row r0+i.
  const float red = transpose_reduce32(x, lane);
  const float d = be * (myv - e * red);                 // valid in even lanes
  const float d_row = __shfl_sync(0xffffffffu, d, lane & ~1);
  if (lane & 1)
    a.o[static_cast<int64_t>(bh) * gdn::kDimV + r0 + (lane >> 1)] =
        __float2bfloat16_rn(a.scale * (e * red + d_row * kq));

  if (out_row >= 0) {
    St* dst = pool + out_row * a.row_stride + head_off + r0 * gdn::kDimK + 4 * lane;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const float di = __shfl_sync(0xffffffffu, d, 2 * i);
      float4 n;
      n.x = e * s[i].x + di * kk[0];
      n.y = e * s[i].y + di * kk[1];
      n.z = e * s[i].z + di * kk[2];
      n.w = e * s[i].w + di * kk[3];
      store4(dst + i * gdn::kDimK, n);
    }
  }
}

}  // namespace

extern "C" int gdn_gated_delta_rule_decode_paged_ex(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                                    const float* g, const float* beta, gdn_bf16* o, int32_t batch,
                                                    int32_t H, int32_t K, int32_t V, float scale, void* state_pool,
                                                    int32_t state_dtype, int32_t num_pages,
                                                    const int32_t* page_indices, const int32_t* page_indptr,
                                                    const int32_t* last_page_len, const gdn_decode_slots* slots,
                                                    int32_t* err_word, void* stream) {
  if (batch < 0 || H < 1 || num_pages < 1) return GDN_ERR_INVALID_ARGUMENT;
  if (state_dtype != GDN_STATE_F32 && state_dtype != GDN_STATE_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (K != gdn::kDimK || V != gdn::kDimV) return GDN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !g || !beta || !o || !state_pool) return GDN_ERR_INVALID_ARGUMENT;
  if (slots) {
    if (!slots->initial_state_indices || !slots->output_state_indices) return GDN_ERR_INVALID_ARGUMENT;
  } else if (!page_indices || !page_indptr || !last_page_len) {
    return GDN_ERR_INVALID_ARGUMENT;
  }
  using gdn_host::aligned16;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(state_pool) ||
      !aligned16(g) || !aligned16(beta))
    return GDN_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(batch) * H > 0x7FFFFFFF) return GDN_ERR_UNSUPPORTED;
  if (batch == 0) return GDN_OK;
  int rc = gdn_host::check_device(nullptr);
  if (rc != GDN_OK) return rc;

  DecodeArgs a;
  a.q = reinterpret_cast<const __nv_bfloat16*>(q);
  a.k = reinterpret_cast<const __nv_bfloat16*>(k);
  a.v = reinterpret_cast<const __nv_bfloat16*>(v);
  a.g = g;
  a.beta = beta;
  a.o = reinterpret_cast<__nv_bfloat16*>(o);
  a.pool = state_pool;
  a.row_stride = static_cast<int64_t>(H) * V * K;
  a.H = H;
  a.num_pages = num_pages;
  a.page_size = 0x7FFFFFFF;  // the decode rows do not depend on page_size; lengths are only range-checked >= 1
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(K));
  a.in_rows = slots ? slots->initial_state_indices : nullptr;
  a.out_rows = slots ? slots->output_state_indices : nullptr;
  a.indptr = page_indptr;
  a.pages = page_indices;
  a.last_len = last_page_len;
  a.err_word = err_word;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (state_dtype == GDN_STATE_BF16)
    decode_kernel<__nv_bfloat16><<<batch * H, kThreads, 0, st>>>(a);
  else
    decode_kernel<float><<<batch * H, kThreads, 0, st>>>(a);
  return gdn_host::launch_status();
}

extern "C" int gdn_gated_delta_rule_decode_paged(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                                 const float* g, const float* beta, gdn_bf16* o, int32_t batch,
                                                 int32_t H, int32_t K, int32_t V, float scale, float* state_pool,
                                                 int32_t num_pages, const int32_t* page_indices,
                                                 const int32_t* page_indptr, const int32_t* last_page_len,
                                                 const gdn_decode_slots* slots, int32_t* err_word, void* stream) {
  return gdn_gated_delta_rule_decode_paged_ex(q, k, v, g, beta, o, batch, H, K, V, scale, state_pool, GDN_STATE_F32,
                                              num_pages, page_indices, page_indptr, last_page_len, slots, err_word,
                                              stream);
}
