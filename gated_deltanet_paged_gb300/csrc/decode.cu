// decode.cu -- single-token paged GDN decode ("flashinfer.gdn_paged",
// gated_delta_rule_decode_paged and the decode paragraph).
//
// For every (sequence b, head h) the 128 x 128 state (fp32, or bf16 in a bf16
// pool: carried in fp32 and rounded to the nearest bf16 on the way out) is read
// once from its read row, updated and written once to its write row:
//     S' = e S + beta (v - e S k) k^T,   o = scale S' q = scale (e S q + d (k.q))
// with e = exp(g) and d = beta (v - e S k) per state row.  Both kernels are a
// streaming read-update-write bound by HBM bandwidth: 16-byte coalesced,
// evict-first loads and streaming stores, all 16 loads of a thread in flight
// before any arithmetic.  In the fp32 kernel each warp owns 16 rows, each
// lane one float4 of every row, and two 4-warp CTAs share a state (rows 0-63
// and 64-127), which spreads a small batch over more SMs; the 32 dot products
// a warp needs (S k and S q of its 16 rows) are reduced together by a
// transpose reduction (31 shuffles instead of 160).  The bf16 kernel is laid
// out below.
//
// Both kernels are launched as programmatic dependents of the kernel before
// them on the stream: a CTA waits (griddepcontrol.wait) until that kernel has
// finished and its writes are visible before it reads anything, so the order
// of the stream is kept, while the launch itself overlaps the previous
// kernel's tail -- a step of many layers' decodes spends less time between
// kernels.
#include <math.h>

#include "common.cuh"

namespace {

constexpr int kThreads = 128;
constexpr int kRowsPerWarp = 16;
static_assert(kThreads / 32 * kRowsPerWarp * 2 == gdn::kDimV, "two CTAs cover one 128-row state");

// Programmatic dependent launch: wait for the previous kernel on the stream to
// complete (its memory visible), then let the next one begin launching.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
}

struct DecodeArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  __nv_bfloat16* o;
  void* pool;  // float (decode_f32_kernel) or __nv_bfloat16 (decode_bf16_kernel) elements
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

// The rows a (sequence b) reads and writes, from the explicit slots or the
// page table: false when the CTA has nothing to do (a bad entry, recorded).
__device__ __forceinline__ bool resolve_rows(const DecodeArgs& a, int b, int& in_row, int& out_row) {
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
      return false;
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
    return false;
  }
  return true;
}

// fp32 pool: two CTAs per state, each 4 warps x 16 rows, each lane one float4
// of every row.
__global__ void __launch_bounds__(kThreads, 4) decode_f32_kernel(const DecodeArgs a) {
  pdl_enter();
  const int bh = blockIdx.x >> 1;  // blockIdx.x & 1: which 64 rows of the state
  const int b = bh / a.H, h = bh % a.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int in_row, out_row;
  if (!resolve_rows(a, b, in_row, out_row)) return;

  const int r0 = (blockIdx.x & 1) * 64 + warp * kRowsPerWarp;
  const int64_t head_off = static_cast<int64_t>(h) * gdn::kDimV * gdn::kDimK;

  float* const pool = static_cast<float*>(a.pool);
  float4 s[kRowsPerWarp];
  if (in_row >= 0) {
    const float* src = pool + in_row * a.row_stride + head_off + r0 * gdn::kDimK + 4 * lane;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) s[i] = __ldcs(reinterpret_cast<const float4*>(src + i * gdn::kDimK));
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
    float* dst = pool + out_row * a.row_stride + head_off + r0 * gdn::kDimK + 4 * lane;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const float di = __shfl_sync(0xffffffffu, d, 2 * i);
      float4 n;
      n.x = e * s[i].x + di * kk[0];
      n.y = e * s[i].y + di * kk[1];
      n.z = e * s[i].z + di * kk[2];
      n.w = e * s[i].w + di * kk[3];
      __stcs(reinterpret_cast<float4*>(dst + i * gdn::kDimK), n);
    }
  }
}

// bf16 pool.  The 32 KB state comes into shared memory by one bulk copy, so
// that the bytes in flight cost no registers (five CTAs per SM, 160 KB of
// state reads in flight).  A 256-byte bf16 row is half a warp of 16-byte
// pieces, so a warp takes two rows per step: lane l (p = l & 15, half
// c = l >> 4) reads elements 8p..8p+7 of rows 2i+c, i < 16, 32 rows per warp
// and four warps per state, once for the dot products and once for the
// update, widening to fp32 as it goes.  A thread has twice the fp32 arithmetic
// of the fp32 kernel's for the same bytes, enough to show against HBM, so the
// products and sums run as paired fp32 operations (fma.rn.f32x2, each half
// rounded like a scalar fma).
constexpr int kBf16Threads = 128;
constexpr int kBf16RowsPerWarp = 32;
static_assert(kBf16Threads / 32 * kBf16RowsPerWarp == gdn::kDimV, "one CTA covers one 128-row state");

__device__ __forceinline__ void widen8(const uint4& u, float2 (&f)[4]) {
  f[0] = gdn::unpack_bf162(u.x), f[1] = gdn::unpack_bf162(u.y);
  f[2] = gdn::unpack_bf162(u.z), f[3] = gdn::unpack_bf162(u.w);
}

__device__ __forceinline__ float dot8(const float2 (&x)[4], const float2 (&w)[4]) {
  float2 r = __fmul2_rn(x[0], w[0]);
#pragma unroll
  for (int j = 1; j < 4; ++j) r = __ffma2_rn(x[j], w[j], r);
  return r.x + r.y;
}

constexpr uint32_t kBf16StateBytes = gdn::kDimV * gdn::kDimK * 2;  // 32 KB

// One bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global into shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   gdn::smem_u32(smem_dst)),
               "l"(src), "r"(bytes), "r"(gdn::smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(kBf16Threads, 5) decode_bf16_kernel(const DecodeArgs a) {
  __shared__ alignas(128) uint4 st[kBf16StateBytes / 16];
  __shared__ uint64_t bar;
  pdl_enter();
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = lane & 15, c = lane >> 4;
  int in_row, out_row;
  if (!resolve_rows(a, b, in_row, out_row)) return;

  const int64_t head_off = static_cast<int64_t>(h) * gdn::kDimV * gdn::kDimK;
  __nv_bfloat16* const pool = static_cast<__nv_bfloat16*>(a.pool);
  // The whole 32 KB state in one bulk copy (a zero state is written in place).
  if (in_row >= 0) {
    if (tid == 0) {
      gdn::mbar_init(&bar, 1);
      gdn::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      gdn::mbar_arrive_expect_tx(&bar, kBf16StateBytes);
      bulk_load(st, pool + in_row * a.row_stride + head_off, kBf16StateBytes, &bar);
    }
  } else {
    for (int i = tid; i < static_cast<int>(kBf16StateBytes / 16); i += kBf16Threads) st[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
  }

  float2 kk[4], qq[4];
  widen8(*reinterpret_cast<const uint4*>(a.k + static_cast<int64_t>(bh) * gdn::kDimK + 8 * p), kk);
  widen8(*reinterpret_cast<const uint4*>(a.q + static_cast<int64_t>(bh) * gdn::kDimK + 8 * p), qq);
  float kq = dot8(kk, qq);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, m);  // both halves hold all of k, q
  const int r0 = warp * kBf16RowsPerWarp;
  const int row = r0 + 2 * p + c;  // the row this lane finishes
  const float e = expf(a.g[bh]);
  const float be = a.beta[bh];
  const float myv = __bfloat162float(a.v[static_cast<int64_t>(bh) * gdn::kDimV + row]);

  if (in_row >= 0) {
    // every lane of a warp takes the same decision, so no shuffle below runs
    // with part of a warp
    const bool landed = __all_sync(0xffffffffu, gdn::mbar_wait(&bar, 0));
    if (!landed) {
      if (lane == 0) gdn::record_error(a.err_word, GDN_DEVERR_TIMEOUT, b);
      gdn::mbar_wait(&bar, 0);  // the copy writes this CTA's shared memory: let it finish (bounded)
      return;
    }
  }
  // this lane's piece of row r0 + 2i + c: srow[32 i] (two 256-byte rows per step)
  const uint4* srow = st + (r0 + c) * 16 + p;

  // 32 partial dot products per lane, value 2i = (S k) and 2i+1 = (S q) of
  // step i, summed over the 16 lanes of each half by a transpose reduction
  // (lane bit 3 pairs value bit 4, ..., lane bit 0 pairs value bit 1).  The
  // first step is taken as the values are formed, so that 16 are live at once.
  float x[16];
  {
    const bool upper = (lane & 8) != 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // steps j and 8 + j: values 2j, 2j + 1 and 2j + 16, 2j + 17
      float2 lo[4], hi[4];
      widen8(srow[32 * j], lo);
      widen8(srow[32 * (8 + j)], hi);
      const float k0 = dot8(lo, kk), k1 = dot8(hi, kk), q0 = dot8(lo, qq), q1 = dot8(hi, qq);
      x[2 * j] = (upper ? k1 : k0) + __shfl_xor_sync(0xffffffffu, upper ? k0 : k1, 8);
      x[2 * j + 1] = (upper ? q1 : q0) + __shfl_xor_sync(0xffffffffu, upper ? q0 : q1, 8);
    }
  }
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 2 * m; ++i) {
      const float send = upper ? x[i] : x[i + 2 * m];
      const float keep = upper ? x[i + 2 * m] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  // x[0] = (S k), x[1] = (S q) of step p in this half, i.e. of row r0 + 2p + c
  const float d = be * (myv - e * x[0]);
  a.o[static_cast<int64_t>(bh) * gdn::kDimV + row] = __float2bfloat16_rn(a.scale * (e * x[1] + d * kq));

  if (out_row >= 0) {
    __nv_bfloat16* dst = pool + out_row * a.row_stride + head_off + (r0 + c) * gdn::kDimK + 8 * p;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float di = __shfl_sync(0xffffffffu, d, (lane & 16) | i);
      float2 f[4];
      widen8(srow[32 * i], f);
      const float2 e2 = make_float2(e, e), d2 = make_float2(di, di);
      float2 n[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) n[j] = __ffma2_rn(e2, f[j], __fmul2_rn(d2, kk[j]));
      uint4 u;
      u.x = gdn::pack_bf162(n[0].x, n[0].y);  // nearest bf16, ties to even
      u.y = gdn::pack_bf162(n[1].x, n[1].y);
      u.z = gdn::pack_bf162(n[2].x, n[2].y);
      u.w = gdn::pack_bf162(n[3].x, n[3].y);
      __stcs(reinterpret_cast<uint4*>(dst + i * 2 * gdn::kDimK), u);
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
  if (static_cast<int64_t>(batch) * H > 0x3FFFFFFF) return GDN_ERR_UNSUPPORTED;  // two fp32 CTAs per state
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
  cudaLaunchConfig_t cfg = {};  // programmatic dependent launch (see the top of this file)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  if (state_dtype == GDN_STATE_BF16) {
    // five 32 KB states per SM: ask for the largest shared-memory carveout
    static std::atomic<uint64_t> carveout_set{0};
    const int rc2 = gdn_host::func_attr_once(decode_bf16_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared, carveout_set);
    if (rc2 != GDN_OK) return rc2;
    cfg.gridDim = dim3(batch * H);
    cfg.blockDim = dim3(kBf16Threads);
    cudaLaunchKernelEx(&cfg, decode_bf16_kernel, a);
  } else {
    cfg.gridDim = dim3(2 * batch * H);
    cfg.blockDim = dim3(kThreads);
    cudaLaunchKernelEx(&cfg, decode_f32_kernel, a);
  }
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
