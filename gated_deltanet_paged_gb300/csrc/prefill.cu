// prefill.cu -- chunked paged GDN prefill on tcgen05 tensor cores.
//
// "flashinfer.gdn_paged": chunk_gated_delta_rule_paged, the prefill bullets,
// the 64-token left-padding paragraph, and "Slot arguments of
// chunk_gated_delta_rule" (read / final / checkpoint rows, -1 = zero state or
// skip, checkpoints at absolute positions (prefix + n) % N == 0).
//
// Method (gated delta rule, chunked).  Per (sequence, head) chain and 64-token
// chunk with rows t = 0..63, cumulative gate G_t = g_0 + ... + g_t (padded
// rows have g = beta = 0 and k = v = 0 in effect, so they are the identity),
// gamma_t = exp(G_t), S0 the V x K state at the chunk start:
//   A[t][j] = beta_t exp(G_t - G_j) (k_t . k_j)      j < t   (strictly lower)
//   T       = (I + A)^-1                             (forward substitution)
//   W       = T diag(beta gamma) K,   U~ = T diag(beta) V
//   U       = U~ - W S0^T                            (the chunk's "new values")
//   O[t]    = scale (gamma_t S0 q_t + sum_{j<=t} exp(G_t - G_j)(q_t . k_j) U[j])
//   S1      = gamma_C S0 + U^T diag(exp(G_C - G_j)) K
// which equals the token-by-token recurrence exactly up to rounding.
//
// Mapping.  One CTA (256 threads) per chain, chains ordered by decreasing
// length so the longest start first.  Q, K, V tiles arrive by TMA (3-D tensor
// map over [T, H, 128], 128-byte swizzle, zero fill outside the tensor); the
// products run as tcgen05.mma (M = 128) with fp32 accumulators in TMEM:
//   [K;Q] K^T (bf16) -> KK^T, QK^T;   W^T, U~^T (fp16);   S0 W^T, S0 Q^T;
//   U^T K~ (state update, N = 128);   U^T P^T (intra-chunk output).
// The fp32 state lives in registers (thread = state row v, half of K) and is
// re-staged as an fp16 MMA operand each chunk.  fp16 (11-bit significand)
// rather than bf16 operands keep written states within 1e-3 relative error.
#include <math.h>

#include "common.cuh"

namespace {

using namespace gdn;

constexpr int kThreads = 256;
constexpr uint32_t kTile = 8192;  // 64 rows x 128 B

// Shared-memory map (byte offsets from a 1024-byte aligned base).
constexpr uint32_t OFF_A1 = 0;           // [kb0: K | Q][kb1: K | Q], 8 KB each; K -> K~, Q -> Q fp16 in place
constexpr uint32_t OFF_V = 32768;        // [vb0 | vb1]; V -> beta V fp16 in place
constexpr uint32_t OFF_BGK = 49152;      // beta gamma K, fp16 [kb0 | kb1]
constexpr uint32_t OFF_T = 65536;        // T fp16, rows t
constexpr uint32_t OFF_P = 73728;        // P fp16, rows t
constexpr uint32_t OFF_WT = 81920;       // W^T fp16, rows k (128)
constexpr uint32_t OFF_U = 98304;        // U^T fp16, rows v (128)
constexpr uint32_t OFF_S = 114688;       // S fp16 [kb0 | kb1], rows v (128 each)
constexpr uint32_t OFF_AM = 147456;      // A matrix fp32 64 x 68 / output staging bf16 64 x 128
constexpr uint32_t OFF_SMALL = OFF_AM + 64 * 68 * 4;
constexpr uint32_t SMEM_USED = OFF_SMALL + 2048;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
constexpr int AM_LD = 68;

// TMEM columns (fp32, 128 lanes).
constexpr uint32_t COL_D1 = 0;    // lanes 0-63: K K^T, lanes 64-127: Q K^T  (64 cols)
constexpr uint32_t COL_WT = 64;   // W^T   (lane = k)
constexpr uint32_t COL_UT = 128;  // U~^T  (lane = v)
constexpr uint32_t COL_X1 = 192;  // S0 W^T
constexpr uint32_t COL_X2 = 256;  // S0 Q^T
constexpr uint32_t COL_SU = 320;  // U^T K~ (128 cols)
constexpr uint32_t COL_Y = 448;   // U^T P^T
constexpr uint32_t TMEM_COLS = 512;

struct PrefillArgs {
  const float* g;
  const float* beta;
  __nv_bfloat16* o;
  const int32_t* cu_seqlens;
  int32_t num_seqs;
  int32_t T;
  int32_t H;
  float scale;
  const float* initial_state;
  const int32_t* state_indices;
  float* output_state;
  const int32_t* output_state_indices;
  float* state_checkpoints;
  const int32_t* checkpoint_state_indices;
  const int32_t* checkpoint_cu_starts;
  const int32_t* prefix_lens;
  int32_t N;
  int64_t row_stride;
  // Paged mode without precomputed slots: rows come from the page table.
  const int32_t* indptr;
  const int32_t* pages;
  const int32_t* last_len;
  int32_t page_size;
  int32_t num_pages;
  int32_t* err_word;
};

struct Small {
  float G[64];
  float gam[64];
  float bet[64];
  int valid[64];
  uint64_t bar_tma;
  uint64_t bar_mma;
  uint32_t tmem_base;
  int seq;
  int flag;
};

__device__ __forceinline__ void cvt8_store(uint8_t* dst, const uint8_t* src_bf16, float sc, bool keep) {
  uint4 out = make_uint4(0u, 0u, 0u, 0u);
  if (keep) {
    const uint4 in = *reinterpret_cast<const uint4*>(src_bf16);
    float2 f0 = unpack_bf162(in.x), f1 = unpack_bf162(in.y), f2 = unpack_bf162(in.z), f3 = unpack_bf162(in.w);
    out.x = pack_half2(f0.x * sc, f0.y * sc);
    out.y = pack_half2(f1.x * sc, f1.y * sc);
    out.z = pack_half2(f2.x * sc, f2.y * sc);
    out.w = pack_half2(f3.x * sc, f3.y * sc);
  }
  *reinterpret_cast<uint4*>(dst) = out;
}

// All threads wait for an mbarrier phase; false (for every thread) if any
// thread timed out.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __syncthreads_or(ok ? 0 : 1) == 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  Small& sh = *reinterpret_cast<Small*>(sm + OFF_SMALL);
  float* AM = reinterpret_cast<float*>(sm + OFF_AM);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  const int rank = blockIdx.x / H, h = blockIdx.x % H;

  // ---- pick the sequence: rank-th longest (ties by index) ----
  if (a.num_seqs > 1 && a.num_seqs <= 4096) {
    int* cu_s = reinterpret_cast<int*>(sm + OFF_AM);
    for (int i = tid; i <= a.num_seqs; i += kThreads) cu_s[i] = a.cu_seqlens[i];
    if (tid == 0) sh.seq = -1;
    __syncthreads();
    for (int s = tid; s < a.num_seqs; s += kThreads) {
      const int ls = cu_s[s + 1] - cu_s[s];
      int r = 0;
      for (int s2 = 0; s2 < a.num_seqs; ++s2) {
        const int l2 = cu_s[s2 + 1] - cu_s[s2];
        r += (l2 > ls) || (l2 == ls && s2 < s);
      }
      if (r == rank) sh.seq = s;
    }
    __syncthreads();
  } else if (tid == 0) {
    sh.seq = rank;
  }
  __syncthreads();
  const int b = sh.seq;
  if (b < 0) return;

  const int cu_b = a.cu_seqlens[b];
  const int L = a.cu_seqlens[b + 1] - cu_b;
  if (L <= 0) return;  // a zero-length sequence reads and writes nothing

  // ---- rows of this sequence ----
  int P, in_row, out_row;
  const int32_t* ck_rows = nullptr;  // j-th checkpoint row = ck_rows[j]
  int N = a.N;
  if (a.indptr) {
    const int i0 = a.indptr[b], i1 = a.indptr[b + 1];
    const int n = i1 - i0;
    const int lpl = a.last_len[b];
    const long long tot = static_cast<long long>(n - 1) * a.page_size + lpl;
    P = static_cast<int>(tot - L);
    bool bad = n < 1 || lpl < 1 || lpl > a.page_size || tot < L;
    if (bad) {
      if (tid == 0) record_error(a.err_word, GDN_DEVERR_PAGE_TABLE, b);
      return;
    }
    in_row = P > 0 ? a.pages[i0 + (P - 1) / a.page_size] : -1;
    out_row = a.pages[i1 - 1];
    ck_rows = a.pages + i0 + P / a.page_size;
    N = a.page_size;
    if (a.err_word) {
      if (tid == 0) {
        int badp = 0;
        for (int i = (P > 0 ? (P - 1) / a.page_size : P / a.page_size); i < n; ++i) {
          const int id = a.pages[i0 + i];
          badp |= (id < 0 || id >= a.num_pages);
        }
        sh.flag = badp;
        if (badp) record_error(a.err_word, GDN_DEVERR_PAGE_ID, b);
      }
      __syncthreads();
      if (sh.flag) return;
    }
  } else {
    P = a.prefix_lens ? a.prefix_lens[b] : 0;
    in_row = a.state_indices ? a.state_indices[b] : -1;
    out_row = a.output_state_indices ? a.output_state_indices[b] : -1;
    if (a.state_checkpoints) ck_rows = a.checkpoint_state_indices + a.checkpoint_cu_starts[b];
    if (P < 0) {
      if (tid == 0) record_error(a.err_word, GDN_DEVERR_PAGE_TABLE, b);
      return;
    }
  }
  if (static_cast<long long>(cu_b) + L > a.T || cu_b < 0) {
    if (tid == 0) record_error(a.err_word, GDN_DEVERR_PAGE_TABLE, b);
    return;
  }
  const float* init_pool = a.initial_state;
  float* out_pool = a.output_state;
  float* ck_pool = a.state_checkpoints;
  if (!init_pool) in_row = -1;
  if (!out_pool) out_row = -1;

  // ---- set-up: barriers, TMEM ----
  if (tid == 0) {
    mbar_init(&sh.bar_tma, 1);
    mbar_init(&sh.bar_mma, 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  const int v_row = tid & 127;        // state row / TMEM lane of this thread
  const int khalf = tid >> 7;         // which 64 columns of K this thread keeps
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  const int64_t head_off = static_cast<int64_t>(h) * kDimV * kDimK;
  const int64_t my_off = head_off + static_cast<int64_t>(v_row) * kDimK + 64 * khalf;

  // ---- initial state: pool row or literal zeros (the pool is never scaled by 0) ----
  float S[64];
  if (in_row >= 0) {
    const float4* src = reinterpret_cast<const float4*>(init_pool + in_row * a.row_stride + my_off);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 x = src[i];
      S[4 * i] = x.x;
      S[4 * i + 1] = x.y;
      S[4 * i + 2] = x.z;
      S[4 * i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) S[i] = 0.f;
  }
  auto stage_state = [&]() {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 u;
      u.x = pack_half2(S[8 * c], S[8 * c + 1]);
      u.y = pack_half2(S[8 * c + 2], S[8 * c + 3]);
      u.z = pack_half2(S[8 * c + 4], S[8 * c + 5]);
      u.w = pack_half2(S[8 * c + 6], S[8 * c + 7]);
      *reinterpret_cast<uint4*>(sm + OFF_S + khalf * 16384 + swz(v_row, c)) = u;
    }
  };
  auto store_state = [&](float* pool, int row) {
    float4* dst = reinterpret_cast<float4*>(pool + row * a.row_stride + my_off);
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
  };
  stage_state();

  const int end_pos = P + L;
  const int first_pos = (P / kChunk) * kChunk;
  const int nchunks = (end_pos + kChunk - 1) / kChunk - P / kChunk;
  const int first_ck = (ck_rows && N > 0) ? P / N : 0;
  uint32_t mma_phase = 0;
  bool failed = false;

  const uint32_t id_bf16_kk = idesc_f16(128, 64, true, true, false, false);
  const uint32_t id_mnA = idesc_f16(128, 64, false, false, true, false);
  const uint32_t id_mnB64 = idesc_f16(128, 64, false, false, false, true);
  const uint32_t id_kk64 = idesc_f16(128, 64, false, false, false, false);
  const uint32_t id_mnB128 = idesc_f16(128, 128, false, false, false, true);

  for (int c = 0; c < nchunks; ++c) {
    const int a0 = first_pos + kChunk * c;   // absolute position of chunk row 0
    const int t_first = cu_b + (a0 - P);     // packed token index of chunk row 0

    // (1) TMA loads of K, Q, V; gates of the 64 rows.
    if (tid == 0) {
      mbar_arrive_expect_tx(&sh.bar_tma, 6 * kTile);
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d(sm + OFF_A1 + kb * 16384, &tm_k, &sh.bar_tma, kb * 64, h, t_first);
        tma_load_3d(sm + OFF_A1 + kb * 16384 + kTile, &tm_q, &sh.bar_tma, kb * 64, h, t_first);
        tma_load_3d(sm + OFF_V + kb * kTile, &tm_v, &sh.bar_tma, kb * 64, h, t_first);
      }
    }
    if (tid < 64) {
      const int pos = a0 + tid;
      const bool valid = pos >= P && pos < end_pos;
      const int64_t t = static_cast<int64_t>(t_first) + tid;
      sh.G[tid] = valid ? a.g[t * H + h] : 0.f;
      sh.bet[tid] = valid ? a.beta[t * H + h] : 0.f;
      sh.valid[tid] = valid;
    }
    __syncthreads();
    if (warp == 0) {
      const float x0 = sh.G[2 * lane], x1 = sh.G[2 * lane + 1];
      float s = x0 + x1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
      }
      const float g0 = s - x1;
      sh.G[2 * lane] = g0;
      sh.G[2 * lane + 1] = s;
      sh.gam[2 * lane] = expf(g0);
      sh.gam[2 * lane + 1] = expf(s);
    }
    if (!wait_all(&sh.bar_tma, c & 1)) {
      failed = true;
      break;
    }
    const float GC = sh.G[63];
    const float gamC = sh.gam[63];

    // (2) MMA1: [K;Q] K^T -> D1 (bf16 operands straight from TMA).
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
        tc_mma(tmem + COL_D1, sdesc(sbase + OFF_A1 + off, 16, 1024), sdesc(sbase + OFF_A1 + off, 16, 1024),
               id_bf16_kk, s > 0);
      }
      tc_commit(&sh.bar_mma);
    }
    // (3) beta gamma K -> BGK, beta V in place (while MMA1 reads K and Q).
    for (int i = tid; i < 2048; i += kThreads) {
      const int r = (i >> 3) & 63, p = i & 7;
      const bool keep = sh.valid[r] != 0;
      if (i < 1024) {
        const int kb = i >> 9;
        cvt8_store(sm + OFF_BGK + kb * kTile + r * 128 + p * 16, sm + OFF_A1 + kb * 16384 + r * 128 + p * 16,
                   sh.bet[r] * sh.gam[r], keep);
      } else {
        const int vb = (i - 1024) >> 9;
        uint8_t* ptr = sm + OFF_V + vb * kTile + r * 128 + p * 16;
        cvt8_store(ptr, ptr, sh.bet[r], keep);
      }
    }
    fence_proxy_async();
    if (!wait_all(&sh.bar_mma, mma_phase)) {
      failed = true;
      break;
    }
    mma_phase ^= 1;
    tc_fence_after();

    // (4) A (fp32, smem) and P (fp16 operand) from D1; Q -> fp16, K -> K~ in place.
    if (warp < 4) {
      const int row = tid;
      float x[32];
      if (row < 64) {
        const int t = row;
        const float Gt = sh.G[t], bt = sh.bet[t];
        const bool vt = sh.valid[t] != 0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tmem_ld32(lane_addr + COL_D1 + 32 * hh, x);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int j = 32 * hh + i;
            AM[t * AM_LD + j] = (vt && j < t && sh.valid[j]) ? bt * expf(Gt - sh.G[j]) * x[i] : 0.f;
          }
        }
      } else {
        const int t = row - 64;
        const float Gt = sh.G[t];
        const bool vt = sh.valid[t] != 0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tmem_ld32(lane_addr + COL_D1 + 32 * hh, x);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = 32 * hh + 8 * q4 + e;
              pv[e] = (vt && j <= t && sh.valid[j]) ? expf(Gt - sh.G[j]) * x[8 * q4 + e] : 0.f;
            }
            uint4 u;
            u.x = pack_half2(pv[0], pv[1]);
            u.y = pack_half2(pv[2], pv[3]);
            u.z = pack_half2(pv[4], pv[5]);
            u.w = pack_half2(pv[6], pv[7]);
            *reinterpret_cast<uint4*>(sm + OFF_P + swz(t, 4 * hh + q4)) = u;
          }
        }
      }
    } else {
      for (int i = tid - 128; i < 2048; i += 128) {
        const int which = i >> 10, j = i & 1023;  // which: 0 = K, 1 = Q
        const int kb = j >> 9, r = (j >> 3) & 63, p = j & 7;
        uint8_t* ptr = sm + OFF_A1 + kb * 16384 + which * kTile + r * 128 + p * 16;
        const bool keep = sh.valid[r] != 0;
        cvt8_store(ptr, ptr, which ? 1.f : expf(GC - sh.G[r]), keep);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // (5) T = (I + A)^-1 by forward substitution, one column per thread.
    if (tid < 64) {
      const int j = tid;
      float col[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) col[i] = 0.f;
#pragma unroll
      for (int t = 0; t < 64; ++t) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < t; i += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(&AM[t * AM_LD + i]);
          acc += a4.x * col[i] + a4.y * col[i + 1] + a4.z * col[i + 2] + a4.w * col[i + 3];
        }
        col[t] = (t == j) ? 1.f : -acc;
      }
      __half* Th = reinterpret_cast<__half*>(sm + OFF_T);
#pragma unroll
      for (int t = 0; t < 64; ++t) Th[(swz(t, j >> 3) >> 1) + (j & 7)] = __float2half_rn(col[t]);
    }
    fence_proxy_async();
    __syncthreads();

    // (6) MMA2: W^T = (beta gamma K)^T T^T,  U~^T = (beta V)^T T^T.
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t bd = sdesc(sbase + OFF_T + s * 32, 16, 1024);
        tc_mma(tmem + COL_WT, sdesc(sbase + OFF_BGK + s * 2048, kTile, 1024), bd, id_mnA, s > 0);
        tc_mma(tmem + COL_UT, sdesc(sbase + OFF_V + s * 2048, kTile, 1024), bd, id_mnA, s > 0);
      }
      tc_commit(&sh.bar_mma);
    }
    if (!wait_all(&sh.bar_mma, mma_phase)) {
      failed = true;
      break;
    }
    mma_phase ^= 1;
    tc_fence_after();

    // (7) W^T -> fp16 operand, rows k.
    {
      float x[32];
      tmem_ld32(lane_addr + COL_WT + 32 * khalf, x);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 u;
        u.x = pack_half2(x[8 * q4], x[8 * q4 + 1]);
        u.y = pack_half2(x[8 * q4 + 2], x[8 * q4 + 3]);
        u.z = pack_half2(x[8 * q4 + 4], x[8 * q4 + 5]);
        u.w = pack_half2(x[8 * q4 + 6], x[8 * q4 + 7]);
        *reinterpret_cast<uint4*>(sm + OFF_WT + swz(v_row, 4 * khalf + q4)) = u;
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // (8) X1 = S0 W^T, X2 = S0 Q^T.
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t koff = (s >> 2) * 16384 + (s & 3) * 32;
        const uint64_t ad = sdesc(sbase + OFF_S + koff, 16, 1024);
        tc_mma(tmem + COL_X1, ad, sdesc(sbase + OFF_WT + s * 2048, kTile, 1024), id_mnB64, s > 0);
        tc_mma(tmem + COL_X2, ad, sdesc(sbase + OFF_A1 + koff + kTile, 16, 1024), id_kk64, s > 0);
      }
      tc_commit(&sh.bar_mma);
    }
    if (!wait_all(&sh.bar_mma, mma_phase)) {
      failed = true;
      break;
    }
    mma_phase ^= 1;
    tc_fence_after();

    // (9) U^T = U~^T - X1 -> fp16 operand, rows v.
    {
      float xu[32], xw[32];
      tmem_ld32(lane_addr + COL_UT + 32 * khalf, xu);
      tmem_ld32(lane_addr + COL_X1 + 32 * khalf, xw);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 u;
        u.x = pack_half2(xu[8 * q4] - xw[8 * q4], xu[8 * q4 + 1] - xw[8 * q4 + 1]);
        u.y = pack_half2(xu[8 * q4 + 2] - xw[8 * q4 + 2], xu[8 * q4 + 3] - xw[8 * q4 + 3]);
        u.z = pack_half2(xu[8 * q4 + 4] - xw[8 * q4 + 4], xu[8 * q4 + 5] - xw[8 * q4 + 5]);
        u.w = pack_half2(xu[8 * q4 + 6] - xw[8 * q4 + 6], xu[8 * q4 + 7] - xw[8 * q4 + 7]);
        *reinterpret_cast<uint4*>(sm + OFF_U + swz(v_row, 4 * khalf + q4)) = u;
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // (10) SU = U^T K~ (state update), Y = U^T P^T (intra-chunk outputs).
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t ad = sdesc(sbase + OFF_U + s * 32, 16, 1024);
        tc_mma(tmem + COL_SU, ad, sdesc(sbase + OFF_A1 + s * 2048, 16384, 1024), id_mnB128, s > 0);
        tc_mma(tmem + COL_Y, ad, sdesc(sbase + OFF_P + s * 32, 16, 1024), id_kk64, s > 0);
      }
      tc_commit(&sh.bar_mma);
    }
    if (!wait_all(&sh.bar_mma, mma_phase)) {
      failed = true;
      break;
    }
    mma_phase ^= 1;
    tc_fence_after();

    // (11) S <- gamma_C S + SU; outputs; checkpoint.
    {
      float x[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        tmem_ld32(lane_addr + COL_SU + 64 * khalf + 32 * hh, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) S[32 * hh + i] = gamC * S[32 * hh + i] + x[i];
      }
      stage_state();
      float x2[32], y[32];
      tmem_ld32(lane_addr + COL_X2 + 32 * khalf, x2);
      tmem_ld32(lane_addr + COL_Y + 32 * khalf, y);
      __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_AM);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = 32 * khalf + i;
        ost[t * 128 + v_row] = __float2bfloat16_rn(a.scale * (sh.gam[t] * x2[i] + y[i]));
      }
      const int a_end = a0 + kChunk;
      if (ck_rows && ck_pool && a_end % N == 0 && a_end <= end_pos) {
        const int row = ck_rows[a_end / N - 1 - first_ck];
        if (row >= 0) store_state(ck_pool, row);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // (12) Output rows of this chunk that belong to the sequence.
    {
      const __nv_bfloat16* ost = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_AM);
      for (int i = tid; i < 64 * 16; i += kThreads) {
        const int r = i >> 4, p = i & 15;
        const int pos = a0 + r;
        if (pos >= P && pos < end_pos) {
          const int64_t t = static_cast<int64_t>(t_first) + r;
          *reinterpret_cast<uint4*>(a.o + (t * H + h) * kDimV + p * 8) =
              *reinterpret_cast<const uint4*>(ost + r * 128 + p * 8);
        }
      }
    }
    __syncthreads();
  }

  if (failed) {
    if (tid == 0) record_error(a.err_word, GDN_DEVERR_TIMEOUT, b);
  } else if (out_row >= 0) {
    store_state(out_pool, out_row);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

int launch(const PrefillArgs& a, const void* q, const void* k, const void* v, cudaStream_t stream) {
  int rc = gdn_host::check_device(nullptr);
  if (rc != GDN_OK) return rc;
  CUtensorMap mq, mk, mv;
  if (gdn_host::encode_tokens_map(&mq, q, a.T, a.H, kDimK) != GDN_OK ||
      gdn_host::encode_tokens_map(&mk, k, a.T, a.H, kDimK) != GDN_OK ||
      gdn_host::encode_tokens_map(&mv, v, a.T, a.H, kDimV) != GDN_OK)
    return GDN_ERR_CUDA;
  if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess) {
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  const long long grid = static_cast<long long>(a.num_seqs) * a.H;
  prefill_kernel<<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, stream>>>(mq, mk, mv, a);
  return gdn_host::launch_status();
}

int check_common(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g, const float* beta,
                 gdn_bf16* o, const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H,
                 int32_t K, int32_t V) {
  if (num_seqs < 0 || total_tokens < 0 || H < 1) return GDN_ERR_INVALID_ARGUMENT;
  if (K != kDimK || V != kDimV) return GDN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_seqs) * H > 0x7FFFFFFFLL) return GDN_ERR_UNSUPPORTED;
  if (num_seqs > 0 && !cu_seqlens) return GDN_ERR_INVALID_ARGUMENT;
  if (total_tokens > 0) {
    using gdn_host::aligned16;
    if (!q || !k || !v || !g || !beta || !o) return GDN_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(g) & 3u) || (reinterpret_cast<uintptr_t>(beta) & 3u))
      return GDN_ERR_INVALID_ARGUMENT;
  }
  return GDN_OK;
}

void fill_common(PrefillArgs& a, const float* g, const float* beta, gdn_bf16* o, const int32_t* cu_seqlens,
                 int32_t num_seqs, int32_t total_tokens, int32_t H, float scale, int32_t* err_word) {
  a = PrefillArgs{};
  a.g = g;
  a.beta = beta;
  a.o = reinterpret_cast<__nv_bfloat16*>(o);
  a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs;
  a.T = total_tokens;
  a.H = H;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(kDimK));
  a.err_word = err_word;
}

}  // namespace

extern "C" int gdn_chunk_gated_delta_rule(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                                          const float* beta, gdn_bf16* o, const int32_t* cu_seqlens,
                                          int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t K, int32_t V,
                                          float scale, const float* initial_state, const int32_t* state_indices,
                                          float* output_state, const int32_t* output_state_indices,
                                          float* state_checkpoints, const int32_t* checkpoint_state_indices,
                                          const int32_t* checkpoint_cu_starts, const int32_t* prefix_lens,
                                          int32_t checkpoint_every_n_tokens, int64_t pool_row_stride,
                                          int32_t* err_word, void* stream) {
  int rc = check_common(q, k, v, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, K, V);
  if (rc != GDN_OK) return rc;
  if ((state_indices != nullptr) != (initial_state != nullptr)) return GDN_ERR_INVALID_ARGUMENT;
  if ((output_state_indices != nullptr) != (output_state != nullptr)) return GDN_ERR_INVALID_ARGUMENT;
  const int nck = (state_checkpoints != nullptr) + (checkpoint_state_indices != nullptr) +
                  (checkpoint_cu_starts != nullptr);
  if (nck != 0 && nck != 3) return GDN_ERR_INVALID_ARGUMENT;
  if (nck == 3 && (!prefix_lens || checkpoint_every_n_tokens <= 0 || checkpoint_every_n_tokens % kChunk != 0))
    return GDN_ERR_INVALID_ARGUMENT;
  const bool any_pool = initial_state || output_state || state_checkpoints;
  if (any_pool && (pool_row_stride < static_cast<int64_t>(H) * kDimV * kDimK || pool_row_stride % 4 != 0))
    return GDN_ERR_INVALID_ARGUMENT;
  using gdn_host::aligned16;
  if ((initial_state && !aligned16(initial_state)) || (output_state && !aligned16(output_state)) ||
      (state_checkpoints && !aligned16(state_checkpoints)))
    return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0 || total_tokens == 0) return GDN_OK;

  PrefillArgs a;
  fill_common(a, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, scale, err_word);
  a.initial_state = initial_state;
  a.state_indices = state_indices;
  a.output_state = output_state;
  a.output_state_indices = output_state_indices;
  a.state_checkpoints = state_checkpoints;
  a.checkpoint_state_indices = checkpoint_state_indices;
  a.checkpoint_cu_starts = checkpoint_cu_starts;
  a.prefix_lens = prefix_lens;
  a.N = nck ? checkpoint_every_n_tokens : 0;
  a.row_stride = any_pool ? pool_row_stride : 0;
  return launch(a, q, k, v, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_chunk_gated_delta_rule_paged(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                                const float* g, const float* beta, gdn_bf16* o,
                                                const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                                int32_t H, int32_t K, int32_t V, float scale, float* state_pool,
                                                int32_t num_pages, const int32_t* page_indices,
                                                const int32_t* page_indptr, int32_t page_size,
                                                const int32_t* last_page_len, const gdn_prefill_slots* slots,
                                                int32_t* err_word, void* stream) {
  int rc = check_common(q, k, v, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, K, V);
  if (rc != GDN_OK) return rc;
  if (page_size <= 0 || page_size % kChunk != 0 || num_pages < 1) return GDN_ERR_INVALID_ARGUMENT;
  if (!state_pool || !gdn_host::aligned16(state_pool)) return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs > 0 && (!page_indices || !page_indptr || !last_page_len)) return GDN_ERR_INVALID_ARGUMENT;
  if (slots && (!slots->state_indices || !slots->output_state_indices || !slots->checkpoint_cu_starts ||
                !slots->prefix_lens))
    return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0 || total_tokens == 0) return GDN_OK;

  PrefillArgs a;
  fill_common(a, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, scale, err_word);
  a.initial_state = state_pool;
  a.output_state = state_pool;
  a.state_checkpoints = state_pool;
  a.checkpoint_state_indices = page_indices;
  a.N = page_size;
  a.row_stride = static_cast<int64_t>(H) * kDimV * kDimK;
  a.num_pages = num_pages;
  a.page_size = page_size;
  if (slots) {
    a.state_indices = slots->state_indices;
    a.output_state_indices = slots->output_state_indices;
    a.checkpoint_cu_starts = slots->checkpoint_cu_starts;
    a.prefix_lens = slots->prefix_lens;
  } else {
    a.indptr = page_indptr;
    a.pages = page_indices;
    a.last_len = last_page_len;
  }
  return launch(a, q, k, v, static_cast<cudaStream_t>(stream));
}
