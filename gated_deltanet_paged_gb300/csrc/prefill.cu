// prefill.cu -- chunked paged GDN prefill on tcgen05 tensor cores.
//
// "flashinfer.gdn_paged": chunk_gated_delta_rule_paged, the prefill bullets,
// the 64-token left-padding paragraph, and "Slot arguments of
// chunk_gated_delta_rule" (read / final / checkpoint rows, -1 = zero state or
// skip, checkpoints at absolute positions (prefix + n) % N == 0).
//
// Method (gated delta rule, chunked).  Per (sequence, head) chain and 64-token
// chunk with rows t = 0..63, cumulative gate G_t = g_0 + ... + g_t (rows outside
// the sequence have g = beta = 0 and k = v = 0, so they are the identity),
// gamma_t = exp(G_t), S0 the V x K state at the chunk start:
//   A[t][j] = beta_t exp(G_t - G_j) (k_t . k_j)      j < t   (strictly lower)
//   T       = (I + A)^-1
//   W       = T diag(beta gamma) K,   U~ = T diag(beta) V
//   U       = U~ - W S0^T                            (the chunk's new values)
//   O[t]    = scale (gamma_t S0 q_t + sum_{j<=t} exp(G_t - G_j)(q_t . k_j) U[j])
//   S1      = gamma_C S0 + U^T diag(exp(G_C - G_j)) K
// which equals the token-by-token recurrence up to rounding.
//
// Mapping.  One CTA (512 threads) per chain, chains ordered by decreasing
// length.  Per chunk the work splits into a state-independent "prep" (TMA of
// Q/K/V, gates, [K;Q]K^T, A and P, the inverse T, W^T and U~^T) and the state
// "chain" (S0 W^T and S0 Q~^T, U, U^T K~ and U^T P^T, the state update and the
// outputs).  The loop runs chain(c) and prep(c+1) in one software-pipelined
// instruction stream: every tcgen05.mma is followed by CUDA-core work that does
// not depend on it, so MMA latency hides behind the other half.  TMA runs two
// chunks ahead into a pair of slots.
//   - MMAs (M = 128, fp32 accumulators in TMEM): [K;Q]K^T on bf16 straight from
//     TMA; everything else on fp16 operands (11-bit significand keeps written
//     states within 1e-3 relative error; bf16 would not).
//   - decay factors exp(G_t - G_j) come from running products of exp(g).
//   - T = (I + A)^-1: the 16x16 diagonal blocks T_d by forward substitution on
//     CUDA cores, the rest as three MMAs: N = -T_d A_o (A_o the block-lower
//     part of A, N^4 = 0), T = (I + N)(I + N^2) T_d = Z + N^2 Z with
//     Z = (I + N) T_d.
//   - beta gamma and beta fold into the columns of T (T', T''), gamma into Q~
//     and exp(G_C - G) into K~, so O = scale (S0 Q~^T + U P^T) is one
//     accumulator and S1 = gamma_C S0 + U^T K~.
//   - the fp32 state lives in registers (thread = state row v, 32 columns) and is
//     restaged as the fp16 MMA operand every chunk; page-boundary and final
//     states go from registers to the pool.
#include <math.h>

#include "common.cuh"

namespace {

using namespace gdn;

constexpr int kThreads = 512;
constexpr uint32_t kTile = 8192;  // 64 rows x 128 B

// Slot: the raw TMA tiles of one chunk (two slots), converted in place.
constexpr uint32_t SLOT_BYTES = 49152;
constexpr uint32_t SL_K0 = 0;      // K cols 0-63   -> K fp16 (MN-major A of W^T)
constexpr uint32_t SL_Q0 = 8192;   // Q cols 0-63   -> A_o, N^2 (inverse operands) -> T' fp16
constexpr uint32_t SL_K1 = 16384;  // K cols 64-127 -> K fp16
constexpr uint32_t SL_Q1 = 24576;  // Q cols 64-127 -> Z (inverse operand) -> T'' fp16
constexpr uint32_t SL_V0 = 32768;  // V cols 0-63   -> V fp16 (MN-major A of U~^T)
constexpr uint32_t SL_V1 = 40960;  // V cols 64-127 -> V fp16
// Other tiles (byte offsets from the 1024-aligned base).
constexpr uint32_t OFF_FREE = 2 * SLOT_BYTES;  // 16 KB scratch (sequence ranking at start-up)
constexpr uint32_t OFF_KT = OFF_FREE + 16384;  // K~ = diag(exp(G_C - G)) K fp16 [kb0 | kb1], rows t
constexpr uint32_t OFF_P = OFF_KT + 16384;     // P fp16, two buffers, rows t
constexpr uint32_t OFF_WT = OFF_P + 16384;     // inverse scratch: fp32 A / T_d, then N | T_d (fp16)
constexpr uint32_t OFF_U = OFF_WT + 16384;     // output / state staging for coalesced stores
constexpr uint32_t OFF_XB = OFF_U + 16384;     // [W | Q~] fp16 per 64-column block: the B operand of S0 [W; Q~]^T
constexpr uint32_t OFF_SMALL = OFF_XB + 32768;
constexpr uint32_t SMEM_USED = OFF_SMALL + 2048;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base

// TMEM columns (fp32, 128 lanes).
constexpr uint32_t COL_D1 = 0;     // [K;Q]K^T, then the inverse's products (cols 0-127)
constexpr uint32_t COL_WT = 64;    // W^T   (lane = k)
constexpr uint32_t COL_U = 64;     // U^T as the fp16 A operand (32 cols; free between W^T uses)
constexpr uint32_t COL_UT = 128;   // U~^T  (lane = v)
constexpr uint32_t COL_X1 = 192;   // S0 W^T       } one N = 128 product
constexpr uint32_t COL_O = 256;    // S0 Q~^T      } + U^T P^T accumulated later
constexpr uint32_t COL_SU = 320;   // U^T K~ (128 cols)
constexpr uint32_t COL_S16 = 448;  // S0 as the fp16 A operand (64 cols)
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

// Per-chunk scalars of the chunk being prepared.
struct Small {
  float G[64];    // cumulative gate
  float e[64];    // exp(g)
  float gam[64];  // exp(G)
  float bet[64];  // beta (0 outside the sequence)
  float sT1[64];  // beta * gamma  (column scale of T')
  float ksc[64];  // exp(G_C - G)  (row scale of K~)
  uint64_t bar_tma[2];
  uint64_t bar_x, bar_1, bar_s, bar_2, bar_l2;
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

__device__ __forceinline__ uint32_t scale_half2(uint32_t u, float sc) {
  __half2 h = *reinterpret_cast<__half2*>(&u);
  const float2 f = __half22float2(h);
  return pack_half2(f.x * sc, f.y * sc);
}

__device__ __forceinline__ uint4 pack8_half(const float* x) {
  uint4 u;
  u.x = pack_half2(x[0], x[1]);
  u.y = pack_half2(x[2], x[3]);
  u.z = pack_half2(x[4], x[5]);
  u.w = pack_half2(x[6], x[7]);
  return u;
}

// fp32 64 x 64 matrix, 16-byte chunk cj of row r stored at chunk cj ^ (r % 16).
__device__ __forceinline__ float* am_chunk(float* AM, int r, int cj) { return AM + r * 64 + ((cj ^ (r & 15)) << 2); }
__device__ __forceinline__ float& am_at(float* AM, int r, int j) {
  return AM[r * 64 + ((((j >> 2) ^ (r & 15)) << 2) | (j & 3))];
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  Small& sh = *reinterpret_cast<Small*>(sm + OFF_SMALL);
  float* AM = reinterpret_cast<float*>(sm + OFF_WT);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  const int rank = blockIdx.x / H, h = blockIdx.x % H;

  // ---- pick the sequence: rank-th longest (ties by index) ----
  if (a.num_seqs > 1 && a.num_seqs < 4096) {
    int* cu_s = reinterpret_cast<int*>(sm + OFF_FREE);
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
    if (n < 1 || lpl < 1 || lpl > a.page_size || tot < L) {
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
        for (int i = (P > 0 ? (P - 1) / a.page_size : 0); i < n; ++i) {
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
    mbar_init(&sh.bar_tma[0], 1);
    mbar_init(&sh.bar_tma[1], 1);
    mbar_init(&sh.bar_x, 1);
    mbar_init(&sh.bar_1, 1);
    mbar_init(&sh.bar_s, 1);
    mbar_init(&sh.bar_2, 1);
    mbar_init(&sh.bar_l2, 1);
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

  // Thread roles: v_row = state row / TMEM lane (0..127), quarter = which 32
  // state columns (and which quarter of a 64-column accumulator) it handles.
  // For tile conversions every thread owns row cr = tid / 8, 16-byte chunk
  // tid % 8, in both 64-column blocks (byte offset tid * 16 in a block).
  const int v_row = tid & 127;
  const int quarter = tid >> 7;
  const int cr = tid >> 3;
  const uint32_t coff = static_cast<uint32_t>(tid) * 16u;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  const int64_t head_off = static_cast<int64_t>(h) * kDimV * kDimK;

  // ---- initial state: pool row or literal zeros (the pool is never scaled by 0) ----
  float S[32];
  if (in_row >= 0) {
    const float4* src =
        reinterpret_cast<const float4*>(init_pool + in_row * a.row_stride + head_off + v_row * kDimK + 32 * quarter);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = src[i];
      S[4 * i] = x.x;
      S[4 * i + 1] = x.y;
      S[4 * i + 2] = x.z;
      S[4 * i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) S[i] = 0.f;
  }
  auto stage_state = [&]() {  // fp16 copy of S as the TMEM A operand
    uint32_t w[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) w[c] = pack_half2(S[2 * c], S[2 * c + 1]);
    tmem_st16(lane_addr + COL_S16 + 16 * quarter, w);
  };
  // Store the fp32 state to a pool row with coalesced 16-byte stores, staging
  // 32 state rows (16 KB) at a time in the U tile (free whenever this runs).
  auto store_state = [&](float* pool, int row) {
    float4* stg = reinterpret_cast<float4*>(sm + OFF_U);
    float4* dst = reinterpret_cast<float4*>(pool + row * a.row_stride + head_off);
#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
      if ((warp & 3) == r) {
        const int rr = v_row - 32 * r;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          stg[rr * 32 + ((8 * quarter + i) ^ rr)] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = tid + k * kThreads;
        dst[r * 1024 + i] = stg[(i >> 5) * 32 + ((i & 31) ^ (i >> 5))];
      }
      __syncthreads();
    }
  };
  stage_state();

  const int end_pos = P + L;
  const int first_pos = (P / kChunk) * kChunk;
  const int nchunks = (end_pos + kChunk - 1) / kChunk - P / kChunk;
  const int first_ck = (ck_rows && N > 0) ? P / N : 0;

  const uint32_t id_bf16_kk = idesc_f16(128, 64, true, true, false, false);
  const uint32_t id_mnA = idesc_f16(128, 64, false, false, true, false);
  const uint32_t id_mnB64 = idesc_f16(128, 64, false, false, false, true);
  const uint32_t id_kk64 = idesc_f16(128, 64, false, false, false, false);
  const uint32_t id_mnB128 = idesc_f16(128, 128, false, false, false, true);
  const uint32_t id_kk128 = idesc_f16(128, 128, false, false, false, false);

  // Geometry of chunk ch: absolute position of row 0, valid rows [lo, hi),
  // packed token index of row 0.
  auto chunk_a0 = [&](int ch) { return first_pos + kChunk * ch; };
  auto chunk_lo = [&](int ch) { return max(P - chunk_a0(ch), 0); };
  auto chunk_hi = [&](int ch) { return min(end_pos - chunk_a0(ch), kChunk); };
  auto chunk_tf = [&](int ch) { return cu_b + (chunk_a0(ch) - P); };
  auto slot_off = [&](int ch) { return static_cast<uint32_t>(ch & 1) * SLOT_BYTES; };
  // Shared-memory descriptors: K-major (8-row groups 1024 B apart) and MN-major.
  auto dK = [&](uint32_t off) { return sdesc(sbase + off, 16, 1024); };
  auto dMN = [&](uint32_t off, uint32_t lbo) { return sdesc(sbase + off, lbo, 1024); };

  uint32_t ph_x = 0, ph_1 = 0, ph_s = 0, ph_2 = 0, ph_l2 = 0;
  bool failed = false;
  // One thread polls the mbarrier; everybody meets at a hardware barrier.
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {
    int bad = 0;
    if (tid == 0) bad = mbar_wait(bar, parity) ? 0 : 1;
    return __syncthreads_or(bad) == 0;
  };

  // ---------------------------------------------------------------- prep ----
  auto issue_tma = [&](int ch) {  // one thread
    const int tf = chunk_tf(ch);
    uint8_t* s = sm + slot_off(ch);
    uint64_t* bar = &sh.bar_tma[ch & 1];
    mbar_arrive_expect_tx(bar, 6 * kTile);
    tma_load_3d(s + SL_K0, &tm_k, bar, 0, h, tf);
    tma_load_3d(s + SL_K1, &tm_k, bar, 64, h, tf);
    tma_load_3d(s + SL_Q0, &tm_q, bar, 0, h, tf);
    tma_load_3d(s + SL_Q1, &tm_q, bar, 64, h, tf);
    tma_load_3d(s + SL_V0, &tm_v, bar, 0, h, tf);
    tma_load_3d(s + SL_V1, &tm_v, bar, 64, h, tf);
  };
  float pg0 = 0.f, pg1 = 0.f, pb0 = 0.f, pb1 = 0.f;  // gates of rows 2*lane, 2*lane+1 (warp 1)
  auto prefetch_gates = [&](int ch) {
    if (warp == 1) {
      const int lo = chunk_lo(ch), hi = chunk_hi(ch);
      const int64_t tf = chunk_tf(ch);
      const int r0 = 2 * lane, r1 = 2 * lane + 1;
      const bool v0 = r0 >= lo && r0 < hi, v1 = r1 >= lo && r1 < hi;
      pg0 = v0 ? a.g[(tf + r0) * H + h] : 0.f;
      pb0 = v0 ? a.beta[(tf + r0) * H + h] : 0.f;
      pg1 = v1 ? a.g[(tf + r1) * H + h] : 0.f;
      pb1 = v1 ? a.beta[(tf + r1) * H + h] : 0.f;
    }
  };
  auto gates = [&]() {  // warp 1: cumulative gate and the per-row scalars
    if (warp == 1) {
      float s = pg0 + pg1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
      }
      const float G0 = s - pg1, G1 = s;
      const float GC = __shfl_sync(0xffffffffu, s, 31);
      const float gm0 = expf(G0), gm1 = expf(G1);
      sh.G[2 * lane] = G0;
      sh.G[2 * lane + 1] = G1;
      sh.e[2 * lane] = expf(pg0);
      sh.e[2 * lane + 1] = expf(pg1);
      sh.gam[2 * lane] = gm0;
      sh.gam[2 * lane + 1] = gm1;
      sh.bet[2 * lane] = pb0;
      sh.bet[2 * lane + 1] = pb1;
      sh.sT1[2 * lane] = pb0 * gm0;
      sh.sT1[2 * lane + 1] = pb1 * gm1;
      sh.ksc[2 * lane] = expf(GC - G0);
      sh.ksc[2 * lane + 1] = expf(GC - G1);
    }
  };
  // Convert this thread's chunk of both 64-column blocks of a bf16 tile.
  auto cvt_tile = [&](uint32_t dst, uint32_t dblk, uint32_t src, uint32_t sblk, float sc, bool keep) {
    cvt8_store(sm + dst + coff, sm + src + coff, sc, keep);
    cvt8_store(sm + dst + dblk + coff, sm + src + sblk + coff, sc, keep);
  };
  auto row_ok = [&](int ch) { return cr >= chunk_lo(ch) && cr < chunk_hi(ch); };
  // The same conversion spread over warps 1-15 only (warp 0 is issuing MMAs).
  auto cvt_tile_w = [&](int ch, uint32_t dst, uint32_t dblk, uint32_t src, uint32_t sblk, const float* rsc) {
    if (warp == 0) return;
    const int lo = chunk_lo(ch), hi = chunk_hi(ch);
    for (int i = tid - 32; i < 1024; i += kThreads - 32) {
      const int kb = i >> 9, r = (i & 511) >> 3;
      const uint32_t o = static_cast<uint32_t>(i & 511) * 16u;
      cvt8_store(sm + dst + kb * dblk + o, sm + src + kb * sblk + o, rsc ? rsc[r] : 1.f, r >= lo && r < hi);
    }
  };
  // A from K K^T rows: the diagonal 16x16 blocks in fp32 (AM, for level 0 of
  // the inverse), the strictly block-lower part as an fp16 operand (slot Q0,
  // diagonal blocks zero); P (fp16 operand) from Q K^T rows.  Decay factors by
  // running products exp(G_t - G_{j-1}) = exp(G_t - G_j) exp(g_j).
  auto build_AP = [&](int ch) {
    const int lo = chunk_lo(ch), hi = chunk_hi(ch);
    const int j0 = 16 * quarter;
    const int t = v_row & 63;
    const bool isA = v_row < 64;
    float x[16];
    tmem_ld16(lane_addr + COL_D1 + j0, x);
    const int jstart = min(j0 + 15, isA ? t - 1 : t);  // last column kept (j < t for A, j <= t for P)
    float out[16];
    if (t >= lo && t < hi && jstart >= j0) {
      float ev[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 e4 = *reinterpret_cast<const float4*>(&sh.e[j0 + 4 * q]);
        ev[4 * q] = e4.x;
        ev[4 * q + 1] = e4.y;
        ev[4 * q + 2] = e4.z;
        ev[4 * q + 3] = e4.w;
      }
      float cur = (isA ? sh.bet[t] : 1.f) * expf(sh.G[t] - sh.G[jstart]);
      if (jstart == j0 + 15 && lo <= j0) {  // whole block inside: no masks
#pragma unroll
        for (int jj = 15; jj >= 0; --jj) {
          out[jj] = cur * x[jj];
          cur *= ev[jj];
        }
      } else {
#pragma unroll
        for (int jj = 15; jj >= 0; --jj) {
          const int j = j0 + jj;
          const bool in = (j <= jstart) && (j >= lo);
          out[jj] = in ? cur * x[jj] : 0.f;
          if (j <= jstart) cur *= ev[jj];
        }
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) out[jj] = 0.f;
    }
    if (isA) {
      const bool diag = (t >> 4) == quarter;
      if (diag) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(am_chunk(AM, t, (j0 >> 2) + q)) =
              make_float4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
      }
      uint8_t* ao = sm + slot_off(ch) + SL_Q0;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        *reinterpret_cast<uint4*>(ao + swz(t, 2 * quarter + q)) =
            diag ? make_uint4(0u, 0u, 0u, 0u) : pack8_half(&out[8 * q]);
    } else {
      uint8_t* pbuf = sm + OFF_P + (ch & 1) * kTile;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        *reinterpret_cast<uint4*>(pbuf + swz(t, 2 * quarter + q)) = pack8_half(&out[8 * q]);
    }
  };
  // Level 0 of the inverse (threads 0-63): T_d = the 16x16 diagonal blocks of
  // (I + A)^-1, one column per thread by forward substitution; then T_d as an
  // fp16 tile (rows t, zeros outside the diagonal blocks) at OFF_WT + 8 KB.
  auto inverse_l0 = [&]() {
    const int bb = tid >> 4, jj = tid & 15;
    float x[16];
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      const int row = 16 * bb + tt;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if (4 * m < tt) {
          const float4 a4 = *reinterpret_cast<const float4*>(am_chunk(AM, row, 4 * bb + m));
          if (4 * m + 0 < tt) acc[0] = fmaf(a4.x, x[4 * m + 0], acc[0]);
          if (4 * m + 1 < tt) acc[1] = fmaf(a4.y, x[4 * m + 1], acc[1]);
          if (4 * m + 2 < tt) acc[2] = fmaf(a4.z, x[4 * m + 2], acc[2]);
          if (4 * m + 3 < tt) acc[3] = fmaf(a4.w, x[4 * m + 3], acc[3]);
        }
      }
      x[tt] = (tt == jj) ? 1.f : (tt > jj ? -((acc[0] + acc[1]) + (acc[2] + acc[3])) : 0.f);
    }
    asm volatile("bar.sync 1, 64;" ::: "memory");  // all of A's diagonal blocks read
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) am_at(AM, 16 * bb + tt, 16 * bb + jj) = x[tt];
    asm volatile("bar.sync 1, 64;" ::: "memory");
    {
      // Row t of T_d (its diagonal block) into registers first: the fp16 tile
      // overlaps rows 32-63 of the fp32 scratch that other threads still read.
      const int t = tid, blk = t >> 4;
      float f[16];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 v4 = *reinterpret_cast<const float4*>(am_chunk(AM, t, 4 * blk + m));
        f[4 * m] = v4.x;
        f[4 * m + 1] = v4.y;
        f[4 * m + 2] = v4.z;
        f[4 * m + 3] = v4.w;
      }
      asm volatile("bar.sync 1, 64;" ::: "memory");
      uint8_t* td = sm + OFF_WT + kTile;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if ((c >> 1) == blk) u = pack8_half(&f[8 * (c & 1)]);
        *reinterpret_cast<uint4*>(td + swz(t, c)) = u;
      }
    }
    fence_proxy_async();  // T_d is an MMA operand
  };
  // Rest of the inverse on the tensor core.  With N = -T_d A_o (A_o = the
  // strictly block-lower part of A; N^4 = 0):
  //   T = (I + N + N^2 + N^3) T_d = Z + N^2 Z,   Z = (I + N) T_d.
  // Round 1: N = -T_d A_o.  Round 2: [N^2 | N T_d] = N [N | T_d] -> Z, N^2.
  // Round 3: T = Z + N^2 Z -> T' = T diag(beta gamma), T'' = T diag(beta).
  // The 64-row products occupy TMEM lanes 0-63; warps 0,1,4,5,8,9,12,13 read
  // them (16 columns each).  Tiles: T_d at OFF_WT + 8 KB, N at OFF_WT (so
  // [N | T_d] is one MN-major operand), A_o / N^2 / T' at slot Q0, Z / T'' at
  // slot Q1.
  auto inverse_rest = [&](int ch) -> bool {
    const uint32_t so = slot_off(ch);
    uint8_t* s = sm + so;
    const bool rt = (warp & 3) < 2;       // this thread reads TMEM lanes 0-63
    const int t = v_row;                  // its row (valid when rt)
    const uint32_t lrow = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    // Round 1.
    if (tid == 0) {
      tc_fence_after();
      tc_mma4(tmem + COL_D1, dK(OFF_WT + kTile), 2, dMN(so + SL_Q0, kTile), 128, id_mnB64, 0);
      tc_commit(&sh.bar_l2);
    }
    if (!wait_bar(&sh.bar_l2, ph_l2)) return false;
    ph_l2 ^= 1;
    tc_fence_after();
    if (rt) {
      float d[16];
      tmem_ld16(lrow + COL_D1 + 16 * quarter, d);
#pragma unroll
      for (int q = 0; q < 16; ++q) d[q] = -d[q];
#pragma unroll
      for (int q = 0; q < 2; ++q)
        *reinterpret_cast<uint4*>(sm + OFF_WT + swz(t, 2 * quarter + q)) = pack8_half(&d[8 * q]);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // Round 2.
    if (tid == 0) {
      tc_fence_after();
      tc_mma4(tmem + COL_D1, dK(OFF_WT), 2, dMN(OFF_WT, kTile), 128, id_mnB128, 0);
      tc_commit(&sh.bar_l2);
    }
    if (!wait_bar(&sh.bar_l2, ph_l2)) return false;
    ph_l2 ^= 1;
    tc_fence_after();
    float z[16];
    if (rt) {
      float n2[16], nt[16];
      tmem_ld16(lrow + COL_D1 + 16 * quarter, n2);
      tmem_ld16(lrow + COL_D1 + 64 + 16 * quarter, nt);
      const uint8_t* td = sm + OFF_WT + kTile;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 u = *reinterpret_cast<const uint4*>(td + swz(t, 2 * quarter + q));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          z[8 * q + 2 * e] = f.x + nt[8 * q + 2 * e];
          z[8 * q + 2 * e + 1] = f.y + nt[8 * q + 2 * e + 1];
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        *reinterpret_cast<uint4*>(s + SL_Q0 + swz(t, 2 * quarter + q)) = pack8_half(&n2[8 * q]);
        *reinterpret_cast<uint4*>(s + SL_Q1 + swz(t, 2 * quarter + q)) = pack8_half(&z[8 * q]);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // Round 3.
    if (tid == 0) {
      tc_fence_after();
      tc_mma4(tmem + COL_D1, dK(so + SL_Q0), 2, dMN(so + SL_Q1, kTile), 128, id_mnB64, 0);
      tc_commit(&sh.bar_l2);
    }
    if (!wait_bar(&sh.bar_l2, ph_l2)) return false;
    ph_l2 ^= 1;
    tc_fence_after();
    if (rt) {
      float d[16], o1[16], o2[16];
      tmem_ld16(lrow + COL_D1 + 16 * quarter, d);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a1 = *reinterpret_cast<const float4*>(&sh.sT1[16 * quarter + 4 * q]);
        const float4 a2 = *reinterpret_cast<const float4*>(&sh.bet[16 * quarter + 4 * q]);
        const float s1[4] = {a1.x, a1.y, a1.z, a1.w}, s2[4] = {a2.x, a2.y, a2.z, a2.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float tv = z[4 * q + e] + d[4 * q + e];
          o1[4 * q + e] = tv * s1[e];
          o2[4 * q + e] = tv * s2[e];
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        *reinterpret_cast<uint4*>(s + SL_Q0 + swz(t, 2 * quarter + q)) = pack8_half(&o1[8 * q]);
        *reinterpret_cast<uint4*>(s + SL_Q1 + swz(t, 2 * quarter + q)) = pack8_half(&o2[8 * q]);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    return true;
  };
  // W (rows t, K-major) from W^T in TMEM (lane k): element (t, k) of this
  // thread's 16 columns t goes to block k / 64 of the [W | Q~] operand.
  auto write_w = [&]() {
    float x[16];
    tmem_ld16(lane_addr + COL_WT + 16 * quarter, x);
    const int k = v_row, kb = k >> 6, kk = k & 63;
    __half* wb = reinterpret_cast<__half*>(sm + OFF_XB + kb * 16384);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t = 16 * quarter + i;
      wb[(swz(t, kk >> 3) >> 1) + (kk & 7)] = __float2half_rn(x[i]);
    }
  };
  // K~ = diag(exp(G_C - G)) K from the fp16 K of the slot.
  auto build_kt = [&](int ch) {  // warps 1-15 (warp 0 is issuing MMA2)
    if (warp == 0) return;
    const uint8_t* src = sm + slot_off(ch) + SL_K0;
    for (int i = tid - 32; i < 1024; i += kThreads - 32) {
      const int kb = i >> 9, r = (i & 511) >> 3;
      const uint32_t o = static_cast<uint32_t>(i & 511) * 16u;
      const float sc = sh.ksc[r];
      uint4 u = *reinterpret_cast<const uint4*>(src + kb * 16384 + o);
      u.x = scale_half2(u.x, sc);
      u.y = scale_half2(u.y, sc);
      u.z = scale_half2(u.z, sc);
      u.w = scale_half2(u.w, sc);
      *reinterpret_cast<uint4*>(sm + OFF_KT + kb * kTile + o) = u;
    }
  };

  // ---- MMA batches (thread 0) ----
  auto issue_mma1 = [&](int ch) {  // D1 = [K;Q] K^T (bf16 from TMA)
    const uint32_t so = slot_off(ch);
    tc_mma4(tmem + COL_D1, dK(so), 2, dK(so), 2, id_bf16_kk, 0);
    tc_mma4(tmem + COL_D1, dK(so + 16384), 2, dK(so + 16384), 2, id_bf16_kk, 1);
    tc_commit(&sh.bar_1);
  };
  auto issue_mma2 = [&](int ch) {  // W^T = K^T T'^T, U~^T = V^T T''^T
    const uint32_t so = slot_off(ch);
    tc_mma4(tmem + COL_WT, dMN(so + SL_K0, 16384), 128, dK(so + SL_Q0), 2, id_mnA, 0);
    tc_mma4(tmem + COL_UT, dMN(so + SL_V0, kTile), 128, dK(so + SL_Q1), 2, id_mnA, 0);
    tc_commit(&sh.bar_2);
  };
  auto issue_x = [&]() {  // [X1 | O] = S0 [W; Q~]^T  (A = S0 from TMEM)
    tc_mma4_ts(tmem + COL_X1, tmem + COL_S16, 8, dK(OFF_XB), 2, id_kk128, 0);
    tc_mma4_ts(tmem + COL_X1, tmem + COL_S16 + 32, 8, dK(OFF_XB + 16384), 2, id_kk128, 1);
    tc_commit(&sh.bar_x);
  };
  auto issue_su = [&](int c) {  // SU = U^T K~, O += U^T P^T  (A = U from TMEM)
    tc_mma4_ts(tmem + COL_SU, tmem + COL_U, 8, dMN(OFF_KT, kTile), 128, id_mnB128, 0);
    tc_mma4_ts(tmem + COL_O, tmem + COL_U, 8, dK(OFF_P + (c & 1) * kTile), 2, id_kk64, 1);
    tc_commit(&sh.bar_s);
  };

  // ------------------------------------------------------------ prologue ----
  if (tid == 0) {
    issue_tma(0);
    if (nchunks > 1) issue_tma(1);
  }
  prefetch_gates(0);
  float gamC = 1.f;
  do {
    if (!wait_bar(&sh.bar_tma[0], 0)) { failed = true; break; }
    gates();
    cvt_tile(SL_V0, kTile, SL_V0, kTile, 1.f, row_ok(0));
    if (tid == 0) {
      tc_fence_after();
      issue_mma1(0);
    }
    __syncthreads();
    cvt_tile(OFF_XB + kTile, 16384, SL_Q0, 16384, sh.gam[cr], row_ok(0));
    if (!wait_bar(&sh.bar_1, ph_1)) { failed = true; break; }
    ph_1 ^= 1;
    tc_fence_after();
    build_AP(0);
    cvt_tile(SL_K0, 16384, SL_K0, 16384, 1.f, row_ok(0));
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid < 64) inverse_l0();
    __syncthreads();
    if (!inverse_rest(0)) { failed = true; break; }
    if (tid == 0) {
      tc_fence_after();
      issue_mma2(0);
    }
    build_kt(0);
    if (!wait_bar(&sh.bar_2, ph_2)) { failed = true; break; }
    ph_2 ^= 1;
    tc_fence_after();
    {
      write_w();
    }
    gamC = sh.gam[63];
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
  } while (0);

  // ---------------------------------------------------------------- loop ----
  // Iteration c runs the state chain of chunk c and the prep of chunk p = c+1.
  // A tcgen05.ld waits for every MMA issued before it, so each TMEM read comes
  // right after the batch it needs, with shared-memory-only work in between.
  for (int c = 0; c < nchunks && !failed; ++c) {
    const int p = c + 1;
    const bool has_p = p < nchunks;
    const uint32_t sop = slot_off(p);
    // [A] TMA two chunks ahead; chain MMAs X1 = S0 W^T, O = S0 Q~^T.
    if (tid == 0) {
      if (c + 2 < nchunks) issue_tma(c + 2);
      tc_fence_after();
      issue_x();
    }
    if (has_p) prefetch_gates(p);
    // [B] prep p (shared memory only): gates, V -> fp16, K~ source rows.
    if (has_p) {
      if (!wait_bar(&sh.bar_tma[p & 1], (p >> 1) & 1)) { failed = true; break; }
      gates();
      cvt_tile_w(p, sop + SL_V0, kTile, sop + SL_V0, kTile, nullptr);
      __syncthreads();
    }
    // [C] chain c: U = U~ - X1; then SU = U^T K~, O += U^T P^T and MMA1 of p.
    if (!wait_bar(&sh.bar_x, ph_x)) { failed = true; break; }
    ph_x ^= 1;
    tc_fence_after();
    {
      float xu[16], xw[16];
      tmem_ld16(lane_addr + COL_UT + 16 * quarter, xu);
      tmem_ld16(lane_addr + COL_X1 + 16 * quarter, xw);
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) w[q] = pack_half2(xu[2 * q] - xw[2 * q], xu[2 * q + 1] - xw[2 * q + 1]);
      tmem_st8(lane_addr + COL_U + 8 * quarter, w);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      issue_su(c);
      if (has_p) issue_mma1(p);
    }
    // [C'] prep p (shared memory only, X(c) has finished reading Q~): Q~ of p.
    if (has_p) cvt_tile_w(p, OFF_XB + kTile, 16384, sop + SL_Q0, 16384, sh.gam);
    // [F1] chain c: S <- gamma_C S + SU (registers), outputs into the U tile.
    if (!wait_bar(&sh.bar_s, ph_s)) { failed = true; break; }
    ph_s ^= 1;
    tc_fence_after();
    {
      float x[32];
      tmem_ld32(lane_addr + COL_SU + 32 * quarter, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] = fmaf(gamC, S[i], x[i]);
      float y[16];
      tmem_ld16(lane_addr + COL_O + 16 * quarter, y);
      __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_U);
#pragma unroll
      for (int i = 0; i < 16; ++i) ost[(16 * quarter + i) * 128 + v_row] = __float2bfloat16_rn(a.scale * y[i]);
    }
    // [D] prep p: A and P from MMA1, K -> fp16 in place.
    if (has_p) {
      if (!wait_bar(&sh.bar_1, ph_1)) { failed = true; break; }
      ph_1 ^= 1;
      tc_fence_after();
      build_AP(p);
      cvt_tile(sop + SL_K0, 16384, sop + SL_K0, 16384, 1.f, row_ok(p));
      fence_proxy_async();
    }
    tc_fence_before();
    __syncthreads();
    // [E0] inverse level 0 (threads 0-63) || output rows of chunk c (the others).
    {
      if (has_p && tid < 64) {
        inverse_l0();
      } else if (tid >= 64) {
        const int lo = chunk_lo(c), hi = chunk_hi(c);
        const int64_t tstride = static_cast<int64_t>(H) * kDimV;
        __nv_bfloat16* obase = a.o + (static_cast<int64_t>(chunk_tf(c)) * H + h) * kDimV;
        const __nv_bfloat16* ost = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_U);
        for (int i = tid - 64; i < 1024; i += kThreads - 64) {
          const int r = i >> 4, part = i & 15;
          if (r >= lo && r < hi)
            *reinterpret_cast<uint4*>(obase + r * tstride + part * 8) =
                *reinterpret_cast<const uint4*>(ost + r * 128 + part * 8);
        }
      }
    }
    __syncthreads();
    stage_state();  // S0 of chunk c+1 into TMEM (X(c) finished reading it)
    // [E] prep p: inverse levels 1-2, T', T''; then MMA2.
    if (has_p) {
      if (!inverse_rest(p)) { failed = true; break; }
      if (tid == 0) {
        tc_fence_after();
        issue_mma2(p);
      }
    }
    // [G1] while MMA2 runs: checkpoint of chunk c, K~ of p (SU(c) has finished).
    {
      const int a_end = chunk_a0(c) + kChunk;
      if (ck_rows && ck_pool && a_end % N == 0 && a_end <= end_pos) {
        const int row = ck_rows[a_end / N - 1 - first_ck];
        if (row >= 0) store_state(ck_pool, row);
      }
    }
    float gamC_next = gamC;
    if (has_p) {
      build_kt(p);
      // [G2] W^T of p -> fp16 rows k.
      if (!wait_bar(&sh.bar_2, ph_2)) { failed = true; break; }
      ph_2 ^= 1;
      tc_fence_after();
      write_w();
      gamC_next = sh.gam[63];
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    gamC = gamC_next;
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
