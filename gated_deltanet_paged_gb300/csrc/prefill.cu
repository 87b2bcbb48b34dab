// prefill.cu -- chunked paged GDN prefill on tcgen05 tensor cores: the state
// chain, plus the C-ABI entry points of the prefill.
//
// "flashinfer.gdn_paged": chunk_gated_delta_rule_paged, the prefill bullets,
// the 64-token left-padding paragraph, and "Slot arguments of
// chunk_gated_delta_rule" (read / final / checkpoint rows, -1 = zero state or
// skip, checkpoints at absolute positions (prefix + n) % N == 0).
//
// Method (gated delta rule, chunked).  Per (sequence, head) chain and 64-token
// chunk with rows t = 0..63, cumulative gate G_t = g_0 + ... + g_t (rows outside
// the sequence have g = beta = 0 and k = v = 0, so they are the identity),
// gamma_t = exp(G_t), S0 the V x K state at the chunk start and
// T'' = (I + A)^-1 diag(beta) and -W from the chunk-local kernel (ut.cu):
//   W     = T'' diag(gamma) K,  U~ = T'' V
//   U     = U~ - W S0^T                            (the chunk's new values)
//   O[t]  = scale (gamma_t S0 q_t + sum_{j<=t} exp(G_t - G_j)(q_t . k_j) U[j])
//   S1    = gamma_C S0 + U^T diag(exp(G_C - G_j)) K
// which equals the token-by-token recurrence up to rounding.
//
// Mapping.  One CTA (16 warps) per chain, chains ordered by decreasing length;
// the warps are specialised and hand work to each other through mbarriers.
// The chain runs transposed: TMEM lane = state row v, so the state and U^T
// are fp16 A operands in TMEM and never pass through shared memory.
//   - warps 0-7, "chain": the fp32 state in registers (thread = state row v,
//     64 columns), U^T packed in place in TMEM, the state update and its fp16
//     copy, the outputs and the page-boundary / final state stores; Q~ and K~
//     of the next chunk, and the -W and K refills they are first to learn
//     about;
//   - warps 8-13, "prep": gates, V -> fp16 and P (decayed, masked Q K^T) of the
//     next chunk while the chain works on the current one;
//   - warp 14 issues the preparation's MMAs, warp 15 the chain's (and the V,
//     T'' and Q refills, off the chain threads' path).  A thread's MMA issue
//     runs almost in step with the tensor core, so one issuer would let a
//     preparation MMA hold up a chain MMA for its whole duration.
// Per chunk (M = 128 = state rows v, fp32 accumulators in TMEM; the U half of
// D_X is its columns 0-63 for even chunks, 64-127 for odd ones):
//   prep : D_P  = Q K^T                        (M = 64, bf16 from TMA)
//          D_X(U half) = V^T T''^T                   (U~^T; the chain threads zero
//                                                      the O half after reading it)
//   chain: D_X += S0 [-W; Q~]^T or S0 [Q~; -W]^T      (U half: U^T; O half:
//                                                      (Q~ S0^T)^T)
//          D_SU = U^T K~;  D_X(O half) += U^T P^T
// T'' arrives by columns (tile row j = column j), i.e. as an N-major B operand.
// Operands are fp16 (an
// 11-bit significand keeps written states within 1e-3 relative error; bf16
// would not) except Q K^T, which uses the bf16 tiles as loaded.
#include <math.h>

#include <atomic>
#include <mutex>

#include "prefill_common.cuh"

namespace {

using namespace gdn;

constexpr int kThreads = 512;
constexpr int kPrepThreads = 192;  // warps 8-13
constexpr int kPrepIssuerWarp = 14;
constexpr int kIssuerWarp = 15;
constexpr uint32_t kTile = 8192;  // 64 rows x 128 B

// Shared memory (byte offsets from the 1024-aligned base).
constexpr uint32_t OFF_Q = 0;         // 2 x Q bf16 [kb0 | kb1], by chunk parity
constexpr uint32_t OFF_K = 32768;     // 2 x K [kb0 | kb1]: bf16 -> K~ (fp16), in place; by chunk parity
constexpr uint32_t OFF_V = 65536;     // 2 x V [kb0 | kb1]: bf16 -> fp16, in place
constexpr uint32_t OFF_TZT = 98304;   // T''(even chunk) | unused 8 KB | T''(odd chunk), by columns
constexpr uint32_t OFF_P = 122880;    // 2 x P (rows t, K-major), by chunk parity
constexpr uint32_t OFF_XA = 139264;   // per K block (32 KB apart): -W (even) | Q~ (even) | Q~ (odd) | -W (odd)
constexpr uint32_t OFF_OST = 204800;  // outputs of a full chunk: 2 KB per chain warp (32 tokens x 32 columns, bf16)
constexpr uint32_t OFF_SMALL = 221184;

// TMEM columns (lane = state row v).
constexpr uint32_t COL_DX = 0;     // two 128-column accumulators S0 [XA rows]^T, by chunk parity
constexpr uint32_t COL_DSU = 256;  // U^T K~
constexpr uint32_t COL_DP = 384;   // Q K^T of the chunk being prepared (M = 64: row t in lane 32 (t / 16) + t % 16)
constexpr uint32_t COL_SA = 448;   // S0 in fp16 pairs: the A operand of S0 [XA rows]^T
constexpr uint32_t TMEM_COLS = 512;

struct Gates {       // of the chunk being prepared
  float G[64];       // cumulative gate
  float e[64];       // exp(g)
  float gam[2][64];  // exp(G), by chunk parity
  float ksc[2][64];  // exp(G_C - G), by chunk parity
};

struct Small {
  Gates gates;
  float gamC[4];  // exp(G_C) by chunk, ring of 3 (read by the chain)
  // TMA completion
  uint64_t bar_q[2], bar_v[2], bar_t[2], bar_k[2], bar_w[2];
  // MMA completion (tcgen05.commit)
  uint64_t bar_p[2], bar_m2[2], bar_x[2], bar_su[2], bar_o[2];
  // hand-offs between warp groups
  uint64_t xa_full, mp_ready, m2_ready, u_ready, s16_ready, gates_ready[2], kt_ready[2], o_read[2];
  uint64_t p_ready[2];          // P of a chunk written (the prep's TMEM readers), by parity
  uint64_t stall;               // the test hook's barrier, never completed
  uint32_t tmem_base;
  int seq;
  int flag;
  int abort;
};
constexpr uint32_t SMALL_BYTES = ((sizeof(Small) + 127) / 128) * 128;
// Dynamic shared memory requested: the tiles, the small block and slack to
// align the base to 1024 B.  Stays below the 227 KB a CTA may use.
constexpr uint32_t SMEM_BYTES = OFF_SMALL + SMALL_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448, "prefill shared memory above the per-CTA limit");

__device__ __forceinline__ uint4 pack8h(const float* x) {
  uint4 u;
  u.x = pack_half2(x[0], x[1]);
  u.y = pack_half2(x[2], x[3]);
  u.z = pack_half2(x[4], x[5]);
  u.w = pack_half2(x[6], x[7]);
  return u;
}

// Largest magnitude an fp16 tensor-core operand holds.
constexpr float kF16Max = 65504.f;

// bf16 x 8 -> fp16 x 8 times sc (zeros unless keep); src may equal dst.  With
// check, an input element of magnitude above the fp16 range sets bad.
__device__ __forceinline__ void cvt8(uint8_t* dst, const uint8_t* src, float sc, bool keep, bool check,
                                     bool& bad) {
  uint4 out = make_uint4(0u, 0u, 0u, 0u);
  if (keep) {
    const uint4 in = *reinterpret_cast<const uint4*>(src);
    const float2 f0 = unpack_bf162(in.x), f1 = unpack_bf162(in.y), f2 = unpack_bf162(in.z), f3 = unpack_bf162(in.w);
    if (check) {
      const float m = fmaxf(fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y))),
                            fmaxf(fmaxf(fabsf(f2.x), fabsf(f2.y)), fmaxf(fabsf(f3.x), fabsf(f3.y))));
      bad |= !(m <= kF16Max);  // NaN inputs too
    }
    out.x = pack_half2(f0.x * sc, f0.y * sc);
    out.y = pack_half2(f1.x * sc, f1.y * sc);
    out.z = pack_half2(f2.x * sc, f2.y * sc);
    out.w = pack_half2(f3.x * sc, f3.y * sc);
  }
  *reinterpret_cast<uint4*>(dst) = out;
}

// The same on a loaded piece, returning the converted one; the products run as
// paired fp32 multiplies (each half rounds as a scalar multiply would).
__device__ __forceinline__ uint4 cvt8v(const uint4 in, float sc, bool keep, bool check, bool& bad) {
  uint4 out = make_uint4(0u, 0u, 0u, 0u);
  if (keep) {
    const float2 f0 = unpack_bf162(in.x), f1 = unpack_bf162(in.y), f2 = unpack_bf162(in.z), f3 = unpack_bf162(in.w);
    if (check) {
      const float m = fmaxf(fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y))),
                            fmaxf(fmaxf(fabsf(f2.x), fabsf(f2.y)), fmaxf(fabsf(f3.x), fabsf(f3.y))));
      bad |= !(m <= kF16Max);  // NaN inputs too
    }
    const float2 s2 = make_float2(sc, sc);
    out.x = pack_half2(__fmul2_rn(f0, s2));
    out.y = pack_half2(__fmul2_rn(f1, s2));
    out.z = pack_half2(__fmul2_rn(f2, s2));
    out.w = pack_half2(__fmul2_rn(f3, s2));
  }
  return out;
}

// kCheck: compiled with the fp16-range and finite-state checks (err_word
// given); without them the hot loops carry no code for the checks.  kBf16:
// pools of bf16 states (else fp32).  The hot loops carry only the code of
// their own variant.
template <bool kCheck, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_t,
                   const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_w,
                   const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  Small& sh = *reinterpret_cast<Small*>(sm + OFF_SMALL);
  volatile int* abort_flag = &sh.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  const int rank = blockIdx.x / H, h = blockIdx.x % H;
  pdl_wait();  // the chunk-local kernel (and everything before it on the stream) is done
  pdl_launch_dependents();

  // ---- pick the sequence: rank-th longest (ties by index) ----
  if (a.num_seqs > 1 && a.num_seqs < 4096) {
    int* cu_s = reinterpret_cast<int*>(sm + OFF_XA);
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
  const void* ck_rows = nullptr;  // j-th checkpoint row = index_at(ck_rows, ck_off + j, ck_wide)
  int64_t ck_off = 0;
  int32_t ck_wide = 0;
  int N = a.N;
  if (a.indptr) {
    const int i0 = a.indptr[b], i1 = a.indptr[b + 1];
    const int n = i1 - i0;
    const int lpl = a.last_len[b];
    const long long tot = static_cast<long long>(n - 1) * a.page_size + lpl;
    if (n < 1 || lpl < 1 || lpl > a.page_size || tot < L || tot > 0x3FFFFFFFLL) {
      if (tid == 0) record_error(a.err_word, GDN_DEVERR_PAGE_TABLE, b);
      return;
    }
    P = static_cast<int>(tot - L);
    in_row = P > 0 ? a.pages[i0 + (P - 1) / a.page_size] : -1;
    out_row = a.pages[i1 - 1];
    ck_rows = a.pages;
    ck_off = i0 + P / a.page_size;
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
    const int64_t p64 = a.prefix_lens ? index_at(a.prefix_lens, b, a.index64) : 0;
    const int64_t in64 = a.state_indices ? index_at(a.state_indices, b, a.index64) : -1;
    const int64_t out64 = a.output_state_indices ? index_at(a.output_state_indices, b, a.index64) : -1;
    if (a.state_checkpoints) {
      ck_rows = a.checkpoint_state_indices;
      ck_off = index_at(a.checkpoint_cu_starts, b, a.index64);
      ck_wide = a.index64;
    }
    if (p64 < 0 || p64 + L > 0x3FFFFFFFLL) {
      if (tid == 0) record_error(a.err_word, GDN_DEVERR_PAGE_TABLE, b);
      return;
    }
    P = static_cast<int>(p64);
    if (a.index64) {
      // int64 slot entries: every row this sequence uses, and its first
      // checkpoint entry, must lie in the int32 range (rows >= -1).
      if (tid == 0) {
        constexpr int64_t kMax = 0x7FFFFFFFLL;
        int bad = in64 < -1 || in64 > kMax || out64 < -1 || out64 > kMax;
        if (ck_rows && a.N > 0) {
          const int64_t nck = (p64 + L) / a.N - p64 / a.N;
          bad |= ck_off < 0 || ck_off > kMax;
          for (int64_t j = 0; j < nck && !bad; ++j) {
            const int64_t r = index_at(ck_rows, ck_off + j, 1);
            bad |= r < -1 || r > kMax;
          }
        }
        sh.flag = bad;
        if (bad) record_error(a.err_word, GDN_DEVERR_INDEX_RANGE, b);
      }
      __syncthreads();
      if (sh.flag) return;
    }
    in_row = static_cast<int>(in64);
    out_row = static_cast<int>(out64);
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

  if (a.debug_stall) {
    // Test hook: one wait that runs out (about 1 ms), taken before any copy,
    // MMA or TMEM allocation, so that nothing is in flight when the CTA leaves.
    if (tid == 0) {
      mbar_init(&sh.stall, 1);
      fence_mbar_init();
      sh.flag = mbar_wait(&sh.stall, 0, 1000000ull) ? 0 : 1;
    }
    __syncthreads();
    if (sh.flag) {
      if (tid == 0) record_error(a.err_word, GDN_DEVERR_TIMEOUT, b);
      return;
    }
  }

  const int end_pos = P + L;
  const int first_pos = (P / kChunk) * kChunk;
  const int nch = chunk_count(P, L);
  const int first_ck = (ck_rows && N > 0) ? P / N : 0;
  const int slot0 = slot_base(cu_b, b);

  // ---- set-up: barriers, TMEM ----
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.bar_q[i], 1);
      mbar_init(&sh.bar_w[i], 1);
      mbar_init(&sh.bar_v[i], 1);
      mbar_init(&sh.bar_t[i], 1);
      mbar_init(&sh.bar_o[i], 1);
      mbar_init(&sh.o_read[i], 256);
      mbar_init(&sh.bar_p[i], 1);
      mbar_init(&sh.bar_x[i], 1);
      mbar_init(&sh.bar_su[i], 1);
      mbar_init(&sh.gates_ready[i], 1);
      mbar_init(&sh.kt_ready[i], 256);
      mbar_init(&sh.bar_m2[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sh.bar_k[i], 1);
    mbar_init(&sh.xa_full, 256);  // every chain thread writes a share of Q~
    mbar_init(&sh.mp_ready, 1);
    mbar_init(&sh.m2_ready, kPrepThreads);  // every preparation thread converts a share of V
    mbar_init(&sh.u_ready, 256);
    mbar_init(&sh.s16_ready, 256);
    mbar_init(&sh.p_ready[0], 128);
    mbar_init(&sh.p_ready[1], 128);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  // Geometry of chunk ch: absolute position of row 0, valid rows [lo, hi),
  // packed token index of row 0.
  auto chunk_a0 = [&](int ch) { return first_pos + kChunk * ch; };
  auto chunk_lo = [&](int ch) { return max(P - chunk_a0(ch), 0); };
  auto chunk_hi = [&](int ch) { return min(end_pos - chunk_a0(ch), kChunk); };
  auto chunk_tf = [&](int ch) { return cu_b + (chunk_a0(ch) - P); };
  auto kslot = [&](int ch) { return OFF_K + static_cast<uint32_t>(ch & 1) * 16384u; };
  auto vslot = [&](int ch) { return OFF_V + static_cast<uint32_t>(ch & 1) * 16384u; };
  auto tslot = [&](int ch) { return OFF_TZT + static_cast<uint32_t>(ch & 1) * 16384u; };
  auto dK = [&](uint32_t off) { return sdesc(sbase + off, 16, 1024); };
  auto dMN = [&](uint32_t off, uint32_t lbo) { return sdesc(sbase + off, lbo, 1024); };
  const int64_t head_off = static_cast<int64_t>(h) * kDimV * kDimK;

  auto tma_rows = [&](const CUtensorMap* map, uint32_t dst, uint64_t* bar, int ch) {
    tma_load_3d(sm + dst, map, bar, 0, h, chunk_tf(ch));
    tma_load_3d(sm + dst + kTile, map, bar, 64, h, chunk_tf(ch));
  };
  auto qslot = [&](int ch) { return OFF_Q + static_cast<uint32_t>(ch & 1) * 16384u; };
  auto tma_q = [&](int ch) {
    mbar_arrive_expect_tx(&sh.bar_q[ch & 1], 16384);
    tma_rows(&tm_q, qslot(ch), &sh.bar_q[ch & 1], ch);
  };
  // Slot refills, each issued by a thread that learns early that the slot is
  // free: -W after X, K after U^T K~ (chain thread 0); V and T'' after U~, Q
  // after Q~ and Q K^T (the chain issuer, after X).
  auto tma_k = [&](int ch) {
    mbar_arrive_expect_tx(&sh.bar_k[ch & 1], 16384);
    tma_rows(&tm_k, kslot(ch), &sh.bar_k[ch & 1], ch);
  };
  auto tma_v = [&](int ch) {
    mbar_arrive_expect_tx(&sh.bar_v[ch & 1], 16384);
    tma_rows(&tm_v, vslot(ch), &sh.bar_v[ch & 1], ch);
  };
  auto tma_t = [&](int ch) {
    mbar_arrive_expect_tx(&sh.bar_t[ch & 1], kTinvBytes);
    tma_load_2d(sm + tslot(ch), &tm_t, &sh.bar_t[ch & 1], 0, ((slot0 + ch) * H + h) * 64);
  };
  // -W of chunk ch straight into its -W buffer of the X operand (by chunk parity).
  auto tma_w = [&](int ch) {
    const uint32_t dst = OFF_XA + static_cast<uint32_t>(ch & 1) * 24576u;
    const int row = ((slot0 + ch) * H + h) * 64;
    uint64_t* bar = &sh.bar_w[ch & 1];
    mbar_arrive_expect_tx(bar, kWBytes);
    tma_load_2d(sm + dst, &tm_w, bar, 0, row);
    tma_load_2d(sm + dst + 32768, &tm_w, bar, 64, row);
  };

  // With err_word: q, k and v elements beyond the fp16 range (the tensor-core
  // operands are fp16) and non-finite stored states are reported.
  constexpr bool check_range = kCheck;
  bool range_bad = false;

  // Two issuing warps, so that an MMA of the preparation never holds up one of
  // the chain (a thread's issue runs almost in step with the tensor core).  Each
  // stream's operations come in a fixed order, so its issuing thread sleeps in
  // the wait for the next one's inputs.
  if (warp == kIssuerWarp) {
    // ========================================================== chain issuer
    // Per chunk (M = 128 = state rows v, fp32 in TMEM; e = chunk parity; the U
    // half of D_X is columns 0-63 for even chunks, 64-127 for odd ones):
    //   D_X  += S0 [XA rows]^T      A: S0 fp16 (TMEM), B: [-W; Q~] or [Q~; -W]
    //   D_SU  = U^T K~              A: U^T fp16 (TMEM, over the U half), B: K~
    //   D_X(O half) += U^T P^T      A: U^T, B: P (rows t)
    // U^T sits in columns [0, 16) and [32, 48) of the U half (each chain thread
    // packs its 32 values in place), so its K = 64 runs as two pairs of steps.
    const uint32_t id_x = idesc_f16(128, 128, false, false, false, false);
    const uint32_t id_su = idesc_f16(128, 128, false, false, false, true);
    const uint32_t id_o = idesc_f16(128, 64, false, false, false, false);
    if (lane == 0) {
      auto w = [&](uint64_t* bar, uint32_t parity) { return mbar_wait_or_abort(bar, parity, abort_flag); };
      for (int c = 0; c < nch; ++c) {
        const uint32_t e = c & 1, ph = (c >> 1) & 1;
        const uint32_t d = tmem + COL_DX + 128 * e;
        const uint32_t ua = d + 64 * e;         // U half
        const uint32_t od = d + 64 * (1 - e);  // O half
        // the state copy (s16_ready) is normally the last of these to complete
        if (!w(&sh.bar_w[e], ph) || !w(&sh.bar_m2[e], ph) || !w(&sh.xa_full, e) || !w(&sh.s16_ready, e)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        tc_mma4_ts(d, tmem + COL_SA, 8, dK(OFF_XA + 16384 * e), 2, id_x, 1);
        tc_mma4_ts(d, tmem + COL_SA + 32, 8, dK(OFF_XA + 32768 + 16384 * e), 2, id_x, 1);
        tc_commit(&sh.bar_x[e]);
        if (c + 2 < nch) {  // U~ of chunk c has read its V and T'' slots
          tma_v(c + 2);
          tma_t(c + 2);
          // Q of chunk c+2 into the slot of chunk c: Q~ of chunk c (waited for
          // above) and Q K^T of chunk c have read it
          if (!w(&sh.bar_p[e], ph)) {
            *abort_flag = 1;
            break;
          }
          tma_q(c + 2);
        }
        if (!w(&sh.kt_ready[e], ph) || !w(&sh.u_ready, e)) {  // U^T (u_ready) is normally last
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint64_t bk = dMN(kslot(c), kTile), bp = dK(OFF_P + 8192 * e);
        tc_mma2_ts(tmem + COL_DSU, ua, 8, bk, 128, id_su, 0);
        tc_mma2_ts(tmem + COL_DSU, ua + 32, 8, bk + 256, 128, id_su, 1);
        tc_commit(&sh.bar_su[e]);
        if (!w(&sh.p_ready[e], ph)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        tc_mma2_ts(od, ua, 8, bp, 2, id_o, 1);
        tc_mma2_ts(od, ua + 32, 8, bp + 4, 2, id_o, 1);
        tc_commit(&sh.bar_o[e]);
      }
    }
    __syncwarp();
  } else if (warp == kPrepIssuerWarp) {
    // =========================================================== prep issuer
    //   D_P  = Q K^T                           (M = 64, bf16 from TMA)
    //   D_X(U half) = V^T T''^T                (U~^T)
    const uint32_t id_m2 = idesc_f16(128, 64, false, false, true, true);
    const uint32_t id_qk = idesc_f16(64, 64, true, true, false, false);
    // Q K^T is committed only once the chunk's V conversion is in (m2_ready):
    // the preparation threads learn of it (bar_p) before they can arrive on
    // m2_ready or mp_ready for the next chunk, so neither barrier can run a
    // phase ahead of this thread.
    if (lane == 0) {
      auto w = [&](uint64_t* bar, uint32_t parity) { return mbar_wait_or_abort(bar, parity, abort_flag); };
      for (int p = 0; p < nch; ++p) {
        const uint32_t e = p & 1, ph = (p >> 1) & 1;
        if (!w(&sh.mp_ready, e) || !w(&sh.bar_q[e], ph) || !w(&sh.bar_k[e], ph)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        tc_mma4(tmem + COL_DP, dK(qslot(p)), 2, dK(kslot(p)), 2, id_qk, 0);
        tc_mma4(tmem + COL_DP, dK(qslot(p) + kTile), 2, dK(kslot(p) + kTile), 2, id_qk, 1);
        // U~ = T'' V once V is in fp16, T'' has landed and the O readout of chunk
        // p-2 has emptied this D_X half
        if (!w(&sh.m2_ready, e)) {
          *abort_flag = 1;
          break;
        }
        tc_commit(&sh.bar_p[e]);
        if (!w(&sh.bar_t[e], ph) || (p >= 2 && !w(&sh.o_read[e], ph ^ 1))) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        tc_mma4(tmem + COL_DX + 192 * e, dMN(vslot(p), kTile), 128, dMN(tslot(p), kTile), 128, id_m2, 0);
        tc_commit(&sh.bar_m2[e]);
      }
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ================================================================== prep
    const int pt = tid - 256, pw = warp - 8;
    const int wq = warp & 3;
    const bool tm_reader = warp < 12;  // warps 8-11: one per TMEM lane quarter (rows 16 wq .. 16 wq + 15 of D_P)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * wq) << 16);
    // Every thread waits for what it needs itself; a thread whose wait fails
    // skips its work, and the group agrees on stopping once per chunk, at the
    // barrier that closes it.
    bool ok = true;
    auto pwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (ok && !mbar_wait_or_abort(bar, parity, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
      tc_fence_after();
      return ok;
    };
    // The same without the tcgen05 fence, for waits followed by shared-memory
    // work only (the next TMEM access or MMA comes after a fenced wait).
    auto pwait_nf = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (ok && !mbar_wait_or_abort(bar, parity, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
      return ok;
    };
    auto pclose = [&]() -> bool {
      uint32_t any;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\t"
          "bar.red.or.pred q, 2, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
          : "=r"(any)
          : "r"(ok ? 1u : 0u), "r"(kPrepThreads)
          : "memory");
      return any == 0;
    };
    if (pt == 0) {
      prefetch_tensormap(&tm_o);
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_t);
      prefetch_tensormap(&tm_w);
      tma_q(0);
      tma_k(0);
      tma_v(0);
      tma_t(0);
      tma_w(0);
      if (nch > 1) {
        tma_q(1);
        tma_k(1);
        tma_v(1);
        tma_t(1);
        tma_w(1);
      }
    }
    // Gates: warp 8 holds g of rows 2 lane and 2 lane + 1 of the next chunk.
    float pg0 = 0.f, pg1 = 0.f;
    auto prefetch_g = [&](int ch) {
      if (pw == 0 && ch < nch) {
        const int lo = chunk_lo(ch), hi = chunk_hi(ch);
        const int64_t tf = chunk_tf(ch);
        const int r0 = 2 * lane, r1 = 2 * lane + 1;
        pg0 = (r0 >= lo && r0 < hi) ? a.g[(tf + r0) * H + h] : 0.f;
        pg1 = (r1 >= lo && r1 < hi) ? a.g[(tf + r1) * H + h] : 0.f;
      }
    };
    prefetch_g(0);
    for (int p = 0; p < nch; ++p) {
      const uint32_t e = p & 1;
      const int lo = chunk_lo(p), hi = chunk_hi(p);
      Gates& gs = sh.gates;
      // 1. warp 8: cumulative gate of chunk p and its tables (slot e: K~ of chunk
      //    p-2 has finished with its exp(G_C - G)); Q K^T may start once Q and K
      //    are in (it has its own TMEM columns)
      if (pw == 0) {
        // warp-uniform, so that the shuffles below see every lane
        const bool go = __all_sync(0xffffffffu, p < 2 || pwait_nf(&sh.kt_ready[e], ((p - 2) >> 1) & 1));
        float s = go ? pg0 + pg1 : 0.f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, s, off);
          if (lane >= off) s += y;
        }
        const float G0 = s - pg1, G1 = s;
        const float GC = __shfl_sync(0xffffffffu, s, 31);
        if (go) {
          gs.G[2 * lane] = G0;
          gs.G[2 * lane + 1] = G1;
          gs.e[2 * lane] = __expf(pg0);
          gs.e[2 * lane + 1] = __expf(pg1);
          gs.gam[e][2 * lane] = __expf(G0);
          gs.gam[e][2 * lane + 1] = __expf(G1);
          gs.ksc[e][2 * lane] = __expf(GC - G0);
          gs.ksc[e][2 * lane + 1] = __expf(GC - G1);
          if (lane == 0) sh.gamC[p % 3] = __expf(GC);
          prefetch_g(p + 1);
        }
        __syncwarp();
        // (Q and K of chunk p are waited for by the threads that read them: the
        // prep issuer before Q K^T, the chain threads before Q~)
        if (lane == 0 && go) {
          mbar_arrive(&sh.mp_ready);
          mbar_arrive(&sh.gates_ready[e]);
        }
      }
      // 2. V -> fp16 in place; U~ = T'' V follows (its issuer waits for T'' and
      //    for the chunk's D_X half)
      if (pwait_nf(&sh.bar_v[e], (p >> 1) & 1)) {
        for (int i = pt; i < 1024; i += kPrepThreads) {
          const int row = (i & 511) >> 3;
          uint8_t* ptr = sm + vslot(p) + (i >> 9) * kTile + (i & 511) * 16;
          cvt8(ptr, ptr, 1.f, row >= lo && row < hi, check_range, range_bad);
        }
        fence_proxy_async();
        mbar_arrive(&sh.m2_ready);
      }
      // 3. P = decayed, masked Q K^T (warps 8-11, a thread per row and half) once U^T P^T of chunk p-2
      //    has read this P tile; warps other than 8 read its gate tables
      if (tm_reader && (p < 2 || pwait_nf(&sh.bar_o[e], ((p - 2) >> 1) & 1)) &&
          (pw == 0 || pwait_nf(&sh.gates_ready[e], (p >> 1) & 1)) &&
          pwait(&sh.bar_p[e], (p >> 1) & 1)) {  // one tcgen05 fence, after the last wait, before the TMEM load
        const int t = 16 * wq + (lane & 15), ph = lane >> 4;  // row t, columns 32 ph ..
        float x[32];
        tmem_ld16x32bx2_32(lane_addr + COL_DP, x);
        float out[32];
        const int j0 = 32 * ph;
        const int jmax = min(j0 + 31, t);
        if (t >= lo && t < hi && jmax >= j0) {
          // exp(G_t - G_j) by a running product downwards from j = jmax; the
          // products with Q K^T in pairs (paired fp32 multiplies)
          float ev[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 e4 = *reinterpret_cast<const float4*>(&gs.e[j0 + 4 * i]);
            ev[4 * i] = e4.x;
            ev[4 * i + 1] = e4.y;
            ev[4 * i + 2] = e4.z;
            ev[4 * i + 3] = e4.w;
          }
          float cur = __expf(gs.G[t] - gs.G[jmax]);
#pragma unroll
          for (int i = 15; i >= 0; --i) {
            const int ja = j0 + 2 * i, jb = ja + 1;
            const float cb = cur;
            if (jb <= jmax) cur *= ev[2 * i + 1];
            const float ca = cur;
            if (ja <= jmax) cur *= ev[2 * i];
            const float2 pr = __fmul2_rn(make_float2(ca, cb), make_float2(x[2 * i], x[2 * i + 1]));
            out[2 * i] = (ja <= jmax && ja >= lo) ? pr.x : 0.f;
            out[2 * i + 1] = (jb <= jmax && jb >= lo) ? pr.y : 0.f;
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) out[jj] = 0.f;
        }
        uint8_t* pb = sm + OFF_P + 8192 * e;
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(pb + swz(t, 4 * ph + c)) = pack8h(&out[8 * c]);
        fence_proxy_async();
        mbar_arrive(&sh.p_ready[e]);  // U^T P^T of chunk p may read it
      }
      tc_fence_before();
      if (!pclose()) break;
    }
    if (range_bad) record_error(a.err_word, GDN_DEVERR_RANGE, b);
  } else {
    // ================================================================= chain
    // Thread (v, hc): state row v (TMEM lane v) and state columns 64 hc .. 64 hc
    // + 63 in registers; of each 64-column half of D_X it reads columns 32 hc ..
    // 32 hc + 31 (tokens t of this chunk).
    const int wq = warp & 3, hc = warp >> 2;
    const int v = 32 * wq + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * wq) << 16);
    bool ok = true;
    // The lanes of a warp wait on the same barrier phase in step, so a wait
    // fails for the whole warp at once and the warp-wide TMEM and stmatrix
    // instructions after it never run with part of the warp.  (Thread 0's
    // extra wait in kt_part can fail alone; the other lanes then meet the abort
    // flag in their next wait, before any warp-wide instruction.)
    auto cwait = [&](uint64_t* bar, uint32_t parity) {
      if (ok && !mbar_wait_or_abort(bar, parity, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
      tc_fence_after();
      return ok;
    };
    // Without the tcgen05 fence: for the waits before the Q~ and K~ conversions,
    // which touch shared memory only.
    auto cwait_nf = [&](uint64_t* bar, uint32_t parity) {
      if (ok && !mbar_wait_or_abort(bar, parity, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
      return ok;
    };
    float S[64];
    // Element offset of this thread's 64 state values (row v, columns 64 hc ..)
    // in pool row `row`; pools hold fp32 or (state_bf16) bf16 elements.
    auto state_off = [&](int row) { return row * a.row_stride + head_off + v * kDimK + 64 * hc; };
    if (in_row >= 0 && kBf16) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(init_pool) +
                                                        state_off(in_row));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 x = src[i];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = unpack_bf162(w[j]);
          S[8 * i + 2 * j] = f.x;
          S[8 * i + 2 * j + 1] = f.y;
        }
      }
    } else if (in_row >= 0) {
      const float4* src = reinterpret_cast<const float4*>(init_pool + state_off(in_row));
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
    // S0 in fp16 pairs: the TMEM A operand of the next S0 [XA rows]^T.
    auto stage_state = [&]() {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_half2(S[32 * hh + 2 * i], S[32 * hh + 2 * i + 1]);
        tmem_st16_nw(lane_addr + COL_SA + 32 * hc + 16 * hh, w);
      }
      tmem_wait_st();
      tc_fence_before();
    };
    // 32 zero columns of this thread's TMEM lane: the O half of D_X, into which X
    // accumulates, is zeroed after each read (and before the first chunks).
    auto zero32 = [&](uint32_t taddr) {
      uint32_t z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0u;
      tmem_st16_nw(taddr, z);
      tmem_st16_nw(taddr + 16, z);
      tmem_wait_st();
    };
    zero32(lane_addr + COL_DX + 64 + 32 * hc);   // O half of even chunks
    zero32(lane_addr + COL_DX + 128 + 32 * hc);  // O half of odd chunks
    stage_state();
    mbar_arrive(&sh.s16_ready);
    // The chain warps' share of the preparation, done while they would otherwise
    // wait.  Q~ of chunk q = diag(gamma) Q goes into its own Q~ tile of XA (by
    // chunk parity; X of chunk q-2 has read it) and releases X of chunk q.  K~
    // of chunk q = diag(exp(G_C - G)) K is converted in place (fp16) once Q K^T
    // has read K, and U^T K~ of chunk q waits for it.  Each thread converts four
    // of the 1024 16-byte pieces of a tile.
    const int ci = tid;  // 0..255
    auto qt_part = [&](int q) -> bool {
      const uint32_t eq = q & 1;
      const int lo = chunk_lo(q), hi = chunk_hi(q);
      if (!cwait_nf(&sh.bar_q[eq], (q >> 1) & 1) || !cwait_nf(&sh.gates_ready[eq], (q >> 1) & 1)) return false;
      const float* gam = sh.gates.gam[eq];
      const uint8_t* src = sm + qslot(q);
      uint4 in[4];
      float sc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // every load before any store
        const int i = ci + 256 * k;
        in[k] = *reinterpret_cast<const uint4*>(src + i * 16);
        sc[k] = gam[(i & 511) >> 3];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = ci + 256 * k;
        const int kb = i >> 9, rc = i & 511, row = rc >> 3;
        *reinterpret_cast<uint4*>(sm + OFF_XA + kb * 32768 + 8192 + 8192 * eq + rc * 16) =
            cvt8v(in[k], sc[k], row >= lo && row < hi, check_range, range_bad);
      }
      fence_proxy_async();
      mbar_arrive(&sh.xa_full);
      return true;
    };
    auto kt_part = [&](int q) -> bool {
      const uint32_t eq = q & 1;
      const int lo = chunk_lo(q), hi = chunk_hi(q);
      // (the gates of chunk q were waited for by qt_part(q), earlier on this thread)
      if (!cwait_nf(&sh.bar_p[eq], (q >> 1) & 1)) return false;
      const float* ksc = sh.gates.ksc[eq];
      uint8_t* kt = sm + kslot(q);
      uint4 in[4];
      float sc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // every load before any store
        const int i = ci + 256 * k;
        in[k] = *reinterpret_cast<const uint4*>(kt + i * 16);
        sc[k] = ksc[(i & 511) >> 3];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = ci + 256 * k;
        const int row = (i & 511) >> 3;
        *reinterpret_cast<uint4*>(kt + i * 16) = cvt8v(in[k], sc[k], row >= lo && row < hi, check_range, range_bad);
      }
      fence_proxy_async();
      mbar_arrive(&sh.kt_ready[eq]);
      return true;
    };
    // A state store goes through this warp's 2 KB output staging block, a few
    // rows at a time, so that every global store instruction writes whole
    // 256-byte (fp32) or 128-byte (bf16) row halves: lanes write their rows into
    // the block (16-byte pieces swizzled by row, free of bank conflicts), then
    // the warp reads the block back in row order and stores it.
    auto store_state = [&](float* pool, int row) {
      if (check_range) {  // an fp16 operand that overflowed leaves a non-finite state
        bool fin = true;
#pragma unroll
        for (int i = 0; i < 64; ++i) fin &= isfinite(S[i]);
        range_bad |= !fin;
      }
      uint8_t* stg = sm + OFF_OST + warp * 2048;
      if (lane == 0) bulk_wait_read();  // this warp's last output store has read the block
      __syncwarp();
      const int v0 = 32 * wq;
      if constexpr (kBf16) {  // nearest bf16, ties to even; 2 passes of 16 rows x 128 B
        __nv_bfloat16* pb = reinterpret_cast<__nv_bfloat16*>(pool);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if ((lane >> 4) == r) {
            const int rr = lane & 15;
#pragma unroll
            for (int f = 0; f < 8; ++f)
              *reinterpret_cast<uint4*>(stg + rr * 128 + ((f ^ (rr & 7)) << 4)) =
                  make_uint4(pack_bf162(S[8 * f], S[8 * f + 1]), pack_bf162(S[8 * f + 2], S[8 * f + 3]),
                             pack_bf162(S[8 * f + 4], S[8 * f + 5]), pack_bf162(S[8 * f + 6], S[8 * f + 7]));
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int pc = 32 * j + lane, rr = pc >> 3, f = pc & 7;
            const uint4 x = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((f ^ (rr & 7)) << 4));
            *reinterpret_cast<uint4*>(pb + row * a.row_stride + head_off + (v0 + 16 * r + rr) * kDimK + 64 * hc + 8 * f) = x;
          }
          __syncwarp();
        }
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // 4 passes of 8 rows x 256 B
          if ((lane >> 3) == r) {
            const int rr = lane & 7;
#pragma unroll
            for (int f = 0; f < 16; ++f)
              *reinterpret_cast<float4*>(stg + rr * 256 + ((f ^ rr) << 4)) =
                  make_float4(S[4 * f], S[4 * f + 1], S[4 * f + 2], S[4 * f + 3]);
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int pc = 32 * j + lane, rr = pc >> 4, f = pc & 15;
            const float4 x = *reinterpret_cast<const float4*>(stg + rr * 256 + ((f ^ rr) << 4));
            *reinterpret_cast<float4*>(pool + row * a.row_stride + head_off + (v0 + 8 * r + rr) * kDimK + 64 * hc + 4 * f) = x;
          }
          __syncwarp();
        }
      }
    };
    if (!qt_part(0) || !kt_part(0)) ok = false;
    for (int c = 0; c < nch && ok; ++c) {
      const uint32_t e = c & 1, ph = (c >> 1) & 1;
      const uint32_t dx = lane_addr + COL_DX + 128 * e;
      const uint32_t uh = dx + 64 * e, oh = dx + 64 * (1 - e);  // U and O halves of D_X
      // U^T, row v: 32 fp32 values packed in place into 16 fp16 pairs (the A
      // operand of U^T K~ and U^T P^T)
      if (!cwait(&sh.bar_x[e], ph)) break;
      {
        float u[32];
        tmem_ld32(uh + 32 * hc, u);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_half2(u[2 * i], u[2 * i + 1]);
        tmem_st16(uh + 32 * hc, w);
      }
      tc_fence_before();
      mbar_arrive(&sh.u_ready);
      if (tid == 0 && c + 2 < nch) tma_w(c + 2);  // X of chunk c has read its -W buffer
      // Q~ of the next chunk while U^T K~ runs
      if (c + 1 < nch && !qt_part(c + 1)) break;
      // S1 = gamma_C S0 + U^T K~, and its fp16 copy for the next chunk
      if (!cwait(&sh.bar_su[e], ph)) break;
      const float gamC = sh.gamC[c % 3];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float su[32];
        tmem_ld32(lane_addr + COL_DSU + 64 * hc + 32 * hh, su);
        const float2 g2 = make_float2(gamC, gamC);
#pragma unroll
        for (int i = 0; i < 16; ++i) {  // paired fp32 FMAs
          const float2 r = __ffma2_rn(g2, make_float2(S[32 * hh + 2 * i], S[32 * hh + 2 * i + 1]),
                                      make_float2(su[2 * i], su[2 * i + 1]));
          S[32 * hh + 2 * i] = r.x;
          S[32 * hh + 2 * i + 1] = r.y;
        }
      }
      stage_state();
      mbar_arrive(&sh.s16_ready);
      if (tid == 0 && c + 2 < nch) tma_k(c + 2);  // U^T K~ of chunk c has read its K slot
      const int a_end = chunk_a0(c) + kChunk;
      if (ck_rows && ck_pool && a_end % N == 0 && a_end <= end_pos) {
        const int row = static_cast<int>(index_at(ck_rows, ck_off + a_end / N - 1 - first_ck, ck_wide));
        if (row >= 0) store_state(ck_pool, row);
      }
      // Outputs of chunk c (columns of O^T).  In a full chunk each warp reads its
      // 32 x 32 block (rows v of its lane quarter x 32 tokens) as 16-lane
      // fragments, which stmatrix stores transposed into a 64B-swizzled staging
      // block (row t: the warp's 32 values v of token t, 16 bytes per store row
      // and no bank conflicts), sent with one TMA store of its own, so no warp
      // waits for another.  A partial chunk (first / last of a sequence) is
      // stored element by element, so that no row of another sequence is touched.
      if (!cwait(&sh.bar_o[e], ph)) break;
      {
        const int lo = chunk_lo(c), hi = chunk_hi(c), tf = chunk_tf(c);
        if (lo == 0 && hi == kChunk) {
          uint32_t f[2][16];
          tmem_ld16x256_x4_nw(oh + 32 * hc, f[0]);               // lanes 32 wq + 0..15
          tmem_ld16x256_x4_nw(oh + 32 * hc + (16u << 16), f[1]);  // lanes 32 wq + 16..31
          tmem_wait_ld2(f[0], f[1]);
          zero32(oh + 32 * hc);
          tc_fence_before();
          mbar_arrive(&sh.o_read[e]);
          uint8_t* stg = sm + OFF_OST + warp * 2048;
          if (lane == 0) bulk_wait_read();  // this warp's previous store has read the block
          __syncwarp();
          const float2 sc2 = make_float2(a.scale, a.scale);
          const int mi = lane >> 3, k = lane & 7;  // this thread's row address: matrix mi, row k
#pragma unroll
          for (int g = 0; g < 2; ++g) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              uint32_t m[4];
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const int j = 2 * jj + q;  // tokens 8 j .. 8 j + 7
                m[2 * q] = pack_bf162(
                    __fmul2_rn(sc2, make_float2(__uint_as_float(f[g][4 * j]), __uint_as_float(f[g][4 * j + 1]))));
                m[2 * q + 1] = pack_bf162(
                    __fmul2_rn(sc2, make_float2(__uint_as_float(f[g][4 * j + 2]), __uint_as_float(f[g][4 * j + 3]))));
              }
              // matrix mi: tokens 8 (2 jj + mi / 2) .., rows v 16 g + 8 (mi % 2) ..
              const int t = 8 * (2 * jj + (mi >> 1)) + k;
              const int piece = 2 * g + (mi & 1);
              stmatrix_x4_trans(smem_u32(stg + t * 64 + ((piece ^ ((t >> 1) & 3)) << 4)), m[0], m[1], m[2], m[3]);
            }
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tm_o, stg, 32 * wq, h, tf + 32 * hc);
            bulk_commit();
          }
        } else {
          float o[32];
          tmem_ld32(oh + 32 * hc, o);
          zero32(oh + 32 * hc);
          tc_fence_before();
          mbar_arrive(&sh.o_read[e]);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int t = 32 * hc + i;
            if (t >= lo && t < hi)
              a.o[(static_cast<int64_t>(tf + t) * H + h) * kDimV + v] = __float2bfloat16_rn(a.scale * o[i]);
          }
        }
      }
      if (c + 1 < nch && !kt_part(c + 1)) break;
    }
    if (ok && out_row >= 0) store_state(out_pool, out_row);
    if (lane == 0) bulk_wait_all();
    if (range_bad) record_error(a.err_word, GDN_DEVERR_RANGE, b);
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && sh.abort) record_error(a.err_word, GDN_DEVERR_TIMEOUT, b);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

std::atomic<int32_t> g_debug_stall{0};

int launch(PrefillArgs& a, const void* q, const void* k, const void* v, void* workspace, size_t workspace_bytes,
           cudaStream_t stream) {
  a.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
  const int64_t ns = num_chunk_slots(a.T, a.num_seqs);
  if (!workspace || workspace_bytes < gdn::workspace_bytes(a.T, a.num_seqs, a.H) || !gdn_host::aligned16(workspace))
    return GDN_ERR_INVALID_ARGUMENT;
  int num_sms = 0;
  int rc = gdn_host::check_device(&num_sms);
  if (rc != GDN_OK) return rc;
  a.num_slots = static_cast<int32_t>(ns);
  a.slot_geo = static_cast<int4*>(workspace);
  a.item_counter = reinterpret_cast<int32_t*>(a.slot_geo + ns);
  a.tinv = reinterpret_cast<__half*>(static_cast<uint8_t*>(workspace) + workspace_map_bytes(ns));
  a.wneg = a.tinv + ns * a.H * (kTinvBytes / 2);
  // (the maps of K, T'' and -W serve both kernels)
  CUtensorMap mq, mk, mv, mt, mo, mw;
  if (gdn_host::encode_tokens_map(&mq, q, a.T, a.H, kDimK) != GDN_OK ||
      gdn_host::encode_tokens_map(&mk, k, a.T, a.H, kDimK) != GDN_OK ||
      gdn_host::encode_tokens_map(&mv, v, a.T, a.H, kDimV) != GDN_OK ||
      gdn_host::encode_tokens_map_32(&mo, a.o, a.T, a.H, kDimV) != GDN_OK ||
      gdn_host::encode_tiles_map_f16(&mt, a.tinv, ns * a.H * 64, 64) != GDN_OK ||
      gdn_host::encode_tiles_map_f16(&mw, a.wneg, ns * a.H * 64, 128) != GDN_OK)
    return GDN_ERR_CUDA;
  rc = host::launch_chunk_inverse(a, mk, mt, mw, num_sms, stream);
  if (rc != GDN_OK) return rc;
  static std::atomic<uint64_t> smem_set[4];
  const int variant = (a.err_word ? 2 : 0) + (a.state_bf16 ? 1 : 0);
  auto kernel = a.err_word ? (a.state_bf16 ? prefill_kernel<true, true> : prefill_kernel<true, false>)
                           : (a.state_bf16 ? prefill_kernel<false, true> : prefill_kernel<false, false>);
  rc = gdn_host::func_attr_once(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES, smem_set[variant]);
  if (rc != GDN_OK) return rc;
  const long long grid = static_cast<long long>(a.num_seqs) * a.H;
  return gdn_host::launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), SMEM_BYTES, stream, mq, mk,
                              mv, mt, mo, mw, a);
}

int check_common(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g, const float* beta,
                 gdn_bf16* o, const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H,
                 int32_t K, int32_t V) {
  if (num_seqs < 0 || total_tokens < 0 || H < 1) return GDN_ERR_INVALID_ARGUMENT;
  if (K != kDimK || V != kDimV) return GDN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_seqs) * H > 0x7FFFFFFFLL || H > 65535) return GDN_ERR_UNSUPPORTED;
  if (num_chunk_slots(total_tokens, num_seqs) * H * 64 > 0x7FFFFFFFLL) return GDN_ERR_UNSUPPORTED;
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

extern "C" void gdn_debug_set_wait_stall(int32_t enable) { g_debug_stall.store(enable != 0 ? 1 : 0); }

extern "C" size_t gdn_prefill_workspace_bytes(int32_t num_seqs, int32_t total_tokens, int32_t H) {
  if (num_seqs < 0 || total_tokens < 0 || H < 1) return 0;
  return gdn::workspace_bytes(total_tokens, num_seqs, H);
}

extern "C" int gdn_chunk_gated_delta_rule_ex(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                             const float* g, const float* beta, gdn_bf16* o,
                                             const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                             int32_t H, int32_t K, int32_t V, float scale, const void* initial_state,
                                             const void* state_indices, void* output_state,
                                             const void* output_state_indices, void* state_checkpoints,
                                             const void* checkpoint_state_indices, const void* checkpoint_cu_starts,
                                             const void* prefix_lens, int32_t checkpoint_every_n_tokens,
                                             int64_t pool_row_stride, int32_t state_dtype, int32_t index_dtype,
                                             void* workspace, size_t workspace_bytes, int32_t* err_word,
                                             void* stream) {
  int rc = check_common(q, k, v, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, K, V);
  if (rc != GDN_OK) return rc;
  if (state_dtype != GDN_STATE_F32 && state_dtype != GDN_STATE_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (index_dtype != GDN_INDEX_I32 && index_dtype != GDN_INDEX_I64) return GDN_ERR_INVALID_ARGUMENT;
  const uintptr_t index_align = index_dtype == GDN_INDEX_I64 ? 8 : 4;
  for (const void* p : {state_indices, output_state_indices, checkpoint_state_indices, checkpoint_cu_starts,
                        prefix_lens})
    if (reinterpret_cast<uintptr_t>(p) % index_align != 0) return GDN_ERR_INVALID_ARGUMENT;
  if ((state_indices != nullptr) != (initial_state != nullptr)) return GDN_ERR_INVALID_ARGUMENT;
  if ((output_state_indices != nullptr) != (output_state != nullptr)) return GDN_ERR_INVALID_ARGUMENT;
  const int nck = (state_checkpoints != nullptr) + (checkpoint_state_indices != nullptr) +
                  (checkpoint_cu_starts != nullptr);
  if (nck != 0 && nck != 3) return GDN_ERR_INVALID_ARGUMENT;
  if (nck == 3 && (!prefix_lens || checkpoint_every_n_tokens <= 0 || checkpoint_every_n_tokens % kChunk != 0))
    return GDN_ERR_INVALID_ARGUMENT;
  const bool any_pool = initial_state || output_state || state_checkpoints;
  const int64_t stride_unit = state_dtype == GDN_STATE_BF16 ? 8 : 4;  // 16-byte rows
  if (any_pool &&
      (pool_row_stride < static_cast<int64_t>(H) * kDimV * kDimK || pool_row_stride % stride_unit != 0))
    return GDN_ERR_INVALID_ARGUMENT;
  using gdn_host::aligned16;
  if ((initial_state && !aligned16(initial_state)) || (output_state && !aligned16(output_state)) ||
      (state_checkpoints && !aligned16(state_checkpoints)))
    return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0 || total_tokens == 0) return GDN_OK;

  PrefillArgs a;
  fill_common(a, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, scale, err_word);
  a.initial_state = static_cast<const float*>(initial_state);
  a.state_indices = state_indices;
  a.output_state = static_cast<float*>(output_state);
  a.output_state_indices = output_state_indices;
  a.state_checkpoints = static_cast<float*>(state_checkpoints);
  a.checkpoint_state_indices = checkpoint_state_indices;
  a.checkpoint_cu_starts = checkpoint_cu_starts;
  a.prefix_lens = prefix_lens;
  a.index64 = index_dtype == GDN_INDEX_I64;
  a.N = nck ? checkpoint_every_n_tokens : 0;
  a.row_stride = any_pool ? pool_row_stride : 0;
  a.state_bf16 = state_dtype == GDN_STATE_BF16;
  return launch(a, q, k, v, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_chunk_gated_delta_rule(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                                          const float* beta, gdn_bf16* o, const int32_t* cu_seqlens,
                                          int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t K, int32_t V,
                                          float scale, const float* initial_state, const int32_t* state_indices,
                                          float* output_state, const int32_t* output_state_indices,
                                          float* state_checkpoints, const int32_t* checkpoint_state_indices,
                                          const int32_t* checkpoint_cu_starts, const int32_t* prefix_lens,
                                          int32_t checkpoint_every_n_tokens, int64_t pool_row_stride,
                                          void* workspace, size_t workspace_bytes, int32_t* err_word,
                                          void* stream) {
  return gdn_chunk_gated_delta_rule_ex(q, k, v, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, K, V, scale,
                                       initial_state, state_indices, output_state, output_state_indices,
                                       state_checkpoints, checkpoint_state_indices, checkpoint_cu_starts, prefix_lens,
                                       checkpoint_every_n_tokens, pool_row_stride, GDN_STATE_F32, GDN_INDEX_I32,
                                       workspace,
                                       workspace_bytes, err_word, stream);
}

extern "C" int gdn_chunk_gated_delta_rule_paged_ex(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                                   const float* g, const float* beta, gdn_bf16* o,
                                                   const int32_t* cu_seqlens, int32_t num_seqs,
                                                   int32_t total_tokens, int32_t H, int32_t K, int32_t V, float scale,
                                                   void* state_pool, int32_t state_dtype, int32_t num_pages,
                                                   const int32_t* page_indices, const int32_t* page_indptr,
                                                   int32_t page_size, const int32_t* last_page_len,
                                                   const gdn_prefill_slots* slots, void* workspace,
                                                   size_t workspace_bytes, int32_t* err_word, void* stream) {
  int rc = check_common(q, k, v, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, K, V);
  if (rc != GDN_OK) return rc;
  if (state_dtype != GDN_STATE_F32 && state_dtype != GDN_STATE_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (page_size <= 0 || page_size % kChunk != 0 || num_pages < 1) return GDN_ERR_INVALID_ARGUMENT;
  if (!state_pool || !gdn_host::aligned16(state_pool)) return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs > 0 && (!page_indices || !page_indptr || !last_page_len)) return GDN_ERR_INVALID_ARGUMENT;
  if (slots && (!slots->state_indices || !slots->output_state_indices || !slots->checkpoint_cu_starts ||
                !slots->prefix_lens))
    return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0 || total_tokens == 0) return GDN_OK;

  PrefillArgs a;
  fill_common(a, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, scale, err_word);
  a.initial_state = static_cast<const float*>(state_pool);
  a.output_state = static_cast<float*>(state_pool);
  a.state_checkpoints = static_cast<float*>(state_pool);
  a.checkpoint_state_indices = page_indices;
  a.N = page_size;
  a.row_stride = static_cast<int64_t>(H) * kDimV * kDimK;
  a.state_bf16 = state_dtype == GDN_STATE_BF16;
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
  return launch(a, q, k, v, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_chunk_gated_delta_rule_paged(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                                const float* g, const float* beta, gdn_bf16* o,
                                                const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                                int32_t H, int32_t K, int32_t V, float scale, float* state_pool,
                                                int32_t num_pages, const int32_t* page_indices,
                                                const int32_t* page_indptr, int32_t page_size,
                                                const int32_t* last_page_len, const gdn_prefill_slots* slots,
                                                void* workspace, size_t workspace_bytes, int32_t* err_word,
                                                void* stream) {
  return gdn_chunk_gated_delta_rule_paged_ex(q, k, v, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, K, V, scale,
                                             state_pool, GDN_STATE_F32, num_pages, page_indices, page_indptr,
                                             page_size, last_page_len, slots, workspace, workspace_bytes, err_word,
                                             stream);
}

// ---------------------------------------------------------------------------
// Paged prefill without a caller-provided workspace.
//
// Some callers cannot call cudaMalloc: a runtime whose device memory is all
// handed out by its own pool, a plugin host that forbids device allocations,
// or a serving loop that cannot afford the device synchronisation an
// allocation may trigger.  For them the workspace of the chunk-local phase
// lives in a fixed array in the library's own device image, reserved on every
// GPU that loads the library for as long as the process runs.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

// The array's device address, looked up once per device (with that device
// current) on the first call made on it.
void* static_workspace() {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int gdn_chunk_gated_delta_rule_paged_static_workspace(
    const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g, const float* beta, gdn_bf16* o,
    const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t K, int32_t V, float scale,
    float* state_pool, int32_t num_pages, const int32_t* page_indices, const int32_t* page_indptr, int32_t page_size,
    const int32_t* last_page_len, const gdn_prefill_slots* slots, int32_t* err_word, void* stream) {
  if (num_seqs >= 0 && total_tokens >= 0 && H >= 1 &&
      gdn::workspace_bytes(total_tokens, num_seqs, H) > kStaticWorkspaceBytes)
    return GDN_ERR_UNSUPPORTED;
  void* ws = nullptr;
  if (num_seqs > 0 && total_tokens > 0) {
    ws = static_workspace();
    if (!ws) return GDN_ERR_CUDA;
  }
  return gdn_chunk_gated_delta_rule_paged(q, k, v, g, beta, o, cu_seqlens, num_seqs, total_tokens, H, K, V, scale,
                                          state_pool, num_pages, page_indices, page_indptr, page_size, last_page_len,
                                          slots, ws, kStaticWorkspaceBytes, err_word, stream);
}
