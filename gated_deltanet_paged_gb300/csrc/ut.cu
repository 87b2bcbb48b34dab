// ut.cu -- the chunk-local part of chunked GDN prefill: for every 64-token chunk
// and head, T'' = (I + A)^-1 diag(beta) and -W = -T'' diag(gamma) K, written to
// the workspace.
//
// "flashinfer.gdn_paged", chunk_gated_delta_rule: the gated delta rule in
// chunked (WY / UT) form.  With rows t = 0..63 of a chunk (rows outside the
// sequence have g = beta = 0 and k = 0), G_t = g_0 + ... + g_t and
//   A[t][j] = beta_t exp(G_t - G_j) (k_t . k_j)   for j < t,  0 otherwise,
// T = (I + A)^-1 is what turns the chunk's sequential rank-1 updates into
// matrix products (W = T diag(beta gamma) K, U~ = T diag(beta) V).  T depends
// only on the chunk's own k, g and beta, never on the state, so every chunk of
// every sequence is computed here at once; the sequential state chain (the
// prefill kernel) then only multiplies.
//
// Mapping: one CTA of 128 threads per (pair of chunk slots, head); thread r is
// row r of the two chunks stacked (rows 0-63 chunk a, 64-127 chunk b), which
// is also its TMEM lane.  All products are M = 128 tcgen05 MMAs on both chunks
// at once:
//   [K_a; K_b] [K_a; K_b]^T   (bf16 straight from TMA; the diagonal 64 x 64
//                              blocks are K_a K_a^T and K_b K_b^T)
//   T_d  = inverse of A's 16 x 16 diagonal blocks, forward substitution (fp32)
//   N    = -T_d A_o           (A_o: A without its diagonal blocks; N^4 = 0)
//   T    = (I + N)(I + N^2) T_d = Z + N^2 Z,  Z = T_d + N T_d
//   W    = [T'_a; 0] K_a + [0; T'_b] K_b,  T' = T diag(beta gamma), K reloaded
//          and converted to fp16 once the inverse no longer needs the space
// The per-chunk B operands sit side by side ([X_a | X_b], N = 128) so one MMA
// serves both chunks (the off-diagonal 64 x 64 result blocks are unused); for
// N [N | T_d] the A operand is padded with a zero tile per chunk instead.
#include <math.h>

#include "prefill_common.cuh"

namespace {

using namespace gdn;

constexpr int kUtThreads = 128;
constexpr uint32_t kTile = 8192;  // 64 rows x 128 B

// Shared memory (offsets from the 1024-aligned base).
//   R2 (24 KB): A_o [a | b] -> N_a | 0 | N_b -> N^2 stack (16 KB) -> T'' staging
//               -> T'_a | 0 | T'_b
//   R0 (32 KB): K stack -> fp32 diagonal blocks (first 8 KB) + T_d stack (last
//               16 KB) -> Z [a | b] (first 16 KB) -> K stack again (fp16) -> -W staging
constexpr uint32_t UT_R2 = 0;
constexpr uint32_t UT_R0 = 24576;
constexpr uint32_t UT_TD = UT_R0 + 16384;
constexpr uint32_t UT_SMALL = UT_R0 + 32768;

struct UtSmall {
  float G[128];    // cumulative gate per stacked row
  float e[128];    // exp(g)
  float bet[128];  // beta
  float gam[128];  // exp(G)
  float wsum[4];   // per-warp gate totals for the scan
  uint64_t bar_tma, bar_mma;
  uint32_t tmem_base;
  int tf[2], lo[2], hi[2], slot[2];
  int flag;
};
constexpr uint32_t UT_SMEM = UT_SMALL + ((sizeof(UtSmall) + 127) / 128) * 128 + 1024;

__device__ __forceinline__ uint4 pack8h(const float* x) {
  uint4 u;
  u.x = pack_half2(x[0], x[1]);
  u.y = pack_half2(x[2], x[3]);
  u.z = pack_half2(x[4], x[5]);
  u.w = pack_half2(x[6], x[7]);
  return u;
}

__device__ __forceinline__ void unpack8h(uint4 u, float* x) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// fp32 16-column rows of the diagonal blocks: float4 q of row r at q ^ (r % 4).
__device__ __forceinline__ float* am_q(float* AM, int r, int q) { return AM + r * 16 + ((q ^ (r & 3)) << 2); }

// Chunk slot -> sequence (or -1 when the slot holds no chunk).
__global__ void slot_map_kernel(const PrefillArgs a) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= a.num_slots) return;
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int cu = a.cu_seqlens[mid];
    if (cu >= 0 && slot_base(cu, mid) <= s)
      lo = mid;
    else
      hi = mid - 1;
  }
  int out = -1, cu_b, L, P;
  if (seq_extent(a, lo, cu_b, L, P)) {
    const int c = s - slot_base(cu_b, lo);
    if (c >= 0 && c < chunk_count(P, L)) out = lo;
  }
  a.slot_seq[s] = out;
}

__global__ void __launch_bounds__(kUtThreads, 3)
    ut_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_t,
              const __grid_constant__ CUtensorMap tm_w, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  UtSmall& sh = *reinterpret_cast<UtSmall*>(sm + UT_SMALL);
  float* AM = reinterpret_cast<float*>(sm + UT_R0);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = tid >> 6, t = tid & 63, r0 = half * 64;
  const int h = blockIdx.y, H = a.H;

  if (t == 0) {
    const int s = 2 * blockIdx.x + half;
    int tf = 0, lo = 0, hi = 0;
    if (s < a.num_slots) {
      const int b = a.slot_seq[s];
      int cu_b, L, P;
      if (b >= 0 && seq_extent(a, b, cu_b, L, P)) {
        const int c = s - slot_base(cu_b, b);
        if (c >= 0 && c < chunk_count(P, L)) {
          const int a0 = (P / 64) * 64 + 64 * c;
          lo = max(P - a0, 0);
          hi = min(P + L - a0, 64);
          tf = cu_b + a0 - P;
        }
      }
    }
    sh.tf[half] = tf;
    sh.lo[half] = lo;
    sh.hi[half] = hi;
    sh.slot[half] = s;
  }
  __syncthreads();
  const bool va = sh.hi[0] > sh.lo[0], vb = sh.hi[1] > sh.lo[1];
  if (!va && !vb) return;
  const int lo = sh.lo[half], hi = sh.hi[half], tf = sh.tf[half];

  if (tid == 0) {
    mbar_init(&sh.bar_tma, 1);
    mbar_init(&sh.bar_mma, 1);
    sh.flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    mbar_arrive_expect_tx(&sh.bar_tma, 16384u * ((va ? 1u : 0u) + (vb ? 1u : 0u)));
    for (int hh = 0; hh < 2; ++hh) {
      if (sh.hi[hh] <= sh.lo[hh]) continue;
      tma_load_3d(sm + UT_R0 + hh * kTile, &tm_k, &sh.bar_tma, 0, h, sh.tf[hh]);
      tma_load_3d(sm + UT_R0 + 16384 + hh * kTile, &tm_k, &sh.bar_tma, 64, h, sh.tf[hh]);
    }
  }
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, 128);
    tmem_relinquish();
  }

  // Gates of this row; inclusive scan over the chunk's 64 rows.
  const bool vme = t >= lo && t < hi;
  float gv = 0.f, bv = 0.f;
  if (vme) {
    const int64_t idx = static_cast<int64_t>(tf + t) * H + h;
    gv = a.g[idx];
    bv = a.beta[idx];
  }
  float s = gv;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, s, off);
    if (lane >= off) s += y;
  }
  if (lane == 31) sh.wsum[warp] = s;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  if (warp & 1) s += sh.wsum[warp - 1];
  sh.G[tid] = s;
  sh.e[tid] = expf(gv);
  sh.bet[tid] = bv;
  sh.gam[tid] = expf(s);

  auto dK = [&](uint32_t off) { return sdesc(sbase + off, 16, 1024); };
  auto dMN = [&](uint32_t off, uint32_t lbo) { return sdesc(sbase + off, lbo, 1024); };
  const uint32_t id_bf16 = idesc_f16(128, 128, true, true, false, false);
  const uint32_t id_mnB = idesc_f16(128, 128, false, false, false, true);

  // Every thread waits for the MMA; a time-out anywhere aborts the CTA.
  auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (!mbar_wait(bar, parity)) sh.flag = 1;
    __syncthreads();
    tc_fence_after();
    return sh.flag == 0;
  };

  // ---- [K_a; K_b] [K_a; K_b]^T ----
  if (tid == 0) {
    if (mbar_wait(&sh.bar_tma, 0)) {
      tc_fence_after();
      tc_mma4(tmem, dK(UT_R0), 2, dK(UT_R0), 2, id_bf16, 0);
      tc_mma4(tmem, dK(UT_R0 + 16384), 2, dK(UT_R0 + 16384), 2, id_bf16, 1);
      tc_commit(&sh.bar_mma);
    } else {
      sh.flag = 1;
    }
  }
  __syncthreads();
  bool ok = sh.flag == 0 && wait_all(&sh.bar_mma, 0);

  // ---- A: fp32 diagonal blocks, fp16 A_o (MN-major B of round 1) ----
  const int dblk = t >> 4;
  if (ok) {
    float x[64];
    tmem_ld64(lane_addr + r0, x);
    const float Gt = sh.G[tid];
    uint8_t* ao = sm + UT_R2 + half * kTile;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float out[16];
      const int jstart = min(16 * q + 15, t - 1);  // last column of the strict lower part
      if (vme && jstart >= 16 * q) {
        float cur = bv * expf(Gt - sh.G[r0 + jstart]);
#pragma unroll
        for (int jj = 15; jj >= 0; --jj) {
          const int j = 16 * q + jj;
          const bool in = (j <= jstart) && (j >= lo);
          out[jj] = in ? cur * x[j] : 0.f;
          if (j <= jstart) cur *= sh.e[r0 + j];
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) out[jj] = 0.f;
      }
      if (q == dblk) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<float4*>(am_q(AM, tid, k)) =
              make_float4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
        *reinterpret_cast<uint4*>(ao + swz(t, 2 * q)) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(ao + swz(t, 2 * q + 1)) = make_uint4(0u, 0u, 0u, 0u);
      } else {
        *reinterpret_cast<uint4*>(ao + swz(t, 2 * q)) = pack8h(&out[0]);
        *reinterpret_cast<uint4*>(ao + swz(t, 2 * q + 1)) = pack8h(&out[8]);
      }
    }
  }
  fence_proxy_async();
  __syncthreads();

  // ---- T_d: thread (chunk, block bb, column jj) solves one column ----
  if (ok) {
    const int bb = (tid >> 4) & 3, jj = tid & 15;
    const int rb = r0 + 16 * bb;
    float xs[16];
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int m4 = 0; m4 < 4; ++m4) {
        if (4 * m4 < tt) {
          const float4 a4 = *reinterpret_cast<const float4*>(am_q(AM, rb + tt, m4));
          if (4 * m4 + 0 < tt) acc[0] = fmaf(a4.x, xs[4 * m4 + 0], acc[0]);
          if (4 * m4 + 1 < tt) acc[1] = fmaf(a4.y, xs[4 * m4 + 1], acc[1]);
          if (4 * m4 + 2 < tt) acc[2] = fmaf(a4.z, xs[4 * m4 + 2], acc[2]);
          if (4 * m4 + 3 < tt) acc[3] = fmaf(a4.w, xs[4 * m4 + 3], acc[3]);
        }
      }
      xs[tt] = (tt == jj) ? 1.f : (tt > jj ? -((acc[0] + acc[1]) + (acc[2] + acc[3])) : 0.f);
    }
    __syncthreads();  // every read of A's diagonal blocks is done
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) am_q(AM, rb + tt, jj >> 2)[jj & 3] = xs[tt];
    __syncthreads();
    float f[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v4 = *reinterpret_cast<const float4*>(am_q(AM, tid, k));
      f[4 * k] = v4.x;
      f[4 * k + 1] = v4.y;
      f[4 * k + 2] = v4.z;
      f[4 * k + 3] = v4.w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if ((c >> 1) == dblk) u = pack8h(&f[8 * (c & 1)]);
      *reinterpret_cast<uint4*>(sm + UT_TD + swz(tid, c)) = u;
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();

  // ---- round 1: N = -T_d A_o ----
  if (ok && tid == 0) {
    tc_fence_after();
    tc_mma4(tmem, dK(UT_TD), 2, dMN(UT_R2, kTile), 128, id_mnB, 0);
    tc_commit(&sh.bar_mma);
  }
  ok = ok && wait_all(&sh.bar_mma, 1);
  if (ok) {
    float d[64];
    tmem_ld64(lane_addr + r0, d);
#pragma unroll
    for (int i = 0; i < 64; ++i) d[i] = -d[i];
    uint8_t* nt = sm + UT_R2 + half * 16384;
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(nt + swz(t, c)) = pack8h(&d[8 * c]);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      reinterpret_cast<uint4*>(sm + UT_R2 + kTile)[tid + 128 * k] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();

  // ---- round 2: [N^2 | N T_d] = [N_a; 0][N_a | T_d,a] + [0; N_b][N_b | T_d,b] ----
  if (ok && tid == 0) {
    tc_fence_after();
    tc_mma4(tmem, dK(UT_R2), 2, dMN(UT_R2, UT_TD - UT_R2), 128, id_mnB, 0);
    tc_mma4(tmem, dK(UT_R2 + kTile), 2, dMN(UT_R2 + 16384, UT_TD + kTile - UT_R2 - 16384), 128, id_mnB, 1);
    tc_commit(&sh.bar_mma);
  }
  ok = ok && wait_all(&sh.bar_mma, 0);
  float z[64];
  if (ok) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float n2[32], nt[32];
      tmem_ld32(lane_addr + 32 * hh, n2);
      tmem_ld32(lane_addr + 64 + 32 * hh, nt);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = 4 * hh + c;
        float td[8];
        unpack8h(*reinterpret_cast<const uint4*>(sm + UT_TD + swz(tid, cc)), td);
#pragma unroll
        for (int i = 0; i < 8; ++i) z[8 * cc + i] = td[i] + nt[8 * c + i];
        *reinterpret_cast<uint4*>(sm + UT_R2 + swz(tid, cc)) = pack8h(&n2[8 * c]);
        *reinterpret_cast<uint4*>(sm + UT_R0 + half * kTile + swz(t, cc)) = pack8h(&z[8 * cc]);
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();

  // ---- round 3: T = Z + N^2 Z;  T'' = T diag(beta) -> workspace ----
  if (ok && tid == 0) {
    tc_fence_after();
    tc_mma4(tmem, dK(UT_R2), 2, dMN(UT_R0, kTile), 128, id_mnB, 0);
    tc_commit(&sh.bar_mma);
  }
  ok = ok && wait_all(&sh.bar_mma, 1);
  // K again (the inverse has released R0), for W.
  if (ok && tid == 0) {
    mbar_arrive_expect_tx(&sh.bar_tma, 16384u * ((va ? 1u : 0u) + (vb ? 1u : 0u)));
    for (int hh = 0; hh < 2; ++hh) {
      if (sh.hi[hh] <= sh.lo[hh]) continue;
      tma_load_3d(sm + UT_R0 + hh * kTile, &tm_k, &sh.bar_tma, 0, h, sh.tf[hh]);
      tma_load_3d(sm + UT_R0 + 16384 + hh * kTile, &tm_k, &sh.bar_tma, 64, h, sh.tf[hh]);
    }
  }
  float tr[64];  // row t of T'' = T diag(beta)
  if (ok) {      // T'' rows into a staging tile per chunk (R2 is free again), then TMA stores
    float d[64];
    tmem_ld64(lane_addr + r0, d);
    uint8_t* stg = sm + UT_R2 + half * kTile;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
#pragma unroll
      for (int i = 0; i < 8; ++i) tr[8 * c + i] = (z[8 * c + i] + d[8 * c + i]) * sh.bet[r0 + 8 * c + i];
      *reinterpret_cast<uint4*>(stg + swz(t, c)) = pack8h(&tr[8 * c]);
    }
  }
  fence_proxy_async();
  __syncthreads();
  if (ok && tid == 0) {
    for (int hh = 0; hh < 2; ++hh)
      if (sh.hi[hh] > sh.lo[hh]) tma_store_2d(&tm_t, sm + UT_R2 + hh * kTile, 0, (sh.slot[hh] * H + h) * 64);
    bulk_commit();
    bulk_wait_read();
  }
  __syncthreads();
  // T' = T'' diag(gamma) as the A operand of W: [T'_a; 0] and [0; T'_b] from T'_a | 0 | T'_b.
  if (ok) {
    uint8_t* tp = sm + UT_R2 + half * 16384;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = tr[8 * c + i] * sh.gam[r0 + 8 * c + i];
      *reinterpret_cast<uint4*>(tp + swz(t, c)) = pack8h(w);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      reinterpret_cast<uint4*>(sm + UT_R2 + kTile)[tid + 128 * k] = make_uint4(0u, 0u, 0u, 0u);
  }
  // K (bf16) -> fp16 in place, rows outside each chunk zero.
  if (ok) {
    if (!mbar_wait(&sh.bar_tma, 1)) sh.flag = 1;
    for (int i = tid; i < 2048; i += kUtThreads) {
      const int box = i >> 9;  // K_a kb0 | K_b kb0 | K_a kb1 | K_b kb1
      const int hh = box & 1, row = (i & 511) >> 3;
      uint8_t* ptr = sm + UT_R0 + box * kTile + (i & 511) * 16;
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (row >= sh.lo[hh] && row < sh.hi[hh]) {
        const uint4 in = *reinterpret_cast<const uint4*>(ptr);
        const float2 f0 = unpack_bf162(in.x), f1 = unpack_bf162(in.y), f2 = unpack_bf162(in.z),
                     f3 = unpack_bf162(in.w);
        out.x = pack_half2(f0.x, f0.y);
        out.y = pack_half2(f1.x, f1.y);
        out.z = pack_half2(f2.x, f2.y);
        out.w = pack_half2(f3.x, f3.y);
      }
      *reinterpret_cast<uint4*>(ptr) = out;
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  ok = ok && sh.flag == 0;

  // ---- W = [T'_a; 0] K_a + [0; T'_b] K_b ----
  if (ok && tid == 0) {
    tc_fence_after();
    tc_mma4(tmem, dK(UT_R2), 2, dMN(UT_R0, 16384), 128, id_mnB, 0);
    tc_mma4(tmem, dK(UT_R2 + kTile), 2, dMN(UT_R0 + kTile, 16384), 128, id_mnB, 1);
    tc_commit(&sh.bar_mma);
  }
  ok = ok && wait_all(&sh.bar_mma, 0);
  // -W rows into staging boxes in R0 (K is no longer needed), then TMA stores.
  if (ok) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float w[64];
      tmem_ld64(lane_addr + 64 * hh, w);
      uint8_t* box = sm + UT_R0 + half * 16384 + hh * kTile;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float nw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) nw[i] = -w[8 * c + i];
        *reinterpret_cast<uint4*>(box + swz(t, c)) = pack8h(nw);
      }
    }
  }
  fence_proxy_async();
  __syncthreads();
  if (ok && tid == 0) {
    for (int hh = 0; hh < 2; ++hh)
      if (sh.hi[hh] > sh.lo[hh]) {
        const int row = (sh.slot[hh] * H + h) * 64;
        tma_store_2d(&tm_w, sm + UT_R0 + hh * 16384, 0, row);
        tma_store_2d(&tm_w, sm + UT_R0 + hh * 16384 + kTile, 64, row);
      }
    bulk_commit();
    bulk_wait_all();
  }
  if (!ok && tid == 0) record_error(a.err_word, GDN_DEVERR_TIMEOUT, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace

namespace gdn {
namespace host {

int launch_chunk_inverse(const PrefillArgs& a, const void* k, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_slots == 0) return GDN_OK;
  slot_map_kernel<<<(a.num_slots + 255) / 256, 256, 0, stream>>>(a);
  CUtensorMap mk, mt, mw;
  const int64_t rows = static_cast<int64_t>(a.num_slots) * a.H * 64;
  if (gdn_host::encode_tokens_map(&mk, k, a.T, a.H, kDimK) != GDN_OK ||
      gdn_host::encode_tiles_map_f16(&mt, a.tinv, rows, 64) != GDN_OK ||
      gdn_host::encode_tiles_map_f16(&mw, a.wneg, rows, 128) != GDN_OK)
    return GDN_ERR_CUDA;
  if (cudaFuncSetAttribute(ut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, UT_SMEM) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  const dim3 grid(static_cast<unsigned>((a.num_slots + 1) / 2), static_cast<unsigned>(a.H));
  ut_kernel<<<grid, kUtThreads, UT_SMEM, stream>>>(mk, mt, mw, a);
  return gdn_host::launch_status();
}

}  // namespace host
}  // namespace gdn
