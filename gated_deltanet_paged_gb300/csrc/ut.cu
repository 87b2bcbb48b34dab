// ut.cu -- the chunk-local part of chunked GDN prefill: for every 64-token chunk
// and head, T'' = (I + A)^-1 diag(beta) (stored by columns: tile row j holds
// column j) and -W = -T'' diag(gamma) K, written to the workspace.
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
// Mapping: one CTA of 128 threads per (pair of chunk slots, head).
//   [K_a; K_b] [K_a; K_b]^T   one M = 128 tcgen05 MMA, bf16 straight from TMA;
//                             thread r (TMEM lane r) reads row r of the stacked
//                             chunks and writes row r of A
//   T_d = diag(T11, T22)      inverses of (I + A)'s two 32 x 32 diagonal blocks
//                             by forward substitution on the CUDA cores in fp32,
//                             one column per thread (2 chunks x 2 blocks x 32
//                             columns = 128 threads, all with equal work):
//                             x_t = [t = c] - sum_{j<t} A[t][j] x_j
//   T21 = -T22 A21 T11        the remaining block of T = (I + A)^-1, by two MMAs:
//                             N21 = -T22 A21, then T21^T = T11^T N21^T (so that
//                             thread j reads column j of T21 from TMEM)
//   T'' = T diag(beta)        written (fp16) by columns into SW128 tiles that are
//                             both the staging of the T'' stores and the
//                             (M-major) A operand of W: a thread writes its column
//                             with 16-byte stores
//   -W = [T''_a; 0] K^_a + [0; T''_b] K^_b,  K^ = -diag(gamma) K converted to
//                             fp16 in place once the first MMA has read K
// The per-chunk B operands sit side by side ([X_a | X_b], N = 128) so one MMA
// serves both chunks (the off-diagonal result blocks are unused).
#include <math.h>

#include "prefill_common.cuh"

namespace {

using namespace gdn;

constexpr int kUtThreads = 128;
constexpr uint32_t kTile = 8192;  // 64 rows x 128 B

// Shared memory (offsets from the 1024-aligned base): two 32 KB regions that
// swap roles from one work item to the next.
//   K region:      K stack (bf16 boxes K_a kb0 | K_b kb0 | K_a kb1 | K_b kb1)
//                  -> K^ = diag(gamma) K (fp16, in place) -> -W staging
//   A-tile region: fp32 diagonal blocks of A (8 KB per chunk: rows 0-31 hold A11,
//                  rows 32-63 hold A22, 128 B per row) -> T_d stack (fp16 by
//                  columns, T_d,a | T_d,b, 64 x 64 SW128 each: tile row j =
//                  column j) in the first 16 KB; A21 of both chunks (fp16,
//                  MN-major B: 32 rows x 64 columns, 4 KB each, columns 32-63
//                  unused) -> N21 of both chunks (fp16, 64 rows: N21_a | N21_b,
//                  only columns 0-31 used) in the second 16 KB; after the second
//                  product T''_a | zero tile | T''_b by columns (24 KB)
// The next item's K lands in this item's A-tile region once its T'' stores
// have read it; this item's -W staging becomes the next item's A-tile region
// once the -W stores have read it.
constexpr uint32_t UT_REGION = 32768;
constexpr uint32_t UT_SMALL = 2 * UT_REGION;

struct UtSmall {
  float G[128];    // cumulative gate per stacked row
  float e[128];    // exp(g)
  float bet[128];  // beta
  float gam[128];  // exp(G)
  float wsum[4];   // per-warp gate totals for the scan
  uint64_t bar_tma, bar_mma;
  uint32_t tmem_base;
  int4 geo[2][2];  // [item parity][chunk]: first token, lo, hi, sequence of the chunk slot
  int next_it[2];  // [item parity]: the item after this one
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
// The same of x times s (paired fp32 multiplies).
__device__ __forceinline__ uint4 pack8h2(const float* x, float2 s) {
  uint4 u;
  u.x = pack_half2(__fmul2_rn(make_float2(x[0], x[1]), s));
  u.y = pack_half2(__fmul2_rn(make_float2(x[2], x[3]), s));
  u.z = pack_half2(__fmul2_rn(make_float2(x[4], x[5]), s));
  u.w = pack_half2(__fmul2_rn(make_float2(x[6], x[7]), s));
  return u;
}

// Byte offset of floats 4q..4q+3 (q < 8) of row r of a chunk's fp32 diagonal
// blocks (rows of 128 B; float4 q of row r sits at q ^ (r % 8), so a warp
// writing 32 rows at one q meets no bank conflict).
__device__ __forceinline__ uint32_t af(int r, int q) { return r * 128 + ((q ^ (r & 7)) << 4); }

// Column c (0..31) of (I + B)^-1 for a 32 x 32 diagonal block B of A whose row 0
// starts at blk (rows 128 B apart, the swizzle of af):
//   x_t = [t = c] - sum_{j<t} B[t][j] x_j.
// Every thread reads the same row at the same time (broadcast); four partial
// sums (j mod 4) keep the FMA chains short, and run as two paired fp32 FMAs
// where both halves of a pair have a term (each half rounds as a scalar FMA).
// hook(t) runs after step t (independent work that fills the steps' latency).
template <typename Hook>
__device__ __forceinline__ void solve32(const uint8_t* blk, int c, float (&x)[32], Hook&& hook) {
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (4 * m < t) {
        const float4 a4 = *reinterpret_cast<const float4*>(blk + af(t, m));
        if (4 * m + 1 < t)
          s01 = __ffma2_rn(make_float2(a4.x, a4.y), make_float2(x[4 * m], x[4 * m + 1]), s01);
        else
          s01.x = fmaf(a4.x, x[4 * m], s01.x);
        if (4 * m + 3 < t)
          s23 = __ffma2_rn(make_float2(a4.z, a4.w), make_float2(x[4 * m + 2], x[4 * m + 3]), s23);
        else if (4 * m + 2 < t)
          s23.x = fmaf(a4.z, x[4 * m + 2], s23.x);
      }
    }
    const float s = (s01.x + s01.y) + (s23.x + s23.y);
    x[t] = t > c ? -s : (t == c ? 1.f : 0.f);
    hook(t);
  }
}

// Chunk slot -> {first token of its 64 rows, lo, hi, sequence}; hi <= lo (and
// sequence -1) when the slot holds no chunk.
__global__ void slot_map_kernel(const PrefillArgs a) {
  pdl_wait();
  pdl_launch_dependents();
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
  int4 out = make_int4(0, 0, 0, -1);
  int cu_b, L, P;
  if (seq_extent(a, lo, cu_b, L, P)) {
    const int c = s - slot_base(cu_b, lo);
    if (c >= 0 && c < chunk_count(P, L)) {
      const int a0 = (P / 64) * 64 + 64 * c;
      out = make_int4(cu_b + a0 - P, max(P - a0, 0), min(P + L - a0, 64), lo);
    }
  }
  a.slot_geo[s] = out;
  if (s == 0) *a.item_counter = 0;
}

__global__ void __launch_bounds__(kUtThreads, 3)
    ut_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_t,
              const __grid_constant__ CUtensorMap tm_w, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  UtSmall& sh = *reinterpret_cast<UtSmall*>(sm + UT_SMALL);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = tid >> 6, t = tid & 63, r0 = half * 64;
  const int H = a.H;
  // Work items (pair of chunk slots, head), item = pair * H + head, taken by
  // persistent CTAs: items b and b + grid by CTA b, the rest one at a time from
  // a counter (item 2 grid + counter), so that CTAs on faster SMs take more
  // items and all finish together.  The two 32 KB regions swap roles from one
  // item to the next (K of item i -> the A tiles of item i+1), so the next
  // item's K is loaded while this one finishes.
  const int nitems = ((a.num_slots + 1) / 2) * H;

  // Geometry of item it's two chunk slots into geo[b] (threads t == 0).
  auto load_geo = [&](int it, int b) {
    const int s = 2 * (it / H) + half;
    sh.geo[b][half] = (it < nitems && s < a.num_slots) ? a.slot_geo[s] : make_int4(0, 0, 0, -1);
  };
  // K of item it (geometry in geo[b]) into the region at kbase (thread 0).
  auto issue_k = [&](int it, int b, uint32_t kbase) {
    const int hd = it % H;
    uint32_t bytes = 0;
    for (int hh = 0; hh < 2; ++hh) bytes += sh.geo[b][hh].z > sh.geo[b][hh].y ? 16384u : 0u;
    mbar_arrive_expect_tx(&sh.bar_tma, bytes);
    for (int hh = 0; hh < 2; ++hh) {
      const int4 g = sh.geo[b][hh];
      if (g.z <= g.y) continue;
      tma_load_3d(sm + kbase + hh * kTile, &tm_k, &sh.bar_tma, 0, hd, g.x);
      tma_load_3d(sm + kbase + 16384 + hh * kTile, &tm_k, &sh.bar_tma, 64, hd, g.x);
    }
  };
  // g and beta of row t of this thread's chunk of item it (geometry in geo[b]).
  float gv_n = 0.f, bv_n = 0.f;
  auto load_gb = [&](int it, int b) {
    const int4 g = sh.geo[b][half];
    gv_n = 0.f;
    bv_n = 0.f;
    if (it < nitems && t >= g.y && t < g.z) {
      const int64_t idx = static_cast<int64_t>(g.x + t) * H + it % H;
      gv_n = a.g[idx];
      bv_n = a.beta[idx];
    }
  };

  pdl_wait();  // the slot map (and everything before it on the stream) is done
  // No early pdl_launch_dependents here: the state chain that follows would
  // then take SMs one by one as this kernel drains, and that placement made it
  // 13% slower (measured); it launches when this kernel completes.
  int it = blockIdx.x;
  if (tid == 0) {
    mbar_init(&sh.bar_tma, 1);
    mbar_init(&sh.bar_mma, 1);
    sh.flag = 0;
    sh.next_it[0] = it + gridDim.x;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_t);
    prefetch_tensormap(&tm_w);
  }
  if (t == 0) load_geo(it, 0);
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  if (tid == 0) issue_k(it, 0, UT_REGION);
  load_gb(it, 0);

  auto dK = [&](uint32_t off) { return sdesc(sbase + off, 16, 1024); };
  auto dMN = [&](uint32_t off, uint32_t lbo) { return sdesc(sbase + off, lbo, 1024); };
  const uint32_t id_bf16 = idesc_f16(128, 128, true, true, false, false);
  const uint32_t id_mnAB = idesc_f16(128, 128, false, false, true, true);
  const uint32_t id_t21 = idesc_f16(128, 64, false, false, false, false);

  // Every thread waits for the MMA; a time-out anywhere aborts the CTA.
  auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (!mbar_wait(bar, parity)) sh.flag = 1;
    __syncthreads();
    tc_fence_after();
    return sh.flag == 0;
  };

  uint32_t mph = 0;  // parity of the next bar_mma phase
  auto wait_mma = [&]() -> bool {
    const bool r = wait_all(&sh.bar_mma, mph);
    mph ^= 1;
    return r;
  };

  bool ok = true;
  for (int i = 0; it < nitems && ok; ++i) {
    const int b = i & 1;
    const uint32_t KB = (i & 1) ? 0u : UT_REGION;  // K, then K^, then the -W staging
    const uint32_t XB = UT_REGION - KB;            // A blocks, T_d, A21 -> N21, then the T'' tiles
    const int pair = it / H, h = it % H, nit = sh.next_it[b];
    // the item after the next one (warp 1 waits for the counter only at the
    // end of this item, where it publishes the number for the next)
    int grabbed = 0;
    auto grab = [&]() {
      if (tid == 32 && nit < nitems) grabbed = atomicAdd(a.item_counter, 1);
    };
    auto publish_next = [&]() {
      if (tid == 32) sh.next_it[b ^ 1] = nit < nitems ? 2 * static_cast<int>(gridDim.x) + grabbed : nitems;
    };
    const int4 ga = sh.geo[b][0], gb = sh.geo[b][1];
    const bool va = ga.z > ga.y, vb = gb.z > gb.y;
    const int lo = half ? gb.y : ga.y, hi = half ? gb.z : ga.z;
    if (va || vb) grab();
    if (t == 0) load_geo(nit, b ^ 1);

    // Gates of this row; inclusive scan over the chunk's 64 rows.
    const bool vme = t >= lo && t < hi;
    const float gv = gv_n, bv = bv_n;
    float s = gv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    if (lane == 31) sh.wsum[warp] = s;
    tc_fence_before();  // the previous item's TMEM reads come before this item's first MMA
    __syncthreads();
    tc_fence_after();
    if (warp & 1) s += sh.wsum[warp - 1];
    sh.G[tid] = s;
    sh.e[tid] = __expf(gv);
    sh.bet[tid] = bv;
    sh.gam[tid] = __expf(s);
    load_gb(nit, b ^ 1);  // in flight during this item

    // K -> K^ = -diag(gamma) K in fp16, in place (the first MMA has read K); its
    // sign makes the W product come out as -W.  The 16 pieces of 16 bytes of a
    // thread (piece i = tid + 128 k of the boxes K_a kb0 | K_b kb0 | K_a kb1 |
    // K_b kb1) are converted between the steps of the 32 x 32 solve, whose
    // dependent chain leaves the issue slots for them: piece k is loaded one
    // hook before it is converted and stored.
    uint4 kin = make_uint4(0u, 0u, 0u, 0u);
    float kg = 0.f;
    auto khat_load = [&](int k) {
      const int i = tid + kUtThreads * k;
      kin = *reinterpret_cast<const uint4*>(sm + KB + i * 16);
      kg = -sh.gam[((i >> 9) & 1) * 64 + ((i & 511) >> 3)];
    };
    auto khat_store = [&](int k, const uint4 in, float g) {
      const int i = tid + kUtThreads * k;
      const int hh = (i >> 9) & 1, row = (i & 511) >> 3;
      const bool keep = hh ? (row >= gb.y && row < gb.z) : (row >= ga.y && row < ga.z);
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (keep) {
        const float2 g2 = make_float2(g, g);
        out.x = pack_half2(__fmul2_rn(unpack_bf162(in.x), g2));
        out.y = pack_half2(__fmul2_rn(unpack_bf162(in.y), g2));
        out.z = pack_half2(__fmul2_rn(unpack_bf162(in.z), g2));
        out.w = pack_half2(__fmul2_rn(unpack_bf162(in.w), g2));
      }
      *reinterpret_cast<uint4*>(sm + KB + i * 16) = out;
    };
    // after odd solve steps t: piece k = t / 2 is stored, piece k + 1 loaded
    auto khat_hook = [&](int t) {
      if ((t & 1) == 0) return;
      const int k = t >> 1;
      const uint4 in = kin;
      const float g = kg;
      if (k + 1 < 16) khat_load(k + 1);
      khat_store(k, in, g);
    };

    // ---- [K_a; K_b] [K_a; K_b]^T ----
    if (tid == 0) {
      if (mbar_wait(&sh.bar_tma, i & 1)) {
        tc_fence_after();
        if (va || vb) {
          tc_mma4(tmem, dK(KB), 2, dK(KB), 2, id_bf16, 0);
          tc_mma4(tmem, dK(KB + 16384), 2, dK(KB + 16384), 2, id_bf16, 1);
          tc_commit(&sh.bar_mma);
        }
      } else {
        sh.flag = 1;
      }
      // the previous item's -W stores have read this item's A-tile region
      // (written after the barrier of the product's wait)
      bulk_wait_read();
    }
    if (!(va || vb)) {  // no chunk in either slot: nothing to compute or store
      grab();
      publish_next();
      __syncthreads();
      ok = sh.flag == 0;
      if (ok && tid == 0 && nit < nitems) issue_k(nit, b ^ 1, XB);
      it = nit;
      continue;
    }
    // (if thread 0's wait for K ran out, the product was never committed: every
    // thread's wait below runs out too, and the barrier inside reports it)
    ok = ok && wait_mma();

    // ---- row t of A: the diagonal block part in fp32, A21 in fp16 ----
    if (ok) {
      float kk[64];
      tmem_ld64(lane_addr + r0, kk);
      const float Gt = sh.G[tid];
      uint8_t* arow = sm + XB + half * 8192;
      uint8_t* a21 = sm + XB + 16384 + half * 4096;
      const bool lower = t >= 32;  // warp-uniform
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q >= 2 && !lower) break;
        float out[16];
        const int jstart = min(16 * q + 15, t - 1);  // last column of the strict lower part
        if (vme && jstart >= 16 * q) {
          // The block's gate values come into registers together (shared-memory
          // loads would otherwise wait behind the previous block's stores).
          float eb[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) eb[jj] = sh.e[r0 + 16 * q + jj];
          // (A21 is kept negated, so that the first small product gives N21 itself)
          float cur = (lower && q < 2 ? -bv : bv) * __expf(Gt - sh.G[r0 + jstart]);
#pragma unroll
          for (int i = 7; i >= 0; --i) {  // a running product downwards from jstart; products in pairs
            const int ja = 16 * q + 2 * i, jb = ja + 1;
            const float cb = cur;
            if (jb <= jstart) cur *= eb[2 * i + 1];
            const float ca = cur;
            if (ja <= jstart) cur *= eb[2 * i];
            const float2 pr = __fmul2_rn(make_float2(ca, cb), make_float2(kk[ja], kk[jb]));
            out[2 * i] = (ja <= jstart && ja >= lo) ? pr.x : 0.f;
            out[2 * i + 1] = (jb <= jstart && jb >= lo) ? pr.y : 0.f;
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) out[jj] = 0.f;
        }
        if (lower && q < 2) {
          *reinterpret_cast<uint4*>(a21 + swz(t - 32, 2 * q)) = pack8h(&out[0]);
          *reinterpret_cast<uint4*>(a21 + swz(t - 32, 2 * q + 1)) = pack8h(&out[8]);
        } else {
          const int qb = 4 * (q & 1);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float4*>(arow + af(t, qb + k)) =
                make_float4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
        }
      }
      // (columns 32-63 of the A21 tile only feed products that are discarded)
    }
    fence_proxy_async();
    // A warp solves the diagonal block whose rows it wrote itself (warp w: chunk
    // w / 2, rows 32 (w % 2) .. + 31), so a warp barrier is enough here; the
    // CTA-wide one before the first small product orders the rest.
    __syncwarp();

    // ---- T_d: thread (chunk, block bk, column c) solves column c of block bk ----
    const int bk = warp & 1;
    float x[32];
    if (ok) {
      khat_load(0);
      solve32(sm + XB + half * 8192 + bk * 32 * 128, lane, x, khat_hook);
    }
    __syncwarp();  // every lane has read this warp's block: the space becomes its T_d columns
    // T_d is kept by columns (tile row j = column j of T_d, 64 rows t in 128
    // bytes), so each thread writes its solved column with four 16-byte stores.
    // Only the diagonal blocks are written: the products below read the blocks
    // off the diagonal only into products that are discarded.
    const int jcol = 32 * bk + lane;
    if (ok) {
      uint8_t* td = sm + XB + half * 8192;
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(td + swz(jcol, 4 * bk + q)) = pack8h(&x[8 * q]);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- N21 = -T22 A21 = T22 (-A21): [T_d,a; T_d,b] (K = 32..63; by columns, so
    //      M-major) x [-A21_a | -A21_b] ----
    if (ok && tid == 0) {
      tc_fence_after();
      tc_mma2(tmem, dMN(XB + 32 * 128, 8192), 128, dMN(XB + 16384, 4096), 128, id_mnAB, 0);
      tc_commit(&sh.bar_mma);
    }
    ok = ok && wait_mma();
    if (ok && bk == 1) {  // rows 32-63 of each chunk -> rows 32 h + i of the N21 stack
      float d[32];
      tmem_ld32(lane_addr + r0, d);
      uint8_t* nt = sm + XB + 16384;  // over A21, which the first small product has read
      const int nr = 32 * half + lane;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) *reinterpret_cast<uint4*>(nt + swz(nr, cc)) = pack8h(&d[8 * cc]);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- T21^T = T11^T N21^T: [T_d,a by columns; T_d,b by columns] (K = rows
    //      0..31) x [N21_a; N21_b]^T (N = 64): lane 64 h + j, column 32 h + i holds
    //      T21[i][j] of chunk h ----
    if (ok && tid == 0) {
      tc_fence_after();
      tc_mma2(tmem, dK(XB), 2, dK(XB + 16384), 2, id_t21, 0);
      tc_commit(&sh.bar_mma);
    }
    ok = ok && wait_mma();

    // ---- T'' = T diag(beta) by columns (tile row j = column j) into T''_a | 0 |
    //      T''_b (T_d, A21 and N21 are dead): thread (chunk, bk, lane) writes
    //      column j = 32 bk + lane, beta_j times its solved block and, for bk = 0,
    //      T21's column from TMEM; zeros above the diagonal block for bk = 1 ----
    if (ok) {
      uint8_t* tile = sm + XB + half * 16384;
      const float bc = sh.bet[tid];
      const float2 bc2 = make_float2(bc, bc);
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(tile + swz(jcol, 4 * bk + q)) = pack8h2(&x[8 * q], bc2);
      if (bk == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(tile + swz(jcol, q)) = make_uint4(0u, 0u, 0u, 0u);
      } else {  // warps 0 and 2: TMEM lanes 64 h + j
        float d[32];
        tmem_ld32(lane_addr + 32 * half, d);
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(tile + swz(jcol, 4 + q)) = pack8h2(&d[8 * q], bc2);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        reinterpret_cast<uint4*>(sm + XB + kTile)[tid + 128 * k] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- -W = [T''_a; 0] K^_a + [0; T''_b] K^_b;  T'' tiles -> workspace ----
    if (ok && tid == 0) {
      tc_fence_after();
      tc_mma4(tmem, dMN(XB, kTile), 128, dMN(KB, 16384), 128, id_mnAB, 0);
      tc_mma4(tmem, dMN(XB + kTile, kTile), 128, dMN(KB + kTile, 16384), 128, id_mnAB, 1);
      tc_commit(&sh.bar_mma);
      for (int hh = 0; hh < 2; ++hh)
        if (hh ? vb : va) tma_store_2d(&tm_t, sm + XB + hh * 16384, 0, ((2 * pair + hh) * H + h) * 64);
      bulk_commit();
    }
    ok = ok && wait_mma();
    // -W rows into staging boxes over K^ (the MMA has read it), then TMA stores.
    if (ok) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float w[64];
        tmem_ld64(lane_addr + 64 * hh, w);
        uint8_t* box = sm + KB + half * 16384 + hh * kTile;
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(box + swz(t, c)) = pack8h(&w[8 * c]);
      }
    }
    // Once the T'' stores (issued with the product, so normally done by now)
    // have read the A-tile region, the next item's K may land there.
    if (ok && tid == 0 && nit < nitems) {
      bulk_wait_read();
      issue_k(nit, b ^ 1, XB);
    }
    fence_proxy_async();
    publish_next();
    __syncthreads();
    it = nit;
    if (tid == 0) {
      if (ok)
        for (int hh = 0; hh < 2; ++hh)
          if (hh ? vb : va) {
            const int row = ((2 * pair + hh) * H + h) * 64;
            tma_store_2d(&tm_w, sm + KB + hh * 16384, 0, row);
            tma_store_2d(&tm_w, sm + KB + hh * 16384 + kTile, 64, row);
          }
      bulk_commit();  // read before the next item writes its A tiles here
    }
  }
  if (tid == 0) bulk_wait_read();
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

int launch_chunk_inverse(const PrefillArgs& a, const CUtensorMap& mk, const CUtensorMap& mt, const CUtensorMap& mw,
                         int num_sms, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_slots == 0) return GDN_OK;
  int rc = gdn_host::launch_pdl(slot_map_kernel, dim3((a.num_slots + 255) / 256), dim3(256), 0, stream, a);
  if (rc != GDN_OK) return rc;
  static std::atomic<uint64_t> smem_set{0};
  rc = gdn_host::func_attr_once(ut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, UT_SMEM, smem_set);
  if (rc != GDN_OK) return rc;
  // Persistent CTAs: three per SM (the shared-memory and register budget), each
  // taking work items in strides of the grid.
  const long long items = static_cast<long long>((a.num_slots + 1) / 2) * a.H;
  const unsigned grid = static_cast<unsigned>(items < 3LL * num_sms ? items : 3LL * num_sms);
  return gdn_host::launch_pdl(ut_kernel, dim3(grid), dim3(kUtThreads), UT_SMEM, stream, mk, mt, mw, a);
}

}  // namespace host
}  // namespace gdn
