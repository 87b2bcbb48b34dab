// prefill_common.cuh -- what the prefill kernels share: the call's arguments,
// the per-sequence geometry (prefix, chunks) and the workspace layout.
//
// "flashinfer.gdn_paged": chunk_gated_delta_rule_paged and "Slot arguments of
// chunk_gated_delta_rule".  Chunks are 64 tokens aligned to ABSOLUTE positions:
// the first chunk of a sequence with prefix P starts at 64 floor(P / 64), its
// rows before P are left padding (the identity step), so page / checkpoint
// boundaries (multiples of 64) always fall on chunk ends.
#pragma once

#include "common.cuh"

namespace gdn {

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
  // The slot arrays: int32, or int64 when index64 is set (index_at reads both).
  const void* state_indices;
  float* output_state;
  const void* output_state_indices;
  float* state_checkpoints;
  const void* checkpoint_state_indices;
  const void* checkpoint_cu_starts;
  const void* prefix_lens;
  int32_t index64;
  int32_t N;
  int64_t row_stride;  // elements of the pools' type
  int32_t state_bf16;  // pools of bf16 (states widened on load, rounded to nearest on store), else fp32
  // Paged mode without precomputed slots: rows come from the page table.
  const int32_t* indptr;
  const int32_t* pages;
  const int32_t* last_len;
  int32_t page_size;
  int32_t num_pages;
  int32_t* err_word;
  // Workspace: per chunk slot its geometry {first token, lo, hi, sequence}
  // (rows lo..hi-1 of the 64 hold tokens first + lo .. first + hi - 1; hi <= lo
  // for a slot without a chunk), then per (chunk slot, head) a 64 x 64 fp16
  // tile T'' = (I + A)^-1 diag(beta) and a 64 x 128 fp16 tile
  // -W = -T'' diag(gamma) K.
  int4* slot_geo;
  int32_t* item_counter;  // the chunk-local kernel's work counter (after the map; zeroed by the slot map)
  __half* tinv;
  __half* wneg;
  int32_t num_slots;
  // Test hook (gdn_debug_set_wait_stall): the state chain's first wait is on a
  // barrier that nothing completes, so that its time-out path runs.
  int32_t debug_stall;
};

// Workspace chunk slots.  Chunk c of sequence b lives in slot
//   base_b + c,  base_b = floor(cu_seqlens[b] / 64) + 2 b.
// A sequence has at most floor(L / 64) + 2 chunks and base_{b+1} - base_b >=
// floor(L_b / 64) + 2, so slots of different sequences never meet, and every
// slot is below floor(T / 64) + 2 S + 2.
__host__ __device__ inline int64_t num_chunk_slots(int64_t T, int64_t num_seqs) { return T / 64 + 2 * num_seqs + 2; }
__device__ inline int slot_base(int cu_b, int b) { return cu_b / 64 + 2 * b; }

constexpr uint32_t kTinvBytes = 64 * 64 * 2;  // one T'' tile
constexpr uint32_t kWBytes = 64 * 128 * 2;    // one -W tile

// The map (16 bytes per slot) and the work counter (16 bytes), rounded up to 1 KB.
__host__ __device__ inline size_t workspace_map_bytes(int64_t num_slots) {
  return static_cast<size_t>((num_slots * 16 + 16 + 1023) / 1024 * 1024);
}
__host__ __device__ inline size_t workspace_bytes(int64_t T, int64_t num_seqs, int64_t H) {
  const int64_t ns = num_chunk_slots(T, num_seqs);
  return workspace_map_bytes(ns) + static_cast<size_t>(ns) * H * (kTinvBytes + kWBytes);
}

// Entry i of a slot array of int32 (wide == 0) or int64 elements.
__device__ inline int64_t index_at(const void* p, int64_t i, int32_t wide) {
  return wide ? static_cast<const int64_t*>(p)[i] : static_cast<int64_t>(static_cast<const int32_t*>(p)[i]);
}

// Prefix length P, start cu_b and new length L of sequence b.  Returns false
// for a zero-length sequence or arguments no kernel may act on (the chain
// kernel reports those in err_word).
__device__ inline bool seq_extent(const PrefillArgs& a, int b, int& cu_b, int& L, int& P) {
  cu_b = a.cu_seqlens[b];
  L = a.cu_seqlens[b + 1] - cu_b;
  if (L <= 0 || cu_b < 0 || static_cast<long long>(cu_b) + L > a.T) return false;
  if (a.indptr) {
    const int n = a.indptr[b + 1] - a.indptr[b];
    const int lpl = a.last_len[b];
    const long long tot = static_cast<long long>(n - 1) * a.page_size + lpl;
    if (n < 1 || lpl < 1 || lpl > a.page_size || tot < L || tot > 0x3FFFFFFFLL) return false;
    P = static_cast<int>(tot - L);
  } else {
    const int64_t p64 = a.prefix_lens ? index_at(a.prefix_lens, b, a.index64) : 0;
    if (p64 < 0 || p64 + L > 0x3FFFFFFFLL) return false;
    P = static_cast<int>(p64);
  }
  return true;
}

__device__ inline int chunk_count(int P, int L) { return (P + L + 63) / 64 - P / 64; }

namespace host {
// Enqueue the slot map and the chunk-local inverse kernels (ut.cu): mk is the
// tensor map of K, mt and mw those of the T'' and -W tiles (shared with the
// state chain), num_sms the device's SM count.
int launch_chunk_inverse(const PrefillArgs& a, const CUtensorMap& mk, const CUtensorMap& mt, const CUtensorMap& mw,
                         int num_sms, cudaStream_t stream);
}  // namespace host

}  // namespace gdn
