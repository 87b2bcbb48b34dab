/*
 * gdn_paged.h -- C ABI of paged Gated Delta-Rule (GDN) prefill and decode on
 * GB300 (sm_103a).
 *
 * Source: "flashinfer.gdn_paged" (docs.flashinfer.ai/api/gdn_paged.html) --
 * the intro, §Page table, the prefill bullets, the decode paragraph, the pool /
 * padding paragraph and "Slot arguments of chunk_gated_delta_rule".  The pages
 * name the method but print no formula for it; the library computes the
 * standard gated delta rule on a V x K state per (sequence, head):
 *     S_t = exp(g_t) S_{t-1} + beta_t (v_t - exp(g_t) S_{t-1} k_t) k_t^T
 *     o_t = scale * S_t q_t
 *
 * Conventions shared by every call
 *   - All array pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no memory and keeps no pointer after a call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronises the host.
 *   - bf16 tensors are passed as raw 16-bit patterns (gdn_bf16).
 *   - Token layout is packed varlen: q, k are [T, H, K], v and o are [T, H, V],
 *     g and beta are [T, H] (fp32, g is the log-space gate applied as exp(g)).
 *     Decode uses [B, H, .] (the same memory as [B, 1, H, .]).
 *   - The state pool is fp32 [rows, H, V, K] (or bf16 through the _ex calls,
 *     see GDN_STATE_BF16); one row is a dense [H, V, K] block at
 *     row * pool_row_stride elements.  Page j of a sequence holds the state
 *     after the last token of that page.
 *   - Page tables are CSR: sequence b owns page_indices[page_indptr[b] ..
 *     page_indptr[b+1]) (any ids, any order) and has
 *     (num_pages_b - 1) * page_size + last_page_len[b] tokens AFTER the call;
 *     its new tokens are the last ones, the ones before are its prefix.
 *   - K and V must be 128.  q, k, v, o, g, beta and every pool must be 16-byte
 *     aligned.
 *   - scale <= 0 selects the default 1/sqrt(K).
 *   - Return value: GDN_OK, or a negative status (no exception crosses the
 *     ABI).  Host-side checks cover scalars, null pointers and alignment only;
 *     nothing is read back from the device.
 *   - err_word (nullable, device int32 the caller zeroes): when given, the
 *     kernels also check device-side data (page ids against [0, num_pages),
 *     page-table consistency) and record the first violation as
 *     (kind << 24) | sequence, kind one of GDN_DEVERR_*; a sequence that fails
 *     a check is skipped.  Without it the data are trusted.
 *   - Preconditions (unchecked): page ids are real ids (-1 is not a padding
 *     value); rows written by one sequence are not read or written by another
 *     sequence of the same call; a decoded sequence holds at least one token
 *     before the decoded one.
 *   - fp16 range of the prefill: its tensor-core products run on fp16
 *     operands, so q, k and v elements must lie within +-65504 and the states
 *     and intermediate values they produce must stay within the fp16 range.
 *     Larger values turn into infinities, and the sequence's outputs and
 *     states then hold non-finite values.  With err_word the prefill kernels
 *     check every q, k and v element they convert and every state they store,
 *     and report a violation as GDN_DEVERR_RANGE (the sequence still runs).
 */
#ifndef GDN_PAGED_H
#define GDN_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gdn_bf16; /* raw bfloat16 bit pattern */

#define GDN_OK 0
#define GDN_ERR_INVALID_ARGUMENT (-1) /* null pointer, bad scalar, misalignment */
#define GDN_ERR_UNSUPPORTED (-2)      /* K or V other than 128, no sm_103a device */
#define GDN_ERR_CUDA (-3)             /* a CUDA launch or driver call failed */

/* Element type of a state pool (the state_dtype of the _ex calls).  The pages
 * ask for a state dtype that prefill and decode both support.  With
 * GDN_STATE_BF16 the kernels still carry every state in fp32 on the chip; a
 * state read from the pool is widened exactly, and a stored state is rounded
 * to the nearest bf16 value (ties to even).  pool_row_stride then counts bf16
 * elements. */
#define GDN_STATE_F32 0
#define GDN_STATE_BF16 1

/* Element type of the slot arrays of gdn_chunk_gated_delta_rule_ex
 * ("Slot arguments of chunk_gated_delta_rule": each is an int32 or int64
 * tensor). */
#define GDN_INDEX_I32 0
#define GDN_INDEX_I64 1

#define GDN_DEVERR_PAGE_ID 1       /* a page id outside [0, num_pages) */
#define GDN_DEVERR_PAGE_TABLE 2    /* no page, last_page_len outside 1..page_size, more new tokens than tokens, or tokens past total_tokens */
#define GDN_DEVERR_NO_PREV_TOKEN 3 /* decode: the decoded token is the sequence's first */
#define GDN_DEVERR_INDEX_RANGE 4   /* an int64 slot entry outside the int32 range (rows below -1) */
#define GDN_DEVERR_RANGE 5         /* prefill: a q, k or v element beyond the fp16 range (|x| > 65504, or NaN), or a stored state that is not finite */
#define GDN_DEVERR_TIMEOUT 15      /* an internal wait ran past its iteration limit */

/* Per-sequence pool rows of a paged prefill batch, each int32 [num_seqs] on
 * the device ("GDNPagedPrefillSlots"). */
typedef struct {
    int32_t *state_indices;        /* row of the page holding the last prefix token, -1 if no prefix */
    int32_t *output_state_indices; /* last page, -1 for a zero-length sequence */
    int32_t *checkpoint_cu_starts; /* index into page_indices of the first page ending after the prefix */
    int32_t *prefix_lens;          /* tokens before the new ones */
} gdn_prefill_slots;

/* Per-sequence pool rows of a paged decode batch, each int32 [B] on the device
 * ("GDNPagedDecodeSlots"). */
typedef struct {
    int32_t *initial_state_indices; /* previous page when last_page_len == 1, else the last page */
    int32_t *output_state_indices;  /* last page */
} gdn_decode_slots;

/* gdn_paged_prefill_slots -- "gdn_paged_prefill_slots(cu_seqlens, ...)" and
 * §Page table: derive the rows the paged prefill uses, in one launch with no
 * host synchronisation.  For sequence b with n_b pages, L_b new tokens and
 * P_b = (n_b - 1) * page_size + last_page_len[b] - L_b prefix tokens:
 *   state_indices[b]        = P_b > 0 ? page_indices[page_indptr[b] + (P_b - 1) / page_size] : -1
 *   output_state_indices[b] = L_b > 0 ? page_indices[page_indptr[b+1] - 1] : -1
 *   checkpoint_cu_starts[b] = page_indptr[b] + P_b / page_size
 *   prefix_lens[b]          = P_b
 * A sequence with no page, a last_page_len outside 1..page_size, P_b < 0, or
 * more than 2^30 - 1 tokens gets -1 rows, prefix 0 (the rows the prefill
 * kernels would skip).
 * Inputs: cu_seqlens [num_seqs+1], page_indptr [num_seqs+1], page_indices,
 * last_page_len [num_seqs]; outputs four int32 [num_seqs] arrays.
 * page_size must be a positive multiple of 64. */
int gdn_paged_prefill_slots(const int32_t *cu_seqlens, const int32_t *page_indptr,
                            const int32_t *page_indices, const int32_t *last_page_len,
                            int32_t num_seqs, int32_t page_size, int32_t *state_indices,
                            int32_t *output_state_indices, int32_t *checkpoint_cu_starts,
                            int32_t *prefix_lens, void *stream);

/* gdn_paged_decode_slots -- "gdn_paged_decode_slots(page_indices, ...)" and the
 * decode paragraph: initial_state_indices[b] is the previous page when the
 * decoded token opens a page (last_page_len[b] == 1), otherwise the last page;
 * output_state_indices[b] is the last page.  A one-page sequence with
 * last_page_len 1 (outside the contract) reads -1, the zero state.
 * Inputs: page_indptr [batch+1], page_indices, last_page_len [batch]; outputs
 * two int32 [batch] arrays. */
int gdn_paged_decode_slots(const int32_t *page_indptr, const int32_t *page_indices,
                           const int32_t *last_page_len, int32_t batch,
                           int32_t *initial_state_indices, int32_t *output_state_indices,
                           void *stream);

/* gdn_chunk_gated_delta_rule -- "Slot arguments of chunk_gated_delta_rule":
 * chunked prefill on explicit rows.  For every sequence b (new tokens
 * cu_seqlens[b] .. cu_seqlens[b+1]-1) and head:
 *   - start from row state_indices[b] of initial_state, or from the zero state
 *     when state_indices is NULL or the row is -1 (the pool is not read);
 *   - after new token n with (prefix_lens[b] + n) % N == 0 (N =
 *     checkpoint_every_n_tokens) store the state to row
 *     checkpoint_state_indices[checkpoint_cu_starts[b] + j] of
 *     state_checkpoints, j counting this call's checkpoints of b from 0; a row
 *     of -1 skips it.  Sequence b has (P_b + L_b) / N - P_b / N checkpoints;
 *   - store the final state to row output_state_indices[b] of output_state
 *     unless that is NULL or -1;
 *   - a zero-length sequence reads and writes nothing.
 * Tokens are processed in 64-token chunks aligned to absolute positions
 * (prefix_lens, 0 when NULL); a prefix that is not a multiple of 64 pads the
 * first chunk on the left.  The checkpoint arrays (state_checkpoints,
 * checkpoint_state_indices, checkpoint_cu_starts) are all given or all NULL;
 * when given, prefix_lens is required and N must be a positive multiple of 64.
 * initial_state, output_state and state_checkpoints may be the same pool;
 * pool_row_stride (elements) is >= H*V*K and a multiple of 4.
 * total_tokens is T, the first dimension of q/k/v/o.
 * workspace: caller-owned device memory of at least
 * gdn_prefill_workspace_bytes(num_seqs, total_tokens, H) bytes, 16-byte
 * aligned (GDN_ERR_INVALID_ARGUMENT otherwise).  The call overwrites it; its
 * contents need no initialisation and mean nothing afterwards, and two calls
 * in flight at once need two workspaces. */
int gdn_chunk_gated_delta_rule(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                               const float *g, const float *beta, gdn_bf16 *o,
                               const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                               int32_t H, int32_t K, int32_t V, float scale,
                               const float *initial_state, const int32_t *state_indices,
                               float *output_state, const int32_t *output_state_indices,
                               float *state_checkpoints, const int32_t *checkpoint_state_indices,
                               const int32_t *checkpoint_cu_starts, const int32_t *prefix_lens,
                               int32_t checkpoint_every_n_tokens, int64_t pool_row_stride,
                               void *workspace, size_t workspace_bytes, int32_t *err_word,
                               void *stream);

/* gdn_chunk_gated_delta_rule_paged -- "chunk_gated_delta_rule_paged(q, k, v,
 * ...)": chunked prefill over a paged pool state_pool[num_pages, H, V, K].  It
 * reads the page holding the last prefix token (zero state for an empty
 * prefix), stores the state at every page boundary the new tokens cross to the
 * page ending there and the final state to the last page, and never writes a
 * page that ends at or before the prefix.  It is the slot-argument call above
 * with state_pool as all three pools, page_indices as checkpoint rows and
 * N = page_size.  slots (nullable): rows from gdn_paged_prefill_slots, e.g.
 * computed once per step and shared by all layers; when NULL the kernels
 * derive them from the page table.  page_size must be a positive multiple of
 * 64.  workspace / workspace_bytes: as for gdn_chunk_gated_delta_rule. */
int gdn_chunk_gated_delta_rule_paged(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                     const float *g, const float *beta, gdn_bf16 *o,
                                     const int32_t *cu_seqlens, int32_t num_seqs,
                                     int32_t total_tokens, int32_t H, int32_t K, int32_t V,
                                     float scale, float *state_pool, int32_t num_pages,
                                     const int32_t *page_indices, const int32_t *page_indptr,
                                     int32_t page_size, const int32_t *last_page_len,
                                     const gdn_prefill_slots *slots, void *workspace,
                                     size_t workspace_bytes, int32_t *err_word, void *stream);

/* gdn_chunk_gated_delta_rule_paged_static_workspace -- no counterpart in the
 * method's published API; it exists for callers that cannot allocate device
 * memory (a runtime whose memory all belongs to its own pool, a plugin host
 * that forbids device allocations, a serving loop that cannot take the device
 * synchronisation an allocation may cause).  Same arguments and result as
 * gdn_chunk_gated_delta_rule_paged without workspace / workspace_bytes: the
 * workspace is a fixed 64 MiB array in the library's device image, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing; it returns GDN_ERR_UNSUPPORTED when
 * gdn_prefill_workspace_bytes(num_seqs, total_tokens, H) exceeds 64 MiB
 * (roughly total_tokens * H <= 170,000).  The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call outside any stream capture.  All calls share
 * the one array: nothing in it needs to start at zero (each call writes what
 * it reads), but calls whose executions overlap on the GPU (other streams,
 * other host threads) race on it and must be serialised by the caller. */
int gdn_chunk_gated_delta_rule_paged_static_workspace(
    const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v, const float *g, const float *beta,
    gdn_bf16 *o, const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H,
    int32_t K, int32_t V, float scale, float *state_pool, int32_t num_pages,
    const int32_t *page_indices, const int32_t *page_indptr, int32_t page_size,
    const int32_t *last_page_len, const gdn_prefill_slots *slots, int32_t *err_word,
    void *stream);

/* gdn_gated_delta_rule_decode_paged -- "gated_delta_rule_decode_paged(q, k, v,
 * ...)": one token per sequence.  When the token opens a new page
 * (last_page_len[b] == 1) the state is read from the previous page and written
 * to the new one; otherwise the last page is updated in place.  q, k are
 * [batch, H, K], v and o [batch, H, V], g and beta [batch, H].  slots
 * (nullable): rows from gdn_paged_decode_slots (or any explicit read / write
 * rows, -1 read = zero state, -1 write = skip); when NULL the kernel derives
 * them from the page table.  The kernel is launched as a programmatic
 * dependent of the previous kernel on the stream (it waits for that kernel to
 * complete before reading anything), so stream order holds as for any launch. */
int gdn_gated_delta_rule_decode_paged(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                      const float *g, const float *beta, gdn_bf16 *o,
                                      int32_t batch, int32_t H, int32_t K, int32_t V, float scale,
                                      float *state_pool, int32_t num_pages,
                                      const int32_t *page_indices, const int32_t *page_indptr,
                                      const int32_t *last_page_len, const gdn_decode_slots *slots,
                                      int32_t *err_word, void *stream);

/* The three calls above with the pool element type as an argument
 * (state_dtype: GDN_STATE_F32 or GDN_STATE_BF16; anything else is
 * GDN_ERR_INVALID_ARGUMENT).  Pools are passed untyped; every pool of one call
 * has that element type.  For bf16 pools pool_row_stride (elements) must be a
 * multiple of 8, so rows stay 16-byte aligned.  The fp32 calls above are these
 * with GDN_STATE_F32.
 * The general call also takes the element type of its five slot arrays
 * (state_indices, output_state_indices, checkpoint_state_indices,
 * checkpoint_cu_starts, prefix_lens: all GDN_INDEX_I32 or all GDN_INDEX_I64,
 * each aligned to its element size; cu_seqlens stays int32).  With int64
 * entries a sequence whose read, final or checkpoint row lies outside
 * [-1, 2^31 - 1], or whose checkpoint start lies outside [0, 2^31 - 1], is
 * skipped (reads and writes nothing) and recorded as GDN_DEVERR_INDEX_RANGE
 * in err_word; the values are otherwise those of the int32 call. */
int gdn_chunk_gated_delta_rule_ex(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                  const float *g, const float *beta, gdn_bf16 *o,
                                  const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                  int32_t H, int32_t K, int32_t V, float scale,
                                  const void *initial_state, const void *state_indices,
                                  void *output_state, const void *output_state_indices,
                                  void *state_checkpoints, const void *checkpoint_state_indices,
                                  const void *checkpoint_cu_starts, const void *prefix_lens,
                                  int32_t checkpoint_every_n_tokens, int64_t pool_row_stride,
                                  int32_t state_dtype, int32_t index_dtype, void *workspace,
                                  size_t workspace_bytes, int32_t *err_word, void *stream);
int gdn_chunk_gated_delta_rule_paged_ex(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                        const float *g, const float *beta, gdn_bf16 *o,
                                        const int32_t *cu_seqlens, int32_t num_seqs,
                                        int32_t total_tokens, int32_t H, int32_t K, int32_t V,
                                        float scale, void *state_pool, int32_t state_dtype,
                                        int32_t num_pages, const int32_t *page_indices,
                                        const int32_t *page_indptr, int32_t page_size,
                                        const int32_t *last_page_len, const gdn_prefill_slots *slots,
                                        void *workspace, size_t workspace_bytes, int32_t *err_word,
                                        void *stream);
int gdn_gated_delta_rule_decode_paged_ex(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                         const float *g, const float *beta, gdn_bf16 *o,
                                         int32_t batch, int32_t H, int32_t K, int32_t V,
                                         float scale, void *state_pool, int32_t state_dtype,
                                         int32_t num_pages, const int32_t *page_indices,
                                         const int32_t *page_indptr, const int32_t *last_page_len,
                                         const gdn_decode_slots *slots, int32_t *err_word,
                                         void *stream);

/* gdn_pool_copy_rows -- "gdn-prefix-cache", §The fix: a cached block's state
 * is kept in that block's page and moved as bit-exact row copies (the
 * request's row into the block after a step that ends on a block boundary,
 * the block back into the request's row before a step that starts from a
 * hit); on this library's pool the same move forks a shared page before a
 * sequence writes it (copy-on-write).  For i < n, row dst_rows[i] of pool
 * receives the row_bytes bytes of row src_rows[i], bit for bit (any element
 * type: fp32 or bf16 states, NaN payloads kept); a -1 on either side skips the
 * pair.  pool rows are pool_row_stride_bytes apart; row_bytes (a full row is
 * H * V * K * element size) and the stride are multiples of 16, pool is
 * 16-byte aligned, src_rows / dst_rows are int32 [n] on the device.  Rows
 * outside [0, num_rows) are skipped and, with err_word, reported as
 * GDN_DEVERR_PAGE_ID with the pair index.  Preconditions (unchecked): no row
 * is the destination of two pairs, and no destination row is the source of
 * another pair.  n <= 65535. */
int gdn_pool_copy_rows(void *pool, int64_t row_bytes, int64_t pool_row_stride_bytes,
                       const int32_t *src_rows, const int32_t *dst_rows, int32_t n, int32_t num_rows,
                       int32_t *err_word, void *stream);

/* gdn_pool_zero_rows -- "gdn-prefix-cache", §The fix: new blocks and rows are
 * zeroed, so that no non-finite value outlives the step that produced it.
 * For i < n, the row_bytes bytes of row rows[i] become zero bits (+0.0 in fp32
 * and bf16: the zero state); -1 skips.  Same layout, checks and limits as
 * gdn_pool_copy_rows. */
int gdn_pool_zero_rows(void *pool, int64_t row_bytes, int64_t pool_row_stride_bytes, const int32_t *rows,
                       int32_t n, int32_t num_rows, int32_t *err_word, void *stream);

/* Bytes of device workspace a prefill call over num_seqs sequences,
 * total_tokens new tokens and H heads needs (0 for invalid arguments).  The
 * prefill runs in two phases: a chunk-local phase computes, for every 64-token
 * chunk and head in parallel, T'' = (I + A)^-1 diag(beta) of the chunked delta
 * rule (A[t][j] = beta_t exp(G_t - G_j) k_t . k_j, j < t) and
 * -W = -T'' diag(exp(G)) K, and stores them as 64 x 64 and 64 x 128 fp16
 * tiles; the sequential state chain then reads them back.  The workspace holds
 * 16 bytes per chunk slot plus 16 (rounded up to 1 KB) and 24 KB per (chunk
 * slot, head), with
 * total_tokens / 64 + 2 num_seqs + 2 chunk slots. */
size_t gdn_prefill_workspace_bytes(int32_t num_seqs, int32_t total_tokens, int32_t H);

/* gdn_debug_set_wait_stall -- fault injection for tests of the bounded waits
 * (no counterpart in the method's API).  While enabled (enable != 0), the
 * state-chain kernel of every prefill call launched afterwards from this
 * process first waits on a barrier that nothing completes; the wait gives up
 * after about 1 ms, before the kernel has issued any copy or tensor-core
 * operation, and the kernel records GDN_DEVERR_TIMEOUT in err_word and
 * returns: the call writes no output and no pool row.  Disabled by default;
 * enable 0 disables it again.  Not for production use. */
void gdn_debug_set_wait_stall(int32_t enable);

/* Static text for a status code. */
const char *gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_PAGED_H */
