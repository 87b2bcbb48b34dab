// slots.cu -- pool rows of a paged prefill / decode batch, derived on the
// device in one launch with no host synchronisation.
//
// "flashinfer.gdn_paged": gdn_paged_prefill_slots / gdn_paged_decode_slots,
// §Page table (sequence b owns page_indices[page_indptr[b]:page_indptr[b+1]]
// and holds (n_b - 1) * page_size + last_page_len[b] tokens after the call),
// the prefill bullets (read the page of the last prefix token, store at every
// crossed boundary and the final state to the last page) and the decode
// paragraph (last_page_len == 1: read the previous page).
#include "common.cuh"

namespace {

__global__ void prefill_slots_kernel(const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ indptr,
                                     const int32_t* __restrict__ pages, const int32_t* __restrict__ last_len,
                                     int32_t num_seqs, int32_t page_size, int32_t* __restrict__ state_indices,
                                     int32_t* __restrict__ output_state_indices,
                                     int32_t* __restrict__ checkpoint_cu_starts, int32_t* __restrict__ prefix_lens) {
  gdn::pdl_wait();
  gdn::pdl_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= num_seqs) return;
  const int32_t i0 = indptr[b], i1 = indptr[b + 1];
  const int64_t n = static_cast<int64_t>(i1) - i0;
  const int64_t len = static_cast<int64_t>(cu_seqlens[b + 1]) - cu_seqlens[b];
  const int32_t lpl = last_len[b];
  const int64_t total = (n - 1) * page_size + lpl;
  const int64_t prefix = total - len;
  // Not a valid sequence (no page, a last page holding no token or more than a
  // page, more new tokens than tokens, or more tokens than the prefill kernels
  // address): nothing to read or write, the same sequences the prefill kernels
  // skip when they derive the rows themselves.
  if (n < 1 || lpl < 1 || lpl > page_size || prefix < 0 || len < 0 || total > 0x3FFFFFFF) {
    state_indices[b] = -1;
    output_state_indices[b] = -1;
    checkpoint_cu_starts[b] = i0;
    prefix_lens[b] = 0;
    return;
  }
  state_indices[b] = prefix > 0 ? pages[i0 + (prefix - 1) / page_size] : -1;
  output_state_indices[b] = len > 0 ? pages[i1 - 1] : -1;
  checkpoint_cu_starts[b] = static_cast<int32_t>(i0 + prefix / page_size);
  prefix_lens[b] = static_cast<int32_t>(prefix);
}

__global__ void decode_slots_kernel(const int32_t* __restrict__ indptr, const int32_t* __restrict__ pages,
                                    const int32_t* __restrict__ last_len, int32_t batch,
                                    int32_t* __restrict__ initial_state_indices,
                                    int32_t* __restrict__ output_state_indices) {
  gdn::pdl_wait();
  gdn::pdl_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int32_t i0 = indptr[b], i1 = indptr[b + 1];
  if (i1 - i0 < 1) {
    initial_state_indices[b] = -1;
    output_state_indices[b] = -1;
    return;
  }
  const int32_t last = pages[i1 - 1];
  output_state_indices[b] = last;
  if (last_len[b] == 1)
    initial_state_indices[b] = (i1 - i0 >= 2) ? pages[i1 - 2] : -1;
  else
    initial_state_indices[b] = last;
}

}  // namespace

extern "C" int gdn_paged_prefill_slots(const int32_t* cu_seqlens, const int32_t* page_indptr,
                                       const int32_t* page_indices, const int32_t* last_page_len,
                                       int32_t num_seqs, int32_t page_size, int32_t* state_indices,
                                       int32_t* output_state_indices, int32_t* checkpoint_cu_starts,
                                       int32_t* prefix_lens, void* stream) {
  if (num_seqs < 0 || page_size <= 0 || page_size % gdn::kChunk != 0) return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return GDN_OK;
  if (!cu_seqlens || !page_indptr || !page_indices || !last_page_len || !state_indices ||
      !output_state_indices || !checkpoint_cu_starts || !prefix_lens)
    return GDN_ERR_INVALID_ARGUMENT;
  const int threads = 128;
  return gdn_host::launch_pdl(prefill_slots_kernel, dim3((num_seqs + threads - 1) / threads), dim3(threads), 0,
                              static_cast<cudaStream_t>(stream), cu_seqlens, page_indptr, page_indices,
                              last_page_len, num_seqs, page_size, state_indices, output_state_indices,
                              checkpoint_cu_starts, prefix_lens);
}

extern "C" int gdn_paged_decode_slots(const int32_t* page_indptr, const int32_t* page_indices,
                                      const int32_t* last_page_len, int32_t batch,
                                      int32_t* initial_state_indices, int32_t* output_state_indices,
                                      void* stream) {
  if (batch < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (batch == 0) return GDN_OK;
  if (!page_indptr || !page_indices || !last_page_len || !initial_state_indices || !output_state_indices)
    return GDN_ERR_INVALID_ARGUMENT;
  const int threads = 128;
  return gdn_host::launch_pdl(decode_slots_kernel, dim3((batch + threads - 1) / threads), dim3(threads), 0,
                              static_cast<cudaStream_t>(stream), page_indptr, page_indices, last_page_len, batch,
                              initial_state_indices, output_state_indices);
}
