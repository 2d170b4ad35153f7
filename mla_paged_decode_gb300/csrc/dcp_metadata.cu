// A DCP rank's per-step decode metadata, built on the device into buffers the
// caller keeps at fixed addresses (sglang pull 33926,
// _apply_dcp_cuda_graph_metadata): global lengths (+ the draft tokens of a
// target-verify step), the rank-local lengths under the round-robin owner
// rule, and the rank-local page table over the rank's compact pool (local
// page i of a request = the pool page of its local token 64 i).  A page table
// can only describe a pool that holds each request's local tokens in whole
// pages, so a slot of local token 64 i that is negative or not the first slot
// of a page pads that page and sets the error word.
//
// A warp per request: lane 0 writes the lengths, the lanes fill the table row.
#include "common.cuh"

namespace mla {

constexpr int kMetaWarps = 4;

__global__ void __launch_bounds__(kMetaWarps * 32)
    dcp_metadata_kernel(const int32_t *__restrict__ seq_lens,
                        const int32_t *__restrict__ req_pool_indices,
                        const int32_t *__restrict__ req_to_token, int batch, int r2t_rows,
                        int r2t_width, int extra, int part_id, int num_parts,
                        int32_t *global_lens, int32_t *local_lens, int32_t *table, int max_pages,
                        int32_t pad, int32_t *error_word) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kMetaWarps + warp;
  if (b >= batch) return;
  const int L = seq_lens[b] + extra;
  const int n = L < 0 ? 0 : local_len(L, num_parts, part_id);
  if (lane == 0) {
    global_lens[b] = L;
    local_lens[b] = n;
  }
  const int npages = (n + kPage - 1) / kPage;
  const int req = req_pool_indices[b];
  const bool ok = L >= 0 && req >= 0 && req < r2t_rows && npages <= max_pages &&
                  (npages == 0 || (long long)(npages - 1) * kPage < r2t_width);
  bool neg = false;
  for (int i = lane; i < max_pages; i += 32) {
    int32_t v = pad;
    if (ok && i < npages) {
      const int32_t slot = req_to_token[size_t(req) * r2t_width + size_t(i) * kPage];
      if (slot < 0 || slot % kPage != 0)
        neg = true;
      else
        v = slot / kPage;
    }
    table[size_t(b) * max_pages + i] = v;
  }
  neg = __any_sync(0xffffffffu, neg);
  if (lane == 0 && (!ok || neg) && error_word) atomicOr(error_word, 1);
}

cudaError_t launch_dcp_metadata(const int32_t *seq_lens, const int32_t *req_pool_indices,
                                const int32_t *req_to_token, int batch, int r2t_rows,
                                int r2t_width, int extra, int part_id, int num_parts,
                                int32_t *global_lens, int32_t *local_lens, int32_t *table,
                                int max_pages, int32_t pad, int32_t *error_word,
                                cudaStream_t stream) {
  const int grid = (batch + kMetaWarps - 1) / kMetaWarps;
  dcp_metadata_kernel<<<grid, kMetaWarps * 32, 0, stream>>>(
      seq_lens, req_pool_indices, req_to_token, batch, r2t_rows, r2t_width, extra, part_id,
      num_parts, global_lens, local_lens, table, max_pages, pad, error_word);
  return cudaGetLastError();
}

}  // namespace mla
