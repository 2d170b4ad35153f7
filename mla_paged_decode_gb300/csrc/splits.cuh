// Split bookkeeping shared by the decode kernels: request walk, neutral outputs
// for requests a partition does not touch, split tickets and the split merge.
#pragma once

#include "common.cuh"

namespace mla {

struct SplitInfo {
  int nsplits;   // CTAs whose tile range meets the request
  int c_first;   // first of them
  int slot;      // this CTA's slot for the request
};

__device__ __forceinline__ SplitInfo split_info(const CtaRange &r, int v, long long pv,
                                                int tiles) {
  SplitInfo s;
  s.c_first = sched_owner(pv, r.total, r.g_eff);
  int c_last = sched_owner(pv + tiles - 1, r.total, r.g_eff);
  s.nsplits = c_last - s.c_first + 1;
  s.slot = 2 * int(blockIdx.x) + (v != r.v_begin ? 1 : 0);
  return s;
}

__device__ __forceinline__ float *slot_lse_ptr(const DecodeParams &p) {
  return reinterpret_cast<float *>(p.ws + p.wl.slot_lse);
}
__device__ __forceinline__ float *slot_out_ptr(const DecodeParams &p) {
  return reinterpret_cast<float *>(p.ws + p.wl.slot_out);
}
__device__ __forceinline__ int4 *info_ptr(const DecodeParams &p) {
  return reinterpret_cast<int4 *>(p.ws + p.wl.info);
}
__device__ __forceinline__ int *error_word(const DecodeParams &p) {
  return reinterpret_cast<int *>(p.ws);
}

__device__ __forceinline__ float lse_out(const DecodeParams &p, float lse2) {
  return p.lse_base2 ? lse2 : lse2 * kLn2;
}

// The neutral pair (0, -inf) for every virtual request with no owned token,
// and its split record {-1, 0, 0} (no splits), so that every record is
// rewritten by each call and the merge reads no lengths.  Virtual request v
// is handled by CTA v mod gridDim.x.  Block-wide.
template <int MULTI = 0>
__device__ inline void write_empty_requests(const DecodeParams &p) {
  const int V = p.batch * p.head_groups;
  int *err = error_word(p);
  for (int v = blockIdx.x; v < V; v += gridDim.x) {
    int b = vreq_row(p, v), g = vreq_group(p, v);  // b: output row
    if (request_len<MULTI>(p, v, threadIdx.x == 0 ? err : nullptr) != 0) continue;
    if (threadIdx.x == 0) info_ptr(p)[v] = make_int4(-1, 0, 0, 0);
    int h0 = g * p.heads_per_group;
    int hn = min(p.heads_per_group, p.heads - h0);
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (size_t(b) * p.heads + h0) * kDv);
    for (int i = threadIdx.x; i < hn * kDv / 8; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < hn; i += blockDim.x)
      p.lse[size_t(b) * p.heads + h0 + i] = -INFINITY;
  }
}

// Called (by one thread) in each CTA that worked on request v: the CTA that
// holds the request's first tile records where its splits are, for the merge
// kernel.  Every request with owned tokens gets a fresh record each call
// (and every other one the empty record of write_empty_requests).
__device__ __forceinline__ void record_split(const DecodeParams &p, int v, const SplitInfo &si) {
  if (int(blockIdx.x) == si.c_first) info_ptr(p)[v] = make_int4(si.c_first, si.nsplits, si.slot, 0);
}

}  // namespace mla
