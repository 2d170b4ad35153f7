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

// Slot CTA c used for request v (which starts at tile pv).
__device__ __forceinline__ int slot_of(const CtaRange &r, int c, int c_first, long long pv) {
  return 2 * c + ((c == c_first && sched_start(c, r.total, r.g_eff) < pv) ? 1 : 0);
}

__device__ __forceinline__ float *slot_lse_ptr(const DecodeParams &p) {
  return reinterpret_cast<float *>(p.ws + p.wl.slot_lse);
}
__device__ __forceinline__ float *slot_out_ptr(const DecodeParams &p) {
  return reinterpret_cast<float *>(p.ws + p.wl.slot_out);
}
__device__ __forceinline__ int *counters_ptr(const DecodeParams &p) {
  return reinterpret_cast<int *>(p.ws + p.wl.counters);
}
__device__ __forceinline__ int *error_word(const DecodeParams &p) {
  return reinterpret_cast<int *>(p.ws);
}

__device__ __forceinline__ float lse_out(const DecodeParams &p, float lse2) {
  return p.lse_base2 ? lse2 : lse2 * kLn2;
}

// The neutral pair (0, -inf) for every virtual request with no owned token.
// Virtual request v is handled by CTA v mod gridDim.x.  Block-wide.
__device__ inline void write_empty_requests(const DecodeParams &p) {
  const int V = p.batch * p.head_groups;
  int *err = error_word(p);
  for (int v = blockIdx.x; v < V; v += gridDim.x) {
    int b = v / p.head_groups, g = v % p.head_groups;
    int L = checked_len(p, b, threadIdx.x == 0 ? err : nullptr);
    if (local_len(L, p.num_parts, p.part_id) != 0) continue;
    int h0 = g * p.heads_per_group;
    int hn = min(p.heads_per_group, p.heads - h0);
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (size_t(b) * p.heads + h0) * kDv);
    for (int i = threadIdx.x; i < hn * kDv / 8; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < hn; i += blockDim.x)
      p.lse[size_t(b) * p.heads + h0 + i] = -INFINITY;
  }
}

// Barrier of every thread of the CTA.
struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Named barrier of `count` threads (a warpgroup that runs the epilogue while
// other warps of the CTA do something else).
struct GroupSync {
  uint32_t id, count;
  __device__ __forceinline__ void operator()() const {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
  }
};

// Called by the `sync` group after this CTA's slot for request v is written
// (`rank` = the caller's index in the group).  Returns true in the CTA that
// completes the request: it must merge.
template <class Sync>
__device__ inline bool split_ticket(const DecodeParams &p, int v, int nsplits, int *s_flag,
                                    int rank, Sync sync) {
  __threadfence();
  sync();
  if (rank == 0) {
    int prev = atomicAdd(counters_ptr(p) + v, 1);
    *s_flag = (prev == nsplits - 1);
  }
  sync();
  bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

// Merge the nsplits slots of request v into out/lse, by the `sync` group of
// `nthreads` threads (`rank` = the caller's index); uses s_m / s_inv
// (kSlotHeads floats each) of shared memory.  Resets the ticket.
template <class Sync>
__device__ inline void merge_splits(const DecodeParams &p, const CtaRange &r, int v, long long pv,
                                    const SplitInfo &si, float *s_m, float *s_inv, int rank,
                                    int nthreads, Sync sync) {
  const int b = v / p.head_groups, g = v % p.head_groups;
  const int h0 = g * p.heads_per_group;
  const int hn = min(p.heads_per_group, p.heads - h0);
  const float *sl = slot_lse_ptr(p);
  const float *so = slot_out_ptr(p);
  for (int h = rank; h < hn; h += nthreads) {
    float mx = -INFINITY;
    for (int k = 0; k < si.nsplits; ++k) {
      int slot = slot_of(r, si.c_first + k, si.c_first, pv);
      mx = fmaxf(mx, __ldcg(sl + slot * kSlotHeads + h));
    }
    float sum = 0.f;
    for (int k = 0; k < si.nsplits; ++k) {
      int slot = slot_of(r, si.c_first + k, si.c_first, pv);
      sum += exp2f(__ldcg(sl + slot * kSlotHeads + h) - mx);
    }
    s_m[h] = mx;
    s_inv[h] = 1.f / sum;
    p.lse[size_t(b) * p.heads + h0 + h] = lse_out(p, mx + log2f(sum));
  }
  sync();
  for (int i = rank; i < hn * (kDv / 4); i += nthreads) {
    int h = i / (kDv / 4), d4 = i % (kDv / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < si.nsplits; ++k) {
      int slot = slot_of(r, si.c_first + k, si.c_first, pv);
      float w = exp2f(__ldcg(sl + slot * kSlotHeads + h) - s_m[h]);
      float4 x = __ldcg(reinterpret_cast<const float4 *>(so + (size_t(slot) * kSlotHeads + h) * kDv) + d4);
      acc.x += w * x.x; acc.y += w * x.y; acc.z += w * x.z; acc.w += w * x.w;
    }
    float inv = s_inv[h];
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(p.out + (size_t(b) * p.heads + h0 + h) * kDv)[d4] = pk;
  }
  if (rank == 0) counters_ptr(p)[v] = 0;
  sync();
}

}  // namespace mla
