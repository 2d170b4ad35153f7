// Merge of the requests that the stream-K schedule cut across CTAs (the
// split-KV reduce inside one partition).  Each split left a normalised fp32
// output and its base-2 LSE in a workspace slot, and the request's first CTA
// recorded {first CTA, number of splits, its slot}; split k > 0 lives in slot
// 2 (first + k).  The merge is the LSE-weighted combine of those splits.
//
// One CTA per (virtual request, 4 heads), a warp per head (few registers,
// so that the whole grid is resident in one wave): each lane owns 16
// of the 512 value dims (64 contiguous bytes of every split's row), issues
// the loads of the first splits before the weights are known, reduces the
// split LSEs with shuffles (max, then the sum of 2^(lse_k - max)), and
// accumulates the remaining splits 2 at a time.
#include "common.cuh"
#include "splits.cuh"

namespace mla {

constexpr int kMergeWarps = 4;  // heads per CTA
constexpr int kMergeBatch = 2;  // splits whose loads are in flight together

__global__ void __launch_bounds__(kMergeWarps * 32, 7) split_merge_kernel(DecodeParams p, int grid) {
  // launched as a programmatic dependent of the decode kernel: wait until its
  // grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int v = blockIdx.x;
  const int b = v / p.head_groups, g = v % p.head_groups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = blockIdx.y * kMergeWarps + warp;  // head within the group
  const int group_heads = min(p.heads_per_group, p.heads - g * p.heads_per_group);
  if (hl >= group_heads) return;
  // both loads in flight together: the record is only current for a request
  // with tiles (an empty one keeps whatever an earlier call left)
  const int4 info = info_ptr(p)[v];
  if ((p.q_len > 1 ? request_tiles<true>(p, v) : request_tiles<false>(p, v)) == 0) return;
  const int ns = info.y;
  // split k > 0 lives in slot 2 (first + k): never past the 2 x grid slots
  if (ns <= 1 || info.x < 0 || info.x + ns > grid) return;
  const float *sl = slot_lse_ptr(p);
  const float *so = slot_out_ptr(p);
  auto slot_of_split = [&](int k) { return k == 0 ? info.z : 2 * (info.x + k); };
  auto part = [&](int k, int i) {  // float4 i (0..3) of this lane's 16 dims in split k
    return reinterpret_cast<const float4 *>(so + (size_t(slot_of_split(k)) * kSlotHeads + hl) * kDv)
        [4 * lane + i];
  };
  auto lse_of = [&](int k) { return sl[slot_of_split(k) * kSlotHeads + hl]; };

  float4 x[kMergeBatch][4];
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u)
#pragma unroll
    for (int i = 0; i < 4; ++i) x[u][i] = u < ns ? part(u, i) : make_float4(0.f, 0.f, 0.f, 0.f);

  float mx = -INFINITY;
  for (int k = lane; k < ns; k += 32) mx = fmaxf(mx, lse_of(k));
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  // a query row that sees no token in any split (several query tokens per
  // request) has mx = -inf: every weight is then 0 and the row the neutral pair
  const float mref = mx == -INFINITY ? 0.f : mx;
  float sum = 0.f;
  for (int k = lane; k < ns; k += 32) sum += exp2f(lse_of(k) - mref);
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < ns; k0 += kMergeBatch) {
    if (k0 > 0) {
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          x[u][i] = k0 + u < ns ? part(k0 + u, i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float w = k0 + u < ns ? exp2f(lse_of(k0 + u) - mref) : 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i].x += w * x[u][i].x; acc[i].y += w * x[u][i].y;
        acc[i].z += w * x[u][i].z; acc[i].w += w * x[u][i].w;
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
    pk[2 * i] = *reinterpret_cast<uint32_t *>(&lo);
    pk[2 * i + 1] = *reinterpret_cast<uint32_t *>(&hi);
  }
  const size_t row = size_t(b) * p.heads + size_t(g) * p.heads_per_group + hl;
  uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kDv + 16 * lane);
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  if (lane == 0) p.lse[row] = sum > 0.f ? lse_out(p, mref + log2f(sum)) : -INFINITY;
}

cudaError_t launch_split_merge(const DecodeParams &p, int grid, cudaStream_t stream) {
  const int V = p.batch * p.head_groups;
  if (V == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(V, (p.heads_per_group + kMergeWarps - 1) / kMergeWarps);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_merge_kernel, p, grid);
}

}  // namespace mla
