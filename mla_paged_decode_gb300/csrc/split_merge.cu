// Merge of the requests that the stream-K schedule cut across CTAs (the
// split-KV reduce inside one partition).  Each split left a normalised fp32
// output and its base-2 LSE in a workspace slot, and the request's first CTA
// recorded {first CTA, number of splits, its slot}; split k > 0 lives in slot
// 2 (first + k).  The merge is the LSE-weighted combine of those splits.
//
// One CTA per (virtual request, 2 heads): a warp per head reduces the split
// LSEs (max, then the weights 2^(lse_k - max) kept in shared memory), then
// each thread owns 4 of the 512 value dims and keeps the loads of 4 splits x 2
// heads in flight before accumulating.
#include "common.cuh"
#include "splits.cuh"

namespace mla {

constexpr int kMergeThreads = 128;  // x 4 dims = 512
constexpr int kMergeHeads = 2;      // heads per CTA
constexpr int kMergeBatch = 4;      // splits whose loads are in flight together

__global__ void __launch_bounds__(kMergeThreads)
    split_merge_kernel(DecodeParams p, int max_splits) {
  extern __shared__ float s_w[];  // [max_splits][kMergeHeads] weights, then [kMergeHeads] 1/sum
  // launched as a programmatic dependent of the decode kernel: wait until its
  // grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int v = blockIdx.x;
  const int b = v / p.head_groups, g = v % p.head_groups;
  const int h_first = blockIdx.y * kMergeHeads;  // within the head group
  const int group_heads = min(p.heads_per_group, p.heads - g * p.heads_per_group);
  if (h_first >= group_heads) return;
  const int hn = min(kMergeHeads, group_heads - h_first);
  if (request_tiles(p, v) == 0) return;
  const int4 info = info_ptr(p)[v];
  const int ns = info.y;
  if (ns <= 1 || ns > max_splits) return;
  const float *sl = slot_lse_ptr(p);
  const float *so = slot_out_ptr(p);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *inv = s_w + max_splits * kMergeHeads;
  const size_t row0 = size_t(b) * p.heads + size_t(g) * p.heads_per_group + h_first;
  auto slot_of_split = [&](int k) { return k == 0 ? info.z : 2 * (info.x + k); };

  if (warp < hn) {  // warp hh: weights of head hh over the splits
    const int hh = warp;
    float mx = -INFINITY;
    for (int k = lane; k < ns; k += 32) mx = fmaxf(mx, sl[slot_of_split(k) * kSlotHeads + h_first + hh]);
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int k = lane; k < ns; k += 32) {
      const float w = exp2f(sl[slot_of_split(k) * kSlotHeads + h_first + hh] - mx);
      s_w[k * kMergeHeads + hh] = w;
      sum += w;
    }
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      inv[hh] = 1.f / sum;
      p.lse[row0 + hh] = lse_out(p, mx + log2f(sum));
    }
  }
  __syncthreads();

  const int d4 = threadIdx.x;  // value dims 4 d4 .. 4 d4 + 3
  float4 acc[kMergeHeads];
#pragma unroll
  for (int hh = 0; hh < kMergeHeads; ++hh) acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < ns; k0 += kMergeBatch) {
    float4 x[kMergeBatch][kMergeHeads];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int k = k0 + u;
      const float4 *src = reinterpret_cast<const float4 *>(
          so + size_t(k < ns ? slot_of_split(k) : 0) * kSlotHeads * kDv);
#pragma unroll
      for (int hh = 0; hh < kMergeHeads; ++hh)
        x[u][hh] = (k < ns && hh < hn) ? src[size_t(h_first + hh) * (kDv / 4) + d4]
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u)
#pragma unroll
      for (int hh = 0; hh < kMergeHeads; ++hh) {
        const float w = (k0 + u < ns) ? s_w[(k0 + u) * kMergeHeads + hh] : 0.f;
        acc[hh].x += w * x[u][hh].x; acc[hh].y += w * x[u][hh].y;
        acc[hh].z += w * x[u][hh].z; acc[hh].w += w * x[u][hh].w;
      }
  }
#pragma unroll
  for (int hh = 0; hh < kMergeHeads; ++hh) {
    if (hh >= hn) break;
    const float sc = inv[hh];
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[hh].x * sc, acc[hh].y * sc);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[hh].z * sc, acc[hh].w * sc);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(p.out + (row0 + hh) * kDv)[d4] = pk;
  }
}

cudaError_t launch_split_merge(const DecodeParams &p, int grid, cudaStream_t stream) {
  const int V = p.batch * p.head_groups;
  if (V == 0) return cudaSuccess;
  dim3 blocks(V, (p.heads_per_group + kMergeHeads - 1) / kMergeHeads);
  const size_t smem = sizeof(float) * (size_t(grid) * kMergeHeads + kMergeHeads);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = blocks;
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_merge_kernel, p, grid);
}

}  // namespace mla
