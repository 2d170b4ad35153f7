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

// One warp merges row hl of request v, which the schedule split into
// info.y >= 2 pieces (info = the record its first CTA left): the
// LSE-weighted combine of the splits' normalised fp32 partials.  Returns this
// lane's 16 output dims as bf16 pairs and the row's base-2 LSE (-inf for a
// row that no split saw).
__device__ __forceinline__ void merge_split_row(const DecodeParams &p, int4 info, int hl,
                                                uint32_t (&pk)[8], float *lse2) {
  const int lane = threadIdx.x & 31;
  const int ns = info.y;
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
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
    pk[2 * i] = *reinterpret_cast<uint32_t *>(&lo);
    pk[2 * i + 1] = *reinterpret_cast<uint32_t *>(&hi);
  }
  *lse2 = sum > 0.f ? mref + log2f(sum) : -INFINITY;
}

__device__ __forceinline__ void store_row(__nv_bfloat16 *row, const uint32_t (&pk)[8]) {
  uint4 *dst = reinterpret_cast<uint4 *>(row + 16 * (threadIdx.x & 31));
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

// The decode rewrote every record this call (requests with no owned token
// get {-1, 0, 0}); split k > 0 lives in slot 2 (first + k): never past the
// 2 x grid slots.
__device__ __forceinline__ bool is_split(int4 info, int grid) {
  return info.y > 1 && info.x >= 0 && info.x + info.y <= grid;
}

__global__ void __launch_bounds__(kMergeWarps * 32, 7) split_merge_kernel(DecodeParams p, int grid) {
  // launched as a programmatic dependent of the decode kernel: wait until its
  // grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int v = blockIdx.x;
  const int b = vreq_row(p, v), g = vreq_group(p, v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = blockIdx.y * kMergeWarps + warp;  // head within the group
  const int group_heads = min(p.heads_per_group, p.heads - g * p.heads_per_group);
  if (hl >= group_heads) return;
  const int4 info = info_ptr(p)[v];
  if (!is_split(info, grid)) return;
  uint32_t pk[8];
  float lse2;
  merge_split_row(p, info, hl, pk, &lse2);
  const size_t row = size_t(b) * p.heads + size_t(g) * p.heads_per_group + hl;
  store_row(p.out + row * kDv, pk);
  if (lane == 0) p.lse[row] = lse2 > -INFINITY ? lse_out(p, lse2) : -INFINITY;
}

// All partitions in one call (the decode ran them in one launch): one CTA
// per (request, row), warp q for partition q.  Warp q completes partition
// q's row -- the split merge when the decode's schedule cut that partition
// of the request across CTAs, else it reads back what the decode wrote --
// and leaves the bf16 row and its base-2 LSE in shared memory; then the CTA
// merges the P partitions with the LSE rule into comb_out / comb_lse: the
// LSE combine (the rank merge of the pages' DCP) fused into the split merge.
constexpr int kDcpMaxParts = 8;

__global__ void __launch_bounds__(kDcpMaxParts * 32) dcp_merge_combine_kernel(DecodeParams p,
                                                                              int grid) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ alignas(16) uint32_t s_val[kDcpMaxParts][kDv / 2];  // bf16 pairs
  __shared__ float s_lse[kDcpMaxParts];
  const int P = p.num_parts, rows = p.heads;
  const int b = blockIdx.x / rows, r = blockIdx.x - b * rows;
  const int g = r / p.heads_per_group, hl = r - g * p.heads_per_group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    const int bv = warp * p.req_batch + b;  // partition `warp` of request b
    const int v = vreq_index(p, bv, g);
    const size_t prow = size_t(bv) * rows + r;
    uint32_t pk[8];
    float l;  // the partition's lse as returned (in the output base)
    const int4 info = info_ptr(p)[v];
    if (is_split(info, grid)) {
      float lse2;
      merge_split_row(p, info, hl, pk, &lse2);
      store_row(p.out + prow * kDv, pk);
      l = lse2 > -INFINITY ? lse_out(p, lse2) : -INFINITY;
      if (lane == 0) p.lse[prow] = l;
    } else {  // written by the decode (the neutral pair if it owned nothing)
      const uint4 *src = reinterpret_cast<const uint4 *>(p.out + prow * kDv + 16 * lane);
      const uint4 a = src[0], c = src[1];
      pk[0] = a.x; pk[1] = a.y; pk[2] = a.z; pk[3] = a.w;
      pk[4] = c.x; pk[5] = c.y; pk[6] = c.z; pk[7] = c.w;
      l = p.lse[prow];
    }
    uint4 *dst = reinterpret_cast<uint4 *>(&s_val[warp][8 * lane]);
    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    if (lane == 0) s_lse[warp] = l;
  }
  __syncthreads();
  // The combine of the returned partials and lses, with the arithmetic of
  // lse_combine_kernel (same expressions, same shuffle tree for the sum), so
  // that the result equals mla_lse_combine's bit for bit.
  const float to2 = p.lse_base2 ? 1.f : kLog2e;
  float mx = -INFINITY;
  for (int q = 0; q < P; ++q) mx = fmaxf(mx, s_lse[q] * to2);
  const size_t orow = size_t(b) * rows + r;
  uint4 *dst = reinterpret_cast<uint4 *>(p.comb_out + orow * kDv);
  constexpr int kChunks = kDv / 8;  // 16-byte chunks of a row
  if (mx == -INFINITY) {  // no partition owned a token of this row: the neutral pair
    for (int c = threadIdx.x; c < kChunks; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    if (p.comb_lse && threadIdx.x == 0) p.comb_lse[orow] = -INFINITY;
    return;
  }
  float w[kDcpMaxParts];
#pragma unroll
  for (int q = 0; q < kDcpMaxParts; ++q) w[q] = q < P ? exp2f(s_lse[q] * to2 - mx) : 0.f;
  const int lane_q = threadIdx.x & 31;
  float sum = lane_q < P ? exp2f(s_lse[lane_q] * to2 - mx) : 0.f;
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.f / sum;
  for (int c = threadIdx.x; c < kChunks; c += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < kDcpMaxParts; ++q) {
      if (w[q] == 0.f) continue;
      const uint4 u = reinterpret_cast<const uint4 *>(s_val[q])[c];
      const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w[q], __uint_as_float(x[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w[q], __uint_as_float(x[i] & 0xffff0000u), acc[2 * i + 1]);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 t2 = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
      o[i] = *reinterpret_cast<uint32_t *>(&t2);
    }
    dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (p.comb_lse && threadIdx.x == 0) {
    const float l2 = mx + log2f(sum);
    p.comb_lse[orow] = p.lse_base2 ? l2 : l2 * kLn2;
  }
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

// The fused-mode merge: split merge and LSE combine in one launch
// (num_parts <= 8), a programmatic dependent of the decode kernel.
cudaError_t launch_dcp_merge_combine(const DecodeParams &p, int grid, cudaStream_t stream) {
  const long long ctas = (long long)p.req_batch * p.heads;
  if (ctas == 0) return cudaSuccess;
  if (p.num_parts < 1 || p.num_parts > kDcpMaxParts || ctas > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ctas));
  cfg.blockDim = dim3(32 * p.num_parts);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dcp_merge_combine_kernel, p, grid);
}

}  // namespace mla
