// LSE-weighted merge of P partial attention results (sglang pull 33364,
// "Modifications", kernel 4: the softmax reduction over all ranks' partials),
// with the LSE base converted at the merge site (sglang pull 33926, step 4).
//
// One warp per output row (token, head).  The row's P LSEs are reduced with
// warp shuffles in the base-2 domain, the weights kept in shared memory, and
// the D values streamed as 16-byte bf16 vectors; a partition whose weight is
// exactly zero (lse = -inf) is not read.  For up to 8 partitions and rows of
// up to 512 values every load of a lane is issued before the first is used
// (one memory round trip per row instead of one per partition and chunk);
// the arithmetic, and so every bit of the result, is the same either way.
#include "common.cuh"

namespace mla {

constexpr int kCombineWarps = 8;
constexpr int kCombineMaxParts = 256;
constexpr int kFastParts = 8;   // partitions whose loads a lane keeps in flight together
constexpr int kFastChunks = 2;  // 16-byte chunks per lane: rows of up to 512 values

__global__ void __launch_bounds__(kCombineWarps * 32)
lse_combine_kernel(const __nv_bfloat16 *__restrict__ partials, const float *__restrict__ lses,
                   int num_parts, __nv_bfloat16 *__restrict__ out, float *__restrict__ out_lse,
                   int rows, int dim, int base2) {
  extern __shared__ float s_w[];  // [kCombineWarps][num_parts]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kCombineWarps + warp;
  if (row >= rows) return;
  float *w = s_w + warp * num_parts;
  const float to2 = base2 ? 1.f : kLog2e;

  float mx = -INFINITY;
  for (int q = lane; q < num_parts; q += 32) mx = fmaxf(mx, lses[size_t(q) * rows + row] * to2);
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

  const int chunks = dim / 8;
  uint4 *dst = reinterpret_cast<uint4 *>(out + size_t(row) * dim);
  if (mx == -INFINITY) {  // every partition owned nothing: the neutral pair
    for (int c = lane; c < chunks; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
    if (out_lse && lane == 0) out_lse[row] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int q = lane; q < num_parts; q += 32) {
    float wq = exp2f(lses[size_t(q) * rows + row] * to2 - mx);
    w[q] = wq;
    sum += wq;
  }
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncwarp();
  const float inv = 1.f / sum;

  if (num_parts <= kFastParts && chunks <= kFastChunks * 32) {
    // this lane's chunks lane + 32 k of every partition with a weight
    uint4 u[kFastChunks][kFastParts];
#pragma unroll
    for (int k = 0; k < kFastChunks; ++k)
#pragma unroll
      for (int q = 0; q < kFastParts; ++q)
        if (lane + 32 * k < chunks && q < num_parts && w[q] != 0.f)
          u[k][q] = __ldg(reinterpret_cast<const uint4 *>(partials + (size_t(q) * rows + row) * dim) +
                          lane + 32 * k);
#pragma unroll
    for (int k = 0; k < kFastChunks; ++k) {
      const int c = lane + 32 * k;
      if (c >= chunks) continue;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kFastParts; ++q) {
        if (q >= num_parts) break;
        const float wq = w[q];
        if (wq == 0.f) continue;
        const uint32_t x[4] = {u[k][q].x, u[k][q].y, u[k][q].z, u[k][q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wq, __uint_as_float(x[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wq, __uint_as_float(x[i] & 0xffff0000u), acc[2 * i + 1]);
        }
      }
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 t2 = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
        pk[i] = *reinterpret_cast<uint32_t *>(&t2);
      }
      dst[c] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  } else for (int c = lane; c < chunks; c += 32) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < num_parts; ++q) {
      const float wq = w[q];
      if (wq == 0.f) continue;
      uint4 u = __ldg(reinterpret_cast<const uint4 *>(partials + (size_t(q) * rows + row) * dim) + c);
      const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wq, __uint_as_float(x[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wq, __uint_as_float(x[i] & 0xffff0000u), acc[2 * i + 1]);
      }
    }
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 t2 = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
      pk[i] = *reinterpret_cast<uint32_t *>(&t2);
    }
    dst[c] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  if (out_lse && lane == 0) {
    float l2 = mx + log2f(sum);
    out_lse[row] = base2 ? l2 : l2 * kLn2;
  }
}

int combine_max_parts() { return kCombineMaxParts; }

cudaError_t launch_lse_combine(const void *partials, const float *lses, int num_parts, void *out,
                               float *out_lse, int rows, int dim, int base2,
                               cudaStream_t stream) {
  const int blocks = (rows + kCombineWarps - 1) / kCombineWarps;
  const size_t smem = sizeof(float) * kCombineWarps * num_parts;
  lse_combine_kernel<<<blocks, kCombineWarps * 32, smem, stream>>>(
      static_cast<const __nv_bfloat16 *>(partials), lses, num_parts,
      static_cast<__nv_bfloat16 *>(out), out_lse, rows, dim, base2);
  return cudaGetLastError();
}

}  // namespace mla
