// The write side of the paged latent cache: each request's new token row
// goes to physical page block_table[b][t / 64], row t % 64, on the partition
// that owns token t (sglang pull 33926, implementation steps 3 and 4: the
// FP8 cache stores the quantised latent with one per-tensor scale; under DCP
// each rank's pool writes only its own rows).
//
// A warp per request.  bf16: 72 chunks of 16 B copied.  e4m3: 36 chunks of
// 16 values, each value fp32(x) / kv_scale (IEEE division) converted by the
// hardware round-to-nearest-even, saturating e4m3 conversion.
#include "common.cuh"

namespace mla {

constexpr int kAppendWarps = 4;
constexpr int kErrAppendBadPage = 1;

// Two fp32 values -> two e4m3 codes (lo in the low byte), nearest even,
// saturated to +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_kernel(const __nv_bfloat16 *__restrict__ kv_new, unsigned char *kv_pages,
                     const int32_t *__restrict__ block_table, const int32_t *__restrict__ positions,
                     int batch, int part_id, int num_parts, int num_pages, int max_pages, int e4m3,
                     float kv_scale, int32_t *error_word) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kAppendWarps + warp;
  if (b >= batch) return;
  const int t = positions[b];
  if (t < 0 || t % num_parts != part_id) return;
  const int lp = t / kPage;
  const int pg = lp < max_pages ? block_table[size_t(b) * max_pages + lp] : -1;
  if (pg < 0 || pg >= num_pages) {
    if (lane == 0 && error_word) atomicOr(error_word, kErrAppendBadPage);
    return;
  }
  const size_t row = size_t(pg) * kPage + size_t(t % kPage);
  const uint4 *src = reinterpret_cast<const uint4 *>(kv_new + size_t(b) * kDqk);  // 72 x 8 values
  if (!e4m3) {
    uint4 *dst = reinterpret_cast<uint4 *>(kv_pages + row * (kDqk * 2));
    for (int i = lane; i < kDqk / 8; i += 32) dst[i] = src[i];
    return;
  }
  uint4 *dst = reinterpret_cast<uint4 *>(kv_pages + row * kDqk);  // 36 x 16 codes
  for (int i = lane; i < kDqk / 16; i += 32) {
    const uint4 a = src[2 * i], c = src[2 * i + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        v[2 * e] = __uint_as_float(w[2 * k + e] << 16) / kv_scale;
        v[2 * e + 1] = __uint_as_float(w[2 * k + e] & 0xffff0000u) / kv_scale;
      }
      o[k] = uint32_t(f32x2_to_e4m3x2(v[0], v[1])) | (uint32_t(f32x2_to_e4m3x2(v[2], v[3])) << 16);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_kv_append(const void *kv_new, void *kv_pages, const int32_t *block_table,
                             const int32_t *positions, int batch, int part_id, int num_parts,
                             int num_pages, int max_pages, int e4m3, float kv_scale,
                             int32_t *error_word, cudaStream_t stream) {
  const int grid = (batch + kAppendWarps - 1) / kAppendWarps;
  kv_append_kernel<<<grid, kAppendWarps * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(kv_new), static_cast<unsigned char *>(kv_pages),
      block_table, positions, batch, part_id, num_parts, num_pages, max_pages, e4m3, kv_scale,
      error_word);
  return cudaGetLastError();
}

}  // namespace mla
