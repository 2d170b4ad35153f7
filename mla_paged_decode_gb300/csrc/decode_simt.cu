// CUDA-core decode kernel: the same split schedule, gather and finalise as the
// tensor-core kernel, with the two contractions on FP32 FMA units.  It serves
// head counts and partition counts the tensor-core kernel does not take.
#include "common.cuh"
#include "splits.cuh"

#include <cuda_fp16.h>

namespace mla {

constexpr int kSimtThreads = 256;
constexpr int kSimtHeads = 32;   // heads per virtual request
constexpr int kKvStride = 584;   // bf16 per shared row: 1168 B, 16-B aligned, bank-skewed

struct SimtSmem {
  float q[kSimtHeads][kDqk];
  __nv_bfloat16 kv[kTile][kKvStride];
  float prob[kSimtHeads][kTile];
  CtaRange range;
  long long scratch[kSimtThreads / 32 + 1];
};

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// 8 e4m3 bytes -> 8 bf16 (exact: every e4m3 value is a bf16 value)
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 raw) {
  uint32_t out[4];
  const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float2 f = e4m3x2_to_float2(uint16_t(w[i] >> (16 * k)));
      __nv_bfloat162 bb = __floats2bfloat162_rn(f.x, f.y);
      out[2 * i + k] = *reinterpret_cast<uint32_t *>(&bb);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(kSimtThreads, 1) decode_simt_kernel(DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem &s = *reinterpret_cast<SimtSmem *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int *err = error_word(p);

  write_empty_requests(p);
  cta_schedule(p, &s.range, s.scratch);
  const CtaRange r = s.range;
  if (r.start >= r.end) return;

  const int V = p.batch * p.head_groups;
  int v = r.v_begin;
  long long pv = r.p_begin;
  while (v < V && pv < r.end) {
    const int tiles = request_tiles(p, v);
    if (tiles == 0) { ++v; continue; }
    const long long t0 = max(r.start, pv) - pv, t1 = min(r.end, pv + tiles) - pv;
    const int b = vreq_row(p, v), g = vreq_group(p, v);
    const int n = local_len(checked_len(p, b, tid == 0 ? err : nullptr), p.num_parts, p.part_id);

    __syncthreads();  // previous request's shared reads are done
    for (int i = tid; i < kSimtHeads * kDqk; i += kSimtThreads) {
      int h = i / kDqk, d = i % kDqk, hg = g * kSimtHeads + h;
      s.q[h][d] = hg < p.heads
          ? __bfloat162float(p.q[(size_t(b) * p.heads + hg) * kDqk + d]) : 0.f;
    }

    float m[4], l[4], acc[4][16];
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      m[hh] = -INFINITY;
      l[hh] = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[hh][k] = 0.f;
    }

    for (long long tile = t0; tile < t1; ++tile) {
      const int j0 = int(tile) * kTile;
      const int nv = min(kTile, n - j0);
      __syncthreads();
      for (int i = tid; i < kTile * (kDqk / 8); i += kSimtThreads) {
        int row = i / (kDqk / 8), ch = i % (kDqk / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (row < nv) {
          long long t = p.part_id + (long long)(j0 + row) * p.num_parts;
          int lp = int(t / kPage), rr = int(t % kPage);
          int page = p.block_table[size_t(b) * p.max_pages + lp];
          if (page < 0 || page >= p.num_pages) {
            if (ch == 0) atomicOr(err, kErrBadPage);
          } else if (!p.kv_e4m3) {
            val = __ldg(reinterpret_cast<const uint4 *>(p.kv) +
                        ((size_t(page) * kPage + rr) * kDqk + ch * 8) / 8);
          } else {
            uint2 raw = __ldg(reinterpret_cast<const uint2 *>(p.kv) +
                              ((size_t(page) * kPage + rr) * kDqk + ch * 8) / 8);
            val = e4m3x8_to_bf16x8(raw);
          }
        }
        *reinterpret_cast<uint4 *>(&s.kv[row][ch * 8]) = val;
      }
      __syncthreads();

      // scores of heads 4*warp .. 4*warp+3 against tokens lane and lane+32
      float sc[4][2];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) sc[hh][0] = sc[hh][1] = 0.f;
      for (int d = 0; d < kDqk; d += 8) {
        float k0[8], k1[8];
        unpack8(*reinterpret_cast<const uint4 *>(&s.kv[lane][d]), k0);
        unpack8(*reinterpret_cast<const uint4 *>(&s.kv[lane + 32][d]), k1);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const float *qq = &s.q[4 * warp + hh][d];
          float4 qa = *reinterpret_cast<const float4 *>(qq);
          float4 qb = *reinterpret_cast<const float4 *>(qq + 4);
          const float qf[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            sc[hh][0] = fmaf(qf[e], k0[e], sc[hh][0]);
            sc[hh][1] = fmaf(qf[e], k1[e], sc[hh][1]);
          }
        }
      }
      const float xs = p.score_scale_log2 * p.kv_scale;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        float x0 = lane < nv ? sc[hh][0] * xs : -INFINITY;
        float x1 = lane + 32 < nv ? sc[hh][1] * xs : -INFINITY;
        float tmax = fmaxf(x0, x1);
        for (int o = 16; o; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
        float mn = fmaxf(m[hh], tmax);
        float alpha = exp2f(m[hh] - mn);
        float p0 = exp2f(x0 - mn), p1 = exp2f(x1 - mn);
        float ps = p0 + p1;
        for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l[hh] = l[hh] * alpha + ps;
        m[hh] = mn;
        s.prob[4 * warp + hh][lane] = p0;
        s.prob[4 * warp + hh][lane + 32] = p1;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[hh][k] *= alpha;
      }
      __syncwarp();
      for (int j = 0; j < nv; ++j) {
        float vf[16];
        unpack8(*reinterpret_cast<const uint4 *>(&s.kv[j][16 * lane]), vf);
        unpack8(*reinterpret_cast<const uint4 *>(&s.kv[j][16 * lane + 8]), vf + 8);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          float pr = s.prob[4 * warp + hh][j];
#pragma unroll
          for (int k = 0; k < 16; ++k) acc[hh][k] = fmaf(pr, vf[k], acc[hh][k]);
        }
      }
    }

    // finalise: the whole request here, or one split of it
    const SplitInfo si = split_info(r, v, pv, tiles);
    const bool split = si.nsplits > 1;
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const int hl = 4 * warp + hh, hg = g * kSimtHeads + hl;
      if (hg >= p.heads) continue;
      const float inv = p.kv_scale / l[hh];
      const float lse2 = m[hh] + log2f(l[hh]);
      if (!split) {
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          __nv_bfloat162 t2 = __floats2bfloat162_rn(acc[hh][2 * k] * inv, acc[hh][2 * k + 1] * inv);
          pk[k] = *reinterpret_cast<uint32_t *>(&t2);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + (size_t(b) * p.heads + hg) * kDv + 16 * lane);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        if (lane == 0) p.lse[size_t(b) * p.heads + hg] = lse_out(p, lse2);
      } else {
        float4 *dst = reinterpret_cast<float4 *>(slot_out_ptr(p) +
                                                 (size_t(si.slot) * kSlotHeads + hl) * kDv + 16 * lane);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_float4(acc[hh][4 * k] * inv, acc[hh][4 * k + 1] * inv,
                               acc[hh][4 * k + 2] * inv, acc[hh][4 * k + 3] * inv);
        if (lane == 0) slot_lse_ptr(p)[si.slot * kSlotHeads + hl] = lse2;
      }
    }
    if (tid == 0) record_split(p, v, si);
    pv += request_cost(tiles, kPieceCost);
    ++v;
  }
}

cudaError_t launch_split_merge(const DecodeParams &p, int grid, cudaStream_t stream);

cudaError_t launch_decode_simt(const DecodeParams &p, int grid, cudaStream_t stream) {
  static SmemLimitOnce smem_limit;
  cudaError_t e = smem_limit.ensure(decode_simt_kernel, int(sizeof(SimtSmem)));
  if (e != cudaSuccess) return e;
  decode_simt_kernel<<<grid, kSimtThreads, sizeof(SimtSmem), stream>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? launch_split_merge(p, grid, stream) : e;
}

}  // namespace mla
