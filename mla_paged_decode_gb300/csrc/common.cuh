// Shared definitions of the MLA paged-decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace mla {

constexpr int kDqk = 576;        // 512 latent + 64 rope
constexpr int kDv = 512;         // latent = value
constexpr int kPage = 64;        // tokens per cache page
constexpr int kTile = 64;        // partition-local tokens per KV tile
constexpr int kSlotHeads = 64;   // heads per split-partial slot in the workspace
// Schedule cost of a request piece's boundary (its Q, the pipeline refill,
// the epilogue), in tiles: an e4m3 piece also splits its Q into two terms,
// and its tiles are shorter, so its boundary weighs more tiles (each value
// the measured best of 4, 8 and 12 on that dtype's workloads).
constexpr int kPieceCost = 4;
constexpr int kPieceCostE4m3 = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device error word bits (workspace header).
constexpr int kErrBadPage = 1;
constexpr int kErrBadLen = 2;
constexpr int kErrTimeout = 4;   // a bounded wait inside the kernel gave up

// Workspace layout (all offsets multiples of 256 bytes):
//   [0, 256)                 header: int32 error word
//   info                     int4[num_virtual_requests]: {first CTA, splits, its slot}
//   slot lse                 fp32[2 * grid][kSlotHeads]   (base-2 lse of a split)
//   slot out                 fp32[2 * grid][kSlotHeads][512] (normalised split output)
struct WorkspaceLayout {
  size_t info, slot_lse, slot_out, total;
};

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ constexpr WorkspaceLayout workspace_layout(int num_virtual, int grid) {
  return WorkspaceLayout{
      256, align256(256 + 16 * size_t(num_virtual)),
      align256(align256(256 + 16 * size_t(num_virtual)) +
               sizeof(float) * size_t(2 * grid) * kSlotHeads),
      align256(align256(align256(256 + 16 * size_t(num_virtual)) +
                        sizeof(float) * size_t(2 * grid) * kSlotHeads) +
               sizeof(float) * size_t(2 * grid) * kSlotHeads * kDv)};
}

struct DecodeParams {
  const __nv_bfloat16 *q;     // [B, 1, H, 576]
  const void *kv;             // [num_pages, 64, 576] bf16 or e4m3
  const int32_t *block_table; // [B, max_pages]
  const int32_t *seq_lens;    // [B]
  __nv_bfloat16 *out;         // [B, 1, H, 512]
  float *lse;                 // [B, 1, H]
  unsigned char *ws;          // workspace base
  WorkspaceLayout wl;
  int batch, heads, head_groups, heads_per_group;
  int num_pages, max_pages;
  int part_id, num_parts;
  // All partitions in one launch (tensor-core kernel only): output row bv of
  // `batch` = num_parts * req_batch rows is request bv % req_batch of
  // partition bv / req_batch; out / lse are then [P, B, ...].  Otherwise
  // fused = 0 and req_batch = batch.
  int fused = 0, req_batch = 0;
  // fused only: the partitions' LSE combine, written by the merge kernel
  // ([B, rows, 512] bf16 and, optionally, [B, rows] fp32 in the lse base)
  __nv_bfloat16 *comb_out = nullptr;
  float *comb_lse = nullptr;
  // Query tokens per request (tensor-core kernel only; 1 elsewhere): the
  // `heads` rows of a request are then q_len x q_heads, row i * q_heads + h
  // for query token i, and token i of T sees the global tokens t < L - T + i + 1.
  int q_len = 1, q_heads = 0;
  // Owner mask (tensor-core kernel only): when own_parts > num_parts the call
  // computes partition own_part of own_parts through the gather of partition
  // part_id = own_part mod num_parts of num_parts (num_parts divides both 8
  // and own_parts), and the softmax drops every gathered token whose global
  // index is not own_part mod own_parts.  Otherwise own_parts = 0.
  int own_parts = 0, own_part = 0;
  // Strided gather (tensor-core kernel, P in {3, 5, 6, 7}):
  // partition r's rows of page lp are y0 + kP (y0 = (r - 64 lp)
  // mod P), landed by TMA with a traversal stride of P in atoms of 8 rows,
  // `apg` atoms per page.  The tile walk then runs over slots: page lp holds
  // slots [8 apg lp, 8 apg (lp + 1)), slot 8 apg lp + k is row y0 + kP when
  // that row is below 64 (else the slot is empty), and a request's length in
  // slots ends just past its last owned token.  Otherwise strided = 0.
  int strided = 0, apg = 0;
  int s_q63 = 0, s_r63 = 0, s_c64 = 0;  // strided: 63 / P, 63 mod P, 64 mod P
  int kv_e4m3;
  float kv_scale;             // 1 for bf16
  float score_scale_log2;     // sm_scale * log2(e): scores kept in the base-2 domain
  int lse_base2;              // output lse in base 2 (else natural)
};

// ---------------------------------------------------------------- host: per-device set-up

// Raises one kernel's dynamic shared-memory limit on each device the first
// time it is launched there.  Thread-safe: host threads that launch on the
// same device for the first time at once take a lock, and later launches
// read only an atomic flag.  One static instance per kernel.
struct SmemLimitOnce {
  std::atomic<uint64_t> done{0};  // bit d: set on device d
  std::mutex mu;
  template <typename Kernel>
  cudaError_t ensure(Kernel kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu);
    if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// ---------------------------------------------------------------- partition rule

// Tokens owned by partition r of P out of a global length L: t < L, t mod P == r.
__host__ __device__ __forceinline__ int local_len(int L, int P, int r) {
  return L / P + (r < L % P ? 1 : 0);
}

// Virtual request v -> its output row b and head group g: group-major,
// v = g * batch + b.  The split schedule cuts the concatenated tile sequence
// of all virtual requests into equal cost ranges, one per CTA; in this order
// the head groups of a request (or the query-token groups of a request with
// several query tokens) sit at the same offset of head_groups equal stretches
// of that sequence, so CTAs c, c + G / head_groups, ... walk the same pages
// at the same time and the later reads of a page find it in L2: the cache
// is read from HBM once for all rows of a request.
__host__ __device__ __forceinline__ int vreq_row(const DecodeParams &p, int v) { return v % p.batch; }
__host__ __device__ __forceinline__ int vreq_group(const DecodeParams &p, int v) { return v / p.batch; }
__host__ __device__ __forceinline__ int vreq_index(const DecodeParams &p, int b, int g) {
  return g * p.batch + b;
}

// Output row bv -> the input request it reads (q, block table, length) and
// the partition it attends for.
__device__ __forceinline__ int req_of(const DecodeParams &p, int bv) {
  return p.fused ? bv % p.req_batch : bv;
}
__device__ __forceinline__ int part_of(const DecodeParams &p, int bv) {
  return p.fused ? bv / p.req_batch : p.part_id;
}

// Clamp a global length to what the block table can hold; flag a bad one.
__device__ __forceinline__ int checked_len(const DecodeParams &p, int b, int *err) {
  int L = p.seq_lens[b];
  int cap = p.max_pages * kPage;
  if (L < 0 || L > cap) {
    if (err) atomicOr(err, kErrBadLen);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

// Global tokens visible to row `row` of a request of length L, and to the
// rows of head group g (its last row sees the most).
__device__ __forceinline__ int row_len(const DecodeParams &p, int L, int row) {
  return p.q_len <= 1 ? L : max(0, L - p.q_len + row / p.q_heads + 1);
}
__device__ __forceinline__ int group_len(const DecodeParams &p, int L, int g) {
  return p.q_len <= 1 ? L : row_len(p, L, min(p.heads, (g + 1) * p.heads_per_group) - 1);
}

// Strided gather: the first row partition `part` owns in logical page lp,
// and the slots of a request of length L (see DecodeParams::strided).
__host__ __device__ __forceinline__ int strided_y0(int part, int P, int lp) {
  return ((part - (kPage % P) * (lp % P)) % P + P) % P;
}
__host__ __device__ __forceinline__ int strided_slots(int L, int P, int r, int apg) {
  const int n = local_len(L, P, r);
  if (n == 0) return 0;
  const int t_last = r + P * (n - 1);
  const int lp = t_last / kPage;
  const int y0 = strided_y0(r, P, lp);
  return 8 * apg * lp + (t_last - kPage * lp - y0) / P + 1;
}
// The slots of consecutive tiles that hold a row (below 64 within its page),
// walked atom by atom without a division: page lp + 1 starts at
// y0 - (64 mod P) (mod P), and a page with start y0 holds 63 / P + 1 rows of
// the partition, one fewer when y0 > 63 mod P.
struct StridedMask {
  int ap, y0;  // the next atom: its index within its page, its page's first row
  __device__ void start(const DecodeParams &p, int part, long long t) {
    const int a = int(8 * t), lp = a / p.apg;
    ap = a - lp * p.apg;
    y0 = strided_y0(part, p.num_parts, lp);
  }
  // bit i set when slot i of the next tile holds a row; moves to the tile after
  __device__ __forceinline__ unsigned long long next(const DecodeParams &p) {
    unsigned long long m = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int rows = p.s_q63 + 1 - (y0 > p.s_r63 ? 1 : 0);
      const int v = min(8, max(0, rows - 8 * ap));
      m |= ((1ull << v) - 1ull) << (8 * k);
      if (++ap == p.apg) {
        ap = 0;
        y0 -= p.s_c64;
        if (y0 < 0) y0 += p.num_parts;
      }
    }
    return m;
  }
};

// Owned tokens of virtual request v (its group's widest row).
// MULTI: rows may differ in the tokens they see (several query tokens, or an
// owner mask); MULTI == 2: the strided gather, whose lengths count slots.  A
// compile-time switch, so that each kernel keeps only its own length rule.
template <int MULTI = 0>
__device__ __forceinline__ int request_len(const DecodeParams &p, int v, int *err) {
  int bv = vreq_row(p, v);
  int L = checked_len(p, req_of(p, bv), err);
  if (MULTI) L = group_len(p, L, vreq_group(p, v));
  // under an owner mask, a request the real partition owns no token of is
  // empty (the neutral pair), however many the gathered partition holds
  if (MULTI && p.own_parts > p.num_parts && local_len(L, p.own_parts, p.own_part) == 0) return 0;
  // strided gather (MULTI == 2): the length in slots
  if (MULTI == 2) return strided_slots(L, p.num_parts, part_of(p, bv), p.apg);
  return local_len(L, p.num_parts, part_of(p, bv));
}

// Kernels whose rows may differ in the tokens they see: several query
// tokens per request, or an owner mask.
__host__ __device__ __forceinline__ bool multi_rows(const DecodeParams &p) {
  return p.q_len > 1 || p.own_parts > p.num_parts || p.strided;
}

// Owner mask of the gathered partition's tiles.  Local token j of partition
// part_id of num_parts is global token part_id + j * num_parts; with
// Q = own_parts / num_parts it belongs to own_part when j = c mod Q,
// c = own_part / num_parts.  bits(t): bit i set when local token 64t + i is
// owned.
struct OwnerMask {
  unsigned long long comb;  // bits 0, Q, 2Q, ... below 64
  int q, c;
  __device__ __forceinline__ unsigned long long bits(long long t) const {
    return comb << int(((long long)c - (64 * t) % q + q) % q);
  }
};

__device__ inline OwnerMask owner_mask_of(const DecodeParams &p) {
  OwnerMask o;
  o.q = p.own_parts / p.num_parts;
  o.c = p.own_part / p.num_parts;
  o.comb = 0;
  for (int j = 0; j < 64; j += o.q) o.comb |= 1ull << j;
  return o;
}

template <int MULTI = 0>
__device__ __forceinline__ int request_tiles(const DecodeParams &p, int v) {
  return (request_len<MULTI>(p, v, nullptr) + kTile - 1) / kTile;
}

// ---------------------------------------------------------------- split schedule
//
// Cost-weighted stream-K split of the concatenated tile sequence of all
// virtual requests v = g * batch + b (tiles_v = ceil(local_len / 64)).
// Every request with tiles costs tiles_v + PC: the extra units stand for the
// per-piece work (Q load, pipeline refill, epilogue), so a CTA whose range
// crosses a request boundary gets fewer tiles.  Request v occupies cost units
// [P_v, P_v + tiles_v) followed by a gap of PC; C = total cost.  PC is a
// compile-time constant of each kernel variant (kPieceCost, or kPieceCostE4m3
// for the e4m3 tensor-core variants): read from the launch parameters instead
// it measured slower.
// G_eff = min(gridDim.x, C) CTAs; CTA c owns the tiles whose cost lies in
// [c*C/G_eff, (c+1)*C/G_eff).  A request crossing a boundary is split; each
// split writes a normalised fp32 partial into slot 2c (the CTA's first
// request) or 2c+1 (its last); the request's first CTA records {itself,
// split count, its slot} and a second kernel merges the splits.

struct CtaRange {
  long long start, end;   // cost range of this CTA
  long long total;        // C
  int g_eff;              // CTAs that own cost units
  int v_begin;            // first virtual request with tiles in range
  long long p_begin;      // cost start of v_begin
};

__device__ __forceinline__ long long sched_start(long long c, long long C, int g_eff) {
  return c * C / g_eff;
}

// Largest c with sched_start(c) <= x.
__device__ __forceinline__ int sched_owner(long long x, long long C, int g_eff) {
  return int(((x + 1) * g_eff - 1) / C);
}

__device__ __forceinline__ long long request_cost(int tiles, int piece_cost) {
  return tiles > 0 ? tiles + piece_cost : 0;
}

// Block-wide: computes this CTA's range.  All threads must call it.
// `scratch` needs blockDim.x / 32 + 1 long longs of shared memory.
template <int MULTI = 0, int PC = kPieceCost>
__device__ inline void cta_schedule(const DecodeParams &p, CtaRange *r, long long *scratch) {
  const int V = p.batch * p.head_groups;
  const int tid = threadIdx.x, nw = blockDim.x / 32, lane = tid & 31, warp = tid >> 5;
  // pass 1: total cost
  long long mine = 0;
  for (int v = tid; v < V; v += blockDim.x) mine += request_cost(request_tiles<MULTI>(p, v), PC);
  for (int o = 16; o; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) scratch[warp] = mine;
  __syncthreads();
  if (tid == 0) {
    long long C = 0;
    for (int w = 0; w < nw; ++w) C += scratch[w];
    r->total = C;
    r->g_eff = int(C < (long long)gridDim.x ? C : (long long)gridDim.x);
    r->v_begin = V;
    r->p_begin = 0;
    if (r->g_eff > 0 && (int)blockIdx.x < r->g_eff) {
      r->start = sched_start(blockIdx.x, C, r->g_eff);
      r->end = sched_start(blockIdx.x + 1, C, r->g_eff);
    } else {
      r->start = r->end = 0;
    }
  }
  __syncthreads();
  const long long start = r->start, end = r->end;
  if (start >= end) return;
  // pass 2: the first request whose tiles end after `start` (chunked block
  // scan of the costs); its predecessor ends at P_v - PC
  long long base = 0;
  for (int v0 = 0; v0 < V; v0 += blockDim.x) {
    int v = v0 + tid;
    const int tiles = v < V ? request_tiles<MULTI>(p, v) : 0;
    const long long cst = request_cost(tiles, PC);
    long long incl = cst;
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    long long wbase = 0, chunk = 0;
    for (int w = 0; w < nw; ++w) {
      if (w < warp) wbase += scratch[w];
      chunk += scratch[w];
    }
    const long long excl = base + wbase + incl - cst;
    if (tiles > 0 && excl + tiles > start && excl - PC <= start) {
      r->v_begin = v;
      r->p_begin = excl;
    }
    base += chunk;
    __syncthreads();
    if (r->v_begin < V) break;  // uniform: read after the barrier
  }
  __syncthreads();
}

// ---------------------------------------------------------------- conversions

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(uint32_t(b) << 16);
}

// Two OCP e4m3 bytes -> two exact f16 values (hardware conversion).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t r;
  asm("{ cvt.rn.f16x2.e4m3x2 %0, %1; }" : "=r"(r) : "h"(two));
  return r;
}

// Two floats -> two OCP e4m3 bytes, round to nearest even, saturated to the
// finite range (hardware conversion): `lo` in the low byte.
__device__ __forceinline__ uint16_t float2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("{ cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2; }" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> two OCP e5m2 bytes (hardware conversion, RNE, saturated):
// `lo` in the low byte.
__device__ __forceinline__ uint16_t float2_to_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("{ cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2; }" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two e5m2 bytes -> two exact floats (through the hardware f16 conversion).
__device__ __forceinline__ float2 e5m2x2_to_float2(uint16_t two) {
  uint32_t h;
  asm("{ cvt.rn.f16x2.e5m2x2 %0, %1; }" : "=r"(h) : "h"(two));
  __half2 hh = *reinterpret_cast<__half2 *>(&h);
  return __half22float2(hh);
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  uint32_t h = e4m3x2_to_f16x2(two);
  __half2 hh = *reinterpret_cast<__half2 *>(&h);
  return __half22float2(hh);
}

}  // namespace mla
