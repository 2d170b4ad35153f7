// Tensor-core decode kernel for sm_103a: one CTA per SM walks its stream-K
// range of 64-token tiles; TMA stages the partition's KV rows, tcgen05 MMAs
// compute S = Q K^T (heads as M = 64) and O^T = V^T P^T (value dims as M =
// 128, heads as N) with fp32 accumulators in TMEM, and a warpgroup runs the
// online softmax between them.
//
// Roles (288 threads):
//   warp 0          TMA producer: Q of each request (bf16: 9 boxes of 64 dims) and,
//                   per tile, the 64/P rows the partition owns of each page
//                   (lane k: page k) into a swizzled [column group][atom]
//                   [dim block][8 rows][128 B] layout that serves both MMAs:
//                   three boxes per page of three dim blocks each when P = 1
//                   (the score MMAs start on the first), else one box.
//   warp 1          TMEM owner (alloc/free).
//   warps 1, 2      lane 0 issues half of the score MMAs (one accumulator each).
//   warps 3, 8      lane 0 issues the PV MMAs of two of the four value chunks.
//   warps 9..11     (e4m3) Q of each request, split into two e4m3 terms.
//   warps 4..7      softmax and epilogue.  The S accumulator (M = 64) puts
//                   head 16q + i in TMEM lane 32q + i (i < 16); read with the
//                   16x256b shape, each lane of warp q gets 2 heads x 16 of the
//                   64 tokens.  For the epilogue every thread owns TMEM lane
//                   32q + lane of O^T: one value dimension.
//
// e4m3 caches (the same kernel with F8 = true, 384 threads): the MMAs are
// kind::f8f6f4 and read the cache's raw rows as landed, in five swizzled
// blocks of 128 dims (three 40 KB stages).  Warps 9..11 read each request's
// Q (bf16) and split 2^k Q into two e4m3 terms, hi + lo, that hold it exactly
// down to 2^-2 of the scaled values (k puts the largest |q| in [2^7, 2^8));
// the score issuers take one term each (S = Q_hi K^T + Q_lo K^T, 18 K-steps
// of 32 dims), the scores carry sm_scale * kv_scale * 2^-k, and the softmax
// writes P as two terms as well (hi e4m3, lo e5m2: P <= 2^8 stays below
// e4m3's maximum), so that each PV step is two MMAs;
// the output is normalised by the sum of P as stored, the LSE takes the sum
// before rounding.  V^T is the raw rows read MN-major.
//
// Partitions: P divides 8 here (64/P owned rows per page), or P in
// {3, 5, 6, 7}: the strided gather (MULTI == 2, DecodeParams::strided), where
// producer lane k loads atom k of the tile, rows y0 + iP of its page through a
// TMA traversal stride, and the softmax masks the tile's empty slots.  A call
// for another P runs the gather of P' = gcd(P, 8) with an owner mask in the
// softmax (DecodeParams::own_parts), through the several-row variants
// (MULTI == 1), which carry the per-row bounds and guards that mask needs.
//
// Pipeline per tile i (stage i mod 2, i mod 3 for e4m3; S buffer i mod 2):
// producer -> kv_full (per column group or block) -> MMA S_i (36 MMAs, two
// accumulators so consecutive MMAs are independent) -> s_full -> softmax
// reads S_i, frees it (s_free), waits for PV_{i-1} (p_free) and rescales
// O^T only when some head's running max grew by more than the threshold
// (2^8), writes P_i -> p_full -> MMA PV_i (4 independent
// value-dim chunks) -> kv_empty + p_free.  The score issuers start S_{i+1} as
// soon as tile i+1 lands, so the score MMAs of the next tile overlap this
// tile's softmax, and the producer keeps the pages of the next tile (two
// ahead when a tile gathers several pages) streaming into L2.  The kernel is
// launched as a programmatic dependent of the stream's previous kernel: its
// prologue overlaps that kernel's tail, and griddepcontrol.wait precedes
// every read of an input.
#pragma once

#include "common.cuh"
#include "sm100.cuh"
#include "splits.cuh"

namespace mla {
using namespace sm100;

namespace tc {
constexpr int kThreads = 288;                // bf16 cache
constexpr int kThreadsF8 = 384;              // e4m3 cache: + 3 warps that split Q
constexpr int kConvWarp0 = 9;                // the first of them
constexpr int kConvThreads = 96;
constexpr int kHeads = 64;                   // heads per virtual request (M of S)
constexpr int kKb = kDqk / 64;               // 9 blocks of 64 bf16 = 128 B
constexpr int kQBytes = kKb * 64 * 128;      // [kb][64 rows][128 B]
constexpr int kAtomBytes = kKb * 1024;       // 8 tokens x 576 dims
constexpr int kStageBytes = 8 * kAtomBytes;  // 64 tokens
// bf16 stage layout: column groups of KBG dim blocks each,
// [group][atom (8 rows)][dim block within the group][8 rows][128 B].
// KBG = 3 (P = 1: a tile is one page): three groups (dims 0..191, 192..383,
// 384..575), each landed by its own TMA box and barrier, so the score MMAs
// start on the first group while the others are in flight.  KBG = 9
// otherwise: one group, one box per page (a tile of P > 1 gathers P pages,
// and three boxes per page cost more than they gain).  P [64 heads][64
// tokens] reuses the rope block (dims 512..575) of the tile's own stage,
// dead once S is computed.  (e4m3: KBG = 4, blocks 0..3 of an atom land
// together and block 4 apart; the layout is below.)
template <bool F8, int AHEAD>
constexpr int stage_kbg() { return F8 ? 4 : AHEAD == 1 ? 3 : kKb; }
template <int KBG>
constexpr int num_groups() { return kKb / KBG; }
template <int KBG>
constexpr uint32_t atom_stride() { return uint32_t(KBG) * 1024u; }
// byte offset of dim block kb of atom 0 within a stage
template <int KBG>
__host__ __device__ constexpr uint32_t kb_off(int kb) {
  return uint32_t(kb / KBG) * 8u * atom_stride<KBG>() + uint32_t(kb % KBG) * 1024u;
}
constexpr int kMaxGroups = 5;
constexpr int kOffQ = 0;
constexpr int kOffKv = kOffQ + kQBytes;
constexpr int kOffMisc = kOffKv + 2 * kStageBytes;

// e4m3 caches, read by fp8 MMAs straight from the raw rows: Q as two e4m3
// terms, hi and lo, each [5 blocks of 128 dims][64 rows][128 B], swizzled
// K-major; three stages of the raw rows as landed, blocks 0..3 as [8
// atoms][block][8 rows][128 B] (one box per page, or per atom for the strided
// gather) and block 4, dims 512..575, as [64 rows][64 B] with the 64-byte
// swizzle after them (a box of its own, issued first: it is the small one, and
// the score MMAs start on it).  The 8 KB block-4 area, dead once the scores
// are computed, then holds P as two terms [64 heads][64 tokens] of 4 KB
// each, hi in e4m3 and lo in e5m2, unswizzled: 8-head x 16-token core
// matrices of 128 B.
constexpr int kFxBlocks = 5;
constexpr int kFxBlock = 64 * 128;                   // one block of 64 rows
constexpr int kFxQTerm = kFxBlocks * kFxBlock;       // 40 KB
constexpr int kFxStageBytes = kFxBlocks * kFxBlock;  // 40 KB
constexpr uint32_t kFxPLbo = 128, kFxPSbo = 512;     // P core matrices along tokens / heads
constexpr uint32_t kFxBlkStride = 1024, kFxAtomStride = 4096;  // raw rows: blocks 0..3, 8-row atoms
constexpr int kFxPTerm = 4096;                       // P lo after P hi
// P is stored as 2^(8 - threshold) p (p <= 2^threshold), below the e4m3
// maximum (448).  Its lo term is e5m2, whose subnormals reach 2^-16: weights
// down to 2^-16 of the running maximum keep a value (e4m3's floor, 2^-9,
// would drop those below 2^-9, and a long context's tail of such weights can
// hold much of the mass).  The sum that normalises the output takes P as
// stored; the LSE takes the sum of P before rounding.  (A lower threshold
// would lower that floor further but rescales O far more often.)
constexpr float kFxRescaleThreshold = 8.f;
constexpr float kFxPLog2Scale = 8.f - kFxRescaleThreshold;
template <bool F8>
constexpr int num_stages() { return F8 ? 3 : 2; }
template <bool F8>
constexpr int stage_bytes() { return F8 ? kFxStageBytes : kStageBytes; }
template <bool F8>
constexpr int off_kv() { return F8 ? 2 * kFxQTerm : kOffKv; }
template <bool F8>
constexpr int off_misc() { return off_kv<F8>() + num_stages<F8>() * stage_bytes<F8>(); }
constexpr int kSmemBytes = 232448;           // per-block maximum on sm_100 parts
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;                // O^T chunk c: columns [64c, 64c + npv)
constexpr uint32_t kColS = 256;              // S(buffer s, chain k): 256 + 64 (2s + k)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr float kRescaleThreshold = 8.f;     // base-2 units
}  // namespace tc

struct TcParams {
  DecodeParams p;
  int npv;              // N of the PV MMA: heads rounded up to 16 (16..64)
  int q_rows;           // rows of one Q box: min(64, H)
  int groups_per_page;  // 8-row atoms one page holds for this partition: 8 / P
};

template <bool F8>
constexpr int tc_threads() { return F8 ? tc::kThreadsF8 : tc::kThreads; }

// Barriers and scratch; NS shared-memory stages (the two S buffers in TMEM
// are separate from them).
template <int NS>
struct TcMisc {
  uint64_t kv_full[NS][tc::kMaxGroups], kv_empty[NS], q_full, q_empty, s_full[2], s_free[2];
  uint64_t p_full[NS], p_free[NS], o_full, o_free, drain;
  uint64_t q_ready;               // e4m3 only: Q split into its two terms
  uint32_t tmem_base;
  int abort;
  float alpha[2][64];
  float ell[64];
  float qinv[4];                 // e4m3 only: 2^-k of Q's scale, by request piece mod 4
  int qinv_v[4];                 // e4m3 only: the virtual request each qinv slot holds
  uint32_t vote[2][4];           // softmax: per-warp flags of the tile, by tile parity
  alignas(16) unsigned char stage_out[4][2048];  // epilogue: per-warp transpose buffer
  uint32_t conv_max[4];
  CtaRange range;
  long long scratch[tc::kThreadsF8 / 32 + 1];
};
static_assert(sizeof(TcMisc<2>) + 1024 <= tc::kSmemBytes - tc::off_misc<false>(), "shared memory budget");
static_assert(sizeof(TcMisc<3>) + 1024 <= tc::kSmemBytes - tc::off_misc<true>(), "shared memory budget");

template <bool F8>
using TcMiscFor = TcMisc<tc::num_stages<F8>()>;

// The split schedule's cost of a request piece's boundary, per cache dtype.
template <bool F8>
constexpr int piece_cost() { return F8 ? kPieceCostE4m3 : kPieceCost; }

// The requests (and tile ranges) this CTA owns, in order; every role walks it.
// FUSED: all partitions in one launch (output row b = partition * B + input
// request); otherwise one partition, p.part_id, and row b is request b.
template <bool FUSED, int MULTI, int PC>
struct Walk {
  const DecodeParams &p;
  const CtaRange &r;
  int V, v, b, g, n, tiles;
  int rb, part, pc;  // input request of output row b, its partition, the map's partition coordinate
  long long pv, t0, t1;
  __device__ Walk(const DecodeParams &p_, const CtaRange &r_)
      : p(p_), r(r_), V(p_.batch * p_.head_groups), v(r_.v_begin), pv(r_.p_begin) {}
  __device__ bool next() {
    while (v < V && pv < r.end) {
      tiles = request_tiles<MULTI>(p, v);
      if (tiles == 0) { ++v; continue; }
      t0 = max(r.start, pv) - pv;
      t1 = min(r.end, pv + tiles) - pv;
      b = vreq_row(p, v);
      g = vreq_group(p, v);
      rb = FUSED ? b % p.req_batch : b;
      part = FUSED ? b / p.req_batch : p.part_id;
      pc = FUSED ? part : 0;
      const int L = checked_len(p, rb, nullptr);
      n = MULTI == 2 ? strided_slots(group_len(p, L, g), p.num_parts, part, p.apg)  // slots
          : MULTI      ? local_len(group_len(p, L, g), p.num_parts, part)
                       : local_len(L, p.num_parts, part);
      return true;
    }
    return false;
  }
  __device__ void advance() { pv += request_cost(tiles, PC); ++v; }
};

// One position in the walk: request + tile.
template <bool FUSED, int MULTI, int PC>
struct TileCursor {
  Walk<FUSED, MULTI, PC> w;
  long long t;
  bool live;
  __device__ TileCursor(const DecodeParams &p, const CtaRange &r) : w(p, r), t(0) {
    live = w.next();
    if (live) t = w.t0;
  }
  __device__ void step() {
    if (++t >= w.t1) {
      w.advance();
      live = w.next();
      if (live) t = w.t0;
    }
  }
  __device__ bool first() const { return t == w.t0; }
  __device__ bool last() const { return t == w.t1 - 1; }
  __device__ int nv() const { return min(kTile, w.n - int(t) * kTile); }
};

__device__ __forceinline__ uint32_t bar_addr(uint64_t &b) { return smem_u32(&b); }

// Logical pages [lp0, lp1] that hold tile t's owned tokens (n tokens owned by
// partition `part`).
__device__ __forceinline__ void tile_pages(const DecodeParams &p, int part, long long t, int n,
                                           int *lp0, int *lp1) {
  const int jl = min(int(t) * kTile + kTile, n) - 1;
  *lp0 = int(t) * p.num_parts;
  *lp1 = int((part + (long long)p.num_parts * jl) / kPage);
}

// The logical page that producer lane `lane` loads for tile t, and the first
// page row of its box: lane k loads page lp0 + k of the tile's pages, or, for
// the strided gather, atom 8t + k (rows row0 + iP, i < 8, of its page).
// False when the lane loads nothing.
template <bool STRIDED>
__device__ __forceinline__ bool lane_page(const DecodeParams &p, int part, long long t, int n, int lane,
                                          int *lp, int *row0) {
  if (STRIDED) {
    const int a = int(8 * t) + lane;
    if (lane >= 8 || 8 * a >= n) return false;
    *lp = a / p.apg;
    *row0 = strided_y0(part, p.num_parts, *lp) + 8 * p.num_parts * (a - *lp * p.apg);
    return true;
  }
  int lp0, lp1;
  tile_pages(p, part, t, n, &lp0, &lp1);
  *lp = lp0 + lane;
  *row0 = 0;
  return lane <= lp1 - lp0;
}

// ------------------------------------------------------------------ producer

// AHEAD: tiles whose pages are pulled into L2 ahead of the stage.  1 when a
// bf16 tile is one page (P = 1), else 2 (each the measured best of 0..4).  It is a template parameter because the same choice
// made at run time costs more than it gains.
template <bool F8, bool FUSED, int MULTI, int AHEAD>
__device__ __forceinline__ void tc_producer(const TcParams &tp, const CtaRange &r, TcMiscFor<F8> &m,
                            uint32_t sQ, uint32_t sKv, const CUtensorMap *tm_q, const CUtensorMap *tm_kv,
                            const CUtensorMap *tm_kvg, const CUtensorMap *tm_kvb, int *err) {
  using namespace tc;
  constexpr bool STRIDED = MULTI == 2;
  constexpr int NS = num_stages<F8>();
  const DecodeParams &p = tp.p;
  volatile int *abort = &m.abort;
  const int lane = threadIdx.x & 31;
  uint32_t kv_it = 0, q_it = 0;
  int last_q = -1, last_kv[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) last_kv[s] = -1;
  // bf16: one 4-D box of groups_per_page swizzled atoms per page; e4m3: per
  // block of 128 dims (one barrier each), one swizzled box of the page's
  // 8 * groups_per_page owned rows (the strided gather: of one atom's rows)
  const int rows_per_page = 8 * tp.groups_per_page;
  constexpr int KBG = stage_kbg<F8, AHEAD>();
  constexpr int kG = F8 ? 2 : num_groups<KBG>();
  // bytes one page lands per barrier: its rows of one block, or one column group
  const uint32_t page_bytes = F8 ? uint32_t(tp.groups_per_page) * 1024u
                                 : uint32_t(tp.groups_per_page) * atom_stride<KBG>();
  bool ok = true;

  // The whole warp produces: lane k handles page k of a tile (a tile spans P
  // pages), so the page-index loads, L2 prefetches and TMA boxes of a tile go
  // out together rather than one after another.  A lane's page index is read
  // one or two tiles early, when the page is prefetched into L2 (the
  // 129 MB L2 gives the two shared-memory stages more HBM requests in
  // flight), and carried in `ring` until its tile is loaded.
  TileCursor<FUSED, MULTI, piece_cost<F8>()> ahead(p, r);
  auto next_ahead = [&]() {
    int pg = -1;
    if (ahead.live) {
      int lp, row0;
      if (lane_page<STRIDED>(p, ahead.w.part, ahead.t, ahead.w.n, lane, &lp, &row0)) {
        pg = p.block_table[size_t(ahead.w.rb) * p.max_pages + lp];
        if (pg >= 0 && pg < p.num_pages) {
          if (F8 && STRIDED) {
            tma_prefetch_3d(tm_kv, 0, row0, pg);
          } else if (F8) {
            if (FUSED)
              tma_prefetch_3d(tm_kv, 0, pg * rows_per_page, ahead.w.pc);
            else
              tma_prefetch_2d(tm_kv, 0, pg * rows_per_page);
          } else if (STRIDED) {
            tma_prefetch_4d(tm_kv, 0, row0, 0, pg);
          } else {
            if (FUSED)
              tma_prefetch_5d(tm_kv, 0, 0, 0, pg * tp.groups_per_page, ahead.w.pc);
            else
              tma_prefetch_4d(tm_kv, 0, 0, 0, pg * tp.groups_per_page);
          }
        }
      }
      ahead.step();
    }
    return pg;
  };
  static_assert(AHEAD == 1 || AHEAD == 2, "prefetch distance");
  int ring[AHEAD];
#pragma unroll
  for (int i = 0; i < AHEAD; ++i) ring[i] = next_ahead();

  TileCursor<FUSED, MULTI, piece_cost<F8>()> cur(p, r);
  while (cur.live) {
    if (!F8 && cur.first()) {  // (e4m3: warps 9..11 load and split Q)
      checked_len(p, cur.w.rb, err);
      if (!__all_sync(0xffffffffu, mbar_wait(bar_addr(m.q_empty), (q_it & 1) ^ 1, abort, kTimeoutNs))) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar_addr(m.q_full), uint32_t(kKb * tp.q_rows * 128));
      __syncwarp();
      if (lane < kKb)
        tma_load_2d(sQ + lane * (64 * 128), tm_q, bar_addr(m.q_full), lane * 64,
                    cur.w.rb * p.heads + cur.w.g * kHeads);
      last_q = q_it & 1;
      ++q_it;
    }
    if (F8 && cur.first()) checked_len(p, cur.w.rb, err);
    const int s = kv_it % NS;
    int lp, row0;
    const bool mine = lane_page<STRIDED>(p, cur.w.part, cur.t, cur.w.n, lane, &lp, &row0);
    int pg = ring[0];
    if (mine && (pg < 0 || pg >= p.num_pages)) {
      atomicOr(err, kErrBadPage);
      pg = -1;
    }
    const bool load = mine && pg >= 0;
    const uint32_t bytes = uint32_t(__popc(__ballot_sync(0xffffffffu, load))) * page_bytes;
    if (!__all_sync(0xffffffffu, mbar_wait(bar_addr(m.kv_empty[s]), ((kv_it / NS) & 1) ^ 1, abort,
                                           kTimeoutNs))) {
      ok = false;
      break;
    }
    // (e4m3: blocks 0..3 on the first barrier, four blocks' bytes; block 4,
    // 64 bytes a row, on the second)
    if (lane < kG)
      mbar_arrive_expect_tx(bar_addr(m.kv_full[s][lane]), F8 ? (lane == 0 ? 4 * bytes : bytes / 2) : bytes);
    __syncwarp();
    if (load) {
      const uint32_t dst = sKv + s * stage_bytes<F8>() + lane * page_bytes;
      if (F8) {
        // this lane's rows (its page's owned rows, or one atom of the strided
        // gather: rows row0 + iP of page pg, traversal stride P): block 4 (64
        // bytes a row) first, then blocks 0..3 as [atom][block][8 rows][128 B]
        // through the grouped map
        const uint32_t d0 = sKv + s * stage_bytes<F8>() + lane * page_bytes * 4;
        const uint32_t d4 = sKv + s * stage_bytes<F8>() + 4 * kFxBlock + lane * (page_bytes / 2);
        if (STRIDED) {
          tma_load_3d(d4, tm_kvg, bar_addr(m.kv_full[s][1]), 512, row0, pg);
          tma_load_4d(d0, tm_kvb, bar_addr(m.kv_full[s][0]), 0, row0, 0, pg);
        } else if (FUSED) {
          tma_load_3d(d4, tm_kvg, bar_addr(m.kv_full[s][1]), 512, pg * rows_per_page, cur.w.pc);
          tma_load_5d(d0, tm_kvb, bar_addr(m.kv_full[s][0]), 0, 0, 0, pg * tp.groups_per_page, cur.w.pc);
        } else {
          tma_load_2d(d4, tm_kvg, bar_addr(m.kv_full[s][1]), 512, pg * rows_per_page);
          tma_load_4d(d0, tm_kvb, bar_addr(m.kv_full[s][0]), 0, 0, 0, pg * tp.groups_per_page);
        }
      } else if (STRIDED) {
        // one atom: rows row0 + iP (traversal stride P) of page pg, all dims
        tma_load_4d(dst, tm_kv, bar_addr(m.kv_full[s][0]), 0, row0, 0, pg);
      } else {
        // group g: dim blocks [KBG g, KBG g + KBG) of the page's atoms
        const CUtensorMap *tm = KBG == kKb ? tm_kv : tm_kvg;
#pragma unroll
        for (int g = 0; g < kG; ++g) {
          const uint32_t dg = dst + uint32_t(g) * 8u * atom_stride<KBG>();
          if (FUSED)
            tma_load_5d(dg, tm, bar_addr(m.kv_full[s][g]), 0, 0, KBG * g, pg * tp.groups_per_page,
                        cur.w.pc);
          else
            tma_load_4d(dg, tm, bar_addr(m.kv_full[s][g]), 0, 0, KBG * g, pg * tp.groups_per_page);
        }
      }
    }
    last_kv[s] = (kv_it / NS) & 1;
    ++kv_it;
#pragma unroll
    for (int i = 0; i + 1 < AHEAD; ++i) ring[i] = ring[i + 1];
    ring[AHEAD - 1] = next_ahead();
    cur.step();
  }
  if (!ok && lane == 0) atomicOr(err, kErrTimeout);
  // never leave the CTA with a copy still in flight into its shared memory
  if (last_q >= 0) mbar_wait_drain(bar_addr(m.q_full), last_q, kDrainNs);
  for (int s = 0; s < NS; ++s)
    if (last_kv[s] >= 0)
      for (int g = 0; g < kG; ++g) mbar_wait_drain(bar_addr(m.kv_full[s][g]), last_kv[s], kDrainNs);
}

// ------------------------------------------------------------------ MMA issuers
//
// A tcgen05.mma costs its issuing thread ~55 cycles whatever its size up to
// N = 128 (measured on this GB300), so one thread cannot keep the tensor core
// fed with M = 64 / N = 64 score MMAs.  Three warps issue: two split the 36
// K-steps of S (one accumulator each), one issues PV.

// Descriptors: an offset is added to the encoded start address (bits 0..13,
// address >> 4), which never carries because shared addresses stay below 256 KB.
template <bool F8, bool FUSED, int MULTI, int KBG>
__device__ __forceinline__ void tc_mma_s(const TcParams &tp, const CtaRange &r, TcMiscFor<F8> &m,
                         uint32_t sQ, uint32_t sKv, uint32_t tmem, int chain, int *err) {
  using namespace tc;
  const DecodeParams &p = tp.p;
  volatile int *abort = &m.abort;
  // bf16: Q once landed, column group g of the stage once its own box has
  // landed; e4m3: Q once split into its two terms, block g once landed
  uint64_t &q_ready = F8 ? m.q_ready : m.q_full;
  if constexpr (F8) {
    // chain 0 scores with Q's hi term, chain 1 with its lo term: 18 K-steps
    // of 32 dims each (blocks 0..3: 4; block 4: 2)
    constexpr int NS = num_stages<F8>();
    const uint32_t idesc_s = idesc_e4m3_f32(64, 64, false, false);
    const uint64_t dq = smem_desc_sw128(sQ + uint32_t(chain) * kFxQTerm, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sKv, 16, kFxAtomStride);        // blocks 0..3
    const uint64_t dk4 = smem_desc_sw64(sKv + 4 * kFxBlock, 16, 512);  // block 4
    constexpr uint64_t kStageEnc = uint64_t(kFxStageBytes) >> 4;
    uint32_t s_it = 0, q_it = 0;
    bool ok = true;
    for (TileCursor<FUSED, MULTI, piece_cost<F8>()> sc(p, r); sc.live; sc.step(), ++s_it) {
      const int st = s_it % NS, sb = s_it & 1;
      const uint32_t ph = (s_it / NS) & 1;
      if (sc.first()) {
        if (!mbar_wait(bar_addr(q_ready), q_it & 1, abort, kTimeoutNs)) { ok = false; break; }
        ++q_it;
      }
      if (!mbar_wait(bar_addr(m.s_free[sb]), ((s_it >> 1) & 1) ^ 1, abort, kTimeoutNs)) {
        ok = false;
        break;
      }
      const uint32_t d = tmem + kColS + 64 * (2 * sb + chain);
      bool landed = true;
#pragma unroll
      for (int j = 0; j < kFxBlocks; ++j) {
        const int kb = (j + 4) % kFxBlocks;  // block 4 first, then blocks 0..3
        if (j < 2) {
          landed = mbar_wait(bar_addr(m.kv_full[st][1 - j]), ph, abort, kTimeoutNs);
          if (!landed) break;
          tc_fence_after();
        }
        const uint64_t dk = (kb < 4 ? dk0 + ((kb * kFxBlkStride) >> 4) : dk4) + st * kStageEnc;
#pragma unroll
        for (int ks = 0; ks < (kb < 4 ? 4 : 2); ++ks)
          mma_f8_ss(d, dq + ((kb * kFxBlock + ks * 32) >> 4), dk + ((ks * 32) >> 4), idesc_s,
                    j > 0 || ks > 0);
      }
      if (!landed) { ok = false; break; }
      mma_commit(bar_addr(m.s_full[sb]));
      if (sc.last()) mma_commit(bar_addr(m.q_empty));
    }
    if (!ok) atomicOr(err, kErrTimeout);
    mma_commit(bar_addr(m.drain));
    mbar_wait_drain(bar_addr(m.drain), 0, kDrainNs);
    return;
  }
  const uint32_t idesc_s = idesc_bf16_f32(64, 64, false, false);
  const uint64_t dq = smem_desc_sw128(sQ, 16, 1024);                         // Q, K-major
  const uint64_t dk0 = smem_desc_sw128(sKv + 32 * chain, 16, atom_stride<KBG>());  // K tile, K-major
  constexpr uint64_t kStageEnc = uint64_t(kStageBytes) >> 4;
  uint32_t s_it = 0, q_it = 0;
  bool ok = true;
  for (TileCursor<FUSED, MULTI, piece_cost<F8>()> sc(p, r); sc.live; sc.step(), ++s_it) {
    const int st = s_it & 1;
    const uint32_t ph = (s_it >> 1) & 1;
    if (!mbar_wait(bar_addr(m.kv_full[st][0]), ph, abort, kTimeoutNs)) {
      ok = false;
      break;
    }
    if (sc.first()) {
      if (!mbar_wait(bar_addr(q_ready), q_it & 1, abort, kTimeoutNs)) { ok = false; break; }
      ++q_it;
    }
    if (!mbar_wait(bar_addr(m.s_free[st]), ph ^ 1, abort, kTimeoutNs)) { ok = false; break; }
    tc_fence_after();
    const uint64_t dk = dk0 + st * kStageEnc;
    const uint32_t d = tmem + kColS + 64 * (2 * st + chain);
    // K-step ks = 2 i + chain: dim block i / 2, 16-dim slice 2 (i % 2) + chain
    bool landed = true;
#pragma unroll
    for (int i = 0; i < kKb * 2; ++i) {
      const int kb = i >> 1;
      if (i > 0 && kb % KBG == 0 && (i & 1) == 0) {
        landed = mbar_wait(bar_addr(m.kv_full[st][kb / KBG]), ph, abort, kTimeoutNs);
        if (!landed) break;
        tc_fence_after();
      }
      const uint32_t sub = 64u * uint32_t(i & 1) + 32u * uint32_t(chain);
      mma_bf16_ss(d, dq + ((kb * (64 * 128) + sub) >> 4),
                  dk + ((kb_off<KBG>(kb) + 64u * uint32_t(i & 1)) >> 4), idesc_s, i > 0);
    }
    if (!landed) { ok = false; break; }
    mma_commit(bar_addr(m.s_full[st]));
    if (sc.last()) mma_commit(bar_addr(m.q_empty));
  }
  if (!ok) atomicOr(err, kErrTimeout);
  mma_commit(bar_addr(m.drain));
  mbar_wait_drain(bar_addr(m.drain), 0, kDrainNs);
}

// O^T(chunk c) (+)= V^T(tile) P^T over ceil(nv/16) steps of 16 tokens; issuer
// `half` takes value chunks 2 half and 2 half + 1.
template <bool F8, bool FUSED, int MULTI, int KBG>
__device__ __forceinline__ void tc_mma_pv(const TcParams &tp, const CtaRange &r, TcMiscFor<F8> &m,
                          uint32_t sKv, uint32_t tmem, int half, int *err) {
  using namespace tc;
  const DecodeParams &p = tp.p;
  volatile int *abort = &m.abort;
  if constexpr (F8) {
    // O^T(chunk c) += V^T P_hi^T + V^T P_lo^T over ceil(nv / 32) steps of 32
    // tokens: V^T of chunk c is block c of the raw rows, MN-major (128 value
    // dims per swizzled row); P's terms (e4m3, e5m2) are K-major, unswizzled
    constexpr int NS = num_stages<F8>();
    const uint32_t idesc_o = idesc_e4m3_f32(128, tp.npv, true, false);
    const uint32_t idesc_o_lo = idesc_f8_f32(128, tp.npv, true, false, kFmtE4M3, kFmtE5M2);
    constexpr uint64_t kStageEnc = uint64_t(kFxStageBytes) >> 4;
    uint64_t dv0[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc)
      dv0[cc] = smem_desc_sw128(sKv + (2 * half + cc) * kFxBlkStride, kFxBlock, kFxAtomStride);
    const uint64_t dp0 = smem_desc_noswz(sKv + 4 * kFxBlock, kFxPLbo, kFxPSbo);
    uint32_t pv_it = 0, o_it = 0;
    bool ok = true;
    for (TileCursor<FUSED, MULTI, piece_cost<F8>()> pc(p, r); pc.live; pc.step(), ++pv_it) {
      const int st = pv_it % NS;
      if (!mbar_wait(bar_addr(m.p_full[st]), (pv_it / NS) & 1, abort, kTimeoutNs)) {
        ok = false;
        break;
      }
      const bool fresh = pc.first();
      if (fresh && !mbar_wait(bar_addr(m.o_free), (o_it & 1) ^ 1, abort, kTimeoutNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t dp = dp0 + st * kStageEnc;
      const int ksteps = (pc.nv() + 31) >> 5;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        if (ks < ksteps) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint32_t dcol = tmem + kColO + 64 * (2 * half + cc);
            const uint64_t dv = dv0[cc] + st * kStageEnc + ((ks * 4 * kFxAtomStride) >> 4);
            mma_f8_ss(dcol, dv, dp + ((ks * 2 * kFxPLbo) >> 4), idesc_o, !(fresh && ks == 0));
            mma_f8_ss(dcol, dv, dp + ((kFxPTerm + ks * 2 * kFxPLbo) >> 4), idesc_o_lo, 1u);
          }
        }
      }
      mma_commit(bar_addr(m.kv_empty[st]));
      mma_commit(bar_addr(m.p_free[st]));
      if (pc.last()) {
        mma_commit(bar_addr(m.o_full));
        ++o_it;
      }
    }
    if (!ok) atomicOr(err, kErrTimeout);
    mma_commit(bar_addr(m.drain));
    mbar_wait_drain(bar_addr(m.drain), 0, kDrainNs);
    return;
  }
  const uint32_t idesc_o = idesc_bf16_f32(128, tp.npv, true, false);
  // V^T of value chunk c (dim blocks 2c, 2c + 1), MN-major; P, K-major
  uint64_t dv0[2];
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int c = 2 * half + cc;
    dv0[cc] = smem_desc_sw128(sKv + kb_off<KBG>(2 * c), kb_off<KBG>(2 * c + 1) - kb_off<KBG>(2 * c),
                              atom_stride<KBG>());
  }
  const uint64_t dp0 = smem_desc_sw128(sKv + kb_off<KBG>(8), 16, atom_stride<KBG>());
  constexpr uint64_t kStageEnc = uint64_t(kStageBytes) >> 4;
  uint32_t pv_it = 0, o_it = 0;
  bool ok = true;
  for (TileCursor<FUSED, MULTI, piece_cost<F8>()> pc(p, r); pc.live; pc.step(), ++pv_it) {
    if (!mbar_wait(bar_addr(m.p_full[pv_it & 1]), (pv_it >> 1) & 1, abort, kTimeoutNs)) {
      ok = false;
      break;
    }
    const bool fresh = pc.first();
    if (fresh && !mbar_wait(bar_addr(m.o_free), (o_it & 1) ^ 1, abort, kTimeoutNs)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const int st = pv_it & 1;
    const uint64_t dp = dp0 + st * kStageEnc;
    const int ksteps = (pc.nv() + 15) >> 4;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (ks < ksteps) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * half + cc;
          mma_bf16_ss(tmem + kColO + 64 * c,
                      dv0[cc] + st * kStageEnc + ((2 * ks * atom_stride<KBG>()) >> 4),
                      dp + ((ks * 32) >> 4), idesc_o, !(fresh && ks == 0));
        }
      }
    }
    mma_commit(bar_addr(m.kv_empty[st]));
    mma_commit(bar_addr(m.p_free[st]));
    if (pc.last()) {
      mma_commit(bar_addr(m.o_full));
      ++o_it;
    }
  }
  if (!ok) atomicOr(err, kErrTimeout);
  mma_commit(bar_addr(m.drain));
  mbar_wait_drain(bar_addr(m.drain), 0, kDrainNs);
}

// ------------------------------------------------------------------ softmax + epilogue

// O^T *= alpha per head (column), for this warp's 32 TMEM lanes.  Rare (a
// head's running maximum grew by more than 2^8): kept out of line so that
// the softmax loop's instruction stream stays short.
static __device__ __noinline__ void rescale_o(uint32_t tq, const float *al, int npv) {
  using namespace tc;
  for (int c = 0; c < 4; ++c)
    for (int hb = 0; hb < npv / 16; ++hb) {
      uint32_t o[16];
      tmem_ld16(tq + kColO + 64 * c + 16 * hb, o);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al[16 * hb + i]);
      tmem_st16(tq + kColO + 64 * c + 16 * hb, o);
    }
  tmem_wait_st();
}

// Packed fp32 pair arithmetic (one instruction per pair on sm_100 parts).
__device__ __forceinline__ unsigned long long f2_bits(float2 a) {
  return *reinterpret_cast<unsigned long long *>(&a);
}
__device__ __forceinline__ float2 bits_f2(unsigned long long b) {
  return *reinterpret_cast<float2 *>(&b);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 2^x by the hardware approximation (relative error far below the bf16 / f16
// rounding that follows); results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Value rows [nv, roundup32(nv)) of a raw e4m3 stage (512 B of value dims
// each, blocks 0..3), zeroed by the softmax warpgroup (rank gt).
static __device__ __noinline__ void zero_value_tail_fx(unsigned char *stage, int nv, int gt) {
  using namespace tc;
  const int nrow = ((nv + 31) & ~31) - nv;
  for (int i = gt; i < nrow * 32; i += 128) {
    const int rr = nv + (i >> 5), kb = (i >> 3) & 3, ch = i & 7;
    *reinterpret_cast<uint4 *>(stage + kb * kFxBlkStride + (rr >> 3) * kFxAtomStride + (rr & 7) * 128 +
                               ch * 16) = make_uint4(0, 0, 0, 0);
  }
}

// Value rows [nv, roundup16(nv)) of a stage (the last tile of a request),
// zeroed by the softmax warpgroup (rank gt): out of line, once per request.
template <int KBG>
static __device__ __noinline__ void zero_value_tail(unsigned char *stage, int nv, int gt) {
  using namespace tc;
  const int r0 = nv, nrow = ((nv + 15) & ~15) - nv;
  for (int i = gt; i < nrow * 64; i += 128) {
    const int rr = r0 + (i >> 6), kb = (i >> 3) & 7, ch = i & 7;
    *reinterpret_cast<uint4 *>(stage + kb_off<KBG>(kb) + (rr >> 3) * atom_stride<KBG>() +
                               (rr & 7) * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
  }
}

template <bool F8, bool FUSED, int MULTI, int KBG>
__device__ __forceinline__ void tc_softmax(const TcParams &tp, const CtaRange &r, TcMiscFor<F8> &m,
                           unsigned char *smem, uint32_t tmem, int *err) {
  using namespace tc;
  constexpr bool STRIDED = MULTI == 2;
  constexpr int NS = num_stages<F8>();
  constexpr float kThreshold = F8 ? kFxRescaleThreshold : kRescaleThreshold;
  const DecodeParams &p = tp.p;
  volatile int *abort = &m.abort;
  const int gt = int(threadIdx.x) - 128;  // rank in the warpgroup
  const int q = gt >> 5, lane = gt & 31;
  // 16x256b view of the M = 64 score accumulator: this lane holds heads
  // row[0] = 16q + lane/4 and row[1] = row[0] + 8, and of every 8 tokens the
  // pair 2 (lane % 4) + {0, 1}; four lanes share a head.
  const int row[2] = {16 * q + (lane >> 2), 16 * q + (lane >> 2) + 8};
  const int pair = 2 * (lane & 3);
  const uint32_t tq = tmem + (uint32_t(32 * q) << 16);
  float cs = p.score_scale_log2 * p.kv_scale;
  uint32_t kv_it = 0, p_it = 0, o_it = 0;
  bool ok = true;
  // an owner mask: the gathered tiles hold other partitions' tokens too
  const bool masked = MULTI && p.own_parts > p.num_parts;
  OwnerMask own{};
  if (masked) own = owner_mask_of(p);

  uint32_t piece = 0;
  Walk<FUSED, MULTI, piece_cost<F8>()> w(p, r);
  for (; ok && w.next(); w.advance(), ++piece) {
    const int hn = min(kHeads, p.heads - w.g * kHeads);
    if (F8) {
      // Q's scale, written by warps 9..11 before the scores of this piece
      // were computed (its slot is checked against the request: bounded)
      const int slot = piece & 3;
      const volatile int *vv = m.qinv_v;
      const uint64_t t0 = globaltimer();
      while (vv[slot] != w.v && globaltimer() - t0 < kTimeoutNs) {
      }
      __threadfence_block();
      const bool have = vv[slot] == w.v;
      if (!have) atomicOr(err, kErrTimeout);
      cs = p.score_scale_log2 * p.kv_scale * (have ? m.qinv[slot] : 0.f);
    }
    // owned tokens each of this lane's two rows sees (all w.n unless a request
    // carries several query tokens, each with its own causal bound)
    int nrow[2] = {w.n, w.n};
    if (MULTI) {  // query token i of T sees the global tokens t < L - T + i + 1
      const int L = checked_len(p, w.rb, nullptr);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int Lr = row_len(p, L, w.g * kHeads + row[h]);
        // strided gather: slots are in token order, so the row's visible
        // slots end just past its last owned token below Lr
        nrow[h] = STRIDED ? strided_slots(Lr, p.num_parts, w.part, p.apg)
                          : local_len(Lr, p.num_parts, w.part);
      }
    }
    StridedMask smask;  // strided gather: the slots of each tile that hold a row
    if (STRIDED) smask.start(p, w.part, w.t0);
    float mrun[2] = {-INFINITY, -INFINITY};  // running max (base-2 units) of each head
    float ellp[2] = {0.f, 0.f};              // this lane's share of each head's sum
    float ellx[2] = {0.f, 0.f};              // e4m3: the same of P before rounding
    for (long long t = w.t0; t < w.t1; ++t, ++kv_it, ++p_it) {
      const int s = kv_it & 1;          // S buffer
      const int st = kv_it % NS;        // shared-memory stage
      const uint32_t ph = (kv_it >> 1) & 1;
      const int nv = min(kTile, w.n - int(t) * kTile);
      // Every wait of the warpgroup is followed by a group vote, so that a
      // wait that gave up in one warp never strands the others at a barrier.
      bool got = __all_sync(0xffffffffu, mbar_wait(bar_addr(m.s_full[s]), ph, abort, kTimeoutNs));
      // unscaled scores in token pairs: xp[2j + h] = head row[h], tokens
      // 8j + pair + {0, 1}
      float2 xp[16];
      if (got) {
        tc_fence_after();
        uint32_t ra[32], rb[32];
        tmem_ld16x256b_x8(tq + kColS + 64 * (2 * s), ra);
        tmem_ld16x256b_x8(tq + kColS + 64 * (2 * s + 1), rb);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k)
          xp[k] = add2(make_float2(__uint_as_float(ra[2 * k]), __uint_as_float(ra[2 * k + 1])),
                       make_float2(__uint_as_float(rb[2 * k]), __uint_as_float(rb[2 * k + 1])));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(m.s_free[s]));
      }
      const int nv0 = MULTI ? nrow[0] - int(t) * kTile : nv, nv1 = MULTI ? nrow[1] - int(t) * kTile : nv;
      if ((MULTI ? min(nv0, nv1) : nv) < kTile) {  // the tile's tail: tokens past a row's last visible one
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int tok = 8 * (k >> 1) + pair, lim = (k & 1) ? nv1 : nv0;
          xp[k].x = tok < lim ? xp[k].x : -INFINITY;
          xp[k].y = tok + 1 < lim ? xp[k].y : -INFINITY;
        }
      }
      if (STRIDED || (MULTI && masked)) {  // empty strided slots; tokens another partition owns
        unsigned long long ob;
        if constexpr (STRIDED) ob = smask.next(p);
        else ob = own.bits(t);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int tok = 8 * (k >> 1) + pair;
          xp[k].x = (ob >> tok) & 1ull ? xp[k].x : -INFINITY;
          xp[k].y = (ob >> (tok + 1)) & 1ull ? xp[k].y : -INFINITY;
        }
      }
      float tmax[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = max3(xp[h].x, xp[h].y, xp[2 + h].x);
        mx = max3(mx, xp[2 + h].y, xp[4 + h].x);
        mx = max3(mx, xp[4 + h].y, xp[6 + h].x);
        mx = max3(mx, xp[6 + h].y, xp[8 + h].x);
        mx = max3(mx, xp[8 + h].y, xp[10 + h].x);
        mx = max3(mx, xp[10 + h].y, xp[12 + h].x);
        mx = max3(mx, xp[12 + h].y, xp[14 + h].x);
        tmax[h] = fmaxf(mx, xp[14 + h].y);
      }
      float mnew[2], alpha[2];
      bool resc = false;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
        const float sm = tmax[h] * cs;  // cs > 0: the scaled maximum
        mnew[h] = mrun[h];
        alpha[h] = 1.f;
        if (t == w.t0) {
          mnew[h] = sm;
        } else if (sm > mrun[h] + kThreshold) {
          mnew[h] = sm;
          alpha[h] = exp2f(mrun[h] - sm);
          resc = true;
        }
      }
      if ((lane & 3) == 0) {
        m.alpha[p_it & 1][row[0]] = alpha[0];
        m.alpha[p_it & 1][row[1]] = alpha[1];
      }
      // One plain group barrier per tile: each warp posts whether one of its
      // heads needs an O rescale (bit 0) or a wait gave up (bit 1), and every
      // branch below follows the OR of the four, so all 128 lanes take it
      // together.  (Flags are double-buffered by tile parity: a warp cannot
      // rewrite a buffer before every warp has passed the next barrier.)
      {
        const uint32_t flag = (__any_sync(0xffffffffu, resc) ? 1u : 0u) | (got ? 0u : 2u);
        if (lane == 0) m.vote[p_it & 1][q] = flag;
      }
      named_sync(1, 128);
      const uint32_t vote = m.vote[p_it & 1][0] | m.vote[p_it & 1][1] | m.vote[p_it & 1][2] |
                            m.vote[p_it & 1][3];
      if (vote & 2u) { ok = false; break; }
      if (vote & 1u) {
        // rescaling O^T needs the previous tile's PV to have finished
        // (one barrier per stage: its phase lags tile p_it - 1 by at most one,
        // as the stage's reload for that tile waited for PV p_it - 1 - NS)
        const bool pv_done =
            mbar_wait(bar_addr(m.p_free[(p_it - 1) % NS]), ((p_it - 1) / NS) & 1, abort, kTimeoutNs);
        if (!named_sync_and(1, 128, pv_done)) { ok = false; break; }
        tc_fence_after();
        rescale_o(tq, m.alpha[p_it & 1], tp.npv);
      }
      // P = 2^(s cs - m), rounded as the MMAs will read it (bf16; two e4m3
      // terms for e4m3 caches); the sum takes the rounded values
      if constexpr (F8) {
        // P scaled by 2^kFxPLog2Scale as hi + lo, hi in e4m3 and lo in e5m2; the sum
        // takes the values the MMAs will read.  Token pair (8j + pair, + 1)
        // of head r: core matrix (r / 8, (8j + pair) / 16), row r % 8, byte
        // (8j + pair) % 16
        unsigned char *pst = smem + off_kv<F8>() + st * kFxStageBytes + 4 * kFxBlock;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float mref = MULTI && mnew[h] == -INFINITY ? 0.f : mnew[h] - kFxPLog2Scale;
          const float2 c2 = make_float2(cs, cs), m2 = make_float2(-mref, -mref);
          unsigned char *prow = pst + (row[h] >> 3) * kFxPSbo + (row[h] & 7) * 16 + pair;
          float2 lsum = make_float2(0.f, 0.f), xsum = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 arg = fma2(xp[2 * j + h], c2, m2);
            const float e0 = ex2(arg.x), e1 = ex2(arg.y);
            const uint16_t hi = float2_to_e4m3x2(e0, e1);
            const float2 bh = e4m3x2_to_float2(hi);
            const uint16_t lo = float2_to_e5m2x2(e0 - bh.x, e1 - bh.y);
            const float2 bl = e5m2x2_to_float2(lo);
            lsum = add2(lsum, add2(bh, bl));
            xsum = add2(xsum, make_float2(e0, e1));
            const int off = (j >> 1) * int(kFxPLbo) + 8 * (j & 1);
            *reinterpret_cast<uint16_t *>(prow + off) = hi;
            *reinterpret_cast<uint16_t *>(prow + kFxPTerm + off) = lo;
          }
          ellp[h] = ellp[h] * alpha[h] + (lsum.x + lsum.y);
          ellx[h] = ellx[h] * alpha[h] + (xsum.x + xsum.y);
          mrun[h] = mnew[h];
        }
        if (nv & 31) zero_value_tail_fx(smem + off_kv<F8>() + st * kFxStageBytes, nv, gt);
      } else {
        // bf16 P [head][token] in the stage's rope block, swizzled K-major:
        // each lane writes 4-byte token pairs
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          unsigned char *prow = smem + kOffKv + s * kStageBytes + kb_off<KBG>(8) +
                                (row[h] >> 3) * atom_stride<KBG>() + (row[h] & 7) * 128 + (lane & 3) * 4;
          // a row that has seen no token yet keeps a -inf max: its P is 0
          const float mref = MULTI && mnew[h] == -INFINITY ? 0.f : mnew[h];
          const float2 c2 = make_float2(cs, cs), m2 = make_float2(-mref, -mref);
          float2 lsum = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 arg = fma2(xp[2 * j + h], c2, m2);
            const float e0 = ex2(arg.x), e1 = ex2(arg.y);
            __nv_bfloat162 v = __floats2bfloat162_rn(e0, e1);
            const uint32_t bits = *reinterpret_cast<uint32_t *>(&v);
            lsum = add2(lsum, make_float2(__uint_as_float(bits << 16), __uint_as_float(bits & 0xffff0000u)));
            *reinterpret_cast<uint32_t *>(prow + ((j ^ (row[h] & 7)) << 4)) = bits;
          }
          ellp[h] = ellp[h] * alpha[h] + (lsum.x + lsum.y);
          mrun[h] = mnew[h];
        }
        // rows [nv, roundup16(nv)) of V are read by the last PV step but hold no
        // owned token (stale or unowned data): zero their 512 value dims
        if (nv & 15) zero_value_tail<KBG>(smem + kOffKv + s * kStageBytes, nv, gt);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(m.p_full[st]));
    }
    if (!ok) break;

    // the four lanes of a head hold parts of its sum
    float ell[2], elx[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      ell[h] = ellp[h] + __shfl_xor_sync(0xffffffffu, ellp[h], 1);
      ell[h] += __shfl_xor_sync(0xffffffffu, ell[h], 2);
      if (F8) {
        elx[h] = ellx[h] + __shfl_xor_sync(0xffffffffu, ellx[h], 1);
        elx[h] += __shfl_xor_sync(0xffffffffu, elx[h], 2);
      } else {
        elx[h] = ell[h];
      }
    }
    // ---- epilogue of this CTA's share of request v
    if ((lane & 3) == 0) {  // per-head output scale: kv_scale / sum (0 for a row that saw nothing)
      m.ell[row[0]] = !MULTI || ell[0] > 0.f ? p.kv_scale / ell[0] : 0.f;
      m.ell[row[1]] = !MULTI || ell[1] > 0.f ? p.kv_scale / ell[1] : 0.f;
    }
    const bool got_o = mbar_wait(bar_addr(m.o_full), o_it & 1, abort, kTimeoutNs);
    if (!named_sync_and(2, 128, got_o)) { ok = false; break; }
    tc_fence_after();
    const SplitInfo si = split_info(r, w.v, w.pv, w.tiles);
    const bool split = si.nsplits > 1;
    const size_t out_row0 = size_t(w.b) * p.heads + size_t(w.g) * kHeads;
    // This warp owns value dims 128c + 32q .. + 31 of each chunk c (its TMEM
    // lanes).  Values go through a 2 KB per-warp buffer, transposed to
    // [head][dim], so that each lane stores 16-byte runs of dims: 8 (bf16)
    // or 16 (fp32 slot) stores per chunk instead of 64.
    unsigned char *stg = m.stage_out[q];
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[4][16];
#pragma unroll
      for (int hb = 0; hb < 4; ++hb) tmem_ld16(tq + kColO + 64 * c + 16 * hb, o[hb]);
      tmem_wait_ld();
      const int d0 = 128 * c + 32 * q;
      if (!split) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // heads 32 half .. + 31
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int hb = 2 * half + hh;
            float sc[16];  // the block's 16 output scales, read before its stores
#pragma unroll
            for (int i = 0; i < 16; ++i) sc[i] = m.ell[16 * hb + i];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              reinterpret_cast<__nv_bfloat16 *>(stg)[(16 * hh + i) * 32 + lane] =
                  __float2bfloat16_rn(__uint_as_float(o[hb][i]) * sc[i]);
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // 32 heads x 4 runs of 8 dims
            const int k = lane + 32 * j, hl = k >> 2, part = k & 3, h = 32 * half + hl;
            const uint4 v = *reinterpret_cast<const uint4 *>(stg + k * 16);
            if (h < hn)
              *reinterpret_cast<uint4 *>(p.out + (out_row0 + h) * kDv + d0 + part * 8) = v;
          }
          __syncwarp();
        }
      } else {
        float *slot = slot_out_ptr(p) + size_t(si.slot) * kSlotHeads * kDv;
#pragma unroll
        for (int hb = 0; hb < 4; ++hb) {  // heads 16 hb .. + 15
          float sc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) sc[i] = m.ell[16 * hb + i];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            reinterpret_cast<float *>(stg)[i * 32 + lane] = __uint_as_float(o[hb][i]) * sc[i];
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // 16 heads x 8 runs of 4 dims
            const int k = lane + 32 * j, hl = k >> 3, part = k & 7, h = 16 * hb + hl;
            const uint4 v = *reinterpret_cast<const uint4 *>(stg + k * 16);
            // the merge reads it back after the rest of the KV stream
            if (h < hn) st_global_keep_l2(slot + size_t(h) * kDv + d0 + part * 4, v);
          }
          __syncwarp();
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(m.o_free));
    ++o_it;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if ((lane & 3) == 0 && row[h] < hn) {
        // (e4m3: the sum is of P scaled by 2^kFxPLog2Scale, before rounding)
        const float lse2 = mrun[h] + log2f(elx[h]) - (F8 ? kFxPLog2Scale : 0.f);
        if (!split)
          p.lse[out_row0 + row[h]] = lse_out(p, lse2);
        else
          slot_lse_ptr(p)[si.slot * kSlotHeads + row[h]] = lse2;
      }
    if (gt == 0) record_split(p, w.v, si);
  }
  if (!ok) atomicOr(err, kErrTimeout);
}

// ------------------------------------------------------------------ Q of an e4m3 cache
//
// Warps 9..11: once per request piece, after the previous piece's score
// MMAs have read Q, they read the piece's Q rows (bf16) from
// global memory, take 2^k with the largest |q| of the piece in [2^7, 2^8),
// and write hi = e4m3(2^k q) and lo = e4m3(2^k q - hi) into the two Q terms
// (rows past the request's heads are zero).  hi + lo equals 2^k q exactly
// down to 2^-2 (below that e4m3's subnormal step, 2^-9, bounds the error), so
// the scores keep bf16 Q's precision; 2^-k goes to the softmax through a
// slot tagged with the request.
// The largest |q| (as bf16 bits without the sign) of a piece's Q rows: the
// three warps' loads go out 16 at a time.  (Asking L2 to keep these lines
// for the split that reads them again measured slower: they crowd out the
// KV lines the other head group reads from L2.)
template <bool FUSED, int MULTI>
__device__ __forceinline__ uint32_t piece_q_max(const DecodeParams &p,
                                                const Walk<FUSED, MULTI, kPieceCostE4m3> &w,
                                                TcMisc<3> &m, int ct) {
  using namespace tc;
  constexpr int kRowChunks = kDqk / 8;
  const int hn = min(kHeads, p.heads - w.g * kHeads), n = hn * kRowChunks;
  const uint4 *qg =
      reinterpret_cast<const uint4 *>(p.q + (size_t(w.rb) * p.heads + size_t(w.g) * kHeads) * kDqk);
  uint32_t mx = 0;
  for (int i0 = ct; i0 < n; i0 += 16 * kConvThreads) {
    uint4 v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = i0 + u * kConvThreads;
      v[u] = i < n ? __ldg(qg + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      mx = __vmaxu2(mx, v[u].x & 0x7fff7fffu);
      mx = __vmaxu2(mx, v[u].y & 0x7fff7fffu);
      mx = __vmaxu2(mx, v[u].z & 0x7fff7fffu);
      mx = __vmaxu2(mx, v[u].w & 0x7fff7fffu);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, max(mx & 0xffffu, mx >> 16));
  if ((ct & 31) == 0) m.conv_max[ct >> 5] = mx;
  named_sync(3, kConvThreads);
  return max(m.conv_max[0], max(m.conv_max[1], m.conv_max[2]));
}

// Warps 9..11, once per request piece: the piece's largest |q| is taken
// while the previous piece runs (its rows are then in L2 as well); after the
// previous piece's score MMAs have read Q (q_empty), the rows are read again,
// 16 loads at a time, split and stored.
template <bool FUSED, int MULTI>
__device__ __forceinline__ void tc_split_q(const TcParams &tp, const CtaRange &r, TcMisc<3> &m,
                                           unsigned char *smem, int *err) {
  using namespace tc;
  const DecodeParams &p = tp.p;
  volatile int *abort = &m.abort;
  const int ct = int(threadIdx.x) - kConvWarp0 * 32;  // 0 .. 95
  const int lane = ct & 31;
  constexpr int kRowChunks = kDqk / 8;                // 72 chunks of 8 dims per row
  constexpr int kPer = kHeads * kRowChunks / kConvThreads;  // 48 chunks per thread
  static_assert(kHeads * kRowChunks % (16 * kConvThreads) == 0, "Q split batches");
  uint32_t q_it = 0;
  bool ok = true;
  Walk<FUSED, MULTI, kPieceCostE4m3> w(p, r), wa(p, r);  // wa: the piece after w
  bool ahead = wa.next();
  uint32_t mx = ahead ? piece_q_max(p, wa, m, ct) : 0u;
  if (ahead) {
    wa.advance();
    ahead = wa.next();
  }
  for (; w.next(); w.advance(), ++q_it) {
    const bool got = mbar_wait(bar_addr(m.q_empty), (q_it & 1) ^ 1, abort, kTimeoutNs);
    if (!named_sync_and(3, kConvThreads, got)) { ok = false; break; }
    const int hn = min(kHeads, p.heads - w.g * kHeads);
    const uint4 *qg =
        reinterpret_cast<const uint4 *>(p.q + (size_t(w.rb) * p.heads + size_t(w.g) * kHeads) * kDqk);
    // |q| bits are ordered like magnitudes; an Inf or NaN keeps k = 0
    int k = 0;
    if (mx < 0x7f80u) k = min(126, max(-126, 134 - int(mx >> 7)));
    const float sc = __int_as_float((127 + k) << 23);
#pragma unroll 1
    for (int u0 = 0; u0 < kPer; u0 += 16) {
      uint4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = ct + (u0 + u) * kConvThreads;
        v[u] = i / kRowChunks < hn ? __ldg(qg + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = ct + (u0 + u) * kConvThreads;
        const int rr = i / kRowChunks, c = i - kRowChunks * rr;
        const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t hw[2] = {0, 0}, lw[2] = {0, 0};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float f0 = __uint_as_float(wv[e] << 16) * sc, f1 = __uint_as_float(wv[e] & 0xffff0000u) * sc;
          const uint16_t h = float2_to_e4m3x2(f0, f1);
          const float2 bh = e4m3x2_to_float2(h);
          const uint16_t l = float2_to_e4m3x2(f0 - bh.x, f1 - bh.y);
          hw[e >> 1] |= uint32_t(h) << (16 * (e & 1));
          lw[e >> 1] |= uint32_t(l) << (16 * (e & 1));
        }
        // dims 8c .. 8c + 7: block c / 16, bytes 8 (c % 16) of the 128-byte
        // row, 16-byte chunk (c % 16) / 2 at its swizzled place
        const int b = c & 15;
        const int off = (c >> 4) * kFxBlock + (rr >> 3) * 1024 + (rr & 7) * 128 +
                        (((b >> 1) ^ (rr & 7)) << 4) + 8 * (b & 1);
        *reinterpret_cast<uint2 *>(smem + off) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2 *>(smem + kFxQTerm + off) = make_uint2(lw[0], lw[1]);
      }
    }
    if (ct == 0) {
      m.qinv[q_it & 3] = __int_as_float((127 - k) << 23);
      __threadfence_block();
      reinterpret_cast<volatile int *>(m.qinv_v)[q_it & 3] = w.v;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(m.q_ready));
    // the next piece's largest |q|, while this one runs
    mx = ahead ? piece_q_max(p, wa, m, ct) : 0u;
    if (ahead) {
      wa.advance();
      ahead = wa.next();
    }
  }
  if (!ok) atomicOr(err, kErrTimeout);
}

// ------------------------------------------------------------------ kernel

template <bool F8, bool FUSED, int MULTI, int AHEAD>
__global__ void __launch_bounds__(tc_threads<F8>(), 1)
    decode_tc_kernel(const __grid_constant__ TcParams tp, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_kv,
                     const __grid_constant__ CUtensorMap tm_kvg,
                     const __grid_constant__ CUtensorMap tm_kvb) {
  using namespace tc;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  unsigned char *smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  constexpr int NS = num_stages<F8>();
  TcMiscFor<F8> &m = *reinterpret_cast<TcMiscFor<F8> *>(smem + off_misc<F8>());
  const DecodeParams &p = tp.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int *err = error_word(p);
  constexpr int KBG = stage_kbg<F8, AHEAD>();

  // Q rows past the request's heads are read by the MMAs but never loaded:
  // they must hold finite values.  (P rows past them are written each tile.)
  for (int i = tid; i < off_kv<F8>() / 16; i += tc_threads<F8>())
    reinterpret_cast<uint4 *>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      for (int g = 0; g < kMaxGroups; ++g) mbar_init(bar_addr(m.kv_full[s][g]), 1);
      mbar_init(bar_addr(m.kv_empty[s]), 2);  // both PV issuers commit
      // one per stage: the softmax runs ahead of the PV issuers, and tile
      // k + NS (same stage) cannot reach the softmax before PV k has been
      // issued
      mbar_init(bar_addr(m.p_full[s]), 4);
      mbar_init(bar_addr(m.p_free[s]), 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_addr(m.s_full[b]), 2);  // both score issuers commit
      mbar_init(bar_addr(m.s_free[b]), 4);
    }
    mbar_init(bar_addr(m.q_full), 1);
    mbar_init(bar_addr(m.q_empty), 2);
    mbar_init(bar_addr(m.o_full), 2);
    mbar_init(bar_addr(m.o_free), 4);
    mbar_init(bar_addr(m.drain), 4);       // all four MMA issuers
    mbar_init(bar_addr(m.q_ready), 3);     // one arrival per Q-splitting warp
    for (int i = 0; i < 4; ++i) m.qinv_v[i] = -1;
    m.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&m.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
    if (F8 || KBG != kKb) tma_prefetch_desc(&tm_kvg);
    if (F8) tma_prefetch_desc(&tm_kvb);
  }
  // While the previous kernel finishes, pull the lengths and the head of the
  // block table into L2 (the KV stream of a previous call evicted them): a
  // hint that reads nothing back, so it may precede the wait below.
  if (warp == 2) {
    if (lane < min(32, (p.req_batch * 4 + 127) / 128))
      prefetch_l2(reinterpret_cast<const char *>(p.seq_lens) + 128 * lane);
    if (lane == 31) prefetch_l2(p.block_table);
  }
  fence_proxy_async_smem();
  // Launched as a programmatic dependent of the stream's previous kernel, so
  // that this prologue overlaps its tail: everything above touches only this
  // CTA's own resources.  Wait for that kernel's completion (and its writes)
  // before reading any input or writing any output.  (Releasing this
  // launch's own dependent, the split merge, early as well measured slower.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  write_empty_requests<MULTI>(p);
  cta_schedule<MULTI, piece_cost<F8>()>(p, &m.range, m.scratch);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;
  const CtaRange r = m.range;

  if (r.start < r.end) {
    const uint32_t sKv = sbase + off_kv<F8>();
    if (warp == 0) {
      tc_producer<F8, FUSED, MULTI, AHEAD>(tp, r, m, sbase + kOffQ, sKv, &tm_q, &tm_kv, &tm_kvg, &tm_kvb,
                                           err);
    } else if (warp == 1 || warp == 2) {
      if (lane == 0) tc_mma_s<F8, FUSED, MULTI, KBG>(tp, r, m, sbase + kOffQ, sKv, tmem, warp - 1, err);
    } else if (warp == 3 || warp == 8) {
      if (lane == 0) tc_mma_pv<F8, FUSED, MULTI, KBG>(tp, r, m, sKv, tmem, warp == 8, err);
    } else if (warp < 8) {
      tc_softmax<F8, FUSED, MULTI, KBG>(tp, r, m, smem, tmem, err);
    } else if constexpr (F8) {
      tc_split_q<FUSED, MULTI>(tp, r, m, smem, err);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t launch_split_merge(const DecodeParams &p, int grid, cudaStream_t stream);
cudaError_t launch_dcp_merge_combine(const DecodeParams &p, int grid, cudaStream_t stream);

template <bool F8, bool FUSED, int MULTI, int AHEAD>
static cudaError_t launch_tc(const TcParams &tp, const CUtensorMap &tm_q, const CUtensorMap &tm_kv,
                             const CUtensorMap &tm_kvg, const CUtensorMap &tm_kvb, int grid,
                             cudaStream_t stream) {
  static SmemLimitOnce smem_limit;
  const cudaError_t e = smem_limit.ensure(decode_tc_kernel<F8, FUSED, MULTI, AHEAD>, tc::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(tc_threads<F8>());
  cfg.dynamicSmemBytes = tc::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<F8, FUSED, MULTI, AHEAD>, tp, tm_q, tm_kv, tm_kvg,
                            tm_kvb);
}

// The variants of one cache dtype: one partition alone with P = 1 (a tile is
// one page: prefetch distance 1), one partition of P > 1, or all P partitions
// in one launch (distance 2); each with one query token or several, and the
// strided gather (one partition or all).
template <bool F8>
cudaError_t launch_tc_variants(const TcParams &tp, const CUtensorMap &tm_q,
                               const CUtensorMap &tm_kv, const CUtensorMap &tm_kvg,
                               const CUtensorMap &tm_kvb, int grid, cudaStream_t stream) {
  if (tp.p.strided)
    return tp.p.fused ? launch_tc<F8, true, 2, 2>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream)
                      : launch_tc<F8, false, 2, 2>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream);
  const bool multi = multi_rows(tp.p);
  if (tp.p.fused)
    return multi ? launch_tc<F8, true, true, 2>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream)
                 : launch_tc<F8, true, false, 2>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream);
  // (a bf16 tile of one page takes distance 1; e4m3 tiles always take 2)
  if (tp.p.num_parts == 1 && !F8)
    return multi ? launch_tc<F8, false, true, 1>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream)
                 : launch_tc<F8, false, false, 1>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream);
  return multi ? launch_tc<F8, false, true, 2>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream)
               : launch_tc<F8, false, false, 2>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream);
}

}  // namespace mla
