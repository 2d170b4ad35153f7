/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA absorbed paged-decode library.
 *
 * Operations, all from the decode-context-parallel (DCP) pages:
 *
 *  mla_decode_partial  one partition's attention over a paged latent KV cache,
 *                      returning the partition-local pair (out, lse).
 *                      sglang pull 33926 (trtllm_mla decode path gains DCP):
 *                      motivation (round-robin owner rule t mod P; a single-token
 *                      decode needs no causal bound), implementation step 3
 *                      (rank-local (out, lse); a rank owning nothing returns the
 *                      neutral (0, -inf)), step 4 (LSE in base 2 or base e).
 *  mla_kv_append       the write side: each request's new token row into the
 *                      paged cache (bf16, or quantised to e4m3 with the
 *                      per-tensor scale), only on the partition that owns it.
 *                      sglang pull 33926, implementation steps 3 (FP8 KV path)
 *                      and 4 (under DCP the fused KV write is off and the
 *                      pool's own write stores the rank's rows).
 *  mla_decode_dcp      all P partitions in one call (one decode launch for P <= 8)
 *                      and their merge: the DCP ranks emulated on one GPU.
 *  mla_lse_combine     the LSE-weighted softmax merge of P partial results.
 *                      sglang pull 33364 ([Attention][DCP] Add symm_a2a ...),
 *                      "Modifications", kernel 4 (wait_lse_combine_kernel), here
 *                      without the cross-GPU exchange: all partials are already
 *                      in one device buffer.
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers of the current CUDA device unless stated.
 *    The caller owns every buffer; the library never allocates, never frees
 *    and never synchronises the host.  Work is enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream).
 *  - The return value is a status: MLA_OK (0) or a negative MLA_ERR_* code.
 *    Argument errors are detected on the host before anything is launched,
 *    and the outputs are then left untouched.  MLA_ERR_CUDA carries the CUDA
 *    error text in mla_last_cuda_error().
 *  - Calls are thread-compatible: concurrent calls must use distinct
 *    workspaces.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mla_stream_t; /* == cudaStream_t */

enum mla_status {
  MLA_OK = 0,
  MLA_ERR_NULL = -1,      /* a required pointer is NULL                           */
  MLA_ERR_SHAPE = -2,     /* unsupported size: q_len outside 1..16 (or > 1 off the
                             tensor-core path), Dqk != 576, Dv != 512,
                             page_size != 64, heads not in [1, 128], ...          */
  MLA_ERR_PARTITION = -3, /* num_parts < 1 or part_id outside [0, num_parts)      */
  MLA_ERR_ALIGN = -4,     /* q / kv_pages / out / partials not 16-byte aligned,
                             workspace not 256-byte aligned                       */
  MLA_ERR_WORKSPACE = -5, /* workspace smaller than mla_decode_workspace_size()   */
  MLA_ERR_ARG = -6,       /* bad enum value, non-finite scale, negative size      */
  MLA_ERR_CUDA = -7,      /* a CUDA call failed; see mla_last_cuda_error()        */
  MLA_ERR_DEVICE = -8,    /* current device is not an sm_103 GPU                  */
  MLA_ERR_BOUNDS = -9,    /* (from mla_decode_check_workspace) the kernel met a
                             block-table entry outside [0, num_pages) or a sequence
                             length outside [0, 64 * max_pages_per_seq]            */
  MLA_ERR_TIMEOUT = -10   /* (from mla_decode_check_workspace) a bounded wait
                             inside the kernel gave up; outputs are unspecified   */
};

enum mla_lse_base {
  MLA_LSE_NATURAL = 0, /* lse = ln(sum_j exp(s_j))                                */
  MLA_LSE_BASE2 = 1    /* lse = log2(sum_j exp(s_j)) = natural * log2(e)          */
};

enum mla_kv_dtype {
  MLA_KV_BF16 = 0, /* cache rows are bf16                                         */
  MLA_KV_E4M3 = 1  /* cache rows are OCP FP8 e4m3, value = e4m3 * kv_scale        */
};

/* Sizes that the ten named arguments of mla_decode_partial leave implicit. */
typedef struct mla_decode_desc {
  int32_t batch;             /* B, number of requests (0 is a no-op)              */
  int32_t num_heads;         /* H, query heads per request, 1..128                */
  int32_t q_len;             /* query tokens per request, 1..16 (see below)       */
  int32_t head_dim_qk;       /* must be 576 (512 latent + 64 rope)                */
  int32_t head_dim_v;        /* must be 512 (the latent)                          */
  int32_t page_size;         /* tokens per cache page; must be 64                 */
  int32_t num_pages;         /* physical pages in kv_pages (>= 1)                 */
  int32_t max_pages_per_seq; /* entries per block_table row (>= 1)                */
  int32_t kv_dtype;          /* enum mla_kv_dtype                                 */
  float kv_scale;            /* per-tensor dequant scale for E4M3 (> 0, finite)   */
} mla_decode_desc;

/*
 * Bytes of scratch workspace mla_decode_partial needs for `d` on a GPU with
 * `num_sms` SMs (num_sms <= 0: ask the current device).  Returns 0 if `d` is
 * NULL or invalid.  The workspace holds a device error word, per-request
 * split records and the fp32 partial results of requests split across CTAs.
 * Its first 256 bytes (the error word) must be zero before the first call;
 * everything else is rewritten by each call before it is read.
 */
size_t mla_decode_workspace_size(const mla_decode_desc *d, int num_sms);

/*
 * Partition `part_id` of `num_parts` of MLA absorbed decode attention.
 *
 *  q           bf16 [B, q_len, H, 576], contiguous.  Dims 0..511 latent, 512..575 rope.
 *  kv_pages    [num_pages, 64, 576] rows of the GLOBAL paged cache, contiguous,
 *              bf16 or e4m3 bytes per d->kv_dtype.  Row dims 0..511 are also
 *              the value (the latent).
 *  block_table int32 [B, max_pages_per_seq]: logical page i of request b lives
 *              in physical page block_table[b][i].  Entries past the request's
 *              last page are never read.
 *  seq_lens    int32 [B]: GLOBAL sequence lengths L_b (tokens 0..L_b-1 exist).
 *  part_id, num_parts
 *              the partition attends exactly to the global tokens t < L_b with
 *              t mod num_parts == part_id (round-robin owner rule).  A real DCP
 *              rank holding a compacted local cache is num_parts = 1 over its
 *              local pages and local lengths.
 *  sm_scale    softmax scale applied to q.k (finite).
 *  lse_base    enum mla_lse_base of the returned lse.
 *  out         bf16 [B, q_len, H, 512]: softmax(sm_scale q K^T) V over the owned
 *              tokens, rounded to nearest even.  All of it is written.
 *  lse         fp32 [B, q_len, H]: log-sum-exp of the scaled scores in `lse_base`.
 *              A request for which the partition owns no token gets out = 0 and
 *              lse = -inf (the neutral pair of the LSE merge).
 *  workspace   scratch of >= mla_decode_workspace_size(d, 0) bytes, 256-byte
 *              aligned, its first 256 bytes zero before first use (see above).
 *
 * Enqueues two kernels on `stream`: the decode kernel and the merge of the
 * requests its schedule split across SMs.  The tensor-core kernel serves
 * every num_parts with num_parts / gcd(num_parts, 8) <= 16.  For num_parts
 * dividing 8 it reads exactly the partition's rows.  For num_parts in
 * {3, 5, 6, 7} it does so too, through a TMA traversal stride of num_parts
 * rows.  Otherwise it gathers partition
 * part_id mod g of g = gcd(num_parts, 8) and drops the tokens the other
 * partitions own (reading num_parts / g times the partition's own bytes).
 * Larger ratios run a CUDA-core kernel.
 *
 * Arithmetic (tensor-core path): fp32 accumulation throughout.  A bf16
 * cache is multiplied as stored by bf16 q and by the softmax weights rounded
 * to bf16.  An e4m3 cache is also multiplied as stored, by e4m3 MMAs:
 *  - q enters as two e4m3 terms of 2^k q, exact for elements down to 2^-9
 *    of the largest |q| of the request's 64-row head group;
 *  - the weights enter as an e4m3 term plus an e5m2 term, relative error
 *    <= 2^-7 for weights down to 2^-6 of the running maximum, 2 to 3 bits
 *    below that; weights below 2^-16 of it drop out of `out`;
 *  - `out` is normalised by the weights as multiplied, and `lse` by their
 *    unrounded sum.
 *
 * Several query tokens (q_len = T > 1; tensor-core path only, else
 * MLA_ERR_SHAPE): the request's queries are its last T tokens, and query
 * token i attends causally to the owned tokens t < L_b - T + i + 1; a query
 * row that sees no owned token gets the neutral pair.
 * Block-table entries outside [0, num_pages) and lengths outside
 * [0, 64 * max_pages_per_seq] are not dereferenced: the kernel skips them and
 * records MLA_ERR_BOUNDS in the workspace (read it with
 * mla_decode_check_workspace); the affected outputs are then unspecified.
 * Outputs are bitwise deterministic for fixed inputs and device.
 */
int mla_decode_partial(const void *q, const void *kv_pages, const int32_t *block_table,
                       const int32_t *seq_lens, int part_id, int num_parts, float sm_scale,
                       int lse_base, void *out, float *lse, const mla_decode_desc *d,
                       void *workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * All partitions of a DCP decode in one call: the partial results of every
 * partition r = 0..num_parts-1 (each exactly what mla_decode_partial with
 * part_id = r returns, up to the rounding order of requests split across
 * SMs) and their LSE-weighted merge.  On the pages each DCP rank returns its
 * partition-local (out, lse) and the ranks' results are merged at the
 * attention output (sglang pull 33926, implementation step 3; pull 33364,
 * "Modifications", kernel 4); this call emulates all the ranks on one GPU.
 *
 *  q, kv_pages, block_table, seq_lens, sm_scale, lse_base, d
 *              as for mla_decode_partial.
 *  partials     bf16 [num_parts, B, 1, H, 512]: partition r's out.
 *  partial_lses fp32 [num_parts, B, 1, H] in lse_base: partition r's lse
 *               (-inf where it owns no token of the request).
 *  out          bf16 [B, 1, H, 512]: the merge over the partitions (as
 *               mla_lse_combine computes it from partials / partial_lses).
 *  out_lse      optional fp32 [B, 1, H]: the merged lse, or NULL.
 *  workspace    >= mla_decode_dcp_workspace_size(d, num_parts, 0) bytes, same
 *               rules as for mla_decode_partial.
 *
 * 2 <= num_parts <= 8: one decode launch covers every (partition, request)
 * pair, then one kernel merges the requests the decode's schedule split
 * across SMs and combines the partitions (two kernels).  num_parts = 1 and
 * num_parts > 8 (up to 256): one mla_decode_partial call per partition, then
 * the combine (for one partition a copy of its result).  Errors and bounds reporting as for mla_decode_partial.
 */
size_t mla_decode_dcp_workspace_size(const mla_decode_desc *d, int num_parts, int num_sms);

int mla_decode_dcp(const void *q, const void *kv_pages, const int32_t *block_table,
                   const int32_t *seq_lens, int num_parts, float sm_scale, int lse_base,
                   void *partials, float *partial_lses, void *out, float *out_lse,
                   const mla_decode_desc *d, void *workspace, size_t workspace_bytes,
                   mla_stream_t stream);

/*
 * mla_decode_partial without a workspace argument.  The method on the pages
 * has no counterpart of this call: it exists for callers that cannot call
 * cudaMalloc -- runtimes that give every byte of HBM to their own KV-cache
 * pool and let no library allocate, decode loops that cannot absorb the
 * device synchronisation an allocation may cause, and plain-C hosts with no
 * allocator of their own.
 *
 * Same arguments, layouts and results as mla_decode_partial, for one query
 * token per request (q_len = 1; other values return MLA_ERR_SHAPE).  Its scratch is
 * a ~40 MB array built into the library, which every GPU that loads the
 * library keeps until the process exits; it calls no cudaMalloc, cudaFree or
 * other allocating routine.  The first call on a device takes that device's
 * address of the array (the device must be current), so make that first call
 * before any stream capture.  Limit: batch * ceil(num_heads / 32) <= 16384;
 * larger batches return MLA_ERR_WORKSPACE without launching.  All calls share
 * the one array: calls that may overlap on the GPU (different streams, or
 * different host threads) race and must be serialised by the caller.  Each
 * call clears the array's error word before its kernels; kernel-side bounds
 * errors are not reported by this variant (use mla_decode_partial with
 * mla_decode_check_workspace to diagnose them).  The kernels are those of
 * mla_decode_partial (tensor cores whenever num_parts / gcd(num_parts, 8)
 * <= 16, else the CUDA-core kernel) on at most 152 CTAs, the number of split
 * partials the array holds: on a GPU with at most 152 SMs the outputs equal
 * mla_decode_partial's bit for bit; with more SMs the split points differ,
 * and so may the rounding of requests cut across CTAs.
 */
int mla_decode_partial_noalloc(const void *q, const void *kv_pages, const int32_t *block_table,
                               const int32_t *seq_lens, int part_id, int num_parts,
                               float sm_scale, int lse_base, void *out, float *lse,
                               const mla_decode_desc *d, mla_stream_t stream);

/*
 * 1 if the library's kernels run on a GPU of compute capability
 * major.minor (they are built for sm_103a only), else 0.  Every entry point
 * that launches returns MLA_ERR_DEVICE on a device this refuses, before
 * launching anything.
 */
int mla_arch_supported(int major, int minor);

/*
 * Self-test of the bounded waits every kernel here uses (no GPU fault
 * involved): launches one CTA whose two warps wait on shared-memory barriers
 * that nothing completes.  Warp 0 gives up after `timeout_ns` (1 us .. 0.1 s)
 * and raises the CTA's abort flag; warp 1, whose own limit is ten times
 * longer, must give up as soon as it sees the flag.  Each warp that gave up
 * sets bit 8 + warp of the workspace's error word, and MLA_ERR_TIMEOUT is
 * reported by mla_decode_check_workspace, which also clears the word.
 *
 *  workspace   any decode workspace (256-byte aligned); only its error word
 *              is written.
 *
 * Returns MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_ARG (timeout out of range),
 * MLA_ERR_CUDA, or MLA_OK once the kernel is enqueued.
 */
int mla_selftest_bounded_wait(void *workspace, int64_t timeout_ns, mla_stream_t stream);

/*
 * Waits for `stream`, reads and clears the device error word of `workspace`.
 * Returns MLA_OK, MLA_ERR_TIMEOUT, MLA_ERR_BOUNDS, or MLA_ERR_CUDA.  (The one call that
 * synchronises; meant for tests and debugging.)
 */
int mla_decode_check_workspace(void *workspace, mla_stream_t stream);

/*
 * Append: writes the new token's cache row of every request (sglang pull
 * 33926, implementation steps 3 and 4; see the top of this file).
 *
 *  kv_new      bf16 [B, 576], contiguous: the new token's latent (dims 0..511)
 *              and rope (512..575) per request, as the model produced them.
 *  kv_pages    the GLOBAL paged cache, [num_pages, 64, 576] bf16 or e4m3 per
 *              d->kv_dtype (written in place).
 *  block_table int32 [B, max_pages_per_seq], as for mla_decode_partial.
 *  positions   int32 [B]: global index t of each request's new token (its
 *              length before the append).  Row t lands in physical page
 *              block_table[b][t / 64], row t % 64.  t < 0 skips the request.
 *  part_id, num_parts
 *              only tokens the partition owns (t mod num_parts == part_id) are
 *              written: each DCP rank stores its own rows.  num_parts = 1
 *              writes every request's row.
 *  d           the decode descriptor of the cache: batch, head_dim_qk (576),
 *              page_size (64), num_pages, max_pages_per_seq, kv_dtype and, for
 *              E4M3, kv_scale; num_heads, q_len and head_dim_v are not used.
 *  error_word  optional device int32: a row whose logical page is past
 *              max_pages_per_seq or whose block-table entry is outside
 *              [0, num_pages) is skipped (never written) and bit 0 is OR-ed in.
 *              NULL: such rows are skipped silently.
 *
 * A bf16 cache receives the row bits unchanged.  An e4m3 cache receives, per
 * value, fp32(x) / kv_scale (an IEEE fp32 division) rounded to the nearest
 * e4m3 value, ties to even, magnitudes past 448 saturated to +-448 (NaN
 * inputs give an e4m3 NaN).  Rows of different requests must not alias (two
 * requests writing the same page row race).  Enqueues one kernel on `stream`;
 * batch 0 enqueues nothing.
 */
int mla_kv_append(const void *kv_new, void *kv_pages, const int32_t *block_table,
                  const int32_t *positions, int part_id, int num_parts,
                  const mla_decode_desc *d, int32_t *error_word, mla_stream_t stream);

/* Sizes of the DCP rank metadata. */
typedef struct mla_dcp_meta_desc {
  int32_t batch;              /* B requests (0 is a no-op)                         */
  int32_t num_req_slots;      /* rows of req_to_token (>= 1)                       */
  int32_t req_to_token_width; /* token slots per row of req_to_token (>= 1)        */
  int32_t max_pages_per_seq;  /* columns of block_table (>= 1)                     */
  int32_t extra_tokens;       /* added to every global length: the draft tokens of
                                 a target-verify step, 0 for decode (>= 0)         */
  int32_t pad_value;          /* block_table entries past a request's pages        */
  int32_t page_size;          /* must be 64                                        */
} mla_dcp_meta_desc;

/*
 * A DCP rank's per-step decode metadata, built on the device (sglang pull
 * 33926, implementation step 1 and the code of _apply_dcp_cuda_graph_metadata:
 * each step writes the global and the rank-local lengths into buffers that a
 * captured CUDA graph keeps reading, then rebuilds the page table over the
 * rank's own slice).  For partition part_id of num_parts and every request b:
 *
 *  global_lens[b] = seq_lens[b] + d->extra_tokens
 *  local_lens[b]  = tokens of global_lens[b] the partition owns
 *                   (t mod num_parts == part_id)
 *  block_table[b][i] = req_to_token[req_pool_indices[b]][64 i] / 64 for the
 *                   request's ceil(local_lens[b] / 64) local pages, then
 *                   d->pad_value up to max_pages_per_seq.
 *
 * req_to_token (int32 [num_req_slots, req_to_token_width]) gives, for a
 * request's j-th LOCAL token, its slot in the rank's compact pool (slot / 64
 * = pool page, slot % 64 = row).  With these, mla_decode_partial(num_parts =
 * 1) over the rank's compact pool with local_lens and block_table returns the
 * rank's (out, lse) -- the same result as the partition of the global cache.
 *
 * A request with a negative global length (local length 0), a pool index
 * outside req_to_token, or more pages than max_pages_per_seq or the width of
 * req_to_token gets a table row of pad_value; a negative slot gives
 * pad_value for its page; either ORs bit 0 into the optional device
 * `error_word`.  All outputs are device int32 arrays written in full; the
 * call allocates nothing and enqueues one kernel.
 */
int mla_dcp_local_metadata(const int32_t *seq_lens, const int32_t *req_pool_indices,
                           const int32_t *req_to_token, int part_id, int num_parts,
                           const mla_dcp_meta_desc *d, int32_t *global_lens,
                           int32_t *local_lens, int32_t *block_table, int32_t *error_word,
                           mla_stream_t stream);

/* Sizes of an LSE combine. */
typedef struct mla_combine_desc {
  int32_t num_tokens; /* T (0 is a no-op)                                         */
  int32_t num_heads;  /* H >= 1                                                   */
  int32_t head_dim;   /* D, a multiple of 8 in [8, 1024]                          */
  int32_t lse_base;   /* enum mla_lse_base of `lses` and of `out_lse`             */
  float *out_lse;     /* optional fp32 [T, H] merged lse (device), or NULL        */
} mla_combine_desc;

/*
 * LSE-weighted merge of `num_parts` partial attention results.
 *
 *  partials  bf16 [num_parts, T, H, D], contiguous.
 *  lses      fp32 [num_parts, T, H] in base d->lse_base; -inf marks a partition
 *            that owned no token (its partial is ignored).
 *  out       bf16 [T, H, D]:  sum_p w_p o_p / sum_p w_p with
 *            w_p = base^(lse_p - max_p lse_p).  Rows whose partitions are all
 *            -inf get out = 0 (and out_lse = -inf), never NaN.
 */
int mla_lse_combine(const void *partials, const float *lses, int num_parts, void *out,
                    const mla_combine_desc *d, mla_stream_t stream);

/* Static text for a status code. */
const char *mla_status_string(int status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char *mla_last_cuda_error(void);

/* Library version as 10000 * major + 100 * minor + patch. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
