// Host side of the C ABI declared in include/mla_decode.h: argument checks,
// workspace sizing, per-device facts, and kernel dispatch.  Nothing here
// allocates device memory or synchronises the host (except the explicit
// mla_decode_check_workspace).
#include "mla_decode.h"

#include <cuda.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace mla {
cudaError_t launch_decode_simt(const DecodeParams &p, int grid, cudaStream_t stream);
cudaError_t launch_dcp_metadata(const int32_t *seq_lens, const int32_t *req_pool_indices,
                                const int32_t *req_to_token, int batch, int r2t_rows,
                                int r2t_width, int extra, int part_id, int num_parts,
                                int32_t *global_lens, int32_t *local_lens, int32_t *table,
                                int max_pages, int32_t pad, int32_t *error_word,
                                cudaStream_t stream);
cudaError_t launch_kv_append(const void *kv_new, void *kv_pages, const int32_t *block_table,
                             const int32_t *positions, int batch, int part_id, int num_parts,
                             int num_pages, int max_pages, int e4m3, float kv_scale,
                             int32_t *error_word, cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeParams &p, int npv, int q_rows, int groups_per_page,
                             const CUtensorMap &tm_q, const CUtensorMap &tm_kv,
                             const CUtensorMap &tm_kvg, const CUtensorMap &tm_kvb, int grid,
                             cudaStream_t stream);
cudaError_t launch_lse_combine(const void *partials, const float *lses, int num_parts, void *out,
                               float *out_lse, int rows, int dim, int base2, cudaStream_t stream);
int combine_max_parts();
}  // namespace mla

namespace {

thread_local char g_cuda_error[256] = "";

int cuda_fail(cudaError_t e) {
  std::snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

struct DeviceFacts {
  int sms = 0;
  int major = 0, minor = 0;
};

constexpr int kMaxDevices = 64;
DeviceFacts g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Facts of the current device; status in *st.
DeviceFacts current_device(int *st, int *dev_out = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = cuda_fail(e);
    return {};
  }
  if (dev_out) *dev_out = dev;
  if (dev < 0 || dev >= kMaxDevices) {
    *st = MLA_ERR_DEVICE;
    return {};
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceFacts &f = g_dev[dev];
  if (f.sms == 0) {
    int sms = 0, mj = 0, mn = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&mj, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&mn, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) {
      *st = cuda_fail(e);
      return {};
    }
    f.sms = sms;
    f.major = mj;
    f.minor = mn;
  }
  *st = mla_arch_supported(f.major, f.minor) ? MLA_OK : MLA_ERR_DEVICE;
  return f;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link the driver library directly).
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  });
  return fn;
}

int tensor_map_fail(const char *what, CUresult r) {
  std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled(%s) failed: %d", what,
                int(r));
  return MLA_ERR_CUDA;
}

constexpr int kTcHeadsPerGroup = 64;

// The tensor-core kernel reads exactly a partition's rows when they form whole
// 8-row groups of a page (P | 8), or through the strided gather below.
// Otherwise it gathers partition r mod g of g = gcd(P, 8) (g divides
// a page's 8 atoms) and, when g < P, drops the tokens other partitions own:
// it reads P / g times the partition's own bytes at the tensor-core rate,
// which beats the CUDA-core kernel while P / g stays small.
int gather_parts(int num_parts) {
  int g = 8, a = num_parts;
  while (a) { const int t = g % a; g = a; a = t; }
  return g;
}
constexpr int kMaxOwnerRatio = 16;  // P / gather_parts(P) served by the tensor cores

bool tensor_core_path(const mla_decode_desc *, int num_parts) {
  return num_parts >= 1 && num_parts / gather_parts(num_parts) <= kMaxOwnerRatio;
}

// P in {3, 5, 6, 7}: the tensor-core kernel gathers exactly the partition's
// rows, with a TMA traversal stride of P rows (at most 8), `strided_apg(P)`
// atoms of 8 rows per page, for bf16 and e4m3 caches and any q_len.  Other P
// not dividing 8 take the owner mask.
bool strided_path(const mla_decode_desc *, int num_parts) {
  return num_parts > 1 && num_parts < 8 && 8 % num_parts != 0;
}
int strided_apg(int num_parts) {
  const int rows = (mla::kPage + num_parts - 1) / num_parts;  // a partition's rows of a page, at most
  return (rows + 7) / 8;
}

// all partitions in one decode launch: P divides 8 (no owner mask), or the
// strided gather
bool fused_path(const mla_decode_desc *d, int num_parts) {
  return num_parts >= 1 && (8 % num_parts == 0 || strided_path(d, num_parts));
}

// Q as [B*H rows, 576] bf16, one 64-column swizzled box of min(64, H) rows;
// partition rows of a bf16 cache as a 5-D view (64 dims, 8 rows of stride P,
// 9 blocks of 64 dims, groups of 8 rows, partitions), one box = one page's
// owned rows; of an e4m3 cache as a 3-D view (576 bytes, rows of stride P,
// partitions), one swizzled box = 128 dims of one page's 64/P owned rows,
// with an unswizzled view of whole 576-byte rows for the L2 prefetch.  The
// strided gather's maps take an atom's rows through a traversal stride P.
// For one partition (`part_id`) the base is offset to its
// first row and the partition dimension is left off (4-D / 2-D maps, the
// faster boxes); for all P partitions (`all_parts`) it is added, with a stride
// of one row (5-D / 3-D maps, coordinate r).
int make_tensor_maps(const void *q, const void *kv, const mla_decode_desc *d, int part_id,
                     int num_parts, bool all_parts, bool strided, CUtensorMap *tm_q,
                     CUtensorMap *tm_kv, CUtensorMap *tm_kvg, CUtensorMap *tm_kvb) {
  EncodeTiled enc = encode_tiled();
  if (!enc) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled unavailable");
    return MLA_ERR_CUDA;
  }
  const cuuint64_t row = cuuint64_t(mla::kDqk) * 2;
  {
    const cuuint64_t qrows = cuuint64_t(d->q_len) * cuuint64_t(d->num_heads);
    cuuint64_t dims[2] = {cuuint64_t(mla::kDqk), cuuint64_t(d->batch) * qrows};
    cuuint64_t strides[1] = {row};
    cuuint32_t box[2] = {64, cuuint32_t(qrows < 64 ? qrows : 64)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("q", r);
  }
  if (d->kv_dtype == MLA_KV_E4M3 && strided) {
    // (144 words of 4 fp8 values, 64 page rows, pages): one box is one atom,
    // raw rows c, c + P, ..., c + 7P of a page (traversal stride P), landing
    // as 8 consecutive 576-byte rows; rows past the page read as zeros
    const cuuint32_t P = cuuint32_t(num_parts);
    const cuuint64_t row8 = cuuint64_t(mla::kDqk);
    cuuint64_t dims[3] = {row8 / 4, cuuint64_t(mla::kPage), cuuint64_t(d->num_pages)};
    cuuint64_t strides[2] = {row8, cuuint64_t(mla::kPage) * row8};
    cuuint32_t box[3] = {cuuint32_t(row8 / 4), 8 * P, 1};
    cuuint32_t es[3] = {1, P, 1};
    CUresult r = enc(tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(kv), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv e4m3 strided", r);
    // block 4 of the kernel's loads (the box above serves the L2 prefetch):
    // (576 bytes, 64 page rows, pages), a box of dims 512..575 of an atom's
    // rows c, c + P, ..., c + 7P with the 64-byte swizzle
    cuuint64_t fdims[3] = {row8, cuuint64_t(mla::kPage), cuuint64_t(d->num_pages)};
    cuuint64_t fstrides[2] = {row8, cuuint64_t(mla::kPage) * row8};
    cuuint32_t fbox[3] = {64, 8 * P, 1};
    r = enc(tm_kvg, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(kv), fdims, fstrides, fbox, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv e4m3 strided blocks", r);
    // blocks 0..3 of an atom in one box, landing [block][8 rows][128 B]:
    // (128 bytes, 64 page rows, 4 blocks, pages)
    cuuint64_t gdims[4] = {128, cuuint64_t(mla::kPage), 4, cuuint64_t(d->num_pages)};
    cuuint64_t gstrides[3] = {row8, 128, cuuint64_t(mla::kPage) * row8};
    cuuint32_t gbox[4] = {128, 8 * P, 4, 1};
    cuuint32_t ges[4] = {1, P, 1, 1};
    r = enc(tm_kvb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(kv), gdims, gstrides, gbox, ges,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv e4m3 strided grouped blocks", r);
  } else if (d->kv_dtype == MLA_KV_E4M3) {
    const cuuint64_t P = cuuint64_t(num_parts);
    const cuuint32_t R = cuuint32_t(mla::kPage / num_parts);
    const cuuint64_t row8 = cuuint64_t(mla::kDqk);
    const char *base = static_cast<const char *>(kv) + (all_parts ? 0 : size_t(part_id) * row8);
    cuuint64_t dims[3] = {row8 / 4, cuuint64_t(d->num_pages) * R, P};
    cuuint64_t strides[2] = {P * row8, row8};
    cuuint32_t box[3] = {cuuint32_t(row8 / 4), R, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT32, all_parts ? 3 : 2,
                     const_cast<char *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv e4m3", r);
    // block 4 of the kernel's loads (the box above serves the L2 prefetch):
    // (576 bytes, owned rows, partitions), a box of dims 512..575 of a page's
    // 64/P owned rows with the 64-byte swizzle
    cuuint64_t fdims[3] = {row8, cuuint64_t(d->num_pages) * R, P};
    cuuint64_t fstrides[2] = {P * row8, row8};
    cuuint32_t fbox[3] = {64, R, 1};
    r = enc(tm_kvg, CU_TENSOR_MAP_DATA_TYPE_UINT8, all_parts ? 3 : 2, const_cast<char *>(base), fdims,
            fstrides, fbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv e4m3 blocks", r);
    {
      // blocks 0..3 of a page's owned atoms in one box, landing
      // [atom][block][8 rows][128 B]: (128 bytes, 8 rows, 4 blocks, 8-row
      // atoms, partitions)
      const cuuint64_t G = 8 / P;
      cuuint64_t gdims[5] = {128, 8, 4, cuuint64_t(d->num_pages) * G, P};
      cuuint64_t gstrides[4] = {P * row8, 128, 8 * P * row8, row8};
      cuuint32_t gbox[5] = {128, 8, 4, cuuint32_t(G), 1};
      cuuint32_t ges[5] = {1, 1, 1, 1, 1};
      r = enc(tm_kvb, CU_TENSOR_MAP_DATA_TYPE_UINT8, all_parts ? 5 : 4, const_cast<char *>(base), gdims,
              gstrides, gbox, ges, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return tensor_map_fail("kv e4m3 grouped blocks", r);
    }
  } else if (strided) {
    // (64 dims, 64 page rows, 9 blocks of 64 dims, pages): one box is one
    // atom, rows c, c + P, ..., c + 7P of a page (traversal stride P), which
    // lands as [9 blocks][8 rows][128 B]; rows past the page are out of
    // bounds and read as zeros.  The partition is in the row coordinate.
    const cuuint32_t P = cuuint32_t(num_parts);
    cuuint64_t dims[4] = {64, cuuint64_t(mla::kPage), cuuint64_t(mla::kDqk / 64),
                          cuuint64_t(d->num_pages)};
    cuuint64_t strides[3] = {row, 128, cuuint64_t(mla::kPage) * row};
    cuuint32_t box[4] = {64, 8 * P, cuuint32_t(mla::kDqk / 64), 1};
    cuuint32_t es[4] = {1, P, 1, 1};
    CUresult r = enc(tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(kv), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv strided", r);
    *tm_kvg = *tm_kv;  // unused: one column group
  } else {
    const cuuint64_t P = cuuint64_t(num_parts);
    const cuuint32_t G = cuuint32_t(8 / num_parts);
    const char *base = static_cast<const char *>(kv) + (all_parts ? 0 : size_t(part_id) * row);
    cuuint64_t dims[5] = {64, 8, cuuint64_t(mla::kDqk / 64), cuuint64_t(d->num_pages) * G, P};
    cuuint64_t strides[4] = {P * row, 128, 8 * P * row, row};
    cuuint32_t box[5] = {64, 8, cuuint32_t(mla::kDqk / 64), G, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, all_parts ? 5 : 4,
                     const_cast<char *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv", r);
    // one column group (3 of the 9 dim blocks) of a page's atoms: the
    // kernel's loads when a tile is one page (P = 1); the full-page box above
    // serves the L2 prefetch and the loads of P > 1
    box[2] = 3;
    r = enc(tm_kvg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, all_parts ? 5 : 4, const_cast<char *>(base),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return tensor_map_fail("kv column group", r);
  }
  if (d->kv_dtype != MLA_KV_E4M3) *tm_kvb = *tm_kv;  // unused: only e4m3 caches take grouped boxes
  return MLA_OK;
}

constexpr int kSimtHeadsPerGroup = 32;
// Query tokens per request: several (multi-token prediction / target verify)
// only on the tensor-core path; the CUDA-core kernel takes one.
constexpr int kMaxQLen = 16;

int check_desc(const mla_decode_desc *d) {
  if (!d) return MLA_ERR_NULL;
  if (d->batch < 0 || d->num_pages < 1 || d->max_pages_per_seq < 1) return MLA_ERR_SHAPE;
  if (d->q_len < 1 || d->q_len > kMaxQLen) return MLA_ERR_SHAPE;
  if (d->head_dim_qk != mla::kDqk || d->head_dim_v != mla::kDv) return MLA_ERR_SHAPE;
  if (d->page_size != mla::kPage) return MLA_ERR_SHAPE;
  if (d->num_heads < 1 || d->num_heads > 128) return MLA_ERR_SHAPE;
  if (d->kv_dtype != MLA_KV_BF16 && d->kv_dtype != MLA_KV_E4M3) return MLA_ERR_ARG;
  if (d->kv_dtype == MLA_KV_E4M3 && !(std::isfinite(d->kv_scale) && d->kv_scale > 0.f))
    return MLA_ERR_ARG;
  return MLA_OK;
}

// The fields of a decode descriptor that describe the cache itself.
int check_cache_desc(const mla_decode_desc *d) {
  if (!d) return MLA_ERR_NULL;
  if (d->batch < 0 || d->num_pages < 1 || d->max_pages_per_seq < 1) return MLA_ERR_SHAPE;
  if (d->head_dim_qk != mla::kDqk || d->page_size != mla::kPage) return MLA_ERR_SHAPE;
  if (d->kv_dtype != MLA_KV_BF16 && d->kv_dtype != MLA_KV_E4M3) return MLA_ERR_ARG;
  if (d->kv_dtype == MLA_KV_E4M3 && !(std::isfinite(d->kv_scale) && d->kv_scale > 0.f))
    return MLA_ERR_ARG;
  return MLA_OK;
}

// Rows of one request: q_len query tokens x num_heads heads.
int rows_of(const mla_decode_desc *d) { return d->q_len * d->num_heads; }

int head_groups_of(const mla_decode_desc *d) {
  return (rows_of(d) + kSimtHeadsPerGroup - 1) / kSimtHeadsPerGroup;
}

// Builds the decode parameters and enqueues the decode kernel and its split
// merge (arguments already validated).  `fused`: all num_parts partitions in
// one launch (tensor-core path only); out / lse are then [P, B, ...].
int enqueue_decode(const void *q, const void *kv_pages, const int32_t *block_table,
                   const int32_t *seq_lens, int part_id, int num_parts, bool fused,
                   float sm_scale, int lse_base, void *out, float *lse, const mla_decode_desc *d,
                   void *workspace, int grid, cudaStream_t s, void *comb_out = nullptr,
                   float *comb_lse = nullptr) {
  const bool tc = tensor_core_path(d, num_parts);
  if (fused && !fused_path(d, num_parts)) return MLA_ERR_ARG;
  if (d->q_len > 1 && !tc) return MLA_ERR_SHAPE;
  const int per_group = tc ? kTcHeadsPerGroup : kSimtHeadsPerGroup;
  const int rows = rows_of(d);
  const int groups = (rows + per_group - 1) / per_group;
  const int vbatch = fused ? num_parts * d->batch : d->batch;
  mla::DecodeParams p;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.kv = kv_pages;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.lse = lse;
  p.ws = static_cast<unsigned char *>(workspace);
  p.wl = mla::workspace_layout(vbatch * groups, grid);
  p.batch = vbatch;
  p.heads = rows;
  p.head_groups = groups;
  p.heads_per_group = per_group;
  p.q_len = d->q_len;
  p.q_heads = d->num_heads;
  p.num_pages = d->num_pages;
  p.max_pages = d->max_pages_per_seq;
  p.part_id = fused ? 0 : part_id;
  p.num_parts = num_parts;
  const bool strided = tc && strided_path(d, num_parts);
  const int gp = tc && !strided ? gather_parts(num_parts) : num_parts;
  if (strided) {
    p.strided = 1;
    p.apg = strided_apg(num_parts);
    p.s_q63 = (mla::kPage - 1) / num_parts;
    p.s_r63 = (mla::kPage - 1) % num_parts;
    p.s_c64 = mla::kPage % num_parts;
  } else if (gp < num_parts) {  // owner mask over the gather of partition part_id mod gp of gp
    p.num_parts = gp;
    p.part_id = part_id % gp;
    p.own_parts = num_parts;
    p.own_part = part_id;
  }
  p.fused = fused ? 1 : 0;
  p.req_batch = d->batch;
  p.comb_out = static_cast<__nv_bfloat16 *>(comb_out);
  p.comb_lse = comb_lse;
  p.kv_e4m3 = d->kv_dtype == MLA_KV_E4M3;
  p.kv_scale = p.kv_e4m3 ? d->kv_scale : 1.f;
  p.score_scale_log2 = sm_scale * mla::kLog2e;
  p.lse_base2 = lse_base == MLA_LSE_BASE2;
  cudaError_t e;
  if (tc) {
    CUtensorMap tm_q, tm_kv, tm_kvg, tm_kvb;
    int st = make_tensor_maps(q, kv_pages, d, p.part_id, p.num_parts, fused, strided, &tm_q,
                              &tm_kv, &tm_kvg, &tm_kvb);
    if (st != MLA_OK) return st;
    const int h = rows < kTcHeadsPerGroup ? rows : kTcHeadsPerGroup;
    const int npv = ((h + 15) / 16) * 16;
    e = mla::launch_decode_tc(p, npv, h, strided ? 1 : 8 / p.num_parts, tm_q, tm_kv, tm_kvg, tm_kvb,
                              grid, s);
  } else {
    e = mla::launch_decode_simt(p, grid, s);
  }
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

}  // namespace

namespace mla {
// The decode partial of one partition on a caller-chosen workspace and grid
// (arguments already validated): the path of the allocation-free entry point.
int enqueue_partial(const void *q, const void *kv_pages, const int32_t *block_table,
                    const int32_t *seq_lens, int part_id, int num_parts, float sm_scale,
                    int lse_base, void *out, float *lse, const mla_decode_desc *d,
                    void *workspace, int grid, cudaStream_t s) {
  return enqueue_decode(q, kv_pages, block_table, seq_lens, part_id, num_parts, false, sm_scale,
                        lse_base, out, lse, d, workspace, grid, s);
}
}  // namespace mla

extern "C" {

int mla_version(void) { return 100; }

// The kernels are built for sm_103a only (arch-specific tcgen05 and TMA
// forms): any other compute capability, sm_100 included, is refused.
int mla_arch_supported(int major, int minor) { return major == 10 && minor == 3 ? 1 : 0; }

const char *mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_NULL: return "a required pointer is NULL";
    case MLA_ERR_SHAPE: return "unsupported shape (q_len 1..16, and 1 off the tensor-core path: num_parts / gcd(num_parts, 8) > 16; Dqk 576, Dv 512, page 64, heads 1..128)";
    case MLA_ERR_PARTITION: return "bad partition (need num_parts >= 1 and 0 <= part_id < num_parts)";
    case MLA_ERR_ALIGN: return "misaligned pointer (16 B for tensors, 256 B for the workspace)";
    case MLA_ERR_WORKSPACE: return "workspace too small";
    case MLA_ERR_ARG: return "bad argument value";
    case MLA_ERR_CUDA: return "CUDA error (see mla_last_cuda_error)";
    case MLA_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case MLA_ERR_BOUNDS: return "block-table entry or sequence length out of bounds";
    case MLA_ERR_TIMEOUT: return "a bounded wait inside the kernel gave up";
    default: return "unknown status";
  }
}

const char *mla_last_cuda_error(void) { return g_cuda_error; }

size_t mla_decode_workspace_size(const mla_decode_desc *d, int num_sms) {
  if (check_desc(d) != MLA_OK) return 0;
  if (num_sms <= 0) {
    int st = 0;
    DeviceFacts f = current_device(&st);
    if (f.sms <= 0) return 0;
    num_sms = f.sms;
  }
  const int virt = d->batch * head_groups_of(d);
  return mla::workspace_layout(virt, num_sms).total;
}

int mla_decode_partial(const void *q, const void *kv_pages, const int32_t *block_table,
                       const int32_t *seq_lens, int part_id, int num_parts, float sm_scale,
                       int lse_base, void *out, float *lse, const mla_decode_desc *d,
                       void *workspace, size_t workspace_bytes, mla_stream_t stream) {
  int st = check_desc(d);
  if (st != MLA_OK) return st;
  if (num_parts < 1 || part_id < 0 || part_id >= num_parts) return MLA_ERR_PARTITION;
  if (d->q_len > 1 && !tensor_core_path(d, num_parts)) return MLA_ERR_SHAPE;
  if (lse_base != MLA_LSE_NATURAL && lse_base != MLA_LSE_BASE2) return MLA_ERR_ARG;
  if (!std::isfinite(sm_scale)) return MLA_ERR_ARG;
  if (d->batch == 0) return MLA_OK;
  if (!q || !kv_pages || !block_table || !seq_lens || !out || !lse || !workspace)
    return MLA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(kv_pages, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256))
    return MLA_ERR_ALIGN;

  DeviceFacts f = current_device(&st);
  if (st != MLA_OK) return st;
  if (workspace_bytes < mla::workspace_layout(d->batch * head_groups_of(d), f.sms).total)
    return MLA_ERR_WORKSPACE;
  return enqueue_decode(q, kv_pages, block_table, seq_lens, part_id, num_parts, false, sm_scale,
                        lse_base, out, lse, d, workspace, f.sms,
                        reinterpret_cast<cudaStream_t>(stream));
}

size_t mla_decode_dcp_workspace_size(const mla_decode_desc *d, int num_parts, int num_sms) {
  if (check_desc(d) != MLA_OK || num_parts < 1) return 0;
  if (num_sms <= 0) {
    int st = 0;
    DeviceFacts f = current_device(&st);
    if (f.sms <= 0) return 0;
    num_sms = f.sms;
  }
  const long long virt = (long long)num_parts * d->batch * head_groups_of(d);
  if (virt > (1LL << 30)) return 0;
  return mla::workspace_layout(int(virt), num_sms).total;
}

int mla_decode_dcp(const void *q, const void *kv_pages, const int32_t *block_table,
                   const int32_t *seq_lens, int num_parts, float sm_scale, int lse_base,
                   void *partials, float *partial_lses, void *out, float *out_lse,
                   const mla_decode_desc *d, void *workspace, size_t workspace_bytes,
                   mla_stream_t stream) {
  int st = check_desc(d);
  if (st != MLA_OK) return st;
  if (num_parts < 1 || num_parts > mla::combine_max_parts()) return MLA_ERR_PARTITION;
  if (lse_base != MLA_LSE_NATURAL && lse_base != MLA_LSE_BASE2) return MLA_ERR_ARG;
  if (!std::isfinite(sm_scale)) return MLA_ERR_ARG;
  if (d->batch == 0) return MLA_OK;
  if ((long long)num_parts * d->batch * rows_of(d) > (1LL << 30)) return MLA_ERR_SHAPE;
  if (d->q_len > 1 && !tensor_core_path(d, num_parts)) return MLA_ERR_SHAPE;
  if (!q || !kv_pages || !block_table || !seq_lens || !partials || !partial_lses || !out ||
      !workspace)
    return MLA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(kv_pages, 16) || !aligned(partials, 16) ||
      !aligned(partial_lses, 4) || !aligned(out, 16) || !aligned(out_lse, 4) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256))
    return MLA_ERR_ALIGN;
  DeviceFacts f = current_device(&st);
  if (st != MLA_OK) return st;
  if (workspace_bytes < mla_decode_dcp_workspace_size(d, num_parts, f.sms))
    return MLA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t rows = size_t(d->batch) * rows_of(d);
  if (num_parts > 1 && fused_path(d, num_parts)) {
    // every partition in one decode launch, then one kernel that merges the
    // splits and combines the partitions (one partition takes the loop below:
    // the single-partition kernel, whose tiles are one page each, and the
    // combine, then a copy)
    return enqueue_decode(q, kv_pages, block_table, seq_lens, 0, num_parts, true, sm_scale,
                          lse_base, partials, partial_lses, d, workspace, f.sms, s, out,
                          out_lse);
  } else {
    for (int r = 0; r < num_parts; ++r) {
      st = enqueue_decode(q, kv_pages, block_table, seq_lens, r, num_parts, false, sm_scale,
                          lse_base, static_cast<__nv_bfloat16 *>(partials) + r * rows * mla::kDv,
                          partial_lses + r * rows, d, workspace, f.sms, s);
      if (st != MLA_OK) return st;
    }
  }
  cudaError_t e = mla::launch_lse_combine(partials, partial_lses, num_parts, out, out_lse,
                                          int(rows), mla::kDv, lse_base == MLA_LSE_BASE2, s);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

int mla_kv_append(const void *kv_new, void *kv_pages, const int32_t *block_table,
                  const int32_t *positions, int part_id, int num_parts,
                  const mla_decode_desc *d, int32_t *error_word, mla_stream_t stream) {
  int st = check_cache_desc(d);
  if (st != MLA_OK) return st;
  if (num_parts < 1 || part_id < 0 || part_id >= num_parts) return MLA_ERR_PARTITION;
  if (d->batch == 0) return MLA_OK;
  if (!kv_new || !kv_pages || !block_table || !positions) return MLA_ERR_NULL;
  if (!aligned(kv_new, 16) || !aligned(kv_pages, 16) || !aligned(block_table, 4) ||
      !aligned(positions, 4) || !aligned(error_word, 4))
    return MLA_ERR_ALIGN;
  current_device(&st);
  if (st != MLA_OK) return st;
  cudaError_t e = mla::launch_kv_append(kv_new, kv_pages, block_table, positions, d->batch,
                                        part_id, num_parts, d->num_pages, d->max_pages_per_seq,
                                        d->kv_dtype == MLA_KV_E4M3, d->kv_scale, error_word,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

int mla_dcp_local_metadata(const int32_t *seq_lens, const int32_t *req_pool_indices,
                           const int32_t *req_to_token, int part_id, int num_parts,
                           const mla_dcp_meta_desc *d, int32_t *global_lens,
                           int32_t *local_lens, int32_t *block_table, int32_t *error_word,
                           mla_stream_t stream) {
  if (!d) return MLA_ERR_NULL;
  if (num_parts < 1 || part_id < 0 || part_id >= num_parts) return MLA_ERR_PARTITION;
  if (d->batch < 0 || d->num_req_slots < 1 || d->req_to_token_width < 1 ||
      d->max_pages_per_seq < 1 || d->page_size != mla::kPage)
    return MLA_ERR_SHAPE;
  if (d->extra_tokens < 0) return MLA_ERR_ARG;
  if (d->batch == 0) return MLA_OK;
  if (!seq_lens || !req_pool_indices || !req_to_token || !global_lens || !local_lens ||
      !block_table)
    return MLA_ERR_NULL;
  if (!aligned(seq_lens, 4) || !aligned(req_pool_indices, 4) || !aligned(req_to_token, 4) ||
      !aligned(global_lens, 4) || !aligned(local_lens, 4) || !aligned(block_table, 4) ||
      !aligned(error_word, 4))
    return MLA_ERR_ALIGN;
  int st = 0;
  current_device(&st);
  if (st != MLA_OK) return st;
  cudaError_t e = mla::launch_dcp_metadata(
      seq_lens, req_pool_indices, req_to_token, d->batch, d->num_req_slots, d->req_to_token_width,
      d->extra_tokens, part_id, num_parts, global_lens, local_lens, block_table,
      d->max_pages_per_seq, d->pad_value, error_word, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

int mla_decode_check_workspace(void *workspace, mla_stream_t stream) {
  if (!workspace) return MLA_ERR_NULL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word & mla::kErrTimeout) return MLA_ERR_TIMEOUT;
  return word ? MLA_ERR_BOUNDS : MLA_OK;
}

int mla_lse_combine(const void *partials, const float *lses, int num_parts, void *out,
                    const mla_combine_desc *d, mla_stream_t stream) {
  if (!d) return MLA_ERR_NULL;
  if (num_parts < 1 || num_parts > mla::combine_max_parts()) return MLA_ERR_PARTITION;
  if (d->num_tokens < 0 || d->num_heads < 1) return MLA_ERR_SHAPE;
  if (d->head_dim < 8 || d->head_dim > 1024 || d->head_dim % 8) return MLA_ERR_SHAPE;
  if (d->lse_base != MLA_LSE_NATURAL && d->lse_base != MLA_LSE_BASE2) return MLA_ERR_ARG;
  if (d->num_tokens == 0) return MLA_OK;
  if (!partials || !lses || !out) return MLA_ERR_NULL;
  if (!aligned(partials, 16) || !aligned(out, 16) || !aligned(lses, 4) ||
      (d->out_lse && !aligned(d->out_lse, 4)))
    return MLA_ERR_ALIGN;
  int st = 0;
  current_device(&st);
  if (st != MLA_OK) return st;
  const long long rows = (long long)d->num_tokens * d->num_heads;
  if (rows > (1LL << 30)) return MLA_ERR_SHAPE;
  cudaError_t e = mla::launch_lse_combine(partials, lses, num_parts, out, d->out_lse, int(rows),
                                          d->head_dim, d->lse_base == MLA_LSE_BASE2,
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

}  // extern "C"
