// mla_decode_partial_noalloc: the decode partial with its scratch in a
// file-scope device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot call cudaMalloc.  Serving runtimes that
// hand every byte of HBM to their own KV-cache pool and forbid libraries from
// allocating, latency-critical decode loops that cannot afford the implicit
// device synchronisation cudaMalloc / cudaFree may cause, and plain-C hosts
// without an allocator of their own.  They pass inputs and outputs only.
//
// The scratch (split records, the device error word and the split partials)
// is g_noalloc_scratch below: ~40 MB that every GPU which loads this library
// keeps until the process exits.  Host code must not use the array's name as
// a device address -- on the host it is only a stand-in -- so each device's
// address is taken once with cudaGetSymbolAddress, with that device current,
// during the entry point's first call on that device.
#include "mla_decode.h"

#include <cmath>
#include <mutex>

#include "common.cuh"

namespace mla {
int enqueue_partial(const void *q, const void *kv_pages, const int32_t *block_table,
                    const int32_t *seq_lens, int part_id, int num_parts, float sm_scale,
                    int lse_base, void *out, float *lse, const mla_decode_desc *d,
                    void *workspace, int grid, cudaStream_t s);
}

namespace {

constexpr int kNoAllocHeadsPerGroup = 32;   // the smaller head group of the two decode kernels
constexpr int kNoAllocMaxVirtual = 16384;   // batch * ceil(heads / 32)
constexpr int kNoAllocMaxGrid = 152;        // CTAs (GPUs with more SMs use 152)

constexpr size_t kNoAllocBytes =
    mla::workspace_layout(kNoAllocMaxVirtual, kNoAllocMaxGrid).total;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

struct NoAllocDevice {
  void *scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sms = 0;
  bool sm103 = false;
};

constexpr int kMaxDevices = 64;
NoAllocDevice g_devices[kMaxDevices];
std::mutex g_devices_mu;

// Once per device, with the device current: the scratch address and SM count.
int noalloc_device(NoAllocDevice *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_devices_mu);
  NoAllocDevice &d = g_devices[dev];
  if (d.scratch == nullptr) {
    int sms = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MLA_ERR_CUDA;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return MLA_ERR_CUDA;
    d.sms = sms;
    d.sm103 = (major == 10 && minor == 3);
    d.scratch = ptr;
  }
  *out = d;
  return MLA_OK;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int mla_decode_partial_noalloc(const void *q, const void *kv_pages,
                                          const int32_t *block_table, const int32_t *seq_lens,
                                          int part_id, int num_parts, float sm_scale,
                                          int lse_base, void *out, float *lse,
                                          const mla_decode_desc *d, mla_stream_t stream) {
  if (!d) return MLA_ERR_NULL;
  if (d->batch < 0 || d->num_pages < 1 || d->max_pages_per_seq < 1 || d->q_len != 1 ||
      d->head_dim_qk != mla::kDqk || d->head_dim_v != mla::kDv || d->page_size != mla::kPage ||
      d->num_heads < 1 || d->num_heads > 128)
    return MLA_ERR_SHAPE;
  if (d->kv_dtype != MLA_KV_BF16 && d->kv_dtype != MLA_KV_E4M3) return MLA_ERR_ARG;
  if (d->kv_dtype == MLA_KV_E4M3 && !(std::isfinite(d->kv_scale) && d->kv_scale > 0.f))
    return MLA_ERR_ARG;
  if (num_parts < 1 || part_id < 0 || part_id >= num_parts) return MLA_ERR_PARTITION;
  if (lse_base != MLA_LSE_NATURAL && lse_base != MLA_LSE_BASE2) return MLA_ERR_ARG;
  if (!std::isfinite(sm_scale)) return MLA_ERR_ARG;
  if (d->batch == 0) return MLA_OK;
  if (!q || !kv_pages || !block_table || !seq_lens || !out || !lse) return MLA_ERR_NULL;
  if (!aligned_to(q, 16) || !aligned_to(kv_pages, 16) || !aligned_to(out, 16) ||
      !aligned_to(lse, 4) || !aligned_to(block_table, 4) || !aligned_to(seq_lens, 4))
    return MLA_ERR_ALIGN;
  const int groups = (d->num_heads + kNoAllocHeadsPerGroup - 1) / kNoAllocHeadsPerGroup;
  const long long virt = (long long)d->batch * groups;
  if (virt > kNoAllocMaxVirtual) return MLA_ERR_WORKSPACE;  // beyond the built-in scratch

  NoAllocDevice dev;
  int st = noalloc_device(&dev);
  if (st != MLA_OK) return st;
  if (!dev.sm103) return MLA_ERR_DEVICE;
  const int grid = dev.sms < kNoAllocMaxGrid ? dev.sms : kNoAllocMaxGrid;
  const mla::WorkspaceLayout wl = mla::workspace_layout(int(virt), grid);
  if (wl.total > kNoAllocBytes) return MLA_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The scratch keeps the previous call's contents: the error word must start
  // at zero (every other part is rewritten before it is read).
  if (cudaMemsetAsync(dev.scratch, 0, 256, s) != cudaSuccess) return MLA_ERR_CUDA;
  // the kernels of mla_decode_partial on the built-in scratch: the
  // tensor-core kernel whenever num_parts / gcd(num_parts, 8) <= 16 (the
  // strided gather and the owner mask included), else the CUDA-core kernel.
  // The split layout depends on the grid, so the outputs equal
  // mla_decode_partial's bit for bit on GPUs with at most 152 SMs.
  return mla::enqueue_partial(q, kv_pages, block_table, seq_lens, part_id, num_parts, sm_scale,
                              lse_base, out, lse, d, dev.scratch, grid, s);
}
