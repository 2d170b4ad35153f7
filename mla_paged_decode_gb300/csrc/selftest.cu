// mla_selftest_bounded_wait: runs the decode kernels' bounded mbarrier wait
// on barriers that nothing completes, so that a test can check, without a
// GPU fault, that such a wait gives up and reports MLA_ERR_TIMEOUT through
// the workspace, and that the context stays usable.
//
// One CTA of two warps.  Warp 0 waits on a barrier that nothing arrives at
// until `timeout_ns` runs out, and then raises the CTA's abort flag.  Warp 1
// waits on another barrier with a limit ten times longer; it must give up as
// soon as it sees the flag (the path that lets the other roles leave when
// one role's wait fails).  Both outcomes go into the error word.
#include "mla_decode.h"

#include "common.cuh"
#include "sm100.cuh"

namespace {

__global__ void __launch_bounds__(64, 1) selftest_wait_kernel(int *err, uint64_t timeout_ns) {
  __shared__ alignas(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mla::sm100::mbar_init(mla::sm100::smem_u32(&bars[0]), 1);
    mla::sm100::mbar_init(mla::sm100::smem_u32(&bars[1]), 1);
    abort_flag = 0;
    mla::sm100::fence_barrier_init();
  }
  __syncthreads();
  volatile int *abort = &abort_flag;
  // phase 0 of either barrier never completes: no thread arrives
  const bool got = mla::sm100::mbar_wait(mla::sm100::smem_u32(&bars[warp]), 0, abort,
                                    warp == 0 ? timeout_ns : 10 * timeout_ns);
  if (lane == 0 && !got) atomicOr(err, mla::kErrTimeout);
  // the wait gave up without completing the phase: record it separately for
  // each warp (bit 8 + warp), so a test sees that both left
  if (lane == 0 && !got) atomicOr(err, 1 << (8 + warp));
}

}  // namespace

extern "C" int mla_selftest_bounded_wait(void *workspace, int64_t timeout_ns,
                                         mla_stream_t stream) {
  if (!workspace) return MLA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return MLA_ERR_ALIGN;
  // at most 0.1 s: even warp 1's own limit (ten times it) ends within a second
  if (timeout_ns < 1000 || timeout_ns > 100000000) return MLA_ERR_ARG;
  selftest_wait_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<int *>(workspace), uint64_t(timeout_ns));
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
