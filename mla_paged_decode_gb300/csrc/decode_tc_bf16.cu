// Tensor-core decode kernel variants for bf16 KV caches (kernel in decode_tc.cuh).
#include "decode_tc.cuh"

namespace mla {
template cudaError_t launch_tc_variants<false>(const TcParams &, const CUtensorMap &,
                                               const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, int, cudaStream_t);
}  // namespace mla
