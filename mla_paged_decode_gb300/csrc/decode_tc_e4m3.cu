// Tensor-core decode kernel variants for e4m3 KV caches (kernel in decode_tc.cuh).
#include "decode_tc.cuh"

namespace mla {
template cudaError_t launch_tc_variants<true>(const TcParams &, const CUtensorMap &,
                                               const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, int, cudaStream_t);
}  // namespace mla
