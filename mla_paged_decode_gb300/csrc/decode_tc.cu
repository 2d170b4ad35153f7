// Host entry of the tensor-core decode partial: picks the variant for the
// cache dtype and queues the split merge behind it.  The kernel and its
// variants are in decode_tc.cuh; the bf16 and e4m3 variants compile in
// decode_tc_bf16.cu and decode_tc_e4m3.cu, side by side.
#include "decode_tc.cuh"

namespace mla {

extern template cudaError_t launch_tc_variants<false>(
    const TcParams &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
    const CUtensorMap &, int, cudaStream_t);
extern template cudaError_t launch_tc_variants<true>(
    const TcParams &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
    const CUtensorMap &, int, cudaStream_t);

cudaError_t launch_decode_tc(const DecodeParams &p, int npv, int q_rows, int groups_per_page,
                             const CUtensorMap &tm_q, const CUtensorMap &tm_kv,
                             const CUtensorMap &tm_kvg, const CUtensorMap &tm_kvb, int grid,
                             cudaStream_t stream) {
  TcParams tp;
  tp.p = p;
  tp.npv = npv;
  tp.q_rows = q_rows;
  tp.groups_per_page = groups_per_page;
  cudaError_t e = p.kv_e4m3 ? launch_tc_variants<true>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream)
                            : launch_tc_variants<false>(tp, tm_q, tm_kv, tm_kvg, tm_kvb, grid, stream);
  if (e != cudaSuccess) return e;
  // all partitions in one launch: the split merge also combines the partitions
  return p.fused && p.comb_out ? launch_dcp_merge_combine(p, grid, stream)
                               : launch_split_merge(p, grid, stream);
}

}  // namespace mla
