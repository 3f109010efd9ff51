// Gram-space skinny kernel with the transposed members' vector path, bf16
// operands (see k_skinny_gs_transposed.cu).
#include "k_skinny_gs.cuh"

namespace muon {

cudaError_t gs_dispatch_transposed_bf16(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  return gs::gs_dispatch_ty<__nv_bfloat16, gs::kVarTransposed>(a, cfg, s, prepare);
}

int gs_max_active_clusters_transposed_bf16(int m, int cl) {
  return gs::gs_clusters_ty<__nv_bfloat16, gs::kVarTransposed>(m, cl);
}

}  // namespace muon
