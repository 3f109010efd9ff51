// Gram-space skinny kernel, Nesterov instantiations (X_0 from U = G + beta M';
// see k_skinny_gs.cuh).
#include "k_skinny_gs.cuh"

namespace muon {

cudaError_t gs_dispatch_nesterov(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  return gs::gs_dispatch_t<gs::kVarNesterov>(a, cfg, s, prepare);
}

int gs_max_active_clusters_nesterov(int ns_type, int m, int cl) {
  return gs::gs_clusters_t<gs::kVarNesterov>(ns_type, m, cl);
}

}  // namespace muon
