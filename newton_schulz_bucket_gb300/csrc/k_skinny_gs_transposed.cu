// Gram-space skinny kernel, the instantiations with the vector path for
// members whose parameter is [n, m] (rows > cols): each 32-column superblock
// of the iterate is 32 contiguous parameter rows (see k_skinny_gs.cuh).
#include "k_skinny_gs.cuh"

namespace muon {

cudaError_t gs_dispatch_transposed(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  return gs::gs_dispatch_t<gs::kVarTransposed>(a, cfg, s, prepare);
}

int gs_max_active_clusters_transposed(int ns_type, int m, int cl) {
  return gs::gs_clusters_t<gs::kVarTransposed>(ns_type, m, cl);
}

}  // namespace muon
