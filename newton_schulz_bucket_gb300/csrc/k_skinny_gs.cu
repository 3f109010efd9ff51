// Gram-space skinny kernel: the plain-momentum instantiations and the
// dispatch between them and the Nesterov ones (k_skinny_gs_nesterov.cu).  The
// kernel itself is in k_skinny_gs.cuh.
#include "k_skinny_gs.cuh"

namespace muon {

cudaError_t gs_dispatch_nesterov(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare);
int gs_max_active_clusters_nesterov(int ns_type, int m, int cl);

cudaError_t gs_dispatch(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  if (prepare) {  // both settings, so that either may run
    const cudaError_t e = gs::gs_dispatch_t<false>(a, cfg, s, true);
    return e != cudaSuccess ? e : gs_dispatch_nesterov(a, cfg, s, true);
  }
  return a.nesterov ? gs_dispatch_nesterov(a, cfg, s, false) : gs::gs_dispatch_t<false>(a, cfg, s, false);
}

int gs_max_active_clusters(int ns_type, int m, int cl) {
  const int p = gs::gs_clusters_t<false>(ns_type, m, cl), q = gs_max_active_clusters_nesterov(ns_type, m, cl);
  return p < q ? p : q;
}

}  // namespace muon
