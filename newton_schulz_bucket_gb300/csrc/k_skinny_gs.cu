// Gram-space skinny kernel: the plain-momentum instantiations and the
// dispatch between the kernel variants (the Nesterov ones in
// k_skinny_gs_nesterov.cu, the ones with the transposed members' vector path
// in k_skinny_gs_transposed.cu).  The kernel itself is in k_skinny_gs.cuh.
#include "k_skinny_gs.cuh"

namespace muon {

cudaError_t gs_dispatch_nesterov(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare);
int gs_max_active_clusters_nesterov(int ns_type, int m, int cl);
cudaError_t gs_dispatch_transposed(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare);
int gs_max_active_clusters_transposed(int ns_type, int m, int cl);

// Nesterov groups take the Nesterov variant; other groups holding a member
// with rows > cols (a.T != 0) take the transposed variant.
cudaError_t gs_dispatch(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  if (prepare) {  // every variant, so that any may run
    cudaError_t e = gs::gs_dispatch_t<gs::kVarPlain>(a, cfg, s, true);
    if (e == cudaSuccess) e = gs_dispatch_nesterov(a, cfg, s, true);
    return e != cudaSuccess ? e : gs_dispatch_transposed(a, cfg, s, true);
  }
  if (a.nesterov) return gs_dispatch_nesterov(a, cfg, s, false);
  return a.T ? gs_dispatch_transposed(a, cfg, s, false) : gs::gs_dispatch_t<gs::kVarPlain>(a, cfg, s, false);
}

int gs_max_active_clusters(int ns_type, int m, int cl) {
  int p = gs::gs_clusters_t<gs::kVarPlain>(ns_type, m, cl);
  const int q = gs_max_active_clusters_nesterov(ns_type, m, cl);
  const int t = gs_max_active_clusters_transposed(ns_type, m, cl);
  p = q < p ? q : p;
  return t < p ? t : p;
}

}  // namespace muon
