// Gram-space skinny kernel, the instantiations with the vector path for
// members whose parameter is [n, m] (rows > cols): each 32-column superblock
// of the iterate is 32 contiguous parameter rows (see k_skinny_gs.cuh).
// fp16 operands here, bf16 operands in k_skinny_gs_transposed_bf16.cu.
#include "k_skinny_gs.cuh"

namespace muon {

cudaError_t gs_dispatch_transposed_bf16(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare);
int gs_max_active_clusters_transposed_bf16(int m, int cl);

cudaError_t gs_dispatch_transposed(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  if (prepare) {
    const cudaError_t e = gs::gs_dispatch_ty<__half, gs::kVarTransposed>(a, cfg, s, true);
    return e != cudaSuccess ? e : gs_dispatch_transposed_bf16(a, cfg, s, true);
  }
  return a.ns_type == NS_F16 ? gs::gs_dispatch_ty<__half, gs::kVarTransposed>(a, cfg, s, false)
                             : gs_dispatch_transposed_bf16(a, cfg, s, false);
}

int gs_max_active_clusters_transposed(int ns_type, int m, int cl) {
  if (m < 1 || m > 64) return -1;
  return ns_type == NS_F16 ? gs::gs_clusters_ty<__half, gs::kVarTransposed>(m, cl)
                           : gs_max_active_clusters_transposed_bf16(m, cl);
}

}  // namespace muon
