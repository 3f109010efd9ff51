// Test hooks (include/muon_testing.h): one tcgen05 product on caller buffers,
// the GEMMs' tile walks, the skinny kernel's cluster occupancy, and a
// bounded wait that times out.
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/muon_testing.h"
#include "internal.h"

using namespace muon;

extern "C" muon_status_t muon_testing_tc_gemm(int32_t op, int32_t ns_dtype, int32_t B, int64_t m,
                                              int64_t n, const void* y, const void* a,
                                              const void* q, void* out, float alpha, float pa,
                                              float pb, float pc, void* stream) {
  if (op < 0 || op > 2 || B < 1 || m < 1 || n < 1 || m % 8 || n % 8 || !out)
    return MUON_ERR_INVALID_ARG;
  if ((op != 1 && !y) || (op == 1 && !a) || (op == 2 && !q)) return MUON_ERR_INVALID_ARG;
  if (ns_dtype != MUON_NS_FP16 && ns_dtype != MUON_NS_BF16) return MUON_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepScalars* sc = nullptr;
  int* err = nullptr;
  if (cudaMalloc(&sc, sizeof(StepScalars)) != cudaSuccess) return MUON_ERR_OOM;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) { cudaFree(sc); return MUON_ERR_OOM; }
  StepScalars h{};
  h.ns_steps = 1;
  h.n_coef = 1;
  h.coef[0][0] = pa; h.coef[0][1] = pb; h.coef[0][2] = pc;
  muon_status_t st = MUON_OK;
  cudaError_t e = cudaMemcpy(sc, &h, sizeof h, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(err, 0, sizeof(int));
  KArgs k{};
  k.sc = sc; k.B = B; k.m = (int32_t)m; k.n = (int32_t)n;
  k.ns_type = ns_dtype == MUON_NS_BF16 ? NS_BF16 : NS_F16;
  k.n_pitch = n; k.m_pitch = m; k.alpha = alpha; k.err = err;
  // the product reads y through y0 and writes its m x n output to y1
  k.y0 = const_cast<void*>(op == 1 ? out : y);
  k.y1 = out;
  k.A = op == 0 ? out : const_cast<void*>(a ? a : out);
  k.Q = op == 1 ? out : const_cast<void*>(q ? q : out);
  TcMaps t;
  if (e == cudaSuccess) e = tc_make_maps(k, &t);
  if (e == cudaSuccess) e = prepare_tc(k.ns_type);
  if (e == cudaSuccess) {
    if (op == 0) e = launch_tc_gram(k, t, 0, s);
    else if (op == 1) e = launch_tc_poly(k, t, 0, s);
    else e = launch_tc_update(k, t, 0, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  int w = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&w, err, sizeof w, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) st = MUON_ERR_CUDA;
  else if (w) st = MUON_ERR_TIMEOUT;
  cudaFree(sc);
  cudaFree(err);
  return st;
}

extern "C" int32_t muon_testing_tile_walk(int32_t op, int64_t m, int64_t n, int32_t bn,
                                          int32_t* tm, int32_t* tn, int32_t cap) {
  return tc_tile_walk(op, m, n, 128, bn, tm, tn, cap);
}

extern "C" int32_t muon_testing_tile_walk_pair(int32_t op, int64_t m, int64_t n, int32_t* tm,
                                               int32_t* tn, int32_t cap) {
  return tc_tile_walk(op, m, n, 256, 256, tm, tn, cap);
}

extern "C" int32_t muon_testing_tc_pair_form(int64_t m) { return tc_pair_form(m) ? 1 : 0; }

extern "C" int32_t muon_testing_skinny_max_clusters(int32_t ns_dtype, int64_t m) {
  if (m < 1 || m > 64) return -1;
  SkinnyCfg cfg;
  if (!skinny_config((int32_t)m, 1024, 64, &cfg)) return -1;
  KArgs k{};
  k.m = (int32_t)m;
  k.ns_type = ns_dtype == MUON_NS_BF16 ? NS_BF16 : NS_F16;
  if (prepare_skinny(k, cfg) != cudaSuccess) return -1;
  return skinny_max_active_clusters(k.ns_type, (int)m, cfg.cluster);
}

extern "C" muon_status_t muon_testing_wait_probe(int32_t arrive, int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > (1ll << 33)) return MUON_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = nullptr;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return MUON_ERR_OOM;
  cudaError_t e = cudaMemset(err, 0, sizeof(int));
  if (e == cudaSuccess) e = launch_wait_probe(err, limit_cycles, arrive ? 1 : 0, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  int w = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&w, err, sizeof w, cudaMemcpyDeviceToHost);
  cudaFree(err);
  if (e != cudaSuccess) return MUON_ERR_CUDA;
  return w ? MUON_ERR_TIMEOUT : MUON_OK;
}
