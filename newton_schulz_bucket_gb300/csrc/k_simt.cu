// SIMT (fp32 FMA) batched products of one Newton-Schulz step, for the FP32
// mode and as the always-available reference path:
//   gram:   A = Y Y^T / alpha^2                     (Gram matrix of the iterate)
//   poly:   Q = a I + b A + c A A                   (the step's polynomial matrix)
//   update: Y' = Q Y                                 (= a Y + (b A + c A A) Y)
// «关于分布式Muon的想法整合及讨论» §2: a Gram matrix and a series of matrix
// products; §6: A is recomputed from the new X every round.
#include "common.cuh"

namespace muon {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, kThreads = 256;

enum Op { OP_GRAM = 0, OP_POLY = 1, OP_UPDATE = 2 };

struct GemmDesc {
  const void* A;    // A-operand base (batch 0)
  const void* B;    // B-operand base
  void* C;          // output base
  const void* Aux;  // poly: the A matrix for the b A term
  int64_t sA, sB, sC;  // batch strides (elements)
  int64_t lda, ldb, ldc;
  int M, N, K;
  int b_trans;  // B(k, j) = B[j * ldb + k] when set, else B[k * ldb + j]
  int step;     // poly: Newton-Schulz step (schedule row)
};

template <typename TI, typename TO, int OP>
__global__ void __launch_bounds__(kThreads) k_simt_gemm(GemmDesc d, KArgs a) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int b = blockIdx.z;
  const TI* Ab = static_cast<const TI*>(d.A) + b * d.sA;
  const TI* Bb = static_cast<const TI*>(d.B) + b * d.sB;
  TO* Cb = static_cast<TO*>(d.C) + b * d.sC;
  const int i0 = blockIdx.y * BM, j0 = blockIdx.x * BN;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d.K; k0 += BK) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int e = tid + t * kThreads;
      const int kk = e & 15, ii = e >> 4;
      const int i = i0 + ii, k = k0 + kk;
      As[kk][ii] = (i < d.M && k < d.K) ? to_f32(Ab[(int64_t)i * d.lda + k]) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int e = tid + t * kThreads;
      int kk, jj;
      if (d.b_trans) { kk = e & 15; jj = e >> 4; } else { jj = e & 63; kk = e >> 6; }
      const int j = j0 + jj, k = k0 + kk;
      float v = 0.f;
      if (j < d.N && k < d.K)
        v = to_f32(d.b_trans ? Bb[(int64_t)j * d.ldb + k] : Bb[(int64_t)k * d.ldb + j]);
      Bs[kk][jj] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) { av[u] = As[kk][ty * 4 + u]; bv[u] = Bs[kk][tx * 4 + u]; }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
  float pa = 0.f, pb = 0.f, pc = 0.f, inv_a2 = 0.f;
  if (OP == OP_POLY) {
    const float* cf = step_coef(a.sc, d.step);
    pa = cf[0]; pb = cf[1]; pc = cf[2];
  }
  if (OP == OP_GRAM) inv_a2 = 1.f / (a.alpha * a.alpha);
  const TI* Aux = static_cast<const TI*>(d.Aux) + b * d.sA;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= d.M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j >= d.N) continue;
      float r = acc[u][v];
      if (OP == OP_GRAM) r *= inv_a2;
      if (OP == OP_POLY) {
        r = fmaf(pc, r, pb * to_f32(Aux[(int64_t)i * d.lda + j]));
        if (i == j) r += pa;
      }
      Cb[(int64_t)i * d.ldc + j] = from_f32<TO>(r);
    }
  }
}

template <int OP>
cudaError_t dispatch(const GemmDesc& d, const KArgs& a, cudaStream_t s) {
  dim3 grid((d.N + BN - 1) / BN, (d.M + BM - 1) / BM, a.B);
  switch (a.ns_type) {
    case NS_F32: k_simt_gemm<float, float, OP><<<grid, kThreads, 0, s>>>(d, a); break;
    case NS_F16: k_simt_gemm<__half, __half, OP><<<grid, kThreads, 0, s>>>(d, a); break;
    default: k_simt_gemm<__nv_bfloat16, __nv_bfloat16, OP><<<grid, kThreads, 0, s>>>(d, a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_gram(const KArgs& a, const void* y, cudaStream_t s) {
  GemmDesc d{};
  d.A = y; d.B = y; d.C = a.A; d.Aux = y;
  d.sA = d.sB = (int64_t)a.m * a.n_pitch; d.sC = (int64_t)a.m * a.m_pitch;
  d.lda = d.ldb = a.n_pitch; d.ldc = a.m_pitch;
  d.M = a.m; d.N = a.m; d.K = a.n; d.b_trans = 1;
  return dispatch<OP_GRAM>(d, a, s);
}

cudaError_t launch_simt_poly(const KArgs& a, int step, cudaStream_t s) {
  GemmDesc d{};
  d.step = step;
  d.A = a.A; d.B = a.A; d.C = a.Q; d.Aux = a.A;
  d.sA = d.sB = d.sC = (int64_t)a.m * a.m_pitch;
  d.lda = d.ldb = d.ldc = a.m_pitch;
  d.M = a.m; d.N = a.m; d.K = a.m; d.b_trans = 0;
  return dispatch<OP_POLY>(d, a, s);
}

cudaError_t launch_simt_update(const KArgs& a, const void* ysrc, void* ydst, cudaStream_t s) {
  GemmDesc d{};
  d.A = a.Q; d.B = ysrc; d.C = ydst; d.Aux = a.Q;
  d.sA = (int64_t)a.m * a.m_pitch; d.sB = d.sC = (int64_t)a.m * a.n_pitch;
  d.lda = a.m_pitch; d.ldb = a.n_pitch; d.ldc = a.n_pitch;
  d.M = a.m; d.N = a.n; d.K = a.m; d.b_trans = 0;
  return dispatch<OP_UPDATE>(d, a, s);
}

}  // namespace muon
