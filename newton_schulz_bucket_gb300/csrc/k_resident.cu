// Resident path (taken on request) for m = min(rows, cols) <= 128 and
// n <= 4096: the whole Muon step of a member in one kernel, its m x n
// iterate held in the shared memory of one cluster for all k Newton-Schulz
// steps.
//
// «MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化: small
// matrices are bound by dispatch and data movement rather than arithmetic,
// and fusing a shape's members into one launch removes the dispatch (Fig. 6,
// Fig. 7).  On this GPU a [128, 4096] member's three products per step take
// microseconds on the tensor cores, while the TENSOR path's three GEMM
// launches per step stream the iterate through HBM (about 50 B per element
// over a step, against the compulsory 14: G, M and P read, M' and P'
// written, in bf16 mode).  Keeping the iterate on chip leaves only the
// compulsory bytes; what bounds this kernel instead is the latency of the
// per-step exchange of partial Gram matrices across the cluster.
//
// The arithmetic per step is the TENSOR path's («关于分布式Muon的想法整合及讨论»
// §1, §2, §6): with Y = alpha X in the operand type,
//   A  = (Y Y^T) / alpha^2          stored in the operand type,
//   Q  = a I + b A + c A A          stored in the operand type,
//   Y' = Q Y                        stored in the operand type,
// fp32 accumulation in TMEM for each product, and the write
// P' = P (1 - lr wd) - lr s Y_k / alpha.
//
// Layout: one cluster of CL CTAs (1, 2, 4 or 8) per member; CTA r owns the
// wide iterate's columns [r W, r W + W), W a multiple of 64 and at most 512.
// Its shared memory holds (1024-byte aligned):
//   Xs  the CTA's slice of Y, 128 rows (rows >= m are zero) x W columns, as
//       W / 64 column chunks of 128 rows x 128 bytes, 128-byte swizzled:
//       K-major for the Gram product (K = the columns) and MN-major for the
//       update product (K = the rows), the same bytes read both ways;
//   AQ  A, then Q in place: 128 x 128 in the operand type, two K-major chunks;
//   GP  the CTA's fp32 partial Gram matrix, 128 x 128, each row's 16-byte
//       units permuted by (row mod 32) so that neither its writers nor its
//       readers meet bank conflicts.
// The partial Gram matrices are added across the cluster by a reduce-scatter
// (CTA r reads rows [r R, r R + R) of every CTA's GP, R = 128 / CL, and adds
// them in one fixed binary tree over the ranks) followed by an all-gather of
// A into every CTA's AQ, both through distributed shared memory.  (Pushing
// the partial rows to their owners with remote stores, and A back with bulk
// copies, measured slower: remote stores drain at about 20 GB/s per SM.)
// Every CTA then forms Q and its slice of Y' on its own.
//
// 512 threads.  Thread 0 issues every tcgen05.mma (M = 128; N = 128 for the
// Gram and A A products, N <= 256 per instruction for the update); all 16
// warps run the epilogues, warp w reading TMEM lanes 32 (w mod 4) .. + 31.
// Each MMA wait is bounded; on timeout the kernel sets the plan's error word
// and runs to its end (every CTA of a cluster takes the same cluster
// barriers whatever happens, so none is left waiting).
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "mbarrier.cuh"
#include "resident.h"
#include "tcgen05.cuh"
#include "warp_mma.cuh"

namespace muon {

namespace {

constexpr int kNT = 512;            // threads per CTA
constexpr int kRows = 128;          // padded m
constexpr int kChunk = kRows * 128; // bytes of one 64-column chunk of Xs
constexpr uint32_t kOffX = 0;
constexpr uint32_t kOffAQ = kOffX + (kResidentMaxWidth / 64) * kChunk;  // 128 KB
constexpr uint32_t kOffGP = kOffAQ + 2 * kChunk;                          // + 32 KB
constexpr uint32_t kOffMisc = kOffGP + kRows * kRows * 4;                 // + 64 KB
constexpr uint32_t kMiscBytes = 256;
constexpr uint32_t kSmem = kOffMisc + kMiscBytes + 1024;  // + alignment slack
static_assert(kSmem <= 227 * 1024, "resident kernel shared memory exceeds the per-CTA limit");
constexpr uint32_t kTmemCols = 512;

// Byte offset of element (i, j) in a 128-byte-swizzled buffer of 64-column
// chunks of 128 rows (Xs and AQ), 16-bit elements.
__device__ __forceinline__ uint32_t sw_off(int i, int j) {
  return (uint32_t)((j >> 6) * kChunk + i * 128 + ((((j & 63) >> 3) ^ (i & 7)) << 4) + ((j & 7) << 1));
}
// Byte offset of the 16-byte unit holding columns 4 c4 .. 4 c4 + 3 of row i
// of GP.
__device__ __forceinline__ uint32_t gp_off(int i, int c4) {
  return (uint32_t)(i * 512 + ((c4 ^ (i & 31)) << 4));
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_u2(uint32_t caddr, uint32_t x, uint32_t y) {
  asm volatile("st.shared::cluster.v2.b32 [%0], {%1,%2};" ::"r"(caddr), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Generic-proxy writes of shared memory made visible to the tensor cores'
// (async proxy) reads that follow.
__device__ __forceinline__ void fence_async() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Sum of the CL (1, 2, 4 or 8) values v[0 .. CL) as the binary tree
// ((v0 + v1) + (v2 + v3)) + ...
__device__ __forceinline__ float rank_tree(const float (&v)[8], int CL) {
  if (CL == 1) return v[0];
  if (CL == 2) return v[0] + v[1];
  if (CL == 4) return (v[0] + v[1]) + (v[2] + v[3]);
  return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

template <typename TY>
__device__ __forceinline__ uint16_t bits16(float v) {
  const TY h = from_f32<TY>(v);
  return *reinterpret_cast<const uint16_t*>(&h);
}
template <typename TY>
__device__ __forceinline__ float from_bits16(uint32_t u) {
  const uint16_t b = (uint16_t)u;
  return to_f32(*reinterpret_cast<const TY*>(&b));
}
template <typename TY>
__device__ __forceinline__ uint4 pack8(const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = (uint32_t)bits16<TY>(v[2 * i]) | ((uint32_t)bits16<TY>(v[2 * i + 1]) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <typename TY>
__device__ __forceinline__ void unpack8(const uint4& u, float* v) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = from_bits16<TY>(w[i] & 0xffffu);
    v[2 * i + 1] = from_bits16<TY>(w[i] >> 16);
  }
}

}  // namespace

}  // namespace muon

namespace muon {

namespace {

// Per-CTA view of one member.
struct RCtx {
  int tid, m, n, W, c0, wv;  // wv: columns of this CTA that hold data (0 .. W)
  bool T;                    // the parameter is [n, m]
  bool vec;                  // 16-byte vectors along the parameter's rows
  const __nv_bfloat16* G;
  float* M;
  __nv_bfloat16* P;
  float beta;
  bool nest;
  // element (i, j) of the wide iterate slice (i < m, j < wv): offset in the parameter
  __device__ __forceinline__ int64_t off(int i, int j) const {
    return T ? (int64_t)(c0 + j) * m + i : (int64_t)i * n + c0 + j;
  }
};

// 1. M' = beta M + G over this CTA's part of the member, stored; returns the
// thread's sum of squares of M' (Nesterov: of U = G + beta M').  The same
// arithmetic per element as the momentum kernel of the other paths.
__device__ __forceinline__ float momentum_pass(const RCtx& c) {
  const uint64_t pin = l2_evict_first(), pout = l2_evict_last();  // M' is read back in pass 2
  float acc = 0.f;
  auto one = [&](float g, float& mv) {
    mv = fmaf(c.beta, mv, g);
    const float x = c.nest ? fmaf(c.beta, mv, g) : mv;
    acc = fmaf(x, x, acc);
  };
  if (c.vec) {
    // non-transposed: m rows of wv / 8 vectors; transposed: the wv rows of
    // the parameter are one contiguous run of wv m / 8 vectors
    const int nv = c.T ? c.wv * c.m / 8 : c.wv / 8;
    const int items = c.T ? nv : c.m * nv;
    // UN vectors' loads in flight per thread, held as raw 16-byte words
    constexpr int UN = 6;
    for (int e0 = c.tid; e0 < items; e0 += UN * kNT) {
      uint4 gr[UN], mr[UN][2];
      int64_t o[UN];
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int e = e0 + u * kNT;
        if (e < items) {
          if (c.T) {
            o[u] = (int64_t)c.c0 * c.m + 8 * (int64_t)e;
          } else {
            const int i = e / nv;
            o[u] = (int64_t)i * c.n + c.c0 + 8 * (e - i * nv);
          }
          gr[u] = ld_hint(c.G + o[u], pin);
          mr[u][0] = ld_hint(c.M + o[u], pin);
          mr[u][1] = ld_hint(c.M + o[u] + 4, pin);
        }
      }
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        if (e0 + u * kNT < items) {
          float g[8], mv[8];
          bf16x8_to_f32(gr[u], g);
          u4_to_f4x2(mr[u][0], mr[u][1], mv);
#pragma unroll
          for (int k = 0; k < 8; ++k) one(g[k], mv[k]);
          st_hint(c.M + o[u], f4_to_u4(mv), pout);
          st_hint(c.M + o[u] + 4, f4_to_u4(mv + 4), pout);
        }
      }
    }
  } else {
    const int items = c.m * c.wv;
    for (int e = c.tid; e < items; e += kNT) {
      // transposed: walk the contiguous run; else row by row
      const int i = c.T ? e % c.m : e / c.wv, j = c.T ? e / c.m : e % c.wv;
      const int64_t o = c.off(i, j);
      float mv = c.M[o];
      one(__bfloat162float(c.G[o]), mv);
      c.M[o] = mv;
    }
  }
  return acc;
}

// 2. Y_0 = cast(x inv) into Xs, x = M' (Nesterov: U = G + beta M'), every
// element of the W columns written once (zero outside the member).
template <typename TY>
__device__ __forceinline__ void load_pass(const RCtx& c, uint8_t* xs, float inv) {
  const uint64_t pol = l2_evict_first();  // the last read of M' and G
  auto x_of = [&](float mv, float g) { return (c.nest ? fmaf(c.beta, mv, g) : mv) * inv; };
  if (c.vec && !c.T) {
    // one 16-byte unit per item: row i, columns 8 v .. 8 v + 7; UN items'
    // loads in flight per thread
    constexpr int UN = 4;
    const int nu = c.W / 8, items = kRows * nu;
    for (int e0 = c.tid; e0 < items; e0 += UN * kNT) {
      uint4 mr[UN][2], gr[UN];
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int e = e0 + u * kNT, i = e / nu, v = e - i * nu;
        if (e < items && i < c.m && 8 * v < c.wv) {
          const int64_t o = c.off(i, 8 * v);
          mr[u][0] = ld_hint(c.M + o, pol);
          mr[u][1] = ld_hint(c.M + o + 4, pol);
          if (c.nest) gr[u] = ld_hint(c.G + o, pol);
        }
      }
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int e = e0 + u * kNT, i = e / nu, v = e - i * nu;
        if (e >= items) break;
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (i < c.m && 8 * v < c.wv) {
          float mv[8], g[8];
          u4_to_f4x2(mr[u][0], mr[u][1], mv);
          if (c.nest) bf16x8_to_f32(gr[u], g);
#pragma unroll
          for (int k = 0; k < 8; ++k) x[k] = x_of(mv[k], c.nest ? g[k] : 0.f);
        }
        *reinterpret_cast<uint4*>(xs + sw_off(i, 8 * v)) = pack8<TY>(x);
      }
    }
  } else if (c.vec) {
    // transposed: an 8 x 8 block per item, parameter rows c0 + 8 jb + t
    // (t < 8) read as 16-byte vectors over columns 8 ib .. 8 ib + 7, written
    // as the 8 units of Xs rows 8 ib + r, columns 8 jb .. 8 jb + 7
    const int nj = c.W / 8;
    for (int e = c.tid; e < (kRows / 8) * nj; e += kNT) {
      const int ib = e / nj, jb = e - ib * nj;
      float x[8][8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int j = 8 * jb + t;
#pragma unroll
        for (int k = 0; k < 8; ++k) x[t][k] = 0.f;
        if (8 * ib < c.m && j < c.wv) {
          const int64_t o = c.off(8 * ib, j);
          float mv[8], g[8];
          u4_to_f4x2(ld_hint(c.M + o, pol), ld_hint(c.M + o + 4, pol), mv);
          if (c.nest) bf16x8_to_f32(ld_hint(c.G + o, pol), g);
#pragma unroll
          for (int k = 0; k < 8; ++k) x[t][k] = x_of(mv[k], c.nest ? g[k] : 0.f);
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float row[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) row[t] = x[t][r];
        *reinterpret_cast<uint4*>(xs + sw_off(8 * ib + r, 8 * jb)) = pack8<TY>(row);
      }
    }
  } else {
    for (int e = c.tid; e < kRows * c.W; e += kNT) {
      const int i = e / c.W, j = e - i * c.W;
      float x = 0.f;
      if (i < c.m && j < c.wv) {
        const int64_t o = c.off(i, j);
        x = x_of(c.M[o], c.nest ? __bfloat162float(c.G[o]) : 0.f);
      }
      *reinterpret_cast<uint16_t*>(xs + sw_off(i, j)) = bits16<TY>(x);
    }
  }
}

// 4. P' = P (1 - lr wd) - coef Y_k, coef = lr s / alpha (the same arithmetic
// per element as the write kernel of the other paths), and the optional fp32
// copy of O = Y_k / alpha.
template <typename TY>
__device__ __forceinline__ void write_pass(const RCtx& c, const uint8_t* xs, float decay, float coef,
                                           float inv_alpha, float* dbg) {
  auto upd = [&](float y, float p) { return fmaf(-coef, y, p * decay); };
  if (c.vec && !c.T) {
    // UN items' parameter loads in flight per thread
    constexpr int UN = 8;
    const int nv = c.wv / 8, items = c.m * nv;
    for (int e0 = c.tid; e0 < items; e0 += UN * kNT) {
      uint4 pr[UN];
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int e = e0 + u * kNT, i = e / nv, v = e - i * nv;
        if (e < items) pr[u] = *reinterpret_cast<const uint4*>(c.P + c.off(i, 8 * v));
      }
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int e = e0 + u * kNT, i = e / nv, v = e - i * nv;
        if (e >= items) break;
        const int64_t o = c.off(i, 8 * v);
        float y[8], p[8], w[8];
        unpack8<TY>(*reinterpret_cast<const uint4*>(xs + sw_off(i, 8 * v)), y);
        bf16x8_to_f32(pr[u], p);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = upd(y[k], p[k]);
        *reinterpret_cast<uint4*>(c.P + o) = f32_to_bf16x8(w);
        if (dbg) {
#pragma unroll
          for (int k = 0; k < 8; ++k) w[k] = y[k] * inv_alpha;
          *reinterpret_cast<uint4*>(dbg + o) = f4_to_u4(w);
          *reinterpret_cast<uint4*>(dbg + o + 4) = f4_to_u4(w + 4);
        }
      }
    }
  } else if (c.vec) {
    const int nj = (c.wv + 7) / 8, ni = c.m / 8;
    for (int e = c.tid; e < ni * nj; e += kNT) {
      const int ib = e / nj, jb = e - ib * nj;
      float y[8][8];  // [Xs row r][column t]
#pragma unroll
      for (int r = 0; r < 8; ++r)
        unpack8<TY>(*reinterpret_cast<const uint4*>(xs + sw_off(8 * ib + r, 8 * jb)), y[r]);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int j = 8 * jb + t;
        if (j >= c.wv) break;
        const int64_t o = c.off(8 * ib, j);
        float p[8], w[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(c.P + o), p);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = upd(y[k][t], p[k]);
        *reinterpret_cast<uint4*>(c.P + o) = f32_to_bf16x8(w);
        if (dbg) {
#pragma unroll
          for (int k = 0; k < 8; ++k) w[k] = y[k][t] * inv_alpha;
          *reinterpret_cast<uint4*>(dbg + o) = f4_to_u4(w);
          *reinterpret_cast<uint4*>(dbg + o + 4) = f4_to_u4(w + 4);
        }
      }
    }
  } else {
    for (int e = c.tid; e < c.m * c.wv; e += kNT) {
      const int i = c.T ? e % c.m : e / c.wv, j = c.T ? e / c.m : e % c.wv;
      const int64_t o = c.off(i, j);
      const float y = from_bits16<TY>(*reinterpret_cast<const uint16_t*>(xs + sw_off(i, j)));
      c.P[o] = __float2bfloat16_rn(upd(y, __bfloat162float(c.P[o])));
      if (dbg) dbg[o] = y * inv_alpha;
    }
  }
}

}  // namespace

}  // namespace muon

namespace muon {

namespace {

constexpr int kErrResidentWait = 64;  // error-word bit of a resident-kernel MMA wait that ran out

template <typename TY>
__global__ void __launch_bounds__(kNT, 1) k_resident(KArgs a, int W) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* xs = smem + kOffX;
  uint8_t* aq = smem + kOffAQ;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffMisc);    // MMA completion
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  float* ss_slot = reinterpret_cast<float*>(smem + kOffMisc + 16);
  float* red = reinterpret_cast<float*>(smem + kOffMisc + 32);  // 33 floats

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster_rank(), CL = (int)cluster_size();
  const int b = blockIdx.x / CL;
  const MemberPtrs mp = a.mem[b];

  RCtx c;
  c.tid = tid; c.m = a.m; c.n = a.n; c.W = W; c.c0 = rank * W;
  c.wv = max(0, min(W, a.n - c.c0));
  c.T = mp.T != 0;
  c.G = static_cast<const __nv_bfloat16*>(mp.G);
  c.M = mp.M;
  c.P = static_cast<__nv_bfloat16*>(mp.P);
  c.vec = (c.T ? a.m % 8 == 0 : a.n % 8 == 0) && aligned16(c.G) && aligned16(c.M) && aligned16(c.P);
  c.beta = a.sc->beta;
  c.nest = a.nesterov != 0;

  if (tid == 0) {
    mbar_init(saddr(bar), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // 1. momentum and the norm: this CTA's sum by a fixed block tree, the
  // member's by the binary tree over the ranks
  const float part = block_sum(momentum_pass(c), red);
  if (tid == 0) *ss_slot = part;
  cluster_sync();
  float sv[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) sv[r] = r < CL ? ld_dsmem_f32(ss_slot, (uint32_t)r) : 0.f;
  const float ss = rank_tree(sv, CL);
  const float inv = a.alpha / (sqrtf(ss) + a.eps);

  // 2. Y_0 into shared memory
  load_pass<TY>(c, xs, inv);
  fence_async();
  __syncthreads();

  // 3. the k steps on chip
  const int ns = a.sc->ns_steps;
  const uint32_t fmt = std::is_same<TY, __nv_bfloat16>::value ? 1u : 0u;
  const uint32_t id_sq = instr_desc(fmt, 128, 128, false);
  const int nkc = max(1, (c.wv + 63) / 64);  // 64-column chunks that hold data
  const float gscale = 1.f / (a.alpha * a.alpha);
  const int R = kRows / CL;                   // rows of A this CTA adds up
  const int q = warp & 3, qpart = warp >> 2;  // TMEM lane quarter, quarter of the columns
  const int row = 32 * q + lane;              // accumulator row of this thread
  const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
  const uint32_t xs_a = saddr(xs), aq_a = saddr(aq), gp_a = saddr(smem + kOffGP);
  uint32_t ph = 0;
  // On a wait that runs out the kernel keeps going (the error word is set):
  // every CTA must still take every cluster barrier.
  auto mma_wait = [&]() {
    mbar_wait(saddr(bar), ph, abort_flag, a.err, kErrResidentWait);
    ph ^= 1;
    tc_fence_after();
  };
  for (int s = 0; s < ns; ++s) {
    const float* cf = step_coef(a.sc, s);
    const float ca = cf[0], cb = cf[1], cc = cf[2];
    // Gram partial of this CTA's columns: D = Y Y^T (K = columns)
    if (tid == 0) {
      tc_fence_after();
      for (int kc = 0; kc < nkc; ++kc)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t d = smem_desc(xs_a + kc * kChunk + kk * 32, 16, 1024);
          umma(tmem, d, d, id_sq, (kc | kk) != 0);
        }
      umma_commit(saddr(bar));
    }
    mma_wait();
    {
      uint32_t v[32];
      tmem_ld32(tq + 32 * qpart, v);
#pragma unroll
      for (int t = 0; t < 8; ++t)
        *reinterpret_cast<uint4*>(smem + kOffGP + gp_off(row, 8 * qpart + t)) =
            make_uint4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
    }
    tc_fence_before();
    cluster_sync();  // every CTA's partial is in its GP
    // reduce-scatter over the ranks (this CTA's rows of A, read from every
    // CTA's GP), then all-gather of those rows, scaled and cast, into every
    // CTA's AQ
    for (int e = tid; e < R * 32; e += kNT) {
      const int i = rank * R + (e >> 5), c4 = e & 31;
      const uint32_t src = gp_a + gp_off(i, c4);
      float vx[8], vy[8], vz[8], vw[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < CL) p = ld_dsmem_f4(map_rank(src, (uint32_t)r));
        vx[r] = p.x; vy[r] = p.y; vz[r] = p.z; vw[r] = p.w;
      }
      const float s0 = rank_tree(vx, CL) * gscale, s1 = rank_tree(vy, CL) * gscale;
      const float s2 = rank_tree(vz, CL) * gscale, s3 = rank_tree(vw, CL) * gscale;
      const uint32_t w0 = (uint32_t)bits16<TY>(s0) | ((uint32_t)bits16<TY>(s1) << 16);
      const uint32_t w1 = (uint32_t)bits16<TY>(s2) | ((uint32_t)bits16<TY>(s3) << 16);
      const uint32_t dst = aq_a + sw_off(i, 4 * c4);
      for (int r = 0; r < CL; ++r) st_dsmem_u2(map_rank(dst, (uint32_t)r), w0, w1);
    }
    fence_async();
    cluster_sync();  // A is complete in every CTA; the GPs may be rewritten
    // A A (A symmetric: B = A as a K-major operand)
    if (tid == 0) {
      fence_async();
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t d = smem_desc(aq_a + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024);
        umma(tmem + 128, d, d, id_sq, kk != 0);
      }
      umma_commit(saddr(bar));
    }
    mma_wait();
    {
      // Q = a I + b A + c A A over this thread's row, 32 columns, in place
      uint32_t v[32];
      tmem_ld32(tq + 128 + 32 * qpart, v);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int col0 = 32 * qpart + 8 * u;
        uint4* p = reinterpret_cast<uint4*>(aq + sw_off(row, col0));
        float av[8], qv[8];
        unpack8<TY>(*p, av);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int col = col0 + k;
          float x = fmaf(cc, __uint_as_float(v[8 * u + k]), cb * av[k]);
          if (col == row) x += ca;
          qv[k] = (row < c.m && col < c.m) ? x : 0.f;
        }
        *p = pack8<TY>(qv);
      }
    }
    tc_fence_before();
    fence_async();
    __syncthreads();
    // Y' = Q Y over this CTA's columns (Y as an MN-major B operand)
    if (tid == 0) {
      tc_fence_after();
      for (int nt = 0; nt * 256 < nkc * 64; ++nt) {
        const int N = min(256, nkc * 64 - nt * 256);
        const uint32_t id_up = instr_desc(fmt, 128, N, true);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = smem_desc(aq_a + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(xs_a + nt * 4 * kChunk + kk * 2048, kChunk, 1024);
          umma(tmem + nt * 256, ad, bd, id_up, kk != 0);
        }
      }
      umma_commit(saddr(bar));
    }
    mma_wait();
    // Y' back into Xs in the operand type: this thread's row, 32-column
    // chunks qpart, qpart + 4, ..., two loads in flight
    for (int ch = qpart; ch < 2 * nkc; ch += 8) {
      uint32_t v[2][32];
      const bool two = ch + 4 < 2 * nkc;
      tmem_ld32_async(tq + 32 * ch, v[0]);
      if (two) tmem_ld32_async(tq + 32 * (ch + 4), v[1]);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h == 1 && !two) break;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float yv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) yv[k] = __uint_as_float(v[h][8 * u + k]);
          *reinterpret_cast<uint4*>(xs + sw_off(row, 32 * (ch + 4 * h) + 8 * u)) = pack8<TY>(yv);
        }
      }
    }
    tc_fence_before();
    fence_async();
    __syncthreads();
  }

  // 4. the write
  const float lr = a.sc->lr;
  const float decay = __fmaf_rn(-lr, a.sc->wd, 1.f);  // one rounding of 1 - lr wd
  const float coef = lr * mp.scale / a.alpha;          // alpha is a power of two
  float* dbg = a.dbg ? a.dbg + (int64_t)b * a.m * a.n : nullptr;
  write_pass<TY>(c, xs, decay, coef, 1.f / a.alpha, dbg);

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

}  // namespace muon

namespace muon {

bool resident_config(int64_t m, int64_t n, ResidentCfg* cfg) {
  if (m < 1 || m > kResidentMaxM || n < m) return false;
  for (int32_t cl = 1; cl <= kResidentMaxCluster; cl *= 2) {
    const int64_t w = ((n + cl - 1) / cl + 63) / 64 * 64;
    if (w <= kResidentMaxWidth) {
      if (cfg) { cfg->cluster = cl; cfg->width = (int32_t)w; }
      return true;
    }
  }
  return false;
}

namespace {
template <typename TY>
cudaError_t prepare_ty() {
  return cudaFuncSetAttribute(k_resident<TY>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
}
template <typename TY>
cudaError_t launch_ty(const KArgs& a, const ResidentCfg& cfg, cudaStream_t st) {
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(a.B * cfg.cluster);
  lc.blockDim = dim3(kNT);
  lc.dynamicSmemBytes = kSmem;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cfg.cluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, k_resident<TY>, a, (int)cfg.width);
}
}  // namespace

cudaError_t prepare_resident(int ns_type) {
  return ns_type == NS_BF16 ? prepare_ty<__nv_bfloat16>() : prepare_ty<__half>();
}

cudaError_t launch_resident(const KArgs& a, const ResidentCfg& cfg, cudaStream_t s) {
  if (a.ns_type == NS_BF16) return launch_ty<__nv_bfloat16>(a, cfg, s);
  return launch_ty<__half>(a, cfg, s);
}


}  // namespace muon
