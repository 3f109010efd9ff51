// Skinny path for m = min(rows, cols) <= 64 (kernel templates; k_skinny_gs.cu,
// k_skinny_gs_nesterov.cu and k_skinny_gs_transposed*.cu instantiate them):
// the whole Muon step of a member in one kernel, with Newton-Schulz evaluated
// in Gram space.
//
// «MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化: for
// shapes such as [24, 10240] the per-parameter iteration is dominated by host
// dispatch, small allocations and synchronisation, and batching every member
// of a shape into one launch removes that (Fig. 7).  On this GPU the batched
// work is bound by bytes moved (HBM, and L2, whose read bandwidth is close to
// HBM's), so the kernel streams the member's data twice however many steps
// are taken:
//
//   1. momentum pass: M' = beta M + G is formed and stored, and from the same
//      registers the sum of squares ||M'||_F^2 and the Gram matrix M' M'^T
//      (tf32 tensor-core products, fp32 accumulation: the norm is not known
//      yet, and tf32 keeps fp32's range with an 11-bit significand);
//   2. in m x m space, fp32: A_0 = M' M'^T / (||M'||_F + eps)^2, then per step
//      Q = a I + b A + c A^2, Pi <- Q Pi, A <- Q A Q (3xTF32 tensor-core
//      tiles up to m = 32, where the stage is latency-bound; fp32 FFMA
//      above, where it is throughput-bound);
//   3. output pass: Y_0 = alpha M' / (||M'||_F + eps) split into an
//      operand-type high part and residual, O = Pi_k Y_0 / alpha with Pi_k
//      split the same way, and P' = P (1 - lr wd) - lr s O.
//
// Each quintic step is X' = Q X with Q = a I + b A + c A^2 and A = X X^T
// («关于分布式Muon的想法整合及讨论» §1, §2, §6).  Q is a polynomial in A, so it
// is symmetric and commutes with A, hence A' = X' X'^T = Q A Q and
// X_k = Pi_k X_0 with Pi_k = Q_{k-1} ... Q_0: in exact arithmetic this is the
// iteration itself; in floating point the data is rounded to the operand
// type once instead of once per step.
//
// Layout: one cluster of CL CTAs per member, CTA r owning one contiguous
// column shard of the wide iterate's columns [r W, (r + 1) W).  Up to m = 32
// a CTA has 16 warps (2-CTA clusters) or 8 warps (4-CTA clusters, two CTAs
// per SM, for batches too small to fill the GPU); beyond, 8 warps, each lane
// keeping Pi's fragments for four 16-row tiles (128 registers).  Both passes
// walk 32-column superblocks.  In the momentum pass warp w of CTA r takes
// one contiguous leaf of the member's superblocks, leaf r NW + w, and the
// leaves' partial sums are added by one fixed binary tree (over warps, then
// over CTAs), so the bits depend only on (rows, cols) and the number of
// leaves, never on the batch or the launch form.  Lane (g, t4) holds rows
// 16 mi + g (+ 8) and the eight consecutive columns 8 t4 .. 8 t4 + 7, which
// stand in tf32 A-fragment slots (see gs_momentum_pass); the output pass
// loads Y_0 straight into B fragments (see gs_out_pass).  The Gram sums over
// all columns and Pi X acts on each column alone, so these fixed
// permutations of a block's columns change nothing, and they turn every
// access into a 16-byte (fp32) or 8/16-byte (bf16) vector.  Operands stream
// through a per-lane cp.async ring.
#pragma once

#include "warp_mma.cuh"

namespace muon {
namespace gs {

// Kernel variants, each instantiated in its own translation unit: plain
// momentum with the vector path for members with rows <= cols (transposed
// members then take the element-wise path); Nesterov (every member with
// rows > cols on the element-wise path); plain momentum with the vector path
// for transposed members too, for groups that hold any (its extra branches
// cost the plain variant registers and time).
constexpr int kVarPlain = 0, kVarNesterov = 1, kVarTransposed = 2;


// Sum of N (a power of two) values as the binary tree
// ((v0 + v1) + (v2 + v3)) + ...: a fixed order, so that a tree over more
// leaves can be split into subtrees computed in different places.
template <int N>
__device__ __forceinline__ float tree_sum(float (&v)[N]) {
#pragma unroll
  for (int s = 1; s < N; s *= 2)
#pragma unroll
    for (int k = 0; k + s < N; k += 2 * s) v[k] += v[k + s];
  return v[0];
}
// The same tree over the value at `local` in each of the cluster's CL CTAs
// (CL = 1, 2, 4 or 8), read through distributed shared memory.
__device__ __forceinline__ float cluster_tree_sum(const float* local, int CL) {
  float v[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) v[r] = r < CL ? ld_dsmem_f32(local, (uint32_t)r) : 0.f;
  if (CL == 1) return v[0];
  if (CL == 2) return v[0] + v[1];
  if (CL == 4) return (v[0] + v[1]) + (v[2] + v[3]);
  return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

template <int MT, int NT, bool HALF>
struct GsLayout {
  static constexpr int MP = 16 * MT;                    // padded m
  static constexpr int LD = MP + 4;                     // fp32 m x m row pitch: 16-byte rows, no bank conflicts
  static constexpr int NW = NT / 32;
  static constexpr int R = 2 * MT - (HALF ? 1 : 0);     // rows g + 8 h a lane holds (momentum pass, output rows)
  static constexpr int KR = 4 * MT - (HALF ? 2 : 0);    // rows 2 t4 + {0, 1, 8, 9} a lane holds (output pass)
  static constexpr int NJ = HALF ? 2 * MT - 1 : 2 * MT; // 8-row groups of the Gram's columns
  using GT = GramTiles<MT, NJ>;
  // Both passes are bound by the bytes a CTA keeps in flight, so each ring
  // takes as many rounds as shared memory holds next to the fixed part
  // (this CTA's Gram partial, misc words, Pi's row scales, the upper-triangle
  // index table).
  static constexpr int kTab = ((MP * (MP + 1) / 2) * 4 + 15) / 16 * 16;
  static constexpr int kCoef = kMaxScheduleRows * 3 * 4;  // the step's (a, b, c) rows
  static constexpr int kFixed = MP * MP * 4 + 64 + MP * 4 + kTab + kCoef;
  // shared memory of one CTA: all of it, or, for the 8-warp form of m <= 32
  // that puts two CTAs on an SM, half the SM's 228 KB less the 1 KB the
  // runtime reserves per CTA
  static constexpr int kBudget = (MT <= 2 && NT == 256) ? 233472 / 2 - 1024 : 227 * 1024;
  static constexpr int kCap = kBudget - kFixed;
  // momentum pass ring: 32 B of M and 16 B of G per row and lane; one round at a time
  static constexpr int LB1 = 48 * R;
  static constexpr int S1 = 4 * NW * 32 * LB1 <= kCap ? 4 : (3 * NW * 32 * LB1 <= kCap ? 3 : 2);
  static constexpr int kRing1 = S1 * NW * 32 * LB1;
  // output pass ring: 16 B of M' per k-row and 16 B of P per output row and lane; one round at a time
  static constexpr int LBO = 16 * (KR + R);
  static constexpr int SO = 4 * NW * 32 * LBO <= kCap ? 4 : (3 * NW * 32 * LBO <= kCap ? 3 : 2);
  static constexpr int kRingO = SO * NW * 32 * LBO;
  // between the passes the ring holds the per-warp Gram partials and sums of
  // squares, then the m x m work arrays: A, Q, T, Pi (two) -- for m <= 32
  // each stored as a tf32 high part and a tf32 residual, else in fp32 -- and
  // Pi's operand-type high / low parts
  static constexpr int kWarpPart = NW * GT::N * 128 * 4 + NW * 4 * 4;
  static constexpr int kMat = MP * LD * 4;
  static constexpr int kPiT = MP * (MP + 8) * 2;
  static constexpr bool TC = MT <= 2;  // m x m products on the tensor cores (else FFMA)
  static constexpr int kMM = (TC ? 10 : 5) * kMat + 2 * kPiT;  // A, Q, T, Pi x2, then Pi high / low
  // the rings, the per-warp partials and the m x m arrays are live one after
  // the other and share the same bytes
  static constexpr int kU0 = kRing1 > kRingO ? kRing1 : kRingO;
  static constexpr int kU1 = kWarpPart > kMM ? kWarpPart : kMM;
  static constexpr int kU = kU0 > kU1 ? kU0 : kU1;
  static constexpr int kCta = kU;                       // this CTA's Gram partial (peer reads it)
  static constexpr int kMisc = kCta + MP * MP * 4;      // [0] sum of squares (peer reads it)
  static constexpr int kRsc = kMisc + 64;               // Pi's row scales
  static constexpr int kTabOff = kRsc + MP * 4;         // (i << 16 | j) of the upper triangle, row-major
  static constexpr int kCoefOff = kTabOff + kTab;       // schedule rows, copied from the step scalars
  static constexpr int kTotal = kCoefOff + kCoef;
  static_assert(kTotal == kU + kFixed, "layout");
  static_assert(kTotal <= kBudget, "Gram-space kernel shared memory exceeds the per-CTA budget");
};

// Wide-iterate element (i, j) in the parameter's memory.
struct Wide {
  int cols, T;
  __device__ __forceinline__ int64_t off(int i, int j) const {
    return T ? (int64_t)j * cols + i : (int64_t)i * cols + j;
  }
};

// Per-thread state of one member's two data passes.
struct GsCtx {
  int lane, warp, g, t4, m, n, c0, NB;  // NB: 16-column blocks of this CTA (even)
  bool vec;            // rows <= cols, cols % 8 == 0, 32 cols < 2^31, M', G and P 16-byte aligned
  bool tvec;           // rows > cols (the parameter is [n, m]), m % 8 == 0, n m < 2^31, 16-byte
                       // aligned, no Nesterov: a superblock is one contiguous block of 32 rows
  float* Mp;
  const __nv_bfloat16* G;
  __nv_bfloat16* P;
  float* dbg;
  int cols;
  Wide wd;
  float beta, inv, decay, coef, inv_alpha;
};

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Momentum pass over this warp's 32-column superblocks: M' = beta M + G
// stored, ss += M'^2 per lane, and gacc += M' M'^T on the upper Gram tiles
// (tf32).  In registers lane (g, t4) holds rows 16 mi + g (+ 8) and columns
// J + 8 t4 .. J + 8 t4 + 7; column J + 8 t4 + 2 st + e stands in the tf32
// A-fragment slot k = t4 + 4 e of k8 step st.  All three streams keep the
// default L2 policy: measured, evict-first reads or evict-last stores here
// only slowed the pass.
template <int MT, int NT, bool HALF, int VAR>
__device__ __forceinline__ void gs_momentum_pass(const GsCtx& c, uint8_t* ring,
                                                 float (&gacc)[GsLayout<MT, NT, HALF>::GT::N][4], float& ss,
                                                 int LS) {
  constexpr bool NEST = VAR == kVarNesterov, TP = VAR == kVarTransposed;
  using L = GsLayout<MT, NT, HALF>;
  using GT = typename L::GT;
  constexpr int NW = L::NW, S = L::S1, LB = L::LB1, R = L::R;
  constexpr uint32_t kSlot = NW * 32 * LB;
  const int lane = c.lane;
  uint8_t* ring_warp = ring + c.warp * 32 * LB;
  const uint32_t ring0 = smem_u32(ring_warp);
  const int nsb = c.NB / 2;  // superblocks of this CTA
  // warp w takes the LS superblocks w LS .. w LS + LS - 1 of the CTA (its
  // leaf of the reduction tree), in order
  const int rounds = LS;
  auto row_of = [&](int s) { return (s >> 1) * 16 + c.g + ((s & 1) ? 8 : 0); };
  const uint64_t pol = l2_evict_normal();
  const float2 beta2 = make_float2(c.beta, c.beta);
  float2 ss2 = make_float2(0.f, 0.f);

  // A round's slot holds the superblock as row-major tiles, so that every
  // global access of a warp moves whole lines: M (later M') rows of 128 B
  // whose 16-byte chunk q sits at q ^ (row & 1) (the fragment reads below are
  // then free of bank conflicts), and G rows of 64 B.  Lanes copy in and out
  // by rows (8 lanes per M row, 4 per G row) and read their fragments after a
  // warp barrier.
  constexpr int RT = 8 * R;  // rows of the tile (rows >= m are zero-filled)
  auto mchunk = [](int row, int q) { return row * 128 + ((q ^ (row & 1)) << 4); };
  // A transposed member's superblock is parameter rows J .. J + 31, one
  // contiguous block: it is staged as such, M at the slot's start (row pitch
  // m floats) and G after 32 m floats (row pitch m bf16), 16-byte chunks
  // spread over the lanes; rows past n are zero-filled.
  const int mq = c.m / 4;  // 16-byte chunks per row of M (transposed member)
  auto issue_t = [&](int r, uint32_t dst) {
    const int sb = c.warp * LS + r;
    if (r < rounds && sb < nsb) {
      const int J = c.c0 + sb * 32, nrows = min(32, c.n - J);
      const float* mb = c.Mp + (int64_t)J * c.m;
      const __nv_bfloat16* gb = c.G + (int64_t)J * c.m;
      for (int k = lane; k < 8 * c.m; k += 32) {
        const bool ok = k / mq < nrows;
        cp_async16_hint(dst + k * 16, ok ? (const void*)(mb + 4 * k) : (const void*)c.Mp, ok ? 16 : 0, pol);
      }
      for (int k = lane; k < 4 * c.m; k += 32) {
        const bool ok = 2 * k / mq < nrows;
        cp_async16_hint(dst + 128 * c.m + k * 16, ok ? (const void*)(gb + 8 * k) : (const void*)c.G,
                        ok ? 16 : 0, pol);
      }
    }
    cp_async_commit();
  };
  auto issue = [&](int r, uint32_t dst) {
    if (TP && c.tvec) {
      issue_t(r, dst);
      return;
    }
    const int sb = c.warp * LS + r;
    if (c.vec && r < rounds && sb < nsb) {
      const int J = c.c0 + sb * 32;
#pragma unroll
      for (int k = 0; k < RT / 4; ++k) {
        const int row = 4 * k + (lane >> 3), q = lane & 7;
        const bool ok = row < c.m && J + 4 * q < c.n;
        cp_async16_hint(dst + mchunk(row, q),
                        ok ? (const void*)(c.Mp + (int64_t)row * c.cols + J + 4 * q) : (const void*)c.Mp,
                        ok ? 16 : 0, pol);
      }
#pragma unroll
      for (int k = 0; k < RT / 8; ++k) {
        const int row = 8 * k + (lane >> 2), q = lane & 3;
        const bool ok = row < c.m && J + 8 * q < c.n;
        cp_async16_hint(dst + RT * 128 + row * 64 + q * 16,
                        ok ? (const void*)(c.G + (int64_t)row * c.cols + J + 8 * q) : (const void*)c.G,
                        ok ? 16 : 0, pol);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int r = 0; r < S; ++r) issue(r, ring0 + r * kSlot);

  auto process = [&](int r, uint8_t* st) {
    const int sb = c.warp * LS + r;
    if (r >= rounds || sb >= nsb) return;
    const int J = c.c0 + sb * 32;
    const int j0 = J + 8 * c.t4;
    // tv[mi][st][h][e]: row 16 mi + g + 8 h, tf32 slot k = t4 + 4 e of k8 step st
    uint32_t tv[MT][4][2][2];
    if (c.vec || (TP && c.tvec)) __syncwarp();  // every lane's copies of this round have landed
    float* tm = reinterpret_cast<float*>(st);                                 // transposed: M, M'
    const __nv_bfloat16* tg = reinterpret_cast<const __nv_bfloat16*>(st + 128 * c.m);  // and G
#pragma unroll
    for (int s = 0; s < R; ++s) {
      const int i = row_of(s);
      float v[8];
      if (TP && c.tvec) {
        // this lane's eight columns of the superblock are parameter rows
        // t4 + 4 q (q = 0..7): for m = 8 mod 16 the 32 lanes then hit 32
        // banks; any fixed assignment serves, since the Gram sums over all
        // columns and both of its operands come from these registers
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int o = (c.t4 + 4 * q) * c.m + i;
          v[q] = 0.f;
          if (i < c.m && J + c.t4 + 4 * q < c.n) {
            v[q] = fmaf(c.beta, tm[o], __bfloat162float(tg[o]));
            tm[o] = v[q];  // M' replaces M in the block
          }
        }
      } else if (c.vec) {
        float4* m0p = reinterpret_cast<float4*>(st + mchunk(i, 2 * c.t4));
        float4* m1p = reinterpret_cast<float4*>(st + mchunk(i, 2 * c.t4 + 1));
        const float4 m0 = *m0p, m1 = *m1p;
        float gf[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(st + RT * 128 + i * 64 + c.t4 * 16), gf);
        const float2 r0 = __ffma2_rn(beta2, make_float2(m0.x, m0.y), make_float2(gf[0], gf[1]));
        const float2 r1 = __ffma2_rn(beta2, make_float2(m0.z, m0.w), make_float2(gf[2], gf[3]));
        const float2 r2 = __ffma2_rn(beta2, make_float2(m1.x, m1.y), make_float2(gf[4], gf[5]));
        const float2 r3 = __ffma2_rn(beta2, make_float2(m1.z, m1.w), make_float2(gf[6], gf[7]));
        v[0] = r0.x; v[1] = r0.y; v[2] = r1.x; v[3] = r1.y;
        v[4] = r2.x; v[5] = r2.y; v[6] = r3.x; v[7] = r3.y;
        *m0p = make_float4(v[0], v[1], v[2], v[3]);  // M' replaces M in the tile
        *m1p = make_float4(v[4], v[5], v[6], v[7]);
        if constexpr (NEST) {
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = fmaf(c.beta, v[q], gf[q]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          v[q] = 0.f;
          if (i < c.m && j0 + q < c.n) {
            const int64_t o = c.wd.off(i, j0 + q);
            const float g = __bfloat162float(c.G[o]);
            v[q] = fmaf(c.beta, c.Mp[o], g);
            c.Mp[o] = v[q];
            if constexpr (NEST) v[q] = fmaf(c.beta, v[q], g);
          }
        }
      }
      // v: this lane's eight values of X (M', or U under Nesterov)
#pragma unroll
      for (int q = 0; q < 4; ++q) ss2 = __ffma2_rn(make_float2(v[2 * q], v[2 * q + 1]),
                                                  make_float2(v[2 * q], v[2 * q + 1]), ss2);
#pragma unroll
      for (int st4 = 0; st4 < 4; ++st4) {
        tv[s >> 1][st4][s & 1][0] = to_tf32(v[2 * st4]);
        tv[s >> 1][st4][s & 1][1] = to_tf32(v[2 * st4 + 1]);
      }
    }
    if (TP && c.tvec) {
      // M' out as the contiguous block
      __syncwarp();
      const int nrows = min(32, c.n - J);
      float* mb = c.Mp + (int64_t)J * c.m;
      for (int k = lane; k < 8 * c.m; k += 32)
        if (k / mq < nrows) st_hint(mb + 4 * k, *reinterpret_cast<const uint4*>(st + k * 16), pol);
      __syncwarp();  // the block is read out before its slot is refilled
    }
    if (c.vec) {
      // M' out by rows, whole lines (each lane stores the chunks it will refill)
      __syncwarp();
#pragma unroll
      for (int k = 0; k < RT / 4; ++k) {
        const int row = 4 * k + (lane >> 3), q = lane & 7;
        if (row < c.m && J + 4 * q < c.n)
          st_hint(c.Mp + (int64_t)row * c.cols + J + 4 * q,
                  *reinterpret_cast<const uint4*>(st + mchunk(row, q)), pol);
      }
    }
    if (HALF) {
#pragma unroll
      for (int st4 = 0; st4 < 4; ++st4) tv[MT - 1][st4][1][0] = tv[MT - 1][st4][1][1] = 0u;
    }
#pragma unroll
    for (int q = 0; q < GT::N; ++q) {
      const int mi = GT::code(q) >> 4, nj = GT::code(q) & 15;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_tf32(gacc[q], tv[mi][k][0][0], tv[mi][k][1][0], tv[mi][k][0][1], tv[mi][k][1][1],
                 tv[nj >> 1][k][nj & 1][0], tv[nj >> 1][k][nj & 1][1]);
    }
  };

  for (int r = 0; r < rounds; ++r) {
    cp_async_wait<S - 1>();
    process(r, ring_warp + (r % S) * kSlot);
    // round r is consumed (its M' copied out): refill its slot
    issue(r + S, ring0 + (r % S) * kSlot);
  }
  cp_async_wait<0>();
  ss += ss2.x + ss2.y;
}

// The output pass's ring and its copies: round r lives in slot r % S.
template <int MT, int NT, bool HALF>
struct GsOutRing {
  using L = GsLayout<MT, NT, HALF>;
  static constexpr int NW = L::NW, S = L::SO, LB = L::LBO, R = L::R, KR = L::KR;
  static constexpr uint32_t kSlot = NW * 32 * LB;
  static __device__ __forceinline__ int slot(int r) { return r % S; }

  // loop-invariant element offsets of this lane's rows (32 cols < 2^31 on the
  // vector path); rows >= m read as zero
  int moff[KR], poff[R];
  uint32_t mok, pok;
  uint32_t ring0;
  int rounds, nsb;

  __device__ __forceinline__ static int krow(const GsCtx& c, int kr) {
    return (kr >> 2) * 16 + 2 * c.t4 + (kr & 1) + ((kr & 2) ? 8 : 0);
  }
  __device__ __forceinline__ static int orow(const GsCtx& c, int s) {
    return (s >> 1) * 16 + c.g + ((s & 1) ? 8 : 0);
  }
  __device__ __forceinline__ GsOutRing(const GsCtx& c, uint8_t* ring) {
    ring0 = smem_u32(ring + c.warp * 32 * LB);
    nsb = c.NB / 2;  // superblocks of this CTA
    rounds = (nsb + NW - 1) / NW;
    mok = pok = 0;
#pragma unroll
    for (int kr = 0; kr < KR; ++kr) {
      moff[kr] = krow(c, kr) * c.cols;
      if (krow(c, kr) < c.m) mok |= 1u << kr;
    }
#pragma unroll
    for (int s = 0; s < R; ++s) {
      poff[s] = orow(c, s) * c.cols;
      if (orow(c, s) < c.m) pok |= 1u << s;
    }
  }
  // round r's M' and P into its slot, as one commit group (empty past the end)
  __device__ __forceinline__ void issue(const GsCtx& c, int r, uint64_t pol) const {
    const int sb = r * NW + c.warp;
    if (c.vec && r < rounds && sb < nsb) {
      const uint32_t dst = ring0 + slot(r) * kSlot;
      const int J = c.c0 + sb * 32, jm = J + 4 * c.g, jp = J + 8 * c.t4;
      const bool cm = jm < c.n, cpp = jp < c.n;  // n % 8 == 0: a lane's columns share fate
#pragma unroll
      for (int kr = 0; kr < KR; ++kr) {
        const bool ok = cm && ((mok >> kr) & 1u);
        cp_async16_hint(dst + kr * 512 + c.lane * 16, c.Mp + (ok ? moff[kr] + jm : 0), ok ? 16 : 0, pol);
      }
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const bool ok = cpp && ((pok >> s) & 1u);
        cp_async16_hint(dst + (KR + s) * 512 + c.lane * 16, c.P + (ok ? poff[s] + jp : 0), ok ? 16 : 0,
                        pol);
      }
    }
    cp_async_commit();
  }
};

// Output pass over this warp's 32-column superblocks: O = (Pi_hi + Pi_lo) Y_0
// and P' = P (1 - lr wd) - lr s O.  Y_0 is loaded straight into B fragments:
// lane (g, t4) holds rows 16 kk + 2 t4 + {0, 1, 8, 9} of columns
// J + 4 g .. J + 4 g + 3, column J + 4 g + q standing at n = g of n-tile q.
// Accumulator n of n-tile q is then column J + 4 n + q, so a lane's outputs
// of a row are the eight consecutive columns J + 8 t4 .. J + 8 t4 + 7.
template <typename TY, int MT, int NT, bool HALF, bool NEST>
__device__ __forceinline__ void gs_out_pass(const GsCtx& c, uint8_t* ring,
                                            const uint32_t (&ph)[MT][MT][4], const uint32_t (&pl)[MT][MT][4],
                                            const float (&rs)[GsLayout<MT, NT, HALF>::R]) {
  using L = GsLayout<MT, NT, HALF>;
  using Ring = GsOutRing<MT, NT, HALF>;
  constexpr int NW = L::NW, S = L::SO, LB = L::LBO, KR = L::KR;
  constexpr uint32_t kSlot = NW * 32 * LB;
  const int lane = c.lane;
  uint8_t* ring_warp = ring + c.warp * 32 * LB;
  const Ring rg(c, ring);
  const int nsb = rg.nsb, rounds = rg.rounds;
  auto krow = [&](int kr) { return Ring::krow(c, kr); };
  auto orow = [&](int s) { return Ring::orow(c, s); };
  const uint64_t last_use = l2_evict_first();
  const float2 inv2 = make_float2(c.inv, c.inv), decay2 = make_float2(c.decay, c.decay);
  const int* poff = rg.poff;

#pragma unroll
  for (int r = 0; r < S; ++r) rg.issue(c, r, last_use);

  auto process = [&](int r, const uint8_t* st) {
    const int sb = r * NW + c.warp;
    if (r >= rounds || sb >= nsb) return;
    const int J = c.c0 + sb * 32, jm = J + 4 * c.g, jp = J + 8 * c.t4;
    // B fragments of k-tile kk: bh[q] / bl[q] = rows (2 t4, 2 t4 + 1) and
    // (2 t4 + 8, 2 t4 + 9) of column jm + q of Y_0, as an operand-type high
    // part and the operand-type residual of Y_0 - high.
    auto make_b = [&](int kk, uint32_t (&bh)[4][2], uint32_t (&bl)[4][2]) {
      const bool half = HALF && kk == MT - 1;
      float v[4][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (half && e >= 2) {
          v[e][0] = v[e][1] = v[e][2] = v[e][3] = 0.f;
          continue;
        }
        if (c.vec) {
          const float4 t = *reinterpret_cast<const float4*>(st + (4 * kk + e) * 512 + lane * 16);
          v[e][0] = t.x; v[e][1] = t.y; v[e][2] = t.z; v[e][3] = t.w;
          if constexpr (NEST) {  // U = G + beta M': G straight from global memory
            const int kr = 4 * kk + e;
            if (((rg.mok >> kr) & 1u) && jm < c.n) {
              const uint2 graw = *reinterpret_cast<const uint2*>(c.G + rg.moff[kr] + jm);
              const float2 g01 = Mma<__nv_bfloat16>::unpack(graw.x), g23 = Mma<__nv_bfloat16>::unpack(graw.y);
              v[e][0] = fmaf(c.beta, v[e][0], g01.x); v[e][1] = fmaf(c.beta, v[e][1], g01.y);
              v[e][2] = fmaf(c.beta, v[e][2], g23.x); v[e][3] = fmaf(c.beta, v[e][3], g23.y);
            }
          }
        } else {
          const int i = krow(4 * kk + e);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float x = 0.f;
            if (i < c.m && jm + q < c.n) {
              const int64_t o = c.wd.off(i, jm + q);
              x = c.Mp[o];
              if constexpr (NEST) x = fmaf(c.beta, x, __bfloat162float(c.G[o]));
            }
            v[e][q] = x;
          }
        }
      }
      // Y_0 = alpha M' / (||M'|| + eps) in fp32, split as high + residual
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (half && h == 1) {
            bh[q][1] = bl[q][1] = 0u;
            continue;
          }
          const float2 y = __fmul2_rn(make_float2(v[2 * h][q], v[2 * h + 1][q]), inv2);
          bh[q][h] = Mma<TY>::pack(y.x, y.y);
          const float2 yh = Mma<TY>::unpack(bh[q][h]);
          bl[q][h] = Mma<TY>::pack(y.x - yh.x, y.y - yh.y);
        }
      }
    };
    // With several 16-row output tiles, each k-tile's fragments are needed
    // once per output tile, and holding both parts of every k-tile in
    // registers would not fit: on the vector path the first output tile forms
    // them and writes them over this lane's own fp32 rows of the ring slot
    // (the same 64 bytes per k-tile: chunk 4 kk + h holds bh[.][h], chunk
    // 4 kk + 2 + h holds bl[.][h]; a half k-tile has chunks 4 kk + {0, 1}
    // only), and the other output tiles read them back.  The scalar path
    // rebuilds them.
    constexpr bool kStage = MT > 1;
    const bool staged = kStage && c.vec;
    auto store_b = [&](int kk, const uint32_t (&bh)[4][2], const uint32_t (&bl)[4][2]) {
      uint8_t* base = const_cast<uint8_t*>(st) + (4 * kk) * 512 + lane * 16;
      if (HALF && kk == MT - 1) {
        *reinterpret_cast<uint4*>(base) = make_uint4(bh[0][0], bh[1][0], bh[2][0], bh[3][0]);
        *reinterpret_cast<uint4*>(base + 512) = make_uint4(bl[0][0], bl[1][0], bl[2][0], bl[3][0]);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          *reinterpret_cast<uint4*>(base + h * 512) = make_uint4(bh[0][h], bh[1][h], bh[2][h], bh[3][h]);
          *reinterpret_cast<uint4*>(base + (2 + h) * 512) = make_uint4(bl[0][h], bl[1][h], bl[2][h], bl[3][h]);
        }
      }
    };
    auto load_b = [&](int kk, uint32_t (&bh)[4][2], uint32_t (&bl)[4][2]) {
      const uint8_t* base = st + (4 * kk) * 512 + lane * 16;
      if (HALF && kk == MT - 1) {
        const uint4 h0 = *reinterpret_cast<const uint4*>(base);
        const uint4 l0 = *reinterpret_cast<const uint4*>(base + 512);
        bh[0][0] = h0.x; bh[1][0] = h0.y; bh[2][0] = h0.z; bh[3][0] = h0.w;
        bl[0][0] = l0.x; bl[1][0] = l0.y; bl[2][0] = l0.z; bl[3][0] = l0.w;
#pragma unroll
        for (int q = 0; q < 4; ++q) bh[q][1] = bl[q][1] = 0u;
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 hv = *reinterpret_cast<const uint4*>(base + h * 512);
          const uint4 lv = *reinterpret_cast<const uint4*>(base + (2 + h) * 512);
          bh[0][h] = hv.x; bh[1][h] = hv.y; bh[2][h] = hv.z; bh[3][h] = hv.w;
          bl[0][h] = lv.x; bl[1][h] = lv.y; bl[2][h] = lv.z; bl[3][h] = lv.w;
        }
      }
    };
    // up to two output tiles the first one stages the fragments as it goes;
    // with more, a separate pass does (it keeps the registers lower)
    constexpr bool kFuse = MT <= 2;
    if (!kFuse && staged) {
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        uint32_t bh[4][2], bl[4][2];
        make_b(kk, bh, bl);
        store_b(kk, bh, bl);
      }
    }
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      float d[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        uint32_t bh[4][2], bl[4][2];
        if (staged && (mi > 0 || !kFuse)) {
          load_b(kk, bh, bl);
        } else {
          make_b(kk, bh, bl);
          if (staged) store_b(kk, bh, bl);
        }
        // O += Pi_hi Y_hi + Pi_lo Y_hi + Pi_hi Y_lo (Pi_lo Y_lo is below fp32's resolution)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (HALF && kk == MT - 1) {  // rows 8..15 of this k-tile are padding
            Mma<TY>::run8(d[q], ph[mi][kk], bh[q][0]);
            Mma<TY>::run8(d[q], pl[mi][kk], bh[q][0]);
            Mma<TY>::run8(d[q], ph[mi][kk], bl[q][0]);
          } else {
            Mma<TY>::run(d[q], ph[mi][kk], bh[q][0], bh[q][1]);
            Mma<TY>::run(d[q], pl[mi][kk], bh[q][0], bh[q][1]);
            Mma<TY>::run(d[q], ph[mi][kk], bl[q][0], bl[q][1]);
          }
        }
      }
      // rows 16 mi + g (h = 0) and 16 mi + g + 8 (h = 1), columns jp .. jp + 7
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (HALF && mi == MT - 1 && h == 1) continue;
        const int s = 2 * mi + h;
        const int i = orow(s);
        if (i >= c.m || jp >= c.n) continue;
        const float o[8] = {d[0][2 * h], d[1][2 * h], d[2][2 * h], d[3][2 * h],
                            d[0][2 * h + 1], d[1][2 * h + 1], d[2][2 * h + 1], d[3][2 * h + 1]};
        const float coef = c.coef * rs[s], oscale = c.inv_alpha * rs[s];  // row scale of Pi undone
        if (c.vec) {
          const uint4 praw = *reinterpret_cast<const uint4*>(st + (KR + s) * 512 + lane * 16);
          float pf[8];
          bf16x8_to_f32(praw, pf);
          const float2 nc2 = make_float2(-coef, -coef);
          float w[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 wv = __ffma2_rn(nc2, make_float2(o[e], o[e + 1]),
                                         __fmul2_rn(make_float2(pf[e], pf[e + 1]), decay2));
            w[e] = wv.x;
            w[e + 1] = wv.y;
          }
          const int off = poff[s] + jp;
          *reinterpret_cast<uint4*>(c.P + off) = f32_to_bf16x8(w);
          if (c.dbg) {
            float* dp = c.dbg + off;
            *reinterpret_cast<float4*>(dp) =
                make_float4(o[0] * oscale, o[1] * oscale, o[2] * oscale, o[3] * oscale);
            *reinterpret_cast<float4*>(dp + 4) =
                make_float4(o[4] * oscale, o[5] * oscale, o[6] * oscale, o[7] * oscale);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (jp + e >= c.n) continue;
            const int64_t off = c.wd.off(i, jp + e);
            c.P[off] = __float2bfloat16_rn(fmaf(-coef, o[e], __bfloat162float(c.P[off]) * c.decay));
            if (c.dbg) c.dbg[off] = o[e] * oscale;
          }
        }
      }
    }
  };

  for (int r = 0; r < rounds; ++r) {
    cp_async_wait<S - 1>();
    uint8_t* st = ring_warp + Ring::slot(r) * kSlot;
    process(r, st);
    // round r now lives in registers / is written: refill its slot
    rg.issue(c, r + S, last_use);
  }
  cp_async_wait<0>();
}

// Output pass of a transposed member (parameter [n, m], m % 8 == 0): each
// superblock is parameter rows J .. J + 31, staged as one contiguous block of
// M' (row pitch m floats) and one of P (row pitch m bf16) in the warp's ring
// slot.  In the parameter's layout the update is O_par = Y_par Pi^T with
// Y_par = alpha M'_par / (||M'|| + eps), so the data is the MMA's A operand
// (rows: parameter rows, K: parameter columns) and Pi^T the constant B
// operand.  Row tile ct (0, 1) covers rows J + 16 ct .. + 15; the accumulator
// of n-tile nt holds rows J + 16 ct + g (+ 8), columns 8 nt + 2 t4 (+ 1).
// Y is split into an operand-type high part and residual as on the vector
// path; P' is formed in the staged P block and written back as the block.
template <typename TY, int MT, int NT, bool HALF>
__device__ __forceinline__ void gs_out_pass_t(const GsCtx& c, uint8_t* ring,
                                              const uint32_t (&bh)[MT][GsLayout<MT, NT, HALF>::NJ][2],
                                              const uint32_t (&bl)[MT][GsLayout<MT, NT, HALF>::NJ][2],
                                              const float* rsc) {
  using L = GsLayout<MT, NT, HALF>;
  constexpr int NW = L::NW, S = L::SO, LB = L::LBO, NJ = L::NJ;
  constexpr uint32_t kSlot = NW * 32 * LB;
  static_assert(192 * 16 * MT - (HALF ? 192 * 8 : 0) <= 32 * LB, "transposed block exceeds the slot");
  const int lane = c.lane, m = c.m, mq = m / 4;
  uint8_t* ring_warp = ring + c.warp * 32 * LB;
  const uint32_t ring0 = smem_u32(ring_warp);
  const int nsb = c.NB / 2, rounds = (nsb + NW - 1) / NW;
  const uint64_t last_use = l2_evict_first();
  const float2 decay2 = make_float2(c.decay, c.decay);

  auto issue = [&](int r) {
    const int sb = r * NW + c.warp;
    if (r < rounds && sb < nsb) {
      const uint32_t dst = ring0 + (r % S) * kSlot;
      const int J = c.c0 + sb * 32, nrows = min(32, c.n - J);
      const float* mb = c.Mp + (int64_t)J * m;
      const __nv_bfloat16* pb = c.P + (int64_t)J * m;
      for (int k = lane; k < 8 * m; k += 32) {
        const bool ok = k / mq < nrows;
        cp_async16_hint(dst + k * 16, ok ? (const void*)(mb + 4 * k) : (const void*)c.Mp, ok ? 16 : 0,
                        last_use);
      }
      for (int k = lane; k < 4 * m; k += 32) {
        const bool ok = 2 * k / mq < nrows;
        cp_async16_hint(dst + 128 * m + k * 16, ok ? (const void*)(pb + 8 * k) : (const void*)c.P,
                        ok ? 16 : 0, last_use);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int r = 0; r < S; ++r) issue(r);

  // with four 16-row tiles, one row tile at a time keeps the accumulators
  // within the register budget
  constexpr int NCT = MT >= 3 ? 1 : 2;
  for (int r = 0; r < rounds; ++r) {
    cp_async_wait<S - 1>();
    __syncwarp();  // every lane's copies of this round have landed
    uint8_t* st = ring_warp + (r % S) * kSlot;
    const int sb = r * NW + c.warp;
    if (sb < nsb) {
      const int J = c.c0 + sb * 32, nrows = min(32, c.n - J);
      const float* ym = reinterpret_cast<const float*>(st);
      __nv_bfloat16* pm = reinterpret_cast<__nv_bfloat16*>(st + 128 * m);
#pragma unroll
      for (int c0 = 0; c0 < 2; c0 += NCT) {
        float d[NCT][NJ][4];
#pragma unroll
        for (int ct = 0; ct < NCT; ++ct)
#pragma unroll
          for (int nt = 0; nt < NJ; ++nt) d[ct][nt][0] = d[ct][nt][1] = d[ct][nt][2] = d[ct][nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
          const bool half = HALF && kk == MT - 1;
#pragma unroll
          for (int ct = 0; ct < NCT; ++ct) {
            // a[f]: rows (16 ct + g, + 8) x columns (16 kk + 2 t4, + 8), pairs of columns
            uint32_t ah[4], al[4];
#pragma unroll
            for (int f = 0; f < 4; ++f) {
              const int row = 16 * (c0 + ct) + c.g + ((f & 1) ? 8 : 0);
              const int col = 16 * kk + 2 * c.t4 + ((f & 2) ? 8 : 0);
              float2 y = make_float2(0.f, 0.f);
              if (!(half && (f & 2)) && col < m)
                y = *reinterpret_cast<const float2*>(ym + row * m + col);
              y = __fmul2_rn(y, make_float2(c.inv, c.inv));
              ah[f] = Mma<TY>::pack(y.x, y.y);
              const float2 yh = Mma<TY>::unpack(ah[f]);
              al[f] = Mma<TY>::pack(y.x - yh.x, y.y - yh.y);
            }
#pragma unroll
            for (int nt = 0; nt < NJ; ++nt) {
              if (half) {  // columns 8..15 of this k-tile are padding
                Mma<TY>::run8(d[ct][nt], ah, bh[kk][nt][0]);
                Mma<TY>::run8(d[ct][nt], ah, bl[kk][nt][0]);
                Mma<TY>::run8(d[ct][nt], al, bh[kk][nt][0]);
              } else {
                Mma<TY>::run(d[ct][nt], ah, bh[kk][nt][0], bh[kk][nt][1]);
                Mma<TY>::run(d[ct][nt], ah, bl[kk][nt][0], bl[kk][nt][1]);
                Mma<TY>::run(d[ct][nt], al, bh[kk][nt][0], bh[kk][nt][1]);
              }
            }
          }
        }
        // P' = P (1 - lr wd) - lr s O in the staged block; O's column i
        // carries Pi's row scale rsc[i]
#pragma unroll
        for (int ct = 0; ct < NCT; ++ct)
#pragma unroll
          for (int nt = 0; nt < NJ; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = 16 * (c0 + ct) + c.g + 8 * h, col = 8 * nt + 2 * c.t4;
              if (row >= nrows || col >= m) continue;
              const float s0 = rsc[col], s1 = rsc[col + 1];
              const float o0 = d[ct][nt][2 * h], o1 = d[ct][nt][2 * h + 1];
              __nv_bfloat162* pp = reinterpret_cast<__nv_bfloat162*>(pm + row * m + col);
              const float2 pv = __bfloat1622float2(*pp);
              const float2 w = __ffma2_rn(make_float2(-c.coef * s0, -c.coef * s1), make_float2(o0, o1),
                                          __fmul2_rn(pv, decay2));
              *pp = __floats2bfloat162_rn(w.x, w.y);
              if (c.dbg) {
                float* dp = c.dbg + (int64_t)(J + row) * m + col;
                dp[0] = o0 * c.inv_alpha * s0;
                dp[1] = o1 * c.inv_alpha * s1;
              }
            }
      }
      __syncwarp();  // the block is complete: P' out as the contiguous block
      __nv_bfloat16* pb = c.P + (int64_t)J * m;
      for (int k = lane; k < 4 * m; k += 32)
        if (2 * k / mq < nrows)
          *reinterpret_cast<uint4*>(pb + 8 * k) = *reinterpret_cast<const uint4*>(st + 128 * m + k * 16);
    }
    __syncwarp();  // the slot is read out before it is refilled
    issue(r + S);
  }
  cp_async_wait<0>();
}

// An m x m fp32 matrix kept as two tf32 parts, x = hi + lo (both exact
// tf32 values, pitch LD), so that the tensor-core products below read their
// operands already split.
struct SplitMat {
  uint32_t* hi;
  uint32_t* lo;
};
template <int LD>
__device__ __forceinline__ void put(const SplitMat& X, int i, int j, float v) {
  const uint32_t h = to_tf32(v);
  X.hi[i * LD + j] = h;
  X.lo[i * LD + j] = to_tf32(v - __uint_as_float(h));
}
template <int LD>
__device__ __forceinline__ float get(const SplitMat& X, int i, int j) {
  return __uint_as_float(X.hi[i * LD + j]) + __uint_as_float(X.lo[i * LD + j]);
}

// One m16 x n8 tile of C = X Y (MP x MP, zero beyond m), on the tensor cores
// with the 3xTF32 split: x y ~ x_hi y_hi + x_hi y_lo + x_lo y_hi (the dropped
// x_lo y_lo is ~2^-22 relative).  k8 steps beyond m (ks of them are live)
// are skipped.  d[0..3] = C at rows 16 mi + g (+ 8), columns 8 nj + 2 t4
// (+ 1).
template <int MP, int LD>
__device__ __forceinline__ void mm_tile(const SplitMat& X, const SplitMat& Y, int tile, int ks, int g,
                                        int t4, float (&d)[4]) {
  const int mi = tile / (MP / 8), nj = tile % (MP / 8);
  // one accumulator per k8 step: independent chains of three products,
  // summed in a fixed order at the end (the stage is latency-bound)
  float acc[MP / 8][4];
#pragma unroll
  for (int kk = 0; kk < MP / 8; ++kk) {
    acc[kk][0] = acc[kk][1] = acc[kk][2] = acc[kk][3] = 0.f;
    if (kk < ks) {
      const int xo = (mi * 16 + g) * LD + kk * 8 + t4;
      const int yo = (kk * 8 + t4) * LD + nj * 8 + g;
      const uint32_t ah0 = X.hi[xo], ah1 = X.hi[xo + 8 * LD], ah2 = X.hi[xo + 4], ah3 = X.hi[xo + 8 * LD + 4];
      const uint32_t al0 = X.lo[xo], al1 = X.lo[xo + 8 * LD], al2 = X.lo[xo + 4], al3 = X.lo[xo + 8 * LD + 4];
      const uint32_t bh0 = Y.hi[yo], bh1 = Y.hi[yo + 4 * LD], bl0 = Y.lo[yo], bl1 = Y.lo[yo + 4 * LD];
      mma_tf32(acc[kk], al0, al1, al2, al3, bh0, bh1);
      mma_tf32(acc[kk], ah0, ah1, ah2, ah3, bl0, bl1);
      mma_tf32(acc[kk], ah0, ah1, ah2, ah3, bh0, bh1);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float v = acc[0][q];
#pragma unroll
    for (int kk = 1; kk < MP / 8; ++kk) v += acc[kk][q];
    d[q] = v;
  }
}

// The m x m stage in plain fp32 (FFMA), for m > 32.  Every left operand there (A, Q and
// Q^2) is symmetric, so C = X Y is formed as C[i][j] = sum_k X[k][i] Y[k][j]:
// both operands read by rows, k ascending, one fixed order per element.
// Thread t < 256 owns the RI x CJ block at rows RI (t / BJ) + r, columns
// CJ (t % BJ) + c.
template <int MP, int NT>
struct MmBlk {
  static constexpr int RI = MP / 16, CJ = RI;
  static constexpr int BI = MP / RI, BJ = MP / CJ;
  static_assert(BI * BJ <= NT, "one block per thread");
};

template <int N>
__device__ __forceinline__ void lds_run(const float* p, float (&v)[N]) {
  if constexpr (N == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else if constexpr (N == 2) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = p[e];
  }
}

// acc[y] = this thread's block of X^T Y_y over k < m, for NY right operands
// sharing the left one.
template <int LD, int RI, int CJ, int NY>
__device__ __forceinline__ void mm_blk(const float* X, const float* const (&Y)[NY], int m, int i0, int j0,
                                       float (&acc)[NY][RI][CJ]) {
#pragma unroll
  for (int y = 0; y < NY; ++y)
#pragma unroll
    for (int r = 0; r < RI; ++r)
#pragma unroll
      for (int c = 0; c < CJ; ++c) acc[y][r][c] = 0.f;
#pragma unroll 2
  for (int k = 0; k < m; ++k) {
    float x[RI];
    lds_run<RI>(X + k * LD + i0, x);
#pragma unroll
    for (int y = 0; y < NY; ++y) {
      float v[CJ];
      lds_run<CJ>(Y[y] + k * LD + j0, v);
#pragma unroll
      for (int r = 0; r < RI; ++r) {
        if constexpr (CJ % 2 == 0) {
#pragma unroll
          for (int c = 0; c < CJ; c += 2) {
            const float2 t = __ffma2_rn(make_float2(x[r], x[r]), make_float2(v[c], v[c + 1]),
                                        make_float2(acc[y][r][c], acc[y][r][c + 1]));
            acc[y][r][c] = t.x;
            acc[y][r][c + 1] = t.y;
          }
        } else {
#pragma unroll
          for (int c = 0; c < CJ; ++c) acc[y][r][c] = fmaf(x[r], v[c], acc[y][r][c]);
        }
      }
    }
  }
}

// The m x m work arrays A, Q, T, Pi (two): matrix k at base, either split
// into tf32 high / low parts (tensor-core form, m <= 32) or plain fp32.
template <int MP, int LD, bool TC>
struct MmMats {
  uint32_t* base;
  static constexpr int kWords = (TC ? 10 : 5) * MP * LD;
  __device__ __forceinline__ SplitMat split(int k) const {
    return SplitMat{base + (2 * k) * MP * LD, base + (2 * k + 1) * MP * LD};
  }
  __device__ __forceinline__ float* plain(int k) const { return reinterpret_cast<float*>(base) + k * MP * LD; }
  __device__ __forceinline__ float get(int k, int i, int j) const {
    if constexpr (TC) return ::muon::gs::get<LD>(split(k), i, j);
    else return plain(k)[i * LD + j];
  }
  __device__ __forceinline__ void put(int k, int i, int j, float v) const {
    if constexpr (TC) ::muon::gs::put<LD>(split(k), i, j, v);
    else plain(k)[i * LD + j] = v;
  }
};

template <typename TY, int MT, int NT, bool HALF, int VAR>
__global__ void __launch_bounds__(NT, (MT <= 2 && NT == 256) ? 2 : 1)
    k_skinny_gs(KArgs a, int W, int NB, int LS) {
  constexpr bool NEST = VAR == kVarNesterov, TP = VAR == kVarTransposed;
  using L = GsLayout<MT, NT, HALF>;
  using GT = typename L::GT;
  constexpr int MP = L::MP, LD = L::LD, NW = L::NW;
  extern __shared__ __align__(128) uint8_t smem[];
  float* cpart = reinterpret_cast<float*>(smem + L::kCta);
  float* misc = reinterpret_cast<float*>(smem + L::kMisc);
  float* rsc = reinterpret_cast<float*>(smem + L::kRsc);         // per-row power-of-two scale of Pi
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + L::kTabOff);  // upper triangle (i << 16 | j)
  float* coef = reinterpret_cast<float*>(smem + L::kCoefOff);        // the schedule's rows

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const int CL = (int)cluster_size();  // CTAs (column shards) per member
  const int b = blockIdx.x / CL;
  const int m = a.m;
  const MemberPtrs mp = a.mem[b];

  GsCtx c;
  c.lane = lane; c.warp = warp; c.g = lane >> 2; c.t4 = lane & 3;
  c.m = m; c.n = a.n; c.c0 = (int)rank * W; c.NB = NB;
  c.Mp = mp.M;
  c.G = static_cast<const __nv_bfloat16*>(mp.G);
  c.P = static_cast<__nv_bfloat16*>(mp.P);
  const bool T = mp.T != 0;  // this member's parameter is [n, m]
  c.cols = T ? m : a.n;      // the parameter's row pitch
  c.wd = Wide{c.cols, (int)T};
  c.vec = !T && (c.cols % 8 == 0) && 32ll * c.cols < (1ll << 31) && aligned16(c.Mp) &&
          aligned16(c.G) && aligned16(c.P);
  c.tvec = TP && T && m % 8 == 0 && (int64_t)a.n * m < (1ll << 31) && aligned16(c.Mp) &&
           aligned16(c.G) && aligned16(c.P);
  c.dbg = a.dbg ? a.dbg + (int64_t)b * m * a.n : nullptr;
  const int ns = a.sc->ns_steps;
  c.beta = a.sc->beta;
  const float lr = a.sc->lr;
  c.decay = __fmaf_rn(-lr, a.sc->wd, 1.f);  // one rounding of 1 - lr wd
  c.inv_alpha = 1.f / a.alpha;
  c.coef = lr * mp.scale * c.inv_alpha;

  // m x m work arrays (aliasing the ring between the two passes)
  float* wpart = reinterpret_cast<float*>(smem);
  float* wss = wpart + NW * GT::N * 128;
  using Mats = MmMats<MP, LD, L::TC>;
  const Mats mats{reinterpret_cast<uint32_t*>(smem)};
  TY* Ph = reinterpret_cast<TY*>(smem + Mats::kWords * 4);
  TY* Pl = Ph + MP * (MP + 8);
  int ip = 3;  // matrix index of the final Pi (3 or 4)
  const int n_coef = min(max(a.sc->n_coef, 1), kMaxScheduleRows);
  for (int e = tid; e < 3 * n_coef; e += NT) coef[e] = a.sc->coef[e / 3][e % 3];
  // (a, b, c) of step s: row s, the last row past the end
  auto step_abc = [&](int s) { return coef + 3 * min(s, n_coef - 1); };
  const int nup = m * (m + 1) / 2;
  for (int e = tid; e < nup; e += NT) {
    // e -> (i, j), i <= j, row-major over the upper triangle
    int i = 0, rem = e;
    while (rem >= m - i) { rem -= m - i; ++i; }
    tab[e] = (uint32_t)(i << 16 | (i + rem));
  }

  // 1. momentum, sum of squares and Gram matrix
  float gacc[GT::N][4];
#pragma unroll
  for (int q = 0; q < GT::N; ++q) gacc[q][0] = gacc[q][1] = gacc[q][2] = gacc[q][3] = 0.f;
  float ss = 0.f;
  gs_momentum_pass<MT, NT, HALF, VAR>(c, smem, gacc, ss, LS);
  // Hint: move this CTA's slice of P into L2 while the m x m work runs.
  if (c.vec && warp == NW - 1 && c.c0 < c.n) {
    const int ncol = min(W, c.n - c.c0);
    const uint32_t bytes = (uint32_t)(ncol * 2) & ~15u;
    if (bytes)
      for (int i = lane; i < m; i += 32) prefetch_l2(c.P + (int64_t)i * c.cols + c.c0, bytes);
  }
  __syncthreads();  // every warp's ring is drained before it is reused
  // per-warp (leaf) partials, then this CTA's partial as the binary tree
  // over its warps' leaves, then (below) the cluster's as the binary tree
  // over its CTAs: one fixed tree over all CL x NW leaves, whatever CL and NW
  ss = warp_sum(ss);
  if (lane == 0) wss[warp] = ss;
#pragma unroll
  for (int q = 0; q < GT::N; ++q) {
    float* dst = wpart + (warp * GT::N + q) * 128;
    dst[c.g * 8 + 2 * c.t4] = gacc[q][0];
    dst[c.g * 8 + 2 * c.t4 + 1] = gacc[q][1];
    dst[(c.g + 8) * 8 + 2 * c.t4] = gacc[q][2];
    dst[(c.g + 8) * 8 + 2 * c.t4 + 1] = gacc[q][3];
  }
  __syncthreads();
  for (int e = tid; e < GT::N * 128; e += NT) {
    const int q = e >> 7, w = e & 127;
    float v[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) v[k] = wpart[(k * GT::N + q) * 128 + w];
    const int code = GT::code(q);
    cpart[((code >> 4) * 16 + (w >> 3)) * MP + (code & 15) * 8 + (w & 7)] = tree_sum<NW>(v);
  }
  if (tid == 0) {
    float v[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) v[k] = wss[k];
    misc[0] = tree_sum<NW>(v);
  }
  cluster_sync();  // (also a CTA barrier: the partials are consumed)
  for (int e = tid; e < Mats::kWords; e += NT) mats.base[e] = 0u;  // m x m arrays, padding included
  __syncthreads();
  // the norm, then A_0 = M' M'^T / (||M'||_F + eps)^2: the CTAs' partials
  // combined by the binary tree over ranks
  const float ssum = cluster_tree_sum(&misc[0], CL);
  const float inv_raw = 1.f / (sqrtf(ssum) + a.eps);
  c.inv = a.alpha * inv_raw;
  const float inv2 = inv_raw * inv_raw;
  for (int e = tid; e < nup; e += NT) {
    const int i = tab[e] >> 16, j = tab[e] & 0xffff;
    const float acc = cluster_tree_sum(&cpart[i * MP + j], CL) * inv2;
    mats.put(0, i, j, acc);
    mats.put(0, j, i, acc);
  }
  cluster_arrive();  // done reading the peer's partials
  __syncthreads();

  // 2. the k steps in m x m space: for m <= 32 m16 x n8 tiles dealt to the
  // warps on the tensor cores (3xTF32; the stage is latency-bound there),
  // else fp32 FFMA blocks, one per thread (throughput-bound)
  if (ns > 0) {
    if constexpr (L::TC) {
      constexpr int TPP = (MP / 16) * (MP / 8);  // tiles of one product
      SplitMat Am = mats.split(0), Qm = mats.split(1), Tm = mats.split(2), Pi0 = mats.split(3);
      SplitMat Pi1 = mats.split(4), Pi = Pi0;
      const int ks = (m + 7) / 8;  // live k8 steps
      // a tile wholly beyond m (rows or columns) stays zero and is skipped
      auto live = [&](int tile) { return (tile / (MP / 8)) * 16 < m && (tile % (MP / 8)) * 8 < m; };
      // element (i, j) of this lane's accumulator slot q in tile `tile`
      auto at = [&](int tile, int q, int& i, int& j) {
        i = (tile / (MP / 8)) * 16 + c.g + ((q & 2) ? 8 : 0);
        j = (tile % (MP / 8)) * 8 + 2 * c.t4 + (q & 1);
      };
      for (int s = 0; s < ns; ++s) {
        const bool more = s + 1 < ns;
        const float* cf = step_abc(s);
        const float ca = cf[0], cb = cf[1], cc = cf[2];
        // Q = a I + b A + c A^2 (zero outside m x m)
        for (int tile = warp; tile < TPP; tile += NW) {
          if (!live(tile)) continue;
          float d[4];
          mm_tile<MP, LD>(Am, Am, tile, ks, c.g, c.t4, d);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            int i, j;
            at(tile, q, i, j);
            float v = 0.f;
            if (i < m && j < m) v = fmaf(cc, d[q], fmaf(cb, get<LD>(Am, i, j), i == j ? ca : 0.f));
            put<LD>(Qm, i, j, v);
          }
        }
        __syncthreads();
        // Pi <- Q Pi (Pi_1 = Q_0) and T = Q^2 (needed for the next A)
        SplitMat Pn = Pi.hi == Pi0.hi ? Pi1 : Pi0;
        for (int t = warp; t < 2 * TPP; t += NW) {
          if (t < TPP) {
            if (!more || !live(t)) continue;
            float d[4];
            mm_tile<MP, LD>(Qm, Qm, t, ks, c.g, c.t4, d);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              int i, j;
              at(t, q, i, j);
              put<LD>(Tm, i, j, d[q]);
            }
            continue;
          }
          const int tile = t - TPP;
          if (!live(tile)) continue;
          float d[4];
          if (s > 0) mm_tile<MP, LD>(Qm, Pi, tile, ks, c.g, c.t4, d);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            int i, j;
            at(tile, q, i, j);
            if (s > 0) {
              put<LD>(Pn, i, j, d[q]);
            } else {
              Pn.hi[i * LD + j] = Qm.hi[i * LD + j];
              Pn.lo[i * LD + j] = Qm.lo[i * LD + j];
            }
          }
        }
        Pi = Pn;
        __syncthreads();
        if (more) {
          // A <- Q^2 A (written over Q, then the two swap roles)
          for (int tile = warp; tile < TPP; tile += NW) {
            if (!live(tile)) continue;
            float d[4];
            mm_tile<MP, LD>(Tm, Am, tile, ks, c.g, c.t4, d);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              int i, j;
              at(tile, q, i, j);
              put<LD>(Qm, i, j, d[q]);
            }
          }
          const SplitMat t = Am; Am = Qm; Qm = t;
          __syncthreads();
        }
      }
      ip = Pi.hi == Pi0.hi ? 3 : 4;
    } else {
      using B = MmBlk<MP, NT>;
      constexpr int RI = B::RI, CJ = B::CJ;
      const int i0 = RI * (tid / B::BJ), j0 = CJ * (tid % B::BJ);
      const bool own = tid < B::BI * B::BJ;
      // this thread's block into C, zero outside m x m
      auto store = [&](float* C, const float (&v)[RI][CJ]) {
#pragma unroll
        for (int r = 0; r < RI; ++r)
#pragma unroll
          for (int q = 0; q < CJ; ++q) {
            const int i = i0 + r, j = j0 + q;
            C[i * LD + j] = (i < m && j < m) ? v[r][q] : 0.f;
          }
      };
      float *Am = mats.plain(0), *Qm = mats.plain(1), *Tm = mats.plain(2);
      float *Pi0 = mats.plain(3), *Pi1 = mats.plain(4), *Pi = Pi0;
      for (int s = 0; s < ns; ++s) {
        const bool more = s + 1 < ns;
        const float* cf = step_abc(s);
        const float ca = cf[0], cb = cf[1], cc = cf[2];
        // Q = a I + b A + c A^2
        if (own) {
          float acc[1][RI][CJ];
          mm_blk<LD, RI, CJ, 1>(Am, {Am}, m, i0, j0, acc);
#pragma unroll
          for (int r = 0; r < RI; ++r)
#pragma unroll
            for (int q = 0; q < CJ; ++q) {
              const int i = i0 + r, j = j0 + q;
              acc[0][r][q] = fmaf(cc, acc[0][r][q], fmaf(cb, Am[i * LD + j], i == j ? ca : 0.f));
            }
          store(Qm, acc[0]);
        }
        __syncthreads();
        // Pi <- Q Pi (Pi_1 = Q_0) and T = Q^2 (needed for the next A)
        float* Pn = Pi == Pi0 ? Pi1 : Pi0;
        if (own) {
          if (s > 0 && more) {
            float acc[2][RI][CJ];
            mm_blk<LD, RI, CJ, 2>(Qm, {Qm, Pi}, m, i0, j0, acc);
            store(Tm, acc[0]);
            store(Pn, acc[1]);
          } else if (s > 0) {
            float acc[1][RI][CJ];
            mm_blk<LD, RI, CJ, 1>(Qm, {Pi}, m, i0, j0, acc);
            store(Pn, acc[0]);
          } else {
            if (more) {
              float acc[1][RI][CJ];
              mm_blk<LD, RI, CJ, 1>(Qm, {Qm}, m, i0, j0, acc);
              store(Tm, acc[0]);
            }
#pragma unroll
            for (int r = 0; r < RI; ++r)
#pragma unroll
              for (int q = 0; q < CJ; ++q) Pn[(i0 + r) * LD + j0 + q] = Qm[(i0 + r) * LD + j0 + q];
          }
        }
        Pi = Pn;
        __syncthreads();
        if (more) {
          // A <- Q^2 A (written over Q, then the two swap roles)
          if (own) {
            float acc[1][RI][CJ];
            mm_blk<LD, RI, CJ, 1>(Tm, {Am}, m, i0, j0, acc);
            store(Qm, acc[0]);
          }
          float* t = Am; Am = Qm; Qm = t;
          __syncthreads();
        }
      }
      ip = Pi == Pi0 ? 3 : 4;
    }
    // Along an exact null direction of X_0 (a zero row, say) Pi grows like
    // a^k while O does not: scale each row i of Pi by 2^-e_i into the operand
    // type's range, and O's row i by 2^e_i in the epilogue.
    for (int i = warp; i < MP; i += NW) {  // one warp per row: lanes over columns
      float mx = 0.f;
      for (int k = lane; k < m && i < m; k += 32) mx = fmaxf(mx, fabsf(mats.get(ip, i, k)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const int ex = mx >= 32768.f ? ((__float_as_int(mx) >> 23) & 0xff) - 127 - 14 : 0;
      if (lane == 0) rsc[i] = exp2f((float)ex);
    }
    __syncthreads();
    // Pi in the operand type: high part and residual, zero outside m x m
    for (int e = tid; e < MP * MP; e += NT) {
      const int i = e / MP, j = e - (e / MP) * MP;
      float v = 0.f;
      if (i < m && j < m) v = mats.get(ip, i, j) / rsc[i];
      const TY hi = from_f32<TY>(v);
      Ph[i * (MP + 8) + j] = hi;
      Pl[i * (MP + 8) + j] = from_f32<TY>(v - to_f32(hi));
    }
  } else {
    // no step: O = X_0 (Pi = I, exact in the operand type)
    for (int i = tid; i < MP; i += NT) rsc[i] = 1.f;
    for (int e = tid; e < MP * MP; e += NT) {
      const int i = e / MP, j = e - (e / MP) * MP;
      Ph[i * (MP + 8) + j] = from_f32<TY>(i == j && i < m ? 1.f : 0.f);
      Pl[i * (MP + 8) + j] = from_f32<TY>(0.f);
    }
  }
  __syncthreads();
  if (TP && c.tvec) {
    // Pi^T as the B operand of the transposed member's product:
    // tb_h[kk][nt] = Pi[8 nt + g][16 kk + 2 t4 (+1)] and [16 kk + 8 + 2 t4 (+1)]
    constexpr int NJ = L::NJ;
    uint32_t tb_h[MT][NJ][2], tb_l[MT][NJ][2];
    const uint32_t hb = smem_u32(Ph), lb = smem_u32(Pl);
#pragma unroll
    for (int kk = 0; kk < MT; ++kk)
#pragma unroll
      for (int nt = 0; nt < NJ; ++nt) {
        const uint32_t o = 2u * ((nt * 8 + (lane & 7)) * (MP + 8) + kk * 16 + ((lane >> 3) & 1) * 8);
        ldsm_x2(hb + o, tb_h[kk][nt]);
        ldsm_x2(lb + o, tb_l[kk][nt]);
      }
    __syncthreads();  // the ring's bytes are reused by the output pass
    gs_out_pass_t<TY, MT, NT, HALF>(c, smem, tb_h, tb_l, rsc);
    cluster_wait();  // the peer may still read this CTA's partials
    return;
  }
  uint32_t ph[MT][MT][4], pl[MT][MT][4];
  {
    const uint32_t hb = smem_u32(Ph), lb = smem_u32(Pl);
#pragma unroll
    for (int mi = 0; mi < MT; ++mi)
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        const uint32_t o = 2u * ((mi * 16 + (lane & 15)) * (MP + 8) + kk * 16 + (lane >> 4) * 8);
        ldsm_x4(hb + o, ph[mi][kk]);
        ldsm_x4(lb + o, pl[mi][kk]);
      }
  }
  float rs[L::R];
#pragma unroll
  for (int s = 0; s < L::R; ++s) rs[s] = rsc[(s >> 1) * 16 + c.g + ((s & 1) ? 8 : 0)];
  __syncthreads();  // the ring's bytes are reused by the output pass

  // 3. O = Pi_k Y_0 and the parameter write
  gs_out_pass<TY, MT, NT, HALF, NEST>(c, smem, ph, pl, rs);
  cluster_wait();  // the peer may still read this CTA's partials
}

// Threads per CTA: 16 warps up to m = 32; beyond, 8 warps, each with the
// registers for Pi's fragments of all 16-row tiles.
template <int MT>
constexpr int gs_threads() { return MT <= 2 ? 512 : 256; }

inline int gs_num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

// One launch in clusters of CL CTAs of NT threads.  The member's superblocks
// go to CL x NW leaves of LS consecutive superblocks each (the last ones
// possibly short or empty), warp w of CTA r taking leaf r NW + w; each CTA
// spans NW LS superblocks.
template <typename TY, int MT, int NT, bool HALF, int VAR>
cudaError_t launch_gs_cl(const KArgs& a, int CL, cudaStream_t st) {
  auto fn = k_skinny_gs<TY, MT, NT, HALF, VAR>;
  constexpr int NW = NT / 32;
  const int sg = (a.n + 31) / 32;
  const int LS = (sg + CL * NW - 1) / (CL * NW);
  const int W = NW * LS * 32;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(a.B * CL);
  lc.blockDim = dim3(NT);
  lc.dynamicSmemBytes = GsLayout<MT, NT, HALF>::kTotal;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, fn, a, W, W / 16, LS);
}

// For m <= 32 with the shard count left to the library, a batch too small
// to fill the GPU with 2-CTA clusters of 16 warps runs 4-CTA clusters of 8
// warps (two CTAs per SM): 32 leaves either way, so the reduction tree and
// every bit of the result are the same, and twice the SMs share the work.
template <typename TY, int MT, bool HALF, int VAR>
cudaError_t launch_gs_t(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prepare) {
  constexpr int NT = gs_threads<MT>();
  if (prepare) {
    cudaError_t e = cudaFuncSetAttribute(k_skinny_gs<TY, MT, NT, HALF, VAR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GsLayout<MT, NT, HALF>::kTotal);
    if constexpr (MT <= 2) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_skinny_gs<TY, MT, 256, HALF, VAR>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GsLayout<MT, 256, HALF>::kTotal);
    }
    return e;
  }
  if constexpr (MT <= 2) {
    if (cfg.auto_shards && cfg.cluster == 2 && 8 * 2 * a.B < 7 * gs_num_sms())
      return launch_gs_cl<TY, MT, 256, HALF, VAR>(a, 4, st);
  }
  return launch_gs_cl<TY, MT, NT, HALF, VAR>(a, cfg.cluster, st);
}

template <typename TY, int MT, bool HALF, int VAR>
int gs_clusters_of(int cl) {
  constexpr int NT = gs_threads<MT>();
  auto fn = k_skinny_gs<TY, MT, NT, HALF, VAR>;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(cl * 1024);
  lc.blockDim = dim3(NT);
  lc.dynamicSmemBytes = GsLayout<MT, NT, HALF>::kTotal;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, fn, &lc) == cudaSuccess ? n : -1;
}

// HALF (a last 16-row tile of at most 8 rows, stored as half a tile) is
// instantiated up to m = 32; beyond, such a tile is padded to 16 rows.
template <typename TY, int VAR>
cudaError_t gs_launch_ty(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prep) {
  const bool half = a.m - 16 * (cfg.mtiles - 1) <= 8;
  switch (cfg.mtiles) {
    case 1:
      return half ? launch_gs_t<TY, 1, true, VAR>(a, cfg, st, prep) : launch_gs_t<TY, 1, false, VAR>(a, cfg, st, prep);
    case 2:
      return half ? launch_gs_t<TY, 2, true, VAR>(a, cfg, st, prep) : launch_gs_t<TY, 2, false, VAR>(a, cfg, st, prep);
    case 3: return launch_gs_t<TY, 3, false, VAR>(a, cfg, st, prep);
    default: return launch_gs_t<TY, 4, false, VAR>(a, cfg, st, prep);
  }
}

template <typename TY, int VAR>
int gs_clusters_ty(int m, int cl) {
  const int mt = (m + 15) / 16;
  const bool half = m - 16 * (mt - 1) <= 8;
  switch (mt) {
    case 1: return half ? gs_clusters_of<TY, 1, true, VAR>(cl) : gs_clusters_of<TY, 1, false, VAR>(cl);
    case 2: return half ? gs_clusters_of<TY, 2, true, VAR>(cl) : gs_clusters_of<TY, 2, false, VAR>(cl);
    case 3: return gs_clusters_of<TY, 3, false, VAR>(cl);
    default: return gs_clusters_of<TY, 4, false, VAR>(cl);
  }
}

// The launcher and occupancy query of one kernel variant (each variant is
// instantiated in its own translation unit).
template <int VAR>
cudaError_t gs_dispatch_t(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  if (a.mode_f32 || cfg.mtiles < 1 || cfg.mtiles > 4) return cudaErrorInvalidValue;
  return a.ns_type == NS_F16 ? gs_launch_ty<__half, VAR>(a, cfg, s, prepare)
                             : gs_launch_ty<__nv_bfloat16, VAR>(a, cfg, s, prepare);
}
// The same for one operand type only (a variant split over two translation
// units to keep each one's compile time short).
template <typename TY, int VAR>
cudaError_t gs_dispatch_ty(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare) {
  if (a.mode_f32 || cfg.mtiles < 1 || cfg.mtiles > 4) return cudaErrorInvalidValue;
  return gs_launch_ty<TY, VAR>(a, cfg, s, prepare);
}

template <int VAR>
int gs_clusters_t(int ns_type, int m, int cl) {
  if (m < 1 || m > 64) return -1;
  return ns_type == NS_F16 ? gs_clusters_ty<__half, VAR>(m, cl) : gs_clusters_ty<__nv_bfloat16, VAR>(m, cl);
}

}  // namespace gs
}  // namespace muon
