// Skinny path, direct iteration: Newton-Schulz for m = min(rows, cols) <= 64,
// one pass over the m x n iterate per step.  It serves step counts beyond the
// Gram-space kernel's range (k_skinny_gs.cuh); the host functions at the end
// choose between the two.
//
// «MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化: for
// shapes such as [24, 10240] the per-parameter iteration is dominated by host
// dispatch, small allocations and synchronisation; batching every member of a
// shape into one launch removes that (Fig. 7).  After the streaming momentum
// kernel (k_elementwise.cu), k_skinny_ns runs one cluster of CL CTAs per
// member (the plan's column shards, 2 by default).  CTA r owns columns
// [r W, (r+1) W) of the wide m x n iterate.  The
// iterate is kept in an L2-resident workspace in the exact register order of
// mma.sync fragments, so each pass is: load fragments -> Y <- Q Y (mma.sync,
// with movmatrix transposes for the B operand) -> accumulate the next Gram
// Y Y^T from the same registers -> store fragments.  Operands of each pass
// stream through a per-thread cp.async ring.  Per step the per-warp Gram
// partials are summed in a fixed warp order, then over the cluster's CTAs in
// rank order (distributed shared memory), and every CTA forms
// Q = a I + b A + c A A in fp32.
//
// Writing aX + (bA + cAA)X as (aI + bA + cAA)X keeps one product per step
// («关于分布式Muon的想法整合及讨论» §2, §6: Gram matrix, then matrix products;
// A changes with X every round).  All reduction orders depend only on
// (rows, cols), so a member gives the same bits in any batch.
#include "warp_mma.cuh"

namespace muon {

namespace {

constexpr int kDefaultShards = 2;  // CTAs (column shards) per member unless the plan says otherwise

// Shared memory (bytes): the cp.async stage ring, per-warp Gram partials, the
// CTA partial (double buffered, read by the peer), A (fp32), Q (operand type).
template <int MT, int NT>
struct NsSmem {
  static constexpr int MP = 16 * MT;
  static constexpr int NW = NT / 32;
  static constexpr int LB = 32 * MT;  // stage bytes per lane and block
  // rounds in flight per warp (MT <= 2 runs 16 warps per CTA); consumed two at a time
  static constexpr int S = MT == 4 ? 2 : 4;
  static constexpr int kStage = 0;
  static constexpr int kWarpPart = kStage + S * NW * 32 * LB;
  static constexpr int kCta = kWarpPart + NW * GramTiles<MT>::N * 128 * 4;
  static constexpr int kA = kCta + 2 * MP * MP * 4;
  static constexpr int kQ = kA + MP * MP * 4;
  static constexpr int kMisc = kQ + MP * (MP + 8) * 2;
  static constexpr int kTotal = kMisc + 64;
  static_assert(kTotal <= 227 * 1024, "skinny kernel shared memory exceeds the per-CTA limit");
};

struct SkArgs {
  int W;        // columns of the wide iterate per CTA (multiple of 16)
  int NB;       // 16-column blocks per CTA
  int blk;      // bytes of one block in the fragment workspace
  uint8_t* ws;  // fragment workspace [B][CL][NB][blk]
};

// Offsets of element (i, j) of the wide iterate in the parameter's memory.
struct Wide {
  int cols, T;
  __device__ __forceinline__ int64_t off(int i, int j) const {
    return T ? (int64_t)j * cols + i : (int64_t)i * cols + j;
  }
};

enum PassKind { PASS_FIRST = 0, PASS_MID = 1, PASS_LAST = 2, PASS_ONLY = 3 };

// Per-thread state shared by the passes of one member.
template <int MT>
struct PassCtx {
  int lane, warp, g, t4, m, n, c0, NB;
  bool pairs;              // M' / P pairs are adjacent and aligned (fast path)
  bool rv[MT][2];          // row 16 mi + g + 8 h is inside the matrix
  int64_t roff[MT][2];     // element offset of (row, column 2 t4) when `pairs`
  const float* Mp;
  __nv_bfloat16* P;
  float* dbg;
  uint8_t* ws;             // this CTA's fragment blocks
  Wide wd;
  float inv, decay, coef, inv_alpha;
};

// One pass over this warp's 16-column blocks (blk = warp + r * NW):
//   FIRST: fragments from M' * inv, next Gram, store fragments
//   MID:   Y <- Q Y, next Gram, store fragments
//   LAST:  Y <- Q Y, P' = P decay - coef Y
//   ONLY:  fragments from M' * inv, P' = P decay - coef Y   (k = 0)
// Operands of the next S rounds stream into this lane's planes of a shared
// ring with cp.async; a lane only reads back what it copied, so the passes
// need no block barrier.  Plane offsets (bytes, lane 0): M' pair k at
// k * 256, fragment tile mi at mi * 512, P pair k at MT * 512 + k * 128.
template <int KIND, typename TY, int MT, int NT, bool HALF>
__device__ __forceinline__ void run_pass(const PassCtx<MT>& c, uint8_t* stage_warp,
                                         const uint32_t (&qf)[MT][MT][4], float (&gacc)[GramTiles<MT>::N][4]) {
  using L = NsSmem<MT, NT>;
  using GT = GramTiles<MT>;
  constexpr int NW = L::NW, S = L::S, LB = L::LB;
  constexpr bool kFromM = KIND == PASS_FIRST || KIND == PASS_ONLY;
  constexpr bool kWriteP = KIND == PASS_LAST || KIND == PASS_ONLY;
  constexpr bool kUpdate = KIND == PASS_MID || KIND == PASS_LAST;
  constexpr int kBlk = (MT - 1) * 512 + (HALF ? 256 : 512);
  constexpr uint32_t kSlot = NW * 32 * LB;  // bytes of one round of the ring
  auto full_tile = [](int mi) { return !(HALF && mi == MT - 1); };
  auto toff = [](int mi) { return mi * 512; };
  const int lane = c.lane;
  const bool stream_p = c.pairs && KIND == PASS_LAST;
  const int rounds = (c.NB + NW - 1) / NW;
  const uint32_t ring0 = static_cast<uint32_t>(__cvta_generic_to_shared(stage_warp));

  auto issue = [&](int r, uint32_t dst) {
    const int blk = r * NW + c.warp;
    if (r < rounds && blk < c.NB) {
      const int jb = c.c0 + blk * 16;
      const bool fullblk = jb + 16 <= c.n;
      if (kFromM) {
        if (c.pairs) {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (!full_tile(mi) && (q & 1)) continue;
              const int dj = (q & 2) ? 8 : 0;
              const bool ok = c.rv[mi][q & 1] && (fullblk || jb + 2 * c.t4 + dj + 1 < c.n);
              cp_async8(dst + (mi * 4 + q) * 256 + lane * 8,
                        ok ? (const void*)(c.Mp + c.roff[mi][q & 1] + jb + dj) : (const void*)c.Mp,
                        ok ? 8 : 0);
            }
        }
      } else {
        const uint8_t* wsb = c.ws + (int64_t)blk * kBlk;
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
          if (full_tile(mi))
            cp_async16(dst + mi * 512 + lane * 16, wsb + toff(mi) + lane * 16, 16);
          else
            cp_async8(dst + mi * 512 + lane * 8, wsb + toff(mi) + lane * 8, 8);
        }
      }
      if (KIND == PASS_LAST && stream_p) {
#pragma unroll
        for (int mi = 0; mi < MT; ++mi)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (!full_tile(mi) && (q & 1)) continue;
            const int dj = (q & 2) ? 8 : 0;
            const bool ok = c.rv[mi][q & 1] && (fullblk || jb + 2 * c.t4 + dj + 1 < c.n);
            cp_async4(dst + MT * 512 + (mi * 4 + q) * 128 + lane * 4,
                      ok ? (const void*)(c.P + c.roff[mi][q & 1] + jb + dj) : (const void*)c.P,
                      ok ? 4 : 0);
          }
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int r = 0; r < S; ++r) issue(r, ring0 + r * kSlot);

  // Two rounds (two blocks per warp) are consumed per iteration so their
  // independent instruction streams can interleave.
  auto process = [&](int r, const uint8_t* st) {
    const int blk = r * NW + c.warp;
    if (r < rounds && blk < c.NB) {
      const int jb = c.c0 + blk * 16;
      const bool fullblk = jb + 16 <= c.n;
      uint8_t* wsb = c.ws + (int64_t)blk * kBlk;
      uint32_t y[MT][4];
      if (kFromM) {
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float v0 = 0.f, v1 = 0.f;
            if (!full_tile(mi) && (q & 1)) {
              y[mi][q] = 0u;
              continue;
            }
            if (c.pairs) {
              const float2 f = *reinterpret_cast<const float2*>(st + (mi * 4 + q) * 256 + lane * 8);
              v0 = f.x; v1 = f.y;
            } else {
              const int i = mi * 16 + c.g + ((q & 1) ? 8 : 0);
              const int j = jb + 2 * c.t4 + ((q & 2) ? 8 : 0);
              if (i < c.m) {
                if (j < c.n) v0 = c.Mp[c.wd.off(i, j)];
                if (j + 1 < c.n) v1 = c.Mp[c.wd.off(i, j + 1)];
              }
            }
            y[mi][q] = Mma<TY>::pack(v0 * c.inv, v1 * c.inv);
          }
        }
      } else {
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
          if (full_tile(mi)) {
            const uint4 v = *reinterpret_cast<const uint4*>(st + mi * 512 + lane * 16);
            y[mi][0] = v.x; y[mi][1] = v.y; y[mi][2] = v.z; y[mi][3] = v.w;
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(st + mi * 512 + lane * 8);
            y[mi][0] = v.x; y[mi][1] = 0u; y[mi][2] = v.y; y[mi][3] = 0u;
          }
        }
      }
      if (kUpdate) {
        // Y <- Q Y: B operand rows are iterate rows, so transpose 8x8 blocks
        uint32_t bt[MT][4];
#pragma unroll
        for (int kk = 0; kk < MT; ++kk)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            bt[kk][q] = (!full_tile(kk) && (q & 1)) ? 0u : movtrans(y[kk][q]);
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
          float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < MT; ++kk) {
            Mma<TY>::run(d0, qf[mi][kk], bt[kk][0], bt[kk][1]);  // columns 0..7
            Mma<TY>::run(d1, qf[mi][kk], bt[kk][2], bt[kk][3]);  // columns 8..15
          }
          y[mi][0] = Mma<TY>::pack(d0[0], d0[1]);
          y[mi][1] = Mma<TY>::pack(d0[2], d0[3]);
          y[mi][2] = Mma<TY>::pack(d1[0], d1[1]);
          y[mi][3] = Mma<TY>::pack(d1[2], d1[3]);
        }
      }
      if (!kWriteP) {
        // next Gram: Y Y^T over this block, upper tiles, B operand = rows of Y
#pragma unroll
        for (int q = 0; q < GT::N; ++q) {
          const int mi = GT::code(q) >> 4, nj = GT::code(q) & 15;
          const uint32_t* src = y[nj >> 1];
          Mma<TY>::run(gacc[q], y[mi], (nj & 1) ? src[1] : src[0], (nj & 1) ? src[3] : src[2]);
        }
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
          if (full_tile(mi))
            *reinterpret_cast<uint4*>(wsb + toff(mi) + lane * 16) =
                make_uint4(y[mi][0], y[mi][1], y[mi][2], y[mi][3]);
          else
            *reinterpret_cast<uint2*>(wsb + toff(mi) + lane * 8) = make_uint2(y[mi][0], y[mi][2]);
        }
      } else {
        // P' = P (1 - lr wd) - lr s Y / alpha on the valid elements
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (!full_tile(mi) && (q & 1)) continue;
            const int dj = (q & 2) ? 8 : 0;
            if (!c.rv[mi][q & 1]) continue;
            const float2 yv = Mma<TY>::unpack(y[mi][q]);
            if (c.pairs) {
              if (!fullblk && jb + 2 * c.t4 + dj >= c.n) continue;
              __nv_bfloat16* pp = c.P + c.roff[mi][q & 1] + jb + dj;
              uint32_t praw = stream_p ? *reinterpret_cast<const uint32_t*>(
                                             st + MT * 512 + (mi * 4 + q) * 128 + lane * 4)
                                       : *reinterpret_cast<const uint32_t*>(pp);
              const float2 pf = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&praw));
              *reinterpret_cast<__nv_bfloat162*>(pp) = __floats2bfloat162_rn(
                  fmaf(-c.coef, yv.x, pf.x * c.decay), fmaf(-c.coef, yv.y, pf.y * c.decay));
              if (c.dbg)
                *reinterpret_cast<float2*>(c.dbg + c.roff[mi][q & 1] + jb + dj) =
                    make_float2(yv.x * c.inv_alpha, yv.y * c.inv_alpha);
            } else {
              const int i = mi * 16 + c.g + ((q & 1) ? 8 : 0);
              const int j = jb + 2 * c.t4 + dj;
              if (j >= c.n) continue;
              const int64_t o0 = c.wd.off(i, j);
              c.P[o0] = __float2bfloat16_rn(fmaf(-c.coef, yv.x, __bfloat162float(c.P[o0]) * c.decay));
              if (c.dbg) c.dbg[o0] = yv.x * c.inv_alpha;
              if (j + 1 < c.n) {
                const int64_t o1 = c.wd.off(i, j + 1);
                c.P[o1] = __float2bfloat16_rn(fmaf(-c.coef, yv.y, __bfloat162float(c.P[o1]) * c.decay));
                if (c.dbg) c.dbg[o1] = yv.y * c.inv_alpha;
              }
            }
          }
        }
      }
    }
  };
  int slot = 0;
  for (int r = 0; r < rounds; r += 2) {
    cp_async_wait<S - 2>();
    const int slot2 = slot + 1 == S ? 0 : slot + 1;
#pragma unroll
    for (int u = 0; u < 2; ++u) process(r + u, stage_warp + (u ? slot2 : slot) * kSlot);
    // the slots of rounds r, r+1 were consumed above (registers): refill them
    issue(r + S, ring0 + slot * kSlot);
    issue(r + 1 + S, ring0 + slot2 * kSlot);
    slot = slot2 + 1 == S ? 0 : slot2 + 1;
  }
  cp_async_wait<0>();
}

template <typename TY, int MT, int NT, bool HALF>
__global__ void __launch_bounds__(NT, 1) k_skinny_ns(KArgs a, SkArgs s) {
  using L = NsSmem<MT, NT>;
  using GT = GramTiles<MT>;
  constexpr int MP = L::MP, NW = L::NW;
  extern __shared__ __align__(16) uint8_t smem[];
  float* wpart = reinterpret_cast<float*>(smem + L::kWarpPart);
  float* cpart = reinterpret_cast<float*>(smem + L::kCta);
  float* Af = reinterpret_cast<float*>(smem + L::kA);
  TY* Qs = reinterpret_cast<TY*>(smem + L::kQ);
  float* misc = reinterpret_cast<float*>(smem + L::kMisc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const int CL = (int)cluster_size();  // CTAs (column shards) per member
  const int b = blockIdx.x / CL;
  const int m = a.m;
  const MemberPtrs mp = a.mem[b];

  PassCtx<MT> c;
  c.lane = lane; c.warp = warp; c.g = lane >> 2; c.t4 = lane & 3;
  c.m = m; c.n = a.n; c.c0 = (int)rank * s.W; c.NB = s.NB;
  // X_0's source: M', or U = G + beta M' written by the momentum kernel
  c.Mp = a.u ? a.u + (int64_t)b * m * a.n : mp.M;
  c.P = static_cast<__nv_bfloat16*>(mp.P);
  const bool T = mp.T != 0;           // this member's parameter is [n, m]
  const int cols = T ? m : a.n;       // the parameter's row pitch
  c.wd = Wide{cols, (int)T};
  // pairs (i, j), (i, j+1) are adjacent in memory (fast path) when the wide
  // iterate is the parameter itself, its rows are even and bases are aligned
  c.pairs = !T && (cols % 2 == 0) &&
            ((reinterpret_cast<uintptr_t>(c.Mp) | reinterpret_cast<uintptr_t>(c.P)) & 7) == 0;
  c.ws = s.ws + ((int64_t)b * CL + rank) * s.NB * s.blk;
  c.dbg = a.dbg ? a.dbg + (int64_t)b * m * a.n : nullptr;
#pragma unroll
  for (int mi = 0; mi < MT; ++mi)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = mi * 16 + c.g + 8 * h;
      c.rv[mi][h] = i < m;
      c.roff[mi][h] = (int64_t)i * cols + 2 * c.t4;
    }

  // Q = 0 outside the m x m block; zero once
  for (int e = tid; e < MP * (MP + 8); e += NT) Qs[e] = from_f32<TY>(0.f);
  // the member's norm from the momentum kernel's fixed-chunk partials
  if (tid == 0) {
    const float* pp = a.part + (int64_t)b * a.n_chunks;
    float s2 = 0.f;
    for (int k = 0; k < a.n_chunks; ++k) s2 += pp[k];
    misc[0] = a.alpha / (sqrtf(s2) + a.eps);
  }
  __syncthreads();
  c.inv = misc[0];

  const int ns = a.sc->ns_steps;
  const float inv_a2 = 1.f / (a.alpha * a.alpha);
  const float lr = a.sc->lr, wdk = a.sc->wd;
  c.decay = __fmaf_rn(-lr, wdk, 1.f);  // one rounding of 1 - lr wd
  c.inv_alpha = 1.f / a.alpha;
  c.coef = lr * mp.scale * c.inv_alpha;
  uint8_t* stage_warp = smem + L::kStage + warp * 32 * L::LB;

  uint32_t qf[MT][MT][4];
  float gacc[GT::N][4];
  auto zero_gacc = [&]() {
#pragma unroll
    for (int q = 0; q < GT::N; ++q) gacc[q][0] = gacc[q][1] = gacc[q][2] = gacc[q][3] = 0.f;
  };
  // sum the Gram partials (warps in fixed order, then CTAs in rank order),
  // form Q = a I + b A + c A A in fp32 (step p's coefficients) and load its
  // fragments
  auto reduce_and_poly = [&](int p) {
    const int g = c.g, t4 = c.t4;
    const float* cf = step_coef(a.sc, p);
    const float ca = cf[0], cb = cf[1], cc = cf[2];
#pragma unroll
    for (int q = 0; q < GT::N; ++q) {
      float* dst = wpart + (warp * GT::N + q) * 128;
      dst[g * 8 + 2 * t4] = gacc[q][0];
      dst[g * 8 + 2 * t4 + 1] = gacc[q][1];
      dst[(g + 8) * 8 + 2 * t4] = gacc[q][2];
      dst[(g + 8) * 8 + 2 * t4 + 1] = gacc[q][3];
    }
    __syncthreads();
    float* cp = cpart + (p & 1) * MP * MP;  // read by the peer after the barrier
    for (int e = tid; e < GT::N * 128; e += NT) {
      const int q = e >> 7, w = e & 127;
      float acc = 0.f;
      for (int k = 0; k < NW; ++k) acc += wpart[(k * GT::N + q) * 128 + w];
      const int code = GT::code(q);
      cp[((code >> 4) * 16 + (w >> 3)) * MP + (code & 15) * 8 + (w & 7)] = acc;
    }
    cluster_sync();
    for (int e = tid; e < m * m; e += NT) {
      const int i = e / m, j = e - (e / m) * m;
      if (i > j) continue;
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < CL; ++r) acc += ld_dsmem_f32(&cp[i * MP + j], (uint32_t)r);
      acc *= inv_a2;
      Af[i * MP + j] = acc;
      Af[j * MP + i] = acc;
    }
    __syncthreads();
    for (int e = tid; e < m * m; e += NT) {
      const int i = e / m, j = e - (e / m) * m;
      if (i > j) continue;
      float acc = 0.f;
      for (int k = 0; k < m; ++k) acc = fmaf(Af[i * MP + k], Af[k * MP + j], acc);
      float q = fmaf(cc, acc, cb * Af[i * MP + j]);
      if (i == j) q += ca;
      const TY qh = from_f32<TY>(q);
      Qs[i * (MP + 8) + j] = qh;
      Qs[j * (MP + 8) + i] = qh;
    }
    __syncthreads();
    const uint32_t qb = smem_u32(Qs);
#pragma unroll
    for (int mi = 0; mi < MT; ++mi)
#pragma unroll
      for (int kk = 0; kk < MT; ++kk)
        ldsm_x4(qb + 2u * ((mi * 16 + (lane & 15)) * (MP + 8) + kk * 16 + (lane >> 4) * 8),
                qf[mi][kk]);
  };

  zero_gacc();
  if (ns == 0) {
    run_pass<PASS_ONLY, TY, MT, NT, HALF>(c, stage_warp, qf, gacc);
  } else {
    run_pass<PASS_FIRST, TY, MT, NT, HALF>(c, stage_warp, qf, gacc);
    for (int p = 1; p < ns; ++p) {
      reduce_and_poly(p - 1);
      zero_gacc();
      run_pass<PASS_MID, TY, MT, NT, HALF>(c, stage_warp, qf, gacc);
    }
    reduce_and_poly(ns - 1);
    run_pass<PASS_LAST, TY, MT, NT, HALF>(c, stage_warp, qf, gacc);
  }
  // the peer may still read this CTA's Gram partial
  cluster_sync();
}

template <typename TY, int MT, int NT, bool HALF>
cudaError_t launch_t(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prepare) {
  auto fn = k_skinny_ns<TY, MT, NT, HALF>;
  constexpr int smem = NsSmem<MT, NT>::kTotal;
  if (prepare) return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  SkArgs s;
  s.W = cfg.width;
  s.NB = cfg.width / 16;
  s.blk = cfg.blk;
  s.ws = static_cast<uint8_t*>(a.y0);
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(a.B * cfg.cluster);
  lc.blockDim = dim3(NT);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cfg.cluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, fn, a, s);
}

template <typename TY, bool HALF>
cudaError_t launch_th(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prep) {
  switch (cfg.mtiles) {
    case 1: return launch_t<TY, 1, 512, HALF>(a, cfg, st, prep);
    case 2: return launch_t<TY, 2, 512, HALF>(a, cfg, st, prep);
    case 3: return launch_t<TY, 3, 256, HALF>(a, cfg, st, prep);
    default: return launch_t<TY, 4, 256, HALF>(a, cfg, st, prep);
  }
}

// HALF: the last m16 tile holds at most 8 rows (stored as half a tile)
bool half_last_tile(int m, int mtiles) { return m - 16 * (mtiles - 1) <= 8; }

template <typename TY>
cudaError_t launch_ty(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prep) {
  return half_last_tile(a.m, cfg.mtiles) ? launch_th<TY, true>(a, cfg, st, prep)
                                         : launch_th<TY, false>(a, cfg, st, prep);
}

cudaError_t dispatch(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prep) {
  if (a.mode_f32) return cudaErrorInvalidValue;  // fp32 parameters use the SIMT path
  return a.ns_type == NS_F16 ? launch_ty<__half>(a, cfg, st, prep)
                             : launch_ty<__nv_bfloat16>(a, cfg, st, prep);
}

template <typename TY, int MT, bool HALF>
int clusters_of(int cl) {
  constexpr int NT = MT <= 2 ? 512 : 256;
  auto fn = k_skinny_ns<TY, MT, NT, HALF>;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(cl * 1024);
  lc.blockDim = dim3(NT);
  lc.dynamicSmemBytes = NsSmem<MT, NT>::kTotal;
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

template <typename TY, bool HALF>
int clusters_mt(int mtiles, int cl) {
  switch (mtiles) {
    case 1: return clusters_of<TY, 1, HALF>(cl);
    case 2: return clusters_of<TY, 2, HALF>(cl);
    case 3: return clusters_of<TY, 3, HALF>(cl);
    default: return clusters_of<TY, 4, HALF>(cl);
  }
}

}  // namespace

bool skinny_config(int32_t rows, int32_t cols, int32_t max_m, SkinnyCfg* cfg, int32_t shards) {
  const int m = rows < cols ? rows : cols, n = rows < cols ? cols : rows;
  if (m < 1 || m > max_m || m > 64) return false;
  const int cl = shards > 0 ? shards : kDefaultShards;
  if (cl != 1 && cl != 2 && cl != 4 && cl != 8) return false;
  cfg->mtiles = (m + 15) / 16;
  cfg->cluster = cl;
  cfg->threads = cfg->mtiles <= 2 ? 512 : 256;
  const int w = (n + cl - 1) / cl;
  cfg->width = (w + 31) / 32 * 32;  // whole 32-column superblocks (Gram-space output pass)
  int blk = 0;
  for (int q = 0; q < cfg->mtiles; ++q) blk += (m - 16 * q > 8) ? 512 : 256;
  cfg->blk = blk;
  cfg->ws_bytes = (int64_t)cl * (cfg->width / 16) * blk;  // per member (direct kernel)
  cfg->smem = 0;
  cfg->gram_space = 1;  // every skinny m (<= 64); the step count decides at launch
  cfg->auto_shards = shards <= 0;
  return true;
}

cudaError_t prepare_skinny(const KArgs& a, const SkinnyCfg& cfg) {
  cudaError_t e = dispatch(a, cfg, nullptr, true);
  if (e == cudaSuccess && cfg.gram_space) e = gs_dispatch(a, cfg, nullptr, true);
  return e;
}

cudaError_t launch_skinny(const KArgs& a, const SkinnyCfg& cfg, int32_t ns_steps, cudaStream_t s) {
  if (cfg.gram_space && ns_steps <= kGramSpaceMaxSteps) return gs_dispatch(a, cfg, s, false);
  const cudaError_t e = launch_momentum_partial(a, s);
  return e == cudaSuccess ? dispatch(a, cfg, s, false) : e;
}

int skinny_max_active_clusters(int ns_type, int m, int cl) {
  const int mt = (m + 15) / 16;
  const bool half = half_last_tile(m, mt);
  const int direct = ns_type == NS_F16
                         ? (half ? clusters_mt<__half, true>(mt, cl) : clusters_mt<__half, false>(mt, cl))
                         : (half ? clusters_mt<__nv_bfloat16, true>(mt, cl)
                                 : clusters_mt<__nv_bfloat16, false>(mt, cl));
  const int gs = gs_max_active_clusters(ns_type, m, cl);  // either kernel may serve a step
  return gs < direct ? gs : direct;
}

}  // namespace muon
