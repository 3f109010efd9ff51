// tcgen05 / TMEM / TMA batched GEMMs of one Newton-Schulz step (TENSOR path).
//
//   GRAM:   A  = (Y Y^T) / alpha^2          M = N = m, K = n   (Gram matrix)
//   POLY:   Q  = a I + b A + c (A A)        M = N = K = m      (step polynomial)
//   UPDATE: Y' = Q Y                        M = m, N = n, K = m
// «关于分布式Muon的想法整合及讨论» §2: the iteration is a Gram matrix and a series
// of matrix products; §6: A is rebuilt from the new X every round.  Writing
// aX + (bA + cAA)X as (aI + bA + cAA)X folds the axpy into the polynomial
// matrix, so each step is three dense products with fused epilogues.
//
// Design (sm_103a): persistent CTAs (one per SM), 320 threads:
//   warp 0      TMA producer: 128-byte-swizzled tiles into a 4-stage ring;
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer (M=128,
//               N=BN, K=16, fp16/bf16 operands, fp32 accumulators in TMEM);
//   warps 2..9  epilogue, two warps per 32-lane TMEM quarter, each on half
//               of the tile's columns: tcgen05.ld of the accumulator (one
//               row per thread), fused scale / polynomial / cast, stores.
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1.  Every wait is bounded: on timeout the kernel sets the plan's error
// word and all roles leave their loops.
//
// GRAM and POLY outputs are symmetric (Y Y^T, and a polynomial in the
// symmetric A), so only the tiles that reach the upper triangle (j >= i) are
// computed; each writes its elements with j >= i in place and mirrors those
// with j > i to (j, i).  Every element is written exactly once and the stored
// matrix is exactly symmetric.  For m = 4096 (BN = 256) that is 272 of 512
// tiles.  Both operands of these two products come from the same matrix, so a
// diagonal tile (whose B panel is its A panel) loads the panel once and reads
// it as both operands.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "mbarrier.cuh"
#include "tcgen05.cuh"

namespace muon {

namespace {

constexpr int BM = 128, BK = 64, kStages = 4;
// Warps of a one-CTA GEMM: a TMA producer, the MMA issuer, and eight
// epilogue warps, two per 32-lane quarter of TMEM, each on half the tile's
// columns (short-K products would otherwise wait on the epilogue).
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;

enum TcOp { TC_GRAM = 0, TC_POLY = 1, TC_UPDATE = 2 };

struct TcArgs {
  int B, M, N, K;
  int tiles_m, tiles_n;
  int tiles_sym;          // GRAM / POLY: tiles per batch reaching the upper triangle (set at launch)
  int64_t ldc, sC;        // output row pitch / batch stride (elements)
  void* C;
  const void* aux;        // POLY: the A matrix (same layout as C)
  const StepScalars* sc;
  int step;               // POLY: Newton-Schulz step (schedule row)
  float scale;            // GRAM: 1 / alpha^2
  int* err;
};

// ---- TMA ----
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t mbar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(mbar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

template <int BN>
struct TcSmem {
  static constexpr uint32_t kA = BM * BK * 2;          // 16 KB
  static constexpr uint32_t kB = BN * BK * 2;          // 32 KB (BN = 256)
  static constexpr uint32_t kStage = kA + kB;
  static constexpr uint32_t kBars = kStages * kStage;  // barrier area offset
  // GRAM / POLY: per epilogue warp a 32 x 32 block of 16-bit values as 32 rows
  // of 17 words (a padded row keeps the column reads free of bank conflicts)
  static constexpr uint32_t kEpi = kBars + 256;
  static constexpr uint32_t kEpiBytes = kEpiWarps * 32 * 17 * 4;
  static constexpr uint32_t kTotal = kEpi + kEpiBytes + 1024;  // + alignment slack
  static_assert(kTotal <= 227 * 1024, "GEMM shared memory exceeds the per-CTA limit");
};

// Tile r of one batch's full output in grouped order: 8 tile-rows share a
// sweep over the tile-columns, so the tiles in flight reuse a compact set of
// operand panels through L2.
__host__ __device__ __forceinline__ void decode_raster(int r, int tiles_m, int tiles_n, int& tm,
                                                       int& tn) {
  constexpr int GM = 8;
  const int group = r / (GM * tiles_n);
  const int first = group * GM;
  const int gsz = tiles_m - first < GM ? tiles_m - first : GM;
  r -= group * GM * tiles_n;
  tm = first + r % gsz;
  tn = r / gsz;
}
__device__ __forceinline__ void decode_tile(int t, const TcArgs& p, int& b, int& tm, int& tn) {
  const int per_b = p.tiles_m * p.tiles_n;
  b = t / per_b;
  decode_raster(t - b * per_b, p.tiles_m, p.tiles_n, tm, tn);
}

// First tile column of tile row tm that reaches the upper triangle (tiles of
// TM rows and BN columns).
template <int BN, int TM = BM>
__host__ __device__ __forceinline__ int first_tn(int tm) { return tm * TM / BN; }
template <int BN, int TM = BM>
__host__ __device__ inline int sym_tiles_per_batch(int tiles_m, int tiles_n) {
  int u = 0;
  for (int tm = 0; tm < tiles_m; ++tm) {
    const int c = tiles_n - first_tn<BN, TM>(tm);
    u += c > 0 ? c : 0;
  }
  return u;
}
// Tile r of one batch's symmetric output: tile rows in order, each from its
// first tile column that reaches the upper triangle.
template <int BN, int TM = BM>
__host__ __device__ __forceinline__ void decode_sym(int r, int tiles_m, int tiles_n, int& tm,
                                                    int& tn) {
  tm = 0;
  while (tm + 1 < tiles_m && r >= tiles_n - first_tn<BN, TM>(tm)) {
    r -= tiles_n - first_tn<BN, TM>(tm);
    ++tm;
  }
  tn = first_tn<BN, TM>(tm) + r;
}
// Tile t of an output: for the symmetric ones batch-major, then decode_sym.
template <int OP, int BN, int TM = BM>
__device__ __forceinline__ void decode(int t, const TcArgs& p, int& b, int& tm, int& tn) {
  if constexpr (OP == TC_UPDATE) {
    decode_tile(t, p, b, tm, tn);
  } else {
    b = t / p.tiles_sym;
    decode_sym<BN, TM>(t - b * p.tiles_sym, p.tiles_m, p.tiles_n, tm, tn);
  }
}

template <typename TY>
__device__ __forceinline__ void store_row32(TY* dst, const float* v, int nvalid) {
  if (nvalid >= 32) {
    uint4 u[4];
    uint32_t* w = reinterpret_cast<uint32_t*>(u);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      TY lo = from_f32<TY>(v[2 * i]), hi = from_f32<TY>(v[2 * i + 1]);
      w[i] = (uint32_t)(*reinterpret_cast<uint16_t*>(&lo)) |
             ((uint32_t)(*reinterpret_cast<uint16_t*>(&hi)) << 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(dst)[i] = u[i];
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nvalid) dst[i] = from_f32<TY>(v[i]);
  }
}

// The epilogue of one output tile for one epilogue warp: rows
// rbase + quarter * 32 + lane (one accumulator row per thread, TMEM lanes
// quarter * 32 ..), columns cbase .. cbase + BN - 1 from the accumulator at
// TMEM column tmem_acc, in chunks of 32 columns (chunks ch0 .. ch1 - 1 of
// the tile, so that two warps can share a row quarter).  GRAM scales by
// 1 / alpha^2, POLY forms a I + b A + c A^2 (A read from p.aux); GRAM and
// POLY write the elements with col >= row in place and mirror those with
// col > row through this warp's 32 x 32 staging block `sw`; UPDATE stores
// the row.
template <typename TY, int OP, int BN>
__device__ __forceinline__ void epilogue_tile(const TcArgs& p, uint32_t tmem_acc, int quarter, int lane,
                                              int b, int rbase, int cbase, float ca, float cb, float cc,
                                              uint32_t* sw, int ch0 = 0, int ch1 = BN / 32) {
  const int row_in_tile = quarter * 32 + lane;
  const int row = rbase + row_in_tile;
  const int row0 = rbase + quarter * 32;  // this warp's first row
  TY* crow = static_cast<TY*>(p.C) + (int64_t)b * p.sC + (int64_t)row * p.ldc;
  const TY* arow = OP == TC_POLY ? static_cast<const TY*>(p.aux) + (int64_t)b * p.sC +
                                       (int64_t)row * p.ldc
                                 : nullptr;
#pragma unroll 1
  for (int ch = ch0; ch < ch1; ++ch) {
    uint32_t r[32];
    const uint32_t taddr = tmem_acc + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ch * 32);
    tmem_ld32(taddr, r);
    const int col0 = cbase + ch * 32;
    if (col0 >= p.N) continue;  // the same for the whole warp
    const bool live = row < p.M;
    if (OP == TC_UPDATE && !live) continue;
    const int nvalid = min(32, p.N - col0);
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    if (OP == TC_GRAM) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= p.scale;
    } else if (OP == TC_POLY) {
      float av[32];
      if (!live) {
#pragma unroll
        for (int i = 0; i < 32; ++i) av[i] = 0.f;
      } else if (nvalid == 32) {
        const uint4* src = reinterpret_cast<const uint4*>(arow + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u = src[q];
          const TY* h = reinterpret_cast<const TY*>(&u);
#pragma unroll
          for (int e = 0; e < 8; ++e) av[q * 8 + e] = to_f32(h[e]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) av[i] = i < nvalid ? to_f32(arow[col0 + i]) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = fmaf(cc, v[i], cb * av[i]);
        if (col0 + i == row) v[i] += ca;
      }
    }
    if constexpr (OP == TC_UPDATE) {
      store_row32<TY>(crow + col0, v, nvalid);
    } else {
      // on and above the diagonal in place
      if (live) {
        if (col0 >= row) {
          store_row32<TY>(crow + col0, v, nvalid);
        } else if (col0 + 31 >= row) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nvalid && col0 + i >= row) crow[col0 + i] = from_f32<TY>(v[i]);
        }
      }
      // strictly above also at (j, i): the warp's 32 x 32 block goes
      // through shared memory, so that lane j then writes row col0 + j of
      // the mirror, 32 values from column row0, as 16-byte stores
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const TY lo = from_f32<TY>(v[2 * q]), hi = from_f32<TY>(v[2 * q + 1]);
        sw[lane * 17 + q] = (uint32_t)(*reinterpret_cast<const uint16_t*>(&lo)) |
                            ((uint32_t)(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
      }
      __syncwarp();
      const int orow = col0 + lane;
      if (lane < nvalid && orow > row0) {
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const uint32_t a0 = sw[(2 * q) * 17 + (lane >> 1)], a1 = sw[(2 * q + 1) * 17 + (lane >> 1)];
          const uint32_t h0 = (lane & 1) ? (a0 >> 16) : (a0 & 0xffffu);
          const uint32_t h1 = (lane & 1) ? (a1 >> 16) : (a1 & 0xffffu);
          w[q] = h0 | (h1 << 16);
        }
        TY* dst = static_cast<TY*>(p.C) + (int64_t)b * p.sC + (int64_t)orow * p.ldc + row0;
        if (col0 >= row0 + 32 && row0 + 32 <= p.M) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        } else {
          const TY* h = reinterpret_cast<const TY*>(w);
#pragma unroll
          for (int r2 = 0; r2 < 32; ++r2)
            if (orow > row0 + r2 && row0 + r2 < p.M) dst[r2] = h[r2];
        }
      }
      __syncwarp();  // the block is overwritten by the next chunk
    }
  }
}

template <typename TY, int OP, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
              TcArgs p) {
  using L = TcSmem<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  // bars: full[kStages], empty[kStages], tfull[2], tempty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* epi = reinterpret_cast<uint32_t*>(smem + L::kEpi);  // GRAM / POLY mirror staging
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = saddr(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
  constexpr uint32_t kCols = 2 * BN;  // two accumulators

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), 32 * kEpiWarps); }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mapA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mapB) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = p.B * (OP == TC_UPDATE ? p.tiles_m * p.tiles_n : p.tiles_sym);
  const int kblocks = (p.K + BK - 1) / BK;
  constexpr bool kMN = OP == TC_UPDATE;  // B operand is N-contiguous (MN-major)
  // GRAM and POLY read both operands from the same matrix (Y, or the
  // symmetric A), so on a diagonal tile the B panel is the A panel
  constexpr bool kSym = OP != TC_UPDATE;

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer ----
      int s = 0;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int b, tm, tn;
        decode<OP, BN>(t, p, b, tm, tn);
        const bool diag = kSym && BN == BM && tm == tn;  // B panel = A panel: load it once
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty(s), ph ^ 1, abort_flag, p.err, 1)) goto producer_done;
          mbar_expect_tx(full(s), diag ? L::kA : L::kStage);
          const uint32_t sa = saddr(smem + s * L::kStage);
          const uint32_t sb = sa + L::kA;
          tma_load_3d(sa, &mapA, full(s), kb * BK, tm * BM, b);
          if (kMN) {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_3d(sb + c * (64 * BK * 2), &mapB, full(s), tn * BN + c * 64, kb * BK, b);
          } else if (!diag) {
            tma_load_3d(sb, &mapB, full(s), kb * BK, tn * BN, b);
          }
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer ----
      constexpr uint32_t idesc =
          instr_desc(std::is_same<TY, __nv_bfloat16>::value ? 1u : 0u, BM, BN, kMN);
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int b, tm, tn;
        decode<OP, BN>(t, p, b, tm, tn);
        const bool diag = kSym && BN == BM && tm == tn;
        if (!mbar_wait(tempty(acc), aph ^ 1, abort_flag, p.err, 2)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(full(s), ph, abort_flag, p.err, 4)) goto mma_done;
          tc_fence_after();
          const uint32_t sa = saddr(smem + s * L::kStage);
          const uint32_t sb = diag ? sa : sa + L::kA;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = kMN ? smem_desc(sb + kk * 2048, 64 * BK * 2, 1024)
                                    : smem_desc(sb + kk * 32, 16, 1024);
            umma(d_tmem, ad, bd, idesc, (kb | kk) != 0);
          }
          umma_commit(empty(s));  // frees the stage once these MMAs retire
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
        umma_commit(tfull(acc));
        if (++acc == 2) { acc = 0; aph ^= 1; }
      }
    mma_done:;
    }
  } else {  // ---- epilogue: warps 2..9, one accumulator row per thread ----
    const int quarter = warp & 3;                 // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;             // which half of the tile's columns
    constexpr int kHalf = BN / 64;                // chunks of 32 columns per half
    float ca = 0.f, cb = 0.f, cc = 0.f;
    if (OP == TC_POLY) {
      const float* cf = step_coef(p.sc, p.step);
      ca = cf[0]; cb = cf[1]; cc = cf[2];
    }
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int b, tm, tn;
      decode<OP, BN>(t, p, b, tm, tn);
      if (!mbar_wait(tfull(acc), aph, abort_flag, p.err, 8)) break;
      tc_fence_after();
      epilogue_tile<TY, OP, BN>(p, tmem_base + (uint32_t)(acc * BN), quarter, lane, b, tm * BM, tn * BN,
                                ca, cb, cc, epi + (warp - 2) * (32 * 17), half * kHalf,
                                half * kHalf + kHalf);
      tc_fence_before();
      mbar_arrive(tempty(acc));
      if (++acc == 2) { acc = 0; aph ^= 1; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kCols)
                 : "memory");
  }
}

// ---- the CTA-pair form (cta_group::2), for m >= 256 ----
//
// A cluster of two CTAs computes one 256 x 256 output tile: the leader (rank
// 0) issues tcgen05.mma.cta_group::2 with M = 256, N = 256, which reads rows
// [r 128, r 128 + 128) of the A tile and columns [r 128, r 128 + 128) of the
// B tile from the shared memory of CTA r, and writes rows [r 128, ..) of the
// accumulator into CTA r's TMEM.  Each CTA stages only half of the B tile, so
// shared-memory traffic per MMA drops by a third against the one-CTA form
// (128 x 256 tiles), and each CTA has room for six stages.  Every CTA loads
// its own halves with TMA from this GPU's memory; the copies of both CTAs
// complete on the leader's `full` barrier (cta_group::2 form of the copy), the
// leader's commits arrive on the `empty` and `tfull` barriers of both CTAs,
// and each epilogue warp tells the leader's `tempty` barrier when it has read
// its part of an accumulator.
constexpr int kStages2 = 6;
constexpr int BM2 = 256;  // rows of a pair tile
// Warps of a pair CTA: a TMA producer, the MMA issuer, and eight epilogue
// warps, two per 32-lane quarter of TMEM, each taking half the tile's
// columns: with short K (m up to ~2048 for the polynomial and Gram
// products) the epilogue would otherwise take longer than the next tile's
// MMAs and set the pace.
constexpr int kEpiWarps2 = 8;
constexpr int kThreads2 = 64 + 32 * kEpiWarps2;

struct TcSmem2 {
  static constexpr uint32_t kA = 128 * BK * 2;           // 16 KB: this CTA's A rows
  static constexpr uint32_t kB = 128 * BK * 2;           // 16 KB: this CTA's half of B
  static constexpr uint32_t kStage = kA + kB;
  static constexpr uint32_t kBars = kStages2 * kStage;   // full, empty, tfull, tempty, done
  static constexpr uint32_t kEpi = kBars + 256;
  static constexpr uint32_t kEpiBytes = kEpiWarps2 * 32 * 17 * 4;
  static constexpr uint32_t kTotal = kEpi + kEpiBytes + 1024;  // + alignment slack
  static_assert(kTotal <= 227 * 1024, "pair GEMM shared memory exceeds the per-CTA limit");
};

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t map_to(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// A tile copy whose completion is counted on an mbarrier that may sit in the
// peer CTA of the pair (`mbar` a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t mbar,
                                                 int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(mbar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the mbarrier at the same shared offset in every CTA of
// `mask` when the MMAs this thread issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t mbar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(mbar),
      "h"(mask)
      : "memory");
}
// Arrival of an epilogue warp on the leader's `tempty` barrier.  It only
// hands the TMEM accumulator back: the tcgen05 fences around it order the
// warp's tcgen05.ld reads before the leader's next MMAs, and the epilogue's
// global stores need no ordering with it, so the arrival is relaxed (a
// release at cluster scope would first wait for those stores to drain).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

template <typename TY, int OP>
__global__ void __launch_bounds__(kThreads2, 1)
    k_tc_gemm2(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
               TcArgs p) {
  constexpr int BN = 256;
  using L = TcSmem2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  // bars: full[kStages2], empty[kStages2], tfull[2], tempty[2], done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages2 + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* epi = reinterpret_cast<uint32_t*>(smem + L::kEpi);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank();
  const uint32_t bar0 = saddr(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages2 + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * kStages2 + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * kStages2 + 2 + a); };
  const uint32_t done = bar0 + 8u * (2 * kStages2 + 4);
  constexpr uint32_t kCols = 2 * BN;  // two accumulators: all 512 TMEM columns

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    // tempty: one arrival per epilogue warp of both CTAs
    for (int a = 0; a < 2; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), 2 * kEpiWarps2); }
    mbar_init(done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mapA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mapB) : "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates, together, the same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_barrier();  // both CTAs' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int num_tiles = p.B * (OP == TC_UPDATE ? p.tiles_m * p.tiles_n : p.tiles_sym);
  const int kblocks = (p.K + BK - 1) / BK;
  constexpr bool kMN = OP == TC_UPDATE;  // B operand is N-contiguous (MN-major)
  // GRAM and POLY read both operands from the same matrix (Y, or the
  // symmetric A), so on a diagonal tile the B panel is the A panel
  constexpr bool kSym = OP != TC_UPDATE;

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer (both CTAs) ----
      int s = 0;
      uint32_t ph = 0;
      for (int t = pair; t < num_tiles; t += npairs) {
        int b, tm, tn;
        decode<OP, BN, BM2>(t, p, b, tm, tn);
        const int arow = tm * BM2 + (int)rank * 128;  // this CTA's A rows
        const int bcol = tn * BN + (int)rank * 128;   // this CTA's half of the B tile
        // on a diagonal tile each CTA's half of B is its own A rows: load them once
        const bool diag = kSym && tm == tn;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty(s), ph ^ 1, abort_flag, p.err, 1)) goto producer_done;
          const uint32_t fb = map_to(full(s), 0);
          if (rank == 0) mbar_expect_tx(full(s), 2 * (diag ? L::kA : L::kStage));
          const uint32_t sa = saddr(smem + s * L::kStage);
          const uint32_t sb = sa + L::kA;
          tma_load_3d_pair(sa, &mapA, fb, kb * BK, arow, b);
          if (kMN) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_3d_pair(sb + c * (64 * BK * 2), &mapB, fb, bcol + c * 64, kb * BK, b);
          } else if (!diag) {
            tma_load_3d_pair(sb, &mapB, fb, kb * BK, bcol, b);
          }
          if (++s == kStages2) { s = 0; ph ^= 1; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // ---- MMA issuer (leader only) ----
      constexpr uint32_t idesc =
          instr_desc(std::is_same<TY, __nv_bfloat16>::value ? 1u : 0u, BM2, BN, kMN);
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      for (int t = pair; t < num_tiles; t += npairs) {
        int b, tm, tn;
        decode<OP, BN, BM2>(t, p, b, tm, tn);
        const bool diag = kSym && tm == tn;
        if (!mbar_wait(tempty(acc), aph ^ 1, abort_flag, p.err, 2)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(full(s), ph, abort_flag, p.err, 4)) goto mma_done;
          tc_fence_after();
          const uint32_t sa = saddr(smem + s * L::kStage);
          const uint32_t sb = diag ? sa : sa + L::kA;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = kMN ? smem_desc(sb + kk * 2048, 64 * BK * 2, 1024)
                                    : smem_desc(sb + kk * 32, 16, 1024);
            umma_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
          }
          umma_commit_pair(empty(s), 3);  // frees the stage in both CTAs once these MMAs retire
          if (++s == kStages2) { s = 0; ph ^= 1; }
        }
        umma_commit_pair(tfull(acc), 3);
        if (++acc == 2) { acc = 0; aph ^= 1; }
      }
    mma_done:
      // every MMA issued has completed before TMEM and shared memory go away
      // (waited for even after an abort, so the wait ignores the abort flag)
      umma_commit_pair(done, 1);
      volatile int keep_waiting = 0;
      mbar_wait(done, 0, &keep_waiting, p.err, 16);
    }
  } else {  // ---- epilogue: warps 2..9 of both CTAs, one accumulator row per thread ----
    const int quarter = warp & 3;                 // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;             // which half of the tile's columns
    constexpr int kHalf = BN / 64;                // chunks of 32 columns per half
    float ca = 0.f, cb = 0.f, cc = 0.f;
    if (OP == TC_POLY) {
      const float* cf = step_coef(p.sc, p.step);
      ca = cf[0]; cb = cf[1]; cc = cf[2];
    }
    int acc = 0;
    uint32_t aph = 0;
    for (int t = pair; t < num_tiles; t += npairs) {
      int b, tm, tn;
      decode<OP, BN, BM2>(t, p, b, tm, tn);
      if (!mbar_wait(tfull(acc), aph, abort_flag, p.err, 8)) break;
      tc_fence_after();
      epilogue_tile<TY, OP, BN>(p, tmem_base + (uint32_t)(acc * BN), quarter, lane, b,
                                tm * BM2 + (int)rank * 128, tn * BN, ca, cb, cc,
                                epi + (warp - 2) * (32 * 17), half * kHalf, half * kHalf + kHalf);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to(tempty(acc), 0));
      if (++acc == 2) { acc = 0; aph ^= 1; }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // neither CTA leaves while the pair's MMAs or copies may touch it
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kCols)
                 : "memory");
  }
}

}  // namespace

// ---------------------------------------------------------------- host side

namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// 3-D map over [B][rows][inner] (logical extents; pitch in elements), 128-byte
// swizzle, zero fill outside the extents.
cudaError_t make_map(CUtensorMap* m, const void* base, int ns_type, int64_t inner, int64_t rows,
                     int64_t B, int64_t pitch, uint32_t box0, uint32_t box1) {
  EncodeFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)(pitch * 2), (cuuint64_t)(rows * pitch * 2)};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, ns_type == NS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int BN, int TM = BM>
static int32_t tile_walk(bool sym, int64_t m, int64_t n, int32_t* tm, int32_t* tn, int32_t cap) {
  const int tiles_m = (int)((m + TM - 1) / TM);
  const int tiles_n = (int)(((sym ? m : n) + BN - 1) / BN);
  const int count = sym ? sym_tiles_per_batch<BN, TM>(tiles_m, tiles_n) : tiles_m * tiles_n;
  for (int t = 0; t < count && t < cap; ++t) {
    int a = 0, b = 0;
    if (sym) decode_sym<BN, TM>(t, tiles_m, tiles_n, a, b);
    else decode_raster(t, tiles_m, tiles_n, a, b);
    tm[t] = a;
    tn[t] = b;
  }
  return count;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <typename TY, int OP, int BN>
cudaError_t run(const CUtensorMap& ma, const CUtensorMap& mb, const TcArgs& p, cudaStream_t s,
                bool prepare) {
  auto fn = k_tc_gemm<TY, OP, BN>;
  if (prepare)
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcSmem<BN>::kTotal);
  TcArgs q = p;
  if (OP != TC_UPDATE) q.tiles_sym = sym_tiles_per_batch<BN>(p.tiles_m, p.tiles_n);
  const int tiles = q.B * (OP == TC_UPDATE ? q.tiles_m * q.tiles_n : q.tiles_sym);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  fn<<<grid, kThreads, TcSmem<BN>::kTotal, s>>>(ma, mb, q);
  return cudaGetLastError();
}

template <int OP, int BN>
cudaError_t run_t(int ns_type, const CUtensorMap& ma, const CUtensorMap& mb, const TcArgs& p,
                  cudaStream_t s, bool prep) {
  return ns_type == NS_BF16 ? run<__nv_bfloat16, OP, BN>(ma, mb, p, s, prep)
                            : run<__half, OP, BN>(ma, mb, p, s, prep);
}

// The CTA-pair form: p.tiles_m counts 256-row tiles; a grid of pairs, at
// most one per two SMs, walks the tiles.
template <typename TY, int OP>
cudaError_t run_pair(const CUtensorMap& ma, const CUtensorMap& mb, const TcArgs& p, cudaStream_t s,
                     bool prepare) {
  auto fn = k_tc_gemm2<TY, OP>;
  if (prepare)
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem2::kTotal);
  TcArgs q = p;
  if (OP != TC_UPDATE) q.tiles_sym = sym_tiles_per_batch<256, BM2>(p.tiles_m, p.tiles_n);
  const int tiles = q.B * (OP == TC_UPDATE ? q.tiles_m * q.tiles_n : q.tiles_sym);
  const int pairs = tiles < num_sms() / 2 ? tiles : num_sms() / 2;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(2 * pairs);
  lc.blockDim = dim3(kThreads2);
  lc.dynamicSmemBytes = TcSmem2::kTotal;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, fn, ma, mb, q);
}

template <int OP>
cudaError_t run_pair_t(int ns_type, const CUtensorMap& ma, const CUtensorMap& mb, const TcArgs& p,
                       cudaStream_t s, bool prep) {
  return ns_type == NS_BF16 ? run_pair<__nv_bfloat16, OP>(ma, mb, p, s, prep)
                            : run_pair<__half, OP>(ma, mb, p, s, prep);
}

template <int OP>
cudaError_t run_bn(int bn, int ns_type, const CUtensorMap& ma, const CUtensorMap& mb,
                   const TcArgs& p, cudaStream_t s, bool prep) {
  return bn == 256 ? run_t<OP, 256>(ns_type, ma, mb, p, s, prep)
                   : run_t<OP, 128>(ns_type, ma, mb, p, s, prep);
}

TcArgs base_args(const KArgs& a) {
  TcArgs p{};
  p.B = a.B;
  p.sc = a.sc;
  p.err = a.err;
  return p;
}

int tc_bn_square(int64_t m) { return m >= 256 ? 256 : 128; }
int tc_bn_update(int64_t n) { return n >= 256 ? 256 : 128; }
// Groups with m >= 256 run every product in the CTA-pair form (256 x 256
// tiles); smaller m would leave most of a 256-row tile empty.
bool tc_pair(int64_t m) { return m >= 256; }

}  // namespace

int32_t tc_tile_walk(int32_t op, int64_t m, int64_t n, int32_t bm, int32_t bn, int32_t* tm,
                     int32_t* tn, int32_t cap) {
  const bool sym = op == TC_GRAM || op == TC_POLY;
  if ((!sym && op != TC_UPDATE) || m < 1 || m > (1ll << 20) || (!sym && (n < 1 || n > (1ll << 20))) ||
      (bn != 128 && bn != 256) || (bm != 128 && bm != 256) || (bm == 256 && bn != 256) || cap < 0 ||
      (cap && (!tm || !tn)))
    return -1;
  if (bm == 256) return tile_walk<256, BM2>(sym, m, n, tm, tn, cap);
  return bn == 256 ? tile_walk<256>(sym, m, n, tm, tn, cap) : tile_walk<128>(sym, m, n, tm, tn, cap);
}

bool tc_pair_form(int64_t m) { return tc_pair(m); }

cudaError_t tc_make_maps(const KArgs& a, TcMaps* t) {
  const int bs = tc_bn_square(a.m), bu = tc_bn_update(a.n);
  void* ys[2] = {a.y0, a.y1};
  cudaError_t e;
  for (int i = 0; i < 2; ++i) {
    if ((e = make_map(&t->y_k128[i], ys[i], a.ns_type, a.n, a.m, a.B, a.n_pitch, 64, 128))) return e;
    if ((e = make_map(&t->y_ksq[i], ys[i], a.ns_type, a.n, a.m, a.B, a.n_pitch, 64, bs))) return e;
    if ((e = make_map(&t->y_mn[i], ys[i], a.ns_type, a.n, a.m, a.B, a.n_pitch, 64, 64))) return e;
  }
  if ((e = make_map(&t->a_k128, a.A, a.ns_type, a.m, a.m, a.B, a.m_pitch, 64, 128))) return e;
  if ((e = make_map(&t->a_ksq, a.A, a.ns_type, a.m, a.m, a.B, a.m_pitch, 64, bs))) return e;
  if ((e = make_map(&t->q_k128, a.Q, a.ns_type, a.m, a.m, a.B, a.m_pitch, 64, 128))) return e;
  t->bn_sq = bs;
  t->bn_up = bu;
  return cudaSuccess;
}

cudaError_t prepare_tc(int ns_type) {
  const CUtensorMap m{};
  const TcArgs p{};
  cudaError_t e;
  for (int bn : {128, 256}) {
    if ((e = run_bn<TC_GRAM>(bn, ns_type, m, m, p, nullptr, true))) return e;
    if ((e = run_bn<TC_POLY>(bn, ns_type, m, m, p, nullptr, true))) return e;
    if ((e = run_bn<TC_UPDATE>(bn, ns_type, m, m, p, nullptr, true))) return e;
  }
  if ((e = run_pair_t<TC_GRAM>(ns_type, m, m, p, nullptr, true))) return e;
  if ((e = run_pair_t<TC_POLY>(ns_type, m, m, p, nullptr, true))) return e;
  return run_pair_t<TC_UPDATE>(ns_type, m, m, p, nullptr, true);
}

cudaError_t launch_tc_gram(const KArgs& a, const TcMaps& t, int src, cudaStream_t s) {
  TcArgs p = base_args(a);
  p.M = a.m; p.N = a.m; p.K = a.n;
  p.tiles_m = (a.m + BM - 1) / BM;
  p.tiles_n = (a.m + t.bn_sq - 1) / t.bn_sq;
  p.ldc = a.m_pitch; p.sC = (int64_t)a.m * a.m_pitch;
  p.C = a.A;
  p.scale = 1.f / (a.alpha * a.alpha);
  if (tc_pair(a.m)) {
    p.tiles_m = p.tiles_n = (a.m + BM2 - 1) / BM2;
    return run_pair_t<TC_GRAM>(a.ns_type, t.y_k128[src], t.y_k128[src], p, s, false);
  }
  return run_bn<TC_GRAM>(t.bn_sq, a.ns_type, t.y_k128[src], t.y_ksq[src], p, s, false);
}

cudaError_t launch_tc_poly(const KArgs& a, const TcMaps& t, int step, cudaStream_t s) {
  TcArgs p = base_args(a);
  p.step = step;
  p.M = a.m; p.N = a.m; p.K = a.m;
  p.tiles_m = (a.m + BM - 1) / BM;
  p.tiles_n = (a.m + t.bn_sq - 1) / t.bn_sq;
  p.ldc = a.m_pitch; p.sC = (int64_t)a.m * a.m_pitch;
  p.C = a.Q;
  p.aux = a.A;
  if (tc_pair(a.m)) {
    p.tiles_m = p.tiles_n = (a.m + BM2 - 1) / BM2;
    return run_pair_t<TC_POLY>(a.ns_type, t.a_k128, t.a_k128, p, s, false);
  }
  return run_bn<TC_POLY>(t.bn_sq, a.ns_type, t.a_k128, t.a_ksq, p, s, false);
}

cudaError_t launch_tc_update(const KArgs& a, const TcMaps& t, int src, cudaStream_t s) {
  TcArgs p = base_args(a);
  p.M = a.m; p.N = a.n; p.K = a.m;
  p.tiles_m = (a.m + BM - 1) / BM;
  p.tiles_n = (a.n + t.bn_up - 1) / t.bn_up;
  p.ldc = a.n_pitch; p.sC = (int64_t)a.m * a.n_pitch;
  p.C = src == 0 ? a.y1 : a.y0;
  if (tc_pair(a.m)) {
    p.tiles_m = (a.m + BM2 - 1) / BM2;
    p.tiles_n = (a.n + 255) / 256;
    return run_pair_t<TC_UPDATE>(a.ns_type, t.q_k128, t.y_mn[src], p, s, false);
  }
  return run_bn<TC_UPDATE>(t.bn_up, a.ns_type, t.q_k128, t.y_mn[src], p, s, false);
}

}  // namespace muon
