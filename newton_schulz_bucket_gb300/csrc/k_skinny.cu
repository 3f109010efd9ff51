// Skinny path: Newton-Schulz for small m = min(rows, cols) <= 64.
//
// «MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化: for
// shapes such as [24, 10240] the per-parameter iteration is dominated by host
// dispatch, small allocations and synchronisation; batching every member of a
// shape into one launch removes that (Fig. 7).  On this GPU the batched work
// is bound by memory traffic and by the latency of the k dependent steps, so
// the path is built around two kernels:
//
//  1. the streaming momentum kernel (k_elementwise.cu) writes M' = beta M + G
//     and fixed-chunk partial sums of squares (HBM bound, fully coalesced);
//  2. k_skinny_ns below: one cluster of kCL CTAs per member.  CTA r owns
//     columns [r W, (r+1) W) of the wide m x n iterate.  The iterate is kept in
//     an L2-resident workspace in the exact register order of mma.sync
//     fragments, so each pass is: load fragments -> Y <- Q Y (mma.sync, with
//     movmatrix transposes for the B operand) -> accumulate the next Gram
//     Y Y^T from the same registers -> store fragments.  No shared-memory
//     round trip of the iterate, one pass over it per Newton-Schulz step.
//     Operands of each pass stream through a per-thread cp.async ring.
//     Per step the per-warp Gram partials are summed in a fixed warp order,
//     then over the cluster's CTAs in rank order (distributed shared memory),
//     and every CTA forms Q = a I + b A + c A A in fp32.
//
// Writing aX + (bA + cAA)X as (aI + bA + cAA)X keeps one product per step
// («关于分布式Muon的想法整合及讨论» §2, §6: Gram matrix, then matrix products;
// A changes with X every round).  All reduction orders depend only on
// (rows, cols), so a member gives the same bits in any batch.
#include "common.cuh"

namespace muon {

namespace {

constexpr int kCL = 2;  // CTAs per member (cluster size), fixed for every shape

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Asynchronous global -> shared copies (per thread, no barrier needed when a
// thread reads back only what it copied).  src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename TY> struct Mma;
template <> struct Mma<__half> {
  static __device__ __forceinline__ void run(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float x, float y) {
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return __half22float2(*reinterpret_cast<__half2*>(&u));
  }
};
template <> struct Mma<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
  }
};

// Gram tiles (m16 x n8) touching the upper triangle, in a fixed order.
template <int MT>
struct GramTiles {
  static constexpr int count() {
    int c = 0;
    for (int mi = 0; mi < MT; ++mi)
      for (int nj = 0; nj < 2 * MT; ++nj)
        if (nj * 8 + 7 >= mi * 16) ++c;
    return c;
  }
  static constexpr int N = count();
  __device__ __forceinline__ static void tile(int t, int& mi, int& nj) {
    int c = 0;
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
      for (int b = 0; b < 2 * MT; ++b)
        if (b * 8 + 7 >= a * 16) {
          if (c == t) { mi = a; nj = b; }
          ++c;
        }
  }
};

// Shared memory (bytes): the cp.async stage ring, per-warp Gram partials, the
// CTA partial (double buffered, read by the peer), A (fp32), Q (operand type).
template <int MT, int NT>
struct NsSmem {
  static constexpr int MP = 16 * MT;
  static constexpr int NW = NT / 32;
  static constexpr int LB = 32 * MT;  // stage bytes per lane and block
  // rounds in flight; MT <= 2 fits two CTAs per SM, so every cluster of a
  // batch of up to ~76 members is resident at once
  static constexpr int S = MT == 1 ? 8 : (MT == 2 ? 5 : (MT == 3 ? 4 : 2));
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
  uint8_t* ws;  // fragment workspace [B][kCL][NB][blk]
};

// Offsets of element (i, j) of the wide iterate in the parameter's memory.
struct Wide {
  int cols, T;
  __device__ __forceinline__ int64_t off(int i, int j) const {
    return T ? (int64_t)j * cols + i : (int64_t)i * cols + j;
  }
};

template <typename TY, int MT, int NT>
__global__ void __launch_bounds__(NT, (MT <= 2 ? 2 : 1)) k_skinny_ns(KArgs a, SkArgs s) {
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
  const int g = lane >> 2, t4 = lane & 3;
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / kCL;
  const int m = a.m, n = a.n;
  const int c0 = (int)rank * s.W;
  const MemberPtrs mp = a.mem[b];
  const float* Mp = mp.M;
  __nv_bfloat16* P = static_cast<__nv_bfloat16*>(mp.P);
  const Wide wd{a.cols, a.T};
  // pairs (i, j), (i, j+1) are adjacent in memory (fast path) when the wide
  // iterate is the parameter itself, its rows are even and bases are aligned
  const bool pairs = !a.T && (a.cols % 2 == 0) &&
                     ((reinterpret_cast<uintptr_t>(Mp) | reinterpret_cast<uintptr_t>(P)) & 7) == 0;
  uint8_t* ws = s.ws + ((int64_t)b * kCL + rank) * s.NB * s.blk;

  // Q = 0 outside the m x m block; zero once
  for (int e = tid; e < MP * (MP + 8); e += NT) Qs[e] = from_f32<TY>(0.f);
  // the member's norm from the momentum kernel's fixed-chunk partials
  if (tid == 0) {
    const float* pp = a.part + (int64_t)b * a.n_chunks;
    float s2 = 0.f;
    for (int c = 0; c < a.n_chunks; ++c) s2 += pp[c];
    misc[0] = a.alpha / (sqrtf(s2) + a.eps);
  }
  __syncthreads();
  const float inv = misc[0];

  const int ns = a.sc->ns_steps;
  const float ca = a.sc->a, cb = a.sc->b, cc = a.sc->c;
  const float inv_a2 = 1.f / (a.alpha * a.alpha);
  const float lr = a.sc->lr, wdk = a.sc->wd;
  const float decay = 1.f - lr * wdk;
  const float inv_alpha = 1.f / a.alpha;
  const float coef = lr * a.scale * inv_alpha;
  float* dbg = a.dbg ? a.dbg + (int64_t)b * a.rows * a.cols : nullptr;

  // rows of m16 tile mi that hold data; a tile with <= 8 stores only a0, a2
  auto tile_off = [&](int mi) {
    int o = 0;
    for (int q = 0; q < mi; ++q) o += (m - 16 * q > 8) ? 512 : 256;
    return o;
  };

  // pass p = 0: fragments from M' / norm;  0 < p: Y <- Q Y;  p = k: write P
  for (int p = 0; p <= ns; ++p) {
    const bool first = p == 0, last = p == ns;
    uint32_t qf[MT][MT][4];
    if (!first) {
      const uint32_t qb = smem_u32(Qs);
#pragma unroll
      for (int mi = 0; mi < MT; ++mi)
#pragma unroll
        for (int kk = 0; kk < MT; ++kk)
          ldsm_x4(qb + 2u * ((mi * 16 + (lane & 15)) * (MP + 8) + kk * 16 + (lane >> 4) * 8),
                  qf[mi][kk]);
    }
    float gacc[GT::N][4];
#pragma unroll
    for (int q = 0; q < GT::N; ++q) gacc[q][0] = gacc[q][1] = gacc[q][2] = gacc[q][3] = 0.f;

    // Round r: warp w handles block r * NW + w.  Each lane streams its own
    // operands of the next S rounds into a shared-memory ring with cp.async
    // (fragments, or M' pairs in the first pass, plus P pairs in the last),
    // and reads back only what it copied, so no block barrier is needed.
    constexpr int S = L::S, LB = L::LB;
    const int rounds = (s.NB + NW - 1) / NW;
    const bool stream_pairs = pairs;                // aligned pair layout: M' via cp.async
    const bool stream_p = pairs && last && !first;  // P pairs via cp.async (own stage area)
    // Stage of one warp and round: 32 * LB bytes as "planes", each plane
    // holding one 4/8/16-byte item for all 32 lanes contiguously, so fills and
    // reads are bank-conflict free.  Plane offsets (bytes, for lane 0):
    //   first pass : M' pair k       at k * 256          (k < 4 MT)
    //   later      : fragment tile mi at mi * 512         (16 or 8 bytes / lane)
    //   last pass  : P pair k        at MT * 512 + k * 128
    const uint32_t stage0 = smem_u32(smem + L::kStage) + (uint32_t)(warp * 32 * LB);
    auto slot = [&](int r) { return stage0 + (uint32_t)((r % S) * NW * 32 * LB); };
    auto issue = [&](int r) {
      const int blk = r * NW + warp;
      if (r < rounds && blk < s.NB) {
        const uint32_t dst = slot(r);
        const int jb = c0 + blk * 16;
        if (first) {
          if (stream_pairs) {
#pragma unroll
            for (int mi = 0; mi < MT; ++mi)
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int i = mi * 16 + g + ((q & 1) ? 8 : 0);
                const int j = jb + 2 * t4 + ((q & 2) ? 8 : 0);
                const bool ok = i < m && j + 1 < n;
                cp_async8(dst + (mi * 4 + q) * 256 + lane * 8,
                          ok ? (const void*)(Mp + wd.off(i, j)) : (const void*)Mp, ok ? 8 : 0);
              }
          }
        } else {
          const uint8_t* wsb = ws + (int64_t)blk * s.blk;
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            const int o = tile_off(mi);
            if (m - 16 * mi > 8)
              cp_async16(dst + mi * 512 + lane * 16, wsb + o + lane * 16, 16);
            else
              cp_async8(dst + mi * 512 + lane * 8, wsb + o + lane * 8, 8);
          }
        }
        if (stream_p) {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = mi * 16 + g + ((q & 1) ? 8 : 0);
              const int j = jb + 2 * t4 + ((q & 2) ? 8 : 0);
              const bool ok = i < m && j + 1 < n;
              cp_async4(dst + MT * 512 + (mi * 4 + q) * 128 + lane * 4,
                        ok ? (const void*)(P + wd.off(i, j)) : (const void*)P, ok ? 4 : 0);
            }
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int r = 0; r < S; ++r) issue(r);

    for (int r = 0; r < rounds; ++r) {
      cp_async_wait<S - 1>();
      const int blk = r * NW + warp;
      if (blk < s.NB) {
        const int jb = c0 + blk * 16;
        uint8_t* wsb = ws + (int64_t)blk * s.blk;
        const uint8_t* st = smem + L::kStage + (r % S) * NW * 32 * LB + warp * 32 * LB;
        uint32_t y[MT][4];
        uint32_t pv[MT][4];  // last pass: P pairs (bf16x2)
        if (first) {
          // fragment registers from M' (fp32) scaled by alpha / ||M'||
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = mi * 16 + g + ((q & 1) ? 8 : 0);
              const int j = jb + 2 * t4 + ((q & 2) ? 8 : 0);
              float v0 = 0.f, v1 = 0.f;
              if (stream_pairs) {
                const float2 f = *reinterpret_cast<const float2*>(st + (mi * 4 + q) * 256 + lane * 8);
                v0 = f.x; v1 = f.y;
              } else if (i < m) {
                if (j < n) v0 = Mp[wd.off(i, j)];
                if (j + 1 < n) v1 = Mp[wd.off(i, j + 1)];
              }
              y[mi][q] = Mma<TY>::pack(v0 * inv, v1 * inv);
            }
          }
        } else {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            if (m - 16 * mi > 8) {
              const uint4 v = *reinterpret_cast<const uint4*>(st + mi * 512 + lane * 16);
              y[mi][0] = v.x; y[mi][1] = v.y; y[mi][2] = v.z; y[mi][3] = v.w;
            } else {
              const uint2 v = *reinterpret_cast<const uint2*>(st + mi * 512 + lane * 8);
              y[mi][0] = v.x; y[mi][1] = 0u; y[mi][2] = v.y; y[mi][3] = 0u;
            }
          }
          // Y <- Q Y: B operand rows are iterate rows, so transpose 8x8 blocks
          uint32_t bt[MT][4];
#pragma unroll
          for (int kk = 0; kk < MT; ++kk)
#pragma unroll
            for (int q = 0; q < 4; ++q) bt[kk][q] = movtrans(y[kk][q]);
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
        if (stream_p) {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              pv[mi][q] = *reinterpret_cast<const uint32_t*>(st + MT * 512 + (mi * 4 + q) * 128 +
                                                            lane * 4);
        }
        if (!last) {
          // next Gram: Y Y^T over this block, upper tiles, B operand = rows of Y
#pragma unroll
          for (int q = 0; q < GT::N; ++q) {
            int mi = 0, nj = 0;
            GT::tile(q, mi, nj);
            const uint32_t* src = y[nj >> 1];
            const uint32_t b0 = (nj & 1) ? src[1] : src[0];
            const uint32_t b1 = (nj & 1) ? src[3] : src[2];
            Mma<TY>::run(gacc[q], y[mi], b0, b1);
          }
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            const int o = tile_off(mi);
            if (m - 16 * mi > 8)
              *reinterpret_cast<uint4*>(wsb + o + lane * 16) =
                  make_uint4(y[mi][0], y[mi][1], y[mi][2], y[mi][3]);
            else
              *reinterpret_cast<uint2*>(wsb + o + lane * 8) = make_uint2(y[mi][0], y[mi][2]);
          }
        } else {
          // P' = P (1 - lr wd) - lr s Y / alpha on the valid elements
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = mi * 16 + g + ((q & 1) ? 8 : 0);
              const int j = jb + 2 * t4 + ((q & 2) ? 8 : 0);
              if (i >= m || j >= n) continue;
              const float2 yv = Mma<TY>::unpack(y[mi][q]);
              if (pairs && j + 1 < n) {
                uint32_t praw = stream_p ? pv[mi][q]
                                         : *reinterpret_cast<const uint32_t*>(P + wd.off(i, j));
                const float2 pf = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&praw));
                *reinterpret_cast<__nv_bfloat162*>(P + wd.off(i, j)) = __floats2bfloat162_rn(
                    fmaf(-coef, yv.x, pf.x * decay), fmaf(-coef, yv.y, pf.y * decay));
                if (dbg)
                  *reinterpret_cast<float2*>(dbg + wd.off(i, j)) =
                      make_float2(yv.x * inv_alpha, yv.y * inv_alpha);
              } else {
                const int64_t o0 = wd.off(i, j);
                P[o0] = __float2bfloat16_rn(fmaf(-coef, yv.x, __bfloat162float(P[o0]) * decay));
                if (dbg) dbg[o0] = yv.x * inv_alpha;
                if (j + 1 < n) {
                  const int64_t o1 = wd.off(i, j + 1);
                  P[o1] = __float2bfloat16_rn(fmaf(-coef, yv.y, __bfloat162float(P[o1]) * decay));
                  if (dbg) dbg[o1] = yv.y * inv_alpha;
                }
              }
            }
          }
        }
      }
      // the slot of round r was consumed above (registers): refill it
      issue(r + S);
    }
    cp_async_wait<0>();
    if (last) break;

    // ---- reduce the Gram partials: warps (fixed order), then CTAs (rank order)
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
      int mi = 0, nj = 0;
      GT::tile(q, mi, nj);
      cp[(mi * 16 + (w >> 3)) * MP + nj * 8 + (w & 7)] = acc;
    }
    cluster_sync();
    for (int e = tid; e < m * m; e += NT) {
      const int i = e / m, j = e - (e / m) * m;
      if (i > j) continue;
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < kCL; ++r) acc += ld_dsmem_f32(&cp[i * MP + j], (uint32_t)r);
      acc *= inv_a2;
      Af[i * MP + j] = acc;
      Af[j * MP + i] = acc;
    }
    __syncthreads();
    // Q = a I + b A + c A A (fp32), cast to the operand type
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
  }
  // the peer may still read this CTA's Gram partial
  cluster_sync();
}

template <typename TY, int MT, int NT>
cudaError_t launch_t(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prepare) {
  auto fn = k_skinny_ns<TY, MT, NT>;
  constexpr int smem = NsSmem<MT, NT>::kTotal;
  if (prepare) return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  SkArgs s;
  s.W = cfg.width;
  s.NB = cfg.width / 16;
  s.blk = cfg.blk;
  s.ws = static_cast<uint8_t*>(a.y0);
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(a.B * kCL);
  lc.blockDim = dim3(NT);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, fn, a, s);
}

template <typename TY>
cudaError_t launch_ty(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prep) {
  switch (cfg.mtiles) {
    case 1: return launch_t<TY, 1, 256>(a, cfg, st, prep);
    case 2: return launch_t<TY, 2, 256>(a, cfg, st, prep);
    case 3: return launch_t<TY, 3, 256>(a, cfg, st, prep);
    default: return launch_t<TY, 4, 256>(a, cfg, st, prep);
  }
}

cudaError_t dispatch(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t st, bool prep) {
  if (a.mode_f32) return cudaErrorInvalidValue;  // fp32 parameters use the SIMT path
  return a.ns_type == NS_F16 ? launch_ty<__half>(a, cfg, st, prep)
                             : launch_ty<__nv_bfloat16>(a, cfg, st, prep);
}

template <typename TY, int MT>
int clusters_of() {
  auto fn = k_skinny_ns<TY, MT, 256>;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(kCL * 1024);
  lc.blockDim = dim3(256);
  lc.dynamicSmemBytes = NsSmem<MT, 256>::kTotal;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, fn, &lc) == cudaSuccess ? n : -1;
}

}  // namespace

bool skinny_config(int32_t rows, int32_t cols, int32_t max_m, SkinnyCfg* cfg) {
  const int m = rows < cols ? rows : cols, n = rows < cols ? cols : rows;
  if (m < 1 || m > max_m || m > 64) return false;
  cfg->mtiles = (m + 15) / 16;
  cfg->cluster = kCL;
  cfg->threads = 256;
  const int w = (n + kCL - 1) / kCL;
  cfg->width = (w + 15) / 16 * 16;
  int blk = 0;
  for (int q = 0; q < cfg->mtiles; ++q) blk += (m - 16 * q > 8) ? 512 : 256;
  cfg->blk = blk;
  cfg->ws_bytes = (int64_t)kCL * (cfg->width / 16) * blk;  // per member
  cfg->smem = 0;
  return true;
}

cudaError_t prepare_skinny(const KArgs& a, const SkinnyCfg& cfg) {
  return dispatch(a, cfg, nullptr, true);
}

cudaError_t launch_skinny(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s) {
  return dispatch(a, cfg, s, false);
}

int skinny_max_active_clusters(int ns_type, int mtiles) {
  if (ns_type == NS_F16)
    switch (mtiles) {
      case 1: return clusters_of<__half, 1>();
      case 2: return clusters_of<__half, 2>();
      case 3: return clusters_of<__half, 3>();
      default: return clusters_of<__half, 4>();
    }
  switch (mtiles) {
    case 1: return clusters_of<__nv_bfloat16, 1>();
    case 2: return clusters_of<__nv_bfloat16, 2>();
    case 3: return clusters_of<__nv_bfloat16, 3>();
    default: return clusters_of<__nv_bfloat16, 4>();
  }
}

}  // namespace muon
