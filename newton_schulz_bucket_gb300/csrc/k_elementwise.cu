// Elementwise passes:
//   momentum + partial sums of squares (every path), norm finalisation,
//   normalise + cast (+ transpose to the wide orientation), and the scaled,
//   decayed write (TENSOR / SIMT paths).
// Momentum M' = beta M + G and the sum-of-squares normaliser follow
// «关于分布式Muon的想法整合及讨论» §1, §2 and §6; the write
// P' = P (1 - lr wd) - lr s O is the scaled, weight-decayed update.
#include "common.cuh"

namespace muon {

namespace {

constexpr int kThreads = 256;

// Eight consecutive elements (16- or 32-byte aligned) to / from fp32.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f) {
  if constexpr (sizeof(T) == 4) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = to_f32(h[e]);
  }
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float* f) {
  if constexpr (sizeof(T) == 4) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
  } else {
    uint4 u;
    T* h = reinterpret_cast<T*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = from_f32<T>(f[e]);
    *reinterpret_cast<uint4*>(p) = u;
  }
}

// One CTA = one fixed chunk of one member: M' = beta M + G (stored), and the
// chunk's sum of squares of X = M' (Nesterov: X = U = G + beta M') by a
// fixed-order tree into part[b][chunk]; with a.u set, U is stored there too.
// G and M are read once (evict-first in L2).  M' is stored evict-last when the
// next kernel reads it back twice (skinny path), so it is still in L2 then.
template <typename TG>
__global__ void __launch_bounds__(kThreads) k_momentum_partial(KArgs a) {
  __shared__ float red[33];
  const int b = blockIdx.y;
  const int64_t total = (int64_t)a.m * a.n;
  const int64_t start = (int64_t)blockIdx.x * kMomentumChunk;
  const int64_t end = min(start + kMomentumChunk, total);
  const MemberPtrs mp = a.mem[b];
  const TG* G = static_cast<const TG*>(mp.G);
  float* M = mp.M;
  const float beta = a.sc->beta;
  const bool nest = a.nesterov != 0;
  float* U = a.u ? a.u + (int64_t)b * total : nullptr;
  float acc = 0.f;
  const bool vec = aligned16(G) && aligned16(M) && (!U || aligned16(U));
  const uint64_t pin = l2_evict_first();
  const uint64_t pout = a.l2_keep_m ? l2_evict_last() : l2_evict_normal();
  auto load8g = [&](const TG* p, float* f) {
    if constexpr (sizeof(TG) == 2) {
      bf16x8_to_f32(ld_hint(p, pin), f);
    } else {
      u4_to_f4x2(ld_hint(p, pin), ld_hint(p + 4, pin), f);
    }
  };
  int64_t i0 = start;
  if (vec) {
    constexpr int UN = 4;  // 4 x 8 elements in flight per thread
    const int64_t stride = (int64_t)8 * kThreads;
    int64_t i = start + 8 * threadIdx.x;
    for (; i + (UN - 1) * stride + 8 <= end; i += UN * stride) {
      float g[UN][8], m[UN][8];
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        load8g(G + i + u * stride, g[u]);
        u4_to_f4x2(ld_hint(M + i + u * stride, pin), ld_hint(M + i + u * stride + 4, pin), m[u]);
      }
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          m[u][e] = fmaf(beta, m[u][e], g[u][e]);
          x[e] = nest ? fmaf(beta, m[u][e], g[u][e]) : m[u][e];
          acc = fmaf(x[e], x[e], acc);
        }
        st_hint(M + i + u * stride, f4_to_u4(m[u]), pout);
        st_hint(M + i + u * stride + 4, f4_to_u4(m[u] + 4), pout);
        if (U) {
          st_hint(U + i + u * stride, f4_to_u4(x), pout);
          st_hint(U + i + u * stride + 4, f4_to_u4(x + 4), pout);
        }
      }
    }
    for (; i + 8 <= end; i += stride) {
      float g[8], m[8], x[8];
      load8g(G + i, g);
      u4_to_f4x2(ld_hint(M + i, pin), ld_hint(M + i + 4, pin), m);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        m[e] = fmaf(beta, m[e], g[e]);
        x[e] = nest ? fmaf(beta, m[e], g[e]) : m[e];
        acc = fmaf(x[e], x[e], acc);
      }
      st_hint(M + i, f4_to_u4(m), pout);
      st_hint(M + i + 4, f4_to_u4(m + 4), pout);
      if (U) {
        st_hint(U + i, f4_to_u4(x), pout);
        st_hint(U + i + 4, f4_to_u4(x + 4), pout);
      }
    }
    i0 = start + ((end - start) / 8) * 8;  // scalar tail below
  }
  for (int64_t i = i0 + threadIdx.x; i < end; i += kThreads) {
    const float g = to_f32(G[i]);
    const float v = fmaf(beta, M[i], g);
    M[i] = v;
    const float x = nest ? fmaf(beta, v, g) : v;
    if (U) U[i] = x;
    acc = fmaf(x, x, acc);
  }
  const float s = block_sum(acc, red);
  if (threadIdx.x == 0) a.part[(int64_t)b * a.n_chunks + blockIdx.x] = s;
}

// invn[b] = alpha / (sqrt(sum of partials) + eps), partials summed in a fixed
// order so the result depends only on the member's data.
__global__ void __launch_bounds__(kThreads) k_norm_finalize(KArgs a) {
  __shared__ float red[33];
  const int b = blockIdx.x;
  const float* p = a.part + (int64_t)b * a.n_chunks;
  float acc = 0.f;
  for (int i = threadIdx.x; i < a.n_chunks; i += kThreads) acc += p[i];
  const float s = block_sum(acc, red);
  if (threadIdx.x == 0) a.invn[b] = a.alpha / (sqrtf(s) + a.eps);
}

// Y[b] = cast(X[b] * invn[b]) in the wide orientation, X = M' (Nesterov:
// U = G + beta M'): Y is m x n with row pitch n_pitch; for T (rows > cols)
// Y = X^T.  64 x 64 tiles through shared memory so both the reads and the
// write of Y are coalesced.
template <typename TY>
__global__ void __launch_bounds__(kThreads) k_normalize_cast(KArgs a, TY* __restrict__ Y) {
  __shared__ float tile[64][65];
  const int b = blockIdx.z;
  const float* Mp = a.mem[b].M;
  const void* Gp = a.mem[b].G;
  const bool nest = a.nesterov != 0;
  const float beta = a.sc->beta;
  const float inv = a.invn[b];
  TY* Yb = Y + (int64_t)b * a.m * a.n_pitch;
  // the grid walks the wide m x n iterate; in parameter coordinates a tile
  // keeps its origin, or swaps it for a transposed member
  const bool T = a.mem[b].T != 0;
  const int rows = T ? a.n : a.m, cols = T ? a.m : a.n;
  const int r0 = (T ? blockIdx.x : blockIdx.y) * 64, c0 = (T ? blockIdx.y : blockIdx.x) * 64;
  // Untransposed member, whole tile width, 8-element alignment: each thread
  // moves rows (t / 8) and (t / 8 + 32), columns 8 (t % 8) .. + 7, as vectors.
  if (!T && c0 + 64 <= cols && cols % 8 == 0 && a.n_pitch % 8 == 0 && aligned16(Mp) && aligned16(Yb) &&
      (!nest || aligned16(Gp))) {
    const int cc = (threadIdx.x & 7) * 8, rr0 = threadIdx.x >> 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r0 + rr0 + 32 * h;
      if (r >= rows) continue;
      const int64_t o = (int64_t)r * cols + c0 + cc;
      float x[8];
      load8(Mp + o, x);
      if (nest) {
        float g[8];
        if (a.mode_f32) load8(static_cast<const float*>(Gp) + o, g);
        else load8(static_cast<const __nv_bfloat16*>(Gp) + o, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = fmaf(beta, x[e], g[e]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= inv;
      store8(Yb + (int64_t)r * a.n_pitch + c0 + cc, x);
    }
    return;
  }
  // Transposed member, 8-element alignment: the 64 x 64 parameter tile comes
  // in as 16-byte row vectors (4 floats of M', 8 bf16 of G), is normalised in
  // shared memory, and leaves as 16-byte vectors along the rows of Y (the
  // parameter's columns).  Y's row pitch is a multiple of 8 >= n, so a last
  // partial vector only touches Y's padding, which nothing reads.
  if (T && cols % 8 == 0 && a.n_pitch % 8 == 0 && aligned16(Mp) && aligned16(Yb) &&
      (!nest || (!a.mode_f32 && aligned16(Gp)))) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // 64 rows x 16 vectors of 4 floats
      const int v = threadIdx.x + k * kThreads, rr = v >> 4, cc = (v & 15) * 4;
      const int r = r0 + rr, c = c0 + cc;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < rows && c < cols) {
        const int64_t o = (int64_t)r * cols + c;
        const float4 t = *reinterpret_cast<const float4*>(Mp + o);
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
        if (nest) {
          const uint2 graw = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(Gp) + o);
          const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.x));
          const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.y));
          x[0] = fmaf(beta, x[0], g01.x); x[1] = fmaf(beta, x[1], g01.y);
          x[2] = fmaf(beta, x[2], g23.x); x[3] = fmaf(beta, x[3], g23.y);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) tile[rr][cc + e] = x[e] * inv;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) {  // 64 rows of Y x 8 vectors of 8
      const int v = threadIdx.x + k * kThreads, cc = v >> 3, rr = (v & 7) * 8;
      const int c = c0 + cc, r = r0 + rr;
      if (c >= cols || r >= rows) continue;
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = tile[rr + e][cc];
      store8(Yb + (int64_t)c * a.n_pitch + r, y);
    }
    return;
  }
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4
  for (int rr = ty; rr < 64; rr += 4) {
    const int r = r0 + rr, c = c0 + tx;
    float x = 0.f;
    if (r < rows && c < cols) {
      const int64_t o = (int64_t)r * cols + c;
      x = Mp[o];
      if (nest) {
        const float g = a.mode_f32 ? static_cast<const float*>(Gp)[o]
                                   : __bfloat162float(static_cast<const __nv_bfloat16*>(Gp)[o]);
        x = fmaf(beta, x, g);
      }
    }
    tile[rr][tx] = x * inv;
  }
  __syncthreads();
  if (!T) {
    for (int rr = ty; rr < 64; rr += 4) {
      const int r = r0 + rr, c = c0 + tx;
      if (r < rows && c < cols) Yb[(int64_t)r * a.n_pitch + c] = from_f32<TY>(tile[rr][tx]);
    }
  } else {
    // Y[c][r] = M'[r][c]: Y row index = parameter column
    for (int cc = ty; cc < 64; cc += 4) {
      const int c = c0 + cc, r = r0 + tx;
      if (r < rows && c < cols) Yb[(int64_t)c * a.n_pitch + r] = from_f32<TY>(tile[tx][cc]);
    }
  }
}

// P' = P (1 - lr wd) - lr s O, O = Y / alpha read back in the parameter's
// orientation.  Optional fp32 copy of O for the test hook.
template <typename TY, typename TP>
__global__ void __launch_bounds__(kThreads) k_write(KArgs a, const TY* __restrict__ Y) {
  __shared__ float tile[64][65];
  const int b = blockIdx.z;
  TP* P = static_cast<TP*>(a.mem[b].P);
  const TY* Yb = Y + (int64_t)b * a.m * a.n_pitch;
  const float lr = a.sc->lr, wd = a.sc->wd;
  const float decay = __fmaf_rn(-lr, wd, 1.f);  // one rounding of 1 - lr wd
  const MemberPtrs mp = a.mem[b];
  const float coef = lr * mp.scale / a.alpha;  // alpha is a power of two
  const float inv_alpha = 1.f / a.alpha;
  const bool T = mp.T != 0;
  const int rows = T ? a.n : a.m, cols = T ? a.m : a.n;
  const int r0 = (T ? blockIdx.x : blockIdx.y) * 64, c0 = (T ? blockIdx.y : blockIdx.x) * 64;
  float* dbg = a.dbg ? a.dbg + (int64_t)b * a.m * a.n : nullptr;
  // Untransposed member, whole tile width, 8-element alignment: vectors, as in
  // k_normalize_cast (the same arithmetic per element as below).
  if (!T && c0 + 64 <= cols && cols % 8 == 0 && a.n_pitch % 8 == 0 && aligned16(P) && aligned16(Yb) &&
      (!dbg || aligned16(dbg))) {
    const int cc = (threadIdx.x & 7) * 8, rr0 = threadIdx.x >> 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r0 + rr0 + 32 * h;
      if (r >= rows) continue;
      const int64_t idx = (int64_t)r * cols + c0 + cc;
      float y[8], pv[8], w[8];
      load8(Yb + (int64_t)r * a.n_pitch + c0 + cc, y);
      load8(P + idx, pv);
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = fmaf(-coef, y[e], pv[e] * decay);
      store8(P + idx, w);
      if (dbg) {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = y[e] * inv_alpha;
        store8(dbg + idx, w);
      }
    }
    return;
  }
  // Transposed member, 8-element alignment: the Y tile Y[c0 .. c0 + 64)
  // [r0 .. r0 + 64) comes in as 16-byte vectors along Y's rows (Y's row pitch
  // is a multiple of 8 >= n, so a last partial vector reads only padding),
  // and the parameter tile is read, updated and written as 16-byte vectors
  // along its rows (the same arithmetic per element as below).
  if (T && cols % 8 == 0 && a.n_pitch % 8 == 0 && aligned16(P) && aligned16(Yb) &&
      (!dbg || aligned16(dbg))) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {  // 64 rows of Y x 8 vectors of 8
      const int v = threadIdx.x + k * kThreads, cc = v >> 3, rr = (v & 7) * 8;
      const int c = c0 + cc, r = r0 + rr;
      float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (c < cols && r < rows) load8(Yb + (int64_t)c * a.n_pitch + r, y);
#pragma unroll
      for (int e = 0; e < 8; ++e) tile[rr + e][cc] = y[e];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) {  // 64 parameter rows x 8 vectors of 8
      const int v = threadIdx.x + k * kThreads, rr = v >> 3, cc = (v & 7) * 8;
      const int r = r0 + rr, c = c0 + cc;
      if (r >= rows || c >= cols) continue;
      const int64_t idx = (int64_t)r * cols + c;
      float y[8], pv[8], w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = tile[rr][cc + e];
      load8(P + idx, pv);
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = fmaf(-coef, y[e], pv[e] * decay);
      store8(P + idx, w);
      if (dbg) {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = y[e] * inv_alpha;
        store8(dbg + idx, w);
      }
    }
    return;
  }
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  if (T) {
    // stage the Y tile Y[c0..c0+64)[r0..r0+64) so reads are coalesced along r
    for (int cc = ty; cc < 64; cc += 4) {
      const int c = c0 + cc, r = r0 + tx;
      tile[tx][cc] = (r < rows && c < cols) ? to_f32(Yb[(int64_t)c * a.n_pitch + r]) : 0.f;
    }
    __syncthreads();
  }
  for (int rr = ty; rr < 64; rr += 4) {
    const int r = r0 + rr, c = c0 + tx;
    if (r >= rows || c >= cols) continue;
    const float y = T ? tile[rr][tx] : to_f32(Yb[(int64_t)r * a.n_pitch + c]);
    const int64_t idx = (int64_t)r * cols + c;
    const float p = to_f32(P[idx]);
    P[idx] = from_f32<TP>(fmaf(-coef, y, p * decay));
    if (dbg) dbg[idx] = y * inv_alpha;
  }
}

// 64 x 64 tiles of the wide m x n iterate (x: columns, y: rows)
dim3 tiles_of(const KArgs& a) {
  return dim3((a.n + 63) / 64, (a.m + 63) / 64, a.B);
}

}  // namespace

cudaError_t launch_momentum_partial(const KArgs& a, cudaStream_t s) {
  dim3 grid(a.n_chunks, a.B);
  if (a.mode_f32)
    k_momentum_partial<float><<<grid, kThreads, 0, s>>>(a);
  else
    k_momentum_partial<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const KArgs& a, cudaStream_t s) {
  k_norm_finalize<<<a.B, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_normalize_cast(const KArgs& a, void* dst, cudaStream_t s) {
  switch (a.ns_type) {
    case NS_F32: k_normalize_cast<float><<<tiles_of(a), kThreads, 0, s>>>(a, (float*)dst); break;
    case NS_F16: k_normalize_cast<__half><<<tiles_of(a), kThreads, 0, s>>>(a, (__half*)dst); break;
    default:
      k_normalize_cast<__nv_bfloat16><<<tiles_of(a), kThreads, 0, s>>>(a, (__nv_bfloat16*)dst);
  }
  return cudaGetLastError();
}

cudaError_t launch_write(const KArgs& a, const void* src, cudaStream_t s) {
  const dim3 g = tiles_of(a);
  if (a.mode_f32) {
    switch (a.ns_type) {
      case NS_F32: k_write<float, float><<<g, kThreads, 0, s>>>(a, (const float*)src); break;
      case NS_F16: k_write<__half, float><<<g, kThreads, 0, s>>>(a, (const __half*)src); break;
      default: k_write<__nv_bfloat16, float><<<g, kThreads, 0, s>>>(a, (const __nv_bfloat16*)src);
    }
  } else {
    switch (a.ns_type) {
      case NS_F32:
        k_write<float, __nv_bfloat16><<<g, kThreads, 0, s>>>(a, (const float*)src);
        break;
      case NS_F16:
        k_write<__half, __nv_bfloat16><<<g, kThreads, 0, s>>>(a, (const __half*)src);
        break;
      default:
        k_write<__nv_bfloat16, __nv_bfloat16><<<g, kThreads, 0, s>>>(
            a, (const __nv_bfloat16*)src);
    }
  }
  return cudaGetLastError();
}

}  // namespace muon
