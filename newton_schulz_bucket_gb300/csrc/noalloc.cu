// muon_step_skinny_static: the skinny-path step for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at step time or at all: code running
// inside a framework's pooled or capped allocator that forbids foreign
// allocations, real-time loops that must not block on the CUDA allocator,
// and embedded hosts that fix all device memory up front.  For them this entry
// point runs the same kernels as the SKINNY path of muon_step, with the same
// arguments, and keeps every byte of scratch in one file-scope device array of
// kStaticScratchBytes.  Up to kGramSpaceMaxSteps Newton-Schulz steps that
// scratch is only the step scalars and the member pointer table (the
// Gram-space kernel keeps everything else on chip); beyond, the direct
// iteration also needs the momentum kernel's partial sums and the
// fragment-ordered iterate.  The array is part of the library image: every
// GPU that loads the library holds it until the process exits.  Every call
// uses the same array, so two calls whose kernels overlap on a GPU race
// (serialise them on one stream).  No byte of the array needs to start at
// zero: each call writes every location it later reads.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/muon.h"
#include "internal.h"

namespace muon {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device, looked up once with that
// device current (the array's host-side name is not a device address), and
// whether the kernel attributes of one (m16 tiles, half last tile) variant
// have been set on that device.
unsigned char* g_scratch_addr[kMaxDevices] = {};
bool g_prepared[kMaxDevices][5][2] = {};
std::mutex g_setup_mu;

// Errors are reported through muon_last_error(), like every other entry point.
muon_status_t static_fail(muon_status_t st, const char* msg) {
  char buf[320];
  std::snprintf(buf, sizeof buf, "muon_step_skinny_static: %s", msg);
  set_last_error(buf);
  return st;
}

// One thread fills the step scalars and the member pointer table from the
// kernel's own arguments (so the call needs neither an allocation nor a host
// staging buffer).
__global__ void k_static_setup(StepScalars sc, void* P, const void* G, float* M, int batch,
                               int64_t per, int32_t T, float scale, StepScalars* sc_out,
                               MemberPtrs* mem_out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  *sc_out = sc;
  for (int b = 0; b < batch; ++b) {
    mem_out[b].P = static_cast<__nv_bfloat16*>(P) + b * per;
    mem_out[b].G = static_cast<const __nv_bfloat16*>(G) + b * per;
    mem_out[b].M = M + b * per;
    mem_out[b].T = T;
    mem_out[b].scale = scale;
  }
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" muon_status_t muon_step_skinny_static(void* params, const void* grads, float* momenta,
                                                 int32_t batch, int64_t rows, int64_t cols,
                                                 float beta, float lr, float wd, int32_t ns_steps,
                                                 float a, float b, float c, float eps,
                                                 int32_t scale_mode, void* stream) {
  if (!params || !grads || !momenta)
    return static_fail(MUON_ERR_INVALID_ARG, "params, grads and momenta must be non-NULL");
  if (batch < 1 || batch > 65535)
    return static_fail(MUON_ERR_INVALID_ARG, "batch must be in [1, 65535]");
  if (rows < 1 || cols < 1 || rows > (1 << 30) || cols > (1 << 30))
    return static_fail(MUON_ERR_INVALID_ARG, "rows and cols must be in [1, 2^30]");
  if (ns_steps < 0 || ns_steps > 1000)
    return static_fail(MUON_ERR_INVALID_ARG, "ns_steps must be in [0, 1000]");
  const float sv[7] = {beta, lr, wd, a, b, c, eps};
  for (float v : sv)
    if (!std::isfinite(v)) return static_fail(MUON_ERR_INVALID_ARG, "non-finite scalar");
  if (eps < 0.f) return static_fail(MUON_ERR_INVALID_ARG, "eps must be >= 0");
  if (scale_mode < MUON_SCALE_SQRT_ASPECT || scale_mode > MUON_SCALE_NONE)
    return static_fail(MUON_ERR_INVALID_ARG, "scale_mode is not a muon_scale_t");
  SkinnyCfg cfg;
  if (!skinny_config((int32_t)rows, (int32_t)cols, 64, &cfg))
    return static_fail(MUON_ERR_UNSUPPORTED, "min(rows, cols) must be <= 64 (skinny path)");

  const int64_t m = rows < cols ? rows : cols, n = rows < cols ? cols : rows;
  const int64_t n_chunks = (rows * cols + kMomentumChunk - 1) / kMomentumChunk;
  // scratch layout: scalars | member table [| partial sums | fragment
  // iterate, for the direct iteration beyond kGramSpaceMaxSteps only]
  const bool gram_space = cfg.gram_space && ns_steps <= kGramSpaceMaxSteps;
  const size_t off_mem = align256(sizeof(StepScalars));
  const size_t off_part = align256(off_mem + (size_t)batch * sizeof(MemberPtrs));
  const size_t off_ws = align256(off_part + (size_t)batch * n_chunks * sizeof(float));
  const size_t total = gram_space ? off_part : off_ws + (size_t)batch * cfg.ws_bytes;
  if (total > kStaticScratchBytes) {
    char msg[200];
    std::snprintf(msg, sizeof msg,
                  "needs %zu bytes of scratch for batch %d of [%lld, %lld] at %d steps; the "
                  "static array holds %zu",
                  total, batch, (long long)rows, (long long)cols, ns_steps, kStaticScratchBytes);
    return static_fail(MUON_ERR_INVALID_ARG, msg);
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return static_fail(MUON_ERR_CUDA, "cudaGetDevice failed");
  {
    // the launches and the array address belong to the current device, so
    // the stream must be one of that device's (the default streams always are)
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int sdev = dev;
    if (cs != nullptr && cs != cudaStreamLegacy && cs != cudaStreamPerThread &&
        cudaStreamGetDevice(cs, &sdev) != cudaSuccess)
      return static_fail(MUON_ERR_INVALID_ARG, "stream is not a valid CUDA stream");
    if (sdev != dev)
      return static_fail(MUON_ERR_INVALID_ARG,
                         "stream belongs to another device than the current one");
  }
  KArgs k{};
  k.B = batch;
  k.rows = (int32_t)rows;
  k.cols = (int32_t)cols;
  k.m = (int32_t)m;
  k.n = (int32_t)n;
  k.T = rows > cols;
  k.mode_f32 = 0;
  k.ns_type = NS_F16;
  k.n_chunks = (int32_t)n_chunks;
  k.eps = eps;
  k.scale = scale_mode == MUON_SCALE_SQRT_ASPECT
                ? (float)std::sqrt(std::max(1.0, (double)rows / (double)cols))
                : (scale_mode == MUON_SCALE_RMS_0_2 ? (float)(0.2 * std::sqrt((double)n)) : 1.f);
  k.alpha = (float)std::ldexp(1.0, (int)std::round(0.5 * std::log2((double)n)));
  k.l2_keep_m = 1;
  {
    // once per device, with that device current: the array's device address;
    // once per device and kernel variant: the kernel attributes (host work
    // only; do the first call before any stream capture)
    const int mt = cfg.mtiles, half = (int)(m - 16 * (mt - 1) <= 8);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
      if (e != cudaSuccess || !ptr)
        return static_fail(MUON_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      g_scratch_addr[dev] = static_cast<unsigned char*>(ptr);
    }
    if (!g_prepared[dev][mt][half]) {
      if (prepare_skinny(k, cfg) != cudaSuccess)
        return static_fail(MUON_ERR_CUDA, "setting the skinny kernel's attributes failed");
      g_prepared[dev][mt][half] = true;
    }
  }
  unsigned char* base = g_scratch_addr[dev];
  StepScalars* sc = reinterpret_cast<StepScalars*>(base);
  MemberPtrs* mem = reinterpret_cast<MemberPtrs*>(base + off_mem);
  k.sc = sc;
  k.mem = mem;
  k.part = gram_space ? nullptr : reinterpret_cast<float*>(base + off_part);
  k.y0 = gram_space ? nullptr : base + off_ws;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepScalars hs{};
  hs.beta = beta; hs.lr = lr; hs.wd = wd;
  hs.ns_steps = ns_steps;
  hs.n_coef = 1;
  hs.coef[0][0] = a; hs.coef[0][1] = b; hs.coef[0][2] = c;
  k_static_setup<<<1, 32, 0, s>>>(hs, params, grads, momenta, batch, rows * cols, k.T, k.scale, sc, mem);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_skinny(k, cfg, ns_steps, s);
  if (e != cudaSuccess) return static_fail(MUON_ERR_CUDA, cudaGetErrorString(e));
  return MUON_OK;
}
