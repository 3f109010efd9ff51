// Internal host/device structures shared by the library's translation units.
// Nothing here is part of the public C ABI (include/muon.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace muon {

// Rows of a per-step coefficient schedule held in the step scalars.
constexpr int32_t kMaxScheduleRows = 64;

// Per-step scalars, rewritten in device memory before every step so that one
// captured CUDA graph serves every step with the same ns_steps.  Newton-Schulz
// step s takes coef[min(s, n_coef - 1)] as (a, b, c).
struct StepScalars {
  float beta, lr, wd;
  int32_t ns_steps;
  int32_t n_coef;
  int32_t pad_[3];
  float coef[kMaxScheduleRows][3];
};

// Per-member device pointers, rewritten before every step (the caller may
// pass different buffers each step).  P and G are bf16 or fp32 by mode.  A
// member's parameter is [m, n] (T = 0) or [n, m] (T = 1) for its group's
// (m, n); scale is its s(rows, cols).
struct MemberPtrs {
  void* P;
  const void* G;
  float* M;
  int32_t T;
  float scale;
};

enum Path : int32_t { PATH_AUTO = 0, PATH_SKINNY = 1, PATH_TENSOR = 2, PATH_SIMT = 3, PATH_RESIDENT = 4 };
// Element type of the Newton-Schulz iterate / Gram / polynomial buffers.
enum NsType : int32_t { NS_F32 = 0, NS_F16 = 1, NS_BF16 = 2 };

// Elements of one member handled by one CTA of the momentum pass; fixed so the
// reduction tree (and thus the norm, bit for bit) depends only on the shape.
constexpr int64_t kMomentumChunk = 16384;

// Arguments of the per-group kernels, passed by value (baked into the graph).
struct KArgs {
  const StepScalars* sc;   // device
  const MemberPtrs* mem;   // device, already offset to the group's first member
  int32_t B;               // members in the group
  int32_t rows, cols;      // parameter dims of the group's first member (kernels use m, n and MemberPtrs::T)
  int32_t m, n;            // min / max of (rows, cols)
  int32_t T;               // rows > cols for the group's first member
  int32_t mode_f32;        // 1: P, G fp32 ; 0: P, G bf16
  int32_t ns_type;         // NsType of y0/y1/A/Q
  int64_t n_pitch;         // row pitch (elements) of the m x n iterate
  int64_t m_pitch;         // row pitch (elements) of the m x m Gram / polynomial
  int32_t n_chunks;        // momentum chunks per member
  float eps;               // added to ||M'||_F
  float scale;             // s(rows, cols)
  float alpha;             // power-of-two factor of the stored iterate (Y = alpha X)
  void* y0;                // [B][m][n_pitch] (skinny path: fragment workspace)
  void* y1;                // [B][m][n_pitch]
  void* A;                 // [B][m][m_pitch]
  void* Q;                 // [B][m][m_pitch]
  float* part;             // [B][n_chunks] partial sums of squares
  float* invn;             // [B] alpha / (||M'||_F + eps)
  float* dbg;              // nullable: [B][rows][cols] fp32 copy of O
  int* err;                // device error word
  int32_t l2_keep_m;       // momentum kernel stores M' evict-last (it is read back soon, twice)
  int32_t nesterov;        // orthogonalise U = G + beta M' instead of M'
  float* u;                // nullable: [B][rows][cols] U written by the momentum kernel (direct kernel's input)
};

// Skinny path configuration of a group (a function of (rows, cols) only).
struct SkinnyCfg {
  int32_t cluster;   // CTAs per matrix
  int32_t width;     // columns of the wide iterate owned by one CTA
  int32_t threads;   // threads per CTA
  int32_t mtiles;    // ceil(m / 16)
  int32_t smem;      // unused (shared memory is fixed per instantiation)
  int32_t blk;       // bytes of one 16-column block in the fragment workspace
  int64_t ws_bytes;  // fragment workspace bytes per member (direct kernel)
  int32_t gram_space;  // the Gram-space kernel serves ns_steps <= kGramSpaceMaxSteps
  int32_t auto_shards; // the plan left column_shards to the library (0): for m <= 32 the
                       // Gram-space kernel may then run 4-CTA clusters of 8 warps for
                       // small batches (the same reduction tree, so the same bits)
};

// Step counts the Gram-space kernel takes: along an exact null direction of
// X_0 its m x m product Pi_k grows like a^k (3.4445^64 < 2^115 stays in fp32).
constexpr int32_t kGramSpaceMaxSteps = 64;

// Newton-Schulz steps allowed on bf16 operands where the iterate itself is
// rounded on every step (tensor and SIMT paths, and the skinny direct
// iteration): with those roundings emulated against the fp64 oracle on
// Gaussian momenta, the relative error of O is 1.1e-2 to 1.2e-2 at 5 steps,
// 1.5e-2 to 1.7e-2 at 6 and 2.1e-2 to 2.4e-2 at 8, against the bf16-mode
// tolerance of 2e-2.
constexpr int32_t kBf16OperandMaxSteps = 5;

// Sets the thread-local message muon_last_error() returns.
void set_last_error(const char* msg);

// ---- launchers (each returns the launch's cudaError_t) ----
cudaError_t launch_momentum_partial(const KArgs& a, cudaStream_t s);
cudaError_t launch_norm_finalize(const KArgs& a, cudaStream_t s);
cudaError_t launch_normalize_cast(const KArgs& a, void* dst, cudaStream_t s);
cudaError_t launch_write(const KArgs& a, const void* src, cudaStream_t s);

// SIMT batched products (fp32 FMA) on the workspace type of `a`:
//   gram:   A = (Y Y^T) / alpha^2
//   poly:   Q = a I + b A + c A A, (a, b, c) of Newton-Schulz step `step`
//   update: Ydst = Q Ysrc
cudaError_t launch_simt_gram(const KArgs& a, const void* y, cudaStream_t s);
cudaError_t launch_simt_poly(const KArgs& a, int step, cudaStream_t s);
cudaError_t launch_simt_update(const KArgs& a, const void* ysrc, void* ydst, cudaStream_t s);

// Skinny path, the whole step of a group: for k <= kGramSpaceMaxSteps one
// kernel (momentum, then Newton-Schulz in Gram space,
// then the write, one cluster per member, no workspace); otherwise the
// momentum kernel, then the direct iteration (iterate in a fragment-ordered
// workspace a.y0).
// shards: CTAs (contiguous column shards) per member, 1, 2, 4 or 8; 0 = 2.
bool skinny_config(int32_t rows, int32_t cols, int32_t max_m, SkinnyCfg* cfg, int32_t shards = 0);
cudaError_t prepare_skinny(const KArgs& a, const SkinnyCfg& cfg);  // function attributes
cudaError_t launch_skinny(const KArgs& a, const SkinnyCfg& cfg, int32_t ns_steps, cudaStream_t s);
cudaError_t gs_dispatch(const KArgs& a, const SkinnyCfg& cfg, cudaStream_t s, bool prepare);
int gs_max_active_clusters(int ns_type, int m, int cl);
// Clusters of the skinny kernel for min dim m that fit on the device at once
// (after prepare_skinny for that m).
int skinny_max_active_clusters(int ns_type, int m, int cl);

// Test hook: one bounded mbarrier wait, completed by a second thread
// (arrive != 0) or by nothing; on giving up it sets bit 16 of *err.
cudaError_t launch_wait_probe(int* err, long long limit, int arrive, cudaStream_t s);

// TENSOR path: tcgen05 GEMMs fed by TMA.  Tensor maps are encoded once per
// group at plan creation (they hold the workspace addresses).
struct TcMaps {
  CUtensorMap y_k128[2];  // iterate y0 / y1, K-major boxes of 128 rows
  CUtensorMap y_ksq[2];   // iterate, K-major boxes of bn_sq rows (Gram B operand)
  CUtensorMap y_mn[2];    // iterate, 64 x 64 boxes read N-contiguous (update B operand)
  CUtensorMap a_k128, a_ksq, q_k128;
  int bn_sq, bn_up;
};
cudaError_t tc_make_maps(const KArgs& a, TcMaps* t);
cudaError_t prepare_tc(int ns_type);  // function attributes
cudaError_t launch_tc_gram(const KArgs& a, const TcMaps& t, int src, cudaStream_t s);
cudaError_t launch_tc_poly(const KArgs& a, const TcMaps& t, int step, cudaStream_t s);  // step: schedule row
// Y[1 - src] = Q Y[src]
cudaError_t launch_tc_update(const KArgs& a, const TcMaps& t, int src, cudaStream_t s);
// The (tile row, tile column) of each tile one batch item of a GEMM computes
// with bm x bn tiles (bm 128: one CTA per tile, bn 128 or 256; bm 256: the
// CTA-pair form, bn 256), in launch order: op 0 / 1 (Gram, polynomial) the
// symmetric walk over the m x m output, op 2 (update) the grouped raster over
// the m x n output.  Returns the tile count (entries past cap are not
// written), -1 on bad arguments.
int32_t tc_tile_walk(int32_t op, int64_t m, int64_t n, int32_t bm, int32_t bn, int32_t* tm,
                     int32_t* tn, int32_t cap);
// True when a group of min dim m runs its products in the CTA-pair form.
bool tc_pair_form(int64_t m);

}  // namespace muon
