/*
 * muon.h -- C ABI of the shape-fused Muon update for one GB300 (sm_103a).
 *
 * What the library computes, per parameter matrix (or per batch slice of a 3-D
 * [E, rows, cols] parameter), all matrices of a step being independent:
 *
 *   M' = beta * M + G                                   (momentum)
 *   X0 = M' / (||M'||_F + eps)                          (Frobenius normalisation)
 *   if rows > cols: X0 = X0^T                           (iterate on the wide side)
 *   k times: A = X X^T ; X = a X + (b A + c A A) X      (quintic Newton-Schulz)
 *   O = X (transposed back if rows > cols)
 *   P' = P * (1 - lr * wd) - lr * s(rows, cols) * O     (scaled, decayed write)
 *
 * Sources: «关于分布式Muon的想法整合及讨论» §1 (momentum, then approximate
 * orthogonalisation of M used as the update direction), §2 (normalise M, Gram
 * matrix, a series of matrix products), §6 (sum-of-squares normaliser, Gram
 * matrix recomputed every round); «MindSpore HyperParallel X 盘古,Muon优化器实现
 * 6倍性能跃升», 三大性能挑战 (5-10 iterations), Muon亲和的专家切分 (Fig. 4: the
 * E slices of an expert tensor are independent), 矩阵融合优化 (Fig. 6-7:
 * parameters sharing their trailing two dims run as one [B, M, N] batch; the
 * unfused version is dominated by host dispatch and small alloc/free, which is
 * why all allocation happens in muon_plan_create and a step is one CUDA-graph
 * replay); HyperParallel-FSDP abstract (arXiv 2609.21594), contribution (3):
 * shape-fused Newton-Schulz iterations.  The exact scalar forms of momentum,
 * eps, weight decay and the scale s are readings: the pages give none.
 *
 * Conventions shared by every entry point:
 *  - Device memory is row-major and contiguous.  One pointer per PARAMETER,
 *    in the order given to muon_plan_create; a 3-D parameter is one pointer to
 *    its [E, rows, cols] block.  The caller owns params, grads and momenta;
 *    the plan owns its workspace, pointer tables and CUDA graphs.
 *  - params and momenta are updated in place; grads are read only; the three
 *    arrays of one parameter must not overlap each other or another parameter.
 *  - Errors are returned as muon_status_t; no entry point aborts or throws.
 *    Argument checks run before any launch.  muon_last_error() returns a
 *    thread-local message for the last failing call of this thread.
 *  - A plan is not thread-safe; distinct plans are independent.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All device work is stream-ordered on it.
 */
#ifndef MUON_GB300_H
#define MUON_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MUON_API __attribute__((visibility("default")))
#else
#define MUON_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct muon_plan_s* muon_plan_t;

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = 1,  /* bad shape, null pointer, bad option        */
  MUON_ERR_UNSUPPORTED = 2,  /* valid request the library cannot run      */
  MUON_ERR_OOM = 3,          /* device or pinned-host allocation failed    */
  MUON_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed          */
  MUON_ERR_TIMEOUT = 5       /* a kernel's bounded wait ran out (see check) */
} muon_status_t;

/* Storage/compute mode of a plan.
 * BF16: params and grads bf16, momenta fp32, Newton-Schulz on 16-bit tensor
 *       core operands with fp32 accumulation.
 * FP32: params, grads and momenta fp32; every product in fp32 FMA (no TF32). */
typedef enum { MUON_MODE_BF16 = 0, MUON_MODE_FP32 = 1 } muon_mode_t;

/* Operand type of the Newton-Schulz products in MUON_MODE_BF16.  FP16 (the
 * default) keeps 3 more mantissa bits at the same tensor-core rate; BF16
 * rounds X, A and the polynomial matrix to bf16, an error that grows with k.
 * With the roundings emulated against the fp64 oracle on Gaussian momenta,
 * the relative Frobenius error of O is about 2e-3 for FP16 up to k = 10 and
 * for BF16 on the skinny path up to k = 64 (the data is rounded once); BF16
 * where the iterate is rounded on every step (tensor and SIMT paths, skinny
 * path beyond 64 steps) is about 1.2e-2 at k = 5, 1.7e-2 at k = 6 and 2.5e-2
 * to 3e-2 at k = 10.  So a step with BF16 operands and more than 5
 * Newton-Schulz steps on such a group fails with MUON_ERR_UNSUPPORTED. */
typedef enum { MUON_NS_FP16 = 0, MUON_NS_BF16 = 1 } muon_ns_dtype_t;

/* Shape-dependent scale s(rows, cols) of the update (a reading; the pages
 * only say "scaled"): sqrt(max(1, rows/cols)), 0.2*sqrt(max(rows, cols)), 1. */
typedef enum {
  MUON_SCALE_SQRT_ASPECT = 0,
  MUON_SCALE_RMS_0_2 = 1,
  MUON_SCALE_NONE = 2
} muon_scale_t;

/* Kernel path of a shape group.  AUTO picks SKINNY when min(rows, cols) <= 64
 * (the skinny_threshold option): up to 64 Newton-Schulz steps that is one
 * kernel per group, a cluster of column_shards CTAs per matrix that streams
 * the data twice (momentum with the Gram matrix and the norm, then the
 * output) and iterates in m x m Gram space on chip; beyond 64 steps, a
 * momentum kernel and the direct iteration on a fragment-ordered, L2-resident
 * workspace.  TENSOR otherwise (tcgen05 GEMMs on TMEM accumulators, fed by
 * TMA).  RESIDENT, only when asked for, takes groups with min(rows, cols)
 * <= 128 and max(rows, cols) <= 4096: one kernel per group, a cluster of up
 * to 8 CTAs per matrix whose shared memory holds the iterate for all k steps
 * (the TENSOR path's arithmetic on tcgen05, partial Gram matrices added
 * through distributed shared memory), so HBM sees only G, M, P read and M',
 * P' written; it is bound by the latency of its per-step cluster exchange.
 * FP32 mode always uses SIMT (fp32 FMA). */
typedef enum {
  MUON_PATH_AUTO = 0,
  MUON_PATH_SKINNY = 1,
  MUON_PATH_TENSOR = 2,
  MUON_PATH_SIMT = 3,
  MUON_PATH_RESIDENT = 4
} muon_path_t;

/* ndim 2: dims = {rows, cols}; ndim 3: dims = {E, rows, cols}. */
typedef struct {
  int32_t ndim;
  int32_t reserved_;
  int64_t dims[3];
} muon_shape_t;

#define MUON_FLAG_KEEP_UPDATE  1u  /* keep O = X_k per member (fp32) for muon_debug_copy_update */
#define MUON_FLAG_NO_GRAPH     2u  /* launch kernels one by one instead of a CUDA-graph replay  */
#define MUON_FLAG_HOST_STAGING 4u  /* allocate device mirrors so muon_step_host can run         */
#define MUON_FLAG_GROUP_TIMING 8u  /* record CUDA events around each group's kernels            */
/* Nesterov look-ahead: orthogonalise U = G + beta M' instead of M' (M' is
 * still the stored momentum).  The pages name no Nesterov form; this is the
 * one that goes with the undamped momentum M' = beta M + G.  Skinny groups
 * then also read G in the output pass, and for ns_steps > 64 (direct
 * iteration) keep U in the workspace (4 bytes per element). */
#define MUON_FLAG_NESTEROV    16u
/* Orientation-canonical buckets: [r, c] and [c, r] parameters share one group
 * keyed by (min, max), so the batch is larger («MindSpore HyperParallel X
 * 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化: fusing more matrices per
 * launch).  Each member keeps its own orientation: it is iterated in the wide
 * form and written back transposed if its rows > cols, with its own scale
 * s(rows, cols), so its result is the same as in an unmerged plan. */
#define MUON_FLAG_MERGE_TRANSPOSED 32u

/* Rows a per-step coefficient schedule may have (muon_step_schedule). */
#define MUON_MAX_SCHEDULE_ROWS 64

typedef struct {
  int32_t mode;              /* muon_mode_t, default BF16                          */
  int32_t scale;             /* muon_scale_t, default SQRT_ASPECT                  */
  float eps;                 /* added to ||M'||_F, default 1e-7                    */
  int32_t skinny_threshold;  /* largest min(rows,cols) for SKINNY; 0 = default 64  */
  int32_t ns_dtype;          /* muon_ns_dtype_t, default FP16                      */
  uint32_t flags;            /* MUON_FLAG_*                                        */
  int32_t path_override;     /* muon_path_t for every group; AUTO = choose         */
  int32_t max_streams;       /* groups run on up to this many graph branches; 0=4  */
  int32_t column_shards;     /* skinny path: CTAs per member (1, 2, 4 or 8), each   */
                             /* owning one contiguous column shard; their partial  */
                             /* Grams and sums of squares are all-reduced through  */
                             /* distributed shared memory («关于分布式Muon的想法整合 */
                             /* 及讨论» §6).  0 = chosen by the library: 2, or 4 for*/
                             /* batches too small to fill the GPU when m <= 32,    */
                             /* with the same bits either way (one fixed reduction */
                             /* tree).  An explicit t fixes the form; the bits then*/
                             /* depend on t, never on the batch                    */
  int32_t reserved[7];       /* must be zero                                       */
} muon_plan_options;

typedef struct {
  int64_t rows, cols;        /* the trailing dims every member shares (with      */
                             /* MUON_FLAG_MERGE_TRANSPOSED: the first member's)   */
  int64_t batch;             /* number of member matrices                         */
  int64_t first_member;      /* index of the group's first member (see below)     */
  int32_t transposed;        /* 1: every member has rows > cols (iterated on its  */
                             /* transpose); 0: none; 2: both orientations (merge) */
  int32_t path;              /* muon_path_t chosen for the group                  */
  int64_t workspace_bytes;   /* device bytes of the group's scratch               */
} muon_group_info_t;

/* Fills *opts with the defaults above.  Never fails for a non-null pointer. */
MUON_API muon_status_t muon_default_options(muon_plan_options* opts);

/* Host-only planning (no device is touched): buckets the parameters by exact
 * trailing shape (rows, cols) in first-seen order, expanding a 3-D parameter
 * into its E slices in E order («MindSpore HyperParallel X 盘古,Muon优化器实现
 * 6倍性能跃升», 矩阵融合优化 Fig. 6 and Muon亲和的专家切分 Fig. 4).
 * groups: caller array of group_cap entries (may be NULL when group_cap = 0);
 * *n_groups receives the group count even when it exceeds group_cap.
 * member_param / member_expert: caller arrays of member_cap entries (or NULL),
 * filled in group order; *n_members receives the member count.
 * *workspace_bytes (nullable) receives the device bytes muon_plan_create will
 * allocate.  INVALID_ARG for ndim not in {2,3}, a dim < 1, n_params < 1,
 * more than 2^31-1 members, or a bad option. */
MUON_API muon_status_t muon_plan_describe(const muon_shape_t* shapes, int32_t n_params,
                                          const muon_plan_options* opts,
                                          muon_group_info_t* groups, int32_t group_cap,
                                          int32_t* n_groups,
                                          int32_t* member_param, int32_t* member_expert,
                                          int64_t member_cap, int64_t* n_members,
                                          size_t* workspace_bytes);

/* Host-only ownership planner for data-parallel replicas: assigns every
 * member matrix (numbered as muon_plan_describe numbers them) to one of
 * n_ranks ranks so that the estimated Newton-Schulz cost is balanced.
 * Matrices are the atomic units, a 3-D parameter's experts are assigned one
 * by one, and the assignment is greedy: members in decreasing cost (then
 * increasing index), each to the rank with the least cost so far (then the
 * lowest rank) («MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升»,
 * HSDP分组去冗余: replicas split the parameters with a greedy algorithm for
 * balance; «关于分布式Muon的想法整合及讨论» §3: whole matrices per owner,
 * balanced by compute cost, not size).  A member's cost is its estimated
 * seconds on this library's path for its group (memory traffic over HBM
 * bandwidth, Newton-Schulz FLOPs over the tensor rate; rates measured on a
 * GB300).  The result is deterministic: a function of the shapes, options,
 * ns_steps and n_ranks only.  owner: member_cap >= member count entries, receives ranks in
 * [0, n_ranks); member_cost (nullable, member_cap entries) and rank_cost
 * (nullable, n_ranks entries) receive seconds.  No communication and no
 * device.  Errors: INVALID_ARG (as muon_plan_describe; n_ranks not in
 * [1, 2^20]; ns_steps not in [0, 1000]; owner NULL or too short). */
MUON_API muon_status_t muon_plan_assign(const muon_shape_t* shapes, int32_t n_params,
                                        const muon_plan_options* opts, int32_t ns_steps,
                                        int32_t n_ranks, int32_t* owner, int64_t member_cap,
                                        double* member_cost, double* rank_cost);

/* Builds a plan on CUDA device `device`: the bucketing above, per-group path
 * and tile choices (functions of (rows, cols) only, never of the batch size,
 * so a matrix gets bit-identical results in any batch), and every device
 * allocation the steps will need (workspace, pointer tables, pinned staging).
 * opts may be NULL (defaults).  *out receives the plan; release it with
 * muon_plan_destroy.  Errors: INVALID_ARG (as muon_plan_describe, or out
 * NULL), OOM, CUDA, UNSUPPORTED (device is not sm_103). */
MUON_API muon_status_t muon_plan_create(const muon_shape_t* shapes, int32_t n_params,
                                        const muon_plan_options* opts, int device,
                                        muon_plan_t* out);

/* One Muon step over every parameter of the plan (the update at the top of
 * this file).  params[i]: bf16 (BF16 mode) or fp32 device pointer to
 * parameter i, updated in place; grads[i]: same type, read only; momenta[i]:
 * fp32, updated in place to M'.  beta, lr, wd: momentum, learning rate,
 * decoupled weight decay.  ns_steps >= 0 (0 = no iteration: O = X0);
 * (a, b, c): quintic coefficients.  Each buffer holds its parameter
 * contiguously, row-major with experts outermost ([E, rows, cols]); buffers
 * must not overlap.  Any alignment of the element type is accepted: a member
 * whose buffers start on 16 bytes, with rows <= cols and cols % 8 == 0,
 * takes the vector paths, and other members take element-wise accesses (the
 * kernels test this per member, so no access leaves the buffers).
 * Never allocates.  The first call with a
 * given ns_steps captures and instantiates a CUDA graph (host work only);
 * later calls copy the scalars and pointers into the plan's device table
 * (one async H2D copy from pinned memory, skipped when they equal those of
 * the previous call) and replay the graph on `stream`.  Successive calls on
 * different streams must be ordered by the caller (the table is shared).
 * Errors (nothing is launched): INVALID_ARG for a null plan/array/pointer,
 * ns_steps < 0 or > 1000, or non-finite scalars; UNSUPPORTED for ns_steps > 5
 * on a group that iterates on BF16 operands (see muon_ns_dtype_t); CUDA on a
 * launch failure. */
MUON_API muon_status_t muon_step(muon_plan_t plan, void* const* params,
                                 const void* const* grads, float* const* momenta,
                                 float beta, float lr, float wd, int32_t ns_steps,
                                 float a, float b, float c, void* stream);

/* muon_step with per-step coefficients («MindSpore HyperParallel X 盘古,Muon
 * 优化器实现6倍性能跃升», 三大性能挑战: 5-10 iterations; the pages give no
 * per-step values): Newton-Schulz step s (0-based) takes row
 * min(s, n_rows - 1) of coeffs, a HOST array of n_rows x 3 floats
 * (a_s, b_s, c_s), row-major, read before the call returns; the last row
 * repeats past the end.  muon_step(..., a, b, c, ...) is the one-row case.
 * The graph captured for ns_steps serves every schedule (the rows travel in
 * the step's scalar table).  Errors: as muon_step, plus INVALID_ARG for
 * coeffs NULL, n_rows not in [1, MUON_MAX_SCHEDULE_ROWS], or a non-finite
 * coefficient. */
MUON_API muon_status_t muon_step_schedule(muon_plan_t plan, void* const* params,
                                          const void* const* grads, float* const* momenta,
                                          float beta, float lr, float wd, int32_t ns_steps,
                                          const float* coeffs, int32_t n_rows, void* stream);

/* The same step on HOST buffers (pinned or pageable): copies each parameter,
 * gradient and momentum to the plan's device mirrors, runs muon_step on them,
 * copies params and momenta back, and returns after `stream` has finished
 * (results are in the host buffers on return).  Needs MUON_FLAG_HOST_STAGING
 * at plan creation (UNSUPPORTED otherwise).  Contiguous host ranges are
 * moved with one copy each.  When every group takes the skinny path the step
 * runs in chunks of parameters, and otherwise in slices of whole members of
 * a group (about 1/16 of the plan's elements each): each unit is copied in,
 * updated and copied out on its own stream order so that copies in both
 * directions and the kernels overlap; every member gets the same kernels as
 * in muon_step, so the results are the same bits.  One (a, b, c) triple per
 * call: a per-step schedule needs device buffers (muon_step_schedule). */
MUON_API muon_status_t muon_step_host(muon_plan_t plan, void* const* host_params,
                                      const void* const* host_grads,
                                      float* const* host_momenta, float beta, float lr,
                                      float wd, int32_t ns_steps, float a, float b,
                                      float c, void* stream);

/* Frees everything the plan owns (synchronises its device first).  NULL ok. */
MUON_API muon_status_t muon_plan_destroy(muon_plan_t plan);

/* Group / member introspection of a created plan (host only). */
MUON_API int32_t muon_plan_num_groups(muon_plan_t plan);
MUON_API muon_status_t muon_plan_group_info(muon_plan_t plan, int32_t group,
                                            muon_group_info_t* info);
MUON_API size_t muon_plan_workspace_bytes(muon_plan_t plan);

/* Test hook: copies O = X_k of (param_index, expert) as fp32 [rows, cols]
 * into dst_host (rows*cols floats) after synchronising the device.  Needs
 * MUON_FLAG_KEEP_UPDATE (UNSUPPORTED otherwise); INVALID_ARG for a bad index. */
MUON_API muon_status_t muon_debug_copy_update(muon_plan_t plan, int32_t param_index,
                                              int64_t expert, float* dst_host);

/* Device time of group `group`'s kernels in the most recent step, from CUDA
 * events recorded inside the step (graph event-record nodes).  Waits for that
 * step to finish.  Needs MUON_FLAG_GROUP_TIMING (UNSUPPORTED otherwise). */
MUON_API muon_status_t muon_plan_group_elapsed_ms(muon_plan_t plan, int32_t group, float* ms);

/* Synchronises the plan's device and reads its error word: MUON_OK, or
 * MUON_ERR_TIMEOUT if any kernel of an earlier step gave up a bounded wait
 * (the word is then cleared). */
MUON_API muon_status_t muon_plan_check_error(muon_plan_t plan);

/* The skinny-path step (min(rows, cols) <= 64) for callers that cannot
 * allocate device memory -- for example code inside a framework whose caching
 * allocator forbids outside cudaMalloc calls, latency-critical loops that must
 * not enter the CUDA allocator, or embedded deployments that fix every
 * device buffer at start-up.  The pages have no counterpart to this call; it
 * exists for those callers.  It applies the update at the top of this file to
 * the `batch` matrices of one [batch, rows, cols] parameter in BF16 mode with
 * fp16 Newton-Schulz operands, and gives bit for bit the results of muon_step
 * on a plan made of that one parameter with default options (same kernels,
 * same arguments, same reduction orders).  params (bf16), grads (bf16) and
 * momenta (fp32) are the caller's device buffers, updated in place as in
 * muon_step.  All scratch lives in one static device array of 8 MiB inside
 * the library: every GPU that loads the library keeps it until the process
 * exits, and it is shared by every call (calls whose work overlaps on a GPU
 * race -- issue them on one stream).  Up to 64 Newton-Schulz steps a call
 * needs 256 + 32 * batch bytes of it (step scalars and member pointers; e.g.
 * any batch, up to 65535, of [24, 10240]); beyond 64 steps the direct
 * iteration also keeps its iterate there (about 2 * rows * cols bytes per
 * member, so about 8 members of [24, 10240]).  A request needing more fails
 * with MUON_ERR_INVALID_ARG and a message giving both sizes.  It calls no
 * allocator.  The current device must be the device of `stream` (checked:
 * INVALID_ARG otherwise).  The first call on each device looks up the array's
 * device address, and the first call for each kernel variant (number of
 * 16-row tiles of min(rows, cols)) sets that kernel's attributes; both are
 * host work: make those calls before any stream capture.  Errors:
 * INVALID_ARG (NULL pointer, batch not in [1, 65535], bad size, scalar or
 * scale_mode, too much scratch, stream of another device), UNSUPPORTED (min(rows, cols) > 64),
 * CUDA. */
MUON_API muon_status_t muon_step_skinny_static(void* params, const void* grads, float* momenta,
                                               int32_t batch, int64_t rows, int64_t cols,
                                               float beta, float lr, float wd, int32_t ns_steps,
                                               float a, float b, float c, float eps,
                                               int32_t scale_mode, void* stream);

MUON_API const char* muon_status_string(muon_status_t status);
MUON_API const char* muon_last_error(void);
/* Library version, e.g. "0.1.0". */
MUON_API const char* muon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H */
