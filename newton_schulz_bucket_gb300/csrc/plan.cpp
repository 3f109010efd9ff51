// Host planner and executor behind the C ABI (include/muon.h).
//
// Planning buckets parameters by exact trailing shape («MindSpore HyperParallel
// X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化, Fig. 6: parameters whose
// trailing two dims agree are stacked into one [B, M, N] batch; Muon亲和的专家
// 切分, Fig. 4: the E slices of an expert tensor are independent members).
// The same article traces the unfused iteration's cost to host dispatch,
// small alloc/free and stream synchronisation, so every allocation happens at
// plan creation and a step is one async copy of scalars + pointers followed by
// one CUDA-graph replay.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <new>
#include <queue>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/muon.h"
#include "internal.h"
#include "resident.h"

namespace muon {
namespace {

thread_local std::string g_last_error;

muon_status_t fail(muon_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(e_ == cudaErrorMemoryAllocation ? MUON_ERR_OOM : MUON_ERR_CUDA,       \
                  "%s failed: %s", #expr, cudaGetErrorString(e_));                      \
  } while (0)

constexpr int kRingSlots = 4;
constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct GroupPlan {
  int64_t rows = 0, cols = 0, batch = 0, first_member = 0;
  int32_t transposed = 0, path = PATH_AUTO;
  int64_t m = 0, n = 0, n_pitch = 0, m_pitch = 0, n_chunks = 0;
  int32_t ns_type = NS_F16;
  float alpha = 1.f, scale = 1.f;
  SkinnyCfg sk{};
  ResidentCfg rc{};     // RESIDENT path: cluster and columns per CTA
  TcMaps tc{};          // TENSOR path: TMA descriptors of the workspace
  size_t off_y0 = 0, off_y1 = 0, off_a = 0, off_q = 0, off_part = 0, off_invn = 0, off_dbg = 0;
  size_t off_u = 0;  // skinny groups under Nesterov: U for the direct kernel (0: none)
  size_t ws_bytes = 0;  // this group's scratch (from the group base)
  size_t base = 0;      // offset of the group's scratch in the plan workspace
  double cost = 0;      // flops-ish estimate, for stream assignment
};

struct PlanDesc {
  muon_plan_options opt{};
  std::vector<GroupPlan> groups;
  std::vector<int32_t> member_param, member_expert;
  std::vector<int64_t> param_E, param_rows, param_cols;
  std::vector<float> param_scale;  // s(rows, cols) of each parameter
  size_t ws_bytes = 0;      // total device scratch incl. tables
  size_t off_scalars = 0;   // StepScalars + MemberPtrs table
  size_t off_err = 0;
  size_t pb_bytes = 0;      // bytes of the per-step parameter block
};

size_t ns_esize(int32_t t) { return t == NS_F32 ? 4 : 2; }

muon_status_t check_options(const muon_plan_options& o) {
  if (o.mode != MUON_MODE_BF16 && o.mode != MUON_MODE_FP32)
    return fail(MUON_ERR_INVALID_ARG, "mode %d is not a muon_mode_t", o.mode);
  if (o.scale < MUON_SCALE_SQRT_ASPECT || o.scale > MUON_SCALE_NONE)
    return fail(MUON_ERR_INVALID_ARG, "scale %d is not a muon_scale_t", o.scale);
  if (!(o.eps >= 0.f) || !std::isfinite(o.eps))
    return fail(MUON_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (o.ns_dtype != MUON_NS_FP16 && o.ns_dtype != MUON_NS_BF16)
    return fail(MUON_ERR_INVALID_ARG, "ns_dtype %d is not a muon_ns_dtype_t", o.ns_dtype);
  if (o.path_override < MUON_PATH_AUTO || o.path_override > MUON_PATH_RESIDENT)
    return fail(MUON_ERR_INVALID_ARG, "path_override %d is not a muon_path_t", o.path_override);
  if (o.mode == MUON_MODE_FP32 && o.path_override != MUON_PATH_AUTO &&
      o.path_override != MUON_PATH_SIMT)
    return fail(MUON_ERR_INVALID_ARG, "FP32 mode runs only the SIMT (fp32 FMA) path");
  if (o.max_streams < 0 || o.max_streams > 16)
    return fail(MUON_ERR_INVALID_ARG, "max_streams must be in [0, 16]");
  if (o.skinny_threshold < -1 || o.skinny_threshold > 64)
    return fail(MUON_ERR_INVALID_ARG, "skinny_threshold must be in [-1, 64]");
  if (o.flags & ~(MUON_FLAG_KEEP_UPDATE | MUON_FLAG_NO_GRAPH | MUON_FLAG_HOST_STAGING |
                  MUON_FLAG_GROUP_TIMING | MUON_FLAG_NESTEROV | MUON_FLAG_MERGE_TRANSPOSED))
    return fail(MUON_ERR_INVALID_ARG, "unknown flag bits 0x%x", o.flags);
  if (o.column_shards != 0 && o.column_shards != 1 && o.column_shards != 2 && o.column_shards != 4 &&
      o.column_shards != 8)
    return fail(MUON_ERR_INVALID_ARG, "column_shards must be 0, 1, 2, 4 or 8");
  for (int i = 0; i < 7; ++i)
    if (o.reserved[i] != 0) return fail(MUON_ERR_INVALID_ARG, "reserved option fields must be 0");
  return MUON_OK;
}

float scale_of(int32_t mode, int64_t rows, int64_t cols) {
  switch (mode) {
    case MUON_SCALE_SQRT_ASPECT:
      return (float)std::sqrt(std::max(1.0, (double)rows / (double)cols));
    case MUON_SCALE_RMS_0_2:
      return (float)(0.2 * std::sqrt((double)std::max(rows, cols)));
    default:
      return 1.f;
  }
}

// Power of two nearest sqrt(n): the stored iterate Y = alpha X keeps its
// entries near 1 in magnitude, far from fp16's subnormal range.
float alpha_of(int64_t n) {
  const double e = std::round(0.5 * std::log2((double)n));
  return (float)std::ldexp(1.0, (int)e);
}

muon_status_t build_desc(const muon_shape_t* shapes, int32_t n_params,
                         const muon_plan_options* opts, PlanDesc* d) {
  muon_plan_options o;
  muon_default_options(&o);
  if (opts) o = *opts;
  if (muon_status_t st = check_options(o)) return st;
  d->opt = o;
  if (!shapes || n_params < 1) return fail(MUON_ERR_INVALID_ARG, "need n_params >= 1 shapes");
  std::map<std::pair<int64_t, int64_t>, int> index;
  std::vector<std::vector<std::pair<int32_t, int32_t>>> members;
  int64_t total_members = 0;
  for (int32_t p = 0; p < n_params; ++p) {
    const muon_shape_t& s = shapes[p];
    int64_t E, r, c;
    if (s.ndim == 2) { E = 1; r = s.dims[0]; c = s.dims[1]; }
    else if (s.ndim == 3) { E = s.dims[0]; r = s.dims[1]; c = s.dims[2]; }
    else return fail(MUON_ERR_INVALID_ARG, "parameter %d: ndim %d (need 2 or 3)", p, s.ndim);
    if (E < 1 || r < 1 || c < 1)
      return fail(MUON_ERR_INVALID_ARG, "parameter %d has an empty dim", p);
    if (r > (1 << 30) || c > (1 << 30) || r * c > ((int64_t)1 << 40))
      return fail(MUON_ERR_UNSUPPORTED, "parameter %d is too large", p);
    d->param_E.push_back(E); d->param_rows.push_back(r); d->param_cols.push_back(c);
    d->param_scale.push_back(scale_of(o.scale, r, c));
    total_members += E;
    if (total_members > INT32_MAX) return fail(MUON_ERR_INVALID_ARG, "too many members");
    // the bucket key: (rows, cols), or (min, max) when [r, c] and [c, r]
    // share a group (each member keeps its orientation)
    auto key = (o.flags & MUON_FLAG_MERGE_TRANSPOSED) ? std::make_pair(std::min(r, c), std::max(r, c))
                                                      : std::make_pair(r, c);
    auto it = index.find(key);
    int g;
    if (it == index.end()) {
      g = (int)members.size();
      index[key] = g;
      members.emplace_back();
      GroupPlan gp;
      gp.rows = r; gp.cols = c;
      d->groups.push_back(gp);
    } else {
      g = it->second;
    }
    for (int64_t e = 0; e < E; ++e) members[g].push_back({p, (int32_t)e});
  }
  size_t off = 0;
  int64_t first = 0;
  const bool f32 = o.mode == MUON_MODE_FP32;
  const int32_t thr = o.skinny_threshold == 0 ? 64 : o.skinny_threshold;
  for (size_t g = 0; g < d->groups.size(); ++g) {
    GroupPlan& gp = d->groups[g];
    gp.batch = (int64_t)members[g].size();
    if (gp.batch > 65535)
      return fail(MUON_ERR_UNSUPPORTED, "group %zu has %lld members (max 65535)", g,
                  (long long)gp.batch);
    gp.first_member = first;
    first += gp.batch;
    for (auto& pe : members[g]) {
      d->member_param.push_back(pe.first);
      d->member_expert.push_back(pe.second);
    }
    int n_t = 0;  // members whose parameter is [n, m]
    for (auto& pe : members[g]) n_t += d->param_rows[pe.first] > d->param_cols[pe.first] ? 1 : 0;
    gp.transposed = n_t == 0 ? 0 : (n_t == (int)members[g].size() ? 1 : 2);
    gp.m = std::min(gp.rows, gp.cols);
    gp.n = std::max(gp.rows, gp.cols);
    gp.ns_type = f32 ? NS_F32 : (o.ns_dtype == MUON_NS_BF16 ? NS_BF16 : NS_F16);
    gp.alpha = f32 ? 1.f : alpha_of(gp.n);
    gp.scale = scale_of(o.scale, gp.rows, gp.cols);
    gp.n_pitch = (int64_t)align_up((size_t)gp.n, 8);
    gp.m_pitch = (int64_t)align_up((size_t)gp.m, 8);
    gp.n_chunks = (gp.rows * gp.cols + kMomentumChunk - 1) / kMomentumChunk;
    const double mm = (double)gp.m, nn = (double)gp.n;
    gp.cost = (double)gp.batch * (4 * mm * mm * nn + 2 * mm * mm * mm + 14 * mm * nn);
    // path
    int32_t path = o.path_override;
    if (f32) {
      path = PATH_SIMT;
    } else if (path == PATH_AUTO) {
      const bool sk = thr > 0 && skinny_config((int32_t)gp.rows, (int32_t)gp.cols, thr, &gp.sk,
                                               o.column_shards);
      // (RESIDENT only on request: under the power cap of a full step it
      // measured slower than TENSOR on every shape it takes)
      path = sk ? PATH_SKINNY : PATH_TENSOR;
    } else if (path == PATH_RESIDENT) {
      if (!resident_config(gp.m, gp.n, &gp.rc))
        return fail(MUON_ERR_UNSUPPORTED, "group %zu [%lld,%lld] does not fit the resident path", g,
                    (long long)gp.rows, (long long)gp.cols);
    } else if (path == PATH_SKINNY) {
      if (!skinny_config((int32_t)gp.rows, (int32_t)gp.cols, 64, &gp.sk, o.column_shards))
        return fail(MUON_ERR_UNSUPPORTED, "group %zu [%lld,%lld] does not fit the skinny path", g,
                    (long long)gp.rows, (long long)gp.cols);
    }
    gp.path = path;
    // scratch
    size_t o2 = 0;
    if (path == PATH_SKINNY) {
      gp.off_y0 = o2; o2 = align_up(o2 + (size_t)gp.batch * gp.sk.ws_bytes, kAlign);
      gp.off_part = o2; o2 = align_up(o2 + (size_t)gp.batch * gp.n_chunks * 4, kAlign);
      if (o.flags & MUON_FLAG_NESTEROV) {  // read only by the direct kernel (k > kGramSpaceMaxSteps)
        gp.off_u = o2; o2 = align_up(o2 + (size_t)gp.batch * gp.rows * gp.cols * 4, kAlign);
      }
    } else if (path == PATH_TENSOR || path == PATH_SIMT) {
      const size_t es = ns_esize(gp.ns_type);
      const size_t yb = (size_t)gp.batch * gp.m * gp.n_pitch * es;
      const size_t ab = (size_t)gp.batch * gp.m * gp.m_pitch * es;
      gp.off_y0 = o2; o2 = align_up(o2 + yb, kAlign);
      gp.off_y1 = o2; o2 = align_up(o2 + yb, kAlign);
      gp.off_a = o2;  o2 = align_up(o2 + ab, kAlign);
      gp.off_q = o2;  o2 = align_up(o2 + ab, kAlign);
      gp.off_part = o2; o2 = align_up(o2 + (size_t)gp.batch * gp.n_chunks * 4, kAlign);
      gp.off_invn = o2; o2 = align_up(o2 + (size_t)gp.batch * 4, kAlign);
    }
    if (o.flags & MUON_FLAG_KEEP_UPDATE) {
      gp.off_dbg = o2;
      o2 = align_up(o2 + (size_t)gp.batch * gp.rows * gp.cols * 4, kAlign);
    }
    gp.ws_bytes = o2;
    gp.base = off;
    off = align_up(off + o2, kAlign);
  }
  d->off_scalars = off;
  d->pb_bytes = align_up(sizeof(StepScalars), 16) + (size_t)first * sizeof(MemberPtrs);
  off = align_up(off + d->pb_bytes, kAlign);
  d->off_err = off;
  off = align_up(off + 16, kAlign);
  d->ws_bytes = off;
  return MUON_OK;
}

}  // namespace

void set_last_error(const char* msg) { g_last_error = msg; }

}  // namespace muon

using namespace muon;

// Chunks of the pipelined host-buffer step (muon_step_host on skinny-only plans).
constexpr int kHostChunks = 4;
// Units of the pipelined muon_step_host for other plans: slices of whole
// members of a group, about 1/kHostUnits of the plan's elements each.
constexpr int kHostUnits = 16;

struct muon_plan_s {
  PlanDesc d;
  int device = 0;
  int num_sms = 1;
  unsigned char* ws = nullptr;        // device scratch
  unsigned char* pinned = nullptr;    // kRingSlots parameter blocks
  std::vector<unsigned char> last_pb; // contents of the last uploaded parameter block
  bool pb_valid = false;
  cudaEvent_t slot_ev[kRingSlots] = {};
  int slot = 0;
  cudaStream_t cap = nullptr;
  std::vector<cudaStream_t> aux;
  cudaEvent_t fork_ev = nullptr;
  std::vector<cudaEvent_t> join_ev;
  std::map<int32_t, cudaGraphExec_t> graphs;
  std::vector<cudaEvent_t> t_start, t_stop;  // per group, MUON_FLAG_GROUP_TIMING
  bool capturing = false;
  // host staging (muon_step_host)
  unsigned char* stage_p = nullptr;
  unsigned char* stage_g = nullptr;
  float* stage_m = nullptr;
  std::vector<size_t> stage_off;      // element offset of each parameter
  // pipelined muon_step_host (skinny-only plans): copy streams and per-chunk events
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t up_ev = nullptr;
  std::vector<cudaEvent_t> in_ev, run_ev, out_ev;
  // pipelined muon_step_host (other plans): members [i0, i0 + cnt) of group g
  // per unit, with the tensor maps of that slice of the group's workspace
  struct HostUnit {
    int32_t g;
    int64_t i0, cnt;
    TcMaps tc;
  };
  std::vector<HostUnit> units;
};

namespace {

KArgs make_args(const muon_plan_s* p, const GroupPlan& g) {
  KArgs a{};
  unsigned char* base = p->ws + g.base;
  a.sc = reinterpret_cast<const StepScalars*>(p->ws + p->d.off_scalars);
  a.mem = reinterpret_cast<const MemberPtrs*>(p->ws + p->d.off_scalars +
                                              align_up(sizeof(StepScalars), 16)) +
          g.first_member;
  a.B = (int32_t)g.batch;
  a.rows = (int32_t)g.rows; a.cols = (int32_t)g.cols;
  a.m = (int32_t)g.m; a.n = (int32_t)g.n;
  a.T = g.transposed;
  a.mode_f32 = p->d.opt.mode == MUON_MODE_FP32;
  a.ns_type = g.ns_type;
  a.n_pitch = g.n_pitch; a.m_pitch = g.m_pitch;
  a.n_chunks = (int32_t)g.n_chunks;
  a.eps = p->d.opt.eps;
  a.scale = g.scale;
  a.alpha = g.alpha;
  a.y0 = base + g.off_y0;
  a.part = reinterpret_cast<float*>(base + g.off_part);
  if (g.path == PATH_TENSOR || g.path == PATH_SIMT) {
    a.y1 = base + g.off_y1;
    a.A = base + g.off_a; a.Q = base + g.off_q;
    a.invn = reinterpret_cast<float*>(base + g.off_invn);
  }
  a.dbg = (p->d.opt.flags & MUON_FLAG_KEEP_UPDATE) ? reinterpret_cast<float*>(base + g.off_dbg)
                                                   : nullptr;
  a.err = reinterpret_cast<int*>(p->ws + p->d.off_err);
  a.l2_keep_m = g.path == PATH_SKINNY;
  a.nesterov = (p->d.opt.flags & MUON_FLAG_NESTEROV) ? 1 : 0;
  a.u = (g.path == PATH_SKINNY && a.nesterov) ? reinterpret_cast<float*>(base + g.off_u) : nullptr;
  return a;
}

// Kernel arguments of members [i0, i0 + cnt) of group g: every per-member
// pointer (the caller's buffers through the member table, and the group's
// scratch) moves by i0 members.
KArgs sub_args(const KArgs& a, const GroupPlan& g, int64_t i0, int64_t cnt) {
  KArgs r = a;
  r.B = (int32_t)cnt;
  r.mem = a.mem + i0;
  const int64_t mn = g.m * g.n;
  if (a.dbg) r.dbg = a.dbg + i0 * mn;
  if (g.path == PATH_SKINNY) {
    r.part = a.part + i0 * a.n_chunks;
    r.y0 = static_cast<unsigned char*>(a.y0) + i0 * g.sk.ws_bytes;
    if (a.u) r.u = a.u + i0 * mn;
  } else if (g.path == PATH_TENSOR || g.path == PATH_SIMT) {
    const size_t es = ns_esize(g.ns_type);
    const size_t yb = (size_t)g.m * g.n_pitch * es, ab = (size_t)g.m * g.m_pitch * es;
    r.y0 = static_cast<unsigned char*>(a.y0) + i0 * yb;
    r.y1 = static_cast<unsigned char*>(a.y1) + i0 * yb;
    r.A = static_cast<unsigned char*>(a.A) + i0 * ab;
    r.Q = static_cast<unsigned char*>(a.Q) + i0 * ab;
    r.part = a.part + i0 * a.n_chunks;
    r.invn = a.invn + i0;
  }
  return r;
}

// Enqueue the whole step of the members `a` describes (a group, or a slice of
// one with its own tensor maps `tc`) on stream s.
cudaError_t enqueue_kernels(const KArgs& a, const GroupPlan& g, const TcMaps& tc, int32_t k,
                            cudaStream_t s) {
  cudaError_t e;
  if (g.path == PATH_SKINNY) return launch_skinny(a, g.sk, k, s);
  if (g.path == PATH_RESIDENT) return launch_resident(a, g.rc, s);
  if ((e = launch_momentum_partial(a, s))) return e;
  if ((e = launch_norm_finalize(a, s))) return e;
  if ((e = launch_normalize_cast(a, a.y0, s))) return e;
  if (g.path == PATH_TENSOR) {
    int src = 0;
    for (int32_t it = 0; it < k; ++it) {
      if ((e = launch_tc_gram(a, tc, src, s))) return e;
      if ((e = launch_tc_poly(a, tc, it, s))) return e;
      if ((e = launch_tc_update(a, tc, src, s))) return e;
      src ^= 1;
    }
    return launch_write(a, src == 0 ? a.y0 : a.y1, s);
  }
  void* ys = a.y0;
  void* yd = a.y1;
  for (int32_t it = 0; it < k; ++it) {
    if ((e = launch_simt_gram(a, ys, s))) return e;
    if ((e = launch_simt_poly(a, it, s))) return e;
    if ((e = launch_simt_update(a, ys, yd, s))) return e;
    std::swap(ys, yd);
  }
  return launch_write(a, ys, s);
}

// Enqueue one group's whole step on stream s.
cudaError_t enqueue_group_kernels(const muon_plan_s* p, const GroupPlan& g, int32_t k,
                                  cudaStream_t s) {
  return enqueue_kernels(make_args(p, g), g, g.tc, k, s);
}

cudaError_t record(const muon_plan_s* p, cudaEvent_t ev, cudaStream_t s) {
  return p->capturing ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                      : cudaEventRecord(ev, s);
}

cudaError_t enqueue_group(const muon_plan_s* p, size_t gi, int32_t k, cudaStream_t s) {
  const bool timed = !p->t_start.empty();
  cudaError_t e;
  if (timed && (e = record(p, p->t_start[gi], s))) return e;
  if ((e = enqueue_group_kernels(p, p->d.groups[gi], k, s))) return e;
  if (timed && (e = record(p, p->t_stop[gi], s))) return e;
  return cudaSuccess;
}

// A group whose kernels alone occupy every SM: its update GEMM has at least
// one 128-row tile per SM (tensor path), or its clusters cover the SMs.
bool fills_gpu(const muon_plan_s* p, const GroupPlan& g) {
  if (g.path == PATH_TENSOR) {
    const int64_t bn = g.n >= 256 ? 256 : 128;
    return g.batch * ((g.m + 127) / 128) * ((g.n + bn - 1) / bn) >= p->num_sms;
  }
  if (g.path == PATH_RESIDENT) return g.batch * g.rc.cluster >= p->num_sms;
  return g.path == PATH_SKINNY && g.batch * g.sk.cluster >= p->num_sms;
}

muon_status_t enqueue_all(muon_plan_s* p, int32_t k, cudaStream_t s, bool fork) {
  std::vector<size_t> order(p->d.groups.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](size_t x, size_t y) {
    return p->d.groups[x].cost > p->d.groups[y].cost;
  });
  // Groups that fill the GPU run one after another on the caller's stream:
  // side by side, persistent kernels would only split the SMs between them
  // and share L2.  The others are dealt to the auxiliary streams, where they
  // overlap with one another and with the big ones.
  const size_t ns = fork ? std::min(order.size(), p->aux.size() + 1) : 1;
  std::vector<size_t> lane_of(order.size(), 0);
  size_t next = 0;
  for (size_t i = 0; i < order.size(); ++i)
    if (ns > 1 && !fills_gpu(p, p->d.groups[order[i]])) lane_of[i] = 1 + (next++ % (ns - 1));
  if (ns > 1) {
    CUDA_TRY(cudaEventRecord(p->fork_ev, s));
    for (size_t i = 0; i + 1 < ns; ++i) CUDA_TRY(cudaStreamWaitEvent(p->aux[i], p->fork_ev, 0));
  }
  for (size_t i = 0; i < order.size(); ++i) {
    const size_t lane = lane_of[i];
    cudaStream_t st = lane == 0 ? s : p->aux[lane - 1];
    cudaError_t e = enqueue_group(p, order[i], k, st);
    if (e != cudaSuccess)
      return fail(MUON_ERR_CUDA, "launch for group %zu failed: %s", order[i], cudaGetErrorString(e));
  }
  if (ns > 1) {
    for (size_t i = 0; i + 1 < ns; ++i) {
      CUDA_TRY(cudaEventRecord(p->join_ev[i], p->aux[i]));
      CUDA_TRY(cudaStreamWaitEvent(s, p->join_ev[i], 0));
    }
  }
  return MUON_OK;
}

muon_status_t get_graph(muon_plan_s* p, int32_t k, cudaGraphExec_t* out) {
  auto it = p->graphs.find(k);
  if (it != p->graphs.end()) { *out = it->second; return MUON_OK; }
  CUDA_TRY(cudaStreamBeginCapture(p->cap, cudaStreamCaptureModeThreadLocal));
  p->capturing = true;
  muon_status_t st = enqueue_all(p, k, p->cap, true);
  p->capturing = false;
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(p->cap, &graph);
  if (st != MUON_OK) { if (graph) cudaGraphDestroy(graph); return st; }
  if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "stream capture failed: %s", cudaGetErrorString(e));
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  p->graphs[k] = exec;
  *out = exec;
  return MUON_OK;
}

void destroy_plan(muon_plan_s* p) {
  if (!p) return;
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  for (auto& kv : p->graphs) cudaGraphExecDestroy(kv.second);
  for (auto& ev : p->slot_ev) if (ev) cudaEventDestroy(ev);
  for (auto ev : p->t_start) cudaEventDestroy(ev);
  for (auto ev : p->t_stop) cudaEventDestroy(ev);
  if (p->fork_ev) cudaEventDestroy(p->fork_ev);
  for (auto ev : p->join_ev) cudaEventDestroy(ev);
  for (auto st : p->aux) cudaStreamDestroy(st);
  if (p->cap) cudaStreamDestroy(p->cap);
  if (p->ws) cudaFree(p->ws);
  if (p->pinned) cudaFreeHost(p->pinned);
  for (auto ev : p->in_ev) cudaEventDestroy(ev);
  for (auto ev : p->run_ev) cudaEventDestroy(ev);
  for (auto ev : p->out_ev) cudaEventDestroy(ev);
  if (p->up_ev) cudaEventDestroy(p->up_ev);
  if (p->h2d) cudaStreamDestroy(p->h2d);
  if (p->d2h) cudaStreamDestroy(p->d2h);
  if (p->stage_p) cudaFree(p->stage_p);
  if (p->stage_g) cudaFree(p->stage_g);
  if (p->stage_m) cudaFree(p->stage_m);
  delete p;
}

size_t p_esize(const muon_plan_s* p) { return p->d.opt.mode == MUON_MODE_FP32 ? 4 : 2; }

int64_t param_elems(const PlanDesc& d, int32_t i) {
  return d.param_E[i] * d.param_rows[i] * d.param_cols[i];
}

}  // namespace

extern "C" {

muon_status_t muon_default_options(muon_plan_options* o) {
  if (!o) return fail(MUON_ERR_INVALID_ARG, "options pointer is NULL");
  std::memset(o, 0, sizeof *o);
  o->mode = MUON_MODE_BF16;
  o->scale = MUON_SCALE_SQRT_ASPECT;
  o->eps = 1e-7f;
  o->skinny_threshold = 0;
  o->ns_dtype = MUON_NS_FP16;
  o->flags = 0;
  o->path_override = MUON_PATH_AUTO;
  o->max_streams = 0;
  return MUON_OK;
}

muon_status_t muon_plan_describe(const muon_shape_t* shapes, int32_t n_params,
                                 const muon_plan_options* opts, muon_group_info_t* groups,
                                 int32_t group_cap, int32_t* n_groups, int32_t* member_param,
                                 int32_t* member_expert, int64_t member_cap, int64_t* n_members,
                                 size_t* workspace_bytes) {
  PlanDesc d;
  if (muon_status_t st = build_desc(shapes, n_params, opts, &d)) return st;
  if (n_groups) *n_groups = (int32_t)d.groups.size();
  if (groups)
    for (int32_t g = 0; g < group_cap && g < (int32_t)d.groups.size(); ++g) {
      const GroupPlan& gp = d.groups[g];
      groups[g] = muon_group_info_t{gp.rows, gp.cols, gp.batch, gp.first_member,
                                    gp.transposed, gp.path, (int64_t)gp.ws_bytes};
    }
  const int64_t nm = (int64_t)d.member_param.size();
  if (n_members) *n_members = nm;
  for (int64_t i = 0; i < member_cap && i < nm; ++i) {
    if (member_param) member_param[i] = d.member_param[i];
    if (member_expert) member_expert[i] = d.member_expert[i];
  }
  if (workspace_bytes) *workspace_bytes = d.ws_bytes;
  return MUON_OK;
}

namespace {

// Estimated seconds of one member's step on this library's path for its
// group: the larger of its compulsory memory traffic over the HBM rate and
// its Newton-Schulz work over the tensor (or fp32 FMA) rate.  Only ratios
// matter to the planner.  The HBM and tensor rates are a GB300's measured
// copy bandwidth and sustained bf16 GEMM rate; the fp32 rate is a nominal
// FFMA figure.
double member_seconds(const GroupPlan& g, int32_t ns_steps, bool f32) {
  constexpr double kHbm = 6.8e12, kTensor = 1.7e15, kFp32 = 6.0e13;
  const double m = (double)g.m, n = (double)g.n;
  const double bytes = m * n * (f32 ? 20.0 : 14.0);
  const double flops = (double)ns_steps * (4 * m * m * n + 2 * m * m * m);
  const double rate = f32 ? kFp32 : kTensor;
  const bool hbm_bound = g.path == PATH_SKINNY || g.path == PATH_RESIDENT;
  return std::max(bytes / kHbm, hbm_bound ? 0.0 : flops / rate);
}

}  // namespace

muon_status_t muon_plan_assign(const muon_shape_t* shapes, int32_t n_params,
                               const muon_plan_options* opts, int32_t ns_steps, int32_t n_ranks,
                               int32_t* owner, int64_t member_cap, double* member_cost,
                               double* rank_cost) {
  if (n_ranks < 1 || n_ranks > (1 << 20))
    return fail(MUON_ERR_INVALID_ARG, "n_ranks %d out of [1, 2^20]", n_ranks);
  if (ns_steps < 0 || ns_steps > 1000)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps %d out of [0, 1000]", ns_steps);
  PlanDesc d;
  if (muon_status_t st = build_desc(shapes, n_params, opts, &d)) return st;
  const int64_t nm = (int64_t)d.member_param.size();
  if (!owner || member_cap < nm)
    return fail(MUON_ERR_INVALID_ARG, "owner must hold %lld members", (long long)nm);
  const bool f32 = d.opt.mode == MUON_MODE_FP32;
  std::vector<double> cost((size_t)nm);
  for (const GroupPlan& g : d.groups) {
    const double t = member_seconds(g, ns_steps, f32);
    for (int64_t i = 0; i < g.batch; ++i) cost[(size_t)(g.first_member + i)] = t;
  }
  // longest processing time first: members by cost (descending, then index),
  // each to the rank with the least load so far (then the lowest rank)
  std::vector<int64_t> order((size_t)nm);
  for (int64_t i = 0; i < nm; ++i) order[(size_t)i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int64_t x, int64_t y) { return cost[(size_t)x] > cost[(size_t)y]; });
  using Slot = std::pair<double, int32_t>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int32_t r = 0; r < n_ranks; ++r) heap.push({0.0, r});
  std::vector<double> load((size_t)n_ranks, 0.0);
  for (int64_t i : order) {
    const Slot s = heap.top();
    heap.pop();
    owner[i] = s.second;
    load[(size_t)s.second] = s.first + cost[(size_t)i];
    heap.push({load[(size_t)s.second], s.second});
  }
  if (member_cost)
    for (int64_t i = 0; i < nm; ++i) member_cost[i] = cost[(size_t)i];
  if (rank_cost)
    for (int32_t r = 0; r < n_ranks; ++r) rank_cost[r] = load[(size_t)r];
  return MUON_OK;
}

muon_status_t muon_plan_create(const muon_shape_t* shapes, int32_t n_params,
                               const muon_plan_options* opts, int device, muon_plan_t* out) {
  if (!out) return fail(MUON_ERR_INVALID_ARG, "out pointer is NULL");
  *out = nullptr;
  muon_plan_s* p = new (std::nothrow) muon_plan_s();
  if (!p) return fail(MUON_ERR_OOM, "host allocation failed");
  if (muon_status_t st = build_desc(shapes, n_params, opts, &p->d)) { delete p; return st; }
  p->device = device;
  auto bail = [&](muon_status_t s) { destroy_plan(p); return s; };
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return bail(fail(MUON_ERR_INVALID_ARG, "device %d is not available", device));
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess)
    return bail(fail(MUON_ERR_CUDA, "cudaGetDeviceProperties failed"));
  if (prop.major != 10 || prop.minor != 3)
    return bail(fail(MUON_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                     device, prop.major, prop.minor));
#define PLAN_TRY(expr)                                                                    \
  do {                                                                                    \
    cudaError_t e_ = (expr);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return bail(fail(e_ == cudaErrorMemoryAllocation ? MUON_ERR_OOM : MUON_ERR_CUDA,    \
                       "%s failed: %s", #expr, cudaGetErrorString(e_)));                  \
  } while (0)
  PLAN_TRY(cudaSetDevice(device));
  PLAN_TRY(cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, device));
  PLAN_TRY(cudaMalloc(&p->ws, p->d.ws_bytes));
  PLAN_TRY(cudaMemset(p->ws, 0, p->d.ws_bytes));
  PLAN_TRY(cudaHostAlloc(&p->pinned, kRingSlots * p->d.pb_bytes, cudaHostAllocDefault));
  p->last_pb.assign(p->d.pb_bytes, 0);
  for (auto& ev : p->slot_ev) PLAN_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
  PLAN_TRY(cudaStreamCreateWithFlags(&p->cap, cudaStreamNonBlocking));
  const int nstreams = p->d.opt.max_streams == 0 ? 4 : p->d.opt.max_streams;
  const int naux = std::min<int>(nstreams, (int)p->d.groups.size()) - 1;
  for (int i = 0; i < naux; ++i) {
    cudaStream_t s;
    PLAN_TRY(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    p->aux.push_back(s);
    cudaEvent_t ev;
    PLAN_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    p->join_ev.push_back(ev);
  }
  PLAN_TRY(cudaEventCreateWithFlags(&p->fork_ev, cudaEventDisableTiming));
  if (p->d.opt.flags & MUON_FLAG_GROUP_TIMING) {
    for (size_t g = 0; g < p->d.groups.size(); ++g) {
      cudaEvent_t e0, e1;
      PLAN_TRY(cudaEventCreate(&e0));
      p->t_start.push_back(e0);
      PLAN_TRY(cudaEventCreate(&e1));
      p->t_stop.push_back(e1);
    }
  }
  bool tc_ready[3] = {false, false, false};
  for (GroupPlan& g : p->d.groups) {
    if (g.path == PATH_SKINNY) PLAN_TRY(prepare_skinny(make_args(p, g), g.sk));
    if (g.path == PATH_RESIDENT) PLAN_TRY(prepare_resident(g.ns_type));
    if (g.path == PATH_TENSOR) {
      if (!tc_ready[g.ns_type]) {
        PLAN_TRY(prepare_tc(g.ns_type));
        tc_ready[g.ns_type] = true;
      }
      PLAN_TRY(tc_make_maps(make_args(p, g), &g.tc));
    }
  }
  if (p->d.opt.flags & MUON_FLAG_HOST_STAGING) {
    size_t tot = 0;
    for (int32_t i = 0; i < (int32_t)p->d.param_E.size(); ++i) {
      p->stage_off.push_back(tot);
      tot += align_up((size_t)param_elems(p->d, i), 64);
    }
    PLAN_TRY(cudaMalloc(&p->stage_p, tot * p_esize(p)));
    PLAN_TRY(cudaMalloc(&p->stage_g, tot * p_esize(p)));
    PLAN_TRY(cudaMalloc(&p->stage_m, tot * 4));
    PLAN_TRY(cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking));
    PLAN_TRY(cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking));
    PLAN_TRY(cudaEventCreateWithFlags(&p->up_ev, cudaEventDisableTiming));
    bool skinny_only = true;
    for (const GroupPlan& g : p->d.groups) skinny_only = skinny_only && g.path == PATH_SKINNY;
    if (!skinny_only) {
      int64_t total = 0;
      for (const GroupPlan& g : p->d.groups) total += g.batch * g.m * g.n;
      const int64_t target = std::max<int64_t>(1, total / kHostUnits);
      for (int32_t gi = 0; gi < (int32_t)p->d.groups.size(); ++gi) {
        const GroupPlan& g = p->d.groups[gi];
        const int64_t nsl = std::min<int64_t>(g.batch, std::max<int64_t>(1, (g.batch * g.m * g.n + target - 1) / target));
        const int64_t per = (g.batch + nsl - 1) / nsl;
        for (int64_t i0 = 0; i0 < g.batch; i0 += per) {
          muon_plan_s::HostUnit u{};
          u.g = gi;
          u.i0 = i0;
          u.cnt = std::min(per, g.batch - i0);
          if (g.path == PATH_TENSOR) PLAN_TRY(tc_make_maps(sub_args(make_args(p, g), g, u.i0, u.cnt), &u.tc));
          p->units.push_back(u);
        }
      }
    }
    const int nev = std::max<int>(kHostChunks, (int)p->units.size());  // chunks or units
    for (int i = 0; i < nev; ++i) {
      cudaEvent_t e0, e1, e2;
      PLAN_TRY(cudaEventCreateWithFlags(&e0, cudaEventDisableTiming));
      p->in_ev.push_back(e0);
      PLAN_TRY(cudaEventCreateWithFlags(&e1, cudaEventDisableTiming));
      p->run_ev.push_back(e1);
      PLAN_TRY(cudaEventCreateWithFlags(&e2, cudaEventDisableTiming));
      p->out_ev.push_back(e2);
    }
  }
  PLAN_TRY(cudaDeviceSynchronize());
#undef PLAN_TRY
  *out = p;
  return MUON_OK;
}

namespace {

// The one step of muon_step and muon_step_schedule: `coef` holds n_coef
// (a, b, c) rows (host memory).
muon_status_t step_impl(muon_plan_t p, void* const* params, const void* const* grads,
                        float* const* momenta, float beta, float lr, float wd, int32_t ns_steps,
                        const float* coef, int32_t n_coef, void* stream, bool launch = true) {
  if (!p) return fail(MUON_ERR_INVALID_ARG, "plan is NULL");
  if (!params || !grads || !momenta) return fail(MUON_ERR_INVALID_ARG, "NULL pointer array");
  if (ns_steps < 0 || ns_steps > 1000)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps %d out of [0, 1000]", ns_steps);
  if (!coef) return fail(MUON_ERR_INVALID_ARG, "coefficient schedule is NULL");
  if (n_coef < 1 || n_coef > kMaxScheduleRows)
    return fail(MUON_ERR_INVALID_ARG, "schedule rows %d out of [1, %d]", n_coef, kMaxScheduleRows);
  const float sc[3] = {beta, lr, wd};
  for (float v : sc)
    if (!std::isfinite(v)) return fail(MUON_ERR_INVALID_ARG, "non-finite step scalar");
  for (int32_t i = 0; i < 3 * n_coef; ++i)
    if (!std::isfinite(coef[i])) return fail(MUON_ERR_INVALID_ARG, "non-finite coefficient");
  const int32_t np = (int32_t)p->d.param_E.size();
  for (int32_t i = 0; i < np; ++i)
    if (!params[i] || !grads[i] || !momenta[i])
      return fail(MUON_ERR_INVALID_ARG, "parameter %d has a NULL pointer", i);
  // bf16 operands rounded on every step (every group but a Gram-space skinny
  // one) drift past the bf16-mode tolerance beyond kBf16OperandMaxSteps
  if (ns_steps > kBf16OperandMaxSteps)
    for (const GroupPlan& g : p->d.groups)
      if (g.ns_type == NS_BF16 && !(g.path == PATH_SKINNY && ns_steps <= kGramSpaceMaxSteps))
        return fail(MUON_ERR_UNSUPPORTED,
                    "group [%lld,%lld] iterates on bf16 operands, which is limited to %d "
                    "Newton-Schulz steps (asked for %d); use fp16 operands",
                    (long long)g.rows, (long long)g.cols, kBf16OperandMaxSteps, ns_steps);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaSetDevice(p->device));
  // fill the next pinned slot once its previous copy has been consumed
  const int slot = p->slot;
  p->slot = (p->slot + 1) % kRingSlots;
  CUDA_TRY(cudaEventSynchronize(p->slot_ev[slot]));
  unsigned char* host = p->pinned + (size_t)slot * p->d.pb_bytes;
  StepScalars ss{};
  ss.beta = beta; ss.lr = lr; ss.wd = wd;
  ss.ns_steps = ns_steps;
  ss.n_coef = n_coef;
  std::memcpy(ss.coef, coef, sizeof(float) * 3 * (size_t)n_coef);
  std::memcpy(host, &ss, sizeof ss);
  MemberPtrs* mp = reinterpret_cast<MemberPtrs*>(host + align_up(sizeof(StepScalars), 16));
  const size_t pes = p_esize(p);
  for (size_t i = 0; i < p->d.member_param.size(); ++i) {
    const int32_t pi = p->d.member_param[i];
    const int64_t e = p->d.member_expert[i];
    const int64_t off = e * p->d.param_rows[pi] * p->d.param_cols[pi];
    mp[i].P = static_cast<unsigned char*>(params[pi]) + off * pes;
    mp[i].G = static_cast<const unsigned char*>(grads[pi]) + off * pes;
    mp[i].M = momenta[pi] + off;
    mp[i].T = p->d.param_rows[pi] > p->d.param_cols[pi] ? 1 : 0;
    mp[i].scale = p->d.param_scale[pi];
  }
  // The device block keeps the last upload (stream order on `s` makes it
  // visible to the steps after it): a step with the same scalars and buffers
  // as the one before it needs no copy.
  if (!p->pb_valid || std::memcmp(host, p->last_pb.data(), p->d.pb_bytes) != 0) {
    std::memcpy(p->last_pb.data(), host, p->d.pb_bytes);
    p->pb_valid = true;
    CUDA_TRY(cudaMemcpyAsync(p->ws + p->d.off_scalars, host, p->d.pb_bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaEventRecord(p->slot_ev[slot], s));
  }
  if (!launch) return MUON_OK;  // the caller enqueues the kernels itself
  if (p->d.opt.flags & MUON_FLAG_NO_GRAPH) return enqueue_all(p, ns_steps, s, false);
  cudaGraphExec_t exec;
  if (muon_status_t st = get_graph(p, ns_steps, &exec)) return st;
  CUDA_TRY(cudaGraphLaunch(exec, s));
  return MUON_OK;
}

bool all_skinny(const muon_plan_s* p) {
  for (const GroupPlan& g : p->d.groups)
    if (g.path != PATH_SKINNY) return false;
  return true;
}

// One cudaMemcpyAsync per run of parameters in [p0, p1) whose host and device
// buffers are both back to back.
cudaError_t copy_param_runs(const muon_plan_s* p, int32_t p0, int32_t p1, const void* const* host,
                            void* const* dev, size_t es, bool to_device, cudaStream_t s) {
  int32_t i = p0;
  while (i < p1) {
    int32_t j = i + 1;
    size_t bytes = (size_t)param_elems(p->d, i) * es;
    while (j < p1 && (const unsigned char*)host[j] == (const unsigned char*)host[i] + bytes &&
           (const unsigned char*)dev[j] == (const unsigned char*)dev[i] + bytes) {
      bytes += (size_t)param_elems(p->d, j) * es;
      ++j;
    }
    const cudaError_t e =
        to_device ? cudaMemcpyAsync(dev[i], host[i], bytes, cudaMemcpyHostToDevice, s)
                  : cudaMemcpyAsync(const_cast<void*>(host[i]), dev[i], bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    i = j;
  }
  return cudaSuccess;
}

// muon_step_host for a plan whose groups all take the skinny path.  The
// parameters go in up to in_ev.size() chunks of about equal size: a chunk's
// inputs are copied in on one stream, its members' kernels run on the
// caller's stream once they have landed, and its results are copied out on
// a third stream.  So one chunk's copy back overlaps the next chunk's copy
// in (the host link carries both directions at once), and the kernels hide
// behind the copies.  Every member gets the same kernels as in a whole-plan
// step, so its results are the same bits.
muon_status_t host_step_pipelined(muon_plan_s* p, void* const* hp, const void* const* hg,
                                  float* const* hm, std::vector<void*>& dp, std::vector<void*>& dg,
                                  std::vector<float*>& dm, float beta, float lr, float wd,
                                  int32_t k, float a, float b, float c, cudaStream_t s) {
  const int32_t np = (int32_t)p->d.param_E.size();
  const float coef[3] = {a, b, c};
  // scalars and member pointers (the staging buffers) to the device, on s
  if (muon_status_t st = step_impl(p, dp.data(), (const void* const*)dg.data(), dm.data(), beta, lr,
                                   wd, k, coef, 1, s, false))
    return st;
  CUDA_TRY(cudaEventRecord(p->up_ev, s));
  CUDA_TRY(cudaStreamWaitEvent(p->h2d, p->up_ev, 0));
  // chunk boundaries: parameter ranges of about equal element counts
  const int nch = std::min<int>((int)p->in_ev.size(), np);
  int64_t total = 0;
  for (int32_t i = 0; i < np; ++i) total += param_elems(p->d, i);
  std::vector<int32_t> cut(nch + 1, np);
  cut[0] = 0;
  {
    int64_t acc = 0;
    int ci = 1;
    for (int32_t i = 0; i < np && ci < nch; ++i) {
      acc += param_elems(p->d, i);
      if (acc * nch >= total * ci) cut[ci++] = i + 1;
    }
  }
  const size_t pes = p_esize(p);
  std::vector<const void*> hpc(hp, hp + np), hmc(hm, hm + np);
  std::vector<void*> dmv(dm.begin(), dm.end());
  for (int ci = 0; ci < nch; ++ci) {
    const int32_t p0 = cut[ci], p1 = cut[ci + 1];
    if (p0 >= p1) continue;
    CUDA_TRY(copy_param_runs(p, p0, p1, hpc.data(), dp.data(), pes, true, p->h2d));
    CUDA_TRY(copy_param_runs(p, p0, p1, hg, dg.data(), pes, true, p->h2d));
    CUDA_TRY(copy_param_runs(p, p0, p1, hmc.data(), dmv.data(), 4, true, p->h2d));
    CUDA_TRY(cudaEventRecord(p->in_ev[ci], p->h2d));
    CUDA_TRY(cudaStreamWaitEvent(s, p->in_ev[ci], 0));
    for (const GroupPlan& g : p->d.groups) {
      int64_t i0 = -1, cnt = 0;  // the chunk's members of g are contiguous in it
      for (int64_t i = 0; i < g.batch; ++i) {
        const int32_t pi = p->d.member_param[g.first_member + i];
        if (pi >= p0 && pi < p1) {
          if (i0 < 0) i0 = i;
          ++cnt;
        }
      }
      if (!cnt) continue;
      const cudaError_t e = launch_skinny(sub_args(make_args(p, g), g, i0, cnt), g.sk, k, s);
      if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    }
    CUDA_TRY(cudaEventRecord(p->run_ev[ci], s));
    CUDA_TRY(cudaStreamWaitEvent(p->d2h, p->run_ev[ci], 0));
    CUDA_TRY(copy_param_runs(p, p0, p1, hpc.data(), dp.data(), pes, false, p->d2h));
    CUDA_TRY(copy_param_runs(p, p0, p1, hmc.data(), dmv.data(), 4, false, p->d2h));
  }
  CUDA_TRY(cudaEventRecord(p->out_ev[0], p->d2h));
  CUDA_TRY(cudaStreamWaitEvent(s, p->out_ev[0], 0));
  CUDA_TRY(cudaStreamSynchronize(s));
  return MUON_OK;
}

// muon_step_host for other plans: the same three-stream pipeline with slices
// of whole members of a group as its units (about 1/kHostUnits of the plan's
// elements each, so that the copy in before the first kernels and the copy
// out after the last ones are short).  Every unit's inputs are queued for
// copy-in at once; its kernels run on the caller's stream once they have
// landed (units one after another), and its parameters and momenta are
// copied back as soon as its kernels are done, so the copies of other units
// hide behind each unit's kernels.  Every member gets the same kernels as in
// a whole-plan step, so its results are the same bits.
muon_status_t host_step_units(muon_plan_s* p, void* const* hp, const void* const* hg,
                              float* const* hm, std::vector<void*>& dp, std::vector<void*>& dg,
                              std::vector<float*>& dm, float beta, float lr, float wd,
                              int32_t k, float a, float b, float c, cudaStream_t s) {
  const float coef[3] = {a, b, c};
  if (muon_status_t st = step_impl(p, dp.data(), (const void* const*)dg.data(), dm.data(), beta, lr,
                                   wd, k, coef, 1, s, false))
    return st;
  CUDA_TRY(cudaEventRecord(p->up_ev, s));
  CUDA_TRY(cudaStreamWaitEvent(p->h2d, p->up_ev, 0));
  const size_t pes = p_esize(p);
  using Unit = muon_plan_s::HostUnit;
  // one copy per run of the unit's members whose host and device bytes are
  // both back to back
  auto copy = [&](const Unit& u, const void* const* host, const void* const* dev, size_t es,
                  bool to_device, cudaStream_t st) -> cudaError_t {
    const GroupPlan& g = p->d.groups[u.g];
    const size_t mb = (size_t)g.m * g.n * es;  // bytes of one member
    auto at = [&](const void* const* base, int64_t i) {
      const int64_t mi = g.first_member + u.i0 + i;
      return static_cast<const unsigned char*>(base[p->d.member_param[mi]]) +
             (size_t)p->d.member_expert[mi] * mb;
    };
    int64_t i = 0;
    while (i < u.cnt) {
      int64_t j = i + 1;
      size_t bytes = mb;
      while (j < u.cnt && at(host, j) == at(host, i) + bytes && at(dev, j) == at(dev, i) + bytes) {
        bytes += mb;
        ++j;
      }
      void* h = const_cast<unsigned char*>(at(host, i));
      void* d = const_cast<unsigned char*>(at(dev, i));
      const cudaError_t e = to_device ? cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice, st)
                                      : cudaMemcpyAsync(h, d, bytes, cudaMemcpyDeviceToHost, st);
      if (e != cudaSuccess) return e;
      i = j;
    }
    return cudaSuccess;
  };
  const void* const* hpc = (const void* const*)hp;
  const void* const* hmc = (const void* const*)hm;
  const void* const* dpc = (const void* const*)dp.data();
  const void* const* dgc = (const void* const*)dg.data();
  const void* const* dmc = (const void* const*)dm.data();
  const size_t nu = p->units.size();
  for (size_t ui = 0; ui < nu; ++ui) {
    const Unit& u = p->units[ui];
    CUDA_TRY(copy(u, hpc, dpc, pes, true, p->h2d));
    CUDA_TRY(copy(u, hg, dgc, pes, true, p->h2d));
    CUDA_TRY(copy(u, hmc, dmc, 4, true, p->h2d));
    CUDA_TRY(cudaEventRecord(p->in_ev[ui], p->h2d));
  }
  for (size_t ui = 0; ui < nu; ++ui) {
    const Unit& u = p->units[ui];
    const GroupPlan& g = p->d.groups[u.g];
    CUDA_TRY(cudaStreamWaitEvent(s, p->in_ev[ui], 0));
    const cudaError_t e = enqueue_kernels(sub_args(make_args(p, g), g, u.i0, u.cnt), g, u.tc, k, s);
    if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    CUDA_TRY(cudaEventRecord(p->run_ev[ui], s));
    CUDA_TRY(cudaStreamWaitEvent(p->d2h, p->run_ev[ui], 0));
    CUDA_TRY(copy(u, hpc, dpc, pes, false, p->d2h));
    CUDA_TRY(copy(u, hmc, dmc, 4, false, p->d2h));
  }
  CUDA_TRY(cudaEventRecord(p->out_ev[0], p->d2h));
  CUDA_TRY(cudaStreamWaitEvent(s, p->out_ev[0], 0));
  CUDA_TRY(cudaStreamSynchronize(s));
  return MUON_OK;
}

}  // namespace

muon_status_t muon_step(muon_plan_t p, void* const* params, const void* const* grads,
                        float* const* momenta, float beta, float lr, float wd, int32_t ns_steps,
                        float a, float b, float c, void* stream) {
  const float coef[3] = {a, b, c};
  return step_impl(p, params, grads, momenta, beta, lr, wd, ns_steps, coef, 1, stream);
}

muon_status_t muon_step_schedule(muon_plan_t p, void* const* params, const void* const* grads,
                                 float* const* momenta, float beta, float lr, float wd,
                                 int32_t ns_steps, const float* coeffs, int32_t n_rows,
                                 void* stream) {
  return step_impl(p, params, grads, momenta, beta, lr, wd, ns_steps, coeffs, n_rows, stream);
}

muon_status_t muon_step_host(muon_plan_t p, void* const* hp, const void* const* hg,
                             float* const* hm, float beta, float lr, float wd, int32_t ns_steps,
                             float a, float b, float c, void* stream) {
  if (!p) return fail(MUON_ERR_INVALID_ARG, "plan is NULL");
  if (!(p->d.opt.flags & MUON_FLAG_HOST_STAGING))
    return fail(MUON_ERR_UNSUPPORTED, "plan was created without MUON_FLAG_HOST_STAGING");
  if (!hp || !hg || !hm) return fail(MUON_ERR_INVALID_ARG, "NULL pointer array");
  const int32_t np = (int32_t)p->d.param_E.size();
  for (int32_t i = 0; i < np; ++i)
    if (!hp[i] || !hg[i] || !hm[i])
      return fail(MUON_ERR_INVALID_ARG, "parameter %d has a NULL pointer", i);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaSetDevice(p->device));
  const size_t pes = p_esize(p);
  std::vector<void*> dp(np), dg(np);
  std::vector<float*> dm(np);
  for (int32_t i = 0; i < np; ++i) {
    dp[i] = p->stage_p + p->stage_off[i] * pes;
    dg[i] = p->stage_g + p->stage_off[i] * pes;
    dm[i] = p->stage_m + p->stage_off[i];
  }
  // one copy per run of parameters whose host buffers are back to back
  auto copy_runs = [&](auto host_at, auto dev_at, size_t es, cudaMemcpyKind kind) -> muon_status_t {
    int32_t i = 0;
    while (i < np) {
      int32_t j = i + 1;
      size_t bytes = (size_t)param_elems(p->d, i) * es;
      while (j < np && (const unsigned char*)host_at(j) == (const unsigned char*)host_at(i) + bytes &&
             (const unsigned char*)dev_at(j) == (const unsigned char*)dev_at(i) + bytes) {
        bytes += (size_t)param_elems(p->d, j) * es;
        ++j;
      }
      if (kind == cudaMemcpyHostToDevice)
        CUDA_TRY(cudaMemcpyAsync((void*)dev_at(i), host_at(i), bytes, kind, s));
      else
        CUDA_TRY(cudaMemcpyAsync((void*)host_at(i), dev_at(i), bytes, kind, s));
      i = j;
    }
    return MUON_OK;
  };
  muon_status_t st;
  if (all_skinny(p) && !p->in_ev.empty() && np > 1)
    return host_step_pipelined(p, hp, hg, hm, dp, dg, dm, beta, lr, wd, ns_steps, a, b, c, s);
  if (p->units.size() > 1 && p->in_ev.size() >= p->units.size())
    return host_step_units(p, hp, hg, hm, dp, dg, dm, beta, lr, wd, ns_steps, a, b, c, s);
  if ((st = copy_runs([&](int32_t i) { return (const void*)hp[i]; },
                      [&](int32_t i) { return (const void*)dp[i]; }, pes, cudaMemcpyHostToDevice)))
    return st;
  if ((st = copy_runs([&](int32_t i) { return (const void*)hg[i]; },
                      [&](int32_t i) { return (const void*)dg[i]; }, pes, cudaMemcpyHostToDevice)))
    return st;
  if ((st = copy_runs([&](int32_t i) { return (const void*)hm[i]; },
                      [&](int32_t i) { return (const void*)dm[i]; }, 4, cudaMemcpyHostToDevice)))
    return st;
  if ((st = muon_step(p, dp.data(), (const void* const*)dg.data(), dm.data(), beta, lr, wd,
                      ns_steps, a, b, c, stream)))
    return st;
  if ((st = copy_runs([&](int32_t i) { return (const void*)hp[i]; },
                      [&](int32_t i) { return (const void*)dp[i]; }, pes, cudaMemcpyDeviceToHost)))
    return st;
  if ((st = copy_runs([&](int32_t i) { return (const void*)hm[i]; },
                      [&](int32_t i) { return (const void*)dm[i]; }, 4, cudaMemcpyDeviceToHost)))
    return st;
  CUDA_TRY(cudaStreamSynchronize(s));
  return MUON_OK;
}

muon_status_t muon_plan_destroy(muon_plan_t p) {
  destroy_plan(p);
  return MUON_OK;
}

int32_t muon_plan_num_groups(muon_plan_t p) { return p ? (int32_t)p->d.groups.size() : 0; }

muon_status_t muon_plan_group_info(muon_plan_t p, int32_t g, muon_group_info_t* info) {
  if (!p || !info) return fail(MUON_ERR_INVALID_ARG, "NULL plan or info");
  if (g < 0 || g >= (int32_t)p->d.groups.size()) return fail(MUON_ERR_INVALID_ARG, "bad group %d", g);
  const GroupPlan& gp = p->d.groups[g];
  *info = muon_group_info_t{gp.rows, gp.cols, gp.batch, gp.first_member,
                            gp.transposed, gp.path, (int64_t)gp.ws_bytes};
  return MUON_OK;
}

size_t muon_plan_workspace_bytes(muon_plan_t p) { return p ? p->d.ws_bytes : 0; }

muon_status_t muon_debug_copy_update(muon_plan_t p, int32_t param_index, int64_t expert,
                                     float* dst) {
  if (!p || !dst) return fail(MUON_ERR_INVALID_ARG, "NULL plan or destination");
  if (!(p->d.opt.flags & MUON_FLAG_KEEP_UPDATE))
    return fail(MUON_ERR_UNSUPPORTED, "plan was created without MUON_FLAG_KEEP_UPDATE");
  if (param_index < 0 || param_index >= (int32_t)p->d.param_E.size() || expert < 0 ||
      expert >= p->d.param_E[param_index])
    return fail(MUON_ERR_INVALID_ARG, "bad (param, expert) = (%d, %lld)", param_index,
                (long long)expert);
  for (const GroupPlan& g : p->d.groups) {
    for (int64_t i = 0; i < g.batch; ++i) {
      const int64_t mi = g.first_member + i;
      if (p->d.member_param[mi] == param_index && p->d.member_expert[mi] == expert) {
        CUDA_TRY(cudaSetDevice(p->device));
        CUDA_TRY(cudaDeviceSynchronize());
        const size_t n = (size_t)g.rows * g.cols;
        CUDA_TRY(cudaMemcpy(dst, p->ws + g.base + g.off_dbg + i * n * 4, n * 4,
                            cudaMemcpyDeviceToHost));
        return MUON_OK;
      }
    }
  }
  return fail(MUON_ERR_INVALID_ARG, "member not found");
}

muon_status_t muon_plan_group_elapsed_ms(muon_plan_t p, int32_t g, float* ms) {
  if (!p || !ms) return fail(MUON_ERR_INVALID_ARG, "NULL plan or output");
  if (p->t_start.empty())
    return fail(MUON_ERR_UNSUPPORTED, "plan was created without MUON_FLAG_GROUP_TIMING");
  if (g < 0 || g >= (int32_t)p->d.groups.size()) return fail(MUON_ERR_INVALID_ARG, "bad group %d", g);
  CUDA_TRY(cudaEventSynchronize(p->t_stop[g]));
  CUDA_TRY(cudaEventElapsedTime(ms, p->t_start[g], p->t_stop[g]));
  return MUON_OK;
}

muon_status_t muon_plan_check_error(muon_plan_t p) {
  if (!p) return fail(MUON_ERR_INVALID_ARG, "plan is NULL");
  CUDA_TRY(cudaSetDevice(p->device));
  CUDA_TRY(cudaDeviceSynchronize());
  int w = 0;
  CUDA_TRY(cudaMemcpy(&w, p->ws + p->d.off_err, sizeof w, cudaMemcpyDeviceToHost));
  if (w != 0) {
    const int zero = 0;
    CUDA_TRY(cudaMemcpy(p->ws + p->d.off_err, &zero, sizeof zero, cudaMemcpyHostToDevice));
    return fail(MUON_ERR_TIMEOUT, "a kernel gave up a bounded wait (code 0x%x)", w);
  }
  return MUON_OK;
}

const char* muon_status_string(muon_status_t s) {
  switch (s) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG";
    case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED";
    case MUON_ERR_OOM: return "MUON_ERR_OOM";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT";
  }
  return "MUON_ERR_UNKNOWN";
}

const char* muon_last_error(void) { return g_last_error.c_str(); }

const char* muon_version(void) { return "0.1.0"; }

}  // extern "C"
