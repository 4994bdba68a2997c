// Host side of liblopt: the C ABI declared in include/lopt.h.
//
// Builds the ragged schedule of a parameter list (one descriptor per tensor,
// one unit table per kernel), keeps the device workspace, and enqueues the
// three launches of a step:
//   K0 rowcol  -- factored row/column second moments (all tensors)
//   K1 stats   -- features + per-feature sum of squares, folded layer-1 weights
//   K2 apply   -- features + normalise + MLP + update (FP32 or tensor cores)
// The page ("PyLO: Towards Accessible Learned Optimizers in PyTorch", section
// "メモリ階層の活用") counts 30-114 launches per step for a whole model with
// its two fused kernels per tensor; here the whole list takes three.
#include <algorithm>
#include <string>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "lopt.h"
#include "lopt_internal.cuh"

namespace lopt {
bool apply_fp32_supported(int hidden);
// k_probe.cu: one block that waits on a barrier nothing completes.
cudaError_t launch_wait_probe(int64_t limit_ns, int32_t* status, cudaStream_t s);

namespace {
// The last CUDA error a call of this thread failed on (lopt_last_cuda_error).
thread_local std::string g_last_cuda;
}  // namespace

int record_cuda_error(cudaError_t e) {
  g_last_cuda = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
  if (e == cudaErrorMemoryAllocation) return LOPT_E_OOM;
  return LOPT_E_CUDA;
}

// Rows per K0 strip.  About kStripTarget elements per strip, but no more
// than kFinalizeCap / cols strips (the last block of a tensor sums
// strips x cols column partials) -- unless strips would then exceed
// kMaxStripElems elements, since a very large tensor in a few huge strips
// leaves the launch waiting on a few blocks; then up to 4 x kFinalizeCap
// partials (1 MB, inside the no-allocation scratch) -- and no more than
// kMaxStripRows rows.
constexpr int64_t kMaxStripElems = 131072;
int strip_rows_for(int64_t R, int64_t C) {
  const int64_t N = R * C;
  const int64_t Cc = std::max<int64_t>(C, 1);
  int64_t strips = std::max<int64_t>(1, (N + kStripTarget - 1) / kStripTarget);
  const int64_t cap = std::max<int64_t>(kFinalizeCap / Cc,
                                        std::min<int64_t>((N + kMaxStripElems - 1) / kMaxStripElems, 4 * kFinalizeCap / Cc));
  strips = std::min<int64_t>(strips, std::max<int64_t>(1, cap));
  strips = std::min<int64_t>(strips, R);
  int64_t rows = (R + strips - 1) / strips;
  rows = std::min<int64_t>(rows, kMaxStripRows);
  return (int)std::max<int64_t>(rows, 1);
}
}  // namespace lopt

using namespace lopt;

struct HostPipe;

struct lopt_ctx {
  int device = 0;
  int hidden = 0;        // caller's width
  int hp = 0;            // padded width used by the kernels
  int n_sets = 0;
  int path = LOPT_MLP_FP32;
  float weight_decay = 0.f;
  float* d_weights = nullptr;  // [n_sets][w_set_size(hp)], zero-padded
  void* d_tcw = nullptr;       // packed FP16 layer-2/3 operands (tensor-core path)
  // workspace
  char* d_ws = nullptr;
  size_t ws_bytes = 0;
  // carved views (valid for the cached schedule)
  TensorDesc* d_desc = nullptr;
  Unit* d_units[3] = {nullptr, nullptr, nullptr};
  TensorAux* d_aux = nullptr;
  int32_t* d_counters = nullptr;   // [2][T]
  float* d_colpart = nullptr;
  double* d_rowpart = nullptr;
  float* d_k1part = nullptr;
  float* d_w1fold = nullptr;
  int32_t* d_status = nullptr;
  int w1fold_stride = 0;
  int n_units[3] = {0, 0, 0};
  int n_tensors = 0;
  // L2-sized groups (lopt_set_sweep_bytes): per group, the first unit and
  // the unit count of each kernel; empty: the whole list in one launch each
  int64_t sweep_bytes = 0;
  int64_t last_sweep = -1;
  struct Group {
    int first[3], count[3];
  };
  std::vector<Group> groups;
  // cached schedule key
  std::vector<lopt_tensor> last_list;
  std::vector<int64_t> last_grows;   // global rows of a row-sharded schedule (empty: plain)
  int last_path = -1;
  // row-sharded step in progress: 0 idle, 1 after begin, 2 after middle
  int shard_phase = 0;
  StepArgs shard_args;
  double* x1 = nullptr;
  double* x2 = nullptr;
  // ordering across calls
  cudaEvent_t done = nullptr;
  bool has_done = false;
  // host-buffer steps: one context per group of tensors, created on first use;
  // the parts share the parent's weights
  HostPipe* pipe = nullptr;
  bool shared_weights = false;
  int host_groups = 2;           // most groups of a host-buffer step (lopt_set_host_groups)
  // optional per-kernel timing: 4 events per timed step
  bool timing = false;
  std::vector<cudaEvent_t> tev;
  size_t tev_used = 0;
};

namespace {

int cuda_fail(cudaError_t e) { return lopt::record_cuda_error(e); }

int padded_hidden(int h) {
  for (int c : {4, 8, 16, 32, 64})
    if (h <= c) return c;
  return -1;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Interval {
  uintptr_t lo, hi;
};

// global_rows: null for a plain step; for a row-sharded step the rows of
// each whole tensor, and a rank may hold none of a tensor's rows.
int validate(const lopt_ctx* h, const lopt_tensor* ts, int n, const int64_t* global_rows = nullptr) {
  std::vector<Interval> iv;
  iv.reserve((size_t)n * 12);
  for (int i = 0; i < n; ++i) {
    const lopt_tensor& t = ts[i];
    if (t.reserved != 0) return LOPT_E_ARG;
    if (t.weight_set < 0 || t.weight_set >= h->n_sets) return LOPT_E_ARG;
    if (global_rows) {
      if (t.rows < 0 || t.cols < 1 || global_rows[i] < 1 || global_rows[i] < t.rows) return LOPT_E_SHAPE;
      if (global_rows[i] > (int64_t)1 << 40) return LOPT_E_SHAPE;
      if (t.rows == 0) {   // only the column accumulators on this rank
        for (int k = 0; k < 3; ++k) {
          if (!t.col[k]) return LOPT_E_ARG;
          if ((uintptr_t)t.col[k] % 4) return LOPT_E_ALIGN;
          iv.push_back({(uintptr_t)t.col[k], (uintptr_t)t.col[k] + (uintptr_t)t.cols * 4});
        }
        continue;
      }
    }
    if (t.rows < 1 || t.cols < 1) return LOPT_E_SHAPE;
    if (t.rows > (int64_t)1 << 31 || t.cols > (int64_t)1 << 31) return LOPT_E_SHAPE;
    const int64_t N = t.rows * t.cols;
    if (N >= ((int64_t)1 << 31)) return LOPT_E_SHAPE;
    const void* ep[6] = {t.param, t.grad, t.mom[0], t.mom[1], t.mom[2], t.rms};
    for (const void* p : ep) {
      if (!p) return LOPT_E_ARG;
      if ((uintptr_t)p % 4) return LOPT_E_ALIGN;
      iv.push_back({(uintptr_t)p, (uintptr_t)p + (uintptr_t)N * 4});
    }
    for (int k = 0; k < 3; ++k) {
      if (!t.row[k] || !t.col[k]) return LOPT_E_ARG;
      if ((uintptr_t)t.row[k] % 4 || (uintptr_t)t.col[k] % 4) return LOPT_E_ALIGN;
      iv.push_back({(uintptr_t)t.row[k], (uintptr_t)t.row[k] + (uintptr_t)t.rows * 4});
      iv.push_back({(uintptr_t)t.col[k], (uintptr_t)t.col[k] + (uintptr_t)t.cols * 4});
    }
  }
  std::sort(iv.begin(), iv.end(), [](const Interval& a, const Interval& b) { return a.lo < b.lo; });
  for (size_t k = 1; k < iv.size(); ++k)
    if (iv[k].lo < iv[k - 1].hi) return LOPT_E_ALIAS;
  return LOPT_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

// The host half of a schedule: one descriptor per tensor, the unit table of
// each kernel in launch order, the L2-sized groups, and the sizes of the
// partial-sum areas.  No device call; the pointers are not dereferenced.
struct Plan {
  std::vector<TensorDesc> desc;
  std::vector<Unit> units[3];
  std::vector<lopt_ctx::Group> groups;
  int64_t colpart = 0, rowpart = 0, k1part = 0;
};

int plan_schedule(const lopt_tensor* ts, int n, int64_t sweep_bytes, const int64_t* global_rows, Plan& pl) {
  std::vector<TensorDesc>& desc = pl.desc;
  std::vector<Unit>* units = pl.units;
  desc.assign(n, TensorDesc{});
  int64_t colpart = 0, rowpart = 0, k1part = 0, x1 = 0;
  for (int i = 0; i < n; ++i) {
    const lopt_tensor& t = ts[i];
    TensorDesc& d = desc[i];
    std::memset(&d, 0, sizeof(d));
    d.p = t.param;
    d.g = t.grad;
    for (int k = 0; k < 3; ++k) {
      d.m[k] = t.mom[k];
      d.r[k] = t.row[k];
      d.c[k] = t.col[k];
    }
    d.v = t.rms;
    d.R = t.rows;
    d.C = t.cols;
    d.N = t.rows * t.cols;
    d.wset = t.weight_set;
    bool v4 = aligned16(t.param) && aligned16(t.grad) && aligned16(t.rms);
    for (int k = 0; k < 3; ++k) v4 = v4 && aligned16(t.mom[k]) && aligned16(t.col[k]);
    d.vec4 = v4 ? 1 : 0;
    d.Rg = global_rows ? global_rows[i] : d.R;
    d.x1_off = x1;
    x1 += d.C + 3;
    d.strip_rows = d.R > 0 ? strip_rows_for(d.R, d.C) : 1;
    d.n_strips = (int)((d.R + d.strip_rows - 1) / d.strip_rows);
    d.k1_units = (int)((d.N + kStatsChunk - 1) / kStatsChunk);
    d.k2_units = (int)((d.N + kApplyChunk - 1) / kApplyChunk);
    colpart = (colpart + 3) / 4 * 4;   // 16-byte aligned start for float4 reads
    d.colpart_off = colpart;
    colpart += (int64_t)d.n_strips * d.C;
    d.rowpart_off = (int32_t)rowpart;
    rowpart += 3 * (int64_t)d.n_strips;
    d.k1_part_off = (int32_t)k1part;
    k1part += (int64_t)kStats * d.k1_units;
    if (rowpart > INT32_MAX || k1part > INT32_MAX) return LOPT_E_SHAPE;
    for (int s = 0; s < d.n_strips; ++s) units[0].push_back({i, s});
    for (int s = 0; s < d.k1_units; ++s) units[1].push_back({i, s});
    for (int s = 0; s < d.k2_units; ++s) units[2].push_back({i, s});
  }
  pl.colpart = colpart;
  pl.rowpart = rowpart;
  pl.k1part = k1part;
  // L2-sized groups: consecutive tensors whose state (p, g, m0..2, v: 24
  // bytes per element) fits in sweep_bytes; a larger tensor is a group of
  // its own.  The units of every kernel are in tensor order here.
  std::vector<lopt_ctx::Group>& groups = pl.groups;
  groups.clear();
  if (sweep_bytes > 0 && !global_rows) {
    int64_t bytes = 0;
    int first[3] = {0, 0, 0}, end[3] = {0, 0, 0};
    for (int i = 0; i < n; ++i) {
      const int64_t b = 24 * desc[i].N;
      if (i > 0 && bytes + b > sweep_bytes) {
        groups.push_back({{first[0], first[1], first[2]},
                          {end[0] - first[0], end[1] - first[1], end[2] - first[2]}});
        for (int k = 0; k < 3; ++k) first[k] = end[k];
        bytes = 0;
      }
      bytes += b;
      end[0] += desc[i].n_strips;
      end[1] += desc[i].k1_units;
      end[2] += desc[i].k2_units;
    }
    groups.push_back({{first[0], first[1], first[2]},
                      {end[0] - first[0], end[1] - first[1], end[2] - first[2]}});
  }
  // K0 blocks are dispatched about in unit order: the largest strips first
  // (whose tensors also have the longest column finalisation), so that the
  // launch ends on small strips -- within each group when there are groups.
  // Results do not depend on this order.
  auto by_strip = [&](const Unit& x, const Unit& y) {
    const TensorDesc& a = desc[x.tensor];
    const TensorDesc& b = desc[y.tensor];
    return (int64_t)a.strip_rows * a.C > (int64_t)b.strip_rows * b.C;
  };
  // K1 blocks likewise take the largest tensors first: the last block of a
  // tensor sums its partials, and a large tensor's sum at the end of the
  // launch would be its tail.
  auto by_size = [&](const Unit& x, const Unit& y) { return desc[x.tensor].N > desc[y.tensor].N; };
  if (groups.empty()) {
    std::stable_sort(units[0].begin(), units[0].end(), by_strip);
    std::stable_sort(units[1].begin(), units[1].end(), by_size);
  } else {
    for (const auto& g : groups) {
      std::stable_sort(units[0].begin() + g.first[0], units[0].begin() + g.first[0] + g.count[0], by_strip);
      std::stable_sort(units[1].begin() + g.first[1], units[1].begin() + g.first[1] + g.count[1], by_size);
    }
  }
  return LOPT_OK;
}

int build_schedule(lopt_ctx* h, const lopt_tensor* ts, int n, cudaStream_t stream,
                   const int64_t* global_rows = nullptr) {
  Plan pl;
  const int prc = plan_schedule(ts, n, h->sweep_bytes, global_rows, pl);
  if (prc != LOPT_OK) return prc;
  const std::vector<TensorDesc>& desc = pl.desc;
  const std::vector<Unit>* units = pl.units;
  const int64_t colpart = pl.colpart, rowpart = pl.rowpart, k1part = pl.k1part;
  h->w1fold_stride = w1fold_floats(h->hp, h->path);
  h->groups = pl.groups;

  // carve the workspace
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t o_desc = take(sizeof(TensorDesc) * n);
  size_t o_units[3];
  for (int k = 0; k < 3; ++k) o_units[k] = take(sizeof(Unit) * units[k].size());
  const size_t o_aux = take(sizeof(TensorAux) * n);
  const size_t o_cnt = take(sizeof(int32_t) * 2 * n);
  const size_t o_col = take(sizeof(float) * colpart);
  const size_t o_row = take(sizeof(double) * rowpart);
  const size_t o_k1 = take(sizeof(float) * k1part);
  const size_t o_w1 = take(sizeof(float) * (size_t)h->w1fold_stride * n);
  const size_t o_st = take(sizeof(int32_t) * 4);
  const size_t need = off;

  if (need > h->ws_bytes) {
    // the previous step may still be reading the old workspace
    if (h->has_done) cudaEventSynchronize(h->done);
    if (h->d_ws) cudaFree(h->d_ws);
    h->d_ws = nullptr;
    h->ws_bytes = 0;
    cudaError_t e = cudaMalloc(&h->d_ws, need);
    if (e != cudaSuccess) {
      cudaGetLastError();
      h->d_ws = nullptr;
      h->last_list.clear();
      return LOPT_E_OOM;
    }
    h->ws_bytes = need;
    e = cudaMemsetAsync(h->d_ws, 0, need, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  } else {
    // counters and status must start at zero for a new layout
    cudaError_t e = cudaMemsetAsync(h->d_ws + o_cnt, 0, sizeof(int32_t) * 2 * n, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemsetAsync(h->d_ws + o_st, 0, sizeof(int32_t) * 4, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  h->d_desc = reinterpret_cast<TensorDesc*>(h->d_ws + o_desc);
  for (int k = 0; k < 3; ++k) h->d_units[k] = reinterpret_cast<Unit*>(h->d_ws + o_units[k]);
  h->d_aux = reinterpret_cast<TensorAux*>(h->d_ws + o_aux);
  h->d_counters = reinterpret_cast<int32_t*>(h->d_ws + o_cnt);
  h->d_colpart = reinterpret_cast<float*>(h->d_ws + o_col);
  h->d_rowpart = reinterpret_cast<double*>(h->d_ws + o_row);
  h->d_k1part = reinterpret_cast<float*>(h->d_ws + o_k1);
  h->d_w1fold = reinterpret_cast<float*>(h->d_ws + o_w1);
  h->d_status = reinterpret_cast<int32_t*>(h->d_ws + o_st);

  // Pageable host sources: the runtime stages them before returning, so the
  // vectors may die right after the calls.
  cudaError_t e = cudaMemcpyAsync(h->d_desc, desc.data(), sizeof(TensorDesc) * n,
                                  cudaMemcpyHostToDevice, stream);
  for (int k = 0; k < 3 && e == cudaSuccess; ++k) {
    if (!units[k].empty())
      e = cudaMemcpyAsync(h->d_units[k], units[k].data(), sizeof(Unit) * units[k].size(),
                          cudaMemcpyHostToDevice, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  for (int k = 0; k < 3; ++k) h->n_units[k] = (int)units[k].size();
  h->n_tensors = n;
  h->last_list.assign(ts, ts + n);
  if (global_rows) h->last_grows.assign(global_rows, global_rows + n);
  else h->last_grows.clear();
  h->last_path = h->path;
  h->last_sweep = h->sweep_bytes;
  return LOPT_OK;
}

// Row-sharded exchange sizes: buffer 1 holds C + 3 doubles per tensor,
// buffer 2 holds 28.
void shard_counts(const lopt_tensor* ts, int n, int64_t* n1, int64_t* n2) {
  int64_t a = 0;
  for (int i = 0; i < n; ++i) a += ts[i].cols + 3;
  *n1 = a;
  *n2 = (int64_t)kStats * n;
}

}  // namespace

namespace {

// Device, ordering and the common launch arguments of one sharded phase.
struct PhaseScope {
  int prev = -1, want = 0;
  ~PhaseScope() { if (prev >= 0 && prev != want) cudaSetDevice(prev); }
};

int enter_phase(lopt_ctx* h, cudaStream_t stream, PhaseScope& sc) {
  cudaError_t e = cudaGetDevice(&sc.prev);
  if (e != cudaSuccess) return cuda_fail(e);
  sc.want = h->device;
  if (sc.prev != h->device && (e = cudaSetDevice(h->device)) != cudaSuccess) return cuda_fail(e);
  if (h->has_done && (e = cudaStreamWaitEvent(stream, h->done, 0)) != cudaSuccess) return cuda_fail(e);
  return LOPT_OK;
}

int leave_phase(lopt_ctx* h, cudaStream_t stream, cudaError_t e) {
  if (e == cudaSuccess) e = cudaEventRecord(h->done, stream);
  if (e != cudaSuccess) {
    h->shard_phase = 0;
    h->last_list.clear();
    return cuda_fail(e);
  }
  h->has_done = true;
  return LOPT_OK;
}

}  // namespace

// ---- host-buffer steps ------------------------------------------------------
constexpr int kHostGroupsMax = 16;             // most groups of tensors per step
constexpr int64_t kHostGroupElems = 1 << 22;   // fewest elements per group

// Consecutive calls alternate between two device staging buffers for the
// gradients, so that the gradient copies of one call can run while the
// kernels of the previous call still read the other buffer.
struct HostPipe {
  std::vector<lopt_ctx*> parts[2];      // per staging buffer, one context per group
  std::vector<int> split;               // group g: tensors [split[g], split[g + 1])
  std::vector<lopt_tensor> list;        // the caller's list the set-up was made for
  std::vector<lopt_tensor> staged[2];   // the same list reading its gradients from buffer q
  float* stage[2] = {nullptr, nullptr};
  size_t stage_floats = 0;
  int q = 0;                            // staging buffer of the next call
  bool any = false;                     // a host-buffer step has been enqueued
  cudaStream_t h2d = nullptr, d2h = nullptr;
  // per group: gradients in (per buffer), kernels done (per buffer), parameters out
  std::vector<cudaEvent_t> ev;
  cudaEvent_t d2h_done = nullptr;       // after the last parameter copy issued
};
constexpr int kGroupEvents = 5;

namespace {

// Consecutive groups of about equal element counts: up to max_groups, at
// least kHostGroupElems elements each (one group for a small list), at
// least one tensor each.
void split_groups(const lopt_tensor* ts, int n, int max_groups, std::vector<int>& split) {
  int64_t total = 0;
  for (int i = 0; i < n; ++i) total += ts[i].rows * ts[i].cols;
  int G = (int)std::min<int64_t>(max_groups, std::max<int64_t>(1, total / kHostGroupElems));
  G = std::min(G, n);
  split.assign(1, 0);
  int64_t acc = 0;
  for (int i = 0; i + 1 < n; ++i) {
    acc += ts[i].rows * ts[i].cols;
    const int g = (int)split.size();   // the boundary that closes group g - 1
    if (g < G && acc * G >= total * g && n - (i + 1) >= G - g) split.push_back(i + 1);
  }
  split.push_back(n);
}

// A context for one group: the parent's weights, its own workspace.
lopt_ctx* make_part(const lopt_ctx* h) {
  lopt_ctx* c = new (std::nothrow) lopt_ctx();
  if (!c) return nullptr;
  c->device = h->device;
  c->hidden = h->hidden;
  c->hp = h->hp;
  c->n_sets = h->n_sets;
  c->d_weights = h->d_weights;
  c->d_tcw = h->d_tcw;
  c->shared_weights = true;
  if (cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return nullptr;
  }
  return c;
}

void destroy_pipe(HostPipe* p);

// Work that reads or writes the device parameters waits for the host-buffer
// steps' parameter copies still in flight.
cudaError_t wait_host_copies(const lopt_ctx* h, cudaStream_t stream) {
  if (!h->pipe || !h->pipe->any) return cudaSuccess;
  return cudaStreamWaitEvent(stream, h->pipe->d2h_done, 0);
}

}  // namespace

extern "C" {

int lopt_version(void) { return 100; }

const char* lopt_last_cuda_error(void) { return g_last_cuda.c_str(); }

const char* lopt_strerror(int code) {
  switch (code) {
    case LOPT_OK: return "ok";
    case LOPT_E_ARG: return "invalid argument";
    case LOPT_E_SHAPE: return "invalid tensor shape";
    case LOPT_E_ALIGN: return "misaligned tensor pointer";
    case LOPT_E_CUDA: return "CUDA runtime error";
    case LOPT_E_OOM: return "device allocation failed";
    case LOPT_E_UNSUPPORTED: return "unsupported configuration";
    case LOPT_E_TIMEOUT: return "device-side wait timed out";
    case LOPT_E_ALIAS: return "tensor buffers overlap";
    case LOPT_E_TOO_LARGE: return "tensor needs more scratch than the static no-allocation buffer";
    default: return "unknown error";
  }
}

int lopt_weight_set_size(int d_feat, int hidden) {
  if (d_feat != LOPT_D_FEAT || hidden < 1 || hidden > LOPT_MAX_HIDDEN) return LOPT_E_ARG;
  return d_feat * hidden + hidden + hidden * hidden + hidden + 2 * hidden + 2;
}

int lopt_create(const float* mlp_weights, int d_feat, int hidden, int n_sets, lopt_handle* out) {
  if (!out) return LOPT_E_ARG;
  *out = nullptr;
  if (!mlp_weights || n_sets < 1 || d_feat != LOPT_D_FEAT) return LOPT_E_ARG;
  if (hidden < 1 || hidden > LOPT_MAX_HIDDEN) return LOPT_E_UNSUPPORTED;
  const int hp = padded_hidden(hidden);
  if (hp < 0 || !apply_fp32_supported(hp)) return LOPT_E_UNSUPPORTED;

  // Re-lay the caller's sets at the padded width (extra units get zero
  // weights and zero biases, so they contribute exactly nothing).
  const int H = hidden, src_sz = lopt_weight_set_size(d_feat, hidden), dst_sz = w_set_size(hp);
  std::vector<float> packed((size_t)n_sets * dst_sz, 0.f);
  for (int s = 0; s < n_sets; ++s) {
    const float* src = mlp_weights + (size_t)s * src_sz;
    float* dst = packed.data() + (size_t)s * dst_sz;
    for (int dd = 0; dd < kDFeat; ++dd)
      for (int x = 0; x < H; ++x) dst[w_off_W1(hp) + dd * hp + x] = src[dd * H + x];
    for (int x = 0; x < H; ++x) dst[w_off_b1(hp) + x] = src[kDFeat * H + x];
    for (int a = 0; a < H; ++a)
      for (int x = 0; x < H; ++x) dst[w_off_W2(hp) + a * hp + x] = src[kDFeat * H + H + a * H + x];
    for (int x = 0; x < H; ++x) dst[w_off_b2(hp) + x] = src[kDFeat * H + H + H * H + x];
    for (int a = 0; a < H; ++a)
      for (int q = 0; q < 2; ++q) dst[w_off_W3(hp) + 2 * a + q] = src[kDFeat * H + 2 * H + H * H + 2 * a + q];
    for (int q = 0; q < 2; ++q) dst[w_off_b3(hp) + q] = src[kDFeat * H + 4 * H + H * H + q];
  }

  lopt_ctx* h = new (std::nothrow) lopt_ctx();
  if (!h) return LOPT_E_OOM;
  h->hidden = hidden;
  h->hp = hp;
  h->n_sets = n_sets;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaMalloc(&h->d_weights, packed.size() * sizeof(float));
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_weights, packed.data(), packed.size() * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->done, cudaEventDisableTiming);
  if (e == cudaSuccess && apply_tc_supported(hp)) {
    e = cudaMalloc(&h->d_tcw, tc_weights_bytes(hp, n_sets));
    if (e == cudaSuccess) e = pack_tc_weights(h->d_weights, hp, n_sets, h->d_tcw, 0);
    if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (h->d_tcw) cudaFree(h->d_tcw);
    if (h->d_weights) cudaFree(h->d_weights);
    if (h->done) cudaEventDestroy(h->done);
    delete h;
    return cuda_fail(e);
  }
  *out = h;
  return LOPT_OK;
}

int lopt_set_mlp_path(lopt_handle h, int path) {
  if (!h) return LOPT_E_ARG;
  if (path == LOPT_MLP_FP32) {
    h->path = path;
    return LOPT_OK;
  }
  if (path == LOPT_MLP_TC) {
    if (!apply_tc_supported(h->hp) || !h->d_tcw) return LOPT_E_UNSUPPORTED;
    h->path = path;
    return LOPT_OK;
  }
  return LOPT_E_ARG;
}

int lopt_selftest_wait(int64_t limit_ns) {
  if (limit_ns <= 0 || limit_ns > 1000000000) return LOPT_E_ARG;
  int32_t* d_status = nullptr;
  cudaError_t e = cudaMalloc(&d_status, sizeof(int32_t));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return LOPT_E_OOM;
  }
  int32_t status = 0;
  e = cudaMemset(d_status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = launch_wait_probe(limit_ns, d_status, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&status, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  cudaFree(d_status);
  if (e != cudaSuccess) return cuda_fail(e);
  return (status & kStatusTimeout) ? LOPT_E_TIMEOUT : LOPT_OK;
}

int lopt_set_sweep_bytes(lopt_handle h, int64_t group_bytes) {
  if (!h || group_bytes < 0) return LOPT_E_ARG;
  h->sweep_bytes = group_bytes;   // a changed setting rebuilds the schedule on the next step
  return LOPT_OK;
}

int lopt_set_weight_decay(lopt_handle h, float weight_decay) {
  if (!h || !(weight_decay >= 0.f) || !std::isfinite(weight_decay)) return LOPT_E_ARG;
  h->weight_decay = weight_decay;
  return LOPT_OK;
}

int lopt_step(lopt_handle h, const lopt_tensor* tensors, int n_tensors, int64_t t, float lr,
              void* stream_ptr) {
  if (!h || n_tensors < 0 || (n_tensors > 0 && !tensors)) return LOPT_E_ARG;
  if (t < 1) return LOPT_E_ARG;
  if (n_tensors == 0) return LOPT_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);

  if (h->shard_phase != 0) return LOPT_E_ARG;   // a row-sharded step is in progress
  const bool same = h->last_path == h->path && h->last_grows.empty() && h->last_sweep == h->sweep_bytes &&
                    (int)h->last_list.size() == n_tensors &&
                    std::memcmp(h->last_list.data(), tensors, sizeof(lopt_tensor) * n_tensors) == 0;
  if (!same) {
    int rc = validate(h, tensors, n_tensors);
    if (rc != LOPT_OK) return rc;
  }
  int prev_device = -1;
  cudaError_t e = cudaGetDevice(&prev_device);
  if (e != cudaSuccess) return cuda_fail(e);
  if (prev_device != h->device) {
    e = cudaSetDevice(h->device);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  struct Restore {
    int dev, want;
    ~Restore() { if (dev >= 0 && dev != want) cudaSetDevice(dev); }
  } restore{prev_device, h->device};
  if (h->has_done) {
    e = cudaStreamWaitEvent(stream, h->done, 0);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  e = wait_host_copies(h, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (!same) {
    int rc = build_schedule(h, tensors, n_tensors, stream);
    if (rc != LOPT_OK) {
      h->last_list.clear();
      return rc;
    }
  }

  StepArgs a;
  std::memset(&a, 0, sizeof(a));
  a.desc = h->d_desc;
  a.hidden = h->hp;
  a.aux = h->d_aux;
  a.colpart = h->d_colpart;
  a.rowpart = h->d_rowpart;
  a.k1part = h->d_k1part;
  a.weights = h->d_weights;
  a.set_size = w_set_size(h->hp);
  a.w1fold = h->d_w1fold;
  a.w1fold_stride = h->w1fold_stride;
  a.path = h->path;
  a.tc_weights = h->d_tcw;
  a.t = (double)t;
  for (int k = 0; k < kTimeFeat; ++k) a.tau[k] = std::tanh((double)t / time_scale(k));
  a.lr = lr;
  a.wd = h->weight_decay;
  a.status = h->d_status;

  // One launch of each kernel over the whole list, or, with L2-sized groups,
  // the three launches per group, group after group.
  const int n_groups = h->groups.empty() ? 1 : (int)h->groups.size();
  for (int gi = 0; gi < n_groups && e == cudaSuccess; ++gi) {
    int first[3] = {0, 0, 0}, count[3] = {h->n_units[0], h->n_units[1], h->n_units[2]};
    if (!h->groups.empty()) {
      for (int k = 0; k < 3; ++k) {
        first[k] = h->groups[gi].first[k];
        count[k] = h->groups[gi].count[k];
      }
    }
    cudaEvent_t* ev = nullptr;   // kernel timing: 4 events per group
    if (h->timing) {
      if (h->tev_used + 4 > h->tev.size()) {
        for (int k = 0; k < 4; ++k) {
          cudaEvent_t x;
          e = cudaEventCreate(&x);
          if (e != cudaSuccess) return cuda_fail(e);
          h->tev.push_back(x);
        }
      }
      ev = h->tev.data() + h->tev_used;
      h->tev_used += 4;
    }
    auto mark = [&](int k) {
      if (ev && e == cudaSuccess) e = cudaEventRecord(ev[k], stream);
    };

    mark(0);
    a.units = h->d_units[0] + first[0];
    a.n_units = count[0];
    a.counters = h->d_counters;
    if (e == cudaSuccess) e = launch_rowcol(a, stream);
    mark(1);
    if (e == cudaSuccess) {
      a.units = h->d_units[1] + first[1];
      a.n_units = count[1];
      a.counters = h->d_counters + n_tensors;
      e = launch_stats(a, stream);
    }
    mark(2);
    if (e == cudaSuccess) {
      a.units = h->d_units[2] + first[2];
      a.n_units = count[2];
      a.counters = nullptr;
      e = (h->path == LOPT_MLP_TC) ? launch_apply_tc(a, stream) : launch_apply_fp32(a, stream);
    }
    mark(3);
  }
  if (e != cudaSuccess) {
    h->last_list.clear();
    return cuda_fail(e);
  }
  e = cudaEventRecord(h->done, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  h->has_done = true;
  return LOPT_OK;
}

int lopt_step_host(lopt_handle h, const lopt_tensor* tensors, int n_tensors, const float* const* grad_host,
                   float* const* param_host, int64_t t, float lr, void* stream_ptr) {
  if (!h || n_tensors < 0 || (n_tensors > 0 && (!tensors || !grad_host || !param_host))) return LOPT_E_ARG;
  if (t < 1 || h->shard_phase != 0 || h->shared_weights) return LOPT_E_ARG;
  for (int i = 0; i < n_tensors; ++i)
    if (tensors[i].rows * tensors[i].cols > 0 && (!grad_host[i] || !param_host[i])) return LOPT_E_ARG;
  if (n_tensors == 0) return LOPT_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);

  PhaseScope sc;
  int rc = enter_phase(h, stream, sc);
  if (rc != LOPT_OK) return rc;
  cudaError_t e = cudaSuccess;
  HostPipe* p = h->pipe;
  if (!p) {
    p = h->pipe = new (std::nothrow) HostPipe();
    if (!p) return LOPT_E_OOM;
    e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->d2h_done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      destroy_pipe(p);
      h->pipe = nullptr;
      return cuda_fail(e);
    }
  }
  const bool same = (int)p->list.size() == n_tensors &&
                    std::memcmp(p->list.data(), tensors, sizeof(lopt_tensor) * n_tensors) == 0;
  if (!same) {
    // a new list: earlier host-buffer steps must be done with the buffers
    p->list.clear();
    if (p->any && (e = cudaEventSynchronize(p->d2h_done)) != cudaSuccess) return cuda_fail(e);
    if (h->has_done && (e = cudaEventSynchronize(h->done)) != cudaSuccess) return cuda_fail(e);
    std::vector<size_t> off((size_t)n_tensors);
    size_t need = 0;
    for (int i = 0; i < n_tensors; ++i) {
      off[i] = need;
      need += ((size_t)(tensors[i].rows * tensors[i].cols) + 3) / 4 * 4;   // 16-byte aligned starts
    }
    need = std::max<size_t>(need, 4);
    if (need > p->stage_floats) {
      for (int q = 0; q < 2; ++q) {
        if (p->stage[q]) cudaFree(p->stage[q]);
        p->stage[q] = nullptr;
      }
      p->stage_floats = 0;
      for (int q = 0; q < 2; ++q) {
        if ((e = cudaMalloc(&p->stage[q], need * sizeof(float))) != cudaSuccess) {
          cudaGetLastError();
          return LOPT_E_OOM;
        }
      }
      p->stage_floats = need;
    }
    for (int q = 0; q < 2; ++q) {
      p->staged[q].assign(tensors, tensors + n_tensors);
      for (int i = 0; i < n_tensors; ++i) p->staged[q][i].grad = p->stage[q] + off[i];
      if ((rc = validate(h, p->staged[q].data(), n_tensors)) != LOPT_OK) return rc;
    }
    split_groups(tensors, n_tensors, h->host_groups, p->split);
    const int G = (int)p->split.size() - 1;
    for (int q = 0; q < 2; ++q) {
      while ((int)p->parts[q].size() < G) {
        lopt_ctx* c = make_part(h);
        if (!c) return LOPT_E_OOM;
        p->parts[q].push_back(c);
      }
    }
    while ((int)p->ev.size() < kGroupEvents * G) {
      cudaEvent_t x;
      if ((e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
      p->ev.push_back(x);
      // recorded once with nothing before it, so that the first waits on it pass
      if ((e = cudaEventRecord(x, p->h2d)) != cudaSuccess) return cuda_fail(e);
    }
    p->q = 0;
    p->list.assign(tensors, tensors + n_tensors);
  }
  const int G = (int)p->split.size() - 1;
  const int q = p->q;
  const lopt_tensor* const st = p->staged[q].data();
  // One copy per run of tensors that follow each other without a gap on
  // both sides (as in flat parameter buffers), else one per tensor.  Two
  // buffers can also touch by chance while being separate allocations; the
  // runtime refuses a copy across them (invalid value, before anything is
  // enqueued), and that run then goes tensor by tensor.
  auto copy_runs = [&](int i0, int i1, auto dst_of, auto src_of, cudaMemcpyKind kind, cudaStream_t cs) {
    cudaError_t err = cudaSuccess;
    float* dst = nullptr;
    const float* src = nullptr;
    size_t n = 0;
    int r0 = i0;   // first tensor of the run
    auto flush = [&](int r1) {
      if (!n) return cudaSuccess;
      cudaError_t x = cudaMemcpyAsync(dst, src, n * sizeof(float), kind, cs);
      if (x != cudaErrorInvalidValue || r1 - r0 < 2) return x;
      cudaGetLastError();
      x = cudaSuccess;
      for (int j = r0; j < r1 && x == cudaSuccess; ++j) {
        const size_t k = (size_t)(tensors[j].rows * tensors[j].cols);
        if (k) x = cudaMemcpyAsync(dst_of(j), src_of(j), k * sizeof(float), kind, cs);
      }
      return x;
    };
    for (int i = i0; i <= i1 && err == cudaSuccess; ++i) {
      const size_t k = i < i1 ? (size_t)(tensors[i].rows * tensors[i].cols) : 0;
      if (i < i1 && k == 0) continue;
      if (i < i1 && n && dst_of(i) == dst + n && src_of(i) == src + n) {
        n += k;
        continue;
      }
      err = flush(i);
      if (i < i1) {
        dst = dst_of(i);
        src = src_of(i);
        n = k;
        r0 = i;
      }
    }
    return err;
  };

  for (int g = 0; g < G && e == cudaSuccess; ++g) {
    const int i0 = p->split[g], i1 = p->split[g + 1];
    cudaEvent_t* ev = p->ev.data() + kGroupEvents * g;   // in[0..1], kernels[2..3], out[4]
    // gradients into staging buffer q once the kernels of the call before the
    // previous one (the last to read it) are done with this group
    e = cudaStreamWaitEvent(p->h2d, ev[2 + q], 0);
    if (e == cudaSuccess)
      e = copy_runs(i0, i1, [&](int i) { return const_cast<float*>(st[i].grad); },
                    [&](int i) { return const_cast<float*>(grad_host[i]); }, cudaMemcpyHostToDevice, p->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(ev[0 + q], p->h2d);
    // the kernels: after the gradients, and after the previous call's
    // parameter copies of this group (they read what the kernels overwrite)
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev[0 + q], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev[4], 0);
    if (e != cudaSuccess) break;
    lopt_ctx* c = p->parts[q][g];
    c->path = h->path;
    c->weight_decay = h->weight_decay;
    rc = lopt_step(c, st + i0, i1 - i0, t, lr, stream);
    if (rc != LOPT_OK) return rc;
    e = cudaEventRecord(ev[2 + q], stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->d2h, ev[2 + q], 0);
    if (e == cudaSuccess)
      e = copy_runs(i0, i1, [&](int i) { return param_host[i]; }, [&](int i) { return tensors[i].param; },
                    cudaMemcpyDeviceToHost, p->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(ev[4], p->d2h);
  }
  if (e == cudaSuccess) e = cudaEventRecord(p->d2h_done, p->d2h);
  if (e == cudaSuccess) {
    p->q ^= 1;
    p->any = true;
  }
  return leave_phase(h, stream, e);
}

int lopt_set_host_groups(lopt_handle h, int max_groups) {
  if (!h || max_groups < 1 || max_groups > kHostGroupsMax || h->shared_weights) return LOPT_E_ARG;
  if (max_groups != h->host_groups) {
    h->host_groups = max_groups;
    if (h->pipe) h->pipe->list.clear();   // split again on the next call
  }
  return LOPT_OK;
}

int lopt_host_sync(lopt_handle h, void* stream_ptr) {
  if (!h) return LOPT_E_ARG;
  if (!h->pipe || !h->pipe->any) return LOPT_OK;
  PhaseScope sc;
  int rc = enter_phase(h, reinterpret_cast<cudaStream_t>(stream_ptr), sc);
  if (rc != LOPT_OK) return rc;
  const cudaError_t e = cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream_ptr), h->pipe->d2h_done, 0);
  return e == cudaSuccess ? LOPT_OK : cuda_fail(e);
}

int lopt_shard_sizes(const lopt_tensor* tensors, int n_tensors, int64_t* n_x1, int64_t* n_x2) {
  if (n_tensors < 0 || (n_tensors > 0 && !tensors) || !n_x1 || !n_x2) return LOPT_E_ARG;
  shard_counts(tensors, n_tensors, n_x1, n_x2);
  return LOPT_OK;
}

int lopt_schedule_info(const lopt_tensor* tensors, int n_tensors, int64_t sweep_bytes,
                       int32_t* n_units, int32_t* units, int32_t* strip_rows,
                       int32_t* n_groups, int32_t* groups) {
  if (n_tensors < 0 || (n_tensors > 0 && !tensors) || !n_units || !n_groups || sweep_bytes < 0)
    return LOPT_E_ARG;
  for (int i = 0; i < n_tensors; ++i) {   // lopt_step's shape rules
    const lopt_tensor& t = tensors[i];
    if (t.reserved != 0) return LOPT_E_ARG;
    if (t.rows < 1 || t.cols < 1) return LOPT_E_SHAPE;
    if (t.rows > (int64_t)1 << 31 || t.cols > (int64_t)1 << 31) return LOPT_E_SHAPE;
    if (t.rows * t.cols >= ((int64_t)1 << 31)) return LOPT_E_SHAPE;
  }
  Plan pl;
  try {
    const int rc = plan_schedule(tensors, n_tensors, sweep_bytes, nullptr, pl);
    if (rc != LOPT_OK) return rc;
  } catch (const std::bad_alloc&) {
    return LOPT_E_OOM;
  }
  for (int k = 0; k < 3; ++k) {
    if (pl.units[k].size() > (size_t)INT32_MAX) return LOPT_E_SHAPE;
    n_units[k] = (int32_t)pl.units[k].size();
  }
  if (units) {
    int64_t o = 0;
    for (int k = 0; k < 3; ++k)
      for (const Unit& u : pl.units[k]) {
        units[2 * o] = u.tensor;
        units[2 * o + 1] = u.local;
        ++o;
      }
  }
  if (strip_rows)
    for (int i = 0; i < n_tensors; ++i) strip_rows[i] = pl.desc[i].strip_rows;
  *n_groups = (int32_t)pl.groups.size();
  if (groups)
    for (size_t gi = 0; gi < pl.groups.size(); ++gi)
      for (int k = 0; k < 3; ++k) {
        groups[6 * gi + 2 * k] = pl.groups[gi].first[k];
        groups[6 * gi + 2 * k + 1] = pl.groups[gi].count[k];
      }
  return LOPT_OK;
}

int lopt_shard_begin(lopt_handle h, const lopt_tensor* tensors, const int64_t* global_rows,
                     int n_tensors, int64_t t, float lr, double* x1, double* x2, void* stream_ptr) {
  if (!h || n_tensors < 1 || !tensors || !global_rows || !x1 || !x2 || t < 1) return LOPT_E_ARG;
  if (h->shard_phase != 0) return LOPT_E_ARG;
  if ((uintptr_t)x1 % 8 || (uintptr_t)x2 % 8) return LOPT_E_ALIGN;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  const bool same = h->last_path == h->path && (int)h->last_list.size() == n_tensors &&
                    (int)h->last_grows.size() == n_tensors &&
                    std::memcmp(h->last_list.data(), tensors, sizeof(lopt_tensor) * n_tensors) == 0 &&
                    std::memcmp(h->last_grows.data(), global_rows, sizeof(int64_t) * n_tensors) == 0;
  if (!same) {
    const int rc = validate(h, tensors, n_tensors, global_rows);
    if (rc != LOPT_OK) return rc;
  }
  PhaseScope sc;
  int rc = enter_phase(h, stream, sc);
  if (rc != LOPT_OK) return rc;
  const cudaError_t ew = wait_host_copies(h, stream);
  if (ew != cudaSuccess) return cuda_fail(ew);
  if (!same) {
    rc = build_schedule(h, tensors, n_tensors, stream, global_rows);
    if (rc != LOPT_OK) {
      h->last_list.clear();
      return rc;
    }
  }
  int64_t n1 = 0, n2 = 0;
  shard_counts(tensors, n_tensors, &n1, &n2);
  StepArgs& a = h->shard_args;
  std::memset(&a, 0, sizeof(a));
  a.desc = h->d_desc;
  a.hidden = h->hp;
  a.aux = h->d_aux;
  a.colpart = h->d_colpart;
  a.rowpart = h->d_rowpart;
  a.k1part = h->d_k1part;
  a.weights = h->d_weights;
  a.set_size = w_set_size(h->hp);
  a.w1fold = h->d_w1fold;
  a.w1fold_stride = h->w1fold_stride;
  a.path = h->path;
  a.tc_weights = h->d_tcw;
  a.t = (double)t;
  for (int k = 0; k < kTimeFeat; ++k) a.tau[k] = std::tanh((double)t / time_scale(k));
  a.lr = lr;
  a.wd = h->weight_decay;
  a.status = h->d_status;
  h->x1 = x1;
  h->x2 = x2;
  cudaError_t e = cudaMemsetAsync(x1, 0, sizeof(double) * n1, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(x2, 0, sizeof(double) * n2, stream);
  StepArgs k0 = a;
  k0.units = h->d_units[0];
  k0.n_units = h->n_units[0];
  k0.counters = h->d_counters;
  k0.xch1 = x1;
  if (e == cudaSuccess) e = launch_rowcol(k0, stream);
  h->shard_phase = 1;
  return leave_phase(h, stream, e);
}

int lopt_shard_middle(lopt_handle h, void* stream_ptr) {
  if (!h || h->shard_phase != 1) return LOPT_E_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  PhaseScope sc;
  const int rc = enter_phase(h, stream, sc);
  if (rc != LOPT_OK) return rc;
  StepArgs f = h->shard_args;
  f.xch1 = h->x1;
  cudaError_t e = launch_rowcol_finish(f, h->n_tensors, stream);
  StepArgs k1 = h->shard_args;
  k1.units = h->d_units[1];
  k1.n_units = h->n_units[1];
  k1.counters = h->d_counters + h->n_tensors;
  k1.xch2 = h->x2;
  if (e == cudaSuccess) e = launch_stats(k1, stream);
  h->shard_phase = 2;
  return leave_phase(h, stream, e);
}

int lopt_shard_end(lopt_handle h, void* stream_ptr) {
  if (!h || h->shard_phase != 2) return LOPT_E_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  PhaseScope sc;
  const int rc = enter_phase(h, stream, sc);
  if (rc != LOPT_OK) return rc;
  StepArgs f = h->shard_args;
  f.xch2 = h->x2;
  cudaError_t e = launch_stats_finish(f, h->n_tensors, stream);
  StepArgs k2 = h->shard_args;
  k2.units = h->d_units[2];
  k2.n_units = h->n_units[2];
  if (e == cudaSuccess) e = (h->path == LOPT_MLP_TC) ? launch_apply_tc(k2, stream) : launch_apply_fp32(k2, stream);
  h->shard_phase = 0;
  return leave_phase(h, stream, e);
}

int lopt_check(lopt_handle h) {
  if (!h) return LOPT_E_ARG;
  if (h->pipe) {
    if (h->pipe->any) {
      const cudaError_t e = cudaEventSynchronize(h->pipe->d2h_done);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    for (int q = 0; q < 2; ++q) {
      for (lopt_ctx* c : h->pipe->parts[q]) {
        const int rc = lopt_check(c);
        if (rc != LOPT_OK) return rc;
      }
    }
  }
  if (!h->has_done) return LOPT_OK;
  cudaError_t e = cudaEventSynchronize(h->done);
  if (e != cudaSuccess) return cuda_fail(e);
  if (!h->d_status) return LOPT_OK;
  int32_t st = 0;
  e = cudaMemcpy(&st, h->d_status, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (st != 0) {
    e = cudaMemset(h->d_status, 0, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(e);
    return LOPT_E_TIMEOUT;
  }
  return LOPT_OK;
}

int lopt_feature_stats(lopt_handle h, int index, double* out) {
  if (!h || !out || index < 0 || index >= h->n_tensors) return LOPT_E_ARG;
  if (h->has_done) {
    cudaError_t e = cudaEventSynchronize(h->done);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  const char* src = reinterpret_cast<const char*>(h->d_aux) + sizeof(TensorAux) * (size_t)index +
                    offsetof(TensorAux, S);
  cudaError_t e = cudaMemcpy(out, src, sizeof(double) * kStats, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? LOPT_OK : cuda_fail(e);
}

int lopt_set_kernel_timing(lopt_handle h, int enable) {
  if (!h) return LOPT_E_ARG;
  h->timing = enable != 0;
  return LOPT_OK;
}

int lopt_kernel_times(lopt_handle h, double* ms, int64_t* launches) {
  if (!h || !ms || !launches) return LOPT_E_ARG;
  for (int k = 0; k < 3; ++k) {
    ms[k] = 0.0;
    launches[k] = 0;
  }
  if (h->tev_used == 0) return LOPT_OK;
  cudaError_t e = cudaEventSynchronize(h->tev[h->tev_used - 1]);
  if (e != cudaSuccess) return cuda_fail(e);
  for (size_t s = 0; s + 4 <= h->tev_used; s += 4) {
    for (int k = 0; k < 3; ++k) {
      float x = 0.f;
      e = cudaEventElapsedTime(&x, h->tev[s + k], h->tev[s + k + 1]);
      if (e != cudaSuccess) return cuda_fail(e);
      ms[k] += x;
      launches[k] += 1;
    }
  }
  h->tev_used = 0;
  return LOPT_OK;
}

int lopt_destroy(lopt_handle h) {
  if (!h) return LOPT_E_ARG;
  if (h->has_done) cudaEventSynchronize(h->done);
  destroy_pipe(h->pipe);
  for (cudaEvent_t x : h->tev) cudaEventDestroy(x);
  if (h->d_ws) cudaFree(h->d_ws);
  if (!h->shared_weights && h->d_weights) cudaFree(h->d_weights);
  if (!h->shared_weights && h->d_tcw) cudaFree(h->d_tcw);
  if (h->done) cudaEventDestroy(h->done);
  delete h;
  return LOPT_OK;
}

}  // extern "C"

namespace {
void destroy_pipe(HostPipe* p) {
  if (!p) return;
  if (p->any) cudaEventSynchronize(p->d2h_done);
  for (int q = 0; q < 2; ++q) {
    for (lopt_ctx* c : p->parts[q]) lopt_destroy(c);
    if (p->stage[q]) cudaFree(p->stage[q]);
  }
  for (cudaEvent_t x : p->ev) cudaEventDestroy(x);
  if (p->d2h_done) cudaEventDestroy(p->d2h_done);
  if (p->h2d) cudaStreamDestroy(p->h2d);
  if (p->d2h) cudaStreamDestroy(p->d2h);
  delete p;
}
}  // namespace
