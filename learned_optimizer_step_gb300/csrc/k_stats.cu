// K1: statistics pass -- per-feature sum of squares over each whole tensor,
// from the squares of the features built in registers.
//
// "PyLO: Towards Accessible Learned Optimizers in PyTorch", section
// "融合カーネル戦略", kernel 1: construct_features() fused with
// compute_squared_average(); features are computed on the fly and never
// stored, every thread keeps a d_feat-wide sum of squares, and only a few
// dozen scalars per tensor leave the kernel.  The page reduces warp ->
// block -> atomicAdd; here the last level is deterministic instead: every
// work unit writes its 28 block sums, and the last unit of a tensor (a
// per-tensor counter, no spin-waits) adds them in unit order in double.
//
// That last block also prepares the apply pass: it divides each row of W1 by
// the feature's RMS (the normalisation folded into the first layer) and adds
// the 11 time features, which are the same for every element, into the first
// bias:  x_hat . W1 = sum_d f_d * (s_d W1[d]) + sum_s tau_s W1[28 + s].
#include "lopt_internal.cuh"
#include "lopt.h"
#include "tc_layout.cuh"

namespace lopt {

// Iteration state for a thread walking a tensor in steps of `stride`
// elements, keeping (row, column) without a division per element.
struct RowColWalker {
  int64_t i, j, C, di, dj;
  __device__ RowColWalker(int64_t e, int64_t stride, int64_t C_) : C(C_) {
    i = e / C; j = e - i * C;
    di = stride / C; dj = stride - di * C;
  }
  __device__ void advance() {
    i += di; j += dj;
    if (j >= C) { j -= C; ++i; }
  }
};

namespace {

constexpr int kT = kStatsThreads;
constexpr int kWarps = kT / 32;
constexpr int kFinalGroups = kT / kStats;   // threads per feature in a tensor's final sum (9)

__device__ __forceinline__ void accumulate_element(const TensorDesc& d, const float inv_rho[3],
                                                   int64_t e, int64_t i, int64_t j,
                                                   float acc[kStats]) {
  const float m[3] = {__ldg(d.m[0] + e), __ldg(d.m[1] + e), __ldg(d.m[2] + e)};
  const float c[3] = {__ldg(d.c[0] + j), __ldg(d.c[1] + j), __ldg(d.c[2] + j)};
  const float r[3] = {__ldg(d.r[0] + i), __ldg(d.r[1] + i), __ldg(d.r[2] + i)};
  lopt_feature_squares(__ldg(d.p + e), __ldg(d.g + e), m, __ldg(d.v + e), r, c, inv_rho, acc);
}

// Normalisation and time features folded into the first layer of tensor T
// (run by a whole block): x_hat . W1 = sum_d f_d (s_d W1[d]) + sum_s tau_s W1[28 + s].
__device__ void fold_first_layer(const StepArgs& a, int T, const TensorDesc& d, const double* scale) {
  const int tid = threadIdx.x;
  const int H = a.hidden;
  const float* W = a.weights + (int64_t)d.wset * a.set_size;
  const float* W1 = W + w_off_W1(H);
  const float* b1 = W + w_off_b1(H);
  float* out = a.w1fold + (int64_t)T * a.w1fold_stride;
  if (a.path == LOPT_MLP_FP32) {
    // layout: W1'[28][H] then b1'[H]
    for (int x = tid; x < kStats * H; x += kT) {
      const int dd = x / H;
      out[x] = (float)(scale[dd] * (double)W1[x]);
    }
    for (int h = tid; h < H; h += kT) {
      double b = (double)b1[h];
      for (int s = 0; s < kTimeFeat; ++s) {
        b += a.tau[s] * (double)W1[(kStats + s) * H + h];
      }
      out[kStats * H + h] = (float)b;
    }
  } else {
    fold_w1_tc(H, W1, b1, a.tau, out);
  }
}

__global__ void __launch_bounds__(kT, 3) k_stats(StepArgs a) {   // 3 blocks per SM for loads in flight
  __shared__ float red[kWarps][kStats];
  __shared__ double fin[kFinalGroups][kStats];
  __shared__ double scale[kStats];
  __shared__ int is_last;

  const Unit u = a.units[blockIdx.x];
  const TensorDesc d = a.desc[u.tensor];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t e0 = (int64_t)u.local * kStatsChunk;
  const int64_t e1 = min(d.N, e0 + (int64_t)kStatsChunk);
  float inv_rho[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) inv_rho[k] = a.aux[u.tensor].inv_rho[k];

  float acc[kStats];
#pragma unroll
  for (int q = 0; q < kStats; ++q) acc[q] = 0.f;

  if (d.vec4 && (d.C % 4 == 0)) {
    // 128-bit path: four consecutive elements share one row.
    int64_t e = e0 + 4 * (int64_t)tid;
    if (e < e1) {
      RowColWalker w(e, 4 * (int64_t)kT, d.C);
      // the element arrays of the next step are loaded before this step's
      // arithmetic, so that a thread always has loads in flight (the last
      // step reloads its own elements)
      float4 p4 = __ldg(reinterpret_cast<const float4*>(d.p + e));
      float4 g4 = __ldg(reinterpret_cast<const float4*>(d.g + e));
      float4 a4 = __ldg(reinterpret_cast<const float4*>(d.m[0] + e));
      float4 b4 = __ldg(reinterpret_cast<const float4*>(d.m[1] + e));
      float4 c4 = __ldg(reinterpret_cast<const float4*>(d.m[2] + e));
      float4 v4 = __ldg(reinterpret_cast<const float4*>(d.v + e));
      for (; e < e1; e += 4 * (int64_t)kT, w.advance()) {
        const int64_t en = e + 4 * (int64_t)kT < e1 ? e + 4 * (int64_t)kT : e;
        const float4 np4 = __ldg(reinterpret_cast<const float4*>(d.p + en));
        const float4 ng4 = __ldg(reinterpret_cast<const float4*>(d.g + en));
        const float4 na4 = __ldg(reinterpret_cast<const float4*>(d.m[0] + en));
        const float4 nb4 = __ldg(reinterpret_cast<const float4*>(d.m[1] + en));
        const float4 nc4 = __ldg(reinterpret_cast<const float4*>(d.m[2] + en));
        const float4 nv4 = __ldg(reinterpret_cast<const float4*>(d.v + en));
        const float4 k0 = __ldg(reinterpret_cast<const float4*>(d.c[0] + w.j));
        const float4 k1 = __ldg(reinterpret_cast<const float4*>(d.c[1] + w.j));
        const float4 k2 = __ldg(reinterpret_cast<const float4*>(d.c[2] + w.j));
        const float r[3] = {__ldg(d.r[0] + w.i), __ldg(d.r[1] + w.i), __ldg(d.r[2] + w.i)};
        const float pp[4] = {p4.x, p4.y, p4.z, p4.w}, gg[4] = {g4.x, g4.y, g4.z, g4.w};
        const float m0[4] = {a4.x, a4.y, a4.z, a4.w}, m1[4] = {b4.x, b4.y, b4.z, b4.w};
        const float m2[4] = {c4.x, c4.y, c4.z, c4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w};
        const float c0[4] = {k0.x, k0.y, k0.z, k0.w}, c1[4] = {k1.x, k1.y, k1.z, k1.w};
        const float c2[4] = {k2.x, k2.y, k2.z, k2.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float m[3] = {m0[q], m1[q], m2[q]};
          const float c[3] = {c0[q], c1[q], c2[q]};
          lopt_feature_squares(pp[q], gg[q], m, vv[q], r, c, inv_rho, acc);
        }
        p4 = np4; g4 = ng4; a4 = na4; b4 = nb4; c4 = nc4; v4 = nv4;
      }
    }
  } else {
    int64_t e = e0 + tid;
    if (e < e1) {
      RowColWalker w(e, (int64_t)kT, d.C);
      for (; e < e1; e += kT, w.advance()) accumulate_element(d, inv_rho, e, w.i, w.j, acc);
    }
  }

  // warp -> block (fixed order), one partial per work unit
#pragma unroll
  for (int q = 0; q < kStats; ++q) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[q] = fadd(acc[q], __shfl_xor_sync(0xffffffffu, acc[q], off));
  }
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < kStats; ++q) red[warp][q] = acc[q];
  }
  __syncthreads();
  if (tid < kStats) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s = fadd(s, red[w][tid]);
    a.k1part[(int64_t)d.k1_part_off + (int64_t)u.local * kStats + tid] = s;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(a.counters + u.tensor, 1);
    is_last = (prev == d.k1_units - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // ---- finalize this tensor: S_d in double, in a fixed order -------------
  // kFinalGroups threads per feature each add, in increasing order, the
  // partials of the units x = g mod kFinalGroups; then their sums are added
  // in g order.  (One thread per feature adding thousands of partials in
  // turn was the tail of the launch for the largest tensors.)
  if (tid < kFinalGroups * kStats) {
    const int f = tid % kStats, g = tid / kStats;
    const float* part = a.k1part + d.k1_part_off;
    double s = 0.0;
    for (int x = g; x < d.k1_units; x += kFinalGroups) s += (double)__ldcg(part + (int64_t)x * kStats + f);
    fin[g][f] = s;
  }
  __syncthreads();
  if (tid < kStats) {
    double s = 0.0;
#pragma unroll
    for (int g = 0; g < kFinalGroups; ++g) s += fin[g][tid];
    if (a.xch2) {   // row-sharded: this rank's sums go out for the exchange
      a.xch2[(int64_t)u.tensor * kStats + tid] = s;
    } else {
      a.aux[u.tensor].S[tid] = s;
      scale[tid] = 1.0 / sqrt(s / (double)d.N + 1e-30);
      a.aux[u.tensor].scale[tid] = (float)scale[tid];
    }
  }
  if (tid == 0) a.counters[u.tensor] = 0;
  if (a.xch2) return;
  __syncthreads();
  fold_first_layer(a, u.tensor, d, scale);
}

// Row-sharded steps: S_d of every tensor from the sums of all ranks (xch2,
// already added up) over the tensor's global element count, then the fold.
__global__ void __launch_bounds__(kT) k_stats_finish(StepArgs a) {
  __shared__ double scale[kStats];
  const int T = blockIdx.x, tid = threadIdx.x;
  const TensorDesc d = a.desc[T];
  if (tid < kStats) {
    const double s = a.xch2[(int64_t)T * kStats + tid];
    a.aux[T].S[tid] = s;
    scale[tid] = 1.0 / sqrt(s / ((double)d.Rg * (double)d.C) + 1e-30);
    a.aux[T].scale[tid] = (float)scale[tid];
  }
  __syncthreads();
  fold_first_layer(a, T, d, scale);
}

}  // namespace

cudaError_t launch_stats(const StepArgs& a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  k_stats<<<a.n_units, kT, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_stats_finish(const StepArgs& a, int n_tensors, cudaStream_t s) {
  if (n_tensors == 0) return cudaSuccess;
  k_stats_finish<<<n_tensors, kT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lopt
