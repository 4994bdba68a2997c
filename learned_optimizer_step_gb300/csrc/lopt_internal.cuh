// Internal definitions shared by the kernels and the host code of liblopt.
//
// Method: "PyLO: Towards Accessible Learned Optimizers in PyTorch" (MLSys 2026
// talk notes), sections "融合カーネル戦略" and "メモリ階層の活用".  The
// feature list, decays and epsilon are this library's small_fc_lopt
// defaults (see the comment on lopt_features below).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace lopt {

// ---- method constants (fp32 on the device) --------------------------------
constexpr int   kStats     = 28;     // per-element (normalised) features
constexpr int   kTimeFeat  = 11;     // tanh(t / x_s)
constexpr int   kDFeat     = kStats + kTimeFeat;   // 39
constexpr float kEps       = 1e-30f; // inside every rsqrt and the normalisation
constexpr float kOutScale  = 1e-3f;  // update = o0 * exp(o1 * 1e-3) * 1e-3

// Momentum / factored decays b (0.1, 0.5, 0.9) and their complements
// (1 - b), as fp32; k is a compile-time index after unrolling.
__host__ __device__ constexpr float beta(int k) { return k == 0 ? 0.1f : (k == 1 ? 0.5f : 0.9f); }
__host__ __device__ constexpr float one_minus_beta(int k) { return k == 0 ? 0.9f : (k == 1 ? 0.5f : 0.1f); }
constexpr float kBeta2 = 0.999f, kOneMinusBeta2 = 0.001f;

// Time-feature scales x_s of tau_s = tanh(t / x_s), s = 0..10.
__host__ __device__ constexpr double time_scale(int s) {
  return s == 0 ? 1.0 : s == 1 ? 3.0 : s == 2 ? 10.0 : s == 3 ? 30.0 : s == 4 ? 100.0
       : s == 5 ? 300.0 : s == 6 ? 1e3 : s == 7 ? 3e3 : s == 8 ? 1e4 : s == 9 ? 3e4 : 1e5;
}

// ---- work decomposition -----------------------------------------------------
constexpr int kRowColThreads = 256;   // K0 block
constexpr int kStatsThreads  = 256;   // K1 block
constexpr int kStatsChunk    = 16384; // elements per K1 work unit
constexpr int kApplyThreads  = 128;   // K2 (FP32 MLP) block
constexpr int kApplyChunk    = 4096;  // elements per K2 work unit
constexpr int kStripTarget   = 32768; // elements per K0 strip, when possible
constexpr int kFinalizeCap   = 65536; // K0: strips * cols bound (column partials one block sums)
constexpr int kMaxStripRows  = 2048;  // K0: rows of one strip (shared row buffer)

// One tensor of a step, as the kernels see it.
struct TensorDesc {
  float*       p;
  const float* g;
  float*       m[3];
  float*       v;
  float*       r[3];
  float*       c[3];
  int64_t      R, C, N;
  int32_t      wset;
  int32_t      vec4;          // all element arrays 16-byte aligned
  int32_t      strip_rows;    // K0: rows per strip
  int32_t      n_strips;      // K0: strips of this tensor
  int32_t      k1_units;      // K1 chunks of this tensor
  int32_t      k2_units;      // K2 chunks of this tensor
  int64_t      colpart_off;   // K0 column partials: n_strips * C floats
  int32_t      rowpart_off;   // K0 row partials: n_strips * 3 doubles
  int32_t      k1_part_off;   // K1 partials: k1_units * kStats floats
  int64_t      Rg;            // row-sharded steps: rows of the whole tensor over all ranks
  int64_t      x1_off;        // row-sharded steps: offset of this tensor in exchange buffer 1
};

// A work unit: tensor index and the unit's index inside the tensor.
struct Unit {
  int32_t tensor;
  int32_t local;
};

// Per-tensor results of the reductions of one step.
struct TensorAux {
  float  inv_rho[3];     // 1 / mean_i r_k[i], or 0 when that mean is 0
  float  pad0;
  double S[kStats];      // sum over elements of feature^2
  float  scale[kStats];  // 1 / sqrt(S / N + eps): the normalisation factors
};

// Everything a launch needs, passed by value.
struct StepArgs {
  const TensorDesc* desc;
  const Unit*       units;       // K0, K1 or K2 unit table
  int32_t           n_units;
  int32_t           hidden;
  TensorAux*        aux;         // [T]
  int32_t*          counters;    // [T] last-block counters (self-resetting)
  float*            colpart;     // K0 column partials
  double*           rowpart;     // K0 row partials
  float*            k1part;      // K1 partials
  const float*      weights;     // [n_sets][set_size], the caller's layout
  int32_t           set_size;
  float*            w1fold;      // [T][w1fold_stride] per-tensor folded W1, b1
  int32_t           w1fold_stride;
  int32_t           path;        // LOPT_MLP_*
  const void*       tc_weights;  // per-set packed FP16 B operands (tensor-core path)
  double            t;           // step count
  double            tau[kTimeFeat];   // tanh(t / x_s), computed once on the host
  float             lr;
  float             wd;          // decoupled weight decay: p -= lr * (update + wd * p)
  // Row-sharded steps only (null otherwise): this rank's sums that the ranks
  // add up between the kernels.  xch1: per tensor, the C column sums of g^2
  // then the 3 sums of the new row accumulators; xch2: per tensor, the 28
  // feature square sums.
  double*           xch1;
  double*           xch2;
  int32_t*          status;      // device-side error flags
};

// ---- exact, contraction-free fp32 helpers ----------------------------------
// Every operation is spelled out with a rounding intrinsic, so that the
// compiler contracts nothing and results do not depend on its choices.
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float ffma(float a, float b, float c) { return __fmaf_rn(a, b, c); }
// Reciprocal square root: the PTX rsqrt.approx instruction (relative error
// below 2^-22.9).  Every argument here is at least kEps = 1e-30, a normal
// number, so flushing subnormals never applies.
__device__ __forceinline__ float frsqrt(float a) {
  float r;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

// Per-row quantities of the factored second moment for one element.
struct RowTerms {
  float rr[3];   // r_k[i] / rho_k
  float sr[3];   // sqrt(r_k[i])
};

// From the three row accumulators r_k[i] of an element's row.
__device__ __forceinline__ RowTerms row_terms_of(const float r[3], const float inv_rho[3]) {
  RowTerms t;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    t.rr[k] = fmul(r[k], inv_rho[k]);
    t.sr[k] = fmul(r[k], frsqrt(fadd(r[k], kEps)));
  }
  return t;
}

__device__ __forceinline__ RowTerms row_terms(const TensorDesc& d, const float inv_rho[3],
                                              int64_t i) {
  const float r[3] = {__ldg(d.r[0] + i), __ldg(d.r[1] + i), __ldg(d.r[2] + i)};
  return row_terms_of(r, inv_rho);
}

// Element-wise accumulator update (EMA of g and g^2), then the 28
// per-element features.  Order of the features:
//   0 p | 1 g | 2-4 m_k | 5 sqrt(v) | 6-8 m_k*rsqrt(v) | 9 g*rsqrt(v)
//   10-12 g*rsqrt(vhat_k) | 13-15 sqrt(r_k[i]) | 16-18 sqrt(c_k[j])
//   19+3a+b m_a*rsqrt(vhat_b),   vhat_k = r_k[i] * c_k[j] / rho_k.
// m and v are updated in place (the apply kernel stores them).
__device__ __forceinline__ void lopt_features(float p, float g, float m[3], float& v,
                                              const RowTerms& rt, const float c[3],
                                              float f[kStats]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) m[k] = ffma(beta(k), m[k], fmul(one_minus_beta(k), g));
  v = ffma(kBeta2, v, fmul(kOneMinusBeta2, fmul(g, g)));
  const float rsv = frsqrt(fadd(v, kEps));
  float rvh[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) rvh[k] = frsqrt(fadd(fmul(rt.rr[k], c[k]), kEps));
  f[0] = p;
  f[1] = g;
#pragma unroll
  for (int k = 0; k < 3; ++k) f[2 + k] = m[k];
  f[5] = fmul(v, rsv);
#pragma unroll
  for (int k = 0; k < 3; ++k) f[6 + k] = fmul(m[k], rsv);
  f[9] = fmul(g, rsv);
#pragma unroll
  for (int k = 0; k < 3; ++k) f[10 + k] = fmul(g, rvh[k]);
#pragma unroll
  for (int k = 0; k < 3; ++k) f[13 + k] = rt.sr[k];
#pragma unroll
  for (int k = 0; k < 3; ++k) f[16 + k] = fmul(c[k], frsqrt(fadd(c[k], kEps)));
#pragma unroll
  for (int a = 0; a < 3; ++a)
#pragma unroll
    for (int b = 0; b < 3; ++b) f[19 + 3 * a + b] = fmul(m[a], rvh[b]);
}

// 1 / a: the PTX rcp.approx instruction (about 1 ulp).  Arguments here are
// at least kEps = 1e-30, a normal number, so flushing never applies.
__device__ __forceinline__ float frcp(float a) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

// The statistics pass needs only the squares of the 28 features, and most of
// them have a cheaper closed form than squaring the feature:
//   (m rsqrt(v+eps))^2 = m^2 / (v+eps),   sqrt(v)^2 ~ v^2 / (v+eps),
//   sqrt(r)^2 = r,   sqrt(c)^2 = c,   (m_a rsqrt(vhat_b+eps))^2 = m_a^2 / (vhat_b+eps).
// This adds, for one element, the squares of its features (order as in
// lopt_features) to acc, after the same accumulator update.
__device__ __forceinline__ void lopt_feature_squares(float p, float g, const float m_old[3], float v_old,
                                                     const float r[3], const float c[3],
                                                     const float inv_rho[3], float acc[kStats]) {
  float m[3], m2[3], ivh[3];
  const float g2 = fmul(g, g);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    m[k] = ffma(beta(k), m_old[k], fmul(one_minus_beta(k), g));
    m2[k] = fmul(m[k], m[k]);
    ivh[k] = frcp(fadd(fmul(fmul(r[k], inv_rho[k]), c[k]), kEps));
  }
  const float v = ffma(kBeta2, v_old, fmul(kOneMinusBeta2, g2));
  const float iv = frcp(fadd(v, kEps));
  acc[0] = ffma(p, p, acc[0]);
  acc[1] = fadd(acc[1], g2);
#pragma unroll
  for (int k = 0; k < 3; ++k) acc[2 + k] = fadd(acc[2 + k], m2[k]);
  acc[5] = ffma(fmul(v, v), iv, acc[5]);
#pragma unroll
  for (int k = 0; k < 3; ++k) acc[6 + k] = ffma(m2[k], iv, acc[6 + k]);
  acc[9] = ffma(g2, iv, acc[9]);
#pragma unroll
  for (int k = 0; k < 3; ++k) acc[10 + k] = ffma(g2, ivh[k], acc[10 + k]);
#pragma unroll
  for (int k = 0; k < 3; ++k) acc[13 + k] = fadd(acc[13 + k], r[k]);
#pragma unroll
  for (int k = 0; k < 3; ++k) acc[16 + k] = fadd(acc[16 + k], c[k]);
#pragma unroll
  for (int a = 0; a < 3; ++a)
#pragma unroll
    for (int b = 0; b < 3; ++b) acc[19 + 3 * a + b] = ffma(m2[a], ivh[b], acc[19 + 3 * a + b]);
}

// Offsets inside one weight set (caller layout).
__host__ __device__ inline int w_off_W1(int) { return 0; }
__host__ __device__ inline int w_off_b1(int H) { return kDFeat * H; }
__host__ __device__ inline int w_off_W2(int H) { return kDFeat * H + H; }
__host__ __device__ inline int w_off_b2(int H) { return kDFeat * H + H + H * H; }
__host__ __device__ inline int w_off_W3(int H) { return kDFeat * H + 2 * H + H * H; }
__host__ __device__ inline int w_off_b3(int H) { return kDFeat * H + 4 * H + H * H; }
__host__ __device__ inline int w_set_size(int H) { return kDFeat * H + 4 * H + H * H + 2; }

// Status flags written by kernels.
enum : int32_t { kStatusTimeout = 1 };

// Records a CUDA error for lopt_last_cuda_error() (this host thread) and
// returns the matching library code (LOPT_E_OOM or LOPT_E_CUDA).
int record_cuda_error(cudaError_t e);

// ---- launchers (one per kernel file) ---------------------------------------
cudaError_t launch_rowcol(const StepArgs& a, cudaStream_t s);
int  strip_rows_for(int64_t R, int64_t C);   // K0 rows per strip of an [R x C] tensor
cudaError_t launch_stats(const StepArgs& a, cudaStream_t s);
// Row-sharded steps: finish every tensor from the exchanged sums.
cudaError_t launch_rowcol_finish(const StepArgs& a, int n_tensors, cudaStream_t s);
cudaError_t launch_stats_finish(const StepArgs& a, int n_tensors, cudaStream_t s);
cudaError_t launch_apply_fp32(const StepArgs& a, cudaStream_t s);
cudaError_t launch_apply_tc(const StepArgs& a, cudaStream_t s);
bool apply_tc_supported(int hidden);
int  w1fold_floats(int hidden, int path);
size_t tc_weights_bytes(int hidden, int n_sets);
cudaError_t pack_tc_weights(const float* weights, int hidden, int n_sets, void* out, cudaStream_t s);

}  // namespace lopt
