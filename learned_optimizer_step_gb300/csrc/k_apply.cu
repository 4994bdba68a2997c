// K2 (FP32 path): apply pass -- recompute the features, normalise, run the
// per-element MLP, apply the update and store the parameter and the
// accumulators.
//
// "PyLO: Towards Accessible Learned Optimizers in PyTorch", section
// "融合カーネル戦略", kernel 2: construct_features() + feature_normalization()
// + apply_lo(); features are recomputed in registers, the MLP is evaluated
// inline with activations in registers, and only the results are written.
// Differences from the page's design: the normalisation statistics and the
// time features are folded into the first layer's weights and bias once per
// tensor (by the statistics pass), and all layer weights sit in shared
// memory, read as warp-wide broadcasts, instead of per-thread __ldg loads.
#include "lopt_internal.cuh"

namespace lopt {
namespace {

constexpr int kT = kApplyThreads;

template <int H>
struct ApplySmem {
  float W1[kStats * H];   // folded: s_d * W1[d][h]
  float b1[H];            // folded: b1 + sum_s tau_s W1[28 + s]
  float W2[H * H];
  float b2[H];
  float W3[H * 2];
  float b3[2];
};

// One element per call; E elements are interleaved by the caller for ILP.
template <int H, int E>
__device__ __forceinline__ void mlp_update(const ApplySmem<H>& w, const float (&f)[E][kStats],
                                           float (&upd)[E]) {
  float h1[E][H];
#pragma unroll
  for (int e = 0; e < E; ++e)
#pragma unroll
    for (int h = 0; h < H; ++h) h1[e][h] = w.b1[h];
#pragma unroll
  for (int dd = 0; dd < kStats; ++dd) {
#pragma unroll
    for (int h = 0; h < H; ++h) {
      const float wv = w.W1[dd * H + h];
#pragma unroll
      for (int e = 0; e < E; ++e) h1[e][h] = fmaf(f[e][dd], wv, h1[e][h]);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e)
#pragma unroll
    for (int h = 0; h < H; ++h) h1[e][h] = fmaxf(h1[e][h], 0.f);

  float o0[E], o1[E];
#pragma unroll
  for (int e = 0; e < E; ++e) { o0[e] = w.b3[0]; o1[e] = w.b3[1]; }
#pragma unroll
  for (int h = 0; h < H; ++h) {
    float z[E];
#pragma unroll
    for (int e = 0; e < E; ++e) z[e] = w.b2[h];
#pragma unroll
    for (int a = 0; a < H; ++a) {
      const float wv = w.W2[a * H + h];
#pragma unroll
      for (int e = 0; e < E; ++e) z[e] = fmaf(h1[e][a], wv, z[e]);
    }
    const float w30 = w.W3[2 * h], w31 = w.W3[2 * h + 1];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float r = fmaxf(z[e], 0.f);
      o0[e] = fmaf(r, w30, o0[e]);
      o1[e] = fmaf(r, w31, o1[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) upd[e] = o0[e] * expf(o1[e] * kOutScale) * kOutScale;
}

template <int H>
__global__ void __launch_bounds__(kT) k_apply_fp32(StepArgs a) {
  constexpr int E = (H <= 32) ? 2 : 1;
  __shared__ ApplySmem<H> w;

  const Unit u = a.units[blockIdx.x];
  const TensorDesc d = a.desc[u.tensor];
  const int tid = threadIdx.x;

  {  // stage the weights of this tensor
    const float* f1 = a.w1fold + (int64_t)u.tensor * a.w1fold_stride;
    for (int x = tid; x < kStats * H; x += kT) w.W1[x] = f1[x];
    for (int x = tid; x < H; x += kT) w.b1[x] = f1[kStats * H + x];
    const float* W = a.weights + (int64_t)d.wset * a.set_size;
    for (int x = tid; x < H * H; x += kT) w.W2[x] = W[w_off_W2(H) + x];
    for (int x = tid; x < H; x += kT) w.b2[x] = W[w_off_b2(H) + x];
    for (int x = tid; x < 2 * H; x += kT) w.W3[x] = W[w_off_W3(H) + x];
    if (tid < 2) w.b3[tid] = W[w_off_b3(H) + tid];
  }
  float inv_rho[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) inv_rho[k] = a.aux[u.tensor].inv_rho[k];
  __syncthreads();

  const int64_t e0 = (int64_t)u.local * kApplyChunk;
  const int64_t e1 = min(d.N, e0 + (int64_t)kApplyChunk);
  const float lr = a.lr, wd = a.wd;

  for (int64_t base = e0 + (int64_t)tid * E; base < e1; base += (int64_t)kT * E) {
    float f[E][kStats];
    float m[E][3], v[E], p[E];
    bool ok[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int64_t x = base + e;
      ok[e] = x < e1;
      const int64_t xs = ok[e] ? x : base;   // keep loads in bounds
      const int64_t i = xs / d.C, j = xs - i * d.C;
      p[e] = d.p[xs];
      const float g = __ldg(d.g + xs);
#pragma unroll
      for (int k = 0; k < 3; ++k) m[e][k] = d.m[k][xs];
      v[e] = d.v[xs];
      const float c[3] = {__ldg(d.c[0] + j), __ldg(d.c[1] + j), __ldg(d.c[2] + j)};
      const RowTerms rt = row_terms(d, inv_rho, i);
      lopt_features(p[e], g, m[e], v[e], rt, c, f[e]);
    }
    float upd[E];
    mlp_update<H, E>(w, f, upd);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (!ok[e]) continue;
      const int64_t x = base + e;
      d.p[x] = p[e] - lr * (upd[e] + wd * p[e]);
#pragma unroll
      for (int k = 0; k < 3; ++k) d.m[k][x] = m[e][k];
      d.v[x] = v[e];
    }
  }
}

}  // namespace

cudaError_t launch_apply_fp32(const StepArgs& a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  switch (a.hidden) {
    case 4:  k_apply_fp32<4><<<a.n_units, kT, 0, s>>>(a); break;
    case 8:  k_apply_fp32<8><<<a.n_units, kT, 0, s>>>(a); break;
    case 16: k_apply_fp32<16><<<a.n_units, kT, 0, s>>>(a); break;
    case 32: k_apply_fp32<32><<<a.n_units, kT, 0, s>>>(a); break;
    case 64: k_apply_fp32<64><<<a.n_units, kT, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

bool apply_fp32_supported(int hidden) {
  return hidden == 4 || hidden == 8 || hidden == 16 || hidden == 32 || hidden == 64;
}

}  // namespace lopt
