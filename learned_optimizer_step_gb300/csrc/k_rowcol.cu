// K0: factored (Adafactor) second moment of every tensor in one launch.
//
// For a tensor viewed as [R x C]:
//   G_i = mean_j g_ij^2,  H_j = mean_i g_ij^2,
//   r_k <- b_k r_k + (1 - b_k) G,   c_k <- b_k c_k + (1 - b_k) H,
//   rho_k = mean_i r_k[i]             (k = 0, 1, 2; b = 0.1, 0.5, 0.9)
// These feed the factored-RMS features of "PyLO: Towards Accessible Learned
// Optimizers in PyTorch" (the Adafactor-style accumulators kept per
// parameter by the optimiser module, section "PyLO のライブラリ設計").  The
// column means need the whole tensor, so they are reduced here, before the
// statistics pass reads them.
//
// Work unit = a strip of consecutive rows.  A block reads its strip once
// (coalesced, 128-bit when the tensor allows), finishes the row means of its
// rows, and writes per-strip column partial sums.  The last strip block of a
// tensor (a per-tensor counter; no spin-waits) sums the column partials and
// row partials in a fixed order, so results do not depend on block timing.
#include "lopt_internal.cuh"

namespace lopt {
namespace {

constexpr int kT = kRowColThreads;
constexpr int kWarps = kT / 32;
constexpr int kRowBatch = 8;         // rows reduced together

template <int W>   // W = 4: float4 columns, W = 1: scalar columns
__device__ void strip_pass(const TensorDesc& d, int64_t r0, int nrows, float* colpart_strip,
                           float* rowacc, float (*wsum)[kWarps][kRowBatch]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t C = d.C;
  for (int i = tid; i < nrows; i += kT) rowacc[i] = 0.f;
  __syncthreads();
  int buf = 0;
  for (int64_t c0 = 0; c0 < C; c0 += (int64_t)kT * W) {
    const int64_t j = c0 + (int64_t)tid * W;
    const bool active = j < C;
    float col[W];
#pragma unroll
    for (int q = 0; q < W; ++q) col[q] = 0.f;
    for (int rb = 0; rb < nrows; rb += kRowBatch) {
      float part[kRowBatch];
#pragma unroll
      for (int q = 0; q < kRowBatch; ++q) {
        part[q] = 0.f;
        const int row = rb + q;
        if (active && row < nrows) {
          const float* src = d.g + (r0 + row) * C + j;
          if constexpr (W == 4) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(src));
            const float s0 = fmul(x.x, x.x), s1 = fmul(x.y, x.y);
            const float s2 = fmul(x.z, x.z), s3 = fmul(x.w, x.w);
            col[0] = fadd(col[0], s0);
            col[1] = fadd(col[1], s1);
            col[2] = fadd(col[2], s2);
            col[3] = fadd(col[3], s3);
            part[q] = fadd(fadd(s0, s1), fadd(s2, s3));
          } else {
            const float x = __ldg(src);
            const float s0 = fmul(x, x);
            col[0] = fadd(col[0], s0);
            part[q] = s0;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kRowBatch; ++q) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          part[q] = fadd(part[q], __shfl_xor_sync(0xffffffffu, part[q], off));
      }
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < kRowBatch; ++q) wsum[buf][warp][q] = part[q];
      }
      __syncthreads();
      if (tid < kRowBatch && rb + tid < nrows) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s = fadd(s, wsum[buf][w][tid]);
        rowacc[rb + tid] = fadd(rowacc[rb + tid], s);
      }
      buf ^= 1;   // the next batch writes the other buffer; one barrier per batch
    }
    if (active) {
#pragma unroll
      for (int q = 0; q < W; ++q) colpart_strip[j + q] = col[q];
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kT) k_rowcol(StepArgs a) {
  __shared__ float rowacc[kMaxStripRows];
  __shared__ float wsum[2][kWarps][kRowBatch];
  __shared__ double red[kWarps][3];
  __shared__ int is_last;

  const Unit u = a.units[blockIdx.x];
  const TensorDesc d = a.desc[u.tensor];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r0 = (int64_t)u.local * d.strip_rows;
  const int nrows = (int)min((int64_t)d.strip_rows, d.R - r0);
  float* colpart_strip = a.colpart + d.colpart_off + (int64_t)u.local * d.C;

  if (d.vec4 && (d.C % 4 == 0))
    strip_pass<4>(d, r0, nrows, colpart_strip, rowacc, wsum);
  else
    strip_pass<1>(d, r0, nrows, colpart_strip, rowacc, wsum);

  // Row means -> row accumulators; partial sums of the new r_k for rho_k.
  double acc[3] = {0.0, 0.0, 0.0};
  for (int i = tid; i < nrows; i += kT) {
    const float G = __fdiv_rn(rowacc[i], (float)d.C);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      float* rp = d.r[k] + r0 + i;
      const float rn = ffma(beta(k), *rp, fmul(one_minus_beta(k), G));
      *rp = rn;
      acc[k] += (double)rn;
    }
  }
#pragma unroll
  for (int k = 0; k < 3; ++k) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
  }
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) red[warp][k] = acc[k];
  }
  __syncthreads();
  if (tid < 3) {
    double s = 0.0;
    for (int w = 0; w < kWarps; ++w) s += red[w][tid];
    a.rowpart[d.rowpart_off + 3 * u.local + tid] = s;
  }

  // Last strip of this tensor finishes the column means and rho.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(a.counters + u.tensor, 1);
    is_last = (prev == d.n_strips - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Column means: every thread owns whole columns and sums their strip
  // partials in strip order (four independent columns per thread when the
  // tensor allows 128-bit access, to keep many loads in flight).
  const float* cp = a.colpart + d.colpart_off;
  const double invR = 1.0 / (double)d.R;
  const int S = d.n_strips;
  if (d.vec4 && (d.C % 4 == 0)) {
    for (int64_t j = 4 * (int64_t)tid; j < d.C; j += 4 * (int64_t)kT) {
      double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
#pragma unroll 8
      for (int st = 0; st < S; ++st) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(cp + (int64_t)st * d.C + j));
        s0 += (double)x.x; s1 += (double)x.y; s2 += (double)x.z; s3 += (double)x.w;
      }
      const float H[4] = {(float)(s0 * invR), (float)(s1 * invR), (float)(s2 * invR), (float)(s3 * invR)};
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        float4* c4 = reinterpret_cast<float4*>(d.c[k] + j);
        float4 c = *c4;
        c.x = ffma(beta(k), c.x, fmul(one_minus_beta(k), H[0]));
        c.y = ffma(beta(k), c.y, fmul(one_minus_beta(k), H[1]));
        c.z = ffma(beta(k), c.z, fmul(one_minus_beta(k), H[2]));
        c.w = ffma(beta(k), c.w, fmul(one_minus_beta(k), H[3]));
        *c4 = c;
      }
    }
  } else {
    for (int64_t j = tid; j < d.C; j += kT) {
      double s = 0.0;
#pragma unroll 8
      for (int st = 0; st < S; ++st) s += (double)__ldcg(cp + (int64_t)st * d.C + j);
      const float H = (float)(s * invR);
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        float* c = d.c[k] + j;
        *c = ffma(beta(k), *c, fmul(one_minus_beta(k), H));
      }
    }
  }
  if (tid < 3) {
    double s = 0.0;
    const double* rp = a.rowpart + d.rowpart_off;
    for (int st = 0; st < d.n_strips; ++st) s += __ldcg(rp + 3 * st + tid);
    const double rho = s * invR;
    a.aux[u.tensor].inv_rho[tid] = rho > 0.0 ? (float)(1.0 / rho) : 0.f;
  }
  if (tid == 0) a.counters[u.tensor] = 0;
}

}  // namespace

cudaError_t launch_rowcol(const StepArgs& a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  k_rowcol<<<a.n_units, kT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lopt
