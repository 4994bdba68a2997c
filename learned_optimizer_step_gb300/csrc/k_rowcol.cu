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
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "lopt.h"
#include "lopt_internal.cuh"

namespace lopt {
namespace {

constexpr int kT = kRowColThreads;

// Compensated (Kahan) fp32 summation: the rounding error of each addition is
// carried into the next one.
struct KahanSum {
  float sum = 0.f, comp = 0.f;
  __device__ void add(float x) {
    const float y = fadd(x, -comp);
    const float t = fadd(sum, y);
    comp = fadd(fadd(t, -sum), -y);
    sum = t;
  }
  __device__ float value() const { return sum; }
};
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

// Row-parallel pass for strips with at least one row per warp: warp w
// reads rows w, w + 8, ... of the strip, one coalesced row segment of up to
// 32 * 4 * kColVec columns at a time; a row's sum is one warp reduction
// added to rowacc by that warp alone, and each lane keeps the column sums
// of its columns in registers until the warps' column sums are combined in
// warp order.  Same results in every run: every sum has a fixed order.
constexpr int kColVec = 4;                 // vectors of W columns per lane and segment
constexpr int kRowUnroll = 2;              // rows whose loads a warp has in flight together

template <int W>
__device__ void strip_rows_pass(const TensorDesc& d, int64_t r0, int nrows, float* colpart_strip,
                                float* rowacc, float* colsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t C = d.C;
  constexpr int kSeg = 32 * W * kColVec;   // columns per segment
  for (int i = tid; i < nrows; i += kT) rowacc[i] = 0.f;
  __syncthreads();
  for (int64_t c0 = 0; c0 < C; c0 += kSeg) {
    float col[kColVec][W];
#pragma unroll
    for (int v = 0; v < kColVec; ++v)
#pragma unroll
      for (int q = 0; q < W; ++q) col[v][q] = 0.f;
    for (int row0 = warp; row0 < nrows; row0 += kRowUnroll * kWarps) {
      // all loads of kRowUnroll row segments first, so that they are in
      // flight together: a row past the strip reads row0 again and a column
      // past the end the segment's first column (both in bounds); neither
      // is counted
      float x[kRowUnroll][kColVec][W];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int row = row0 + u * kWarps < nrows ? row0 + u * kWarps : row0;
        const float* src = d.g + (r0 + row) * C + c0;
#pragma unroll
        for (int v = 0; v < kColVec; ++v) {
          const int64_t j = (int64_t)(v * 32 + lane) * W;   // column offset in the segment
          const int64_t js = c0 + j < C ? j : 0;
          if constexpr (W == 4) {
            const float4 y = __ldg(reinterpret_cast<const float4*>(src + js));
            x[u][v][0] = y.x; x[u][v][1] = y.y; x[u][v][2] = y.z; x[u][v][3] = y.w;
          } else {
            x[u][v][0] = __ldg(src + js);
          }
        }
      }
      // rows in increasing order, as one row at a time would add them
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int row = row0 + u * kWarps;
        if (row >= nrows) break;
        float rs = 0.f;
#pragma unroll
        for (int v = 0; v < kColVec; ++v) {
          const int64_t j = (int64_t)(v * 32 + lane) * W;
          if (c0 + j < C) {
            if constexpr (W == 4) {
              const float s0 = fmul(x[u][v][0], x[u][v][0]), s1 = fmul(x[u][v][1], x[u][v][1]);
              const float s2 = fmul(x[u][v][2], x[u][v][2]), s3 = fmul(x[u][v][3], x[u][v][3]);
              col[v][0] = fadd(col[v][0], s0);
              col[v][1] = fadd(col[v][1], s1);
              col[v][2] = fadd(col[v][2], s2);
              col[v][3] = fadd(col[v][3], s3);
              rs = fadd(rs, fadd(fadd(s0, s1), fadd(s2, s3)));
            } else {
              const float s0 = fmul(x[u][v][0], x[u][v][0]);
              col[v][0] = fadd(col[v][0], s0);
              rs = fadd(rs, s0);
            }
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) rs = fadd(rs, __shfl_xor_sync(0xffffffffu, rs, off));
        if (lane == 0) rowacc[row] = fadd(rowacc[row], rs);
      }
    }
    // this warp's column sums, then the warps' sums in warp order
#pragma unroll
    for (int v = 0; v < kColVec; ++v)
#pragma unroll
      for (int q = 0; q < W; ++q) colsum[warp * kSeg + (v * 32 + lane) * W + q] = col[v][q];
    __syncthreads();
    for (int jj = tid; jj < kSeg && c0 + jj < C; jj += kT) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s = fadd(s, colsum[w * kSeg + jj]);
      colpart_strip[c0 + jj] = s;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kT, 4) k_rowcol(StepArgs a) {   // 4 blocks per SM
  __shared__ float rowacc[kMaxStripRows];
  __shared__ float wsum[2][kWarps][kRowBatch];
  __shared__ __align__(16) float colsum[kWarps * 32 * 4 * kColVec];   // 16 KB
  __shared__ double red[kWarps][3];
  __shared__ int is_last;

  const Unit u = a.units[blockIdx.x];
  const TensorDesc d = a.desc[u.tensor];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r0 = (int64_t)u.local * d.strip_rows;
  const int nrows = (int)min((int64_t)d.strip_rows, d.R - r0);
  float* colpart_strip = a.colpart + d.colpart_off + (int64_t)u.local * d.C;

  const bool v4 = d.vec4 && (d.C % 4 == 0);
  if (nrows >= kWarps) {   // a row or more per warp
    if (v4) strip_rows_pass<4>(d, r0, nrows, colpart_strip, rowacc, colsum);
    else    strip_rows_pass<1>(d, r0, nrows, colpart_strip, rowacc, colsum);
  } else {                 // few long rows: all threads across the columns
    if (v4) strip_pass<4>(d, r0, nrows, colpart_strip, rowacc, wsum);
    else    strip_pass<1>(d, r0, nrows, colpart_strip, rowacc, wsum);
  }

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
  double* const xout = a.xch1 ? a.xch1 + d.x1_off : nullptr;   // row-sharded: sums go out
  if (xout) {
    for (int64_t j = tid; j < d.C; j += kT) {
      double s = 0.0;
#pragma unroll 8
      for (int st = 0; st < S; ++st) s += (double)__ldcg(cp + (int64_t)st * d.C + j);
      xout[j] = s;
    }
    if (tid < 3) {
      double s = 0.0;
      const double* rp = a.rowpart + d.rowpart_off;
      for (int st = 0; st < d.n_strips; ++st) s += __ldcg(rp + 3 * st + tid);
      xout[d.C + tid] = s;
    }
  } else if (d.vec4 && (d.C % 4 == 0)) {
    // compensated fp32 sums (FP64 is slow on this part; the error stays a
    // few ulp whatever the number of strips)
    const float invRf = (float)invR;
    for (int64_t j = 4 * (int64_t)tid; j < d.C; j += 4 * (int64_t)kT) {
      KahanSum s0, s1, s2, s3;
#pragma unroll 8
      for (int st = 0; st < S; ++st) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(cp + (int64_t)st * d.C + j));
        s0.add(x.x); s1.add(x.y); s2.add(x.z); s3.add(x.w);
      }
      const float H[4] = {fmul(s0.value(), invRf), fmul(s1.value(), invRf), fmul(s2.value(), invRf),
                          fmul(s3.value(), invRf)};
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
    const float invRf = (float)invR;
    for (int64_t j = tid; j < d.C; j += kT) {
      KahanSum s;
#pragma unroll 8
      for (int st = 0; st < S; ++st) s.add(__ldcg(cp + (int64_t)st * d.C + j));
      const float H = fmul(s.value(), invRf);
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        float* c = d.c[k] + j;
        *c = ffma(beta(k), *c, fmul(one_minus_beta(k), H));
      }
    }
  }
  if (!xout && tid < 3) {
    double s = 0.0;
    const double* rp = a.rowpart + d.rowpart_off;
    for (int st = 0; st < d.n_strips; ++st) s += __ldcg(rp + 3 * st + tid);
    const double rho = s * invR;
    a.aux[u.tensor].inv_rho[tid] = rho > 0.0 ? (float)(1.0 / rho) : 0.f;
  }
  if (tid == 0) a.counters[u.tensor] = 0;
}

// Row-sharded steps: the column means and rho of every tensor from the sums
// of all ranks (xch1, already added up), with the tensor's global row count.
__global__ void __launch_bounds__(kT) k_rowcol_finish(StepArgs a) {
  const TensorDesc d = a.desc[blockIdx.x];
  const double* x = a.xch1 + d.x1_off;
  const double invR = 1.0 / (double)d.Rg;
  for (int64_t j = threadIdx.x; j < d.C; j += kT) {
    const float H = (float)(x[j] * invR);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      float* c = d.c[k] + j;
      *c = ffma(beta(k), *c, fmul(one_minus_beta(k), H));
    }
  }
  if (threadIdx.x < 3) {
    const double rho = x[d.C + threadIdx.x] * invR;
    a.aux[blockIdx.x].inv_rho[threadIdx.x] = rho > 0.0 ? (float)(1.0 / rho) : 0.f;
  }
}

}  // namespace

cudaError_t launch_rowcol(const StepArgs& a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  k_rowcol<<<a.n_units, kT, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rowcol_finish(const StepArgs& a, int n_tensors, cudaStream_t s) {
  if (n_tensors == 0) return cudaSuccess;
  k_rowcol_finish<<<n_tensors, kT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace lopt

// ---- no-allocation entry point ----------------------------------------------
// lopt_rowcol_static() runs the kernel above for one tensor with all of its
// scratch (descriptor, unit table, per-tensor results, counter, column and
// row partials) carved from one fixed array in device memory, so it never
// calls cudaMalloc.  The array belongs to the library image: every GPU that
// loads the library holds LOPT_STATIC_SCRATCH_BYTES for it until the process
// exits, and all calls on a device share it.
namespace lopt {
namespace {

__device__ __align__(256) unsigned char g_rowcol_scratch[LOPT_STATIC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxScratchDevices] = {};

// Device address of the scratch array on the current device.  Host code may
// not use the symbol itself (it names a host-side stand-in), so the address
// is looked up once per device, with that device current, and cached.
int scratch_address(void** out) {
  int dev = -1;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) {
    cudaGetLastError();
    return record_cuda_error(ge);
  }
  if (dev < 0 || dev >= kMaxScratchDevices) return LOPT_E_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_rowcol_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LOPT_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Fills the scratch for one call from the kernel's parameters: the tensor's
// descriptor, its unit table (one unit per strip) and the zeroed counter
// and status words.  No host memory is involved.
__global__ void k_static_setup(TensorDesc d, TensorDesc* desc, Unit* units, int n_strips, int32_t* words) {
  const int tid = threadIdx.x;
  if (tid == 0) *desc = d;
  if (tid < 64) words[tid] = 0;
  for (int s = tid; s < n_strips; s += blockDim.x) units[s] = Unit{0, s};
}

}  // namespace
}  // namespace lopt

extern "C" int lopt_rowcol_static(const float* grad, float* const* row, float* const* col,
                                  int64_t rows, int64_t cols, float* inv_rho, void* stream_ptr) {
  using namespace lopt;
  if (!grad || !row || !col || !inv_rho) return LOPT_E_ARG;
  if (rows < 1 || cols < 1) return LOPT_E_SHAPE;
  if (rows > ((int64_t)1 << 31) || cols > ((int64_t)1 << 31) || rows * cols >= ((int64_t)1 << 31))
    return LOPT_E_SHAPE;
  struct Span { uintptr_t lo, hi; };
  std::vector<Span> spans = {{(uintptr_t)grad, (uintptr_t)grad + (uintptr_t)(rows * cols) * 4},
                             {(uintptr_t)inv_rho, (uintptr_t)inv_rho + 12}};
  for (int k = 0; k < 3; ++k) {
    if (!row[k] || !col[k]) return LOPT_E_ARG;
    spans.push_back({(uintptr_t)row[k], (uintptr_t)row[k] + (uintptr_t)rows * 4});
    spans.push_back({(uintptr_t)col[k], (uintptr_t)col[k] + (uintptr_t)cols * 4});
  }
  for (const Span& sp : spans)
    if (sp.lo % 4) return LOPT_E_ALIGN;
  std::sort(spans.begin(), spans.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
  for (size_t k = 1; k < spans.size(); ++k)
    if (spans[k].lo < spans[k - 1].hi) return LOPT_E_ALIAS;

  // Same strips as lopt_step(); with 16-byte aligned arrays both take the
  // 128-bit route, and then the results are the same bits.
  const int strip_rows = strip_rows_for(rows, cols);
  const int n_strips = (int)((rows + strip_rows - 1) / strip_rows);
  const size_t o_desc = 0;
  const size_t o_units = o_desc + round256(sizeof(TensorDesc));
  const size_t o_aux = o_units + round256(sizeof(Unit) * (size_t)n_strips);
  const size_t o_cnt = o_aux + round256(sizeof(TensorAux));
  const size_t o_row = o_cnt + 256;                       // counter + status
  const size_t o_col = o_row + round256(sizeof(double) * 3 * (size_t)n_strips);
  const size_t need = o_col + sizeof(float) * (size_t)n_strips * (size_t)cols;
  if (need > LOPT_STATIC_SCRATCH_BYTES) return LOPT_E_TOO_LARGE;

  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc != LOPT_OK) return rc;
  char* sc = static_cast<char*>(base);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);

  TensorDesc d;
  std::memset(&d, 0, sizeof(d));
  d.g = grad;
  for (int k = 0; k < 3; ++k) {
    d.r[k] = row[k];
    d.c[k] = col[k];
  }
  d.R = rows;
  d.C = cols;
  d.N = rows * cols;
  bool v4 = ((uintptr_t)grad & 15) == 0;
  for (int k = 0; k < 3; ++k) v4 = v4 && (((uintptr_t)col[k] & 15) == 0);
  d.vec4 = v4 ? 1 : 0;
  d.strip_rows = strip_rows;
  d.n_strips = n_strips;
  d.colpart_off = 0;
  d.rowpart_off = 0;
  cudaError_t e = cudaSuccess;
  {
    k_static_setup<<<1, 256, 0, stream>>>(d, reinterpret_cast<TensorDesc*>(sc + o_desc),
                                          reinterpret_cast<Unit*>(sc + o_units), n_strips,
                                          reinterpret_cast<int32_t*>(sc + o_cnt));
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    StepArgs a;
    std::memset(&a, 0, sizeof(a));
    a.desc = reinterpret_cast<const TensorDesc*>(sc + o_desc);
    a.units = reinterpret_cast<const Unit*>(sc + o_units);
    a.n_units = n_strips;
    a.aux = reinterpret_cast<TensorAux*>(sc + o_aux);
    a.counters = reinterpret_cast<int32_t*>(sc + o_cnt);
    a.status = reinterpret_cast<int32_t*>(sc + o_cnt + 16);
    a.rowpart = reinterpret_cast<double*>(sc + o_row);
    a.colpart = reinterpret_cast<float*>(sc + o_col);
    e = launch_rowcol(a, stream);
  }
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(inv_rho, sc + o_aux + offsetof(TensorAux, inv_rho), 3 * sizeof(float),
                        cudaMemcpyDeviceToDevice, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return record_cuda_error(e);
  }
  return LOPT_OK;
}
