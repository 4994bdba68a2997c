// K2 (tensor-core path): apply pass with the per-element MLP on tcgen05.
//
// Same computation as the FP32 apply kernel ("PyLO: Towards Accessible
// Learned Optimizers in PyTorch", section "融合カーネル戦略", kernel 2:
// features recomputed in registers, normalised, MLP, update written back),
// but the MLP layers run as batched GEMMs on the 5th-generation tensor cores:
// the page's design evaluates the MLP on CUDA cores with __ldg weights, which
// on GB300 is ALU-bound (about 4.7 kFLOP per element against 44 bytes).
//
// One CTA = 128 threads = one 128-lane tensor-memory accumulator.  A round
// covers 512 consecutive elements: thread t owns elements 4t..4t+3 and row t
// of four M=128 tiles (tile q holds elements 4t+q).  Per round:
//   features -> smem A1 (TF32) -> MMA layer 1 -> TMEM
//   TMEM -> ReLU/FP16 -> smem A2 -> MMA layer 2 -> TMEM
//   TMEM -> ReLU/FP16 -> smem A3 -> MMA layer 3 -> TMEM -> update, store.
// One elected thread issues the MMAs; completion is tracked by an mbarrier
// (tcgen05.commit).  Every wait is bounded; on timeout the kernel raises the
// status flag, stops issuing work, frees its tensor memory and returns.
// The CTA grid is persistent (a contiguous range of work units per CTA), so
// layer weights are reloaded only when the tensor changes.
#include <cuda_fp16.h>

#include "lopt.h"
#include "lopt_internal.cuh"
#include "tc_layout.cuh"

namespace lopt {
namespace {

constexpr int kT = 128;
constexpr int kTiles = 4;
constexpr int kRound = kT * kTiles;   // 512 elements
constexpr uint64_t kWaitNs = 1000000000ull;

template <int NP>
struct Geom {
  static constexpr int K2 = tc_k2(NP);
  static constexpr int A1 = 128 * 32 * 4;
  static constexpr int A2 = 128 * K2 * 2;
  static constexpr int Tile = ((A1 > A2 ? A1 : A2) + 1023) / 1024 * 1024;
  static constexpr int B1 = NP * 32 * 4;
  static constexpr int B2 = NP * K2 * 2;
  static constexpr int B3 = 16 * K2 * 2;
  static constexpr int B23 = (B2 + B3 + 1023) / 1024 * 1024;   // packed per-set stride
  static constexpr int oB1 = kTiles * Tile;
  static constexpr int oB2 = oB1 + B1;
  static constexpr int oB3 = oB2 + B2;
  static constexpr int oBar = (oB3 + B3 + 15) / 16 * 16;
  static constexpr int Smem = oBar + 64;
  static constexpr int Cols = kTiles * NP;
  static constexpr int TmemCols = Cols <= 32 ? 32 : Cols <= 64 ? 64 : Cols <= 128 ? 128 : 256;
  static constexpr int SBO2 = K2 * 16;                 // bytes between 8-row groups (f16)
  static constexpr uint32_t ID1 = instr_desc(2, 128, NP);
  static constexpr uint32_t ID2 = instr_desc(0, 128, NP);
  static constexpr uint32_t ID3 = instr_desc(0, 128, 16);
};

// Copy `bytes` (multiple of 16) from global to shared memory.
__device__ __forceinline__ void copy_g2s(uint8_t* dst, const uint8_t* src, int bytes) {
  for (int o = threadIdx.x * 16; o < bytes; o += kT * 16)
    *reinterpret_cast<uint4*>(dst + o) = __ldg(reinterpret_cast<const uint4*>(src + o));
}

// Writes one FP16 A-operand row (h values of this thread's tile row), with
// the constant-1 bias column at k = NP and zeros up to K2.
template <int NP>
__device__ __forceinline__ void store_h_row(uint32_t tile_addr, int row, const uint32_t* h) {
  using G = Geom<NP>;
  const uint32_t base = tile_addr + (row >> 3) * G::SBO2 + (row & 7) * 16;
#pragma unroll
  for (int kc = 0; kc < NP / 8; ++kc) {
    const float* f = reinterpret_cast<const float*>(h + 8 * kc);
    st_shared_v4(base + kc * 128, relu_f16x2(f[0], f[1]), relu_f16x2(f[2], f[3]),
                 relu_f16x2(f[4], f[5]), relu_f16x2(f[6], f[7]));
  }
  st_shared_v4(base + (NP / 8) * 128, 0x3C00u /* 1.0h, 0 */, 0u, 0u, 0u);
#pragma unroll
  for (int kc = NP / 8 + 1; kc < G::K2 / 8; ++kc) st_shared_v4(base + kc * 128, 0u, 0u, 0u, 0u);
}

template <int NP>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[NP]) {
  if constexpr (NP == 16) {
    tmem_ld16(taddr, r);
  } else {
#pragma unroll
    for (int c = 0; c < NP / 32; ++c)
      tmem_ld32(taddr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
  }
}

struct Elems {
  float p[4], g[4], m[3][4], v[4], c[3][4];
  RowTerms rt[4];
  bool ok[4];
};

__device__ __forceinline__ void load_elems(const TensorDesc& d, const float inv_rho[3], int64_t eb,
                                           int64_t e1, int64_t i, int64_t j, bool vec, Elems& x) {
  if (vec && eb + 3 < e1) {
    const float4 p4 = __ldg(reinterpret_cast<const float4*>(d.p + eb));
    const float4 g4 = __ldg(reinterpret_cast<const float4*>(d.g + eb));
    const float4 v4 = __ldg(reinterpret_cast<const float4*>(d.v + eb));
    x.p[0] = p4.x; x.p[1] = p4.y; x.p[2] = p4.z; x.p[3] = p4.w;
    x.g[0] = g4.x; x.g[1] = g4.y; x.g[2] = g4.z; x.g[3] = g4.w;
    x.v[0] = v4.x; x.v[1] = v4.y; x.v[2] = v4.z; x.v[3] = v4.w;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const float4 m4 = __ldg(reinterpret_cast<const float4*>(d.m[k] + eb));
      x.m[k][0] = m4.x; x.m[k][1] = m4.y; x.m[k][2] = m4.z; x.m[k][3] = m4.w;
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(d.c[k] + j));
      x.c[k][0] = c4.x; x.c[k][1] = c4.y; x.c[k][2] = c4.z; x.c[k][3] = c4.w;
    }
    const RowTerms rt = row_terms(d, inv_rho, i);
#pragma unroll
    for (int q = 0; q < 4; ++q) { x.rt[q] = rt; x.ok[q] = true; }
    return;
  }
  int64_t ii = i, jj = j;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int64_t e = eb + q;
    x.ok[q] = e < e1;
    const int64_t es = x.ok[q] ? e : (eb < e1 ? eb : e1 - 1);
    const int64_t iq = x.ok[q] ? ii : 0, jq = x.ok[q] ? jj : 0;   // in-bounds for idle lanes
    x.p[q] = __ldg(d.p + es);
    x.g[q] = __ldg(d.g + es);
    x.v[q] = __ldg(d.v + es);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      x.m[k][q] = __ldg(d.m[k] + es);
      x.c[k][q] = __ldg(d.c[k] + jq);
    }
    x.rt[q] = row_terms(d, inv_rho, iq);
    if (++jj == d.C) { jj = 0; ++ii; }
  }
}

template <int NP>
__global__ void __launch_bounds__(kT) k_apply_tc(StepArgs a) {
  using G = Geom<NP>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + G::oBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::oBar + 8);

  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t s_b1 = s_base + G::oB1, s_b2 = s_base + G::oB2, s_b3 = s_base + G::oB3;

  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, G::TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);

  // Descriptor of every operand at K-step 0; step s adds s*256 bytes, i.e.
  // 16 to the start-address field (no carry: all addresses < 256 KB).
  const uint64_t dA1 = smem_desc(s_base, 128, 1024), dA2 = smem_desc(s_base, 128, G::SBO2);
  const uint64_t dB1 = smem_desc(s_b1, 128, 1024), dB2 = smem_desc(s_b2, 128, G::SBO2);
  const uint64_t dB3 = smem_desc(s_b3, 128, G::SBO2);
  constexpr uint64_t kTileStep = (uint64_t)(G::Tile >> 4);

  const int64_t U = a.n_units;
  const int64_t u0 = (int64_t)blockIdx.x * U / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * U / gridDim.x;
  uint32_t phase = 0;
  int timed_out = 0;
  int cur_tensor = -1, cur_set = -1;
  float inv_rho[3] = {0.f, 0.f, 0.f};
  const float lr = a.lr;

  for (int64_t ui = u0; ui < u1; ++ui) {
    const Unit u = a.units[ui];
    const TensorDesc& d = a.desc[u.tensor];
    const int64_t N = d.N, C = d.C;
    const bool vec = d.vec4 && (C % 4 == 0);
    if (u.tensor != cur_tensor) {
      // No MMA is in flight here: every round waits for its last commit.
      const int wset = d.wset;
      copy_g2s(smem + G::oB1,
               reinterpret_cast<const uint8_t*>(a.w1fold + (int64_t)u.tensor * a.w1fold_stride), G::B1);
      if (wset != cur_set) {
        copy_g2s(smem + G::oB2, reinterpret_cast<const uint8_t*>(a.tc_weights) + (int64_t)wset * G::B23,
                 G::B2 + G::B3);
        cur_set = wset;
      }
#pragma unroll
      for (int k = 0; k < 3; ++k) inv_rho[k] = a.aux[u.tensor].inv_rho[k];
      cur_tensor = u.tensor;
      fence_proxy_async();
    }
    const int64_t e0 = (int64_t)u.local * kApplyChunk;
    const int64_t e1 = min(N, e0 + (int64_t)kApplyChunk);
    int64_t eb = e0 + 4 * tid;
    int64_t i = min(eb, N - 1) / C;
    int64_t j = min(eb, N - 1) - i * C;
    const int64_t di = kRound / C, dj = kRound - di * C;

    for (int64_t base = e0; base < e1; base += kRound, eb += kRound) {
      if (vec && tid < 6 && base + 2 * kRound <= e1) {
        // bring the next round's element arrays into L2 while this one runs
        const float* arr = tid == 0 ? d.p : tid == 1 ? d.g : tid == 2 ? d.v : d.m[tid - 3];
        prefetch_l2(arr + base + kRound, kRound * 4);
      }
      Elems x;
      load_elems(d, inv_rho, eb, e1, i, j, vec, x);
      // ---- features -> A1 (TF32), one row per tile -------------------------
#pragma unroll
      for (int q = 0; q < kTiles; ++q) {
        float f[kStats];
        float m[3] = {x.m[0][q], x.m[1][q], x.m[2][q]};
        float v = x.v[q];
        const float c[3] = {x.c[0][q], x.c[1][q], x.c[2][q]};
        lopt_features(x.p[q], x.g[q], m, v, x.rt[q], c, f);
#pragma unroll
        for (int k = 0; k < 3; ++k) x.m[k][q] = m[k];
        x.v[q] = v;
        const uint32_t row = s_base + q * G::Tile + (tid >> 3) * 1024 + (tid & 7) * 16;
#pragma unroll
        for (int kc = 0; kc < 7; ++kc) {
          st_shared_v4(row + kc * 128, __float_as_uint(tf32_round(f[4 * kc])),
                       __float_as_uint(tf32_round(f[4 * kc + 1])),
                       __float_as_uint(tf32_round(f[4 * kc + 2])),
                       __float_as_uint(tf32_round(f[4 * kc + 3])));
        }
        st_shared_v4(row + 7 * 128, __float_as_uint(1.0f), 0u, 0u, 0u);
      }
      fence_proxy_async();
      tc_fence_before();
      if (__syncthreads_or(timed_out)) goto bail;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < kTiles; ++q) {
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_tf32(tmem + q * NP, dA1 + q * kTileStep + 16 * s, dB1 + 16 * s, G::ID1, s > 0);
        }
        mma_commit(bar);
      }
      if (!mbar_wait_bounded(bar, phase, kWaitNs)) timed_out = 1;
      phase ^= 1;
      tc_fence_after();
      // ---- layer-1 epilogue: ReLU, FP16 -> A2 -------------------------------
#pragma unroll
      for (int q = 0; q < kTiles; ++q) {
        uint32_t h[NP];
        tmem_ld_row<NP>(t_lane + q * NP, h);
        tmem_wait_ld();
        store_h_row<NP>(s_base + q * G::Tile, tid, h);
      }
      fence_proxy_async();
      tc_fence_before();
      if (__syncthreads_or(timed_out)) goto bail;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < kTiles; ++q) {
#pragma unroll
          for (int s = 0; s < G::K2 / 16; ++s)
            mma_f16(tmem + q * NP, dA2 + q * kTileStep + 16 * s, dB2 + 16 * s, G::ID2, s > 0);
        }
        mma_commit(bar);
      }
      if (!mbar_wait_bounded(bar, phase, kWaitNs)) timed_out = 1;
      phase ^= 1;
      tc_fence_after();
      // ---- layer-2 epilogue -> A3 --------------------------------------------
#pragma unroll
      for (int q = 0; q < kTiles; ++q) {
        uint32_t h[NP];
        tmem_ld_row<NP>(t_lane + q * NP, h);
        tmem_wait_ld();
        store_h_row<NP>(s_base + q * G::Tile, tid, h);
      }
      fence_proxy_async();
      tc_fence_before();
      if (__syncthreads_or(timed_out)) goto bail;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < kTiles; ++q) {
#pragma unroll
          for (int s = 0; s < G::K2 / 16; ++s)
            mma_f16(tmem + q * NP, dA2 + q * kTileStep + 16 * s, dB3 + 16 * s, G::ID3, s > 0);
        }
        mma_commit(bar);
      }
      if (!mbar_wait_bounded(bar, phase, kWaitNs)) timed_out = 1;
      phase ^= 1;
      tc_fence_after();
      // ---- output: update and store ------------------------------------------
      float pn[4];
#pragma unroll
      for (int q = 0; q < kTiles; ++q) {
        uint32_t o[2];
        tmem_ld2(t_lane + q * NP, o);
        tmem_wait_ld();
        const float o0 = __uint_as_float(o[0]), o1 = __uint_as_float(o[1]);
        const float upd = o0 * expf(o1 * kOutScale) * kOutScale;
        pn[q] = x.p[q] - lr * upd;
      }
      tc_fence_before();
      if (!timed_out) {
        if (vec && eb + 3 < e1) {
          *reinterpret_cast<float4*>(d.p + eb) = make_float4(pn[0], pn[1], pn[2], pn[3]);
          *reinterpret_cast<float4*>(d.v + eb) = make_float4(x.v[0], x.v[1], x.v[2], x.v[3]);
#pragma unroll
          for (int k = 0; k < 3; ++k)
            *reinterpret_cast<float4*>(d.m[k] + eb) =
                make_float4(x.m[k][0], x.m[k][1], x.m[k][2], x.m[k][3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (!x.ok[q]) continue;
            d.p[eb + q] = pn[q];
            d.v[eb + q] = x.v[q];
#pragma unroll
            for (int k = 0; k < 3; ++k) d.m[k][eb + q] = x.m[k][q];
          }
        }
      }
      // advance (row, column) by one round
      i += di;
      j += dj;
      if (j >= C) { j -= C; ++i; }
    }
  }

bail:
  if (timed_out) {
    atomicOr(a.status, kStatusTimeout);
    // give an MMA that may still be in flight one more bounded chance
    mbar_wait_bounded(bar, phase, kWaitNs / 10);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TmemCols);
  }
}

// Packs the layer-2 and layer-3 B operands of every weight set (FP16,
// canonical K-major) from the caller-layout weights at padded width hp.
template <int NP>
__global__ void k_pack_tc(const float* weights, int hp, int set_size, int n_sets, uint8_t* out) {
  using G = Geom<NP>;
  const int per = NP * G::K2 + 16 * G::K2;
  const int64_t total = (int64_t)n_sets * per;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int s = (int)(x / per);
    int r = (int)(x - (int64_t)s * per);
    const float* W = weights + (int64_t)s * set_size;
    __half* dst = reinterpret_cast<__half*>(out + (int64_t)s * G::B23);
    float v = 0.f;
    if (r < NP * G::K2) {            // B2[n][k]
      const int n = r / G::K2, k = r % G::K2;
      if (n < hp && k < hp) v = W[w_off_W2(hp) + k * hp + n];
      else if (n < hp && k == NP) v = W[w_off_b2(hp) + n];
      dst[f16_off(n, k, G::K2)] = __float2half_rn(v);
    } else {                         // B3[n][k], n < 16
      r -= NP * G::K2;
      const int n = r / G::K2, k = r % G::K2;
      if (n < 2 && k < hp) v = W[w_off_W3(hp) + 2 * k + n];
      else if (n < 2 && k == NP) v = W[w_off_b3(hp) + n];
      dst[G::B2 / 2 + f16_off(n, k, G::K2)] = __float2half_rn(v);
    }
  }
}

template <int NP>
cudaError_t launch_np(const StepArgs& a, cudaStream_t s) {
  using G = Geom<NP>;
  static int blocks = 0;
  if (blocks == 0) {
    cudaError_t e = cudaFuncSetAttribute(k_apply_tc<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_apply_tc<NP>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, occ = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_apply_tc<NP>, kT, G::Smem);
    if (e != cudaSuccess) return e;
    occ = occ < 512 / G::TmemCols ? occ : 512 / G::TmemCols;   // tensor-memory columns per SM
    blocks = (occ < 1 ? 1 : occ) * sms;
  }
  const int grid = a.n_units < blocks ? a.n_units : blocks;
  k_apply_tc<NP><<<grid, kT, G::Smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool apply_tc_supported(int hidden) {
  return hidden == 4 || hidden == 8 || hidden == 16 || hidden == 32 || hidden == 64;
}

int w1fold_floats(int hidden, int path) {
  if (path == LOPT_MLP_TC) return tc_np(hidden) * 32;
  return (kStats + 1) * hidden;
}

size_t tc_weights_bytes(int hidden, int n_sets) {
  switch (tc_np(hidden)) {
    case 16: return (size_t)n_sets * Geom<16>::B23;
    case 32: return (size_t)n_sets * Geom<32>::B23;
    case 64: return (size_t)n_sets * Geom<64>::B23;
  }
  return 0;
}

cudaError_t pack_tc_weights(const float* weights, int hidden, int n_sets, void* out, cudaStream_t s) {
  const int ss = w_set_size(hidden);
  switch (tc_np(hidden)) {
    case 16: k_pack_tc<16><<<64, 256, 0, s>>>(weights, hidden, ss, n_sets, (uint8_t*)out); break;
    case 32: k_pack_tc<32><<<64, 256, 0, s>>>(weights, hidden, ss, n_sets, (uint8_t*)out); break;
    case 64: k_pack_tc<64><<<64, 256, 0, s>>>(weights, hidden, ss, n_sets, (uint8_t*)out); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_apply_tc(const StepArgs& a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  switch (tc_np(a.hidden)) {
    case 16: return launch_np<16>(a, s);
    case 32: return launch_np<32>(a, s);
    case 64: return launch_np<64>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lopt
