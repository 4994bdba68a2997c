// K2 (tensor-core path): apply pass with the per-element MLP on tcgen05.
//
// Same computation as the FP32 apply kernel ("PyLO: Towards Accessible
// Learned Optimizers in PyTorch", section "融合カーネル戦略", kernel 2:
// features recomputed in registers, normalised, MLP, update written back),
// but the three MLP layers run as batched GEMMs on the 5th-generation tensor
// cores: the page's design evaluates the MLP on CUDA cores with __ldg
// weights, which on GB300 is ALU-bound (about 4.7 kFLOP per element against
// 44 bytes of traffic).
//
// One persistent CTA per SM, warp-specialised, linked by mbarriers:
//   warp 16      producer: bulk-copies (cp.async.bulk) p, g, m0..2, v of the
//                next tiles into a ring of shared-memory stages;
//   warps 8-15   two feature warpgroups (alternate tiles): EMA update,
//                features, normalisation, FP16 A tile of layer 1 into a tile
//                slot; they also store the updated accumulators m and v;
//   warp 17      MMA issuer (one thread);
//   warps 0-7    two epilogue warpgroups (alternate tiles; tensor-memory
//                lanes 0-127): ReLU + FP16 A tiles of layers 2 and 3, the
//                b2 preset of the layer-2 accumulator, and the update of p.
// A tile is 128 consecutive elements of one tensor (one per TMEM lane).
//
// Small MMAs (M=128, N<=32) cost about 40 cycles of the SM's MMA pipe each,
// whatever their K, so a tile uses as few as possible: FP16 operands with
// K = 32 for layer 1 (2 MMAs) and K = NP for layers 2 and 3 (2 MMAs each at
// NP = 32), biases without extra K columns, and one tcgen05.commit per
// issue iteration.  Stages of different tiles overlap with fixed lags: in
// iteration k the MMA thread issues layer 1 of tile k, layer 2 of tile k-5
// and layer 3 of tile k-11 (K-steps interleaved), then commits once; in step
// m an epilogue group finishes layer 1 of tile m-2, layer 2 of tile m-8 and
// the update of tile m-14.  No role waits on work issued in the same
// iteration, and at most 15 tiles are in flight (16 slots).
//
// The tiles of a CTA are processed in sessions: maximal runs of tiles whose
// tensors share one MLP weight set.  Between sessions the pipeline drains,
// the weights of the next set are loaded and the barriers restart.
//
// Every wait is bounded: on timeout the kernel raises the status flag, all
// roles stop, in-flight copies and MMAs are waited for (bounded) and tensor
// memory is freed.
#include <cuda_fp16.h>

#include "lopt.h"
#include "lopt_internal.cuh"
#include "tc_layout.cuh"

namespace lopt {
namespace {

constexpr int kTile = 128;                // elements per tile (= TMEM lanes)
constexpr int kThreads = 18 * 32;         // 8 epilogue + 8 feature + producer + MMA warps
constexpr int kSlots = 16;                // tiles in flight
constexpr int kRingStages = 20;           // input stages (one tile each)
constexpr int kStageBytes = 6 * kTile * 4;
constexpr int kDone = 8;                  // commit barriers (one per MMA iteration)
constexpr int kLag2 = 5, kLag3 = 11;      // MMA: layer 2 / 3 of tiles k-5 / k-11
constexpr int kE1 = 2, kE2 = 8, kE3 = 14; // epilogue step m: tiles m-2, m-8, m-14
constexpr int kProducerWarp = 16, kMmaWarp = 17;
constexpr uint64_t kWaitNs = 1000000000ull;

template <int NP>
struct Geom {
  static constexpr int Slot = kTile * 32 * 2;          // 8 KB: largest A tile (layer 1)
  static constexpr int SBO1 = 32 * 16;                 // layer-1 operands: K = 32
  static constexpr int SBO = NP * 16;                  // layer-2/3 operands: K = NP
  static constexpr int B1 = NP * 32 * 2;
  static constexpr int B2 = NP * NP * 2;
  static constexpr int B3 = 16 * NP * 2;
  static constexpr int Bias = (NP + 4) * 4;            // b2[NP], b3[2], pad
  static constexpr int Set = (B2 + B3 + Bias + 1023) / 1024 * 1024;   // packed per-set stride
  static constexpr int oSlots = 0;
  static constexpr int oRing = kSlots * Slot;
  static constexpr int oB1 = oRing + kRingStages * kStageBytes;
  static constexpr int oB2 = oB1 + B1;                  // B2, B3, b2, b3 as packed
  static constexpr int oBar = (oB2 + Set + 15) / 16 * 16;
  static constexpr int nBars = 2 * kRingStages + 4 * kSlots + kDone;
  static constexpr int oInfo = oBar + nBars * 8;
  static constexpr int Smem = oInfo + 64;
  static constexpr int TmemCols = kSlots * NP <= 256 ? 256 : 512;
  static constexpr uint32_t ID12 = instr_desc(0, 128, NP);
  static constexpr uint32_t ID3 = instr_desc(0, 128, 16);
  static_assert(Smem <= 232448, "shared memory of one CTA");
  static_assert(kSlots * NP <= 512, "tensor memory columns");
};

// Walks tiles in order: units [u, u1), 128-element tiles each.
struct TileWalk {
  const Unit* units;
  const TensorDesc* desc;
  int64_t u, u1;
  int tensor;
  int64_t start, end;
  __device__ void init(const Unit* un, const TensorDesc* de, int64_t b, int64_t e) {
    units = un; desc = de; u = b; u1 = e;
    load();
  }
  __device__ void load() {
    if (u < u1) {
      const Unit x = units[u];
      tensor = x.tensor;
      start = (int64_t)x.local * kApplyChunk;
      end = min(desc[tensor].N, start + (int64_t)kApplyChunk);
    }
  }
  __device__ void next() {
    start += kTile;
    if (start >= end) { ++u; load(); }
  }
};

__device__ __forceinline__ int64_t unit_tiles(const StepArgs& a, int64_t u) {
  const Unit x = a.units[u];
  const int64_t st = (int64_t)x.local * kApplyChunk;
  const int64_t en = min(a.desc[x.tensor].N, st + (int64_t)kApplyChunk);
  return (en - st + kTile - 1) / kTile;
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15) == 0 && global_ns() - t0 > limit_ns) return;
  }
}

// One FP16 A-operand row of layer 2 or 3: ReLU(h) in columns 0..NP-1.
template <int NP>
__device__ __forceinline__ void store_h_row(uint32_t slot_addr, int row, const uint32_t* h) {
  const uint32_t base = slot_addr + (row >> 3) * Geom<NP>::SBO + (row & 7) * 16;
#pragma unroll
  for (int kc = 0; kc < NP / 8; ++kc) {
    const float* f = reinterpret_cast<const float*>(h + 8 * kc);
    st_shared_v4(base + kc * 128, relu_f16x2(f[0], f[1]), relu_f16x2(f[2], f[3]),
                 relu_f16x2(f[4], f[5]), relu_f16x2(f[6], f[7]));
  }
}

template <int NP>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[NP]) {
  if constexpr (NP == 16) tmem_ld16(taddr, r);
  else tmem_ld32(taddr, r);
}
template <int NP>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint32_t (&r)[NP]) {
  if constexpr (NP == 16) tmem_st16(taddr, r);
  else tmem_st32(taddr, r);
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) k_apply_tc(StepArgs a) {
  static_assert(NP == 16 || NP == 32, "tensor-core path: padded hidden width 16 or 32");
  using G = Geom<NP>;
  constexpr int S = kSlots, R = kRingStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  float* ring = reinterpret_cast<float*>(smem + G::oRing);
  uint64_t* ring_full = reinterpret_cast<uint64_t*>(smem + G::oBar);
  uint64_t* ring_empty = ring_full + R;
  uint64_t* a1_full = ring_empty + R;
  uint64_t* a2_full = a1_full + S;
  uint64_t* a3_full = a2_full + S;
  uint64_t* slot_empty = a3_full + S;
  uint64_t* done = slot_empty + S;
  int64_t* info = reinterpret_cast<int64_t*>(smem + G::oInfo);   // session: end unit, tiles
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::oInfo + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::oInfo + 40);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t s_base = smem_u32(smem);

  if (tid == 0) *abort_flag = 0;
  if (warp == 0) tmem_alloc(tmem_slot, G::TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t U = a.n_units;
  const int64_t u_first = (int64_t)blockIdx.x * U / gridDim.x;
  const int64_t u_last = (int64_t)(blockIdx.x + 1) * U / gridDim.x;

  for (int64_t u0 = u_first; u0 < u_last;) {
    // ---- session set-up: tiles sharing one weight set --------------------------
    if (tid == 0) {
      const int wset = a.desc[a.units[u0].tensor].wset;
      int64_t u1 = u0, K = 0;
      while (u1 < u_last && a.desc[a.units[u1].tensor].wset == wset) K += unit_tiles(a, u1++);
      info[0] = u1;
      info[1] = K;
      for (int r = 0; r < R; ++r) {
        mbar_init(ring_full + r, 1);
        mbar_init(ring_empty + r, kTile);
      }
      for (int s = 0; s < S; ++s) {
        mbar_init(a1_full + s, kTile);
        mbar_init(a2_full + s, kTile);
        mbar_init(a3_full + s, kTile);
        mbar_init(slot_empty + s, kTile);
      }
      for (int s = 0; s < kDone; ++s) mbar_init(done + s, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {  // weights of the session's set: layer-1 operand of its first tensor,
       // then the packed layer-2/3 operands and biases
      const int t0 = a.units[u0].tensor;
      const uint4* src1 = reinterpret_cast<const uint4*>(a.w1fold + (int64_t)t0 * a.w1fold_stride);
      const uint4* src2 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.tc_weights) +
                                                         (int64_t)a.desc[t0].wset * G::Set);
      for (int o = tid; o < G::B1 / 16; o += kThreads) reinterpret_cast<uint4*>(smem + G::oB1)[o] = __ldg(src1 + o);
      for (int o = tid; o < G::Set / 16; o += kThreads) reinterpret_cast<uint4*>(smem + G::oB2)[o] = __ldg(src2 + o);
    }
    fence_proxy_async();
    __syncthreads();
    const int64_t u1 = info[0], K = info[1];
    if (*abort_flag) break;

    if (warp == kProducerWarp) {
      // ------------------------------ producer -------------------------------
      if (lane == 0) {
        TileWalk w;
        w.init(a.units, a.desc, u0, u1);
        int64_t k = 0;
        for (; k < K; ++k, w.next()) {
          const int st = (int)(k % R);
          if (!mbar_wait_or_abort(ring_empty + st, (uint32_t)((k / R) & 1) ^ 1u, kWaitNs, abort_flag)) break;
          const TensorDesc& d = a.desc[w.tensor];
          if (d.vec4 && (d.C % 4 == 0)) {
            const uint32_t bytes = (uint32_t)(min((int64_t)kTile, w.end - w.start) * 4);
            mbar_arrive_expect_tx(ring_full + st, 6 * bytes);
            float* dst = ring + st * (6 * kTile);
            bulk_g2s(dst + 0 * kTile, d.p + w.start, bytes, ring_full + st);
            bulk_g2s(dst + 1 * kTile, d.g + w.start, bytes, ring_full + st);
            bulk_g2s(dst + 2 * kTile, d.m[0] + w.start, bytes, ring_full + st);
            bulk_g2s(dst + 3 * kTile, d.m[1] + w.start, bytes, ring_full + st);
            bulk_g2s(dst + 4 * kTile, d.m[2] + w.start, bytes, ring_full + st);
            bulk_g2s(dst + 5 * kTile, d.v + w.start, bytes, ring_full + st);
          } else {
            mbar_arrive(ring_full + st);   // feature warps read global memory directly
          }
        }
        if (*abort_flag) {   // let copies already issued land before teardown
          for (int64_t kk = (k > R ? k - R : 0); kk < k; ++kk)
            mbar_drain(ring_full + kk % R, (uint32_t)((kk / R) & 1), kWaitNs / 10);
        }
      }
    } else if (warp >= 8 && warp < 16) {
      // --------------------------- feature warpgroups ------------------------
      const int grp = (warp - 8) >> 2;
      const int t = tid - 256 - 128 * grp;
      TileWalk w;
      w.init(a.units, a.desc, u0, u1);
      int cur = -1;
      bool vec = false, have_ij = false;
      int64_t i = 0, j = 0, last_e = 0, di = 0, dj = 0;
      float inv_rho[3] = {0.f, 0.f, 0.f};
      float sc[kStats];
#pragma unroll
      for (int q = 0; q < kStats; ++q) sc[q] = 0.f;
      for (int64_t k = 0; k < K; ++k, w.next()) {
        if ((int)(k & 1) != grp) continue;
        const int s = (int)(k % S), st = (int)(k % R);
        if (!mbar_wait_or_abort(slot_empty + s, (uint32_t)((k / S) & 1) ^ 1u, kWaitNs, abort_flag)) break;
        if (!mbar_wait_or_abort(ring_full + st, (uint32_t)((k / R) & 1), kWaitNs, abort_flag)) break;
        const TensorDesc& d = a.desc[w.tensor];
        if (w.tensor != cur) {
          cur = w.tensor;
          vec = d.vec4 && (d.C % 4 == 0);
#pragma unroll
          for (int q = 0; q < 3; ++q) inv_rho[q] = a.aux[cur].inv_rho[q];
#pragma unroll
          for (int q = 0; q < kStats; ++q) sc[q] = a.aux[cur].scale[q];
          di = (2 * kTile) / d.C;
          dj = (2 * kTile) - di * d.C;
          have_ij = false;
        }
        const int64_t e = w.start + t;
        const bool valid = e < w.end;
        float p = 0.f, g = 0.f, m[3] = {0.f, 0.f, 0.f}, v = 0.f;
        if (vec) {
          const float* rs = ring + st * (6 * kTile);
          if (valid) {
            p = rs[t]; g = rs[kTile + t]; m[0] = rs[2 * kTile + t]; m[1] = rs[3 * kTile + t];
            m[2] = rs[4 * kTile + t]; v = rs[5 * kTile + t];
          }
        } else if (valid) {
          p = __ldg(d.p + e); g = __ldg(d.g + e); v = __ldg(d.v + e);
#pragma unroll
          for (int q = 0; q < 3; ++q) m[q] = __ldg(d.m[q] + e);
        }
        mbar_arrive(ring_empty + st);
        float c[3] = {0.f, 0.f, 0.f};
        RowTerms rt;
#pragma unroll
        for (int q = 0; q < 3; ++q) { rt.rr[q] = 0.f; rt.sr[q] = 0.f; }
        if (valid) {
          if (have_ij && e == last_e + 2 * kTile) {
            i += di; j += dj;
            if (j >= d.C) { j -= d.C; ++i; }
          } else {
            i = e / d.C; j = e - i * d.C;
          }
          last_e = e;
          have_ij = true;
#pragma unroll
          for (int q = 0; q < 3; ++q) c[q] = __ldg(d.c[q] + j);
          rt = row_terms(d, inv_rho, i);
        } else {
          have_ij = false;
        }
        float f[kStats];
        lopt_features(p, g, m, v, rt, c, f);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 3; ++q) d.m[q][e] = m[q];
          d.v[e] = v;
        }
        // normalised features, FP16, into row t of the slot (K = 32)
        const uint32_t row = s_base + G::oSlots + s * G::Slot + (t >> 3) * G::SBO1 + (t & 7) * 16;
#pragma unroll
        for (int kc = 0; kc < 3; ++kc) {
          const int b = 8 * kc;
          st_shared_v4(row + kc * 128, f16x2(f[b] * sc[b], f[b + 1] * sc[b + 1]),
                       f16x2(f[b + 2] * sc[b + 2], f[b + 3] * sc[b + 3]),
                       f16x2(f[b + 4] * sc[b + 4], f[b + 5] * sc[b + 5]),
                       f16x2(f[b + 6] * sc[b + 6], f[b + 7] * sc[b + 7]));
        }
        st_shared_v4(row + 3 * 128, f16x2(f[24] * sc[24], f[25] * sc[25]),
                     f16x2(f[26] * sc[26], f[27] * sc[27]), 0x00003C00u /* 1.0h, 0 */, 0u);
        fence_proxy_async();
        mbar_arrive(a1_full + s);
      }
    } else if (warp == kMmaWarp) {
      // ------------------------------- MMA issuer ----------------------------
      if (lane == 0) {
        const uint32_t s_slots = s_base + G::oSlots;
        const uint64_t dB1 = smem_desc(s_base + G::oB1, 128, G::SBO1);
        const uint64_t dB2 = smem_desc(s_base + G::oB2, 128, G::SBO);
        const uint64_t dB3 = smem_desc(s_base + G::oB2 + G::B2, 128, G::SBO);
        int64_t k = 0;
        for (; k < K + kLag3; ++k) {
          if (*abort_flag) break;
          const bool do1 = k < K;
          const bool do2 = k >= kLag2 && k - kLag2 < K;
          const bool do3 = k >= kLag3 && k - kLag3 < K;
          const int64_t k2 = k - kLag2, k3 = k - kLag3;
          const int s1 = (int)(k % S), s2 = do2 ? (int)(k2 % S) : 0, s3 = do3 ? (int)(k3 % S) : 0;
          if (do1 && !mbar_wait_or_abort(a1_full + s1, (uint32_t)((k / S) & 1), kWaitNs, abort_flag)) break;
          if (do2 && !mbar_wait_or_abort(a2_full + s2, (uint32_t)((k2 / S) & 1), kWaitNs, abort_flag)) break;
          if (do3 && !mbar_wait_or_abort(a3_full + s3, (uint32_t)((k3 / S) & 1), kWaitNs, abort_flag)) break;
          tc_fence_after();
          const uint64_t dA1 = smem_desc(s_slots + s1 * G::Slot, 128, G::SBO1);
          const uint64_t dA2 = smem_desc(s_slots + s2 * G::Slot, 128, G::SBO);
          const uint64_t dA3 = smem_desc(s_slots + s3 * G::Slot, 128, G::SBO);
          // K-steps of the three layers interleaved (independent accumulators)
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            if (do1) mma_f16(tmem + s1 * NP, dA1 + 16 * kk, dB1 + 16 * kk, G::ID12, kk > 0);
            if (kk < NP / 16) {
              if (do2) mma_f16(tmem + s2 * NP, dA2 + 16 * kk, dB2 + 16 * kk, G::ID12, 1u);   // onto b2
              if (do3) mma_f16(tmem + s3 * NP, dA3 + 16 * kk, dB3 + 16 * kk, G::ID3, kk > 0);
            }
          }
          mma_commit(done + (k % kDone));   // tracks every MMA issued so far
        }
        // nothing of ours may still be running when the session ends
        if (k > 0) mbar_drain(done + ((k - 1) % kDone), (uint32_t)(((k - 1) / kDone) & 1), kWaitNs / 10);
      }
    } else if (warp < 8) {
      // ------------------------------ epilogue -------------------------------
      // Group h takes the tiles k with k % 2 == h.  In step m it finishes
      // layer 1 of tile m-2 (and presets the layer-2 accumulator to b2),
      // layer 2 of tile m-8 and the update of tile m-14; it loads p of tile
      // m-12 for the update two steps later.
      const int h = warp >> 2;
      const int t = tid - 128 * h;
      const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t s_slots = s_base + G::oSlots;
      const float* bias = reinterpret_cast<const float*>(smem + G::oB2 + G::B2 + G::B3);
      uint32_t b2[NP];
#pragma unroll
      for (int q = 0; q < NP; ++q) b2[q] = __float_as_uint(bias[q]);
      const float b30 = bias[NP], b31 = bias[NP + 1];
      TileWalk wp;   // tile m-12 of this group
      wp.init(a.units, a.desc, u0, u1);
      if (h == 1) wp.next();
      const float lr = a.lr;
      float* p_ptr_prev = nullptr;
      float p_prev = 0.f;
      for (int64_t m = h; m - kE3 < K; m += 2) {
        if (*abort_flag) break;
        const int64_t t1 = m - kE1, t2 = m - kE2, t3 = m - kE3, tp = m - (kE3 - 2);
        float* p_ptr_next = nullptr;
        float p_next = 0.f;
        if (tp >= 0 && tp < K) {
          const int64_t e = wp.start + t;
          if (e < wp.end) {
            p_ptr_next = a.desc[wp.tensor].p + e;
            p_next = *p_ptr_next;
          }
          wp.next();
          wp.next();
        }
        if (t1 >= 0 && t1 < K) {
          const int s = (int)(t1 % S);
          if (!mbar_wait_or_abort(done + (t1 % kDone), (uint32_t)((t1 / kDone) & 1), kWaitNs, abort_flag)) break;
          tc_fence_after();
          uint32_t hv[NP];
          tmem_ld_row<NP>(t_lane + s * NP, hv);
          tmem_wait_ld();
          store_h_row<NP>(s_slots + s * G::Slot, t, hv);
          tmem_st_row<NP>(t_lane + s * NP, b2);
          tmem_wait_st();
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(a2_full + s);
        }
        if (t2 >= 0 && t2 < K) {
          const int s = (int)(t2 % S);
          const int64_t it = t2 + kLag2;
          if (!mbar_wait_or_abort(done + (it % kDone), (uint32_t)((it / kDone) & 1), kWaitNs, abort_flag)) break;
          tc_fence_after();
          uint32_t hv[NP];
          tmem_ld_row<NP>(t_lane + s * NP, hv);
          tmem_wait_ld();
          store_h_row<NP>(s_slots + s * G::Slot, t, hv);
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(a3_full + s);
        }
        if (t3 >= 0 && t3 < K) {
          const int s = (int)(t3 % S);
          const int64_t it = t3 + kLag3;
          if (!mbar_wait_or_abort(done + (it % kDone), (uint32_t)((it / kDone) & 1), kWaitNs, abort_flag)) break;
          tc_fence_after();
          uint32_t o[2];
          tmem_ld2(t_lane + s * NP, o);
          tmem_wait_ld();
          if (p_ptr_prev) {
            const float o0 = __uint_as_float(o[0]) + b30, o1 = __uint_as_float(o[1]) + b31;
            const float upd = o0 * expf(o1 * kOutScale) * kOutScale;
            *p_ptr_prev = p_prev - lr * upd;
          }
          tc_fence_before();
          mbar_arrive(slot_empty + s);
        }
        p_ptr_prev = p_ptr_next;
        p_prev = p_next;
      }
    }
    // ---- session end: every role has finished its tiles --------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    u0 = u1;
  }

  // ------------------------------- teardown ----------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TmemCols);
  }
  if (tid == 0 && *abort_flag) atomicOr(a.status, kStatusTimeout);
}

// Packs the layer-2 and layer-3 operands of every weight set (FP16,
// canonical K-major) and its biases b2, b3 (FP32) from the caller-layout
// weights at padded width hp.
template <int NP>
__global__ void k_pack_tc(const float* weights, int hp, int set_size, int n_sets, uint8_t* out) {
  using G = Geom<NP>;
  const int per = NP * NP + 16 * NP + NP + 4;
  const int64_t total = (int64_t)n_sets * per;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int s = (int)(x / per);
    int r = (int)(x - (int64_t)s * per);
    const float* W = weights + (int64_t)s * set_size;
    uint8_t* base = out + (int64_t)s * G::Set;
    if (r < NP * NP) {                        // B2[n][k] = W2[k][n]
      const int n = r / NP, k = r % NP;
      const float v = (n < hp && k < hp) ? W[w_off_W2(hp) + k * hp + n] : 0.f;
      reinterpret_cast<__half*>(base)[f16_off(n, k, NP)] = __float2half_rn(v);
    } else if ((r -= NP * NP) < 16 * NP) {    // B3[n][k] = W3[k][n], n < 2
      const int n = r / NP, k = r % NP;
      const float v = (n < 2 && k < hp) ? W[w_off_W3(hp) + 2 * k + n] : 0.f;
      reinterpret_cast<__half*>(base + G::B2)[f16_off(n, k, NP)] = __float2half_rn(v);
    } else {                                  // b2[NP], b3[2], pad
      r -= 16 * NP;
      float v = 0.f;
      if (r < NP) v = r < hp ? W[w_off_b2(hp) + r] : 0.f;
      else if (r < NP + 2) v = W[w_off_b3(hp) + (r - NP)];
      reinterpret_cast<float*>(base + G::B2 + G::B3)[r] = v;
    }
  }
}

template <int NP>
cudaError_t launch_np(const StepArgs& a, cudaStream_t s) {
  using G = Geom<NP>;
  static int sms = 0;
  if (sms == 0) {
    cudaError_t e = cudaFuncSetAttribute(k_apply_tc<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::Smem);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  // one persistent CTA per SM (its shared memory and tensor memory fill the SM)
  const int grid = a.n_units < sms ? a.n_units : sms;
  k_apply_tc<NP><<<grid, kThreads, G::Smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool apply_tc_supported(int hidden) {
  return hidden == 4 || hidden == 8 || hidden == 16 || hidden == 32;
}

int w1fold_floats(int hidden, int path) {
  if (path == LOPT_MLP_TC) return tc_np(hidden) * 16;   // FP16 [NP x 32]
  return (kStats + 1) * hidden;
}

size_t tc_weights_bytes(int hidden, int n_sets) {
  switch (tc_np(hidden)) {
    case 16: return (size_t)n_sets * Geom<16>::Set;
    case 32: return (size_t)n_sets * Geom<32>::Set;
  }
  return 0;
}

cudaError_t pack_tc_weights(const float* weights, int hidden, int n_sets, void* out, cudaStream_t s) {
  const int ss = w_set_size(hidden);
  switch (tc_np(hidden)) {
    case 16: k_pack_tc<16><<<64, 256, 0, s>>>(weights, hidden, ss, n_sets, (uint8_t*)out); break;
    case 32: k_pack_tc<32><<<64, 256, 0, s>>>(weights, hidden, ss, n_sets, (uint8_t*)out); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_apply_tc(const StepArgs& a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  switch (tc_np(a.hidden)) {
    case 16: return launch_np<16>(a, s);
    case 32: return launch_np<32>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lopt
