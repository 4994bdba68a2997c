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
//   warp 16      producer: bulk-copies (cp.async.bulk, one array per lane) p,
//                g, m0..2, v of the next 8 tiles of a work unit into a ring
//                of shared-memory stages;
//   warps 8-15   two feature warpgroups (alternate tiles): EMA update,
//                features, normalisation, FP16 A operand of layer 1 into the
//                tile slot's tensor memory; they also store the updated
//                accumulators m and v;
//   warp 17      MMA issuer (one thread);
//   warps 0-7    two epilogue warpgroups (alternate tiles): ReLU + FP16 A
//                operand of layer 2 (in tensor memory) and the b2 preset of
//                its accumulator; then ReLU(h2), the two-unit output layer in
//                FP32 on the CUDA cores, and the update of p.
// A tile is 128 consecutive elements of one tensor (one per TMEM lane).  A
// tile slot is a set of tensor-memory columns: the FP32 accumulator (NP
// columns) and the FP16 A operand of the next MMA (16 columns); the A
// operands never pass through shared memory.
//
// Small MMAs (M=128, N<=32) cost about 40-50 cycles of the SM's MMA pipe
// each, whatever their K, and an MMA's result reaches a waiting thread about
// a thousand cycles after issue.  So a tile uses few MMAs (FP16 operands,
// K = 32 for layer 1 and K = NP for layer 2: 4 MMAs at NP = 32, biases
// without extra K columns, one tcgen05.commit per issue iteration) and only
// two MMA round trips: the output layer (two units) runs on the CUDA cores.
// Stages of different tiles overlap with fixed lags chosen for the largest
// slack around that latency: in iteration k the MMA thread issues layer 1 of
// tile k and layer 2 of tile k-5 (K-steps interleaved), then commits once;
// in step m an epilogue group finishes layer 1 of tile m-4 and the rest of
// tile m-8.  At most 9 tiles are in flight (10 slots at NP = 32).
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
constexpr int kStageTiles = 8;            // tiles per input stage (4 KB per array)
constexpr int kStageElems = kStageTiles * kTile;
constexpr int kRingStages = 5;            // input stages
constexpr int kStageBytes = 6 * kStageElems * 4;
constexpr int kDone = 8;                  // commit barriers (one per MMA iteration)
constexpr int kLag2 = 5;                  // MMA iteration k: layer 2 of tile k-5
constexpr int kE1 = 4, kE2 = 8;           // epilogue step m: tiles m-4, m-8
constexpr int kProducerWarp = 16, kMmaWarp = 17;
constexpr uint64_t kWaitNs = 1000000000ull;

template <int NP>
struct Geom {
  static constexpr int ACols = 16;                     // A operand: 32 FP16 per row
  static constexpr int SlotCols = NP + ACols;          // accumulator + A operand
  static constexpr int S = 512 / SlotCols < 16 ? 512 / SlotCols : 16;   // tiles in flight
  static constexpr int SBO1 = 32 * 16;                 // layer-1 B operand: K = 32
  static constexpr int SBO = NP * 16;                  // layer-2/3 B operands: K = NP
  static constexpr int B1 = NP * 32 * 2;
  static constexpr int B2 = NP * NP * 2;
  static constexpr int Aux = (3 * NP + 4) * 4;         // b2[NP], W3 pairs[NP][2], b3[2], pad
  static constexpr int Set = (B2 + Aux + 1023) / 1024 * 1024;   // packed per-set stride
  static constexpr int oRing = 0;
  static constexpr int oB1 = oRing + kRingStages * kStageBytes;
  static constexpr int oB2 = oB1 + B1;                  // B2, b2, W3, b3 as packed
  static constexpr int oBar = (oB2 + Set + 15) / 16 * 16;
  static constexpr int nBars = 2 * kRingStages + 3 * S + kDone;
  static constexpr int oInfo = oBar + nBars * 8;
  static constexpr int Smem = oInfo + 64;
  static constexpr int TmemCols = 512;
  static constexpr uint32_t ID12 = instr_desc(0, 128, NP);
  static_assert(Smem <= 232448, "shared memory of one CTA");
  static_assert(S * SlotCols <= 512 && S > kE2, "tensor memory columns / pipeline depth");
};

// Walks tiles in order: units [u, u1), 128-element tiles each.
struct TileWalk {
  const Unit* units;
  const TensorDesc* desc;
  int64_t u, u1;
  int tensor;
  int64_t ustart, start, end;   // unit start, tile start, unit end
  __device__ void init(const Unit* un, const TensorDesc* de, int64_t b, int64_t e) {
    units = un; desc = de; u = b; u1 = e;
    load();
  }
  __device__ void load() {
    if (u < u1) {
      const Unit x = units[u];
      tensor = x.tensor;
      ustart = start = (int64_t)x.local * kApplyChunk;
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

// ReLU + FP16 of one accumulator row, packed two per 32-bit column (16
// columns: the A operand of the next layer, zero-padded past NP).
template <int NP>
__device__ __forceinline__ void pack_relu_row(const uint32_t (&h)[NP], uint32_t (&av)[16]) {
#pragma unroll
  for (int q = 0; q < 16; ++q)
    av[q] = 2 * q < NP ? relu_f16x2(__uint_as_float(h[2 * q]), __uint_as_float(h[2 * q + 1])) : 0u;
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
  constexpr int S = G::S, R = kRingStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  float* ring = reinterpret_cast<float*>(smem + G::oRing);
  uint64_t* ring_full = reinterpret_cast<uint64_t*>(smem + G::oBar);
  uint64_t* ring_empty = ring_full + R;
  uint64_t* a1_full = ring_empty + R;
  uint64_t* a2_full = a1_full + S;
  uint64_t* slot_empty = a2_full + S;
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
        mbar_init(ring_empty + r, 2 * kTile);   // every feature thread, once per stage
      }
      for (int s = 0; s < S; ++s) {
        mbar_init(a1_full + s, kTile);
        mbar_init(a2_full + s, kTile);
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
      // A stage holds up to 8 consecutive tiles of one work unit; lane q < 6
      // copies array q of the stage.
      int64_t n_st = 0;
      for (int64_t u = u0; u < u1 && !*abort_flag; ++u) {
        const Unit x = a.units[u];
        const TensorDesc& d = a.desc[x.tensor];
        const bool vec = d.vec4 && (d.C % 4 == 0);
        const int64_t ue = min(d.N, (int64_t)x.local * kApplyChunk + kApplyChunk);
        const float* src = lane == 0 ? d.p : lane == 1 ? d.g : lane == 2 ? d.m[0] : lane == 3 ? d.m[1]
                         : lane == 4 ? d.m[2] : d.v;
        bool stop = false;
        for (int64_t e0 = (int64_t)x.local * kApplyChunk; e0 < ue; e0 += kStageElems, ++n_st) {
          const int st = (int)(n_st % R);
          if (!mbar_wait_or_abort(ring_empty + st, (uint32_t)((n_st / R) & 1) ^ 1u, kWaitNs, abort_flag)) {
            stop = true;
            break;
          }
          const uint32_t bytes = (uint32_t)(min((int64_t)kStageElems, ue - e0) * 4);
          if (lane == 0) {
            if (vec) mbar_arrive_expect_tx(ring_full + st, 6 * bytes);
            else mbar_arrive(ring_full + st);   // feature warps read global memory directly
          }
          __syncwarp();
          if (vec && lane < 6) bulk_g2s(ring + st * (6 * kStageElems) + lane * kStageElems, src + e0, bytes,
                                        ring_full + st);
        }
        if (stop) break;
      }
      if (*abort_flag) {   // let copies already issued land before teardown
        for (int64_t kk = (n_st > R ? n_st - R : 0); kk < n_st; ++kk)
          mbar_drain(ring_full + kk % R, (uint32_t)((kk / R) & 1), kWaitNs / 10);
      }
    } else if (warp >= 8 && warp < 16) {
      // --------------------------- feature warpgroups ------------------------
      const int grp = (warp - 8) >> 2;
      const int t = tid - 256 - 128 * grp;
      const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      TileWalk w;
      w.init(a.units, a.desc, u0, u1);
      int cur = -1;
      bool vec = false, have_ij = false;
      int64_t i = 0, j = 0, last_e = 0, di = 0, dj = 0;
      float inv_rho[3] = {0.f, 0.f, 0.f};
      float sc[kStats];
#pragma unroll
      for (int q = 0; q < kStats; ++q) sc[q] = 0.f;
      // input stage of the current tile: counter, ring index, offset in it
      int64_t n_st = -1;
      int st = 0, st_off = 0;
      int64_t k = 0;
      for (; k < K; ++k, w.next()) {
        const int64_t in_unit = w.start - w.ustart;
        if (in_unit % kStageElems == 0) {   // this tile opens a new stage
          if (n_st >= 0) mbar_arrive(ring_empty + st);   // done with the previous one
          ++n_st;
          st = (int)(n_st % R);
        }
        st_off = (int)(in_unit % kStageElems);
        if ((int)(k & 1) != grp) continue;
        const int s = (int)(k % S);
        if (!mbar_wait_or_abort(slot_empty + s, (uint32_t)((k / S) & 1) ^ 1u, kWaitNs, abort_flag)) break;
        if (!mbar_wait_or_abort(ring_full + st, (uint32_t)((n_st / R) & 1), kWaitNs, abort_flag)) break;
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
          const float* rs = ring + st * (6 * kStageElems) + st_off + t;
          if (valid) {
            p = rs[0]; g = rs[kStageElems]; m[0] = rs[2 * kStageElems]; m[1] = rs[3 * kStageElems];
            m[2] = rs[4 * kStageElems]; v = rs[5 * kStageElems];
          }
        } else if (valid) {
          p = __ldg(d.p + e); g = __ldg(d.g + e); v = __ldg(d.v + e);
#pragma unroll
          for (int q = 0; q < 3; ++q) m[q] = __ldg(d.m[q] + e);
        }
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
        // normalised features, FP16, into this lane's row of the slot's A
        // operand in tensor memory (K = 32: 28 features, 1 for the bias, 0s)
        uint32_t av[16];
#pragma unroll
        for (int q = 0; q < 14; ++q) av[q] = f16x2(f[2 * q] * sc[2 * q], f[2 * q + 1] * sc[2 * q + 1]);
        av[14] = 0x00003C00u;   // 1.0h, 0
        av[15] = 0u;
        tmem_st16(t_lane + s * G::SlotCols + NP, av);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(a1_full + s);
      }
      if (k == K && n_st >= 0) mbar_arrive(ring_empty + st);
    } else if (warp == kMmaWarp) {
      // ------------------------------- MMA issuer ----------------------------
      if (lane == 0) {
        const uint64_t dB1 = smem_desc(s_base + G::oB1, 128, G::SBO1);
        const uint64_t dB2 = smem_desc(s_base + G::oB2, 128, G::SBO);
        const int k_end = (int)K + kLag2;
        // slot index and phase of tile k and of tile k - kLag2, kept incrementally
        int s1 = 0, s2 = S - kLag2;
        uint32_t p1 = 0, p2 = 1;
        int k = 0;
        for (; k < k_end; ++k) {
          const bool do1 = k < (int)K;
          const bool do2 = k >= kLag2;
          if (do1 && !mbar_wait_or_abort(a1_full + s1, p1, kWaitNs, abort_flag)) break;
          if (do2 && !mbar_wait_or_abort(a2_full + s2, p2, kWaitNs, abort_flag)) break;
          tc_fence_after();
          const uint32_t d1 = tmem + s1 * G::SlotCols, d2 = tmem + s2 * G::SlotCols;
          // K-steps of the two layers interleaved (independent accumulators);
          // one K-step of 16 FP16 values = 8 tensor-memory columns of A
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            if (do1) mma_f16_ts(d1, d1 + NP + 8 * kk, dB1 + 16 * kk, G::ID12, kk > 0);
            if (do2 && kk < NP / 16) mma_f16_ts(d2, d2 + NP + 8 * kk, dB2 + 16 * kk, G::ID12, 1u);  // onto b2
          }
          mma_commit(done + (k % kDone));   // tracks every MMA issued so far
          if (++s1 == S) { s1 = 0; p1 ^= 1; }
          if (++s2 == S) { s2 = 0; p2 ^= 1; }
        }
        // nothing of ours may still be running when the session ends
        if (k > 0) mbar_drain(done + ((k - 1) % kDone), (uint32_t)(((k - 1) / kDone) & 1), kWaitNs / 10);
      }
    } else if (warp < 8) {
      // ------------------------------ epilogue -------------------------------
      // Group h takes the tiles k with k % 2 == h.  In step m it finishes
      // layer 1 of tile m-4 (ReLU, FP16 A operand of layer 2, b2 preset of
      // its accumulator) and the rest of tile m-8 (ReLU(h2), output layer,
      // update); it loads p of tile m-6 for the update two steps later.
      const int h = warp >> 2;
      const int t = tid - 128 * h;
      const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const float* aux = reinterpret_cast<const float*>(smem + G::oB2 + G::B2);
      const float4* w3 = reinterpret_cast<const float4*>(aux + NP);   // {w0_j, w0_j+1, w1_j, w1_j+1}
      const float b30 = aux[3 * NP], b31 = aux[3 * NP + 1];
      TileWalk wp;   // tile m-6 of this group
      wp.init(a.units, a.desc, u0, u1);
      if (h == 1) wp.next();
      const float lr = a.lr;
      float* p_ptr_prev = nullptr;
      float p_prev = 0.f;
      for (int64_t m = h; m - kE2 < K; m += 2) {
        if (*abort_flag) break;
        const int64_t t1 = m - kE1, t2 = m - kE2, tp = m - (kE2 - 2);
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
          const uint32_t col = t_lane + s * G::SlotCols;
          uint32_t hv[NP], av[16], b2[NP];
          tmem_ld_row<NP>(col, hv);
#pragma unroll
          for (int q = 0; q < NP; q += 4) {
            const float4 b = *reinterpret_cast<const float4*>(aux + q);
            b2[q] = __float_as_uint(b.x); b2[q + 1] = __float_as_uint(b.y);
            b2[q + 2] = __float_as_uint(b.z); b2[q + 3] = __float_as_uint(b.w);
          }
          tmem_wait_ld();
          pack_relu_row<NP>(hv, av);
          tmem_st16(col + NP, av);
          tmem_st_row<NP>(col, b2);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(a2_full + s);
        }
        if (t2 >= 0 && t2 < K) {
          const int s = (int)(t2 % S);
          const int64_t it = t2 + kLag2;
          if (!mbar_wait_or_abort(done + (it % kDone), (uint32_t)((it / kDone) & 1), kWaitNs, abort_flag)) break;
          tc_fence_after();
          uint32_t hv[NP];
          tmem_ld_row<NP>(t_lane + s * G::SlotCols, hv);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(slot_empty + s);   // the slot's tensor memory is no longer read
          if (p_ptr_prev) {
            // output layer: (direction, magnitude) = ReLU(h2) . W3 + b3
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NP / 2; ++q) {
              const float2 r = make_float2(fmaxf(__uint_as_float(hv[2 * q]), 0.f),
                                           fmaxf(__uint_as_float(hv[2 * q + 1]), 0.f));
              const float4 w = w3[q];
              acc0 = __ffma2_rn(r, make_float2(w.x, w.y), acc0);
              acc1 = __ffma2_rn(r, make_float2(w.z, w.w), acc1);
            }
            const float o0 = acc0.x + acc0.y + b30, o1 = acc1.x + acc1.y + b31;
            const float upd = o0 * expf(o1 * kOutScale) * kOutScale;
            *p_ptr_prev = p_prev - lr * upd;
          }
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

// Packs, per weight set, the layer-2 B operand (FP16, canonical K-major) and
// the FP32 vectors the epilogue needs: b2[NP], the output weights as pairs
// {W3[j][0], W3[j+1][0], W3[j][1], W3[j+1][1]} for even j, and b3[2]; padded
// hidden units get zeros.
template <int NP>
__global__ void k_pack_tc(const float* weights, int hp, int set_size, int n_sets, uint8_t* out) {
  using G = Geom<NP>;
  const int per = NP * NP + 3 * NP + 4;
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
      continue;
    }
    r -= NP * NP;
    float v = 0.f;
    if (r < NP) {                             // b2
      v = r < hp ? W[w_off_b2(hp) + r] : 0.f;
    } else if (r < 3 * NP) {                  // W3 pairs
      const int q = r - NP;                   // 4 floats per pair of hidden units
      const int j = (q >> 2) * 2 + (q & 1), col = (q >> 1) & 1;
      v = j < hp ? W[w_off_W3(hp) + 2 * j + col] : 0.f;
    } else if (r < 3 * NP + 2) {              // b3
      v = W[w_off_b3(hp) + (r - 3 * NP)];
    }
    reinterpret_cast<float*>(base + G::B2)[r] = v;
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
