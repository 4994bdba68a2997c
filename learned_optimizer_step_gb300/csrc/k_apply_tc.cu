// K2 (tensor-core path): apply pass with the per-element MLP on tcgen05.
//
// Same computation as the FP32 apply kernel ("PyLO: Towards Accessible
// Learned Optimizers in PyTorch", section "融合カーネル戦略", kernel 2:
// features recomputed in registers, normalised, MLP, update written back),
// but the two hidden layers run as batched GEMMs on the 5th-generation
// tensor cores: the page's design evaluates the MLP on CUDA cores with __ldg
// weights, which on GB300 is ALU-bound (about 4.7 kFLOP per element against
// 44 bytes of traffic).
//
// One persistent CTA per SM, warp-specialised, linked by mbarriers:
//   warp 16      producer: bulk-copies (cp.async.bulk, one array per lane) p,
//                g, m0..2, v of up to 8 tiles (a stage) of a work unit into a
//                ring of shared-memory stages, and writes p, m0..2, v of a
//                stage back with bulk copies once its two groups are done;
//   warps 8-15   two feature warpgroups, owning alternate stages: EMA
//                update, features, normalisation, FP16 A operand of layer 1
//                into the tile slot's tensor memory (the updated m and v go
//                back into the stage), two elements (two tiles) at a time;
//   warps 17-18  MMA issuers, one thread each: layer 1 and layer 2, two
//                tiles and one commit at a time;
//   warps 0-7    two epilogue warpgroups, owning alternate stages, two
//                tiles at a time: ReLU + FP16 A operand of layer 2 (in
//                tensor memory) and the b2 preset of its accumulator; and,
//                two pairs later, ReLU(h2), the two-unit output layer in
//                FP32 on the CUDA cores and the update of p in the stage.
// A tile is 128 elements of one tensor (one per TMEM lane); four tiles
// cover 512 consecutive elements, lane t of each holding one of elements
// 4t..4t+3, so that a feature thread finds the row of four consecutive
// elements once and loads them in pairs.  A tile slot is a set of
// tensor-memory columns: the FP32 accumulator (NP columns) and the FP16 A
// operand of the next MMA (16 columns); the A operands never pass through
// shared memory.  Per-tensor data (scales,
// 1/rho, row/column accumulator addresses) travel with each stage in a
// small record, so the feature warps keep no per-tensor state.  Owning whole
// stages keeps the per-tile control flow of the warps small.
//
// Issuing is the scarce resource of the tensor-core side: measured on one
// SM, a thread that issues two small MMAs (M=128, N=32, K=16) per tile
// spends about 150 cycles on them and about 185 more on a commit, while
// threads of different warps issue side by side.  So a tile uses few MMAs
// (FP16 operands, K = 32 for layer 1 with b1 against a constant 1 in the A
// operand, K = NP for layer 2 onto the preset b2: 4 MMAs at NP = 32), a
// commit covers two tiles, and only two MMA round trips are made: the
// output layer (two units) runs on the CUDA cores.  (More issuer warps were
// measured to slow the kernel: their polling takes issue slots from the
// feature warps.)  At most S tiles are in flight (10 slots at NP = 32), and
// a tile keeps its slot from its features to the read of its layer-2
// result (its release is a barrier per tile in rotation, so that no wait
// can mistake an older release of the same slot for it), so S tiles per
// slot lifetime bound the throughput; hence the
// epilogue's lag of two pairs between layer 1 and the rest of a pair (by
// then layer 2 has usually completed), and no third MMA for the output
// layer: its round trip lengthens the lifetime more than it shortens the
// epilogue.
//
// The tiles of a CTA are processed in sessions: maximal runs of tiles whose
// tensors share one MLP weight set.  Between sessions the pipeline drains,
// the weights of the next set are loaded and the barriers restart.
//
// Every wait is bounded: on timeout the kernel raises the status flag, all
// roles stop, in-flight copies and MMAs are waited for (bounded) and tensor
// memory is freed.
//
// Code of the rare routes (the per-element feature builder of tensors that
// are not staged, the polling loop of a bounded wait) is kept out of line,
// so that the hot loops stay compact in the instruction cache: the kernel's
// unrolled code is large, and stalls on instruction fetch were measured to
// move its time by a few per cent.
#include <cuda_fp16.h>

#include "lopt.h"
#include "lopt_internal.cuh"
#include "tc_layout.cuh"

namespace lopt {
namespace {

constexpr int kTile = 128;                // elements per tile (= TMEM lanes)
constexpr int kEpiGroups = 2;             // epilogue warpgroups (stages in rotation)
constexpr int kFeatGroups = 2;            // feature warpgroups (stages in rotation)
// Measured on the ViT-B/16 list: three epilogue groups (80 registers per
// thread) are slower than two; three feature groups deadlock in the slot
// rotation, so the pipeline is built for two of each.
static_assert(kFeatGroups == 2 && kEpiGroups >= 2, "pipeline depth analysis assumes two feature groups");
constexpr int kFeatWarp0 = 4 * kEpiGroups;                    // first feature warp
constexpr int kProducerWarp = kFeatWarp0 + 4 * kFeatGroups;   // then the producer
constexpr int kMma1Warp = kProducerWarp + 1, kMma2Warp = kProducerWarp + 2;
constexpr int kThreads = (kMma2Warp + 1) * 32;
constexpr int kStageTiles = 8;            // tiles per stage (4 KB per array)
constexpr int kStageElems = kStageTiles * kTile;
constexpr int kArrays = 6;                // p, g, m0, m1, m2, v
constexpr int kRingStages = 6;            // stages held in shared memory
constexpr int kStageBytes = kArrays * kStageElems * 4;
constexpr int kStageUsers = 2 * kTile;    // the feature group (m, v) and the epilogue group (p) of a stage
// An epilogue group finishes a pair of tiles this many pairs after its layer 1.
constexpr int kLag = 2;
// Commit barriers per layer, one per pair of tiles in rotation; a waiter
// must never see its barrier lapped.  While an epilogue thread waits for
// pair j, the slots of j and of the later tiles of its stage stay taken, so
// the MMA threads can get no further ahead than the stages the other
// epilogue groups own plus one slot round: fewer than kEpiGroups *
// kStageTiles + S tiles, well under kDone pairs.
// Slot releases likewise have one barrier per tile in rotation, not one
// per slot: a waiter for the release of tile k - S (waited for by parity)
// must find the release of tile k - S - kDone complete, which a per-slot
// barrier (kDone = S) would not guarantee -- that earlier release may come
// from the other epilogue group, arbitrarily late.  Tile k - S - kDone lies
// in a stage at least kRingStages before tile k's, and such a stage is done
// before tile k's stage is loaded; and tile k - S + kDone cannot be
// released before tile k is handed over.
constexpr int kDone = 64;
constexpr uint64_t kWaitNs = 1000000000ull;

// Where stage array q (p, g, m0, m1, m2, v) of a tensor lives.
__device__ __forceinline__ float* stage_array(const TensorDesc& d, int q) {
  return q == 0 ? d.p : q == 1 ? const_cast<float*>(d.g) : q == 5 ? d.v : d.m[q - 2];
}

// A tensor's tiles move through shared memory by bulk copies when every
// array is 16-byte aligned and every stage is a whole number of 16-byte
// words; otherwise the feature and epilogue warps read and write its
// arrays in global memory themselves.
__device__ __forceinline__ bool staged(const TensorDesc& d) { return d.vec4 && (d.N & 3) == 0; }

// What the tiles of one ring slot need to know about their tensor, written
// by the producer when it loads the slot (and read again when it writes the
// slot back): the feature warps then keep no per-tensor state.
struct StageRec {
  float        sc[kStats];   // normalisation scales
  float        inv_rho[3];
  int32_t      tensor;
  const float* c[3];         // column accumulators
  const float* r[3];         // row accumulators
  int64_t      e0;           // first element of the stage
  int64_t      i0;           // its row and column
  int32_t      j0;
  int32_t      C;
  uint32_t     bytes;        // bytes per array; 0: not staged (nothing to write back)
  float        invC;         // 1 / C
  int32_t      quad;         // staged, C % 4 == 0 and the column accumulators 16-byte aligned:
                             // the four elements of a lane share a row, c is read in pairs
  int32_t      pad_[3];
};
static_assert(sizeof(StageRec) % 16 == 0, "stage records stay 16-byte aligned");

template <int NP>
struct Geom {
  static constexpr int ACols = 16;                     // A operand: 32 FP16 per row
  static constexpr int SlotCols = NP + ACols;          // accumulator + A operand
  static constexpr int S = 512 / SlotCols < 16 ? 512 / SlotCols : 16;   // tiles in flight
  static constexpr int SBO1 = 32 * 16;                 // layer-1 B operand: K = 32
  static constexpr int SBO = NP * 16;                  // layer-2 B operand: K = NP
  static constexpr int B1 = NP * 32 * 2;
  static constexpr int B2 = NP * NP * 2;
  static constexpr int Aux = (3 * NP + 4) * 4;         // b2[NP], W3 pairs[NP][2], b3[2], pad
  static constexpr int Set = (B2 + Aux + 1023) / 1024 * 1024;   // packed per-set stride
  static constexpr int oRing = 0;
  static constexpr int oB1 = oRing + kRingStages * kStageBytes;
  static constexpr int oB2 = oB1 + B1;                  // B2, b2, W3, b3 as packed
  static constexpr int oBar = (oB2 + Set + 15) / 16 * 16;
  static constexpr int nBars = 2 * kRingStages + 2 * S + 3 * kDone;
  static constexpr int oRec = (oBar + nBars * 8 + 15) / 16 * 16;   // records are read as float4
  static constexpr int oInfo = oRec + kRingStages * (int)sizeof(StageRec);
  static constexpr int Smem = oInfo + 64;
  static constexpr int TmemCols = 512;
  static constexpr uint32_t ID12 = instr_desc(0, 128, NP);
  static_assert(Smem <= 232448, "shared memory of one CTA");
  // a feature group emits all tiles of a stage before it finishes any: the
  // stage's last tile must not wait for a slot of its own
  static_assert(S % 2 == 0, "tile pairs start on even slots");
  static_assert(S * SlotCols <= 512 && S > kStageTiles && kDone >= kEpiGroups * kStageTiles + S,
                "tensor memory columns / pipeline depth");
  static_assert(S + kDone > kRingStages * kStageTiles && kDone - S >= kRingStages * kStageTiles,
                "slot releases are never waited for a round behind nor lapped");
  static_assert(oRec % 16 == 0 && sizeof(StageRec) % 16 == 0, "16-byte aligned stage records");
};

// Element layout of a stage: its tiles go in groups of four (a quad, 512
// consecutive elements); lane t of tile 4q + e holds element 512q + 4t + e,
// so that one thread builds the features of four consecutive elements from
// 64-bit loads and shares their row terms.  A stage of n elements has
// 4 * ceil(n / 512) tiles.
constexpr int kQuadElems = 4 * kTile;
static_assert(kStageElems % kQuadElems == 0 && kApplyChunk % kStageElems == 0,
              "units are whole stages but the last, stages whole quads but the last");
__device__ __forceinline__ int32_t stage_tiles(int32_t n) { return ((n + kQuadElems - 1) / kQuadElems) * 4; }

// Walks the stages of a session in order.  A stage holds up to kStageTiles
// consecutive tiles of one work unit; stage n of a session lives in ring
// slot n % kRingStages, round n / kRingStages.
struct StageIter {
  const Unit* units;
  const TensorDesc* desc;
  int32_t u, u1;
  int32_t soff, ulen;   // the stage's offset in its unit, the unit's length (elements)
  int32_t n;            // elements in the stage
  int32_t k0;           // its first tile, counted in the session
  int32_t st;           // ring slot
  uint32_t ph;          // round parity of the slot
  __device__ void init(const Unit* un, const TensorDesc* de, int32_t b, int32_t e) {
    units = un; desc = de; u = b; u1 = e; k0 = 0; st = 0; ph = 0;
    load_unit();
  }
  __device__ void load_unit() {
    if (u < u1) {
      const Unit x = units[u];
      const int64_t base = (int64_t)x.local * kApplyChunk;
      ulen = (int32_t)min(desc[x.tensor].N - base, (int64_t)kApplyChunk);
      soff = 0;
      n = min(ulen, kStageElems);
    }
  }
  __device__ bool valid() const { return u < u1; }
  __device__ void next() {
    k0 += stage_tiles(n);
    soff += kStageElems;
    if (soff >= ulen) {
      ++u;
      load_unit();
    } else {
      n = min(ulen - soff, kStageElems);
    }
    if (++st == kRingStages) { st = 0; ph ^= 1u; }
  }
};

__device__ __forceinline__ int32_t unit_tiles(const StepArgs& a, int32_t u) {
  const Unit x = a.units[u];
  const int64_t st = (int64_t)x.local * kApplyChunk;
  const int32_t len = (int32_t)min(a.desc[x.tensor].N - st, (int64_t)kApplyChunk);
  return (len / kStageElems) * stage_tiles(kStageElems) + stage_tiles(len % kStageElems);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return;
    if (global_ns() - t0 > limit_ns) return;
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

// Row and column of the element at offset xi of a stage: j0 + xi < C +
// kStageElems, so a float quotient is exact to within one.
__device__ __forceinline__ void stage_row_col(const StageRec& rc, int xi, int64_t& i, uint32_t& jc) {
  const uint32_t C = (uint32_t)rc.C;
  i = rc.i0;
  jc = (uint32_t)rc.j0 + (uint32_t)xi;
  if (jc >= C) {
    uint32_t q = (uint32_t)((float)jc * rc.invC);
    int32_t rem = (int32_t)(jc - q * C);
    if (rem < 0) { --q; rem += (int32_t)C; }
    else if (rem >= (int32_t)C) { ++q; rem -= (int32_t)C; }
    i += q;
    jc = (uint32_t)rem;
  }
}

__device__ __forceinline__ float2 ld_f2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ void st_f2(float* p, const float2& v) { *reinterpret_cast<float2*>(p) = v; }

// Per-row terms of one element's features: rr = r / rho and sr = sqrt(r)
// (as r * rsqrt(r + eps)), shared by every element of a row.
__device__ __forceinline__ void row_terms_f16(const float (&r)[3], const float (&inv_rho)[3], float (&rr)[3],
                                              float (&sr)[3]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    rr[k] = fmul(r[k], inv_rho[k]);
    sr[k] = fmul(r[k], frsqrt(fadd(r[k], kEps)));
  }
}

// The accumulator update and the 28 features of one element, normalised by
// the scales sc and packed as FP16 pairs (feature order as in lopt_features).
// m and v get exactly lopt_features' arithmetic (they are stored); the
// features themselves, which go to FP16, use paired FP32 multiplies where two
// neighbouring features share the operation, and a fused multiply-add
// inside rsqrt(r c / rho + eps).  rr, sr: the element's row terms.
__device__ __noinline__ void features_f16(float p, float g, float (&m)[3], float& v, const float (&rr)[3],
                                             const float (&sr)[3], const float (&c)[3], const float* sc,
                                             uint32_t (&av)[16]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) m[k] = ffma(beta(k), m[k], fmul(one_minus_beta(k), g));
  v = ffma(kBeta2, v, fmul(kOneMinusBeta2, fmul(g, g)));
  const float rsv = frsqrt(fadd(v, kEps));
  float rvh[3], sq[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    rvh[k] = frsqrt(fmaf(rr[k], c[k], kEps));
    sq[k] = fmul(c[k], frsqrt(fadd(c[k], kEps)));
  }
  float2 q[14];
  q[0] = make_float2(p, g);
  q[1] = make_float2(m[0], m[1]);
  q[2] = make_float2(m[2], fmul(v, rsv));
  q[3] = __fmul2_rn(make_float2(m[0], m[1]), make_float2(rsv, rsv));
  q[4] = __fmul2_rn(make_float2(m[2], g), make_float2(rsv, rsv));
  q[5] = __fmul2_rn(make_float2(g, g), make_float2(rvh[0], rvh[1]));
  q[6] = make_float2(fmul(g, rvh[2]), sr[0]);
  q[7] = make_float2(sr[1], sr[2]);
  q[8] = make_float2(sq[0], sq[1]);
  q[9] = make_float2(sq[2], fmul(m[0], rvh[0]));
  q[10] = __fmul2_rn(make_float2(m[0], m[0]), make_float2(rvh[1], rvh[2]));
  q[11] = __fmul2_rn(make_float2(m[1], m[1]), make_float2(rvh[0], rvh[1]));
  q[12] = __fmul2_rn(make_float2(m[1], m[2]), make_float2(rvh[2], rvh[0]));
  q[13] = __fmul2_rn(make_float2(m[2], m[2]), make_float2(rvh[1], rvh[2]));
  const float4* sc4 = reinterpret_cast<const float4*>(sc);
#pragma unroll
  for (int k = 0; k < 7; ++k) {
    const float4 s = sc4[k];
    const float2 lo = __fmul2_rn(q[2 * k], make_float2(s.x, s.y));
    const float2 hi = __fmul2_rn(q[2 * k + 1], make_float2(s.z, s.w));
    av[2 * k] = f16x2(lo.x, lo.y);
    av[2 * k + 1] = f16x2(hi.x, hi.y);
  }
  av[14] = 0x00003C00u;   // 1.0h (against b1 in the B operand), 0
  av[15] = 0u;
}

// features_f16 for two neighbouring elements of one row at once, one in
// each half of every float2 (x: the first, y: the second), with the paired
// FP32 instructions.  Every result is the same single-element operation as
// in features_f16, so both elements get exactly its values.  srn: the row's
// sqrt(r_k) features already normalised (sr_k * sc[13 + k]).  The FP16 words
// come in two halves, to keep fewer registers live: words 0-7 (features
// 0-15) of both elements go to store_lo(loA, loB), which returns false to
// stop; words 8-15 (features 16-27, the constant 1, zeros) are returned.
template <typename StoreLo>
__device__ __forceinline__ bool features_f16_pair(float2 P, float2 G, float2 (&M)[3], float2& V,
                                                  const float (&rr)[3], const float (&srn)[3],
                                                  const float2 (&C)[3], const float* sc, StoreLo&& store_lo,
                                                  uint32_t (&hiA)[8], uint32_t (&hiB)[8]) {
  const auto dup = [](float x) { return make_float2(x, x); };
#pragma unroll
  for (int k = 0; k < 3; ++k) M[k] = __ffma2_rn(dup(beta(k)), M[k], __fmul2_rn(dup(one_minus_beta(k)), G));
  V = __ffma2_rn(dup(kBeta2), V, __fmul2_rn(dup(kOneMinusBeta2), __fmul2_rn(G, G)));
  const float2 ve = __fadd2_rn(V, dup(kEps));
  const float2 rsv = make_float2(frsqrt(ve.x), frsqrt(ve.y));
  float2 rvh[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const float2 h = __ffma2_rn(dup(rr[k]), C[k], dup(kEps));
    rvh[k] = make_float2(frsqrt(h.x), frsqrt(h.y));
  }
  // features 0-27 in order, normalised, two at a time into FP16 pairs
  const float4* sc4 = reinterpret_cast<const float4*>(sc);
  auto put = [&](uint32_t (&oa)[8], uint32_t (&ob)[8], int w, float2 f0, float2 f1, float s0, float s1) {
    const float2 n0 = __fmul2_rn(f0, dup(s0)), n1 = __fmul2_rn(f1, dup(s1));
    oa[w] = f16x2(n0.x, n1.x);
    ob[w] = f16x2(n0.y, n1.y);
  };
  {
    uint32_t loA[8], loB[8];
    float4 s;
    s = sc4[0];
    put(loA, loB, 0, P, G, s.x, s.y);
    put(loA, loB, 1, M[0], M[1], s.z, s.w);
    s = sc4[1];
    put(loA, loB, 2, M[2], __fmul2_rn(V, rsv), s.x, s.y);
    put(loA, loB, 3, __fmul2_rn(M[0], rsv), __fmul2_rn(M[1], rsv), s.z, s.w);
    s = sc4[2];
    put(loA, loB, 4, __fmul2_rn(M[2], rsv), __fmul2_rn(G, rsv), s.x, s.y);
    put(loA, loB, 5, __fmul2_rn(G, rvh[0]), __fmul2_rn(G, rvh[1]), s.z, s.w);
    s = sc4[3];
    {  // g rsqrt(vhat_2), then the first normalised sqrt(r) of the row
      const float2 n0 = __fmul2_rn(__fmul2_rn(G, rvh[2]), dup(s.x));
      loA[6] = f16x2(n0.x, srn[0]);
      loB[6] = f16x2(n0.y, srn[0]);
    }
    loA[7] = loB[7] = f16x2(srn[1], srn[2]);
    if (!store_lo(loA, loB)) return false;
  }
  float2 sq[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const float2 ce = __fadd2_rn(C[k], dup(kEps));
    sq[k] = __fmul2_rn(C[k], make_float2(frsqrt(ce.x), frsqrt(ce.y)));
  }
  float4 s;
  s = sc4[4];
  put(hiA, hiB, 0, sq[0], sq[1], s.x, s.y);
  put(hiA, hiB, 1, sq[2], __fmul2_rn(M[0], rvh[0]), s.z, s.w);
  s = sc4[5];
  put(hiA, hiB, 2, __fmul2_rn(M[0], rvh[1]), __fmul2_rn(M[0], rvh[2]), s.x, s.y);
  put(hiA, hiB, 3, __fmul2_rn(M[1], rvh[0]), __fmul2_rn(M[1], rvh[1]), s.z, s.w);
  s = sc4[6];
  put(hiA, hiB, 4, __fmul2_rn(M[1], rvh[2]), __fmul2_rn(M[2], rvh[0]), s.x, s.y);
  put(hiA, hiB, 5, __fmul2_rn(M[2], rvh[1]), __fmul2_rn(M[2], rvh[2]), s.z, s.w);
  hiA[6] = hiB[6] = 0x00003C00u;   // 1.0h (against b1 in the B operand), 0
  hiA[7] = hiB[7] = 0u;
  return true;
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
  uint64_t* stage_done = ring_full + R;
  uint64_t* a1_full = stage_done + R;
  uint64_t* a2_full = a1_full + S;
  uint64_t* freed = a2_full + S;       // per tile in rotation: its slot is free again
  uint64_t* done1 = freed + kDone;
  uint64_t* done2 = done1 + kDone;
  StageRec* rec = reinterpret_cast<StageRec*>(smem + G::oRec);
  int32_t* info = reinterpret_cast<int32_t*>(smem + G::oInfo);   // session: end unit, tiles
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

  const int32_t U = a.n_units;
  const int32_t u_first = (int32_t)((int64_t)blockIdx.x * U / gridDim.x);
  const int32_t u_last = (int32_t)((int64_t)(blockIdx.x + 1) * U / gridDim.x);

  // ---- sessions: maximal runs of tiles that share one MLP weight set --------
  // Every role runs the same sequence of sessions and meets the same
  // barriers; set-up and tear-down of a session are common to all.
  auto begin_session = [&](int32_t u0, int32_t& u1, int32_t& K) -> bool {
    if (tid == 0) {
      const int wset = a.desc[a.units[u0].tensor].wset;
      int32_t e = u0, n = 0;
      while (e < u_last && a.desc[a.units[e].tensor].wset == wset) n += unit_tiles(a, e++);
      info[0] = e;
      info[1] = n;
      for (int r = 0; r < R; ++r) {
        mbar_init(ring_full + r, 1);
        mbar_init(stage_done + r, kStageUsers);
      }
      for (int s = 0; s < S; ++s) {
        mbar_init(a1_full + s, kTile);
        mbar_init(a2_full + s, kTile);

      }
      for (int x = 0; x < kDone; ++x) mbar_init(freed + x, kTile);
      for (int s = 0; s < 2 * kDone; ++s) mbar_init(done1 + s, 1);
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
    u1 = info[0];
    K = info[1];
    return !*abort_flag;
  };
  auto sessions = [&](auto&& role) {
    for (int32_t u0 = u_first, u1 = 0, K = 0; u0 < u_last; u0 = u1) {
      if (!begin_session(u0, u1, K)) break;
      role(u0, u1, K);
      // ---- session end: every role has finished its tiles
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  };

  if (warp >= kProducerWarp) {
    sessions([&](int32_t u0, int32_t u1, int32_t K) {
      if (warp == kProducerWarp) {

          // ------------------------------ producer -------------------------------
          // Lane q < 6 moves array q of every stage.  Before a slot is loaded
          // again, the stage it held is written back (p, m0..2, v) once every
          // feature and epilogue thread has left it.
          auto write_back = [&](int st) {
            const StageRec r = rec[st];
            if (r.bytes != 0 && lane < kArrays && lane != 1) {
              bulk_s2g(stage_array(a.desc[r.tensor], lane) + r.e0, ring + st * (kArrays * kStageElems) + lane * kStageElems,
                       r.bytes);
              bulk_commit();
              bulk_wait_read_all();   // the slot may be refilled once its contents have been read
            }
            __syncwarp();
          };
          int32_t n = 0;      // stages issued
          int st = 0;         // slot of stage n
          uint32_t ph = 0;    // its round parity
          bool stop = false;
          for (int32_t u = u0; u < u1 && !stop; ++u) {
            const Unit x = a.units[u];
            const TensorDesc& d = a.desc[x.tensor];
            const bool stg = staged(d);
            const int64_t ub = (int64_t)x.local * kApplyChunk;
            const int64_t ue = min(d.N, ub + kApplyChunk);
            const float* src = stage_array(d, lane < kArrays ? lane : 0);
            for (int64_t e0 = ub; e0 < ue; e0 += kStageElems) {
              if (n >= R) {   // the slot's previous stage: round ph ^ 1
                if (!mbar_wait_or_abort(stage_done + st, ph ^ 1u, kWaitNs, abort_flag)) {
                  stop = true;
                  break;
                }
                write_back(st);
              }
              const uint32_t bytes = (uint32_t)(min((int64_t)kStageElems, ue - e0) * 4);
              StageRec& rc = rec[st];
              if (lane < kStats) rc.sc[lane] = a.aux[x.tensor].scale[lane];
              else if (lane < kStats + 3) rc.inv_rho[lane - kStats] = a.aux[x.tensor].inv_rho[lane - kStats];
              else if (lane == 31) {
                rc.tensor = x.tensor;
                rc.e0 = e0;
                rc.i0 = e0 / d.C;
                rc.j0 = (int32_t)(e0 - rc.i0 * d.C);
                rc.C = (int32_t)d.C;
                rc.invC = 1.0f / (float)d.C;
                rc.bytes = stg ? bytes : 0u;
                rc.quad = stg && (d.C & 3) == 0 &&
                          (((uintptr_t)d.c[0] | (uintptr_t)d.c[1] | (uintptr_t)d.c[2]) & 15) == 0;
              }
              if (lane < 3) rc.c[lane] = d.c[lane];
              else if (lane < 6) rc.r[lane - 3] = d.r[lane - 3];
              __syncwarp();
              if (lane == 0) {
                if (stg) mbar_arrive_expect_tx(ring_full + st, kArrays * bytes);
                else mbar_arrive(ring_full + st);
              }
              __syncwarp();
              if (stg && lane < kArrays)
                bulk_g2s(ring + st * (kArrays * kStageElems) + lane * kStageElems, src + e0, bytes, ring_full + st);
              ++n;
              if (++st == R) { st = 0; ph ^= 1u; }
            }
          }
          // the stages still in the ring, oldest first
          for (int32_t x = (n > R ? n - R : 0); x < n && !stop; ++x) {
            const int xs = x % R;
            if (!mbar_wait_or_abort(stage_done + xs, (uint32_t)((x / R) & 1), kWaitNs, abort_flag)) {
              stop = true;
              break;
            }
            write_back(xs);
          }
          if (stop) {   // let loads already issued land before teardown
            for (int32_t x = (n > R ? n - R : 0); x < n; ++x)
              mbar_drain(ring_full + x % R, (uint32_t)((x / R) & 1), kWaitNs / 10);
          }
          bulk_wait_all();   // every write-back complete before the session ends
      } else if (warp == kMma1Warp || warp == kMma2Warp) {

          // ------------------------------ MMA issuers ----------------------------
          // One thread per layer, two tiles at a time (tiles come in pairs):
          // layer 1 of tiles k, k + 1 once their A operands are in tensor
          // memory, committed to done1[k / 2]; layer 2 once their A operands
          // and b2 presets are, committed to done2[k / 2].  A commit keeps the
          // issuing thread about as long as two MMAs, so one per pair.
          if (lane == 0) {
            const bool l1 = warp == kMma1Warp;
            const uint64_t dB = l1 ? smem_desc(s_base + G::oB1, 128, G::SBO1) : smem_desc(s_base + G::oB2, 128, G::SBO);
            uint64_t* const full = l1 ? a1_full : a2_full;
            uint64_t* const fin = l1 ? done1 : done2;
            const int ksteps = l1 ? 2 : NP / 16;   // K-steps of 16 FP16 values (8 A columns)
            int s = 0;
            uint32_t ph = 0;
            int32_t k = 0;
            for (; k < K; k += 2) {
              const int s1 = s + 1;   // S is even and pairs start on even tiles
              if (!mbar_wait_or_abort(full + s, ph, kWaitNs, abort_flag) ||
                  !mbar_wait_or_abort(full + s1, ph, kWaitNs, abort_flag))
                break;
              tc_fence_after();
#pragma unroll
              for (int tt = 0; tt < 2; ++tt) {
                const uint32_t d = tmem + (tt ? s1 : s) * G::SlotCols;
                // layer 1 overwrites its accumulator; layer 2 adds onto the b2 preset
                mma_f16_ts(d, d + NP, dB, G::ID12, l1 ? 0u : 1u);
                if (ksteps > 1) mma_f16_ts(d, d + NP + 8, dB + 16, G::ID12, 1u);
              }
              mma_commit(fin + ((k >> 1) & (kDone - 1)));   // tracks every MMA of this thread so far
              s += 2;
              if (s == S) { s = 0; ph ^= 1u; }
            }
            // nothing of ours may still be running when the session ends
            if (k > 0) {
              const int32_t kp = (k - 2) >> 1;
              mbar_drain(fin + (kp & (kDone - 1)), (uint32_t)((kp / kDone) & 1), kWaitNs / 10);
            }
          }
      }
    });
  } else if (warp >= kFeatWarp0) {
    sessions([&](int32_t u0, int32_t u1, int32_t K) {

        // --------------------------- feature warpgroups ------------------------
        // Group grp owns the stages n with n % 2 == grp: it updates m and v
        // in the stage and builds the A operand of layer 1 for each of their
        // tiles in order.
        const int grp = (warp - kFeatWarp0) >> 2;
        const int t = tid - 32 * kFeatWarp0 - 128 * grp;
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        StageIter si;
        si.init(a.units, a.desc, u0, u1);
        bool ok = true;
        for (int32_t ns = 0; ok && si.valid(); ++ns, si.next()) {
          if (ns % kFeatGroups != grp) continue;
          if (!mbar_wait_or_abort(ring_full + si.st, si.ph, kWaitNs, abort_flag)) { ok = false; break; }
          const StageRec& rc = rec[si.st];
          const bool stg = rc.bytes != 0;
          float* const sbase = ring + si.st * (kArrays * kStageElems);
          const int nq = stage_tiles(si.n) / 4;
          int s = si.k0 % S;                          // slot of the stage's first tile
          // The next tile, k, may use its slot once tile k - S has released
          // it.  Releases have a barrier per tile in rotation (kDone), so that
          // a release that is waited for by parity cannot be confused with a
          // late release of an earlier tile of the same slot.  fj, fph: the
          // rotation index and phase parity of tile k - S (floor semantics:
          // for the first S tiles of a session, parity 1 of a fresh barrier,
          // which passes at once).
          int fj = (si.k0 - S) & (kDone - 1);
          uint32_t fph = (uint32_t)((si.k0 - S) >> 6) & 1u;
          static_assert(kDone == 64, "rotation parity by shift");
          // Hands a tile's A operand to its slot and tells the layer-1 MMA
          // thread at once.  The slot is waited for only now, so that loads
          // and arithmetic overlap the wait.  (Announcing a tile only at the
          // next tile, to avoid waiting for the store, was measured to delay
          // the layer-1 MMA by about 450 cycles.)
          auto emit = [&](const uint32_t (&av)[16]) -> bool {
            if (!mbar_wait_or_abort(freed + fj, fph, kWaitNs, abort_flag)) return false;
            tmem_st16(t_lane + s * G::SlotCols + NP, av);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(a1_full + s);
            if (++s == S) s = 0;
            if (++fj == kDone) { fj = 0; fph ^= 1u; }
            return true;
          };
          // The same for two tiles at once (one wait for both stores), in two
          // steps: the slots are waited for and the first half of each A
          // operand stored once it is built, then the second half stored and
          // both tiles announced.
          auto store_lo_pair = [&](const uint32_t (&loA)[8], const uint32_t (&loB)[8]) -> bool {
            const int s1 = s + 1 == S ? 0 : s + 1;
            const int fj1 = fj + 1 == kDone ? 0 : fj + 1;
            const uint32_t fph1 = fj1 == 0 ? fph ^ 1u : fph;
            if (!mbar_wait_or_abort(freed + fj, fph, kWaitNs, abort_flag) ||
                !mbar_wait_or_abort(freed + fj1, fph1, kWaitNs, abort_flag))
              return false;
            tmem_st8(t_lane + s * G::SlotCols + NP, loA);
            tmem_st8(t_lane + s1 * G::SlotCols + NP, loB);
            return true;
          };
          auto finish_emit_pair = [&](const uint32_t (&hiA)[8], const uint32_t (&hiB)[8]) {
            const int s1 = s + 1 == S ? 0 : s + 1;
            tmem_st8(t_lane + s * G::SlotCols + NP + 8, hiA);
            tmem_st8(t_lane + s1 * G::SlotCols + NP + 8, hiB);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(a1_full + s);
            mbar_arrive(a1_full + s1);
            s = s1 + 1 == S ? 0 : s1 + 1;
            const int fj1 = fj + 1 == kDone ? 0 : fj + 1;
            fj = fj1 + 1 == kDone ? 0 : fj1 + 1;
            if (fj1 == 0 || fj == 0) fph ^= 1u;   // passed the end of the rotation
          };
          for (int qd = 0; ok && qd < nq; ++qd) {
            const int x0 = qd * kQuadElems + 4 * t;   // this lane's first element in the stage
            if (rc.quad) {
              // four consecutive elements of one row (C % 4 == 0 and x0 % 4 ==
              // 0); past the end: unused stage words, and the row and columns
              // of the stage's last four elements
              int64_t i;
              uint32_t jc;
              stage_row_col(rc, min(x0, si.n - 4), i, jc);
              float r[3], inv_rho[3], rr[3], sr[3];
#pragma unroll
              for (int q = 0; q < 3; ++q) {
                r[q] = __ldg(rc.r[q] + i);
                inv_rho[q] = rc.inv_rho[q];
              }
              row_terms_f16(r, inv_rho, rr, sr);
              float srn[3];
#pragma unroll
              for (int q = 0; q < 3; ++q) srn[q] = fmul(sr[q], rc.sc[13 + q]);
              // two pairs of elements, 64-bit loads and stores; each pair is
              // built at once and handed to tiles 4 qd + h and 4 qd + h + 1
#pragma unroll
              for (int h = 0; h < 4; h += 2) {
                const int xh = x0 + h;
                const float2 P = ld_f2(sbase + xh), Gr = ld_f2(sbase + kStageElems + xh);
                float2 M[3] = {ld_f2(sbase + 2 * kStageElems + xh), ld_f2(sbase + 3 * kStageElems + xh),
                               ld_f2(sbase + 4 * kStageElems + xh)};
                float2 V = ld_f2(sbase + 5 * kStageElems + xh);
                float2 c2[3];
#pragma unroll
                for (int q = 0; q < 3; ++q) c2[q] = __ldg(reinterpret_cast<const float2*>(rc.c[q] + jc + h));
                // normalised features, FP16, for this lane's row of the A
                // operands (K = 32: 28 features, 1, 0s)
                uint32_t hiA[8], hiB[8];
                if (!features_f16_pair(P, Gr, M, V, rr, srn, c2, rc.sc, store_lo_pair, hiA, hiB)) {
                  ok = false;
                  break;
                }
                st_f2(sbase + 2 * kStageElems + xh, M[0]); st_f2(sbase + 3 * kStageElems + xh, M[1]);
                st_f2(sbase + 4 * kStageElems + xh, M[2]); st_f2(sbase + 5 * kStageElems + xh, V);
                finish_emit_pair(hiA, hiB);
              }
              if (!ok) break;
            } else {
#pragma unroll 1
              for (int e = 0; e < 4; ++e) {
                const int x = x0 + e;                // element offset in the stage
                const int xi = min(x, si.n - 1);     // past the end: index math of the last element
                float p, g, m[3], v;
                if (stg) {   // elements past the end read and write unused stage words
                  p = sbase[x]; g = sbase[kStageElems + x]; m[0] = sbase[2 * kStageElems + x];
                  m[1] = sbase[3 * kStageElems + x]; m[2] = sbase[4 * kStageElems + x];
                  v = sbase[5 * kStageElems + x];
                } else {
                  const TensorDesc& d = a.desc[rc.tensor];
                  const int64_t el = rc.e0 + xi;
                  p = d.p[el]; g = __ldg(d.g + el); v = d.v[el];
#pragma unroll
                  for (int q = 0; q < 3; ++q) m[q] = d.m[q][el];
                }
                int64_t i;
                uint32_t jc;
                stage_row_col(rc, xi, i, jc);
                float c[3], r[3], inv_rho[3], rr[3], sr[3];
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                  c[q] = __ldg(rc.c[q] + jc);
                  r[q] = __ldg(rc.r[q] + i);
                  inv_rho[q] = rc.inv_rho[q];
                }
                row_terms_f16(r, inv_rho, rr, sr);
                uint32_t av[16];
                features_f16(p, g, m, v, rr, sr, c, rc.sc, av);
                if (stg) {
                  sbase[2 * kStageElems + x] = m[0]; sbase[3 * kStageElems + x] = m[1];
                  sbase[4 * kStageElems + x] = m[2]; sbase[5 * kStageElems + x] = v;
                } else if (x < si.n) {
                  const TensorDesc& d = a.desc[rc.tensor];
                  const int64_t el = rc.e0 + x;
#pragma unroll
                  for (int q = 0; q < 3; ++q) d.m[q][el] = m[q];
                  d.v[el] = v;
                }
                if (!emit(av)) { ok = false; break; }
              }
            }
          }
          if (!ok) break;
          fence_proxy_async();   // m, v in the stage, before its write-back
          mbar_arrive(stage_done + si.st);
        }
    });
  } else {
    sessions([&](int32_t u0, int32_t u1, int32_t K) {

        // ------------------------------ epilogue -------------------------------
        // Group h owns the stages n with n % 2 == h.  For each pair of tiles
        // of a stage it finishes layer 1 (ReLU, FP16 A operand of layer 2, b2
        // preset of its accumulator) and, kLag pairs later, the rest (ReLU(h2),
        // output layer, update of p in the stage): by then the pair's layer 2
        // has usually completed, so neither step waits for the tensor cores.
        const int h = warp >> 2;
        const int t = tid - 128 * h;
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float* aux = reinterpret_cast<const float*>(smem + G::oB2 + G::B2);
        const float4* w3 = reinterpret_cast<const float4*>(aux + NP);   // {w0_j, w0_j+1, w1_j, w1_j+1}
        const float b30 = aux[3 * NP], b31 = aux[3 * NP + 1];
        const float lr = a.lr, wd = a.wd;
        StageIter si;
        si.init(a.units, a.desc, u0, u1);
        bool ok = true;
        for (int32_t ns = 0; ok && si.valid(); ++ns, si.next()) {
          if (ns % kEpiGroups != h) continue;
          // the stage's record and p (loaded before any of its tiles was built)
          if (!mbar_wait_or_abort(ring_full + si.st, si.ph, kWaitNs, abort_flag)) { ok = false; break; }
          const StageRec& rc = rec[si.st];
          const bool stg = rc.bytes != 0;
          float* const pst = ring + si.st * (kArrays * kStageElems);
          const int ntl = stage_tiles(si.n);
          const int s0 = si.k0 % S;

          // ---- layer 1 of tiles j, j + 1: the b2 preset is read from shared
          // memory once for both
          auto layer1 = [&](int j) -> bool {
            const int s = (s0 + j) % S;
            const int s1 = s + 1 == S ? 0 : s + 1;
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
              const int32_t k = si.k0 + j + tt;
              if (tt == 0 && !mbar_wait_or_abort(done1 + ((k >> 1) & (kDone - 1)), (uint32_t)(((k >> 1) / kDone) & 1),
                                                 kWaitNs, abort_flag))
                return false;
              tc_fence_after();
              const uint32_t col = t_lane + (tt ? s1 : s) * G::SlotCols;
              uint32_t av[16];
              {
                uint32_t h1[NP];
                tmem_ld_row<NP>(col, h1);
                tmem_wait_ld();
                pack_relu_row<NP>(h1, av);
              }
              tmem_st16(col + NP, av);
            }
#pragma unroll
            for (int hf = 0; hf < NP / 16; ++hf) {   // 16 columns at a time (fewer live registers)
              uint32_t b2[16];
#pragma unroll
              for (int q = 0; q < 16; q += 4) {
                const float4 b = *reinterpret_cast<const float4*>(aux + 16 * hf + q);
                b2[q] = __float_as_uint(b.x); b2[q + 1] = __float_as_uint(b.y);
                b2[q + 2] = __float_as_uint(b.z); b2[q + 3] = __float_as_uint(b.w);
              }
              tmem_st16(t_lane + s * G::SlotCols + 16 * hf, b2);
              tmem_st16(t_lane + s1 * G::SlotCols + 16 * hf, b2);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(a2_full + s);
            mbar_arrive(a2_full + s1);
            return true;
          };

          // ---- the rest of tiles j, j + 1, so that every output-layer weight
          // read from shared memory serves two elements; their slots are freed
          // as soon as h2 is read.  Lane t of the stage's tiles holds this
          // thread's elements.
          auto finish = [&](int j) -> bool {
            const int32_t k = si.k0 + j;
            if (!mbar_wait_or_abort(done2 + ((k >> 1) & (kDone - 1)), (uint32_t)(((k >> 1) / kDone) & 1), kWaitNs,
                                    abort_flag))
              return false;
            tc_fence_after();
            const int s = (s0 + j) % S;
            const int s1 = s + 1 == S ? 0 : s + 1;
            // output layer: (direction, magnitude) = ReLU(h2) . W3 + b3 for
            // both tiles, over 16 hidden units at a time, two FMA chains each
            float2 acc[2][4];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[0][q] = acc[1][q] = make_float2(0.f, 0.f);
#pragma unroll
            for (int hf = 0; hf < NP / 16; ++hf) {
              uint32_t ha[16], hb[16];
              tmem_ld16(t_lane + s * G::SlotCols + 16 * hf, ha);
              tmem_ld16(t_lane + s1 * G::SlotCols + 16 * hf, hb);
              tmem_wait_ld();
              if (hf == NP / 16 - 1) {
                tc_fence_before();
                mbar_arrive(freed + (k & (kDone - 1)));
                mbar_arrive(freed + ((k + 1) & (kDone - 1)));
              }
#pragma unroll
              for (int ch = 0; ch < 2; ++ch) {   // 8 hidden units
                float4 w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = w3[4 * (2 * hf + ch) + q];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const int u = 8 * ch + 2 * q;
                  const float2 w0 = make_float2(w[q].x, w[q].y), w1 = make_float2(w[q].z, w[q].w);
                  const float2 ra = make_float2(fmaxf(__uint_as_float(ha[u]), 0.f), fmaxf(__uint_as_float(ha[u + 1]), 0.f));
                  const float2 rb = make_float2(fmaxf(__uint_as_float(hb[u]), 0.f), fmaxf(__uint_as_float(hb[u + 1]), 0.f));
                  acc[0][(q & 1) * 2] = __ffma2_rn(ra, w0, acc[0][(q & 1) * 2]);
                  acc[0][(q & 1) * 2 + 1] = __ffma2_rn(ra, w1, acc[0][(q & 1) * 2 + 1]);
                  acc[1][(q & 1) * 2] = __ffma2_rn(rb, w0, acc[1][(q & 1) * 2]);
                  acc[1][(q & 1) * 2 + 1] = __ffma2_rn(rb, w1, acc[1][(q & 1) * 2 + 1]);
                }
              }
            }
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
              const float o0 = (acc[tt][0].x + acc[tt][0].y) + (acc[tt][2].x + acc[tt][2].y) + b30;
              const float o1 = (acc[tt][1].x + acc[tt][1].y) + (acc[tt][3].x + acc[tt][3].y) + b31;
              // exp(x) = 2^(x log2 e) with the PTX ex2.approx instruction
              // (relative error below 2^-22); here |x| = |o1| * 1e-3 is small
              float ex;
              asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ex) : "f"(o1 * (kOutScale * 1.44269504088896341f)));
              const float upd = o0 * ex * kOutScale;
              const int jt = j + tt;
              const int x = (jt >> 2) * kQuadElems + 4 * t + (jt & 3);   // this lane's element of tile jt
              if (stg) {   // past the end: an unused stage word
                pst[x] = pst[x] - lr * (upd + wd * pst[x]);
              } else if (x < si.n) {
                float* pp = a.desc[rc.tensor].p + (rc.e0 + x);
                *pp = *pp - lr * (upd + wd * *pp);
              }
            }
            return true;
          };

          for (int j = 0; ok && j < ntl; j += 2) {
            ok = layer1(j);
            if (ok && j >= 2 * kLag) ok = finish(j - 2 * kLag);
          }
          for (int j = ntl > 2 * kLag ? ntl - 2 * kLag : 0; ok && j < ntl; j += 2) ok = finish(j);
          if (!ok) break;
          fence_proxy_async();   // p in the stage, before its write-back
          mbar_arrive(stage_done + si.st);
        }
    });
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
