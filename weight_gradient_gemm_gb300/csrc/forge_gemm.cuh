// The tensor-core weight-gradient kernel, in two modes:
//   kModeFused : G = dY^T X per 128 x BN weight tile, then AdamW on the tile
//                straight from the tensor-memory accumulator; only W, m, v
//                (and int8 scales) are written back.  This is the FORGE step
//                ("FORGE: Fused On-Register Gradient Elimination", section 2.2,
//                Eq. 4 and Algorithm 1), with the accumulator in TMEM.
//   kModeStoreG: the same main loop, storing G (fp32 or bf16): the unfused
//                gradient ("store-G control", Appendix D).
//   kModeDgrad : the layer's input gradient dX = dY W (the other half of the
//                backward pass of Y = X W^T, which Algorithm 1 computes from
//                the weight before the update): M = tokens, N = d_in,
//                K = d_out, A = dY K-major, B = W MN-major, bf16 dX stored as
//                in kModeStoreG.
//
// One persistent CTA per SM (or one CTA pair per two SMs, CG = 2) walks the
// tile queue t = unit, unit + units, ... over all layers of the launch.
// Warp roles (384 threads):
//   warp 0      TMA producer: dY and X chunks of BK tokens into a STAGES ring,
//               one lane per box so a stage is one warp-wide TMA issue
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma 128 x BN x 16 (256 x BN
//               on a pair), bf16 in, fp32 accumulate, into one of two TMEM
//               accumulators (the next tile's main loop overlaps this tile's
//               epilogue)
//   warp 2      state loader (fused mode): W/m/v slices of the tile, TMA into
//               an NS-slot ring, issued ahead of the epilogue
//   warp 3      store warp: lane j TMA-stores what the epilogue left in slot j
//               and frees the slot once the store has read it
//   warps 4-11  epilogue: TMEM -> registers, AdamW in fp32, results written in
//               place into the slot (two warps per TMEM lane quadrant)
// How shared memory is split between operand stages and state slots is the
// pipeline profile (forge_internal.h), chosen by token count on the host.
//
// Operands: A = dY^T (M = weight rows) and B = X (N = weight columns) are both
// contiguous along M/N, so both are fed to the MMA MN-major, straight from the
// TMA boxes [BK tokens][64 elements] with the 128-byte swizzle.
//
// Every wait is bounded (GemmParams::timeout_ns).  When a bound runs out the
// CTA raises a shared abort flag, records FORGE_ERR_DEVICE_TIMEOUT in the
// device error word, lets its in-flight copies and MMAs land, frees its
// tensor memory and returns.  Nothing traps.
#pragma once

#include "forge_internal.h"
#include "forge_ptx.cuh"

namespace forge {

constexpr int kSmemLimit = 232448;   // max dynamic shared memory per CTA (227 KB)


// BN is the accumulator width per CTA (the MMA N).  With CG = 2 a pair of
// CTAs computes a 256 x BN tile with one tcgen05.mma.cta_group::2: each CTA
// loads its 128 rows of A and BN/2 columns of B and holds 128 x BN of D.
template <int MODE, int FMT, int BN, int PROF, int CG = 1>
struct GemmTraits {
  static constexpr int SW = slice_cols(MODE, FMT);     // columns per epilogue slice
  static constexpr int RPS = slot_rows(MODE, FMT, PROF);   // rows per state slot
  static constexpr int PARTS = kBM / RPS;              // slots per 128-row column slice
  // slots per tile, ordered (column slice, part) with the part varying fastest
  static constexpr int SLICES = PARTS * (BN / SW);
  static constexpr int HALF = SW / 2;                  // columns per epilogue thread per slice
  static constexpr int TM = kBM * CG;                  // weight rows per tile
  static constexpr int BNL = BN / CG;                  // B columns loaded per CTA
  static constexpr int BK = bk_of(CG);                 // tokens per operand stage
  static constexpr int A_BYTES = kBM * BK * 2;
  static constexpr int B_BYTES = BNL * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int W_ELEM =
      ((MODE == kModeStoreG || MODE == kModeAccum) && FMT == kFmtF32) ? 4 : 2;
  static constexpr int SFMT = state_elem_fmt(FMT);
  static constexpr int MOM_ELEM =
      (!has_state(MODE) || FMT == kFmtNone) ? 0
                                            : (SFMT == kFmtF32 ? 4 : (SFMT == kFmtBF16 ? 2 : 1));
  // 8-bit moments (int8 blocks or fp8): 128-column slices whose W is two
  // 64-column boxes
  static constexpr bool Q8 = (MODE == kModeFused && (FMT == kFmtI8 || FMT == kFmtF8));
  static constexpr bool F8 = (MODE == kModeFused && FMT == kFmtF8);
  static constexpr int W_BYTES = RPS * SW * W_ELEM;
  static constexpr int M_BYTES = RPS * SW * MOM_ELEM;
  // the fused step with an addend: an fp32 box of the accumulator after m, v
  static constexpr int ADD_BYTES = (MODE == kModeFused && has_addend(FMT)) ? RPS * SW * 4 : 0;
  static constexpr int SLOT_BYTES = W_BYTES + state_boxes(FMT) * M_BYTES + ADD_BYTES;
  // every box of a slot starts 1024-byte aligned (the 128-byte swizzle's atom)
  static_assert(W_BYTES % 1024 == 0 && M_BYTES % 1024 == 0 && SLOT_BYTES % 1024 == 0,
                "state boxes must stay 1024-byte aligned");
  static constexpr bool I8 = (MODE == kModeFused && FMT == kFmtI8);
  // int8 row-halves exchange: [2 halves][2 kinds][128 rows] floats
  static constexpr int XCH_BYTES = I8 ? 2 * 2 * kBM * 4 : 0;
  static constexpr int MAX_BARS = 2 * 6 + 4 + 3 * 6 + 5;
  static constexpr int BUDGET = kSmemLimit - (8 * MAX_BARS + 16 + XCH_BYTES);
  static constexpr int NS_CAP = 6;
  // state slots that fit next to `st` operand stages, a multiple of PARTS
  static constexpr int slots_beside(int st) {
    const int n = (BUDGET - st * STAGE_BYTES) / SLOT_BYTES;
    return ((n > NS_CAP ? NS_CAP : n) / PARTS) * PARTS;
  }
  static constexpr int stages_mma() {
    int st = 6;
    while (st > 2 && slots_beside(st) < 2) --st;
    return st;
  }
  static constexpr int stages_balanced() {
    int st = 6;
    while (st > 2 && slots_beside(st) < st) --st;
    return st;
  }
  static constexpr int STAGES =
      (PROF == kProfStream) ? 2
                            : (PROF == kProfMma || PROF == kProfDeep ? stages_mma() : stages_balanced());
  static constexpr int NS = slots_beside(STAGES);
  static_assert(NS >= 2, "shared memory does not fit two state slots");
  // int8 with 128-wide accumulators: the spare 256 tensor-memory columns hold
  // the epilogue's m', r' between its two passes
  static constexpr bool STASH = I8 && BN == 128;
  static constexpr int TMEM_COLS = STASH ? 512 : 2 * BN;
  // shared-memory carve (offsets from the 1024-aligned base)
  static constexpr int OFF_SLOTS = STAGES * STAGE_BYTES;
  static constexpr int OFF_BARS = OFF_SLOTS + NS * SLOT_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 3 * NS + 5;
  static constexpr int OFF_TMEM = OFF_BARS + 8 * NUM_BARS;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int OFF_XCH = (OFF_ABORT + 4 + 15) & ~15;
  static constexpr int SMEM_USED = OFF_XCH + XCH_BYTES;
  // Ask for 1 KB of slack to align the base; where that would pass the limit
  // the kernel checks at run time that its window is aligned well enough.
  static constexpr int SMEM_ALLOC =
      (SMEM_USED + 1024 < kSmemLimit) ? SMEM_USED + 1024 : kSmemLimit;
  static_assert(SMEM_USED <= kSmemLimit, "shared memory budget exceeded");
  static_assert(BN % SW == 0 && BNL % 64 == 0, "tile width");
  // the input-gradient mode loads A as K-major boxes 64 elements deep: one per stage
  static_assert(MODE != kModeDgrad || BK == 64, "K-major A boxes hold 64 elements of K");
  static_assert(MODE != kModeOpt || (FMT != kFmtI8 && FMT != kFmtF8),
                "the other optimizers keep fp32 or bf16 state");
  static_assert(MODE != kModeAccum || FMT == kFmtF32, "the accumulation buffer is fp32");
  static_assert(CG == 1 || (CG == 2 && BN == 256), "CTA pairs use 256 x 256 tiles");
  static_assert(TMEM_COLS <= 512, "tensor memory has 512 columns");
  // with half-tile slots each half of the epilogue owns every other slot
  static_assert(PARTS == 1 || (NS % PARTS == 0 && SLICES % PARTS == 0), "slot ownership");
};

struct WaitCtx {
  volatile uint32_t* abort_flag;
  int* err;
  int* site;          // where the first timeout happened (diagnostics)
  uint64_t timeout_ns;
};

// Wait sites, recorded as site*100000 + blockIdx.x*100 + index on a timeout.
enum WaitSite : int {
  kSiteProducerEmpty = 1, kSiteMmaTmemEmpty = 2, kSiteMmaFull = 3, kSiteLoaderEmpty = 4,
  kSiteEpiTmemFull = 5, kSiteEpiSlotFull = 6, kSiteEpiSlotFree = 7, kSiteDrainOperands = 8,
  kSiteDrainState = 9, kSiteDrainMma = 10, kSiteStoreSlotDone = 11, kSiteEpiExchange = 12
};

// Wait until the phase of `bar` with `parity` completes.  Gives up (returns
// false) when the CTA's abort flag is raised, if `honor_abort`, or when the
// time limit runs out, in which case it raises the abort flag and records the
// timeout in the device error word.
//
// The first test is inlined; only a wait that has to spin calls the bounded
// loop.  The MMA issuer passes through one wait per pipeline stage, and a
// call there (frame set-up, argument moves) sits between two stages' MMAs
// long enough for the tensor core to run dry: with the call the plain GEMM
// main loop ran 11 % slower.
static __device__ __noinline__ bool wait_spin(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                              int site, bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      *w.abort_flag = 1u;
      atomicCAS(w.err, 0, kErrDeviceTimeout);
      atomicCAS(w.site, 0, site * 100000 + static_cast<int>(blockIdx.x) * 100);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                             int site, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_spin(bar, parity, w, site, honor_abort);
}

// The operand-stage waits of the producer and the MMA issuer.  On one CTA
// they first poll with the non-blocking test (at most kSpinTests times)
// before the bounded wait, which may suspend the thread: the hand-off of a
// stage between the two threads is then quicker, worth 3 % at BT = 512 where
// two stages have to keep the main loop fed.  On CTA pairs, whose main loop
// reads shared memory at full rate, the polling costs more than it saves.
constexpr int kSpinTests = 4096;
template <bool SPIN>
__device__ __forceinline__ bool wait_stage(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                           int site) {
  if constexpr (SPIN) {
#pragma unroll 1
    for (int i = 0; i < kSpinTests; ++i)
      if (mbar_test_wait(bar, parity)) return true;
  }
  return wait_bounded(bar, parity, w, site);
}

// A bounded wait that polls with a short sleep between tests: quicker to
// notice a completed phase than a suspended wait, but issues few
// instructions while it waits.  Used by the store lanes where the host asks
// for it (GemmParams::poll_store).
__device__ __forceinline__ bool wait_poll(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                          int site) {
#pragma unroll 1
  for (int i = 0; i < kSpinTests; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    __nanosleep(32);
  }
  return wait_bounded(bar, parity, w, site);
}

// The k-steps [kb, ke) of work unit u of layer pi: split u % splits of the
// layer's num_k steps (never empty: the host keeps splits <= num_k).
__device__ __forceinline__ void split_range(int u, int pi, const GemmParams& p, int& kb,
                                            int& ke) {
  const int z = u % p.splits;
  const int nk = p.prob[pi].num_k;
  kb = (z * nk) / p.splits;
  ke = ((z + 1) * nk) / p.splits;
}

// Global tile index -> (layer, tile row, tile column).  Layers are laid out
// one after another in the queue; inside a layer, groups of group_m tile rows
// are walked column by column so that concurrent tiles share operand panels
// in L2.
__device__ __forceinline__ int tile_coords(int t, const GemmParams& p, int& tm, int& tn) {
  int pi = 0;
#pragma unroll
  for (int i = 1; i < kMaxGroup; ++i)
    if (i < p.nprob && t >= p.prob[i].tile_start) pi = i;
  const GemmProblem& q = p.prob[pi];
  const int lt = t - q.tile_start;
  const int per_group = p.group_m * q.tiles_n;
  const int g = lt / per_group;
  const int first_m = g * p.group_m;
  const int gsize = min(q.tiles_m - first_m, p.group_m);
  const int r = lt - g * per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
  return pi;
}

// ---------------------------------------------------------------------------
// Epilogue slice bodies.  Each epilogue thread owns one tile row (`row`, the
// TMEM lane) and HALF consecutive columns of the slice.
// ---------------------------------------------------------------------------

// The thread's 16 columns of one state box in the slot: fp32 boxes have
// 128-byte rows (128-byte swizzle), bf16 boxes 64-byte rows (64-byte swizzle).
template <int FMT>
__device__ __forceinline__ void state_ld16(const uint8_t* box, uint32_t row, int h,
                                           float (&x)[16]) {
  if constexpr (FMT == kFmtF32) {
    float4 q[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      q[c] = *reinterpret_cast<const float4*>(box + sw128_off(row, 4 * h + c));
    const float* f = reinterpret_cast<const float*>(q);
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = f[i];
  } else {
    uint4 q[2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
      q[c] = *reinterpret_cast<const uint4*>(box + sw64_off(row, 2 * h + c));
    const uint32_t* u = reinterpret_cast<const uint32_t*>(q);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_lo(u[i]);
      x[2 * i + 1] = bf16_hi(u[i]);
    }
  }
}
template <int FMT>
__device__ __forceinline__ void state_st16(uint8_t* box, uint32_t row, int h,
                                           const float (&x)[16]) {
  if constexpr (FMT == kFmtF32) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<float4*>(box + sw128_off(row, 4 * h + c)) =
          make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
  } else {
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
#pragma unroll
    for (int c = 0; c < 2; ++c)
      *reinterpret_cast<uint4*>(box + sw64_off(row, 2 * h + c)) =
          make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
  }
}

// fp32 or bf16 moments; SW = 32, HALF = 16.
// `row` is the thread's row inside the RPS-row slot (its TMEM lane is in
// `taddr`); the slot holds the W, m and v boxes of RPS rows back to back.
// With `sr` the weight is committed by stochastic rounding: the random bits
// of the thread's 16 columns are the Philox block with counter (grow, gcol16,
// sr_step, 0), grow the global weight row and gcol16 the first column / 16.
template <int SLOT_FMT, int RPS>
__device__ __forceinline__ void epi_slice_fused_16(uint32_t taddr, bool zero_grad, uint8_t* slot,
                                                   uint32_t row, int h, const AdamWConsts& hc,
                                                   bool sr, uint64_t sr_seed, uint32_t sr_step,
                                                   uint32_t grow, uint32_t gcol16) {
  constexpr int FMT = state_elem_fmt(SLOT_FMT);   // fp32 or bf16 moments
  constexpr int kWBytes = RPS * 32 * 2;
  constexpr int kMBytes = RPS * 32 * (FMT == kFmtF32 ? 4 : 2);
  // the accumulator load runs while the slot's W, m and v are read from
  // shared memory; its registers are read only after the wait
  uint32_t graw[16];
  tmem_ld_x16(taddr, graw);
  float g[16], w[16], m[16], v[16];

  uint8_t* wbox = slot;                 // [RPS][32] bf16: 64-byte rows
  uint8_t* mbox = slot + kWBytes;
  uint8_t* vbox = mbox + kMBytes;
  uint4 wq[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) wq[c] = *reinterpret_cast<const uint4*>(wbox + sw64_off(row, 2 * h + c));
  const uint32_t* wu = reinterpret_cast<const uint32_t*>(wq);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w[2 * i] = bf16_lo(wu[i]);
    w[2 * i + 1] = bf16_hi(wu[i]);
  }
  if constexpr (FMT == kFmtF32) {        // [RPS][32] fp32: 128-byte rows
    float4 mq[4], vq[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      mq[c] = *reinterpret_cast<const float4*>(mbox + sw128_off(row, 4 * h + c));
      vq[c] = *reinterpret_cast<const float4*>(vbox + sw128_off(row, 4 * h + c));
    }
    const float* mf = reinterpret_cast<const float*>(mq);
    const float* vf = reinterpret_cast<const float*>(vq);
#pragma unroll
    for (int i = 0; i < 16; ++i) { m[i] = mf[i]; v[i] = vf[i]; }
  } else {                               // [RPS][32] bf16: 64-byte rows
    uint4 mq[2], vq[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      mq[c] = *reinterpret_cast<const uint4*>(mbox + sw64_off(row, 2 * h + c));
      vq[c] = *reinterpret_cast<const uint4*>(vbox + sw64_off(row, 2 * h + c));
    }
    const uint32_t* mu = reinterpret_cast<const uint32_t*>(mq);
    const uint32_t* vu = reinterpret_cast<const uint32_t*>(vq);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      m[2 * i] = bf16_lo(mu[i]); m[2 * i + 1] = bf16_hi(mu[i]);
      v[2 * i] = bf16_lo(vu[i]); v[2 * i + 1] = bf16_hi(vu[i]);
    }
  }
  float b[16];   // the addend (accumulator of the earlier micro-batches)
  if constexpr (has_addend(SLOT_FMT)) state_ld16<kFmtF32>(mbox + 2 * kMBytes, row, h, b);
  tmem_ld_wait();
  if (zero_grad) {   // warp-uniform: no accumulator was written
#pragma unroll
    for (int i = 0; i < 16; ++i) graw[i] = 0u;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) g[i] = __uint_as_float(graw[i]);
  if constexpr (has_addend(SLOT_FMT)) {
    // the gradient the step reads: fp32(B + G), as the accumulate mode forms it
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = __fadd_rn(b[i], g[i]);
  }
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float2 w2 = make_float2(w[i], w[i + 1]), m2 = make_float2(m[i], m[i + 1]);
    float2 v2 = make_float2(v[i], v[i + 1]), r2;
    adamw_elem2(make_float2(g[i], g[i + 1]), w2, m2, v2, r2, hc);
    w[i] = w2.x; w[i + 1] = w2.y;
    m[i] = m2.x; m[i + 1] = m2.y;
    v[i] = v2.x; v[i + 1] = v2.y;
  }
  uint32_t wo[8];
  if (sr) {
    uint64_t rb[4] = {grow, gcol16, sr_step, 0ull};
    philox4x64_10(rb, sr_seed, 0ull);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t r0 = static_cast<uint32_t>(rb[(2 * i) >> 2] >> (16 * ((2 * i) & 3))) & 0xFFFFu;
      const uint32_t r1 =
          static_cast<uint32_t>(rb[(2 * i + 1) >> 2] >> (16 * ((2 * i + 1) & 3))) & 0xFFFFu;
      wo[i] = sr_bf16_bits(w[2 * i], r0) | (sr_bf16_bits(w[2 * i + 1], r1) << 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) wo[i] = pack_bf16x2(w[2 * i], w[2 * i + 1]);
  }
#pragma unroll
  for (int c = 0; c < 2; ++c)
    *reinterpret_cast<uint4*>(wbox + sw64_off(row, 2 * h + c)) =
        make_uint4(wo[4 * c], wo[4 * c + 1], wo[4 * c + 2], wo[4 * c + 3]);
  if constexpr (FMT == kFmtF32) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      *reinterpret_cast<float4*>(mbox + sw128_off(row, 4 * h + c)) =
          make_float4(m[4 * c], m[4 * c + 1], m[4 * c + 2], m[4 * c + 3]);
      *reinterpret_cast<float4*>(vbox + sw128_off(row, 4 * h + c)) =
          make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
  } else {
    uint32_t mo[8], vo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mo[i] = pack_bf16x2(m[2 * i], m[2 * i + 1]);
      vo[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      *reinterpret_cast<uint4*>(mbox + sw64_off(row, 2 * h + c)) =
          make_uint4(mo[4 * c], mo[4 * c + 1], mo[4 * c + 2], mo[4 * c + 3]);
      *reinterpret_cast<uint4*>(vbox + sw64_off(row, 2 * h + c)) =
          make_uint4(vo[4 * c], vo[4 * c + 1], vo[4 * c + 2], vo[4 * c + 3]);
    }
  }
}

// 32 int8 codes (two 16-byte chunks) as 16 pairs of floats, without
// conversion instructions (i8_code_pair).
__device__ __forceinline__ void load_code_pairs32(const uint8_t* box, uint32_t row, int chunk0,
                                                  float2 (&q)[16]) {
  const uint4 a = *reinterpret_cast<const uint4*>(box + sw128_off(row, chunk0));
  const uint4 b = *reinterpret_cast<const uint4*>(box + sw128_off(row, chunk0 + 1));
  const uint32_t words[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t off = words[i] ^ 0x80808080u;
    q[2 * i] = i8_code_pair(off, 0);
    q[2 * i + 1] = i8_code_pair(off, 2);
  }
}
// Store 32 codes, each in the low byte of its word (quant_m_bits / quant_r_bits).
__device__ __forceinline__ void store_codes32(uint8_t* box, uint32_t row, int chunk0,
                                              const uint32_t (&q)[32]) {
  uint32_t words[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    words[i] = pack_low_bytes4(q[4 * i], q[4 * i + 1], q[4 * i + 2], q[4 * i + 3]);
  *reinterpret_cast<uint4*>(box + sw128_off(row, chunk0)) =
      make_uint4(words[0], words[1], words[2], words[3]);
  *reinterpret_cast<uint4*>(box + sw128_off(row, chunk0 + 1)) =
      make_uint4(words[4], words[5], words[6], words[7]);
}

// int8 moments; SW = 128 (one quantisation block), HALF = 64.  Two passes
// over the thread's 64 columns: the first updates W and finds the block
// absmax of m' and r' = sqrt(v') (combined with the partner thread, in the
// other epilogue warp of the same TMEM lane quadrant, that holds the other 64
// columns of the row), the second recomputes m', r' and writes their codes.
// The two halves meet at an mbarrier (bounded wait).  `xch` is one buffer:
// before writing it a thread waits until every thread has read the previous
// block's values (bar_xch_read), so a fast thread cannot overwrite them.
// Returns false (warp-uniform) if a wait timed out.
// `row` is the thread's row inside the RPS-row slot, `trow` its TMEM lane.
// STASH: the first pass parks m' and r' (fp32) in 128 spare tensor-memory
// columns at `saddr` (this thread's lane) and the second pass reads them back
// instead of dequantising and updating the moments a second time; possible
// when the accumulators leave 256 of the 512 columns free (128-wide tiles).
// sm_old, sv_old: the block's current scales (0 for rows outside the weight).
template <int RPS, bool STASH>
__device__ __forceinline__ bool epi_slice_fused_i8(uint32_t taddr, uint32_t saddr, bool zero_grad,
                                                   bool active, uint8_t* slot, float* xch,
                                                   uint32_t bar_xch, uint32_t bar_xch_read,
                                                   uint32_t xphase, const WaitCtx& wc,
                                                   uint32_t row, uint32_t trow, int h,
                                                   float sm_old, float sv_old,
                                                   float* m_scale_rc, float* v_scale_rc,
                                                   const AdamWConsts& hc) {
  constexpr int kWBytes = RPS * 128 * 2;
  constexpr int kMBytes = RPS * 128;
  uint8_t* wbox = slot + h * (RPS * 64 * 2);   // box h: [RPS][64] bf16, 128-byte rows
  uint8_t* mbox = slot + kWBytes;              // [RPS][128] int8
  uint8_t* vbox = mbox + kMBytes;
  float amax_m = 0.0f, amax_r = 0.0f;
  const float2 sm2 = dup2(sm_old), sv2 = dup2(sv_old);
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t graw[32];
    tmem_ld_x32(taddr + 32 * c, graw);   // in flight while the codes and W are read
    float2 qm[16], qv[16];
    load_code_pairs32(mbox, row, 4 * h + 2 * c, qm);
    load_code_pairs32(vbox, row, 4 * h + 2 * c, qv);
    uint4 wq[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      wq[k] = *reinterpret_cast<const uint4*>(wbox + sw128_off(row, 4 * c + k));
    const uint32_t* wu = reinterpret_cast<const uint32_t*>(wq);
    tmem_ld_wait();
    if (zero_grad) {   // warp-uniform: no accumulator was written
#pragma unroll
      for (int i = 0; i < 32; ++i) graw[i] = 0u;
    }
    uint32_t wo[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float2 w2 = make_float2(bf16_lo(wu[i]), bf16_hi(wu[i]));
      const float2 g2 = make_float2(__uint_as_float(graw[2 * i]), __uint_as_float(graw[2 * i + 1]));
      float2 m2 = dequant_m2(qm[i], sm2), v2 = dequant_v2(qv[i], sv2), r2;
      adamw_elem2(g2, w2, m2, v2, r2, hc);
      amax_m = max3_abs(amax_m, m2.x, m2.y);
      amax_r = max3(amax_r, r2.x, r2.y);
      wo[i] = pack_bf16x2(w2.x, w2.y);
      if constexpr (STASH) {   // the old codes are consumed: reuse their registers
        qm[i] = m2;
        qv[i] = r2;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint4*>(wbox + sw128_off(row, 4 * c + k)) =
          make_uint4(wo[4 * k], wo[4 * k + 1], wo[4 * k + 2], wo[4 * k + 3]);
    if constexpr (STASH) {
      uint32_t su[32], sv[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        su[2 * i] = __float_as_uint(qm[i].x);
        su[2 * i + 1] = __float_as_uint(qm[i].y);
        sv[2 * i] = __float_as_uint(qv[i].x);
        sv[2 * i + 1] = __float_as_uint(qv[i].y);
      }
      tmem_st_x32(saddr + 64 * c, su);
      tmem_st_x32(saddr + 64 * c + 32, sv);
    }
  }
  // the second pass's first stash chunk (this thread's own m', r') is read
  // from tensor memory while the row's two halves meet
  uint32_t ms[32], rs[32];
  if constexpr (STASH) {
    tmem_st_wait();
    tmem_ld_x32(saddr, ms);
    tmem_ld_x32(saddr + 32, rs);
  }
  // combine the row's two halves
  bool ok = wait_bounded(bar_xch_read, xphase ^ 1u, wc, kSiteEpiExchange);
  if (!__all_sync(0xffffffffu, ok)) return false;
  xch[(h * 2 + 0) * kBM + trow] = amax_m;
  xch[(h * 2 + 1) * kBM + trow] = amax_r;
  mbar_arrive(bar_xch);
  ok = wait_bounded(bar_xch, xphase, wc, kSiteEpiExchange);
  if (!__all_sync(0xffffffffu, ok)) return false;
  amax_m = fmaxf(amax_m, xch[((1 - h) * 2 + 0) * kBM + trow]);
  amax_r = fmaxf(amax_r, xch[((1 - h) * 2 + 1) * kBM + trow]);
  mbar_arrive(bar_xch_read);
  const float inv_m = int8_inv_step(amax_m), inv_r = int8_inv_step(amax_r);
  const float2 inv_m2 = dup2(inv_m), inv_r2 = dup2(inv_r);
  const float r_floor = amax_r > 0.0f ? 1.0f : 0.0f;   // codes >= 1 in a non-zero block
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t bm[32], bv[32];
    if constexpr (STASH) {
      if (c == 1) {
        tmem_ld_x32(saddr + 64, ms);
        tmem_ld_x32(saddr + 96, rs);
      }
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        quant_m_bits2(make_float2(__uint_as_float(ms[i]), __uint_as_float(ms[i + 1])), inv_m2,
                      bm[i], bm[i + 1]);
        quant_r_bits2(make_float2(__uint_as_float(rs[i]), __uint_as_float(rs[i + 1])), inv_r2,
                      r_floor, bv[i], bv[i + 1]);
      }
    } else {
      uint32_t graw[32];
      tmem_ld_x32(taddr + 32 * c, graw);
      float2 qm[16], qv[16];
      load_code_pairs32(mbox, row, 4 * h + 2 * c, qm);
      load_code_pairs32(vbox, row, 4 * h + 2 * c, qv);
      tmem_ld_wait();
      if (zero_grad) {
#pragma unroll
        for (int i = 0; i < 32; ++i) graw[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 g = make_float2(__uint_as_float(graw[2 * i]), __uint_as_float(graw[2 * i + 1]));
        float2 w = make_float2(0.0f, 0.0f), r;
        float2 m = dequant_m2(qm[i], sm2), v = dequant_v2(qv[i], sv2);
        adamw_elem2(g, w, m, v, r, hc);
        quant_m_bits2(m, inv_m2, bm[2 * i], bm[2 * i + 1]);
        quant_r_bits2(r, inv_r2, r_floor, bv[2 * i], bv[2 * i + 1]);
      }
    }
    store_codes32(mbox, row, 4 * h + 2 * c, bm);
    store_codes32(vbox, row, 4 * h + 2 * c, bv);
  }
  if (active && h == 0) {
    *m_scale_rc = int8_scale(amax_m);
    *v_scale_rc = int8_scale(amax_r);
  }
  return true;
}

// fp8 moments with per-tensor scales; SW = 128, HALF = 64.  One pass: the
// scales are the caller's (delayed scaling), so no block absmax is needed
// before the codes are written.  The thread's running amaxes of m' and
// r' = sqrt(v') are raised for the caller's next scales.
template <int RPS>
__device__ __forceinline__ void epi_slice_fused_f8(uint32_t taddr, bool zero_grad, uint8_t* slot,
                                                   uint32_t row, int h, const AdamWConsts& hc,
                                                   const Fp8Step& fm, const Fp8Step& fr,
                                                   float& amax_m, float& amax_r) {
  constexpr int kWBytes = RPS * 128 * 2;
  constexpr int kMBytes = RPS * 128;
  uint8_t* wbox = slot + h * (RPS * 64 * 2);   // box h: [RPS][64] bf16, 128-byte rows
  uint8_t* mbox = slot + kWBytes;              // [RPS][128] e4m3
  uint8_t* vbox = mbox + kMBytes;
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t graw[32];
    tmem_ld_x32(taddr + 32 * c, graw);
    // the first 16 columns' codes and W are read while the accumulator load
    // is in flight
    uint4 mq = *reinterpret_cast<const uint4*>(mbox + sw128_off(row, 4 * h + 2 * c));
    uint4 rq = *reinterpret_cast<const uint4*>(vbox + sw128_off(row, 4 * h + 2 * c));
    uint4 wq[2];
#pragma unroll
    for (int k = 0; k < 2; ++k)
      wq[k] = *reinterpret_cast<const uint4*>(wbox + sw128_off(row, 4 * c + k));
    tmem_ld_wait();
    if (zero_grad) {
#pragma unroll
      for (int i = 0; i < 32; ++i) graw[i] = 0u;
    }
#pragma unroll
    for (int p16 = 0; p16 < 2; ++p16) {
      const int chunk = 4 * h + 2 * c + p16;     // 16 codes of m and of r
      if (p16 == 1) {
        mq = *reinterpret_cast<const uint4*>(mbox + sw128_off(row, chunk));
        rq = *reinterpret_cast<const uint4*>(vbox + sw128_off(row, chunk));
#pragma unroll
        for (int k = 0; k < 2; ++k)
          wq[k] = *reinterpret_cast<const uint4*>(wbox + sw128_off(row, 4 * c + 2 + k));
      }
      const uint32_t* wu = reinterpret_cast<const uint32_t*>(wq);
      float g[16], w[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        w[2 * i] = bf16_lo(wu[i]);
        w[2 * i + 1] = bf16_hi(wu[i]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) g[i] = __uint_as_float(graw[16 * p16 + i]);
      adamw_fp8_x16(g, w, mq, rq, fm, fr, hc, amax_m, amax_r);
      uint32_t wo[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) wo[i] = pack_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
      for (int k = 0; k < 2; ++k)
        *reinterpret_cast<uint4*>(wbox + sw128_off(row, 4 * c + 2 * p16 + k)) =
            make_uint4(wo[4 * k], wo[4 * k + 1], wo[4 * k + 2], wo[4 * k + 3]);
      *reinterpret_cast<uint4*>(mbox + sw128_off(row, chunk)) = mq;
      *reinterpret_cast<uint4*>(vbox + sw128_off(row, chunk)) = rq;
    }
  }
}

// Store-G: write the fp32 accumulator as fp32 or bf16.  SW = 32, HALF = 16.
template <int FMT>
__device__ __forceinline__ void epi_slice_store(uint32_t taddr, bool zero_grad, uint8_t* slot,
                                                uint32_t row, int h) {
  uint32_t graw[16];
  tmem_ld_x16(taddr, graw);
  tmem_ld_wait();
  float g[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) g[i] = zero_grad ? 0.0f : __uint_as_float(graw[i]);
  if constexpr (FMT == kFmtF32) {        // [128][32] fp32: 128-byte rows
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<float4*>(slot + sw128_off(row, 4 * h + c)) =
          make_float4(g[4 * c], g[4 * c + 1], g[4 * c + 2], g[4 * c + 3]);
  } else {                               // [128][32] bf16: 64-byte rows
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(g[2 * i], g[2 * i + 1]);
#pragma unroll
    for (int c = 0; c < 2; ++c)
      *reinterpret_cast<uint4*>(slot + sw64_off(row, 2 * h + c)) =
          make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
  }
}

// The other optimizers (kModeOpt): the slice of epi_slice_fused_16 with
// optimizer OPT's element update, touching only the states OPT has.
template <int SLOT_FMT, int RPS, int OPT>
__device__ __forceinline__ void epi_slice_opt(uint32_t taddr, bool zero_grad, uint8_t* slot,
                                              uint32_t row, int h, const OptConsts& oc) {
  constexpr int FMT = state_elem_fmt(SLOT_FMT);
  constexpr int kWBytes = RPS * 32 * 2;
  constexpr int kMBytes = RPS * 32 * (FMT == kFmtF32 ? 4 : 2);
  constexpr int NST = opt_states(OPT);
  uint32_t graw[16];
  tmem_ld_x16(taddr, graw);   // in flight while the slot's state is read
  float w[16], s1[16], s2[16];
  state_ld16<kFmtBF16>(slot, row, h, w);
  if constexpr (NST >= 1) state_ld16<FMT>(slot + kWBytes, row, h, s1);
  if constexpr (NST >= 2) state_ld16<FMT>(slot + kWBytes + kMBytes, row, h, s2);
  tmem_ld_wait();
  if (zero_grad) {
#pragma unroll
    for (int i = 0; i < 16; ++i) graw[i] = 0u;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) opt_elem<OPT>(__uint_as_float(graw[i]), w[i], s1[i], s2[i], oc);
  state_st16<kFmtBF16>(slot, row, h, w);
  if constexpr (NST >= 1) state_st16<FMT>(slot + kWBytes, row, h, s1);
  if constexpr (NST >= 2) state_st16<FMT>(slot + kWBytes + kMBytes, row, h, s2);
}
// Dispatch on the launch's optimizer (uniform across the grid); stateless
// slots (kFmtNone) only ever run SGD.
template <int FMT, int RPS>
__device__ __forceinline__ void epi_slice_opt_any(const OptConsts& oc, uint32_t taddr,
                                                  bool zero_grad, uint8_t* slot, uint32_t row,
                                                  int h) {
  if constexpr (FMT == kFmtNone) {
    epi_slice_opt<FMT, RPS, kOptSgd>(taddr, zero_grad, slot, row, h, oc);
    return;
  } else if constexpr (state_boxes(FMT) == 1) {
    // one-state slots: SGD with momentum, Adagrad, RMSprop, Lion
    switch (oc.opt) {
      case kOptSgdMomentum:
        epi_slice_opt<FMT, RPS, kOptSgdMomentum>(taddr, zero_grad, slot, row, h, oc);
        break;
      case kOptAdagrad: epi_slice_opt<FMT, RPS, kOptAdagrad>(taddr, zero_grad, slot, row, h, oc); break;
      case kOptRmsprop: epi_slice_opt<FMT, RPS, kOptRmsprop>(taddr, zero_grad, slot, row, h, oc); break;
      default: epi_slice_opt<FMT, RPS, kOptLion>(taddr, zero_grad, slot, row, h, oc); break;
    }
    return;
  }
  switch (oc.opt) {
    case kOptSgd: epi_slice_opt<FMT, RPS, kOptSgd>(taddr, zero_grad, slot, row, h, oc); break;
    case kOptSgdMomentum:
      epi_slice_opt<FMT, RPS, kOptSgdMomentum>(taddr, zero_grad, slot, row, h, oc);
      break;
    case kOptAdagrad: epi_slice_opt<FMT, RPS, kOptAdagrad>(taddr, zero_grad, slot, row, h, oc); break;
    case kOptRmsprop: epi_slice_opt<FMT, RPS, kOptRmsprop>(taddr, zero_grad, slot, row, h, oc); break;
    case kOptLion: epi_slice_opt<FMT, RPS, kOptLion>(taddr, zero_grad, slot, row, h, oc); break;
    case kOptNadam: epi_slice_opt<FMT, RPS, kOptNadam>(taddr, zero_grad, slot, row, h, oc); break;
    default: epi_slice_opt<FMT, RPS, kOptRadam>(taddr, zero_grad, slot, row, h, oc); break;
  }
}

// Accumulate mode: B' = beta B + G into the slot's fp32 box (B loaded there
// by the state loader unless beta = 0, when the old B is not read).
__device__ __forceinline__ void epi_slice_accum(uint32_t taddr, bool zero_grad, uint8_t* slot,
                                                uint32_t row, int h, float beta, bool load) {
  uint32_t graw[16];
  tmem_ld_x16(taddr, graw);   // in flight while B is read
  float b[16], o[16];
  if (load) state_ld16<kFmtF32>(slot, row, h, b);
  tmem_ld_wait();
  if (zero_grad) {
#pragma unroll
    for (int i = 0; i < 16; ++i) graw[i] = 0u;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float g = __uint_as_float(graw[i]);
    o[i] = load ? __fmaf_rn(beta, b[i], g) : g;
  }
  state_st16<kFmtF32>(slot, row, h, o);
}

// Split reduction of the input gradient.  A CTA's fp32 partial tile (128 rows
// x BN) is laid out so that a warp's accesses are contiguous: column slice cb,
// half h and quarter j of a thread's 16 columns form a run of 128 float4, one
// per row, at float4 index ((cb * 2 + h) * 4 + j) * 128 + row.  The reduce
// kernel (forge_dgrad_reduce.cu) reads the same layout.
__device__ __forceinline__ void epi_part_write(uint32_t taddr, float* part, int cb, int h,
                                               uint32_t row) {
  uint32_t g[16];
  tmem_ld_x16(taddr, g);
  tmem_ld_wait();
  float4* dst = reinterpret_cast<float4*>(part) + (cb * 2 + h) * 4 * kBM + row;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    __stcg(dst + j * kBM, make_float4(__uint_as_float(g[4 * j]), __uint_as_float(g[4 * j + 1]),
                                      __uint_as_float(g[4 * j + 2]), __uint_as_float(g[4 * j + 3])));
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int MODE, int FMT, int BN, int PROF, int CG>
__global__ void __launch_bounds__(kNumThreads, 1)
    forge_gemm_kernel(const __grid_constant__ GemmArgs a) {
  const GemmParams& p = a.p;
  using T = GemmTraits<MODE, FMT, BN, PROF, CG>;
  constexpr bool kPair = (CG == 2);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  {
    uint32_t dyn;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (base - raw + T::SMEM_USED > dyn) {   // uniform across the CTA: nothing started yet
      if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrDeviceConfig);
      return;
    }
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A CTA pair walks the tiles as one unit; rank 0 issues the pair's MMAs.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  const int unit0 = kPair ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  // work unit -> tile: the input gradient's split reduction gives each tile
  // `splits` consecutive units; elsewhere a unit is a tile
  auto tile_of = [&](int u) { return MODE == kModeDgrad ? u / p.splits : u; };

  const uint32_t bars = base + T::OFF_BARS;
  auto bar_full = [&](int s) { return bars + 8u * s; };
  auto bar_empty = [&](int s) { return bars + 8u * (T::STAGES + s); };
  auto bar_tfull = [&](int b) { return bars + 8u * (2 * T::STAGES + b); };
  auto bar_tempty = [&](int b) { return bars + 8u * (2 * T::STAGES + 2 + b); };
  auto bar_sfull = [&](int j) { return bars + 8u * (2 * T::STAGES + 4 + j); };
  auto bar_sempty = [&](int j) { return bars + 8u * (2 * T::STAGES + 4 + T::NS + j); };
  auto bar_sdone = [&](int j) { return bars + 8u * (2 * T::STAGES + 4 + 2 * T::NS + j); };
  const uint32_t bar_drain = bars + 8u * (2 * T::STAGES + 4 + 3 * T::NS);
  // int8 row-half exchange barriers, one pair per slot part: [xch0, xch1, read0, read1]
  const uint32_t bar_xch0 = bar_drain + 8u;
  const uint32_t bar_xch_read0 = bar_drain + 24u;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + T::OFF_ABORT);
  const WaitCtx wc{abort_flag, p.err, p.err_site, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < T::STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull(b), 1);
      mbar_init(bar_tempty(b), CG * (kEpiThreads / 32));   // one arrival per epilogue warp
    }
    for (int j = 0; j < T::NS; ++j) {
      mbar_init(bar_sfull(j), 1);
      mbar_init(bar_sempty(j), 1);
      mbar_init(bar_sdone(j), kEpiThreads / T::PARTS);
    }
    mbar_init(bar_drain, 1);
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar_xch0 + 8u * g, kEpiThreads / T::PARTS);
      mbar_init(bar_xch_read0 + 8u * g, kEpiThreads / T::PARTS);
    }
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.nprob; ++i) {
      if (p.num_k > 0) {   // with no tokens the operand descriptors are never encoded
        tma_prefetch_desc(&a.maps[i].dy);
        tma_prefetch_desc(&a.maps[i].x);
      }
      tma_prefetch_desc(&a.maps[i].w);
      if (MODE == kModeFused || (MODE == kModeOpt && p.nstate >= 1)) tma_prefetch_desc(&a.maps[i].m);
      if (MODE == kModeFused || (MODE == kModeOpt && p.nstate >= 2)) tma_prefetch_desc(&a.maps[i].v);
      if (T::ADD_BYTES) tma_prefetch_desc(&a.maps[i].b);
    }
  }
  // the peer's barriers must be initialised before any cross-CTA arrival
  if constexpr (kPair) cluster_sync_all(); else __syncthreads();
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(base + T::OFF_TMEM, T::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(base + T::OFF_TMEM, T::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gbase + T::OFF_TMEM);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lanes 0..NBOX-1 each issue one box per stage (A rows 0-63 and 64-127,
    // then the B column blocks), so one warp-wide TMA instruction carries all
    // of a stage's loads; four back-to-back single-lane issues measured 3 %
    // slower on the plain GEMM.
    constexpr int NBOX = 2 + T::BNL / 64;
    if (lane < NBOX) {
      const uint64_t pol = l2_policy_evict_last();
      uint32_t cnt = 0;
      int32_t last_armed[T::STAGES];
#pragma unroll
      for (int s = 0; s < T::STAGES; ++s) last_armed[s] = -1;
      bool ok = true;
      for (int t = unit0; ok && t < p.num_units; t += units) {
        int tm, tn;
        const int pi = tile_coords(tile_of(t), p, tm, tn);
        const GemmMaps& maps = a.maps[pi];
        int kb, ke;
        split_range(t, pi, p, kb, ke);
        for (int k = kb; k < ke; ++k, ++cnt) {
          const int s = cnt % T::STAGES;
          const uint32_t ph = (cnt / T::STAGES) & 1u;
          if (!wait_stage<!kPair>(bar_empty(s), ph ^ 1u, wc, kSiteProducerEmpty)) { ok = false; break; }
          if (p.drop_first_arrival && cnt == 0) continue;   // testing aid
          const uint32_t dst = base + s * T::STAGE_BYTES;
          const int ya = tm * T::TM + static_cast<int>(rank) * kBM;      // this CTA's A rows
          const int xb = tn * BN + static_cast<int>(rank) * T::BNL;      // this CTA's B columns
          // A boxes: 64 rows of M x 64 of K (dgrad, K-major: x = K, y = rows) or
          // 64 of M x 64 tokens (MN-major: x = M, y = tokens); B boxes: 64 of N
          // x 64 of K, MN-major in both
          const CUtensorMap* bm = lane < 2 ? &maps.dy : &maps.x;
          const bool a_kmaj = (MODE == kModeDgrad) && lane < 2;
          const int bx = a_kmaj ? k * T::BK : (lane < 2 ? ya + 64 * lane : xb + 64 * (lane - 2));
          const int by = a_kmaj ? ya + 64 * lane : k * T::BK;
          const uint32_t bdst = lane < 2 ? dst + lane * 64 * T::BK * 2
                                         : dst + T::A_BYTES + (lane - 2) * 64 * T::BK * 2;
          if constexpr (kPair) {
            // both CTAs' loads complete on the leader's barrier, which expects both
            const uint32_t fb = mapa_shared(bar_full(s), 0);
            if (leader && lane == 0) mbar_arrive_expect_tx(bar_full(s), 2 * T::STAGE_BYTES);
            tma_load_2d_pair(bdst, bm, bx, by, fb, pol);
          } else {
            if (lane == 0) mbar_arrive_expect_tx(bar_full(s), T::STAGE_BYTES);
            tma_load_2d(bdst, bm, bx, by, bar_full(s), pol);
          }
          if (leader) last_armed[s] = static_cast<int32_t>(cnt);
        }
      }
      // let every armed load land before the CTA can exit
      for (int s = 0; s < T::STAGES; ++s)
        if (last_armed[s] >= 0)
          wait_bounded(bar_full(s), (static_cast<uint32_t>(last_armed[s]) / T::STAGES) & 1u, wc,
                       kSiteDrainOperands, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr bool kAK = (MODE == kModeDgrad);   // A (dY) is K-major
      constexpr uint32_t idesc = make_idesc_bf16(T::TM, BN, !kAK, true);
      constexpr uint32_t kLBO = T::BK * 128;   // next 64-element group along M/N
      constexpr uint32_t kSBO = 1024;        // next 8-token group
      uint32_t cnt = 0;
      bool ok = true;
      int it = 0;
      for (int t = unit0; ok && t < p.num_units; t += units, ++it) {
        const int buf = it & 1;
        const uint32_t use = (it >> 1) & 1;
        if (!wait_bounded(bar_tempty(buf), use ^ 1u, wc, kSiteMmaTmemEmpty)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d = tmem_base + buf * BN;
        int kb, ke;
        {
          int tm_, tn_;
          split_range(t, tile_coords(tile_of(t), p, tm_, tn_), p, kb, ke);
        }
        for (int k = kb; k < ke; ++k, ++cnt) {
          const int s = cnt % T::STAGES;
          const uint32_t ph = (cnt / T::STAGES) & 1u;
          if (!wait_stage<!kPair>(bar_full(s), ph, wc, kSiteMmaFull)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a0 = base + s * T::STAGE_BYTES;
          const uint32_t b0 = a0 + T::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < T::BK / 16; ++kk) {
            const uint64_t ad = kAK ? make_sdesc_k_sw128(a0 + kk * 32, kSBO)
                                    : make_sdesc_mn_sw128(a0 + kk * 2048, kLBO, kSBO);
            const uint64_t bd = make_sdesc_mn_sw128(b0 + kk * 2048, kLBO, kSBO);
            if constexpr (kPair)
              umma_bf16_pair(d, ad, bd, idesc, (k != kb || kk != 0) ? 1u : 0u);
            else
              umma_bf16(d, ad, bd, idesc, (k != kb || kk != 0) ? 1u : 0u);
          }
          // frees stage s in both CTAs once these MMAs have read it
          if constexpr (kPair) umma_commit_pair_mc(bar_empty(s), 0x3); else umma_commit(bar_empty(s));
        }
        if (!ok) break;
        if constexpr (kPair) {
          umma_commit_pair_mc(bar_tfull(buf), 0x3);
        } else {
          if (ke > kb)
            umma_commit(bar_tfull(buf));
          else
            mbar_arrive(bar_tfull(buf));
        }
      }
      // every MMA issued must complete before the tensor memory is freed
      if constexpr (kPair) umma_commit_pair_mc(bar_drain, 0x1); else umma_commit(bar_drain);
      wait_bounded(bar_drain, 0u, wc, kSiteDrainMma, false);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ state loader
    if ((has_state(MODE) || MODE == kModeAccum) && lane == 0) {
      // Normal priority, not evict-first: a 32-column slice covers only half
      // of a 128-byte line of W (and of bf16 m, v), and the slice after it
      // reads the other half a moment later.  Marked evict-first, the line
      // is often gone by then and DRAM serves it twice (measured: 24 % more
      // DRAM reads at BT = 512 with fp32 moments, 69 % with bf16 moments);
      // at normal priority the reads equal the state's size.
      const uint64_t pol = l2_policy_evict_normal();
      const uint64_t pol_first = l2_policy_evict_first();
      uint32_t cnt = 0;
      int32_t last_armed[T::NS];
#pragma unroll
      for (int j = 0; j < T::NS; ++j) last_armed[j] = -1;
      bool ok = true;
      // L2 prefetch of the state boxes `state_prefetch` slices ahead, so that
      // a slot's load finds them in L2 and the slot ring turns over faster
      // than DRAM latency would let it
      auto prefetch_ahead = [&](uint32_t c) {
        const int tt = unit0 + static_cast<int>(c / T::SLICES) * units;
        if (tt >= p.num_units) return;
        const int sp = static_cast<int>(c % T::SLICES);
        int tm2, tn2;
        const int pi2 = tile_coords(tile_of(tt), p, tm2, tn2);
        const GemmProblem& q2 = p.prob[pi2];
        const int x = tn2 * BN + (sp / T::PARTS) * T::SW;
        const int y = tm2 * T::TM + static_cast<int>(rank) * kBM + (sp % T::PARTS) * T::RPS;
        if (x >= q2.d_in || y >= q2.d_out) return;
        const GemmMaps& m2 = a.maps[pi2];
        tma_prefetch_l2_2d(&m2.w, x, y);
        if constexpr (T::Q8) tma_prefetch_l2_2d(&m2.w, x + 64, y);
        const int nst2 = (MODE == kModeOpt) ? p.nstate : (MODE == kModeAccum ? 0 : 2);
        if (nst2 >= 1) tma_prefetch_l2_2d(&m2.m, x, y);
        if (nst2 >= 2) tma_prefetch_l2_2d(&m2.v, x, y);
      };
      const uint32_t pf = static_cast<uint32_t>(p.state_prefetch);
      const bool do_pf = pf > 0 && !(MODE == kModeAccum && !p.accum_load);
      if (do_pf)
        for (uint32_t c = 0; c < pf; ++c) prefetch_ahead(c);
      for (int t = unit0; ok && t < p.num_units; t += units) {
        int tm, tn;
        const int pi = tile_coords(tile_of(t), p, tm, tn);
        const GemmMaps& maps = a.maps[pi];
        const GemmProblem& pr = p.prob[pi];
        for (int s = 0; s < T::SLICES; ++s, ++cnt) {
          const int j = cnt % T::NS;
          const uint32_t ph = (cnt / T::NS) & 1u;
          if (do_pf) prefetch_ahead(cnt + pf);
          if (!wait_bounded(bar_sempty(j), ph ^ 1u, wc, kSiteLoaderEmpty)) { ok = false; break; }
          const int x0 = tn * BN + (s / T::PARTS) * T::SW;
          const int y0 = tm * T::TM + static_cast<int>(rank) * kBM + (s % T::PARTS) * T::RPS;
          last_armed[j] = static_cast<int32_t>(cnt);   // latest phase started on slot j
          if (x0 >= pr.d_in || y0 >= pr.d_out) {   // slice entirely outside the weight
            mbar_arrive(bar_sfull(j));
            continue;
          }
          if (MODE == kModeAccum && !p.accum_load) {   // beta = 0: B is not read
            mbar_arrive(bar_sfull(j));
            continue;
          }
          const uint32_t slot = base + T::OFF_SLOTS + j * T::SLOT_BYTES;
          // kModeOpt loads only the states its optimizer has; kModeAccum only B
          const int nst = (MODE == kModeOpt) ? p.nstate : (MODE == kModeAccum ? 0 : 2);
          mbar_arrive_expect_tx(bar_sfull(j), T::W_BYTES + nst * T::M_BYTES + T::ADD_BYTES);
          if constexpr (T::Q8) {
            tma_load_2d(slot, &maps.w, x0, y0, bar_sfull(j), pol);
            tma_load_2d(slot + T::RPS * 64 * 2, &maps.w, x0 + 64, y0, bar_sfull(j), pol);
          } else {
            tma_load_2d(slot, &maps.w, x0, y0, bar_sfull(j), pol);
          }
          // m, v boxes whose rows are whole 128-byte lines may be marked
          // evict-first (nothing reads them again in this launch)
          const uint64_t mpol = (T::SW * T::MOM_ELEM >= 128 && (p.l2_hints & 2)) ? pol_first : pol;
          if (nst >= 1) tma_load_2d(slot + T::W_BYTES, &maps.m, x0, y0, bar_sfull(j), mpol);
          if (nst >= 2)
            tma_load_2d(slot + T::W_BYTES + T::M_BYTES, &maps.v, x0, y0, bar_sfull(j), mpol);
          if constexpr (T::ADD_BYTES > 0)   // the accumulator's box (read, never stored)
            tma_load_2d(slot + T::W_BYTES + 2 * T::M_BYTES, &maps.b, x0, y0, bar_sfull(j), mpol);
        }
      }
      // let the loads of each slot's latest phase land before the CTA can exit
      for (int j = 0; j < T::NS; ++j)
        if (last_armed[j] >= 0)
          wait_bounded(bar_sfull(j), (static_cast<uint32_t>(last_armed[j]) / T::NS) & 1u, wc,
                       kSiteDrainState, false);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ store warp
    // Lane j TMA-stores the slices that land in state slot j and frees the
    // slot as soon as its store has read it, off the epilogue's critical
    // path; the lanes wait on their own bulk groups, so one slow store does
    // not hold back the release of the other slots.
    // (a split input-gradient launch writes only fp32 partials: no slots)
    const bool split_launch = (MODE == kModeDgrad) && p.splits > 1;
    if (lane < T::NS && !split_launch) {
      const bool hint_first = has_state(MODE) && (p.l2_hints & 1);
      const uint64_t spol = l2_policy_evict_first();
      uint32_t cnt = 0;
      bool ok = true;
      for (int t = unit0; ok && t < p.num_units; t += units) {
        int tm, tn;
        const int pi = tile_coords(tile_of(t), p, tm, tn);
        const GemmMaps& maps = a.maps[pi];
        const GemmProblem& pr = p.prob[pi];
        for (int s = 0; s < T::SLICES; ++s, ++cnt) {
          const int j = cnt % T::NS;
          if (j != lane) continue;
          const uint32_t ph = (cnt / T::NS) & 1u;
          const bool done = p.poll_store ? wait_poll(bar_sdone(j), ph, wc, kSiteStoreSlotDone)
                                         : wait_bounded(bar_sdone(j), ph, wc, kSiteStoreSlotDone);
          if (!done) { ok = false; break; }
          const int x0 = tn * BN + (s / T::PARTS) * T::SW;
          const int y0 = tm * T::TM + static_cast<int>(rank) * kBM + (s % T::PARTS) * T::RPS;
          if (x0 < pr.d_in && y0 < pr.d_out) {
            const uint32_t sl = base + T::OFF_SLOTS + j * T::SLOT_BYTES;
            // optionally evict-first: nothing reads the new state again here
            auto st2d = [&](const CUtensorMap* mp, int x, int y, uint32_t src) {
              if (hint_first) tma_store_2d_hint(mp, x, y, src, spol);
              else tma_store_2d(mp, x, y, src);
            };
            if constexpr (T::Q8) {
              st2d(&maps.w, x0, y0, sl);
              st2d(&maps.w, x0 + 64, y0, sl + T::RPS * 64 * 2);
            } else {
              st2d(&maps.w, x0, y0, sl);
            }
            if constexpr (MODE == kModeFused) {
              st2d(&maps.m, x0, y0, sl + T::W_BYTES);
              st2d(&maps.v, x0, y0, sl + T::W_BYTES + T::M_BYTES);
            } else if constexpr (MODE == kModeOpt) {
              if (p.nstate >= 1) st2d(&maps.m, x0, y0, sl + T::W_BYTES);
              if (p.nstate >= 2) st2d(&maps.v, x0, y0, sl + T::W_BYTES + T::M_BYTES);
            }
            bulk_commit_group();
            bulk_wait_group_read<0>();
          }
          mbar_arrive(bar_sempty(j));
        }
      }
      bulk_wait_group<0>();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quadrant this warp may read
    const int h = (warp - 4) >> 2;           // column half of each slice
    const uint32_t row = q * 32 + lane;      // tile row = TMEM lane
    // with half-tile slots, quadrants 0-1 take part 0 (even slots) and 2-3 part 1
    const int part = (T::PARTS == 1) ? 0 : (q >> 1);
    const uint32_t srow = (T::PARTS == 1) ? row : static_cast<uint32_t>((q & 1) * 32 + lane);
    const uint32_t bar_xch = bar_xch0 + 8u * part;
    const uint32_t bar_xch_read = bar_xch_read0 + 8u * part;
    const bool zero_grad = (p.num_k == 0);
    float* xch = reinterpret_cast<float*>(gbase + T::OFF_XCH);
    // int8: the old block scales of this thread's row are read one tile ahead,
    // so their global-memory latency is not paid at the start of each slice
    constexpr int NCB = BN / T::SW;   // 1 or 2 for int8 (slices are selected, not indexed)
    static_assert(!T::I8 || NCB <= 2, "int8 tiles hold at most two 128-column blocks");
    float sc_m[NCB], sc_v[NCB], nx_m[NCB], nx_v[NCB];
    auto load_scales = [&](int tt, float (&om)[NCB], float (&ov)[NCB]) {
#pragma unroll
      for (int cb = 0; cb < NCB; ++cb) om[cb] = ov[cb] = 0.0f;
      if (tt >= p.num_units) return;
      int tm2, tn2;
      const GemmProblem& q2 = p.prob[tile_coords(tile_of(tt), p, tm2, tn2)];
      const int y = tm2 * T::TM + static_cast<int>(rank) * kBM + part * T::RPS +
                    static_cast<int>(srow);
      if (y >= q2.d_out) return;
#pragma unroll
      for (int cb = 0; cb < NCB; ++cb) {
        const int x = tn2 * BN + cb * T::SW;
        if (x < q2.d_in) {
          const size_t idx = static_cast<size_t>(y) * (q2.d_in / 128) + (x >> 7);
          om[cb] = q2.m_scale[idx];
          ov[cb] = q2.v_scale[idx];
        }
      }
    };
    if constexpr (T::I8) load_scales(unit0, nx_m, nx_v);
    // fp8: this thread's running amaxes of the current layer's new moments,
    // raised into the layer's amax words whenever the layer changes (tiles
    // of one layer are consecutive in the queue) and at the end
    float am_m = 0.0f, am_r = 0.0f;
    int am_layer = -1;
    auto flush_amax = [&]() {
      if constexpr (T::F8) {
        if (am_layer >= 0) {
          warp_raise_amax(p.prob[am_layer].m_scale + kFp8Amax, am_m, lane);
          warp_raise_amax(p.prob[am_layer].v_scale + kFp8Amax, am_r, lane);
        }
        am_m = am_r = 0.0f;
      }
    };
    uint32_t scnt = 0, xcnt = 0;
    int it = 0;
    bool ok = true;
    for (int t = unit0; ok && t < p.num_units; t += units, ++it) {
      int tm, tn;
      const int pi = tile_coords(tile_of(t), p, tm, tn);
      const GemmProblem& pr = p.prob[pi];
      const int scale_cols = pr.d_in / 128;
      Fp8Step f8m, f8r;
      if constexpr (T::F8) {
        if (pi != am_layer) {
          flush_amax();
          am_layer = pi;
        }
        f8m = fp8_step_of(pr.m_scale);
        f8r = fp8_step_of(pr.v_scale);
      }
      if constexpr (T::I8) {
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) {
          sc_m[cb] = nx_m[cb];
          sc_v[cb] = nx_v[cb];
        }
        load_scales(t + units, nx_m, nx_v);
      }
      const int buf = it & 1;
      const uint32_t use = (it >> 1) & 1;
      bool good = wait_bounded(bar_tfull(buf), use, wc, kSiteEpiTmemFull);
      // tcgen05.ld is warp-collective: the whole warp takes the same branch
      if (!__all_sync(0xffffffffu, good)) { ok = false; break; }
      tc_fence_after_sync();
      // split input gradient: the unit writes its fp32 partial tile and frees
      // the accumulator; the reduce kernel adds the splits afterwards
      if constexpr (MODE == kModeDgrad) {
        if (p.splits > 1) {
          // partials indexed by tile row and column (not queue order)
          const size_t ctile =
              (static_cast<size_t>(pr.part_tile0) + static_cast<size_t>(tm) * pr.tiles_n + tn) * CG +
              rank;
          const size_t part_elems = static_cast<size_t>(kBM) * BN;
          float* mine = p.part + (ctile * p.splits + t % p.splits) * part_elems;
#pragma unroll 1
          for (int cb = 0; cb < BN / T::SW; ++cb)
            epi_part_write(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN +
                               cb * T::SW + h * T::HALF,
                           mine, cb, h, row);
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kPair) mbar_arrive_cluster(mapa_shared(bar_tempty(buf), 0));
            else mbar_arrive(bar_tempty(buf));
          }
          continue;
        }
      }
      for (int s = 0; s < T::SLICES; ++s, ++scnt) {
        if (T::PARTS > 1 && (s % T::PARTS) != part) continue;   // the other half's slot
        const int j = scnt % T::NS;
        const uint32_t ph = (scnt / T::NS) & 1u;
        if (has_state(MODE) || MODE == kModeAccum)
          good = wait_bounded(bar_sfull(j), ph, wc, kSiteEpiSlotFull);
        else
          good = wait_bounded(bar_sempty(j), ph ^ 1u, wc, kSiteEpiSlotFree);
        if (!__all_sync(0xffffffffu, good)) { ok = false; break; }
        const int cb = s / T::PARTS;             // column slice
        const int x0 = tn * BN + cb * T::SW;
        const int y0 = tm * T::TM + static_cast<int>(rank) * kBM + part * T::RPS;
        const bool active = x0 < pr.d_in && y0 < pr.d_out;
        uint8_t* slot = gbase + T::OFF_SLOTS + j * T::SLOT_BYTES;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN +
                               cb * T::SW + h * T::HALF;
        if constexpr (T::I8) {
          const bool row_ok = active && (y0 + static_cast<int>(srow)) < pr.d_out;
          const size_t sidx = row_ok ? static_cast<size_t>(y0 + srow) * scale_cols + (x0 >> 7) : 0;
          const uint32_t saddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + 2 * BN +
                                 static_cast<uint32_t>(h) * 128u;
          const bool xok = epi_slice_fused_i8<T::RPS, T::STASH>(
              taddr, saddr, zero_grad, row_ok, slot, xch, bar_xch, bar_xch_read, xcnt & 1u, wc,
              srow, row, h, cb == 0 ? sc_m[0] : sc_m[NCB - 1], cb == 0 ? sc_v[0] : sc_v[NCB - 1],
              pr.m_scale + sidx, pr.v_scale + sidx, p.h);
          ++xcnt;
          if (!xok) { ok = false; break; }
        } else if constexpr (T::F8) {
          if (active)
            epi_slice_fused_f8<T::RPS>(taddr, zero_grad, slot, srow, h, p.h, f8m, f8r, am_m, am_r);
        } else if (active) {
          if constexpr (MODE == kModeFused) {
            epi_slice_fused_16<FMT, T::RPS>(taddr, zero_grad, slot, srow, h, p.h, p.sr != 0,
                                            pr.sr_seed, static_cast<uint32_t>(p.sr_step),
                                            static_cast<uint32_t>(y0) + srow,
                                            static_cast<uint32_t>(x0 >> 4) + h);
          } else if constexpr (MODE == kModeOpt) {
            epi_slice_opt_any<FMT, T::RPS>(p.o, taddr, zero_grad, slot, srow, h);
          } else if constexpr (MODE == kModeAccum) {
            epi_slice_accum(taddr, zero_grad, slot, srow, h, p.accum_beta, p.accum_load != 0);
          } else {
            epi_slice_store<FMT>(taddr, zero_grad, slot, srow, h);
          }
        }
        if (s == T::SLICES - T::PARTS + part) {   // this warp has read the whole accumulator
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kPair) mbar_arrive_cluster(mapa_shared(bar_tempty(buf), 0));
            else mbar_arrive(bar_tempty(buf));
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_sdone(j));
      }
    }
    flush_amax();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before_sync();
  if constexpr (kPair) {
    // after a timeout, give copies still in flight into this CTA's shared
    // memory time to land (their completions go to the leader's barriers)
    if (*abort_flag) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 200000ull) {
      }
    }
    // neither CTA leaves while its peer may still read its shared memory or
    // arrive on its barriers
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, T::TMEM_COLS);
    else tmem_dealloc(tmem_base, T::TMEM_COLS);
  }
}

template <int MODE, int FMT, int BN, int PROF, int CG>
cudaError_t launch_gemm_t(const GemmConfig& cfg, const GemmArgs& args, cudaStream_t stream) {
  using T = GemmTraits<MODE, FMT, BN, PROF, CG>;
  auto kern = forge_gemm_kernel<MODE, FMT, BN, PROF, CG>;
  static int attr_done[64] = {0};     // per device: attributes set, pair count known
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < 64 && attr_done[dev];
  if (!cached) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t lc = {};
  lc.blockDim = dim3(kNumThreads, 1, 1);
  lc.dynamicSmemBytes = T::SMEM_ALLOC;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  int grid = cfg.grid;
  if constexpr (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int pairs = cached ? max_pairs[dev] : 0;
    if (!cached) {
      lc.gridDim = dim3(2 * 76, 1, 1);
      cudaError_t e = cudaOccupancyMaxActiveClusters(&pairs, kern, &lc);
      if (e != cudaSuccess || pairs <= 0) return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
      if (dev >= 0 && dev < 64) max_pairs[dev] = pairs;
    }
    grid = 2 * (cfg.grid / 2 < pairs ? cfg.grid / 2 : pairs);
  } else {
    lc.attrs = nullptr;
    lc.numAttrs = 0;
  }
  if (!cached && dev >= 0 && dev < 64) attr_done[dev] = 1;
  lc.gridDim = dim3(grid, 1, 1);
  return cudaLaunchKernelEx(&lc, kern, args);
}

template <int MODE, int FMT, int PROF>
cudaError_t launch_gemm_prof(const GemmConfig& cfg, const GemmArgs& args, cudaStream_t stream) {
  if (cfg.cg == 1 && cfg.bn == 128)
    return launch_gemm_t<MODE, FMT, 128, PROF, 1>(cfg, args, stream);
  // 256-wide accumulators use all 512 tensor-memory columns (two buffers).
  // Not built for 1-CTA 8-bit moments, whose 64 KB state slots do not fit
  // twice next to the wider 1-CTA operand stages.
  if constexpr (!(MODE == kModeFused && (FMT == kFmtI8 || FMT == kFmtF8))) {
    if (cfg.cg == 1 && cfg.bn == 256)
      return launch_gemm_t<MODE, FMT, 256, PROF, 1>(cfg, args, stream);
  }
  if (cfg.cg == 2 && cfg.bn == 256)
    return launch_gemm_t<MODE, FMT, 256, PROF, 2>(cfg, args, stream);
  return cudaErrorInvalidValue;
}

template <int MODE, int FMT>
cudaError_t launch_gemm_fmt(const GemmConfig& cfg, const GemmArgs& args, cudaStream_t stream) {
  switch (cfg.prof) {
    case kProfStream: return launch_gemm_prof<MODE, FMT, kProfStream>(cfg, args, stream);
    case kProfMma: return launch_gemm_prof<MODE, FMT, kProfMma>(cfg, args, stream);
    case kProfBalanced: return launch_gemm_prof<MODE, FMT, kProfBalanced>(cfg, args, stream);
    case kProfDeep:
      // 8-bit moments already use half-tile slots in the mma profile, and
      // store-G has no state slots: both run the deep profile as mma
      if constexpr (has_state(MODE) && FMT != kFmtI8 && FMT != kFmtF8)
        return launch_gemm_prof<MODE, FMT, kProfDeep>(cfg, args, stream);
      else
        return launch_gemm_prof<MODE, FMT, kProfMma>(cfg, args, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace forge
