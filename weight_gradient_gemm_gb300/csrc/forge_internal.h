// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "forge_math.cuh"

namespace forge {

// Device error word values (match forge_status).
constexpr int kErrDeviceTimeout = 9;
constexpr int kErrDeviceConfig = 11;

// Tile geometry of the tensor-core kernels.
constexpr int kBM = 128;     // weight rows per tile (MMA M)
constexpr int kBK = 64;      // tokens per pipeline stage on one CTA
constexpr int kBKPair = 64;  // tokens per pipeline stage on a CTA pair
constexpr int kNumThreads = 384;   // 4 role warps + 8 epilogue warps
constexpr int kEpiThreads = 256;

// kModeDgrad computes the layer's input gradient dX = dY W with the same
// pipeline: A = dY read K-major (rows = tokens), B = W read MN-major, the
// bf16 result stored like the gradient of kModeStoreG.
// kModeOpt is kModeFused with one of the other coordinate-wise optimizers
// (OptKind, chosen at run time) in place of AdamW: the same W, m, v slots,
// with the states the optimizer does not have left unread and unwritten.
// kModeAccum accumulates into an fp32 buffer B (B' = beta B + G): store-G
// with fp32 output whose slots are first loaded with B (unless beta = 0).
enum Mode : int { kModeFused = 0, kModeStoreG = 1, kModeDgrad = 2, kModeOpt = 3, kModeAccum = 4 };
// Modes that stream optimizer state through the state slots.
__host__ __device__ constexpr bool has_state(int mode) {
  return mode == kModeFused || mode == kModeOpt;
}
// Pipeline profiles, i.e. how shared memory is split between operand stages
// and state slots: kProfStream (small token counts, HBM-bound epilogue) keeps
// two operand stages and gives the rest to state slots; kProfMma (large token
// counts, tensor-bound main loop) keeps as many operand stages as fit next to
// two state slots; kProfBalanced keeps as many stages as slots, for the range
// where the main loop and the epilogue take about the same time; kProfDeep
// (the largest token counts) keeps as many operand stages as fit next to two
// half-tile state slots.
enum Prof : int { kProfStream = 0, kProfMma = 1, kProfBalanced = 2, kProfDeep = 3 };
// Epilogue formats: fused moment formats 0..3 (fp32, bf16, int8 blocks of
// 128, fp8 e4m3 with per-tensor scales); store-G dW formats 0..1 (fp32, bf16);
// kFmtNone: an optimizer without state (SGD), whose slots hold W alone;
// kFmtF32S1, kFmtBF16S1: an optimizer with one state (fp32 or bf16), whose
// slots hold W and that state only.  kFmtF32A, kFmtBF16A: the fused AdamW
// step with fp32 or bf16 moments whose gradient is G plus an fp32 addend
// (the accumulator of the earlier micro-batches), which each slot holds as a
// third fp32 box after m and v.
enum Fmt : int { kFmtF32 = 0, kFmtBF16 = 1, kFmtI8 = 2, kFmtF8 = 3, kFmtNone = 4,
                 kFmtF32S1 = 5, kFmtBF16S1 = 6, kFmtF32A = 7, kFmtBF16A = 8 };
// The element format of an optimizer state format (fp32 or bf16).
__host__ __device__ constexpr int state_elem_fmt(int fmt) {
  return (fmt == kFmtF32S1 || fmt == kFmtF32A) ? kFmtF32
         : (fmt == kFmtBF16S1 || fmt == kFmtBF16A) ? kFmtBF16 : fmt;
}
// Whether the format's slots carry an fp32 gradient addend.
__host__ __device__ constexpr bool has_addend(int fmt) {
  return fmt == kFmtF32A || fmt == kFmtBF16A;
}
// State boxes a slot holds.
__host__ __device__ constexpr int state_boxes(int fmt) {
  return fmt == kFmtNone ? 0 : ((fmt == kFmtF32S1 || fmt == kFmtBF16S1) ? 1 : 2);
}

// Most linear layers one launch can step (a grouped launch walks one tile
// queue across all of them).
constexpr int kMaxGroup = 8;

// One linear layer of a launch.
struct GemmProblem {
  int32_t d_in, d_out;
  int32_t tiles_m, tiles_n;
  int32_t tile_start;         // first index of this layer's tiles in the launch's queue
  int32_t num_k;              // k-steps of this layer's reduction (tokens, or d_out for dX)
  int32_t part_tile0;         // split input gradient: first partial tile of this layer
  uint64_t sr_seed;           // stochastic rounding: this layer's Philox key
  float* m_scale;             // int8: scales [d_out, d_in/128]; fp8: the moment's
  float* v_scale;             // four words (read scale, write scale, amax)
};

struct GemmParams {
  int32_t bt;                 // shared token count of every layer in the launch
  int32_t num_k;              // the largest layer's k-steps (0: no tokens, G = 0)
  int32_t nprob, num_tiles;   // layers, and tiles over all of them
  // Split reduction (input gradient only; 1 elsewhere): each tile's k-steps
  // are cut into `splits` contiguous ranges, one work unit each, so the queue
  // holds num_units = num_tiles * splits units, the splits of a tile next to
  // each other.  Every unit writes its fp32 partial tile to `part`; the
  // reduce kernel then adds the partials in split order and stores dX.
  int32_t splits, num_units;
  float* part;                // per layer from part_tile0: [tile row][tile column][CTA of
                              // the pair][split][128 x BN] fp32
  int32_t group_m;            // tile-order swizzle: rows of tiles per group
  AdamWConsts h;
  OptConsts o;                // kModeOpt: the optimizer and its step constants
  int32_t nstate;             // kModeOpt: state tensors read and written (0..2)
  float accum_beta;           // kModeAccum: beta
  int32_t accum_load;         // kModeAccum: B is read (beta != 0)
  // kModeFused: commit W by stochastic rounding (Philox4x64-10 key (the
  // layer's sr_seed, 0), counter (row, column / 16, sr_step, 0)) instead of
  // to nearest even
  int32_t sr, sr_step;
  GemmProblem prob[kMaxGroup];
  int* err;                   // device error word
  int* err_site;              // device word: where a wait first timed out
  uint64_t timeout_ns;
  int32_t drop_first_arrival;  // testing aid, see forge_debug_drop_first_arrival
  int32_t poll_store;         // store lanes poll for finished slots (see choose_config)
  // L2 hints of the state stream: bit 0, the stores of W, m, v are marked
  // evict-first; bit 1, loads of m and v boxes with whole 128-byte rows (fp32,
  // 8-bit codes) are marked evict-first
  int32_t l2_hints;
  // the state loader prefetches into L2 the boxes of the slice this many
  // slices ahead of the one it loads (0: no prefetch)
  int32_t state_prefetch;
};

struct GemmMaps {
  CUtensorMap dy, x;      // operands
  CUtensorMap w, m, v;    // fused: state; store-G: w is dW
  CUtensorMap b;          // fused with an addend: the fp32 accumulator
};

// Everything a launch reads from its parameter space (about 6.5 KB).
struct GemmArgs {
  GemmMaps maps[kMaxGroup];
  GemmParams p;
};

// Launch configuration chosen on the host.
struct GemmConfig {
  int cg;        // CTAs per tile: 1, or 2 for a CTA pair (cta_group::2, 256-row tiles)
  int bn;        // accumulator width per CTA (MMA N)
  int prof;      // pipeline profile: 0 stream (HBM-bound), 1 mma (tensor-bound)
  int grid;      // persistent CTAs (even for CTA pairs)
  int group_m;
  int poll_store;  // store lanes poll the slot-done barrier instead of suspending
  int splits;      // input gradient: k-ranges per tile (GemmParams::splits); 1 elsewhere
  int l2_hints;    // GemmParams::l2_hints
  int state_prefetch;  // GemmParams::state_prefetch
};

// Tokens per operand pipeline stage (the TMA box height of dY and X), used
// both to encode the operand descriptors and inside the kernels.
__host__ __device__ constexpr int bk_of(int cg) { return cg == 2 ? kBKPair : kBK; }

// Box widths (columns per epilogue slice) by mode/format, used both to
// encode the TMA descriptors and inside the kernels.
__host__ __device__ constexpr int slice_cols(int mode, int fmt) {
  return (mode == kModeFused && (fmt == kFmtI8 || fmt == kFmtF8)) ? 128 : 32;
}

// Rows of one state slot.  A whole 128-row tile, except in the deep profile
// and for 8-bit moments (int8, fp8) outside the stream profile: there a slot
// holds half a tile (64 rows; 8-bit 32 KB instead of 64 KB, fp32 20 KB
// instead of 40 KB),
// processed by the four epilogue warps of its two TMEM lane quadrants, which
// leaves shared memory for more operand stages.
__host__ __device__ constexpr int slot_rows(int mode, int fmt, int prof) {
  return (has_state(mode) &&
          (((fmt == kFmtI8 || fmt == kFmtF8) && prof != kProfStream) || prof == kProfDeep))
             ? 64 : 128;
}

// Launchers (one per instantiated kernel family); return a CUDA error.
cudaError_t launch_gemm(int mode, int fmt, const GemmConfig& cfg, const GemmArgs& args,
                        cudaStream_t stream);

// The input gradient's split reduction: dX[r][c] = sum over z of the fp32
// partials (in split order), rounded once to bf16.
cudaError_t launch_dgrad_reduce(const float* part, int splits, int cg, int bn, int tiles_m,
                                int tiles_n, int64_t rows, int64_t d_in, void* dX, int num_sms,
                                cudaStream_t stream);

cudaError_t launch_adamw(const void* dW, int dw_fmt, void* W, void* m, void* v, float* m_scale,
                         float* v_scale, int64_t d_in, int64_t d_out, int fmt,
                         const AdamWConsts& h, int num_sms, cudaStream_t stream);

// fp8 moments: the scale roll between steps (see forge_fp8_roll_scales).
cudaError_t launch_fp8_roll(float* words, int n, int stride, float headroom,
                            cudaStream_t stream);

}  // namespace forge
