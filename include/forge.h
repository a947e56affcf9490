/*
 * libforge: the fused weight-gradient + AdamW step of a linear layer on a
 * GB300 (sm_103a).  C ABI.
 *
 * Source of the operation: "FORGE: Fused On-Register Gradient Elimination for
 * Memory-Efficient LLM Training" (arXiv 2606.22932).
 *   - section 2.1, Eq. 3: the weight gradient of Y = X W^T is G = dY^T X;
 *   - section 2.2, Eq. 4: G is accumulated per weight tile over chunks of the
 *     token axis, in fp32;
 *   - section 2.2, Algorithm 1: AdamW is applied to each accumulator tile and
 *     only W, m and v return to memory; G is never stored;
 *   - section 1, Eq. 1 and Appendix B "INT8 states": moments stored as fp32,
 *     bf16 or blockwise-absmax int8;
 *   - the weight-error table's "FORGE fp8 states (per-tensor scale)" row and
 *     the delayed scaling described with it: moments stored as fp8 with one
 *     scale per tensor.
 *
 * Layout.  Every matrix is dense, row-major, with no padding between rows:
 *   X  [bt,    d_in ]  bf16   activations of the layer's forward pass
 *   dY [bt,    d_out]  bf16   gradient of the loss with respect to Y
 *   W  [d_out, d_in ]  bf16   weight, updated in place
 *   dW [d_out, d_in ]  fp32 or bf16 (forge_wgrad output, forge_adamw input)
 *   m, v [d_out, d_in] moments in the chosen format, updated in place
 *   int8 scales [d_out, d_in/128] fp32, one per row and 128-column block.
 *   fp8 scales: one forge_fp8_scales (four fp32 words) per moment tensor.
 *
 * Ownership.  The caller owns every buffer (device memory).  The library
 * keeps a small host-side cache of TMA descriptors keyed by pointer and
 * shape.  Only forge_dgrad (and so forge_linear_backward) uses device memory
 * of its own: when it splits the reduction (few tokens), it takes a
 * workspace for fp32 partial tiles from a stream-ordered pool the library
 * owns (one per device) and gives it back in stream order after the launch,
 * so calls on different streams never share one.  The pool keeps freed
 * memory for later calls.  The grouped input-gradient calls
 * (forge_dgrad_grouped, forge_linear_backward_grouped) take that workspace
 * from the caller instead and allocate nothing.
 *
 * Tuning.  The tile configuration is chosen from the token count and the
 * moment format (forge_describe_config shows it).  forge_set_tuning
 * overrides the choice for measurements; its initial value comes from these
 * environment variables, read once, at the library's first call that
 * chooses a configuration: FORGE_PROFILE=stream|balanced|mma|deep (how
 * shared memory is split between operand stages and state slots),
 * FORGE_CG=1|2 (one CTA or a CTA pair per tile), FORGE_BN=128|256
 * (accumulator width on one CTA), FORGE_GROUP_M=1..64 (tile rows per raster
 * group), FORGE_POLL_STORE=0|1 (the store lanes poll for finished state
 * slots), FORGE_SPLITS=1..8 (forge_dgrad: k-ranges per tile),
 * FORGE_L2_HINTS=0..3 (L2 eviction hints of the state stream),
 * FORGE_STATE_PREFETCH=0..32 (L2 prefetch distance of the state stream, in
 * slices).  Every choice
 * computes the same step to the same accuracy; only the speed differs.
 *
 * Errors.  Argument errors are returned synchronously, before anything is
 * enqueued.  Launch failures return FORGE_ERR_LAUNCH.  Kernels never trap:
 * every wait inside a kernel is bounded, and when a bound runs out the kernel
 * records FORGE_ERR_DEVICE_TIMEOUT in a per-library device word and returns;
 * forge_device_error() reads and clears it (FORGE_ERR_DEVICE_CONFIG is reported
 * the same way).
 *
 * Ordering precondition (documented, not checked).  W is overwritten in
 * place, so the layer's input gradient dX = dY W must already have been
 * computed, or enqueued earlier on the same stream, before forge_wgrad_adamw
 * or forge_adamw runs (section 2.2 and Appendix A, Remark 2).  A weight read
 * by more than one backward path (tied weights) must not use the fused call.
 */
#ifndef FORGE_H_
#define FORGE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FORGE_OK = 0,
  FORGE_ERR_NULL = 1,           /* a required pointer is NULL                         */
  FORGE_ERR_ALIGN = 2,          /* a pointer is not 16-byte aligned                   */
  FORGE_ERR_SHAPE = 3,          /* bt < 0, d_in/d_out <= 0 or not a multiple of 8,
                                   int8 moments with d_in % 128 != 0, fp8 moments
                                   with d_in % 16 != 0, or a size over the 32-bit
                                   index range of the kernels                        */
  FORGE_ERR_FORMAT = 4,         /* unknown moment format or dtype                     */
  FORGE_ERR_HYPER = 5,          /* step < 1, beta outside [0,1), lr/wd < 0 or NaN, eps neither
                                   0 nor a normal fp32 number at most 2^64 */
  FORGE_ERR_ALIAS = 6,          /* an input overlaps an output                        */
  FORGE_ERR_ARCH = 7,           /* current device is not sm_103 (no fallback exists)  */
  FORGE_ERR_LAUNCH = 8,         /* a kernel launch or TMA descriptor encode failed    */
  FORGE_ERR_DEVICE_TIMEOUT = 9, /* a bounded wait inside a kernel ran out             */
  FORGE_ERR_CUDA = 10,          /* a CUDA runtime call failed                         */
  FORGE_ERR_DEVICE_CONFIG = 11  /* a kernel found its shared-memory window unusable
                                   (not 1 KB aligned) and did no work               */
} forge_status;

typedef enum {
  FORGE_MOM_FP32 = 0,       /* k = 8 bytes of state per parameter                   */
  FORGE_MOM_BF16 = 1,       /* k = 4, round to nearest even                          */
  FORGE_MOM_INT8_B128 = 2,  /* k = 2 (+ scales): per row and 128-column block an
                               absmax scale s = a/127 and codes round(x/s) in
                               [-127,127]; the second moment is stored as
                               r = sqrt(v) with codes in [1,127] when a > 0       */
  FORGE_MOM_FP8_E4M3 = 3    /* k = 2 (+ 16 bytes per tensor): e4m3 codes (OCP
                               "fn": bias 7, largest finite 448, no infinities)
                               with one scale per tensor, delayed scaling; the
                               second moment is stored as r = sqrt(v).  Value =
                               e4m3(code) * read_scale; a new value x is stored
                               as e4m3(x * (1 / write_scale)), rounded to nearest
                               even and saturated at +-448 (see forge_fp8_scales) */
} forge_moment_fmt;

typedef enum { FORGE_DT_FP32 = 0, FORGE_DT_BF16 = 1 } forge_dtype;

/* One moment tensor.  data: fp32, bf16, int8 or e4m3 codes [d_out, d_in].
 * scale: for FORGE_MOM_INT8_B128 fp32 [d_out, d_in/128]; for
 * FORGE_MOM_FP8_E4M3 a forge_fp8_scales (cast to float*); ignored (may be
 * NULL) otherwise. */
typedef struct {
  void* data;
  float* scale;
} forge_moment;

/* The per-tensor words of an fp8 moment, in device memory, 16-byte aligned.
 * A step reads the stored codes with read_scale, writes the new codes with
 * write_scale (both > 0 and finite: they live in device memory and are not
 * checked), and raises amax to at least max |m'| (first moment) or
 * max sqrt(v') (second moment) of this step's new, unrounded moments; amax
 * is only ever raised, so the caller clears it between steps
 * (forge_fp8_roll_scales does).  The caller forms write_scale from earlier
 * steps' amaxes (delayed scaling); the first step's scales are the caller's
 * choice, since no history exists yet. */
typedef struct {
  float read_scale;
  float write_scale;
  float amax;
  float reserved;
} forge_fp8_scales;

/* A cudaStream_t passed as an opaque pointer; NULL is the legacy default stream. */
typedef void* forge_stream;

/*
 * forge_wgrad_adamw: one fused step for one linear layer (Algorithm 1).
 *   G = dY^T X (fp32 accumulation over all bt tokens inside the GPU's tensor
 *   memory, never written to global memory), then per element
 *     m' = beta1 m + (1 - beta1) G
 *     v' = beta2 v + (1 - beta2) G^2
 *     W' = (1 - lr wd) W - (lr / (1 - beta1^step)) m' / (sqrt(v' / (1 - beta2^step)) + eps)
 *   and W', m', v' are stored (W' bf16 round-to-nearest-even).  The weight update
 *   reads the unrounded m', v' of this step.
 * Arguments: X, dY device pointers (read only); W, m, v device pointers (read
 *   and written); bt >= 0 tokens (bt = 0 means G = 0); d_in, d_out > 0 and
 *   multiples of 8; step >= 1 is the 1-based count of this step.
 *   Pointers 16-byte aligned.  X and dY must not overlap W, m, v or scales.
 * Asynchronous on `stream`.
 */
forge_status forge_wgrad_adamw(const void* X, const void* dY, void* W,
                               forge_moment m, forge_moment v,
                               int64_t bt, int64_t d_in, int64_t d_out,
                               float lr, float beta1, float beta2, float eps,
                               float weight_decay, int64_t step,
                               forge_moment_fmt fmt, forge_stream stream);

/* Most layers one grouped call can step. */
#define FORGE_MAX_GROUP 8

/* One linear layer of a grouped call; the fields have the meaning of the
 * same-named arguments of forge_wgrad_adamw. */
typedef struct {
  const void* X;        /* [bt, d_in]  bf16, read only (may be shared by layers) */
  const void* dY;       /* [bt, d_out] bf16, read only                           */
  void* W;              /* [d_out, d_in] bf16, updated in place                  */
  forge_moment m, v;    /* moments (and int8 scales), updated in place           */
  int64_t d_in, d_out;
} forge_linear;

/*
 * forge_wgrad_adamw_sr: forge_wgrad_adamw with the new bf16 weight committed
 * by stochastic rounding (the page's SR-store recipe, after Gupta et al.:
 * no fp32 master copy; the weight rounds up with probability equal to the
 * dropped fraction, so its expected value is the fp32 update).  The update is
 * rounded to fp32 first.  The random bits come from Philox4x64-10 (Salmon
 * et al. 2011) with key (seed, 0): weight (p, q) at step t takes bits
 * 16 j .. 16 j + 15 of word k of the block with counter (p, q / 16, t, 0),
 * where q % 16 = 4 k + j.  Give each layer its own seed.  The moments round
 * to nearest as in forge_wgrad_adamw.  fp32 or bf16 moments (int8:
 * FORGE_ERR_FORMAT); step <= 2^31 - 1.  Otherwise the arguments and errors of
 * forge_wgrad_adamw.  Asynchronous on `stream`.
 */
forge_status forge_wgrad_adamw_sr(const void* X, const void* dY, void* W, forge_moment m,
                                  forge_moment v, int64_t bt, int64_t d_in, int64_t d_out,
                                  float lr, float beta1, float beta2, float eps,
                                  float weight_decay, int64_t step, forge_moment_fmt fmt,
                                  uint64_t seed, forge_stream stream);

/*
 * forge_wgrad_adamw_grouped: forge_wgrad_adamw on n (1..FORGE_MAX_GROUP)
 * independent linear layers with the same token count bt, hyperparameters,
 * step and moment format, in ONE kernel launch whose persistent CTAs walk a
 * single tile queue over all layers (largest first).  Results are those of n
 * separate forge_wgrad_adamw calls, bit for bit.  Inputs may be shared between
 * layers (e.g. the q, k, v projections read the same X); no layer's W, m, v or
 * scales may overlap any layer's inputs or outputs (FORGE_ERR_ALIAS).
 * FORGE_ERR_NULL if `layers` is NULL, FORGE_ERR_SHAPE if n is out of range;
 * otherwise the errors of forge_wgrad_adamw.  Asynchronous on `stream`.
 */
forge_status forge_wgrad_adamw_grouped(const forge_linear* layers, int n, int64_t bt,
                                       float lr, float beta1, float beta2, float eps,
                                       float weight_decay, int64_t step,
                                       forge_moment_fmt fmt, forge_stream stream);

/*
 * The other coordinate-wise optimizers FORGE fuses: the families the page
 * lists as entering their state one coordinate at a time (section 1; the
 * definition of a tile-local state update, section 2; the appendix table of
 * optimizer families, regime 1).  The page checks each against a reference
 * PyTorch implementation; these are torch.optim's definitions with default
 * options, and Chen et al.'s for Lion.  With G the accumulator tile and
 * g = G + weight_decay * W (L2 decay, the pre-update W):
 *   SGD           W -= lr g                                          no state
 *   SGD_MOMENTUM  b = momentum b + g;  W -= lr b                     s1 = b
 *   ADAGRAD       s += g^2;  W -= lr g / (sqrt(s) + eps)             s1 = s
 *   RMSPROP       s = alpha s + (1 - alpha) g^2;
 *                 W -= lr g / (sqrt(s) + eps)                        s1 = s
 *   LION          c = beta1 m + (1 - beta1) G;
 *                 W = (1 - lr weight_decay) W - lr sign(c)  (decoupled decay);
 *                 m = beta2 m + (1 - beta2) G                        s1 = m
 *   NADAM         torch.optim.NAdam: m, v moving averages of g, g^2;
 *                 mu_i = beta1 (1 - 0.5 * 0.96^(i momentum_decay)), P_t = prod_{i<=t} mu_i;
 *                 W -= lr [(1 - mu_t)/(1 - P_t) g + mu_{t+1}/(1 - P_t mu_{t+1}) m]
 *                      / (sqrt(v / (1 - beta2^t)) + eps)             s1 = m, s2 = v
 *   RADAM         torch.optim.RAdam: m, v as NAdam; with rho_t > 5,
 *                 W -= lr r_t sqrt(1 - beta2^t) m / ((1 - beta1^t)(sqrt(v) + eps)),
 *                 else W -= lr m / (1 - beta1^t)                     s1 = m, s2 = v
 * States start at zero.  Every stored value is rounded once to nearest even.
 */
typedef enum {
  FORGE_OPT_SGD = 0,
  FORGE_OPT_SGD_MOMENTUM = 1,
  FORGE_OPT_ADAGRAD = 2,
  FORGE_OPT_RMSPROP = 3,
  FORGE_OPT_LION = 4,
  FORGE_OPT_NADAM = 5,
  FORGE_OPT_RADAM = 6
} forge_optimizer;

/* Hyperparameters of forge_wgrad_opt; an optimizer reads only its own. */
typedef struct {
  float lr, weight_decay;   /* all; >= 0 and finite                                 */
  float beta1, beta2;       /* LION, NADAM, RADAM; in [0, 1)                        */
  float eps;                /* ADAGRAD, RMSPROP, NADAM, RADAM: 0, or a normal fp32
                               number at most 2^64 (FORGE_ERR_HYPER otherwise)    */
  float momentum;           /* SGD_MOMENTUM; in [0, 1)                              */
  float alpha;              /* RMSPROP; in [0, 1)                                   */
  float momentum_decay;     /* NADAM (torch's psi, 0.004 by default); >= 0, finite  */
} forge_opt_hyper;

/*
 * forge_wgrad_opt: the fused step of forge_wgrad_adamw with optimizer `opt`
 * in place of AdamW: G = dY^T X accumulated on chip, the update applied in
 * the epilogue, only W and the optimizer's states written back.
 *   s1, s2  the optimizer's states (see the table above), fmt FORGE_MOM_FP32
 *           or FORGE_MOM_BF16, [d_out, d_in], updated in place; the `scale`
 *           fields are unused, and so are states the optimizer does not have
 *           (they may be NULL).
 * Errors: FORGE_ERR_HYPER for an unknown optimizer, a NULL `hyper`, step < 1
 * or a hyperparameter out of range; FORGE_ERR_FORMAT for int8 states; the
 * shape, NULL, alignment and overlap errors of forge_wgrad_adamw.
 * Asynchronous on `stream`; the ordering precondition on dX applies.
 */
forge_status forge_wgrad_opt(const void* X, const void* dY, void* W, forge_moment s1,
                             forge_moment s2, int64_t bt, int64_t d_in, int64_t d_out,
                             forge_optimizer opt, const forge_opt_hyper* hyper, int64_t step,
                             forge_moment_fmt fmt, forge_stream stream);

/*
 * forge_wgrad_opt_grouped: forge_wgrad_opt on n (1..FORGE_MAX_GROUP) linear
 * layers with one token count, optimizer, hyperparameters, step and state
 * format, in one launch (one tile queue over all layers, largest first).
 * Each layer's m and v fields are its s1 and s2 (scale fields unused).
 * Results are those of n separate calls, bit for bit.  Errors as
 * forge_wgrad_opt, plus those of forge_wgrad_adamw_grouped's layer checks.
 */
forge_status forge_wgrad_opt_grouped(const forge_linear* layers, int n, int64_t bt,
                                     forge_optimizer opt, const forge_opt_hyper* hyper,
                                     int64_t step, forge_moment_fmt fmt, forge_stream stream);

/*
 * forge_wgrad_adamw_sr_grouped: forge_wgrad_adamw_sr on n layers in one
 * launch; layer i draws its random bits with key (seeds[i], 0).  Results are
 * those of n separate calls with those seeds, bit for bit.
 */
forge_status forge_wgrad_adamw_sr_grouped(const forge_linear* layers, const uint64_t* seeds,
                                          int n, int64_t bt, float lr, float beta1, float beta2,
                                          float eps, float weight_decay, int64_t step,
                                          forge_moment_fmt fmt, forge_stream stream);

/*
 * forge_wgrad_accumulate: B = beta * B + dY^T X into an fp32 buffer, the
 * gradient accumulated on chip and added to B in the epilogue, rounded once
 * per call.  The FORGE page uses it twice: Muon's momentum B <- mu B + G
 * accumulates through the GEMM's beta (its optimizer regimes, regime 2), and
 * the exact-accumulation mode (Appendix N.5) keeps an fp32 gradient-shaped
 * accumulator across micro-batches (beta = 0 for the first, 1 for the
 * others) and steps once at the last one: forge_adamw then reads B as its
 * fp32 gradient.
 *   X [bt, d_in], dY [bt, d_out] bf16; B [d_out, d_in] fp32, updated in
 *   place (16-byte aligned).  beta = 0 does not read B (it may hold anything).
 * Errors: FORGE_ERR_HYPER for a non-finite beta; the shape, NULL, alignment
 * and overlap (B over X or dY) errors of forge_wgrad.  bt = 0 scales B by
 * beta.  Asynchronous on `stream`.
 */
forge_status forge_wgrad_accumulate(const void* X, const void* dY, float* B, float beta,
                                    int64_t bt, int64_t d_in, int64_t d_out,
                                    forge_stream stream);

/* One linear layer of forge_wgrad_accumulate_grouped; fields as the
 * same-named arguments of forge_wgrad_accumulate. */
typedef struct {
  const void* X;   /* [bt, d_in] bf16, read only (may be shared)     */
  const void* dY;  /* [bt, d_out] bf16, read only                    */
  float* B;        /* [d_out, d_in] fp32, updated in place           */
  int64_t d_in, d_out;
} forge_accum_item;

/* forge_wgrad_accumulate on n (1..FORGE_MAX_GROUP) layers with one token
 * count and beta, in one launch; no B may overlap an input or another B. */
forge_status forge_wgrad_accumulate_grouped(const forge_accum_item* items, int n, int64_t bt,
                                            float beta, forge_stream stream);

/*
 * forge_wgrad_adamw_acc: the step at the final micro-batch of the
 * exact-accumulation mode (the FORGE page, Appendix N.5) in one launch.  The
 * gradient the AdamW step reads is fp32(B + dY^T X): B holds the earlier
 * micro-batches' sum (forge_wgrad_accumulate), the last micro-batch's tile is
 * added to it on chip, and W, m, v are updated as forge_wgrad_adamw updates
 * them.  The result equals forge_wgrad_accumulate(beta = 1) followed by
 * forge_adamw on B, bit for bit, without writing B back or reading it twice.
 *   Arguments as forge_wgrad_adamw; B [d_out, d_in] fp32, 16-byte aligned,
 *   read only (the caller clears or reuses it for the next step).
 *   fmt: FORGE_MOM_FP32 or FORGE_MOM_BF16.
 * Errors: as forge_wgrad_adamw; FORGE_ERR_FORMAT for other moment formats;
 * FORGE_ERR_ALIAS if B overlaps W, m or v.  bt = 0 steps on B alone.
 * Asynchronous on `stream`.
 */
forge_status forge_wgrad_adamw_acc(const void* X, const void* dY, void* W, forge_moment m,
                                   forge_moment v, const float* B, int64_t bt, int64_t d_in,
                                   int64_t d_out, float lr, float beta1, float beta2, float eps,
                                   float weight_decay, int64_t step, forge_moment_fmt fmt,
                                   forge_stream stream);
/* forge_wgrad_adamw_acc on n (1..FORGE_MAX_GROUP) layers in one launch;
 * B[i] is layer i's accumulator.  No B may overlap any layer's W, m or v. */
forge_status forge_wgrad_adamw_acc_grouped(const forge_linear* layers, const float* const* B,
                                           int n, int64_t bt, float lr, float beta1, float beta2,
                                           float eps, float weight_decay, int64_t step,
                                           forge_moment_fmt fmt, forge_stream stream);

/*
 * forge_wgrad: the unfused gradient, dW = dY^T X stored to global memory
 * (the "store-G control" of the FORGE page's Appendix D).  It runs the same
 * tensor-core main loop as forge_wgrad_adamw, so with dw_dtype = FORGE_DT_FP32
 * it produces bit for bit the accumulator the fused call consumes.
 * dw_dtype FORGE_DT_BF16 rounds dW to bf16 (the standard bf16 pipeline).
 * dW must not overlap X or dY.  bt = 0 writes zeros.  Asynchronous on `stream`.
 */
forge_status forge_wgrad(const void* X, const void* dY, void* dW, forge_dtype dw_dtype,
                         int64_t bt, int64_t d_in, int64_t d_out, forge_stream stream);

/*
 * forge_dgrad: the layer's input gradient dX = dY W (the other half of the
 * backward pass of Y = X W^T, section 2.1), bf16 in, fp32 accumulation over
 * d_out, bf16 out (rounded to nearest even).
 *   dY [bt, d_out] bf16, W [d_out, d_in] bf16 (read only), dX [bt, d_in] bf16
 *   (written).  Row-major, 16-byte aligned, d_in and d_out multiples of 8.
 * dX must not overlap dY or W.  bt = 0 does nothing.  Asynchronous on
 * `stream`; argument errors are returned before anything is enqueued.
 * With few tiles (few tokens) the reduction over d_out is split into up to 8
 * k-ranges whose fp32 partials are added in a fixed order, so the result is
 * the same on every run; the partials live in a workspace from the library's
 * pool (see Ownership), and if that memory cannot be had the launch runs
 * unsplit.
 */
forge_status forge_dgrad(const void* dY, const void* W, void* dX,
                         int64_t bt, int64_t d_in, int64_t d_out, forge_stream stream);

/* One projection of a grouped input-gradient call. */
typedef struct {
  const void* dY;  /* [bt, d_out] bf16, read only                   */
  const void* W;   /* [d_out, d_in] bf16, read only                 */
  void* dX;        /* [bt, d_in] bf16, written                       */
  int64_t d_in, d_out;
} forge_dgrad_item;

/*
 * forge_dgrad_grouped: forge_dgrad for n (1..FORGE_MAX_GROUP) projections
 * with one token count in one launch: one tile queue over all of them, the
 * projections with the most work first (their reductions over d_out differ
 * in length).  When the launch splits the reductions (few tiles), the fp32
 * partials go to the caller's `workspace` (device, 16-byte aligned,
 * `workspace_bytes` long; forge_dgrad_workspace_bytes gives the size the
 * library's choice needs); with less, or NULL, it splits less or not at all
 * (same accuracy).  Nothing is allocated.  With the same split count each
 * dX is bit for bit that of forge_dgrad.  The workspace must not be used by
 * another call until this one has run.  Errors as forge_dgrad; no dX may
 * overlap any projection's dY, W or another dX (FORGE_ERR_ALIAS).
 */
forge_status forge_dgrad_grouped(const forge_dgrad_item* items, int n, int64_t bt,
                                 void* workspace, size_t workspace_bytes, forge_stream stream);

/* Bytes of workspace forge_dgrad_grouped wants for these projections (0 if
 * it would not split, or for invalid arguments). */
size_t forge_dgrad_workspace_bytes(const forge_dgrad_item* items, int n, int64_t bt);

/*
 * forge_dgrad_noalloc: forge_dgrad that allocates nothing, for callers that
 * cannot allocate device memory while they run: an engine that plans and
 * owns every byte of the device up front, or code that runs where an
 * allocation call is not allowed.  When it splits the reduction, the fp32 partials go to a
 * 32 MiB scratch array that lives in the library's own module (a file-scope
 * device array) instead of the pool; a split that needs more runs with
 * fewer splits (down to none).  With the same split count the result is bit
 * for bit that of forge_dgrad.  Same arguments, layout and errors as
 * forge_dgrad.
 * When the scratch is reserved: under CUDA's default lazy module loading the
 * array (and the kernels' code) is placed on a device at the first libforge
 * call there that needs it, not when the library is loaded; a caller that
 * needs even the first forge_dgrad_noalloc call on a device to take no
 * device memory makes one warm-up call (any libforge call that launches on
 * that device) beforehand.  Every GPU that loads the module holds the 32 MiB
 * until the process exits.
 * Precondition (documented, not checked): the scratch is one per device, so
 * two forge_dgrad_noalloc calls on one device must not run at the same time
 * (issue them on one stream, or order the streams); forge_dgrad calls may
 * run beside them.
 */
forge_status forge_dgrad_noalloc(const void* dY, const void* W, void* dX, int64_t bt,
                                 int64_t d_in, int64_t d_out, forge_stream stream);

/*
 * forge_linear_backward: the layer's whole backward step with the fused
 * update: dX = dY W from the weight before the update (Algorithm 1 computes
 * the input gradient first; Appendix A, Remark 2), then forge_wgrad_adamw.
 * Both run on `stream` in that order, so the caller no longer has to order
 * dX before the update.  Arguments as forge_dgrad and forge_wgrad_adamw;
 * dX [bt, d_in] bf16 must not overlap X, dY, W, m, v or the scales.  Every
 * argument of both halves is checked before anything is enqueued.
 */
forge_status forge_linear_backward(const void* X, const void* dY, void* W, void* dX,
                                   forge_moment m, forge_moment v,
                                   int64_t bt, int64_t d_in, int64_t d_out,
                                   float lr, float beta1, float beta2, float eps,
                                   float weight_decay, int64_t step,
                                   forge_moment_fmt fmt, forge_stream stream);

/*
 * forge_linear_backward_grouped: forge_linear_backward for n layers with one
 * token count: one grouped input-gradient launch (dX[i] = dY_i W_i from the
 * weights before the update; split partials in the caller's workspace, as
 * forge_dgrad_grouped), then forge_wgrad_adamw_grouped, both on `stream`.
 * dX[i] [bt, d_in_i] bf16 must not overlap any layer's X, dY, W, m, v,
 * scales or another dX.  Every argument of both halves is checked before
 * anything is enqueued.  Nothing is allocated.
 */
forge_status forge_linear_backward_grouped(const forge_linear* layers, void* const* dX, int n,
                                           int64_t bt, float lr, float beta1, float beta2,
                                           float eps, float weight_decay, int64_t step,
                                           forge_moment_fmt fmt, void* workspace,
                                           size_t workspace_bytes, forge_stream stream);

/*
 * forge_adamw: the unfused optimizer step on a stored gradient dW (fp32 or
 * bf16), with exactly the per-element arithmetic of forge_wgrad_adamw.
 * forge_wgrad(FP32) followed by forge_adamw gives the same bits as
 * forge_wgrad_adamw (Appendix A, "Floating-point characterization").
 * dW may be NULL, which means a zero gradient.  dW must not overlap W, m, v.
 */
forge_status forge_adamw(const void* dW, forge_dtype dw_dtype, void* W,
                         forge_moment m, forge_moment v,
                         int64_t d_in, int64_t d_out,
                         float lr, float beta1, float beta2, float eps,
                         float weight_decay, int64_t step,
                         forge_moment_fmt fmt, forge_stream stream);

/*
 * forge_fp8_roll_scales: the scale roll between two steps of fp8 moments,
 * for n tensors' forge_fp8_scales (a device array, consecutive): read_scale
 * <- write_scale (the codes were just written with it); write_scale <-
 * amax * headroom / 448 in fp32 (product rounded, then quotient), or
 * unchanged when amax is 0; amax <- 0.  headroom >= 1 leaves room for the
 * moments to grow by that factor before they saturate.  One small kernel on
 * `stream`, so the whole delayed-scaling loop stays on the device.
 * Errors: FORGE_ERR_SHAPE for n < 0, FORGE_ERR_NULL, FORGE_ERR_ALIGN,
 * FORGE_ERR_HYPER for headroom < 1 or not finite.
 */
forge_status forge_fp8_roll_scales(forge_fp8_scales* scales, int n, float headroom,
                                   forge_stream stream);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device: FORGE_OK, FORGE_ERR_DEVICE_TIMEOUT if a kernel gave up on a
 * bounded wait since the last call, or FORGE_ERR_DEVICE_CONFIG.  FORGE_ERR_CUDA
 * if the sync failed. */
forge_status forge_device_error(forge_stream stream);

/* A static, human-readable name for a status code. */
const char* forge_status_string(forge_status status);

/* The tile configuration the fused kernel would use for a shape, written as
 * text into buf (at most len bytes, always NUL-terminated).  Returns the
 * number of bytes needed, or -1 for an invalid shape or format. */
int forge_describe_config(int64_t bt, int64_t d_in, int64_t d_out,
                          forge_moment_fmt fmt, char* buf, int len);

/* The same for forge_dgrad on a [bt, d_out] x [d_out, d_in] problem: tile,
 * CTA grouping, profile, grid and the number of k-ranges the reduction over
 * d_out is split into.  Returns the bytes needed, or -1 for an invalid shape. */
int forge_describe_dgrad_config(int64_t bt, int64_t d_in, int64_t d_out, char* buf, int len);

/* Diagnostics for FORGE_ERR_DEVICE_TIMEOUT: where the first timed-out wait
 * since the last call happened, as site*100000 + block*100 (site 1 operand
 * slot free, 2 accumulator free, 3 operands landed, 4 state slot free,
 * 5 accumulator ready, 6 state landed, 7 output slot free, 8-10 teardown
 * drains), or 0 if none; -1 if the device cannot be queried.  Reading clears
 * it.  Call after forge_device_error() has synchronised. */
int forge_debug_timeout_site(void);

/* Bounded-wait limit for the kernels' internal waits, in nanoseconds
 * (default 2e9).  Applies to launches made after the call. */
void forge_set_wait_limit_ns(uint64_t ns);

/* Testing aid for the timeout path: when enabled, the next fused or forge_wgrad
 * launch skips its first operand-load arrival, so its waits run out, the kernel
 * records FORGE_ERR_DEVICE_TIMEOUT and returns with its outputs unspecified.
 * The flag clears itself after that one launch. */
void forge_debug_drop_first_arrival(int enable);

/* Pipeline profiles: how a tensor-core kernel splits shared memory between
 * operand stages and optimizer-state slots. */
typedef enum {
  FORGE_PROFILE_AUTO = -1,     /* chosen from the token count and format       */
  FORGE_PROFILE_STREAM = 0,    /* two operand stages, the rest state slots      */
  FORGE_PROFILE_MMA = 1,       /* as many operand stages as fit beside 2 slots  */
  FORGE_PROFILE_BALANCED = 2,  /* as many operand stages as state slots         */
  FORGE_PROFILE_DEEP = 3       /* as many stages as fit beside 2 half-tile slots */
} forge_profile;

/* Tuning overrides; a field at its automatic value (FORGE_PROFILE_AUTO, 0 or
 * -1 as stated) leaves that choice to the library.  Out-of-range values are
 * ignored. */
typedef struct {
  int profile;     /* a forge_profile                                          */
  int cta_group;   /* 0 automatic; 1 one CTA per tile; 2 a CTA pair (256 x 256) */
  int bn;          /* 0 automatic; 128 or 256: accumulator width on one CTA     */
  int group_m;     /* 0 automatic; 1..64 tile rows per raster group             */
  int poll_store;  /* -1 automatic; 0 or 1: store lanes poll for finished slots */
  int splits;      /* 0 automatic; 1..8 k-ranges per tile for forge_dgrad       */
  int l2_hints;    /* -1 automatic; 0..3: bit 0 marks the optimizer state's
                      stores evict-first in L2, bit 1 its m, v loads whose rows
                      are whole 128-byte lines                                  */
  int state_prefetch; /* -1 automatic; 0..32: the state loader prefetches into L2
                         the boxes this many state slices ahead (0: none)         */
} forge_tuning;

/* Replace the tuning overrides (NULL: everything automatic).  Applies to
 * calls made after it returns, from any thread; thread-safe.  Every setting
 * computes the same results; only the speed differs. */
void forge_set_tuning(const forge_tuning* tuning);

/* The tuning overrides now in force (the environment's, until the first
 * forge_set_tuning). */
void forge_get_tuning(forge_tuning* tuning);

#ifdef __cplusplus
}
#endif

#endif /* FORGE_H_ */
