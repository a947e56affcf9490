// The C ABI of libforge: argument validation, TMA descriptor encoding (cached),
// tile configuration, launches and the device error word.
#include <algorithm>
#include <cstdint>
#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/forge.h"
#include "forge_internal.h"

// Scratch of forge_dgrad_noalloc: the fp32 split partials of one call, in
// static device memory the library reserves on each device when its module
// loads, so that the call itself allocates nothing.  32 MiB holds the
// partials of the Llama-3.1-8B projections at 512 tokens with up to 4
// splits; a split that needs more runs with fewer splits.
constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;
static __device__ __align__(256) float g_dgrad_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace forge {

cudaError_t launch_gemm_fused_f32(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_fused_bf16(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_fused_i8(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_fused_f8(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_store_f32(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_store_bf16(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_dgrad(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_opt_f32(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_opt_bf16(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_opt_none(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_opt_f32s1(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_opt_bf16s1(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_fused_f32a(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_fused_bf16a(const GemmConfig&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_accum(const GemmConfig&, const GemmArgs&, cudaStream_t);

cudaError_t launch_gemm(int mode, int fmt, const GemmConfig& cfg, const GemmArgs& args,
                        cudaStream_t stream) {
  if (mode == kModeFused) {
    switch (fmt) {
      case kFmtF32: return launch_gemm_fused_f32(cfg, args, stream);
      case kFmtBF16: return launch_gemm_fused_bf16(cfg, args, stream);
      case kFmtI8: return launch_gemm_fused_i8(cfg, args, stream);
      case kFmtF8: return launch_gemm_fused_f8(cfg, args, stream);
      case kFmtF32A: return launch_gemm_fused_f32a(cfg, args, stream);
      case kFmtBF16A: return launch_gemm_fused_bf16a(cfg, args, stream);
    }
  } else if (mode == kModeStoreG) {
    switch (fmt) {
      case kFmtF32: return launch_gemm_store_f32(cfg, args, stream);
      case kFmtBF16: return launch_gemm_store_bf16(cfg, args, stream);
    }
  } else if (mode == kModeDgrad && fmt == kFmtBF16) {
    return launch_gemm_dgrad(cfg, args, stream);
  } else if (mode == kModeAccum && fmt == kFmtF32) {
    return launch_gemm_accum(cfg, args, stream);
  } else if (mode == kModeOpt) {
    switch (fmt) {
      case kFmtF32: return launch_gemm_opt_f32(cfg, args, stream);
      case kFmtBF16: return launch_gemm_opt_bf16(cfg, args, stream);
      case kFmtNone: return launch_gemm_opt_none(cfg, args, stream);
      case kFmtF32S1: return launch_gemm_opt_f32s1(cfg, args, stream);
      case kFmtBF16S1: return launch_gemm_opt_bf16s1(cfg, args, stream);
    }
  }
  return cudaErrorInvalidValue;
}

// One error word per device; a kernel that gives up on a bounded wait writes
// FORGE_ERR_DEVICE_TIMEOUT here.
__device__ int g_forge_device_error;
// Where the first timeout since the last read happened (diagnostics).
__device__ int g_forge_device_error_site;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int cc_major = 0, cc_minor = 0, num_sms = 0;
  int* err_word = nullptr;
  int* site_word = nullptr;
  // stream-ordered pool for launch workspaces (the input gradient's split
  // partials); it keeps freed memory for the next call instead of returning it
  cudaMemPool_t pool = nullptr;
  float* scratch = nullptr;   // this device's g_dgrad_scratch
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
uint64_t g_wait_limit_ns = 2000000000ull;
int g_drop_first_arrival = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Cache of encoded descriptors keyed by everything that goes into them (a
// whole model's linears fit; it is cleared if it ever grows past kCacheMax).
struct MapKey {
  const void* ptr;
  int dtype;
  uint64_t inner, outer, stride;
  uint32_t box_inner, box_outer;
  int swizzle;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && dtype == o.dtype && inner == o.inner && outer == o.outer &&
           stride == o.stride && box_inner == o.box_inner && box_outer == o.box_outer &&
           swizzle == o.swizzle;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = reinterpret_cast<uintptr_t>(k.ptr) * 0x9E3779B97F4A7C15ull;
    for (uint64_t v : {static_cast<uint64_t>(k.dtype), k.inner, k.outer, k.stride,
                       static_cast<uint64_t>(k.box_inner) << 32 | k.box_outer,
                       static_cast<uint64_t>(k.swizzle)})
      h = (h ^ v) * 0x100000001B3ull;
    return static_cast<size_t>(h);
  }
};
constexpr size_t kCacheMax = 8192;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_cache;

forge_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FORGE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FORGE_ERR_CUDA;
    if (d.cc_major != 10 || d.cc_minor != 3) return FORGE_ERR_ARCH;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_forge_device_error) != cudaSuccess) return FORGE_ERR_CUDA;
    d.err_word = static_cast<int*>(addr);
    if (cudaGetSymbolAddress(&addr, g_forge_device_error_site) != cudaSuccess) return FORGE_ERR_CUDA;
    d.site_word = static_cast<int*>(addr);
    if (cudaGetSymbolAddress(&addr, g_dgrad_scratch) != cudaSuccess) return FORGE_ERR_CUDA;
    d.scratch = static_cast<float*>(addr);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FORGE_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return FORGE_OK;
}

// The device's workspace pool, created on first use.
cudaMemPool_t workspace_pool(DeviceInfo& d) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!d.pool) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = UINT64_MAX;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    d.pool = pool;
  }
  return d.pool;
}

// Encode (or fetch from the cache) a 2-D row-major tensor map.
bool get_map(CUtensorMap* out, const void* ptr, CUtensorMapDataType dt, uint64_t inner,
             uint64_t outer, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer,
             CUtensorMapSwizzle sw) {
  MapKey key{ptr, static_cast<int>(dt), inner, outer, stride_bytes, box_inner, box_outer,
             static_cast<int>(sw)};
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_cache.find(key);
  if (it != g_cache.end()) {
    *out = it->second;
    return true;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  CUresult r = g_encode(&m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (g_cache.size() >= kCacheMax) g_cache.clear();
  g_cache.emplace(key, m);
  *out = m;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

int mom_elem_bytes(forge_moment_fmt f) {
  return f == FORGE_MOM_FP32 ? 4 : (f == FORGE_MOM_BF16 ? 2 : 1);
}

bool valid_fmt(forge_moment_fmt f) {
  return f == FORGE_MOM_FP32 || f == FORGE_MOM_BF16 || f == FORGE_MOM_INT8_B128 ||
         f == FORGE_MOM_FP8_E4M3;
}

// Bytes of one moment's scale storage: int8 one fp32 per row and 128-column
// block; fp8 the four words of forge_fp8_scales.
uint64_t scale_bytes(forge_moment_fmt f, uint64_t n) {
  return f == FORGE_MOM_INT8_B128 ? n / 128 * 4
                                  : (f == FORGE_MOM_FP8_E4M3 ? sizeof(forge_fp8_scales) : 0);
}

forge_status check_shape(int64_t bt, int64_t d_in, int64_t d_out) {
  const int64_t lim = (1LL << 31) - 1;
  if (bt < 0 || d_in <= 0 || d_out <= 0) return FORGE_ERR_SHAPE;
  if (bt > lim || d_in > lim || d_out > lim) return FORGE_ERR_SHAPE;
  if (d_in % 8 != 0 || d_out % 8 != 0) return FORGE_ERR_SHAPE;
  return FORGE_OK;
}

// eps is 0 or a normal fp32 number at most 2^64: the kernels' reciprocal of
// the AdamW-style denominator flushes subnormals, which then never occur.
bool eps_ok(float eps) { return eps == 0.0f || (eps >= FLT_MIN && eps <= 0x1p64f); }

forge_status check_hyper(float lr, float b1, float b2, float eps, float wd, int64_t step) {
  if (step < 1) return FORGE_ERR_HYPER;
  if (!(b1 >= 0.0f && b1 < 1.0f) || !(b2 >= 0.0f && b2 < 1.0f)) return FORGE_ERR_HYPER;
  if (!(lr >= 0.0f) || !(wd >= 0.0f) || !eps_ok(eps)) return FORGE_ERR_HYPER;
  if (!std::isfinite(lr) || !std::isfinite(wd)) return FORGE_ERR_HYPER;
  return FORGE_OK;
}

// Validation shared by the fused call and forge_adamw (state side).
forge_status check_state(void* W, const forge_moment& m, const forge_moment& v, int64_t d_in,
                         int64_t d_out, forge_moment_fmt fmt) {
  if (!valid_fmt(fmt)) return FORGE_ERR_FORMAT;
  if (!W || !m.data || !v.data) return FORGE_ERR_NULL;
  if (fmt == FORGE_MOM_INT8_B128 || fmt == FORGE_MOM_FP8_E4M3) {
    if (!m.scale || !v.scale) return FORGE_ERR_NULL;
    // int8: whole 128-column blocks; fp8: rows of codes 16-byte aligned (TMA strides)
    if (d_in % (fmt == FORGE_MOM_INT8_B128 ? 128 : 16) != 0) return FORGE_ERR_SHAPE;
    if (!aligned16(m.scale) || !aligned16(v.scale)) return FORGE_ERR_ALIGN;
  }
  if (!aligned16(W) || !aligned16(m.data) || !aligned16(v.data)) return FORGE_ERR_ALIGN;
  const uint64_t n = static_cast<uint64_t>(d_in) * static_cast<uint64_t>(d_out);
  const uint64_t nm = n * mom_elem_bytes(fmt);
  const uint64_t ns = scale_bytes(fmt, n);
  // the three (five) state tensors must be distinct
  if (overlaps(W, 2 * n, m.data, nm) || overlaps(W, 2 * n, v.data, nm) ||
      overlaps(m.data, nm, v.data, nm))
    return FORGE_ERR_ALIAS;
  if (ns && (overlaps(m.scale, ns, v.scale, ns) || overlaps(m.scale, ns, W, 2 * n) ||
             overlaps(v.scale, ns, W, 2 * n) || overlaps(m.scale, ns, m.data, nm) ||
             overlaps(m.scale, ns, v.data, nm) || overlaps(v.scale, ns, m.data, nm) ||
             overlaps(v.scale, ns, v.data, nm)))
    return FORGE_ERR_ALIAS;
  return FORGE_OK;
}

bool input_overlaps_state(const void* in, uint64_t nin, void* W, const forge_moment& m,
                          const forge_moment& v, int64_t d_in, int64_t d_out,
                          forge_moment_fmt fmt) {
  const uint64_t n = static_cast<uint64_t>(d_in) * static_cast<uint64_t>(d_out);
  const uint64_t nm = n * mom_elem_bytes(fmt);
  const uint64_t ns = scale_bytes(fmt, n);
  return overlaps(in, nin, W, 2 * n) || overlaps(in, nin, m.data, nm) ||
         overlaps(in, nin, v.data, nm) || (ns && overlaps(in, nin, m.scale, ns)) ||
         (ns && overlaps(in, nin, v.scale, ns));
}

AdamWConsts make_consts(float lr, float b1, float b2, float eps, float wd, int64_t step) {
  const double db1 = b1, db2 = b2, dlr = lr, dwd = wd;
  const double bc1 = 1.0 - std::pow(db1, static_cast<double>(step));
  const double bc2 = 1.0 - std::pow(db2, static_cast<double>(step));
  AdamWConsts h;
  h.beta1 = b1;
  h.beta2 = b2;
  h.omb1 = static_cast<float>(1.0 - db1);
  h.omb2 = static_cast<float>(1.0 - db2);
  h.eps = eps;
  h.decay = static_cast<float>(1.0 - dlr * dwd);
  h.neg_step_size = static_cast<float>(-dlr / bc1);
  h.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  return h;
}

// forge_wgrad_opt: the hyperparameters its optimizer reads, in range.
forge_status check_opt_hyper(int opt, const forge_opt_hyper& h, int64_t step) {
  if (opt < kOptSgd || opt > kOptRadam || step < 1) return FORGE_ERR_HYPER;
  auto nonneg = [](float x) { return x >= 0.0f && std::isfinite(x); };
  auto unit = [](float x) { return x >= 0.0f && x < 1.0f; };
  if (!nonneg(h.lr) || !nonneg(h.weight_decay)) return FORGE_ERR_HYPER;
  if ((opt == kOptLion || opt == kOptNadam || opt == kOptRadam) &&
      (!unit(h.beta1) || !unit(h.beta2)))
    return FORGE_ERR_HYPER;
  if (opt != kOptSgd && opt != kOptSgdMomentum && opt != kOptLion && !eps_ok(h.eps))
    return FORGE_ERR_HYPER;
  if (opt == kOptSgdMomentum && !unit(h.momentum)) return FORGE_ERR_HYPER;
  if (opt == kOptRmsprop && !unit(h.alpha)) return FORGE_ERR_HYPER;
  if (opt == kOptNadam && !nonneg(h.momentum_decay)) return FORGE_ERR_HYPER;
  return FORGE_OK;
}

// The step constants of forge_wgrad_opt, formed in fp64 from the float32
// hyperparameters and rounded once each to fp32.
OptConsts make_opt_consts(int opt, const forge_opt_hyper& h, int64_t step) {
  OptConsts c;
  std::memset(&c, 0, sizeof(c));
  const double lr = h.lr, t = static_cast<double>(step);
  c.opt = opt;
  c.lr = h.lr;
  c.wd = h.weight_decay;
  c.eps = h.eps;
  switch (opt) {
    case kOptSgdMomentum: c.a = h.momentum; break;
    case kOptRmsprop:
      c.a = h.alpha;
      c.oma = static_cast<float>(1.0 - static_cast<double>(h.alpha));
      break;
    case kOptLion:
    case kOptNadam:
    case kOptRadam: {
      const double b1 = h.beta1, b2 = h.beta2;
      c.a = h.beta1;
      c.oma = static_cast<float>(1.0 - b1);
      c.b = h.beta2;
      c.omb = static_cast<float>(1.0 - b2);
      if (opt == kOptLion) {
        c.decay = static_cast<float>(1.0 - lr * static_cast<double>(h.weight_decay));
      } else if (opt == kOptNadam) {
        // mu_i = beta1 (1 - 0.5 * 0.96^(i psi)); the running product falls
        // below fp64's range within a few thousand steps and then stays zero
        const double psi = h.momentum_decay;
        auto mu = [&](double i) { return b1 * (1.0 - 0.5 * std::pow(0.96, i * psi)); };
        double prod = 1.0;
        for (int64_t i = 1; i <= step && prod != 0.0; ++i) prod *= mu(static_cast<double>(i));
        const double mu_t = mu(t), mu_next = mu(t + 1.0);
        c.k1 = static_cast<float>(-lr * (1.0 - mu_t) / (1.0 - prod));
        c.k2 = static_cast<float>(-lr * mu_next / (1.0 - prod * mu_next));
        c.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(1.0 - std::pow(b2, t)));
      } else {
        const double bc1 = 1.0 - std::pow(b1, t), bc2 = 1.0 - std::pow(b2, t);
        const double rho_inf = 2.0 / (1.0 - b2) - 1.0;
        const double rho_t = rho_inf - 2.0 * t * std::pow(b2, t) / bc2;
        if (rho_t > 5.0) {
          const double r = std::sqrt((rho_t - 4.0) * (rho_t - 2.0) * rho_inf /
                                     ((rho_inf - 4.0) * (rho_inf - 2.0) * rho_t));
          c.rect = 1;
          c.k1 = static_cast<float>(-lr * r * std::sqrt(bc2) / bc1);
        } else {
          c.k1 = static_cast<float>(-lr / bc1);
        }
      }
      break;
    }
    default: break;
  }
  return c;
}

// Tile configuration, from measured sweeps over the Llama-3.1-8B projections
// on GB300.  At a few hundred tokens the fused step streams W, m, v through
// HBM: 128 x 128 tiles on one CTA, with two operand stages and four state
// slots for fp32 moments up to 512 tokens, equal stage and slot depths
// otherwise (int8 moments in half-tile slots).  From about a thousand tokens
// (768 for bf16 moments) the main loop matters and 256 x 256 tiles on a CTA
// pair (tcgen05 cta_group::2) win, since each SM then reads only half of the
// B operand from shared memory: balanced depths up to 1536 tokens, then as
// many operand stages as fit next to two state slots, and above 3072 tokens
// next to two half-tile slots.  The store-G kernel (fmt = dW dtype) keeps the
// 768-token split.  forge_set_tuning (or the FORGE_* environment variables,
// read once) overrides the choice.
GemmConfig finish_config(GemmConfig c, int64_t bt, int fmt, int mode);
forge_tuning current_tuning();

GemmConfig choose_config(int64_t bt, int fmt, int mode) {
  GemmConfig c;
  // (fp8 moments move the bytes of int8 ones and take int8's choices)
  const int64_t one_cta_upto = (mode == kModeFused && fmt == kFmtBF16) ? 640 : 768;
  if (bt <= one_cta_upto) {
    c.cg = 1;
    if (mode == kModeFused)
      c.prof = (fmt == kFmtF32 && bt <= 512) ? kProfStream : kProfBalanced;
    else
      c.prof = (fmt == kFmtBF16) ? kProfBalanced : kProfStream;
  } else {
    c.cg = 2;
    c.prof = bt <= 1536 ? kProfBalanced : (bt <= 3072 ? kProfMma : kProfDeep);
  }
  return finish_config(c, bt, fmt, mode);
}

// The fused step at the final micro-batch (an fp32 addend in every slot):
// the fused choice for the moment format; its slots are larger by the
// addend's fp32 box.
GemmConfig choose_acc_step_config(int64_t bt, int fmt) {
  return choose_config(bt, fmt, kModeFused);
}

// forge_wgrad_opt: the fused tile choice with two changes, from sweeps over
// the Llama-3.1-8B projections with zero, one and two states.  With fewer
// state bytes than AdamW the epilogue gains less from extra state slots, so
// one CTA always runs the balanced profile (SGD at 512 tokens: -9 %), and
// bf16 states keep balanced depths on pairs up to 3072 tokens (-2 to -5 %
// at 2048).
GemmConfig choose_opt_config(int64_t bt, int fmt, int nstate) {
  const int efmt = state_elem_fmt(fmt);   // fp32 or bf16 (kFmtNone for SGD)
  GemmConfig c;
  const int64_t one_cta_upto = (efmt == kFmtBF16) ? 640 : 768;
  if (bt <= one_cta_upto) {
    c.cg = 1;
    c.prof = kProfBalanced;
  } else {
    c.cg = 2;
    c.prof = bt <= 1536 ? kProfBalanced
           : bt <= 3072 ? (efmt == kFmtBF16 ? kProfBalanced : kProfMma)
                        : kProfDeep;
  }
  if (nstate == 1 && bt <= one_cta_upto && efmt == kFmtF32) c.prof = kProfStream;
  c = finish_config(c, bt, efmt, kModeFused);
  if (nstate <= 1 && bt <= one_cta_upto && current_tuning().bn != 128) {
    // Slots that hold W alone (SGD, 8 KB) or W and one state (24 KB fp32,
    // 16 KB bf16) leave room for 256-wide tiles on one CTA, which halve the
    // main loop's A re-reads.  Sweeps over the layer at 512 tokens, against
    // AdamW's slot layout and 128-wide tiles: SGD 0.41 -> 0.59 of HBM
    // (balanced); SGD with momentum, Adagrad, RMSprop and Lion with fp32
    // states 0.68-0.82 -> 0.90-0.93 (stream profile), bf16 states
    // 0.55-0.72 -> 0.70-0.79 (balanced).
    c.bn = 256;
  }
  // the state stream's L2 prefetch was measured for AdamW only
  if (current_tuning().state_prefetch < 0) c.state_prefetch = 0;
  return c;
}

// Tuning overrides.  The FORGE_* environment variables are read once, at the
// first call that chooses a configuration; afterwards only forge_set_tuning
// changes them.  Reading the environment on every call would cost host time
// per launch and race with setenv in other threads.
std::once_flag g_tune_once;
forge_tuning g_tune = {FORGE_PROFILE_AUTO, 0, 0, 0, -1, 0, -1, -1};

void tuning_from_env() {
  forge_tuning t = {FORGE_PROFILE_AUTO, 0, 0, 0, -1, 0, -1, -1};
  if (const char* e = std::getenv("FORGE_PROFILE")) {
    if (std::strcmp(e, "stream") == 0) t.profile = FORGE_PROFILE_STREAM;
    if (std::strcmp(e, "mma") == 0) t.profile = FORGE_PROFILE_MMA;
    if (std::strcmp(e, "balanced") == 0) t.profile = FORGE_PROFILE_BALANCED;
    if (std::strcmp(e, "deep") == 0) t.profile = FORGE_PROFILE_DEEP;
  }
  if (const char* e = std::getenv("FORGE_CG")) t.cta_group = std::atoi(e);
  if (const char* e = std::getenv("FORGE_BN")) t.bn = std::atoi(e);
  if (const char* e = std::getenv("FORGE_GROUP_M")) t.group_m = std::atoi(e);
  if (const char* e = std::getenv("FORGE_POLL_STORE")) t.poll_store = std::atoi(e) != 0;
  if (const char* e = std::getenv("FORGE_SPLITS")) t.splits = std::atoi(e);
  if (const char* e = std::getenv("FORGE_L2_HINTS")) t.l2_hints = std::atoi(e);
  if (const char* e = std::getenv("FORGE_STATE_PREFETCH")) t.state_prefetch = std::atoi(e);
  std::lock_guard<std::mutex> lk(g_mu);
  g_tune = t;
}

forge_tuning current_tuning() {
  std::call_once(g_tune_once, tuning_from_env);
  std::lock_guard<std::mutex> lk(g_mu);
  return g_tune;
}

// The accumulate mode: store-G's split between one CTA and pairs, but on one
// CTA 256-wide tiles with balanced depths (a sweep over the layer at 512
// tokens: beta = 1 from 0.63 to 0.76 of HBM, beta = 0 from 0.36 to 0.54;
// the light epilogue leaves the main loop in charge, and 256-wide tiles halve
// its A re-reads).
GemmConfig choose_accum_config(int64_t bt) {
  GemmConfig c;
  if (bt <= 768) {
    c.cg = 1;
    c.prof = kProfBalanced;
    c = finish_config(c, bt, kFmtF32, kModeAccum);
    const forge_tuning tu = current_tuning();
    if (tu.bn != 128) c.bn = 256;
    return c;
  }
  c.cg = 2;
  c.prof = bt <= 1536 ? kProfBalanced : (bt <= 3072 ? kProfMma : kProfDeep);
  return finish_config(c, bt, kFmtF32, kModeAccum);
}

// The tile width, the raster order and the store-lane wait follow from the
// grouping, profile and format; the tuning overrides apply last.
GemmConfig finish_config(GemmConfig c, int64_t bt, int fmt, int mode) {
  const forge_tuning tu = current_tuning();
  c.bn = (c.cg == 2) ? 256 : 128;
  if (tu.profile >= kProfStream && tu.profile <= kProfDeep) c.prof = tu.profile;
  if (tu.cta_group == 1 || tu.cta_group == 2) c.cg = tu.cta_group;
  if (tu.bn == 128 || tu.bn == 256) c.bn = tu.bn;
  if (c.cg == 2) c.bn = 256;                    // pairs always use 256 x 256 tiles
  if (c.cg == 1 && (fmt == kFmtI8 || fmt == kFmtF8)) c.bn = 128;   // 1-CTA 8-bit moments: 128-wide tiles
  // Tile rows per raster group (the kernel's tile_coords): 4 for 128 x 128
  // tiles; 8 for the weight-gradient modes on pairs (a sweep of 1, 2, 4, 8,
  // 16 and 32 over the layer at 2048-8192 tokens: 8 was fastest or tied, by
  // 4.8 % at 8192 with bf16 moments and 2 % at 4096 with int8 against plain
  // row-major order); 1 (row-major) for the input gradient, whose tile rows
  // are tokens and where a column-wise walk measured slower at 4096-8192.
  c.group_m = (c.cg == 1) ? 4 : (mode == kModeDgrad ? 1 : 8);
  // The store lanes poll for finished slots (instead of a suspending wait)
  // where the slot ring is short against the state stream: bf16 moments up
  // to 576 tokens on one CTA (+12 % at BT = 512), fp32 moments in the stream
  // profile (+0.3-1.4 %) and on CTA pairs (+2 % at 1024 and 4096 tokens).
  // Elsewhere it measured neutral or slower.
  c.poll_store = mode == kModeFused &&
                 ((c.cg == 1 && ((fmt == kFmtBF16 && bt <= 576) ||
                                 (fmt == kFmtF32 && c.prof == kProfStream))) ||
                  (c.cg == 2 && fmt == kFmtF32));
  if (tu.poll_store == 0 || tu.poll_store == 1) c.poll_store = tu.poll_store;
  if (tu.group_m >= 1 && tu.group_m <= 64) c.group_m = tu.group_m;
  c.l2_hints = 0;
  if (tu.l2_hints >= 0 && tu.l2_hints <= 3) c.l2_hints = tu.l2_hints;
  // L2 prefetch of the state stream two slices ahead: only fp32 moments in
  // the deep profile up to 6144 tokens gained (layer at 4096 tokens: -4.7 %;
  // neutral at 6144 and 8192); every other format and token count measured
  // slower with it (at 512 tokens by up to a third: the prefetches add DRAM
  // requests to a stream that is already bandwidth-bound)
  c.state_prefetch = (mode == kModeFused && fmt == kFmtF32 && c.prof == kProfDeep && bt <= 6144)
                         ? 2 : 0;
  if (tu.state_prefetch >= 0 && tu.state_prefetch <= 32) c.state_prefetch = tu.state_prefetch;
  c.grid = 0;
  c.splits = 1;
  return c;
}

// How many k-ranges to cut each tile of the input gradient into.  With few
// tiles (few tokens) most SMs would sit idle through a long reduction over
// d_out; splitting it gives every SM work, at the price of writing one fp32
// partial tile per unit and of the reduce kernel that adds them.  Estimated
// time, in nanoseconds: waves x k-steps per unit x 400 (one 64-deep k-step of
// a 256 x 256 tile on a CTA pair), plus, when split, 5000 (the reduce
// launch and the last partial write) and the partials' bytes at 4 TB/s
// (mostly L2 hits).  Splits are at most 8 and at least 8 k-steps
// long (shorter units cannot hide their 128 KB partial write behind the next
// unit's main loop), and only for queues shorter than two waves.
// The tuning's `splits` overrides (clamped to the same length limits).
int choose_splits(int64_t tiles, int64_t num_k, int64_t slots, int64_t ctile_bytes) {
  const int64_t max_s = std::max<int64_t>(1, std::min<int64_t>(8, num_k / 8));
  const int64_t f = current_tuning().splits;
  if (f >= 1) return static_cast<int>(std::min(f, max_s));
  if (tiles >= 2 * slots) return 1;
  auto cost = [&](int64_t s) {
    const int64_t waves = (tiles * s + slots - 1) / slots;
    int64_t ns = waves * ((num_k + s - 1) / s) * 400;
    if (s > 1) ns += 5000 + s * tiles * ctile_bytes / 4000;
    return ns;
  };
  int pick = 1;
  int64_t best = cost(1);
  for (int64_t s = 2; s <= max_s; ++s)
    if (cost(s) < best) {
      best = cost(s);
      pick = static_cast<int>(s);
    }
  return pick;
}

// The input-gradient GEMM dX = dY W (rows = tokens, K = d_out): a light
// epilogue, so the deepest operand pipeline on CTA pairs (256 x 256 tiles,
// measured faster than one CTA at every token count from 512 to 8192), with
// the reduction split where there are too few tiles for the SMs.
GemmConfig choose_dgrad_config(int64_t rows, int64_t d_in, int64_t d_out, int num_sms) {
  GemmConfig c;
  c.cg = 2;
  c.prof = kProfMma;
  c = finish_config(c, d_out, kFmtBF16, kModeDgrad);
  const int64_t tiles = ((rows + kBM * c.cg - 1) / (kBM * c.cg)) * ((d_in + c.bn - 1) / c.bn);
  const int64_t num_k = (d_out + bk_of(c.cg) - 1) / bk_of(c.cg);
  c.splits = choose_splits(tiles, num_k, num_sms / c.cg,
                           static_cast<int64_t>(c.cg) * kBM * c.bn * sizeof(float));
  return c;
}

int64_t tiles_of(const GemmConfig& c, int64_t d_in, int64_t d_out) {
  return ((d_out + kBM * c.cg - 1) / (kBM * c.cg)) * ((d_in + c.bn - 1) / c.bn);
}

// Persistent grid: one CTA (or CTA pair) per SM (pair of SMs), at most one per tile.
void set_grid(GemmConfig& c, int64_t tiles, int num_sms) {
  const int64_t units = num_sms / c.cg;
  c.grid = static_cast<int>(c.cg * (tiles < units ? tiles : units));
}

GemmParams base_params(int64_t bt, const GemmConfig& cfg, const DeviceInfo& d) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.bt = static_cast<int32_t>(bt);
  const int bk = bk_of(cfg.cg);
  p.num_k = static_cast<int32_t>((bt + bk - 1) / bk);
  p.group_m = cfg.group_m;
  p.err = d.err_word;
  p.err_site = d.site_word;
  p.timeout_ns = g_wait_limit_ns;
  p.poll_store = cfg.poll_store;
  p.l2_hints = cfg.l2_hints;
  p.state_prefetch = cfg.state_prefetch;
  p.splits = 1;
  return p;
}

// Appends one linear layer to a launch's tile queue.
void add_problem(GemmParams& p, const GemmConfig& cfg, int64_t d_in, int64_t d_out,
                 float* m_scale, float* v_scale) {
  GemmProblem& q = p.prob[p.nprob];
  q.d_in = static_cast<int32_t>(d_in);
  q.d_out = static_cast<int32_t>(d_out);
  q.tiles_m = static_cast<int32_t>((d_out + kBM * cfg.cg - 1) / (kBM * cfg.cg));
  q.tiles_n = static_cast<int32_t>((d_in + cfg.bn - 1) / cfg.bn);
  q.tile_start = p.num_tiles;
  q.num_k = p.num_k;
  q.part_tile0 = p.num_tiles;
  q.m_scale = m_scale;
  q.v_scale = v_scale;
  p.num_tiles += q.tiles_m * q.tiles_n;
  p.num_units = p.num_tiles * p.splits;
  p.nprob += 1;
}

// Operand descriptors: dY [bt, d_out] and X [bt, d_in], boxes of 64 columns x
// bk tokens with the 128-byte swizzle.
bool operand_maps(GemmMaps& maps, const void* X, const void* dY, int64_t bt, int64_t d_in,
                  int64_t d_out, int bk) {
  return get_map(&maps.dy, dY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_out, bt, d_out * 2, 64, bk,
                 CU_TENSOR_MAP_SWIZZLE_128B) &&
         get_map(&maps.x, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_in, bt, d_in * 2, 64, bk,
                 CU_TENSOR_MAP_SWIZZLE_128B);
}

// State descriptors of one layer for the fused kernel: W (bf16) and the two
// moments, boxes of one epilogue slice (32 columns, or 128 for 8-bit moments)
// x the slot's rows.
bool state_maps(GemmMaps& maps, void* W, const forge_moment& m, const forge_moment& v,
                int64_t d_in, int64_t d_out, forge_moment_fmt fmt, int prof) {
  if (fmt == FORGE_MOM_INT8_B128 || fmt == FORGE_MOM_FP8_E4M3) {   // 8-bit codes
    const uint32_t rows = static_cast<uint32_t>(slot_rows(kModeFused, static_cast<int>(fmt), prof));
    return get_map(&maps.w, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_in, d_out, d_in * 2, 64, rows,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
           get_map(&maps.m, m.data, CU_TENSOR_MAP_DATA_TYPE_UINT8, d_in, d_out, d_in, 128, rows,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
           get_map(&maps.v, v.data, CU_TENSOR_MAP_DATA_TYPE_UINT8, d_in, d_out, d_in, 128, rows,
                   CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const bool f32 = fmt == FORGE_MOM_FP32;
  const CUtensorMapDataType mdt =
      f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle msw = f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const int eb = f32 ? 4 : 2;
  const uint32_t rows =
      static_cast<uint32_t>(slot_rows(kModeFused, f32 ? kFmtF32 : kFmtBF16, prof));
  return get_map(&maps.w, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_in, d_out, d_in * 2, 32, rows,
                 CU_TENSOR_MAP_SWIZZLE_64B) &&
         get_map(&maps.m, m.data, mdt, d_in, d_out, d_in * eb, 32, rows, msw) &&
         get_map(&maps.v, v.data, mdt, d_in, d_out, d_in * eb, 32, rows, msw);
}

uint64_t state_bytes_of(const forge_linear& L, forge_moment_fmt fmt) {
  const uint64_t n = static_cast<uint64_t>(L.d_in) * static_cast<uint64_t>(L.d_out);
  return n * (2 + 2 * mom_elem_bytes(fmt));
}

// The launch order of a group's layers: largest first, so the small ones
// fill the last wave (a stable insertion sort on the state bytes).
void largest_first(const forge_linear* layers, int n, forge_moment_fmt fmt, int* order) {
  for (int i = 0; i < n; ++i) order[i] = i;
  for (int i = 1; i < n; ++i)
    for (int j = i; j > 0 && state_bytes_of(layers[order[j]], fmt) >
                                 state_bytes_of(layers[order[j - 1]], fmt); --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
}

// Checks one layer of a fused launch (everything but cross-layer aliasing).
forge_status check_linear(const forge_linear& L, int64_t bt, forge_moment_fmt fmt) {
  forge_status s = check_shape(bt, L.d_in, L.d_out);
  if (s != FORGE_OK) return s;
  if (bt > 0 && (!L.X || !L.dY)) return FORGE_ERR_NULL;
  s = check_state(L.W, L.m, L.v, L.d_in, L.d_out, fmt);
  if (s != FORGE_OK) return s;
  if (bt > 0 && (!aligned16(L.X) || !aligned16(L.dY))) return FORGE_ERR_ALIGN;
  return FORGE_OK;
}

// The outputs (W, m, v, scales) of layer b overlap an input or an output of layer a.
bool layers_clash(const forge_linear& a, const forge_linear& b, int64_t bt, forge_moment_fmt fmt,
                  bool same) {
  if (bt > 0 && (input_overlaps_state(a.X, 2ull * bt * a.d_in, b.W, b.m, b.v, b.d_in, b.d_out, fmt) ||
                 input_overlaps_state(a.dY, 2ull * bt * a.d_out, b.W, b.m, b.v, b.d_in, b.d_out,
                                      fmt)))
    return true;
  if (same) return false;
  const uint64_t n = static_cast<uint64_t>(a.d_in) * static_cast<uint64_t>(a.d_out);
  const uint64_t nm = n * mom_elem_bytes(fmt);
  const uint64_t ns = scale_bytes(fmt, n);
  return input_overlaps_state(a.W, 2 * n, b.W, b.m, b.v, b.d_in, b.d_out, fmt) ||
         input_overlaps_state(a.m.data, nm, b.W, b.m, b.v, b.d_in, b.d_out, fmt) ||
         input_overlaps_state(a.v.data, nm, b.W, b.m, b.v, b.d_in, b.d_out, fmt) ||
         (ns && input_overlaps_state(a.m.scale, ns, b.W, b.m, b.v, b.d_in, b.d_out, fmt)) ||
         (ns && input_overlaps_state(a.v.scale, ns, b.W, b.m, b.v, b.d_in, b.d_out, fmt));
}

int take_drop_flag() {
  std::lock_guard<std::mutex> lk(g_mu);
  const int f = g_drop_first_arrival;
  g_drop_first_arrival = 0;
  return f;
}

}  // namespace
}  // namespace forge

using namespace forge;

extern "C" {

forge_status forge_wgrad_adamw_grouped(const forge_linear* layers, int n, int64_t bt, float lr,
                                       float beta1, float beta2, float eps, float weight_decay,
                                       int64_t step, forge_moment_fmt fmt, forge_stream stream) {
  if (!layers) return FORGE_ERR_NULL;
  if (n < 1 || n > FORGE_MAX_GROUP) return FORGE_ERR_SHAPE;
  for (int i = 0; i < n; ++i) {
    forge_status s = check_linear(layers[i], bt, fmt);
    if (s != FORGE_OK) return s;
  }
  forge_status s = check_hyper(lr, beta1, beta2, eps, weight_decay, step);
  if (s != FORGE_OK) return s;
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j)
      if (layers_clash(layers[i], layers[j], bt, fmt, i == j)) return FORGE_ERR_ALIAS;
  DeviceInfo* d = nullptr;
  s = device_info(&d);
  if (s != FORGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AdamWConsts h = make_consts(lr, beta1, beta2, eps, weight_decay, step);
  const int ifmt = static_cast<int>(fmt);
  if (bt == 0) {   // G = 0: the moments decay and W takes decay and the m-driven update
    for (int i = 0; i < n; ++i) {
      const forge_linear& L = layers[i];
      if (launch_adamw(nullptr, 0, L.W, L.m.data, L.v.data, L.m.scale, L.v.scale, L.d_in,
                       L.d_out, ifmt, h, d->num_sms, st) != cudaSuccess)
        return FORGE_ERR_LAUNCH;
    }
    return FORGE_OK;
  }
  GemmConfig cfg = choose_config(bt, ifmt, kModeFused);
  int order[FORGE_MAX_GROUP];
  largest_first(layers, n, fmt, order);
  GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  args.p = base_params(bt, cfg, *d);
  args.p.h = h;
  for (int k = 0; k < n; ++k) {
    const forge_linear& L = layers[order[k]];
    GemmMaps& maps = args.maps[k];
    if (!operand_maps(maps, L.X, L.dY, bt, L.d_in, L.d_out, bk_of(cfg.cg)) ||
        !state_maps(maps, L.W, L.m, L.v, L.d_in, L.d_out, fmt, cfg.prof))
      return FORGE_ERR_LAUNCH;
    add_problem(args.p, cfg, L.d_in, L.d_out, L.m.scale, L.v.scale);
  }
  set_grid(cfg, args.p.num_units, d->num_sms);
  args.p.drop_first_arrival = take_drop_flag();
  return launch_gemm(kModeFused, ifmt, cfg, args, st) == cudaSuccess ? FORGE_OK
                                                                      : FORGE_ERR_LAUNCH;
}

forge_status forge_wgrad_adamw_acc_grouped(const forge_linear* layers, const float* const* B,
                                           int n, int64_t bt, float lr, float beta1, float beta2,
                                           float eps, float weight_decay, int64_t step,
                                           forge_moment_fmt fmt, forge_stream stream) {
  if (!layers || !B) return FORGE_ERR_NULL;
  if (n < 1 || n > FORGE_MAX_GROUP) return FORGE_ERR_SHAPE;
  if (fmt != FORGE_MOM_FP32 && fmt != FORGE_MOM_BF16) return FORGE_ERR_FORMAT;
  for (int i = 0; i < n; ++i) {
    forge_status s = check_linear(layers[i], bt, fmt);
    if (s != FORGE_OK) return s;
    if (!B[i]) return FORGE_ERR_NULL;
    if (!aligned16(B[i])) return FORGE_ERR_ALIGN;
  }
  forge_status s = check_hyper(lr, beta1, beta2, eps, weight_decay, step);
  if (s != FORGE_OK) return s;
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      if (layers_clash(layers[i], layers[j], bt, fmt, i == j)) return FORGE_ERR_ALIAS;
      // the accumulators are read while the states are written
      const forge_linear& L = layers[j];
      const uint64_t nb = 4ull * layers[i].d_in * layers[i].d_out;
      if (input_overlaps_state(B[i], nb, L.W, L.m, L.v, L.d_in, L.d_out, fmt))
        return FORGE_ERR_ALIAS;
    }
  DeviceInfo* d = nullptr;
  s = device_info(&d);
  if (s != FORGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AdamWConsts h = make_consts(lr, beta1, beta2, eps, weight_decay, step);
  if (bt == 0) {   // G = 0: the step reads the accumulator alone, as forge_adamw does
    for (int i = 0; i < n; ++i) {
      const forge_linear& L = layers[i];
      if (launch_adamw(B[i], 0, L.W, L.m.data, L.v.data, nullptr, nullptr, L.d_in, L.d_out,
                       static_cast<int>(fmt), h, d->num_sms, st) != cudaSuccess)
        return FORGE_ERR_LAUNCH;
    }
    return FORGE_OK;
  }
  const int afmt = (fmt == FORGE_MOM_FP32) ? kFmtF32A : kFmtBF16A;
  GemmConfig cfg = choose_acc_step_config(bt, static_cast<int>(fmt));
  int order[FORGE_MAX_GROUP];
  largest_first(layers, n, fmt, order);
  GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  args.p = base_params(bt, cfg, *d);
  args.p.h = h;
  const uint32_t rows = static_cast<uint32_t>(slot_rows(kModeFused, afmt, cfg.prof));
  for (int k = 0; k < n; ++k) {
    const forge_linear& L = layers[order[k]];
    GemmMaps& maps = args.maps[k];
    if (!operand_maps(maps, L.X, L.dY, bt, L.d_in, L.d_out, bk_of(cfg.cg)) ||
        !state_maps(maps, L.W, L.m, L.v, L.d_in, L.d_out, fmt, cfg.prof) ||
        !get_map(&maps.b, B[order[k]], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, L.d_in, L.d_out,
                 L.d_in * 4, 32, rows, CU_TENSOR_MAP_SWIZZLE_128B))
      return FORGE_ERR_LAUNCH;
    add_problem(args.p, cfg, L.d_in, L.d_out, nullptr, nullptr);
  }
  set_grid(cfg, args.p.num_units, d->num_sms);
  args.p.drop_first_arrival = take_drop_flag();
  return launch_gemm(kModeFused, afmt, cfg, args, st) == cudaSuccess ? FORGE_OK
                                                                     : FORGE_ERR_LAUNCH;
}

forge_status forge_wgrad_adamw_acc(const void* X, const void* dY, void* W, forge_moment m,
                                   forge_moment v, const float* B, int64_t bt, int64_t d_in,
                                   int64_t d_out, float lr, float beta1, float beta2, float eps,
                                   float weight_decay, int64_t step, forge_moment_fmt fmt,
                                   forge_stream stream) {
  forge_linear L;
  std::memset(&L, 0, sizeof(L));
  L.X = X;
  L.dY = dY;
  L.W = W;
  L.m = m;
  L.v = v;
  L.d_in = d_in;
  L.d_out = d_out;
  return forge_wgrad_adamw_acc_grouped(&L, &B, 1, bt, lr, beta1, beta2, eps, weight_decay, step,
                                       fmt, stream);
}

forge_status forge_wgrad_adamw_sr_grouped(const forge_linear* layers, const uint64_t* seeds,
                                          int n, int64_t bt, float lr, float beta1, float beta2,
                                          float eps, float weight_decay, int64_t step,
                                          forge_moment_fmt fmt, forge_stream stream) {
  if (!layers || !seeds) return FORGE_ERR_NULL;
  if (n < 1 || n > FORGE_MAX_GROUP) return FORGE_ERR_SHAPE;
  for (int i = 0; i < n; ++i) {
    forge_status s = check_linear(layers[i], bt, fmt);
    if (s != FORGE_OK) return s;
  }
  if (fmt == FORGE_MOM_INT8_B128 || fmt == FORGE_MOM_FP8_E4M3)
    return FORGE_ERR_FORMAT;   // fp32 or bf16 moments
  forge_status s = check_hyper(lr, beta1, beta2, eps, weight_decay, step);
  if (s != FORGE_OK) return s;
  if (step > INT32_MAX) return FORGE_ERR_HYPER;   // the step is a 32-bit Philox counter word
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j)
      if (layers_clash(layers[i], layers[j], bt, fmt, i == j)) return FORGE_ERR_ALIAS;
  DeviceInfo* d = nullptr;
  s = device_info(&d);
  if (s != FORGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ifmt = static_cast<int>(fmt);
  // the tensor-core kernel even without tokens (G = 0): the separate
  // optimizer kernel rounds W to nearest
  GemmConfig cfg = choose_config(bt, ifmt, kModeFused);
  int order[FORGE_MAX_GROUP];
  largest_first(layers, n, fmt, order);
  GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  args.p = base_params(bt, cfg, *d);
  args.p.h = make_consts(lr, beta1, beta2, eps, weight_decay, step);
  args.p.sr = 1;
  args.p.sr_step = static_cast<int32_t>(step);
  for (int k = 0; k < n; ++k) {
    const forge_linear& L = layers[order[k]];
    GemmMaps& maps = args.maps[k];
    if ((bt > 0 && !operand_maps(maps, L.X, L.dY, bt, L.d_in, L.d_out, bk_of(cfg.cg))) ||
        !state_maps(maps, L.W, L.m, L.v, L.d_in, L.d_out, fmt, cfg.prof))
      return FORGE_ERR_LAUNCH;
    add_problem(args.p, cfg, L.d_in, L.d_out, L.m.scale, L.v.scale);
    args.p.prob[k].sr_seed = seeds[order[k]];
  }
  set_grid(cfg, args.p.num_units, d->num_sms);
  args.p.drop_first_arrival = take_drop_flag();
  return launch_gemm(kModeFused, ifmt, cfg, args, st) == cudaSuccess ? FORGE_OK
                                                                      : FORGE_ERR_LAUNCH;
}

forge_status forge_wgrad_adamw_sr(const void* X, const void* dY, void* W, forge_moment m,
                                  forge_moment v, int64_t bt, int64_t d_in, int64_t d_out,
                                  float lr, float beta1, float beta2, float eps,
                                  float weight_decay, int64_t step, forge_moment_fmt fmt,
                                  uint64_t seed, forge_stream stream) {
  forge_linear L;
  L.X = X;
  L.dY = dY;
  L.W = W;
  L.m = m;
  L.v = v;
  L.d_in = d_in;
  L.d_out = d_out;
  return forge_wgrad_adamw_sr_grouped(&L, &seed, 1, bt, lr, beta1, beta2, eps, weight_decay,
                                      step, fmt, stream);
}

forge_status forge_wgrad_adamw(const void* X, const void* dY, void* W, forge_moment m,
                               forge_moment v, int64_t bt, int64_t d_in, int64_t d_out, float lr,
                               float beta1, float beta2, float eps, float weight_decay,
                               int64_t step, forge_moment_fmt fmt, forge_stream stream) {
  forge_linear L;
  L.X = X;
  L.dY = dY;
  L.W = W;
  L.m = m;
  L.v = v;
  L.d_in = d_in;
  L.d_out = d_out;
  return forge_wgrad_adamw_grouped(&L, 1, bt, lr, beta1, beta2, eps, weight_decay, step, fmt,
                                   stream);
}

forge_status forge_wgrad(const void* X, const void* dY, void* dW, forge_dtype dw_dtype,
                         int64_t bt, int64_t d_in, int64_t d_out, forge_stream stream) {
  forge_status s = check_shape(bt, d_in, d_out);
  if (s != FORGE_OK) return s;
  if (dw_dtype != FORGE_DT_FP32 && dw_dtype != FORGE_DT_BF16) return FORGE_ERR_FORMAT;
  if (!dW || (bt > 0 && (!X || !dY))) return FORGE_ERR_NULL;
  if (!aligned16(dW) || (bt > 0 && (!aligned16(X) || !aligned16(dY)))) return FORGE_ERR_ALIGN;
  const uint64_t nbytes =
      static_cast<uint64_t>(d_in) * d_out * (dw_dtype == FORGE_DT_FP32 ? 4 : 2);
  if (bt > 0 && (overlaps(dW, nbytes, X, 2ull * bt * d_in) ||
                 overlaps(dW, nbytes, dY, 2ull * bt * d_out)))
    return FORGE_ERR_ALIAS;
  DeviceInfo* d = nullptr;
  s = device_info(&d);
  if (s != FORGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bt == 0) return cudaMemsetAsync(dW, 0, nbytes, st) == cudaSuccess ? FORGE_OK : FORGE_ERR_CUDA;
  const int ifmt = dw_dtype == FORGE_DT_FP32 ? kFmtF32 : kFmtBF16;
  GemmConfig cfg = choose_config(bt, ifmt, kModeStoreG);
  GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  GemmMaps& maps = args.maps[0];
  bool ok = operand_maps(maps, X, dY, bt, d_in, d_out, bk_of(cfg.cg));
  if (dw_dtype == FORGE_DT_FP32)
    ok = ok && get_map(&maps.w, dW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d_in, d_out, d_in * 4, 32, kBM,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok = ok && get_map(&maps.w, dW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_in, d_out, d_in * 2, 32,
                       kBM, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return FORGE_ERR_LAUNCH;
  args.p = base_params(bt, cfg, *d);
  add_problem(args.p, cfg, d_in, d_out, nullptr, nullptr);
  set_grid(cfg, args.p.num_units, d->num_sms);
  args.p.drop_first_arrival = take_drop_flag();
  return launch_gemm(kModeStoreG, ifmt, cfg, args, st) == cudaSuccess ? FORGE_OK
                                                                       : FORGE_ERR_LAUNCH;
}

}  // extern "C"

namespace {

// Where a split input-gradient launch keeps its fp32 partials: the library's
// stream-ordered pool (forge_dgrad), its static scratch (forge_dgrad_noalloc),
// or the caller's workspace (the grouped calls; none means unsplit).
enum WsMode { kWsPool, kWsStatic, kWsCaller };

// The k-steps of one projection's reduction over d_out.
int64_t dgrad_num_k(const forge_dgrad_item& it, const GemmConfig& c) {
  return (it.d_out + bk_of(c.cg) - 1) / bk_of(c.cg);
}

// Checks the projections of an input-gradient call: shapes, pointers, and
// that no dX overlaps any projection's dY, W or another dX.
forge_status check_dgrad_items(const forge_dgrad_item* items, int n, int64_t bt) {
  if (!items) return FORGE_ERR_NULL;
  if (n < 1 || n > FORGE_MAX_GROUP) return FORGE_ERR_SHAPE;
  for (int i = 0; i < n; ++i) {
    const forge_dgrad_item& a = items[i];
    forge_status s = check_shape(bt, a.d_in, a.d_out);
    if (s != FORGE_OK) return s;
    if (bt == 0) continue;
    if (!a.dY || !a.W || !a.dX) return FORGE_ERR_NULL;
    if (!aligned16(a.dY) || !aligned16(a.W) || !aligned16(a.dX)) return FORGE_ERR_ALIGN;
  }
  if (bt == 0) return FORGE_OK;
  for (int i = 0; i < n; ++i) {
    const uint64_t ndx = 2ull * bt * items[i].d_in;
    for (int j = 0; j < n; ++j) {
      const forge_dgrad_item& b = items[j];
      if (overlaps(items[i].dX, ndx, b.dY, 2ull * bt * b.d_out) ||
          overlaps(items[i].dX, ndx, b.W, 2ull * b.d_in * b.d_out) ||
          (j != i && overlaps(items[i].dX, ndx, b.dX, 2ull * bt * b.d_in)))
        return FORGE_ERR_ALIAS;
    }
  }
  return FORGE_OK;
}

// The launch configuration, the order of the projections in the tile queue
// (most work first, so the short reductions fill the last wave) and the split
// count the library would choose, before any workspace limit.
struct DgradPlan {
  GemmConfig cfg;
  int order[FORGE_MAX_GROUP];
  int64_t tiles;
  size_t ctile_bytes;
};
DgradPlan plan_dgrad(const forge_dgrad_item* items, int n, int64_t bt, int num_sms) {
  DgradPlan pl;
  int64_t max_din = 0, max_dout = 0;
  for (int i = 0; i < n; ++i) {
    max_din = std::max<int64_t>(max_din, items[i].d_in);
    max_dout = std::max<int64_t>(max_dout, items[i].d_out);
  }
  pl.cfg = choose_dgrad_config(bt, max_din, max_dout, num_sms);
  const GemmConfig& c = pl.cfg;
  auto tiles_of_item = [&](const forge_dgrad_item& it) {
    return ((bt + kBM * c.cg - 1) / (kBM * c.cg)) * ((it.d_in + c.bn - 1) / c.bn);
  };
  pl.tiles = 0;
  int64_t max_k = 0, min_k = INT64_MAX;
  for (int i = 0; i < n; ++i) {
    pl.tiles += tiles_of_item(items[i]);
    max_k = std::max(max_k, dgrad_num_k(items[i], c));
    min_k = std::min(min_k, dgrad_num_k(items[i], c));
    pl.order[i] = i;
  }
  for (int i = 1; i < n; ++i)
    for (int j = i; j > 0; --j) {
      const forge_dgrad_item &a = items[pl.order[j]], &b = items[pl.order[j - 1]];
      if (tiles_of_item(a) * dgrad_num_k(a, c) <= tiles_of_item(b) * dgrad_num_k(b, c)) break;
      std::swap(pl.order[j], pl.order[j - 1]);
    }
  pl.ctile_bytes = static_cast<size_t>(c.cg) * kBM * c.bn * sizeof(float);
  // one split count for the launch: from the longest reduction, never more
  // k-ranges than the shortest one has k-steps
  pl.cfg.splits = static_cast<int>(std::min<int64_t>(
      choose_splits(pl.tiles, max_k, num_sms / c.cg, static_cast<int64_t>(pl.ctile_bytes)),
      min_k));
  return pl;
}

forge_status dgrad_run(const forge_dgrad_item* items, int n, int64_t bt, WsMode mode, void* cws,
                       size_t cws_bytes, forge_stream stream) {
  forge_status s = check_dgrad_items(items, n, bt);
  if (s != FORGE_OK) return s;
  if (bt == 0) return FORGE_OK;   // no tokens: every dX is empty
  DeviceInfo* d = nullptr;
  s = device_info(&d);
  if (s != FORGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DgradPlan pl = plan_dgrad(items, n, bt, d->num_sms);
  GemmConfig& cfg = pl.cfg;
  GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  int64_t max_dout = 0;
  for (int i = 0; i < n; ++i) max_dout = std::max<int64_t>(max_dout, items[i].d_out);
  args.p = base_params(max_dout, cfg, *d);   // the reductions run over d_out
  args.p.splits = cfg.splits;
  const int bk = bk_of(cfg.cg);
  for (int k = 0; k < n; ++k) {
    const forge_dgrad_item& it = items[pl.order[k]];
    GemmMaps& maps = args.maps[k];
    // A = dY read K-major: 64 of d_out x 64 token rows per box; B = W read
    // MN-major: 64 of d_in x bk of d_out per box; dX stored in 32 x 128 boxes
    const bool ok =
        get_map(&maps.dy, it.dY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, it.d_out, bt, it.d_out * 2, 64,
                64, CU_TENSOR_MAP_SWIZZLE_128B) &&
        get_map(&maps.x, it.W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, it.d_in, it.d_out, it.d_in * 2,
                64, bk, CU_TENSOR_MAP_SWIZZLE_128B) &&
        get_map(&maps.w, it.dX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, it.d_in, bt, it.d_in * 2, 32,
                kBM, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return FORGE_ERR_LAUNCH;
    add_problem(args.p, cfg, it.d_in, bt, nullptr, nullptr);   // tile rows are tokens
    args.p.prob[k].num_k = static_cast<int32_t>(dgrad_num_k(it, cfg));
  }
  // Split partials: taken from the pool in stream order and given back after
  // the reduce kernels, or placed in the static scratch or the caller's
  // workspace with as many splits as fit.  Without the memory the launch runs
  // unsplit (same accuracy, slower).
  void* ws = nullptr;
  auto need = [&](int sp) { return static_cast<size_t>(args.p.num_tiles) * sp * pl.ctile_bytes; };
  if (mode == kWsPool) {
    if (args.p.splits > 1) {
      cudaMemPool_t pool = workspace_pool(*d);
      if (pool && cudaMallocFromPoolAsync(&ws, need(args.p.splits), pool, st) == cudaSuccess) {
        args.p.part = static_cast<float*>(ws);
      } else {
        (void)cudaGetLastError();
        ws = nullptr;
        args.p.splits = 1;
      }
    }
  } else {
    float* base = mode == kWsStatic ? d->scratch : static_cast<float*>(cws);
    const size_t cap = mode == kWsStatic ? kNoAllocScratchBytes : (cws ? cws_bytes : 0);
    while (args.p.splits > 1 && need(args.p.splits) > cap) --args.p.splits;
    if (args.p.splits > 1) args.p.part = base;
  }
  args.p.num_units = args.p.num_tiles * args.p.splits;
  set_grid(cfg, args.p.num_units, d->num_sms);
  args.p.drop_first_arrival = take_drop_flag();
  cudaError_t e = launch_gemm(kModeDgrad, kFmtBF16, cfg, args, st);
  for (int k = 0; e == cudaSuccess && args.p.splits > 1 && k < n; ++k) {
    const GemmProblem& q = args.p.prob[k];
    const forge_dgrad_item& it = items[pl.order[k]];
    e = launch_dgrad_reduce(args.p.part + static_cast<size_t>(q.part_tile0) * args.p.splits *
                                              (pl.ctile_bytes / sizeof(float)),
                            args.p.splits, cfg.cg, cfg.bn, q.tiles_m, q.tiles_n, bt, it.d_in,
                            it.dX, d->num_sms, st);
  }
  if (ws) cudaFreeAsync(ws, st);
  return e == cudaSuccess ? FORGE_OK : FORGE_ERR_LAUNCH;
}

forge_dgrad_item dgrad_item(const void* dY, const void* W, void* dX, int64_t d_in,
                            int64_t d_out) {
  forge_dgrad_item it;
  it.dY = dY;
  it.W = W;
  it.dX = dX;
  it.d_in = d_in;
  it.d_out = d_out;
  return it;
}

}  // namespace

extern "C" {

forge_status forge_dgrad(const void* dY, const void* W, void* dX, int64_t bt, int64_t d_in,
                         int64_t d_out, forge_stream stream) {
  const forge_dgrad_item it = dgrad_item(dY, W, dX, d_in, d_out);
  return dgrad_run(&it, 1, bt, kWsPool, nullptr, 0, stream);
}

forge_status forge_dgrad_grouped(const forge_dgrad_item* items, int n, int64_t bt,
                                 void* workspace, size_t workspace_bytes, forge_stream stream) {
  if (workspace && !aligned16(workspace)) return FORGE_ERR_ALIGN;
  return dgrad_run(items, n, bt, kWsCaller, workspace, workspace_bytes, stream);
}

size_t forge_dgrad_workspace_bytes(const forge_dgrad_item* items, int n, int64_t bt) {
  if (!items || n < 1 || n > FORGE_MAX_GROUP || bt <= 0) return 0;
  for (int i = 0; i < n; ++i)
    if (check_shape(bt, items[i].d_in, items[i].d_out) != FORGE_OK) return 0;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
  }
  const DgradPlan pl = plan_dgrad(items, n, bt, sms);
  return pl.cfg.splits > 1 ? static_cast<size_t>(pl.tiles) * pl.cfg.splits * pl.ctile_bytes : 0;
}

forge_status forge_wgrad_accumulate_grouped(const forge_accum_item* items, int n, int64_t bt,
                                            float beta, forge_stream stream) {
  if (!items) return FORGE_ERR_NULL;
  if (n < 1 || n > FORGE_MAX_GROUP) return FORGE_ERR_SHAPE;
  if (!std::isfinite(beta)) return FORGE_ERR_HYPER;
  for (int i = 0; i < n; ++i) {
    const forge_accum_item& a = items[i];
    forge_status s = check_shape(bt, a.d_in, a.d_out);
    if (s != FORGE_OK) return s;
    if (!a.B || (bt > 0 && (!a.X || !a.dY))) return FORGE_ERR_NULL;
    if (!aligned16(a.B) || (bt > 0 && (!aligned16(a.X) || !aligned16(a.dY))))
      return FORGE_ERR_ALIGN;
  }
  // no B overlaps any item's inputs or another B
  for (int i = 0; i < n; ++i) {
    const uint64_t nb = 4ull * static_cast<uint64_t>(items[i].d_in) *
                        static_cast<uint64_t>(items[i].d_out);
    for (int j = 0; j < n; ++j) {
      const forge_accum_item& b = items[j];
      if (bt > 0 && (overlaps(items[i].B, nb, b.X, 2ull * bt * b.d_in) ||
                     overlaps(items[i].B, nb, b.dY, 2ull * bt * b.d_out)))
        return FORGE_ERR_ALIAS;
      if (j != i && overlaps(items[i].B, nb, b.B, 4ull * b.d_in * b.d_out)) return FORGE_ERR_ALIAS;
    }
  }
  DeviceInfo* d = nullptr;
  forge_status s = device_info(&d);
  if (s != FORGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmConfig cfg = choose_accum_config(bt);
  // largest first
  int order[FORGE_MAX_GROUP];
  for (int i = 0; i < n; ++i) order[i] = i;
  for (int i = 1; i < n; ++i)
    for (int j = i; j > 0 && items[order[j]].d_in * items[order[j]].d_out >
                                 items[order[j - 1]].d_in * items[order[j - 1]].d_out; --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
  GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  args.p = base_params(bt, cfg, *d);
  args.p.accum_beta = beta;
  args.p.accum_load = beta != 0.0f;
  for (int k = 0; k < n; ++k) {
    const forge_accum_item& a = items[order[k]];
    GemmMaps& maps = args.maps[k];
    const bool ok = (bt == 0 || operand_maps(maps, a.X, a.dY, bt, a.d_in, a.d_out,
                                             bk_of(cfg.cg))) &&
                    get_map(&maps.w, a.B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.d_in, a.d_out,
                            a.d_in * 4, 32, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return FORGE_ERR_LAUNCH;
    add_problem(args.p, cfg, a.d_in, a.d_out, nullptr, nullptr);
  }
  set_grid(cfg, args.p.num_units, d->num_sms);
  args.p.drop_first_arrival = take_drop_flag();
  return launch_gemm(kModeAccum, kFmtF32, cfg, args, st) == cudaSuccess ? FORGE_OK
                                                                         : FORGE_ERR_LAUNCH;
}

forge_status forge_wgrad_accumulate(const void* X, const void* dY, float* B, float beta,
                                    int64_t bt, int64_t d_in, int64_t d_out,
                                    forge_stream stream) {
  forge_accum_item a;
  a.X = X;
  a.dY = dY;
  a.B = B;
  a.d_in = d_in;
  a.d_out = d_out;
  return forge_wgrad_accumulate_grouped(&a, 1, bt, beta, stream);
}

forge_status forge_wgrad_opt_grouped(const forge_linear* layers, int n, int64_t bt,
                                     forge_optimizer opt, const forge_opt_hyper* hyper,
                                     int64_t step, forge_moment_fmt fmt, forge_stream stream) {
  if (!layers) return FORGE_ERR_NULL;
  if (n < 1 || n > FORGE_MAX_GROUP) return FORGE_ERR_SHAPE;
  if (!hyper) return FORGE_ERR_HYPER;
  forge_status s = check_opt_hyper(static_cast<int>(opt), *hyper, step);
  if (s != FORGE_OK) return s;
  if (fmt != FORGE_MOM_FP32 && fmt != FORGE_MOM_BF16) return FORGE_ERR_FORMAT;
  const int ns = opt_states(static_cast<int>(opt));
  // the states the optimizer does not have are neither read nor checked
  forge_linear L[FORGE_MAX_GROUP];
  for (int i = 0; i < n; ++i) {
    L[i] = layers[i];
    if (ns < 1) L[i].m.data = nullptr;
    if (ns < 2) L[i].v.data = nullptr;
    L[i].m.scale = L[i].v.scale = nullptr;
    const forge_linear& a = L[i];
    s = check_shape(bt, a.d_in, a.d_out);
    if (s != FORGE_OK) return s;
    if (!a.W || (ns >= 1 && !a.m.data) || (ns >= 2 && !a.v.data)) return FORGE_ERR_NULL;
    if (bt > 0 && (!a.X || !a.dY)) return FORGE_ERR_NULL;
    if (!aligned16(a.W) || (a.m.data && !aligned16(a.m.data)) || (a.v.data && !aligned16(a.v.data)))
      return FORGE_ERR_ALIGN;
    if (bt > 0 && (!aligned16(a.X) || !aligned16(a.dY))) return FORGE_ERR_ALIGN;
    const uint64_t ne = static_cast<uint64_t>(a.d_in) * static_cast<uint64_t>(a.d_out);
    const uint64_t nm = ne * mom_elem_bytes(fmt);
    if (overlaps(a.W, 2 * ne, a.m.data, nm) || overlaps(a.W, 2 * ne, a.v.data, nm) ||
        overlaps(a.m.data, nm, a.v.data, nm))
      return FORGE_ERR_ALIAS;
  }
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j)
      if (layers_clash(L[i], L[j], bt, fmt, i == j)) return FORGE_ERR_ALIAS;
  DeviceInfo* d = nullptr;
  s = device_info(&d);
  if (s != FORGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the slots hold W and as many state boxes as the optimizer has
  const bool f32s = fmt == FORGE_MOM_FP32;
  const int ifmt = ns == 0 ? kFmtNone
                 : ns == 1 ? (f32s ? kFmtF32S1 : kFmtBF16S1)
                           : (f32s ? kFmtF32 : kFmtBF16);
  GemmConfig cfg = choose_opt_config(bt, ifmt, ns);
  const bool f32 = fmt == FORGE_MOM_FP32;
  const CUtensorMapDataType mdt =
      f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle msw = f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const int eb = f32 ? 4 : 2;
  const uint32_t rows = static_cast<uint32_t>(slot_rows(kModeOpt, ifmt, cfg.prof));
  int order[FORGE_MAX_GROUP];
  largest_first(L, n, fmt, order);
  GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  args.p = base_params(bt, cfg, *d);
  args.p.o = make_opt_consts(static_cast<int>(opt), *hyper, step);
  args.p.nstate = ns;
  for (int k = 0; k < n; ++k) {
    const forge_linear& a = L[order[k]];
    GemmMaps& maps = args.maps[k];
    bool ok = (bt == 0 || operand_maps(maps, a.X, a.dY, bt, a.d_in, a.d_out, bk_of(cfg.cg))) &&
              get_map(&maps.w, a.W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.d_in, a.d_out,
                      a.d_in * 2, 32, rows, CU_TENSOR_MAP_SWIZZLE_64B);
    if (ok && ns >= 1)
      ok = get_map(&maps.m, a.m.data, mdt, a.d_in, a.d_out, a.d_in * eb, 32, rows, msw);
    if (ok && ns >= 2)
      ok = get_map(&maps.v, a.v.data, mdt, a.d_in, a.d_out, a.d_in * eb, 32, rows, msw);
    if (!ok) return FORGE_ERR_LAUNCH;
    add_problem(args.p, cfg, a.d_in, a.d_out, nullptr, nullptr);
  }
  set_grid(cfg, args.p.num_units, d->num_sms);
  args.p.drop_first_arrival = take_drop_flag();
  return launch_gemm(kModeOpt, ifmt, cfg, args, st) == cudaSuccess ? FORGE_OK
                                                                      : FORGE_ERR_LAUNCH;
}

forge_status forge_wgrad_opt(const void* X, const void* dY, void* W, forge_moment s1,
                             forge_moment s2, int64_t bt, int64_t d_in, int64_t d_out,
                             forge_optimizer opt, const forge_opt_hyper* hyper, int64_t step,
                             forge_moment_fmt fmt, forge_stream stream) {
  forge_linear L;
  L.X = X;
  L.dY = dY;
  L.W = W;
  L.m = s1;
  L.v = s2;
  L.d_in = d_in;
  L.d_out = d_out;
  return forge_wgrad_opt_grouped(&L, 1, bt, opt, hyper, step, fmt, stream);
}

forge_status forge_dgrad_noalloc(const void* dY, const void* W, void* dX, int64_t bt,
                                 int64_t d_in, int64_t d_out, forge_stream stream) {
  const forge_dgrad_item it = dgrad_item(dY, W, dX, d_in, d_out);
  return dgrad_run(&it, 1, bt, kWsStatic, nullptr, 0, stream);
}

forge_status forge_linear_backward(const void* X, const void* dY, void* W, void* dX,
                                   forge_moment m, forge_moment v, int64_t bt, int64_t d_in,
                                   int64_t d_out, float lr, float beta1, float beta2, float eps,
                                   float weight_decay, int64_t step, forge_moment_fmt fmt,
                                   forge_stream stream) {
  // every argument of both halves is checked before anything is enqueued
  forge_linear L;
  L.X = X;
  L.dY = dY;
  L.W = W;
  L.m = m;
  L.v = v;
  L.d_in = d_in;
  L.d_out = d_out;
  forge_status s = check_linear(L, bt, fmt);
  if (s != FORGE_OK) return s;
  s = check_hyper(lr, beta1, beta2, eps, weight_decay, step);
  if (s != FORGE_OK) return s;
  if (layers_clash(L, L, bt, fmt, true)) return FORGE_ERR_ALIAS;
  if (bt > 0) {
    if (!dX) return FORGE_ERR_NULL;
    if (!aligned16(dX)) return FORGE_ERR_ALIGN;
    const uint64_t ndx = 2ull * bt * d_in;
    if (overlaps(dX, ndx, X, 2ull * bt * d_in) || overlaps(dX, ndx, dY, 2ull * bt * d_out) ||
        input_overlaps_state(dX, ndx, W, m, v, d_in, d_out, fmt))
      return FORGE_ERR_ALIAS;
  }
  // dX reads W before the fused step overwrites it (Algorithm 1): same stream
  s = forge_dgrad(dY, W, dX, bt, d_in, d_out, stream);
  if (s != FORGE_OK) return s;
  return forge_wgrad_adamw(X, dY, W, m, v, bt, d_in, d_out, lr, beta1, beta2, eps, weight_decay,
                           step, fmt, stream);
}

forge_status forge_linear_backward_grouped(const forge_linear* layers, void* const* dX, int n,
                                           int64_t bt, float lr, float beta1, float beta2,
                                           float eps, float weight_decay, int64_t step,
                                           forge_moment_fmt fmt, void* workspace,
                                           size_t workspace_bytes, forge_stream stream) {
  // every argument of both halves is checked before anything is enqueued
  if (!layers || !dX) return FORGE_ERR_NULL;
  if (n < 1 || n > FORGE_MAX_GROUP) return FORGE_ERR_SHAPE;
  for (int i = 0; i < n; ++i) {
    forge_status s = check_linear(layers[i], bt, fmt);
    if (s != FORGE_OK) return s;
  }
  forge_status s = check_hyper(lr, beta1, beta2, eps, weight_decay, step);
  if (s != FORGE_OK) return s;
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j)
      if (layers_clash(layers[i], layers[j], bt, fmt, i == j)) return FORGE_ERR_ALIAS;
  forge_dgrad_item items[FORGE_MAX_GROUP];
  for (int i = 0; i < n; ++i) {
    const forge_linear& L = layers[i];
    items[i] = dgrad_item(L.dY, L.W, dX[i], L.d_in, L.d_out);
    if (bt == 0) continue;
    if (!dX[i]) return FORGE_ERR_NULL;
    if (!aligned16(dX[i])) return FORGE_ERR_ALIGN;
    // no dX overlaps any layer's inputs, state or scales
    const uint64_t ndx = 2ull * bt * L.d_in;
    for (int j = 0; j < n; ++j) {
      const forge_linear& b = layers[j];
      if (overlaps(dX[i], ndx, b.X, 2ull * bt * b.d_in) ||
          input_overlaps_state(dX[i], ndx, b.W, b.m, b.v, b.d_in, b.d_out, fmt))
        return FORGE_ERR_ALIAS;
    }
  }
  if (workspace && !aligned16(workspace)) return FORGE_ERR_ALIGN;
  s = check_dgrad_items(items, n, bt);
  if (s != FORGE_OK) return s;
  // dX reads W before the fused step overwrites it (Algorithm 1): same stream
  s = dgrad_run(items, n, bt, kWsCaller, workspace, workspace_bytes, stream);
  if (s != FORGE_OK) return s;
  return forge_wgrad_adamw_grouped(layers, n, bt, lr, beta1, beta2, eps, weight_decay, step,
                                   fmt, stream);
}

forge_status forge_adamw(const void* dW, forge_dtype dw_dtype, void* W, forge_moment m,
                         forge_moment v, int64_t d_in, int64_t d_out, float lr, float beta1,
                         float beta2, float eps, float weight_decay, int64_t step,
                         forge_moment_fmt fmt, forge_stream stream) {
  forge_status s = check_shape(0, d_in, d_out);
  if (s != FORGE_OK) return s;
  if (dw_dtype != FORGE_DT_FP32 && dw_dtype != FORGE_DT_BF16) return FORGE_ERR_FORMAT;
  s = check_state(W, m, v, d_in, d_out, fmt);
  if (s != FORGE_OK) return s;
  if (dW && !aligned16(dW)) return FORGE_ERR_ALIGN;
  s = check_hyper(lr, beta1, beta2, eps, weight_decay, step);
  if (s != FORGE_OK) return s;
  const uint64_t nbytes =
      static_cast<uint64_t>(d_in) * d_out * (dw_dtype == FORGE_DT_FP32 ? 4 : 2);
  if (dW && input_overlaps_state(dW, nbytes, W, m, v, d_in, d_out, fmt)) return FORGE_ERR_ALIAS;
  DeviceInfo* d = nullptr;
  s = device_info(&d);
  if (s != FORGE_OK) return s;
  const AdamWConsts h = make_consts(lr, beta1, beta2, eps, weight_decay, step);
  return launch_adamw(dW, dw_dtype == FORGE_DT_FP32 ? 0 : 1, W, m.data, v.data, m.scale, v.scale,
                      d_in, d_out, static_cast<int>(fmt), h, d->num_sms,
                      static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FORGE_OK
             : FORGE_ERR_LAUNCH;
}

forge_status forge_device_error(forge_stream stream) {
  DeviceInfo* d = nullptr;
  forge_status s = device_info(&d);
  if (s != FORGE_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FORGE_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, d->err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FORGE_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(d->err_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return FORGE_ERR_CUDA;
    return static_cast<forge_status>(word);
  }
  return FORGE_OK;
}

const char* forge_status_string(forge_status status) {
  switch (status) {
    case FORGE_OK: return "FORGE_OK";
    case FORGE_ERR_NULL: return "FORGE_ERR_NULL: a required pointer is NULL";
    case FORGE_ERR_ALIGN: return "FORGE_ERR_ALIGN: a pointer is not 16-byte aligned";
    case FORGE_ERR_SHAPE: return "FORGE_ERR_SHAPE: unsupported shape";
    case FORGE_ERR_FORMAT: return "FORGE_ERR_FORMAT: unknown moment format or dtype";
    case FORGE_ERR_HYPER: return "FORGE_ERR_HYPER: hyperparameter out of range";
    case FORGE_ERR_ALIAS: return "FORGE_ERR_ALIAS: an input overlaps an output";
    case FORGE_ERR_ARCH: return "FORGE_ERR_ARCH: the current device is not sm_103";
    case FORGE_ERR_LAUNCH: return "FORGE_ERR_LAUNCH: kernel launch or descriptor encode failed";
    case FORGE_ERR_DEVICE_TIMEOUT:
      return "FORGE_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel ran out";
    case FORGE_ERR_CUDA: return "FORGE_ERR_CUDA: a CUDA runtime call failed";
    case FORGE_ERR_DEVICE_CONFIG:
      return "FORGE_ERR_DEVICE_CONFIG: a kernel found its shared-memory window unusable";
  }
  return "FORGE: unknown status";
}

int forge_describe_config(int64_t bt, int64_t d_in, int64_t d_out, forge_moment_fmt fmt, char* buf,
                          int len) {
  if (check_shape(bt, d_in, d_out) != FORGE_OK) return -1;
  if (!valid_fmt(fmt)) return -1;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      sms = n;
  }
  const int fm = static_cast<int>(fmt);
  GemmConfig c = choose_config(bt, fm, kModeFused);
  set_grid(c, tiles_of(c, d_in, d_out), sms);
  const int sw = slice_cols(kModeFused, fm);
  const int need = std::snprintf(buf, buf ? len : 0,
                                 "tile=%dx%d ctas=%d bk=%d slice=%d grid=%d group_m=%d threads=%d "
                                 "poll_store=%d profile=%s",
                                 kBM * c.cg, c.bn, c.cg, bk_of(c.cg), sw, c.grid, c.group_m, kNumThreads,
                                 c.poll_store,
                                 c.prof == kProfStream ? "stream"
                                 : c.prof == kProfMma  ? "mma"
                                 : c.prof == kProfDeep ? "deep"
                                                       : "balanced");
  return need + 1;
}

int forge_describe_dgrad_config(int64_t bt, int64_t d_in, int64_t d_out, char* buf, int len) {
  if (check_shape(bt, d_in, d_out) != FORGE_OK) return -1;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      sms = n;
  }
  GemmConfig c = choose_dgrad_config(bt, d_in, d_out, sms);
  const int64_t tiles = ((bt + kBM * c.cg - 1) / (kBM * c.cg)) * ((d_in + c.bn - 1) / c.bn);
  set_grid(c, tiles * c.splits, sms);
  const int need = std::snprintf(buf, buf ? len : 0,
                                 "tile=%dx%d ctas=%d bk=%d grid=%d splits=%d profile=%s",
                                 kBM * c.cg, c.bn, c.cg, bk_of(c.cg), c.grid, c.splits,
                                 c.prof == kProfStream ? "stream"
                                 : c.prof == kProfMma  ? "mma"
                                 : c.prof == kProfDeep ? "deep"
                                                       : "balanced");
  return need + 1;
}

int forge_debug_timeout_site(void) {
  DeviceInfo* d = nullptr;
  if (device_info(&d) != FORGE_OK) return -1;
  int word = 0;
  if (cudaMemcpy(&word, d->site_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return -1;
  const int zero = 0;
  if (cudaMemcpy(d->site_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return -1;
  return word;
}

void forge_set_wait_limit_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_wait_limit_ns = ns;
}

void forge_debug_drop_first_arrival(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_drop_first_arrival = enable ? 1 : 0;
}

forge_status forge_fp8_roll_scales(forge_fp8_scales* scales, int n, float headroom,
                                   forge_stream stream) {
  if (n < 0) return FORGE_ERR_SHAPE;
  if (n == 0) return FORGE_OK;
  if (!scales) return FORGE_ERR_NULL;
  if (!aligned16(scales)) return FORGE_ERR_ALIGN;
  if (!(headroom >= 1.0f) || !std::isfinite(headroom)) return FORGE_ERR_HYPER;
  DeviceInfo* d = nullptr;
  forge_status s = device_info(&d);
  if (s != FORGE_OK) return s;
  return launch_fp8_roll(reinterpret_cast<float*>(scales), n,
                         static_cast<int>(sizeof(forge_fp8_scales) / sizeof(float)), headroom,
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FORGE_OK
             : FORGE_ERR_LAUNCH;
}

void forge_set_tuning(const forge_tuning* t) {
  std::call_once(g_tune_once, tuning_from_env);   // a later first read must not undo this
  const forge_tuning automatic = {FORGE_PROFILE_AUTO, 0, 0, 0, -1, 0, -1, -1};
  std::lock_guard<std::mutex> lk(g_mu);
  g_tune = t ? *t : automatic;
}

void forge_get_tuning(forge_tuning* t) {
  if (t) *t = current_tuning();
}

}  // extern "C"
