// Per-element optimizer arithmetic shared by the fused kernel's epilogue and
// the unfused AdamW kernel.  Both call exactly these functions, so for the
// same fp32 gradient they produce the same bits (the FORGE page, Appendix A,
// "Floating-point characterization").  Every operation is an explicit
// round-to-nearest intrinsic, so the compiler cannot contract or reorder it
// differently in the two call sites.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace forge {

// AdamW constants for one step (Algorithm 1), prepared on the host in fp64
// and rounded once to fp32.
struct AdamWConsts {
  float beta1, beta2;
  float omb1, omb2;        // 1 - beta1, 1 - beta2
  float eps;
  float decay;             // 1 - lr * wd
  float neg_step_size;     // -lr / (1 - beta1^t)
  float inv_sqrt_bc2;      // 1 / sqrt(1 - beta2^t)
};

// Square root and reciprocal on the special-function unit (PTX sqrt.approx /
// rcp.approx: relative error about 2^-23).  The update they feed is added to
// a weight rounded to bf16 (2^-8 relative), so their error is far below what
// the stored result can show; the moments themselves use only exact-rounded
// multiply-adds.
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// The reciprocal flushes subnormal inputs and results (.ftz), which skips the
// subnormal handling of the plain form.  Every denominator it is given is
// sqrt(.) * c + eps or sqrt(.) + eps with c in [1, 2^12] (c = 1/sqrt(1 -
// beta2^t), beta2 < 1 in fp32), sqrt(.) below 2^64 and eps either 0 or a
// normal number at most 2^64 (the host rejects other eps): so the input is
// 0, infinite, NaN or normal and below 2^77, the result is never subnormal,
// and the flush never changes a bit.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One AdamW element.  In: g (fp32 gradient), w, m, v.  Out: w', m', v' and
// r' = sqrt(v').  The weight update reads the unrounded m' and v'.
//   m' = beta1 m + (1-beta1) g
//   v' = beta2 v + (1-beta2) g^2
//   w' = (1 - lr wd) w - (lr/bc1) m' / (sqrt(v') / sqrt(bc2) + eps)
__device__ __forceinline__ void adamw_elem(float g, float& w, float& m, float& v, float& r,
                                           const AdamWConsts& c) {
  const float m1 = __fmaf_rn(c.beta1, m, __fmul_rn(c.omb1, g));
  const float v1 = __fmaf_rn(c.beta2, v, __fmul_rn(c.omb2, __fmul_rn(g, g)));
  const float r1 = sqrt_approx(v1);
  const float denom = __fmaf_rn(r1, c.inv_sqrt_bc2, c.eps);
  const float upd = __fmul_rn(m1, rcp_approx(denom));
  w = __fmaf_rn(c.neg_step_size, upd, __fmul_rn(w, c.decay));
  m = m1;
  v = v1;
  r = r1;
}

// Paired fp32 arithmetic (PTX mul/add/fma .rn.f32x2, sm_100 and later): each
// lane is an IEEE round-to-nearest multiply, add or fused multiply-add, so the
// results are those of __fmul_rn / __fadd_rn / __fmaf_rn bit for bit, in half
// the instructions.  Unlike the scalar forms with an explicit rounding, a
// paired multiply whose result feeds a paired add was measured to come out
// as one fused multiply-add (a single rounding; 30 of 16.8 M int8 codes
// differed by one level from the scalar pair); so no paired multiply here
// feeds an add: where that arithmetic is wanted it is an explicit fma2.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }

// max(a, b, c) and max(|a|, |b|, |c|) in one instruction (three-input PTX
// max, sm_100 and later).  Like fmaxf, a NaN input is ignored when another
// input is a number.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// adamw_elem on two elements at once: the same operations in the same order
// on each lane (paired multiplies and multiply-adds), so each lane's results
// equal adamw_elem's bit for bit.
__device__ __forceinline__ void adamw_elem2(float2 g, float2& w, float2& m, float2& v,
                                            float2& r, const AdamWConsts& c) {
  const float2 m1 = fma2(dup2(c.beta1), m, mul2(dup2(c.omb1), g));
  const float2 v1 = fma2(dup2(c.beta2), v, mul2(dup2(c.omb2), mul2(g, g)));
  const float2 r1 = make_float2(sqrt_approx(v1.x), sqrt_approx(v1.y));
  const float2 den = fma2(r1, dup2(c.inv_sqrt_bc2), dup2(c.eps));
  const float2 upd = mul2(m1, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
  w = fma2(dup2(c.neg_step_size), upd, mul2(w, dup2(c.decay)));
  m = m1;
  v = v1;
  r = r1;
}

// ---------------------------------------------------------------------------
// The other coordinate-wise optimizers FORGE fuses (the page's regime 1):
// SGD, SGD with momentum, Adagrad and RMSprop (PyTorch's definitions with
// default options: L2 decay through the gradient, g = G + wd W), Lion (Chen et
// al.: sign update, decoupled decay), NAdam and RAdam (PyTorch's definitions).
// ---------------------------------------------------------------------------
enum OptKind : int {
  kOptSgd = 0, kOptSgdMomentum = 1, kOptAdagrad = 2, kOptRmsprop = 3, kOptLion = 4,
  kOptNadam = 5, kOptRadam = 6
};
// per-coordinate state tensors: none; the momentum buffer, Adagrad's sum,
// RMSprop's average or Lion's m; NAdam's and RAdam's m and v
__host__ __device__ constexpr int opt_states(int opt) {
  return opt == kOptSgd ? 0 : (opt >= kOptNadam ? 2 : 1);
}

// Per-step constants, formed in fp64 on the host and rounded once to fp32.
struct OptConsts {
  int32_t opt;           // OptKind
  int32_t rect;          // RAdam: the variance rectification applies at this step
  float lr, wd;          // learning rate; weight decay (L2: g = G + wd W)
  float a, oma;          // momentum | RMSprop alpha | beta1, and 1 - that
  float b, omb;          // beta2, 1 - beta2
  float eps;
  float k1, k2;          // NAdam: -lr (1 - mu_t) / (1 - P_t), -lr mu_{t+1} / (1 - P_t mu_{t+1});
                         // RAdam: -lr r_t sqrt(1 - beta2^t) / (1 - beta1^t) (rectified)
                         //        or -lr / (1 - beta1^t)
  float inv_sqrt_bc2;    // NAdam: 1 / sqrt(1 - beta2^t)
  float decay;           // Lion: 1 - lr wd
};

// One element of optimizer OPT: G from the accumulator, the weight w and the
// states s1, s2 (fp32, updated in place; unused ones are left alone).
template <int OPT>
__device__ __forceinline__ void opt_elem(float G, float& w, float& s1, float& s2,
                                         const OptConsts& c) {
  if constexpr (OPT == kOptLion) {
    const float dir = __fmaf_rn(c.a, s1, __fmul_rn(c.oma, G));
    const float sg = dir > 0.0f ? 1.0f : (dir < 0.0f ? -1.0f : 0.0f);
    w = __fmaf_rn(-c.lr, sg, __fmul_rn(w, c.decay));
    s1 = __fmaf_rn(c.b, s1, __fmul_rn(c.omb, G));
  } else {
    const float g = __fmaf_rn(c.wd, w, G);
    if constexpr (OPT == kOptSgd) {
      w = __fmaf_rn(-c.lr, g, w);
    } else if constexpr (OPT == kOptSgdMomentum) {
      s1 = __fmaf_rn(c.a, s1, g);
      w = __fmaf_rn(-c.lr, s1, w);
    } else if constexpr (OPT == kOptAdagrad || OPT == kOptRmsprop) {
      s1 = (OPT == kOptAdagrad) ? __fmaf_rn(g, g, s1)
                                : __fmaf_rn(c.a, s1, __fmul_rn(c.oma, __fmul_rn(g, g)));
      const float d = __fadd_rn(sqrt_approx(s1), c.eps);
      w = __fmaf_rn(-c.lr, __fmul_rn(g, rcp_approx(d)), w);
    } else {   // NAdam, RAdam
      const float m = __fmaf_rn(c.a, s1, __fmul_rn(c.oma, g));
      const float v = __fmaf_rn(c.b, s2, __fmul_rn(c.omb, __fmul_rn(g, g)));
      if constexpr (OPT == kOptNadam) {
        const float d = __fmaf_rn(sqrt_approx(v), c.inv_sqrt_bc2, c.eps);
        w = __fmaf_rn(__fmaf_rn(c.k1, g, __fmul_rn(c.k2, m)), rcp_approx(d), w);
      } else if (c.rect) {
        const float d = __fadd_rn(sqrt_approx(v), c.eps);
        w = __fmaf_rn(c.k1, __fmul_rn(m, rcp_approx(d)), w);
      } else {
        w = __fmaf_rn(c.k1, m, w);
      }
      s1 = m;
      s2 = v;
    }
  }
}

// ---------------------------------------------------------------------------
// Stochastic-rounding store of the bf16 weight (the page's SR-store recipe,
// Gupta et al.): the random bits come from Philox4x64-10 (Salmon, Moraes,
// Dror, Shaw 2011), one block of 4 x 64 bits per 16 weights.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t hi0 = __umul64hi(kM0, c[0]), lo0 = kM0 * c[0];
    const uint64_t hi1 = __umul64hi(kM1, c[2]), lo1 = kM1 * c[2];
    const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// fp32 -> bf16 bit pattern by stochastic rounding with a uniform 16-bit r:
// r is added to the low 16 bits of the magnitude and the upper 16 kept, so
// the magnitude rounds up with probability (dropped bits) / 2^16; past the
// largest finite value it becomes infinity.  NaN and infinity pass through.
__device__ __forceinline__ uint32_t sr_bf16_bits(float x, uint32_t r16) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t mag = b & 0x7FFFFFFFu, sign = (b >> 16) & 0x8000u;
  if (mag >= 0x7F800000u) return (mag > 0x7F800000u ? 0x7FC0u : 0x7F80u) | sign;
  const uint32_t up = (mag + r16) >> 16;   // mag + r16 < 2^32
  return (up > 0x7F80u ? 0x7F80u : up) | sign;
}

// bf16 <-> fp32 (round to nearest even on the way down).
__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) {
  return __uint_as_float(packed & 0xFFFF0000u);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Blockwise absmax int8 (128 columns of one row per block).
//   scale s = a / 127; code = round(x / s) computed as round(x * (127 / a)),
//   ties to even, in [-127, 127].  The second moment is stored as r = sqrt(v)
//   with codes of at least 1 in a block whose absmax is non-zero.
__device__ __forceinline__ float int8_scale(float absmax) { return __fdiv_rn(absmax, 127.0f); }
__device__ __forceinline__ float int8_inv_step(float absmax) {
  return absmax > 0.0f ? __fdiv_rn(127.0f, absmax) : 0.0f;
}
// Codes without conversion instructions.  y = x * (127 / a) with |x| <= a
// (a the block's absmax of the same fp32 values) satisfies |y| < 127.0001,
// so round(y) is already in [-127, 127].  One fused multiply-add forms
// x * inv + 1.5 * 2^23 with a single rounding to the nearest integer (ties to
// even), which leaves round(x * inv) in the low bits of the sum: the low
// byte of its bit pattern is the two's-complement code.  (The product is not
// rounded on its own first: the code is the integer nearest to the exact
// x * inv, inv = 127 / a rounded to fp32.)  The second moment's floor of one
// level in a non-zero block is a max after rounding: max(round(y), 1) equals
// round(max(y, 1)) for y >= 0.
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23
__device__ __forceinline__ uint32_t quant_m_bits(float x, float inv) {
  return __float_as_uint(__fmaf_rn(x, inv, kRoundMagic));
}
__device__ __forceinline__ uint32_t quant_r_bits(float r, float inv, float floor_level) {
  return __float_as_uint(fmaxf(__fmaf_rn(r, inv, kRoundMagic), kRoundMagic + floor_level));
}
// The low bytes of four words, in order, as one word of four codes.
__device__ __forceinline__ uint32_t pack_low_bytes4(uint32_t a, uint32_t b, uint32_t c,
                                                    uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}
// Codes k and k + 1 (k = 0 or 2) of a word of four int8 codes, as floats:
// with the word's bytes offset by 128 (w ^ 0x80808080), 2^23 + (code + 128)
// is assembled by a byte permute and 2^23 + 128 subtracted exactly (one
// paired add).
__device__ __forceinline__ float2 i8_code_pair(uint32_t w_offset, int k) {
  const float2 biased =
      make_float2(__uint_as_float(__byte_perm(w_offset, 0x4B000000u, 0x7540u | k)),
                  __uint_as_float(__byte_perm(w_offset, 0x4B000000u, 0x7540u | (k + 1))));
  return add2(biased, dup2(-8388736.0f));
}
// quant_m_bits / quant_r_bits on two values with one paired multiply-add.
__device__ __forceinline__ void quant_m_bits2(float2 x, float2 inv, uint32_t& b0, uint32_t& b1) {
  const float2 q = fma2(x, inv, dup2(kRoundMagic));
  b0 = __float_as_uint(q.x);
  b1 = __float_as_uint(q.y);
}
__device__ __forceinline__ void quant_r_bits2(float2 r, float2 inv, float floor_level,
                                              uint32_t& b0, uint32_t& b1) {
  const float2 q = fma2(r, inv, dup2(kRoundMagic));
  const float lo = kRoundMagic + floor_level;
  b0 = __float_as_uint(fmaxf(q.x, lo));
  b1 = __float_as_uint(fmaxf(q.y, lo));
}

// Decoded int8 values (two codes as floats): m = code * s; v = (code * s)^2.
__device__ __forceinline__ float2 dequant_m2(float2 code, float2 s) { return mul2(code, s); }
__device__ __forceinline__ float2 dequant_v2(float2 code, float2 s) {
  const float2 r = mul2(code, s);
  return mul2(r, r);
}

// ---------------------------------------------------------------------------
// fp8 moments (e4m3, the OCP "fn" variant: bias 7, largest finite 448, no
// infinities) with one scale per tensor and delayed scaling.  Per tensor the
// caller keeps four fp32 words in device memory: the scale the stored codes
// are read with, the scale the new codes are written with, and the amax of
// the new moments (max |m'|, or max sqrt(v') for the second moment, whose
// codes hold r = sqrt(v)), which a step raises and the caller resets.
// ---------------------------------------------------------------------------
constexpr int kFp8ReadScale = 0, kFp8WriteScale = 1, kFp8Amax = 2;
constexpr float kE4m3Max = 448.0f;

// Two e4m3 codes (low byte first) to two floats: exact (e4m3 -> f16 -> f32).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t codes16) {
  uint32_t h2;
  const uint16_t c = static_cast<uint16_t>(codes16);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  __half2 hh;
  *reinterpret_cast<uint32_t*>(&hh) = h2;
  return __half22float2(hh);
}
// Two floats to two e4m3 codes (lo in the low byte): round to nearest even,
// saturating at +-448.
__device__ __forceinline__ uint32_t float2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The per-tensor constants of one fp8 moment for a step.
struct Fp8Step {
  float read;      // decode: value = e4m3(code) * read
  float inv_write; // encode: code = e4m3(value * inv_write), 1 / write rounded to fp32
};
__device__ __forceinline__ Fp8Step fp8_step_of(const float* words) {
  Fp8Step f;
  f.read = __ldg(words + kFp8ReadScale);
  f.inv_write = __frcp_rn(__ldg(words + kFp8WriteScale));
  return f;
}

// 16 fp8 AdamW elements: codes of m and r = sqrt(v) (one uint4 each, 16
// codes, element i in byte i), w and g as floats.  Updates w; returns the
// new codes and raises the running amaxes.
__device__ __forceinline__ void adamw_fp8_x16(const float (&g)[16], float (&w)[16], uint4& mq,
                                              uint4& rq, const Fp8Step& fm, const Fp8Step& fr,
                                              const AdamWConsts& h, float& amax_m, float& amax_r) {
  uint32_t mw[4] = {mq.x, mq.y, mq.z, mq.w};
  uint32_t rw[4] = {rq.x, rq.y, rq.z, rq.w};
  uint32_t mo[4], ro[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t mpack = 0, rpack = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const float2 m2 = e4m3x2_to_float2(mw[k] >> (16 * half));
      const float2 r2 = e4m3x2_to_float2(rw[k] >> (16 * half));
      const int i = 4 * k + 2 * half;
      float2 mm = mul2(m2, dup2(fm.read));
      const float2 q = mul2(r2, dup2(fr.read));
      float2 vv = mul2(q, q);
      float2 ww = make_float2(w[i], w[i + 1]), rr;
      adamw_elem2(make_float2(g[i], g[i + 1]), ww, mm, vv, rr, h);
      w[i] = ww.x;
      w[i + 1] = ww.y;
      amax_m = max3_abs(amax_m, mm.x, mm.y);
      amax_r = max3(amax_r, rr.x, rr.y);
      const float2 me = mul2(mm, dup2(fm.inv_write));
      const float2 re = mul2(rr, dup2(fr.inv_write));
      mpack |= float2_to_e4m3x2(me.x, me.y) << (16 * half);
      rpack |= float2_to_e4m3x2(re.x, re.y) << (16 * half);
    }
    mo[k] = mpack;
    ro[k] = rpack;
  }
  mq = make_uint4(mo[0], mo[1], mo[2], mo[3]);
  rq = make_uint4(ro[0], ro[1], ro[2], ro[3]);
}

// Raise *word (an fp32 amax, >= 0) to at least the warp's largest x (>= 0):
// non-negative floats order like their bit patterns.  Warp-collective.
__device__ __forceinline__ void warp_raise_amax(float* word, float x, int lane) {
  const unsigned u = __reduce_max_sync(0xffffffffu, __float_as_uint(x));
  if (lane == 0 && u != 0u) atomicMax(reinterpret_cast<unsigned int*>(word), u);
}

}  // namespace forge
