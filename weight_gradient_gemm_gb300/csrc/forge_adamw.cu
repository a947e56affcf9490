// The unfused optimizer step: AdamW on a stored gradient dW (fp32 or bf16, or
// none for a zero gradient), with the per-element arithmetic of the fused
// kernel's epilogue (forge_math.cuh).  This is the second kernel of the
// two-kernel path the FORGE page compares against ("cuBLAS + FORGE optimizer
// kernel", Appendix E; "store-G control" plus update, Appendix D).
//
// An HBM-streaming kernel: grid-stride over 16-byte vectors, loads and stores
// marked streaming (each byte is touched once).
#include <cuda_bf16.h>

#include "forge_internal.h"

namespace forge {

// dW formats: 0 fp32, 1 bf16, 2 no gradient (zero).
template <int DW>
__device__ __forceinline__ void load_grad8(const void* dW, int64_t i8, float (&g)[8]) {
  if constexpr (DW == 0) {
    const float4* p = reinterpret_cast<const float4*>(dW) + 2 * i8;
    const float4 a = __ldcs(p), b = __ldcs(p + 1);
    g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
    g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
  } else if constexpr (DW == 1) {
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(dW) + i8);
    const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) { g[2 * k] = bf16_lo(u[k]); g[2 * k + 1] = bf16_hi(u[k]); }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) g[k] = 0.0f;
  }
}

// fp32 or bf16 moments: one thread per 8 consecutive elements.
template <int FMT, int DW>
__global__ void __launch_bounds__(256) adamw_vec8_kernel(const void* __restrict__ dW,
                                                         uint16_t* __restrict__ W,
                                                         void* __restrict__ m,
                                                         void* __restrict__ v, int64_t n8,
                                                         const AdamWConsts h) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += stride) {
    float g[8], w[8], mm[8], vv[8];
    load_grad8<DW>(dW, i, g);
    uint4* wp = reinterpret_cast<uint4*>(W) + i;
    const uint4 wq = __ldcs(wp);
    const uint32_t wu[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) { w[2 * k] = bf16_lo(wu[k]); w[2 * k + 1] = bf16_hi(wu[k]); }
    if constexpr (FMT == kFmtF32) {
      float4* mp = reinterpret_cast<float4*>(m) + 2 * i;
      float4* vp = reinterpret_cast<float4*>(v) + 2 * i;
      const float4 m0 = __ldcs(mp), m1 = __ldcs(mp + 1), v0 = __ldcs(vp), v1 = __ldcs(vp + 1);
      mm[0] = m0.x; mm[1] = m0.y; mm[2] = m0.z; mm[3] = m0.w;
      mm[4] = m1.x; mm[5] = m1.y; mm[6] = m1.z; mm[7] = m1.w;
      vv[0] = v0.x; vv[1] = v0.y; vv[2] = v0.z; vv[3] = v0.w;
      vv[4] = v1.x; vv[5] = v1.y; vv[6] = v1.z; vv[7] = v1.w;
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        float2 w2 = make_float2(w[k], w[k + 1]), m2 = make_float2(mm[k], mm[k + 1]);
        float2 v2 = make_float2(vv[k], vv[k + 1]), r2;
        adamw_elem2(make_float2(g[k], g[k + 1]), w2, m2, v2, r2, h);
        w[k] = w2.x; w[k + 1] = w2.y;
        mm[k] = m2.x; mm[k + 1] = m2.y;
        vv[k] = v2.x; vv[k + 1] = v2.y;
      }
      __stcs(mp, make_float4(mm[0], mm[1], mm[2], mm[3]));
      __stcs(mp + 1, make_float4(mm[4], mm[5], mm[6], mm[7]));
      __stcs(vp, make_float4(vv[0], vv[1], vv[2], vv[3]));
      __stcs(vp + 1, make_float4(vv[4], vv[5], vv[6], vv[7]));
    } else {
      uint4* mp = reinterpret_cast<uint4*>(m) + i;
      uint4* vp = reinterpret_cast<uint4*>(v) + i;
      const uint4 mq = __ldcs(mp), vq = __ldcs(vp);
      const uint32_t mu[4] = {mq.x, mq.y, mq.z, mq.w};
      const uint32_t vu[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mm[2 * k] = bf16_lo(mu[k]); mm[2 * k + 1] = bf16_hi(mu[k]);
        vv[2 * k] = bf16_lo(vu[k]); vv[2 * k + 1] = bf16_hi(vu[k]);
      }
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        float2 w2 = make_float2(w[k], w[k + 1]), m2 = make_float2(mm[k], mm[k + 1]);
        float2 v2 = make_float2(vv[k], vv[k + 1]), r2;
        adamw_elem2(make_float2(g[k], g[k + 1]), w2, m2, v2, r2, h);
        w[k] = w2.x; w[k + 1] = w2.y;
        mm[k] = m2.x; mm[k + 1] = m2.y;
        vv[k] = v2.x; vv[k + 1] = v2.y;
      }
      __stcs(mp, make_uint4(pack_bf16x2(mm[0], mm[1]), pack_bf16x2(mm[2], mm[3]),
                            pack_bf16x2(mm[4], mm[5]), pack_bf16x2(mm[6], mm[7])));
      __stcs(vp, make_uint4(pack_bf16x2(vv[0], vv[1]), pack_bf16x2(vv[2], vv[3]),
                            pack_bf16x2(vv[4], vv[5]), pack_bf16x2(vv[6], vv[7])));
    }
    __stcs(wp, make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                          pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7])));
  }
}

// int8 moments: one warp per 128-column block of one row; lane l owns
// columns 4l..4l+3.  The block absmax is a warp max.
template <int DW>
__global__ void __launch_bounds__(256) adamw_int8_kernel(const void* __restrict__ dW,
                                                         uint16_t* __restrict__ W,
                                                         int8_t* __restrict__ mq,
                                                         int8_t* __restrict__ vq,
                                                         float* __restrict__ m_scale,
                                                         float* __restrict__ v_scale,
                                                         int64_t nblocks, const AdamWConsts h) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       b < nblocks; b += warps) {
    const int64_t e0 = b * 128 + 4 * lane;   // first element of this lane
    float g[4], w[4], mm[4], rr[4];
    if constexpr (DW == 0) {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(dW) + e0 / 4);
      g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
    } else if constexpr (DW == 1) {
      const uint2 a = __ldcs(reinterpret_cast<const uint2*>(dW) + e0 / 4);
      g[0] = bf16_lo(a.x); g[1] = bf16_hi(a.x); g[2] = bf16_lo(a.y); g[3] = bf16_hi(a.y);
    } else {
      g[0] = g[1] = g[2] = g[3] = 0.0f;
    }
    uint2* wp = reinterpret_cast<uint2*>(W) + e0 / 4;
    const uint2 wv = __ldcs(wp);
    w[0] = bf16_lo(wv.x); w[1] = bf16_hi(wv.x); w[2] = bf16_lo(wv.y); w[3] = bf16_hi(wv.y);
    uint32_t* mp = reinterpret_cast<uint32_t*>(mq) + e0 / 4;
    uint32_t* vp = reinterpret_cast<uint32_t*>(vq) + e0 / 4;
    const uint32_t mc = __ldcs(mp), vc = __ldcs(vp);
    const float2 sm = dup2(m_scale[b]), sv = dup2(v_scale[b]);
    float amax_m = 0.0f, amax_r = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; k += 2) {
      float2 w2 = make_float2(w[k], w[k + 1]);
      float2 m2 = dequant_m2(i8_code_pair(mc ^ 0x80808080u, k), sm);
      float2 v2 = dequant_v2(i8_code_pair(vc ^ 0x80808080u, k), sv), r2;
      adamw_elem2(make_float2(g[k], g[k + 1]), w2, m2, v2, r2, h);
      w[k] = w2.x; w[k + 1] = w2.y;
      mm[k] = m2.x; mm[k + 1] = m2.y;
      rr[k] = r2.x; rr[k + 1] = r2.y;
      amax_m = max3_abs(amax_m, mm[k], mm[k + 1]);
      amax_r = max3(amax_r, rr[k], rr[k + 1]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      amax_m = fmaxf(amax_m, __shfl_xor_sync(0xffffffffu, amax_m, o));
      amax_r = fmaxf(amax_r, __shfl_xor_sync(0xffffffffu, amax_r, o));
    }
    const float inv_m = int8_inv_step(amax_m), inv_r = int8_inv_step(amax_r);
    const float r_floor = amax_r > 0.0f ? 1.0f : 0.0f;
    const uint32_t mo = pack_low_bytes4(quant_m_bits(mm[0], inv_m), quant_m_bits(mm[1], inv_m),
                                        quant_m_bits(mm[2], inv_m), quant_m_bits(mm[3], inv_m));
    const uint32_t vo =
        pack_low_bytes4(quant_r_bits(rr[0], inv_r, r_floor), quant_r_bits(rr[1], inv_r, r_floor),
                        quant_r_bits(rr[2], inv_r, r_floor), quant_r_bits(rr[3], inv_r, r_floor));
    __stcs(mp, mo);
    __stcs(vp, vo);
    __stcs(wp, make_uint2(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3])));
    if (lane == 0) {
      m_scale[b] = int8_scale(amax_m);
      v_scale[b] = int8_scale(amax_r);
    }
  }
}

// fp8 moments with per-tensor scales: one thread per 16 consecutive
// elements, the same per-element arithmetic and encoding as the fused
// kernel's fp8 epilogue; each warp raises the tensors' amax words once.
template <int DW>
__global__ void __launch_bounds__(256) adamw_fp8_kernel(const void* __restrict__ dW,
                                                        uint16_t* __restrict__ W,
                                                        uint8_t* __restrict__ mq,
                                                        uint8_t* __restrict__ rq,
                                                        float* __restrict__ m_words,
                                                        float* __restrict__ r_words,
                                                        int64_t n16, const AdamWConsts h) {
  const Fp8Step fm = fp8_step_of(m_words), fr = fp8_step_of(r_words);
  float amax_m = 0.0f, amax_r = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride) {
    float g[16], w[16], ga[8], gb[8];
    load_grad8<DW>(dW, 2 * i, ga);
    load_grad8<DW>(dW, 2 * i + 1, gb);
#pragma unroll
    for (int k = 0; k < 8; ++k) { g[k] = ga[k]; g[8 + k] = gb[k]; }
    uint4* wp = reinterpret_cast<uint4*>(W) + 2 * i;
    const uint4 w0 = __ldcs(wp), w1 = __ldcs(wp + 1);
    const uint32_t wu[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) { w[2 * k] = bf16_lo(wu[k]); w[2 * k + 1] = bf16_hi(wu[k]); }
    uint4* mp = reinterpret_cast<uint4*>(mq) + i;
    uint4* rp = reinterpret_cast<uint4*>(rq) + i;
    uint4 mc = __ldcs(mp), rc = __ldcs(rp);
    adamw_fp8_x16(g, w, mc, rc, fm, fr, h, amax_m, amax_r);
    __stcs(mp, mc);
    __stcs(rp, rc);
    __stcs(wp, make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                          pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7])));
    __stcs(wp + 1, make_uint4(pack_bf16x2(w[8], w[9]), pack_bf16x2(w[10], w[11]),
                              pack_bf16x2(w[12], w[13]), pack_bf16x2(w[14], w[15])));
  }
  const int lane = threadIdx.x & 31;
  warp_raise_amax(m_words + kFp8Amax, amax_m, lane);
  warp_raise_amax(r_words + kFp8Amax, amax_r, lane);
}

// The scale roll between steps for n fp8 moment tensors (four words each,
// `stride` floats apart): read <- write; write <- amax * headroom / 448
// when amax > 0; amax <- 0.
__global__ void fp8_roll_kernel(float* words, int n, int stride, float headroom) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float* w = words + static_cast<int64_t>(i) * stride;
  const float amax = w[kFp8Amax];
  const float write = w[kFp8WriteScale];
  w[kFp8ReadScale] = write;
  if (amax > 0.0f) w[kFp8WriteScale] = __fdiv_rn(__fmul_rn(amax, headroom), kE4m3Max);
  w[kFp8Amax] = 0.0f;
}

cudaError_t launch_fp8_roll(float* words, int n, int stride, float headroom,
                            cudaStream_t stream) {
  fp8_roll_kernel<<<(n + 127) / 128, 128, 0, stream>>>(words, n, stride, headroom);
  return cudaGetLastError();
}

template <int FMT, int DW>
static cudaError_t launch_vec8(const void* dW, void* W, void* m, void* v, int64_t n, int grid,
                               const AdamWConsts& h, cudaStream_t stream) {
  adamw_vec8_kernel<FMT, DW><<<grid, 256, 0, stream>>>(dW, static_cast<uint16_t*>(W), m, v, n / 8,
                                                      h);
  return cudaGetLastError();
}

template <int DW>
static cudaError_t launch_i8(const void* dW, void* W, void* m, void* v, float* ms, float* vs,
                             int64_t n, int grid, const AdamWConsts& h, cudaStream_t stream) {
  adamw_int8_kernel<DW><<<grid, 256, 0, stream>>>(dW, static_cast<uint16_t*>(W),
                                                 static_cast<int8_t*>(m), static_cast<int8_t*>(v),
                                                 ms, vs, n / 128, h);
  return cudaGetLastError();
}

cudaError_t launch_adamw(const void* dW, int dw_fmt, void* W, void* m, void* v, float* m_scale,
                         float* v_scale, int64_t d_in, int64_t d_out, int fmt,
                         const AdamWConsts& h, int num_sms, cudaStream_t stream) {
  const int64_t n = d_in * d_out;
  const int dw = dW == nullptr ? 2 : dw_fmt;
  if (fmt == kFmtF8) {   // n is a multiple of 64 (d_in, d_out multiples of 8)
    const int64_t n16 = n / 16;
    const int64_t want = (n16 + 255) / 256;
    const int grid = static_cast<int>(want < 8LL * num_sms ? (want > 0 ? want : 1) : 8LL * num_sms);
    auto* Wp = static_cast<uint16_t*>(W);
    auto* mp = static_cast<uint8_t*>(m);
    auto* vp = static_cast<uint8_t*>(v);
    switch (dw) {
      case 0: adamw_fp8_kernel<0><<<grid, 256, 0, stream>>>(dW, Wp, mp, vp, m_scale, v_scale, n16, h); break;
      case 1: adamw_fp8_kernel<1><<<grid, 256, 0, stream>>>(dW, Wp, mp, vp, m_scale, v_scale, n16, h); break;
      default: adamw_fp8_kernel<2><<<grid, 256, 0, stream>>>(dW, Wp, mp, vp, m_scale, v_scale, n16, h); break;
    }
    return cudaGetLastError();
  }
  if (fmt == kFmtI8) {
    const int64_t nb = n / 128;
    const int64_t want = (nb + 7) / 8;
    const int grid = static_cast<int>(want < 8LL * num_sms ? (want > 0 ? want : 1) : 8LL * num_sms);
    switch (dw) {
      case 0: return launch_i8<0>(dW, W, m, v, m_scale, v_scale, n, grid, h, stream);
      case 1: return launch_i8<1>(dW, W, m, v, m_scale, v_scale, n, grid, h, stream);
      default: return launch_i8<2>(dW, W, m, v, m_scale, v_scale, n, grid, h, stream);
    }
  }
  const int64_t n8 = n / 8;
  const int64_t want = (n8 + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * num_sms ? (want > 0 ? want : 1) : 8LL * num_sms);
  if (fmt == kFmtF32) {
    switch (dw) {
      case 0: return launch_vec8<kFmtF32, 0>(dW, W, m, v, n, grid, h, stream);
      case 1: return launch_vec8<kFmtF32, 1>(dW, W, m, v, n, grid, h, stream);
      default: return launch_vec8<kFmtF32, 2>(dW, W, m, v, n, grid, h, stream);
    }
  }
  switch (dw) {
    case 0: return launch_vec8<kFmtBF16, 0>(dW, W, m, v, n, grid, h, stream);
    case 1: return launch_vec8<kFmtBF16, 1>(dW, W, m, v, n, grid, h, stream);
    default: return launch_vec8<kFmtBF16, 2>(dW, W, m, v, n, grid, h, stream);
  }
}

}  // namespace forge
