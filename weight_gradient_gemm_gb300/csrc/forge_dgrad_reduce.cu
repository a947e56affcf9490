// The input gradient's split reduction.  When forge_dgrad cuts the reduction
// over d_out into k-ranges ("splits"), the tensor-core kernel writes one fp32
// partial tile per split and this kernel adds them:
//   dX[r][c] = bf16_rn( (((0 + P_0[r][c]) + P_1[r][c]) + ...) + P_{S-1}[r][c] )
// in split order, so the result does not depend on which split finished
// first, and it is rounded once.
//
// Partial layout (written by the kernel's epilogue): for CTA tile `ctile`
// (tile row, tile column, CTA of the pair) and split z, a 128 x BN fp32 block
// at float offset (ctile * splits + z) * 128 * BN, in which column slice cb
// (32 columns), half h and quarter j of a row's 16 columns form a run of 128
// float4, one per row, at float4 index ((cb * 2 + h) * 4 + j) * 128 + row.
#include <cuda_bf16.h>

#include "forge_internal.h"

namespace forge {
namespace {

constexpr int kRedThreads = 256;

// One block per 128-row x 32-column slice of a CTA tile (grid-stride): the
// splits' partials of the slice are read with contiguous whole-warp accesses
// (a warp covers 32 rows of one 4-column group), added in split order,
// rounded to bf16 and turned row-major through shared memory, so that dX is
// written in 64-byte row segments.
__global__ void __launch_bounds__(kRedThreads)
    dgrad_reduce_kernel(const float4* __restrict__ part, int splits, int cg, int bn,
                        int tiles_n, int64_t nslices, int64_t rows, int64_t d_in,
                        __nv_bfloat16* __restrict__ dX) {
  __shared__ uint32_t tile[kBM][17];   // 128 rows x 32 bf16 (16 words) + 1 word of padding
  constexpr int kSlice4 = kBM * 8;     // float4 per 32-column slice of a partial
  const int slices_per_tile = bn / 32;
  const int64_t part4 = static_cast<int64_t>(kBM) * bn / 4;   // float4 per partial
  for (int64_t sl = blockIdx.x; sl < nslices; sl += gridDim.x) {
    const int64_t ctile = sl / slices_per_tile;
    const int cb = static_cast<int>(sl % slices_per_tile);
    const float4* src = part + ctile * splits * part4 + cb * kSlice4;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int z = 0; z < splits; ++z) {
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __ldcs(src + z * part4 + threadIdx.x + kRedThreads * i);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i].x += v[i].x;
        acc[i].y += v[i].y;
        acc[i].z += v[i].z;
        acc[i].w += v[i].w;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int w = threadIdx.x + kRedThreads * i;   // (h * 4 + j) * 128 + row
      const int row = w & (kBM - 1);
      const int g = w >> 7;                          // 4-column group 0..7
      tile[row][2 * g] = pack_bf16x2(acc[i].x, acc[i].y);
      tile[row][2 * g + 1] = pack_bf16x2(acc[i].z, acc[i].w);
    }
    __syncthreads();
    const int64_t t = ctile / cg;
    const int rank = static_cast<int>(ctile % cg);
    const int64_t r0 = (t / tiles_n) * kBM * cg + rank * kBM;
    const int64_t c0 = (t % tiles_n) * bn + cb * 32;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int row = (threadIdx.x >> 2) + 64 * k;
      const int seg = threadIdx.x & 3;                // 8 bf16 (16 bytes) of the row
      const int64_t r = r0 + row;
      const int64_t c = c0 + seg * 8;
      if (r < rows && c < d_in)                       // d_in is a multiple of 8
        *reinterpret_cast<uint4*>(dX + r * d_in + c) =
            make_uint4(tile[row][4 * seg], tile[row][4 * seg + 1], tile[row][4 * seg + 2],
                       tile[row][4 * seg + 3]);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_dgrad_reduce(const float* part, int splits, int cg, int bn, int tiles_m,
                                int tiles_n, int64_t rows, int64_t d_in, void* dX, int num_sms,
                                cudaStream_t stream) {
  const int64_t nslices = static_cast<int64_t>(tiles_m) * tiles_n * cg * (bn / 32);
  const int64_t cap = 8LL * num_sms;
  const int grid = static_cast<int>(nslices < cap ? nslices : cap);
  if (grid <= 0) return cudaSuccess;
  dgrad_reduce_kernel<<<grid, kRedThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(part), splits, cg, bn, tiles_n, nslices, rows, d_in,
      static_cast<__nv_bfloat16*>(dX));
  return cudaGetLastError();
}

}  // namespace forge
