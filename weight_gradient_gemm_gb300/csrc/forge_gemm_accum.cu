// Instantiates the tensor-core kernel in its accumulate mode (B' = beta B + G
// into an fp32 buffer); one translation unit so it compiles in parallel.
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_accum(const GemmConfig& cfg, const GemmArgs& args, cudaStream_t stream) {
  return launch_gemm_fmt<kModeAccum, kFmtF32>(cfg, args, stream);
}

}  // namespace forge
