// Instantiates the tensor-core kernel for the fused step at the final
// micro-batch of the exact-accumulation mode with fp32 moments: every state
// slot also holds the fp32 accumulator's box, which the epilogue adds to the
// tile's gradient before AdamW.
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_fused_f32a(const GemmConfig& cfg, const GemmArgs& args,
                                  cudaStream_t stream) {
  return launch_gemm_fmt<kModeFused, kFmtF32A>(cfg, args, stream);
}

}  // namespace forge
