// Instantiates the tensor-core weight-gradient kernel for one mode and format
// (one translation unit each, so they compile in parallel).
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_fused_f8(const GemmConfig& cfg, const GemmArgs& args,
                                 cudaStream_t stream) {
  return launch_gemm_fmt<kModeFused, kFmtF8>(cfg, args, stream);
}

}  // namespace forge
