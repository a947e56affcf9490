// Instantiates the tensor-core kernel in its input-gradient mode (dX = dY W,
// bf16 out); one translation unit per mode and format so they compile in
// parallel.
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_dgrad(const GemmConfig& cfg, const GemmArgs& args, cudaStream_t stream) {
  return launch_gemm_fmt<kModeDgrad, kFmtBF16>(cfg, args, stream);
}

}  // namespace forge
