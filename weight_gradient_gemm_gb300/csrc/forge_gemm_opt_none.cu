// Instantiates the tensor-core kernel for SGD, the optimizer without state:
// its state slots hold W alone, which leaves shared memory for more operand
// stages and slots.
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_opt_none(const GemmConfig& cfg, const GemmArgs& args, cudaStream_t stream) {
  return launch_gemm_fmt<kModeOpt, kFmtNone>(cfg, args, stream);
}

}  // namespace forge
