// Instantiates the tensor-core kernel for the optimizers with one fp32
// state (SGD with momentum, Adagrad, RMSprop, Lion): their state slots hold
// W and that state alone, which leaves shared memory for more operand stages
// and slots.
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_opt_f32s1(const GemmConfig& cfg, const GemmArgs& args,
                                  cudaStream_t stream) {
  return launch_gemm_fmt<kModeOpt, kFmtF32S1>(cfg, args, stream);
}

}  // namespace forge
