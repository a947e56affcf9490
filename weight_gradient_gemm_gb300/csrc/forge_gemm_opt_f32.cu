// Instantiates the tensor-core kernel with the other coordinate-wise
// optimizers (SGD, SGD with momentum, Adagrad, RMSprop, Lion, NAdam, RAdam)
// in the epilogue and fp32 optimizer state; one translation unit per
// state format so they compile in parallel.
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_opt_f32(const GemmConfig& cfg, const GemmArgs& args, cudaStream_t stream) {
  return launch_gemm_fmt<kModeOpt, kFmtF32>(cfg, args, stream);
}

}  // namespace forge
