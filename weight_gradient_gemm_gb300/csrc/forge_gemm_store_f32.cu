// Instantiates the tensor-core weight-gradient kernel for one mode and format
// (one translation unit each, so they compile in parallel).
#include "forge_gemm.cuh"

namespace forge {

cudaError_t launch_gemm_store_f32(const GemmConfig& cfg, const GemmArgs& args,
                                cudaStream_t stream) {
  return launch_gemm_fmt<kModeStoreG, kFmtF32>(cfg, args, stream);
}


}  // namespace forge
