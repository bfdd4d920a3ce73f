// gemm_swap128.cu -- instantiates the GEMM launchers of: launch_bn<true, 128>.
#include "gemm_impl.cuh"

namespace fp8bq {

cudaError_t launch_gemm_swap128(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_bn<true, 128>(p, g, stream);
}

}  // namespace fp8bq
