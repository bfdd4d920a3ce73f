// gemm_i8.cu -- instantiates the GEMM launchers of: launch_i8<8>, launch_i8<16>, launch_i8<32>, launch_i8<64>, launch_i8<128>.
#include "gemm_impl.cuh"

namespace fp8bq {

cudaError_t launch_gemm_i8_8(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_i8<8>(p, g, stream);
}

cudaError_t launch_gemm_i8_16(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_i8<16>(p, g, stream);
}

cudaError_t launch_gemm_i8_32(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_i8<32>(p, g, stream);
}

cudaError_t launch_gemm_i8_64(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_i8<64>(p, g, stream);
}

cudaError_t launch_gemm_i8_128(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_i8<128>(p, g, stream);
}

}  // namespace fp8bq
