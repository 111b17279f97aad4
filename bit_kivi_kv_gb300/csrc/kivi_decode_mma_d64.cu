// Instantiations of the tensor-core decode kernel for head_dim 64.
#include "kivi_decode_mma.cuh"

namespace kivi {

namespace {
template <int BB, int NN, int GG>
cudaError_t launch_one(const mma_detail::Args& a, dim3 grid, cudaStream_t st) {
    using namespace mma_detail;
    using C = Cfg<64, BB, NN, GG>;
    // opt in to the dynamic shared memory of the copy ring once per instance
    static const cudaError_t attr = cudaFuncSetAttribute(
        decode_mma_kernel<64, BB, NN, GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
    if (attr != cudaSuccess) return attr;
    decode_mma_kernel<64, BB, NN, GG><<<grid, kThreads, C::DYN_SMEM, st>>>(a);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_mma_d64(const mma_detail::Args& a, int bits, int nq, int G, dim3 grid,
                                  cudaStream_t st) {
#define KIVI_MMA(BB, NN, GG) \
    if (bits == BB && nq == NN && G == GG) return launch_one<BB, NN, GG>(a, grid, st);
#define KIVI_MMA_G(BB, NN) KIVI_MMA(BB, NN, 32) KIVI_MMA(BB, NN, 64) 
    KIVI_MMA_G(2, 1) KIVI_MMA_G(2, 2) KIVI_MMA_G(2, 4)
    KIVI_MMA_G(4, 1) KIVI_MMA_G(4, 2) KIVI_MMA_G(4, 4)
#undef KIVI_MMA_G
#undef KIVI_MMA
    return cudaErrorInvalidValue;
}

}  // namespace kivi
