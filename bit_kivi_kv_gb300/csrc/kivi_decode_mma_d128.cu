// Instantiations of the tensor-core decode kernel for head_dim 128.
#include "kivi_decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d128(const mma_detail::Args& a, int bits, int nq, int G, dim3 grid,
                                  cudaStream_t st) {
    using namespace mma_detail;
#define KIVI_MMA(BB, NN, GG)                                                          \
    if (bits == BB && nq == NN && G == GG) {                                          \
        decode_mma_kernel<128, BB, NN, GG><<<grid, kThreads, 0, st>>>(a);             \
        return cudaGetLastError();                                                    \
    }
#define KIVI_MMA_G(BB, NN) KIVI_MMA(BB, NN, 32) KIVI_MMA(BB, NN, 64) KIVI_MMA(BB, NN, 128)
    KIVI_MMA_G(2, 1) KIVI_MMA_G(2, 2) KIVI_MMA_G(2, 4)
    KIVI_MMA_G(4, 1) KIVI_MMA_G(4, 2) KIVI_MMA_G(4, 4)
#undef KIVI_MMA_G
#undef KIVI_MMA
    return cudaErrorInvalidValue;
}

}  // namespace kivi
