// Instantiations of the tensor-core decode kernel: head_dim 64, decode calls with a fused append.
#include "kivi_decode_mma_launch.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d64f(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st) {
    return mma_launch::dispatch<64, mma_detail::kModeFused>(a, bits, nq, G, num_sms, st);
}

}  // namespace kivi
