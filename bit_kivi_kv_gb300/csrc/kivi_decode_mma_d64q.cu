// Instantiations of the tensor-core decode kernel: head_dim 64, caches whose value residual is a queue.
#include "kivi_decode_mma_launch.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d64q(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st) {
    return mma_launch::dispatch<64, mma_detail::kModeFifo>(a, bits, nq, G, num_sms, st);
}

}  // namespace kivi
