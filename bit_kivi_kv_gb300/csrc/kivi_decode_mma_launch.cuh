// Launch of one tensor-core decode kernel instance (persistent grid, dynamic
// shared memory, programmatic dependent launch) and the dispatch over the
// instances of one head_dim; included by the per-head_dim instantiation files.
#pragma once

#include <mutex>

#include "kivi_decode_mma.cuh"

namespace kivi {
namespace mma_launch {

// Per-device set-up of one kernel instance: the opt-in to its dynamic shared
// memory and its resident CTAs per SM are properties of a device, so they are
// taken once per device (with that device current) and kept per device.
constexpr int kMaxDevices = 64;
struct InstanceSetup {
    std::mutex mu;
    int per_sm[kMaxDevices] = {};        // 0: not set up on that device yet
};

template <int D, int BB, int NN, int GG, int MODE>
cudaError_t launch_one(typename mma_detail::ArgsOf<MODE>::type& a, int num_sms, cudaStream_t st) {
    using namespace mma_detail;
    using C = Cfg<D, BB, NN, GG>;
    constexpr int kDyn = C::DYN_SMEM + (MODE == kModeFifo ? kMixBytes : 0);
    static InstanceSetup setup;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int per_sm;
    {
        std::lock_guard<std::mutex> lock(setup.mu);
        per_sm = setup.per_sm[dev];
        if (per_sm == 0) {
            // opt in to the dynamic shared memory of the copy ring and size the
            // persistent grid from the occupancy on this device
            e = cudaFuncSetAttribute(decode_mma_kernel<D, BB, NN, GG, MODE>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mma_kernel<D, BB, NN, GG, MODE>,
                                                                  kThreads, kDyn);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) per_sm = 1;
            setup.per_sm[dev] = per_sm;
        }
    }
    // the workers of the map are warps: the resident warps of a persistent grid
    // (or the caller's cap on CTAs, times the warps of a CTA)
    const long long slots = a.wm.Ws > 0 ? a.wm.Wt / a.wm.Ws : 1;   // slots of the largest weight
    long long n = (long long)num_sms * per_sm * kWarps;
    if (a.wm.n > 0 && a.wm.n * kWarps < n) n = a.wm.n * kWarps;
    // (a warp whose range holds no unit start inside a slot writes an empty
    // partial; at most kMaxSplits partials per slot)
    if (n > (kMaxSplits - 1) * slots) n = (kMaxSplits - 1) * slots;
    const long long units = a.wm.Wt / (a.wm.wq < a.wm.wr ? a.wm.wq : a.wm.wr);
    if (n > units) n = units;                                          // no more warps than units
    if (n < 1) n = 1;
    a.wm.n = n;
    const long long ctas = (n + kWarps - 1) / kWarps;
    // a programmatic dependent of the preceding kernel: the kernel's prologue
    // and first cache copies overlap that kernel's tail
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3((unsigned)ctas);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = kDyn;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, decode_mma_kernel<D, BB, NN, GG, MODE>, a);
}

// every (bits, q heads per kv head, G) instance of head_dim D
template <int D, int MODE>
cudaError_t dispatch(typename mma_detail::ArgsOf<MODE>::type& a, int bits, int nq, int G, int num_sms,
                     cudaStream_t st) {
#define KIVI_MMA(BB, NN, GG) \
    if (bits == BB && nq == NN && G == GG) return launch_one<D, BB, NN, GG, MODE>(a, num_sms, st);
#define KIVI_MMA_G(BB, NN) KIVI_MMA(BB, NN, 32) KIVI_MMA(BB, NN, 64) if constexpr (D >= 128) { KIVI_MMA(BB, NN, 128) }
    KIVI_MMA_G(2, 1) KIVI_MMA_G(2, 2) KIVI_MMA_G(2, 4)
    KIVI_MMA_G(4, 1) KIVI_MMA_G(4, 2) KIVI_MMA_G(4, 4)
    KIVI_MMA_G(8, 1) KIVI_MMA_G(8, 2) KIVI_MMA_G(8, 4)
#undef KIVI_MMA_G
#undef KIVI_MMA
    return cudaErrorInvalidValue;
}

}  // namespace mma_launch
}  // namespace kivi
