// Quantize-and-pack kernels: prefill blocks, residual flush, residual row copies.
//
// Method: uniform asymmetric B-bit group quantization ("KV cache quantization
// axis selection guide", unite.ai, section on what quantization error is made
// of): zero = group minimum, step = range / (2^B - 1), nearest level.  Keys are
// grouped per channel over G tokens, values per token over G channels (same
// guide, keys and values sections; KIVI explainer, discosf.com, 3.1).  The
// arithmetic is the fixed fp32 formula written out in kivi.h.
#include "kivi_common.cuh"

namespace kivi {
namespace {

constexpr int kQuantThreads = 128;

// Step and zero of one group from its fp32 min / max (fp16 inputs, exact).
// A -0 min or max becomes +0; every operation is a separately rounded RN op.
__device__ __forceinline__ void group_step_zero(float mn, float mx, int L, float* s, float* z,
                                                __half* s_out, __half* z_out) {
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    const float s32 = __fdiv_rn(__fsub_rn(mx, mn), (float)L);
    const __half s16 = __float2half_rn(s32);
    const __half z16 = __float2half_rn(mn);
    *s = __half2float(s16);
    *z = __half2float(z16);
    *s_out = s16;
    *z_out = z16;
}

// Nearest level of the stored grid: clamp(rint((x - z) / s), 0, L); 0 when s == 0.
__device__ __forceinline__ uint32_t nearest_code(float x, float s, float z, int L) {
    if (s == 0.0f) return 0u;
    const int c = __float2int_rn(__fdiv_rn(__fsub_rn(x, z), s));
    return (uint32_t)min(max(c, 0), L);
}

struct QuantArgs {
    uint8_t* cache;
    const __half* src_k;
    const __half* src_v;
    long long src_slot_elems;
    long long first_block;
    long long NB, part_bytes, slot_bytes, tile_bytes;
    int G;
};

// One CTA quantizes one block (G tokens x D channels) of keys and of values.
template <int D, int BITS>
__global__ void __launch_bounds__(kQuantThreads) quantize_blocks_kernel(QuantArgs a) {
    constexpr int L = (1 << BITS) - 1;
    constexpr int W = D * BITS / 64;        // words per lane per tile
    constexpr int PER = 16 / BITS;          // code pairs per word
    constexpr int TILE_WORDS = 32 * W;
    extern __shared__ __align__(16) unsigned char smem[];
    const int G = a.G;
    __half* xs = reinterpret_cast<__half*>(smem);            // [G][D]
    float* sf = reinterpret_cast<float*>(xs + G * D);         // [D] steps
    float* zf = sf + D;                                       // [D] zeros

    const int tid = threadIdx.x;
    const long long slot = blockIdx.y;
    const long long j = blockIdx.x;
    uint8_t* part_k = a.cache + slot * a.slot_bytes + (a.first_block + j) * a.part_bytes;
    uint8_t* part_v = part_k + a.NB * a.part_bytes;
    const long long tiles_bytes = (long long)(G / 16) * a.tile_bytes;
    const int n_vec = G * D / 8;

    // ---------------- keys: per channel over the block's G tokens ----------------
    {
        const uint4* src = reinterpret_cast<const uint4*>(a.src_k + slot * a.src_slot_elems + j * G * D);
        for (int v = tid; v < n_vec; v += kQuantThreads) reinterpret_cast<uint4*>(xs)[v] = src[v];
    }
    __syncthreads();
    for (int c = tid; c < D; c += kQuantThreads) {
        float mn = INFINITY, mx = -INFINITY;
        for (int t = 0; t < G; ++t) {
            const float v = __half2float(xs[t * D + c]);
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
        }
        __half* ent = reinterpret_cast<__half*>(part_k + tiles_bytes);   // D steps, then D zeros
        group_step_zero(mn, mx, L, &sf[c], &zf[c], &ent[c], &ent[D + c]);
    }
    __syncthreads();
    for (int w = tid; w < (G / 16) * TILE_WORDS; w += kQuantThreads) {
        const int tt = w / TILE_WORDS, lane = (w % TILE_WORDS) / W, wl = w % W;
        const int g = lane >> 2, i = lane & 3;
        uint32_t word = 0;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            using PP = PairPlace<BITS, false>;
            const int k = PP::k_of(wl, u), r = PP::r_of(wl, u), bit = PP::bit(k, r);
            const int tok = tt * 16 + g + 8 * (r & 1);
            const int ch = 16 * k + 2 * i + 8 * (r >> 1);
            const uint32_t c0 = nearest_code(__half2float(xs[tok * D + ch]), sf[ch], zf[ch], L);
            const uint32_t c1 = nearest_code(__half2float(xs[tok * D + ch + 1]), sf[ch + 1], zf[ch + 1], L);
            word |= (c0 << bit) | (c1 << (16 + bit));
        }
        reinterpret_cast<uint32_t*>(part_k)[w] = word;
    }
    __syncthreads();

    // ---------------- values: per token over groups of G channels ----------------
    {
        const uint4* src = reinterpret_cast<const uint4*>(a.src_v + slot * a.src_slot_elems + j * G * D);
        for (int v = tid; v < n_vec; v += kQuantThreads) reinterpret_cast<uint4*>(xs)[v] = src[v];
    }
    __syncthreads();
    const int ngrp = D / G;                 // channel groups per token; G * ngrp == D entries
    for (int e = tid; e < D; e += kQuantThreads) {
        const int t = e / ngrp, gr = e % ngrp;
        const __half* row = xs + t * D + gr * G;
        float mn = INFINITY, mx = -INFINITY;
        for (int jj = 0; jj < G; ++jj) {
            const float v = __half2float(row[(jj + tid) & (G - 1)]);   // rotated start: fewer bank conflicts
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
        }
        // entry tile of the token's code tile: ngrp rows of 16 steps, then the zeros
        __half* ent = reinterpret_cast<__half*>(part_v + tiles_bytes + (long long)(t / 16) * 64 * ngrp);
        const int at = gr * 16 + entry_pos(t % 16);
        group_step_zero(mn, mx, L, &sf[e], &zf[e], &ent[at], &ent[16 * ngrp + at]);
    }
    __syncthreads();
    for (int w = tid; w < (G / 16) * TILE_WORDS; w += kQuantThreads) {
        const int tt = w / TILE_WORDS, lane = (w % TILE_WORDS) / W, wl = w % W;
        const int g = lane >> 2, i = lane & 3;
        uint32_t word = 0;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            using PP = PairPlace<BITS, true>;
            const int k = PP::k_of(wl, u), r = PP::r_of(wl, u), bit = PP::bit(k, r);
            const int ch = 16 * k + g + 8 * (r & 1);
            const int tok0 = tt * 16 + 2 * i + 8 * (r >> 1);
            const int e0 = tok0 * ngrp + ch / G, e1 = e0 + ngrp;
            const uint32_t c0 = nearest_code(__half2float(xs[tok0 * D + ch]), sf[e0], zf[e0], L);
            const uint32_t c1 = nearest_code(__half2float(xs[(tok0 + 1) * D + ch]), sf[e1], zf[e1], L);
            word |= (c0 << bit) | (c1 << (16 + bit));
        }
        reinterpret_cast<uint32_t*>(part_v)[w] = word;
    }
}

// Copy nrows rows of D fp16 (keys and values) per slot into the residual.
__global__ void __launch_bounds__(128) copy_rows_kernel(uint8_t* cache, const __half* src_k,
                                                        const __half* src_v, long long src_slot_elems,
                                                        long long k_off, long long v_off,
                                                        long long resid_slot_bytes, int D, int row0,
                                                        int nrows) {
    // a following decode launched as a programmatic dependent may start its
    // prologue now; it waits for this kernel before it reads residual rows
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long slot = blockIdx.x;
    const int n_vec = nrows * D / 8;
    const uint4* sk = reinterpret_cast<const uint4*>(src_k + slot * src_slot_elems);
    const uint4* sv = reinterpret_cast<const uint4*>(src_v + slot * src_slot_elems);
    uint4* dk = reinterpret_cast<uint4*>(cache + k_off + slot * resid_slot_bytes + (long long)row0 * D * 2);
    uint4* dv = reinterpret_cast<uint4*>(cache + v_off + slot * resid_slot_bytes + (long long)row0 * D * 2);
    for (int v = threadIdx.x; v < n_vec; v += blockDim.x) {
        dk[v] = sk[v];
        dv[v] = sv[v];
    }
}

}  // namespace

cudaError_t launch_quantize_blocks(const Geometry& g, uint8_t* cache, const __half* src_k,
                                   const __half* src_v, long long src_slot_elems,
                                   long long first_block, long long nblk, cudaStream_t st) {
    QuantArgs a{cache, src_k, src_v, src_slot_elems, first_block, g.NB, g.part_bytes,
                g.slot_bytes, g.tile_bytes, g.G};
    const dim3 grid((unsigned)nblk, (unsigned)(g.B * g.Hkv));
    const size_t smem = (size_t)g.G * g.D * 2 + 2 * (size_t)g.D * 4;
    if (g.D == 128 && g.bits == 2) quantize_blocks_kernel<128, 2><<<grid, kQuantThreads, smem, st>>>(a);
    else if (g.D == 128 && g.bits == 4) quantize_blocks_kernel<128, 4><<<grid, kQuantThreads, smem, st>>>(a);
    else if (g.D == 64 && g.bits == 2) quantize_blocks_kernel<64, 2><<<grid, kQuantThreads, smem, st>>>(a);
    else if (g.D == 64 && g.bits == 4) quantize_blocks_kernel<64, 4><<<grid, kQuantThreads, smem, st>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_copy_rows(const Geometry& g, uint8_t* cache, const __half* src_k,
                             const __half* src_v, long long src_slot_elems, int row0, int nrows,
                             cudaStream_t st) {
    copy_rows_kernel<<<g.B * g.Hkv, 128, 0, st>>>(cache, src_k, src_v, src_slot_elems, g.k_resid_off,
                                                  g.v_resid_off, g.resid_slot_bytes, g.D, row0, nrows);
    return cudaGetLastError();
}

}  // namespace kivi
