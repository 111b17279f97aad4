// Split-KV decode attention over the quantized cache and the fp16 residual.
//
// Method: at each generated token the whole KV cache is read and the output is
// the softmax-weighted sum of the values ("KV cache quantization axis selection
// guide", unite.ai, sections on why the KV cache is the problem and on values).
// The split-KV partial results (m, l, o) are merged by log-sum-exp.
//
// Key-side algebra used here: with per-(block, channel) step s_c and zero z_c,
//   q . k_hat_t = sum_c (q_c s_c) code_tc + sum_c q_c z_c,
// so the query is folded with the block's steps once per block and the zero
// term is one scalar per block.  Logits are kept in the log2 domain
// (scale * log2(e) folded into q) so the softmax uses exp2.
#include <math.h>

#include "kivi_common.cuh"
#include "kivi_decode_mma.cuh"

namespace kivi {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

struct DecodeArgs {
    const uint8_t* cache;
    const __half* q;
    float* ws;
    long long NB, part_bytes, slot_bytes, tile_bytes, k_resid_off, v_resid_off;
    int R, G, Hq, Hkv;
    int n_qtiles, n_resid;
    int tiles_per_split, n_qsplits;
    float scale_log2;
};

template <int N>
__device__ __forceinline__ void load_words(const uint32_t* p, uint32_t (&w)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int v = 0; v < N / 4; ++v) {
            const uint4 x = reinterpret_cast<const uint4*>(p)[v];
            w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int v = 0; v < N / 2; ++v) {
            const uint2 x = reinterpret_cast<const uint2*>(p)[v];
            w[2 * v] = x.x; w[2 * v + 1] = x.y;
        }
    }
}

// Online-softmax update of one warp for one head over a 16-token tile.
// sc0 / sc1: logits of tokens g and g+8 (same in the 4 lanes of group g).
// On return pr[0..3] hold the probabilities of tokens 2i, 2i+1, 2i+8, 2i+9.
template <int VCH>
__device__ __forceinline__ void softmax_tile(float sc0, float sc1, float& m, float& l,
                                             float (&acc)[VCH], float (&pr)[4], int i) {
    float mt = fmaxf(sc0, sc1);
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
    const float mn = fmaxf(m, mt);
    const float alpha = exp2f(m - mn);
    const float p0 = exp2f(sc0 - mn), p1 = exp2f(sc1 - mn);
    float ps = p0 + p1;
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int v = 0; v < VCH; ++v) acc[v] *= alpha;
    pr[0] = __shfl_sync(0xffffffffu, p0, 8 * i);
    pr[1] = __shfl_sync(0xffffffffu, p0, 8 * i + 4);
    pr[2] = __shfl_sync(0xffffffffu, p1, 8 * i);
    pr[3] = __shfl_sync(0xffffffffu, p1, 8 * i + 4);
}

// One CTA: one (batch, kv-head) slot, one split of its tokens, all NQ query
// heads of the slot.  Warps take the split's 16-token tiles round-robin.
template <int D, int BITS, int NQ>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeArgs a) {
    constexpr int L = (1 << BITS) - 1;
    constexpr int W = D * BITS / 64;
    constexpr int PAIRS = D / 4;
    constexpr int VCH = D / 8;           // value channels per lane
    __shared__ float qf[NQ][D];
    __shared__ float qt[kWarps][NQ][D];
    __shared__ float red_m[kWarps][NQ], red_l[kWarps][NQ];
    __shared__ __align__(16) float red_o[kWarps][NQ][D];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, i = lane & 3;
    const int slot = blockIdx.y, split = blockIdx.x;
    const int b = slot / a.Hkv, hk = slot % a.Hkv;
    const int G = a.G, ngrp = D / G;

    for (int idx = tid; idx < NQ * D; idx += kThreads) {
        const int j = idx / D, c = idx % D;
        qf[j][c] = __half2float(a.q[((long long)b * a.Hq + hk * NQ + j) * D + c]) * a.scale_log2;
    }
    __syncthreads();

    float m[NQ], l[NQ], acc[NQ][VCH];
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
        m[j] = -INFINITY; l[j] = 0.f;
#pragma unroll
        for (int v = 0; v < VCH; ++v) acc[j][v] = 0.f;
    }

    const uint8_t* slot_base = a.cache + (long long)slot * a.slot_bytes;
    if (split < a.n_qsplits) {
        const int t0 = split * a.tiles_per_split;
        const int t1 = min(t0 + a.tiles_per_split, a.n_qtiles);
        int cur_blk = -1;
        float beta[NQ];
        for (int T = t0 + warp; T < t1; T += kWarps) {
            const int blk = T * 16 / G, tin = (T * 16 % G) / 16;
            const uint8_t* kpart = slot_base + (long long)blk * a.part_bytes;
            const uint8_t* vpart = kpart + a.NB * a.part_bytes;
            const long long tiles_bytes = (long long)(G / 16) * a.tile_bytes;
            if (blk != cur_blk) {            // fold this block's key steps into q
                cur_blk = blk;
                __syncwarp();                // all lanes are done reading the previous block's qt
                const __half* ks = reinterpret_cast<const __half*>(kpart + tiles_bytes);   // D steps, D zeros
                float bp[NQ];
#pragma unroll
                for (int j = 0; j < NQ; ++j) bp[j] = 0.f;
                for (int c = lane; c < D; c += 32) {
                    const float2 sz = make_float2(__half2float(ks[c]), __half2float(ks[D + c]));
#pragma unroll
                    for (int j = 0; j < NQ; ++j) {
                        qt[warp][j][c] = qf[j][c] * sz.x;
                        bp[j] = fmaf(qf[j][c], sz.y, bp[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) bp[j] += __shfl_xor_sync(0xffffffffu, bp[j], o);
                    beta[j] = bp[j];
                }
                __syncwarp();
            }
            // ---- scores of tokens g and g+8 ----
            uint32_t kw[W];
            load_words(reinterpret_cast<const uint32_t*>(kpart + tin * a.tile_bytes) + lane * W, kw);
            float part[NQ][2];
#pragma unroll
            for (int j = 0; j < NQ; ++j) part[j][0] = part[j][1] = 0.f;
#pragma unroll
            for (int p = 0; p < PAIRS; ++p) {
                using PP = PairPlace<BITS, false>;
                const int k = p >> 2, r = p & 3, bit = PP::bit(k, r);
                const uint32_t w = kw[PP::word(k, r)];
                const float c0 = (float)((w >> bit) & L);
                const float c1 = (float)((w >> (16 + bit)) & L);
                const int ch = 16 * k + 2 * i + 8 * (r >> 1);
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
                    part[j][r & 1] = fmaf(qt[warp][j][ch], c0, part[j][r & 1]);
                    part[j][r & 1] = fmaf(qt[warp][j][ch + 1], c1, part[j][r & 1]);
                }
            }
            float pr[NQ][4];
#pragma unroll
            for (int j = 0; j < NQ; ++j) {
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    part[j][s] += __shfl_xor_sync(0xffffffffu, part[j][s], 1);
                    part[j][s] += __shfl_xor_sync(0xffffffffu, part[j][s], 2);
                }
                softmax_tile<VCH>(part[j][0] + beta[j], part[j][1] + beta[j], m[j], l[j], acc[j], pr[j], i);
            }
            // ---- weighted values ----
            uint32_t vw[W];
            load_words(reinterpret_cast<const uint32_t*>(vpart + tin * a.tile_bytes) + lane * W, vw);
            // this tile's entry tile: ngrp rows of 16 steps, then the zeros
            const __half* vse = reinterpret_cast<const __half*>(vpart + tiles_bytes + (long long)tin * 64 * ngrp);
#pragma unroll
            for (int p = 0; p < PAIRS; ++p) {
                using PP = PairPlace<BITS, true>;
                const int k = p >> 2, r = p & 3, bit = PP::bit(k, r);
                const uint32_t w = vw[PP::word(k, r)];
                const float c0 = (float)((w >> bit) & L);
                const float c1 = (float)((w >> (16 + bit)) & L);
                const int ch = 16 * k + g + 8 * (r & 1);
                const int e0 = (ch / G) * 16 + entry_pos(2 * i + 8 * (r >> 1)), e1 = e0 + 1;   // tokens tau, tau+1
                const float2 sz0 = make_float2(__half2float(vse[e0]), __half2float(vse[16 * ngrp + e0]));
                const float2 sz1 = make_float2(__half2float(vse[e1]), __half2float(vse[16 * ngrp + e1]));
                const float v0 = fmaf(c0, sz0.x, sz0.y), v1 = fmaf(c1, sz1.x, sz1.y);
                const int vl = 2 * k + (r & 1), ts = 2 * (r >> 1);
#pragma unroll
                for (int j = 0; j < NQ; ++j)
                    acc[j][vl] = fmaf(pr[j][ts], v0, fmaf(pr[j][ts + 1], v1, acc[j][vl]));
            }
        }
    } else {
        // ---- the fp16 residual rows [0, n_resid) ----
        const __half* kr = reinterpret_cast<const __half*>(a.cache + a.k_resid_off) + (long long)slot * a.R * D;
        const __half* vr = reinterpret_cast<const __half*>(a.cache + a.v_resid_off) + (long long)slot * a.R * D;
        const int n = a.n_resid;
        for (int sub = warp; sub * 16 < n; sub += kWarps) {
            float part[NQ][2];
#pragma unroll
            for (int j = 0; j < NQ; ++j) part[j][0] = part[j][1] = 0.f;
#pragma unroll
            for (int ts = 0; ts < 2; ++ts) {
                const int tok = sub * 16 + g + 8 * ts;
                if (tok < n) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int ch = 16 * k + 2 * i + 8 * h;
                            const float2 kv = __half22float2(*reinterpret_cast<const __half2*>(kr + (long long)tok * D + ch));
#pragma unroll
                            for (int j = 0; j < NQ; ++j)
                                part[j][ts] = fmaf(qf[j][ch], kv.x, fmaf(qf[j][ch + 1], kv.y, part[j][ts]));
                        }
                    }
                }
            }
            const bool ok0 = sub * 16 + g < n, ok1 = sub * 16 + g + 8 < n;
            float pr[NQ][4];
#pragma unroll
            for (int j = 0; j < NQ; ++j) {
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    part[j][s] += __shfl_xor_sync(0xffffffffu, part[j][s], 1);
                    part[j][s] += __shfl_xor_sync(0xffffffffu, part[j][s], 2);
                }
                softmax_tile<VCH>(ok0 ? part[j][0] : -INFINITY, ok1 ? part[j][1] : -INFINITY, m[j], l[j],
                                  acc[j], pr[j], i);
            }
#pragma unroll
            for (int p = 0; p < PAIRS; ++p) {
                const int k = p >> 2, r = p & 3;
                const int ch = 16 * k + g + 8 * (r & 1);
                const int tok0 = sub * 16 + 2 * i + 8 * (r >> 1);
                const float v0 = tok0 < n ? __half2float(vr[(long long)tok0 * D + ch]) : 0.f;
                const float v1 = tok0 + 1 < n ? __half2float(vr[(long long)(tok0 + 1) * D + ch]) : 0.f;
                const int vl = 2 * k + (r & 1), ts = 2 * (r >> 1);
#pragma unroll
                for (int j = 0; j < NQ; ++j)
                    acc[j][vl] = fmaf(pr[j][ts], v0, fmaf(pr[j][ts + 1], v1, acc[j][vl]));
            }
        }
    }

    // ---- merge the warps, write this split's partial (m, l, o) ----
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
#pragma unroll
        for (int v = 0; v < VCH; ++v) {
            acc[j][v] += __shfl_xor_sync(0xffffffffu, acc[j][v], 1);
            acc[j][v] += __shfl_xor_sync(0xffffffffu, acc[j][v], 2);
        }
        if (i == 0) {
#pragma unroll
            for (int v = 0; v < VCH; ++v) red_o[warp][j][16 * (v >> 1) + g + 8 * (v & 1)] = acc[j][v];
        }
        if (lane == 0) { red_m[warp][j] = m[j]; red_l[warp][j] = l[j]; }
    }
    __syncthreads();
    for (int idx = tid; idx < NQ * D; idx += kThreads) {
        const int j = idx / D, c = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][j]);
        float o = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float e = red_m[w][j] == -INFINITY ? 0.f : exp2f(red_m[w][j] - M);
            o = fmaf(red_o[w][j][c], e, o);
            lsum = fmaf(red_l[w][j], e, lsum);
        }
        float* pw = a.ws + ((long long)(b * a.Hq + hk * NQ + j) * kPartialSlots + split) * partial_stride(D);
        if (c == 0) { pw[0] = M; pw[1] = lsum; }
        if (c == 1) pw[2] = 0.f;
        pw[4 + c] = o;
    }
}

// Log-sum-exp merge of a head's split partials -> fp16 output.
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(const float* ws, __half* out, int n_splits) {
    const long long bh = blockIdx.x;
    const int c = threadIdx.x;
    const float* base = ws + bh * kPartialSlots * partial_stride(D);
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, base[s * partial_stride(D)]);
    float o = 0.f, lsum = 0.f;
    bool failed = false;
    for (int s = 0; s < n_splits; ++s) {
        const float* ps = base + s * partial_stride(D);
        failed |= ps[2] != 0.f;            // a split whose data copy timed out
        if (ps[0] == -INFINITY) continue;
        const float e = exp2f(ps[0] - M);
        lsum = fmaf(ps[1], e, lsum);
        o = fmaf(ps[4 + c], e, o);
    }
    out[bh * D + c] = failed ? __float2half_rn(NAN) : __float2half_rn(o / lsum);
}

template <int D, int BITS, int NQ>
cudaError_t launch_t(const DecodeArgs& a, int n_splits, int slots, __half* out, int Hq, int B,
                     cudaStream_t st) {
    decode_split_kernel<D, BITS, NQ><<<dim3(n_splits, slots), kThreads, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    combine_kernel<D><<<B * Hq, D, 0, st>>>(a.ws, out, n_splits);
    return cudaGetLastError();
}

}  // namespace

DecodePlan plan_decode(const Geometry& g, long long n_quant, long long n_resid, int num_sms) {
    DecodePlan p{};
    const long long n_qtiles = n_quant / 16;
    const long long slots = (long long)g.B * g.Hkv;
    const long long target = 4LL * (num_sms > 0 ? num_sms : 1);
    const long long per_slot = (target + slots - 1) / slots;
    long long tps = (n_qtiles + per_slot - 1) / per_slot;
    if (tps < 8) tps = 8;
    const long long cap = (n_qtiles + kMaxSplits - 1) / kMaxSplits;
    if (tps < cap) tps = cap;
    tps = (tps + 1) & ~1LL;   // whole tile pairs (the tensor-core kernel takes two tiles per stage)
    p.tiles_per_split = (int)tps;
    p.n_qsplits = n_qtiles ? (int)((n_qtiles + tps - 1) / tps) : 0;
    p.n_splits = p.n_qsplits + (n_resid > 0 ? 1 : 0);
    p.num_sms = num_sms > 0 ? num_sms : 1;
    return p;
}

// Launch the tensor-core kernel on a persistent grid; fills a.wm.n.
cudaError_t launch_decode_mma_d128(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st);
cudaError_t launch_decode_mma_d64(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st);
cudaError_t launch_decode_mma_d128f(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st);
cudaError_t launch_decode_mma_d64f(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st);
cudaError_t launch_decode_mma_d128p(mma_detail::PagedArgs& a, int bits, int nq, int G, int num_sms, cudaStream_t st);
cudaError_t launch_decode_mma_d128q(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st);
cudaError_t launch_decode_mma_d64q(mma_detail::Args& a, int bits, int nq, int G, int num_sms, cudaStream_t st);
cudaError_t launch_decode_mma_d64p(mma_detail::PagedArgs& a, int bits, int nq, int G, int num_sms, cudaStream_t st);

namespace {

// The merge's form: a warp per head when no slot has more partials than the
// warp form loads in one round trip (a slot meets at most Ws * n / Wt + 2
// workers), else a CTA per head.
inline bool merge_by_warp(const WorkMap& wm) {
    return (double)wm.Ws * (double)wm.n / (double)wm.Wt + 2.0 <= (double)mma_detail::kMergeAhead;
}

// Launch the merge kernel as a programmatic dependent of the decode kernel.
template <typename K, typename A>
cudaError_t launch_finish(K kernel, const A& f, long long ctas, cudaStream_t st) {
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3((unsigned)ctas);
    lc.blockDim = dim3(mma_detail::kMergeThreads);
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&lc, kernel, f);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_paged(const PagedGeometry& pg, const uint8_t* buf, const PagedSeq* seqs, int n,
                                const __half* q, __half* out, float scale_log2, float* workspace,
                                const __half* new_k, const __half* new_v, int early_ok, int num_sms, int max_ctas,
                                cudaStream_t st, int* launches) {
    const Geometry& g = pg.g;
    *launches = 0;
    if (n < 1 || n > kMaxCallSeqs) return cudaErrorInvalidValue;
    const int nq = g.Hq / g.Hkv;
    WorkMap wm{};
    wm.wq = (long long)g.D * g.bits / 4 + 8LL * g.D / g.G;
    wm.wr = 5LL * g.D / 2;   // the dense call's weights (below), so equal lengths split alike
    long long wt0 = 0, ws_min = -1;
    for (int i = 0; i < n; ++i) {
        if (seqs[i].P + seqs[i].n_resid <= 0) return cudaErrorInvalidValue;   // a sequence without tokens
        const long long w = slot_weight(wm, seqs[i].P, 0, (seqs[i].n_resid + 31) / 32);
        wt0 += g.Hkv * w;
        if (ws_min < 0 || w < ws_min) ws_min = w;
    }
    wm.S0 = segment_lead(wm.wq, ws_min, wt0, num_sms);
    mma_detail::PagedArgs m;   // ~12 KB of kernel parameters
    long long start = 0, ws_max = 0;
    for (int i = 0; i < n; ++i) {
        PagedSeq s = seqs[i];
        const long long Ws = wm.S0 + slot_weight(wm, s.P, 0, (s.n_resid + 31) / 32);
        s.start = start;
        start += g.Hkv * Ws;
        if (Ws > ws_max) ws_max = Ws;
        m.seqs[i] = s;
    }
    wm.Ws = ws_max;
    wm.Wt = start;
    wm.n = max_ctas;   // 0: the launch sizes the grid
    static_cast<mma_detail::Args&>(m) =
        mma_detail::Args{buf, q, workspace, g.NB, g.part_bytes, 0, g.tile_bytes, g.k_resid_off, g.v_resid_off,
                         g.R, g.Hq, g.Hkv, 0, wm, scale_log2, new_k, new_v, -1, early_ok};
    m.table = reinterpret_cast<const int*>(buf + pg.table_off);
    m.max_blocks = (int)g.NB;
    m.n_pages = (int)pg.n_pages;
    m.n_seqs = n;
    cudaError_t e = (g.D == 128 ? launch_decode_mma_d128p : launch_decode_mma_d64p)(m, g.bits, nq, g.G, num_sms, st);
    if (e != cudaSuccess) return e;
    *launches = 1;
    mma_detail::PagedFinishArgs f;
    f.ws = workspace;
    f.out = out;
    f.Hq = g.Hq;
    f.Hkv = g.Hkv;
    f.nq = nq;
    f.wm = m.wm;   // with the grid size the launch chose
    f.heads = (long long)n * g.Hq;
    f.n_seqs = n;
    for (int i = 0; i < n; ++i) f.seqs[i] = m.seqs[i];
    if (merge_by_warp(m.wm)) {
        const long long ctas = (f.heads + mma_detail::kMergeWarps - 1) / mma_detail::kMergeWarps;
        e = g.D == 128 ? launch_finish(mma_detail::finish_paged_kernel<128, true>, f, ctas, st)
                       : launch_finish(mma_detail::finish_paged_kernel<64, true>, f, ctas, st);
    } else {
        e = g.D == 128 ? launch_finish(mma_detail::finish_paged_kernel<128, false>, f, f.heads, st)
                       : launch_finish(mma_detail::finish_paged_kernel<64, false>, f, f.heads, st);
    }
    if (e != cudaSuccess) return e;
    *launches = 2;
    return cudaSuccess;
}



cudaError_t launch_decode(const Geometry& g, const uint8_t* cache, long long n_quant,
                          long long n_resid, const __half* q, __half* out, float scale_log2,
                          float* workspace, const DecodePlan& plan, int variant, cudaStream_t st,
                          int* launches, const FusedAppend& fa) {
    if ((fa.row >= 0 || fa.lqv >= 0) && variant != KIVI_DECODE_TENSOR_CORE)
        return cudaErrorInvalidValue;   // fused append and value queue: tensor cores only
    if (variant == KIVI_DECODE_TENSOR_CORE) {
        const int nq = g.Hq / g.Hkv;
        const long long slots = (long long)g.B * g.Hkv;
        WorkMap wm{};
        wm.P = n_quant / 32;
        wm.PR = (n_resid + 31) / 32;
        wm.wq = (long long)g.D * g.bits / 4 + 8LL * g.D / g.G;   // bytes of a quantized pair / 32
        // a residual pair reads 128 D bytes (weight 4 D), but its rows come
        // through plain loads that the SM overlaps with the bulk copies of the
        // warps beside it: weighted as 80 D bytes, measured best on the 7B
        // layer shape (4 D: +2% per call; GQA and long context within 1%).
        // With the value queue the warps at slot ends also hold the mixed
        // pairs, and the full 4 D measured best.
        wm.wr = fa.lqv >= 0 ? 4LL * g.D : 5LL * g.D / 2;
        if (fa.lqv >= 0) {
            // value queue: pairs from lqv / 32 on also read up to 32 fp16 value
            // rows, 64 D bytes, weighted as 48 D bytes: measured on the 7B layer
            // shape, with the full weight the warps that read them finish early
            wm.M = wm.P - (fa.lqv / 32 < wm.P ? fa.lqv / 32 : wm.P);
            wm.wx = 3LL * g.D / 2;
        }
        const long long ws0 = slot_weight(wm, wm.P, wm.M, wm.PR);
        wm.S0 = segment_lead(wm.wq, ws0, slots * ws0, plan.num_sms);
        wm.Ws = wm.S0 + ws0;
        wm.n = plan.max_ctas;   // 0: the launch sizes the grid
        wm.Wt = slots * wm.Ws;
        mma_detail::Args m{cache, q, workspace, g.NB, g.part_bytes, g.slot_bytes, g.tile_bytes,
                           g.k_resid_off, g.v_resid_off, g.R, g.Hq, g.Hkv, (int)n_resid, wm, scale_log2,
                           fa.k, fa.v, fa.row, fa.early_ok, fa.lqv, fa.pop, fa.stall_bytes};
        const bool fused = fa.row >= 0, fifo = fa.lqv >= 0;
        using L = cudaError_t (*)(mma_detail::Args&, int, int, int, int, cudaStream_t);
        const L launch = g.D == 128 ? (fifo ? launch_decode_mma_d128q : fused ? launch_decode_mma_d128f
                                                                              : launch_decode_mma_d128)
                                    : (fifo ? launch_decode_mma_d64q : fused ? launch_decode_mma_d64f
                                                                             : launch_decode_mma_d64);
        cudaError_t e = launch(m, g.bits, nq, g.G, plan.num_sms, st);
        if (e != cudaSuccess) return e;
        const long long heads = (long long)g.B * g.Hq;
        mma_detail::FinishArgs f{workspace, out, g.Hq, g.Hkv, nq, m.wm, heads};
        // the merge may start while the main kernel drains; it waits for it on the GPU
        if (merge_by_warp(m.wm)) {
            const long long ctas = (heads + mma_detail::kMergeWarps - 1) / mma_detail::kMergeWarps;
            e = g.D == 128 ? launch_finish(mma_detail::finish_kernel<128, true>, f, ctas, st)
                           : launch_finish(mma_detail::finish_kernel<64, true>, f, ctas, st);
        } else {
            e = g.D == 128 ? launch_finish(mma_detail::finish_kernel<128, false>, f, heads, st)
                           : launch_finish(mma_detail::finish_kernel<64, false>, f, heads, st);
        }
        *launches = 2;
        return e;
    }
    DecodeArgs a{cache, q, workspace, g.NB, g.part_bytes, g.slot_bytes, g.tile_bytes,
                 g.k_resid_off, g.v_resid_off, g.R, g.G, g.Hq, g.Hkv,
                 (int)(n_quant / 16), (int)n_resid, plan.tiles_per_split, plan.n_qsplits, scale_log2};
    const int slots = g.B * g.Hkv, nq = g.Hq / g.Hkv;
    *launches = 2;
#define KIVI_DISPATCH(DD, BB, NN)                                                            \
    if (g.D == DD && g.bits == BB && nq == NN)                                               \
        return launch_t<DD, BB, NN>(a, plan.n_splits, slots, out, g.Hq, g.B, st);
    KIVI_DISPATCH(128, 2, 1) KIVI_DISPATCH(128, 2, 2) KIVI_DISPATCH(128, 2, 4)
    KIVI_DISPATCH(128, 4, 1) KIVI_DISPATCH(128, 4, 2) KIVI_DISPATCH(128, 4, 4)
    KIVI_DISPATCH(64, 2, 1) KIVI_DISPATCH(64, 2, 2) KIVI_DISPATCH(64, 2, 4)
    KIVI_DISPATCH(64, 4, 1) KIVI_DISPATCH(64, 4, 2) KIVI_DISPATCH(64, 4, 4)
    KIVI_DISPATCH(128, 8, 1) KIVI_DISPATCH(128, 8, 2) KIVI_DISPATCH(128, 8, 4)
    KIVI_DISPATCH(64, 8, 1) KIVI_DISPATCH(64, 8, 2) KIVI_DISPATCH(64, 8, 4)
#undef KIVI_DISPATCH
    *launches = 0;
    return cudaErrorInvalidValue;
}

}  // namespace kivi
