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

// The same code as nearest_code with the division done as a multiply by
// r = rn(1/s) plus one FMA correction, which lands within 1.5 ulp of the IEEE
// quotient rn((x - z) / s).  Rounding to the nearest level can then differ
// only when the quotient is within 2^-17 of a half-integer (ulp <= 2^-19 below
// 16; 2^-15 with 8-bit codes, ulp <= 2^-16 below 256); those elements, and no
// others, take the IEEE division.  Quotients >= L + 1 round to L either way.
__device__ __forceinline__ uint32_t nearest_code_r(float x, float s, float r, float z, int L) {
    const float near = L > 15 ? 0x1p-15f : 0x1p-17f;
    if (s == 0.0f) return 0u;
    const float d = __fsub_rn(x, z);
    const float q0 = __fmul_rn(d, r);
    const float q = __fmaf_rn(__fmaf_rn(-s, q0, d), r, q0);
    if (q >= (float)L + 1.0f) return (uint32_t)L;
    const int c = __float2int_rn(q);                      // q >= 0: x >= z, the group minimum
    if (fabsf(__fsub_rn(q, __int2float_rn(c))) >= 0.5f - near) return nearest_code(x, s, z, L);
    return (uint32_t)min(c, L);
}

// ---- 2-bit codes from per-group thresholds ----
// The fixed formula code(x) = clamp(rint(rn(rn(x - z) / s)), 0, L) is
// non-decreasing in x (each rounded step is monotone for s > 0), so a group's
// code of x is the number of levels c = 1..L whose threshold T_c, the least
// fp16 value with code(T_c) >= c, x reaches.  T_c is found next to the real
// crossing z + (c - 1/2) s by evaluating the formula itself (IEEE division) on
// fp16 neighbours, so the codes are those of the formula bit for bit; the
// elements are then compared with the thresholds two at a time in fp16.

// fp16 values in order as integers (-0 and +0 both 0) and back
__device__ __forceinline__ int half_ord(__half h) {
    const int b = __half_as_ushort(h);
    return (b & 0x8000) ? -(b & 0x7FFF) : b;
}
__device__ __forceinline__ __half ord_half(int o) {
    return __ushort_as_half((unsigned short)(o >= 0 ? o : (0x8000 | -o)));
}

// T_c of a group with stored step s > 0 and zero z (fp32 values of fp16
// entries).  The probes sit next to a half-step by construction, so they take
// the IEEE division directly.
__device__ __forceinline__ __half level_threshold(int c, float s, float z, int L) {
    // The real crossing is y = z + (c - 1/2) s.  rn(x - z) and rn(. / s) each
    // move the quotient by at most 2^-24 of itself, so an fp16 x more than
    // (c - 1/2) s 2^-23 (plus y's own rounding, |y| 2^-24) above y has
    // code(x) >= c, and one as far below has code(x) < c; delta = (c s + |y|)
    // 2^-22 covers that twice.  So when no fp16 value lies within delta of y,
    // T_c is the least fp16 >= y: the least fp16 >= y - delta, when that is
    // above y + delta (the fp32 rounding of y -/+ delta is far inside the slack).
    const float y = __fmaf_rn((float)c - 0.5f, s, z);
    const float delta = __fmaf_rn((float)c, s, fabsf(y)) * 0x1p-22f;
    const __half a = __float2half_ru(y - delta);
    if (__half2float(a) > y + delta) return a;
    // Otherwise search, probing with the formula itself: code(x) does not
    // decrease with x, so gallop from the fp16 nearest y to neighbours lo < hi
    // with code(lo) < c <= code(hi), then bisect.  The finite fp16 range holds
    // both ends (code(-65504) = 0 < c <= L = code(65504) for s > 0), and
    // near 0, where fp16 values are far denser than the rounding band, the
    // threshold can be hundreds of fp16 steps from y.
    constexpr int kMin = -0x7BFF, kMax = 0x7BFF;
    auto reaches = [&](int o) { return (int)nearest_code(__half2float(ord_half(o)), s, z, L) >= c; };
    const int o = min(max(half_ord(__float2half_rn(y)), kMin), kMax);
    int lo, hi;
    if (reaches(o)) {
        hi = o;
        for (int step = 1;; step *= 2) {
            lo = max(hi - step, kMin);
            if (!reaches(lo)) break;
            hi = lo;
            if (lo == kMin) return ord_half(kMin);   // (not reached for s > 0)
        }
    } else {
        lo = o;
        for (int step = 1;; step *= 2) {
            hi = min(lo + step, kMax);
            if (reaches(hi)) break;
            lo = hi;
            if (hi == kMax) return __ushort_as_half(0x7C00);   // no finite x reaches c (not for s > 0)
        }
    }
    while (hi - lo > 1) {
        const int mid = lo + (hi - lo) / 2;
        if (reaches(mid)) hi = mid; else lo = mid;
    }
    return ord_half(hi);
}

// Two 2-bit codes (lo and hi halves) of x against half2 thresholds, OR-ed into
// word at bit b of each half.  The code is the number of thresholds x reaches;
// T_1 <= T_2 <= T_3, so the ones reached are a prefix: bit 1 of the code is
// [x >= T_2] and bit 0 the parity of the three comparisons.
__device__ __forceinline__ uint32_t place_codes2(uint32_t word, __half2 x, __half2 t1, __half2 t2, __half2 t3, int b) {
    const uint32_t m1 = __hge2_mask(x, t1), m2 = __hge2_mask(x, t2), m3 = __hge2_mask(x, t3);
    return word | ((m1 ^ m2 ^ m3) & (0x00010001u << b)) | (m2 & (0x00020002u << b));
}

// With 2-bit codes the bit of a word's code pair u does not depend on the
// word's column: 8 (u / 4) + 2 (u % 4) for keys and values alike.
__host__ __device__ constexpr int code2_bit(int u) { return 8 * (u >> 2) + 2 * (u & 3); }
template <bool VALUES>
constexpr bool code2_bits_hold() {
    using PP = PairPlace<2, VALUES>;
    for (int wl = 0; wl < 128 * 2 / 64; ++wl)
        for (int u = 0; u < 8; ++u)
            if (PP::bit(PP::k_of(wl, u), PP::r_of(wl, u)) != code2_bit(u)) return false;
    return true;
}
static_assert(code2_bits_hold<false>() && code2_bits_hold<true>(), "2-bit code placement");

struct QuantArgs {
    uint8_t* cache;
    const __half* src_k;
    const __half* src_v;
    long long src_slot_elems;
    long long first_block;
    long long NB, part_bytes, slot_bytes, tile_bytes;
    long long vlimit;   // value tokens at or after this slot position stay unquantized (zero codes, step, zero)
    int G;
};

// Paged form: CTA (j, h) quantizes job j's block of kv head h into its page.
struct PagedQuantArgs {
    uint8_t* pool;
    int* table;
    const __half* src_k;
    const __half* src_v;
    long long src_head_elems;
    long long part_bytes, tile_bytes;
    int Hkv, G;
    QJob jobs[kMaxQJobs];
};

template <bool PAGED>
struct QuantArgsOf { using type = QuantArgs; };
template <>
struct QuantArgsOf<true> { using type = PagedQuantArgs; };

// One CTA quantizes one block (G tokens x D channels) of keys and of values.
// The block's rows are staged in shared memory with a stride of D + 8 halves,
// so lanes reading one channel of different tokens hit different banks.  A
// thread packs the same word position of every 16-token tile, so the
// coordinates of its codes (and, for keys, their steps and zeros) are fixed
// once per block.
template <int D, int BITS, int G, bool PAGED>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_blocks_kernel(const __grid_constant__ typename QuantArgsOf<PAGED>::type a) {
    constexpr int L = (1 << BITS) - 1;
    constexpr int W = D * BITS / 64;        // words per lane per tile
    constexpr int PER = 16 / BITS;          // code pairs per word
    constexpr int TILE_WORDS = 32 * W;
    constexpr int DP = D + 8;               // staged row stride, halves
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int TPB = G / 16;
    __half* xs = reinterpret_cast<__half*>(smem);            // [G][DP]
    // per group: (step, rn(1 / step), zero, unused); D groups for keys and for values
    float4* szr = reinterpret_cast<float4*>(xs + G * DP);
    // 2-bit codes: the groups' level thresholds T_1..T_3 (fp16), [3][D] each:
    // keys by channel, values by (channel group, token)
    __half* thr = reinterpret_cast<__half*>(szr + D);

    const int tid = threadIdx.x;
    const __half* blk_k;   // the block's G rows of keys / values
    const __half* blk_v;
    uint8_t* part_k;
    uint8_t* part_v;
    if constexpr (PAGED) {
        const QJob& jb = a.jobs[blockIdx.x];
        const int h = blockIdx.y;
        const long long off = jb.src_off + h * a.src_head_elems;
        blk_k = a.src_k + off;
        blk_v = a.src_v + off;
        part_k = a.pool + ((long long)jb.page * a.Hkv + h) * 2 * a.part_bytes;
        part_v = part_k + a.part_bytes;
        if (h == 0 && tid == 0) a.table[jb.tbl_idx] = jb.page;
    } else {
        const long long slot = blockIdx.y;
        const long long j = blockIdx.x;
        const long long off = slot * a.src_slot_elems + j * G * D;
        blk_k = a.src_k + off;
        blk_v = a.src_v + off;
        part_k = a.cache + slot * a.slot_bytes + (a.first_block + j) * a.part_bytes;
        part_v = part_k + a.NB * a.part_bytes;
    }
    const long long tiles_bytes = (long long)TPB * a.tile_bytes;
    auto stage_rows = [&](const __half* src) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        for (int v = tid; v < G * D / 8; v += kQuantThreads) {
            const int row = v / (D / 8), c8 = v - row * (D / 8);
            *reinterpret_cast<uint4*>(xs + row * DP + 8 * c8) = s4[v];
        }
    };

    // ---------------- keys: per channel over the block's G tokens ----------------
    stage_rows(blk_k);
    __syncthreads();
    // min / max of channel pairs (2cp, 2cp+1) over the G tokens on fp16 pairs (exact);
    // adjacent threads take alternate blocks of 4 tokens (rows 4 apart fall 16
    // banks apart, so the pair's reads do not conflict) and combine
    for (int idx = tid; idx < D; idx += kQuantThreads) {
        const int cp = idx >> 1, half = idx & 1;
        __half2 mn2 = __half2half2(__ushort_as_half(0x7C00)), mx2 = __half2half2(__ushort_as_half(0xFC00));
        for (int jt = 0; jt < G / 2; ++jt) {
            const int t = 8 * (jt >> 2) + 4 * half + (jt & 3);
            const __half2 v = *reinterpret_cast<const __half2*>(xs + t * DP + 2 * cp);
            mn2 = __hmin2(mn2, v);
            mx2 = __hmax2(mx2, v);
        }
        mn2 = __hmin2(mn2, __shfl_xor_sync(0xffffffffu, mn2, 1));
        mx2 = __hmax2(mx2, __shfl_xor_sync(0xffffffffu, mx2, 1));
        const float2 mn = __half22float2(mn2), mx = __half22float2(mx2);
        const int c = 2 * cp + half;                    // each thread of the pair finishes one channel
        __half* ent = reinterpret_cast<__half*>(part_k + tiles_bytes);   // D steps, then D zeros
        float sc, zc;
        group_step_zero(half ? mn.y : mn.x, half ? mx.y : mx.x, L, &sc, &zc, &ent[c], &ent[D + c]);
        szr[c] = make_float4(sc, sc != 0.0f ? __frcp_rn(sc) : 0.0f, zc, 0.0f);
        if constexpr (BITS == 2) {
#pragma unroll
            for (int lv = 1; lv <= 3; ++lv)
                thr[(lv - 1) * D + c] = sc == 0.0f ? __ushort_as_half(0x7C00) : level_threshold(lv, sc, zc, L);
        }
    }
    __syncthreads();
    if constexpr (BITS == 2) {
        // each thread packs one word position of every tile: 8 code pairs, each
        // two adjacent channels of one token, compared with their thresholds.  A
        // warp takes one word column (wl) of all 32 lanes, so its rows (tokens g,
        // g + 8) and channel pairs fall in distinct banks.
        using PP = PairPlace<BITS, false>;
        for (int wt = tid; wt < TILE_WORDS; wt += kQuantThreads) {
            const int lane = wt & 31, wl = wt >> 5;
            const int g = lane >> 2, i = lane & 3;
            int off[PER];
            __half2 t1[PER], t2[PER], t3[PER];
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int k = PP::k_of(wl, u), r = PP::r_of(wl, u);
                const int ch = 16 * k + 2 * i + 8 * (r >> 1);
                off[u] = (g + 8 * (r & 1)) * DP + ch;
                t1[u] = *reinterpret_cast<const __half2*>(thr + ch);
                t2[u] = *reinterpret_cast<const __half2*>(thr + D + ch);
                t3[u] = *reinterpret_cast<const __half2*>(thr + 2 * D + ch);
            }
            for (int tt = 0; tt < TPB; ++tt) {
                uint32_t word = 0;
#pragma unroll
                for (int u = 0; u < PER; ++u) {
                    const __half2 x = *reinterpret_cast<const __half2*>(xs + tt * 16 * DP + off[u]);
                    word = place_codes2(word, x, t1[u], t2[u], t3[u], code2_bit(u));
                }
                reinterpret_cast<uint32_t*>(part_k)[tt * TILE_WORDS + lane * W + wl] = word;
            }
        }
    } else
    for (int wt = tid; wt < TILE_WORDS; wt += kQuantThreads) {
        using PP = PairPlace<BITS, false>;
        const int lane = wt / W, wl = wt - lane * W;
        const int g = lane >> 2, i = lane & 3;
        int off[PER], bit[PER];
        float s0[PER], z0[PER], s1[PER], z1[PER], q0r[PER], q1r[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int k = PP::k_of(wl, u), r = PP::r_of(wl, u);
            const int ch = 16 * k + 2 * i + 8 * (r >> 1);
            off[u] = (g + 8 * (r & 1)) * DP + ch;
            bit[u] = PP::bit(k, r);
            const float4 e0 = szr[ch], e1 = szr[ch + 1];
            s0[u] = e0.x; q0r[u] = e0.y; z0[u] = e0.z;
            s1[u] = e1.x; q1r[u] = e1.y; z1[u] = e1.z;
        }
        for (int tt = 0; tt < TPB; ++tt) {
            uint32_t word = 0;
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const float2 x = __half22float2(*reinterpret_cast<const __half2*>(xs + tt * 16 * DP + off[u]));
                const uint32_t c0 = nearest_code_r(x.x, s0[u], q0r[u], z0[u], L);
                const uint32_t c1 = nearest_code_r(x.y, s1[u], q1r[u], z1[u], L);
                word |= (c0 << bit[u]) | (c1 << (16 + bit[u]));
            }
            reinterpret_cast<uint32_t*>(part_k)[tt * TILE_WORDS + wt] = word;
        }
    }
    __syncthreads();

    // ---------------- values: per token over groups of G channels ----------------
    stage_rows(blk_v);
    __syncthreads();
    const int ngrp = D / G;                 // channel groups per token; G * ngrp == D entries
    long long vfirst = 0;                   // slot position of the block's first token (value limit)
    if constexpr (!PAGED) vfirst = (a.first_block + (long long)blockIdx.x) * G;
    for (int e = tid; e < D; e += kQuantThreads) {
        const int t = e / ngrp, gr = e % ngrp;
        const __half* row = xs + t * DP + gr * G;
        __half2 mn2 = __half2half2(__ushort_as_half(0x7C00)), mx2 = __half2half2(__ushort_as_half(0xFC00));
        for (int jj = 0; jj < G / 8; ++jj) {           // 8 channels a load; the rotated start spreads banks
            const uint4 v4 = *reinterpret_cast<const uint4*>(row + 8 * ((jj + tid) & (G / 8 - 1)));
            const __half2* h = reinterpret_cast<const __half2*>(&v4);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mn2 = __hmin2(mn2, h[q]);
                mx2 = __hmax2(mx2, h[q]);
            }
        }
        const float2 mnf = __half22float2(mn2), mxf = __half22float2(mx2);
        float mn = fminf(mnf.x, mnf.y), mx = fmaxf(mxf.x, mxf.y);
        if constexpr (!PAGED) {
            // a value token not quantized yet: step 0 and zero point 0, so codes 0
            if (vfirst + t >= a.vlimit) mn = mx = 0.0f;
        }
        // entry tile of the token's code tile: ngrp rows of 16 steps, then the zeros
        __half* ent = reinterpret_cast<__half*>(part_v + tiles_bytes + (long long)(t / 16) * 64 * ngrp);
        const int at = gr * 16 + entry_pos(t % 16);
        float se, ze;
        group_step_zero(mn, mx, L, &se, &ze, &ent[at], &ent[16 * ngrp + at]);
        szr[e] = make_float4(se, se != 0.0f ? __frcp_rn(se) : 0.0f, ze, 0.0f);
        if constexpr (BITS == 2) {
#pragma unroll
            for (int lv = 1; lv <= 3; ++lv)
                thr[(lv - 1) * D + gr * G + t] = se == 0.0f ? __ushort_as_half(0x7C00) : level_threshold(lv, se, ze, L);
        }
    }
    __syncthreads();
    if constexpr (BITS == 2) {
        // each thread packs one word position of every tile: 8 code pairs, each
        // one channel of two consecutive tokens, compared with the tokens'
        // thresholds; a warp takes one word column of all 32 lanes
        using PP = PairPlace<BITS, true>;
        for (int wt = tid; wt < TILE_WORDS; wt += kQuantThreads) {
            const int lane = wt & 31, wl = wt >> 5;
            const int g = lane >> 2, i = lane & 3;
            // the word's channels 16k + g (+8), k in {2wl, 2wl+1}, lie in one group of
            // G >= 32 channels; its tokens are 2i, 2i+1 (r < 2) and 2i+8, 2i+9 (r >= 2)
            int off[PER];
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int k = PP::k_of(wl, u), r = PP::r_of(wl, u);
                const int ch = 16 * k + g + 8 * (r & 1);
                off[u] = (2 * i + 8 * (r >> 1)) * DP + ch;
            }
            const int tgrp = ((16 * PP::k_of(wl, 0)) / G) * G + 2 * i;   // thresholds of (group, token 2i)
            for (int tt = 0; tt < TPB; ++tt) {
                const __half* tp = thr + tgrp + tt * 16;
                const __half2 a1 = *reinterpret_cast<const __half2*>(tp);
                const __half2 a2 = *reinterpret_cast<const __half2*>(tp + D);
                const __half2 a3 = *reinterpret_cast<const __half2*>(tp + 2 * D);
                const __half2 b1 = *reinterpret_cast<const __half2*>(tp + 8);
                const __half2 b2 = *reinterpret_cast<const __half2*>(tp + 8 + D);
                const __half2 b3 = *reinterpret_cast<const __half2*>(tp + 8 + 2 * D);
                uint32_t word = 0;
#pragma unroll
                for (int u = 0; u < PER; ++u) {
                    // r = PP::r_of(wl, u) = (u & 1) + 2 * (u >> 2) for 2-bit codes (wl * 4 is even)
                    const bool first_tokens = (u >> 2) == 0;
                    const __half* xp = xs + tt * 16 * DP + off[u];
                    const __half2 x = __halves2half2(xp[0], xp[DP]);
                    word = first_tokens ? place_codes2(word, x, a1, a2, a3, code2_bit(u))
                                        : place_codes2(word, x, b1, b2, b3, code2_bit(u));
                }
                reinterpret_cast<uint32_t*>(part_v)[tt * TILE_WORDS + lane * W + wl] = word;
            }
        }
    } else
    for (int wt = tid; wt < TILE_WORDS; wt += kQuantThreads) {
        using PP = PairPlace<BITS, true>;
        const int lane = wt / W, wl = wt - lane * W;
        const int g = lane >> 2, i = lane & 3;
        int off[PER], bit[PER], ent0[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int k = PP::k_of(wl, u), r = PP::r_of(wl, u);
            const int ch = 16 * k + g + 8 * (r & 1);
            const int tok0 = 2 * i + 8 * (r >> 1);
            off[u] = tok0 * DP + ch;
            bit[u] = PP::bit(k, r);
            ent0[u] = tok0 * ngrp + ch / G;   // (step, zero) entry of the first token; the second's is ngrp on
        }
        for (int tt = 0; tt < TPB; ++tt) {
            uint32_t word = 0;
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const __half* xp = xs + tt * 16 * DP + off[u];
                const int e0 = tt * 16 * ngrp + ent0[u], e1 = e0 + ngrp;
                const float4 f0 = szr[e0], f1 = szr[e1];
                const uint32_t c0 = nearest_code_r(__half2float(xp[0]), f0.x, f0.y, f0.z, L);
                const uint32_t c1 = nearest_code_r(__half2float(xp[DP]), f1.x, f1.y, f1.z, L);
                word |= (c0 << bit[u]) | (c1 << (16 + bit[u]));
            }
            reinterpret_cast<uint32_t*>(part_v)[tt * TILE_WORDS + wt] = word;
        }
    }
}

// One value token per slot leaves the queue: token t (slot position) is read
// from residual row t % R, quantized per group of G channels with the fixed
// formula, and its codes and (step, zero) entries are written into block t / G,
// whose value part holds zeros for it until now (the codes are OR-ed in).
struct PopArgs {
    uint8_t* cache;
    long long t;
    long long NB, part_bytes, slot_bytes, tile_bytes, v_resid_off;
    int R, G;
};

template <int D, int BITS>
__global__ void __launch_bounds__(D) pop_value_kernel(PopArgs a) {
    constexpr int L = (1 << BITS) - 1;
    constexpr int W = D * BITS / 64;
    using PP = PairPlace<BITS, true>;
    __shared__ float x[D];
    __shared__ float s_g[D], z_g[D];       // per group (at most D / 32 used)
    const int c = threadIdx.x;
    const long long slot = blockIdx.x;
    const __half* row = reinterpret_cast<const __half*>(a.cache + a.v_resid_off) + (slot * a.R + a.t % a.R) * D;
    x[c] = __half2float(row[c]);
    __syncthreads();
    const int G = a.G, ngrp = D / G, gr = c / G;
    const long long blk = a.t / G;
    const int tt = (int)(a.t % G), tile = tt / 16, tok = tt % 16;
    uint8_t* part_v = a.cache + slot * a.slot_bytes + (a.NB + blk) * a.part_bytes;
    if (c % G == 0) {
        float mn = x[c], mx = x[c];
        for (int j = 1; j < G; ++j) { mn = fminf(mn, x[c + j]); mx = fmaxf(mx, x[c + j]); }
        __half* ent = reinterpret_cast<__half*>(part_v + (long long)(G / 16) * a.tile_bytes + (long long)tile * 64 * ngrp);
        const int at = gr * 16 + entry_pos(tok);
        float s, z;
        group_step_zero(mn, mx, L, &s, &z, &ent[at], &ent[16 * ngrp + at]);
        s_g[gr] = s;
        z_g[gr] = z;
    }
    __syncthreads();
    const uint32_t code = nearest_code(x[c], s_g[gr], z_g[gr], L);
    // value tile placement: channel c = 16k + g + 8(r%2), token tok = 2i + 8(r/2) + half
    const int k = c / 16, cc = c % 16, g = cc % 8;
    const int r = (cc / 8) + 2 * (tok / 8), i = (tok % 8) / 2, half = tok % 2;
    const int lane = 4 * g + i;
    uint32_t* words = reinterpret_cast<uint32_t*>(part_v + (long long)tile * a.tile_bytes);
    atomicOr(&words[lane * W + PP::word(k, r)], code << (PP::bit(k, r) + 16 * half));
}

// Copy nk key rows (source rows k_src0.., residual rows k_row0..) and nv value
// rows (source rows v_src0.., tokens v_tok0.. at residual rows token % R) per slot.
__global__ void __launch_bounds__(128) copy_rows_ring_kernel(uint8_t* cache, const __half* src_k,
                                                             const __half* src_v, long long src_slot_elems,
                                                             long long k_off, long long v_off,
                                                             long long resid_slot_bytes, int D, int R,
                                                             int k_row0, long long k_src0, int nk,
                                                             long long v_tok0, long long v_src0, int nv) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long slot = blockIdx.x;
    const int cpr = D / 8;      // 16-byte chunks per row
    const uint4* sk = reinterpret_cast<const uint4*>(src_k + slot * src_slot_elems + k_src0 * D);
    const uint4* sv = reinterpret_cast<const uint4*>(src_v + slot * src_slot_elems + v_src0 * D);
    uint4* dk = reinterpret_cast<uint4*>(cache + k_off + slot * resid_slot_bytes);
    uint4* dv = reinterpret_cast<uint4*>(cache + v_off + slot * resid_slot_bytes);
    for (int v = threadIdx.x; v < nk * cpr; v += blockDim.x) dk[(long long)k_row0 * cpr + v] = sk[v];
    for (int v = threadIdx.x; v < nv * cpr; v += blockDim.x) {
        const int j = v / cpr, c = v % cpr;
        dv[((v_tok0 + j) % R) * cpr + c] = sv[v];
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

template <bool PAGED>
cudaError_t launch_q(const typename QuantArgsOf<PAGED>::type& a, const Geometry& g, dim3 grid, cudaStream_t st) {
    // staged rows + (step, 1/step, zero) per group + three fp16 level thresholds per group
    const size_t smem = (size_t)g.G * (g.D + 8) * 2 + 16 * (size_t)g.D + 6 * (size_t)g.D;
#define KIVI_Q(DD, BB, GG)                                                                      \
    if (g.D == DD && g.bits == BB && g.G == GG) {                                               \
        quantize_blocks_kernel<DD, BB, GG, PAGED><<<grid, kQuantThreads, smem, st>>>(a);        \
        return cudaGetLastError();                                                              \
    }
#define KIVI_QG(DD, BB) KIVI_Q(DD, BB, 32) KIVI_Q(DD, BB, 64) if (DD >= 128) { KIVI_Q(128, BB, 128) }
    KIVI_QG(128, 2) KIVI_QG(128, 4) KIVI_QG(128, 8) KIVI_QG(64, 2) KIVI_QG(64, 4) KIVI_QG(64, 8)
#undef KIVI_QG
#undef KIVI_Q
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_quantize_blocks(const Geometry& g, uint8_t* cache, const __half* src_k,
                                   const __half* src_v, long long src_slot_elems,
                                   long long first_block, long long nblk, cudaStream_t st, long long vlimit) {
    QuantArgs a{cache, src_k, src_v, src_slot_elems, first_block, g.NB, g.part_bytes,
                g.slot_bytes, g.tile_bytes, vlimit, g.G};
    const dim3 grid((unsigned)nblk, (unsigned)(g.B * g.Hkv));
    return launch_q<false>(a, g, grid, st);
}

cudaError_t launch_quantize_pages(const PagedGeometry& pg, uint8_t* buf, const __half* src_k,
                                  const __half* src_v, long long src_head_elems, const QJob* jobs,
                                  int njobs, cudaStream_t st, int* launches) {
    const Geometry& g = pg.g;
    PagedQuantArgs a;          // ~16 KB of kernel parameters
    a.pool = buf;
    a.table = reinterpret_cast<int*>(buf + pg.table_off);
    a.src_k = src_k;
    a.src_v = src_v;
    a.src_head_elems = src_head_elems;
    a.part_bytes = g.part_bytes;
    a.tile_bytes = g.tile_bytes;
    a.Hkv = g.Hkv;
    a.G = g.G;
    *launches = 0;
    for (int j0 = 0; j0 < njobs; j0 += kMaxQJobs) {
        const int nj = njobs - j0 < kMaxQJobs ? njobs - j0 : kMaxQJobs;
        for (int j = 0; j < nj; ++j) a.jobs[j] = jobs[j0 + j];
        const cudaError_t e = launch_q<true>(a, g, dim3((unsigned)nj, (unsigned)g.Hkv), st);
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

cudaError_t launch_copy_rows_slots(const Geometry& g, uint8_t* cache, const __half* src_k,
                                   const __half* src_v, long long src_slot_elems, long long first_slot,
                                   int nslots, int row0, int nrows, cudaStream_t st) {
    const long long skip = first_slot * g.resid_slot_bytes;
    copy_rows_kernel<<<nslots, 128, 0, st>>>(cache, src_k, src_v, src_slot_elems, g.k_resid_off + skip,
                                             g.v_resid_off + skip, g.resid_slot_bytes, g.D, row0, nrows);
    return cudaGetLastError();
}

cudaError_t launch_pop_values(const Geometry& g, uint8_t* cache, long long t, cudaStream_t st) {
    PopArgs a{cache, t, g.NB, g.part_bytes, g.slot_bytes, g.tile_bytes, g.v_resid_off, g.R, g.G};
    const unsigned slots = (unsigned)((long long)g.B * g.Hkv);
#define KIVI_POP(DD, BB) \
    if (g.D == DD && g.bits == BB) { pop_value_kernel<DD, BB><<<slots, DD, 0, st>>>(a); return cudaGetLastError(); }
    KIVI_POP(128, 2) KIVI_POP(128, 4) KIVI_POP(128, 8) KIVI_POP(64, 2) KIVI_POP(64, 4) KIVI_POP(64, 8)
#undef KIVI_POP
    return cudaErrorInvalidValue;
}

cudaError_t launch_copy_rows_ring(const Geometry& g, uint8_t* cache, const __half* src_k, const __half* src_v,
                                  long long src_slot_elems, int k_row0, long long k_src0, int nk,
                                  long long v_tok0, long long v_src0, int nv, cudaStream_t st) {
    copy_rows_ring_kernel<<<g.B * g.Hkv, 128, 0, st>>>(cache, src_k, src_v, src_slot_elems, g.k_resid_off,
                                                       g.v_resid_off, g.resid_slot_bytes, g.D, g.R, k_row0,
                                                       k_src0, nk, v_tok0, v_src0, nv);
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
