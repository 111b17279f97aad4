// Tensor-core split-KV decode over the quantized cache and the fp16 residual.
//
// Same computation as the CUDA-core kernel (softmax-weighted sum of the
// dequantized values over every cached token; "KV cache quantization axis
// selection guide", unite.ai), arranged for mma.sync.m16n8k16 (fp16 x fp16 ->
// fp32) with the cache as the M operand:
//
//   keys   : S[t][n]   = sum_c code[t][c] * Qt[c][n] + beta[n]
//            Qt[c][2h] + Qt[c][2h+1] = q_h[c] * step_c (fp16 hi + lo parts,
//            about 22 significant bits); beta = sum_c q_h[c] * zero_c is
//            added to the MMA's sums (the block's zero-point term).
//   values : O^T[c][n] = sum_t code[c][t] * Pt[t][n]  (+ sum_t p_t zero_t per
//            channel group, accumulated on the side in fp32)
//            Pt[t][n] = p_h(t) * step(t, group) as fp16 hi + lo parts.  Column
//            n = 2*(h*GB + j) + {hi, lo} carries group j of the GB groups one
//            B fragment covers, so for one query head all channel groups share
//            one fragment per 16-token tile; a lane keeps the accumulators of
//            the column pair that matches its channels' group.
//
// Codes enter the MMA straight from the tile words: a code pair masked in
// place (one AND per A register, plus one 8-bit shift per word for the pairs
// in the upper byte) is a pair of fp16 subnormals code * 2^(BITS*pos - 24),
// exact, with pos = (channel / 8) % (8 / BITS) set by the cache layout.  For
// keys the channel is the MMA's k index, so 2^-(BITS*pos) is folded into the
// query side once per slot and the 2^-24 into the softmax; for values it is
// the output row, so the accumulators are rescaled once after the quantized
// tiles.  The integer pipe, the busiest one, does one mask per code pair.
// Online softmax per warp in the log2 domain.  Each warp of a persistent grid
// owns a balanced, weight-proportional share of the call's work (tile pairs of
// 32 tokens, then fp16 residual pairs, per (batch row, kv head) slot) and
// writes one partial result per slot it works on; a merge kernel combines a
// slot's partials by log-sum-exp.
#pragma once

#include <math.h>

#include "kivi_common.cuh"

namespace kivi {
namespace mma_detail {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr unsigned kFull = 0xffffffffu;

struct Args {
    const uint8_t* cache;
    const __half* q;
    float* ws;
    long long NB, part_bytes, slot_bytes, tile_bytes, k_resid_off, v_resid_off;
    int R, Hq, Hkv, n_resid;
    WorkMap wm;
    float scale_log2;
    // append fused into the call: residual row new_row (< n_resid) of every
    // slot is the token new_k / new_v [slot][D]; the kernel reads it from there
    // and writes it into the cache.  new_row < 0: no fused append.
    const __half* new_k;
    const __half* new_v;
    int new_row;
    // 1: the preceding kernel writes no quantized block, so the first bulk
    // copies may go out before waiting for it
    int early_ok;
    // value queue (kModeFifo): values of slot positions >= lqv are in the
    // residual ring (row = position % R), those below are quantized
    long long lqv = -1;
    // value queue with a fused append: position pop (== lqv - 1) leaves the
    // queue in this call, so it counts as quantized already; -1: none
    long long pop = -1;
    // failure-detection test hook: the first ring stage of CTA 0, warp 0 expects
    // this many bytes more than its copies bring, so its bounded wait runs out
    int stall_bytes = 0;
};

struct FinishArgs {
    const float* ws;
    __half* out;
    int Hq, Hkv, nq;
    WorkMap wm;
    long long heads;   // query rows x query heads
};

// Kernel modes: plain decode; decode with a fused append; paged cache with
// ragged sequences (fused append optional per sequence).
// kModeFifo: dense cache whose values are a queue of R fp16 rows (a ring).
constexpr int kModePlain = 0, kModeFused = 1, kModePaged = 2, kModeFifo = 3;
// value queue: tile pairs with quantized keys but queued values, per warp at
// most R / 32 (R <= 128); their logits wait in shared memory for the second pass
constexpr int kMaxMixPairs = 4;
// paged: a warp's block-table entries turned into block offsets, kept per segment
constexpr int kPageCache = 128;
struct PageCache {
    long long off[kPageCache];   // byte offset of block (first + j)'s key part
    const int* trow;             // the sequence's block-table row
    long long hoff;              // byte offset of the kv head's block in a page
    int first;                   // block of off[0]
    int last;                    // the segment's last block
    int bad;                     // an entry was outside the pool (read as page 0)
};
// Fill a warp's page cache with blocks [first, first + n) of table row trow
// (n <= kPageCache); entries outside the pool become page 0 and set bad.
// Called by all lanes (lane_step 32) or by one lane alone (lane_step 1).
__device__ __forceinline__ void fill_pages(PageCache& pc, const int* trow, int first, int n, int max_blocks,
                                           int n_pages, long long pstride, long long hoff, int lane0, int lane_step) {
    bool bad = false;
    for (int j = lane0; j < n; j += lane_step) {
        const int pg = __ldg(trow + min(first + j, max_blocks - 1));
        const bool ok = (unsigned)pg < (unsigned)n_pages;
        bad |= !ok;
        pc.off[j] = (long long)(ok ? pg : 0) * pstride + hoff;
    }
    if (bad) pc.bad = 1;
}
constexpr int kMixBytes = kWarps * kMaxMixPairs * 32 * 16;

// Paged call: cache = the page pool (and the buffer holding residual rows and
// the block table); q / out / ws / new_k / new_v are indexed by the call's
// sequence i in place of the batch row; wm.Ws is the largest slot weight.
// NB, slot_bytes, n_resid and new_row of Args are unused.
struct PagedArgs : Args {
    const int* table;
    int max_blocks;
    int n_pages;
    int n_seqs;
    PagedSeq seqs[kMaxCallSeqs];
};

struct PagedFinishArgs {
    const float* ws;
    __half* out;
    int Hq, Hkv, nq;
    WorkMap wm;
    long long heads;   // call sequences x query heads
    int n_seqs;
    PagedSeq seqs[kMaxCallSeqs];
};

template <int MODE>
struct ArgsOf { using type = Args; };
template <>
struct ArgsOf<kModePaged> { using type = PagedArgs; };

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t d;   // low 16 bits <- lo
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
__device__ __forceinline__ uint32_t neg_f16x2(uint32_t v) {
    uint32_t d;
    asm("neg.f16x2 %0, %1;" : "=r"(d) : "r"(v));
    return d;
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Transpose of an 8x8 matrix of 16-bit elements held as one fragment (lane l:
// row l/4, columns 2(l%4), 2(l%4)+1) into the same fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
    return d;
}

// A fragment (m16n8k16) of V^T for m-tile mt from 16 fp16 rows (tokens) of D
// channels: vg / vg8 are rows g and g+8 of the tile (ok: the row exists, else
// zeros).  Each lane loads the row-major 8x8 fragments of rows x channels
// like a key tile, and movmatrix transposes them to channels x rows.
template <int D>
__device__ __forceinline__ void vt_frag_rows(const __half* vg, const __half* vg8, bool okg, bool okg8, int mt, int i,
                                             uint32_t (&af)[4]) {
    const int ch = 16 * mt + 2 * i;
    const uint32_t x0 = okg ? *reinterpret_cast<const uint32_t*>(vg + ch) : 0u;        // tokens 0-7, channels 0-7
    const uint32_t x1 = okg8 ? *reinterpret_cast<const uint32_t*>(vg8 + ch) : 0u;      // tokens 8-15, channels 0-7
    const uint32_t x2 = okg ? *reinterpret_cast<const uint32_t*>(vg + ch + 8) : 0u;    // tokens 0-7, channels 8-15
    const uint32_t x3 = okg8 ? *reinterpret_cast<const uint32_t*>(vg8 + ch + 8) : 0u;  // tokens 8-15, channels 8-15
    af[0] = movmatrix_trans(x0);   // channels 0-7, tokens 0-7
    af[1] = movmatrix_trans(x2);   // channels 8-15, tokens 0-7
    af[2] = movmatrix_trans(x1);   // channels 0-7, tokens 8-15
    af[3] = movmatrix_trans(x3);   // channels 8-15, tokens 8-15
}

// ---- shared-memory loads through 32-bit shared addresses ----
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// ---- 1-D bulk copies (TMA) into shared memory, completed on an mbarrier ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// raise the phase's expected byte count without arriving
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_u32(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_1d_u32(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).  L2
// is coherent for the whole GPU, so a prefetch may run ahead of the kernel
// that writes the data: the later loads still see the written bytes.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// rows [first, first + n) (mod R, n <= R) of a ring of R rows of D fp16 at base
template <int D>
__device__ __forceinline__ void prefetch_ring_rows(const __half* base, int first, int n, int R) {
    if (n <= 0) return;
    const int a0 = first % R, n0 = min(n, R - a0);
    prefetch_l2(base + (long long)a0 * D, (uint32_t)(n0 * D * 2));
    if (n > n0) prefetch_l2(base, (uint32_t)((n - n0) * D * 2));
}
// 16 bytes global -> shared, asynchronous (completed by cp_async_wait_all)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for phase `parity` of an mbarrier, giving up after about 2 seconds
// (or 2^26 polls); returns false on time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_try(addr, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try(addr, parity)) return true;
        if ((it & 63u) == 63u && global_ns() - t0 > 2000000000ull) return false;
    }
    return false;
}
// programmatic dependent launch: wait for the preceding kernel's completion
// and memory; let the next kernel in the stream start launching
__device__ __forceinline__ void griddepcontrol_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddepcontrol_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }   // 2^e, |e| < 127
__device__ __forceinline__ float fast_exp2(float x) {   // hardware 2^x (ex2.approx, rel. err ~2^-22)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A fragment (4 registers) of k-step / m-tile t from a lane's tile words
// (w8 = w >> 8): each register is one code pair masked in place, i.e. two fp16
// subnormals code * 2^(BITS*pos - 24), pos = (channel / 8) % (8 / BITS).
template <int BITS, bool VALUES, int W>
__device__ __forceinline__ void a_frag(const uint32_t (&w)[W], const uint32_t (&w8)[W], int t, uint32_t (&a)[4]) {
    using PP = PairPlace<BITS, VALUES>;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int x = PP::word(t, r);
        const uint32_t field = ((1u << BITS) - 1u) * 0x00010001u << (BITS * (PP::cls(t, r) % PP::P));
        a[r] = (PP::order(r) ? w8[x] : w[x]) & field;
    }
}

// The same fragment with the 8-bit shifts done in place (no shifted copy of
// the words kept): 8-bit codes give a lane 4x the words of 2-bit ones.
template <int BITS, bool VALUES, int W>
__device__ __forceinline__ void a_frag_inline(const uint32_t (&w)[W], int t, uint32_t (&a)[4]) {
    using PP = PairPlace<BITS, VALUES>;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint32_t word = w[PP::word(t, r)];
        const uint32_t field = ((1u << BITS) - 1u) * 0x00010001u << (BITS * (PP::cls(t, r) % PP::P));
        a[r] = (PP::order(r) ? word >> 8 : word) & field;
    }
}

template <int W>
__device__ __forceinline__ void load_tile_words(const uint8_t* p, uint32_t (&w)[W]) {
    if constexpr (W % 4 == 0) {
#pragma unroll
        for (int v = 0; v < W / 4; ++v) {
            const uint4 x = ldg_stream(p + 16 * v);
            w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
    } else {
        const uint2 x = ldg_stream2(p);
        w[0] = x.x; w[1] = x.y;
    }
}

template <int D, int BITS, int NQ, int G>
struct Cfg {
    static constexpr int KSTEPS = D / 16;             // k-steps (keys) = m-tiles (values)
    static constexpr int W = D * BITS / 64;           // words per lane per tile
    static constexpr int NGRP = D / G;                // value channel groups per token
    static constexpr int GB = (NQ * NGRP <= 4) ? NGRP : 1;   // groups per B fragment
    static constexpr int NBF = NGRP / GB;             // B fragments per tile (values)
    static constexpr int QSTRIDE = 2 * KSTEPS + 4;    // u32 per lane row of the Qt fragment table
    static constexpr int TPB = G / 16;                // tiles per block
    static constexpr int TILE = 2 * D * BITS;         // bytes of one code tile
    static constexpr int ENT = 16 * NGRP * 4;         // value (step, zero) entries of one tile
    static constexpr int KSZ = 4 * D;                 // key (step, zero) entries of one block
    static constexpr int STAGES = 2;                  // ring depth per warp (stages of 2 tiles)
    // a stage: key words of 2 tiles, the block's key entries, value words of
    // 2 tiles, their value entries.  With G = 32 a tile pair is a whole block,
    // and the key part and the value part of a block are each one contiguous
    // run in this order, so a stage takes two bulk copies.
    static constexpr int KT = 0, KE = 2 * TILE, VT = 2 * TILE + KSZ, VE = 4 * TILE + KSZ;
    static constexpr int STAGE_BYTES = 4 * TILE + 2 * ENT + KSZ;
    static constexpr int DYN_SMEM = kWarps * STAGES * STAGE_BYTES;
    static constexpr bool WHOLE = TPB == 2;
};

// Build this warp's Qt B fragments (fp16 hi + lo parts of q_h * step) and
// its beta = sum_c q_h[c] * zero_c, from the block's key steps and zeros
// (D fp16 steps, then D fp16 zeros); entries == nullptr means step 1, zero 0
// (the fp16 residual: the parts are split from the fp32 query qf).  qh/ql hold
// the fp16 hi/lo parts of the scaled query per channel pair, already
// multiplied by the channel's code scale 2^-(BITS*pos); with s exact in fp16, hi = rn(qh*s)
// and lo = rn(ql*s + (qh*s - hi)), the inner residual exact, so hi + lo =
// q*s to about 22 bits.  Lane l handles channel pairs CPL*l + j; off[j] is
// the table offset of pair CPL*l + j (head 0, hi column).  With entries,
// beta is returned times 2^-24, the unit of the masked codes.  KEEP: the
// fragments are also loaded into qb; otherwise they stay in the table and the
// MMAs read each k-step's pair from it.  Measured per instance: with one query
// head per kv head, reading from the table (fewer registers held across the
// pair loop) made the calls 1-2% faster (7B layer, 13B layer, 131k context,
// the value queue, the paged cache); with grouped heads the registers were
// faster (by 0.7%).
template <class C, int D, int NQ, bool KEEP>
__device__ __forceinline__ void build_q_frags(const uint8_t* entries, const float (*qf)[D],
                                              const uint32_t (*qh)[D / 2], const uint32_t (*ql)[D / 2],
                                              const int (&off)[D / 64], uint32_t* qfrag, int lane,
                                              uint32_t (&qb)[2 * C::KSTEPS], float& beta) {
    constexpr int CPL = D / 64;               // channel pairs per lane
    constexpr int HEAD = 8 * C::QSTRIDE;      // table distance between heads' hi columns
    constexpr int LOC = 4 * C::QSTRIDE;       // hi column -> lo column
    float bp[NQ];
#pragma unroll
    for (int h = 0; h < NQ; ++h) bp[h] = 0.f;
    __syncwarp();
    if (entries) {
        uint32_t sw[CPL], zw[CPL];             // steps / zeros of channels 2*CPL*l ..
        if constexpr (CPL == 2) {
            const uint2 sv = *reinterpret_cast<const uint2*>(entries + 8 * lane);
            const uint2 zv = *reinterpret_cast<const uint2*>(entries + 2 * D + 8 * lane);
            sw[0] = sv.x; sw[1] = sv.y; zw[0] = zv.x; zw[1] = zv.y;
        } else {
            sw[0] = *reinterpret_cast<const uint32_t*>(entries + 4 * lane);
            zw[0] = *reinterpret_cast<const uint32_t*>(entries + 2 * D + 4 * lane);
        }
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int cp = CPL * lane + j;
            const float2 z = unpack_f16x2(zw[j]);
#pragma unroll
            for (int h = 0; h < NQ; ++h) {
                const uint32_t hi = hmul2(qh[h][cp], sw[j]);
                const uint32_t lo = hfma2(ql[h][cp], sw[j], hfma2(qh[h][cp], sw[j], neg_f16x2(hi)));
                const float2 q2 = *reinterpret_cast<const float2*>(&qf[h][2 * cp]);
                bp[h] = fmaf(q2.x, z.x, fmaf(q2.y, z.y, bp[h]));
                qfrag[off[j] + h * HEAD] = hi;
                qfrag[off[j] + h * HEAD + LOC] = lo;
            }
        }
    } else {
        // the fp16 residual: hi / lo parts of the scaled query itself
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int cp = CPL * lane + j;
#pragma unroll
            for (int h = 0; h < NQ; ++h) {
                const float2 x = *reinterpret_cast<const float2*>(&qf[h][2 * cp]);
                const uint32_t hi = pack_f16x2(x.x, x.y);
                const float2 hf = unpack_f16x2(hi);
                qfrag[off[j] + h * HEAD] = hi;
                qfrag[off[j] + h * HEAD + LOC] = pack_f16x2(x.x - hf.x, x.y - hf.y);
            }
        }
    }
    const int i = lane & 3;
    beta = 0.f;
    if (entries) {
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) bp[h] += __shfl_xor_sync(kFull, bp[h], o);
            if (i == h) beta = bp[h] * 0x1p-24f;
        }
    }
    __syncwarp();
    if constexpr (KEEP) {
        const uint4* row = reinterpret_cast<const uint4*>(qfrag + lane * C::QSTRIDE);
#pragma unroll
        for (int v = 0; v < C::KSTEPS / 2; ++v) {
            const uint4 x = row[v];
            qb[4 * v] = x.x; qb[4 * v + 1] = x.y; qb[4 * v + 2] = x.z; qb[4 * v + 3] = x.w;
        }
    }
}

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// Register budget: four CTAs per SM (128 registers a thread); at head_dim 128
// with four query heads per kv head three, which leaves enough registers.
template <int D, int NQ>
struct MinCtas {
    static constexpr int value = (D == 128 && NQ == 4) ? 3 : 4;
};

// The value queue's pop, done by one warp: quantize the value of the popped
// token (block token tt; its fp16 row xs, a shared copy of ring row `row`)
// per token over groups of G channels with the shared formula, write its
// steps / zeros into its entry tile and OR its codes into its code tile
// (placement as in kivi.h, "Code tile": channel c = 16k + g + 8(r%2) and token
// tt%16 = 2i + 8(r/2) + half go to lane 4g + i, word PairPlace::word(k, r),
// bit PairPlace::bit(k, r) + 16 half), keep the codes (codes[c]) and the group
// steps / zeros (sz[j], sz[NGRP + j]) for queue_patch, then overwrite the ring
// row with ns (a shared copy of the appended value, which takes that row).
// Lane l handles channels [l*D/32, (l+1)*D/32).
template <int D, int BITS, int G>
__device__ __forceinline__ void queue_pop(uint8_t* part_v, __half* row, const __half* xs, const __half* ns, int tt,
                                          int lane, uint8_t* codes, __half* sz) {
    constexpr int CPL = D / 32, L = (1 << BITS) - 1, NGRP = D / G, W = D * BITS / 64;
    constexpr int TILE = 2 * D * BITS;
    using PP = PairPlace<BITS, true>;
    float x[CPL];
#pragma unroll
    for (int j = 0; j < CPL; j += 2) {
        const float2 v = unpack_f16x2(*reinterpret_cast<const uint32_t*>(xs + CPL * lane + j));
        x[j] = v.x;
        x[j + 1] = v.y;
    }
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int j = 1; j < CPL; ++j) { mn = fminf(mn, x[j]); mx = fmaxf(mx, x[j]); }
#pragma unroll
    for (int o = 1; o < G / CPL; o <<= 1) {     // the lanes of one channel group
        mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    }
    const int c0 = CPL * lane, gr = c0 / G, tile = tt / 16, tok = tt % 16;
    float s, z;
    __half s16, z16;
    group_step_zero(mn, mx, L, &s, &z, &s16, &z16);
    if (c0 % G == 0) {
        __half* ent = reinterpret_cast<__half*>(part_v + (G / 16) * TILE + tile * 64 * NGRP);
        const int at = gr * 16 + entry_pos(tok);
        ent[at] = s16;
        ent[16 * NGRP + at] = z16;
        sz[gr] = s16;
        sz[NGRP + gr] = z16;
    }
    uint32_t* words = reinterpret_cast<uint32_t*>(part_v + tile * TILE);
    const int r_hi = 2 * (tok / 8), ii = (tok % 8) / 2, half = tok % 2;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const int c = c0 + j, k = c / 16, cc = c % 16;
        const int r = cc / 8 + r_hi;
        const uint32_t code = nearest_code(x[j], s, z, L);
        codes[c] = (uint8_t)code;
        atomicOr(&words[(4 * (cc % 8) + ii) * W + PP::word(k, r)], code << (PP::bit(k, r) + 16 * half));
    }
    if constexpr (D == 128)
        *reinterpret_cast<uint2*>(row + 4 * lane) = *reinterpret_cast<const uint2*>(ns + 4 * lane);
    else
        *reinterpret_cast<uint32_t*>(row + 2 * lane) = *reinterpret_cast<const uint32_t*>(ns + 2 * lane);
}

// The popped token in the warp's staged copy of its tile pair (value code
// tiles at vt, their entry tiles at ve; tp = the token's index in the pair):
// the copy may predate the pop's writes, so its codes and entries go in here
// too (OR and equal stores: a copy that already has them is unchanged).
template <int D, int BITS, int G>
__device__ __forceinline__ void queue_patch(uint8_t* vt, uint8_t* ve, int tp, int lane, const uint8_t* codes,
                                            const __half* sz) {
    constexpr int CPL = D / 32, NGRP = D / G, W = D * BITS / 64, TILE = 2 * D * BITS;
    using PP = PairPlace<BITS, true>;
    const int tile = tp / 16, tok = tp % 16;
    uint32_t* words = reinterpret_cast<uint32_t*>(vt + tile * TILE);
    const int r_hi = 2 * (tok / 8), ii = (tok % 8) / 2, half = tok % 2;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const int c = CPL * lane + j, k = c / 16, cc = c % 16;
        const int r = cc / 8 + r_hi;
        atomicOr(&words[(4 * (cc % 8) + ii) * W + PP::word(k, r)], (uint32_t)codes[c] << (PP::bit(k, r) + 16 * half));
    }
    if (lane < NGRP) {
        __half* ent = reinterpret_cast<__half*>(ve + tile * 64 * NGRP);
        ent[lane * 16 + entry_pos(tok)] = sz[lane];
        ent[16 * NGRP + lane * 16 + entry_pos(tok)] = sz[NGRP + lane];
    }
}

// MODE kModeFused: the call appends a token (Args::new_row) the kernel reads
// from its inputs and stores in the cache; kModePaged: blocks are addressed
// through the block table and every sequence has its own length and appended
// row.  Separate instances, so that plain decode calls carry none of that code.
template <int D, int BITS, int NQ, int G, int MODE>
__global__ void __launch_bounds__(kThreads, MinCtas<D, NQ>::value)
    decode_mma_kernel(const __grid_constant__ typename ArgsOf<MODE>::type a) {
    constexpr bool FUSED = MODE != kModePlain, PAGED = MODE == kModePaged, FIFO = MODE == kModeFifo;
    using C = Cfg<D, BITS, NQ, G>;
    constexpr int KS = C::KSTEPS, W = C::W, NGRP = C::NGRP, GB = C::GB, NBF = C::NBF;
    // per warp: the scaled query (fp32) and the fp16 hi / lo parts of it times
    // the code scale 2^-(BITS*pos), for the slot the warp works on
    __shared__ __align__(16) float qf_all[kWarps][NQ][D];
    __shared__ uint32_t qhc_all[kWarps][NQ][D / 2], qlc_all[kWarps][NQ][D / 2];
    __shared__ __align__(16) uint32_t qfrag_all[kWarps][32 * C::QSTRIDE];
    __shared__ __align__(8) uint64_t full_bar[kWarps][C::STAGES];
    // paged, per warp: the segment's block-table entries as byte offsets of the
    // blocks' key parts (refilled past kPageCache blocks) and the sticky flag
    // of an entry outside the pool
    __shared__ PageCache pc_all[PAGED ? kWarps : 1];
    // value queue, per warp: the popped token's fp16 row and the appended value
    // (shared copies), its codes and group steps / zeros
    __shared__ __align__(16) __half poprow_all[FIFO ? kWarps : 1][2][D];
    __shared__ uint8_t popc_all[FIFO ? kWarps : 1][D];
    __shared__ __half popsz_all[FIFO ? kWarps : 1][2 * NGRP];
    extern __shared__ __align__(128) uint8_t dyn_smem[];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, i = lane & 3;
#define qf (qf_all[warp])
#define qhc_s (qhc_all[warp])
#define qlc_s (qlc_all[warp])
    uint32_t* qfrag = qfrag_all[warp];
    uint8_t* ring = dyn_smem + warp * C::STAGES * C::STAGE_BYTES;
    // value queue: the warp's logits of its mixed pairs, kept for the second pass
    auto mixbuf = [&](int idx) {
        return reinterpret_cast<float4*>(dyn_smem + C::DYN_SMEM) + warp * kMaxMixPairs * 32 + idx;
    };
    uint64_t* bars = full_bar[warp];
    for (int idx = lane; idx < 32 * C::QSTRIDE; idx += 32) qfrag[idx] = 0u;   // unused columns stay 0
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < C::STAGES; ++st) mbar_init(&bars[st], 1);
        // failure-detection test hook: warp 0 of CTA 0 expects bytes that never come
        // on its first stage, so its first bounded wait runs out
        if (a.stall_bytes && blockIdx.x == 0 && warp == 0) mbar_expect_tx_only(smem_u32(&bars[0]), (uint32_t)a.stall_bytes);
        fence_mbar_init();
        if constexpr (PAGED) pc_all[warp].bad = 0;
    }
    __syncwarp();

    int qoff[D / 64];     // this lane's Qt table offsets (channel pairs (D/64)*lane + j)
#pragma unroll
    for (int j = 0; j < D / 64; ++j) {
        const int cp = (D / 64) * lane + j, cc = (2 * cp) & 15;
        qoff[j] = ((cc & 7) >> 1) * C::QSTRIDE + 2 * (cp >> 3) + (cc >> 3);
    }
    const uint32_t ring_u32 = smem_u32(ring), bars_u32 = smem_u32(bars);
    const long long vdelta = PAGED ? a.part_bytes : a.NB * a.part_bytes;   // key part -> value part of a block
    // this lane's B column for the values: head hP, group slot jP, hi/lo
    const int colP = g >> 1, hP = colP / GB, jP = colP % GB;
    const bool lo_col = (g & 1) != 0;
    const bool col_ok = hP < NQ;
    // this lane's output columns (2i, 2i+1): head hO, group slot jO
    const int hO = i / GB, jO = i % GB;
    // byte offset, inside an entry tile, of the steps of this lane's tokens
    // 2i, 2i+1, 2i+8, 2i+9 (adjacent in the row order) for group fragment 0;
    // the zeros follow 32*NGRP bytes later, fragment f adds 32*f*GB
    const uint32_t eoff = 32u * jP + 8u * i;
    const long long tiles_bytes = (long long)C::TPB * a.tile_bytes;

    float m = -INFINITY, l = 0.f;
    bool fresh = true;    // no tile of the current segment has been counted yet
    float o[KS][4];
    float zeta[NBF];
    // the key B fragments, held in registers or read from the warp's table
    constexpr bool QB_REGS = NQ > 1;
    uint32_t qb[2 * KS];
    // the key B fragment of k-step kk (see build_q_frags)
    auto qbk = [&](const int kk) -> uint2 {
        if constexpr (QB_REGS)
            return make_uint2(qb[2 * kk], qb[2 * kk + 1]);
        else
            return *reinterpret_cast<const uint2*>(qfrag + lane * C::QSTRIDE + 2 * kk);
    };
    float beta = 0.f;
    uint32_t status = 0;  // 1: a bulk copy did not complete in time (sticky)
    uint32_t item = 0;    // ring stages this warp has consumed (stage index and phase)

    // Online softmax step over two tiles: sc * unit = logits of tokens g, g+8
    // of tile A and of tile B (head i); p receives their probabilities.
    auto softmax = [&](const float (&sc)[4], float (&p)[4], float unit) {
        float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
        const float mn = fmaxf(m, mt * unit);
        if (fresh) {
            m = mn;          // the segment's first tiles: o, zeta and l are still zero
            fresh = false;
        } else if (__any_sync(kFull, mn > m)) {
            const float alpha = fast_exp2(m - mn);
            l *= alpha;
            const float ao = __shfl_sync(kFull, alpha, (lane & ~3) | (hO < NQ ? hO : 0));
#pragma unroll
            for (int t = 0; t < KS; ++t) { o[t][0] *= ao; o[t][1] *= ao; o[t][2] *= ao; o[t][3] *= ao; }
            const float az = __shfl_sync(kFull, alpha, col_ok ? hP : 0);
#pragma unroll
            for (int f = 0; f < NBF; ++f) zeta[f] *= az;
            m = mn;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = fast_exp2(fmaf(sc[j], unit, -m));
        l += (p[0] + p[1]) + (p[2] + p[3]);
    };
    // probabilities of tokens 2i, 2i+1, 2i+8, 2i+9 of head hP from (p0, p1) =
    // the probabilities of tokens g, g+8 held by every lane
    auto gather = [&](float p0, float p1, float (&pr)[4]) {
        const int src = 8 * i + (col_ok ? hP : 0);
        pr[0] = __shfl_sync(kFull, p0, src);        // token 2i
        pr[1] = __shfl_sync(kFull, p0, src + 4);    // token 2i+1
        pr[2] = __shfl_sync(kFull, p1, src);        // token 2i+8
        pr[3] = __shfl_sync(kFull, p1, src + 4);    // token 2i+9
        if (!col_ok) pr[0] = pr[1] = pr[2] = pr[3] = 0.f;
    };
    // B fragment of P*step for one value fragment from the 4 tokens' (s, z) entries.
    auto p_frag = [&](const float (&pr)[4], uint32_t ph01, uint32_t ph89, uint32_t pl01, uint32_t pl89,
                      uint2 sv, uint2 zv, uint32_t& b0, uint32_t& b1, float& z) {
        const uint32_t s01 = sv.x, s89 = sv.y;
        const uint32_t h01 = hmul2(ph01, s01), h89 = hmul2(ph89, s89);
        const uint32_t l01 = hfma2(pl01, s01, hfma2(ph01, s01, neg_f16x2(h01)));
        const uint32_t l89 = hfma2(pl89, s89, hfma2(ph89, s89, neg_f16x2(h89)));
        b0 = lo_col ? l01 : h01;
        b1 = lo_col ? l89 : h89;
        const float2 z01 = unpack_f16x2(zv.x);
        const float2 z89 = unpack_f16x2(zv.y);
        z = fmaf(pr[0], z01.x, fmaf(pr[1], z01.y, fmaf(pr[2], z89.x, fmaf(pr[3], z89.y, z))));
    };
    auto split_p = [&](const float (&pr)[4], uint32_t& ph01, uint32_t& ph89, uint32_t& pl01, uint32_t& pl89) {
        ph01 = pack_f16x2(pr[0], pr[1]);
        ph89 = pack_f16x2(pr[2], pr[3]);
        const float2 f01 = unpack_f16x2(ph01), f89 = unpack_f16x2(ph89);
        pl01 = pack_f16x2(pr[0] - f01.x, pr[1] - f01.y);
        pl89 = pack_f16x2(pr[2] - f89.x, pr[3] - f89.y);
    };
    const uint32_t lane_words = (uint32_t)(lane * W * 4);
    auto lds_words = [&](uint32_t src, uint32_t (&w)[W]) {   // this lane's words of a tile at src
        if constexpr (W % 4 == 0) {
#pragma unroll
            for (int v = 0; v < W / 4; ++v) {
                const uint4 x = lds128(src + lane_words + 16 * v);
                w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
            }
        } else {
            const uint2 x = lds64(src + lane_words);
            w[0] = x.x; w[1] = x.y;
        }
    };

    // This warp's share of the call's work: the units starting in its weight
    // range [pos, pe); one partial result per slot it touches.  Warps are the
    // workers of the map (wm.n of them); the warps of a CTA share nothing but
    // the SM.
    const WorkMap& wm = a.wm;
    const long long cta = blockIdx.x;
    const long long gw = cta * kWarps + warp;
    long long pos = gw < wm.n ? map_begin(wm, gw) : wm.Wt;
    const long long pe = gw < wm.n ? map_begin(wm, gw + 1) : wm.Wt;
    bool first_seg = true;
    // The programmatic-dependent launch point: wait for the preceding kernel,
    // let the merge kernel start launching, store the fused append's rows.
    // Every warp passes it once (its first segment, or after its loop if it
    // has none), after issuing its first copies: with early_ok those read only
    // quantized blocks, which the preceding kernel never writes (the library's
    // last kernel on a cache copies residual rows, or is a decode's merge,
    // which lets this kernel launch only after that decode, a writer of blocks
    // when it pops the value queue, has finished); the query, the residual
    // rows and the workspace are touched only after it.
    auto dependency_point = [&]() {
        griddepcontrol_wait();
        griddepcontrol_launch_dependents();       // the merge kernel may start launching
        if constexpr (PAGED) {
            // the fused append of a paged call: each sequence's own new row
            constexpr int CPR = D * 2 / 16;
            if (a.new_k != nullptr) {
                const long long nsl = (long long)a.n_seqs * a.Hkv;
                for (long long idx = cta * kThreads + tid; idx < nsl * 2 * CPR;
                     idx += (long long)gridDim.x * kThreads) {
                    const long long sl = idx / (2 * CPR);
                    const int rem = (int)(idx - sl * 2 * CPR), is_v = rem >= CPR, c16 = rem % CPR;
                    const int si = (int)(sl / a.Hkv), h2 = (int)(sl % a.Hkv);
                    const int nr = a.seqs[si].new_row;
                    if (nr < 0) continue;
                    const uint4* src = reinterpret_cast<const uint4*>((is_v ? a.new_v : a.new_k) + sl * D) + c16;
                    uint8_t* rows = const_cast<uint8_t*>(a.cache) + (is_v ? a.v_resid_off : a.k_resid_off);
                    const long long drow = ((long long)a.seqs[si].seq * a.Hkv + h2) * a.R + nr;
                    reinterpret_cast<uint4*>(reinterpret_cast<__half*>(rows) + drow * D)[c16] = *src;
                }
            }
        } else if (FUSED && a.new_row >= 0) {
            // the fused append: store every slot's new row in the cache, 16
            // bytes a thread over the grid (this call reads that row from the
            // inputs, never from the cache)
            constexpr int CPR = D * 2 / 16;       // 16-byte chunks per row
            const long long nslots = (long long)(wm.Wt / wm.Ws);
            for (long long idx = cta * kThreads + tid; idx < nslots * 2 * CPR;
                 idx += (long long)gridDim.x * kThreads) {
                const long long sl = idx / (2 * CPR);
                const int rem = (int)(idx - sl * 2 * CPR), is_v = rem >= CPR, c16 = rem % CPR;
                // value queue with a pop: the new value takes the popped token's
                // ring row, written by the warp that quantizes that token
                if (FIFO && is_v && a.pop >= 0) continue;
                const uint4* src = reinterpret_cast<const uint4*>((is_v ? a.new_v : a.new_k) + sl * D) + c16;
                uint8_t* rows = const_cast<uint8_t*>(a.cache) + (is_v ? a.v_resid_off : a.k_resid_off);
                // value queue: the new value goes to ring row (its slot position) % R
                const long long vr_row = FIFO && is_v ? (32 * wm.P + a.new_row) % a.R : a.new_row;
                reinterpret_cast<uint4*>(reinterpret_cast<__half*>(rows) + (sl * a.R + vr_row) * D)[c16] = *src;
            }
        }
    };
    while (pos < pe) {
        // the slot holding weight position pos: weights [w0, w0 + Ws), P quantized
        // pairs then PR residual pairs
        long long w0, Ws, P, PR, M = 0;   // M: mixed pairs (value queue)
        int b, hk;               // query / output row (batch row or call sequence), kv head
        long long rslot, islot;  // residual slot; row of the fused append's inputs
        int n_res, nrow;         // residual rows; the fused append's row (-1: none)
        long long trow = 0;      // paged: offset of the sequence's block-table row
        if constexpr (PAGED) {
            int lo = 0, hi = a.n_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.seqs[mid].start <= pos) lo = mid; else hi = mid - 1;
            }
            const PagedSeq& sq = a.seqs[lo];
            P = sq.P;
            PR = (sq.n_resid + 31) / 32;
            Ws = wm.S0 + slot_weight(wm, P, 0, PR);
            hk = (int)((pos - sq.start) / Ws);
            w0 = sq.start + hk * Ws;
            b = lo;
            rslot = (long long)sq.seq * a.Hkv + hk;
            islot = (long long)lo * a.Hkv + hk;
            n_res = sq.n_resid;
            nrow = sq.new_row;
            trow = (long long)sq.seq * a.max_blocks;
        } else {
            const long long slot = pos / wm.Ws;
            w0 = slot * wm.Ws;
            Ws = wm.Ws;
            P = wm.P;
            PR = wm.PR;
            M = wm.M;
            b = (int)(slot / a.Hkv);
            hk = (int)(slot % a.Hkv);
            rslot = islot = slot;
            n_res = a.n_resid;
            nrow = a.new_row;
        }
        const long long NU = P + PR;
        const long long u0 = first_unit_at_p(wm, P, M, pos - w0);
        if (u0 >= NU) { pos = w0 + Ws; continue; }
        if (w0 + unit_start_p(wm, P, M, u0) >= pe) {
            // no unit of the slot starts in this warp's range: if the range lies
            // between the slot's first and last unit starts, the slot still
            // counts this warp's partial, so write it empty (weight 0)
            if (u0 > 0) {
                // (the workspace only after the preceding kernel, which may read it)
                if (first_seg) {
                    first_seg = false;
                    dependency_point();
                }
                const long long part = gw - map_owner(wm, w0 + wm.S0);
                for (int idx = lane; idx < NQ * (D + 4); idx += 32) {
                    const int h = idx / (D + 4), c = idx % (D + 4);
                    float* pw = a.ws + ((long long)(b * a.Hq + hk * NQ + h) * kPartialSlots + part) * partial_stride(D);
                    pw[c] = c == 0 ? -INFINITY : 0.f;
                }
            }
            break;
        }
        const long long u1 = first_unit_at_p(wm, P, M, min(pe - w0, Ws));
        const int p0 = (int)min(u0, P), p1 = (int)min(u1, P);                  // quantized pairs
        const int r0 = (int)(max(u0, P) - P), r1 = (int)(max(u1, P) - P);      // residual pairs
        const int part = (int)(gw - map_owner(wm, w0 + wm.S0));
        // ---- this warp's run of pairs, two tiles per ring stage ----
        const int wb = p0, we = p1;
        const int npairs = status ? 0 : we - wb;   // after a failed copy: no more copies
        // value queue: this warp's pairs from mix_first() on have quantized keys
        // and queued values (recomputed where used, not held across the loop)
        auto mix_first = [&]() { return max(wb, (int)(a.lqv >> 5)); };
        auto need_ksz = [&](int pr) { return pr == wb || ((2 * pr) % C::TPB) == 0; };
        // the preceding kernel wrote blocks (and, paged, block-table entries): wait
        // before the first copy and before the first table read
        if (first_seg && !a.early_ok) griddepcontrol_wait();
        // lane 0's copy cursor: key part of the block of the next pair to fetch, tile in block
        // (paged: the block's offset in the warp's page cache, which the whole
        // warp fills from the table at the segment start, so no copy waits on a
        // table load of its own)
        const uint8_t* kcur;
        int pidx = 0;            // paged: lane 0's entry of the page cache
        // the pairs whose copies may be issued: paged, those whose blocks are in
        // the page cache (a longer segment runs in parts, the cache refilled
        // between them, so that the pair loop carries no refill)
        int kiss = npairs;
        if constexpr (PAGED) {
            kcur = a.cache;
            if (npairs > 0) {
                PageCache& pcw = pc_all[warp];
                const int blk0 = (2 * wb) / C::TPB;
                const int nb = min((2 * we - 1) / C::TPB - blk0 + 1, kPageCache);
                const long long pstride = (long long)a.Hkv * 2 * a.part_bytes, hoff = (long long)hk * 2 * a.part_bytes;
                fill_pages(pcw, a.table + trow, blk0, nb, a.max_blocks, a.n_pages, pstride, hoff, lane, 32);
                if (lane == 0) {
                    pcw.trow = a.table + trow;
                    pcw.hoff = hoff;
                    pcw.first = blk0;
                    pcw.last = (2 * we - 1) / C::TPB;
                }
                __syncwarp();
                kiss = min(npairs, (blk0 + kPageCache) * (C::TPB / 2) - wb);
            }
        } else {
            kcur = a.cache + rslot * a.slot_bytes + (long long)((2 * wb) / C::TPB) * a.part_bytes;
        }
        int tcur = (2 * wb) % C::TPB;
        bool first = true;
        auto issue_next = [&](uint32_t it) {          // lane 0: next pair -> ring stage of item it
            const uint32_t st = it % C::STAGES;
            const uint32_t dst = ring_u32 + st * C::STAGE_BYTES, bar = bars_u32 + 8 * st;
            const bool kz = first || tcur == 0;
            const uint8_t* kp;
            if constexpr (PAGED) {
                // (an entry outside the pool was flagged and turned into page 0)
                kp = a.cache + pc_all[warp].off[pidx];
            } else {
                kp = kcur;
            }
            const uint8_t* vcur = kp + vdelta;
            if constexpr (C::WHOLE) {
                // the block's key part and value part, each one contiguous copy
                mbar_expect_tx_u32(bar, C::STAGE_BYTES);
                tma_1d_u32(dst + C::KT, kp, 2 * C::TILE + C::KSZ, bar);
                tma_1d_u32(dst + C::VT, vcur, 2 * C::TILE + 2 * C::ENT, bar);
            } else {
                mbar_expect_tx_u32(bar, 4 * C::TILE + 2 * C::ENT + (kz ? C::KSZ : 0));
                tma_1d_u32(dst + C::KT, kp + tcur * C::TILE, 2 * C::TILE, bar);
                if (kz) tma_1d_u32(dst + C::KE, kp + tiles_bytes, C::KSZ, bar);
                tma_1d_u32(dst + C::VT, vcur + tcur * C::TILE, 2 * C::TILE, bar);
                tma_1d_u32(dst + C::VE, vcur + tiles_bytes + tcur * C::ENT, 2 * C::ENT, bar);
            }
            first = false;
            tcur += 2;
            if (tcur == C::TPB) {
                tcur = 0;
                if constexpr (PAGED) {
                    ++pidx;
                } else {
                    kcur += a.part_bytes;
                }
            }
        };
        if (lane == 0) {
            for (int k = 0; k < C::STAGES && k < kiss; ++k) issue_next(item + k);
            // the fp16 rows this segment reads with plain loads, into L2 ahead
            // of them: its residual pairs' key and value rows (value queue:
            // ring rows) and, with the value queue, the queued values of its
            // mixed pairs and the popped token's row
            const __half* kr0 = reinterpret_cast<const __half*>(a.cache + a.k_resid_off) + rslot * a.R * D;
            const __half* vr0 = reinterpret_cast<const __half*>(a.cache + a.v_resid_off) + rslot * a.R * D;
            const int nr = min(32 * r1, n_res) - 32 * r0;
            if (nr > 0) {
                prefetch_l2(kr0 + 32LL * r0 * D, (uint32_t)(nr * D * 2));
                if constexpr (FIFO) prefetch_ring_rows<D>(vr0, (int)(32 * P) + 32 * r0, nr, a.R);
                else prefetch_l2(vr0 + 32LL * r0 * D, (uint32_t)(nr * D * 2));
            }
            if constexpr (FIFO) {
                const int tlo = (int)max(a.lqv, 32LL * mix_first()), thi = 32 * we;
                prefetch_ring_rows<D>(vr0, tlo, thi - tlo, a.R);
                if (a.pop >= 0 && wb <= a.pop / 32 && a.pop / 32 < we) prefetch_ring_rows<D>(vr0, (int)a.pop, 1, a.R);
            }
        }
        if (first_seg) {
            first_seg = false;
            dependency_point();
        }
        // value queue: the warp owning the pair of position a.pop quantizes that
        // value into its block after the query setup below (the ring row then
        // takes the appended value); both rows are copied to shared memory
        // meanwhile
        const int tpop = FIFO && a.pop >= 0 && wb <= a.pop / 32 && a.pop / 32 < we ? (int)(a.pop / 32) : -1;
        if constexpr (FIFO) {
            constexpr int CPR = D * 2 / 16;          // 16-byte chunks per row
            if (tpop >= 0 && lane < 2 * CPR) {
                const __half* src = lane < CPR ? reinterpret_cast<const __half*>(a.cache + a.v_resid_off) +
                                                     (rslot * a.R + (int)a.pop % a.R) * D
                                               : a.new_v + islot * D;
                cp_async16(&poprow_all[warp][lane / CPR][8 * (lane % CPR)], src + 8 * (lane % CPR));
            }
        }
        __syncwarp();
        for (int idx = lane; idx < NQ * D / 2; idx += 32) {
            const int j = idx / (D / 2), cp = idx % (D / 2);
            const float2 qv = __half22float2(
                *reinterpret_cast<const __half2*>(a.q + ((long long)b * a.Hq + hk * NQ + j) * D + 2 * cp));
            const float x0 = qv.x * a.scale_log2, x1 = qv.y * a.scale_log2;
            qf[j][2 * cp] = x0;
            qf[j][2 * cp + 1] = x1;
            // channels 2cp, 2cp+1 have class cp / 4: their codes read as code * 2^(BITS*pos - 24)
            const float cs = pow2i(-BITS * ((cp >> 2) % (8 / BITS)));
            const float y0 = x0 * cs, y1 = x1 * cs;
            const uint32_t hic = pack_f16x2(y0, y1);
            const float2 hcf = unpack_f16x2(hic);
            qhc_s[j][cp] = hic;
            qlc_s[j][cp] = pack_f16x2(y0 - hcf.x, y1 - hcf.y);
        }
        if constexpr (FIFO) {
            if (tpop >= 0) {
                // the pop (this pair's staged copy gets its codes in the pair loop)
                cp_async_wait_all();
                __syncwarp();
                uint8_t* part_v = const_cast<uint8_t*>(a.cache) + rslot * a.slot_bytes + (a.NB + a.pop / G) * a.part_bytes;
                __half* row = reinterpret_cast<__half*>(const_cast<uint8_t*>(a.cache) + a.v_resid_off) +
                              (rslot * a.R + (int)a.pop % a.R) * D;
                queue_pop<D, BITS, G>(part_v, row, poprow_all[warp][0], poprow_all[warp][1], (int)(a.pop % G), lane,
                                      popc_all[warp], popsz_all[warp]);
            }
        }
        __syncwarp();

        m = -INFINITY; l = 0.f;
        fresh = true;
#pragma unroll
        for (int t = 0; t < KS; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
#pragma unroll
        for (int f = 0; f < NBF; ++f) zeta[f] = 0.f;

        int k = 0;
        // The pair loop, in two runs for the value queue: pairs from kq on (the
        // mixed pairs and the popped token's pair) take the queue's steps, the
        // pairs before them the plain body, so that the common case carries none
        // of the queue's branches.
        int kq = npairs;
        if constexpr (FIFO) {
            int first = (int)(a.lqv >> 5);                 // the first pair with queued values
            if (tpop >= 0 && tpop < first) first = tpop;
            kq = min(max(first - wb, 0), npairs);
        }
        auto pair_run = [&](auto queue_steps, int kend) {
        constexpr bool QS = decltype(queue_steps)::value;
        for (; k < kend; ++k) {
            const uint32_t it = item + k;
            const int st = (int)(it % C::STAGES);
            if (!__all_sync(kFull, mbar_wait(&bars[st], (it / C::STAGES) & 1u))) break;
            const uint8_t* stage = ring + st * C::STAGE_BYTES;
            const uint32_t stage_u32 = ring_u32 + st * C::STAGE_BYTES;
            const int pr = wb + k;
            if constexpr (FIFO && QS) {
                if (a.pop >= 0 && pr == (int)(a.pop >> 5)) {   // only the popping warp has this pair
                    // the popped token's codes into this pair's staged copy
                    queue_patch<D, BITS, G>(const_cast<uint8_t*>(stage) + C::VT, const_cast<uint8_t*>(stage) + C::VE,
                                            (int)(a.pop % 32), lane, popc_all[warp], popsz_all[warp]);
                    __syncwarp();
                }
            }
            if (need_ksz(pr))
                build_q_frags<C, D, NQ, QB_REGS>(stage + C::KE, qf, qhc_s, qlc_s, qoff, qfrag, lane, qb, beta);
            // keys: logits of tokens g, g+8 of both tiles for head i
            float sc[4];
            if constexpr (BITS == 8) {
                // one tile at a time: a lane's 16 words per tile, shifted in place
                float ca[4] = {0.f, 0.f, 0.f, 0.f};
                float cb[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    uint32_t w[W];
                    lds_words(stage_u32 + C::KT, w);
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        uint32_t fa[4];
                        a_frag_inline<BITS, false, W>(w, kk, fa);
                        const uint2 bq = qbk(kk);
                        mma16816(ca, fa, bq.x, bq.y);
                    }
                }
                {
                    uint32_t w[W];
                    lds_words(stage_u32 + C::KT + C::TILE, w);
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        uint32_t fb[4];
                        a_frag_inline<BITS, false, W>(w, kk, fb);
                        const uint2 bq = qbk(kk);
                        mma16816(cb, fb, bq.x, bq.y);
                    }
                }
                // the block's zero-point term joins after the MMAs, so its
                // reduction over the lanes runs beside them
                sc[0] = ca[0] + (ca[1] + beta);
                sc[1] = ca[2] + (ca[3] + beta);
                sc[2] = cb[0] + (cb[1] + beta);
                sc[3] = cb[2] + (cb[3] + beta);
            } else {
                uint32_t wa[W], wbw[W], wa8[W], wb8[W];
                lds_words(stage_u32 + C::KT, wa);
                lds_words(stage_u32 + C::KT + C::TILE, wbw);
#pragma unroll
                for (int x = 0; x < W; ++x) { wa8[x] = wa[x] >> 8; wb8[x] = wbw[x] >> 8; }
                float ca[4] = {0.f, 0.f, 0.f, 0.f};
                float cb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t fa[4], fb[4];
                    a_frag<BITS, false, W>(wa, wa8, kk, fa);
                    a_frag<BITS, false, W>(wbw, wb8, kk, fb);
                    const uint2 bq = qbk(kk);
                    mma16816(ca, fa, bq.x, bq.y);
                    mma16816(cb, fb, bq.x, bq.y);
                }
                // the block's zero-point term joins after the MMAs, so its
                // reduction over the lanes runs beside them
                sc[0] = ca[0] + (ca[1] + beta);
                sc[1] = ca[2] + (ca[3] + beta);
                sc[2] = cb[0] + (cb[1] + beta);
                sc[3] = cb[2] + (cb[3] + beta);
            }
            bool live = true;                          // the pair has a token to count in this pass
            if constexpr (FIFO && QS) {
                const long long t0 = 32LL * pr;
                if (t0 + 32 > a.lqv) {
                    // keys quantized, some values still in the queue: keep the logits
                    // for the second pass; here only the value-quantized tokens count
                    *mixbuf((pr - mix_first()) * 32 + lane) = make_float4(sc[0], sc[1], sc[2], sc[3]);
                    if (t0 + g >= a.lqv) sc[0] = -INFINITY;
                    if (t0 + g + 8 >= a.lqv) sc[1] = -INFINITY;
                    if (t0 + 16 + g >= a.lqv) sc[2] = -INFINITY;
                    if (t0 + 24 + g >= a.lqv) sc[3] = -INFINITY;
                    live = t0 < a.lqv;
                }
            }
            if (live) {
                // small tiles (at most four words a lane): both value tiles' words
                // are loaded before the softmax, whose shuffles then hide their
                // latency; the entries too in the fused and queue instances
                // (plain decode calls measured 0.5-1.2% faster loading them after
                // it, paged calls 1%; the other two were faster as here)
                constexpr bool HOIST = BITS != 8 && W <= 4, HOIST_E = HOIST && FUSED && !PAGED;
                uint32_t wvh[2][W];
                uint2 svh[2][NBF], zvh[2][NBF];
                if constexpr (HOIST) {
                    lds_words(stage_u32 + C::VT, wvh[0]);
                    lds_words(stage_u32 + C::VT + C::TILE, wvh[1]);
                }
                if constexpr (HOIST_E) {
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint32_t ve = stage_u32 + C::VE + t * C::ENT + eoff;
#pragma unroll
                        for (int f = 0; f < NBF; ++f) {
                            svh[t][f] = lds64(ve + 32u * GB * f);
                            zvh[t][f] = lds64(ve + 32u * (NGRP + GB * f));
                        }
                    }
                }
                float p[4];
                softmax(sc, p, 0x1p24f);                   // scores are in units of 2^-24
                // values, tile by tile
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    float prb[4];
                    gather(p[2 * t], p[2 * t + 1], prb);
                    uint32_t ph01, ph89, pl01, pl89;
                    split_p(prb, ph01, ph89, pl01, pl89);
                    const uint32_t ve = stage_u32 + C::VE + t * C::ENT + eoff;
                    uint32_t pb[NBF][2];
#pragma unroll
                    for (int f = 0; f < NBF; ++f) {
                        const uint2 sv = HOIST_E ? svh[t][f] : lds64(ve + 32u * GB * f);
                        const uint2 zv = HOIST_E ? zvh[t][f] : lds64(ve + 32u * (NGRP + GB * f));
                        p_frag(prb, ph01, ph89, pl01, pl89, sv, zv, pb[f][0], pb[f][1], zeta[f]);
                    }
                    uint32_t wv[W];
                    if constexpr (HOIST) {
#pragma unroll
                        for (int x = 0; x < W; ++x) wv[x] = wvh[t][x];
                    } else {
                        lds_words(stage_u32 + C::VT + t * C::TILE, wv);
                    }
                    if constexpr (BITS == 8) {
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            uint32_t af[4];
                            a_frag_inline<BITS, true, W>(wv, mt, af);
                            const int f = (16 * mt / G) / GB;
                            mma16816(o[mt], af, pb[f][0], pb[f][1]);
                        }
                    } else {
                        uint32_t wv8[W];
#pragma unroll
                        for (int x = 0; x < W; ++x) wv8[x] = wv[x] >> 8;
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            uint32_t af[4];
                            a_frag<BITS, true, W>(wv, wv8, mt, af);
                            const int f = (16 * mt / G) / GB;
                            mma16816(o[mt], af, pb[f][0], pb[f][1]);
                        }
                    }
                }
            }
            __syncwarp();                              // every lane is done with this stage
            if (lane == 0 && k + C::STAGES < kiss) {
                fence_proxy_async();
                issue_next(it + C::STAGES);
            }
        }
        };
        if constexpr (PAGED) {
            for (;;) {
                pair_run(BoolTag<false>{}, kiss);
                if (k < kiss || kiss >= npairs) break;   // a copy timed out, or the segment is done
                // the segment's next blocks into the page cache (up to its last
                // block: later table entries are not the sequence's), then the
                // next part's first copies
                PageCache& pcw = pc_all[warp];
                const int f = pcw.first + kPageCache;
                fill_pages(pcw, pcw.trow, f, min(pcw.last - f + 1, kPageCache), a.max_blocks, a.n_pages,
                           (long long)a.Hkv * 2 * a.part_bytes, pcw.hoff, lane, 32);
                __syncwarp();
                if (lane == 0) pcw.first = f;
                pidx = 0;
                kiss = min(npairs, (f + kPageCache) * (C::TPB / 2) - wb);
                if (lane == 0) {
                    fence_proxy_async();
                    for (int u = k; u < k + C::STAGES && u < kiss; ++u) issue_next(item + u);
                }
                __syncwarp();
            }
        } else {
            pair_run(BoolTag<false>{}, kq);
            if constexpr (FIFO) {
                if (k == kq) pair_run(BoolTag<true>{}, npairs);
            }
        }
        if (k < npairs) {
            // a copy timed out: flag it, wait (bounded) for this warp's copies in
            // flight, and issue no more copies in this kernel
            status = 1;
            for (int u = k; u < kiss && u < k + C::STAGES; ++u)
                mbar_wait(&bars[(item + u) % C::STAGES], ((item + u) / C::STAGES) & 1u);
        }
        item += (uint32_t)npairs;
        // the quantized tiles' value sums are in units of 2^(BITS*pos - 24),
        // pos = (channel / 8) % (8 / BITS): rows g and g+8 of m-tile mt have
        // classes 2mt and 2mt+1
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const float u0 = pow2i(24 - BITS * ((2 * mt) % (8 / BITS)));
            const float u1 = pow2i(24 - BITS * ((2 * mt + 1) % (8 / BITS)));
            o[mt][0] *= u0; o[mt][1] *= u0; o[mt][2] *= u1; o[mt][3] *= u1;
        }
        if constexpr (FIFO) {
            // ---- value queue: the queued tokens of this warp's mixed pairs, with the
            // logits kept in the first pass and the values from the ring's fp16 rows ----
            const int me = wb + k;                    // pairs this warp processed
            const __half* ring_v = reinterpret_cast<const __half*>(a.cache + a.v_resid_off) + rslot * a.R * D;
            const int mix0 = mix_first();
            for (int pr = mix0; pr < me; ++pr) {
                const float4 s4 = *mixbuf((pr - mix0) * 32 + lane);
                float sc[4] = {s4.x, s4.y, s4.z, s4.w};
                const long long t0 = 32LL * pr;       // the first pass counted the tokens below lqv
                if (t0 + g < a.lqv) sc[0] = -INFINITY;
                if (t0 + g + 8 < a.lqv) sc[1] = -INFINITY;
                if (t0 + 16 + g < a.lqv) sc[2] = -INFINITY;
                if (t0 + 24 + g < a.lqv) sc[3] = -INFINITY;
                float p[4];
                softmax(sc, p, 0x1p24f);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    float prb[4];
                    gather(p[2 * t], p[2 * t + 1], prb);
                    uint32_t ph01, ph89, pl01, pl89;
                    split_p(prb, ph01, ph89, pl01, pl89);
                    const uint32_t pb0 = lo_col ? pl01 : ph01, pb1 = lo_col ? pl89 : ph89;
                    // rows g, g+8 of the 16 tokens: queued values sit at ring row token % R
                    const long long tg = t0 + 16 * t + g, tg8 = tg + 8;
                    const __half* vg = ring_v + (long long)((int)tg % a.R) * D;
                    const __half* vg8 = ring_v + (long long)((int)tg8 % a.R) * D;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        uint32_t af[4];
                        vt_frag_rows<D>(vg, vg8, tg >= a.lqv, tg8 >= a.lqv, mt, i, af);
                        mma16816(o[mt], af, pb0, pb1);
                    }
                }
            }
        }
        // ---- the segment's residual pairs: 32 fp16 rows each, A operands straight from memory ----
        const int rb = r0, re = r1;
        if (rb < re) {
            const __half* kr = reinterpret_cast<const __half*>(a.cache + a.k_resid_off) + rslot * a.R * D;
            const __half* vr = reinterpret_cast<const __half*>(a.cache + a.v_resid_off) + rslot * a.R * D;
            const int n = n_res;
            // row rr of the residual: the fused append's token comes from its input
            auto krow = [&](int rr) {
                return FUSED && rr == nrow ? a.new_k + islot * D : kr + (long long)rr * D;
            };
            auto vrow = [&](int rr) {
                if constexpr (FIFO)   // residual row rr is slot position 32P + rr: ring row (32P + rr) % R
                    return rr == nrow ? a.new_v + islot * D : vr + (long long)(((int)(32 * P) + rr) % a.R) * D;
                return FUSED && rr == nrow ? a.new_v + islot * D : vr + (long long)rr * D;
            };
            build_q_frags<C, D, NQ, QB_REGS>(nullptr, qf, qhc_s, qlc_s, qoff, qfrag, lane, qb, beta);   // step 1, zero 0
            for (int rp = rb; rp < re; ++rp) {
                float sc[4];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int r0w = 32 * rp + 16 * t;
                    const bool okg = r0w + g < n, okg8 = r0w + g + 8 < n;
                    const __half* kg = FUSED ? krow(r0w + g) : kr + (long long)(r0w + g) * D;
                    const __half* kg8 = FUSED ? krow(r0w + g + 8) : kr + (long long)(r0w + g + 8) * D;
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const int ch = 16 * kk + 2 * i;
                        uint32_t af[4];
                        af[0] = okg ? *reinterpret_cast<const uint32_t*>(kg + ch) : 0u;
                        af[1] = okg8 ? *reinterpret_cast<const uint32_t*>(kg8 + ch) : 0u;
                        af[2] = okg ? *reinterpret_cast<const uint32_t*>(kg + ch + 8) : 0u;
                        af[3] = okg8 ? *reinterpret_cast<const uint32_t*>(kg8 + ch + 8) : 0u;
                        const uint2 bq = qbk(kk);
                        mma16816(c, af, bq.x, bq.y);
                    }
                    sc[2 * t] = okg ? c[0] + c[1] : -INFINITY;
                    sc[2 * t + 1] = okg8 ? c[2] + c[3] : -INFINITY;
                }
                float p[4];
                softmax(sc, p, 1.f);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    float prb[4];
                    gather(p[2 * t], p[2 * t + 1], prb);
                    uint32_t ph01, ph89, pl01, pl89;
                    split_p(prb, ph01, ph89, pl01, pl89);
                    const uint32_t pb0 = lo_col ? pl01 : ph01, pb1 = lo_col ? pl89 : ph89;
                    const int r0w = 32 * rp + 16 * t;
                    const bool okg = r0w + g < n, okg8 = r0w + g + 8 < n;
                    const __half* vg = FUSED ? vrow(r0w + g) : vr + (long long)(r0w + g) * D;
                    const __half* vg8 = FUSED ? vrow(r0w + g + 8) : vr + (long long)(r0w + g + 8) * D;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        uint32_t af[4];
                        vt_frag_rows<D>(vg, vg8, okg, okg8, mt, i, af);
                        mma16816(o[mt], af, pb0, pb1);
                    }
                }
            }
        }

        // ---- the segment's partial result (m, l, status, o) per query head ----
        const uint32_t st_all = (uint32_t)__reduce_or_sync(kFull, status | (PAGED && pc_all[warp].bad ? 2u : 0u));
#pragma unroll
        for (int f = 0; f < NBF; ++f) {
            zeta[f] += __shfl_xor_sync(kFull, zeta[f], 1);
            zeta[f] += __shfl_xor_sync(kFull, zeta[f], 2);
        }
        float lt = l;
        lt += __shfl_xor_sync(kFull, lt, 4);
        lt += __shfl_xor_sync(kFull, lt, 8);
        lt += __shfl_xor_sync(kFull, lt, 16);
        // the zero-point sums of this lane's output column i sit in lanes 8i .. 8i+3
        float zo[NBF];
#pragma unroll
        for (int f = 0; f < NBF; ++f) zo[f] = __shfl_sync(kFull, zeta[f], 8 * i);
        auto partial = [&](int h) -> float* {
            return a.ws + ((long long)(b * a.Hq + hk * NQ + h) * kPartialSlots + part) * partial_stride(D);
        };
        if (hO < NQ) {
            float* pw = partial(hO);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int gr = 16 * mt / G;
                if (gr % GB == jO) {
                    const float z = zo[gr / GB];
                    pw[4 + 16 * mt + g] = o[mt][0] + o[mt][1] + z;
                    pw[4 + 16 * mt + g + 8] = o[mt][2] + o[mt][3] + z;
                }
            }
        }
        if (g == 0 && i < NQ) {
            float* pw = partial(i);
            pw[0] = m;
            pw[1] = lt;
            pw[2] = (float)st_all;
        }
        pos = u1 >= NU ? w0 + Ws : w0 + unit_start_p(wm, P, M, u1);
    }
    if (first_seg) dependency_point();   // a warp without a segment still stores its share of the rows
}

#undef qf
#undef qhc_s
#undef qlc_s

// The log-sum-exp merge of a head's nparts partial results -> fp16 output, in
// two forms; a partial whose status is set (a cache copy timed out, a bad
// table entry) makes the head's output NaN.
//
// merge_head_warp: one warp per (query row, query head), for calls whose slots
// have at most kMergeAhead partials.  The (m, l, status) of every partial and
// the values of the first kMergeAhead partials are loaded together, so the
// merge is one round trip; the weights 2^(m_j - M) and the sum L come from
// shuffles, and the values are summed in partial order.
constexpr int kMergeThreads = 128;
constexpr int kMergeWarps = kMergeThreads / 32;   // heads per merge CTA in the warp form
constexpr int kMergeAhead = 16;
template <int D>
__device__ __forceinline__ void merge_head_warp(const float* base, int nparts, __half* out, int lane) {
    constexpr int S = partial_stride(D);
    constexpr int CPL = D / 32;                   // channels per lane
    static_assert(kPartialSlots <= 96, "partials held three to a lane");
    auto load_v = [&](int j, float (&v)[CPL]) {
        const float* ps = base + j * S + 4 + CPL * lane;
        if constexpr (CPL == 4) {
            const float4 x = *reinterpret_cast<const float4*>(ps);
            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2*>(ps);
            v[0] = x.x; v[1] = x.y;
        }
    };
    float v[kMergeAhead][CPL];
#pragma unroll
    for (int u = 0; u < kMergeAhead; ++u)
        if (u < nparts) load_v(u, v[u]);
    float mj[3], lj[3];
    bool bad = false;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const int j = lane + 32 * r;
        mj[r] = -INFINITY;
        lj[r] = 0.f;
        if (j < nparts) {
            const float* ps = base + j * S;
            mj[r] = ps[0];
            lj[r] = ps[1];
            bad |= ps[2] != 0.f;
        }
    }
    float M = fmaxf(fmaxf(mj[0], mj[1]), mj[2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float e[3], ls = 0.f;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        // a weight of 0 (an empty partial, m = -inf) adds nothing, whatever its values hold
        e[r] = mj[r] == -INFINITY ? 0.f : fast_exp2(mj[r] - M);
        ls = fmaf(lj[r], e[r], ls);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(kFull, ls, o);
    bad = __any_sync(kFull, bad);
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
#pragma unroll
    for (int u = 0; u < kMergeAhead; ++u) {
        const float eu = __shfl_sync(kFull, e[0], u);
        if (u < nparts && eu != 0.f) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fmaf(v[u][c], eu, acc[c]);
        }
    }
    for (int j = kMergeAhead; j < nparts; ++j) {  // beyond the values loaded ahead
        const float ej = __shfl_sync(kFull, j < 32 ? e[0] : (j < 64 ? e[1] : e[2]), j & 31);
        if (ej != 0.f) {
            float vj[CPL];
            load_v(j, vj);
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fmaf(vj[c], ej, acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < CPL; c += 2) {
        const __half2 h = bad ? __float2half2_rn(NAN) : __floats2half2_rn(acc[c] / ls, acc[c + 1] / ls);
        *reinterpret_cast<__half2*>(out + CPL * lane + c) = h;
    }
}

// merge_head_cta: one CTA (kMergeThreads threads) per head, for calls with
// more partials per slot.  The values of the partials a warp sums go out first,
// together with the (m, l) loads; one warp turns the m's into weights and the
// sum L; warp w sums partials w, w + 4, ... and the four warps' sums are added
// in warp order.
template <int D>
__device__ __forceinline__ void merge_head_cta(const float* base, int nparts, __half* out) {
    constexpr int S = partial_stride(D);
    constexpr int CPL = D / 32;                                 // channels per lane
    constexpr int NR = (kPartialSlots + kMergeWarps - 1) / kMergeWarps;   // partials per warp, at most
    __shared__ float e_s[kPartialSlots], l_s[kPartialSlots];
    __shared__ __align__(16) float red[kMergeWarps][D];
    __shared__ float lsum_s;
    __shared__ int bad_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float v[NR][CPL];
#pragma unroll
    for (int u = 0; u < NR; ++u) {
        const int j = warp + u * kMergeWarps;
        if (j < nparts) {
            const float* ps = base + j * S + 4 + CPL * lane;
            if constexpr (CPL == 4) {
                const float4 x = *reinterpret_cast<const float4*>(ps);
                v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2*>(ps);
                v[u][0] = x.x; v[u][1] = x.y;
            }
        }
    }
    if (tid == 0) bad_s = 0;
    __syncthreads();
    bool bad = false;
    for (int j = tid; j < nparts; j += kMergeThreads) {
        const float* ps = base + j * S;
        e_s[j] = ps[0];
        l_s[j] = ps[1];
        bad |= ps[2] != 0.f;
    }
    if (bad) bad_s = 1;
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
        for (int j = lane; j < nparts; j += 32) M = fmaxf(M, e_s[j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        float ls = 0.f;
        for (int j = lane; j < nparts; j += 32) {
            const float m = e_s[j];
            const float e = m == -INFINITY ? 0.f : fast_exp2(m - M);
            e_s[j] = e;
            ls = fmaf(l_s[j], e, ls);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(kFull, ls, o);
        if (lane == 0) lsum_s = ls;
    }
    __syncthreads();
    float acc[CPL];
#pragma unroll
    for (int r = 0; r < CPL; ++r) acc[r] = 0.f;
#pragma unroll
    for (int u = 0; u < NR; ++u) {
        const int j = warp + u * kMergeWarps;
        // a weight of 0 (an empty partial, m = -inf) adds nothing, whatever its values hold
        const float e = j < nparts ? e_s[j] : 0.f;
        if (e != 0.f) {
#pragma unroll
            for (int r = 0; r < CPL; ++r) acc[r] = fmaf(v[u][r], e, acc[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < CPL; ++r) red[warp][CPL * lane + r] = acc[r];
    __syncthreads();
    for (int c = tid; c < D; c += kMergeThreads) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) sum += red[w][c];
        out[c] = bad_s ? __float2half_rn(NAN) : __float2half_rn(sum / lsum_s);
    }
}

// Merge of the partials of each (batch, query head) of a dense call: WARP, one
// warp per head (four to a CTA), else one CTA per head.
template <int D, bool WARP>
__global__ void __launch_bounds__(kMergeThreads) finish_kernel(FinishArgs a) {
    // launched as a programmatic dependent of the main kernel: wait until its
    // partial results are complete and visible
    griddepcontrol_wait();
    griddepcontrol_launch_dependents();   // the next decode call may start its prologue
    const long long bh = WARP ? (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5) : (long long)blockIdx.x;
    if (bh >= a.heads) return;
    const long long slot = (bh / a.Hq) * a.Hkv + (bh % a.Hq) / a.nq;
    const float* base = a.ws + bh * kPartialSlots * partial_stride(D);
    if constexpr (WARP)
        merge_head_warp<D>(base, slot_parts(a.wm, slot), a.out + bh * D, threadIdx.x & 31);
    else
        merge_head_cta<D>(base, slot_parts(a.wm, slot), a.out + bh * D);
}

// The same for a paged call, per (call sequence, query head).
template <int D, bool WARP>
__global__ void __launch_bounds__(kMergeThreads) finish_paged_kernel(const __grid_constant__ PagedFinishArgs a) {
    griddepcontrol_wait();
    griddepcontrol_launch_dependents();
    const long long bh = WARP ? (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5) : (long long)blockIdx.x;
    if (bh >= a.heads) return;
    const int i = (int)(bh / a.Hq), hk = (int)((bh % a.Hq) / a.nq);
    const PagedSeq& sq = a.seqs[i];
    const long long P = sq.P, PR = (sq.n_resid + 31) / 32;
    const long long w0 = sq.start + hk * (a.wm.S0 + slot_weight(a.wm, P, 0, PR));
    const long long last = w0 + unit_start_p(a.wm, P, 0, P + PR - 1);
    const int nparts = (int)(map_owner(a.wm, last) - map_owner(a.wm, w0 + a.wm.S0) + 1);
    const float* base = a.ws + bh * kPartialSlots * partial_stride(D);
    if constexpr (WARP)
        merge_head_warp<D>(base, nparts, a.out + bh * D, threadIdx.x & 31);
    else
        merge_head_cta<D>(base, nparts, a.out + bh * D);
}

}  // namespace mma_detail
}  // namespace kivi
