// Internal declarations shared by the host API and the kernels of the KIVI
// KV-cache library.  The public contract (argument meaning, buffer layout,
// errors) is in include/kivi.h.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kivi.h"

namespace kivi {

// Everything derived from a kivi_config that kernels need to address the cache.
struct Geometry {
    int B, Hq, Hkv, D, bits, G, R;
    long long max_tokens;
    long long NB;              // quantized blocks per (batch, kv-head) slot
    long long tile_bytes;      // one 16-token code tile: 2*D*bits
    long long part_bytes;      // one block's key or value part: (G/16)*tile + 4*D
    long long slot_bytes;      // 2 * NB * part
    long long k_resid_off;     // byte offset of the key residual region
    long long v_resid_off;     // byte offset of the value residual region
    long long resid_slot_bytes;// R * D * 2
    long long total_bytes;
};

// Validates cfg; on failure returns the status and writes a reason.
kivi_status derive_geometry(const kivi_config* cfg, Geometry* g, const char** why);

// Upper bound on decode partial results per (batch, query head).
constexpr int kMaxSplits = 64;          // quantized-token splits
constexpr int kPartialSlots = kMaxSplits + 1;  // + one split for the fp16 residual

// Floats per partial result (m, l, status, pad, o[D]); D + 4 keeps o 16-byte aligned.
// status != 0 marks a split whose cache copy did not complete (its output is NaN).
__host__ __device__ constexpr int partial_stride(int D) { return D + 4; }

// ---- code-tile placement (kivi.h, "Code tile") ----
// A lane's code pair (k, r) has class c and order h; it sits in lane word
// c / P, P = 8 / BITS, at bit 8*h + BITS*(c % P) of each 16-bit half.  Keys:
// c = 2k + r/2, h = r%2; values: c = 2k + r%2, h = r/2.  In both cases
// c = channel / 8, so a code masked in place is the fp16 value
// code * 2^(BITS*((channel/8) % P) - 24).
template <int BITS, bool VALUES>
struct PairPlace {
    static constexpr int P = 8 / BITS;
    __host__ __device__ static constexpr int cls(int k, int r) { return 2 * k + (VALUES ? (r & 1) : (r >> 1)); }
    __host__ __device__ static constexpr int order(int r) { return VALUES ? (r >> 1) : (r & 1); }
    __host__ __device__ static constexpr int word(int k, int r) { return cls(k, r) / P; }
    __host__ __device__ static constexpr int bit(int k, int r) { return 8 * order(r) + BITS * (cls(k, r) % P); }
    // inverse: the pair in lane word wl, slot u (byte u / P, position u % P)
    __host__ __device__ static constexpr int k_of(int wl, int u) { return (wl * P + u % P) >> 1; }
    __host__ __device__ static constexpr int r_of(int wl, int u) {
        return VALUES ? ((wl * P + u % P) & 1) + 2 * (u / P) : 2 * ((wl * P + u % P) & 1) + u / P;
    }
};

// Position of token t (0..15) of a tile inside a row of its value entry tile.
__host__ __device__ constexpr int entry_pos(int t) { return 4 * ((t & 7) >> 1) + 2 * (t >> 3) + (t & 1); }

// ---- the quantization arithmetic written out at the top of kivi.h, shared
// by every kernel that writes codes ----

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

// Balanced partition of a decode call's work over the warps of the
// tensor-core kernel (the map's workers; a CTA's warps work independently).
// Per (batch, kv-head) slot the work is a row of units: P quantized tile pairs
// (32 tokens) of weight wq, the last M of them of weight wq + wx (value queue:
// pairs that also read their queued values as fp16 rows), then PR fp16
// residual pairs (32 rows) of weight wr (weights proportional to the bytes each
// reads), after a lead-in of weight S0 that stands for the fixed cost a worker
// pays per slot it works on (query setup, ring fill, partial write): the
// worker whose range takes in a slot's start is given that much less of the
// units.  Slots follow each other; worker c covers weight positions
// [c*Wt/n, (c+1)*Wt/n) and owns the units that start there.  A worker whose
// range lies inside a slot without holding a unit start writes an empty
// partial for it.
struct WorkMap {
    long long P, PR, wq, wr, Ws, Wt, n, S0;
    long long M = 0, wx = 0;   // dense calls: the slots' mixed pairs and their extra weight
};
// The lead-in in quantized pairs, used when the call's shortest slot is shorter
// than a worker's share (with ~16 warps per SM), so that workers cover several
// slot starts.
constexpr long long kSegmentLeadPairs = 4;
__host__ inline long long segment_lead(long long wq, long long ws_min, long long wt, int num_sms) {
    const long long n_est = 16LL * (num_sms > 0 ? num_sms : 1);
    return ws_min * n_est < wt ? kSegmentLeadPairs * wq : 0;
}
// weight of a slot's units (without the lead-in): P quantized pairs, the last M
// of them mixed, and PR residual pairs
__host__ __device__ inline long long slot_weight(const WorkMap& m, long long P, long long M, long long PR) {
    return P * m.wq + M * m.wx + PR * m.wr;
}
// unit u of a slot of P quantized pairs, the last M of them mixed (slots of
// ragged sequences differ; they have no mixed pairs)
__host__ __device__ inline long long unit_start_p(const WorkMap& m, long long P, long long M, long long u) {
    const long long Q = P - M, wm = m.wq + m.wx;
    if (u <= Q) return m.S0 + u * m.wq;
    if (u <= P) return m.S0 + Q * m.wq + (u - Q) * wm;
    return m.S0 + Q * m.wq + M * wm + (u - P) * m.wr;
}
// first unit of a slot starting at or after weight offset y (0 <= y <= Ws); P + PR if none
__host__ __device__ inline long long first_unit_at_p(const WorkMap& m, long long P, long long M, long long y) {
    y -= m.S0;
    if (y <= 0) return 0;
    const long long Q = P - M, wm = m.wq + m.wx;
    if (y <= Q * m.wq) return (y + m.wq - 1) / m.wq;
    y -= Q * m.wq;
    if (y <= M * wm) return Q + (y + wm - 1) / wm;
    y -= M * wm;
    return P + (y + m.wr - 1) / m.wr;
}
__host__ __device__ inline long long unit_start(const WorkMap& m, long long u) {
    return unit_start_p(m, m.P, m.M, u);
}
__host__ __device__ inline long long first_unit_at(const WorkMap& m, long long y) {
    return first_unit_at_p(m, m.P, m.M, y);
}
__host__ __device__ inline long long map_begin(const WorkMap& m, long long c) { return c * m.Wt / m.n; }
// the worker whose range holds weight position x
__host__ __device__ inline long long map_owner(const WorkMap& m, long long x) {
    return ((x + 1) * m.n + m.Wt - 1) / m.Wt - 1;
}
// partials of slot s: workers [owner of its first unit's start, owner of its last unit's start]
__host__ __device__ inline long long slot_first_worker(const WorkMap& m, long long s) {
    return map_owner(m, s * m.Ws + m.S0);
}
__host__ __device__ inline int slot_parts(const WorkMap& m, long long s) {
    if (m.P + m.PR == 0) return 0;
    return (int)(map_owner(m, s * m.Ws + unit_start(m, m.P + m.PR - 1)) - slot_first_worker(m, s) + 1);
}

// ---- launchers (defined in the .cu files; return the launch status) -------

// Quantize nblk whole blocks per slot.  Block j of slot s is read from
// src_k/src_v + s*src_slot_elems + j*G*D (rows of D fp16, consecutive tokens)
// and written to block first_block + j of that slot.  Value tokens at slot
// positions >= vlimit are written as not yet quantized (zero codes, step and
// zero point); the value queue fills them in later.
constexpr long long kNoValueLimit = 1LL << 62;
cudaError_t launch_quantize_blocks(const Geometry& g, uint8_t* cache, const __half* src_k,
                                   const __half* src_v, long long src_slot_elems,
                                   long long first_block, long long nblk, cudaStream_t st,
                                   long long vlimit = kNoValueLimit);

// Value queue: quantize value token t of every slot from residual row t % R
// into its block (whose value part holds zeros for it).
cudaError_t launch_pop_values(const Geometry& g, uint8_t* cache, long long t, cudaStream_t st);

// Residual copies with the values kept as a ring of R rows: per slot, nk key
// rows (source rows k_src0.. into residual rows k_row0..) and nv value rows
// (source rows v_src0.., tokens v_tok0.. into rows token % R).
cudaError_t launch_copy_rows_ring(const Geometry& g, uint8_t* cache, const __half* src_k, const __half* src_v,
                                  long long src_slot_elems, int k_row0, long long k_src0, int nk,
                                  long long v_tok0, long long v_src0, int nv, cudaStream_t st);

// Copy nrows token rows per slot (K and V) into residual rows [row0, row0+nrows).
cudaError_t launch_copy_rows(const Geometry& g, uint8_t* cache, const __half* src_k,
                             const __half* src_v, long long src_slot_elems, int row0, int nrows,
                             cudaStream_t st);

struct DecodePlan {
    int tiles_per_split;   // CUDA-core kernel: 16-token tiles of quantized cache per split
    int n_qsplits;         // CUDA-core kernel: splits over the quantized tokens
    int n_splits;          // CUDA-core kernel: n_qsplits + (residual split ? 1 : 0)
    int num_sms;           // tensor-core kernel: sizes its persistent grid
    int max_ctas;          // tensor-core kernel: cap on that grid (0: none)
};

DecodePlan plan_decode(const Geometry& g, long long n_quant, long long n_resid, int num_sms);

// An append fused into a decode call (tensor-core kernel only): residual row
// `row` of every slot is the token k / v ([B*Hkv][D] fp16); the decode kernel
// reads it from there and stores it in the cache.  row < 0: none.  early_ok: the
// kernel preceding the decode on the stream writes no quantized block.
struct FusedAppend {
    const __half* k = nullptr;
    const __half* v = nullptr;
    int row = -1;
    int early_ok = 1;
    // value queue (tensor-core kernel only): >= 0 selects it; values of slot
    // positions below lqv are quantized, the rest sit in the residual ring
    long long lqv = -1;
    // value queue with a fused append: slot position pop (== lqv - 1) leaves
    // the queue in this call (the kernel quantizes its value into its block,
    // and the appended value takes its ring row); -1: no pop
    long long pop = -1;
    // failure-detection test hook (kivi_cache_set_fault): bytes the first ring
    // stage of CTA 0, warp 0 waits for beyond its copies
    int stall_bytes = 0;
};

// variant: KIVI_DECODE_CUDA_CORE or KIVI_DECODE_TENSOR_CORE (resolved, never AUTO).
// n_resid counts the fused append's row, if any.
cudaError_t launch_decode(const Geometry& g, const uint8_t* cache, long long n_quant,
                          long long n_resid, const __half* q, __half* out, float scale_log2,
                          float* workspace, const DecodePlan& plan, int variant, cudaStream_t st,
                          int* launches, const FusedAppend& fa = FusedAppend{});

// ---- paged cache (kivi.h, "Paged cache with ragged sequences") ----

constexpr int kMaxCallSeqs = KIVI_PAGED_MAX_CALL_SEQS;

// Geometry of a paged cache: g.B = max_seqs, g.NB = max_blocks_per_seq; the
// residual offsets and resid_slot_bytes keep their meaning per (sequence, kv
// head) slot; slot_bytes is unused.
struct PagedGeometry {
    Geometry g;
    long long n_pages, page_bytes, table_off;
};

// One sequence of a paged decode call.  Its Hkv slots take weight positions
// [start, start + Hkv * Ws), Ws = P * wq + ceil(n_resid / 32) * wr.
struct PagedSeq {
    long long start;
    int seq;       // sequence slot: residual rows and block-table row
    int P;         // quantized tile pairs (Lq / 32)
    int n_resid;   // residual rows, the fused append's included
    int new_row;   // the fused append's residual row, -1: none
};

// One block quantized into a page: head h's G rows start at
// src + src_off + h * src_head_elems; table entry tbl_idx is set to page.
struct QJob {
    long long src_off;
    int page;
    int tbl_idx;
};
constexpr int kMaxQJobs = 1024;   // per launch

// Quantize njobs blocks (any number; launched in chunks of kMaxQJobs).
cudaError_t launch_quantize_pages(const PagedGeometry& pg, uint8_t* buf, const __half* src_k,
                                  const __half* src_v, long long src_head_elems, const QJob* jobs,
                                  int njobs, cudaStream_t st, int* launches);

// Copy nrows rows per slot into residual rows [row0, row0 + nrows) of slots
// [first_slot, first_slot + nslots); slot j's rows come from src + j * src_slot_elems.
cudaError_t launch_copy_rows_slots(const Geometry& g, uint8_t* cache, const __half* src_k,
                                   const __half* src_v, long long src_slot_elems, long long first_slot,
                                   int nslots, int row0, int nrows, cudaStream_t st);

// Tensor-core decode over the n sequences of a paged call (+ its merge).
// new_k / new_v: the fused append's tokens [n][Hkv][D], or null.
cudaError_t launch_decode_paged(const PagedGeometry& pg, const uint8_t* buf, const PagedSeq* seqs, int n,
                                const __half* q, __half* out, float scale_log2, float* workspace,
                                const __half* new_k, const __half* new_v, int early_ok, int num_sms, int max_ctas,
                                cudaStream_t st, int* launches);

// Host-side helpers of the C ABI (kivi_api.cu): set the calling thread's
// error string and return st; the decode workspace bytes a handle needs.
kivi_status report_error(kivi_status st, const char* msg);
void count_launches(int n);   // adds to kivi_launch_count()
size_t decode_workspace_need(const struct ::kivi_cache* c);
// Checks that the cache's device is current (recording it at the first call).
kivi_status cache_device(struct ::kivi_cache* c);

}  // namespace kivi
