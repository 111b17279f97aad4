/*
 * kivi.h - C ABI of a KIVI-style low-bit KV cache with single-query decode
 * attention, for NVIDIA GB300 (sm_103a).
 *
 * The method (three web pages describe it):
 *   [explainer]  KIVI explainer, discosf.com/news/3594501, sections 2.1-3.2, 5.2
 *   [axis-guide] "KV cache quantization axis selection guide", unite.ai
 *   [survey]     "3.2.3 KV Cache Quantization", blog.csdn.net
 *
 *   - Keys are quantized per channel over groups of G consecutive tokens;
 *     values per token over groups of G consecutive channels ([axis-guide]
 *     "keys: outliers sit in fixed channels" and "values: where intuition
 *     breaks"; [explainer] 3.1 pseudo-code; [survey]).
 *   - Each group is quantized uniformly and asymmetrically to B bits: the
 *     zero point is the group minimum, the step is (max - min) / (2^B - 1),
 *     every element goes to the nearest step ([axis-guide] "what
 *     quantization error is made of").  The exact arithmetic is:
 *         mn, mx   = group min / max (fp16 values, taken exactly; -0 -> +0)
 *         z        = (fp16) mn
 *         s        = (fp16) ((fp32)(mx - mn) / (2^B - 1))        IEEE fp32, RN
 *         code(x)  = s == 0 ? 0 : clamp(rint(((fp32)x - z) / s), 0, 2^B - 1)
 *     each fp32 operation rounded to nearest-even separately (no FMA); the
 *     rint tie rule is ties-to-even.  The dequantized value is the exact real
 *     number x_hat = code * s + z of the stored fp16 s and z: the decode
 *     kernels never round it to a float of their own (they fold s into the
 *     query or the attention weights and add z on the side), and their output
 *     is held to attention over these exact values.
 *   - The newest tokens (at most R) stay in an fp16 residual window; when the
 *     window is full it is quantized as one batch and emptied ([explainer]
 *     3.1, [axis-guide] "the system tax").  A prompt of L tokens keeps
 *     Lq = G * ceil(max(L - R, 0) / G) tokens quantized and r = L - Lq in the
 *     residual; an append that finds r == R first flushes all R residual
 *     tokens (keys and values together), then stores the new token.
 *   - Decode attention reads every cached token for each new query
 *     ([axis-guide] "why the KV cache is the problem"):
 *         o = sum_t softmax_t(scale * q . k_hat_t) * v_hat_t,
 *     scale = 1/sqrt(D) by default, no mask, query head h reads kv head
 *     h / (Hq / Hkv).  Accumulation is fp32; the output is fp16.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses on the current device.  The
 *     caller allocates and owns ALL device memory: the cache buffer, inputs,
 *     outputs and workspace.  The library owns only the small host handle.
 *   - A handle's device is the device current at its first call that launches
 *     work; every later launching call must find that device current
 *     (KIVI_ERR_INVALID_ARG otherwise).  Handles on different devices may be
 *     used in one process.
 *   - Calls that take a stream enqueue kernels on it and return without
 *     synchronizing.  Token counts live on the host handle, so no call reads
 *     device memory back.  Buffers passed in must stay valid until the
 *     enqueued work finishes.
 *   - All tensors are fp16, dense, row-major, 16-byte aligned.
 *   - Errors are return codes; nothing is launched when a call fails its
 *     checks, and the handle's state is then unchanged.  A failed launch
 *     returns KIVI_ERR_CUDA.  kivi_last_error_string() describes the last
 *     failure on the calling thread.
 *   - One handle must not be used from two threads at once.  One handle is
 *     one layer's cache; a model with several layers uses several handles.
 *   - There is no CPU fallback: every computation runs in the library's
 *     sm_103a kernels.
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same type as cudaStream_t); NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* kivi_stream_t;

typedef enum {
    KIVI_OK = 0,
    KIVI_ERR_INVALID_ARG = 1,   /* null or misaligned pointer, bad size or config */
    KIVI_ERR_UNSUPPORTED = 2,   /* valid in principle, not built (e.g. head_dim 96) */
    KIVI_ERR_CAPACITY = 3,      /* the cache or workspace is too small */
    KIVI_ERR_STATE = 4,         /* call out of order (prefill twice, decode on empty) */
    KIVI_ERR_CUDA = 5           /* a CUDA call failed; see kivi_last_error_string() */
} kivi_status;

/*
 * Cache shape.  Supported: bits in {2, 4, 8}; head_dim in {64, 128};
 * group in {32, 64, 128} with head_dim % group == 0 (value groups) and
 * residual % group == 0, residual >= group; n_q_heads / n_kv_heads in
 * {1, 2, 4}; batch * n_kv_heads <= 65535; 1 <= max_tokens <= 2^30 is the
 * most tokens (quantized + residual) one sequence may hold.  All sequences of
 * the batch have the same length (sequences of different lengths: the paged
 * cache below).
 * Typical group sizes 32-128 and residual lengths 64-128 follow
 * [explainer] 5.2.
 */
typedef struct {
    int batch;
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    int bits;
    int group;
    int residual;
    long long max_tokens;
} kivi_config;

/*
 * Byte layout of the cache buffer (all offsets from the buffer start).
 *
 *   NB   = floor(max_tokens / G)      quantized blocks per (batch, kv-head) slot
 *   TILE = 2 * D * bits               bytes of one 16-token code tile
 *   PART = (G / 16) * TILE + 4 * D    bytes of one block's key part or value part
 *
 *   blocks  : [B][Hkv][2][NB][PART] at offset 0; index 2: 0 = keys, 1 = values
 *   k_resid : [B][Hkv][R][D] fp16 at k_resid_offset
 *   v_resid : [B][Hkv][R][D] fp16 at v_resid_offset
 *
 * Block n of a slot holds that slot's tokens [n*G, (n+1)*G).  Residual row j
 * holds token Lq + j.
 *   key part  : G/16 code tiles (tokens in order), then the D channel steps
 *               s[c] (fp16), then the D channel zeros z[c] (fp16); s[c], z[c]
 *               hold for channel c over the block's G tokens.
 *   value part: G/16 code tiles, then G/16 entry tiles of 64*(D/G) bytes,
 *               one per code tile: the steps of the tile's 16 tokens as D/G
 *               rows of 16 fp16 (row j: channels [j*G, (j+1)*G)), then their
 *               zeros in the same form.  Inside a row, token t (0..15) of the
 *               tile sits at position 4*((t%8)/2) + 2*(t/8) + t%2, i.e. the
 *               order 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15.
 *
 * Code tile: 16 tokens x D channels of b-bit codes in D*b/2 little-endian
 * 32-bit words.  Lane l (0..31) owns words [l*W, (l+1)*W), W = D*b/64.
 * Write l = 4*g + i and P = 8/b.  The lane's D/4 code pairs are (k, r),
 * k = 0..D/16-1, r = 0..3:
 *   key tile  : both codes are token g + 8*(r%2); the first is channel
 *               16k + 2i + 8*(r/2), the second the next channel;
 *               class c = 2k + r/2, order h = r%2.
 *   value tile: both codes are channel 16k + g + 8*(r%2); the first is token
 *               2i + 8*(r/2), the second the next token;
 *               class c = 2k + r%2, order h = r/2.
 * Pair (k, r) is in the lane's word c/P, in byte h of each 16-bit half, at
 * bits [b*(c%P), b*(c%P) + b) of that byte: the first code in the low half
 * (bits 0-15), the second in the high half.
 * (Each lane's words are thereby the fragments of a 16x16 fp16 A operand of
 * an m16n8k16 MMA: keys as [token][channel], values as [channel][token].
 * The class of a code is its channel / 8, so a code masked in place reads as
 * the fp16 value code * 2^(b*((ch/8)%P) - 24), a scale set by the channel.)
 */
typedef struct {
    size_t total_bytes;       /* == kivi_cache_bytes() */
    long long blocks_per_slot;/* NB */
    size_t tile_bytes;        /* TILE */
    size_t part_bytes;        /* PART */
    size_t slot_bytes;        /* 2 * NB * PART: one (batch, kv-head) slot */
    size_t k_resid_offset;    /* 256-byte aligned */
    size_t v_resid_offset;    /* 256-byte aligned */
    size_t resid_slot_bytes;  /* R * D * 2: one slot's residual rows */
} kivi_layout;

typedef struct kivi_cache* kivi_cache_t;

/* Bytes of device memory a cache of this shape needs; 0 if cfg is invalid.
 * Host-only. */
size_t kivi_cache_bytes(const kivi_config* cfg);

/* Fill *out with the buffer layout described above.  Host-only.
 * KIVI_ERR_INVALID_ARG / KIVI_ERR_UNSUPPORTED for a bad config. */
kivi_status kivi_cache_layout(const kivi_config* cfg, kivi_layout* out);

/* Create a handle over the caller's device buffer dev_buf (256-byte aligned,
 * at least kivi_cache_bytes(cfg) bytes; the contents need no initialization).
 * The cache starts empty.  Host-only: no CUDA call is made.  The buffer stays
 * owned by the caller and must outlive the handle. */
kivi_status kivi_cache_create(const kivi_config* cfg, void* dev_buf, size_t bytes,
                              kivi_cache_t* out);

/* Free the host handle (not the buffer).  Work already enqueued is unaffected. */
kivi_status kivi_cache_destroy(kivi_cache_t cache);

/* Forget all cached tokens (host counters only; no device work). */
kivi_status kivi_cache_reset(kivi_cache_t cache);

/* Token counts: *n_quant = Lq (quantized), *n_resid = r (fp16 residual). */
kivi_status kivi_cache_counts(kivi_cache_t cache, long long* n_quant, long long* n_resid);

/*
 * Prefill ([explainer] 3.1): K, V are fp16 [B][Hkv][L][D] device tensors.
 * Quantizes tokens [0, Lq) into blocks and copies tokens [Lq, L) bit for bit
 * into the residual, Lq = G * ceil(max(L - R, 0) / G).  Only on an empty
 * cache (KIVI_ERR_STATE otherwise); L may be 0.  KIVI_ERR_CAPACITY if
 * L > max_tokens.
 */
kivi_status kivi_prefill(kivi_cache_t cache, const void* K, const void* V, long long L,
                         kivi_stream_t stream);

/*
 * Append one token ([explainer] 3.1, [axis-guide] "the system tax"): k, v are
 * fp16 [B][Hkv][D] device tensors.  If the residual holds R tokens they are
 * first quantized into blocks (R/G key groups, R value tokens) and the
 * residual is emptied; then k, v become the newest residual row.
 * KIVI_ERR_CAPACITY if the cache already holds max_tokens tokens.
 */
kivi_status kivi_append(kivi_cache_t cache, const void* k, const void* v,
                        kivi_stream_t stream);

/* Bytes of decode workspace needed for any context of this shape on any
 * device; 0 if cfg is invalid.  Host-only. */
size_t kivi_decode_workspace_bytes(const kivi_config* cfg);

/*
 * Decode attention ([axis-guide] "why the KV cache is the problem", "values:
 * where intuition breaks"): q fp16 [B][Hq][D] device tensor; out fp16
 * [B][Hq][D] device tensor.  softmax_scale <= 0 selects 1/sqrt(D).
 * workspace: device scratch of ws_bytes >= kivi_decode_workspace_bytes(cfg)
 * bytes, 256-byte aligned; its contents need no initialization and are
 * garbage afterwards.  Reads all Lq + r cached tokens.  KIVI_ERR_STATE on an
 * empty cache; KIVI_ERR_CAPACITY if ws_bytes is too small.
 */
kivi_status kivi_decode_attn(kivi_cache_t cache, const void* q, void* out, float softmax_scale,
                             void* workspace, size_t ws_bytes, kivi_stream_t stream);

/*
 * Append one token, then decode attention over the cache holding it, in one
 * call: the same arguments, result and cache state as kivi_append(cache, k, v)
 * followed by kivi_decode_attn(cache, q, out, softmax_scale, workspace,
 * ws_bytes, stream) (the method's description has them as two steps; this
 * fuses them).  With the tensor-core decode kernel the new token's residual
 * row is written by the decode kernel itself, one launch fewer than the two
 * calls, and with the value queue (kivi_cache_set_value_residual) the decode
 * kernel also quantizes the value that leaves the queue, another launch
 * fewer; with the CUDA-core kernel selected the two calls run in sequence.
 * Errors as for those two calls; every check runs before anything is
 * launched.
 */
kivi_status kivi_append_decode(kivi_cache_t cache, const void* k, const void* v, const void* q, void* out,
                               float softmax_scale, void* workspace, size_t ws_bytes, kivi_stream_t stream);

/*
 * Which decode kernel kivi_decode_attn uses.  Both compute the same result
 * within the same tolerance: the CUDA-core kernel accumulates fp32 products of
 * the codes with q * step; the tensor-core kernel feeds exact fp16 codes and
 * fp16 hi + lo splits of q * step (and of p * step) to mma.sync with fp32
 * accumulation.  AUTO picks the faster one for the shape (the tensor-core
 * kernel on sm_103a for every supported shape, from measurement).
 */
typedef enum {
    KIVI_DECODE_AUTO = 0,
    KIVI_DECODE_CUDA_CORE = 1,
    KIVI_DECODE_TENSOR_CORE = 2
} kivi_decode_kernel;

kivi_status kivi_cache_set_decode_kernel(kivi_cache_t cache, int kernel);

/*
 * Cap the tensor-core decode kernel's persistent grid at max_ctas CTAs (0, the
 * default: SMs x resident CTAs per SM), e.g. to leave SMs to other work on the
 * GPU.  The result does not depend on the grid beyond fp32 summation order
 * (the split of a slot over CTAs changes, the arithmetic per token does not).
 * Host-only; KIVI_ERR_INVALID_ARG for a negative cap.
 */
kivi_status kivi_cache_set_max_ctas(kivi_cache_t cache, int max_ctas);

/*
 * Value residual as a queue ([explainer] 3.2): new value tokens enter an fp16
 * queue of R rows; once it holds R tokens, each append quantizes the oldest
 * value on its own (per token, groups of G channels, the formula above) and
 * drops it, so after every call the newest min(L, R) values are fp16 and the
 * first Lv = max(L - R, 0) are quantized.  Keys keep the flush-all rule, so
 * Lv <= Lq and tokens [Lv, Lq) have quantized keys with fp16 values.
 *
 *   KIVI_VALUE_FLUSH (default): values flush with the keys (the rule above).
 *   KIVI_VALUE_QUEUE          : the queue.  Layout changes: v_resid row j of a
 *       slot holds the value of token p with p % R == j, for p in [Lv, L);
 *       in the value part of a block, tokens not quantized yet have all-zero
 *       codes and step = zero = +0.  Decode runs on the tensor-core kernel only
 *       (KIVI_ERR_UNSUPPORTED with the CUDA-core kernel selected); residual
 *       must be <= 128.  kivi_cache_counts still reports (Lq, r) of the keys.
 *
 * Set on an empty cache (after create or reset; KIVI_ERR_STATE otherwise); a
 * reset keeps the mode.  Host-only.
 */
typedef enum {
    KIVI_VALUE_FLUSH = 0,
    KIVI_VALUE_QUEUE = 1
} kivi_value_residual;

kivi_status kivi_cache_set_value_residual(kivi_cache_t cache, int mode);

/*
 * Decode attention with a workspace owned by the library (the method's
 * description has no counterpart; this is an integration aid).
 *
 * For callers that cannot allocate device memory: a plugin inside a host
 * framework that owns all device memory through its own pool (a raw
 * cudaMalloc is refused there, or would synchronize the device), or code that
 * only receives device pointers.  Same arguments and result as
 * kivi_decode_attn, minus the workspace: the library keeps one 16 MiB
 * workspace per device in a static device array, which every device that
 * loads the library holds until the process exits.  Shapes whose
 * kivi_decode_workspace_bytes() exceeds 16 MiB (batch * n_q_heads above 488
 * at head_dim 128, above 948 at head_dim 64) get KIVI_ERR_CAPACITY.
 * The cache's device must be current (KIVI_ERR_INVALID_ARG otherwise).
 * The first call on a device looks up the array's device address (with that
 * device current).  The library's device code loads lazily, so that first
 * call is also when the driver loads the array onto the device and reserves
 * its 16 MiB there; it can fail (KIVI_ERR_CUDA, with a message naming the
 * workspace) if the device is out of memory, and it may synchronize.  Make
 * that first call during set-up, before any stream capture and before a
 * framework takes the device's free memory.  After it no call allocates
 * memory.  All calls on a device share the one workspace, so two calls whose
 * kernels overlap on the GPU (different streams, no ordering between them)
 * race and may return wrong results; serialize them.
 */
kivi_status kivi_decode_attn_static_ws(kivi_cache_t cache, const void* q, void* out,
                                       float softmax_scale, kivi_stream_t stream);

/* ===================== Paged cache with ragged sequences =====================
 *
 * The same quantized cache for a changing set of sequences of different
 * lengths, as a serving engine runs it: quantized blocks live in pages of a
 * shared pool and each sequence has a block table (the explainer's pointer to
 * PagedAttention, section 7; the method itself is unchanged).  Every sequence
 * follows the streaming rule above on its own: Lq = G * ceil(max(L - R, 0) / G)
 * after its prompt, a flush of its R residual tokens when an append finds
 * r == R.
 *
 * A page holds one block (G tokens) of one sequence for every kv head:
 *
 *   pages   : [n_pages][Hkv][2][PART] at offset 0; index 2: 0 = keys, 1 = values
 *             (each part exactly as in a block of the dense cache above)
 *   k_resid : [max_seqs][Hkv][R][D] fp16 at k_resid_offset
 *   v_resid : [max_seqs][Hkv][R][D] fp16 at v_resid_offset
 *   table   : [max_seqs][max_blocks_per_seq] int32 at table_offset; entry n of
 *             row s is the page of block n of sequence s (tokens [n*G, (n+1)*G)),
 *             valid for n < Lq / G
 *
 * Pages and sequence slots are handed out by an allocator on the host handle
 * (free lists; a released sequence's pages are reused in any order).  The
 * library writes table entries from its kernels when it fills a page; the
 * host keeps its own copy, so no call reads device memory back.
 *
 * Conventions as for the dense cache (caller-owned device memory, stream
 * ordering, errors before launch, no CPU fallback).
 */
typedef struct {
    int max_seqs;             /* sequence slots */
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    int bits;
    int group;
    int residual;
    int max_blocks_per_seq;   /* a sequence holds at most max_blocks_per_seq * group + residual tokens */
    long long n_pages;        /* pages in the pool */
} kivi_paged_config;

typedef struct {
    size_t total_bytes;       /* == kivi_paged_bytes() */
    size_t tile_bytes;        /* TILE */
    size_t part_bytes;        /* PART */
    size_t page_bytes;        /* Hkv * 2 * PART */
    size_t k_resid_offset;    /* 256-byte aligned */
    size_t v_resid_offset;    /* 256-byte aligned */
    size_t resid_seq_bytes;   /* Hkv * R * D * 2: one sequence's residual rows (keys or values) */
    size_t table_offset;      /* 256-byte aligned */
} kivi_paged_layout;

typedef struct kivi_paged* kivi_paged_t;

/* Most sequences one kivi_paged_append_decode call may take. */
#define KIVI_PAGED_MAX_CALL_SEQS 512

/* Bytes of device memory a paged cache of this shape needs; 0 if cfg is
 * invalid.  The shape limits are those of the dense cache, plus max_seqs,
 * max_blocks_per_seq and n_pages >= 1, n_pages < 2^31 and
 * max_seqs * max_blocks_per_seq < 2^31.  Host-only. */
size_t kivi_paged_bytes(const kivi_paged_config* cfg);

/* Fill *out with the layout above.  Host-only. */
kivi_status kivi_paged_cache_layout(const kivi_paged_config* cfg, kivi_paged_layout* out);

/* Create a handle over the caller's device buffer (256-byte aligned, at least
 * kivi_paged_bytes(cfg) bytes, no initialization needed): no sequences, every
 * page free.  Host-only. */
kivi_status kivi_paged_create(const kivi_paged_config* cfg, void* dev_buf, size_t bytes,
                              kivi_paged_t* out);

/* Free the host handle (not the buffer). */
kivi_status kivi_paged_destroy(kivi_paged_t cache);

/*
 * Add a sequence with a prompt of L >= 0 tokens: K, V fp16 [Hkv][L][D] device
 * tensors (may be NULL when L == 0).  Takes a free sequence slot (its id is
 * written to *seq) and ceil(Lq / G) pages, quantizes tokens [0, Lq) into
 * them and copies [Lq, L) into the sequence's residual rows, as kivi_prefill
 * does for one batch row.  KIVI_ERR_CAPACITY when no slot is free, the pool
 * has too few free pages, or Lq / G > max_blocks_per_seq.
 */
kivi_status kivi_paged_add(kivi_paged_t cache, const void* K, const void* V, long long L,
                           kivi_stream_t stream, int* seq);

/* Release a sequence: its slot and pages return to the free lists (host only,
 * no device work; work already enqueued that reads them must finish before the
 * next call that reuses them is enqueued on another stream). */
kivi_status kivi_paged_release(kivi_paged_t cache, int seq);

/* Token counts of one live sequence. */
kivi_status kivi_paged_seq_counts(kivi_paged_t cache, int seq, long long* n_quant, long long* n_resid);

/* The pages of a live sequence's blocks, in block order: writes
 * min(count, cap) entries to pages[] and the count to *n. */
kivi_status kivi_paged_seq_pages(kivi_paged_t cache, int seq, int* pages, int cap, int* n);

/* Free pages and free sequence slots. */
kivi_status kivi_paged_free(kivi_paged_t cache, long long* free_pages, int* free_seqs);

/* Cap the decode kernel's persistent grid at max_ctas CTAs for this cache's
 * calls (0, the default: SMs x resident CTAs per SM); as
 * kivi_cache_set_max_ctas.  Host-only; KIVI_ERR_INVALID_ARG for a negative cap. */
kivi_status kivi_paged_set_max_ctas(kivi_paged_t cache, int max_ctas);

/* Workspace bytes of a call over n sequences (n <= KIVI_PAGED_MAX_CALL_SEQS);
 * 0 if cfg or n is invalid.  Host-only. */
size_t kivi_paged_workspace_bytes(const kivi_paged_config* cfg, int n);

/*
 * For each of the n distinct live sequences seqs[0..n-1] (host array): append
 * token k[i], v[i] (fp16 [n][Hkv][D]) with the flush rule above, then decode
 * attention of q[i] (fp16 [n][Hq][D]) over that sequence's cached tokens into
 * out[i] (fp16 [n][Hq][D]).  k and v both NULL: decode only, no append (a
 * sequence must then hold a token).  softmax_scale and workspace as for
 * kivi_decode_attn (ws_bytes >= kivi_paged_workspace_bytes(cfg, n)).  Runs on
 * the tensor-core kernel (one decode launch and one merge launch, plus one
 * quantize launch when a sequence flushes).  KIVI_ERR_CAPACITY when a flush
 * needs more free pages than the pool has or a sequence is full; every check
 * runs before anything is launched or allocated.
 */
kivi_status kivi_paged_append_decode(kivi_paged_t cache, const int* seqs, int n, const void* k,
                                     const void* v, const void* q, void* out, float softmax_scale,
                                     void* workspace, size_t ws_bytes, kivi_stream_t stream);

/*
 * Failure detection.  Every wait of the tensor-core decode kernel on its bulk
 * copies is bounded (about 2 s); a copy that does not complete in time marks
 * the waiting warp's partial results, and the merge writes NaN for every query
 * head of the slots that warp covered (the warp then issues no more copies,
 * finishes and returns; the context stays usable).  The paged kernel also
 * marks a block-table entry outside the pool the same way.
 *
 * Test hook: KIVI_FAULT_COPY_STALL makes the next tensor-core decode call on
 * this cache (kivi_decode_attn or kivi_append_decode) expect 16 bytes more on
 * the first copy stage of CTA 0, warp 0 than its copies bring, so that wait
 * runs out: that call takes about 4 s more and returns NaN for the heads of the
 * slots that warp covers, correct outputs elsewhere.  One call only; host-only.
 */
typedef enum {
    KIVI_FAULT_NONE = 0,
    KIVI_FAULT_COPY_STALL = 1
} kivi_fault;

kivi_status kivi_cache_set_fault(kivi_cache_t cache, int fault);

/* Description of the last failure on the calling thread ("" if none). */
const char* kivi_last_error_string(void);

/* Number of kernel launches this library has issued in this process. */
unsigned long long kivi_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KIVI_H */
