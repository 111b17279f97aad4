// Host side of the C ABI declared in include/kivi.h: argument checks, the
// streaming state (quantized / residual token counts), and kernel launches.
//
// Streaming rule (KIVI explainer, discosf.com, 3.1; "KV cache quantization
// axis selection guide", unite.ai, "the system tax"): a prompt keeps its
// G-aligned prefix quantized and at most R tokens in fp16; an append that
// finds R residual tokens quantizes them as one batch first.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <new>

#include "kivi_common.cuh"

struct kivi_cache {
    kivi::Geometry geo;
    uint8_t* buf;
    long long n_quant;
    long long n_resid;
    int device;      // -1 until the first launching call records the current device
    int num_sms;
    int decode_kernel;   // kivi_decode_kernel
    int value_queue;     // 1: the value residual is a queue ([explainer] 3.2)
    int fault;           // kivi_fault for the next tensor-core decode call (test hook)
    int max_ctas;        // cap on the tensor-core decode kernel's grid (0: none)
};

namespace {

thread_local char g_err[512] = "";
std::atomic<unsigned long long> g_launches{0};

kivi_status fail(kivi_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

kivi_status ok() {
    g_err[0] = '\0';
    return KIVI_OK;
}

kivi_status cuda_fail(cudaError_t e, const char* what) {
    return fail(KIVI_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }

// The cache's device: the device current at the handle's first call that
// launches work (its SM count is taken then too).  Every later launching call
// must find that device current, since the kernels run on the current device
// and the cache buffer lives on its own.
kivi_status ensure_device(kivi_cache_t c) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    if (c->device < 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "device query");
        c->device = dev;
        c->num_sms = sms;
    } else if (dev != c->device) {
        return fail(KIVI_ERR_INVALID_ARG, "the cache is on device %d but device %d is current", c->device, dev);
    }
    return KIVI_OK;
}

}  // namespace

// Value queue, before an append stores its token: flush the key residual when
// full (its blocks get their values as not quantized yet: they are all still
// queued), then, with pop, quantize the oldest queued value, whose ring row
// the new token takes (a fused append-and-decode leaves that to its decode
// kernel).  *wrote: a kernel that writes quantized blocks was launched.
static kivi_status queue_before_append(kivi_cache* c, cudaStream_t st, bool pop, bool* wrote);

namespace kivi {

kivi_status derive_geometry(const kivi_config* c, Geometry* g, const char** why) {
    if (!c) { *why = "null config"; return KIVI_ERR_INVALID_ARG; }
    if (c->batch < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 1 ||
        c->group < 1 || c->residual < 1 || c->max_tokens < 1) {
        *why = "batch, heads, head_dim, group, residual and max_tokens must be positive";
        return KIVI_ERR_INVALID_ARG;
    }
    if (c->bits != 2 && c->bits != 4 && c->bits != 8) { *why = "bits must be 2, 4 or 8"; return KIVI_ERR_UNSUPPORTED; }
    if (c->head_dim != 64 && c->head_dim != 128) { *why = "head_dim must be 64 or 128"; return KIVI_ERR_UNSUPPORTED; }
    if (c->group != 32 && c->group != 64 && c->group != 128) { *why = "group must be 32, 64 or 128"; return KIVI_ERR_UNSUPPORTED; }
    if (c->head_dim % c->group) { *why = "head_dim must be a multiple of group (value groups)"; return KIVI_ERR_INVALID_ARG; }
    if (c->residual % c->group || c->residual < c->group) { *why = "residual must be a positive multiple of group"; return KIVI_ERR_INVALID_ARG; }
    if (c->n_q_heads % c->n_kv_heads) { *why = "n_q_heads must be a multiple of n_kv_heads"; return KIVI_ERR_INVALID_ARG; }
    const int nq = c->n_q_heads / c->n_kv_heads;
    if (nq != 1 && nq != 2 && nq != 4) { *why = "n_q_heads / n_kv_heads must be 1, 2 or 4"; return KIVI_ERR_UNSUPPORTED; }
    if ((long long)c->batch * c->n_kv_heads > 65535) { *why = "batch * n_kv_heads must be <= 65535"; return KIVI_ERR_UNSUPPORTED; }
    if ((long long)c->batch * c->n_q_heads > 0x7fffffffLL) { *why = "batch * n_q_heads too large"; return KIVI_ERR_UNSUPPORTED; }
    if (c->max_tokens > (1LL << 30)) { *why = "max_tokens must be <= 2^30"; return KIVI_ERR_UNSUPPORTED; }
    g->B = c->batch; g->Hq = c->n_q_heads; g->Hkv = c->n_kv_heads; g->D = c->head_dim;
    g->bits = c->bits; g->G = c->group; g->R = c->residual; g->max_tokens = c->max_tokens;
    g->NB = c->max_tokens / c->group;
    g->tile_bytes = 2LL * g->D * g->bits;
    g->part_bytes = (g->G / 16) * g->tile_bytes + 4LL * g->D;
    g->slot_bytes = 2 * g->NB * g->part_bytes;
    const long long slots = (long long)g->B * g->Hkv;
    g->resid_slot_bytes = (long long)g->R * g->D * 2;
    g->k_resid_off = round_up(slots * g->slot_bytes, 256);
    g->v_resid_off = round_up(g->k_resid_off + slots * g->resid_slot_bytes, 256);
    g->total_bytes = round_up(g->v_resid_off + slots * g->resid_slot_bytes, 256);
    *why = "";
    return KIVI_OK;
}

}  // namespace kivi

extern "C" {

size_t kivi_cache_bytes(const kivi_config* cfg) {
    kivi::Geometry g;
    const char* why;
    if (kivi::derive_geometry(cfg, &g, &why) != KIVI_OK) { fail(KIVI_ERR_INVALID_ARG, "%s", why); return 0; }
    return (size_t)g.total_bytes;
}

kivi_status kivi_cache_layout(const kivi_config* cfg, kivi_layout* out) {
    if (!out) return fail(KIVI_ERR_INVALID_ARG, "null layout pointer");
    kivi::Geometry g;
    const char* why;
    const kivi_status st = kivi::derive_geometry(cfg, &g, &why);
    if (st != KIVI_OK) return fail(st, "%s", why);
    out->total_bytes = (size_t)g.total_bytes;
    out->blocks_per_slot = g.NB;
    out->tile_bytes = (size_t)g.tile_bytes;
    out->part_bytes = (size_t)g.part_bytes;
    out->slot_bytes = (size_t)g.slot_bytes;
    out->k_resid_offset = (size_t)g.k_resid_off;
    out->v_resid_offset = (size_t)g.v_resid_off;
    out->resid_slot_bytes = (size_t)g.resid_slot_bytes;
    return ok();
}

kivi_status kivi_cache_create(const kivi_config* cfg, void* dev_buf, size_t bytes, kivi_cache_t* out) {
    if (!out) return fail(KIVI_ERR_INVALID_ARG, "null output handle pointer");
    *out = nullptr;
    kivi::Geometry g;
    const char* why;
    const kivi_status st = kivi::derive_geometry(cfg, &g, &why);
    if (st != KIVI_OK) return fail(st, "%s", why);
    if (!dev_buf) return fail(KIVI_ERR_INVALID_ARG, "null cache buffer");
    if (!aligned(dev_buf, 256)) return fail(KIVI_ERR_INVALID_ARG, "cache buffer must be 256-byte aligned");
    if (bytes < (size_t)g.total_bytes)
        return fail(KIVI_ERR_CAPACITY, "cache buffer has %zu bytes, needs %lld", bytes, g.total_bytes);
    kivi_cache* c = new (std::nothrow) kivi_cache{g, static_cast<uint8_t*>(dev_buf), 0, 0, -1, 0, KIVI_DECODE_AUTO, 0, KIVI_FAULT_NONE, 0};
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "out of host memory");
    *out = c;
    return ok();
}

kivi_status kivi_cache_destroy(kivi_cache_t c) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    delete c;
    return ok();
}

kivi_status kivi_cache_reset(kivi_cache_t c) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    c->n_quant = 0;
    c->n_resid = 0;
    return ok();
}

kivi_status kivi_cache_counts(kivi_cache_t c, long long* n_quant, long long* n_resid) {
    if (!c || !n_quant || !n_resid) return fail(KIVI_ERR_INVALID_ARG, "null argument");
    *n_quant = c->n_quant;
    *n_resid = c->n_resid;
    return ok();
}

kivi_status kivi_prefill(kivi_cache_t c, const void* K, const void* V, long long L, kivi_stream_t stream) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    if (c->n_quant || c->n_resid) return fail(KIVI_ERR_STATE, "prefill needs an empty cache");
    if (L < 0) return fail(KIVI_ERR_INVALID_ARG, "negative length");
    if (L > c->geo.max_tokens) return fail(KIVI_ERR_CAPACITY, "prompt of %lld tokens exceeds max_tokens %lld", L, c->geo.max_tokens);
    if (L == 0) return ok();
    if (!K || !V) return fail(KIVI_ERR_INVALID_ARG, "null K or V");
    if (!aligned(K, 16) || !aligned(V, 16)) return fail(KIVI_ERR_INVALID_ARG, "K and V must be 16-byte aligned");
    const kivi_status sdev = ensure_device(c);
    if (sdev != KIVI_OK) return sdev;
    const kivi::Geometry& g = c->geo;
    const long long over = L > g.R ? L - g.R : 0;
    const long long Lq = (over + g.G - 1) / g.G * g.G;
    const long long r = L - Lq;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const __half* k = static_cast<const __half*>(K);
    const __half* v = static_cast<const __half*>(V);
    if (c->value_queue) {
        // values: all but the newest R are quantized (per token); the newest sit
        // in the ring at row position % R; keys as below
        const long long Lv = L > g.R ? L - g.R : 0;
        if (Lq) {
            const cudaError_t e = kivi::launch_quantize_blocks(g, c->buf, k, v, L * g.D, 0, Lq / g.G, st, Lv);
            if (e != cudaSuccess) return cuda_fail(e, "prefill quantize launch");
            g_launches++;
        }
        const cudaError_t e = kivi::launch_copy_rows_ring(g, c->buf, k, v, L * g.D, 0, Lq, (int)r, Lv, Lv,
                                                          (int)(L - Lv), st);
        if (e != cudaSuccess) return cuda_fail(e, "prefill residual copy launch");
        g_launches++;
        c->n_quant = Lq;
        c->n_resid = r;
        return ok();
    }
    if (Lq) {
        const cudaError_t e = kivi::launch_quantize_blocks(g, c->buf, k, v, L * g.D, 0, Lq / g.G, st);
        if (e != cudaSuccess) return cuda_fail(e, "prefill quantize launch");
        g_launches++;
    }
    if (r) {
        const cudaError_t e = kivi::launch_copy_rows(g, c->buf, k + Lq * g.D, v + Lq * g.D, L * g.D, 0, (int)r, st);
        if (e != cudaSuccess) return cuda_fail(e, "prefill residual copy launch");
        g_launches++;
    }
    c->n_quant = Lq;
    c->n_resid = r;
    return ok();
}

kivi_status kivi_append(kivi_cache_t c, const void* k, const void* v, kivi_stream_t stream) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    if (!k || !v) return fail(KIVI_ERR_INVALID_ARG, "null k or v");
    if (!aligned(k, 16) || !aligned(v, 16)) return fail(KIVI_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    const kivi::Geometry& g = c->geo;
    if (c->n_quant + c->n_resid + 1 > g.max_tokens)
        return fail(KIVI_ERR_CAPACITY, "cache already holds max_tokens (%lld) tokens", g.max_tokens);
    const kivi_status sdev = ensure_device(c);
    if (sdev != KIVI_OK) return sdev;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (c->value_queue) {
        bool unused;
        const kivi_status sq = queue_before_append(c, st, true, &unused);
        if (sq != KIVI_OK) return sq;
        const long long L = c->n_quant + c->n_resid;
        const cudaError_t e = kivi::launch_copy_rows_ring(g, c->buf, static_cast<const __half*>(k),
                                                          static_cast<const __half*>(v), g.D, (int)c->n_resid, 0, 1,
                                                          L, 0, 1, st);
        if (e != cudaSuccess) return cuda_fail(e, "append copy launch");
        g_launches++;
        c->n_resid += 1;
        return ok();
    }
    if (c->n_resid == g.R) {
        const __half* rk = reinterpret_cast<const __half*>(c->buf + g.k_resid_off);
        const __half* rv = reinterpret_cast<const __half*>(c->buf + g.v_resid_off);
        const cudaError_t e = kivi::launch_quantize_blocks(g, c->buf, rk, rv, (long long)g.R * g.D,
                                                           c->n_quant / g.G, g.R / g.G, st);
        if (e != cudaSuccess) return cuda_fail(e, "residual flush launch");
        g_launches++;
        c->n_quant += g.R;
        c->n_resid = 0;
    }
    const cudaError_t e = kivi::launch_copy_rows(g, c->buf, static_cast<const __half*>(k),
                                                 static_cast<const __half*>(v), g.D, (int)c->n_resid, 1, st);
    if (e != cudaSuccess) return cuda_fail(e, "append copy launch");
    g_launches++;
    c->n_resid += 1;
    return ok();
}

size_t kivi_decode_workspace_bytes(const kivi_config* cfg) {
    kivi::Geometry g;
    const char* why;
    if (kivi::derive_geometry(cfg, &g, &why) != KIVI_OK) { fail(KIVI_ERR_INVALID_ARG, "%s", why); return 0; }
    return (size_t)g.B * g.Hq * kivi::kPartialSlots * kivi::partial_stride(g.D) * sizeof(float);
}

}  // extern "C"

namespace {

// Checks of a decode call that do not depend on the cache's token counts.
kivi_status decode_checks(kivi_cache_t c, const void* q, void* out, float softmax_scale, void* workspace,
                          size_t ws_bytes) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    if (!q || !out || !workspace) return fail(KIVI_ERR_INVALID_ARG, "null q, out or workspace");
    if (!aligned(q, 16) || !aligned(out, 16)) return fail(KIVI_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return fail(KIVI_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (!(softmax_scale == softmax_scale) || isinf(softmax_scale)) return fail(KIVI_ERR_INVALID_ARG, "softmax_scale must be finite");
    const kivi::Geometry& g = c->geo;
    const size_t need = (size_t)g.B * g.Hq * kivi::kPartialSlots * kivi::partial_stride(g.D) * sizeof(float);
    if (ws_bytes < need) return fail(KIVI_ERR_CAPACITY, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    return KIVI_OK;
}


// Launch a decode call over n_resid residual rows (fa.row < n_resid: a fused append's row).
kivi_status decode_launch(kivi_cache_t c, const void* q, void* out, float softmax_scale, void* workspace,
                          long long n_resid, int variant, kivi_stream_t stream, const kivi::FusedAppend& fa) {
    const kivi::Geometry& g = c->geo;
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)g.D);
    const float scale_log2 = scale * 1.4426950408889634f;
    kivi::DecodePlan plan = kivi::plan_decode(g, c->n_quant, n_resid, c->num_sms);
    plan.max_ctas = c->max_ctas;
    int launches = 0;
    kivi::FusedAppend f2 = fa;
    if (variant == KIVI_DECODE_TENSOR_CORE && c->fault == KIVI_FAULT_COPY_STALL) {
        f2.stall_bytes = 16;
        c->fault = KIVI_FAULT_NONE;   // one call
    }
    const cudaError_t e = kivi::launch_decode(g, c->buf, c->n_quant, n_resid, static_cast<const __half*>(q),
                                              static_cast<__half*>(out), scale_log2, static_cast<float*>(workspace),
                                              plan, variant, reinterpret_cast<cudaStream_t>(stream), &launches, f2);
    g_launches += (unsigned long long)launches;
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ok();
}

}  // namespace

extern "C" {

kivi_status kivi_decode_attn(kivi_cache_t c, const void* q, void* out, float softmax_scale,
                             void* workspace, size_t ws_bytes, kivi_stream_t stream) {
    const kivi_status st = decode_checks(c, q, out, softmax_scale, workspace, ws_bytes);
    if (st != KIVI_OK) return st;
    if (c->n_quant + c->n_resid == 0) return fail(KIVI_ERR_STATE, "decode on an empty cache");
    const int variant = c->decode_kernel == KIVI_DECODE_AUTO ? KIVI_DECODE_TENSOR_CORE : c->decode_kernel;
    if (c->value_queue && variant != KIVI_DECODE_TENSOR_CORE)
        return fail(KIVI_ERR_UNSUPPORTED, "the value queue is decoded by the tensor-core kernel only");
    const kivi_status sdev = ensure_device(c);
    if (sdev != KIVI_OK) return sdev;
    kivi::FusedAppend fa;
    if (c->value_queue) {
        const long long L = c->n_quant + c->n_resid;
        fa.lqv = L > c->geo.R ? L - c->geo.R : 0;
    }
    return decode_launch(c, q, out, softmax_scale, workspace, c->n_resid, variant, stream, fa);
}

kivi_status kivi_append_decode(kivi_cache_t c, const void* k, const void* v, const void* q, void* out,
                               float softmax_scale, void* workspace, size_t ws_bytes, kivi_stream_t stream) {
    const kivi_status st = decode_checks(c, q, out, softmax_scale, workspace, ws_bytes);
    if (st != KIVI_OK) return st;
    if (!k || !v) return fail(KIVI_ERR_INVALID_ARG, "null k or v");
    if (!aligned(k, 16) || !aligned(v, 16)) return fail(KIVI_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    const kivi::Geometry& g = c->geo;
    if (c->n_quant + c->n_resid + 1 > g.max_tokens)
        return fail(KIVI_ERR_CAPACITY, "cache already holds max_tokens (%lld) tokens", g.max_tokens);
    const int variant = c->decode_kernel == KIVI_DECODE_AUTO ? KIVI_DECODE_TENSOR_CORE : c->decode_kernel;
    if (c->value_queue && variant != KIVI_DECODE_TENSOR_CORE)
        return fail(KIVI_ERR_UNSUPPORTED, "the value queue is decoded by the tensor-core kernel only");
    if (variant != KIVI_DECODE_TENSOR_CORE) {
        // the CUDA-core kernel has no fused form: append, then decode
        const kivi_status sa = kivi_append(c, k, v, stream);
        if (sa != KIVI_OK) return sa;
        return kivi_decode_attn(c, q, out, softmax_scale, workspace, ws_bytes, stream);
    }
    const kivi_status sdev = ensure_device(c);
    if (sdev != KIVI_OK) return sdev;
    cudaStream_t sp = reinterpret_cast<cudaStream_t>(stream);
    bool flushed = false;
    if (c->value_queue) {
        const kivi_status sq = queue_before_append(c, sp, false, &flushed);
        if (sq != KIVI_OK) return sq;
        // the decode kernel pops position L - R (quantizes that value into its
        // block, counts it as quantized) and stores the new value in its ring row
        const long long L = c->n_quant + c->n_resid;   // before the new token
        kivi::FusedAppend fa;
        fa.k = static_cast<const __half*>(k);
        fa.v = static_cast<const __half*>(v);
        fa.row = (int)c->n_resid;
        fa.early_ok = flushed ? 0 : 1;
        fa.lqv = L >= g.R ? L + 1 - g.R : 0;
        fa.pop = L >= g.R ? L - g.R : -1;
        const kivi_status sd = decode_launch(c, q, out, softmax_scale, workspace, c->n_resid + 1, variant, stream, fa);
        if (sd != KIVI_OK) return sd;
        c->n_resid += 1;
        return ok();
    }
    if (c->n_resid == g.R) {
        const __half* rk = reinterpret_cast<const __half*>(c->buf + g.k_resid_off);
        const __half* rv = reinterpret_cast<const __half*>(c->buf + g.v_resid_off);
        const cudaError_t e = kivi::launch_quantize_blocks(g, c->buf, rk, rv, (long long)g.R * g.D,
                                                           c->n_quant / g.G, g.R / g.G, sp);
        if (e != cudaSuccess) return cuda_fail(e, "residual flush launch");
        g_launches++;
        c->n_quant += g.R;
        c->n_resid = 0;
        flushed = true;
    }
    kivi::FusedAppend fa;
    fa.k = static_cast<const __half*>(k);
    fa.v = static_cast<const __half*>(v);
    fa.row = (int)c->n_resid;
    fa.early_ok = flushed ? 0 : 1;   // the flush writes blocks right before the decode
    const kivi_status sd = decode_launch(c, q, out, softmax_scale, workspace, c->n_resid + 1, variant, stream, fa);
    if (sd != KIVI_OK) return sd;
    c->n_resid += 1;
    return ok();
}

kivi_status kivi_cache_set_value_residual(kivi_cache_t c, int mode) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    if (mode != KIVI_VALUE_FLUSH && mode != KIVI_VALUE_QUEUE) return fail(KIVI_ERR_INVALID_ARG, "unknown value residual mode %d", mode);
    if (c->n_quant || c->n_resid) return fail(KIVI_ERR_STATE, "the value residual mode is set on an empty cache");
    if (mode == KIVI_VALUE_QUEUE && c->geo.R > 128)
        return fail(KIVI_ERR_UNSUPPORTED, "the value queue needs residual <= 128 (residual is %d)", c->geo.R);
    c->value_queue = mode == KIVI_VALUE_QUEUE;
    return ok();
}

kivi_status kivi_cache_set_max_ctas(kivi_cache_t c, int max_ctas) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    if (max_ctas < 0) return fail(KIVI_ERR_INVALID_ARG, "max_ctas must be >= 0");
    c->max_ctas = max_ctas;
    return ok();
}

kivi_status kivi_cache_set_fault(kivi_cache_t c, int fault) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    if (fault != KIVI_FAULT_NONE && fault != KIVI_FAULT_COPY_STALL) return fail(KIVI_ERR_INVALID_ARG, "unknown fault %d", fault);
    c->fault = fault;
    return ok();
}

kivi_status kivi_cache_set_decode_kernel(kivi_cache_t c, int kernel) {
    if (!c) return fail(KIVI_ERR_INVALID_ARG, "null handle");
    if (kernel != KIVI_DECODE_AUTO && kernel != KIVI_DECODE_CUDA_CORE && kernel != KIVI_DECODE_TENSOR_CORE)
        return fail(KIVI_ERR_INVALID_ARG, "unknown decode kernel %d", kernel);
    c->decode_kernel = kernel;
    return ok();
}

const char* kivi_last_error_string(void) { return g_err; }

unsigned long long kivi_launch_count(void) { return g_launches.load(); }

}  // extern "C"

namespace kivi {

kivi_status report_error(kivi_status st, const char* msg) { return fail(st, "%s", msg); }

void count_launches(int n) { g_launches += (unsigned long long)n; }

kivi_status cache_device(kivi_cache* c) { return ensure_device(c); }

size_t decode_workspace_need(const kivi_cache* c) {
    const Geometry& g = c->geo;
    return (size_t)g.B * g.Hq * kPartialSlots * partial_stride(g.D) * sizeof(float);
}

}  // namespace kivi

static kivi_status queue_before_append(kivi_cache* c, cudaStream_t st, bool pop, bool* wrote) {
    const kivi::Geometry& g = c->geo;
    *wrote = false;
    const long long L = c->n_quant + c->n_resid;
    const long long Lv = L > g.R ? L - g.R : 0;   // values quantized so far
    if (c->n_resid == g.R) {
        // keys [Lq, Lq + R) into blocks; their values are all >= Lv, so written as
        // not quantized yet (the value source is not read for them)
        const __half* rk = reinterpret_cast<const __half*>(c->buf + g.k_resid_off);
        const cudaError_t e = kivi::launch_quantize_blocks(g, c->buf, rk, rk, (long long)g.R * g.D,
                                                           c->n_quant / g.G, g.R / g.G, st, Lv);
        if (e != cudaSuccess) return cuda_fail(e, "residual flush launch");
        g_launches++;
        c->n_quant += g.R;
        c->n_resid = 0;
        *wrote = true;
    }
    if (pop && L >= g.R) {
        const cudaError_t e = kivi::launch_pop_values(g, c->buf, L - g.R, st);
        if (e != cudaSuccess) return cuda_fail(e, "value queue launch");
        g_launches++;
        *wrote = true;
    }
    return ok();
}

