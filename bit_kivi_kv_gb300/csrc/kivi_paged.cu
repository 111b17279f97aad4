// Host side of the paged cache (include/kivi.h, "Paged cache with ragged
// sequences"): shape checks, the page and sequence-slot allocator, each
// sequence's streaming state, and the launches.
//
// Each sequence follows the streaming rule of the dense cache on its own
// (KIVI explainer, discosf.com, 3.1; "KV cache quantization axis selection
// guide", unite.ai, "the system tax"); blocks live in pool pages addressed
// through a block table (the same explainer, section 7, points to
// PagedAttention for this).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <new>
#include <vector>

#include "kivi_common.cuh"

namespace {

struct SeqState {
    bool live = false;
    long long n_quant = 0;   // Lq
    int n_resid = 0;         // r
    std::vector<int> pages;  // page of block n, n < Lq / G
};

long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kivi_status failf(kivi_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kivi_status failf(kivi_status st, const char* fmt, ...) {
    char msg[400];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    return kivi::report_error(st, msg);
}

kivi_status ok() { return kivi::report_error(KIVI_OK, ""); }

kivi_status cuda_fail(cudaError_t e, const char* what) {
    return failf(KIVI_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

kivi_status derive_paged(const kivi_paged_config* c, kivi::PagedGeometry* pg, const char** why) {
    if (!c) { *why = "null config"; return KIVI_ERR_INVALID_ARG; }
    if (c->max_seqs < 1 || c->max_blocks_per_seq < 1 || c->n_pages < 1) {
        *why = "max_seqs, max_blocks_per_seq and n_pages must be positive";
        return KIVI_ERR_INVALID_ARG;
    }
    if (c->n_pages >= (1LL << 31)) { *why = "n_pages must be < 2^31"; return KIVI_ERR_UNSUPPORTED; }
    if ((long long)c->max_seqs * c->max_blocks_per_seq >= (1LL << 31)) {
        *why = "max_seqs * max_blocks_per_seq must be < 2^31";
        return KIVI_ERR_UNSUPPORTED;
    }
    // the per-sequence shape rules are those of a dense cache of max_seqs rows
    kivi_config dc{c->max_seqs, c->n_q_heads, c->n_kv_heads, c->head_dim, c->bits, c->group, c->residual,
                   (long long)c->max_blocks_per_seq * (c->group > 0 ? c->group : 1) + c->residual};
    kivi::Geometry& g = pg->g;
    const kivi_status st = kivi::derive_geometry(&dc, &g, why);
    if (st != KIVI_OK) return st;
    g.NB = c->max_blocks_per_seq;
    g.slot_bytes = 0;
    const long long slots = (long long)g.B * g.Hkv;
    pg->n_pages = c->n_pages;
    pg->page_bytes = (long long)g.Hkv * 2 * g.part_bytes;
    g.k_resid_off = round_up(pg->n_pages * pg->page_bytes, 256);
    g.v_resid_off = round_up(g.k_resid_off + slots * g.resid_slot_bytes, 256);
    pg->table_off = round_up(g.v_resid_off + slots * g.resid_slot_bytes, 256);
    g.total_bytes = round_up(pg->table_off + (long long)g.B * g.NB * 4, 256);
    *why = "";
    return KIVI_OK;
}

size_t paged_ws_need(const kivi::Geometry& g, int n) {
    return (size_t)n * g.Hq * kivi::kPartialSlots * kivi::partial_stride(g.D) * sizeof(float);
}

}  // namespace

struct kivi_paged {
    kivi::PagedGeometry pg;
    uint8_t* buf;
    std::vector<int> free_pages;   // stack: the next page handed out is at the back
    std::vector<int> free_seqs;
    std::vector<SeqState> seqs;
    std::vector<unsigned> mark;    // call stamp per sequence (duplicate check)
    unsigned stamp = 0;
    int device = -1;
    int num_sms = 0;
    int max_ctas = 0;              // decode grid cap (0: the launch sizes it)
};

namespace {

// The cache's device: the device current at the handle's first launching
// call; later launching calls must find it current.
kivi_status paged_device(kivi_paged* c) {
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
        return failf(KIVI_ERR_INVALID_ARG, "the cache is on device %d but device %d is current", c->device, dev);
    }
    return KIVI_OK;
}

bool live_seq(const kivi_paged* c, int s) {
    return s >= 0 && s < (int)c->seqs.size() && c->seqs[s].live;
}

}  // namespace

extern "C" {

size_t kivi_paged_bytes(const kivi_paged_config* cfg) {
    kivi::PagedGeometry pg;
    const char* why;
    if (derive_paged(cfg, &pg, &why) != KIVI_OK) { failf(KIVI_ERR_INVALID_ARG, "%s", why); return 0; }
    return (size_t)pg.g.total_bytes;
}

kivi_status kivi_paged_cache_layout(const kivi_paged_config* cfg, kivi_paged_layout* out) {
    if (!out) return failf(KIVI_ERR_INVALID_ARG, "null layout pointer");
    kivi::PagedGeometry pg;
    const char* why;
    const kivi_status st = derive_paged(cfg, &pg, &why);
    if (st != KIVI_OK) return failf(st, "%s", why);
    out->total_bytes = (size_t)pg.g.total_bytes;
    out->tile_bytes = (size_t)pg.g.tile_bytes;
    out->part_bytes = (size_t)pg.g.part_bytes;
    out->page_bytes = (size_t)pg.page_bytes;
    out->k_resid_offset = (size_t)pg.g.k_resid_off;
    out->v_resid_offset = (size_t)pg.g.v_resid_off;
    out->resid_seq_bytes = (size_t)(pg.g.Hkv * pg.g.resid_slot_bytes);
    out->table_offset = (size_t)pg.table_off;
    return ok();
}

kivi_status kivi_paged_create(const kivi_paged_config* cfg, void* dev_buf, size_t bytes, kivi_paged_t* out) {
    if (!out) return failf(KIVI_ERR_INVALID_ARG, "null output handle pointer");
    *out = nullptr;
    kivi::PagedGeometry pg;
    const char* why;
    const kivi_status st = derive_paged(cfg, &pg, &why);
    if (st != KIVI_OK) return failf(st, "%s", why);
    if (!dev_buf) return failf(KIVI_ERR_INVALID_ARG, "null cache buffer");
    if (!aligned(dev_buf, 256)) return failf(KIVI_ERR_INVALID_ARG, "cache buffer must be 256-byte aligned");
    if (bytes < (size_t)pg.g.total_bytes)
        return failf(KIVI_ERR_CAPACITY, "cache buffer has %zu bytes, needs %lld", bytes, pg.g.total_bytes);
    kivi_paged* c = new (std::nothrow) kivi_paged;
    if (!c) return failf(KIVI_ERR_INVALID_ARG, "out of host memory");
    try {
        c->pg = pg;
        c->buf = static_cast<uint8_t*>(dev_buf);
        c->free_pages.resize((size_t)pg.n_pages);
        for (long long p = 0; p < pg.n_pages; ++p) c->free_pages[(size_t)p] = (int)(pg.n_pages - 1 - p);
        c->free_seqs.resize((size_t)pg.g.B);
        for (int s = 0; s < pg.g.B; ++s) c->free_seqs[(size_t)s] = pg.g.B - 1 - s;
        c->seqs.resize((size_t)pg.g.B);
        c->mark.assign((size_t)pg.g.B, 0u);
    } catch (const std::bad_alloc&) {
        delete c;
        return failf(KIVI_ERR_INVALID_ARG, "out of host memory");
    }
    *out = c;
    return ok();
}

kivi_status kivi_paged_destroy(kivi_paged_t c) {
    if (!c) return failf(KIVI_ERR_INVALID_ARG, "null handle");
    delete c;
    return ok();
}

kivi_status kivi_paged_add(kivi_paged_t c, const void* K, const void* V, long long L, kivi_stream_t stream,
                           int* seq) {
    if (!c || !seq) return failf(KIVI_ERR_INVALID_ARG, "null handle or sequence pointer");
    if (L < 0) return failf(KIVI_ERR_INVALID_ARG, "negative length");
    if (L > 0 && (!K || !V)) return failf(KIVI_ERR_INVALID_ARG, "null K or V");
    if (L > 0 && (!aligned(K, 16) || !aligned(V, 16)))
        return failf(KIVI_ERR_INVALID_ARG, "K and V must be 16-byte aligned");
    const kivi::Geometry& g = c->pg.g;
    if (c->free_seqs.empty()) return failf(KIVI_ERR_CAPACITY, "all %d sequence slots are in use", g.B);
    const long long over = L > g.R ? L - g.R : 0;
    const long long Lq = (over + g.G - 1) / g.G * g.G;
    const long long r = L - Lq;
    const long long nblk = Lq / g.G;
    if (nblk > g.NB)
        return failf(KIVI_ERR_CAPACITY, "prompt of %lld tokens needs %lld blocks, max_blocks_per_seq is %lld", L,
                     nblk, g.NB);
    if (nblk > (long long)c->free_pages.size())
        return failf(KIVI_ERR_CAPACITY, "prompt needs %lld pages, %zu are free", nblk, c->free_pages.size());
    if (L > 0) {
        const kivi_status sdev = paged_device(c);
        if (sdev != KIVI_OK) return sdev;
    }
    const int s = c->free_seqs.back();
    SeqState& sq = c->seqs[(size_t)s];
    sq.pages.clear();
    sq.pages.reserve((size_t)nblk);
    std::vector<kivi::QJob> jobs((size_t)nblk);
    for (long long j = 0; j < nblk; ++j) {
        const int page = c->free_pages[c->free_pages.size() - 1 - (size_t)j];
        sq.pages.push_back(page);
        jobs[(size_t)j] = kivi::QJob{j * g.G * g.D, page, (int)((long long)s * g.NB + j)};
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const __half* k = static_cast<const __half*>(K);
    const __half* v = static_cast<const __half*>(V);
    if (nblk) {
        int n = 0;
        const cudaError_t e = kivi::launch_quantize_pages(c->pg, c->buf, k, v, L * g.D, jobs.data(), (int)nblk, st, &n);
        kivi::count_launches(n);
        if (e != cudaSuccess) { sq.pages.clear(); return cuda_fail(e, "prompt quantize launch"); }
    }
    if (r) {
        const cudaError_t e = kivi::launch_copy_rows_slots(g, c->buf, k + Lq * g.D, v + Lq * g.D, L * g.D,
                                                           (long long)s * g.Hkv, g.Hkv, 0, (int)r, st);
        kivi::count_launches(1);
        if (e != cudaSuccess) { sq.pages.clear(); return cuda_fail(e, "prompt residual copy launch"); }
    }
    c->free_pages.resize(c->free_pages.size() - (size_t)nblk);
    c->free_seqs.pop_back();
    sq.live = true;
    sq.n_quant = Lq;
    sq.n_resid = (int)r;
    *seq = s;
    return ok();
}

kivi_status kivi_paged_release(kivi_paged_t c, int s) {
    if (!c) return failf(KIVI_ERR_INVALID_ARG, "null handle");
    if (!live_seq(c, s)) return failf(KIVI_ERR_INVALID_ARG, "sequence %d is not live", s);
    SeqState& sq = c->seqs[(size_t)s];
    for (size_t j = sq.pages.size(); j-- > 0;) c->free_pages.push_back(sq.pages[j]);
    sq.pages.clear();
    sq.live = false;
    sq.n_quant = 0;
    sq.n_resid = 0;
    c->free_seqs.push_back(s);
    return ok();
}

kivi_status kivi_paged_seq_counts(kivi_paged_t c, int s, long long* n_quant, long long* n_resid) {
    if (!c || !n_quant || !n_resid) return failf(KIVI_ERR_INVALID_ARG, "null argument");
    if (!live_seq(c, s)) return failf(KIVI_ERR_INVALID_ARG, "sequence %d is not live", s);
    *n_quant = c->seqs[(size_t)s].n_quant;
    *n_resid = c->seqs[(size_t)s].n_resid;
    return ok();
}

kivi_status kivi_paged_seq_pages(kivi_paged_t c, int s, int* pages, int cap, int* n) {
    if (!c || !n || (cap > 0 && !pages)) return failf(KIVI_ERR_INVALID_ARG, "null argument");
    if (!live_seq(c, s)) return failf(KIVI_ERR_INVALID_ARG, "sequence %d is not live", s);
    const std::vector<int>& pv = c->seqs[(size_t)s].pages;
    for (int j = 0; j < cap && j < (int)pv.size(); ++j) pages[j] = pv[(size_t)j];
    *n = (int)pv.size();
    return ok();
}

kivi_status kivi_paged_free(kivi_paged_t c, long long* free_pages, int* free_seqs) {
    if (!c || !free_pages || !free_seqs) return failf(KIVI_ERR_INVALID_ARG, "null argument");
    *free_pages = (long long)c->free_pages.size();
    *free_seqs = (int)c->free_seqs.size();
    return ok();
}

kivi_status kivi_paged_set_max_ctas(kivi_paged_t c, int max_ctas) {
    if (!c) return failf(KIVI_ERR_INVALID_ARG, "null handle");
    if (max_ctas < 0) return failf(KIVI_ERR_INVALID_ARG, "max_ctas must be >= 0");
    c->max_ctas = max_ctas;
    return ok();
}

size_t kivi_paged_workspace_bytes(const kivi_paged_config* cfg, int n) {
    kivi::PagedGeometry pg;
    const char* why;
    if (derive_paged(cfg, &pg, &why) != KIVI_OK) { failf(KIVI_ERR_INVALID_ARG, "%s", why); return 0; }
    if (n < 1 || n > kivi::kMaxCallSeqs) {
        failf(KIVI_ERR_INVALID_ARG, "n must be in [1, %d]", kivi::kMaxCallSeqs);
        return 0;
    }
    return paged_ws_need(pg.g, n);
}

kivi_status kivi_paged_append_decode(kivi_paged_t c, const int* seqs, int n, const void* k, const void* v,
                                     const void* q, void* out, float softmax_scale, void* workspace,
                                     size_t ws_bytes, kivi_stream_t stream) {
    if (!c) return failf(KIVI_ERR_INVALID_ARG, "null handle");
    if (!seqs) return failf(KIVI_ERR_INVALID_ARG, "null sequence list");
    if (n < 1 || n > kivi::kMaxCallSeqs) return failf(KIVI_ERR_INVALID_ARG, "n must be in [1, %d]", kivi::kMaxCallSeqs);
    if (!q || !out || !workspace) return failf(KIVI_ERR_INVALID_ARG, "null q, out or workspace");
    if (!aligned(q, 16) || !aligned(out, 16)) return failf(KIVI_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return failf(KIVI_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (!(softmax_scale == softmax_scale) || isinf(softmax_scale))
        return failf(KIVI_ERR_INVALID_ARG, "softmax_scale must be finite");
    if ((k == nullptr) != (v == nullptr)) return failf(KIVI_ERR_INVALID_ARG, "k and v must both be given or both be null");
    const bool append = k != nullptr;
    if (append && (!aligned(k, 16) || !aligned(v, 16))) return failf(KIVI_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    const kivi::Geometry& g = c->pg.g;
    const size_t need = paged_ws_need(g, n);
    if (ws_bytes < need) return failf(KIVI_ERR_CAPACITY, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    // every check before any launch or state change
    if (++c->stamp == 0) {   // stamp wrapped: clear the marks
        c->mark.assign(c->mark.size(), 0u);
        c->stamp = 1;
    }
    long long flush_pages = 0;
    for (int i = 0; i < n; ++i) {
        const int s = seqs[i];
        if (!live_seq(c, s)) return failf(KIVI_ERR_INVALID_ARG, "sequence %d (entry %d) is not live", s, i);
        if (c->mark[(size_t)s] == c->stamp) return failf(KIVI_ERR_INVALID_ARG, "sequence %d is listed twice", s);
        c->mark[(size_t)s] = c->stamp;
        const SeqState& sq = c->seqs[(size_t)s];
        if (append && sq.n_resid == g.R) {
            if (sq.n_quant / g.G + g.R / g.G > g.NB)
                return failf(KIVI_ERR_CAPACITY, "sequence %d is full (%lld tokens)", s, sq.n_quant + sq.n_resid);
            flush_pages += g.R / g.G;
        }
        if (!append && sq.n_quant + sq.n_resid == 0)
            return failf(KIVI_ERR_STATE, "decode of sequence %d, which holds no token", s);
    }
    if (flush_pages > (long long)c->free_pages.size())
        return failf(KIVI_ERR_CAPACITY, "flushes need %lld pages, %zu are free", flush_pages, c->free_pages.size());
    const kivi_status sdev = paged_device(c);
    if (sdev != KIVI_OK) return sdev;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // flushes: the R residual rows of each full sequence become R / G blocks in new pages
    std::vector<kivi::QJob> jobs;
    std::vector<kivi::PagedSeq> call((size_t)n);
    size_t taken = 0;
    if (flush_pages) {
        jobs.reserve((size_t)flush_pages);
        for (int i = 0; i < n; ++i) {
            const int s = seqs[i];
            const SeqState& sq = c->seqs[(size_t)s];
            if (!(append && sq.n_resid == g.R)) continue;
            for (int jj = 0; jj < g.R / g.G; ++jj) {
                const int page = c->free_pages[c->free_pages.size() - 1 - taken++];
                jobs.push_back(kivi::QJob{(long long)s * g.Hkv * g.R * g.D + (long long)jj * g.G * g.D, page,
                                          (int)((long long)s * g.NB + sq.n_quant / g.G + jj)});
            }
        }
        const __half* rk = reinterpret_cast<const __half*>(c->buf + g.k_resid_off);
        const __half* rv = reinterpret_cast<const __half*>(c->buf + g.v_resid_off);
        int nl = 0;
        const cudaError_t e = kivi::launch_quantize_pages(c->pg, c->buf, rk, rv, (long long)g.R * g.D, jobs.data(),
                                                          (int)jobs.size(), st, &nl);
        kivi::count_launches(nl);
        if (e != cudaSuccess) return cuda_fail(e, "residual flush launch");
    }
    for (int i = 0; i < n; ++i) {
        const SeqState& sq = c->seqs[(size_t)seqs[i]];
        const bool fl = append && sq.n_resid == g.R;
        const long long lq = sq.n_quant + (fl ? g.R : 0);
        const int r = fl ? 0 : sq.n_resid;
        call[(size_t)i] = kivi::PagedSeq{0, seqs[i], (int)(lq / 32), r + (append ? 1 : 0), append ? r : -1};
    }
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)g.D);
    int nl = 0;
    const cudaError_t e = kivi::launch_decode_paged(
        c->pg, c->buf, call.data(), n, static_cast<const __half*>(q), static_cast<__half*>(out),
        scale * 1.4426950408889634f, static_cast<float*>(workspace), static_cast<const __half*>(k),
        static_cast<const __half*>(v), flush_pages ? 0 : 1, c->num_sms, c->max_ctas, st, &nl);
    kivi::count_launches(nl);
    // the flushes were enqueued: their pages belong to the sequences whatever the decode launch did
    size_t used = 0;
    for (int i = 0; i < n && flush_pages; ++i) {
        SeqState& sq = c->seqs[(size_t)seqs[i]];
        if (!(append && sq.n_resid == g.R)) continue;
        for (int jj = 0; jj < g.R / g.G; ++jj) sq.pages.push_back(c->free_pages[c->free_pages.size() - 1 - used++]);
        sq.n_quant += g.R;
        sq.n_resid = 0;
    }
    c->free_pages.resize(c->free_pages.size() - used);
    if (e != cudaSuccess) return cuda_fail(e, "paged decode launch");
    if (append)
        for (int i = 0; i < n; ++i) c->seqs[(size_t)seqs[i]].n_resid += 1;
    return ok();
}

}  // extern "C"
