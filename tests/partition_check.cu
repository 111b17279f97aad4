// Host-only check of the decode partition (the work map in kivi_common.cuh),
// built and run by tests/test_partition.py.  For random dense and ragged calls
// (dense ones with mixed pairs, as a value-queue cache has) it walks every
// worker's (warp's) weight range the way the decode kernel does
// and checks that every unit (tile pair or residual pair) of every slot is
// owned by exactly one worker, that a slot's partial indices (workers with
// units, and workers inside the slot without a unit start, which write an
// empty partial) are 0 .. parts-1 once each, and that no slot has more
// partials than the workspace holds.
#include <cstdio>
#include <random>
#include <vector>

#include "kivi_common.cuh"

using namespace kivi;

namespace {

struct Slot {
    long long P, PR, w0, Ws, M = 0;   // M: mixed pairs (the last M of the P)
};

// the worker-count rule of the launch: resident warps (4 a CTA), or the
// caller's cap on CTAs times 4, then the two bounds
long long grid_size(long long Wt, long long wmin, long long slots_of_max, long long resident, long long cap) {
    long long n = resident * 4;
    if (cap > 0 && cap * 4 < n) n = cap * 4;
    if (n > (kMaxSplits - 1) * slots_of_max) n = (kMaxSplits - 1) * slots_of_max;
    if (n > Wt / wmin) n = Wt / wmin;
    return n < 1 ? 1 : n;
}

bool check(const std::vector<Slot>& slots, const WorkMap& wm, int trial) {
    std::vector<std::vector<int>> owner(slots.size()), part(slots.size()), empty(slots.size());
    for (size_t s = 0; s < slots.size(); ++s) {
        owner[s].assign((size_t)(slots[s].P + slots[s].PR), -1);
        part[s].assign((size_t)(slots[s].P + slots[s].PR), -1);
    }
    size_t si = 0;
    for (long long c = 0; c < wm.n; ++c) {
        long long pos = map_begin(wm, c);
        const long long pe = map_begin(wm, c + 1);
        while (pos < pe) {
            while (si + 1 < slots.size() && slots[si + 1].w0 <= pos) ++si;   // the slot holding pos
            while (si > 0 && slots[si].w0 > pos) --si;
            const Slot& sl = slots[si];
            const long long NU = sl.P + sl.PR;
            const long long u0 = first_unit_at_p(wm, sl.P, sl.M, pos - sl.w0);
            if (u0 >= NU) { pos = sl.w0 + sl.Ws; continue; }
            if (sl.w0 + unit_start_p(wm, sl.P, sl.M, u0) >= pe) {
                // no unit start in the range: inside the slot, an empty partial
                if (u0 > 0) empty[si].push_back((int)(c - map_owner(wm, sl.w0 + wm.S0)));
                break;
            }
            const long long u1 = first_unit_at_p(wm, sl.P, sl.M, pe - sl.w0 < sl.Ws ? pe - sl.w0 : sl.Ws);
            const long long p = c - map_owner(wm, sl.w0 + wm.S0);
            for (long long u = u0; u < u1; ++u) {
                if (owner[si][(size_t)u] != -1) { std::printf("trial %d: unit owned twice\n", trial); return false; }
                owner[si][(size_t)u] = (int)c;
                part[si][(size_t)u] = (int)p;
            }
            pos = u1 >= NU ? sl.w0 + sl.Ws : sl.w0 + unit_start_p(wm, sl.P, sl.M, u1);
        }
    }
    for (size_t s = 0; s < slots.size(); ++s) {
        const Slot& sl = slots[s];
        const long long last = sl.w0 + unit_start_p(wm, sl.P, sl.M, sl.P + sl.PR - 1);
        const long long nparts = map_owner(wm, last) - map_owner(wm, sl.w0 + wm.S0) + 1;
        if (nparts < 1 || nparts > kPartialSlots) { std::printf("trial %d: %lld parts\n", trial, nparts); return false; }
        std::vector<int> seen((size_t)nparts, 0);
        for (size_t u = 0; u < owner[s].size(); ++u) {
            if (owner[s][u] < 0) { std::printf("trial %d: unit not owned\n", trial); return false; }
            if (part[s][u] < 0 || part[s][u] >= nparts) { std::printf("trial %d: part out of range\n", trial); return false; }
            seen[(size_t)part[s][u]] = 1;
        }
        for (int p : empty[s]) {
            if (p < 0 || p >= nparts || seen[(size_t)p]) { std::printf("trial %d: bad empty part %d\n", trial, p); return false; }
            seen[(size_t)p] = 1;
        }
        for (long long p = 0; p < nparts; ++p)
            if (!seen[(size_t)p]) { std::printf("trial %d: part %lld has no unit\n", trial, p); return false; }
    }
    return true;
}

}  // namespace

int main() {
    std::mt19937_64 rng(12345);
    auto pick = [&](long long lo, long long hi) { return lo + (long long)(rng() % (unsigned long long)(hi - lo + 1)); };
    const long long wqs[] = {40, 64, 96, 136, 288}, wrs[] = {160, 256, 320, 512}, wxs[] = {1, 128, 256};
    for (int trial = 0; trial < 4000; ++trial) {
        WorkMap wm{};
        wm.wq = wqs[pick(0, 4)];
        wm.wr = wrs[pick(0, 3)];
        const bool ragged = trial % 2 == 1;
        const long long nslots = pick(1, trial % 7 == 0 ? 2000 : 300);
        std::vector<Slot> slots((size_t)nslots);
        long long start = 0, ws_min = -1, ws_max = 0;
        const long long P0 = pick(0, 400), PR0 = pick(P0 == 0 ? 1 : 0, 4);
        // dense calls of a value-queue cache: the last M0 (<= 4) pairs are mixed
        const long long M0 = ragged || trial % 3 == 0 ? 0 : pick(0, P0 < 4 ? P0 : 4);
        wm.M = M0;
        wm.wx = M0 ? wxs[pick(0, 2)] : 0;
        for (auto& s : slots) {
            s.P = ragged ? pick(0, 400) : P0;
            s.PR = ragged ? pick(s.P == 0 ? 1 : 0, 4) : PR0;
            s.M = M0;
            const long long w = slot_weight(wm, s.P, s.M, s.PR);
            if (ws_min < 0 || w < ws_min) ws_min = w;
        }
        long long wt0 = 0;
        for (auto& s : slots) wt0 += slot_weight(wm, s.P, s.M, s.PR);
        const int num_sms = (int)pick(1, 152);
        wm.S0 = segment_lead(wm.wq, ws_min, wt0, num_sms);
        for (auto& s : slots) {
            s.w0 = start;
            s.Ws = wm.S0 + slot_weight(wm, s.P, s.M, s.PR);
            start += s.Ws;
            if (s.Ws > ws_max) ws_max = s.Ws;
        }
        wm.Wt = start;
        wm.Ws = ws_max;
        wm.P = slots[0].P;
        wm.PR = slots[0].PR;
        const long long resident = (long long)num_sms * pick(1, 4);
        wm.n = grid_size(wm.Wt, wm.wq < wm.wr ? wm.wq : wm.wr, wm.Wt / ws_max, resident,
                         trial % 5 == 0 ? pick(1, 64) : 0);
        if (!check(slots, wm, trial)) return 1;
        if (!ragged) {
            // the dense helpers agree with the walk
            for (long long s = 0; s < nslots; ++s) {
                if (slot_first_worker(wm, s) != map_owner(wm, slots[(size_t)s].w0 + wm.S0)) { std::printf("first worker\n"); return 1; }
                const long long last = slots[(size_t)s].w0 + unit_start(wm, wm.P + wm.PR - 1);
                if (slot_parts(wm, s) != (int)(map_owner(wm, last) - slot_first_worker(wm, s) + 1)) { std::printf("parts\n"); return 1; }
            }
        }
    }
    std::printf("ok\n");
    return 0;
}
