// tq_kernel.cu -- shared-memory plan, tensor maps and launch of the
// persistent GEMV / FFN kernel.
#include <algorithm>
#include <atomic>

#include "tq.h"
#include "tq_kernel.cuh"
#include "tq_kernel_launch.h"
#include "tq_kernel_run.cuh"
#include "tq_tmap.h"

namespace tq {

namespace {

constexpr int kPrologueSlots = 16;     // units in flight before the input is staged

struct DevInfo {
    int sms = 0;
    int smem_optin = 0;
};

cudaError_t dev_info(DevInfo *out) {
    static std::atomic<int> cached_sms[kMaxDev] = {};
    static std::atomic<int> cached_smem[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDev && cached_sms[dev].load() > 0) {
        out->sms = cached_sms[dev].load();
        out->smem_optin = cached_smem[dev].load();
        return cudaSuccess;
    }
    if ((e = cudaDeviceGetAttribute(&out->sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&out->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    if (dev < kMaxDev) {
        cached_smem[dev].store(out->smem_optin);
        cached_sms[dev].store(out->sms);
    }
    return cudaSuccess;
}

struct Plan {
    uint32_t off_scales, off_act, off_sn, off_acth, off_snh, off_part, off_tcnt, off_scr;
    size_t bytes;
    int slots, lanes, grid, tiles_max, nseg_max;
    Deal deal_a, deal_b;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// A phase-B-only launch splits tiles between CTAs (equal shares of the
// units) when the caller gave it the global segment sums and counts, their
// scratch stays small, and it pays: the whole-tile deal's busiest CTA has
// more than 1.15 x the average share, and a share spans at least two tiles
// and 24 units, so that the cross-CTA fold of the shared tiles hides behind
// other units (measured on GB300: a 5120 x 17408 GEMV, 2 or 3 tiles of 17
// units per CTA, 17.3 -> 15.9 us at m = 1; GEMVs of 512 to 5120 rows with k
// of 4096 or 5120, shares of 1 to 9 units, slower by 1.6 to 2.4 us).
bool split_b(const Call &c, int sms) {
    if (c.do_a || c.gcnt == nullptr || c.gpart == nullptr) return false;
    const int uptB = ceil_div(c.wb.k / kBlock, kSegBlocks);
    if (static_cast<size_t>(2) * uptB * c.m * kTileRows * 4 > 32768) return false;
    const long long tiles = ceil_div(c.wb.n, kTileRows);
    const long long G = std::min<long long>(sms, tiles);
    const double share = static_cast<double>(tiles) / static_cast<double>(sms);     // tiles per CTA when split
    const double busiest = static_cast<double>((tiles + G - 1) / G);
    return share >= 2.0 && share * uptB >= 24.0 && busiest > 1.15 * share;
}


// q or q + 1 tiles per CTA.
Deal uniform_deal(int ntiles, int G) {
    const int q = ntiles / G, r = ntiles % G;
    return Deal{{q + 1, q, q, q}, {r, G, G}};
}

// Phase A's deal for a launch running both phases, phase B dealt uniformly
// in reverse (the last ntB % G CTAs of phase A's order hold one more phase-B
// tile).  Per CTA load = uA * (phase-A tiles) + uB * (phase-B tiles) units;
// the deal takes the smallest bound L on every CTA's load that leaves room
// for all ntA tiles, and gives the tiles beyond ntA back from the end of each
// group, keeping the counts non-increasing in dealing order.
Deal balanced_deal_a(int ntA, int uA, int ntB, int uB, int G) {
    const int bq = ntB / G, rB = ntB % G;
    const int nL = G - rB, nH = rB;
    const long long total = static_cast<long long>(ntA) * uA + static_cast<long long>(ntB) * uB;
    for (long long L = (total + G - 1) / G;; ++L) {
        const long long A1 = std::max(0ll, (L - static_cast<long long>(bq) * uB) / uA);
        const long long A2 = nH > 0 ? std::max(0ll, (L - static_cast<long long>(bq + 1) * uB) / uA) : A1;
        const long long room = nL * A1 + nH * A2;
        if (room < ntA) continue;
        // each step of L adds at most G tiles of room, so the excess is below
        // G unless the first bound tried already had room to spare
        if (room - ntA >= G) return uniform_deal(ntA, G);
        const int E = static_cast<int>(room - ntA);
        const int a1 = static_cast<int>(A1), a2 = static_cast<int>(A2);
        if (a1 == a2) return Deal{{a1, a1 - 1, a1 - 1, a1 - 1}, {G - E, G, G}};
        const int e1 = std::min(E, nL), e2 = E - e1;
        if (e2 > 0 && a2 == 0) return uniform_deal(ntA, G);
        return Deal{{a1, a1 - 1, a2, a2 - 1}, {nL - e1, nL, G - e2}};
    }
}

// Shared-memory plan: ring slots as many as fit (at most kMaxSlots), after
// both phases' activations and (scale, magic - sum) pairs, the segment sums
// of the largest per-CTA share of units of each phase and the counters.
bool make_plan(const Call &c, const DevInfo &d, Plan *p) {
    const int nA = c.do_a ? c.wa[0].n : 0, kA = c.do_a ? c.wa[0].k : 0;
    const int nB = c.do_b ? c.wb.n : 0, kB = c.do_b ? c.wb.k : 0;
    const int tilesA = ceil_div(nA, kTileRows), tilesB = ceil_div(nB, kTileRows);
    // a launch running both phases needs every CTA resident (phase B waits on
    // blocks of h other CTAs rotate): one CTA per SM
    p->grid = (c.do_a && c.do_b) ? d.sms
              : split_b(c, d.sms) ? std::max(1, std::min(d.sms, tilesB * ceil_div(kB / kBlock, kSegBlocks)))
                           : std::max(1, std::min(d.sms, std::max(tilesA, tilesB)));
    const int G = p->grid;
    const int nbA = kA / kBlock, nbB = kB / kBlock;
    const int uptA = 2 * ceil_div(nbA, kSegBlocks), uptB = ceil_div(nbB, kSegBlocks);
    p->deal_b = uniform_deal(tilesB, G);
    p->deal_a = c.do_a && c.do_b ? balanced_deal_a(tilesA, uptA, tilesB, uptB, G) : uniform_deal(tilesA, G);
    const int tpcA = c.do_a ? p->deal_a.lv[0] : 0, tpcB = c.do_b ? p->deal_b.lv[0] : 0;
    p->tiles_max = std::max(1, std::max(tpcA, tpcB));
    p->nseg_max = std::max(1, uptB);
    // a phase-B-only launch with split tiles: an equal share of the units
    // spans at most ceil(share / upt) + 1 tiles; two of them may be shared
    // and folded from a scratch of all their segment sums
    size_t scr = 0;
    if (split_b(c, d.sms)) {
        const long long U = static_cast<long long>(tilesB) * uptB;
        const int share = static_cast<int>((U + G - 1) / G);
        p->tiles_max = std::max(p->tiles_max, ceil_div(share, uptB) + 1);
        scr = static_cast<size_t>(2) * uptB * c.m * kTileRows * 4;
    }
    const size_t actA = static_cast<size_t>(nbA) * kBlock * c.m, snA = static_cast<size_t>(nbA) * c.m * 8;
    const size_t actB = static_cast<size_t>(nbB) * kBlock * c.m, snB = static_cast<size_t>(nbB) * c.m * 8;
    const size_t part = static_cast<size_t>(tpcA * uptA + tpcB * uptB) * c.m * kTileRows * 4;
    const size_t ints = static_cast<size_t>(2 * p->tiles_max + p->nseg_max) * 4;
    // every region starts on a 128-byte boundary (the activations are read
    // and written 16 bytes at a time)
    constexpr size_t kAlign = 128;
    const size_t fixed = 1024 /* alignment slack */ + align_up(actA, kAlign) + align_up(snA, kAlign) + align_up(actB, kAlign) +
                         align_up(snB, kAlign) + align_up(part, kAlign) + align_up(ints, kAlign) + align_up(scr, kAlign);
    const size_t budget = static_cast<size_t>(d.smem_optin) - 2048;   // static shared memory < 1 KB
    if (fixed >= budget) return false;
    int slots = static_cast<int>(std::min<size_t>(kMaxSlots, (budget - fixed) / (kCodesSlot + kScalesSlot)));
    // one or two rows: 6 producer lanes where 12 slots or more fit
    const int lanes = c.m <= 2 && slots - slots % kProducerLanesMax >= 2 * kProducerLanesMax ? kProducerLanesMax : 4;
    slots -= slots % lanes;               // each slot filled by one producer lane
    if (slots < 2 * lanes) return false;
    p->slots = slots;
    p->lanes = lanes;
    size_t off = static_cast<size_t>(slots) * kCodesSlot;
    p->off_scales = static_cast<uint32_t>(off);
    off += static_cast<size_t>(slots) * kScalesSlot;
    p->off_act = static_cast<uint32_t>(off);
    off = align_up(off + actA, kAlign);
    p->off_sn = static_cast<uint32_t>(off);
    off = align_up(off + snA, kAlign);
    p->off_acth = static_cast<uint32_t>(off);
    off = align_up(off + actB, kAlign);
    p->off_snh = static_cast<uint32_t>(off);
    off = align_up(off + snB, kAlign);
    p->off_part = static_cast<uint32_t>(off);
    off = align_up(off + part, kAlign);
    p->off_tcnt = static_cast<uint32_t>(off);
    off = align_up(off + ints, kAlign);
    p->off_scr = static_cast<uint32_t>(off);
    off = align_up(off + scr, kAlign);
    p->bytes = off + 1024;
    return true;
}

cudaError_t make_mat(MatDesc *md, const WeightRef &w, int fmt) {
    md->codes = w.codes;
    md->scales = w.scales;
    md->n = w.n;
    md->k = w.k;
    const uint64_t row_bytes = static_cast<uint64_t>(w.k) / (fmt == TQ_FMT_TERNARY2 ? 4 : 8);
    // 2-bit rows that are whole 128-byte planes take one 3D copy per unit
    md->codes3d = fmt == TQ_FMT_TERNARY2 && row_bytes % 128 == 0;
    cudaError_t e = md->codes3d
                        ? make_codes_tmap_3d(&md->tm_codes, w.codes, row_bytes, static_cast<uint64_t>(w.n))
                        : make_tmap_2d(&md->tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, row_bytes,
                                       static_cast<uint64_t>(w.n), row_bytes, 128, kTileRows,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int nb = w.k / kBlock;
    // the scales rows are 16-byte multiples only when nb % 8 == 0; otherwise
    // the consumers read them from global memory
    md->scales_tma = (nb % kSegBlocks == 0) && (reinterpret_cast<uintptr_t>(w.scales) % 16 == 0);
    if (md->scales_tma)
        e = make_tmap_2d(&md->tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, w.scales, static_cast<uint64_t>(nb),
                         static_cast<uint64_t>(w.n), static_cast<uint64_t>(nb) * 2, kSegBlocks, kTileRows,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    return e;
}

}  // namespace

bool call_fits(const Call &c, cudaError_t *err) {
    DevInfo d;
    *err = dev_info(&d);
    if (*err != cudaSuccess) return false;
    Plan p;
    return make_plan(c, d, &p);
}

cudaError_t launch_call(const Call &c, cudaStream_t stream) {
    DevInfo d;
    cudaError_t e = dev_info(&d);
    if (e != cudaSuccess) return e;
    Plan p;
    if (!make_plan(c, d, &p)) return cudaErrorInvalidConfiguration;
    KArgs a{};
    if (c.do_a) {
        if ((e = make_mat(&a.mat[0], c.wa[0], c.fmt)) != cudaSuccess) return e;
        if ((e = make_mat(&a.mat[1], c.wa[1], c.fmt)) != cudaSuccess) return e;
    }
    if (c.do_b && (e = make_mat(&a.mat[2], c.wb, c.fmt)) != cudaSuccess) return e;
    a.do_a = c.do_a;
    a.do_b = c.do_b;
    a.deal_a = p.deal_a;
    a.deal_b = p.deal_b;
    a.slots = p.slots;
    a.lanes = p.lanes;
    // a phase-B-only launch of one or two rows over a long input (64 blocks
    // or more) stages the input by segments on demand: measured 15.5 -> 14.2
    // us for the 5120 x 17408 GEMV; shorter inputs and more rows (one warp
    // then stages a segment of up to 4 rows alone) measured slower
    a.lazy_b = !c.do_a && c.do_b && c.m <= 2 && c.wb.k / kBlock >= 64;
    a.prologue_slots = std::min(p.slots, kPrologueSlots);
    a.off_scales = p.off_scales;
    a.off_act = p.off_act;
    a.off_sn = p.off_sn;
    a.off_acth = p.off_acth;
    a.off_snh = p.off_snh;
    a.off_part = p.off_part;
    a.off_tcnt = p.off_tcnt;
    a.off_scr = p.off_scr;
    if (split_b(c, d.sms)) {
        a.gpart = c.gpart;
        a.gcnt = c.gcnt;
    }
    a.tiles_max = p.tiles_max;
    a.nseg_max = p.nseg_max;
    a.in_mode = c.in_mode;
    a.x = c.x;
    a.y_in = c.y_in;
    a.eps = c.eps;
    a.qa = c.qa;
    a.sa = c.sa;
    a.qx = c.qx;
    a.sx = c.sx;
    a.h = c.h;
    a.rotate_h = c.rotate_h;
    a.qh = c.qh;
    a.sh = c.sh;
    a.hst = c.hst;
    a.hsn = c.hsn;
    a.hp = c.hp;
    a.hcount = c.hcount;
    a.bst = c.bst;
    a.bsn = c.bsn;
    a.qb = c.qb;
    a.sb = c.sb;
    a.y = c.y;
    a.dots = c.dots;
    a.segready = c.segready;
    a.ticket = c.ticket;
    a.err = c.err;
    if (!c.do_a) return launch_b_only(a, c.fmt, c.m, p.grid, p.bytes, stream);
    const bool coop = c.do_b;     // phase B waits on other CTAs' rotations
    if (c.fmt == TQ_FMT_TERNARY2) {
        switch (c.m) {
            case 1: return launch_t<0, 1, false>(a, p.grid, p.bytes, coop, stream);
            case 2: return launch_t<0, 2, false>(a, p.grid, p.bytes, coop, stream);
            case 3: return launch_t<0, 3, false>(a, p.grid, p.bytes, coop, stream);
            default: return launch_t<0, 4, false>(a, p.grid, p.bytes, coop, stream);
        }
    }
    switch (c.m) {
        case 1: return launch_t<1, 1, false>(a, p.grid, p.bytes, coop, stream);
        case 2: return launch_t<1, 2, false>(a, p.grid, p.bytes, coop, stream);
        case 3: return launch_t<1, 3, false>(a, p.grid, p.bytes, coop, stream);
        default: return launch_t<1, 4, false>(a, p.grid, p.bytes, coop, stream);
    }
}

}  // namespace tq
