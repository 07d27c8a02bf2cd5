// tq_tc.cu -- host side of the tensor-core GEMV / FFN kernel
// (tq_tc_kernel.cuh): applicability, shared-memory plan, tensor maps and the
// launch; plus the kernel that lays plain int8 rows out as the MMA's B
// operand (the input of a phase-B-only launch).
#include <algorithm>
#include <atomic>
#include <mutex>

#include "tq.h"
#include "tq_launch.h"
#include "tq_tc.h"
#include "tq_tc_kernel.cuh"
#include "tq_tmap.h"

namespace tq {

namespace {

constexpr int kMaxDev = 64;

struct DevLimits {
    int sms = 0;
    int smem_optin = 0;
};

cudaError_t dev_limits(DevLimits *out) {
    static std::atomic<int> c_sms[kMaxDev] = {};
    static std::atomic<int> c_smem[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDev && c_sms[dev].load() > 0) {
        out->sms = c_sms[dev].load();
        out->smem_optin = c_smem[dev].load();
        return cudaSuccess;
    }
    if ((e = cudaDeviceGetAttribute(&out->sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&out->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    if (dev < kMaxDev) {
        c_smem[dev].store(out->smem_optin);
        c_sms[dev].store(out->sms);
    }
    return cudaSuccess;
}

int cdiv(int a, int b) { return (a + b - 1) / b; }
size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int pass_m(int m) { return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : 8; }

struct TcPlan {
    int grid, ring, sc_slots, b_slots;
    uint32_t off_sc, off_ba, off_bap, off_bb, off_bbp, off_fold;
    size_t bytes;
};

// Shared memory: as many 16 KB code planes as fit after the fixed regions
// (at least 4); 4 scales slots; 2 operand slots for phase B.
bool tc_plan(const TcCall &c, const DevLimits &d, TcPlan *p) {
    const int M = pass_m(c.m);
    const int bblk = M <= 4 ? 1024 : 2048;
    const int nbA = c.do_a ? c.wa[0].k / kBlock : 0;
    const int ua = c.do_a ? 2 * cdiv(c.wa[0].n, tc::kTile) * cdiv(nbA, tc::kSeg) : 0;
    const int nbB = c.do_b ? c.wb.k / kBlock : 0;
    const int ub = c.do_b ? cdiv(c.wb.n, tc::kTile) * cdiv(nbB, tc::kSeg) : 0;
    const int total = ua + ub;
    if (total == 0) return false;
    p->grid = (c.do_a && c.do_b) ? d.sms : std::max(1, std::min(d.sms, total));
    // fold jobs per CTA are bounded by its units (+ the closing job)
    if (cdiv(total, p->grid) + 1 > tc::kQueue) return false;
    p->sc_slots = 4;
    p->b_slots = c.do_b ? 2 : 1;
    constexpr size_t A = 1024;
    size_t off = 0;
    // ring first (1024-aligned planes), sized last
    size_t fixed = 0;
    fixed += up(static_cast<size_t>(p->sc_slots) * tc::kScBytes, A);
    fixed += up(static_cast<size_t>(nbA) * bblk + 256, A);                  // + the MMA's over-read of N = 16
    fixed += up(static_cast<size_t>(std::max(nbA, 1)) * M * 8, A);
    fixed += up(static_cast<size_t>(p->b_slots) * tc::kSeg * bblk + 256, A);
    fixed += up(static_cast<size_t>(p->b_slots) * tc::kSeg * M * 8, 128);
    fixed += up(static_cast<size_t>(M) * tc::kTile * 4 + bblk, 128);
    const size_t budget = static_cast<size_t>(d.smem_optin) - 3072 /* static shared memory */ - 1024 /* alignment */;
    if (fixed + 4 * static_cast<size_t>(tc::kPlane) > budget) return false;
    p->ring = static_cast<int>(std::min<size_t>(tc::kMaxRing, (budget - fixed) / tc::kPlane));
    off = static_cast<size_t>(p->ring) * tc::kPlane;
    p->off_sc = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(p->sc_slots) * tc::kScBytes, A);
    p->off_ba = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(nbA) * bblk + 256, A);
    p->off_bap = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(std::max(nbA, 1)) * M * 8, A);
    p->off_bb = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(p->b_slots) * tc::kSeg * bblk + 256, A);
    p->off_bbp = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(p->b_slots) * tc::kSeg * M * 8, 128);
    p->off_fold = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(M) * tc::kTile * 4 + bblk, 128);
    p->bytes = off + 1024;
    return p->bytes <= static_cast<size_t>(d.smem_optin) - 3072;
}

cudaError_t make_mat(tc::TcMat *md, const WeightRef &w, int fmt) {
    md->scales = w.scales;
    md->n = w.n;
    md->k = w.k;
    md->nb = w.k / kBlock;
    md->nseg = cdiv(md->nb, tc::kSeg);
    md->ntiles = cdiv(w.n, tc::kTile);
    const uint64_t row_bytes = static_cast<uint64_t>(w.k) / (fmt == TQ_FMT_TERNARY2 ? 4 : 8);
    cudaError_t e = make_tmap_2d(&md->tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, row_bytes,
                                 static_cast<uint64_t>(w.n), row_bytes, 128, tc::kTile, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    md->scales_tma = (md->nb % tc::kSeg == 0) && (reinterpret_cast<uintptr_t>(w.scales) % 16 == 0);
    if (md->scales_tma)
        e = make_tmap_2d(&md->tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, w.scales, static_cast<uint64_t>(md->nb),
                         static_cast<uint64_t>(w.n), static_cast<uint64_t>(md->nb) * 2, tc::kSeg, tc::kTile,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    return e;
}

template <int FMT, int M>
cudaError_t launch_tc_t(const tc::TcArgs &a, int grid, size_t bytes, bool coop, cudaStream_t stream) {
    auto kernel = tc::tc_kernel<FMT, M>;
    // the attribute is raised once per device to the largest size any launch
    // can ask for, under a lock, so concurrent first calls cannot lower it
    static std::mutex mu;
    static bool configured[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= kMaxDev || !configured[dev]) {
            int optin = 0;
            if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
                return e;
            if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 3072)) !=
                cudaSuccess)
                return e;
            if (dev < kMaxDev) configured[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(tc::kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (coop) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess && coop) {
        (void)cudaGetLastError();
        cfg.attrs = attr + 1;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, a);
    }
    return e;
}

// ---------------------------------------------------------------------------
// Plain int8 rows q [m][k] (+ fp32 s [m][k/128]) -> B operand blocks of
// bblk bytes (hi / lo e4m3 rows in staged order; rows m.. zero) and
// (scale, sum q) pairs [blocks][M].  One warp per block; blocks up to a whole
// number of segments (the padding blocks are zero).
// ---------------------------------------------------------------------------
template <int FMT, int M>
__global__ void tc_operand_kernel(const int8_t *__restrict__ q, const float *__restrict__ s, int m, int k, int nblocks,
                                  uint8_t *__restrict__ bst, float2 *__restrict__ bsn) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (b >= nblocks) return;
    pdl_wait();
    const int nb = k / kBlock;
    constexpr int kRowsInBlock = tc::kBBlk<M> / 256;      // activation rows the block holds (hi + lo each)
    uint8_t *blk = bst + static_cast<size_t>(b) * tc::kBBlk<M>;
    for (int r = 0; r < kRowsInBlock; ++r) {
        int qq[4] = {0, 0, 0, 0};
        float sc = 0.0f;
        if (r < m && b < nb) {
            const signed char *src = reinterpret_cast<const signed char *>(q) + static_cast<size_t>(r) * k + b * kBlock;
#pragma unroll
            for (int c = 0; c < 4; ++c) qq[c] = src[staged_elem<FMT>(4 * lane + c)];
            sc = s[static_cast<size_t>(r) * nb + b];
        }
        const int sum = __reduce_add_sync(0xffffffffu, qq[0] + qq[1] + qq[2] + qq[3]);
        uint32_t whi, wlo;
        tc::hilo_words(qq, whi, wlo);
        *reinterpret_cast<uint32_t *>(blk + tc::b_off<M>(2 * r, 4 * lane)) = whi;
        *reinterpret_cast<uint32_t *>(blk + tc::b_off<M>(2 * r + 1, 4 * lane)) = wlo;
        if (lane == 0 && r < M) bsn[static_cast<size_t>(b) * M + r] = make_float2(sc, static_cast<float>(sum));
    }
}

template <int FMT, int M>
cudaError_t launch_operand_t(const int8_t *q, const float *s, int m, int k, uint8_t *bst, float2 *bsn,
                             cudaStream_t stream) {
    const int nblocks = cdiv(k / kBlock, tc::kSeg) * tc::kSeg;
    return launch_pdl(tc_operand_kernel<FMT, M>, dim3(cdiv(nblocks, 8)), dim3(256), 0, stream, q, s, m, k, nblocks, bst, bsn);
}

}  // namespace

size_t tc_operand_bytes(int k) {
    return static_cast<size_t>(cdiv(k / kBlock, tc::kSeg) * tc::kSeg) * 2048;
}

size_t tc_pairs_bytes(int k) {
    return static_cast<size_t>(cdiv(k / kBlock, tc::kSeg) * tc::kSeg) * 8 * 8;
}

size_t tc_partials_bytes(int n, int k) {
    return static_cast<size_t>(cdiv(n, tc::kTile)) * cdiv(k / kBlock, tc::kSeg) * 8 * tc::kTile * 4;
}

int tc_tiles(int n) { return cdiv(n, tc::kTile); }

bool tc_applicable(const TcCall &c, cudaError_t *err) {
    *err = cudaSuccess;
    if (c.m < 1 || c.m > 8) return false;
    if (c.do_a && cdiv(c.wa[0].k / kBlock, tc::kSeg) > tc::kMaxSegs) return false;
    if (c.do_b && cdiv(c.wb.k / kBlock, tc::kSeg) > tc::kMaxSegs) return false;
    if (c.do_a && c.rotate_h && c.wa[0].n % kBlock != 0) return false;
    DevLimits d;
    if ((*err = dev_limits(&d)) != cudaSuccess) return false;
    TcPlan p;
    return tc_plan(c, d, &p);
}

cudaError_t tc_stage_operand(int fmt, int m, const int8_t *q, const float *s, int k, uint8_t *bst, float2 *bsn,
                             cudaStream_t stream) {
    const int M = pass_m(m);
    if (fmt == TQ_FMT_TERNARY2) {
        switch (M) {
            case 1: return launch_operand_t<0, 1>(q, s, m, k, bst, bsn, stream);
            case 2: return launch_operand_t<0, 2>(q, s, m, k, bst, bsn, stream);
            case 4: return launch_operand_t<0, 4>(q, s, m, k, bst, bsn, stream);
            default: return launch_operand_t<0, 8>(q, s, m, k, bst, bsn, stream);
        }
    }
    switch (M) {
        case 1: return launch_operand_t<1, 1>(q, s, m, k, bst, bsn, stream);
        case 2: return launch_operand_t<1, 2>(q, s, m, k, bst, bsn, stream);
        case 4: return launch_operand_t<1, 4>(q, s, m, k, bst, bsn, stream);
        default: return launch_operand_t<1, 8>(q, s, m, k, bst, bsn, stream);
    }
}

cudaError_t tc_launch(const TcCall &c, cudaStream_t stream) {
    DevLimits d;
    cudaError_t e = dev_limits(&d);
    if (e != cudaSuccess) return e;
    TcPlan p;
    if (!tc_plan(c, d, &p)) return cudaErrorInvalidConfiguration;
    tc::TcArgs a{};
    if (c.do_a) {
        if ((e = make_mat(&a.mat[0], c.wa[0], c.fmt)) != cudaSuccess) return e;
        if ((e = make_mat(&a.mat[1], c.wa[1], c.fmt)) != cudaSuccess) return e;
    }
    if (c.do_b && (e = make_mat(&a.mat[2], c.wb, c.fmt)) != cudaSuccess) return e;
    a.do_a = c.do_a;
    a.do_b = c.do_b;
    a.m = c.m;
    a.ua = c.do_a ? 2 * a.mat[0].ntiles * a.mat[0].nseg : 0;
    a.ub = c.do_b ? a.mat[2].ntiles * a.mat[2].nseg : 0;
    a.ring = p.ring;
    a.sc_slots = p.sc_slots;
    a.b_slots = p.b_slots;
    a.off_sc = p.off_sc;
    a.off_ba = p.off_ba;
    a.off_bap = p.off_bap;
    a.off_bb = p.off_bb;
    a.off_bbp = p.off_bbp;
    a.off_fold = p.off_fold;
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
    a.bst = c.bst;
    a.bsn = c.bsn;
    a.y = c.y;
    a.dots = c.dots;
    a.part_a = c.part_a;
    a.part_b = c.part_b;
    a.cnt_a = c.cnt_a;
    a.cnt_b = c.cnt_b;
    a.segready = c.segready;
    a.ticket = c.ticket;
    a.err = c.err;
    const bool coop = c.do_a && c.do_b;
    const int M = pass_m(c.m);
    if (c.fmt == TQ_FMT_TERNARY2) {
        switch (M) {
            case 1: return launch_tc_t<0, 1>(a, p.grid, p.bytes, coop, stream);
            case 2: return launch_tc_t<0, 2>(a, p.grid, p.bytes, coop, stream);
            case 4: return launch_tc_t<0, 4>(a, p.grid, p.bytes, coop, stream);
            default: return launch_tc_t<0, 8>(a, p.grid, p.bytes, coop, stream);
        }
    }
    switch (M) {
        case 1: return launch_tc_t<1, 1>(a, p.grid, p.bytes, coop, stream);
        case 2: return launch_tc_t<1, 2>(a, p.grid, p.bytes, coop, stream);
        case 4: return launch_tc_t<1, 4>(a, p.grid, p.bytes, coop, stream);
        default: return launch_tc_t<1, 8>(a, p.grid, p.bytes, coop, stream);
    }
}

}  // namespace tq
