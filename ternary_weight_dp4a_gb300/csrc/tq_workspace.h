// tq_workspace.h -- layout of the caller-owned workspaces of the FFN entry
// points and of tq_gemv (every section 256-byte aligned).
//
// FFN workspace (m rows, hidden, inter):
//   qx int8 [m][hidden] | sx f32 [m][hidden/128] | h bf16 [m][inter] |
//   qh int8 [m][inter]  | sh f32 [m][inter/128]  | counters u32 [inter/128] |
//   ybuf f32 [m][hidden] | err u32 (nonzero: a kernel's bounded wait ran out) |
//   sync: u64 launch ticket, then u32 [inter/1024] per 1024-wide segment of h,
//   its rotated 128-blocks (both count up over every step kernel launched on
//   the workspace) |
//   hst i8 [m*inter] | hsn (f32, i32) [m][inter/128] | hp f32 [m][inter]
//     (the dp4a kernel's staged copies of h: quantised again in the order its
//     down phase reads, with per-block (scale, magic - sum q), and h after the
//     transform's first four butterfly stages)
//   -- end of the dp4a kernel's part --
//   tc_hst: h as the tensor-core kernel's B operand, per pass of <= 8 rows 2 KB
//     per 128-block (whole segments) | tc_hsn: per pass (f32 scale, f32 sum q)
//     [blocks][8] |
//   part_a f32 [2][inter/128 tiles][hidden/1024 segments][8][128] |
//   part_b f32 [hidden/128 tiles][inter/1024 segments][8][128] (segment sums) |
//   cnt_a u32 [inter/128 tiles] | cnt_b u32 [hidden/16] (units counted per
//     tile, 128-row tiles of the tensor-core kernel or 16-row tiles of the
//     dp4a kernel's down projection alone, whose segment sums share part_b;
//     zero between launches) | ybuf2 f32 [m][hidden] (the stack's second
//     activation buffer: layers alternate between ybuf and ybuf2)
//
// GEMV workspace (m rows, n x k):
//   err u32 | cnt u32 [n/16] (units counted per tile: 128-row tiles of the
//   tensor-core kernel, 16-row tiles the dp4a kernel shares between CTAs) |
//   operand (2 KB per 128-block of k, whole segments) | pairs (f32 scale, f32
//   sum q) [blocks][8] | part f32 [n/128 tiles][k/1024 segments][8][128]
//   (segment sums; the dp4a kernel's [n/16][k/1024][m <= 4][16] fit in it)
#pragma once

#include <cstddef>
#include <cstdint>

namespace tq {

constexpr size_t kWsAlign = 256;

constexpr size_t ws_round(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }
constexpr int64_t ws_cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// tensor-core kernel scratch sizes (tq_tc.h restates them for the launch code)
constexpr size_t tc_ws_operand(int64_t k) { return static_cast<size_t>(ws_cdiv(k / 128, 8) * 8) * 2048; }
constexpr size_t tc_ws_pairs(int64_t k) { return static_cast<size_t>(ws_cdiv(k / 128, 8) * 8) * 8 * 8; }
constexpr size_t tc_ws_partials(int64_t n, int64_t k) {
    return static_cast<size_t>(ws_cdiv(n, 128) * ws_cdiv(k / 128, 8)) * 8 * 128 * 4;
}

struct FfnWorkspace {
    size_t qx, sx, h, qh, sh, counters, ybuf, err, sync, hst, hsn, hp, dp4a_total;
    size_t tc_hst, tc_hsn, part_a, part_b, cnt_a, cnt_b, ybuf2, total;
};

constexpr FfnWorkspace ffn_layout(int64_t m, int64_t hidden, int64_t inter) {
    FfnWorkspace w{};
    size_t off = 0;
    w.qx = off; off = ws_round(off + static_cast<size_t>(m * hidden));
    w.sx = off; off = ws_round(off + static_cast<size_t>(m * (hidden / 128)) * 4);
    w.h = off;  off = ws_round(off + static_cast<size_t>(m * inter) * 2);
    w.qh = off; off = ws_round(off + static_cast<size_t>(m * inter));
    w.sh = off; off = ws_round(off + static_cast<size_t>(m * (inter / 128)) * 4);
    w.counters = off; off = ws_round(off + static_cast<size_t>(inter / 128) * 4);
    w.ybuf = off; off = ws_round(off + static_cast<size_t>(m * hidden) * 4);
    w.err = off; off = ws_round(off + 4);
    w.sync = off; off = ws_round(off + static_cast<size_t>(2 + (inter + 1023) / 1024) * 4);
    w.hst = off; off = ws_round(off + static_cast<size_t>(m * inter));
    w.hsn = off; off = ws_round(off + static_cast<size_t>(m * (inter / 128)) * 8);
    w.hp = off;  off = ws_round(off + static_cast<size_t>(m * inter) * 4);
    w.dp4a_total = off;
    const int64_t passes = ws_cdiv(m, 8);
    w.tc_hst = off; off = ws_round(off + static_cast<size_t>(passes) * tc_ws_operand(inter));
    w.tc_hsn = off; off = ws_round(off + static_cast<size_t>(passes) * tc_ws_pairs(inter));
    w.part_a = off; off = ws_round(off + 2 * tc_ws_partials(inter, hidden));
    w.part_b = off; off = ws_round(off + tc_ws_partials(hidden, inter));
    w.cnt_a = off; off = ws_round(off + static_cast<size_t>(ws_cdiv(inter, 128)) * 4);
    w.cnt_b = off; off = ws_round(off + static_cast<size_t>(ws_cdiv(hidden, 16)) * 4);
    w.ybuf2 = off; off = ws_round(off + static_cast<size_t>(m * hidden) * 4);
    w.total = off;
    return w;
}

struct GemvWorkspace {
    size_t err, cnt, operand, pairs, part, total;
};

constexpr GemvWorkspace gemv_layout(int64_t n, int64_t k) {
    GemvWorkspace w{};
    size_t off = 0;
    w.err = off; off = ws_round(off + 4);
    w.cnt = off; off = ws_round(off + static_cast<size_t>(ws_cdiv(n, 16)) * 4);
    w.operand = off; off = ws_round(off + tc_ws_operand(k));
    w.pairs = off; off = ws_round(off + tc_ws_pairs(k));
    w.part = off; off = ws_round(off + tc_ws_partials(n, k));
    w.total = off;
    return w;
}

}  // namespace tq
