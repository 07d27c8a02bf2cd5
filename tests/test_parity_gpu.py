"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, on
both kernels (the tensor-core kernel and the dp4a kernel; every test runs
once per engine).

Bars (per the method's exactness): int8 codes, fp32 activation scales and int32
block dots bit-exact; fp32 outputs bit-exact against the oracle's documented
fold order (so their relative error against that oracle is 0); against the
fp64 definition, within 1e-4 of the summed magnitude of each output's block
terms, and the plain relative error with the floor max(|r|, 1e-3 rms(r))
reported and bounded (see REL_FLOOR_BOUND); every row of a packed step
bit-identical to its single-row run; repeated runs bit-identical.
"""
import numpy as np
import pytest

from _util import Mat, bf16_bits, bf16_tensor, ffn_mats, fold_rel_err, rel_err, ws_offsets
from ternary_weight_dp4a_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4
# The plain relative error against the fp64 definition, with the floor
# max(|r|, 1e-3 rms(r)), of ANY binary32 evaluation of the documented fold:
# outputs that cancel to within the floor keep the rounding error of the
# terms they cancelled (measured on the oracle's fp32 fold, which these
# kernels match bit for bit: at most 1.7e-4 on the 5120 x 17408 down GEMV and
# 1.4e-4 on the 17408 x 5120 gate GEMV, with 99.9 % of outputs below 4e-5).
REL_FLOOR_BOUND = 5e-4


@pytest.fixture(scope="module", params=[2, 1], ids=["tcgen05", "dp4a"])
def tq(request):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ternary_weight_dp4a_gb300 import build, tq as tqmod
    build.build()
    tqmod.load()
    before = tqmod.get_engine()
    tqmod.set_engine(request.param)
    yield tqmod
    tqmod.set_engine(before)


def _acts(m, k, outliers=0.01, seed=synth.SEED_ACT_BASE):
    return synth.activation(m, k, seed=seed, outlier_frac=outliers)


# ----------------------------------------------------------------------------
# packing and rotation
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n,k", [(512, 256), (77, 1152), (300, 5120)])
def test_pack_bit_exact(tq, orc, fmt, n, k):
    w = Mat(n, k, fmt, seed=5)
    assert np.array_equal(w.dev.codes.cpu().numpy(), w.orc_packed(orc))


@pytest.mark.parametrize("m,k,outliers", [(1, 256, 0.0), (8, 5120, 0.01), (3, 17408, 0.01),
                                          (5, 128, 0.0), (13, 384, 0.01)])
def test_rotate_quant_bit_exact(tq, orc, m, k, outliers):
    x = _acts(m, k, outliers)
    if m >= 3:
        x[1, :128] = 0                      # an all-zero block
        x[2, 128:256] = 0x4f00 if k >= 256 else x[2, 128:256]   # large bf16 values (2^31)
    q, s = tq.rotate_quant(bf16_tensor(x))
    q_ref, s_ref = orc.rotate_quant(x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


# ----------------------------------------------------------------------------
# GEMV
# ----------------------------------------------------------------------------

# the tiny config, ragged and multi-tile shapes, the FFN's K, and the
# full-attention projections of the model family the pages describe
# (head_dim 256, 8:1 GQA with 2 KV heads: q 4096 x 5120, k/v 512 x 5120,
# o 5120 x 4096), and the FFN's down projection alone (5120 x 17408: the
# dp4a kernel shares its 320 tiles between CTAs in equal shares of units)
GEMV_SHAPES = [(512, 256), (1000, 384), (77, 1152), (4101, 5120), (96, 17408),
               (4096, 5120), (512, 5120), (5120, 4096), (5120, 17408)]


# m = 1, 2 over an input of 64 blocks or more (k = 17408) stage it by segments
# on demand; the other cases stage it up front
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n,k", GEMV_SHAPES)
@pytest.mark.parametrize("m", [1, 2, 3, 8])
def test_gemv_bit_exact(tq, orc, fmt, n, k, m):
    import torch
    w = Mat(n, k, fmt, seed=synth.SEED_TINY_WEIGHT)
    x = _acts(m, k, 0.01)
    q_ref, s_ref = orc.rotate_quant(x)
    q = torch.from_numpy(q_ref).cuda()
    s = torch.from_numpy(s_ref).cuda()
    y, dots = tq.gemv(w.dev, q, s, blockdots=True)
    torch.cuda.synchronize()
    packed = w.orc_packed(orc)
    d_ref = orc.blockdots(packed, fmt, n, k, q_ref)
    assert np.array_equal(dots.cpu().numpy(), d_ref)
    y_ref = orc.gemv(packed, w.scales, fmt, n, k, q_ref, s_ref)
    yg = y.cpu().numpy()
    assert np.array_equal(yg.view(np.uint32), y_ref.view(np.uint32))
    y64 = orc.gemv_f64(packed, w.scales, fmt, n, k, q_ref, s_ref)
    assert fold_rel_err(yg, y64, orc, packed, w.scales, fmt, n, k, q_ref, s_ref) <= TOL
    assert rel_err(yg, y64) <= REL_FLOOR_BOUND


def test_gemv_error_word_is_zero_after_a_good_call(tq):
    import torch
    n, k, m = 4101, 5120, 3
    w = Mat(n, k, 0, seed=31)
    q, s = tq.rotate_quant(bf16_tensor(_acts(m, k, 0.01)))
    ws = tq.gemv_workspace(m, n, k)
    tq.gemv(w.dev, q, s, workspace=ws)
    assert tq.read_error_word(ws[:4]) == 0
    # and again on the same workspace (its tile counts return to zero)
    y1 = tq.gemv(w.dev, q, s, workspace=ws)
    y2 = tq.gemv(w.dev, q, s, workspace=ws)
    assert tq.read_error_word(ws[:4]) == 0
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("fmt", [0, 1])
def test_gemv_wide_shape_sampled_rows(tq, orc, fmt):
    """A wide GEMV at LM-head scale (N = 131072, K = 5120) in the launch the
    bench times: 64 sampled output rows against the oracle, which computes
    them from their own rows of the weights (rows are independent)."""
    import torch
    n, k, m = 131072, 5120, 2
    codes_d, scales_d = synth.weight(n, k, fmt, synth.SEED_TINY_WEIGHT + 17, device="cuda")
    wdev = tq.pack_weights(codes_d, fmt, scales_d)
    x = _acts(m, k, 0.01)
    q_ref, s_ref = orc.rotate_quant(x)
    q = torch.from_numpy(q_ref).cuda()
    s = torch.from_numpy(s_ref).cuda()
    y, dots = tq.gemv(wdev, q, s, blockdots=True)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(5).choice(n - 1, 63, replace=False))
    rows = np.append(rows, n - 1)                               # the last tile's last row
    ridx = torch.from_numpy(rows).cuda()
    sub_codes = codes_d[ridx].cpu().numpy()
    sub_scales = scales_d[ridx].cpu().numpy()
    packed = orc.pack(sub_codes, fmt)
    d_ref = orc.blockdots(packed, fmt, len(rows), k, q_ref)
    assert np.array_equal(dots.cpu().numpy()[:, rows, :], d_ref)
    y_ref = orc.gemv(packed, sub_scales, fmt, len(rows), k, q_ref, s_ref)
    assert np.array_equal(y.cpu().numpy()[:, rows].view(np.uint32), y_ref.view(np.uint32))


@pytest.mark.parametrize("fmt", [0, 1])
def test_gemv_tiny_config_edge_cases(tq, orc, fmt):
    """K=256, N=512 (the tiny GEMV), plus zero activations and zero weights."""
    import torch
    n, k = 512, 256
    w = Mat(n, k, fmt, seed=synth.SEED_TINY_WEIGHT)
    q = torch.zeros((2, k), dtype=torch.int8, device="cuda")
    s = torch.zeros((2, k // 128), dtype=torch.float32, device="cuda")
    assert torch.all(tq.gemv(w.dev, q, s) == 0)
    if fmt == 0:
        zero_codes = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
        scales = torch.from_numpy(w.scales).cuda()
        wz = tq.pack_weights(zero_codes, 0, scales)
        x = _acts(1, k, 0.0)
        qq, ss = tq.rotate_quant(bf16_tensor(x))
        assert torch.all(tq.gemv(wz, qq, ss) == 0)


@pytest.mark.parametrize("fmt", [0, 1])
def test_gemv_packed_rows_bit_identical_to_single(tq, fmt):
    import torch
    n, k = 2053, 5120
    w = Mat(n, k, fmt, seed=17)
    x = bf16_tensor(_acts(8, k, 0.01))
    q, s = tq.rotate_quant(x)
    singles = [tq.gemv(w.dev, q[r:r + 1].contiguous(), s[r:r + 1].contiguous()) for r in range(8)]
    for m in (2, 3, 4, 5, 6, 7, 8):
        y = tq.gemv(w.dev, q[:m].contiguous(), s[:m].contiguous())
        for r in range(m):
            assert torch.equal(y[r].view(torch.int32), singles[r][0].view(torch.int32)), (m, r)


@pytest.mark.parametrize("fmt", [0, 1])
def test_gemv_verify_blocks_up_to_64_rows(tq, orc, fmt):
    """9..64 rows (verify / prefill blocks) run as passes of at most 4 rows:
    every row bit-exact against the oracle and bit-identical to its
    single-row run, including ragged last passes (9, 33 rows)."""
    import torch
    n, k = 300, 1152
    w = Mat(n, k, fmt, seed=23)
    x = _acts(64, k, 0.01)
    q_ref, s_ref = orc.rotate_quant(x)
    q = torch.from_numpy(q_ref).cuda()
    s = torch.from_numpy(s_ref).cuda()
    singles = [tq.gemv(w.dev, q[r:r + 1].contiguous(), s[r:r + 1].contiguous()) for r in range(64)]
    y_ref = orc.gemv(w.orc_packed(orc), w.scales, fmt, n, k, q_ref, s_ref)
    for m in (9, 16, 33, 64):
        y = tq.gemv(w.dev, q[:m].contiguous(), s[:m].contiguous())
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref[:m].view(np.uint32)), m
        for r in range(m):
            assert torch.equal(y[r].view(torch.int32), singles[r][0].view(torch.int32)), (m, r)


# ----------------------------------------------------------------------------
# FFN step
# ----------------------------------------------------------------------------

def _ffn_gpu(tq, mats, x_bits):
    import torch
    g, u, d = mats
    m, hidden = x_bits.shape
    ws = tq.ffn_workspace(m, hidden, g.n)
    y = tq.ffn_step(g.dev, u.dev, d.dev, bf16_tensor(x_bits), workspace=ws)
    torch.cuda.synchronize()
    return y.cpu().numpy(), ws


def _ffn_orc(orc, mats, x_bits):
    g, u, d = mats
    return orc.ffn_step(g.orc_packed(orc), g.scales, u.orc_packed(orc), u.scales,
                        d.orc_packed(orc), d.scales, g.fmt, d.n, g.n, x_bits)


def _check_ffn(tq, orc, mats, x_bits):
    m, hidden = x_bits.shape
    inter = mats[0].n
    y, ws = _ffn_gpu(tq, mats, x_bits)
    ref = _ffn_orc(orc, mats, x_bits)
    # stage-wise first (diagnoses which stage differs), then the output
    o = ws_offsets(m, hidden, inter)
    wsn = ws.cpu().numpy()
    assert np.array_equal(wsn[o["qx"]:o["qx"] + m * hidden].view(np.int8).reshape(m, hidden),
                          ref["qx"])
    h = wsn[o["h"]:o["h"] + 2 * m * inter].view(np.uint16).reshape(m, inter)
    assert np.array_equal(h, ref["h"])
    assert np.array_equal(wsn[o["qh"]:o["qh"] + m * inter].view(np.int8).reshape(m, inter),
                          ref["qh"])
    assert np.array_equal(y.view(np.uint32), ref["y"].view(np.uint32))
    d = mats[2]
    y64 = orc.gemv_f64(d.orc_packed(orc), d.scales, d.fmt, d.n, d.k, ref["qh"], ref["sh"])
    assert fold_rel_err(y, y64, orc, d.orc_packed(orc), d.scales, d.fmt, d.n, d.k,
                        ref["qh"], ref["sh"]) <= TOL
    assert rel_err(y, y64) <= REL_FLOOR_BOUND
    assert tq.ffn_workspace_error(ws, m, hidden, inter) == 0
    return y


# a single tile, a ragged segment count (k = 384, 1152), several tiles and
# segments; m = 5 and 8 are one pass on the tensor-core kernel and two on the
# dp4a kernel
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("hidden,inter", [(256, 512), (384, 1152), (1024, 2816), (2048, 4096)])
@pytest.mark.parametrize("m", [1, 2, 5, 8])
def test_ffn_step_bit_exact(tq, orc, fmt, hidden, inter, m):
    mats = ffn_mats(hidden, inter, fmt)
    _check_ffn(tq, orc, mats, _acts(m, hidden, 0.01))


@pytest.mark.parametrize("m", [9, 33, 64])
def test_ffn_step_verify_blocks(tq, orc, m):
    """An FFN step of 9..64 rows (passes of at most 4 rows on one workspace),
    bit-exact against the oracle row by row."""
    mats = ffn_mats(256, 1024, 0)
    _check_ffn(tq, orc, mats, _acts(m, 256, 0.01))


@pytest.mark.parametrize("fmt", [0, 1])
def test_ffn_full_size_layer_and_packed_rows(tq, orc, fmt):
    """One full FFN layer (hidden 5120, intermediate 17408): m = 1 and the
    packed m = 8 step against the oracle, and each packed row against its
    single-row GPU run."""
    import torch
    hidden, inter = 5120, 17408
    mats = ffn_mats(hidden, inter, fmt)
    x8 = _acts(8, hidden, 0.01)
    y1 = _check_ffn(tq, orc, mats, x8[:1])
    y8 = _check_ffn(tq, orc, mats, x8)
    assert np.array_equal(y8[0].view(np.uint32), y1[0].view(np.uint32))
    for m in (2, 4):
        ym, _ = _ffn_gpu(tq, mats, x8[:m])
        assert np.array_equal(ym.view(np.uint32), y8[:m].view(np.uint32))
    for r in range(1, 8):
        yr, _ = _ffn_gpu(tq, mats, x8[r:r + 1])
        assert np.array_equal(yr[0].view(np.uint32), y8[r].view(np.uint32)), r


def test_ffn_workspace_counters_return_to_zero_and_stages_match_step(tq, orc):
    """The per-block completion counters are zero after every step, the launch
    ticket and the segment ready counters count exactly one launch, and the
    three stage calls compute exactly the one-launch step."""
    import torch
    hidden, inter, m = 1024, 3072, 2
    mats = ffn_mats(hidden, inter, 0)
    x = _acts(m, hidden, 0.01)
    y_step, ws = _ffn_gpu(tq, mats, x)
    o = ws_offsets(m, hidden, inter)
    wsn = ws.cpu().numpy()
    cnt = wsn[o["counters"]:o["counters"] + 4 * (inter // 128)].view(np.uint32)
    assert np.all(cnt == 0)
    # the tensor-core kernel's per-tile unit counts are zero again too
    for name, tiles in (("cnt_a", inter // 128), ("cnt_b", hidden // 128)):
        assert np.all(wsn[o[name]:o[name] + 4 * tiles].view(np.uint32) == 0), name
    assert wsn[o["err"]:o["err"] + 4].view(np.uint32)[0] == 0     # no wait ran out
    # one launch: one ticket per CTA (one CTA per SM), and every segment's
    # ready counter counted each of its 128-blocks once
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert int(wsn[o["sync"]:o["sync"] + 8].view(np.uint64)[0]) == sms
    nseg = (inter + 1023) // 1024
    seg = wsn[o["sync"] + 8:o["sync"] + 8 + 4 * nseg].view(np.uint32)
    assert list(seg) == [min(8, inter // 128 - 8 * j) for j in range(nseg)]
    g, u, d = mats
    ws2 = tq.ffn_workspace(m, hidden, inter)
    y2 = torch.empty((m, hidden), dtype=torch.float32, device="cuda")
    for _ in range(2):
        tq.ffn_stage_input(bf16_tensor(x), inter, ws2)
        tq.ffn_stage_gateup(g.dev, u.dev, m, ws2)
        tq.ffn_stage_down(d.dev, m, y2, ws2)
    torch.cuda.synchronize()
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), y_step.view(np.uint32))


@pytest.mark.parametrize("m", [1, 2])
def test_ffn_stages_long_intermediate_match_step(tq, orc, m):
    """The down stage over a long staged h (intermediate 8192: 64 blocks,
    staged by segments on demand at one or two rows) computes exactly the
    one-launch step, and the step matches the oracle."""
    import torch
    hidden, inter = 1024, 8192
    mats = ffn_mats(hidden, inter, 0)
    x = _acts(m, hidden, 0.01)
    y_step, _ = _ffn_gpu(tq, mats, x)
    g, u, d = mats
    ws2 = tq.ffn_workspace(m, hidden, inter)
    y2 = torch.empty((m, hidden), dtype=torch.float32, device="cuda")
    tq.ffn_stage_input(bf16_tensor(x), inter, ws2)
    tq.ffn_stage_gateup(g.dev, u.dev, m, ws2)
    tq.ffn_stage_down(d.dev, m, y2, ws2)
    torch.cuda.synchronize()
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), y_step.view(np.uint32))
    ref = _ffn_orc(orc, mats, x)
    assert np.array_equal(y_step.view(np.uint32), ref["y"].view(np.uint32))


def test_ffn_gateup_standalone_matches_oracle(tq, orc):
    import torch
    hidden, inter, m = 1024, 2816, 2
    g, u, _ = ffn_mats(hidden, inter, 0)
    x = _acts(m, hidden, 0.01)
    qx, sx = orc.rotate_quant(x)
    h = tq.ffn_gateup(g.dev, u.dev, torch.from_numpy(qx).cuda(), torch.from_numpy(sx).cuda())
    gref = orc.gemv(g.orc_packed(orc), g.scales, 0, inter, hidden, qx, sx)
    uref = orc.gemv(u.orc_packed(orc), u.scales, 0, inter, hidden, qx, sx)
    assert np.array_equal(bf16_bits(h), orc.silu_mul_bf16(gref, uref))


def test_ffn_repeat_runs_bit_identical(tq):
    import torch
    mats = ffn_mats(1024, 2816, 0)
    x = _acts(4, 1024, 0.01)
    first, _ = _ffn_gpu(tq, mats, x)
    for _ in range(5):
        again, _ = _ffn_gpu(tq, mats, x)
        assert np.array_equal(again.view(np.uint32), first.view(np.uint32))


def test_ffn_wait_that_runs_out_sets_error_and_workspace_recovers(tq, orc):
    """Failure detection without a fault: the workspace's launch ticket is set
    1000 launches ahead, so the count the down phase waits for on every
    segment of h is one that no launch reaches.  Each such wait is bounded
    (about 0.5 s): the kernel finishes, the error word carries bit 6, the
    context stays usable, and after tq_ffn_workspace_init the same step is
    bit-exact against the oracle again."""
    import torch
    hidden, inter, m = 256, 2048, 1
    mats = ffn_mats(hidden, inter, 0)
    g, u, d = mats
    x = _acts(m, hidden, 0.01)
    ws = tq.ffn_workspace(m, hidden, inter)
    o = ws_offsets(m, hidden, inter)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ticket = np.array([1000 * sms], dtype=np.uint64).view(np.uint8)
    ws[o["sync"]:o["sync"] + 8].copy_(torch.from_numpy(ticket).cuda())
    tq.ffn_step(g.dev, u.dev, d.dev, bf16_tensor(x), workspace=ws)
    torch.cuda.synchronize()
    err = tq.ffn_workspace_error(ws, m, hidden, inter)
    assert err & 64, hex(err)
    # the boundary reports it as TQ_ERR_TIMEOUT
    off = tq.load().tq_ffn_workspace_error_offset(m, hidden, inter)
    with pytest.raises(tq.TQError) as ei:
        tq.read_error_word(ws[off:off + 4])
    assert ei.value.status == tq.TQ_ERR_TIMEOUT
    tq.ffn_workspace_init(ws)
    y = tq.ffn_step(g.dev, u.dev, d.dev, bf16_tensor(x), workspace=ws)
    torch.cuda.synchronize()
    assert tq.ffn_workspace_error(ws, m, hidden, inter) == 0
    assert tq.read_error_word(ws[off:off + 4]) == 0
    ref = _ffn_orc(orc, mats, x)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), ref["y"].view(np.uint32))


def test_ffn_zero_activation(tq):
    import torch
    mats = ffn_mats(256, 512, 0)
    y, _ = _ffn_gpu(tq, mats, np.zeros((2, 256), np.uint16))
    assert np.all(y == 0)


# ----------------------------------------------------------------------------
# RMS-normalise and the layer stack
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("m,n", [(1, 5120), (8, 5120), (3, 300)])
def test_rmsnorm_bit_exact(tq, orc, m, n):
    import torch
    rng = np.random.default_rng(3)
    y = (rng.standard_normal((m, n)) * 7).astype(np.float32)
    x = tq.rmsnorm_bf16(torch.from_numpy(y).cuda(), 1e-6)
    assert np.array_equal(bf16_bits(x), orc.rmsnorm_bf16(y, 1e-6))


@pytest.mark.parametrize("fmt", [0, 1])
def test_stack_full_width(tq, orc, fmt):
    """Three stacked full-width layers, rmsnorm between them, m = 1 and 2."""
    import torch
    hidden, inter, L = 5120, 17408, 3
    layers = [ffn_mats(hidden, inter, fmt, layer=l) for l in range(L)]
    x = _acts(2, hidden, 0.01)
    xt = bf16_tensor(x)
    for l, mats in enumerate(layers):
        g, u, d = mats
        y = tq.ffn_step(g.dev, u.dev, d.dev, xt)
        if l + 1 < L:
            xt = tq.rmsnorm_bf16(y, 1e-6)
    # the fused stack entry point (norm + rotation kernel between layers)
    ys = tq.ffn_stack([(g.dev, u.dev, d.dev) for g, u, d in layers], bf16_tensor(x), 1e-6)
    torch.cuda.synchronize()
    ref = orc.ffn_stack([(g.orc_packed(orc), g.scales, u.orc_packed(orc), u.scales,
                          d.orc_packed(orc), d.scales) for g, u, d in layers],
                        fmt, hidden, inter, x, 1e-6)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(ys.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # each packed row equals its single-row stack
    for r in range(2):
        yr = tq.ffn_stack([(g.dev, u.dev, d.dev) for g, u, d in layers],
                          bf16_tensor(x[r:r + 1]), 1e-6)
        assert torch.equal(yr[0].view(torch.int32), ys[r].view(torch.int32))
