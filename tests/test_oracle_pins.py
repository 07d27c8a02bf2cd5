"""Pins for the CPU oracle: closed forms, library routines, invariants, brute force
and hand-derived worked examples (tests/golden/*.txt).  No GPU.

Each pin is chosen so that a plausible mistake in the oracle (a wrong bit order,
a dropped normalisation, a wrong sign, a transposed operand, a changed reduction
order, a swapped gate/up) fails at least one of them.  The "mutant" tests check
that the pins really do reject such mistakes, by feeding deliberately wrong
results through the same comparisons.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg

from ternary_weight_dp4a_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
B = 128


def _golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = vals
    return rows


def _hadamard_normalised():
    return scipy.linalg.hadamard(B).astype(np.float64) / math.sqrt(B)


def _bf16_bits(x):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# scalar conversions
# ----------------------------------------------------------------------------

def test_f16_decode_matches_numpy_all_patterns(orc):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = orc.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_round_to_nearest_even_matches_torch(orc):
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(37.0),
        # exact ties and near-ties around bf16 boundaries
        (np.array([0x3f808000, 0x3f818000, 0x3f80ffff, 0x3f817fff, 0x00008000,
                   0x7f7fffff, 0x80018000], dtype=np.uint32)).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -3.3e38], dtype=np.float32)])
    ours = orc.f32_to_bf16(x)
    assert np.array_equal(ours, _bf16_bits(x))
    # and the decode is the top-16-bit embedding
    assert np.array_equal(orc.bf16_to_f32(ours).view(np.uint32),
                          ours.astype(np.uint32) << 16)


# ----------------------------------------------------------------------------
# layout
# ----------------------------------------------------------------------------

def test_layout_2bit_golden(orc):
    g = _golden("layout_2bit.txt")
    codes = np.array([[int(v) for v in g["codes"]]], dtype=np.uint8)
    packed = orc.pack(codes, orc.FMT_TERNARY2)
    assert [int(b) for b in packed[0]] == [int(v, 16) for v in g["bytes"]]
    assert orc.unpack(packed, 8, orc.FMT_TERNARY2)[0].tolist() == [int(v) for v in g["values"]]


def test_layout_1bit_golden(orc):
    g = _golden("layout_1bit.txt")
    bits = np.array([[int(v) for v in g["bits"]]], dtype=np.uint8)
    packed = orc.pack(bits, orc.FMT_BINARY1)
    assert [int(b) for b in packed[0]] == [int(v, 16) for v in g["bytes"]]
    assert orc.unpack(packed, 16, orc.FMT_BINARY1)[0].tolist() == [int(v) for v in g["values"]]


def _indep_pack2(codes):
    # the layout written out a second way: weights k = 4j+t -> bits 2t of byte j
    c = codes.astype(np.uint32).reshape(codes.shape[0], -1, 4)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def _indep_pack1(bits):
    return np.packbits(bits.astype(np.uint8), axis=1, bitorder="little")


@pytest.mark.parametrize("fmt", [0, 1])
def test_pack_roundtrip_random(orc, fmt):
    codes, _ = synth.weight(16, 512, fmt, seed=3)
    packed = orc.pack(codes, fmt)
    indep = _indep_pack2(codes) if fmt == 0 else _indep_pack1(codes)
    assert np.array_equal(packed, indep)
    vals = orc.unpack(packed, 512, fmt)
    if fmt == 0:
        expect = np.choose(codes, [0, 1, -1]).astype(np.int8)
    else:
        expect = (2 * codes.astype(np.int8) - 1)
    assert np.array_equal(vals, expect)
    # the distribution recipe: p(0)=0.4, p(+1)=p(-1)=0.3 (2-bit); 0.5/0.5 (1-bit)
    if fmt == 0:
        assert abs((vals == 0).mean() - 0.4) < 0.02
        assert abs((vals == 1).mean() - 0.3) < 0.02


def test_unused_code_3_reads_as_zero(orc):
    codes = np.full((1, 128), 3, dtype=np.uint8)
    packed = orc.pack(codes, 0)
    assert np.all(packed == 0xFF)
    assert np.all(orc.unpack(packed, 128, 0) == 0)


# ----------------------------------------------------------------------------
# Walsh-Hadamard rotation
# ----------------------------------------------------------------------------

def test_wht_unit_vectors_give_hadamard_rows(orc):
    H = _hadamard_normalised()              # scipy's Sylvester construction
    E = np.eye(B, dtype=np.float32)
    rows = orc.wht128(E)
    assert np.allclose(rows, H, atol=1e-7, rtol=0)
    # H H^T = I
    assert np.allclose(rows.astype(np.float64) @ rows.T.astype(np.float64), np.eye(B),
                       atol=1e-6)


def test_wht_matches_dense_fp64_and_is_involution(orc):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((6, B)) * np.array([[1], [10], [1e-3], [1], [100], [1]])
         ).astype(np.float32)
    y = orc.wht128(x)
    ref = x.astype(np.float64) @ _hadamard_normalised().T
    scale = np.abs(x).max(axis=1, keepdims=True).astype(np.float64)
    assert np.all(np.abs(y - ref) <= 2e-6 * scale * math.sqrt(B))
    # normalised H is symmetric and orthogonal: applying it twice gives x back
    z = orc.wht128(y)
    assert np.all(np.abs(z - x) <= 4e-6 * scale * math.sqrt(B))
    # norm preserved
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)


def test_wht_unnormalised_integer_inputs_exact(orc):
    # on small integers every butterfly is exact, so y*sqrt(128) is the exact
    # integer matrix product; check H(Hx) = x exactly through the normalisation
    rng = np.random.default_rng(2)
    x = rng.integers(-8, 9, size=(4, B)).astype(np.float32)
    y = orc.wht128(x).astype(np.float64)
    exact = x.astype(np.float64) @ scipy.linalg.hadamard(B).T.astype(np.float64)
    c = np.float64(np.float32(1.0 / math.sqrt(128.0)))
    # one rounding (the final multiply): |y - exact*c| <= ulp/2
    assert np.all(np.abs(y - exact * c) <= np.abs(exact * c) * 2.0 ** -24 + 1e-30)


# ----------------------------------------------------------------------------
# quantisation
# ----------------------------------------------------------------------------

def test_quant_golden_ties(orc):
    g = _golden("quant_ties.txt")
    v = np.zeros(B, np.float32)
    vals = np.array([float(t) for t in g["v"]], np.float32)
    v[:len(vals)] = vals
    q, s = orc.quant_block(v)
    assert s == np.float32(float(g["s"][0]))
    assert q[:len(vals)].tolist() == [int(t) for t in g["q"]]
    assert np.all(q[len(vals):] == 0)


def test_quant_bounds_and_zero_block(orc):
    rng = np.random.default_rng(7)
    for trial in range(200):
        v = (rng.standard_normal(B) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        if trial % 7 == 0:
            v[rng.integers(0, B)] *= 50
        q, s = orc.quant_block(v)
        amax = np.abs(v).max()
        assert s == np.float32(amax / np.float32(127.0))
        assert np.abs(q.astype(int)).max() == 127
        assert np.all(np.abs(q.astype(int)) <= 127)
        err = np.abs(v.astype(np.float64) - q.astype(np.float64) * np.float64(s))
        assert np.all(err <= np.float64(s) * 0.5 * (1 + 2.0 ** -20) + 1e-30)
    q, s = orc.quant_block(np.zeros(B, np.float32))
    assert s == 0.0 and np.all(q == 0)


def test_rotate_quant_dequantises_to_dense_rotation(orc):
    x = synth.activation(3, 512, seed=synth.SEED_ACT_BASE, outlier_frac=0.01)
    q, s = orc.rotate_quant(x)
    xf = _bf16_value(x).astype(np.float64).reshape(3, 4, B)
    rot = xf @ _hadamard_normalised().T                      # [3][4][128]
    deq = q.reshape(3, 4, B).astype(np.float64) * s[..., None].astype(np.float64)
    assert np.all(np.abs(deq - rot) <= 0.5 * s[..., None] * (1 + 1e-5) + 1e-6)


# ----------------------------------------------------------------------------
# GEMV
# ----------------------------------------------------------------------------

def _dense_values(codes, fmt):
    return np.choose(codes, [0, 1, -1]) if fmt == 0 else 2 * codes.astype(np.int64) - 1


@pytest.mark.parametrize("fmt", [0, 1])
def test_blockdots_brute_force(orc, fmt):
    n, k, m = 12, 384, 3
    codes, _ = synth.weight(n, k, fmt, seed=21)
    rng = np.random.default_rng(22)
    q = rng.integers(-127, 128, size=(m, k)).astype(np.int8)
    packed = orc.pack(codes, fmt)
    d = orc.blockdots(packed, fmt, n, k, q)
    W = _dense_values(codes, fmt).astype(np.int64)
    for r in range(m):
        for row in range(n):
            for b in range(k // B):
                sl = slice(b * B, (b + 1) * B)
                assert d[r, row, b] == int(np.dot(W[row, sl], q[r, sl].astype(np.int64)))


def test_gemv_identity_like_closed_form(orc):
    # K = N = 128, code 1 (+1) on the diagonal: y_i = (float)q_i * (sw * s) exactly
    codes = np.eye(B, dtype=np.uint8)
    packed = orc.pack(codes, 0)
    sw = np.full((B, 1), 0.03125, np.float16)
    rng = np.random.default_rng(1)
    q = rng.integers(-127, 128, size=(1, B)).astype(np.int8)
    s = np.array([[0.0123]], np.float32)
    y = orc.gemv(packed, sw, 0, B, B, q, s)
    ws = np.float32(np.float32(0.03125) * s[0, 0])
    assert np.array_equal(y[0], q[0].astype(np.float32) * ws)


def test_gemv_all_plus_one_and_zero_weights(orc):
    k = 1024
    plus = np.ones((4, k), np.uint8)
    zero = np.zeros((4, k), np.uint8)
    sw = np.full((4, k // B), 1.0, np.float16)
    rng = np.random.default_rng(4)
    q = rng.integers(-127, 128, size=(1, k)).astype(np.int8)
    s = np.ones((1, k // B), np.float32)
    y = orc.gemv(orc.pack(plus, 0), sw, 0, 4, k, q, s)
    assert np.all(y == np.float32(q.astype(np.int64).sum()))   # small ints: exact
    y0 = orc.gemv(orc.pack(zero, 0), sw, 0, 4, k, q, s)
    assert np.all(y0 == 0.0)
    # zero activation
    yz = orc.gemv(orc.pack(plus, 0), sw, 0, 4, k, np.zeros_like(q), np.zeros_like(s))
    assert np.all(yz == 0.0)


def test_gemv_fold_order_golden(orc):
    g = _golden("fold_order.txt")
    nb = int(g["blocks"][0])
    dots = [int(v) for v in g["dots"]]
    act_s = np.array([[float(v) for v in g["act_scales"]]], np.float32)
    k = nb * B
    codes = np.zeros((1, k), np.uint8)
    for b, d in enumerate(dots):
        codes[0, b * B: b * B + abs(d)] = 1 if d > 0 else 2
    q = np.ones((1, k), np.int8)
    sw = np.full((1, nb), 1.0, np.float16)
    packed = orc.pack(codes, 0)
    assert orc.blockdots(packed, 0, 1, k, q)[0, 0].tolist() == dots
    y = orc.gemv(packed, sw, 0, 1, k, q, act_s)
    assert y[0, 0] == np.float32(float(g["expected_fp32"][0]))
    y64 = orc.gemv_f64(packed, sw, 0, 1, k, q, act_s)
    assert y64[0, 0] == float(g["expected_f64"][0])


@pytest.mark.parametrize("fmt", [0, 1])
def test_gemv_matches_dense_fp64_einsum(orc, fmt):
    n, k, m = 64, 640, 2
    codes, sw = synth.weight(n, k, fmt, seed=31)
    x = synth.activation(m, k, seed=synth.SEED_ACT_BASE, outlier_frac=0.01)
    q, s = orc.rotate_quant(x)
    y = orc.gemv(orc.pack(codes, fmt), sw, fmt, n, k, q, s)
    W = _dense_values(codes, fmt).astype(np.float64).reshape(n, k // B, B)
    A = q.astype(np.float64).reshape(m, k // B, B)
    ref = np.einsum("nbk,mbk,nb,mb->mn", W, A, sw.astype(np.float64), s.astype(np.float64))
    # binary32 error bound of the fold: two roundings per block term and at most
    # nb + 3 roundings along any summation path, each <= 2^-24 relative
    dots = np.einsum("nbk,mbk->mnb", W, A)
    mag = np.einsum("mnb,nb,mb->mn", np.abs(dots), sw.astype(np.float64), s.astype(np.float64))
    nb = k // B
    assert np.all(np.abs(y - ref) <= (nb + 5) * 2.0 ** -24 * mag + 1e-30)
    y64 = orc.gemv_f64(orc.pack(codes, fmt), sw, fmt, n, k, q, s)
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


# ----------------------------------------------------------------------------
# exp / SiLU
# ----------------------------------------------------------------------------

def _ulp32(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, np.finfo(np.float32).tiny)))
    return 2.0 ** (e - 23)


def test_expf_within_two_ulp_of_fp64(orc):
    x = np.concatenate([np.linspace(-87.0, 88.5, 20001), np.linspace(-1, 1, 2001),
                        np.array([0.0, 1e-8, -1e-8, 0.5, -0.5])]).astype(np.float32)
    e = orc.expf(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    err = np.abs(e - ref) / _ulp32(ref)
    assert err.max() <= 2.0
    assert orc.expf(np.float32([0.0]))[0] == 1.0
    assert np.isinf(orc.expf(np.float32([89.0]))[0])
    assert orc.expf(np.float32([-110.0]))[0] == 0.0
    # subnormal results stay within 2 units of the subnormal spacing
    xs = np.linspace(-103.5, -88.0, 501).astype(np.float32)
    assert np.all(np.abs(orc.expf(xs).astype(np.float64) - np.exp(xs.astype(np.float64)))
                  <= 2.0 * 2.0 ** -149 + 2 * _ulp32(np.exp(xs.astype(np.float64))))


def test_silu_against_fp64(orc):
    g = np.concatenate([np.linspace(-40, 40, 8001),
                        np.array([0.0, 1e-20, -1e-20, 90.0, -90.0, -200.0])]).astype(np.float32)
    s = orc.silu(g).astype(np.float64)
    gd = g.astype(np.float64)
    ref = gd / (1.0 + np.exp(-gd))
    # below g = -88.7, exp(-g) overflows and the formula gives -0 where the exact
    # value is under 2^-120 in magnitude: compare those absolutely
    err = np.abs(s - ref) / np.maximum(_ulp32(ref), 2.0 ** -120)
    assert err.max() <= 4.0
    assert orc.silu(np.float32([0.0]))[0] == 0.0
    assert orc.silu(np.float32([90.0]))[0] == np.float32(90.0)


def test_silu_mul_bf16_against_fp64(orc):
    rng = np.random.default_rng(9)
    g = (rng.standard_normal(5000) * 3).astype(np.float32)
    u = (rng.standard_normal(5000) * 3).astype(np.float32)
    h = orc.silu_mul_bf16(g, u)
    gd, ud = g.astype(np.float64), u.astype(np.float64)
    ref = gd / (1 + np.exp(-gd)) * ud
    hv = _bf16_value(h).astype(np.float64)
    # within one bf16 ulp of the exact value (rounding + a few fp32 ulps)
    assert np.all(np.abs(hv - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    # swapping the operands is a different function (guards a gate/up swap)
    assert not np.array_equal(h, orc.silu_mul_bf16(u, g))


# ----------------------------------------------------------------------------
# RMS-normalise
# ----------------------------------------------------------------------------

def test_rmsnorm_against_fp64(orc):
    rng = np.random.default_rng(12)
    y = (rng.standard_normal((3, 5120)) * np.array([[1.0], [40.0], [1e-3]])).astype(np.float32)
    x = orc.rmsnorm_bf16(y, 1e-6)
    yd = y.astype(np.float64)
    ref = yd / np.sqrt((yd ** 2).mean(axis=1, keepdims=True) + 1e-6)
    xv = _bf16_value(x).astype(np.float64)
    assert np.all(np.abs(xv - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    # constant input: mean square is c^2 exactly, output bf16(c / sqrt(c^2+eps))
    c = np.full((1, 256), 2.0, np.float32)
    xc = _bf16_value(orc.rmsnorm_bf16(c, 0.0))
    assert np.all(xc == 1.0)


# ----------------------------------------------------------------------------
# FFN step: stage-wise against independent fp64 math
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [0, 1])
def test_ffn_step_stagewise(orc, fmt):
    hidden, inter, m = 256, 512, 2
    (gc, gs), (uc, us), (dc, ds) = (synth.weight(*shape, fmt, seed=synth.ffn_weight_seed(0, j))
                                    for j, shape in enumerate([(inter, hidden), (inter, hidden),
                                                               (hidden, inter)]))
    x = synth.activation(m, hidden, seed=synth.SEED_ACT_BASE, outlier_frac=0.01)
    out = orc.ffn_step(orc.pack(gc, fmt), gs, orc.pack(uc, fmt), us, orc.pack(dc, fmt), ds,
                       fmt, hidden, inter, x)
    Hn = _hadamard_normalised()

    def dense_ok(y, codes, sc, qq, ss, K):
        # fp64 dense product with the binary32 error bound of the fold
        W = _dense_values(codes, fmt).astype(np.float64).reshape(codes.shape[0], K // B, B)
        A = qq.astype(np.float64).reshape(qq.shape[0], K // B, B)
        dots = np.einsum("nbk,mbk->mnb", W, A)
        w = np.einsum("nb,mb->mnb", sc.astype(np.float64), ss.astype(np.float64))
        ref = (dots * w).sum(axis=2)
        mag = (np.abs(dots) * w).sum(axis=2)
        return np.all(np.abs(y - ref) <= (K // B + 5) * 2.0 ** -24 * mag + 1e-30)

    # rotation of x
    xr = _bf16_value(x).astype(np.float64).reshape(m, -1, B) @ Hn.T
    assert np.all(np.abs(out["qx"].reshape(m, -1, B) * out["sx"][..., None] - xr)
                  <= 0.5 * out["sx"][..., None] * (1 + 1e-5) + 1e-7)
    # gate and up use their own matrices
    assert dense_ok(out["g"], gc, gs, out["qx"], out["sx"], hidden)
    assert dense_ok(out["u"], uc, us, out["qx"], out["sx"], hidden)
    # h = bf16(silu(g) * u), not silu(u) * g
    g64, u64 = out["g"].astype(np.float64), out["u"].astype(np.float64)
    href = g64 / (1 + np.exp(-g64)) * u64
    assert np.all(np.abs(_bf16_value(out["h"]) - href) <= np.abs(href) * 2.0 ** -7 + 1e-30)
    # h is rotated and quantised like x
    hr = _bf16_value(out["h"]).astype(np.float64).reshape(m, -1, B) @ Hn.T
    assert np.all(np.abs(out["qh"].reshape(m, -1, B) * out["sh"][..., None] - hr)
                  <= 0.5 * out["sh"][..., None] * (1 + 1e-5) + 1e-7)
    # down
    assert dense_ok(out["y"], dc, ds, out["qh"], out["sh"], inter)


def test_ffn_identity_like_closed_form(orc):
    # hidden = inter = 128; gate, up, down all +1 on the diagonal with scales a, b, c.
    # g_i = q_i*(a*s), u_i = q_i*(b*s); y ~ H h within the quantisation error.
    n = B
    eye = np.eye(n, dtype=np.uint8)
    P = orc.pack(eye, 0)
    a, b_, c = (np.full((n, 1), v, np.float16) for v in (0.5, 0.25, 2.0))
    x = synth.activation(1, n, seed=synth.SEED_ACT_BASE)
    out = orc.ffn_step(P, a, P, b_, P, c, 0, n, n, x)
    s = out["sx"][0, 0]
    assert np.array_equal(out["g"][0], out["qx"][0].astype(np.float32) * np.float32(0.5 * s))
    assert np.array_equal(out["u"][0], out["qx"][0].astype(np.float32) * np.float32(0.25 * s))
    hv = _bf16_value(out["h"][0]).astype(np.float64)
    rot = _hadamard_normalised() @ hv
    y = out["y"][0].astype(np.float64)
    assert np.all(np.abs(y - 2.0 * rot) <= 2.0 * 0.5 * out["sh"][0, 0] * (1 + 1e-5) + 1e-7)


# ----------------------------------------------------------------------------
# the pins reject planted mistakes
# ----------------------------------------------------------------------------

def test_mutants_are_rejected(orc):
    # a flipped sign of code 2 (remap codes 1<->2) breaks the brute-force dot pin
    n, k = 4, 256
    codes, sw = synth.weight(n, k, 0, seed=41)
    rng = np.random.default_rng(42)
    q = rng.integers(-127, 128, size=(1, k)).astype(np.int8)
    swapped = np.choose(codes, [0, 2, 1]).astype(np.uint8)
    d_mut = orc.blockdots(orc.pack(swapped, 0), 0, n, k, q)
    W = _dense_values(codes, 0).astype(np.int64).reshape(n, 2, B)
    ref = np.einsum("nbk,bk->nb", W, q.astype(np.int64).reshape(2, B))
    assert not np.array_equal(d_mut[0], ref)
    # a transposed scale index (block-major scales) breaks the dense einsum pin
    x = synth.activation(1, k, seed=synth.SEED_ACT_BASE)
    qq, ss = orc.rotate_quant(x)
    sw4 = np.ascontiguousarray(sw.reshape(-1)[::-1].reshape(sw.shape))
    y_mut = orc.gemv(orc.pack(codes, 0), sw4, 0, n, k, qq, ss)
    Wd = W.astype(np.float64)
    good = np.einsum("nbk,bk,nb,b->n", Wd, qq.astype(np.float64).reshape(2, B),
                     sw.astype(np.float64), ss[0].astype(np.float64))
    assert np.abs(y_mut[0] - good).max() > 1e-3 * np.abs(good).max()
    # other fold orders give other values on the fold-order worked example,
    # so the golden pin rejects each of them
    g = _golden("fold_order.txt")
    t = [np.float32(int(d)) * np.float32(float(sv)) for d, sv in zip(g["dots"], g["act_scales"])]
    want = np.float32(float(g["expected_fp32"][0]))
    acc = np.float32(0)                                  # one sequential walk over all blocks
    for v in t:
        acc = np.float32(acc + v)
    assert acc == np.float32(float(g["expected_sequential_blocks"][0])) and acc != want
    segs = []                                            # segment sums, then a sequential combine
    for j in range(0, len(t), 8):
        a = np.float32(0)
        for v in t[j:j + 8]:
            a = np.float32(a + v)
        segs.append(a)
    acc = np.float32(0)
    for v in segs:
        acc = np.float32(acc + v)
    assert acc == np.float32(float(g["expected_sequential_segments"][0])) and acc != want
    parts = []                                           # eight strided chains and a fixed tree
    for p in range(8):
        a = np.float32(0)
        for v in t[p::8]:
            a = np.float32(a + v)
        parts.append(a)
    old = np.float32(np.float32(np.float32(parts[0] + parts[1]) + np.float32(parts[2] + parts[3]))
                     + np.float32(np.float32(parts[4] + parts[5]) + np.float32(parts[6] + parts[7])))
    assert old == np.float32(2.0) and old != want

# ----------------------------------------------------------------------------
# the layer stack: layer l + 1 reads the RMS-normalised output of layer l
# ----------------------------------------------------------------------------

def _stack_identity_closed_form(c, n_layers, eps, sg, su, sd):
    """y of a stack of identity-weight layers (hidden = inter = 128, +1 on the
    diagonal; every gate / up / down scale sg / su / sd) fed x = c * e_0, derived
    by hand from the definitions, step by step in binary32:

    * rotation of c * e_0: every butterfly adds or subtracts an exact zero, so
      all 128 values are c, times k = (float)(1/sqrt(128)); absmax = |c k|,
      s = absmax / 127, and every code is rint((c k) / s) = +-127.
    * gate / up: one block, one segment, so g = 0 + 127 (sg s) and
      u = 127 (su s) in every output (with the sign of c).
    * h = bf16(silu(g) u) is the same in all 128 outputs; its rotation is
      128 h k at index 0 and exact zeros elsewhere, so s_h = |128 h k| / 127,
      code 0 is +-127 and the rest 0: y = (127 (sd s_h) sign, 0, ..., 0).
    * RMS-normalise of that y: the sum of squares is y_0^2 exactly, so the next
      input is bf16(y_0 / sqrt(y_0^2 / 128 + eps)) * e_0.
    The last layer's y is not normalised."""
    f = np.float32
    k = np.uint32(0x3DB504F3).view(np.float32)
    x0 = f(c)
    y0 = None
    for layer in range(n_layers):
        v = f(x0 * k)
        s = f(abs(v) / f(127))
        q = f(127) if v > 0 else f(-127)
        g = f(q * f(f(sg) * s))
        u = f(q * f(f(su) * s))
        gd, ud = float(g), float(u)
        h64 = gd / (1.0 + math.exp(-gd)) * ud
        hb = _bf16_bits(np.array([h64], np.float32))[0]
        hv = _bf16_value(np.array([hb]))[0]
        # the fp32 chain of the oracle rounds to the same bf16 value unless
        # h64 sits within an fp32 ulp or two of a bf16 rounding midpoint
        lo, hi = sorted((float(_bf16_value(np.array([hb - 1]))[0]), float(_bf16_value(np.array([hb + 1]))[0])))
        assert abs(h64 - (hv + lo) / 2) > 1e-5 * abs(h64) and abs(h64 - (hv + hi) / 2) > 1e-5 * abs(h64)
        vh = f(f(f(128) * hv) * k)
        sh = f(abs(vh) / f(127))
        qh = f(127) if vh > 0 else f(-127)
        y0 = f(qh * f(f(sd) * sh))
        if layer + 1 < n_layers:
            ms = f(f(y0 * y0) / f(128))
            inv = f(f(1) / np.sqrt(f(ms + f(eps)), dtype=np.float32))
            x0 = _bf16_value(_bf16_bits(np.array([f(y0 * inv)], np.float32)))[0]
    y = np.zeros(128, np.float32)
    y[0] = y0
    return y


def _identity_stack_layers(orc, n_layers, sg, su, sd):
    n = B
    P = orc.pack(np.eye(n, dtype=np.uint8), 0)
    sc = [np.full((n, 1), v, np.float16) for v in (sg, su, sd)]
    return [(P, sc[0], P, sc[1], P, sc[2])] * n_layers


@pytest.mark.parametrize("c,eps", [(3.0, 1e-6), (-0.75, 0.01)])
def test_ffn_stack_identity_closed_form(orc, c, eps):
    sg, su, sd = 1.0, 0.5, 2.0
    x = _bf16_bits(np.array([[c] + [0.0] * (B - 1)], np.float32))
    for n_layers in (1, 2, 3):
        layers = _identity_stack_layers(orc, n_layers, sg, su, sd)
        y = orc.ffn_stack(layers, 0, B, B, x, eps)
        want = _stack_identity_closed_form(c, n_layers, eps, sg, su, sd)
        assert np.array_equal(y[0].view(np.uint32), want.view(np.uint32)), (n_layers, y[0][:2], want[:2])


def test_ffn_stack_mutants_are_rejected(orc):
    """Plausible mistakes in the stack's composition fail the closed-form pin:
    normalising after the last layer, feeding layer 2 the raw input instead of
    the normalised output of layer 1, and dropping (or misplacing) eps."""
    sg, su, sd, c, eps = 1.0, 0.5, 2.0, 3.0, 0.01
    x = _bf16_bits(np.array([[c] + [0.0] * (B - 1)], np.float32))
    layers = _identity_stack_layers(orc, 2, sg, su, sd)
    want = _stack_identity_closed_form(c, 2, eps, sg, su, sd)
    good = orc.ffn_stack(layers, 0, B, B, x, eps)[0]
    assert np.array_equal(good.view(np.uint32), want.view(np.uint32))
    # the last layer normalised as well
    normed_last = _bf16_value(orc.rmsnorm_bf16(good[None, :], eps))[0]
    assert not np.array_equal(normed_last, want)
    # layer 2 fed x instead of rmsnorm(y_1)
    y1 = orc.ffn_step(*layers[0], 0, B, B, x)["y"]
    raw = orc.ffn_step(*layers[1], 0, B, B, x)["y"][0]
    assert not np.array_equal(raw, want)
    # layer 2 fed y_1 rounded to bf16 without the normalisation
    unnormed = orc.ffn_step(*layers[1], 0, B, B, _bf16_bits(y1))["y"][0]
    assert not np.array_equal(unnormed, want)
    # eps dropped (0 instead of the argument)
    no_eps = orc.ffn_stack(layers, 0, B, B, x, 0.0)[0]
    assert not np.array_equal(no_eps, want)
