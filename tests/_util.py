"""Helpers shared by the GPU tests: seeded inputs on both sides of the parity check.

Inputs come from ``ternary_weight_dp4a_gb300.synth`` (numpy PCG64 on the host).
The oracle packs the raw codes itself; the CUDA path packs them with its own
kernel.  Nothing the CUDA path produces is ever fed to the oracle.
"""
import numpy as np

from ternary_weight_dp4a_gb300 import synth

B = 128


def round_up(x, a):
    return (x + a - 1) // a * a


def ws_offsets(m, hidden, inter):
    """Offsets of the FFN-step intermediates inside the workspace (qx, sx, h,
    qh, sh, counters, ybuf, ..., and the tensor-core kernel's sections), as
    tq_ffn_step lays them out; used only to read intermediates and the
    synchronisation state back for diagnosis."""
    def cdiv(a, b):
        return (a + b - 1) // b
    seg_blocks = cdiv(inter // B, 8) * 8
    passes = cdiv(m, 8)
    off, o = 0, {}
    for name, nbytes in (("qx", m * hidden), ("sx", m * (hidden // B) * 4),
                         ("h", m * inter * 2), ("qh", m * inter), ("sh", m * (inter // B) * 4),
                         ("counters", (inter // B) * 4), ("ybuf", m * hidden * 4), ("err", 4),
                         ("sync", (2 + (inter + 1023) // 1024) * 4), ("hst", m * inter), ("hsn", m * (inter // B) * 8),
                         ("hp", m * inter * 4),
                         ("tc_hst", passes * seg_blocks * 2048), ("tc_hsn", passes * seg_blocks * 64),
                         ("part_a", 2 * cdiv(inter, B) * cdiv(hidden // B, 8) * 8 * B * 4),
                         ("part_b", cdiv(hidden, B) * cdiv(inter // B, 8) * 8 * B * 4),
                         ("cnt_a", cdiv(inter, B) * 4), ("cnt_b", cdiv(hidden, 16) * 4),
                         ("ybuf2", m * hidden * 4)):
        o[name] = off
        off = round_up(off + nbytes, 256)
    o["total"] = off
    return o


class Mat:
    """One weight matrix: raw codes + fp16 scales on the host, packed on the GPU."""

    def __init__(self, n, k, fmt, seed):
        import torch
        from ternary_weight_dp4a_gb300 import tq
        self.n, self.k, self.fmt = n, k, fmt
        self.codes, self.scales = synth.weight(n, k, fmt, seed)
        codes_d = torch.from_numpy(self.codes).cuda()
        scales_d = torch.from_numpy(self.scales).cuda()
        self.dev = tq.pack_weights(codes_d, fmt, scales_d)
        del codes_d
        self._orc_packed = None

    def orc_packed(self, orc):
        if self._orc_packed is None:
            self._orc_packed = orc.pack(self.codes, self.fmt)
        return self._orc_packed


def ffn_mats(hidden, inter, fmt, layer=0):
    return (Mat(inter, hidden, fmt, synth.ffn_weight_seed(layer, 0)),
            Mat(inter, hidden, fmt, synth.ffn_weight_seed(layer, 1)),
            Mat(hidden, inter, fmt, synth.ffn_weight_seed(layer, 2)))


def bf16_tensor(bits_np):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits_np).view(np.int16)).cuda().view(torch.bfloat16)


def bf16_bits(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def fold_rel_err(y, ref64, orc, packed, scales, fmt, n, k, q, s):
    """max |y - ref| / sum_b |t_b|: the error relative to the magnitude of the
    block terms being summed (t_b = d_b * sw * s), which stays meaningful for
    outputs whose terms cancel."""
    d = orc.blockdots(packed, fmt, n, k, q).astype(np.float64)          # [m][n][nb]
    sw = np.asarray(scales, np.float16).astype(np.float64)               # [n][nb]
    sa = np.asarray(s, np.float64).reshape(d.shape[0], 1, -1)            # [m][1][nb]
    mag = (np.abs(d) * sw[None] * sa).sum(axis=2)
    err = np.abs(np.asarray(y, np.float64) - ref64)
    return float((err / np.maximum(mag, 1e-30)).max()) if err.size else 0.0


def rel_err(y, ref):
    """max |y - ref| / max(|ref|, 1e-3 * rms(ref)) (the floor keeps outputs that
    cancel to near zero from dominating)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = 1e-3 * np.sqrt(np.mean(ref ** 2)) if ref.size else 1.0
    return float((np.abs(y - ref) / np.maximum(np.abs(ref), max(floor, 1e-30))).max()) \
        if ref.size else 0.0
