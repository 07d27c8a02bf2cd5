"""GPU parity of the 64-layer FFN stacks the benchmark times (hidden 5120,
intermediate 17408): the 2-bit stack at one row and the 1-bit stack at 1, 2,
4 and 8 packed rows, bit for bit against the oracle's stack (layer l + 1
reads the RMS-normalised output of layer l, the last layer's output is not
normalised), on both kernels.

The weights are drawn on the GPU (seeded, as the benchmark draws them) and
copied to the host one layer at a time for the oracle, so the host never
holds more than one layer.
"""
import numpy as np
import pytest

from _util import bf16_tensor
from ternary_weight_dp4a_gb300 import synth

pytestmark = pytest.mark.gpu
HIDDEN, INTER, LAYERS, EPS = 5120, 17408, 64, 1e-6


@pytest.fixture(scope="module")
def tq():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ternary_weight_dp4a_gb300 import build, tq as tqmod
    build.build()
    tqmod.load()
    return tqmod


class _HostLayers:
    """The oracle's view of the device layers: packed on the host on demand."""

    def __init__(self, orc, raw, fmt):
        self.orc, self.raw, self.fmt = orc, raw, fmt

    def __len__(self):
        return len(self.raw)

    def __iter__(self):
        for mats in self.raw:
            out = []
            for codes_d, scales_d in mats:
                out += [self.orc.pack(codes_d.cpu().numpy(), self.fmt), scales_d.cpu().numpy()]
            yield tuple(out)


@pytest.fixture(scope="module")
def stacks(tq):
    import torch
    made = {}

    def get(fmt):
        if fmt not in made:
            made.clear()
            torch.cuda.empty_cache()
            raw, dev = [], []
            for layer in range(LAYERS):
                mats, packed = [], []
                for j, (n, k) in enumerate([(INTER, HIDDEN), (INTER, HIDDEN), (HIDDEN, INTER)]):
                    codes, scales = synth.weight(n, k, fmt, synth.ffn_weight_seed(layer, j), device="cuda")
                    packed.append(tq.pack_weights(codes, fmt, scales))
                    mats.append((codes, scales))
                raw.append(mats)
                dev.append(tuple(packed))
                # keep the unpacked codes only as long as the oracle needs them
            made[fmt] = (raw, dev)
        return made[fmt]
    return get


@pytest.mark.parametrize("fmt,rows", [(0, (1,)), (1, (1, 2, 4, 8))], ids=["ternary2", "binary1"])
def test_64_layer_stack_bit_exact(tq, orc, stacks, fmt, rows):
    """The oracle runs once for the largest row count (its rows are computed
    independently of one another); every GPU run, on either kernel, must give
    the oracle's bits for its rows."""
    import torch
    raw, dev = stacks(fmt)
    x = synth.activation(max(rows), HIDDEN, seed=synth.SEED_ACT_BASE, outlier_frac=0.01)
    ref = orc.ffn_stack(_HostLayers(orc, raw, fmt), fmt, HIDDEN, INTER, x, EPS)
    before = tq.get_engine()
    try:
        for engine in (tq.ENGINE_TCGEN05, tq.ENGINE_DP4A):
            tq.set_engine(engine)
            for m in rows:
                y = tq.ffn_stack(list(dev), bf16_tensor(x[:m]), EPS)
                torch.cuda.synchronize()
                assert np.array_equal(y.cpu().numpy().view(np.uint32), ref[:m].view(np.uint32)), (engine, fmt, m)
    finally:
        tq.set_engine(before)
