"""tq_ffn_step_static: the FFN step for callers that cannot allocate device
memory when they run it (a plugin whose host application owns every device
allocation, a real-time loop that may not call the allocator after start-up).
Its scratch is an array built into the library instead of a caller-supplied
workspace.  It must give exactly the bits tq_ffn_step gives with a
caller-owned workspace, call after call, and refuse sizes beyond the array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest

from _util import bf16_tensor, ffn_mats
from ternary_weight_dp4a_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ternary_weight_dp4a_gb300 import build, tq as tqmod
    build.build()
    tqmod.load()
    return tqmod


# one row; 3 rows (one pass); 5 and 8 rows (two passes over the one array: the
# launch ticket, the segment counters and the per-block counts carry from the
# first pass to the second after a single zero-fill)
@pytest.mark.parametrize("hidden,inter,m", [(1024, 3072, 1), (1024, 2816, 3), (1024, 2816, 5), (2048, 4096, 8)])
def test_static_scratch_step_matches_workspace_step(tq, hidden, inter, m):
    import torch
    g, u, d = (w.dev for w in ffn_mats(hidden, inter, 0))
    for call in range(2):          # two calls in a row share the built-in scratch
        x = bf16_tensor(synth.activation(m, hidden, seed=synth.SEED_ACT_BASE + 100 * call,
                                         outlier_frac=0.01))
        y_static = tq.ffn_step_static(g, u, d, x)
        y_ref = tq.ffn_step(g, u, d, x)
        torch.cuda.synchronize()
        assert torch.equal(y_static.view(torch.int32), y_ref.view(torch.int32)), call


def test_static_scratch_call_allocates_nothing(tq):
    """After a first call (which looks the array up once), a raw C-ABI call
    changes neither PyTorch's allocation counters nor the device's free
    memory: the entry point allocates nothing."""
    import torch
    hidden, inter, m = 1024, 2816, 2
    g, u, d = (w.dev for w in ffn_mats(hidden, inter, 0))
    x = bf16_tensor(synth.activation(m, hidden, seed=synth.SEED_ACT_BASE, outlier_frac=0.01))
    y = torch.empty((m, hidden), dtype=torch.float32, device="cuda")
    lib = tq.load()
    gs, us, ds = g.c_struct(), u.c_struct(), d.c_struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        return lib.tq_ffn_step_static(ctypes.byref(gs), ctypes.byref(us), ctypes.byref(ds),
                                      ctypes.c_void_p(x.data_ptr()), m, ctypes.c_void_p(y.data_ptr()), stream)
    assert call() == 0
    torch.cuda.synchronize()
    stats0 = torch.cuda.memory_stats()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert call() == 0
    torch.cuda.synchronize()
    stats1 = torch.cuda.memory_stats()
    free1 = torch.cuda.mem_get_info()[0]
    for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key
    assert free1 == free0
    ref = tq.ffn_step(g, u, d, x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))


def test_static_scratch_refuses_sizes_beyond_its_limit(tq):
    from _util import ws_offsets
    lib = tq.load()
    # the array holds the part of the FFN workspace the step it runs uses (the
    # dp4a kernel's, which ends where the tensor-core sections begin) at the
    # largest sizes it serves
    assert lib.tq_ffn_static_workspace_bytes() == ws_offsets(8, 8192, 32768)["tc_hst"]
    # shapes only: nothing is read when the call refuses
    big = dict(hidden=8192 + 1024, inter=17408)
    g = tq._Weight(0x1000, 0x2000, big["inter"], big["hidden"], 0)
    u = tq._Weight(0x3000, 0x4000, big["inter"], big["hidden"], 0)
    d = tq._Weight(0x5000, 0x6000, big["hidden"], big["inter"], 0)
    p = ctypes.c_void_p(0x7000)
    st = lib.tq_ffn_step_static(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), p, 1, p,
                                ctypes.c_void_p(0))
    assert st == 3                 # TQ_ERR_UNSUPPORTED
