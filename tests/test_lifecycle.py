"""Host-side lifecycle policy of the ternary weight copy (include/tq_lifecycle.h),
run in libtq against a fake device with a fixed memory budget.  No GPU needed.

The rules under test come from the review that rejected the first ternary copy
(sparkinfer PR #1154, "long-context serving regression" closing comment) and
the fix after it (PR #1160, commit message): skip the copy at load when what
is left after it cannot hold the reserve other work needs; release it on any
allocation failure it causes and retry; rebuild it once memory is free again.
"""
import pytest

from ternary_weight_dp4a_gb300 import build as tqbuild
from ternary_weight_dp4a_gb300 import tq

MB = 1 << 20
GB = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def lib():
    tqbuild.build()
    return tq.load()


class FakeDevice:
    """Device memory of `total` bytes; every allocation and release logged."""

    def __init__(self, total):
        self.total = total
        self.used = 0
        self.live = {}
        self.next = 0x10000
        self.log = []
        self.fail_builds = 0
        self.raise_in = None

    def _maybe_raise(self, hook):
        if self.raise_in == hook:
            raise RuntimeError("hook failure")

    def alloc(self, nbytes, purpose):
        self._maybe_raise("alloc")
        if self.used + nbytes > self.total:
            self.log.append(("oom", nbytes, purpose))
            return 0
        addr = self.next
        self.next += (nbytes + 4095) // 4096 * 4096 + 4096
        self.live[addr] = (nbytes, purpose)
        self.used += nbytes
        self.log.append(("alloc", nbytes, purpose))
        return addr

    def release(self, ptr, nbytes, purpose):
        assert self.live.pop(ptr) == (nbytes, purpose)
        self.used -= nbytes
        self.log.append(("release", nbytes, purpose))

    def free_bytes(self):
        self._maybe_raise("free_bytes")
        return self.total - self.used

    def build(self, ptr, nbytes):
        self._maybe_raise("build")
        assert self.live[ptr] == (nbytes, tq.CopyLifecycle.COPY)
        if self.fail_builds:
            self.fail_builds -= 1
            return False
        return True

    def hold(self, nbytes):
        """Memory taken by something outside the policy (e.g. a cache pool)."""
        self.used += nbytes


def _lc(dev, copy=30, reserve=20, margin=0, after=0):
    return tq.CopyLifecycle(copy, reserve, dev, rebuild_margin=margin, rebuild_after=after)


def test_load_builds_when_copy_and_reserve_fit():
    dev = FakeDevice(100)
    lc = _lc(dev)
    assert lc.state == "absent" and lc.copy is None
    assert lc.load() == "resident"
    assert lc.copy is not None and dev.live[lc.copy] == (30, tq.CopyLifecycle.COPY)
    assert dev.used == 30
    assert lc.counters()["builds"] == 1 and lc.counters()["rebuilds"] == 0


def test_load_skips_when_reserve_would_not_fit():
    dev = FakeDevice(100)
    dev.hold(51)                                   # free 49 < copy 30 + reserve 20
    lc = _lc(dev)
    assert lc.load() == "skipped"
    assert lc.copy is None
    assert not any(e[0] == "alloc" for e in dev.log)     # the copy was never allocated


def test_load_exactly_at_the_limit_builds():
    dev = FakeDevice(100)
    dev.hold(50)                                   # free 50 == 30 + 20
    assert _lc(dev).load() == "resident"


def test_failed_allocation_releases_copy_and_retries_once():
    dev = FakeDevice(100)
    lc = _lc(dev)
    lc.load()
    p = lc.alloc(60)                               # free 70: fits beside the copy
    assert p is not None and lc.state == "resident"
    lc.free(p, 60)
    p = lc.alloc(80)                               # free 70: fails, copy released, retry fits
    assert p is not None
    assert lc.state == "released" and lc.copy is None
    c = lc.counters()
    assert (c["alloc_failures"], c["releases"], c["retries_ok"]) == (1, 1, 1)
    assert [e[0] for e in dev.log[-3:]] == ["oom", "release", "alloc"]


def test_allocation_too_large_even_without_copy():
    dev = FakeDevice(100)
    lc = _lc(dev)
    lc.load()
    assert lc.alloc(120) is None
    assert lc.state == "released"                  # released for the retry, which still failed
    c = lc.counters()
    assert (c["alloc_failures"], c["releases"], c["retries_ok"]) == (1, 1, 0)


def test_failed_allocation_without_copy_changes_nothing():
    dev = FakeDevice(100)
    dev.hold(60)
    lc = _lc(dev)
    lc.load()                                      # skipped
    assert lc.alloc(50) is None
    assert lc.state == "skipped"
    assert lc.counters()["releases"] == 0 and lc.counters()["alloc_failures"] == 1


def test_rebuild_once_memory_is_free_again():
    dev = FakeDevice(100)
    lc = _lc(dev)
    lc.load()
    p = lc.alloc(80)                               # forces a release
    assert lc.state == "released"
    for _ in range(3):                             # scratch still held: free 20 < 50
        assert lc.poll() == "released"
    lc.free(p, 80)
    assert lc.poll() == "resident"
    assert lc.copy is not None and dev.used == 30
    c = lc.counters()
    assert (c["builds"], c["rebuilds"]) == (2, 1)


def test_rebuild_waits_the_configured_polls():
    dev = FakeDevice(100)
    lc = _lc(dev, after=3)
    lc.load()
    lc.release()
    assert [lc.poll() for _ in range(4)] == ["released", "released", "released", "resident"]


def test_rebuild_margin_is_hysteresis():
    dev = FakeDevice(100)
    lc = _lc(dev, margin=10)
    lc.load()                                      # load needs only copy + reserve
    assert lc.state == "resident"
    lc.release()
    dev.hold(45)                                   # free 55 < 30 + 20 + 10
    assert lc.poll() == "released"
    dev.hold(-5)                                   # free 60 == 30 + 20 + 10
    assert lc.poll() == "resident"


def test_skipped_copy_is_built_when_memory_allows():
    dev = FakeDevice(100)
    dev.hold(60)
    lc = _lc(dev)
    assert lc.load() == "skipped"
    assert lc.poll() == "skipped"
    dev.hold(-60)
    assert lc.poll() == "resident"
    assert lc.counters()["rebuilds"] == 1


def test_build_failure_frees_the_copy_and_retries_later():
    dev = FakeDevice(100)
    dev.fail_builds = 1
    lc = _lc(dev)
    assert lc.load() == "failed"
    assert dev.used == 0 and lc.copy is None
    assert lc.counters()["build_failures"] == 1
    assert lc.poll() == "resident"


def test_copy_allocation_failure_is_a_build_failure():
    dev = FakeDevice(100)
    lc = _lc(dev, copy=30, reserve=0)
    # free memory says yes, the allocation says no (fragmentation, a race)
    dev.free_bytes = lambda: 100
    dev.hold(80)
    assert lc.load() == "failed"
    assert lc.counters()["build_failures"] == 1


def test_explicit_release_and_destroy():
    dev = FakeDevice(100)
    lc = _lc(dev)
    lc.load()
    lc.release()
    assert lc.state == "released" and dev.used == 0
    lc.release()                                   # no-op
    assert lc.counters()["releases"] == 1
    assert lc.poll() == "resident"
    lc.destroy()
    assert dev.used == 0 and lc.state == "absent" and lc.copy is None


def test_load_only_once():
    dev = FakeDevice(100)
    lc = _lc(dev)
    lc.load()
    with pytest.raises(tq.TQError):
        lc.load()


@pytest.mark.parametrize("copy,after", [(0, 0), (10, -1)])
def test_init_rejects_bad_config(copy, after):
    with pytest.raises(tq.TQError):
        tq.CopyLifecycle(copy, 0, FakeDevice(100), rebuild_after=after)


@pytest.mark.parametrize("hook", ["alloc", "build", "free_bytes"])
def test_raising_hooks_count_as_failures(hook):
    dev = FakeDevice(100)
    dev.raise_in = hook
    lc = _lc(dev)
    state = lc.load()
    if hook == "free_bytes":
        assert state == "skipped"                  # 0 bytes free
    else:
        assert state == "failed"
    assert dev.used == 0


def test_long_context_serving_scenario():
    """The rejected copy's failure, replayed with the page's figures: a 32 GB
    card, a ~3.85 GB copy, a KV pool that leaves 60-100 MB free after startup,
    and prefill scratch allocations that then fail.  With the policy the copy
    is skipped at load when the prefill reserve cannot fit; when it is built
    (short context), a prefill allocation releases it and succeeds, and the
    copy comes back after the prefill frees its scratch."""
    copy = int(3.85 * GB)
    prefill = 1731 * MB                            # the scratch the failing prefill asked for
    # long context: the cache pool leaves less than copy + reserve
    dev = FakeDevice(32 * GB)
    dev.hold(32 * GB - copy - 80 * MB)             # after startup ~80 MB would be free
    lc = tq.CopyLifecycle(copy, prefill, dev)
    assert lc.load() == "skipped"
    p = lc.alloc(prefill)                          # prefill's scratch fits: nothing was built
    assert p is not None
    lc.free(p, prefill)
    # short context: room for copy + reserve, so it is built
    dev = FakeDevice(32 * GB)
    dev.hold(20 * GB)
    lc = tq.CopyLifecycle(copy, prefill, dev, rebuild_after=1)
    assert lc.load() == "resident"
    dev.hold(32 * GB - dev.used - 80 * MB)         # later, sessions grow the pool
    p = lc.alloc(prefill)                          # fails, copy released, retry succeeds
    assert p is not None and lc.state == "released"
    assert lc.poll() == "released"                 # waits one poll
    assert lc.poll() == "released"                 # prefill still holds its scratch
    lc.free(p, prefill)
    dev.hold(-(prefill + 2 * GB))                  # sessions end: 7.6 GB free
    assert lc.poll() == "resident"
    c = lc.counters()
    assert (c["builds"], c["rebuilds"], c["releases"], c["retries_ok"]) == (2, 1, 1, 1)


@pytest.mark.gpu
def test_torch_hooks_build_a_copy_the_gemv_reads():
    """The PyTorch adapter on a real device (small allocations only): the copy
    the policy builds is what a GEMV reads, bit-identical to the original; an
    impossible reserve skips it."""
    import ctypes
    import numpy as np
    import torch
    from ternary_weight_dp4a_gb300 import synth
    n, k = 512, 256
    codes, scales = synth.weight(n, k, 0, synth.SEED_TINY_WEIGHT, device="cuda")
    w = tq.pack_weights(codes, 0, scales)
    nbytes = w.codes.numel()

    def build_fn(t):
        t.copy_(w.codes.view(-1))
        return True

    hooks = tq.TorchDeviceHooks(build_fn)
    lc = tq.CopyLifecycle(nbytes, 0, hooks)
    assert lc.load() == "resident"
    t = hooks.tensor(lc.copy)
    assert t is not None and t.data_ptr() == lc.copy
    wc = tq.PackedWeight(t.view(n, k // 4), w.scales, n, k, 0)
    x = synth.activation(1, k, synth.SEED_ACT_BASE, 0.01, device="cuda")
    q, s = tq.rotate_quant(x)
    y0 = tq.gemv(w, q, s)
    y1 = tq.gemv(wc, q, s)
    torch.cuda.synchronize()
    assert np.array_equal(y0.cpu().numpy().view(np.uint32), y1.cpu().numpy().view(np.uint32))
    lc.destroy()
    assert hooks.tensor(int(t.data_ptr())) is None
    skipped = tq.CopyLifecycle(nbytes, 1 << 62, tq.TorchDeviceHooks(build_fn))
    assert skipped.load() == "skipped"
