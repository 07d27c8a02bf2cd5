"""The C-ABI library loads and exports every entry point include/*.h declare,
and rejects bad arguments before touching the GPU.  No GPU needed."""
import ctypes
import os
import re

import pytest

from ternary_weight_dp4a_gb300 import build as tqbuild
from ternary_weight_dp4a_gb300 import tq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tqbuild.build()
    return tq.load()


def _declared():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        # function declarations only (not the hook members "(*name)(")
        names |= set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_and_binding_agree():
    assert sorted(tq.EXPORTS) == _declared()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.tq_status_string(0) == b"ok"
    assert lib.tq_status_string(4) == b"workspace too small"
    assert lib.tq_status_string(6).startswith(b"a bounded wait")
    assert lib.tq_status_string(99) == b"unknown status"


def test_error_word_maps_to_timeout_status(lib):
    assert lib.tq_error_status(0) == 0
    for bit in range(9):
        assert lib.tq_error_status(1 << bit) == tq.TQ_ERR_TIMEOUT
    assert lib.tq_read_error_word(None, None, ctypes.c_void_p(0)) == 1


def test_engine_setting_round_trips_and_rejects_unknown(lib):
    before = lib.tq_get_engine()
    try:
        for e in (tq.ENGINE_DP4A, tq.ENGINE_TCGEN05, tq.ENGINE_AUTO):
            assert lib.tq_set_engine(e) == 0 and lib.tq_get_engine() == e
        assert lib.tq_set_engine(7) == 1 and lib.tq_get_engine() == tq.ENGINE_AUTO
    finally:
        lib.tq_set_engine(before)


def test_workspace_bytes(lib):
    # dp4a part: qx 5120 | sx 160->256 | h 34816 | qh 17408 | sh 544->768 |
    # counters 544->768 | ybuf 20480 | err 4->256 | sync 76->256 | hst 17408 |
    # hsn 1088->1280 | hp 69632, each 256-aligned
    dp4a = 5120 + 256 + 34816 + 17408 + 768 + 768 + 20480 + 256 + 256 + 17408 + 1280 + 69632
    # tensor-core part: operand copy of h, 136 blocks x 2 KB | its pairs 136 x 8 x 8 |
    # segment sums of gate and up, 2 x 136 tiles x 5 segments x 8 rows x 128 x 4 |
    # of down, 40 tiles x 17 segments x 4096 | tile counts 136 x 4 -> 768, 320 x 4 -> 1280 |
    # second stack buffer 20480
    tc = 136 * 2048 + 136 * 64 + 2 * 136 * 5 * 4096 + 40 * 17 * 4096 + 768 + 1280 + 20480
    assert lib.tq_ffn_workspace_bytes(1, 5120, 17408) == dp4a + tc
    assert lib.tq_ffn_workspace_bytes(0, 5120, 17408) == 0
    # GEMV: err 256 | tile counts 1088 x 4 = 4352 | operand 40 blocks x 2 KB |
    # pairs 40 x 64 | segment sums 136 tiles x 5 segments x 4096
    assert lib.tq_gemv_workspace_bytes(1, 17408, 5120) == 256 + 4352 + 40 * 2048 + 40 * 64 + 136 * 5 * 4096
    assert lib.tq_gemv_workspace_bytes(0, 17408, 5120) == 0


def test_workspace_error_offset(lib):
    from _util import ws_offsets
    for m, hidden, inter in ((1, 5120, 17408), (8, 5120, 17408), (3, 256, 512)):
        off = lib.tq_ffn_workspace_error_offset(m, hidden, inter)
        assert off == ws_offsets(m, hidden, inter)["err"]
        assert off % 4 == 0 and off + 4 <= lib.tq_ffn_workspace_bytes(m, hidden, inter)
    assert lib.tq_ffn_workspace_error_offset(1, 0, 512) == 0


def _w(codes=0x1000, scales=0x2000, n=512, k=256, fmt=0):
    return tq._Weight(codes, scales, n, k, fmt)


def test_gemv_rejects_bad_arguments_before_any_launch(lib):
    good_q, good_s, good_y = ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000), ctypes.c_void_p(0x5000)
    st = ctypes.c_void_p(0)
    ws, wsb = ctypes.c_void_p(0x100000), lib.tq_gemv_workspace_bytes(1, 512, 256)
    call = lambda w, q=good_q, s=good_s, m=1, y=good_y, ws=ws, wsb=wsb: lib.tq_gemv(
        ctypes.byref(w), q, s, m, y, None, ws, wsb, st)
    assert call(_w(codes=0)) == 1                       # null codes
    assert call(_w(k=200)) == 1                         # k not a multiple of 128
    assert call(_w(n=0)) == 1                           # empty output
    assert call(_w(fmt=7)) == 1                         # unknown format
    assert call(_w(), m=0) == 1 and call(_w(), m=65) == 1
    assert call(_w(), q=ctypes.c_void_p(0)) == 1
    assert call(_w(codes=0x1010)) == 2                  # codes not 32-byte aligned
    assert call(_w(), q=ctypes.c_void_p(0x3008)) == 2   # q not 16-byte aligned
    assert call(_w(), ws=ctypes.c_void_p(0)) == 1       # no workspace
    assert call(_w(), ws=ctypes.c_void_p(0x100010)) == 2  # workspace not 256-byte aligned
    assert call(_w(), wsb=wsb - 1) == 4                 # workspace too small
    assert lib.tq_gemv(None, good_q, good_s, 1, good_y, None, ws, wsb, st) == 1
    g, u = _w(n=512, k=256), _w(n=512, k=256)
    fw = lib.tq_ffn_workspace_bytes(1, 256, 512)
    assert lib.tq_ffn_gateup(ctypes.byref(g), ctypes.byref(u), good_q, good_s, 1, good_y, ws, fw - 1, st) == 4
    assert lib.tq_ffn_gateup(ctypes.byref(g), ctypes.byref(u), good_q, good_s, 1, good_y, None, fw, st) == 1


def test_ffn_step_rejects_bad_arguments(lib):
    st = ctypes.c_void_p(0)
    g, u, d = _w(n=512, k=256), _w(n=512, k=256), _w(n=256, k=512)
    x, y, ws = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    need = lib.tq_ffn_workspace_bytes(1, 256, 512)
    call = lambda g=g, u=u, d=d, m=1, wsb=need, ws=ws: lib.tq_ffn_step(
        ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), x, m, y, ws, wsb, st)
    assert call(d=_w(n=256, k=384)) == 1                # down shape mismatch
    assert call(u=_w(n=512, k=256, fmt=1)) == 1         # mixed formats
    assert call(m=65) == 1
    assert call(wsb=need - 1) == 4                      # workspace too small
    assert call(ws=ctypes.c_void_p(0x30010)) == 2       # workspace not 256-byte aligned


def test_other_entry_points_reject_bad_arguments(lib):
    st = ctypes.c_void_p(0)
    p = ctypes.c_void_p(0x1000)
    assert lib.tq_pack_weights(None, 4, 128, 0, p, st) == 1
    assert lib.tq_pack_weights(p, 4, 100, 0, p, st) == 1
    assert lib.tq_pack_weights(p, 4, 128, 0, ctypes.c_void_p(0x1001), st) == 2
    assert lib.tq_rotate_quant(p, 0, 128, p, p, st) == 1
    assert lib.tq_rotate_quant(p, 1, 130, p, p, st) == 1
    assert lib.tq_rmsnorm_bf16(None, 1, 128, ctypes.c_float(1e-6), p, st) == 1
    assert lib.tq_ffn_workspace_init(None, 16, st) == 1
    assert lib.tq_ffn_stage_input(p, 1, 256, 512, None, 4096, st) == 1
    assert lib.tq_ffn_stage_input(p, 65, 256, 512, p, 1 << 20, st) == 1
    big = ctypes.c_void_p(0x100000)
    assert lib.tq_ffn_stage_input(p, 1, 256, 512, big, 16, st) == 4
    assert lib.tq_ffn_stack(None, 1, p, 1, ctypes.c_float(1e-6), p, big, 1 << 20, st) == 1
    w = (tq._Weight * 3)(_w(n=512, k=256), _w(n=512, k=256), _w(n=256, k=512))
    assert lib.tq_ffn_stack(w, 0, p, 1, ctypes.c_float(1e-6), p, big, 1 << 20, st) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(tq, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(tq, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        tq.load()


def test_headers_are_c11_and_a_c_program_links(lib, tmp_path):
    """include/*.h compile as pedantic C11 with no warnings, and a C program
    links against libtq and calls its host-only entry points (no GPU work)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(r'''
#include "tq.h"
#include "tq_lifecycle.h"
#include <stdio.h>
static void *a(void *c, size_t b, int32_t p) { (void)c; (void)b; (void)p; return 0; }
static void r(void *c, void *q, size_t b, int32_t p) { (void)c; (void)q; (void)b; (void)p; }
static size_t f(void *c) { (void)c; return 0; }
static int32_t bd(void *c, void *q, size_t b) { (void)c; (void)q; (void)b; return 0; }
int main(void) {
    tq_lifecycle lc;
    tq_lifecycle_config cfg = {100, 10, 0, 0};
    tq_lifecycle_hooks h = {a, r, f, bd, 0};
    if (tq_lifecycle_init(&lc, &cfg, &h) != TQ_OK) return 1;
    if (tq_lifecycle_load(&lc) != TQ_OK) return 2;
    if (tq_set_engine(TQ_ENGINE_DP4A) != TQ_OK || tq_get_engine() != TQ_ENGINE_DP4A) return 3;
    if (tq_error_status(64u) != TQ_ERR_TIMEOUT) return 4;
    printf("%s %d %zu %zu %zu\n", tq_status_string(TQ_OK), lc.state,
           tq_ffn_workspace_bytes(1, 5120, 17408), tq_ffn_workspace_error_offset(1, 5120, 17408),
           tq_gemv_workspace_bytes(1, 17408, 5120));
    return 0;
}
''')
    libdir = os.path.dirname(tq.LIB_PATH)
    exe = tmp_path / "abi"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    f"-I{os.path.join(ROOT, 'include')}", str(src), f"-L{libdir}", "-ltq",
                    "-o", str(exe)], check=True, capture_output=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")
    env = dict(os.environ, LD_LIBRARY_PATH=os.pathsep.join(
        [libdir, cuda_lib, os.environ.get("LD_LIBRARY_PATH", "")]))
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, env=env).stdout.split()
    assert out[0] == "ok" and int(out[1]) == 2              # skipped: no free memory
    assert int(out[2]) == lib.tq_ffn_workspace_bytes(1, 5120, 17408)
    assert int(out[3]) == lib.tq_ffn_workspace_error_offset(1, 5120, 17408)
    assert int(out[4]) == lib.tq_gemv_workspace_bytes(1, 17408, 5120)
