"""Python face of the CPU oracle (``tq_oracle.c``) for the ternary FFN decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The product library
(``ternary_weight_dp4a_gb300``) never imports it and shares no code with it.

Every function here marshals numpy arrays into the plain-C oracle (compiled with
gcc, ``-O2 -ffp-contract=off``) and back.  The arithmetic lives in the C file;
each C function cites the passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtq_oracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 128
FMT_TERNARY2 = 0
FMT_BINARY1 = 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, portable C, no intrinsics)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u8, u16, i8, i32, f32, f64 = (ctypes.c_uint8, ctypes.c_uint16, ctypes.c_int8,
                                          ctypes.c_int32, ctypes.c_float, ctypes.c_double)
            ci = ctypes.c_int
            L.orc_bf16_to_f32.argtypes = [u16]; L.orc_bf16_to_f32.restype = f32
            L.orc_f32_to_bf16.argtypes = [f32]; L.orc_f32_to_bf16.restype = u16
            L.orc_f16_to_f32.argtypes = [u16]; L.orc_f16_to_f32.restype = f32
            L.orc_pack2.argtypes = [_P(u8), ci, ci, _P(u8)]
            L.orc_unpack2.argtypes = [_P(u8), ci, ci, _P(i8)]
            L.orc_pack1.argtypes = [_P(u8), ci, ci, _P(u8)]
            L.orc_unpack1.argtypes = [_P(u8), ci, ci, _P(i8)]
            L.orc_wht128.argtypes = [_P(f32)]
            L.orc_quant_block.argtypes = [_P(f32), _P(i8), _P(f32)]
            L.orc_rotate_quant.argtypes = [_P(u16), ci, ci, _P(i8), _P(f32)]
            L.orc_blockdots.argtypes = [_P(u8), ci, ci, ci, _P(i8), ci, _P(i32)]
            L.orc_gemv.argtypes = [_P(u8), _P(u16), ci, ci, ci, _P(i8), _P(f32), ci, _P(f32)]
            L.orc_gemv_f64.argtypes = [_P(u8), _P(u16), ci, ci, ci, _P(i8), _P(f32), ci,
                                       _P(f64)]
            L.orc_expf.argtypes = [f32]; L.orc_expf.restype = f32
            L.orc_silu.argtypes = [f32]; L.orc_silu.restype = f32
            L.orc_silu_mul_bf16.argtypes = [_P(f32), _P(f32), ctypes.c_size_t, _P(u16)]
            L.orc_ffn_step.argtypes = [_P(u8), _P(u16), _P(u8), _P(u16), _P(u8), _P(u16), ci,
                                       ci, ci, _P(u16), ci, _P(f32),
                                       _P(i8), _P(f32), _P(f32), _P(f32), _P(u16), _P(i8),
                                       _P(f32)]
            L.orc_rmsnorm_bf16.argtypes = [_P(f32), ci, ci, f32, _P(u16)]
            L.orc_set_threads.argtypes = [ci]
            L.orc_get_threads.restype = ci
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(t: int) -> None:
    lib().orc_set_threads(int(t))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# --- scalar conversions -----------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = _c(bits, np.uint16)
    L = lib()
    return np.array([L.orc_bf16_to_f32(int(v)) for v in b.ravel()],
                    dtype=np.float32).reshape(b.shape)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    f = _c(x, np.float32)
    L = lib()
    return np.array([L.orc_f32_to_bf16(float(v)) for v in f.ravel()],
                    dtype=np.uint16).reshape(f.shape)


def f16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = _c(bits, np.uint16)
    L = lib()
    return np.array([L.orc_f16_to_f32(int(v)) for v in b.ravel()],
                    dtype=np.float32).reshape(b.shape)


# --- layout -----------------------------------------------------------------

def pack(codes: np.ndarray, fmt: int) -> np.ndarray:
    """codes [n][k] (2-bit: values 0/1/2; 1-bit: 0/1) -> packed bytes."""
    c = _c(codes, np.uint8)
    n, k = c.shape
    per = 4 if fmt == FMT_TERNARY2 else 8
    out = np.empty((n, k // per), dtype=np.uint8)
    fn = lib().orc_pack2 if fmt == FMT_TERNARY2 else lib().orc_pack1
    fn(_ptr(c, ctypes.c_uint8), n, k, _ptr(out, ctypes.c_uint8))
    return out


def unpack(packed: np.ndarray, k: int, fmt: int) -> np.ndarray:
    """packed bytes -> int8 weight values [n][k] in {-1, 0, +1}."""
    p = _c(packed, np.uint8)
    n = p.shape[0]
    out = np.empty((n, k), dtype=np.int8)
    fn = lib().orc_unpack2 if fmt == FMT_TERNARY2 else lib().orc_unpack1
    fn(_ptr(p, ctypes.c_uint8), n, k, _ptr(out, ctypes.c_int8))
    return out


# --- rotation / quantisation ----------------------------------------------------

def wht128(v: np.ndarray) -> np.ndarray:
    """Normalised 128-point WHT of each 128-row of ``v`` (fp32)."""
    a = _c(v, np.float32).reshape(-1, BLOCK).copy()
    L = lib()
    for row in a:
        L.orc_wht128(_ptr(row, ctypes.c_float))
    return a.reshape(np.shape(v))


def quant_block(v: np.ndarray):
    a = _c(v, np.float32)
    assert a.shape == (BLOCK,)
    q = np.empty(BLOCK, dtype=np.int8)
    s = np.zeros(1, dtype=np.float32)
    lib().orc_quant_block(_ptr(a, ctypes.c_float), _ptr(q, ctypes.c_int8),
                          _ptr(s, ctypes.c_float))
    return q, np.float32(s[0])


def rotate_quant(x_bf16: np.ndarray):
    """x bf16 bits [m][k] -> (q int8 [m][k], s fp32 [m][k/128])."""
    x = _c(x_bf16, np.uint16)
    m, k = x.shape
    q = np.empty((m, k), dtype=np.int8)
    s = np.empty((m, k // BLOCK), dtype=np.float32)
    lib().orc_rotate_quant(_ptr(x, ctypes.c_uint16), m, k, _ptr(q, ctypes.c_int8),
                           _ptr(s, ctypes.c_float))
    return q, s


# --- GEMV -----------------------------------------------------------------------

def blockdots(packed: np.ndarray, fmt: int, n: int, k: int, q: np.ndarray) -> np.ndarray:
    p = _c(packed, np.uint8)
    qq = _c(q, np.int8).reshape(-1, k)
    m = qq.shape[0]
    out = np.empty((m, n, k // BLOCK), dtype=np.int32)
    lib().orc_blockdots(_ptr(p, ctypes.c_uint8), fmt, n, k, _ptr(qq, ctypes.c_int8), m,
                        _ptr(out, ctypes.c_int32))
    return out


def gemv(packed, scales, fmt, n, k, q, s) -> np.ndarray:
    """fp32 outputs [m][n] in the documented fold/reduction order."""
    p = _c(packed, np.uint8)
    sc = _c(scales, np.uint16) if np.asarray(scales).dtype != np.float16 else \
        np.ascontiguousarray(scales).view(np.uint16)
    qq = _c(q, np.int8).reshape(-1, k)
    ss = _c(s, np.float32).reshape(qq.shape[0], k // BLOCK)
    m = qq.shape[0]
    y = np.empty((m, n), dtype=np.float32)
    lib().orc_gemv(_ptr(p, ctypes.c_uint8), _ptr(sc, ctypes.c_uint16), fmt, n, k,
                   _ptr(qq, ctypes.c_int8), _ptr(ss, ctypes.c_float), m,
                   _ptr(y, ctypes.c_float))
    return y


def gemv_f64(packed, scales, fmt, n, k, q, s) -> np.ndarray:
    """The plain definition in fp64 (sequential block order)."""
    p = _c(packed, np.uint8)
    sc = _c(scales, np.uint16) if np.asarray(scales).dtype != np.float16 else \
        np.ascontiguousarray(scales).view(np.uint16)
    qq = _c(q, np.int8).reshape(-1, k)
    ss = _c(s, np.float32).reshape(qq.shape[0], k // BLOCK)
    m = qq.shape[0]
    y = np.empty((m, n), dtype=np.float64)
    lib().orc_gemv_f64(_ptr(p, ctypes.c_uint8), _ptr(sc, ctypes.c_uint16), fmt, n, k,
                       _ptr(qq, ctypes.c_int8), _ptr(ss, ctypes.c_float), m,
                       _ptr(y, ctypes.c_double))
    return y


# --- SiLU -----------------------------------------------------------------------

def expf(x: np.ndarray) -> np.ndarray:
    f = _c(x, np.float32)
    L = lib()
    return np.array([L.orc_expf(float(v)) for v in f.ravel()],
                    dtype=np.float32).reshape(f.shape)


def silu(x: np.ndarray) -> np.ndarray:
    f = _c(x, np.float32)
    L = lib()
    return np.array([L.orc_silu(float(v)) for v in f.ravel()],
                    dtype=np.float32).reshape(f.shape)


def silu_mul_bf16(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    gg = _c(g, np.float32)
    uu = _c(u, np.float32)
    assert gg.shape == uu.shape
    h = np.empty(gg.shape, dtype=np.uint16)
    lib().orc_silu_mul_bf16(_ptr(gg, ctypes.c_float), _ptr(uu, ctypes.c_float), gg.size,
                            _ptr(h, ctypes.c_uint16))
    return h


# --- FFN step / norm / stack ------------------------------------------------------

def _scales_u16(s):
    a = np.asarray(s)
    return np.ascontiguousarray(a).view(np.uint16) if a.dtype == np.float16 else _c(a, np.uint16)


def ffn_step(gate, gate_s, up, up_s, down, down_s, fmt, hidden, inter, x_bf16):
    """One FFN step for m rows.  Returns a dict with every intermediate."""
    x = _c(x_bf16, np.uint16).reshape(-1, hidden)
    m = x.shape[0]
    g_p, u_p, d_p = (_c(a, np.uint8) for a in (gate, up, down))
    g_s, u_s, d_s = (_scales_u16(a) for a in (gate_s, up_s, down_s))
    out = dict(
        y=np.empty((m, hidden), np.float32),
        qx=np.empty((m, hidden), np.int8), sx=np.empty((m, hidden // BLOCK), np.float32),
        g=np.empty((m, inter), np.float32), u=np.empty((m, inter), np.float32),
        h=np.empty((m, inter), np.uint16),
        qh=np.empty((m, inter), np.int8), sh=np.empty((m, inter // BLOCK), np.float32))
    c = ctypes
    lib().orc_ffn_step(_ptr(g_p, c.c_uint8), _ptr(g_s, c.c_uint16), _ptr(u_p, c.c_uint8),
                       _ptr(u_s, c.c_uint16), _ptr(d_p, c.c_uint8), _ptr(d_s, c.c_uint16),
                       fmt, hidden, inter, _ptr(x, c.c_uint16), m, _ptr(out["y"], c.c_float),
                       _ptr(out["qx"], c.c_int8), _ptr(out["sx"], c.c_float),
                       _ptr(out["g"], c.c_float), _ptr(out["u"], c.c_float),
                       _ptr(out["h"], c.c_uint16), _ptr(out["qh"], c.c_int8),
                       _ptr(out["sh"], c.c_float))
    return out


def rmsnorm_bf16(y: np.ndarray, eps: float) -> np.ndarray:
    yy = _c(y, np.float32)
    m, n = yy.shape
    out = np.empty((m, n), np.uint16)
    lib().orc_rmsnorm_bf16(_ptr(yy, ctypes.c_float), m, n, ctypes.c_float(eps),
                           _ptr(out, ctypes.c_uint16))
    return out


def ffn_stack(layers, fmt, hidden, inter, x_bf16, eps):
    """layers: list of (gate, gate_s, up, up_s, down, down_s) packed numpy arrays.
    Layer l's output y_l feeds layer l+1 as rmsnorm_bf16(y_l)."""
    x = _c(x_bf16, np.uint16).reshape(-1, hidden)
    y = None
    for li, (g, gs, u, us, d, ds) in enumerate(layers):
        y = ffn_step(g, gs, u, us, d, ds, fmt, hidden, inter, x)["y"]
        if li + 1 < len(layers):
            x = rmsnorm_bf16(y, eps)
    return y
