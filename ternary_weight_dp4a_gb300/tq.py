"""ctypes binding of libtq (include/tq.h).  Argument marshalling only.

Every function takes torch CUDA tensors (PyTorch provides device memory and
streams), passes raw device pointers to the C ABI and raises ``TQError`` on a
non-OK status.  Work is enqueued on the current torch CUDA stream unless a
``stream`` is given.  There is no CPU path: if ``libtq.so`` has not been built
(``python -m ternary_weight_dp4a_gb300.build``), the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtq.so")

FMT_TERNARY2 = 0
FMT_BINARY1 = 1
ENGINE_AUTO, ENGINE_DP4A, ENGINE_TCGEN05 = 0, 1, 2
TQ_ERR_TIMEOUT = 6
BLOCK = 128
MAX_ROWS = 64

# every entry point include/tq.h and include/tq_lifecycle.h declare
EXPORTS = ("tq_status_string", "tq_last_cuda_error", "tq_set_engine", "tq_get_engine",
           "tq_error_status", "tq_read_error_word", "tq_workspace_init", "tq_pack_weights",
           "tq_rotate_quant", "tq_gemv_workspace_bytes", "tq_gemv", "tq_ffn_gateup",
           "tq_ffn_workspace_bytes", "tq_ffn_workspace_error_offset", "tq_ffn_workspace_init",
           "tq_ffn_step", "tq_ffn_stage_input", "tq_ffn_stage_gateup", "tq_ffn_stage_down",
           "tq_ffn_stack", "tq_ffn_static_workspace_bytes", "tq_ffn_step_static",
           "tq_rmsnorm_bf16",
           "tq_lifecycle_init", "tq_lifecycle_load", "tq_lifecycle_copy", "tq_lifecycle_alloc",
           "tq_lifecycle_free", "tq_lifecycle_poll", "tq_lifecycle_release", "tq_lifecycle_destroy")

_lock = threading.Lock()
_lib = None


class TQError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = load().tq_status_string(status).decode()
        extra = f" (cudaError {cuda_error})" if status == 5 else ""
        super().__init__(f"{fn}: {name}{extra}")


class _Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("n", ctypes.c_int32), ("k", ctypes.c_int32), ("fmt", ctypes.c_int32)]


# tq_lifecycle.h
_LC_ALLOC = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32)
_LC_RELEASE = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32)
_LC_FREE_BYTES = ctypes.CFUNCTYPE(ctypes.c_size_t, ctypes.c_void_p)
_LC_BUILD = ctypes.CFUNCTYPE(ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t)


class _LcHooks(ctypes.Structure):
    _fields_ = [("alloc", _LC_ALLOC), ("release", _LC_RELEASE), ("free_bytes", _LC_FREE_BYTES),
                ("build", _LC_BUILD), ("ctx", ctypes.c_void_p)]


class _LcConfig(ctypes.Structure):
    _fields_ = [("copy_bytes", ctypes.c_size_t), ("reserve_bytes", ctypes.c_size_t),
                ("rebuild_margin", ctypes.c_size_t), ("rebuild_after", ctypes.c_int32)]


class _Lifecycle(ctypes.Structure):
    _fields_ = [("cfg", _LcConfig), ("hooks", _LcHooks), ("copy", ctypes.c_void_p),
                ("state", ctypes.c_int32), ("polls_since_change", ctypes.c_int32),
                ("builds", ctypes.c_int64), ("rebuilds", ctypes.c_int64), ("releases", ctypes.c_int64),
                ("alloc_failures", ctypes.c_int64), ("retries_ok", ctypes.c_int64),
                ("build_failures", ctypes.c_int64)]


def load():
    """Load libtq.so (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libtq.so not found at {LIB_PATH}: build it with "
                    "`python -m ternary_weight_dp4a_gb300.build` (needs nvcc); "
                    "there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
            W = ctypes.POINTER(_Weight)
            L.tq_status_string.argtypes = [ctypes.c_int]
            L.tq_status_string.restype = ctypes.c_char_p
            L.tq_last_cuda_error.restype = ctypes.c_int
            L.tq_pack_weights.argtypes = [vp, i32, i32, i32, vp, vp]
            L.tq_rotate_quant.argtypes = [vp, i32, i32, vp, vp, vp]
            L.tq_set_engine.argtypes = [i32]
            L.tq_get_engine.argtypes = []
            L.tq_error_status.argtypes = [ctypes.c_uint32]
            L.tq_read_error_word.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
            L.tq_workspace_init.argtypes = [vp, sz, vp]
            L.tq_gemv_workspace_bytes.argtypes = [i32, i32, i32]
            L.tq_gemv_workspace_bytes.restype = sz
            L.tq_gemv.argtypes = [W, vp, vp, i32, vp, vp, vp, sz, vp]
            L.tq_ffn_gateup.argtypes = [W, W, vp, vp, i32, vp, vp, sz, vp]
            L.tq_ffn_workspace_bytes.argtypes = [i32, i32, i32]
            L.tq_ffn_workspace_bytes.restype = sz
            L.tq_ffn_workspace_error_offset.argtypes = [i32, i32, i32]
            L.tq_ffn_workspace_error_offset.restype = sz
            L.tq_ffn_workspace_init.argtypes = [vp, sz, vp]
            L.tq_ffn_step.argtypes = [W, W, W, vp, i32, vp, vp, sz, vp]
            L.tq_ffn_stage_input.argtypes = [vp, i32, i32, i32, vp, sz, vp]
            L.tq_ffn_stage_gateup.argtypes = [W, W, i32, vp, sz, vp]
            L.tq_ffn_stage_down.argtypes = [W, i32, vp, vp, sz, vp]
            L.tq_ffn_stack.argtypes = [W, i32, vp, i32, f32, vp, vp, sz, vp]
            L.tq_rmsnorm_bf16.argtypes = [vp, i32, i32, f32, vp, vp]
            L.tq_ffn_static_workspace_bytes.argtypes = []
            L.tq_ffn_static_workspace_bytes.restype = sz
            L.tq_ffn_step_static.argtypes = [W, W, W, vp, i32, vp, vp]
            LC = ctypes.POINTER(_Lifecycle)
            L.tq_lifecycle_init.argtypes = [LC, ctypes.POINTER(_LcConfig), ctypes.POINTER(_LcHooks)]
            L.tq_lifecycle_load.argtypes = [LC]
            L.tq_lifecycle_copy.argtypes = [LC]
            L.tq_lifecycle_copy.restype = vp
            L.tq_lifecycle_alloc.argtypes = [LC, sz, i32]
            L.tq_lifecycle_alloc.restype = vp
            L.tq_lifecycle_free.argtypes = [LC, vp, sz, i32]
            L.tq_lifecycle_free.restype = None
            L.tq_lifecycle_poll.argtypes = [LC]
            L.tq_lifecycle_release.argtypes = [LC]
            L.tq_lifecycle_release.restype = None
            L.tq_lifecycle_destroy.argtypes = [LC]
            L.tq_lifecycle_destroy.restype = None
            for name in EXPORTS:
                if name not in ("tq_status_string", "tq_last_cuda_error", "tq_ffn_workspace_bytes",
                                "tq_gemv_workspace_bytes",
                                "tq_ffn_workspace_error_offset", "tq_ffn_static_workspace_bytes", "tq_lifecycle_copy", "tq_lifecycle_alloc",
                                "tq_lifecycle_free", "tq_lifecycle_release", "tq_lifecycle_destroy"):
                    getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise TQError(fn, status, load().tq_last_cuda_error())


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


@dataclass
class PackedWeight:
    """A packed weight matrix on the device: codes [n][k/4] (2-bit) or
    [n][k/8] (1-bit) uint8, scales [n][k/128] float16."""
    codes: "object"
    scales: "object"
    n: int
    k: int
    fmt: int

    def c_struct(self) -> _Weight:
        return _Weight(self.codes.data_ptr(), self.scales.data_ptr(), self.n, self.k, self.fmt)

    @property
    def nbytes(self) -> int:
        return self.codes.numel() + 2 * self.scales.numel()


def pack_weights(codes, fmt: int, scales, stream=None) -> PackedWeight:
    """codes: uint8 CUDA tensor [n][k]; scales: float16 CUDA tensor [n][k/128]."""
    import torch
    n, k = codes.shape
    per = 4 if fmt == FMT_TERNARY2 else 8
    packed = torch.empty((n, k // per), dtype=torch.uint8, device=codes.device)
    _check("tq_pack_weights", load().tq_pack_weights(_ptr(codes), n, k, fmt, _ptr(packed),
                                                      _stream(stream)))
    return PackedWeight(packed, scales.contiguous(), n, k, fmt)


def rotate_quant(x, q=None, s=None, stream=None):
    """x: bf16 CUDA tensor [m][k] -> (q int8 [m][k], s float32 [m][k/128])."""
    import torch
    m, k = x.shape
    if q is None:
        q = torch.empty((m, k), dtype=torch.int8, device=x.device)
    if s is None:
        s = torch.empty((m, k // BLOCK), dtype=torch.float32, device=x.device)
    _check("tq_rotate_quant", load().tq_rotate_quant(_ptr(x), m, k, _ptr(q), _ptr(s),
                                                      _stream(stream)))
    return q, s


def set_engine(engine: int) -> None:
    """Process-wide kernel choice: ENGINE_AUTO, ENGINE_DP4A or ENGINE_TCGEN05."""
    _check("tq_set_engine", load().tq_set_engine(engine))


def get_engine() -> int:
    return int(load().tq_get_engine())


def read_error_word(word_tensor, stream=None) -> int:
    """Read a workspace's error word (a 4-byte slice of the workspace tensor)
    through tq_read_error_word: synchronises the stream; raises TQError with
    status TQ_ERR_TIMEOUT when the word is not zero, else returns 0."""
    v = ctypes.c_uint32(0)
    st = load().tq_read_error_word(_ptr(word_tensor), ctypes.byref(v), _stream(stream))
    _check("tq_read_error_word", st)
    return int(v.value)


def gemv_workspace_bytes(m: int, n: int, k: int) -> int:
    return int(load().tq_gemv_workspace_bytes(m, n, k))


def gemv_workspace(m: int, n: int, k: int, device="cuda"):
    """A zero-filled GEMV workspace (its first 4 bytes are the error word)."""
    import torch
    return torch.zeros(gemv_workspace_bytes(m, n, k), dtype=torch.uint8, device=device)


def gemv(w: PackedWeight, q, s, y=None, blockdots: bool = False, workspace=None, stream=None):
    """y[m][n] (float32); with ``blockdots`` also the int32 [m][n][k/128] dots."""
    import torch
    m = q.shape[0]
    if y is None:
        y = torch.empty((m, w.n), dtype=torch.float32, device=q.device)
    d = torch.empty((m, w.n, w.k // BLOCK), dtype=torch.int32, device=q.device) \
        if blockdots else None
    if workspace is None:
        workspace = gemv_workspace(m, w.n, w.k, q.device)
    ws = w.c_struct()
    _check("tq_gemv", load().tq_gemv(ctypes.byref(ws), _ptr(q), _ptr(s), m, _ptr(y), _ptr(d),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))
    return (y, d) if blockdots else y


def ffn_gateup(gate: PackedWeight, up: PackedWeight, qx, sx, h=None, workspace=None, stream=None):
    """Fused gate/up GEMVs + SiLU(g)*u: qx int8 [m][hidden] -> h bf16 [m][inter]."""
    import torch
    m = qx.shape[0]
    if h is None:
        h = torch.empty((m, gate.n), dtype=torch.bfloat16, device=qx.device)
    if workspace is None:
        workspace = ffn_workspace(m, gate.k, gate.n, qx.device)
    g, u = gate.c_struct(), up.c_struct()
    _check("tq_ffn_gateup", load().tq_ffn_gateup(ctypes.byref(g), ctypes.byref(u), _ptr(qx),
                                                 _ptr(sx), m, _ptr(h), _ptr(workspace),
                                                 workspace.numel(), _stream(stream)))
    return h


def ffn_workspace_bytes(m: int, hidden: int, inter: int) -> int:
    return int(load().tq_ffn_workspace_bytes(m, hidden, inter))


def ffn_workspace(m: int, hidden: int, inter: int, device="cuda"):
    """A zero-filled FFN workspace (zero is the state tq_ffn_workspace_init sets)."""
    import torch
    return torch.zeros(ffn_workspace_bytes(m, hidden, inter), dtype=torch.uint8, device=device)


def ffn_workspace_init(workspace, stream=None):
    _check("tq_ffn_workspace_init", load().tq_ffn_workspace_init(
        _ptr(workspace), workspace.numel(), _stream(stream)))


def ffn_workspace_error(workspace, m: int, hidden: int, inter: int) -> int:
    """The workspace's error word (bits of the waits that ran out; see
    tq_ffn_workspace_error_offset).  Reads 4 bytes back, so it synchronises."""
    off = load().tq_ffn_workspace_error_offset(m, hidden, inter)
    return int(workspace[off:off + 4].cpu().numpy().view("<u4")[0])


def ffn_stage_input(x, inter: int, workspace, stream=None):
    m, hidden = x.shape
    _check("tq_ffn_stage_input", load().tq_ffn_stage_input(
        _ptr(x), m, hidden, inter, _ptr(workspace), workspace.numel(), _stream(stream)))


def ffn_stage_gateup(gate: PackedWeight, up: PackedWeight, m: int, workspace, stream=None):
    g, u = gate.c_struct(), up.c_struct()
    _check("tq_ffn_stage_gateup", load().tq_ffn_stage_gateup(
        ctypes.byref(g), ctypes.byref(u), m, _ptr(workspace), workspace.numel(), _stream(stream)))


def ffn_stage_down(down: PackedWeight, m: int, y, workspace, stream=None):
    d = down.c_struct()
    _check("tq_ffn_stage_down", load().tq_ffn_stage_down(
        ctypes.byref(d), m, _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)))


def ffn_stack(layers, x, eps: float = 1e-6, y=None, workspace=None, stream=None):
    """layers: list of (gate, up, down) PackedWeight; x bf16 [m][hidden] ->
    the last layer's y float32 [m][hidden]."""
    import torch
    m, hidden = x.shape
    inter = layers[0][0].n
    if y is None:
        y = torch.empty((m, hidden), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = ffn_workspace(m, hidden, inter, x.device)
    arr = (_Weight * (3 * len(layers)))(*[w.c_struct() for layer in layers for w in layer])
    _check("tq_ffn_stack", load().tq_ffn_stack(arr, len(layers), _ptr(x), m, eps, _ptr(y),
                                               _ptr(workspace), workspace.numel(),
                                               _stream(stream)))
    return y


def ffn_step(gate: PackedWeight, up: PackedWeight, down: PackedWeight, x, y=None,
             workspace=None, stream=None):
    """x: bf16 CUDA tensor [m][hidden] -> y float32 [m][hidden]."""
    import torch
    m, hidden = x.shape
    if y is None:
        y = torch.empty((m, hidden), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = ffn_workspace(m, hidden, gate.n, x.device)
    g, u, d = gate.c_struct(), up.c_struct(), down.c_struct()
    _check("tq_ffn_step", load().tq_ffn_step(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d),
                                             _ptr(x), m, _ptr(y), _ptr(workspace),
                                             workspace.numel(), _stream(stream)))
    return y


def ffn_step_static(gate: PackedWeight, up: PackedWeight, down: PackedWeight, x, y=None,
                    stream=None):
    """The FFN step with the library's built-in scratch (no workspace argument;
    see tq_ffn_step_static in include/tq.h for who needs it and its limits)."""
    import torch
    m, hidden = x.shape
    if y is None:
        y = torch.empty((m, hidden), dtype=torch.float32, device=x.device)
    g, u, d = gate.c_struct(), up.c_struct(), down.c_struct()
    _check("tq_ffn_step_static", load().tq_ffn_step_static(
        ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), _ptr(x), m, _ptr(y), _stream(stream)))
    return y


def rmsnorm_bf16(y, eps: float = 1e-6, x_out=None, stream=None):
    """y float32 [m][n] -> bf16 [m][n]."""
    import torch
    m, n = y.shape
    if x_out is None:
        x_out = torch.empty((m, n), dtype=torch.bfloat16, device=y.device)
    _check("tq_rmsnorm_bf16", load().tq_rmsnorm_bf16(_ptr(y), m, n, eps, _ptr(x_out),
                                                     _stream(stream)))
    return x_out


# ---------------------------------------------------------------------------
# lifecycle of the ternary weight copy (include/tq_lifecycle.h)
# ---------------------------------------------------------------------------

class CopyLifecycle:
    """The host-side policy of include/tq_lifecycle.h around a caller's hooks.

    ``hooks`` has ``alloc(nbytes, purpose) -> address or 0``,
    ``release(address, nbytes, purpose)``, ``free_bytes() -> int`` and
    ``build(address, nbytes) -> bool``; the policy itself runs in libtq.
    A hook that raises counts as a failure (alloc/build) or as 0 free bytes.
    """

    STATES = ("absent", "resident", "skipped", "released", "failed")
    COPY, OTHER = 0, 1

    def __init__(self, copy_bytes: int, reserve_bytes: int, hooks, rebuild_margin: int = 0,
                 rebuild_after: int = 0):
        L = load()

        def _alloc(_ctx, nbytes, purpose):
            try:
                return hooks.alloc(int(nbytes), int(purpose)) or None
            except Exception:
                return None

        def _release(_ctx, ptr, nbytes, purpose):
            try:
                hooks.release(int(ptr or 0), int(nbytes), int(purpose))
            except Exception:
                pass

        def _free_bytes(_ctx):
            try:
                return max(0, int(hooks.free_bytes()))
            except Exception:
                return 0

        def _build(_ctx, ptr, nbytes):
            try:
                return 0 if hooks.build(int(ptr or 0), int(nbytes)) else 1
            except Exception:
                return 1

        # the callbacks must outlive the struct that points at them
        self._cbs = (_LC_ALLOC(_alloc), _LC_RELEASE(_release), _LC_FREE_BYTES(_free_bytes),
                     _LC_BUILD(_build))
        self._hooks = _LcHooks(*self._cbs, None)
        self._cfg = _LcConfig(copy_bytes, reserve_bytes, rebuild_margin, rebuild_after)
        self._lc = _Lifecycle()
        _check("tq_lifecycle_init",
               L.tq_lifecycle_init(ctypes.byref(self._lc), ctypes.byref(self._cfg),
                                   ctypes.byref(self._hooks)))

    def load(self) -> str:
        _check("tq_lifecycle_load", load().tq_lifecycle_load(ctypes.byref(self._lc)))
        return self.state

    @property
    def copy(self):
        """Address of the resident copy, or None."""
        return load().tq_lifecycle_copy(ctypes.byref(self._lc))

    def alloc(self, nbytes: int, purpose: int = OTHER):
        """Memory for other work; releases the copy and retries once on failure."""
        return load().tq_lifecycle_alloc(ctypes.byref(self._lc), nbytes, purpose)

    def free(self, ptr, nbytes: int, purpose: int = OTHER) -> None:
        load().tq_lifecycle_free(ctypes.byref(self._lc), ptr, nbytes, purpose)

    def poll(self) -> str:
        _check("tq_lifecycle_poll", load().tq_lifecycle_poll(ctypes.byref(self._lc)))
        return self.state

    def release(self) -> None:
        load().tq_lifecycle_release(ctypes.byref(self._lc))

    def destroy(self) -> None:
        load().tq_lifecycle_destroy(ctypes.byref(self._lc))

    @property
    def state(self) -> str:
        return self.STATES[self._lc.state]

    def counters(self) -> dict:
        return {k: int(getattr(self._lc, k)) for k in
                ("builds", "rebuilds", "releases", "alloc_failures", "retries_ok", "build_failures")}


class TorchDeviceHooks:
    """Lifecycle hooks over PyTorch's CUDA allocator.  ``build_fn(tensor)``
    fills a uint8 tensor of the copy's size (e.g. packs weights into it) and
    returns True on success.  Free memory counts the driver's free bytes plus
    what PyTorch holds cached but unused."""

    def __init__(self, build_fn, device="cuda"):
        self.build_fn = build_fn
        self.device = device
        self._live = {}

    def alloc(self, nbytes, purpose):
        import torch
        try:
            t = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        except torch.cuda.OutOfMemoryError:
            return 0
        self._live[t.data_ptr()] = t
        return t.data_ptr()

    def release(self, ptr, nbytes, purpose):
        self._live.pop(ptr, None)

    def free_bytes(self):
        import torch
        free, _total = torch.cuda.mem_get_info(self.device)
        return free + torch.cuda.memory_reserved(self.device) - torch.cuda.memory_allocated(self.device)

    def build(self, ptr, nbytes):
        return bool(self.build_fn(self._live[ptr]))

    def tensor(self, ptr):
        """The tensor behind an address alloc returned (None once released)."""
        return self._live.get(ptr)
