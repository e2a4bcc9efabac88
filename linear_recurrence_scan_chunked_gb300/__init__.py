"""Python binding of the GB300 chunked linear-recurrence library (liblrscan.so).

Argument marshalling only: every step of every operation runs in the CUDA
kernels behind the C ABI declared in ``include/lrscan.h``.  PyTorch provides
device memory (output tensors are allocated with ``torch.empty`` when not
given) and the current CUDA stream.  There is no CPU fallback: if the shared
library has not been built, every call raises.

Tensors are CUDA, contiguous, [T, B, D] for sequences, [B, D] for states and
[D] fp32 for per-feature parameters; the storage dtype is float32 or bfloat16.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liblrscan.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "lrscan.h")

LR_F32, LR_BF16 = 0, 1
(LR_OK, LR_ERR_INVALID_ARG, LR_ERR_ALIGN, LR_ERR_CUDA, LR_ERR_TIMEOUT, LR_ERR_NONFINITE,
 LR_ERR_NOT_CONVERGED, LR_ERR_TOO_LARGE) = range(8)

_lib = None


class LrError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"lrscan status {status}: {msg}")
        self.status = status


def build(force: bool = False) -> str:
    # the compiler driver lives in a module of another name: importing a
    # submodule binds it as an attribute of the package, which would replace
    # this function after its first call
    from ._nvcc_build import build as _build
    return _build(force=force)


def load():
    """Load the shared library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                           "(linear_recurrence_scan_chunked_gb300.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.lr_scan_fwd.argtypes = [P, P, P, P, I64, I64, I64, I, P]
    lib.lr_scan_bwd.argtypes = [P] * 7 + [I64, I64, I64, I, P]
    lib.sru_fwd.argtypes = [P] * 9 + [I64, I64, I64, I, P]
    lib.sru_bwd.argtypes = [P] * 16 + [I64, I64, I64, I, P]
    lib.lstm_cell_fwd.argtypes = [P] * 11 + [I64, I64, I64, I, P]
    lib.lstm_cell_bwd.argtypes = [P] * 20 + [I64, I64, I64, I, P]
    lib.deer_diag_solve.argtypes = [P, P, P, P, I64, I64, I64, ctypes.c_float, I, P, P, P, I, P]
    lib.deer_diag_solve_ex.argtypes = [P, P, P, P, P, I64, I64, I64, ctypes.c_float, I, I, P, P,
                                       P, P, P, P, I, P]
    lib.deer_ode_solve.argtypes = [P, P, P, P, P, I64, I64, I64, ctypes.c_float, I, P, P, P, P,
                                   I, P]
    lib.deer_diag_bwd.argtypes = [P] * 7 + [I64, I64, I64, I, P]
    lib.lr_last_error.argtypes = []
    lib.lr_status_str.argtypes = [I]
    lib.lr_status_str.restype = ctypes.c_char_p
    lib.lr_cuda_error_string.restype = ctypes.c_char_p
    lib.lr_workspace_bytes.restype = I64
    lib.lr_test_lookback_timeout.argtypes = [ctypes.c_uint32, P]
    lib.lr_test_activations.argtypes = [P, P, P, P, I64, P]
    lib.lr_test_fail_after_enqueue.argtypes = [P, I64, ctypes.c_float, ctypes.c_uint64, P]
    lib.lr_test_fail_after_enqueue.restype = I
    lib.lr_plan_info.argtypes = [I, I, I, I64, I64, P, P, P, P]
    lib.lr_plan_info.restype = I
    for f in ("lr_scan_fwd", "lr_scan_bwd", "sru_fwd", "sru_bwd", "deer_diag_solve", "deer_diag_bwd",
              "lr_last_error", "lr_test_lookback_timeout", "lr_test_activations"):
        getattr(lib, f).restype = I
    _lib = lib
    return lib


def declared_functions() -> list[str]:
    """Names of the functions declared in include/lrscan.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s*([A-Za-z_]\w*)\s*\(", src, flags=re.M)


def status_str(st: int) -> str:
    return load().lr_status_str(int(st)).decode()


def _check(st: int):
    if st != LR_OK:
        msg = status_str(st)
        if st == LR_ERR_CUDA:
            msg += ": " + load().lr_cuda_error_string().decode()
        raise LrError(st, msg)


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LR_F32
    if t.dtype == torch.bfloat16:
        return LR_BF16
    raise TypeError(f"storage dtype must be float32 or bfloat16, got {t.dtype}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, ref=None):
    """The stream handle for a call on `ref`'s tensors: those tensors must be on
    the current CUDA device (the library launches there) and an explicit
    stream must belong to it."""
    if ref is not None and ref.device.index != torch.cuda.current_device():
        raise ValueError(f"the tensors are on {ref.device} but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}: call under torch.cuda.device({ref.device})")
    s = stream if stream is not None else torch.cuda.current_stream()
    if ref is not None and s.device != ref.device:
        raise ValueError(f"the stream belongs to {s.device}, the tensors to {ref.device}")
    return ctypes.c_void_p(s.cuda_stream)


def _seq(name, t, like=None):
    if t.dim() != 3:
        raise ValueError(f"{name} must be [T, B, D], got shape {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if like is not None and (t.shape != like.shape or t.dtype != like.dtype or t.device != like.device):
        raise ValueError(f"{name} must match shape/dtype/device of the first input")
    return t


def _state(name, t, ref):
    if t is None:
        return None
    T, B, D = ref.shape
    if tuple(t.shape) != (B, D) or t.dtype != ref.dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, D] CUDA tensor of the storage dtype")
    if t.device != ref.device:
        raise ValueError(f"{name} is on {t.device}, the sequence tensors on {ref.device}")
    return t


def _param(name, t, D, ref):
    if t.dtype != torch.float32 or tuple(t.shape) != (D,) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous fp32 [D] CUDA tensor")
    if t.device != ref.device:
        raise ValueError(f"{name} is on {t.device}, the sequence tensors on {ref.device}")
    return t


def lr_scan_fwd(a, b, h0=None, h=None, stream=None):
    """h_t = a_t * h_{t-1} + b_t (h_{-1} = h0). Returns h."""
    _seq("a", a)
    _seq("b", b, a)
    _state("h0", h0, a)
    h = torch.empty_like(a) if h is None else _seq("h", h, a)
    T, B, D = a.shape
    _check(load().lr_scan_fwd(_p(a), _p(b), _p(h0), _p(h), B, T, D, _code(a), _stream(stream, a)))
    return h


def lr_scan_bwd(a, h, dh, h0=None, da=None, db=None, dh0=None, want_dh0=True, stream=None):
    """BPTT of the forward scan. Returns (da, db, dh0 or None)."""
    _seq("a", a)
    _seq("h", h, a)
    _seq("dh", dh, a)
    _state("h0", h0, a)
    T, B, D = a.shape
    da = torch.empty_like(a) if da is None else _seq("da", da, a)
    db = torch.empty_like(a) if db is None else _seq("db", db, a)
    if dh0 is None and want_dh0:
        dh0 = torch.empty((B, D), dtype=a.dtype, device=a.device)
    _state("dh0", dh0, a)
    _check(load().lr_scan_bwd(_p(a), _p(h), _p(h0), _p(dh), _p(da), _p(db), _p(dh0), B, T, D,
                              _code(a), _stream(stream, a)))
    return da, db, dh0


def sru_fwd(xt, uf, ur, x, bf, br, c0=None, h=None, c=None, stream=None):
    """Fused linear-form SRU forward. Returns (h, c)."""
    _seq("xt", xt)
    for n, t in (("uf", uf), ("ur", ur), ("x", x)):
        _seq(n, t, xt)
    T, B, D = xt.shape
    _param("bf", bf, D, xt)
    _param("br", br, D, xt)
    _state("c0", c0, xt)
    h = torch.empty_like(xt) if h is None else _seq("h", h, xt)
    c = torch.empty_like(xt) if c is None else _seq("c", c, xt)
    _check(load().sru_fwd(_p(xt), _p(uf), _p(ur), _p(x), _p(bf), _p(br), _p(c0), _p(h), _p(c),
                          B, T, D, _code(xt), _stream(stream, xt)))
    return h, c


def sru_bwd(xt, uf, ur, x, bf, br, c, dh, c0=None, out=None, want_dc0=True, stream=None):
    """SRU backward. Returns dict dxt, duf, dur, dx, dbf, dbr, dc0."""
    _seq("xt", xt)
    for n, t in (("uf", uf), ("ur", ur), ("x", x), ("c", c), ("dh", dh)):
        _seq(n, t, xt)
    T, B, D = xt.shape
    _param("bf", bf, D, xt)
    _param("br", br, D, xt)
    _state("c0", c0, xt)
    o = dict(out or {})
    for k in ("dxt", "duf", "dur", "dx"):
        o[k] = torch.empty_like(xt) if o.get(k) is None else _seq(k, o[k], xt)
    for k in ("dbf", "dbr"):
        o[k] = torch.empty(D, dtype=torch.float32, device=xt.device) if o.get(k) is None else _param(k, o[k], D, xt)
    if o.get("dc0") is None and want_dc0:
        o["dc0"] = torch.empty((B, D), dtype=xt.dtype, device=xt.device)
    _state("dc0", o.get("dc0"), xt)
    _check(load().sru_bwd(_p(xt), _p(uf), _p(ur), _p(x), _p(bf), _p(br), _p(c0), _p(c), _p(dh),
                          _p(o["dxt"]), _p(o["duf"]), _p(o["dur"]), _p(o["dx"]), _p(o["dbf"]),
                          _p(o["dbr"]), _p(o.get("dc0")), B, T, D, _code(xt), _stream(stream, xt)))
    return o


def lstm_cell_fwd(zf, zi, zc, zo, bf, bi, bc, bo, c0=None, h=None, c=None, stream=None):
    """LSTM cell-state scan with its gates (forget, input, candidate, output
    pre-activations [T, B, D]; biases [D] fp32). Returns (h, c)."""
    _seq("zf", zf)
    for n, t in (("zi", zi), ("zc", zc), ("zo", zo)):
        _seq(n, t, zf)
    T, B, D = zf.shape
    for n, t in (("bf", bf), ("bi", bi), ("bc", bc), ("bo", bo)):
        _param(n, t, D, zf)
    _state("c0", c0, zf)
    h = torch.empty_like(zf) if h is None else _seq("h", h, zf)
    c = torch.empty_like(zf) if c is None else _seq("c", c, zf)
    _check(load().lstm_cell_fwd(_p(zf), _p(zi), _p(zc), _p(zo), _p(bf), _p(bi), _p(bc), _p(bo),
                                _p(c0), _p(h), _p(c), B, T, D, _code(zf), _stream(stream, zf)))
    return h, c


def lstm_cell_bwd(zf, zi, zc, zo, bf, bi, bc, bo, c, dh, c0=None, out=None, want_dc0=True,
                  stream=None):
    """LSTM cell backward. Returns dict dzf, dzi, dzc, dzo, dbf, dbi, dbc, dbo, dc0."""
    _seq("zf", zf)
    for n, t in (("zi", zi), ("zc", zc), ("zo", zo), ("c", c), ("dh", dh)):
        _seq(n, t, zf)
    T, B, D = zf.shape
    for n, t in (("bf", bf), ("bi", bi), ("bc", bc), ("bo", bo)):
        _param(n, t, D, zf)
    _state("c0", c0, zf)
    o = dict(out or {})
    for k in ("dzf", "dzi", "dzc", "dzo"):
        o[k] = torch.empty_like(zf) if o.get(k) is None else _seq(k, o[k], zf)
    for k in ("dbf", "dbi", "dbc", "dbo"):
        o[k] = torch.empty(D, dtype=torch.float32, device=zf.device) if o.get(k) is None else _param(k, o[k], D, zf)
    if o.get("dc0") is None and want_dc0:
        o["dc0"] = torch.empty((B, D), dtype=zf.dtype, device=zf.device)
    _state("dc0", o.get("dc0"), zf)
    _check(load().lstm_cell_bwd(_p(zf), _p(zi), _p(zc), _p(zo), _p(bf), _p(bi), _p(bc), _p(bo),
                                _p(c0), _p(c), _p(dh), _p(o["dzf"]), _p(o["dzi"]), _p(o["dzc"]),
                                _p(o["dzo"]), _p(o["dbf"]), _p(o["dbi"]), _p(o["dbc"]),
                                _p(o["dbo"]), _p(o.get("dc0")), B, T, D, _code(zf),
                                _stream(stream, zf)))
    return o


def deer_diag_solve(w, u, h0=None, y=None, eps=1e-5, kmax=20, stream=None):
    """DEER solve of h_t = tanh(w h_{t-1} + u_t).

    Returns (y, iters, resid, resid_history, status); status is LR_OK,
    LR_ERR_NOT_CONVERGED or LR_ERR_NONFINITE (other statuses raise)."""
    _seq("u", u)
    T, B, D = u.shape
    _param("w", w, D, u)
    _state("h0", h0, u)
    y = torch.empty_like(u) if y is None else _seq("y", y, u)
    iters = ctypes.c_int(0)
    resid = ctypes.c_float(0.0)
    hist = (ctypes.c_float * max(1, int(kmax)))()
    st = load().deer_diag_solve(_p(w), _p(u), _p(h0), _p(y), B, T, D, ctypes.c_float(eps),
                                int(kmax), ctypes.byref(iters), ctypes.byref(resid), hist,
                                _code(u), _stream(stream, u))
    if st not in (LR_OK, LR_ERR_NOT_CONVERGED, LR_ERR_NONFINITE):
        _check(st)
    k = iters.value
    return y, k, resid.value, [hist[i] for i in range(k)], st


def deer_diag_solve_ex(w, u, h0=None, y=None, y_init=None, eps=1e-5, kmax=20,
                       per_sequence=False, stream=None):
    """DEER solve from an initial guess (None = zeros; it may be y itself) with
    one stopping test for the batch or one per sequence.  Returns a dict: y,
    iters (largest K), resid, hist (per iteration), status, seq_iters[B],
    seq_resid[B], launches (kernels the solve enqueued)."""
    _seq("u", u)
    T, B, D = u.shape
    _param("w", w, D, u)
    _state("h0", h0, u)
    if y_init is not None:
        _seq("y_init", y_init, u)
    y = torch.empty_like(u) if y is None else _seq("y", y, u)
    it = ctypes.c_int(0)
    rho = ctypes.c_float(0.0)
    hist = (ctypes.c_float * int(kmax))()
    sk = (ctypes.c_int * max(1, B))()
    sr = (ctypes.c_float * max(1, B))()
    nl = ctypes.c_int(0)
    st = load().deer_diag_solve_ex(_p(w), _p(u), _p(h0), _p(y_init), _p(y), B, T, D,
                                   ctypes.c_float(eps), int(kmax), 1 if per_sequence else 0,
                                   ctypes.byref(it), ctypes.byref(rho), hist, sk, sr,
                                   ctypes.byref(nl), _code(u), _stream(stream, u))
    if st not in (LR_OK, LR_ERR_NOT_CONVERGED, LR_ERR_NONFINITE):
        _check(st)
    k = int(it.value)
    return {"y": y, "iters": k, "resid": float(rho.value), "hist": list(hist)[:k], "status": int(st),
            "seq_iters": list(sk)[:B], "seq_resid": list(sr)[:B], "launches": int(nl.value)}


def deer_ode_solve(w, u, dt, h0=None, y=None, eps=1e-5, kmax=20, stream=None):
    """DEER in the ODE form (dy/dt = -y + tanh(w y + u) on steps dt[T], G
    clamped to [-10, 10]).  Returns (y, iters, resid, resid_history, status,
    clamps of the last iteration)."""
    _seq("u", u)
    T, B, D = u.shape
    _param("w", w, D, u)
    _param("dt", dt, T, u)
    _state("h0", h0, u)
    y = torch.empty_like(u) if y is None else _seq("y", y, u)
    iters = ctypes.c_int(0)
    resid = ctypes.c_float(0.0)
    clamps = ctypes.c_int64(0)
    hist = (ctypes.c_float * max(1, int(kmax)))()
    st = load().deer_ode_solve(_p(w), _p(u), _p(dt), _p(h0), _p(y), B, T, D, ctypes.c_float(eps),
                               int(kmax), ctypes.byref(iters), ctypes.byref(resid), hist,
                               ctypes.byref(clamps), _code(u), _stream(stream, u))
    if st not in (LR_OK, LR_ERR_NOT_CONVERGED, LR_ERR_NONFINITE):
        _check(st)
    k = iters.value
    return y, k, resid.value, [hist[i] for i in range(k)], st, int(clamps.value)


def deer_diag_bwd(w, y, dy, h0=None, du=None, dw=None, dh0=None, want_dh0=True, stream=None):
    """Gradient through the DEER solution y for the upstream dy = dL/dy.
    Returns (du, dw, dh0 or None)."""
    _seq("y", y)
    _seq("dy", dy, y)
    T, B, D = y.shape
    _param("w", w, D, y)
    _state("h0", h0, y)
    du = torch.empty_like(y) if du is None else _seq("du", du, y)
    dw = torch.empty(D, dtype=torch.float32, device=y.device) if dw is None else _param("dw", dw, D, y)
    if dh0 is None and want_dh0:
        dh0 = torch.empty((B, D), dtype=y.dtype, device=y.device)
    _state("dh0", dh0, y)
    _check(load().deer_diag_bwd(_p(w), _p(y), _p(h0), _p(dy), _p(du), _p(dw), _p(dh0), B, T, D,
                                _code(y), _stream(stream, y)))
    return du, dw, dh0


def last_error() -> int:
    """Reads and clears the device error word (synchronises the device)."""
    return int(load().lr_last_error())


def workspace_bytes() -> int:
    return int(load().lr_workspace_bytes())


# lr_op and lr_protocol of the header
OPS = ("scan_fwd", "scan_bwd", "sru_fwd", "sru_bwd", "deer", "deer_bwd", "lstm_fwd", "lstm_bwd",
       "deer_ode")
PROTOCOLS = ("chain", "walk", "look", "cluster")


def plan_info(op: str, dtype: str, vec: bool, T: int, C: int) -> dict:
    """The carry protocol a call of `op` plans for T steps and C = B*D
    channels (lr_plan_info; host only, no device): {"protocol", "tma",
    "tile_rows", "n_chunks"}.  Raises ValueError on an argument error."""
    lib = load()
    proto, tma = ctypes.c_int(-1), ctypes.c_int(-1)
    rows, nch = ctypes.c_int64(-1), ctypes.c_int64(-1)
    if dtype not in ("f32", "bf16"):
        raise ValueError(f"dtype must be 'f32' or 'bf16', got {dtype!r}")
    st = lib.lr_plan_info(OPS.index(op), LR_F32 if dtype == "f32" else LR_BF16, 1 if vec else 0, int(T), int(C),
                          ctypes.byref(proto), ctypes.byref(tma), ctypes.byref(rows),
                          ctypes.byref(nch))
    if st != LR_OK:
        raise ValueError(f"lr_plan_info: {status_str(st)}")
    return {"protocol": PROTOCOLS[proto.value], "tma": bool(tma.value), "tile_rows": rows.value,
            "n_chunks": nch.value}


def test_activations(x, stream=None, with_expm1=False):
    """tanh and sigmoid (and e^x - 1) of a contiguous fp32 CUDA tensor as the
    fused kernels evaluate them. Returns (tanh, sigmoid) or (tanh, sigmoid,
    expm1)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 CUDA tensor")
    th, sg = torch.empty_like(x), torch.empty_like(x)
    em = torch.empty_like(x) if with_expm1 else None
    _check(load().lr_test_activations(_p(x), _p(th), _p(sg), _p(em), x.numel(), _stream(stream, x)))
    return (th, sg, em) if with_expm1 else (th, sg)


def test_lookback_timeout(spin_limit: int = 1000, stream=None) -> int:
    """Runs the bounded-wait test launch; returns its enqueue status."""
    return int(load().lr_test_lookback_timeout(ctypes.c_uint32(spin_limit), _stream(stream)))


def test_fail_after_enqueue(x, value: float, sleep_ns: int, stream=None) -> int:
    """Enqueues a kernel that sleeps ~sleep_ns and then fills the fp32 CUDA
    tensor x with `value`, and returns the LR_ERR_CUDA of a call whose later
    launch failed (the call-ordering test after an error)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 CUDA tensor")
    return int(load().lr_test_fail_after_enqueue(_p(x), x.numel(), ctypes.c_float(value),
                                                  ctypes.c_uint64(sleep_ns), _stream(stream, x)))
