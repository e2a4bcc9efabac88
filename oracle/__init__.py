"""fp64 CPU oracle for the linear-recurrence hot path -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it.  The arithmetic lives in ``lr_oracle.c`` (plain C,
fp64, sequential in time); this module only compiles it with gcc, loads it with
ctypes and converts numpy arrays to contiguous fp64.

Every function here follows the pages cited in ``lr_oracle.c``:
  scan_fwd / scan_bwd  -- the diagonal linear recurrence and its BPTT gradient
  sru_fwd / sru_bwd    -- the linear-form SRU layer and its gradient
  lstm_fwd / lstm_bwd  -- the LSTM cell-state scan with its gates, and its gradient
  deer / deer_step     -- DEER Newton iteration on a diagonal tanh RNN (from a
                          given initial guess or zeros)
  deer_per_sequence    -- the same with each batch sequence stopping on its own
  deer_ode / deer_ode_step / rollout_ode -- DEER's ODE form (exp(-G dt)
                          coefficients, G clamped) and its exponential-Euler
                          fixed point
  rollout_tanh         -- the direct sequential tanh RNN
Each is pinned by tests in ``tests/test_oracle_pins.py`` against closed forms,
library linear solves, finite differences and brute-force evaluation orders.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lr_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liblroracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts give the same
# bits; -O2 keeps IEEE semantics (no -ffast-math).
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile lr_oracle.c into a shared library (idempotent)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.lro_scan_fwd.argtypes = [I64, I64, P, P, P, P]
        lib.lro_scan_bwd.argtypes = [I64, I64, P, P, P, P, P, P, P]
        lib.lro_sru_fwd.argtypes = [I64, I64, I64] + [P] * 9
        lib.lro_sru_bwd.argtypes = [I64, I64, I64] + [P] * 15
        lib.lro_sru_bwd.restype = ctypes.c_int
        lib.lro_lstm_fwd.argtypes = [I64, I64, I64] + [P] * 11
        lib.lro_lstm_bwd.argtypes = [I64, I64, I64] + [P] * 20
        lib.lro_lstm_bwd.restype = ctypes.c_int
        lib.lro_rollout_tanh.argtypes = [I64, I64, I64, P, P, P, P]
        lib.lro_deer_step.argtypes = [I64, I64, I64, P, P, P, P, P, P]
        lib.lro_deer.argtypes = [I64, I64, I64, P, P, P, P, ctypes.c_double, ctypes.c_int, P, P, P]
        lib.lro_deer_bwd.argtypes = [I64, I64, I64] + [P] * 7
        lib.lro_deer_bwd.restype = ctypes.c_int
        lib.lro_rollout_ode.argtypes = [I64, I64, I64] + [P] * 6
        lib.lro_deer_ode_step.argtypes = [I64, I64, I64] + [P] * 8
        lib.lro_deer_ode.argtypes = [I64, I64, I64, P, P, P, P, ctypes.c_double, ctypes.c_int,
                                     P, P, P, P]
        lib.lro_deer_ode.restype = ctypes.c_int
        lib.lro_deer.restype = ctypes.c_int
        lib.lro_num_threads.restype = ctypes.c_int
        lib.lro_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def set_num_threads(n: int) -> None:
    """0 = OpenMP default (all cores)."""
    _load().lro_set_num_threads(int(n))


def num_threads() -> int:
    return int(_load().lro_num_threads())


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _tc(x):
    """[T, B, D] or [T, C] -> (T, C)."""
    T = x.shape[0]
    return T, int(np.prod(x.shape[1:])) if x.ndim > 1 else 1


def _shapes(ref, seqs=(), feats=(), states=(), steps=()):
    """(T, C) of sequence tensor `ref`, after checking the shapes the C code
    trusts: every other sequence tensor shaped like ref, the per-feature
    arrays one length D dividing C, the initial states C values, the
    per-step arrays T values (None = absent)."""
    T, C = _tc(ref)
    for x in seqs:
        if x is not None and x.shape != ref.shape:
            raise ValueError(f"sequence tensor of shape {x.shape}, expected {ref.shape}")
    lens = {x.size for x in feats}
    if feats and (len(lens) != 1 or any(x.ndim != 1 for x in feats)):
        raise ValueError("per-feature arrays must be 1-D and of one length")
    if feats and C and (next(iter(lens)) == 0 or C % next(iter(lens))):
        raise ValueError(f"per-feature length {next(iter(lens))} does not divide {C} channels")
    for x in states:
        if x is not None and x.size != C:
            raise ValueError(f"initial state of {x.size} values, expected {C}")
    for x in steps:
        if x.shape != (T,):
            raise ValueError(f"per-step array of shape {x.shape}, expected ({T},)")
    return T, C


def scan_fwd(a, b, h0=None):
    """h_t = a_t h_{t-1} + b_t along axis 0; returns fp64 h shaped like a."""
    a, b, h0 = _f64(a), _f64(b), _f64(h0)
    T, C = _shapes(a, seqs=(b,), states=(h0,))
    h = np.empty_like(a)
    _load().lro_scan_fwd(T, C, _p(a), _p(b), _p(h0), _p(h))
    return h


def scan_bwd(a, h, g, h0=None):
    """Returns (da, db, dh0) for loss sum(g * h), given the forward h."""
    a, h, g, h0 = _f64(a), _f64(h), _f64(g), _f64(h0)
    T, C = _shapes(a, seqs=(h, g), states=(h0,))
    da, db = np.empty_like(a), np.empty_like(a)
    dh0 = np.empty(a.shape[1:], dtype=np.float64)
    _load().lro_scan_bwd(T, C, _p(a), _p(h), _p(h0), _p(g), _p(da), _p(db), _p(dh0))
    return da, db, dh0


def sru_fwd(xt, uf, ur, x, bf, br, c0=None):
    """Returns (h, c). Sequence tensors [T, B, D]; bf, br [D]."""
    xt, uf, ur, x, bf, br, c0 = map(_f64, (xt, uf, ur, x, bf, br, c0))
    T, C = _shapes(xt, seqs=(uf, ur, x), feats=(bf, br), states=(c0,))
    D = bf.shape[0]
    h, c = np.empty_like(xt), np.empty_like(xt)
    _load().lro_sru_fwd(T, C, D, *map(_p, (xt, uf, ur, x, bf, br, c0, h, c)))
    return h, c


def sru_bwd(xt, uf, ur, x, bf, br, c, dh, c0=None):
    """Returns (dxt, duf, dur, dx, dbf, dbr, dc0) given the forward c."""
    xt, uf, ur, x, bf, br, c, dh, c0 = map(_f64, (xt, uf, ur, x, bf, br, c, dh, c0))
    T, C = _shapes(xt, seqs=(uf, ur, x, c, dh), feats=(bf, br), states=(c0,))
    D = bf.shape[0]
    dxt, duf, dur, dx = (np.empty_like(xt) for _ in range(4))
    dbf, dbr = np.empty(D), np.empty(D)
    dc0 = np.empty(xt.shape[1:], dtype=np.float64)
    st = _load().lro_sru_bwd(T, C, D, *map(_p, (xt, uf, ur, x, bf, br, c0, c, dh,
                                                 dxt, duf, dur, dx, dbf, dbr, dc0)))
    if st != 0:
        raise MemoryError("oracle sru_bwd: allocation failed")
    return dxt, duf, dur, dx, dbf, dbr, dc0


def lstm_fwd(zf, zi, zc, zo, bf, bi, bc, bo, c0=None):
    """LSTM cell-state scan with its gates; returns (h, c).  Pre-activations
    [T, B, D]; biases [D]; c0 [B, D] (None = zeros)."""
    zf, zi, zc, zo, bf, bi, bc, bo, c0 = map(_f64, (zf, zi, zc, zo, bf, bi, bc, bo, c0))
    T, C = _shapes(zf, seqs=(zi, zc, zo), feats=(bf, bi, bc, bo), states=(c0,))
    D = bf.shape[0]
    h, c = np.empty_like(zf), np.empty_like(zf)
    _load().lro_lstm_fwd(T, C, D, *map(_p, (zf, zi, zc, zo, bf, bi, bc, bo, c0, h, c)))
    return h, c


def lstm_bwd(zf, zi, zc, zo, bf, bi, bc, bo, c, dh, c0=None):
    """Gradient of sum(dh * h) for lstm_fwd given its cell states c.
    Returns (dzf, dzi, dzc, dzo, dbf, dbi, dbc, dbo, dc0)."""
    zf, zi, zc, zo, bf, bi, bc, bo, c, dh, c0 = map(
        _f64, (zf, zi, zc, zo, bf, bi, bc, bo, c, dh, c0))
    T, C = _shapes(zf, seqs=(zi, zc, zo, c, dh), feats=(bf, bi, bc, bo), states=(c0,))
    D = bf.shape[0]
    dz = [np.empty_like(zf) for _ in range(4)]
    db = [np.empty(D) for _ in range(4)]
    dc0 = np.empty(zf.shape[1:]) if zf.ndim == 3 else np.empty(C)
    st = _load().lro_lstm_bwd(T, C, D, *map(_p, (zf, zi, zc, zo, bf, bi, bc, bo, c0, c, dh,
                                                 *dz, *db, dc0)))
    if st < 0:
        raise MemoryError("oracle lstm_bwd: allocation failed")
    return (*dz, *db, dc0)


def rollout_tanh(w, u, h0=None):
    """Direct sequential h_t = tanh(w h_{t-1} + u_t)."""
    w, u, h0 = _f64(w), _f64(u), _f64(h0)
    T, C = _shapes(u, feats=(w,), states=(h0,))
    y = np.empty_like(u)
    _load().lro_rollout_tanh(T, C, w.shape[0], _p(w), _p(u), _p(h0), _p(y))
    return y


def deer_step(w, u, yprev=None, h0=None):
    """One Newton step from yprev (None = all-zero guess); returns (ynew, rho)."""
    w, u, yprev, h0 = _f64(w), _f64(u), _f64(yprev), _f64(h0)
    T, C = _shapes(u, seqs=(yprev,), feats=(w,), states=(h0,))
    y = np.empty_like(u)
    rho = ctypes.c_double(0.0)
    _load().lro_deer_step(T, C, w.shape[0], _p(w), _p(u), _p(h0), _p(yprev), _p(y),
                          ctypes.byref(rho))
    return y, rho.value


def deer_bwd(w, y, g, h0=None):
    """Gradient through the DEER solution y (the tanh-RNN rollout) for the
    upstream dL/dy = g. Returns (du, dw, dh0)."""
    w, y, g, h0 = _f64(w), _f64(y), _f64(g), _f64(h0)
    T, C = _shapes(y, seqs=(g,), feats=(w,), states=(h0,))
    D = w.shape[0]
    du = np.empty_like(y)
    dw = np.zeros(D)
    dh0 = np.empty(y.shape[1:]) if y.ndim == 3 else np.empty(C)
    st = _load().lro_deer_bwd(T, C, D, _p(w), _p(y), _p(h0), _p(g), _p(du), _p(dw), _p(dh0))
    if st != 0:
        raise MemoryError("oracle deer_bwd: allocation failed")
    return du, dw, dh0


DEER_CONVERGED, DEER_NOT_CONVERGED, DEER_NONFINITE = 0, 1, 2


def deer(w, u, h0=None, eps=1e-5, kmax=20, y_init=None):
    """Returns (y, iters, rho_history, status) -- status 0 converged, 1 hit kmax,
    2 not finite.  y_init: the initial guess (None = zeros)."""
    w, u, h0, y_init = _f64(w), _f64(u), _f64(h0), _f64(y_init)
    T, C = _shapes(u, seqs=(y_init,), feats=(w,), states=(h0,))
    y = np.empty_like(u)
    hist = np.zeros(kmax, dtype=np.float64)
    iters = ctypes.c_int(0)
    st = _load().lro_deer(T, C, w.shape[0], _p(w), _p(u), _p(h0), _p(y_init), float(eps),
                          int(kmax), _p(y), _p(hist), ctypes.byref(iters))
    if st < 0:
        raise MemoryError("oracle deer: allocation failed")
    return y, int(iters.value), hist[: iters.value].copy(), int(st)


def deer_per_sequence(w, u, h0=None, eps=1e-5, kmax=20, y_init=None):
    """Per-sequence stopping: every batch sequence u[:, b] is its own DEER
    problem with its own stopping test.  Returns (y, iters[B], status[B],
    rho_histories[B])."""
    u = _f64(u)
    T, B, D = u.shape
    y = np.empty_like(u)
    iters, status, hists = [], [], []
    for b in range(B):
        yb, kb, hb, sb = deer(w, u[:, b:b + 1], None if h0 is None else _f64(h0)[b:b + 1], eps, kmax,
                              None if y_init is None else _f64(y_init)[:, b:b + 1])
        y[:, b:b + 1] = yb
        iters.append(kb)
        status.append(sb)
        hists.append(hb)
    return y, iters, status, hists


def rollout_ode(w, u, dt, h0=None):
    """Exponential-Euler rollout of dy/dt = -y + tanh(w y + u) on steps dt[t]
    (G clamped to [-10, 10]).  Returns (y, clamps)."""
    w, u, dt, h0 = _f64(w), _f64(u), _f64(dt), _f64(h0)
    T, C = _shapes(u, feats=(w,), states=(h0,), steps=(dt,))
    y = np.empty_like(u)
    n = ctypes.c_int64(0)
    _load().lro_rollout_ode(T, C, w.shape[0], _p(w), _p(u), _p(dt), _p(h0), _p(y), ctypes.byref(n))
    return y, int(n.value)


def deer_ode_step(w, u, dt, yprev=None, h0=None):
    """One ODE-form DEER iteration from yprev (None = zeros): (ynew, rho, clamps)."""
    w, u, dt, yprev, h0 = _f64(w), _f64(u), _f64(dt), _f64(yprev), _f64(h0)
    T, C = _shapes(u, seqs=(yprev,), feats=(w,), states=(h0,), steps=(dt,))
    y = np.empty_like(u)
    rho = ctypes.c_double(0.0)
    n = ctypes.c_int64(0)
    _load().lro_deer_ode_step(T, C, w.shape[0], _p(w), _p(u), _p(dt), _p(h0), _p(yprev), _p(y),
                              ctypes.byref(rho), ctypes.byref(n))
    return y, rho.value, int(n.value)


def deer_ode(w, u, dt, h0=None, eps=1e-5, kmax=20):
    """ODE-form DEER: (y, iters, rho_history, status, clamps of the last iteration)."""
    w, u, dt, h0 = _f64(w), _f64(u), _f64(dt), _f64(h0)
    T, C = _shapes(u, feats=(w,), states=(h0,), steps=(dt,))
    y = np.empty_like(u)
    hist = np.zeros(kmax, dtype=np.float64)
    iters = ctypes.c_int(0)
    n = ctypes.c_int64(0)
    st = _load().lro_deer_ode(T, C, w.shape[0], _p(w), _p(u), _p(dt), _p(h0), float(eps), int(kmax),
                              _p(y), _p(hist), ctypes.byref(iters), ctypes.byref(n))
    if st < 0:
        raise MemoryError("oracle deer_ode: allocation failed")
    return y, int(iters.value), hist[: iters.value].copy(), int(st), int(n.value)


def rel_err(got, ref) -> float:
    """max|got - ref| / max(1, max|ref|) -- the parity measure, per tensor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)) / max(1.0, float(np.max(np.abs(ref)))))
