"""Seeded synthetic inputs for the linear-recurrence hot path.

This module is the one piece shared by the CUDA-path tests, the oracle tests
and the benchmark.  It holds no arithmetic of the method: it draws random
numbers, applies the input distributions (e.g. a = sigmoid(z) is how the
coefficients are *distributed*, not a step of the scan) and converts storage
formats.

Generator: numpy's Philox4x64-10 counter-based bit generator (Salmon et al.,
SC'11).  Every tensor role has a fixed id; the tensor is filled in blocks of
2**22 elements and block j of tensor `tid` uses key (seed, tid << 32 | j), so
the values do not depend on the number of threads used to draw them.

Storage formats: "f32" -> numpy float32; "bf16" -> numpy uint16 holding the
bfloat16 bit pattern, rounded to nearest-even from the float32 value.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK = 1 << 22

# fixed ids of the tensor roles (part of the input recipe)
TID = {"a": 1, "b": 2, "h0": 3, "g": 4, "xt": 5, "uf": 6, "ur": 7, "x": 8,
       "dh": 9, "w": 10, "u": 11, "zf": 12, "zi": 13, "zc": 14, "zo": 15,
       "bf": 16, "bi": 17, "bc": 18, "bo": 19}


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill(seed: int, tid: int, n: int, draw) -> np.ndarray:
    """Fill n values block by block; draw(gen, count) -> float array."""
    out = np.empty(n, dtype=np.float32)
    nblk = (n + BLOCK - 1) // BLOCK

    def work(j):
        lo, hi = j * BLOCK, min(n, (j + 1) * BLOCK)
        key = np.array([seed, (tid << 32) | j], dtype=np.uint64)
        gen = np.random.Generator(np.random.Philox(key=key))
        out[lo:hi] = draw(gen, hi - lo)

    if nblk <= 1:
        for j in range(nblk):
            work(j)
    else:
        with ThreadPoolExecutor(min(nblk, _threads())) as ex:
            list(ex.map(work, range(nblk)))
    return out


def normal(seed, tid, shape, mean=0.0, std=1.0) -> np.ndarray:
    """float32 N(mean, std) (std is the standard deviation)."""
    n = int(np.prod(shape))
    if mean == 0.0 and std == 1.0:
        f = lambda g, m: g.standard_normal(m, dtype=np.float32)
    else:
        f = lambda g, m: (g.standard_normal(m, dtype=np.float32).astype(np.float64) * std + mean)
    return _fill(seed, tid, n, f).reshape(shape)


def uniform(seed, tid, shape, lo, hi) -> np.ndarray:
    """float32 U[lo, hi) drawn in fp64 then rounded."""
    n = int(np.prod(shape))
    return _fill(seed, tid, n, lambda g, m: g.random(m) * (hi - lo) + lo).reshape(shape)


def sigmoid_of_normal(seed, tid, shape, mean=0.0, std=1.0) -> np.ndarray:
    """float32 sigmoid(z), z ~ N(mean, std); sigmoid taken in fp64 then rounded."""
    n = int(np.prod(shape))

    def f(g, m):
        z = g.standard_normal(m, dtype=np.float32).astype(np.float64) * std + mean
        return 1.0 / (1.0 + np.exp(-z))

    return _fill(seed, tid, n, f).reshape(shape)


# ------------------------------------------------------------ storage formats

def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even); returns uint16 bit patterns.
    A NaN stays a NaN (the quiet NaN 0x7FC0, sign kept): adding the rounding
    bias to a NaN with a small payload would carry into an infinity."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    u = x32.view(np.uint32)
    r = ((u.astype(np.uint64) + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x32)
    if nan.any():
        r = np.where(nan, ((u >> 16) & 0x8000).astype(np.uint16) | np.uint16(0x7FC0), r)
    return r


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored values (f32 array or bf16 bit patterns) to float64 exactly."""
    if dtype == "bf16":
        return bf16_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


# ------------------------------------------------------------------ workloads

@dataclass
class Workload:
    name: str
    kind: str               # "scan" | "sru" | "deer" | "lstm"
    T: int
    B: int
    D: int
    dtype: str = "f32"      # storage format
    backward: bool = True
    extra: dict = field(default_factory=dict)

    @property
    def C(self) -> int:
        return self.B * self.D

    @property
    def N(self) -> int:
        return self.T * self.B * self.D

    def describe(self) -> str:
        return f"{self.name}: {self.kind} T={self.T} B={self.B} D={self.D} {self.dtype}"


# The five full-size workloads of the hot path (layout [T, B, D]).
SCAN_TINY = Workload("scan_tiny_f32", "scan", 1024, 4, 256, "f32", True,
                     {"a": ("sigmoid_normal", 0.0, 1.0), "h0": "zero"})
SRU = Workload("sru_f32", "sru", 2048, 32, 1024, "f32", True)
SCAN_LONG = Workload("scan_long_f32", "scan", 1 << 20, 1, 128, "f32", False,
                     {"a": ("uniform", 0.9, 1.0), "b_std": 0.01, "h0": "normal"})
SCAN_BF16 = Workload("scan_large_bf16", "scan", 8192, 16, 4096, "bf16", True,
                     {"a": ("sigmoid_normal", 2.0, 1.0), "h0": "zero"})
DEER = Workload("deer_tanh_f32", "deer", 65536, 4, 256, "f32", False,
                {"eps": 1e-5, "kmax": 20})
FULL = [SCAN_TINY, SRU, SCAN_LONG, SCAN_BF16, DEER]
# The LSTM cell-state scan at the SRU layer's size (the pages give no LSTM
# sizes; same [T, B, D] and the same number of gate projections per element).
LSTM = Workload("lstm_cell_f32", "lstm", 2048, 32, 1024, "f32", True)


def like(base: Workload, T=None, B=None, D=None, dtype=None, name=None) -> Workload:
    """Same distributions as `base` at another shape (small parity cases)."""
    return Workload(name or f"{base.name}[{T or base.T}x{B or base.B}x{D or base.D}]",
                    base.kind, T or base.T, B or base.B, D or base.D,
                    dtype or base.dtype, base.backward, dict(base.extra))


def make_inputs(wl: Workload, seed: int = 0) -> dict:
    """Seeded inputs in storage format; sequence tensors are [T, B, D]."""
    shp = (wl.T, wl.B, wl.D)
    st = lambda x: store(x, wl.dtype)
    out = {}
    if wl.kind == "scan":
        am = wl.extra.get("a", ("sigmoid_normal", 0.0, 1.0))
        if am[0] == "uniform":
            out["a"] = st(uniform(seed, TID["a"], shp, am[1], am[2]))
        else:
            out["a"] = st(sigmoid_of_normal(seed, TID["a"], shp, am[1], am[2]))
        out["b"] = st(normal(seed, TID["b"], shp, 0.0, wl.extra.get("b_std", 1.0)))
        if wl.extra.get("h0", "zero") == "normal":
            out["h0"] = st(normal(seed, TID["h0"], (wl.B, wl.D)))
        else:
            out["h0"] = st(np.zeros((wl.B, wl.D), np.float32))
        if wl.backward:
            out["g"] = st(normal(seed, TID["g"], shp))
    elif wl.kind == "sru":
        for k in ("xt", "uf", "ur", "x"):
            out[k] = st(normal(seed, TID[k], shp))
        out["bf"] = np.full(wl.D, wl.extra.get("bf", 1.0), np.float32)
        out["br"] = np.full(wl.D, wl.extra.get("br", -1.0), np.float32)
        out["c0"] = st(np.zeros((wl.B, wl.D), np.float32))
        if wl.backward:
            out["dh"] = st(normal(seed, TID["dh"], shp))
    elif wl.kind == "lstm":
        for k in ("zf", "zi", "zc", "zo"):
            out[k] = st(normal(seed, TID[k], shp))
        # biases: forget gate biased open (mean 1), the others around 0
        out["bf"] = normal(seed, TID["bf"], (wl.D,), 1.0, 0.5)
        for k in ("bi", "bc", "bo"):
            out[k] = normal(seed, TID[k], (wl.D,), 0.0, 0.5)
        out["c0"] = st(np.zeros((wl.B, wl.D), np.float32))
        if wl.backward:
            out["dh"] = st(normal(seed, TID["dh"], shp))
    elif wl.kind == "deer":
        out["w"] = uniform(seed, TID["w"], (wl.D,), -0.9, 0.9)
        out["u"] = st(normal(seed, TID["u"], shp))
        out["h0"] = st(np.zeros((wl.B, wl.D), np.float32))
    else:
        raise ValueError(wl.kind)
    return out
