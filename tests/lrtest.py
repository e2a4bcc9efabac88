"""Shared helpers of the parity tests: device transfer of the seeded inputs,
the comparison measure, and the oracle runs on (sampled) channels."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

# per-feature parameters: always fp32, whatever the storage type
PARAMS = ("w", "bf", "br", "bi", "bc", "bo")

# max|gpu - oracle| / max(1, max|oracle|) per output tensor
TOL = {"f32": 1e-5, "bf16": 2e-2}


def to_dev(arr: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return W.to_f64(t.view(torch.int16).numpy().view(np.uint16), "bf16")
    return t.numpy().astype(np.float64)


def dev_inputs(inp: dict, dtype: str) -> dict:
    out = {}
    for k, v in inp.items():
        if k in PARAMS:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()
        else:
            out[k] = to_dev(v, dtype)
    return out


def f64_inputs(inp: dict, dtype: str) -> dict:
    return {k: (np.asarray(v, np.float64) if k in PARAMS else W.to_f64(v, dtype))
            for k, v in inp.items()}


def rel_err(got, ref) -> float:
    return oracle.rel_err(got, ref)


def assert_close(name, got, ref, dtype):
    e = rel_err(got, ref)
    assert e <= TOL[dtype], f"{name}: rel err {e:.3e} > {TOL[dtype]:.0e}"
    return e


def cols(x: np.ndarray, sel) -> np.ndarray:
    """[T, B, D] or [B, D] -> the selected flat channels, as [T, n] / [n]."""
    if x.ndim == 3:
        return np.ascontiguousarray(x.reshape(x.shape[0], -1)[:, sel])
    return np.ascontiguousarray(x.reshape(-1)[sel])


def dev_cols(t: torch.Tensor, sel) -> np.ndarray:
    idx = torch.as_tensor(np.asarray(sel), device=t.device)
    if t.dim() == 3:
        return to_f64(t.reshape(t.shape[0], -1).index_select(1, idx))
    return to_f64(t.reshape(-1).index_select(0, idx))
