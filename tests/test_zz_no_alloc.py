"""lr_scan_fwd_noalloc: the forward scan for callers that may not allocate
device memory (engines or plugins that own every device byte, latency-critical
loops where a cudaFree would synchronise the device).  Its scratch lives in a
fixed __device__ array, so this file checks, through the C ABI, that it gives
the same bits as lr_scan_fwd on two calls in a row with different inputs (the
second call reuses the array the first one left behind), with and without a
caller-supplied error word, and that oversize problems are refused.

Collected last on purpose (file name), so a failure here does not hide the
results of the other GPU tests; it also passes when run alone."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _lib(cuda):
    lib = cuda.load()
    f = lib.lr_scan_fwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_void_p,
                                                                 ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _dev(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


@pytest.mark.parametrize("dtype,shape", [# cluster kernel (8 and 16 CTAs); look-back kernel
                                         ("f32", (1024, 4, 256)), ("bf16", (777, 3, 512)),
                                         ("f32", (2048, 4, 256)),
                                         ("f32", (2100, 2, 256)), ("f32", (3001, 2, 100)),
                                         # strip kernel; walker kernels (register, segmented)
                                         ("bf16", (2100, 16, 1024)), ("f32", (20000, 1, 128)),
                                         ("bf16", (20000, 1, 128))])
@pytest.mark.parametrize("with_err", [True, False])
def test_noalloc_matches_allocating_scan_twice(cuda, dtype, shape, with_err):
    """Two calls in a row, each on new inputs (a stale packet left by the first
    call would show in the second), with and without a caller error word:
    each result has the same bits as lr_scan_fwd's on the same inputs (both
    run the same kernel on the same shape)."""
    T, B, D = shape
    wl = W.like(W.SCAN_TINY, T, B, D, dtype)
    f = _lib(cuda)
    code = 1 if dtype == "bf16" else 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda") if with_err else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed in (21, 22):
        inp = W.make_inputs(wl, seed)
        inp["h0"] = W.store(W.normal(seed, 77, (B, D)), dtype)
        a, b, h0 = (_dev(inp[k], dtype) for k in ("a", "b", "h0"))
        ref = cuda.lr_scan_fwd(a, b, h0)
        h = torch.full_like(a, float("nan"))
        st = f(_p(a), _p(b), _p(h0), _p(h), B, T, D, code, _p(err), stream)
        assert st == cuda.LR_OK, cuda.status_str(st)
        torch.cuda.synchronize()
        assert torch.equal(h, ref), (h.float() - ref.float()).abs().max().item()
    if with_err:
        assert int(err.item()) == 0
    assert cuda.last_error() == cuda.LR_OK


def test_noalloc_refuses_oversize(cuda):
    f = _lib(cuda)
    T, B, D = 1 << 20, 1, 128  # 16384 tiles: beyond the fixed scratch
    a = torch.empty(T, B, D, device="cuda")
    st = f(_p(a), _p(a), None, _p(a), B, T, D, 0, None,
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == cuda.LR_ERR_TOO_LARGE
