"""The C-ABI library: it builds, loads and exports every function that
include/lrscan.h declares; argument errors are reported before any CUDA call.
CPU only (no compute call)."""
import ctypes

import pytest

import linear_recurrence_scan_chunked_gb300 as lrs


@pytest.fixture(scope="module")
def lib():
    lrs.build()
    return lrs.load()


def test_every_declared_function_is_exported(lib):
    names = lrs.declared_functions()
    for required in ("lr_scan_fwd", "lr_scan_bwd", "sru_fwd", "sru_bwd", "deer_diag_solve",
                     "deer_diag_bwd", "lstm_cell_fwd", "lstm_cell_bwd", "lr_scan_fwd_noalloc",
                     "lr_last_error", "lr_status_str"):
        assert required in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for st in range(8):
        assert lrs.status_str(st)
    assert lrs.status_str(999) == "unknown status"


def test_argument_errors_before_cuda(lib):
    P = None
    # null required pointers, bad dtype, negative sizes
    assert lib.lr_scan_fwd(P, P, P, P, 2, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.lr_scan_fwd(P, P, P, P, 2, 3, 4, 7, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.lr_scan_fwd(P, P, P, P, -1, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.lr_scan_bwd(P, P, P, P, P, P, P, 2, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.sru_fwd(*([P] * 9), 2, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.sru_bwd(*([P] * 16), 2, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.lstm_cell_fwd(*([P] * 11), 2, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.lstm_cell_bwd(*([P] * 20), 2, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.lstm_cell_fwd(*([P] * 11), 2, 3, 4, 1, P) == lrs.LR_ERR_INVALID_ARG
    iters = ctypes.c_int(0)
    assert lib.deer_diag_solve(P, P, P, P, 2, 3, 4, ctypes.c_float(1e-5), 20, ctypes.byref(iters),
                               P, P, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.deer_diag_solve(P, P, P, P, 2, 3, 4, ctypes.c_float(1e-5), 0, ctypes.byref(iters),
                               P, P, 0, P) == lrs.LR_ERR_INVALID_ARG
    # the DEER variants: null required pointers, kmax out of range, a bad mode
    it, nl = ctypes.c_int(0), ctypes.c_int(0)
    eps = ctypes.c_float(1e-5)
    assert lib.deer_diag_solve_ex(P, P, P, P, P, 2, 3, 4, eps, 20, 0, ctypes.byref(it), P, P, P, P,
                                  ctypes.byref(nl), 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.deer_diag_solve_ex(P, P, P, P, P, 2, 3, 4, eps, 20, 2, ctypes.byref(it), P, P, P, P,
                                  P, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.deer_diag_solve_ex(P, P, P, P, P, 2, 3, 4, eps, 0, 0, ctypes.byref(it), P, P, P, P,
                                  P, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.deer_ode_solve(P, P, P, P, P, 2, 3, 4, eps, 20, ctypes.byref(it), P, P, P, 0,
                              P) == lrs.LR_ERR_INVALID_ARG
    assert lib.deer_ode_solve(P, P, P, P, P, 2, 3, 4, ctypes.c_float(-1.0), 20, ctypes.byref(it), P,
                              P, P, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.deer_diag_bwd(*([P] * 7), 2, 3, 4, 0, P) == lrs.LR_ERR_INVALID_ARG
    assert lib.lr_test_activations(P, P, P, P, -1, P) == lrs.LR_ERR_INVALID_ARG
    # sizes beyond 2^62 elements
    assert lib.lr_scan_fwd(P, P, P, P, 1 << 31, 1 << 31, 4, 0, P) == lrs.LR_ERR_TOO_LARGE
    # misaligned (odd byte address) fp32 pointer
    buf = ctypes.create_string_buffer(64)
    odd = ctypes.c_void_p(ctypes.addressof(buf) + 1)
    assert lib.lr_scan_fwd(odd, odd, P, odd, 1, 1, 1, 0, P) == lrs.LR_ERR_ALIGN


def test_empty_problem_is_a_no_op(lib):
    # B*T*D == 0 returns before touching the device
    assert lib.lr_scan_fwd(None, None, None, None, 0, 5, 4, 0, None) == lrs.LR_OK
    assert lib.sru_fwd(*([None] * 9), 3, 0, 4, 0, None) == lrs.LR_OK
    assert lib.lstm_cell_fwd(*([None] * 11), 3, 0, 4, 0, None) == lrs.LR_OK


def test_binding_checks_tensors_before_the_library():
    """The binding rejects host tensors, wrong shapes and wrong dtypes with
    ValueError before any call into the library (no device needed)."""
    import torch
    u = torch.zeros(5, 2, 4)
    w = torch.zeros(4)
    with pytest.raises(ValueError):
        lrs.deer_ode_solve(w, u, torch.zeros(5))
    with pytest.raises(ValueError):
        lrs.deer_diag_solve_ex(w, u)
    with pytest.raises(ValueError):
        lrs.lstm_cell_fwd(u, u, u, u, w, w, w, w)
    with pytest.raises(ValueError):
        lrs.test_activations(torch.zeros(3))


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(lrs, "_lib", None)
    monkeypatch.setattr(lrs, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        lrs.load()


def _fake_cuda_tensor(shape, dtype, device):
    """Stands in for a CUDA tensor in the binding's checks (no device here)."""
    import types
    import torch
    return types.SimpleNamespace(shape=torch.Size(shape), dtype=dtype, device=torch.device(device),
                                 is_cuda=True, dim=lambda: len(shape), is_contiguous=lambda: True)


def test_binding_rejects_tensors_on_another_device(monkeypatch):
    """States, per-feature parameters and the stream must be on the sequence
    tensors' device, and that device must be the current one (the library
    launches on the current device)."""
    import types
    import torch
    f32 = torch.float32
    u = _fake_cuda_tensor((5, 2, 4), f32, "cuda:0")
    assert lrs._state("h0", _fake_cuda_tensor((2, 4), f32, "cuda:0"), u) is not None
    assert lrs._param("w", _fake_cuda_tensor((4,), f32, "cuda:0"), 4, u) is not None
    with pytest.raises(ValueError, match="cuda:1"):
        lrs._state("h0", _fake_cuda_tensor((2, 4), f32, "cuda:1"), u)
    with pytest.raises(ValueError, match="cuda:1"):
        lrs._param("w", _fake_cuda_tensor((4,), f32, "cuda:1"), 4, u)
    with pytest.raises(ValueError, match="match"):
        lrs._seq("b", _fake_cuda_tensor((5, 2, 4), f32, "cuda:1"), u)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    s0 = types.SimpleNamespace(device=torch.device("cuda:0"), cuda_stream=0)
    s1 = types.SimpleNamespace(device=torch.device("cuda:1"), cuda_stream=0)
    assert lrs._stream(s0, u).value is None  # handle 0: the legacy default stream
    with pytest.raises(ValueError, match="stream belongs"):
        lrs._stream(s1, u)
    with pytest.raises(ValueError, match="current CUDA device"):
        lrs._stream(s1, _fake_cuda_tensor((5, 2, 4), f32, "cuda:1"))


def test_binding_call_paths_reach_the_library(lib, monkeypatch):
    """Every public call marshals its arguments through the real library's
    prototypes (ctypes checks their count and types).  With stand-in CUDA
    tensors at address 0 the library answers LR_ERR_INVALID_ARG before any
    CUDA call, and the binding raises it as LrError."""
    import types
    import torch
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream",
                        lambda *a, **k: types.SimpleNamespace(device=torch.device("cuda:0"), cuda_stream=0))
    T, B, D = 5, 2, 4

    def t(*shape):
        x = _fake_cuda_tensor(shape, torch.float32, "cuda:0")
        x.data_ptr = lambda: 0
        return x

    def seq():
        return t(T, B, D)

    calls = [
        lambda: lrs.lr_scan_fwd(seq(), seq(), t(B, D), h=seq()),
        lambda: lrs.lr_scan_bwd(seq(), seq(), seq(), t(B, D), da=seq(), db=seq(), dh0=t(B, D)),
        lambda: lrs.sru_fwd(seq(), seq(), seq(), seq(), t(D), t(D), t(B, D), h=seq(), c=seq()),
        lambda: lrs.sru_bwd(seq(), seq(), seq(), seq(), t(D), t(D), seq(), seq(), t(B, D),
                            out={"dxt": seq(), "duf": seq(), "dur": seq(), "dx": seq(), "dbf": t(D),
                                 "dbr": t(D), "dc0": t(B, D)}),
        lambda: lrs.lstm_cell_fwd(seq(), seq(), seq(), seq(), t(D), t(D), t(D), t(D), t(B, D),
                                  h=seq(), c=seq()),
        lambda: lrs.lstm_cell_bwd(seq(), seq(), seq(), seq(), t(D), t(D), t(D), t(D), seq(), seq(),
                                  t(B, D), out={"dzf": seq(), "dzi": seq(), "dzc": seq(), "dzo": seq(),
                                                "dbf": t(D), "dbi": t(D), "dbc": t(D), "dbo": t(D),
                                                "dc0": t(B, D)}),
        lambda: lrs.deer_diag_solve(t(D), seq(), t(B, D), y=seq()),
        lambda: lrs.deer_diag_solve_ex(t(D), seq(), t(B, D), y=seq(), y_init=seq()),
        lambda: lrs.deer_diag_solve_ex(t(D), seq(), y=seq(), per_sequence=True),
        lambda: lrs.deer_ode_solve(t(D), seq(), t(T), t(B, D), y=seq()),
        lambda: lrs.deer_diag_bwd(t(D), seq(), seq(), t(B, D), du=seq(), dw=t(D), dh0=t(B, D)),
    ]
    for call in calls:
        with pytest.raises(lrs.LrError) as e:
            call()
        assert e.value.status == lrs.LR_ERR_INVALID_ARG


_C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "lrscan.h"

int main(void) {
    int bad = 0, it = 0;
    float eps = 1e-5f;
    if (lr_scan_fwd(NULL, NULL, NULL, NULL, 2, 3, 4, LR_F32, NULL) != LR_ERR_INVALID_ARG) bad |= 1;
    if (lr_scan_fwd(NULL, NULL, NULL, NULL, 0, 3, 4, LR_F32, NULL) != LR_OK) bad |= 2;
    if (lr_scan_fwd(NULL, NULL, NULL, NULL, 2, 3, 4, 9, NULL) != LR_ERR_INVALID_ARG) bad |= 4;
    if (deer_diag_solve(NULL, NULL, NULL, NULL, 2, 3, 4, eps, 0, &it, NULL, NULL, LR_F32, NULL)
        != LR_ERR_INVALID_ARG) bad |= 8;
    if (strcmp(lr_status_str(LR_OK), lr_status_str(LR_ERR_INVALID_ARG)) == 0) bad |= 16;
    printf("%s\n", lr_status_str(LR_ERR_INVALID_ARG));
    return bad;
}
"""


def test_c_program_links_against_the_header_and_library(lib):
    """The boundary as a C caller sees it: a C99 program includes the header,
    links the shared library, and gets the documented status codes (argument
    errors only: no device is needed)."""
    import os
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lrs.LIB_PATH)
    root = os.path.dirname(os.path.dirname(os.path.abspath(lrs.__file__)))
    src = os.path.join(libdir, f"c_caller.{os.getpid()}.c")
    exe = src[:-2]
    with open(src, "w") as f:
        f.write(_C_CALLER)
    try:
        subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"), src,
                        "-o", exe, "-L", libdir, "-llrscan", f"-Wl,-rpath,{libdir}"],
                       check=True, capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
        assert r.stdout.strip() == lrs.status_str(lrs.LR_ERR_INVALID_ARG)
    finally:
        for p in (src, exe):
            if os.path.exists(p):
                os.remove(p)
