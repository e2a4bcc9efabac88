"""Parity at the full benchmark sizes, through the same C-ABI calls and launch
configuration that bench.py times.  Channels are independent, so the oracle
checks a sample of whole channels (every time step of each sampled channel,
which exercises every chunk boundary along time); the small scan is checked
in full, and DEER's iteration count -- a global quantity -- against the full
oracle solve."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from lrtest import TOL, assert_close, cols, dev_cols, dev_inputs, f64_inputs, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample(C, n, seed):
    r = np.random.default_rng(seed)
    s = set(r.choice(C, size=min(n, C), replace=False).tolist())
    s.update({0, C - 1})
    return np.array(sorted(s))


def test_scan_tiny_full(cuda):
    wl = W.SCAN_TINY
    inp = W.make_inputs(wl, 0)
    dv, f = dev_inputs(inp, wl.dtype), f64_inputs(inp, wl.dtype)
    h = cuda.lr_scan_fwd(dv["a"], dv["b"], dv["h0"])
    href = oracle.scan_fwd(f["a"], f["b"], f["h0"])
    assert_close("h", to_f64(h), href, wl.dtype)
    da, db, dh0 = cuda.lr_scan_bwd(dv["a"], h, dv["g"], dv["h0"])
    rda, rdb, rdh0 = oracle.scan_bwd(f["a"], href, f["g"], f["h0"])
    for n, g_, r_ in (("da", da, rda), ("db", db, rdb), ("dh0", dh0, rdh0)):
        assert_close(n, to_f64(g_), r_, wl.dtype)


@pytest.mark.parametrize("wl", [W.SCAN_LONG, W.SCAN_BF16], ids=lambda w: w.name)
def test_scan_large_sampled(cuda, wl):
    inp = W.make_inputs(wl, 0)
    dv = dev_inputs(inp, wl.dtype)
    h = cuda.lr_scan_fwd(dv["a"], dv["b"], dv["h0"])
    sel = _sample(wl.C, 24, 1)
    a, b = (W.to_f64(cols(inp[k], sel), wl.dtype) for k in ("a", "b"))
    h0 = W.to_f64(cols(inp["h0"], sel), wl.dtype)
    href = oracle.scan_fwd(a, b, h0)
    assert_close("h", dev_cols(h, sel), href, wl.dtype)
    if wl.backward:
        da, db, dh0 = cuda.lr_scan_bwd(dv["a"], h, dv["g"], dv["h0"])
        g = W.to_f64(cols(inp["g"], sel), wl.dtype)
        rda, rdb, rdh0 = oracle.scan_bwd(a, href, g, h0)
        assert_close("da", dev_cols(da, sel), rda, wl.dtype)
        assert_close("db", dev_cols(db, sel), rdb, wl.dtype)
        assert_close("dh0", dev_cols(dh0, sel), rdh0, wl.dtype)


def test_sru_sampled(cuda):
    wl = W.SRU
    inp = W.make_inputs(wl, 0)
    dv = dev_inputs(inp, wl.dtype)
    h, c = cuda.sru_fwd(dv["xt"], dv["uf"], dv["ur"], dv["x"], dv["bf"], dv["br"], dv["c0"])
    g = cuda.sru_bwd(dv["xt"], dv["uf"], dv["ur"], dv["x"], dv["bf"], dv["br"], c, dv["dh"], dv["c0"])
    dsel = _sample(wl.D, 12, 2)  # features; every batch row of each (bias sums need all b)
    sub = lambda x: np.ascontiguousarray(x[:, :, dsel]) if x.ndim == 3 else np.ascontiguousarray(x[:, dsel])
    f = {k: (np.asarray(v, np.float64)[dsel] if k in ("bf", "br") else sub(np.asarray(v, np.float64)))
         for k, v in inp.items()}
    rh, rc = oracle.sru_fwd(f["xt"], f["uf"], f["ur"], f["x"], f["bf"], f["br"], f["c0"])
    ref = oracle.sru_bwd(f["xt"], f["uf"], f["ur"], f["x"], f["bf"], f["br"], rc, f["dh"], f["c0"])
    dsel_t = torch.as_tensor(dsel, device="cuda")
    pick = lambda t: to_f64(t.index_select(t.dim() - 1, dsel_t))
    assert_close("h", pick(h), rh, wl.dtype)
    assert_close("c", pick(c), rc, wl.dtype)
    for k, r in zip(("dxt", "duf", "dur", "dx", "dbf", "dbr", "dc0"), ref):
        assert_close(k, pick(g[k]), r, wl.dtype)


def test_deer_full(cuda):
    wl = W.DEER
    inp = W.make_inputs(wl, 0)
    dv, f = dev_inputs(inp, wl.dtype), f64_inputs(inp, wl.dtype)
    y, k, resid, hist, st = cuda.deer_diag_solve(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20)
    ry, rk, rhist, rst = oracle.deer(f["w"], f["u"], f["h0"], eps=1e-5, kmax=20)
    # the count is robust only if no residual sits near eps: require > 0.3 decades
    margin = float(np.min(np.abs(np.log10(rhist / 1e-5))))
    assert margin > 0.3, f"residual history too close to eps: {rhist}"
    assert (k, st) == (rk, rst), (k, hist, list(rhist))
    np.testing.assert_allclose(hist, rhist, rtol=1e-3, atol=1e-6)
    assert_close("y", to_f64(y), ry, wl.dtype)
