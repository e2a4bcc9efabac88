"""Parity of the next rows at the full sizes bench.py times them, through
the same C-ABI calls: the LSTM cell at the SRU layer's size, the DEER
backward and the ODE form of DEER at the DEER workload's size, on the bench's
own seeded inputs.  Features are independent in the cell and in the DEER
backward, so the oracle checks a sample of whole features (every batch row
and time step of each, which the parameter-gradient sums need); the ODE
solve's iteration count is a global quantity, so its oracle solves the full
problem.  Collected after the other GPU tests (file name), so a failure here
does not hide their results; it also passes when run alone."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from lrtest import assert_close, dev_inputs, f64_inputs, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _features(D, n, seed):
    r = np.random.default_rng(seed)
    s = set(r.choice(D, size=min(n, D), replace=False).tolist())
    s.update({0, D - 1})
    return np.array(sorted(s))


def _sub(x, dsel):
    """The selected features of a [T, B, D], [B, D] or [D] array."""
    return np.ascontiguousarray(np.asarray(x, np.float64)[..., dsel])


def _pick(t, dsel):
    return to_f64(t.index_select(t.dim() - 1, torch.as_tensor(dsel, device=t.device)))


def test_lstm_cell_full_sampled(cuda):
    wl = W.LSTM
    inp = W.make_inputs(wl, 0)
    dv, f = dev_inputs(inp, wl.dtype), f64_inputs(inp, wl.dtype)
    gates = ("zf", "zi", "zc", "zo")
    biases = ("bf", "bi", "bc", "bo")
    args = [dv[k] for k in gates + biases]
    h, c = cuda.lstm_cell_fwd(*args, dv["c0"])
    g = cuda.lstm_cell_bwd(*args, c, dv["dh"], dv["c0"])
    dsel = _features(wl.D, 12, 5)
    sf = {k: _sub(v, dsel) for k, v in f.items()}
    rh, rc = oracle.lstm_fwd(*(sf[k] for k in gates + biases), sf["c0"])
    ref = oracle.lstm_bwd(*(sf[k] for k in gates + biases), rc, sf["dh"], sf["c0"])
    assert_close("h", _pick(h, dsel), rh, wl.dtype)
    assert_close("c", _pick(c, dsel), rc, wl.dtype)
    for k, r in zip(("dzf", "dzi", "dzc", "dzo", "dbf", "dbi", "dbc", "dbo", "dc0"), ref):
        assert_close(k, _pick(g[k], dsel), r, wl.dtype)


def test_deer_bwd_full_sampled(cuda):
    """The gradient through the solution, with the solution y made by the
    oracle's rollout (stored in fp32 for both sides) and the bench's upstream
    gradient."""
    wl = W.DEER
    inp = W.make_inputs(wl, 0)
    w = np.asarray(inp["w"], np.float64)
    y = W.store(oracle.rollout_tanh(w, W.to_f64(inp["u"], wl.dtype), W.to_f64(inp["h0"], wl.dtype)),
                wl.dtype)
    dy = W.store(W.normal(0, 90, (wl.T, wl.B, wl.D)), wl.dtype)
    data = {"w": inp["w"], "y": y, "dy": dy, "h0": inp["h0"]}
    dv, f = dev_inputs(data, wl.dtype), f64_inputs(data, wl.dtype)
    du, dw, dh0 = cuda.deer_diag_bwd(dv["w"], dv["y"], dv["dy"], dv["h0"])
    dsel = _features(wl.D, 12, 6)
    rdu, rdw, rdh0 = oracle.deer_bwd(_sub(f["w"], dsel), _sub(f["y"], dsel), _sub(f["dy"], dsel),
                                     _sub(f["h0"], dsel))
    assert_close("du", _pick(du, dsel), rdu, wl.dtype)
    assert_close("dw", to_f64(dw)[dsel], rdw, wl.dtype)
    assert_close("dh0", _pick(dh0, dsel), rdh0, wl.dtype)


def test_deer_ode_full(cuda):
    """The ODE form on the DEER workload with the bench's steps dt ~ U(0.1, 1):
    the same iteration count and status as the fp64 oracle, the residual
    history and the solution within the fp32 tolerance."""
    wl = W.DEER
    inp = W.make_inputs(wl, 0)
    dv, f = dev_inputs(inp, wl.dtype), f64_inputs(inp, wl.dtype)
    dts = W.uniform(0, 44, (wl.T,), 0.1, 1.0)
    y, k, resid, hist, st, cl = cuda.deer_ode_solve(dv["w"], dv["u"], torch.from_numpy(dts).cuda(),
                                                    dv["h0"], eps=1e-5, kmax=20)
    ry, rk, rhist, rst, rcl = oracle.deer_ode(f["w"], f["u"], dts.astype(np.float64), f["h0"],
                                              eps=1e-5, kmax=20)
    assert _margin_ok(rhist), f"residual history too close to eps: {list(rhist)}"
    assert (k, st == cuda.LR_OK) == (rk, rst == oracle.DEER_CONVERGED), (hist, list(rhist))
    np.testing.assert_allclose(hist, rhist, rtol=1e-3, atol=1e-6)
    assert_close("y", to_f64(y), ry, wl.dtype)
    assert cl == rcl == 0


def _margin_ok(hist, eps=1e-5):
    """No fp64 residual within 2e-6 of eps.  The fp32 residuals carry ~1e-7 of
    rounding (differences of stored iterates of magnitude ~1), so at that
    distance the stopping test takes the same decision in both precisions."""
    h = np.asarray(hist, np.float64)
    return h.size == 0 or float(np.min(np.abs(h - eps))) > 2e-6


@pytest.mark.parametrize("shape", [(77, 2, 5), (1, 1, 4), (1, 3, 7), (300, 2, 9)])
def test_deer_variants_scalar_path_and_single_step(cuda, shape):
    """The ODE form, the warm start and per-sequence stopping on odd D (the
    scalar path) and at T = 1, against the oracle: the same counts, and the
    solutions within the fp32 tolerance."""
    T, B, D = shape
    wl = W.like(W.DEER, T, B, D, "f32")
    inp = W.make_inputs(wl, 12)
    inp["h0"] = W.normal(12, 43, (B, D))
    dv, f = dev_inputs(inp, "f32"), f64_inputs(inp, "f32")
    # ODE form
    dts = W.uniform(12, 44, (T,), 0.1, 1.0)
    y, k, resid, hist, st, cl = cuda.deer_ode_solve(dv["w"], dv["u"], torch.from_numpy(dts).cuda(),
                                                    dv["h0"], eps=1e-5, kmax=20)
    ry, rk, rhist, rst, rcl = oracle.deer_ode(f["w"], f["u"], dts.astype(np.float64), f["h0"],
                                              eps=1e-5, kmax=20)
    assert _margin_ok(rhist), list(rhist)
    assert (k, st == cuda.LR_OK) == (rk, rst == oracle.DEER_CONVERGED), (hist, list(rhist))
    assert_close("ode y", to_f64(y), ry, "f32")
    # warm start from the solution of a nearby problem
    near = oracle.rollout_tanh(f["w"], f["u"] + 1e-3 * np.sin(np.arange(f["u"].size)).reshape(f["u"].shape),
                               f["h0"]).astype(np.float32)
    r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], y_init=torch.from_numpy(near).cuda(),
                                eps=1e-5, kmax=20)
    wy, wk, whist, wst = oracle.deer(f["w"], f["u"], f["h0"], eps=1e-5, kmax=20,
                                     y_init=near.astype(np.float64))
    assert _margin_ok(whist), list(whist)
    assert (r["iters"], r["status"] == cuda.LR_OK) == (wk, wst == oracle.DEER_CONVERGED)
    assert_close("warm y", to_f64(r["y"]), wy, "f32")
    # per-sequence stopping
    r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20, per_sequence=True)
    sy, sks, ssts, shists = oracle.deer_per_sequence(f["w"], f["u"], f["h0"], eps=1e-5, kmax=20)
    assert all(_margin_ok(h) for h in shists), shists
    assert r["seq_iters"] == sks
    assert_close("per-sequence y", to_f64(r["y"]), sy, "f32")
