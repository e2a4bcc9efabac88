"""GPU vs fp64 oracle, element by element, on seeded inputs at sizes the oracle
finishes in seconds: several tiles along time and channels, ragged time and
channel tails, the scalar (unaligned / odd D) path, bf16 storage, and the
degenerate cases (T = 1, one channel, empty problems).  All calls go through
the C ABI (via the thin binding)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from lrtest import assert_close, dev_inputs, f64_inputs, to_dev, to_f64, TOL

pytestmark = pytest.mark.gpu

# (T, B, D).  The scans of up to 2048 steps run the cluster kernel (128 rows,
# 32 channels per CTA; up to 16 CTAs per cluster); the cells take their tiles of
# 32-64 rows and 128 channels.
SHAPES = [(1, 1, 4), (5, 2, 8), (64, 1, 128), (65, 1, 128), (200, 3, 96), (1000, 2, 64),
          (333, 4, 40), (77, 3, 5), (513, 1, 129), (2048, 2, 256), (3, 1, 1)]
# long, narrow problems run the walker protocol; 200 channels need more walker
# warps than there are SMs, so the forward takes the register kernel there
LONG = [(100003, 1, 4), (20000, 1, 128), (20000, 1, 200)]
# wide problems (at least 128 channel tiles) run the strip kernel: one strip
# per CTA with a ragged last strip, and two strips per CTA (more strips than
# resident CTAs)
WIDE = [(70, 33, 520), (45, 40, 1000)]
# the scans' own protocols past the cluster kernel's 2048 steps: look-back
# (fp32 TMA tiles of 32 rows, 4 channel tiles), strip (135 channel tiles of
# 128), register chain (scalar path: D = 7)
SCAN_MID = [(2100, 2, 256), (2100, 33, 520), (2100, 3, 7)]
# the cluster kernel's vector path with a ragged last channel tile (C = 20, 36:
# lanes past the channels idle, 2 channels a lane)
SCAN_RAGGED = [(300, 1, 20), (1000, 3, 12)]


def _scan_case(cuda, T, B, D, dtype, seed=0):
    wl = W.like(W.SCAN_TINY, T, B, D, dtype)
    inp = W.make_inputs(wl, seed)
    inp["h0"] = W.store(W.normal(seed, 99, (B, D)), dtype)  # nonzero initial state
    dv, f = dev_inputs(inp, dtype), f64_inputs(inp, dtype)
    h = cuda.lr_scan_fwd(dv["a"], dv["b"], dv["h0"])
    href = oracle.scan_fwd(f["a"], f["b"], f["h0"])
    assert_close("h", to_f64(h), href, dtype)
    da, db, dh0 = cuda.lr_scan_bwd(dv["a"], h, dv["g"], dv["h0"])
    rda, rdb, rdh0 = oracle.scan_bwd(f["a"], href, f["g"], f["h0"])
    assert_close("da", to_f64(da), rda, dtype)
    assert_close("db", to_f64(db), rdb, dtype)
    assert_close("dh0", to_f64(dh0), rdh0, dtype)


@pytest.mark.parametrize("shape", SHAPES + LONG + WIDE + SCAN_MID + SCAN_RAGGED)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scan_fwd_bwd(cuda, shape, dtype):
    _scan_case(cuda, *shape, dtype)


@pytest.mark.parametrize("shape", SHAPES[:9] + WIDE + [(6001, 1, 256)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sru_fwd_bwd(cuda, shape, dtype):
    T, B, D = shape
    wl = W.like(W.SRU, T, B, D, dtype)
    inp = W.make_inputs(wl, 3)
    inp["bf"] = W.normal(3, 40, (D,))
    inp["br"] = W.normal(3, 41, (D,))
    inp["c0"] = W.store(W.normal(3, 42, (B, D)), dtype)
    dv, f = dev_inputs(inp, dtype), f64_inputs(inp, dtype)
    h, c = cuda.sru_fwd(dv["xt"], dv["uf"], dv["ur"], dv["x"], dv["bf"], dv["br"], dv["c0"])
    rh, rc = oracle.sru_fwd(f["xt"], f["uf"], f["ur"], f["x"], f["bf"], f["br"], f["c0"])
    assert_close("h", to_f64(h), rh, dtype)
    assert_close("c", to_f64(c), rc, dtype)
    g = cuda.sru_bwd(dv["xt"], dv["uf"], dv["ur"], dv["x"], dv["bf"], dv["br"], c, dv["dh"], dv["c0"])
    ref = oracle.sru_bwd(f["xt"], f["uf"], f["ur"], f["x"], f["bf"], f["br"], rc, f["dh"], f["c0"])
    for k, r in zip(("dxt", "duf", "dur", "dx", "dbf", "dbr", "dc0"), ref):
        # the bias gradients are sums over T*B terms: compare against the
        # magnitude of the sum's terms, scaled like the other tensors
        assert_close(k, to_f64(g[k]), r, dtype)


def _lstm_case(cuda, T, B, D, dtype, seed=6):
    wl = W.like(W.LSTM, T, B, D, dtype)
    inp = W.make_inputs(wl, seed)
    inp["c0"] = W.store(W.normal(seed, 44, (B, D)), dtype)  # nonzero initial state
    dv, f = dev_inputs(inp, dtype), f64_inputs(inp, dtype)
    z = [dv[k] for k in ("zf", "zi", "zc", "zo")]
    bias = [dv[k] for k in ("bf", "bi", "bc", "bo")]
    zr = [f[k] for k in ("zf", "zi", "zc", "zo")]
    br = [f[k] for k in ("bf", "bi", "bc", "bo")]
    h, c = cuda.lstm_cell_fwd(*z, *bias, dv["c0"])
    rh, rc = oracle.lstm_fwd(*zr, *br, f["c0"])
    assert_close("h", to_f64(h), rh, dtype)
    assert_close("c", to_f64(c), rc, dtype)
    g = cuda.lstm_cell_bwd(*z, *bias, c, dv["dh"], dv["c0"])
    ref = oracle.lstm_bwd(*zr, *br, rc, f["dh"], f["c0"])
    for k, r in zip(("dzf", "dzi", "dzc", "dzo", "dbf", "dbi", "dbc", "dbo", "dc0"), ref):
        assert_close(k, to_f64(g[k]), r, dtype)
    return g


@pytest.mark.parametrize("shape", SHAPES[:9] + WIDE + [(6001, 1, 256), (20000, 1, 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lstm_cell_fwd_bwd(cuda, shape, dtype):
    _lstm_case(cuda, *shape, dtype)


def test_lstm_cell_gilr_tie_matches_sru(cuda):
    """i = 1 - f (zi = -zf, bi = -bf) and the candidate as SRU's input with
    a zero highway input: the LSTM cell's c and h are the SRU layer's, on the
    GPU, up to the rounding of sigmoid(-z) against 1 - sigmoid(z)."""
    T, B, D = 3000, 2, 256
    r = np.random.default_rng(17)
    zf = torch.from_numpy(r.standard_normal((T, B, D)).astype(np.float32)).cuda()
    zc = torch.from_numpy(r.standard_normal((T, B, D)).astype(np.float32)).cuda()
    zo = torch.from_numpy(r.standard_normal((T, B, D)).astype(np.float32)).cuda()
    bf, bc, bo = (torch.from_numpy(r.standard_normal(D).astype(np.float32)).cuda() for _ in range(3))
    c0 = torch.from_numpy(r.standard_normal((B, D)).astype(np.float32)).cuda()
    h, c = cuda.lstm_cell_fwd(zf, -zf, zc, zo, bf, -bf, bc, bo, c0)
    xt = torch.tanh(zc + bc)
    hs, cs = cuda.sru_fwd(xt, zf, zo, torch.zeros_like(zf), bf, bo, c0)
    assert float((c - cs).abs().max()) < 1e-4
    assert float((h - hs).abs().max()) < 1e-4


def test_lstm_cell_bwd_is_deterministic(cuda):
    T, B, D = 4000, 8, 256
    wl = W.like(W.LSTM, T, B, D, "f32")
    dv = dev_inputs(W.make_inputs(wl, 2), "f32")
    z = [dv[k] for k in ("zf", "zi", "zc", "zo")]
    bias = [dv[k] for k in ("bf", "bi", "bc", "bo")]
    h, c = cuda.lstm_cell_fwd(*z, *bias)
    g1 = cuda.lstm_cell_bwd(*z, *bias, c, dv["dh"])
    g2 = cuda.lstm_cell_bwd(*z, *bias, c, dv["dh"])
    for k in g1:
        if g1[k] is not None:
            assert torch.equal(g1[k], g2[k]), k


@pytest.mark.parametrize("shape", [(1, 1, 4), (64, 2, 8), (300, 3, 40), (77, 2, 5), (5000, 1, 128),
                                   (9000, 2, 512)] + WIDE)
@pytest.mark.parametrize("dtype", ["f32"])
def test_deer(cuda, shape, dtype):
    T, B, D = shape
    wl = W.like(W.DEER, T, B, D, dtype)
    inp = W.make_inputs(wl, 5)
    inp["h0"] = W.store(W.normal(5, 43, (B, D)), dtype)
    dv, f = dev_inputs(inp, dtype), f64_inputs(inp, dtype)
    y, k, resid, hist, st = cuda.deer_diag_solve(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20)
    ry, rk, rhist, rst = oracle.deer(f["w"], f["u"], f["h0"], eps=1e-5, kmax=20)
    assert (k, st) == (rk, rst), (k, rk, hist, list(rhist))
    assert_close("y", to_f64(y), ry, dtype)
    np.testing.assert_allclose(hist, rhist, rtol=1e-3, atol=1e-6)


def _deer_case(shape, seed, scales=None):
    """DEER inputs in fp32; scales[b] multiplies sequence b's u and h0."""
    T, B, D = shape
    wl = W.like(W.DEER, T, B, D, "f32")
    inp = W.make_inputs(wl, seed)
    inp["h0"] = W.normal(seed, 43, (B, D))
    if scales is not None:
        sc = np.asarray(scales, np.float32)
        inp["u"] = (inp["u"] * sc[None, :, None]).astype(np.float32)
        inp["h0"] = (inp["h0"] * sc[:, None]).astype(np.float32)
    return inp, dev_inputs(inp, "f32"), f64_inputs(inp, "f32")


DEER_SHAPES = [(300, 3, 40), (2000, 2, 256), (9000, 2, 512), (5000, 1, 128)]


@pytest.mark.parametrize("shape", DEER_SHAPES)
def test_deer_warm_start(cuda, shape):
    """Warm start from the solution of a nearby problem (the previous step's):
    same K, status and residuals as the oracle from the same guess, fewer
    iterations than the cold start; the guess may be y itself."""
    inp, dv, f = _deer_case(shape, 7)
    near = oracle.rollout_tanh(f["w"], f["u"] + 1e-3 * np.sin(np.arange(f["u"].size)).reshape(f["u"].shape),
                               f["h0"]).astype(np.float32)
    guess = torch.from_numpy(near).cuda()
    r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], y_init=guess, eps=1e-5, kmax=20)
    ry, rk, rhist, rst = oracle.deer(f["w"], f["u"], f["h0"], eps=1e-5, kmax=20,
                                     y_init=near.astype(np.float64))
    assert (r["iters"], r["status"]) == (rk, rst), (r["hist"], list(rhist))
    assert_close("y", to_f64(r["y"]), ry, "f32")
    np.testing.assert_allclose(r["hist"], rhist, rtol=1e-3, atol=1e-6)
    _, kc, _, _ = oracle.deer(f["w"], f["u"], f["h0"], eps=1e-5, kmax=20)
    assert rk < kc
    # in place: the guess in the output buffer
    y = guess.clone()
    r2 = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], y=y, y_init=y, eps=1e-5, kmax=20)
    assert r2["iters"] == rk and torch.equal(y, r["y"])


@pytest.mark.parametrize("shape", DEER_SHAPES)
def test_deer_per_sequence_stopping(cuda, shape):
    """Per-sequence stopping against the oracle's per-sequence solve: each
    sequence's K, final residual and iterate; a quiet sequence stops early."""
    T, B, D = shape
    scales = [0.01] + [1.5] * (B - 1) if B > 1 else [1.5]
    inp, dv, f = _deer_case(shape, 8, scales)
    r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20, per_sequence=True)
    ry, rks, rsts, rhists = oracle.deer_per_sequence(f["w"], f["u"], f["h0"], eps=1e-5, kmax=20)
    assert r["seq_iters"] == rks, (r["seq_iters"], rks)
    assert r["status"] == (cuda.LR_OK if all(s == 0 for s in rsts) else r["status"])
    assert r["iters"] == max(rks)
    for b in range(B):
        np.testing.assert_allclose(r["seq_resid"][b], rhists[b][-1], rtol=1e-3, atol=1e-6)
    assert_close("y", to_f64(r["y"]), ry, "f32")
    if B > 1:
        assert rks[0] < max(rks)


def test_deer_per_sequence_kmax(cuda):
    """kmax reached by the loud sequences, not by the quiet one: NOT_CONVERGED,
    and each sequence's iterate is its own last one."""
    shape = (9000, 3, 256)
    inp, dv, f = _deer_case(shape, 9, [0.01, 1.5, 1.5])
    r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=3, per_sequence=True)
    ry, rks, rsts, rhists = oracle.deer_per_sequence(f["w"], f["u"], f["h0"], eps=1e-5, kmax=3)
    assert rsts[1] == oracle.DEER_NOT_CONVERGED and rsts[0] == oracle.DEER_CONVERGED
    assert r["status"] == cuda.LR_ERR_NOT_CONVERGED
    assert r["seq_iters"] == rks
    assert_close("y", to_f64(r["y"]), ry, "f32")


def test_deer_per_sequence_nonfinite_sequence(cuda):
    """A NaN input stops its own sequence at K = 1 (not finite) and the solve
    reports LR_ERR_NONFINITE, while the other sequences run to their own
    convergence and match the oracle's per-sequence solve."""
    shape = (9000, 3, 256)
    inp, dv, f = _deer_case(shape, 10, [0.01, 1.5, 1.5])
    dv["u"][4000, 2, 17] = float("nan")
    u = f["u"].copy()
    u[4000, 2, 17] = np.nan
    r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20, per_sequence=True)
    ry, rks, rsts, rhists = oracle.deer_per_sequence(f["w"], u, f["h0"], eps=1e-5, kmax=20)
    assert rsts == [oracle.DEER_CONVERGED, oracle.DEER_CONVERGED, oracle.DEER_NONFINITE]
    assert r["status"] == cuda.LR_ERR_NONFINITE
    assert r["seq_iters"] == rks and rks[2] == 1
    assert np.isnan(r["seq_resid"][2])
    y = to_f64(r["y"])
    assert_close("y of the finite sequences", y[:, :2], ry[:, :2], "f32")
    # sequence 2 holds its first iterate: NaN from the bad step on, in its channel only
    bad = np.zeros(shape, bool)
    bad[4000:, 2, 17] = True
    assert np.isnan(y[bad]).all() and np.isfinite(y[~bad]).all()
    assert_close("y of the stopped sequence", np.where(bad, 0.0, y)[:, 2], np.where(bad, 0.0, ry)[:, 2], "f32")


@pytest.mark.parametrize("shape", [(2000, 2, 256), (9000, 2, 512)])
def test_deer_bf16_warm_start_and_per_sequence(cuda, shape):
    """bf16 storage: the warm start converges in fewer iterations than the
    cold start, per-sequence stopping stops the quiet sequence first, and both
    solutions match the fp64 fixed point within the bf16 tolerance (the
    iteration counts can differ from the oracle's by the stored rounding)."""
    T, B, D = shape
    wl = W.like(W.DEER, T, B, D, "bf16")
    inp = W.make_inputs(wl, 24)
    sc = np.asarray([0.01] + [1.5] * (B - 1), np.float32)
    inp["u"] = W.store(W.to_f64(inp["u"], "bf16").astype(np.float32) * sc[None, :, None], "bf16")
    dv, f = dev_inputs(inp, "bf16"), f64_inputs(inp, "bf16")
    star = oracle.rollout_tanh(f["w"], f["u"])
    near = W.store(oracle.rollout_tanh(f["w"], f["u"] * 1.001).astype(np.float32), "bf16")
    guess = dev_inputs({"y": near}, "bf16")["y"]
    warm = cuda.deer_diag_solve_ex(dv["w"], dv["u"], None, y_init=guess, eps=1e-2, kmax=20)
    cold = cuda.deer_diag_solve_ex(dv["w"], dv["u"], None, eps=1e-2, kmax=20)
    assert warm["status"] == cold["status"] == cuda.LR_OK
    assert warm["iters"] < cold["iters"]
    assert_close("y warm", to_f64(warm["y"]), star, "bf16")
    seq = cuda.deer_diag_solve_ex(dv["w"], dv["u"], None, eps=1e-2, kmax=20, per_sequence=True)
    assert seq["status"] == cuda.LR_OK
    assert seq["seq_iters"][0] < max(seq["seq_iters"])
    assert_close("y per sequence", to_f64(seq["y"]), star, "bf16")


@pytest.mark.parametrize("shape", [(300, 3, 40), (9000, 2, 512)])
def test_deer_repeat_uses_the_last_count(cuda, shape):
    """A solve remembers its K: the next solve of the same shape enqueues K
    iterations before its first read-back and writes iterate K straight into
    y.  Solves that stop later (eps 1e-5 after 1e-2) or earlier (1e-2 after
    1e-5) than the remembered count match the oracle; a repeat takes exactly
    K iteration launches and gives the same bits."""
    inp, dv, f = _deer_case(shape, 14)

    def solve_and_check(eps):
        r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], eps=eps, kmax=20)
        ry, rk, rhist, rst = oracle.deer(f["w"], f["u"], f["h0"], eps=eps, kmax=20)
        assert (r["iters"], r["status"]) == (rk, rst), (eps, r["hist"], list(rhist))
        assert_close(f"y eps={eps}", to_f64(r["y"]), ry, "f32")
        return r

    short = solve_and_check(1e-2)
    long_ = solve_and_check(1e-5)  # later than remembered
    assert long_["iters"] > short["iters"]
    y1 = long_["y"].clone()
    again = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20)
    # the long, narrow shape adds two kernels to its K iterations: the pass that
    # publishes iteration 1's segment aggregates and the one closing the solve
    extra = 2 if shape == (9000, 2, 512) else 0
    assert again["iters"] == long_["iters"] == again["launches"] - extra
    assert torch.equal(again["y"], y1)
    solve_and_check(1e-2)  # earlier than remembered


def test_deer_ex_global_matches_deer_diag_solve(cuda):
    inp, dv, f = _deer_case((9000, 2, 512), 10)
    y, k, resid, hist, st = cuda.deer_diag_solve(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20)
    r = cuda.deer_diag_solve_ex(dv["w"], dv["u"], dv["h0"], eps=1e-5, kmax=20)
    assert (r["iters"], r["status"]) == (k, st) and torch.equal(r["y"], y)
    assert r["seq_iters"] == [k, k]


def _ode_case(shape, seed, w_value=None, u_scale=1.0, dt=None):
    T, B, D = shape
    wl = W.like(W.DEER, T, B, D, "f32")
    inp = W.make_inputs(wl, seed)
    inp["h0"] = W.normal(seed, 43, (B, D))
    inp["u"] = (inp["u"] * np.float32(u_scale)).astype(np.float32)
    if w_value is not None:
        inp["w"] = np.full(D, w_value, np.float32)
    dts = W.uniform(seed, 44, (T,), 0.1, 1.0) if dt is None else np.full(T, dt, np.float32)
    dv, f = dev_inputs(inp, "f32"), f64_inputs(inp, "f32")
    return dv, f, torch.from_numpy(dts).cuda(), dts.astype(np.float64)


@pytest.mark.parametrize("shape", DEER_SHAPES)
def test_deer_ode(cuda, shape):
    """ODE form against the oracle: K, status, residual history, iterate."""
    dv, f, dt, dtf = _ode_case(shape, 11)
    y, k, resid, hist, st, cl = cuda.deer_ode_solve(dv["w"], dv["u"], dt, dv["h0"], eps=1e-5, kmax=20)
    ry, rk, rhist, rst, rcl = oracle.deer_ode(f["w"], f["u"], dtf, f["h0"], eps=1e-5, kmax=20)
    assert (k, st) == (rk, rst), (hist, list(rhist))
    assert_close("y", to_f64(y), ry, "f32")
    np.testing.assert_allclose(hist, rhist, rtol=1e-3, atol=1e-6)
    assert cl == rcl == 0


def test_deer_ode_nonfinite_stops(cuda):
    """A NaN input makes the ODE form's first residual NaN: the solve stops at
    K = 1 with LR_ERR_NONFINITE, as the oracle does, and y holds iterate 1
    (NaN from the bad step on, in its channel only).  A clean solve of the
    same shape runs first, so the remembered count enqueues several iterations
    and the later ones must pass the residual on."""
    shape = (2000, 2, 256)
    dv, f, dt, dtf = _ode_case(shape, 14)
    _, k0, _, _, st0, _ = cuda.deer_ode_solve(dv["w"], dv["u"], dt, dv["h0"], eps=1e-5, kmax=20)
    assert st0 == cuda.LR_OK and k0 > 2
    dv["u"][700, 1, 33] = float("nan")
    u = f["u"].copy()
    u[700, 1, 33] = np.nan
    y, k, resid, hist, st, cl = cuda.deer_ode_solve(dv["w"], dv["u"], dt, dv["h0"], eps=1e-5, kmax=20)
    ry, rk, rhist, rst, rcl = oracle.deer_ode(f["w"], u, dtf, f["h0"], eps=1e-5, kmax=20)
    assert (rk, rst) == (1, oracle.DEER_NONFINITE)
    assert (k, st) == (1, cuda.LR_ERR_NONFINITE)
    assert np.isnan(resid) and np.isnan(hist[0]) and np.isnan(rhist[0])
    assert cl == rcl == 0
    y = to_f64(y)
    bad = np.zeros(shape, bool)
    bad[700:, 1, 33] = True
    assert np.isnan(y[bad]).all() and np.isfinite(y[~bad]).all()
    assert_close("y", np.where(bad, 0.0, y), np.where(bad, 0.0, ry), "f32")


def test_deer_ode_repeat_and_bf16(cuda):
    """A repeated ODE solve (the remembered count: iterate K written straight
    into y) gives the same bits; bf16 storage converges to the fp64 fixed point
    within the bf16 tolerance."""
    dv, f, dt, dtf = _ode_case((9000, 2, 512), 13)
    a = cuda.deer_ode_solve(dv["w"], dv["u"], dt, dv["h0"], eps=1e-5, kmax=20)
    ya = a[0].clone()
    b = cuda.deer_ode_solve(dv["w"], dv["u"], dt, dv["h0"], eps=1e-5, kmax=20)
    assert (b[1], b[4]) == (a[1], a[4]) and torch.equal(b[0], ya)
    ry, rk, rhist, rst, _ = oracle.deer_ode(f["w"], f["u"], dtf, f["h0"], eps=1e-5, kmax=20)
    assert (a[1], a[4]) == (rk, rst)
    assert_close("y", to_f64(ya), ry, "f32")
    T, B, D = 4000, 2, 256
    wl = W.like(W.DEER, T, B, D, "bf16")
    inp = W.make_inputs(wl, 15)
    dvb, fb = dev_inputs(inp, "bf16"), f64_inputs(inp, "bf16")
    dts = W.uniform(15, 44, (T,), 0.1, 1.0)
    y, k, resid, hist, st, cl = cuda.deer_ode_solve(dvb["w"], dvb["u"], torch.from_numpy(dts).cuda(),
                                                    None, eps=1e-2, kmax=20)
    ry, rk, rhist, rst, _ = oracle.deer_ode(fb["w"], fb["u"], dts.astype(np.float64), None, eps=1e-2,
                                            kmax=20)
    assert st == cuda.LR_OK and rst == oracle.DEER_CONVERGED and abs(k - rk) <= 1
    assert_close("y bf16", to_f64(y), oracle.rollout_ode(fb["w"], fb["u"], dts.astype(np.float64))[0],
                 "bf16")


def test_deer_ode_clamp(cuda):
    """w = -12: G = 1 + 12 (1 - tanh^2) exceeds 10 for small pre-activations
    and is clamped.  The count decides, per element, G > 10 in fp32 on the
    GPU and in fp64 in the oracle from iterates that differ by ~1e-6: the
    elements within that band of the bound may fall either way.  The
    iteration count is exact: the case (steps of 0.1) keeps every residual
    more than 0.3 decades from eps, far beyond fp32's ~1e-7 in the residual."""
    dv, f, dt, dtf = _ode_case((3000, 2, 128), 12, w_value=-12.0, u_scale=0.3, dt=0.1)
    y, k, resid, hist, st, cl = cuda.deer_ode_solve(dv["w"], dv["u"], dt, dv["h0"], eps=1e-5, kmax=60)
    ry, rk, rhist, rst, rcl = oracle.deer_ode(f["w"], f["u"], dtf, f["h0"], eps=1e-5, kmax=60)
    margin = float(np.min(np.abs(np.log10(np.asarray(rhist[:rk]) / 1e-5))))
    assert margin > 0.3, f"residual history too close to eps: {list(rhist[:rk])}"
    assert (k, st) == (rk, rst) and rst == oracle.DEER_CONVERGED, (k, hist, list(rhist))
    np.testing.assert_allclose(hist, rhist, rtol=1e-3, atol=1e-6)
    assert_close("y", to_f64(y), ry, "f32")
    assert rcl > 0 and abs(cl - rcl) <= max(4, rcl // 10000), (cl, rcl)


def test_scan_integer_valued_is_bit_exact(cuda):
    """a in {0, +1, -1}, b small integers: every association order is exact,
    so the chunked scan must equal the sequential oracle bit for bit."""
    r = np.random.default_rng(11)
    for (T, B, D) in [(4097, 2, 128), (50000, 1, 8), (999, 3, 7), (2100, 3, 7)]:
        a = r.choice([0.0, 1.0, 1.0, 1.0, -1.0], size=(T, B, D)).astype(np.float32)
        b = r.integers(-3, 4, size=(T, B, D)).astype(np.float32)
        h0 = r.integers(-5, 6, size=(B, D)).astype(np.float32)
        g = r.integers(-3, 4, size=(T, B, D)).astype(np.float32)
        ta, tb, th0, tg = (torch.from_numpy(x).cuda() for x in (a, b, h0, g))
        h = cuda.lr_scan_fwd(ta, tb, th0)
        href = oracle.scan_fwd(a, b, h0)
        assert np.array_equal(to_f64(h), href)
        da, db, dh0 = cuda.lr_scan_bwd(ta, h, tg, th0)
        rda, rdb, rdh0 = oracle.scan_bwd(a, href, g, h0)
        assert np.array_equal(to_f64(db), rdb)
        assert np.array_equal(to_f64(da), rda)
        assert np.array_equal(to_f64(dh0), rdh0)


def _dyadic(rng, T, C):
    """Coefficients a in {0, +-1/2, +-1, 2} and b, g, h0 small integers, with
    every 1/2 paired with a 2 next to it ((+-1/2, 2) or (2, +-1/2)): the running
    products stay within a factor 2 of +-1, so every partial sum the scan can
    form, in any association, is a dyadic of a few bits -- exact in fp32.
    Zeros (3%) cut the chains; the signs and pairs keep the carries nontrivial
    across every chunk boundary."""
    a = np.empty((T, C), np.float32)
    pend = np.zeros(C, np.int8)  # 1: the next step must be 2; 2: must be +-1/2
    vals = np.array([0.0, 1.0, -1.0, 0.5, -0.5, 2.0], np.float32)
    cum = np.array([0.03, 0.33, 0.63, 0.80, 0.90, 1.0])
    for t in range(T):
        pick = vals[np.searchsorted(cum, rng.random(C), side="right").clip(0, 5)]
        half = np.where(rng.random(C) < 0.5, 0.5, -0.5).astype(np.float32)
        row = np.where(pend == 1, 2.0, np.where(pend == 2, half, pick)).astype(np.float32)
        pend = np.where(pend != 0, 0, np.where(np.abs(pick) == 0.5, 1, np.where(pick == 2.0, 2, 0)))
        a[t] = row
    b = rng.integers(-3, 4, size=(T, C)).astype(np.float32)
    g = rng.integers(-3, 4, size=(T, C)).astype(np.float32)
    h0 = rng.integers(-5, 6, size=C).astype(np.float32)
    return a, b, g, h0


# every carry protocol: cluster (five shapes: clusters of 8 and of 16 CTAs,
# one-chunk clusters of many channel tiles, ragged steps and channels on the
# scalar path and on the vector path), look-back (two shapes), TMA chain (past
# the look-back budget), register walker, segmented walker (bf16 forward, both
# backwards), strip (wide), register chain (scalar path)
DYADIC_SHAPES = [(1024, 4, 256), (2048, 4, 256), (64, 40, 1000), (999, 3, 7), (1000, 3, 12), (2100, 2, 256),
                 (3001, 2, 100), (4097, 2, 128), (20000, 1, 128), (50000, 1, 8), (2100, 33, 520), (2100, 3, 7)]


@pytest.mark.parametrize("shape", DYADIC_SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scan_dyadic_is_bit_exact(cuda, shape, dtype):
    """Dyadic inputs make every association order exact, so the chunked scan
    must equal the sequential oracle bit for bit -- the chunk folds, the
    carried states and the look-back / walker aggregates included.  bf16:
    inputs are exact in bf16 and every fp32 intermediate is exact, so each
    stored output is the round-to-nearest-even of the exact value; the
    backward reads the bf16 h it stored, and so does its oracle."""
    T, B, D = shape
    C = B * D
    a, b, g, h0 = _dyadic(np.random.default_rng(101), T, C)
    sh = lambda x: x.reshape((T, B, D) if x.ndim == 2 else (B, D))
    a, b, g, h0 = (sh(x) for x in (a, b, g, h0))
    ta, tb, tg, th0 = (to_dev(W.store(x, dtype), dtype) for x in (a, b, g, h0))
    a64, b64, g64, h064 = (x.astype(np.float64) for x in (a, b, g, h0))
    h = cuda.lr_scan_fwd(ta, tb, th0)
    href = oracle.scan_fwd(a64, b64, h064)
    hs = W.store(href, dtype)  # exact for fp32; the rounding the kernel's store does for bf16
    got = h.cpu()
    if dtype == "bf16":
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), hs)
    else:
        assert np.array_equal(got.numpy(), hs)
    da, db, dh0 = cuda.lr_scan_bwd(ta, h, tg, th0)
    rda, rdb, rdh0 = oracle.scan_bwd(a64, W.to_f64(hs, dtype), g64, h064)
    for name, x, r in (("da", da, rda), ("db", db, rdb), ("dh0", dh0, rdh0)):
        xs = x.cpu()
        xs = xs.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else xs.numpy()
        assert np.array_equal(xs, W.store(r, dtype)), name


@pytest.mark.parametrize("shape", [(1024, 4, 256), (2048, 4, 256), (2100, 2, 256), (4097, 2, 128),
                                   (20000, 1, 128), (64, 40, 1000), (2100, 33, 520)])
def test_scan_back_to_back_fresh_inputs(cuda, shape):
    """Calls of one shape back to back with different inputs, on one stream:
    every launch takes a fresh epoch on the device, so no tile may accept a
    packet the previous call left in the same slot."""
    T, B, D = shape
    for seed in (31, 32, 33):
        _scan_case(cuda, T, B, D, "f32", seed=seed)


@pytest.mark.parametrize("shape", [(1024, 4, 256), (2048, 4, 256), (2100, 2, 256), (4097, 2, 128),
                                   (20000, 1, 128), (70, 33, 520), (2100, 33, 520)])
def test_scan_graph_replay_takes_fresh_inputs(cuda, shape):
    """The forward and backward scans captured into a CUDA graph: each replay,
    with new values copied into the captured buffers, matches the oracle (the
    launches take their epochs on the device, so a replay never accepts the
    previous replay's packets)."""
    T, B, D = shape
    wl = W.like(W.SCAN_TINY, T, B, D, "f32")

    def inputs(seed):
        inp = W.make_inputs(wl, seed)
        inp["h0"] = W.store(W.normal(seed, 99, (B, D)), "f32")
        return inp

    first = dev_inputs(inputs(40), "f32")
    a, b, h0, gg = (first[k].clone() for k in ("a", "b", "h0", "g"))
    h, da, db = (torch.empty_like(a) for _ in range(3))
    dh0 = torch.empty_like(h0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # uncaptured first call: sizes the workspace
        cuda.lr_scan_fwd(a, b, h0, h)
        cuda.lr_scan_bwd(a, h, gg, h0, da, db, dh0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cuda.lr_scan_fwd(a, b, h0, h)
        cuda.lr_scan_bwd(a, h, gg, h0, da, db, dh0)
    for seed in (41, 42, 43):
        inp = inputs(seed)
        dv, f = dev_inputs(inp, "f32"), f64_inputs(inp, "f32")
        for dst, k in ((a, "a"), (b, "b"), (h0, "h0"), (gg, "g")):
            dst.copy_(dv[k])
        graph.replay()
        torch.cuda.synchronize()
        href = oracle.scan_fwd(f["a"], f["b"], f["h0"])
        assert_close("h", to_f64(h), href, "f32")
        rda, rdb, rdh0 = oracle.scan_bwd(f["a"], href, f["g"], f["h0"])
        assert_close("da", to_f64(da), rda, "f32")
        assert_close("db", to_f64(db), rdb, "f32")
        assert_close("dh0", to_f64(dh0), rdh0, "f32")
    assert cuda.last_error() == cuda.LR_OK


def test_error_return_still_orders_the_next_call(cuda):
    """A call that returns an error after it began enqueueing still records
    the workspace event: the next call, on another stream, waits for what the
    failed call enqueued.  The failure is injected on the host (the hook
    enqueues a kernel that sleeps ~50 ms then fills b with 7, and returns
    LR_ERR_CUDA); the next call scans a = 0, so h must be b = 7."""
    T, B, D = 1024, 4, 256
    b = torch.zeros(T, B, D, device="cuda")
    a = torch.zeros_like(b)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    assert cuda.test_fail_after_enqueue(b, 7.0, 50_000_000, stream=s1) == cuda.LR_ERR_CUDA
    h = torch.empty_like(b)
    with torch.cuda.stream(s2):
        cuda.lr_scan_fwd(a, b, None, h, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(h, torch.full_like(h, 7.0))


def test_scan_a_zero_gives_b_bit_exact(cuda):
    b = torch.randn(3000, 2, 64, device="cuda")
    h = cuda.lr_scan_fwd(torch.zeros_like(b), b, torch.randn(2, 64, device="cuda"))
    assert torch.equal(h, b)


def test_unaligned_pointers_take_scalar_path(cuda):
    T, B, D = 300, 2, 64
    wl = W.like(W.SCAN_TINY, T, B, D, "f32")
    inp = W.make_inputs(wl, 8)
    n = T * B * D
    buf_a = torch.empty(n + 1, device="cuda")
    buf_b = torch.empty(n + 1, device="cuda")
    buf_h = torch.empty(n + 1, device="cuda")
    a = buf_a[1:].view(T, B, D)
    b = buf_b[1:].view(T, B, D)
    h = buf_h[1:].view(T, B, D)
    a.copy_(torch.from_numpy(inp["a"]))
    b.copy_(torch.from_numpy(inp["b"]))
    cuda.lr_scan_fwd(a, b, None, h)
    assert_close("h", to_f64(h), oracle.scan_fwd(inp["a"], inp["b"]), "f32")


def test_null_optional_states(cuda):
    T, B, D = 130, 2, 16
    wl = W.like(W.SCAN_TINY, T, B, D, "f32")
    inp = W.make_inputs(wl, 9)
    dv, f = dev_inputs(inp, "f32"), f64_inputs(inp, "f32")
    h = cuda.lr_scan_fwd(dv["a"], dv["b"], None)
    href = oracle.scan_fwd(f["a"], f["b"])
    assert_close("h", to_f64(h), href, "f32")
    da, db, dh0 = cuda.lr_scan_bwd(dv["a"], h, dv["g"], None, want_dh0=False)
    assert dh0 is None
    rda, rdb, _ = oracle.scan_bwd(f["a"], href, f["g"])
    assert_close("da", to_f64(da), rda, "f32")


def test_empty_problems(cuda):
    e = torch.empty(0, 3, 8, device="cuda")
    h = cuda.lr_scan_fwd(e, e)
    assert h.shape == (0, 3, 8)
    dh0 = torch.full((3, 8), 7.0, device="cuda")
    cuda.lr_scan_bwd(e, e, e, dh0=dh0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dh0) == 0
    y, k, resid, hist, st = cuda.deer_diag_solve(torch.zeros(8, device="cuda"), e)
    assert (k, st) == (0, cuda.LR_OK)
    # LSTM cell: the bias gradients and dc0 of an empty sequence are zero
    bias = [torch.zeros(8, device="cuda") for _ in range(4)]
    h, c = cuda.lstm_cell_fwd(e, e, e, e, *bias)
    assert h.shape == (0, 3, 8)
    out = {k: torch.full((8,), 7.0, device="cuda") for k in ("dbf", "dbi", "dbc", "dbo")}
    out["dc0"] = torch.full((3, 8), 7.0, device="cuda")
    g = cuda.lstm_cell_bwd(e, e, e, e, *bias, e, e, out=out)
    torch.cuda.synchronize()
    for k in ("dbf", "dbi", "dbc", "dbo", "dc0"):
        assert torch.count_nonzero(g[k]) == 0, k


def test_lstm_cell_null_initial_state(cuda):
    T, B, D = 130, 2, 16
    wl = W.like(W.LSTM, T, B, D, "f32")
    inp = W.make_inputs(wl, 9)
    dv, f = dev_inputs(inp, "f32"), f64_inputs(inp, "f32")
    z = [dv[k] for k in ("zf", "zi", "zc", "zo")] + [dv[k] for k in ("bf", "bi", "bc", "bo")]
    zr = [f[k] for k in ("zf", "zi", "zc", "zo")] + [f[k] for k in ("bf", "bi", "bc", "bo")]
    h, c = cuda.lstm_cell_fwd(*z, None)
    rh, rc = oracle.lstm_fwd(*zr)
    assert_close("h", to_f64(h), rh, "f32")
    g = cuda.lstm_cell_bwd(*z, c, dv["dh"], None, want_dc0=False)
    assert g.get("dc0") is None
    ref = oracle.lstm_bwd(*zr, rc, f["dh"])
    assert_close("dzf", to_f64(g["dzf"]), ref[0], "f32")
    assert_close("dbf", to_f64(g["dbf"]), ref[4], "f32")


@pytest.mark.parametrize("shape", [(2048, 4, 256), (64, 40, 1000)])
def test_repeat_is_bitwise_deterministic(cuda, shape):
    T, B, D = shape
    wl = W.like(W.SRU, T, B, D, "f32")
    inp = W.make_inputs(wl, 4)
    dv = dev_inputs(inp, "f32")
    outs = []
    for _ in range(3):
        h, c = cuda.sru_fwd(dv["xt"], dv["uf"], dv["ur"], dv["x"], dv["bf"], dv["br"], dv["c0"])
        g = cuda.sru_bwd(dv["xt"], dv["uf"], dv["ur"], dv["x"], dv["bf"], dv["br"], c, dv["dh"], dv["c0"])
        outs.append([h.clone(), c.clone()] + [g[k].clone() for k in sorted(g)])
    for o in outs[1:]:
        for x, y in zip(outs[0], o):
            assert torch.equal(x, y)


def test_long_scan_is_bitwise_deterministic(cuda):
    """Many chunks along time: tiles and walkers interleave differently from
    run to run, yet every carry is folded in an order fixed by position."""
    T, B, D = 300000, 1, 128
    wl = W.like(W.SCAN_LONG, T, B, D)
    dv = dev_inputs(W.make_inputs(wl, 13), "f32")
    hs = [cuda.lr_scan_fwd(dv["a"], dv["b"], dv["h0"]).clone() for _ in range(4)]
    for h in hs[1:]:
        assert torch.equal(h, hs[0])


def test_calls_on_two_streams(cuda):
    T, B, D = 4096, 2, 128
    wl = W.like(W.SCAN_TINY, T, B, D, "f32")
    inp = W.make_inputs(wl, 12)
    dv, f = dev_inputs(inp, "f32"), f64_inputs(inp, "f32")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    for i in range(6):
        s = s1 if i % 2 else s2
        with torch.cuda.stream(s):
            outs.append(cuda.lr_scan_fwd(dv["a"], dv["b"], dv["h0"], stream=s))
    torch.cuda.synchronize()
    href = oracle.scan_fwd(f["a"], f["b"], f["h0"])
    for h in outs:
        assert_close("h", to_f64(h), href, "f32")


def test_lookback_wait_runs_out_cleanly(cuda):
    """A chunk whose predecessor never publishes gives up after the poll limit,
    records LR_ERR_TIMEOUT, and the context stays usable."""
    assert cuda.last_error() == cuda.LR_OK
    assert cuda.test_lookback_timeout(2000) == cuda.LR_OK
    assert cuda.last_error() == cuda.LR_ERR_TIMEOUT
    assert cuda.last_error() == cuda.LR_OK  # cleared by the read
    _scan_case(cuda, 500, 2, 64, "f32")


def test_argument_errors(cuda):
    a = torch.randn(10, 2, 8, device="cuda")
    with pytest.raises(ValueError):
        cuda.lr_scan_fwd(a, torch.randn(10, 2, 7, device="cuda"))
    with pytest.raises(TypeError):
        cuda.lr_scan_fwd(a.double(), a.double())
    lib = cuda.load()
    assert lib.lr_scan_fwd(None, None, None, None, 2, 10, 8, 0, None) == cuda.LR_ERR_INVALID_ARG
    bad = a.view(-1)[1:].view(torch.uint8)[1:]  # byte-offset pointer
    import ctypes
    st = lib.lr_scan_fwd(ctypes.c_void_p(bad.data_ptr()), ctypes.c_void_p(a.data_ptr()), None,
                         ctypes.c_void_p(a.data_ptr()), 1, 1, 1, 0, None)
    assert st == cuda.LR_ERR_ALIGN


def test_activations_error_bound(cuda):
    """The kernels' tanh and sigmoid (exponential forms on the hardware
    exponential) against fp64 on a dense grid, the saturated tails, signed
    zeros, infinities and NaN: absolute error below 1e-6 everywhere."""
    grid = np.concatenate([np.linspace(-30, 30, 600001), np.linspace(-1e-3, 1e-3, 20001),
                           np.array([0.0, -0.0, 88.0, -88.0, 200.0, -200.0, np.inf, -np.inf])])
    x = grid.astype(np.float32)
    th, sg = cuda.test_activations(torch.from_numpy(x).cuda())
    th, sg = th.cpu().numpy().astype(np.float64), sg.cpu().numpy().astype(np.float64)
    xd = x.astype(np.float64)
    with np.errstate(over="ignore"):
        ref_sg = 1.0 / (1.0 + np.exp(-xd))
    assert np.max(np.abs(th - np.tanh(xd))) < 1e-6
    assert np.max(np.abs(sg - ref_sg)) < 1e-6
    assert np.all(th * xd >= 0)  # odd: never the wrong sign
    assert th[-2] == 1.0 and th[-1] == -1.0 and sg[-2] == 1.0 and sg[-1] == 0.0
    nan_th, nan_sg = cuda.test_activations(torch.tensor([float("nan")], device="cuda"))
    assert torch.isnan(nan_th).all() and torch.isnan(nan_sg).all()


def test_expm1_error_bound(cuda):
    """The kernels' e^x - 1 (Taylor series below |x| = 1/4, the hardware
    exponential above) against fp64: relative error below 2e-6 on a dense grid
    through the switch, tiny arguments and the range the ODE form uses; the
    limits at +-inf and NaN."""
    grid = np.concatenate([np.linspace(-12, 12, 480001), np.linspace(-0.3, 0.3, 60001),
                           np.geomspace(1e-30, 1e-2, 2001), -np.geomspace(1e-30, 1e-2, 2001),
                           np.array([0.25, -0.25, np.nextafter(np.float32(0.25), np.float32(0)),
                                     -np.nextafter(np.float32(0.25), np.float32(0))])])
    x = grid.astype(np.float32)
    _, _, em = cuda.test_activations(torch.from_numpy(x).cuda(), with_expm1=True)
    em = em.cpu().numpy().astype(np.float64)
    ref = np.expm1(x.astype(np.float64))
    rel = np.abs(em - ref) / np.maximum(np.abs(ref), 1e-300)
    assert np.max(rel) < 2e-6, (x[np.argmax(rel)], np.max(rel))
    special = torch.tensor([float("inf"), float("-inf"), float("nan")], device="cuda")
    _, _, es = cuda.test_activations(special, with_expm1=True)
    es = es.cpu().numpy()
    assert es[0] == np.inf and es[1] == -1.0 and np.isnan(es[2])


@pytest.mark.parametrize("kmax", [1, 3, 4, 5, 6])
def test_deer_kmax_across_launch_batches(cuda, kmax):
    """Iterations are enqueued four at a time and those past the stopping test
    do nothing: stopping at kmax inside, at the end of and past a batch gives
    the oracle's iterate, count, status and residual history."""
    T, B, D = 3001, 2, 128
    wl = W.like(W.DEER, T, B, D, "f32")
    inp = W.make_inputs(wl, 21)
    dv, f = dev_inputs(inp, "f32"), f64_inputs(inp, "f32")
    y, k, resid, hist, st = cuda.deer_diag_solve(dv["w"], dv["u"], None, eps=1e-5, kmax=kmax)
    ry, rk, rhist, rst = oracle.deer(f["w"], f["u"], None, eps=1e-5, kmax=kmax)
    assert (k, st == cuda.LR_OK) == (rk, rst == oracle.DEER_CONVERGED), (k, st, rk, rst)
    assert_close("y", to_f64(y), ry, "f32")
    np.testing.assert_allclose(hist[:k], rhist, rtol=1e-3, atol=1e-6)


def test_deer_nonfinite_stops_the_batch(cuda):
    """A NaN input makes the first residual non-finite: the solve stops there
    (the rest of the batch returns at once) and reports LR_ERR_NONFINITE."""
    T, B, D = 2000, 1, 128
    wl = W.like(W.DEER, T, B, D, "f32")
    inp = W.make_inputs(wl, 22)
    dv = dev_inputs(inp, "f32")
    dv["u"][100, 0, 7] = float("nan")
    y, k, resid, hist, st = cuda.deer_diag_solve(dv["w"], dv["u"], None, eps=1e-5, kmax=20)
    assert st == cuda.LR_ERR_NONFINITE and k == 1
    assert cuda.last_error() == cuda.LR_OK


@pytest.mark.parametrize("shape", [(300, 3, 40), (9000, 2, 512), (45, 40, 1000)])
def test_deer_bf16(cuda, shape):
    """bf16 storage (the iterates are stored in bf16, so the stopping test sees
    bf16 iterates): converges, and the solution matches the fp64 fixed point
    within the bf16 tolerance.  The iteration count can differ from the fp64
    oracle's by the rounding of the stored iterate; fp32 checks it exactly."""
    T, B, D = shape
    wl = W.like(W.DEER, T, B, D, "bf16")
    inp = W.make_inputs(wl, 23)
    dv, f = dev_inputs(inp, "bf16"), f64_inputs(inp, "bf16")
    y, k, resid, hist, st = cuda.deer_diag_solve(dv["w"], dv["u"], None, eps=1e-2, kmax=20)
    ry, rk, rhist, rst = oracle.deer(f["w"], f["u"], None, eps=1e-2, kmax=20)
    assert st == cuda.LR_OK and rst == oracle.DEER_CONVERGED
    assert abs(k - rk) <= 1, (k, rk, hist, list(rhist))
    assert_close("y", to_f64(y), ry, "bf16")


@pytest.mark.parametrize("shape", SHAPES[:9] + WIDE + [(20000, 1, 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_deer_bwd(cuda, shape, dtype):
    """Gradient through the DEER solution: du, dw, dh0 against the oracle on
    the same stored solution y and upstream gradient."""
    T, B, D = shape
    wl = W.like(W.DEER, T, B, D, dtype)
    inp = W.make_inputs(wl, 31)
    h0 = W.store(W.normal(31, 44, (B, D)), dtype)
    y = W.store(oracle.rollout_tanh(np.asarray(inp["w"], np.float64), W.to_f64(inp["u"], dtype),
                                    W.to_f64(h0, dtype)), dtype)
    g = W.store(W.normal(31, 45, (T, B, D)), dtype)
    dv = dev_inputs({"w": inp["w"], "y": y, "h0": h0, "g": g}, dtype)
    f = f64_inputs({"w": inp["w"], "y": y, "h0": h0, "g": g}, dtype)
    du, dw, dh0 = cuda.deer_diag_bwd(dv["w"], dv["y"], dv["g"], dv["h0"])
    rdu, rdw, rdh0 = oracle.deer_bwd(f["w"], f["y"], f["g"], f["h0"])
    assert_close("du", to_f64(du), rdu, dtype)
    assert_close("dw", to_f64(dw), rdw, dtype)
    assert_close("dh0", to_f64(dh0), rdh0, dtype)
