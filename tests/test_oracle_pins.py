"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each test checks the oracle against something other than its own loop: a
closed form, a library linear solve (scipy), a library filter, central finite
differences, a brute-force evaluation of the associative operator in random
tree orders, Newton's method written from the residual function, or a
hand-worked example under tests/golden/.  A plausible slip in the oracle (a
dropped term, a wrong sign or time index, a transposed operand) fails at least
one of them.  CPU only.
"""
import os
import random

import numpy as np
import pytest
import scipy.linalg
import scipy.signal

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _bidiag_solve(a, rhs):
    """Solve (I - S_a) h = rhs for one channel, S_a having a_t at (t, t-1)."""
    T = a.shape[0]
    ab = np.zeros((2, T))
    ab[0] = 1.0
    ab[1, :-1] = -a[1:]
    return scipy.linalg.solve_banded((1, 0), ab, rhs)


def _bidiag_solve_T(a, rhs):
    """Solve (I - S_a)^T x = rhs (upper bidiagonal) for one channel."""
    T = a.shape[0]
    ab = np.zeros((2, T))
    ab[1] = 1.0
    ab[0, 1:] = -a[1:]
    return scipy.linalg.solve_banded((0, 1), ab, rhs)


# ------------------------------------------------------------ forward scan

def test_golden_dyadic_example():
    vals = {}
    with open(os.path.join(GOLDEN, "scan_dyadic_T4.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                vals[k] = np.array([float(x) for x in v])
    a, b, g = (vals[k].reshape(4, 1) for k in ("a", "b", "g"))
    h0 = vals["h0"].reshape(1)
    h = oracle.scan_fwd(a, b, h0)
    assert np.array_equal(h[:, 0], vals["h"])
    da, db, dh0 = oracle.scan_bwd(a, h, g, h0)
    assert np.array_equal(db[:, 0], vals["db"])
    assert np.array_equal(da[:, 0], vals["da"])
    assert np.array_equal(dh0, vals["dh0"])


def test_scan_a_zero_gives_b_exactly():
    b = rng.standard_normal((37, 3, 5))
    h = oracle.scan_fwd(np.zeros_like(b), b, rng.standard_normal((3, 5)))
    assert np.array_equal(h, b)


def test_scan_a_one_is_running_sum():
    b = rng.standard_normal((200, 7))
    h0 = rng.standard_normal(7)
    h = oracle.scan_fwd(np.ones_like(b), b, h0)
    np.testing.assert_allclose(h, h0 + np.cumsum(b, axis=0), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("alpha", [0.3, -0.7, 0.99, 1.5])
def test_scan_constant_coefficients_geometric_series(alpha):
    T, beta, h0 = 60, 0.25, -1.5
    h = oracle.scan_fwd(np.full((T, 1), alpha), np.full((T, 1), beta), np.array([h0]))
    t = np.arange(T) + 1.0
    closed = alpha ** t * h0 + beta * (1 - alpha ** t) / (1 - alpha)
    np.testing.assert_allclose(h[:, 0], closed, rtol=1e-11, atol=1e-12)


def test_scan_constant_a_matches_iir_filter():
    alpha = 0.87
    b = rng.standard_normal((300, 4))
    h0 = rng.standard_normal(4)
    h = oracle.scan_fwd(np.full_like(b, alpha), b, h0)
    for c in range(4):
        ref, _ = scipy.signal.lfilter([1.0], [1.0, -alpha], b[:, c], zi=[alpha * h0[c]])
        np.testing.assert_allclose(h[:, c], ref, rtol=1e-12, atol=1e-12)


def test_scan_time_varying_matches_banded_solve():
    T, C = 150, 6
    a = rng.uniform(-1.2, 1.2, (T, C))
    b = rng.standard_normal((T, C))
    h0 = rng.standard_normal(C)
    h = oracle.scan_fwd(a, b, h0)
    for c in range(C):
        rhs = b[:, c].copy()
        rhs[0] += a[0, c] * h0[c]
        np.testing.assert_allclose(h[:, c], _bidiag_solve(a[:, c], rhs), rtol=1e-10, atol=1e-10)


def _combine(x, y):
    """(a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2), earlier element on the left."""
    return (x[0] * y[0], y[0] * x[1] + y[1])


def _random_tree(elems, r):
    if len(elems) == 1:
        return elems[0]
    k = r.randint(1, len(elems) - 1)
    return _combine(_random_tree(elems[:k], r), _random_tree(elems[k:], r))


def _blelloch_inclusive(elems):
    """Up-sweep / down-sweep (work-efficient) exclusive scan, made inclusive."""
    n = len(elems)
    x = list(elems)
    d = 1
    while d < n:
        for i in range(2 * d - 1, n, 2 * d):
            x[i] = _combine(x[i - d], x[i])
        d *= 2
    x[n - 1] = (1.0, 0.0)  # identity
    d = n // 2
    while d >= 1:
        for i in range(2 * d - 1, n, 2 * d):
            left = x[i - d]
            x[i - d] = x[i]
            x[i] = _combine(x[i], left)
        d //= 2
    return [_combine(x[i], elems[i]) for i in range(n)]


def test_scan_brute_force_tree_orders_dyadic():
    """Every parenthesisation of the operator reproduces the sequential oracle
    bit for bit on dyadic inputs (all intermediate values exact)."""
    r = random.Random(7)
    for trial in range(40):
        T = r.randint(1, 16)
        a = np.array([r.choice([0.0, 0.5, -0.5, 1.0, -1.0, 2.0]) for _ in range(T)])
        b = np.array([float(r.randint(-4, 4)) for _ in range(T)])
        h0 = float(r.randint(-3, 3))
        h = oracle.scan_fwd(a.reshape(T, 1), b.reshape(T, 1), np.array([h0]))[:, 0]
        elems = [(0.0, h0)] + [(a[t], b[t]) for t in range(T)]
        for t in range(T):
            for _ in range(3):
                assert _random_tree(elems[: t + 2], r)[1] == h[t]
        if T in (1, 2, 4, 8, 16):
            # element 0 carries h0; pad to a power of two with identities
            seq = [(a[0], a[0] * h0 + b[0])] + [(a[t], b[t]) for t in range(1, T)]
            inc = _blelloch_inclusive(seq)
            assert [v[1] for v in inc] == list(h)


# ----------------------------------------------------------- backward scan

def _fd(fun, x, eps=1e-6):
    g = np.zeros_like(x)
    flat = x.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + eps
        fp = fun()
        flat[i] = old - eps
        fm = fun()
        flat[i] = old
        g.reshape(-1)[i] = (fp - fm) / (2 * eps)
    return g


def test_scan_bwd_finite_differences():
    T, C = 9, 3
    a = rng.uniform(-0.9, 0.9, (T, C))
    b = rng.standard_normal((T, C))
    h0 = rng.standard_normal(C)
    g = rng.standard_normal((T, C))
    loss = lambda: float(np.sum(g * oracle.scan_fwd(a, b, h0)))
    h = oracle.scan_fwd(a, b, h0)
    da, db, dh0 = oracle.scan_bwd(a, h, g, h0)
    np.testing.assert_allclose(da, _fd(loss, a), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(db, _fd(loss, b), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(dh0, _fd(loss, h0), rtol=1e-7, atol=1e-8)


def test_scan_bwd_is_transposed_solve():
    T, C = 120, 4
    a = rng.uniform(-1.1, 1.1, (T, C))
    b = rng.standard_normal((T, C))
    g = rng.standard_normal((T, C))
    h = oracle.scan_fwd(a, b)
    da, db, dh0 = oracle.scan_bwd(a, h, g)
    for c in range(C):
        np.testing.assert_allclose(db[:, c], _bidiag_solve_T(a[:, c], g[:, c]), rtol=1e-10, atol=1e-10)
    # h0 absent means zeros: da_0 = 0
    assert np.all(da[0] == 0.0)


# --------------------------------------------------------------------- SRU

def _sru_inputs(T, B, D, seed=5):
    r = np.random.default_rng(seed)
    return dict(xt=r.standard_normal((T, B, D)), uf=r.standard_normal((T, B, D)),
                ur=r.standard_normal((T, B, D)), x=r.standard_normal((T, B, D)),
                bf=r.standard_normal(D), br=r.standard_normal(D),
                c0=r.standard_normal((B, D)))


def test_sru_forget_closed_gives_c_equal_xt():
    p = _sru_inputs(20, 2, 3)
    p["uf"][:] = -40.0
    p["bf"][:] = 0.0
    h, c = oracle.sru_fwd(**p)
    np.testing.assert_allclose(c, p["xt"], rtol=0, atol=1e-15)


def test_sru_reset_gate_limits():
    p = _sru_inputs(20, 2, 3)
    p["br"][:] = 0.0
    p["ur"][:] = 40.0
    h, c = oracle.sru_fwd(**p)
    np.testing.assert_allclose(h, np.tanh(c), rtol=0, atol=1e-15)
    p["ur"][:] = -40.0
    h, c = oracle.sru_fwd(**p)
    np.testing.assert_allclose(h, p["x"], rtol=0, atol=1e-15)


def test_sru_memory_is_linear_recurrence_solve():
    p = _sru_inputs(80, 2, 3)
    h, c = oracle.sru_fwd(**p)
    f = 1.0 / (1.0 + np.exp(-(p["uf"] + p["bf"])))
    for bb in range(2):
        for d in range(3):
            a = f[:, bb, d]
            rhs = (1 - a) * p["xt"][:, bb, d]
            rhs[0] += a[0] * p["c0"][bb, d]
            np.testing.assert_allclose(c[:, bb, d], _bidiag_solve(a, rhs), rtol=1e-11, atol=1e-12)


def test_sru_bwd_finite_differences():
    T, B, D = 7, 2, 3
    p = _sru_inputs(T, B, D)
    dh = np.random.default_rng(9).standard_normal((T, B, D))
    loss = lambda: float(np.sum(dh * oracle.sru_fwd(**p)[0]))
    h, c = oracle.sru_fwd(**p)
    dxt, duf, dur, dx, dbf, dbr, dc0 = oracle.sru_bwd(c=c, dh=dh, **p)
    for got, key in ((dxt, "xt"), (duf, "uf"), (dur, "ur"), (dx, "x"),
                     (dbf, "bf"), (dbr, "br"), (dc0, "c0")):
        np.testing.assert_allclose(got, _fd(loss, p[key]), rtol=1e-6, atol=1e-8, err_msg=key)


# ---------------------------------------------------- LSTM cell-state scan

def _lstm_inputs(T, B, D, seed=21):
    r = np.random.default_rng(seed)
    p = {k: r.standard_normal((T, B, D)) for k in ("zf", "zi", "zc", "zo")}
    p.update({k: r.standard_normal(D) for k in ("bf", "bi", "bc", "bo")})
    p["c0"] = r.standard_normal((B, D))
    return p


def _gilr(p):
    """Tie the input gate to the forget gate: i = sigma(-(zf + bf)) = 1 - f."""
    q = dict(p)
    q["zi"], q["bi"] = -p["zf"], -p["bf"]
    return q


def test_lstm_gilr_tie_is_the_sru_cell():
    # with i = 1 - f and the candidate as SRU's xt, the cell is SRU's memory
    # c_t = f c_{t-1} + (1 - f) xt, and h = o tanh(c) is SRU's output with
    # reset gate o and highway input x = 0
    p = _gilr(_lstm_inputs(40, 2, 3))
    h, c = oracle.lstm_fwd(**p)
    xt = np.tanh(p["zc"] + p["bc"])
    zero = np.zeros_like(xt)
    hs, cs = oracle.sru_fwd(xt, p["zf"], p["zo"], zero, p["bf"], p["bo"], p["c0"])
    np.testing.assert_allclose(c, cs, rtol=0, atol=1e-13)
    np.testing.assert_allclose(h, hs, rtol=0, atol=1e-13)


def test_lstm_bwd_gilr_tie_is_the_sru_gradient():
    # chain rule through the tie zi = -zf: SRU's duf = dzf - dzi, its dxt
    # times (1 - xt^2) is dzc (xt = tanh(zc + bc)), its dur is dzo
    T, B, D = 30, 2, 3
    p = _gilr(_lstm_inputs(T, B, D))
    dh = np.random.default_rng(4).standard_normal((T, B, D))
    h, c = oracle.lstm_fwd(**p)
    dzf, dzi, dzc, dzo, dbf, dbi, dbc, dbo, dc0 = oracle.lstm_bwd(c=c, dh=dh, **p)
    xt = np.tanh(p["zc"] + p["bc"])
    zero = np.zeros_like(xt)
    dxt, duf, dur, _, sbf, sbr, sc0 = oracle.sru_bwd(xt, p["zf"], p["zo"], zero, p["bf"],
                                                     p["bo"], c, dh, p["c0"])
    tol = dict(rtol=0, atol=1e-12)
    np.testing.assert_allclose(dzf - dzi, duf, **tol)
    np.testing.assert_allclose(dzc, dxt * (1 - xt * xt), **tol)
    np.testing.assert_allclose(dzo, dur, **tol)
    np.testing.assert_allclose(dbf - dbi, sbf, **tol)
    np.testing.assert_allclose(dbo, sbr, **tol)
    np.testing.assert_allclose(dc0, sc0, **tol)


def test_lstm_gates_open_is_running_sum():
    # f = i = o = 1 exactly (sigmoid of +1000 rounds to 1): C = c0 + cumsum(C~)
    p = _lstm_inputs(50, 2, 3)
    for k in ("zf", "zi", "zo"):
        p[k][:] = 1000.0
    h, c = oracle.lstm_fwd(**p)
    ref = p["c0"][None] + np.cumsum(np.tanh(p["zc"] + p["bc"]), axis=0)
    np.testing.assert_allclose(c, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(h, np.tanh(ref), rtol=1e-13, atol=1e-13)


def test_lstm_forget_closed_has_no_memory():
    # f = 0 exactly (sigmoid of -1000 is 0): every row is its own one-step
    # problem whatever came before
    T, B, D = 12, 2, 3
    p = _lstm_inputs(T, B, D)
    p["zf"][:] = -1000.0
    h, c = oracle.lstm_fwd(**p)
    for t in range(T):
        row = {k: (v[t:t + 1] if v.ndim == 3 else v) for k, v in p.items() if k != "c0"}
        c0 = np.random.default_rng(t).standard_normal((B, D))
        ht, ct = oracle.lstm_fwd(**row, c0=c0)
        np.testing.assert_array_equal(ct[0], c[t])
        np.testing.assert_array_equal(ht[0], h[t])


def test_lstm_cell_is_linear_recurrence_solve():
    T, B, D = 80, 2, 3
    p = _lstm_inputs(T, B, D)
    h, c = oracle.lstm_fwd(**p)
    sig = lambda z: 1.0 / (1.0 + np.exp(-z))
    f = sig(p["zf"] + p["bf"])
    ig = sig(p["zi"] + p["bi"]) * np.tanh(p["zc"] + p["bc"])
    for bb in range(B):
        for d in range(D):
            rhs = ig[:, bb, d].copy()
            rhs[0] += f[0, bb, d] * p["c0"][bb, d]
            np.testing.assert_allclose(c[:, bb, d], _bidiag_solve(f[:, bb, d], rhs),
                                       rtol=1e-11, atol=1e-12)


def test_lstm_bwd_finite_differences():
    T, B, D = 7, 2, 3
    p = _lstm_inputs(T, B, D)
    dh = np.random.default_rng(9).standard_normal((T, B, D))
    loss = lambda: float(np.sum(dh * oracle.lstm_fwd(**p)[0]))
    h, c = oracle.lstm_fwd(**p)
    got = oracle.lstm_bwd(c=c, dh=dh, **p)
    keys = ("zf", "zi", "zc", "zo", "bf", "bi", "bc", "bo", "c0")
    for g, key in zip(got, keys):
        np.testing.assert_allclose(g, _fd(loss, p[key]), rtol=1e-6, atol=1e-8, err_msg=key)


# -------------------------------------------------------------------- DEER

def test_rollout_w_zero_is_tanh():
    u = rng.standard_normal((50, 2, 4))
    y = oracle.rollout_tanh(np.zeros(4), u, rng.standard_normal((2, 4)))
    np.testing.assert_allclose(y, np.tanh(u), rtol=0, atol=1e-15)


def test_rollout_small_signal_is_linear_recurrence():
    """|tanh z - z| <= |z|^3 / 3: at amplitude 1e-6 the rollout equals the
    linear recurrence y_t = w y_{t-1} + u_t within that term, carried through
    the recurrence (a factor 1 / (1 - max|w|)), plus rounding."""
    T, D = 200, 5
    r = np.random.default_rng(38)
    w = r.uniform(-0.9, 0.9, D)
    u = 1e-6 * r.standard_normal((T, 1, D))
    y = oracle.rollout_tanh(w, u)
    for d in range(D):
        lin = _bidiag_solve(np.full(T, w[d]), u[:, 0, d])
        zmax = np.abs(w[d] * np.concatenate([[0.0], lin[:-1]]) + u[:, 0, d]).max()
        bound = 2 * zmax ** 3 / 3 / (1 - abs(w[d])) + 1e-19
        assert bound < 1e-3 * np.abs(lin).max()
        np.testing.assert_allclose(y[:, 0, d], lin, rtol=0, atol=bound)


def test_deer_step_is_newton_on_residual():
    """One iteration equals y - J_F(y)^{-1} F(y) for F(y)_t = y_t - tanh(w y_{t-1} + u_t),
    with J_F formed by differentiating F and solved by a banded library solve."""
    T, B, D = 40, 2, 3
    w = rng.uniform(-0.9, 0.9, D)
    u = rng.standard_normal((T, B, D))
    h0 = rng.standard_normal((B, D))
    y = rng.standard_normal((T, B, D)) * 0.5
    ynew, rho = oracle.deer_step(w, u, y, h0)
    ref = np.empty_like(y)
    for bb in range(B):
        for d in range(D):
            yc = y[:, bb, d]
            prev = np.concatenate([[h0[bb, d]], yc[:-1]])
            s = w[d] * prev + u[:, bb, d]
            F = yc - np.tanh(s)
            sub = -w[d] * (1 - np.tanh(s) ** 2)  # dF_t / dy_{t-1}
            ab = np.zeros((2, T))
            ab[0] = 1.0
            ab[1, :-1] = sub[1:]
            ref[:, bb, d] = yc - scipy.linalg.solve_banded((1, 0), ab, F)
    np.testing.assert_allclose(ynew, ref, rtol=1e-10, atol=1e-12)
    assert rho == pytest.approx(np.max(np.abs(ref - y)), rel=1e-12)


def test_deer_prefix_exact_after_k_iterations():
    """After k iterations from zero, y^(k)_t is exact for t < k."""
    T, D = 12, 4
    w = rng.uniform(-0.9, 0.9, D)
    u = rng.standard_normal((T, 1, D))
    h0 = rng.standard_normal((1, D))
    roll = oracle.rollout_tanh(w, u, h0)
    y = None
    for k in range(1, T + 1):
        y, _ = oracle.deer_step(w, u, y, h0)
        np.testing.assert_allclose(y[:k], roll[:k], rtol=0, atol=1e-14)
    np.testing.assert_allclose(y, roll, rtol=0, atol=1e-14)


def test_deer_converges_to_rollout():
    T, B, D = 3000, 2, 8
    w = rng.uniform(-0.9, 0.9, D)
    u = rng.standard_normal((T, B, D))
    y, k, hist, st = oracle.deer(w, u, eps=1e-12, kmax=60)
    assert st == oracle.DEER_CONVERGED
    np.testing.assert_allclose(y, oracle.rollout_tanh(w, u), rtol=0, atol=1e-11)
    assert hist[-1] < 1e-12 <= hist[-2]


def test_deer_w_zero_takes_two_iterations():
    u = rng.standard_normal((100, 2, 3))
    y, k, hist, st = oracle.deer(np.zeros(3), u, eps=1e-5, kmax=20)
    assert (k, st) == (2, oracle.DEER_CONVERGED)
    assert hist[1] == 0.0
    np.testing.assert_allclose(y, np.tanh(u), rtol=0, atol=1e-15)


def test_deer_warm_start_from_the_solution_takes_one_iteration():
    # Newton's method started at the root returns it: one scan, residual ~0
    T, B, D = 400, 2, 5
    r = np.random.default_rng(31)
    w, u, h0 = r.uniform(-0.9, 0.9, D), r.standard_normal((T, B, D)), r.standard_normal((B, D))
    ystar = oracle.rollout_tanh(w, u, h0)
    y, k, hist, st = oracle.deer(w, u, h0, eps=1e-10, kmax=20, y_init=ystar)
    assert (k, st) == (1, oracle.DEER_CONVERGED)
    assert hist[0] < 1e-13
    np.testing.assert_allclose(y, ystar, rtol=0, atol=1e-13)


def test_deer_warm_start_first_iteration_is_newton_from_the_guess():
    T, B, D = 200, 2, 4
    r = np.random.default_rng(32)
    w, u = r.uniform(-0.9, 0.9, D), r.standard_normal((T, B, D))
    guess = r.standard_normal((T, B, D))
    y, k, hist, st = oracle.deer(w, u, eps=0.0, kmax=1, y_init=guess)
    ystep, rho = oracle.deer_step(w, u, guess)
    np.testing.assert_array_equal(y, ystep)
    assert hist[0] == rho == np.max(np.abs(ystep - guess))


def test_deer_warm_start_zero_is_the_cold_start():
    r = np.random.default_rng(33)
    w, u = r.uniform(-0.9, 0.9, 3), r.standard_normal((300, 2, 3))
    a = oracle.deer(w, u, eps=1e-8, kmax=30)
    b = oracle.deer(w, u, eps=1e-8, kmax=30, y_init=np.zeros_like(u))
    np.testing.assert_array_equal(a[0], b[0])
    assert a[1] == b[1] and a[3] == b[3]
    np.testing.assert_array_equal(a[2], b[2])


def test_deer_per_sequence_stopping():
    # a quiet sequence (small u: nearly linear, converges fast), a loud one,
    # and a copy of the loud one
    T, D = 2000, 6
    r = np.random.default_rng(34)
    w = r.uniform(-0.9, 0.9, D)
    loud = r.standard_normal((T, D)) * 2.0
    u = np.stack([1e-3 * r.standard_normal((T, D)), loud, loud], axis=1)
    y, ks, sts, hists = oracle.deer_per_sequence(w, u, eps=1e-9, kmax=40)
    assert sts == [oracle.DEER_CONVERGED] * 3
    assert ks[0] < ks[1] == ks[2]
    # each sequence reached its own rollout; the global stopping test takes as
    # many iterations as the slowest sequence
    np.testing.assert_allclose(y, oracle.rollout_tanh(w, u), rtol=0, atol=1e-8)
    yg, kg, hg, stg = oracle.deer(w, u, eps=1e-9, kmax=40)
    assert kg == max(ks)
    np.testing.assert_array_equal(y[:, 1:], yg[:, 1:])


def test_deer_per_sequence_nonfinite_sequence_stops_alone():
    # a NaN in one sequence's input makes its first residual NaN: that
    # sequence stops (not finite) at K = 1, the other converges untouched
    T, D = 500, 4
    r = np.random.default_rng(35)
    w = r.uniform(-0.9, 0.9, D)
    u = r.standard_normal((T, 2, D))
    u[100, 1, 2] = np.nan
    y, ks, sts, hists = oracle.deer_per_sequence(w, u, eps=1e-9, kmax=30)
    assert sts[1] == oracle.DEER_NONFINITE and ks[1] == 1
    assert sts[0] == oracle.DEER_CONVERGED
    np.testing.assert_allclose(y[:, 0], oracle.rollout_tanh(w, u[:, :1])[:, 0], rtol=0, atol=1e-8)


def test_deer_ode_nonfinite_input_stops_at_once():
    # the ODE form's residual carries a NaN through the max-abs norm as well
    T, D = 300, 4
    r = np.random.default_rng(36)
    w = r.uniform(-0.9, 0.9, D)
    u = r.standard_normal((T, 1, D))
    u[50, 0, 1] = np.nan
    dt = np.full(T, 0.1)
    y, k, hist, st, ncl = oracle.deer_ode(w, u, dt, eps=1e-9, kmax=30)
    assert st == oracle.DEER_NONFINITE and k == 1 and np.isnan(hist[0])


def test_deer_stopping_rule_edges():
    w = rng.uniform(-0.9, 0.9, 3)
    u = rng.standard_normal((64, 1, 3))
    _, k, hist, st = oracle.deer(w, u, eps=1e9, kmax=20)
    assert (k, st, len(hist)) == (1, oracle.DEER_CONVERGED, 1)
    _, k, hist, st = oracle.deer(w, u, eps=0.0, kmax=5)
    assert (k, st, len(hist)) == (5, oracle.DEER_NOT_CONVERGED, 5)


def test_deer_stopping_test_is_strict():
    # the test is rho < eps: a residual equal to eps does not stop.  With
    # w = 0 iteration 2 repeats iteration 1 exactly (rho_2 = 0), so eps = 0
    # never stops; with eps = rho_2 of a random problem, iteration 2 goes on
    _, k, hist, st = oracle.deer(np.zeros(3), rng.standard_normal((40, 1, 3)), eps=0.0, kmax=4)
    assert hist[1] == 0.0 and (k, st) == (4, oracle.DEER_NOT_CONVERGED)
    w = rng.uniform(-0.9, 0.9, 3)
    u = rng.standard_normal((64, 1, 3))
    _, _, hist, _ = oracle.deer(w, u, eps=0.0, kmax=3)
    assert hist[2] < hist[1]
    _, k, _, st = oracle.deer(w, u, eps=hist[1], kmax=20)
    assert k > 2 and st == oracle.DEER_CONVERGED


# ----------------------------------------------------------- DEER backward

def test_deer_bwd_finite_differences_of_the_rollout():
    """The gradient through the solution, against central differences of
    L = sum g . rollout(w, u, h0) -- the quantity the gradient is of, computed
    by the direct sequential tanh RNN, not by the backward code."""
    T, B, D = 6, 2, 3
    r = np.random.default_rng(21)
    p = {"w": r.uniform(-0.9, 0.9, D), "u": r.standard_normal((T, B, D)),
         "h0": r.standard_normal((B, D))}
    g = r.standard_normal((T, B, D))
    loss = lambda: float(np.sum(g * oracle.rollout_tanh(**p)))
    y = oracle.rollout_tanh(**p)
    du, dw, dh0 = oracle.deer_bwd(p["w"], y, g, p["h0"])
    for got, key in ((du, "u"), (dw, "w"), (dh0, "h0")):
        np.testing.assert_allclose(got, _fd(loss, p[key]), rtol=1e-6, atol=1e-8, err_msg=key)


def test_deer_bwd_w_zero_is_tanh_derivative():
    """w = 0: no time coupling, du = g tanh'(u) (numpy's tanh), dh0 = 0."""
    T, B, D = 30, 2, 4
    u = rng.standard_normal((T, B, D))
    g = rng.standard_normal((T, B, D))
    y = np.tanh(u)
    du, dw, dh0 = oracle.deer_bwd(np.zeros(D), y, g, rng.standard_normal((B, D)))
    np.testing.assert_allclose(du, g * (1.0 - np.tanh(u) ** 2), rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(dh0, np.zeros((B, D)))


def test_deer_bwd_small_signal_is_linear_scan_backward():
    """At amplitude 1e-6 tanh is the identity to O(1e-12), so the gradient is
    the linear scan's (coefficient w): du ~ db and dh0 ~ dh0 of the transposed
    bidiagonal solve."""
    T, D = 120, 4
    r = np.random.default_rng(23)
    w = r.uniform(-0.9, 0.9, D)
    u = 1e-6 * r.standard_normal((T, 1, D))
    y = oracle.rollout_tanh(w, u)
    g = r.standard_normal((T, 1, D))
    du, dw, dh0 = oracle.deer_bwd(w, y, g)
    for d in range(D):
        a = np.full(T, w[d])
        delta = _bidiag_solve_T(a, g[:, 0, d])
        scale = np.max(np.abs(delta))  # rounding of the two solves, relative to the vector
        np.testing.assert_allclose(du[:, 0, d], delta, rtol=0, atol=1e-10 * scale)
        np.testing.assert_allclose(dh0[0, d], w[d] * delta[0], rtol=0, atol=1e-10 * scale)


# --------------------------------------------------------- DEER, ODE form

def _ode_exact_piecewise(w, u, dt, h0, fun):
    """Integrate dy/dt = fun(y, u_t) step by step with scipy (DOP853, tight
    tolerances), the input held over each step."""
    import scipy.integrate
    T, C = u.shape
    y = np.empty_like(u)
    cur = h0.copy()
    for t in range(T):
        sol = scipy.integrate.solve_ivp(lambda _, yy: fun(yy, u[t]), (0.0, dt[t]), cur,
                                        method="DOP853", rtol=1e-13, atol=1e-15)
        cur = sol.y[:, -1]
        y[t] = cur
    return y


def test_deer_ode_linear_case_is_exact():
    # w = 0: f = -y + tanh(u) is linear in y, so the exponential step is the
    # exact solution over each step and DEER is exact after one iteration
    T, C = 40, 3
    r = np.random.default_rng(41)
    u, h0 = r.standard_normal((T, C)), r.standard_normal(C)
    dt = r.uniform(0.05, 2.0, T)
    ref = _ode_exact_piecewise(np.zeros(C), u, dt, h0, lambda yy, ut: -yy + np.tanh(ut))
    y, clamps = oracle.rollout_ode(np.zeros(C), u, dt, h0)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-11)
    yd, k, hist, st, _ = oracle.deer_ode(np.zeros(C), u, dt, h0, eps=1e-12, kmax=10)
    assert (k, st) == (2, oracle.DEER_CONVERGED) and hist[1] < 1e-15
    np.testing.assert_allclose(yd, ref, rtol=0, atol=1e-11)


def test_deer_ode_small_signal_is_the_linearised_ode():
    # at amplitude 1e-6 tanh(x) = x to 1e-18: f = -(1 - w) y + u, linear, so
    # the exponential step with G = 1 - w is exact (a wrong sign or a dropped
    # term in G's w part is first order in dt here)
    T, C = 30, 4
    r = np.random.default_rng(42)
    w = r.uniform(-0.9, 0.9, C)
    u, h0 = 1e-6 * r.standard_normal((T, C)), 1e-6 * r.standard_normal(C)
    dt = r.uniform(0.1, 1.5, T)
    ref = _ode_exact_piecewise(w, u, dt, h0, lambda yy, ut: -(1.0 - w) * yy + ut)
    y, _ = oracle.rollout_ode(w, u, dt, h0)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-16)


def test_deer_ode_small_step_is_forward_euler():
    # dt -> 0: the exponential step is y + dt f(y) + O(dt^2)
    T, C = 100, 3
    r = np.random.default_rng(43)
    w = r.uniform(-0.9, 0.9, C)
    u, h0 = r.standard_normal((T, C)), r.standard_normal(C)
    dt = np.full(T, 1e-5)
    y, _ = oracle.rollout_ode(w, u, dt, h0)
    fe = np.empty_like(u)
    cur = h0.copy()
    for t in range(T):
        cur = cur + dt[t] * (-cur + np.tanh(w * cur + u[t]))
        fe[t] = cur
    np.testing.assert_allclose(y, fe, rtol=0, atol=1e-7)


def test_deer_ode_converges_to_the_rollout():
    T, B, D = 2000, 2, 5
    r = np.random.default_rng(44)
    w = r.uniform(-0.9, 0.9, D)
    u, h0 = r.standard_normal((T, B, D)), r.standard_normal((B, D))
    dt = r.uniform(0.1, 1.0, T)
    y, k, hist, st, _ = oracle.deer_ode(w, u, dt, h0, eps=1e-12, kmax=60)
    assert st == oracle.DEER_CONVERGED
    np.testing.assert_allclose(y, oracle.rollout_ode(w, u, dt, h0)[0], rtol=0, atol=1e-11)
    # iteration 1 from zeros is one step of the iteration
    y1, rho1, _ = oracle.deer_ode_step(w, u, dt)
    assert abs(rho1 - np.max(np.abs(y1))) == 0.0


def test_deer_ode_stopping_test_is_strict():
    # as the tanh form: a residual equal to eps does not stop the iteration
    T, D = 300, 4
    r = np.random.default_rng(45)
    w = r.uniform(-0.9, 0.9, D)
    u = r.standard_normal((T, 1, D))
    dt = r.uniform(0.1, 1.0, T)
    _, _, hist, _, _ = oracle.deer_ode(w, u, dt, eps=0.0, kmax=3)
    assert hist[2] < hist[1]
    _, k, _, st, _ = oracle.deer_ode(w, u, dt, eps=hist[1], kmax=20)
    assert k > 2 and st == oracle.DEER_CONVERGED


def test_deer_ode_clamp():
    # w = -12: G = 1 + 12 (1 - tanh^2) reaches 13 where the pre-activation is
    # small; clamped to 10 and counted (the count is that of the rollout, at
    # the fixed point), every value finite
    T, C = 500, 4
    r = np.random.default_rng(45)
    w = np.full(C, -12.0)
    u, dt = 0.3 * r.standard_normal((T, C)), np.full(T, 0.2)
    y, clamps = oracle.rollout_ode(w, u, dt, np.zeros(C))
    assert np.all(np.isfinite(y))
    prev = np.vstack([np.zeros((1, C)), y[:-1]])
    g = 1.0 - w * (1.0 - np.tanh(w * prev + u) ** 2)
    assert clamps == int(np.sum(np.abs(g) > 10.0)) > 0
    yd, k, hist, st, cl = oracle.deer_ode(w, u, dt, np.zeros(C), eps=1e-10, kmax=60)
    assert st == oracle.DEER_CONVERGED and cl == clamps
    np.testing.assert_allclose(yd, y, rtol=0, atol=1e-9)


def test_oracle_threads_do_not_change_results():
    a = rng.uniform(-1, 1, (300, 33))
    b = rng.standard_normal((300, 33))
    oracle.set_num_threads(1)
    h1 = oracle.scan_fwd(a, b)
    oracle.set_num_threads(4)
    h4 = oracle.scan_fwd(a, b)
    oracle.set_num_threads(0)
    assert np.array_equal(h1, h4)


def test_oracle_rejects_shapes_it_would_misread():
    # the C code trusts its sizes: the wrappers check them first
    u = np.zeros((6, 2, 4))
    w = np.zeros(4)
    with pytest.raises(ValueError):
        oracle.scan_fwd(u, np.zeros((6, 2, 3)))
    with pytest.raises(ValueError):
        oracle.scan_fwd(u, u, np.zeros(7))
    with pytest.raises(ValueError):
        oracle.deer(np.zeros(3), u)
    with pytest.raises(ValueError):
        oracle.deer(w, u, y_init=np.zeros((5, 2, 4)))
    with pytest.raises(ValueError):
        oracle.deer_ode(w, u, np.zeros(5))
    with pytest.raises(ValueError):
        oracle.sru_fwd(u, u, u, u, w, np.zeros(2))
    # per-feature arrays shorter than the channel count repeat over the batch
    y, _, _, _ = oracle.deer(np.zeros(2), np.zeros((6, 8)))
    assert y.shape == (6, 8)
