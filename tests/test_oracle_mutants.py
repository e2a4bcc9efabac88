"""Planted mistakes in the oracle: the pins must catch them.

Each entry of MUTANTS turns one expression of oracle/lr_oracle.c into a
plausible slip -- a time index shifted by one, a flipped sign, a dropped
factor or initial state, swapped operands or biases, a loosened stopping
test, a NaN left out of the residual.  The mutant is compiled with the
oracle's own flags into the oracle's (git-ignored) build folder, loaded in
place of the oracle's library, and every pin named beside it in
test_oracle_pins.py must fail.  The unmutated source, built and loaded the
same way, passes every named pin, so a failure belongs to the planted
mistake and not to the harness.  The module-wide generator of the pins is
reseeded before each call, so a pin sees the same inputs under every build.

CPU only: nothing here loads the CUDA library.
"""

import concurrent.futures
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

_SRC = os.path.join(os.path.dirname(oracle.__file__), "lr_oracle.c")
_OUT = os.path.join(os.path.dirname(oracle.__file__), "_build", "mutants")
_SEED = 20250921

_FD_SCAN = "test_scan_bwd_finite_differences"
_FD_SRU = "test_sru_bwd_finite_differences"
_FD_LSTM = "test_lstm_bwd_finite_differences"
_TIE_LSTM_BWD = "test_lstm_bwd_gilr_tie_is_the_sru_gradient"
_NEWTON = "test_deer_step_is_newton_on_residual"
_FD_DEER = "test_deer_bwd_finite_differences_of_the_rollout"
_ODE_LIN = "test_deer_ode_linear_case_is_exact"

# (id, text in lr_oracle.c, replacement, which occurrence, pins that must fail)
MUTANTS = [
    # ---- forward scan
    ("scan_fwd-a_prev_for_a_t",
     "h[t * C + c] = a[t * C + c] * h[(t - 1) * C + c]",
     "h[t * C + c] = a[(t - 1) * C + c] * h[(t - 1) * C + c]", 0,
     ["test_golden_dyadic_example", "test_scan_time_varying_matches_banded_solve"]),
    ("scan_fwd-h0_dropped",
     "h[c] = a[c] * (h0 ? h0[c] : 0.0) + b[c];", "h[c] = b[c];", 0,
     ["test_golden_dyadic_example", "test_scan_a_one_is_running_sum"]),
    # ---- backward scan
    ("scan_bwd-a_t_for_a_next",
     "db[t * C + c] = g[t * C + c] + a[(t + 1) * C + c] * db[(t + 1) * C + c];",
     "db[t * C + c] = g[t * C + c] + a[t * C + c] * db[(t + 1) * C + c];", 0,
     [_FD_SCAN, "test_scan_bwd_is_transposed_solve"]),
    ("scan_bwd-h_t_for_h_prev_in_da",
     "double hprev = t > 0 ? h[(t - 1) * C + c]", "double hprev = t > 0 ? h[t * C + c]", 0,
     ["test_golden_dyadic_example", _FD_SCAN]),
    ("scan_bwd-h0_dropped_in_da",
     "double hprev = t > 0 ? h[(t - 1) * C + c] : (h0 ? h0[c] : 0.0);",
     "double hprev = t > 0 ? h[(t - 1) * C + c] : 0.0;", 0, [_FD_SCAN]),
    ("scan_bwd-a0_dropped_in_dh0", "dh0[c] = a[c] * db[c];", "dh0[c] = db[c];", 0,
     ["test_golden_dyadic_example", _FD_SCAN]),
    # ---- SRU
    ("sigmoid-sign_of_exponent",
     "return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));", 0,
     ["test_sru_reset_gate_limits", "test_lstm_gates_open_is_running_sum"]),
    ("sru_fwd-f_for_one_minus_f",
     "c[i] = f * cprev + (1.0 - f) * xt[i];", "c[i] = f * cprev + f * xt[i];", 0,
     ["test_sru_forget_closed_gives_c_equal_xt", "test_sru_memory_is_linear_recurrence_solve"]),
    ("sru_fwd-tanh_dropped",
     "h[i] = r * tanh(c[i]) + (1.0 - r) * x[i];", "h[i] = r * c[i] + (1.0 - r) * x[i];", 0,
     ["test_sru_reset_gate_limits"]),
    ("sru_fwd-c0_dropped",
     "double cprev = t > 0 ? c[i - C] : (c0 ? c0[k] : 0.0);",
     "double cprev = t > 0 ? c[i - C] : 0.0;", 0, ["test_sru_memory_is_linear_recurrence_solve"]),
    ("sru_fwd-bf_for_br",
     "double r = sigm(ur[i] + br[d]);", "double r = sigm(ur[i] + bf[d]);", 0,
     [_FD_SRU, "test_lstm_gilr_tie_is_the_sru_cell"]),
    ("sru_bwd-operand_order_in_dUf",
     "duf[i] = dc[i] * (cprev - xt[i]) * f * (1.0 - f);",
     "duf[i] = dc[i] * (xt[i] - cprev) * f * (1.0 - f);", 0, [_FD_SRU, _TIE_LSTM_BWD]),
    ("sru_bwd-tanh_derivative_dropped",
     "double e = dh[i] * r * (1.0 - th * th);", "double e = dh[i] * r;", 0, [_FD_SRU]),
    ("sru_bwd-f_t_for_f_next",
     "if (t + 1 < T) carry = sigm(uf[i + C] + bf[d]) * dc[i + C];",
     "if (t + 1 < T) carry = sigm(uf[i] + bf[d]) * dc[i + C];", 0, [_FD_SRU]),
    ("sru_bwd-bias_sums_swapped",
     "dbf[k % D] += sf[k]; dbr[k % D] += sr[k];", "dbf[k % D] += sr[k]; dbr[k % D] += sf[k];", 0,
     [_FD_SRU]),
    ("sru_bwd-bf_for_br",
     "double r = sigm(ur[i] + br[d]);", "double r = sigm(ur[i] + bf[d]);", 2, [_FD_SRU]),
    ("sru_bwd-c0_dropped_in_dUf",
     "double cprev = t > 0 ? c[i - C] : (c0 ? c0[k] : 0.0);",
     "double cprev = t > 0 ? c[i - C] : 0.0;", 1, [_FD_SRU]),
    ("sru_bwd-f0_dropped_in_dc0",
     "dc0[k] = sigm(uf[k] + bf[k % D]) * dc[k];", "dc0[k] = dc[k];", 0, [_FD_SRU]),
    # ---- LSTM cell
    ("lstm_fwd-h_from_C_prev", "h[n] = o * tanh(c[n]);", "h[n] = o * tanh(cprev);", 0,
     ["test_lstm_gates_open_is_running_sum", "test_lstm_gilr_tie_is_the_sru_cell"]),
    ("lstm_fwd-i_and_f_swapped", "c[n] = f * cprev + i * g;", "c[n] = i * cprev + f * g;", 0,
     ["test_lstm_cell_is_linear_recurrence_solve", "test_lstm_forget_closed_has_no_memory"]),
    ("lstm_fwd-c0_dropped",
     "double cprev = t > 0 ? c[n - C] : (c0 ? c0[k] : 0.0);",
     "double cprev = t > 0 ? c[n - C] : 0.0;", 0,
     ["test_lstm_cell_is_linear_recurrence_solve", "test_lstm_gates_open_is_running_sum"]),
    ("lstm_fwd-bi_for_bo",
     "double o = sigm(zo[n] + bo[d]);", "double o = sigm(zo[n] + bi[d]);", 0,
     ["test_lstm_gilr_tie_is_the_sru_cell"]),
    ("lstm_bwd-i_dropped_in_dzc",
     "dzc[n] = dc[n] * i * (1.0 - g * g);", "dzc[n] = dc[n] * (1.0 - g * g);", 0,
     [_FD_LSTM, _TIE_LSTM_BWD]),
    ("lstm_bwd-C_t_for_C_prev_in_dzf",
     "dzf[n] = dc[n] * cprev * f * (1.0 - f);", "dzf[n] = dc[n] * c[n] * f * (1.0 - f);", 0,
     [_FD_LSTM, _TIE_LSTM_BWD]),
    ("lstm_bwd-f0_dropped_in_dc0",
     "dc0[k] = sigm(zf[k] + bf[k % D]) * dc[k];", "dc0[k] = dc[k];", 0, [_FD_LSTM, _TIE_LSTM_BWD]),
    ("lstm_bwd-o_dropped_in_dC",
     "dc[n] = dh[n] * o * (1.0 - th * th) + carry;", "dc[n] = dh[n] * (1.0 - th * th) + carry;", 0,
     [_FD_LSTM, _TIE_LSTM_BWD]),
    ("lstm_bwd-bi_for_bo",
     "double o = sigm(zo[n] + bo[d]);", "double o = sigm(zo[n] + bi[d]);", 1, [_FD_LSTM]),
    ("lstm_bwd-c0_dropped_in_dzf",
     "double cprev = t > 0 ? c[n - C] : (c0 ? c0[k] : 0.0);",
     "double cprev = t > 0 ? c[n - C] : 0.0;", 1, [_FD_LSTM]),
    # ---- tanh rollout and DEER
    ("rollout-h0_dropped",
     "double prev = t > 0 ? y[i - C] : (h0 ? h0[k] : 0.0);",
     "double prev = t > 0 ? y[i - C] : 0.0;", 0, ["test_deer_prefix_exact_after_k_iterations"]),
    ("deer_step-sign_of_rhs", "double rhs = th - J * ytil;", "double rhs = th + J * ytil;", 0,
     [_NEWTON, "test_deer_converges_to_rollout"]),
    ("deer_step-tanh_derivative_dropped_in_J",
     "double J = wk * (1.0 - th * th);", "double J = wk;", 0, [_NEWTON]),
    ("deer_step-ytil_t_for_ytil_prev",
     "double ytil = t > 0 ? (yprev ? yprev[i - C] : 0.0) : init;\n                double s = wk",
     "double ytil = yprev ? yprev[i] : init;\n                double s = wk", 0,
     [_NEWTON, "test_deer_prefix_exact_after_k_iterations"]),
    ("deer_step-h0_dropped", "double init = h0 ? h0[k] : 0.0;", "double init = 0.0;", 1, [_NEWTON]),
    ("deer_step-nan_left_out_of_residual",
     "if (isnan(diff)) nan_seen = 1;", "if (0) nan_seen = 1;", 1,
     ["test_deer_per_sequence_nonfinite_sequence_stops_alone"]),
    ("deer-stopping_test_not_strict",
     "if (rho < eps) { status = 0; break; }", "if (rho <= eps) { status = 0; break; }", 1,
     ["test_deer_stopping_test_is_strict"]),
    ("deer-guess_ignored", "k == 1 ? y_init : prev", "k == 1 ? NULL : prev", 0,
     ["test_deer_warm_start_first_iteration_is_newton_from_the_guess",
      "test_deer_warm_start_from_the_solution_takes_one_iteration"]),
    # ---- DEER backward
    ("deer_bwd-y_t_for_y_next_in_carry",
     "delta = g[i] + wk * (1.0 - y[i + C] * y[i + C]) * delta;",
     "delta = g[i] + wk * (1.0 - y[i] * y[i]) * delta;", 0, [_FD_DEER]),
    ("deer_bwd-y_t_for_y_prev_in_dw",
     "const double yprev = t > 0 ? y[i - C]", "const double yprev = t > 0 ? y[i]", 0, [_FD_DEER]),
    ("deer_bwd-h0_dropped_in_dw",
     "const double yprev = t > 0 ? y[i - C] : (h0 ? h0[k] : 0.0);",
     "const double yprev = t > 0 ? y[i - C] : 0.0;", 0, [_FD_DEER]),
    ("deer_bwd-w_dropped_in_dh0",
     "dh0[k] = T > 0 ? wk * (1.0 - y[k] * y[k]) * delta : 0.0;",
     "dh0[k] = T > 0 ? (1.0 - y[k] * y[k]) * delta : 0.0;", 0,
     [_FD_DEER, "test_deer_bwd_small_signal_is_linear_scan_backward"]),
    # ---- DEER, ODE form
    ("ode-sign_of_w_term_in_G",
     "double g = 1.0 - wk * (1.0 - th * th);", "double g = 1.0 + wk * (1.0 - th * th);", 0,
     ["test_deer_ode_small_signal_is_the_linearised_ode"]),
    ("ode-clamp_bound", "if (g > 10.0) { g = 10.0; ++*ncl; }", "if (g > 1.0) { g = 1.0; ++*ncl; }", 0,
     ["test_deer_ode_clamp"]),
    ("ode-phi_sign",
     "return g != 0.0 ? -expm1(-g * dt) / g : dt;", "return g != 0.0 ? expm1(-g * dt) / g : dt;", 0,
     [_ODE_LIN, "test_deer_ode_small_step_is_forward_euler"]),
    ("ode_rollout-sign_of_minus_y",
     "y[i] = yp + ode_phi(g, dt[t]) * (th - yp);", "y[i] = yp + ode_phi(g, dt[t]) * (th + yp);", 0,
     [_ODE_LIN, "test_deer_ode_small_step_is_forward_euler"]),
    ("ode_rollout-h0_dropped",
     "double yp = t > 0 ? y[i - C] : (h0 ? h0[k] : 0.0);",
     "double yp = t > 0 ? y[i - C] : 0.0;", 0, [_ODE_LIN]),
    ("ode_step-minus_ytil_dropped_in_z",
     "double z = (th - ytil) + g * ytil;", "double z = th + g * ytil;", 0,
     [_ODE_LIN, "test_deer_ode_converges_to_the_rollout"]),
    ("ode_step-sign_of_exponent", "double a = exp(-g * dt[t]);", "double a = exp(g * dt[t]);", 0,
     [_ODE_LIN]),
    ("ode_step-h0_dropped", "double init = h0 ? h0[k] : 0.0;", "double init = 0.0;", 0,
     ["test_deer_ode_converges_to_the_rollout"]),
    ("ode_step-nan_left_out_of_residual",
     "if (isnan(diff)) nan_seen = 1;", "if (0) nan_seen = 1;", 0,
     ["test_deer_ode_nonfinite_input_stops_at_once"]),
    ("ode-stopping_test_not_strict",
     "if (rho < eps) { status = 0; break; }", "if (rho <= eps) { status = 0; break; }", 0,
     ["test_deer_ode_stopping_test_is_strict"]),
]


def _mutate(src: str, old: str, new: str, occurrence: int) -> str:
    assert src.count(old) > occurrence, f"{old!r} occurs {src.count(old)} times in the oracle"
    pos = -1
    for _ in range(occurrence + 1):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


@pytest.fixture(scope="module")
def libraries():
    """The control build and every mutant, compiled in parallel; tag -> path."""
    with open(_SRC) as f:
        src = f.read()
    os.makedirs(_OUT, exist_ok=True)
    jobs = [("control", src)]
    jobs += [(m[0], _mutate(src, m[1], m[2], m[3])) for m in MUTANTS]
    tag = f"{os.getpid()}"

    def compile_one(job):
        name, text = job
        c = os.path.join(_OUT, f"{name}.{tag}.c")
        so = os.path.join(_OUT, f"{name}.{tag}.so")
        with open(c, "w") as f:
            f.write(text)
        subprocess.run(["gcc", *oracle.CFLAGS, c, "-o", so, "-lm"], check=True, capture_output=True)
        os.remove(c)
        return name, so

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        libs = dict(ex.map(compile_one, jobs))
    yield libs
    for so in libs.values():
        os.remove(so)


def _run(monkeypatch, so: str, pin: str) -> None:
    """Runs pin `pin` with the oracle's functions bound to library `so`."""
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: so)
    monkeypatch.setattr(pins, "rng", np.random.default_rng(_SEED))
    getattr(pins, pin)()


def test_mutant_table_is_well_formed():
    ids = [m[0] for m in MUTANTS]
    assert len(set(ids)) == len(ids)
    for m in MUTANTS:
        assert m[4] and all(callable(getattr(pins, p, None)) for p in m[4]), m[0]


def test_control_build_passes_every_named_pin(libraries, monkeypatch):
    for pin in sorted({p for m in MUTANTS for p in m[4]}):
        _run(monkeypatch, libraries["control"], pin)


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_its_pins(libraries, monkeypatch, mutant):
    name, _, _, _, names = mutant
    for pin in names:
        with pytest.raises(AssertionError):
            _run(monkeypatch, libraries[name], pin)
