/*
 * lr_oracle.c -- plain, sequential, fp64 CPU oracle for the linear-recurrence
 * hot path.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg, never by the product path.
 * It shares no code, header or constant with the CUDA library.
 *
 * Sources (four blog pages from blog.hotdry.top, all dated 2025-09-21):
 *   [P1] "CUDA并行化RNN训练：从O(T)到O(log T)的工程实践与参数调优"
 *        (CUDA-parallel RNN training, O(T) -> O(log T)): the SRU paragraph
 *        (forget gate, highway reset gate) and the parallel-scan paragraph
 *        (an associative operation evaluated for forward and backward).
 *   [P2] "RNN CUDA内核优化：实现序列长度无关的恒定推理延迟"
 *        (RNN CUDA kernel optimisation): the paragraph that isolates the
 *        linear part C_t = f_t*C_{t-1} + i_t*C~_t and solves it by tree
 *        reduction in log2(T) stages.
 *   [P4] the DEER page (.../cuda-parallel-rnn-training-logt-optimization),
 *        section "核心原理：DEER 框架与牛顿法的工程映射" (Newton form, the
 *        three steps: f and Jacobian J, G_p times a vector, the linear inverse
 *        solved as a prefix scan) and section "工程实现" (the stopping rule
 *        ||y^(i+1) - y^(i)|| < eps or K_max).
 *
 * Everything is the plain definition: strictly sequential in t, fp64, libm
 * exp/tanh only.  No blocking, no re-association.  Channels are independent,
 * so threads (OpenMP) split the channel range and nothing else.
 *
 * Layout: every sequence tensor is [T, C] row-major with C = B*D channels
 * contiguous; channel c uses the per-feature parameter index d = c % D.
 * A NULL initial state means zeros.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- threads */

static int g_threads = 0; /* 0: OpenMP default */

void lro_set_num_threads(int n) { g_threads = n; }

int lro_num_threads(void) {
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/* Channel range [*c0, *c1) owned by thread `tid` of `nt`. */
static void chan_range(int64_t C, int tid, int nt, int64_t* c0, int64_t* c1) {
    int64_t per = C / nt, rem = C % nt;
    *c0 = tid * per + (tid < rem ? tid : rem);
    *c1 = *c0 + per + (tid < rem ? 1 : 0);
}

#ifdef _OPENMP
#define PAR_BEGIN                                                     \
    _Pragma("omp parallel num_threads(lro_num_threads())") {          \
        int tid_ = omp_get_thread_num(), nt_ = omp_get_num_threads(); \
        int64_t c0_, c1_;                                             \
        chan_range(C, tid_, nt_, &c0_, &c1_);
#define PAR_END }
#else
#define PAR_BEGIN                 \
    {                             \
        int64_t c0_ = 0, c1_ = C;
#define PAR_END }
#endif

/* ------------------------------------------------------- forward (row a1) */
/*
 * h_t = a_t * h_{t-1} + b_t,  h_{-1} = h0  (elementwise per channel).
 * [P2] LSTM paragraph: the state update is a linear recurrence with
 * time-varying coefficient; [P1] parallel-scan paragraph.
 */
void lro_scan_fwd(int64_t T, int64_t C, const double* a, const double* b,
                  const double* h0, double* h) {
    PAR_BEGIN
    for (int64_t c = c0_; c < c1_; ++c) h[c] = a[c] * (h0 ? h0[c] : 0.0) + b[c];
    for (int64_t t = 1; t < T; ++t)
        for (int64_t c = c0_; c < c1_; ++c)
            h[t * C + c] = a[t * C + c] * h[(t - 1) * C + c] + b[t * C + c];
    PAR_END
}

/* ------------------------------------------------------ backward (row a2) */
/*
 * Given the forward states h and the upstream gradient g = dL/dh_t for every
 * t, back-propagation through time of h_t = a_t h_{t-1} + b_t:
 *   delta_{T-1} = g_{T-1},   delta_t = g_t + a_{t+1} * delta_{t+1}
 *   dL/db_t = delta_t,   dL/da_t = delta_t * h_{t-1},   dL/dh0 = a_0 * delta_0
 * [P1] parallel-scan paragraph: the same associative evaluation serves the
 * backward pass, which is this recurrence run in reverse time.
 * dh0 may be NULL (skipped).
 */
void lro_scan_bwd(int64_t T, int64_t C, const double* a, const double* h,
                  const double* h0, const double* g, double* da, double* db,
                  double* dh0) {
    PAR_BEGIN
    for (int64_t c = c0_; c < c1_; ++c) db[(T - 1) * C + c] = g[(T - 1) * C + c];
    for (int64_t t = T - 2; t >= 0; --t)
        for (int64_t c = c0_; c < c1_; ++c)
            db[t * C + c] = g[t * C + c] + a[(t + 1) * C + c] * db[(t + 1) * C + c];
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = c0_; c < c1_; ++c) {
            double hprev = t > 0 ? h[(t - 1) * C + c] : (h0 ? h0[c] : 0.0);
            da[t * C + c] = db[t * C + c] * hprev;
        }
    if (dh0)
        for (int64_t c = c0_; c < c1_; ++c) dh0[c] = a[c] * db[c];
    PAR_END
}

/* --------------------------------------------------- SRU forward (row a3) */

static double sigm(double z) { return 1.0 / (1.0 + exp(-z)); }

/*
 * SRU in its linear form (v_f = 0), per [P1] SRU paragraph (forget gate from
 * the current input only; highway reset gate mixing input and memory):
 *   f_t = sigma(U_f,t + b_f),  r_t = sigma(U_r,t + b_r)
 *   c_t = f_t c_{t-1} + (1 - f_t) xt_t,        c_{-1} = c0
 *   h_t = r_t tanh(c_t) + (1 - r_t) x_t
 * U_f, U_r, xt are the precomputed projections; bf, br are [D].
 */
void lro_sru_fwd(int64_t T, int64_t C, int64_t D, const double* xt,
                 const double* uf, const double* ur, const double* x,
                 const double* bf, const double* br, const double* c0,
                 double* h, double* c) {
    PAR_BEGIN
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = c0_; k < c1_; ++k) {
            int64_t i = t * C + k, d = k % D;
            double cprev = t > 0 ? c[i - C] : (c0 ? c0[k] : 0.0);
            double f = sigm(uf[i] + bf[d]);
            double r = sigm(ur[i] + br[d]);
            c[i] = f * cprev + (1.0 - f) * xt[i];
            h[i] = r * tanh(c[i]) + (1.0 - r) * x[i];
        }
    PAR_END
}

/* -------------------------------------------------- SRU backward (row a4) */
/*
 * Gradients of the SRU forward above given the memory states c and the
 * upstream dh = dL/dh_t (the only upstream gradient):
 *   dr_t   = dh_t (tanh c_t - x_t),     dU_r = dr_t r_t (1 - r_t)
 *   dx_t   = dh_t (1 - r_t)
 *   dc_t   = dh_t r_t (1 - tanh^2 c_t) + f_{t+1} dc_{t+1}    (reverse in t)
 *   dxt_t  = dc_t (1 - f_t)
 *   dU_f,t = dc_t (c_{t-1} - xt_t) f_t (1 - f_t)
 *   dc0    = f_0 dc_0
 *   db_f[d] = sum over t and batch of dU_f,  db_r[d] likewise of dU_r.
 * dc0 may be NULL.  Returns -1 when scratch allocation fails.
 */
int lro_sru_bwd(int64_t T, int64_t C, int64_t D, const double* xt,
                const double* uf, const double* ur, const double* x,
                const double* bf, const double* br, const double* c0,
                const double* c, const double* dh, double* dxt, double* duf,
                double* dur, double* dx, double* dbf, double* dbr,
                double* dc0) {
    double* dc = (double*)malloc(sizeof(double) * (size_t)(T * C > 0 ? T * C : 1));
    double* sf = (double*)calloc((size_t)(C > 0 ? C : 1), sizeof(double));
    double* sr = (double*)calloc((size_t)(C > 0 ? C : 1), sizeof(double));
    if (!dc || !sf || !sr) {
        free(dc);
        free(sf);
        free(sr);
        return -1;
    }
    PAR_BEGIN
    /* memory-state gradient, reverse in time */
    for (int64_t t = T - 1; t >= 0; --t)
        for (int64_t k = c0_; k < c1_; ++k) {
            int64_t i = t * C + k, d = k % D;
            double r = sigm(ur[i] + br[d]);
            double th = tanh(c[i]);
            double e = dh[i] * r * (1.0 - th * th);
            double carry = 0.0;
            if (t + 1 < T) carry = sigm(uf[i + C] + bf[d]) * dc[i + C];
            dc[i] = e + carry;
        }
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = c0_; k < c1_; ++k) {
            int64_t i = t * C + k, d = k % D;
            double f = sigm(uf[i] + bf[d]);
            double r = sigm(ur[i] + br[d]);
            double th = tanh(c[i]);
            double cprev = t > 0 ? c[i - C] : (c0 ? c0[k] : 0.0);
            double dr = dh[i] * (th - x[i]);
            dur[i] = dr * r * (1.0 - r);
            dx[i] = dh[i] * (1.0 - r);
            dxt[i] = dc[i] * (1.0 - f);
            duf[i] = dc[i] * (cprev - xt[i]) * f * (1.0 - f);
            sf[k] += duf[i];
            sr[k] += dur[i];
        }
    if (dc0)
        for (int64_t k = c0_; k < c1_; ++k) dc0[k] = sigm(uf[k] + bf[k % D]) * dc[k];
    PAR_END
    /* bias gradients: sum the per-channel sums over the batch, serially */
    for (int64_t d = 0; d < D; ++d) { dbf[d] = 0.0; dbr[d] = 0.0; }
    for (int64_t k = 0; k < C; ++k) { dbf[k % D] += sf[k]; dbr[k % D] += sr[k]; }
    free(dc);
    free(sf);
    free(sr);
    return 0;
}

/* ------------------------------------------- LSTM cell-state scan (next) */
/*
 * [P2] LSTM paragraph: the cell state of a standard LSTM unit evolves by
 *   C_t = f_t * C_{t-1} + i_t * C~_t,
 * a linear recurrence in C whose coefficients f_t (forget gate) and i_t
 * (input gate) vary with t, and C~_t is the candidate state; the input,
 * forget and output gates are sigmoids and the candidate a tanh of their
 * pre-activations.  The plain reading taken here (the GILR-style cell of
 * [P2] checklist item 1): the pre-activations zf, zi, zc, zo come
 * precomputed from the input only (no h_{t-1} term), so the gates do not
 * depend on the state and the recurrence is linear:
 *   f = sigma(zf + bf),  i = sigma(zi + bi),  C~ = tanh(zc + bc),
 *   o = sigma(zo + bo),
 *   C_t = f_t C_{t-1} + i_t C~_t,   C_{-1} = c0,
 *   h_t = o_t tanh(C_t)             (the LSTM output).
 * zf..zo are [T, C]; bf..bo are [D].
 */
void lro_lstm_fwd(int64_t T, int64_t C, int64_t D, const double* zf,
                  const double* zi, const double* zc, const double* zo,
                  const double* bf, const double* bi, const double* bc,
                  const double* bo, const double* c0, double* h, double* c) {
    PAR_BEGIN
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = c0_; k < c1_; ++k) {
            int64_t n = t * C + k, d = k % D;
            double cprev = t > 0 ? c[n - C] : (c0 ? c0[k] : 0.0);
            double f = sigm(zf[n] + bf[d]);
            double i = sigm(zi[n] + bi[d]);
            double g = tanh(zc[n] + bc[d]);
            double o = sigm(zo[n] + bo[d]);
            c[n] = f * cprev + i * g;
            h[n] = o * tanh(c[n]);
        }
    PAR_END
}

/*
 * Gradients of lro_lstm_fwd given the cell states c and the upstream
 * dh = dL/dh_t (back-propagation through time, the reverse-time form of the
 * same linear recurrence):
 *   dC_t  = dh_t o_t (1 - tanh^2 C_t) + f_{t+1} dC_{t+1}     (reverse in t)
 *   dzf_t = dC_t C_{t-1} f_t (1 - f_t)
 *   dzi_t = dC_t C~_t i_t (1 - i_t)
 *   dzc_t = dC_t i_t (1 - C~_t^2)
 *   dzo_t = dh_t tanh(C_t) o_t (1 - o_t)
 *   dc0   = f_0 dC_0
 *   db*[d] = sum over t and batch of dz*.
 * dc0 may be NULL.  Returns -1 when scratch allocation fails.
 */
int lro_lstm_bwd(int64_t T, int64_t C, int64_t D, const double* zf,
                 const double* zi, const double* zc, const double* zo,
                 const double* bf, const double* bi, const double* bc,
                 const double* bo, const double* c0, const double* c,
                 const double* dh, double* dzf, double* dzi, double* dzc,
                 double* dzo, double* dbf, double* dbi, double* dbc,
                 double* dbo, double* dc0) {
    double* dc = (double*)malloc(sizeof(double) * (size_t)(T * C > 0 ? T * C : 1));
    double* sum = (double*)calloc((size_t)(4 * C > 0 ? 4 * C : 1), sizeof(double));
    if (!dc || !sum) {
        free(dc);
        free(sum);
        return -1;
    }
    PAR_BEGIN
    for (int64_t t = T - 1; t >= 0; --t)
        for (int64_t k = c0_; k < c1_; ++k) {
            int64_t n = t * C + k, d = k % D;
            double o = sigm(zo[n] + bo[d]);
            double th = tanh(c[n]);
            double carry = 0.0;
            if (t + 1 < T) carry = sigm(zf[n + C] + bf[d]) * dc[n + C];
            dc[n] = dh[n] * o * (1.0 - th * th) + carry;
        }
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = c0_; k < c1_; ++k) {
            int64_t n = t * C + k, d = k % D;
            double cprev = t > 0 ? c[n - C] : (c0 ? c0[k] : 0.0);
            double f = sigm(zf[n] + bf[d]);
            double i = sigm(zi[n] + bi[d]);
            double g = tanh(zc[n] + bc[d]);
            double o = sigm(zo[n] + bo[d]);
            dzf[n] = dc[n] * cprev * f * (1.0 - f);
            dzi[n] = dc[n] * g * i * (1.0 - i);
            dzc[n] = dc[n] * i * (1.0 - g * g);
            dzo[n] = dh[n] * tanh(c[n]) * o * (1.0 - o);
            sum[k] += dzf[n];
            sum[C + k] += dzi[n];
            sum[2 * C + k] += dzc[n];
            sum[3 * C + k] += dzo[n];
        }
    if (dc0)
        for (int64_t k = c0_; k < c1_; ++k) dc0[k] = sigm(zf[k] + bf[k % D]) * dc[k];
    PAR_END
    for (int64_t d = 0; d < D; ++d) { dbf[d] = 0.0; dbi[d] = 0.0; dbc[d] = 0.0; dbo[d] = 0.0; }
    for (int64_t k = 0; k < C; ++k) {
        dbf[k % D] += sum[k];
        dbi[k % D] += sum[C + k];
        dbc[k % D] += sum[2 * C + k];
        dbo[k % D] += sum[3 * C + k];
    }
    free(dc);
    free(sum);
    return 0;
}

/* ------------------------------------------- DEER, ODE form (next row) */
/*
 * [P4] "监控与调优", third check: in the ODE form of DEER the linear inverse
 * operator's coefficients are exp(-G_i Delta_i), which overflow when G_i is
 * large, so the elements of G_i are clamped to [-10, 10] (and the clamps
 * counted).  Reading: the continuous-time form of the same diagonal tanh RNN,
 *     dy/dt = f(y, u) = -y + tanh(w y + u),
 * on steps of length dt[t] with the input held at u_t over step t and
 * y_{-1} = h0.  Each iteration linearises f at the previous iterate at the
 * start of the step,
 *     G_t = -df/dy = 1 - w (1 - tanh^2(w ytil_{t-1} + u_t)),  clamped to [-10, 10],
 *     z_t = f(ytil_{t-1}, u_t) + G_t ytil_{t-1},
 * and solves dy/dt + G_t y = z_t exactly over the step,
 *     y_t = exp(-G_t dt_t) y_{t-1} + (1 - exp(-G_t dt_t)) / G_t z_t
 * (dt_t z_t when G_t = 0): a linear recurrence, the scan.  At the fixed point
 * (ytil = y) this is the exponential-Euler rollout
 *     y_t = y_{t-1} + (1 - exp(-G_t dt_t)) / G_t f(y_{t-1}, u_t).
 * (1 - exp(-x)) is evaluated as -expm1(-x).  The clamp counts are of the
 * evaluations where G left [-10, 10].
 */
static double ode_g(double wk, double th, int64_t* ncl) {
    double g = 1.0 - wk * (1.0 - th * th);
    if (g > 10.0) { g = 10.0; ++*ncl; }
    else if (g < -10.0) { g = -10.0; ++*ncl; }
    return g;
}

/* (1 - exp(-g dt)) / g, and its g = 0 limit dt */
static double ode_phi(double g, double dt) { return g != 0.0 ? -expm1(-g * dt) / g : dt; }

void lro_rollout_ode(int64_t T, int64_t C, int64_t D, const double* w,
                     const double* u, const double* dt, const double* h0,
                     double* y, int64_t* clamps) {
    int64_t ncl = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(lro_num_threads()) reduction(+ : ncl)
#endif
    {
        int64_t c0_ = 0, c1_ = C;
#ifdef _OPENMP
        chan_range(C, omp_get_thread_num(), omp_get_num_threads(), &c0_, &c1_);
#endif
        for (int64_t t = 0; t < T; ++t)
            for (int64_t k = c0_; k < c1_; ++k) {
                int64_t i = t * C + k;
                double wk = w[k % D];
                double yp = t > 0 ? y[i - C] : (h0 ? h0[k] : 0.0);
                double th = tanh(wk * yp + u[i]);
                double g = ode_g(wk, th, &ncl);
                y[i] = yp + ode_phi(g, dt[t]) * (th - yp);
            }
    }
    if (clamps) *clamps = ncl;
}

/* One iteration from yprev (NULL = the all-zero guess); rho = max |ynew - yprev|,
 * NaN when any difference is NaN (as lro_deer_step). */
void lro_deer_ode_step(int64_t T, int64_t C, int64_t D, const double* w,
                       const double* u, const double* dt, const double* h0,
                       const double* yprev, double* ynew, double* rho,
                       int64_t* clamps) {
    double best = 0.0;
    int64_t ncl = 0;
    int nan_seen = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(lro_num_threads()) reduction(max : best) reduction(+ : ncl) reduction(| : nan_seen)
#endif
    {
        int64_t c0_ = 0, c1_ = C;
#ifdef _OPENMP
        chan_range(C, omp_get_thread_num(), omp_get_num_threads(), &c0_, &c1_);
#endif
        for (int64_t t = 0; t < T; ++t)
            for (int64_t k = c0_; k < c1_; ++k) {
                int64_t i = t * C + k;
                double wk = w[k % D];
                double init = h0 ? h0[k] : 0.0;
                double ytil = t > 0 ? (yprev ? yprev[i - C] : 0.0) : init;
                double th = tanh(wk * ytil + u[i]);
                double g = ode_g(wk, th, &ncl);
                double z = (th - ytil) + g * ytil;
                double a = exp(-g * dt[t]);
                double b = ode_phi(g, dt[t]) * z;
                double ylast = t > 0 ? ynew[i - C] : init;
                ynew[i] = a * ylast + b;
                double diff = fabs(ynew[i] - (yprev ? yprev[i] : 0.0));
                if (isnan(diff)) nan_seen = 1;
                else if (diff > best) best = diff;
            }
    }
    *rho = nan_seen ? NAN : best;
    if (clamps) *clamps = ncl;
}

/*
 * The ODE-form iteration from the all-zero guess with the stopping rule of
 * lro_deer; clamps: the clamp count of the last iteration.  Returns as
 * lro_deer.
 */
int lro_deer_ode(int64_t T, int64_t C, int64_t D, const double* w, const double* u,
                 const double* dt, const double* h0, double eps, int kmax,
                 double* y, double* rho_hist, int* iters, int64_t* clamps) {
    size_t n = (size_t)(T * C);
    double* prev = (double*)malloc(sizeof(double) * (n ? n : 1));
    if (!prev) return -1;
    int status = 1, k;
    for (k = 1; k <= kmax; ++k) {
        double rho = 0.0;
        lro_deer_ode_step(T, C, D, w, u, dt, h0, k == 1 ? NULL : prev, y, &rho, clamps);
        rho_hist[k - 1] = rho;
        if (!isfinite(rho)) { status = 2; break; }
        if (rho < eps) { status = 0; break; }
        memcpy(prev, y, sizeof(double) * n);
    }
    *iters = k > kmax ? kmax : k;
    free(prev);
    return status;
}

/* -------------------------------------------------- DEER (row a5), tanh RNN */
/*
 * Target recurrence: h_t = tanh(w (.) h_{t-1} + u_t), h_{-1} = h0, w in [D].
 *
 * The direct sequential evaluation ([P1]/[P4]: the O(T) serial RNN).
 */
void lro_rollout_tanh(int64_t T, int64_t C, int64_t D, const double* w,
                      const double* u, const double* h0, double* y) {
    PAR_BEGIN
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = c0_; k < c1_; ++k) {
            int64_t i = t * C + k;
            double prev = t > 0 ? y[i - C] : (h0 ? h0[k] : 0.0);
            y[i] = tanh(w[k % D] * prev + u[i]);
        }
    PAR_END
}

/*
 * One DEER / Newton step ([P4] "核心原理": (1) evaluate f and its Jacobian J at
 * the current guess, (2) form G_p times the guess, G_p = -J, (3) apply the
 * linear inverse operator, which for an RNN is a linear recurrence with an
 * initial condition).  For the diagonal tanh cell, with ytil_{t-1} the
 * previous iterate shifted by one step (ytil_{-1} = h0):
 *   s_t   = w ytil_{t-1} + u_t
 *   J_t   = w (1 - tanh^2 s_t)
 *   rhs_t = tanh(s_t) - J_t ytil_{t-1}
 *   ynew_t = J_t ynew_{t-1} + rhs_t,   ynew_{-1} = h0     (sequential here)
 * yprev == NULL means the all-zero initial guess.  Returns, through *rho,
 * max |ynew - yprev| over all B*T*D entries; NaN when any entry's difference
 * is NaN (the max-abs norm of a vector holding a NaN is NaN, so the stopping
 * test sees it as not finite).
 */
void lro_deer_step(int64_t T, int64_t C, int64_t D, const double* w,
                   const double* u, const double* h0, const double* yprev,
                   double* ynew, double* rho) {
    double best = 0.0;
    int nan_seen = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(lro_num_threads()) reduction(max : best) reduction(| : nan_seen)
#endif
    {
        int64_t c0_ = 0, c1_ = C;
#ifdef _OPENMP
        chan_range(C, omp_get_thread_num(), omp_get_num_threads(), &c0_, &c1_);
#endif
        for (int64_t t = 0; t < T; ++t)
            for (int64_t k = c0_; k < c1_; ++k) {
                int64_t i = t * C + k;
                double wk = w[k % D];
                double init = h0 ? h0[k] : 0.0;
                double ytil = t > 0 ? (yprev ? yprev[i - C] : 0.0) : init;
                double s = wk * ytil + u[i];
                double th = tanh(s);
                double J = wk * (1.0 - th * th);
                double rhs = th - J * ytil;
                double ylast = t > 0 ? ynew[i - C] : init;
                ynew[i] = J * ylast + rhs;
                double diff = fabs(ynew[i] - (yprev ? yprev[i] : 0.0));
                if (isnan(diff)) nan_seen = 1;
                else if (diff > best) best = diff;
            }
    }
    *rho = nan_seen ? NAN : best;
}

/*
 * DEER fixed-point iteration ([P4] "工程实现": stop when
 * ||y^(i+1) - y^(i)|| < eps, here the max-abs norm over all entries, or after
 * kmax iterations) from the initial guess y_init, NULL meaning the all-zero
 * guess ([P4] "核心原理": a guess close to the solution -- in training, the
 * previous step's -- keeps the iteration count small; the residual of
 * iteration 1 is measured against the guess).  K counts the scans performed,
 * including the one whose residual fell below eps.  rho_hist[k-1] = residual
 * of iteration k.  Returns 0 when converged, 1 when kmax was reached without
 * convergence, 2 when a residual was not finite, -1 on allocation failure.
 */
int lro_deer(int64_t T, int64_t C, int64_t D, const double* w, const double* u,
             const double* h0, const double* y_init, double eps, int kmax,
             double* y, double* rho_hist, int* iters) {
    size_t n = (size_t)(T * C);
    double* prev = (double*)malloc(sizeof(double) * (n ? n : 1));
    if (!prev) return -1;
    int status = 1, k;
    for (k = 1; k <= kmax; ++k) {
        double rho = 0.0;
        /* iteration 1 starts from the initial guess: y_init, or zeros */
        lro_deer_step(T, C, D, w, u, h0, k == 1 ? y_init : prev, y, &rho);
        rho_hist[k - 1] = rho;
        if (!isfinite(rho)) { status = 2; break; }
        if (rho < eps) { status = 0; break; }
        memcpy(prev, y, sizeof(double) * n);
    }
    *iters = k > kmax ? kmax : k;
    free(prev);
    return status;
}

/* ------------------------------------- DEER backward (next row), tanh RNN */
/*
 * Gradient through the solution y of h_t = tanh(w (.) h_{t-1} + u_t)
 * ([P4] "核心原理": at the fixed point y is the rollout, so the gradient is
 * back-propagation through the rollout evaluated at y):
 *   s_t = w y_{t-1} + u_t, y_t = tanh(s_t), dy_t/dy_{t-1} = w (1 - y_t^2);
 *   delta_{T-1} = g_{T-1},  delta_t = g_t + w (1 - y_{t+1}^2) delta_{t+1}
 *     (delta_t: total derivative of L = sum g.y with respect to y_t);
 *   du_t = delta_t (1 - y_t^2);  dw_d = sum over t and the channels of
 *   feature d of du_t y_{t-1} (y_{-1} = h0);  dh0 = w (1 - y_0^2) delta_0.
 * g is the upstream gradient dL/dy.  dh0 may be NULL.  Returns -1 when
 * scratch allocation fails.
 */
int lro_deer_bwd(int64_t T, int64_t C, int64_t D, const double* w,
                 const double* y, const double* h0, const double* g, double* du,
                 double* dw, double* dh0) {
    double* sw = (double*)calloc((size_t)(C > 0 ? C : 1), sizeof(double));
    if (!sw) return -1;
    PAR_BEGIN
    for (int64_t k = c0_; k < c1_; ++k) {
        const double wk = w[k % D];
        double delta = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            const int64_t i = t * C + k;
            if (t == T - 1) delta = g[i];
            else delta = g[i] + wk * (1.0 - y[i + C] * y[i + C]) * delta;
            du[i] = delta * (1.0 - y[i] * y[i]);
            const double yprev = t > 0 ? y[i - C] : (h0 ? h0[k] : 0.0);
            sw[k] += du[i] * yprev;
        }
        if (dh0) dh0[k] = T > 0 ? wk * (1.0 - y[k] * y[k]) * delta : 0.0;
    }
    PAR_END
    for (int64_t d = 0; d < D; ++d) dw[d] = 0.0;
    for (int64_t k = 0; k < C; ++k) dw[k % D] += sw[k];
    free(sw);
    return 0;
}
