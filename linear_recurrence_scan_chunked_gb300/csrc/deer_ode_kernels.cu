// deer_ode_kernels.cu -- one DEER iteration in the ODE form (next row on the
// same scan), page [P4] (.../cuda-parallel-rnn-training-logt-optimization),
// section "监控与调优", third check: the coefficients of the linear inverse
// operator are exp(-G_i dt_i), and the elements of G_i are clamped to
// [-10, 10] (counted) so that they cannot overflow.
//
// The ODE is the continuous-time form of the diagonal tanh RNN,
//     dy/dt = f(y, u) = -y + tanh(w y + u),
// on steps dt[t] with the input held at u_t over step t.  One iteration
// linearises f at the previous iterate at the start of each step (ytil_{t-1},
// ytil_{-1} = h0):
//     G_t = -df/dy = 1 - w (1 - tanh^2(w ytil_{t-1} + u_t)),  clamped to [-10, 10],
//     z_t = f(ytil_{t-1}, u_t) + G_t ytil_{t-1},
// and solves dy/dt + G_t y = z_t exactly over the step: the scan element is
//     (a_t, b_t) = (exp(-G_t dt_t), (1 - exp(-G_t dt_t)) / G_t z_t)
// (b_t = dt_t z_t when G_t = 0), both from one e^x - 1 (act_expm1).  The
// epilogue writes y and folds max |y - yold| as the tanh form does, and on the
// segmented walker kernel also builds the next iteration's coefficients at
// row t from the y_{t-1} just computed (as stored) and folds them into the next
// iteration's aggregates, which then needs no reduce pass (NextAgg).
#include "lr_act.cuh"
#include "lr_launch.h"
#include "lr_persist.cuh"

namespace lrs {

template <typename S>
struct DeerOdeParams {
    const float* w;
    const S* u;
    const float* dt;  // [T] step lengths
    const S* h0;
    const S* yold;
    S* ynew;
    uint32_t* resid;
    const uint32_t* prev_resid;  // residual of the previous iteration (nullptr: first)
    float eps;
    unsigned long long* clamps;  // clamped G evaluations of this iteration
    NextAgg nx;                  // next iteration's aggregates (segmented walker kernel only)
};

constexpr float kOdeGClamp = 10.f;

template <typename S_, int VEC_, int NW_, int R_>
struct DeerOdeOp {
    using S = S_;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, MINB = 2;
    static constexpr bool REV = false;
    static constexpr int IN_ARRAYS = 2;  // u, previous iterate
    static constexpr bool SCRATCH_IN_CARRY = false;
    static constexpr bool NEXT_AGG = true;
    using Params = DeerOdeParams<S>;
    struct Regs {
        Pack<S, VEC> u[R];
        Pack<S, VEC> yo[R + 1];  // previous iterate at rows t0-1 .. t0+R-1 (row -1 is h0)
    };
    struct Work {
        float J[R][VEC], Rh[R][VEC];  // (a_t, b_t)
        float DT[R];                  // step lengths of the rows
        uint32_t ncl;                 // clamps among this thread's rows (counted once per element)
        float NA[VEC], NB[VEC];       // next iteration's aggregate of this thread's rows
    };
    struct Smem {
        uint32_t mx[NW];
    };
    struct Acc {
        uint32_t mx;  // max |y - yold| as bits
    };
    __device__ static void acc_init(Acc& a) { a.mx = 0; }
    // as the tanh form: an iteration enqueued after the solve stopped passes
    // its predecessor's residual on and does nothing else
    __device__ static bool skip(const Params& p) {
        if (p.prev_resid == nullptr) return false;
        const uint32_t bits = *(volatile const uint32_t*)p.prev_resid;
        const float rho = __uint_as_float(bits);
        const bool stop = rho < p.eps || !(rho <= 3.4e38f);
        if (stop && blockIdx.x == 0 && threadIdx.x == 0) *p.resid = bits;
        return stop;
    }
    __device__ static const S* init_ptr(const Params& p) { return p.h0; }
    __host__ __device__ static NextAgg next_agg(const Params& p) { return p.nx; }

    // The step's coefficients from the linearisation point yt (the state
    // entering the step), the input and the step length: clamps G, counts it.
    // w4 = 4 w: G = 1 - w (1 - tanh^2) = 1 - 4 w q (the same bits as with w).
    __device__ static void coeffs(float wv, float w4, float yt, float uv, float dtt, float& a,
                                  float& b, uint32_t& ncl) {
        float q1;
        const float th = act_tanh_q(wv * yt + uv, q1);
        float gv = fmaf(-w4, q1, 1.f);
        if (gv > kOdeGClamp) {  // (a NaN fails both tests and stays NaN)
            gv = kOdeGClamp;
            ++ncl;
        } else if (gv < -kOdeGClamp) {
            gv = -kOdeGClamp;
            ++ncl;
        }
        const float z = (th - yt) + gv * yt;
        const float em = act_expm1(-gv * dtt);  // exp(-G dt) - 1
        a = 1.f + em;
        b = (gv != 0.f ? __fdividef(-em, gv) : dtt) * z;
    }

    static constexpr int TMA_N = 2;  // staged: u, previous iterate (rows t0-1 .. t0+L-1)
    __host__ __device__ static constexpr int tma_shift(int k) { return k == 1 ? -1 : 0; }
    __host__ __device__ static constexpr int tma_extra(int k) { return k == 1 ? 1 : 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.u;
        ptr[1] = p.yold;  // nullptr on the first iteration: not staged
    }

    template <class Src>
    __device__ static void load(const Src& src, const Params& p, const Geom& g,
                                const TileCoord& tc, Regs& rg) {
#pragma unroll
        for (int i = 0; i <= R; ++i) {
            const int64_t t = tc.t0 - 1 + i;
            if (!tc.cok || t >= g.T) rg.yo[i].ident(0.f);
            else if (t < 0) {
                if (p.h0 != nullptr) rg.yo[i].load(p.h0 + tc.c);
                else rg.yo[i].ident(0.f);
            } else if (p.yold != nullptr) src.ld(rg.yo[i], 1, p.yold, t);
            else rg.yo[i].ident(0.f);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            if (tc.cok && t < g.T) src.ld(rg.u[r], 0, p.u, t);
            else rg.u[r].ident(0.f);
        }
    }
    __device__ static void aggregate(const Params& p, const Geom& g, const TileCoord& tc,
                                     const Regs& rg, Work& w, float (&A)[VEC], float (&B)[VEC],
                                     bool side) {
        float wv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) wv[v] = 0.f;
        if (tc.cok) load_param<VEC>(p.w + tc.cd, wv);
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
        uint32_t ncl = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            const bool ok = tc.cok && t < g.T;
            const float dtt = ok ? __ldg(p.dt + t) : 0.f;
            w.DT[r] = dtt;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                float a, b;
                uint32_t n = 0;
                coeffs(wv[v], 4.f * wv[v], rg.yo[r].get(v), rg.u[r].get(v), dtt, a, b, n);
                ncl += ok ? n : 0u;
                w.J[r][v] = ok ? a : 1.f;
                w.Rh[r][v] = ok ? b : 0.f;
                B[v] = w.J[r][v] * B[v] + w.Rh[r][v];
                A[v] *= w.J[r][v];
            }
        }
        w.ncl = side ? ncl : 0u;
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work& w, float (&s)[VEC], Smem&, Acc& acc) {
        const bool nxt = p.nx.agg != nullptr;
        float wv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { wv[v] = 0.f; w.NA[v] = 1.f; w.NB[v] = 0.f; }
        if (nxt && tc.cok) load_param<VEC>(p.w + tc.cd, wv);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            if (nxt && tc.cok && t < g.T) {
                // next iteration, row t: linearised at y_{t-1} (s, as stored)
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    float yp = s[v];
                    if constexpr (sizeof(S) == 2) yp = bf_lo(bf_bits(yp));
                    float a, b;
                    uint32_t n = 0;  // counted by the next iteration itself
                    coeffs(wv[v], 4.f * wv[v], yp, rg.u[r].get(v), w.DT[r], a, b, n);
                    w.NB[v] = a * w.NB[v] + b;
                    w.NA[v] *= a;
                }
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) s[v] = w.J[r][v] * s[v] + w.Rh[r][v];
            if (tc.cok && t < g.T) {
                store_vec<S, VEC>(p.ynew + t * g.C + tc.c, s);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    float yv = s[v];  // the stored (rounded) value is what the next step reads
                    if constexpr (sizeof(S) == 2) yv = bf_lo(bf_bits(yv));
                    const uint32_t bits = __float_as_uint(fabsf(yv - rg.yo[r + 1].get(v)));
                    acc.mx = bits > acc.mx ? bits : acc.mx;
                }
            }
        }
        // clamp count: one atomic per warp, only when it clamped
        uint32_t n = w.ncl;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
        if ((threadIdx.x & 31) == 0 && n) atomicAdd(p.clamps, (unsigned long long)n);
    }
    __device__ static void at_exit(const Params& p, Smem& xs, Acc& acc) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        uint32_t mx = acc.mx;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, mx, off);
            mx = o > mx ? o : mx;
        }
        if (lane == 0) xs.mx[warp] = mx;
        csync<NW>();
        if (threadIdx.x == 0) {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < NW; ++i) m = xs.mx[i] > m ? xs.mx[i] : m;
            if (m) atomicMax(p.resid, m);
        }
    }
};

template <typename S, bool VP, int M>
using DeerOdeOpT = DeerOdeOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_DEER_ODE, sizeof(S) == 2, M).NW,
                             kcfg(OP_DEER_ODE, sizeof(S) == 2, M).R>;

template <typename S, bool VP>
static cudaError_t deer_ode_t(const DeerOdeParams<S>& p, const Geom& g, const Carry& cr,
                              cudaStream_t s) {
    return launch_persist<DeerOdeOpT<S, VP, CARRY_CHAIN>, DeerOdeOpT<S, VP, CARRY_WALK>,
                          DeerOdeOpT<S, VP, TILE_TMA>, kcfg(OP_DEER_ODE, sizeof(S) == 2, TILE_TMA).ST>(
        p, g, cr, s);
}

template <typename S>
static cudaError_t deer_ode_s(bool vec, const float* w, const void* u, const float* dt,
                              const void* h0, const void* yold, void* ynew, uint32_t* resid,
                              const uint32_t* prev_resid, float eps, unsigned long long* clamps,
                              const NextAgg& nx, const Geom& g, const Carry& cr, cudaStream_t s) {
    const DeerOdeParams<S> p{w, (const S*)u, dt, (const S*)h0, (const S*)yold, (S*)ynew,
                             resid, prev_resid, eps, clamps, nx};
    return vec ? deer_ode_t<S, true>(p, g, cr, s) : deer_ode_t<S, false>(p, g, cr, s);
}

cudaError_t launch_deer_ode_iter(int dtype, bool vec, const float* w, const void* u,
                                 const float* dt, const void* h0, const void* yold, void* ynew,
                                 uint32_t* resid, const uint32_t* prev_resid, float eps,
                                 unsigned long long* clamps, const NextAgg& nx, const Geom& g,
                                 const Carry& cr, cudaStream_t s) {
    return dtype == 0 ? deer_ode_s<float>(vec, w, u, dt, h0, yold, ynew, resid, prev_resid, eps,
                                          clamps, nx, g, cr, s)
                      : deer_ode_s<__nv_bfloat16>(vec, w, u, dt, h0, yold, ynew, resid,
                                                  prev_resid, eps, clamps, nx, g, cr, s);
}

}  // namespace lrs
