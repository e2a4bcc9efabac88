// deer_kernels.cu -- one fused DEER / Newton iteration for the diagonal tanh
// RNN h_t = tanh(w h_{t-1} + u_t) (row a5).
//
// Page [P4] (.../cuda-parallel-rnn-training-logt-optimization), section
// "核心原理：DEER 框架与牛顿法的工程映射": each iteration (1) evaluates f and its
// Jacobian J at the current guess, (2) multiplies G_p = -J by the guess, and
// (3) applies the linear inverse operator, which for an RNN is a linear
// recurrence with an initial condition, solved by a prefix scan.  Here all
// three happen in one launch: the producer builds, for row t, from the
// previous iterate shifted by one step (ytil_{t-1}, ytil_{-1} = h0)
//     s_t = w ytil_{t-1} + u_t,  J_t = w (1 - tanh^2 s_t),
//     rhs_t = tanh(s_t) - J_t ytil_{t-1},
// the scan solves y_t = J_t y_{t-1} + rhs_t, and the epilogue writes y and
// folds max |y_t - yold_t| into one residual word (the stopping test of the
// section "工程实现": ||y^(i+1) - y^(i)|| < eps, here the max-abs norm).
// yold == nullptr is the all-zero initial guess (not read).
//
// On the segmented walker kernel the epilogue also builds the next
// iteration's J and rhs at row t from the value just computed at row t-1 (as
// stored: bf16-rounded for bf16 storage) and u_t, exactly what the next
// iteration would read, and folds them into the next iteration's segment
// aggregates; the next iteration then needs no reduce pass (NextAgg).
#include "lr_act.cuh"
#include "lr_launch.h"
#include "lr_persist.cuh"

namespace lrs {

template <typename S>
struct DeerParams {
    const float* w;
    const S* u;
    const S* h0;
    const S* yold;
    S* ynew;
    uint32_t* resid;
    const uint32_t* prev_resid;  // residual of the previous iteration (nullptr: first)
    float eps;
    NextAgg nx;  // next iteration's aggregates (segmented walker kernel only)
    // Per-sequence stopping (nullptr: one stopping test for the whole batch).
    uint32_t* seq_resid;        // [B] this iteration's residual bits, per sequence
    const uint32_t* seq_done;   // [B] nonzero: the sequence stopped (its y is not written)
    const uint32_t* all_done;   // nonzero: every sequence stopped (the launch does nothing)
};

template <typename S_, int VEC_, int NW_, int R_>
struct DeerOp {
    using S = S_;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, MINB = 2;
    static constexpr bool REV = false;
    static constexpr int IN_ARRAYS = 2;  // u, previous iterate
    static constexpr bool SCRATCH_IN_CARRY = false;
    static constexpr bool NEXT_AGG = true;
    using Params = DeerParams<S>;
    struct Regs {
        Pack<S, VEC> u[R];
        Pack<S, VEC> yo[R + 1];  // previous iterate at rows t0-1 .. t0+R-1 (row -1 is h0)
    };
    struct Work {
        float J[R][VEC], Rh[R][VEC];
        float NA[VEC], NB[VEC];  // next iteration's aggregate of this thread's rows
    };
    struct Smem {
        uint32_t mx[NW];
    };
    __host__ __device__ static NextAgg next_agg(const Params& p) { return p.nx; }
    struct Acc {
        uint32_t mx;  // max |y - yold| as bits: fp32 order of non-negative values, NaN on top
    };
    __device__ static void acc_init(Acc& a) { a.mx = 0; }
    // The iterations of a solve are enqueued in batches; one whose predecessor
    // already stopped the solve (residual below eps, or not finite) does
    // nothing but pass that residual on, so that its own successor stops too.
    __device__ static bool skip(const Params& p) {
        if (p.all_done != nullptr) return *(volatile const uint32_t*)p.all_done != 0;
        if (p.prev_resid == nullptr) return false;
        const uint32_t bits = *(volatile const uint32_t*)p.prev_resid;
        const float rho = __uint_as_float(bits);
        const bool stop = rho < p.eps || !(rho <= 3.4e38f);
        if (stop && blockIdx.x == 0 && threadIdx.x == 0) *p.resid = bits;
        return stop;
    }
    __device__ static const S* init_ptr(const Params& p) { return p.h0; }
    // This thread's rows and the row before them are all inside the problem:
    // no per-row bounds checks (the previous iterate is staged, or it is the
    // all-zero first guess).
    __device__ static bool interior(const Params&, const Geom& g, const TileCoord& tc) {
        return tc.cok && tc.t0 >= 1 && tc.t0 + R <= g.T;
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
        if (interior(p, g, tc)) {
            if (p.yold != nullptr) {
#pragma unroll
                for (int i = 0; i <= R; ++i) src.ld(rg.yo[i], 1, p.yold, tc.t0 - 1 + i);
            } else {
#pragma unroll
                for (int i = 0; i <= R; ++i) rg.yo[i].ident(0.f);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) src.ld(rg.u[r], 0, p.u, tc.t0 + r);
            return;
        }
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
                                     bool) {
        float wv[VEC], w4[VEC];  // w, and 4 w for the Jacobian w (1 - tanh^2) = 4 w q
#pragma unroll
        for (int v = 0; v < VEC; ++v) wv[v] = 0.f;
        if (tc.cok) load_param<VEC>(p.w + tc.cd, wv);
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; w4[v] = 4.f * wv[v]; }
        if (interior(p, g, tc)) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float yt = rg.yo[r].get(v);
                    float q1;
                    const float th = act_tanh_q(wv[v] * yt + rg.u[r].get(v), q1);
                    const float jac = w4[v] * q1;
                    w.J[r][v] = jac;
                    w.Rh[r][v] = th - jac * yt;
                    B[v] = jac * B[v] + w.Rh[r][v];
                    A[v] *= jac;
                }
            return;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool ok = tc.cok && tc.t0 + r < g.T;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float yt = rg.yo[r].get(v);
                float q1;
                const float th = act_tanh_q(wv[v] * yt + rg.u[r].get(v), q1);
                const float jac = w4[v] * q1;
                w.J[r][v] = ok ? jac : 1.f;
                w.Rh[r][v] = ok ? th - jac * yt : 0.f;
                B[v] = w.J[r][v] * B[v] + w.Rh[r][v];
                A[v] *= w.J[r][v];
            }
        }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work& w, float (&s)[VEC], Smem&, Acc& acc) {
        const bool nxt = p.nx.agg != nullptr;
        // per-sequence stopping: the lane's channels belong to one sequence
        // (VEC divides D); a stopped sequence keeps its iterate
        const bool per_seq = p.seq_done != nullptr;
        uint32_t seq = 0;
        bool live = true;
        if (per_seq && tc.cok) {
            seq = (uint32_t)chan_seq(g, tc.c);
            live = p.seq_done[seq] == 0;
        }
        uint32_t mx = 0;  // this tile's residual bits (per-sequence stopping)
        float wv[VEC], w4[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { wv[v] = 0.f; w.NA[v] = 1.f; w.NB[v] = 0.f; }
        if (nxt && tc.cok) load_param<VEC>(p.w + tc.cd, wv);
#pragma unroll
        for (int v = 0; v < VEC; ++v) w4[v] = 4.f * wv[v];
        if (nxt && !per_seq && interior(p, g, tc)) {  // the iterations' common case
            S* out = p.ynew + tc.t0 * g.C + tc.c;
#pragma unroll
            for (int r = 0; r < R; ++r, out += g.C) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    float yp = s[v];
                    if constexpr (sizeof(S) == 2) yp = bf_lo(bf_bits(yp));
                    float q1;
                    const float th = act_tanh_q(wv[v] * yp + rg.u[r].get(v), q1);
                    const float jac = w4[v] * q1;
                    w.NB[v] = jac * w.NB[v] + (th - jac * yp);
                    w.NA[v] *= jac;
                    s[v] = w.J[r][v] * s[v] + w.Rh[r][v];
                }
                store_vec<S, VEC>(out, s);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    float yv = s[v];
                    if constexpr (sizeof(S) == 2) yv = bf_lo(bf_bits(yv));
                    const uint32_t bits = __float_as_uint(fabsf(yv - rg.yo[r + 1].get(v)));
                    mx = bits > mx ? bits : mx;
                }
            }
            acc.mx = mx > acc.mx ? mx : acc.mx;
            return;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            if (nxt && tc.cok && t < g.T) {
                // next iteration, row t: from y_{t-1} (s, as stored) and u_t
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    float yp = s[v];
                    if constexpr (sizeof(S) == 2) yp = bf_lo(bf_bits(yp));
                    float q1;
                    const float th = act_tanh_q(wv[v] * yp + rg.u[r].get(v), q1);
                    const float jac = w4[v] * q1;
                    w.NB[v] = jac * w.NB[v] + (th - jac * yp);
                    w.NA[v] *= jac;
                }
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) s[v] = w.J[r][v] * s[v] + w.Rh[r][v];
            if (tc.cok && t < g.T && live) {
                store_vec<S, VEC>(p.ynew + t * g.C + tc.c, s);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    // the stored (rounded) value is the iterate the next step reads
                    float yv = s[v];
                    if constexpr (sizeof(S) == 2) yv = bf_lo(bf_bits(yv));
                    const uint32_t bits = __float_as_uint(fabsf(yv - rg.yo[r + 1].get(v)));
                    mx = bits > mx ? bits : mx;
                }
            }
        }
        acc.mx = mx > acc.mx ? mx : acc.mx;
        if (per_seq) {
            // one atomic per warp when its lanes share a sequence, else per lane
            const uint32_t key = tc.cok && live ? seq : 0xffffffffu;
            const uint32_t k0 = __shfl_sync(0xffffffffu, key, 0);
            if (__all_sync(0xffffffffu, key == k0)) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const uint32_t o = __shfl_xor_sync(0xffffffffu, mx, off);
                    mx = o > mx ? o : mx;
                }
                if ((threadIdx.x & 31) == 0 && k0 != 0xffffffffu && mx) atomicMax(p.seq_resid + k0, mx);
            } else if (key != 0xffffffffu && mx) {
                atomicMax(p.seq_resid + key, mx);
            }
        }
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

// DEER backward (next row of the same scan): the gradient through the
// solution y of h_t = tanh(w h_{t-1} + u_t).  At the fixed point y is the
// rollout ([P4] "核心原理"), so the gradient is back-propagation through it:
// with the upstream g = dL/dy and J_t = dy_t/dy_{t-1} = w (1 - y_t^2),
//     delta_t = g_t + J_{t+1} delta_{t+1}   (reverse scan, as the linear BPTT,
//                                           on u_t = J_t delta_t),
//     du_t = delta_t (1 - y_t^2),   dw = sum_{t,b} du_t y_{t-1},
//     dh0 = u_0 = J_0 delta_0      (y_{-1} = h0).
// dw: per-tile channel sums, then the fixed-order reduction of the SRU bias
// gradients.
template <typename S>
struct DeerBwdParams {
    const float* w;
    const S* y;
    const S* h0;
    const S* dy;
    S* du;
    S* dh0;
    float* partials;  // [n_chunks][C]
};

template <typename S_, int VEC_, int NW_, int R_>
struct DeerBwdOp {
    using S = S_;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, MINB = 2;
    static constexpr bool REV = true;
    static constexpr int IN_ARRAYS = 2;  // y (rows t and t-1), dy
    using Params = DeerBwdParams<S>;
    struct Regs {
        Pack<S, VEC> y[R + 1];  // y at times t0, t0-1, ..., t0-R (row -1 is h0)
        Pack<S, VEC> g[R];
    };
    struct Work {
        float J[R][VEC], D1[R][VEC];  // J_t and 1 - y_t^2
    };
    struct Smem {
        float pw[NW][32][VEC];
    };
    // the partial sums may overlay the carry's warp aggregates: finish() writes
    // them only after a barrier that every warp reaches once done with those
    static constexpr bool SCRATCH_IN_CARRY = true;
    struct Acc {
        float sw[VEC];  // dw sums over a run of tiles (acc_run)
    };
    __device__ static void acc_init(Acc& a) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) a.sw[v] = 0.f;
    }
    __device__ static bool skip(const Params&) { return false; }
    __device__ static const S* init_ptr(const Params&) { return nullptr; }  // u_T = 0

    static constexpr int TMA_N = 2;  // staged: dy, y (rows t0-1 .. t0+L-1 of the chunk)
    __host__ __device__ static constexpr int tma_shift(int k) { return k == 1 ? -1 : 0; }
    __host__ __device__ static constexpr int tma_extra(int k) { return k == 1 ? 1 : 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.dy;
        ptr[1] = p.y;
    }

    template <class Src>
    __device__ static void load(const Src& src, const Params& p, const Geom& g,
                                const TileCoord& tc, Regs& rg) {
#pragma unroll
        for (int i = 0; i <= R; ++i) {
            const int64_t t = tc.t0 - i;
            if (!tc.cok || t >= g.T) rg.y[i].ident(0.f);
            else if (t < 0) {
                if (p.h0 != nullptr) rg.y[i].load(p.h0 + tc.c);
                else rg.y[i].ident(0.f);
            } else src.ld(rg.y[i], 1, p.y, t);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            if (tc.cok && t < g.T) src.ld(rg.g[r], 0, p.dy, t);
            else rg.g[r].ident(0.f);
        }
    }
    __device__ static void aggregate(const Params& p, const Geom& g, const TileCoord& tc,
                                     const Regs& rg, Work& w, float (&A)[VEC], float (&B)[VEC],
                                     bool) {
        float wv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) wv[v] = 0.f;
        if (tc.cok) load_param<VEC>(p.w + tc.cd, wv);
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool ok = tc.cok && tc.t0 - r < g.T;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float yt = rg.y[r].get(v);
                const float d1 = 1.f - yt * yt;
                w.D1[r][v] = d1;
                w.J[r][v] = ok ? wv[v] * d1 : 1.f;
                B[v] = w.J[r][v] * (rg.g[r].get(v) + B[v]);
                A[v] *= w.J[r][v];
            }
        }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work& w, float (&s)[VEC], Smem& xs, Acc& acc) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        float sum[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) sum[v] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            const bool ok = tc.cok && t < g.T;
            float du[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float delta = rg.g[r].get(v) + s[v];
                du[v] = delta * w.D1[r][v];
                s[v] = w.J[r][v] * delta;
                if (ok) sum[v] += du[v] * rg.y[r + 1].get(v);
            }
            if (ok) store_vec<S, VEC>(p.du + t * g.C + tc.c, du);
        }
        // row 0 is the last row of the last warp of time chunk 0: s = u_0 = dh0
        if (tc.tchunk == 0 && warp == NW - 1 && p.dh0 != nullptr && tc.cok)
            store_vec<S, VEC>(p.dh0 + tc.c, s);
        if (tc.acc_run) {
            // a run of tiles of these channels through this CTA: the sums run
            // over it in registers; a tile's partial row is zeros and the
            // run's last tile writes the total (the reduction over chunks is
            // unchanged)
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc.sw[v] += sum[v];
            if (!tc.acc_flush) {
                if (warp == 0 && tc.cok) {
                    float* pp = p.partials + tc.tchunk * g.C + tc.c;
#pragma unroll
                    for (int v = 0; v < VEC; ++v) pp[v] = 0.f;
                }
                return;
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sum[v] = acc.sw[v];
                acc.sw[v] = 0.f;
            }
        }
        // dw partials of this tile (or run): fixed warp order
        csync<NW>();  // every warp is past its reads of the carry smem
#pragma unroll
        for (int v = 0; v < VEC; ++v) xs.pw[warp][lane][v] = sum[v];
        csync<NW>();
        if (warp == 0 && tc.cok) {
            float pw[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) pw[v] = 0.f;
#pragma unroll
            for (int ww = 0; ww < NW; ++ww)
#pragma unroll
                for (int v = 0; v < VEC; ++v) pw[v] += xs.pw[ww][lane][v];
            float* pp = p.partials + tc.tchunk * g.C + tc.c;
#pragma unroll
            for (int v = 0; v < VEC; ++v) pp[v] = pw[v];
        }
    }
    __device__ static void at_exit(const Params&, Smem&, Acc&) {}
};

template <typename S, bool VP, int M>
using DeerOpT = DeerOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_DEER, sizeof(S) == 2, M).NW,
                       kcfg(OP_DEER, sizeof(S) == 2, M).R>;

template <typename S, bool VP>
static cudaError_t deer_t(const float* w, const void* u, const void* h0, const void* yold,
                          void* ynew, uint32_t* resid, const uint32_t* prev_resid, float eps,
                          const NextAgg& nx, const DeerSeq& sq, const Geom& g, const Carry& cr,
                          cudaStream_t s) {
    return launch_persist<DeerOpT<S, VP, CARRY_CHAIN>, DeerOpT<S, VP, CARRY_WALK>,
                          DeerOpT<S, VP, TILE_TMA>, kcfg(OP_DEER, sizeof(S) == 2, TILE_TMA).ST>(
        {w, (const S*)u, (const S*)h0, (const S*)yold, (S*)ynew, resid, prev_resid, eps, nx,
         sq.resid, sq.done, sq.all_done},
        g, cr, s);
}

cudaError_t launch_deer_iter(int dtype, bool vec, const float* w, const void* u, const void* h0,
                             const void* yold, void* ynew, uint32_t* resid,
                             const uint32_t* prev_resid, float eps, const NextAgg& nx,
                             const DeerSeq& sq, const Geom& g, const Carry& cr, cudaStream_t s) {
    if (dtype == 0)
        return vec ? deer_t<float, true>(w, u, h0, yold, ynew, resid, prev_resid, eps, nx, sq, g,
                                         cr, s)
                   : deer_t<float, false>(w, u, h0, yold, ynew, resid, prev_resid, eps, nx, sq, g,
                                          cr, s);
    return vec ? deer_t<__nv_bfloat16, true>(w, u, h0, yold, ynew, resid, prev_resid, eps, nx, sq,
                                             g, cr, s)
               : deer_t<__nv_bfloat16, false>(w, u, h0, yold, ynew, resid, prev_resid, eps, nx,
                                              sq, g, cr, s);
}

// Per-sequence stopping, after iteration k: a running sequence whose residual
// of iteration k is below eps (or not finite) stops at K = k; all_done is set
// when no sequence runs.  One block.
__global__ void __launch_bounds__(1024)
    k_deer_seq_update(const uint32_t* __restrict__ resid, uint32_t* done, int32_t* iters,
                      uint32_t* all_done, int64_t B, float eps, int k) {
    __shared__ int any_live;
    if (threadIdx.x == 0) any_live = 0;
    __syncthreads();
    int live = 0;
    for (int64_t b = threadIdx.x; b < B; b += blockDim.x) {
        if (done[b]) continue;
        const float rho = __uint_as_float(resid[b]);
        if (rho < eps || !(rho <= 3.4e38f)) {
            done[b] = 1u;
            iters[b] = k;
        } else {
            live = 1;
        }
    }
    if (live) atomicOr(&any_live, 1);
    __syncthreads();
    if (threadIdx.x == 0) *all_done = any_live ? 0u : 1u;
}

// Per-sequence solve, at the end: sequence b's last iterate (K_b, or
// `launched` when it never stopped) is in the second buffer when K_b is even;
// copy those channels into y.  Threads own channels, blocks stride over rows.
template <typename S>
__global__ void __launch_bounds__(256)
    k_deer_seq_gather(const S* __restrict__ ybuf, S* __restrict__ y, const int32_t* __restrict__ iters,
                      int launched, int64_t T, int64_t C, int64_t D) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    const int kb = iters[c / D] > 0 ? iters[c / D] : launched;
    if (kb & 1) return;
    for (int64_t t = blockIdx.y; t < T; t += gridDim.y) y[t * C + c] = ybuf[t * C + c];
}

cudaError_t launch_deer_seq_gather(const void* ybuf, void* y, const int32_t* iters, int launched,
                                   int64_t T, int64_t C, int64_t D, int dtype, cudaStream_t s) {
    const dim3 grid((unsigned)((C + 255) / 256), (unsigned)(T < 1024 ? T : 1024));
    if (dtype == 0)
        k_deer_seq_gather<float><<<grid, 256, 0, s>>>((const float*)ybuf, (float*)y, iters, launched,
                                                      T, C, D);
    else
        k_deer_seq_gather<__nv_bfloat16><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16*)ybuf, (__nv_bfloat16*)y, iters, launched, T, C, D);
    return cudaGetLastError();
}

cudaError_t launch_deer_seq_update(const uint32_t* resid, uint32_t* done, int32_t* iters,
                                   uint32_t* all_done, int64_t B, float eps, int k,
                                   cudaStream_t s) {
    k_deer_seq_update<<<1, 1024, 0, s>>>(resid, done, iters, all_done, B, eps, k);
    return cudaGetLastError();
}

template <typename S, bool VP, int M>
using DeerBwdOpT = DeerBwdOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_DEER_BWD, sizeof(S) == 2, M).NW,
                             kcfg(OP_DEER_BWD, sizeof(S) == 2, M).R>;

template <typename S, bool VP>
static cudaError_t deer_bwd_t(const float* w, const void* y, const void* h0, const void* dy,
                              void* du, void* dh0, float* partials, const Geom& g, const Carry& cr,
                              cudaStream_t s) {
    return launch_persist<DeerBwdOpT<S, VP, CARRY_CHAIN>, DeerBwdOpT<S, VP, CARRY_WALK>,
                          DeerBwdOpT<S, VP, TILE_TMA>, kcfg(OP_DEER_BWD, sizeof(S) == 2, TILE_TMA).ST>(
        {w, (const S*)y, (const S*)h0, (const S*)dy, (S*)du, (S*)dh0, partials}, g, cr, s);
}

cudaError_t launch_deer_bwd(int dtype, bool vec, const float* w, const void* y, const void* h0,
                            const void* dy, void* du, void* dh0, float* partials, const Geom& g,
                            const Carry& cr, cudaStream_t s) {
    if (dtype == 0)
        return vec ? deer_bwd_t<float, true>(w, y, h0, dy, du, dh0, partials, g, cr, s)
                   : deer_bwd_t<float, false>(w, y, h0, dy, du, dh0, partials, g, cr, s);
    return vec ? deer_bwd_t<__nv_bfloat16, true>(w, y, h0, dy, du, dh0, partials, g, cr, s)
               : deer_bwd_t<__nv_bfloat16, false>(w, y, h0, dy, du, dh0, partials, g, cr, s);
}

}  // namespace lrs
