// lstm_kernels.cu -- LSTM cell-state scan with a fused gate producer, forward
// and backward, page [P2] "RNN CUDA内核优化：实现序列长度无关的恒定推理延迟":
// the LSTM paragraph (the cell update C_t = f_t C_{t-1} + i_t C~_t is a linear
// recurrence whose time-varying coefficients are the forget and input gates)
// and checklist item 1 (make the recurrent path linear: the GILR-style cell,
// whose gates come from the input only).  The sigmoid / tanh of the four
// precomputed pre-activations, the scan and the output gate run in one kernel,
// so each element crosses HBM once.
//
// Forward, per element: f = sigmoid(zf + bf), i = sigmoid(zi + bi),
//   C~ = tanh(zc + bc), o = sigmoid(zo + bo),
//   C_t = f C_{t-1} + i C~  -- the scan with (a, b) = (f, i C~) --
//   h_t = o tanh(C_t).
// Backward, reverse time on u_t = f_t dC_t (what row t passes to row t-1):
//   e_t = dh o (1 - tanh^2 C_t),  dC_t = e_t + u_{t+1},  u_t = f_t dC_t,
//   dzf = dC C_{t-1} f (1-f),  dzi = dC C~ i (1-i),  dzc = dC i (1 - C~^2),
//   dzo = dh tanh(C_t) o (1-o)  (no scan needed: written before the carry is
//   known),  dc0 = u_0,
//   dbf, dbi, dbc, dbo: per-tile channel sums -> [4][n_chunks][C] partials ->
//   the fixed-order reduction over chunks, then over the batch.
#include "lr_act.cuh"
#include "lr_launch.h"
#include "lr_persist.cuh"

namespace lrs {

template <typename S>
struct LstmFwdParams {
    const S* zf;
    const S* zi;
    const S* zc;
    const S* zo;
    const float* bf;
    const float* bi;
    const float* bc;
    const float* bo;
    const S* c0;
    S* h;
    S* c;
};

template <typename S_, int VEC_, int NW_, int R_>
struct LstmFwdOp {
    using S = S_;
    static constexpr bool STRIP_ONE_BARRIER = LR_STRIP_ONEB != 0;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, MINB = 2;
    static constexpr bool REV = false;
    static constexpr int IN_ARRAYS = 4;  // zf, zi, zc, zo
    static constexpr bool SCRATCH_IN_CARRY = false;
    using Params = LstmFwdParams<S>;
    struct Regs {
        Pack<S, VEC> zf[R], zi[R], zc[R], zo[R];
    };
    struct Work {
        float fa[R][VEC], fb[R][VEC];  // scan element (f, i C~)
    };
    struct Smem {
        int unused;
    };
    struct Acc {};
    __device__ static void acc_init(Acc&) {}
    __device__ static bool skip(const Params&) { return false; }
    __device__ static const S* init_ptr(const Params& p) { return p.c0; }

    static constexpr int TMA_N = 4;  // staged: zf, zi, zc, zo
    __host__ __device__ static constexpr int tma_shift(int) { return 0; }
    __host__ __device__ static constexpr int tma_extra(int) { return 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.zf;
        ptr[1] = p.zi;
        ptr[2] = p.zc;
        ptr[3] = p.zo;
    }

    template <class Src>
    __device__ static void load(const Src& src, const Params& p, const Geom& g,
                                const TileCoord& tc, Regs& rg) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            if (tc.cok && t < g.T) {
                src.ld(rg.zf[r], 0, p.zf, t);
                src.ld(rg.zi[r], 1, p.zi, t);
                src.ld(rg.zc[r], 2, p.zc, t);
                src.ld(rg.zo[r], 3, p.zo, t);
            } else {
                rg.zf[r].ident(0.f);
                rg.zi[r].ident(0.f);
                rg.zc[r].ident(0.f);
                rg.zo[r].ident(0.f);
            }
        }
    }
    __device__ static void aggregate(const Params& p, const Geom& g, const TileCoord& tc,
                                     const Regs& rg, Work& w, float (&A)[VEC], float (&B)[VEC],
                                     bool) {
        float bfv[VEC], biv[VEC], bcv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { bfv[v] = 0.f; biv[v] = 0.f; bcv[v] = 0.f; }
        if (tc.cok) {
            load_param<VEC>(p.bf + tc.cd, bfv);
            load_param<VEC>(p.bi + tc.cd, biv);
            load_param<VEC>(p.bc + tc.cd, bcv);
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool ok = tc.cok && tc.t0 + r < g.T;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float f = act_sigmoid(rg.zf[r].get(v) + bfv[v]);
                const float i = act_sigmoid(rg.zi[r].get(v) + biv[v]);
                const float cand = act_tanh(rg.zc[r].get(v) + bcv[v]);
                w.fa[r][v] = ok ? f : 1.f;
                w.fb[r][v] = ok ? i * cand : 0.f;
                B[v] = w.fa[r][v] * B[v] + w.fb[r][v];
                A[v] *= w.fa[r][v];
            }
        }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work& w, float (&s)[VEC], Smem&, Acc&) {
        float bov[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) bov[v] = 0.f;
        if (tc.cok) load_param<VEC>(p.bo + tc.cd, bov);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            float hv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                s[v] = w.fa[r][v] * s[v] + w.fb[r][v];
                const float o = act_sigmoid(rg.zo[r].get(v) + bov[v]);
                hv[v] = o * act_tanh(s[v]);
            }
            if (tc.cok && t < g.T) {
                store_vec<S, VEC>(p.c + t * g.C + tc.c, s);
                store_vec<S, VEC>(p.h + t * g.C + tc.c, hv);
            }
        }
    }
    __device__ static void at_exit(const Params&, Smem&, Acc&) {}
};

template <typename S>
struct LstmBwdParams {
    const S* zf;
    const S* zi;
    const S* zc;
    const S* zo;
    const float* bf;
    const float* bi;
    const float* bc;
    const float* bo;
    const S* c0;
    const S* c;
    const S* dh;
    S* dzf;
    S* dzi;
    S* dzc;
    S* dzo;
    S* dc0;
    float* partials;  // [4][n_chunks][C]: f, i, c, o
};

template <typename S_, int VEC_, int NW_, int R_>
struct LstmBwdOp {
    using S = S_;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, MINB = 2;
    static constexpr bool REV = true;
    static constexpr int IN_ARRAYS = 7;  // zf, zi, zc, zo, C, C_{t-1}, dh
    using Params = LstmBwdParams<S>;
    struct Regs {
        Pack<S, VEC> zf[R], zi[R], zc[R], zo[R], c[R], cp[R], dh[R];
    };
    struct Work {
        float F[R][VEC], E[R][VEC];
        float sum_o[VEC];
    };
    // Two of the four partial-sum arrays at a time (8 KB), over the carry's
    // warp aggregates: finish() writes them only after a barrier that every
    // warp reaches once it is done with those.
    struct Smem {
        float p0[NW][32][VEC];
        float p1[NW][32][VEC];
    };
    static constexpr bool SCRATCH_IN_CARRY = true;
    struct Acc {
        float sf[VEC], si[VEC], sc[VEC], so[VEC];  // bias sums over a run of tiles (acc_run)
    };
    __device__ static void acc_init(Acc& a) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) { a.sf[v] = 0.f; a.si[v] = 0.f; a.sc[v] = 0.f; a.so[v] = 0.f; }
    }
    __device__ static bool skip(const Params&) { return false; }
    __device__ static const S* init_ptr(const Params&) { return nullptr; }  // u_T = 0

    static constexpr int TMA_N = 6;  // staged: zf, zi, zc, zo, dh, C (rows t0-1 .. t0+L-1)
    __host__ __device__ static constexpr int tma_shift(int k) { return k == 5 ? -1 : 0; }
    __host__ __device__ static constexpr int tma_extra(int k) { return k == 5 ? 1 : 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.zf;
        ptr[1] = p.zi;
        ptr[2] = p.zc;
        ptr[3] = p.zo;
        ptr[4] = p.dh;
        ptr[5] = p.c;
    }

    template <class Src>
    __device__ static void load(const Src& src, const Params& p, const Geom& g,
                                const TileCoord& tc, Regs& rg) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            if (tc.cok && t < g.T) {
                src.ld(rg.zf[r], 0, p.zf, t);
                src.ld(rg.zi[r], 1, p.zi, t);
                src.ld(rg.zc[r], 2, p.zc, t);
                src.ld(rg.zo[r], 3, p.zo, t);
                src.ld(rg.dh[r], 4, p.dh, t);
                src.ld(rg.c[r], 5, p.c, t);
                if (t > 0) src.ld(rg.cp[r], 5, p.c, t - 1);
                else if (p.c0 != nullptr) rg.cp[r].load(p.c0 + tc.c);
                else rg.cp[r].ident(0.f);
            } else {
                rg.zf[r].ident(0.f);
                rg.zi[r].ident(0.f);
                rg.zc[r].ident(0.f);
                rg.zo[r].ident(0.f);
                rg.dh[r].ident(0.f);
                rg.c[r].ident(0.f);
                rg.cp[r].ident(0.f);
            }
        }
    }
    __device__ static void aggregate(const Params& p, const Geom& g, const TileCoord& tc,
                                     const Regs& rg, Work& w, float (&A)[VEC], float (&B)[VEC],
                                     bool side) {
        float bfv[VEC], bov[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { bfv[v] = 0.f; bov[v] = 0.f; w.sum_o[v] = 0.f; }
        if (tc.cok) {
            load_param<VEC>(p.bf + tc.cd, bfv);
            load_param<VEC>(p.bo + tc.cd, bov);
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            const bool ok = tc.cok && t < g.T;
            float dzov[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float f = act_sigmoid(rg.zf[r].get(v) + bfv[v]);
                const float o = act_sigmoid(rg.zo[r].get(v) + bov[v]);
                float d1;
                const float th = act_tanh_d(rg.c[r].get(v), d1);
                const float gv = rg.dh[r].get(v);
                dzov[v] = gv * th * o * (1.f - o);
                if (ok) w.sum_o[v] += dzov[v];
                w.F[r][v] = ok ? f : 1.f;
                w.E[r][v] = ok ? gv * o * d1 : 0.f;
                B[v] = w.F[r][v] * (w.E[r][v] + B[v]);
                A[v] *= w.F[r][v];
            }
            if (ok && side) store_vec<S, VEC>(p.dzo + t * g.C + tc.c, dzov);
        }
    }
    // Sum the NW warps' rows of one channel pair of arrays (fixed warp order)
    // and write them as this tile's partials of arrays k0 and k0 + 1.
    __device__ static void flush_pair(const Params& p, const Geom& g, const TileCoord& tc,
                                      const Smem& xs, int k0, int lane) {
        float s0[VEC], s1[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { s0[v] = 0.f; s1[v] = 0.f; }
#pragma unroll
        for (int ww = 0; ww < NW; ++ww)
#pragma unroll
            for (int v = 0; v < VEC; ++v) { s0[v] += xs.p0[ww][lane][v]; s1[v] += xs.p1[ww][lane][v]; }
        float* q0 = p.partials + ((int64_t)k0 * g.n_chunks + tc.tchunk) * g.C + tc.c;
        float* q1 = q0 + g.n_chunks * g.C;
#pragma unroll
        for (int v = 0; v < VEC; ++v) { q0[v] = s0[v]; q1[v] = s1[v]; }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work& w, float (&s)[VEC], Smem& xs, Acc& acc) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        float biv[VEC], bcv[VEC];
        float sum_f[VEC], sum_i[VEC], sum_c[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            biv[v] = 0.f;
            bcv[v] = 0.f;
            sum_f[v] = 0.f;
            sum_i[v] = 0.f;
            sum_c[v] = 0.f;
        }
        if (tc.cok) {
            load_param<VEC>(p.bi + tc.cd, biv);
            load_param<VEC>(p.bc + tc.cd, bcv);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            const bool ok = tc.cok && t < g.T;
            float dzfv[VEC], dziv[VEC], dzcv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float dc = w.E[r][v] + s[v];
                const float f = w.F[r][v];
                const float i = act_sigmoid(rg.zi[r].get(v) + biv[v]);
                const float cand = act_tanh(rg.zc[r].get(v) + bcv[v]);
                dzfv[v] = dc * rg.cp[r].get(v) * f * (1.f - f);
                dziv[v] = dc * cand * i * (1.f - i);
                dzcv[v] = dc * i * (1.f - cand * cand);
                s[v] = f * dc;
                if (ok) {
                    sum_f[v] += dzfv[v];
                    sum_i[v] += dziv[v];
                    sum_c[v] += dzcv[v];
                }
            }
            if (ok) {
                store_vec<S, VEC>(p.dzf + t * g.C + tc.c, dzfv);
                store_vec<S, VEC>(p.dzi + t * g.C + tc.c, dziv);
                store_vec<S, VEC>(p.dzc + t * g.C + tc.c, dzcv);
            }
        }
        if (tc.tchunk == 0 && warp == NW - 1 && p.dc0 != nullptr && tc.cok)
            store_vec<S, VEC>(p.dc0 + tc.c, s);
        if (tc.acc_run) {
            // a run of tiles of these channels through this CTA: the sums run
            // over it in registers; a tile's partial rows are zeros and the
            // run's last tile writes the totals (the reduction over chunks is
            // unchanged)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                acc.sf[v] += sum_f[v];
                acc.si[v] += sum_i[v];
                acc.sc[v] += sum_c[v];
                acc.so[v] += w.sum_o[v];
            }
            if (!tc.acc_flush) {
                if (warp == 0 && tc.cok) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float* q = p.partials + ((int64_t)k * g.n_chunks + tc.tchunk) * g.C + tc.c;
#pragma unroll
                        for (int v = 0; v < VEC; ++v) q[v] = 0.f;
                    }
                }
                return;
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sum_f[v] = acc.sf[v];
                sum_i[v] = acc.si[v];
                sum_c[v] = acc.sc[v];
                w.sum_o[v] = acc.so[v];
                acc.sf[v] = acc.si[v] = acc.sc[v] = acc.so[v] = 0.f;
            }
        }
        // bias-gradient partials of this tile (or strip), two arrays per round
        csync<NW>();  // every warp is past its reads of the carry smem
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            xs.p0[warp][lane][v] = sum_f[v];
            xs.p1[warp][lane][v] = sum_i[v];
        }
        csync<NW>();
        if (warp == 0 && tc.cok) flush_pair(p, g, tc, xs, 0, lane);
        csync<NW>();  // warp 0 has read round one
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            xs.p0[warp][lane][v] = sum_c[v];
            xs.p1[warp][lane][v] = w.sum_o[v];
        }
        csync<NW>();
        if (warp == NW - 1 && tc.cok) flush_pair(p, g, tc, xs, 2, lane);
    }
    __device__ static void at_exit(const Params&, Smem&, Acc&) {}
};

// The LSTM cell's kernels take the SRU cell's tile shapes: the same number of
// staged arrays per direction (4 forward; 6 backward, C read at two rows).
template <typename S, bool VP, int M>
using LstmFwdOpT = LstmFwdOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_LSTM_FWD, sizeof(S) == 2, M).NW,
                             kcfg(OP_LSTM_FWD, sizeof(S) == 2, M).R>;
template <typename S, bool VP, int M>
using LstmBwdOpT = LstmBwdOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_LSTM_BWD, sizeof(S) == 2, M).NW,
                             kcfg(OP_LSTM_BWD, sizeof(S) == 2, M).R>;

template <typename S, bool VP>
static cudaError_t lstm_fwd_t(const LstmFwdParams<S>& p, const Geom& g, const Carry& cr,
                              cudaStream_t s) {
    return launch_persist<LstmFwdOpT<S, VP, CARRY_CHAIN>, LstmFwdOpT<S, VP, CARRY_WALK>,
                          LstmFwdOpT<S, VP, TILE_TMA>, kcfg(OP_LSTM_FWD, sizeof(S) == 2, TILE_TMA).ST>(
        p, g, cr, s);
}

template <typename S, bool VP>
static cudaError_t lstm_bwd_t(const LstmBwdParams<S>& p, const Geom& g, const Carry& cr,
                              cudaStream_t s) {
    return launch_persist<LstmBwdOpT<S, VP, CARRY_CHAIN>, LstmBwdOpT<S, VP, CARRY_WALK>,
                          LstmBwdOpT<S, VP, TILE_TMA>, kcfg(OP_LSTM_BWD, sizeof(S) == 2, TILE_TMA).ST>(
        p, g, cr, s);
}

template <typename S>
static cudaError_t lstm_fwd_s(bool vec, const LstmGates& z, const LstmBias& b, const void* c0,
                              void* h, void* c, const Geom& g, const Carry& cr, cudaStream_t s) {
    const LstmFwdParams<S> p{(const S*)z.f, (const S*)z.i, (const S*)z.c, (const S*)z.o,
                             b.f, b.i, b.c, b.o, (const S*)c0, (S*)h, (S*)c};
    return vec ? lstm_fwd_t<S, true>(p, g, cr, s) : lstm_fwd_t<S, false>(p, g, cr, s);
}

template <typename S>
static cudaError_t lstm_bwd_s(bool vec, const LstmGates& z, const LstmBias& b, const void* c0,
                              const void* c, const void* dh, const LstmGates& dz, void* dc0,
                              float* partials, const Geom& g, const Carry& cr, cudaStream_t s) {
    const LstmBwdParams<S> p{(const S*)z.f, (const S*)z.i, (const S*)z.c, (const S*)z.o,
                             b.f, b.i, b.c, b.o, (const S*)c0, (const S*)c, (const S*)dh,
                             (S*)dz.f, (S*)dz.i, (S*)dz.c, (S*)dz.o, (S*)dc0, partials};
    return vec ? lstm_bwd_t<S, true>(p, g, cr, s) : lstm_bwd_t<S, false>(p, g, cr, s);
}

cudaError_t launch_lstm_fwd(int dtype, bool vec, const LstmGates& z, const LstmBias& b,
                            const void* c0, void* h, void* c, const Geom& g, const Carry& cr,
                            cudaStream_t s) {
    return dtype == 0 ? lstm_fwd_s<float>(vec, z, b, c0, h, c, g, cr, s)
                      : lstm_fwd_s<__nv_bfloat16>(vec, z, b, c0, h, c, g, cr, s);
}

cudaError_t launch_lstm_bwd(int dtype, bool vec, const LstmGates& z, const LstmBias& b,
                            const void* c0, const void* c, const void* dh, const LstmGates& dz,
                            void* dc0, float* partials, const Geom& g, const Carry& cr,
                            cudaStream_t s) {
    return dtype == 0
               ? lstm_bwd_s<float>(vec, z, b, c0, c, dh, dz, dc0, partials, g, cr, s)
               : lstm_bwd_s<__nv_bfloat16>(vec, z, b, c0, c, dh, dz, dc0, partials, g, cr, s);
}

}  // namespace lrs
