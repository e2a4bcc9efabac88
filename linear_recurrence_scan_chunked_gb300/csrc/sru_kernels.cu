// sru_kernels.cu -- fused linear-form SRU layer, forward and backward (rows a3,
// a4), page [P1] "CUDA并行化RNN训练：从O(T)到O(log T)的工程实践与参数调优":
// SRU paragraph (the forget gate depends on the current input only, v_f = 0
// here; the highway reset gate mixes input and memory) and checklist item 2
// (all sigmoid / tanh / multiply-add work of the layer in one kernel, so each
// element crosses HBM once).
//
// Forward, per element: f = sigmoid(uf + bf), r = sigmoid(ur + br),
//   c_t = f c_{t-1} + (1-f) xt  -- the scan with (a, b) = (f, (1-f) xt) --
//   h_t = r tanh(c_t) + (1-r) x.
// Backward, reverse time on u_t = f_t dc_t (what row t passes to row t-1):
//   e_t = dh r (1 - tanh^2 c_t),  u_t = f_t (e_t + u_{t+1}),  dc_t = e_t + u_{t+1},
//   dxt = dc (1-f),  duf = dc (c_{t-1} - xt) f (1-f),  dc0 = u_0,
//   dur = dh (tanh c - x) r (1-r),  dx = dh (1-r)  (no scan needed: written
//   before the carry is known),
//   dbf, dbr: per-tile channel sums -> [2][n_chunks][C] partials -> a
//   fixed-order reduction over chunks, then over the batch (deterministic).
#include "lr_act.cuh"
#include "lr_launch.h"
#include "lr_persist.cuh"

namespace lrs {

template <typename S>
struct SruFwdParams {
    const S* xt;
    const S* uf;
    const S* ur;
    const S* x;
    const float* bf;
    const float* br;
    const S* c0;
    S* h;
    S* c;
};

template <typename S_, int VEC_, int NW_, int R_>
struct SruFwdOp {
    using S = S_;
    static constexpr bool STRIP_ONE_BARRIER = LR_STRIP_ONEB != 0;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, MINB = 2;
    static constexpr bool REV = false;
    static constexpr int IN_ARRAYS = 4;  // xt, uf, ur, x
    static constexpr bool SCRATCH_IN_CARRY = false;
    using Params = SruFwdParams<S>;
    struct Regs {
        Pack<S, VEC> xt[R], uf[R], ur[R], x[R];
    };
    struct Work {
        float fa[R][VEC], fb[R][VEC];  // scan element (f, (1-f) xt)
    };
    struct Smem {
        int unused;
    };
    struct Acc {};
    __device__ static void acc_init(Acc&) {}
    __device__ static bool skip(const Params&) { return false; }
    __device__ static const S* init_ptr(const Params& p) { return p.c0; }

    static constexpr int TMA_N = 4;  // staged: xt, uf, ur, x
    __host__ __device__ static constexpr int tma_shift(int) { return 0; }
    __host__ __device__ static constexpr int tma_extra(int) { return 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.xt;
        ptr[1] = p.uf;
        ptr[2] = p.ur;
        ptr[3] = p.x;
    }

    template <class Src>
    __device__ static void load(const Src& src, const Params& p, const Geom& g,
                                const TileCoord& tc, Regs& rg) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            if (tc.cok && t < g.T) {
                src.ld(rg.xt[r], 0, p.xt, t);
                src.ld(rg.uf[r], 1, p.uf, t);
                src.ld(rg.ur[r], 2, p.ur, t);
                src.ld(rg.x[r], 3, p.x, t);
            } else {
                rg.xt[r].ident(0.f);
                rg.uf[r].ident(0.f);
                rg.ur[r].ident(0.f);
                rg.x[r].ident(0.f);
            }
        }
    }
    __device__ static void aggregate(const Params& p, const Geom& g, const TileCoord& tc,
                                     const Regs& rg, Work& w, float (&A)[VEC], float (&B)[VEC],
                                     bool side) {
        float bfv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) bfv[v] = 0.f;
        if (tc.cok) load_param<VEC>(p.bf + tc.cd, bfv);
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool ok = tc.cok && tc.t0 + r < g.T;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float f = act_sigmoid(rg.uf[r].get(v) + bfv[v]);
                w.fa[r][v] = ok ? f : 1.f;
                w.fb[r][v] = ok ? (1.f - f) * rg.xt[r].get(v) : 0.f;
                B[v] = w.fa[r][v] * B[v] + w.fb[r][v];
                A[v] *= w.fa[r][v];
            }
        }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work& w, float (&s)[VEC], Smem&, Acc&) {
        float brv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) brv[v] = 0.f;
        if (tc.cok) load_param<VEC>(p.br + tc.cd, brv);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            float hv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                s[v] = w.fa[r][v] * s[v] + w.fb[r][v];
                const float rg_ = act_sigmoid(rg.ur[r].get(v) + brv[v]);
                hv[v] = rg_ * act_tanh(s[v]) + (1.f - rg_) * rg.x[r].get(v);
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
struct SruBwdParams {
    const S* xt;
    const S* uf;
    const S* ur;
    const S* x;
    const float* bf;
    const float* br;
    const S* c0;
    const S* c;
    const S* dh;
    S* dxt;
    S* duf;
    S* dur;
    S* dx;
    S* dc0;
    float* partials;  // [2][n_chunks][C]
};

template <typename S_, int VEC_, int NW_, int R_>
struct SruBwdOp {
    using S = S_;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, MINB = 2;
    static constexpr bool REV = true;
    static constexpr int IN_ARRAYS = 7;  // xt, uf, ur, x, c, c_{t-1}, dh
    using Params = SruBwdParams<S>;
    struct Regs {
        Pack<S, VEC> xt[R], uf[R], ur[R], x[R], c[R], cp[R], dh[R];
    };
    struct Work {
        float F[R][VEC], E[R][VEC], XT[R][VEC], CP[R][VEC];
        float sum_r[VEC];
    };
    struct Smem {
        float pf[NW][32][VEC];
        float pr[NW][32][VEC];
    };
    // The 8 KB of partial sums may overlay the carry's warp aggregates (the
    // TMA kernels do that to keep two CTAs per SM): finish() writes them only
    // after a barrier that every warp reaches once it is done with those.
    static constexpr bool SCRATCH_IN_CARRY = true;
    struct Acc {
        float sf[VEC], sr[VEC];  // bias sums over a run of tiles (acc_run)
    };
    __device__ static void acc_init(Acc& a) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) { a.sf[v] = 0.f; a.sr[v] = 0.f; }
    }
    __device__ static bool skip(const Params&) { return false; }
    __device__ static const S* init_ptr(const Params&) { return nullptr; }  // u_T = 0

    static constexpr int TMA_N = 6;  // staged: xt, uf, ur, x, dh, c (rows t0-1 .. t0+L-1)
    __host__ __device__ static constexpr int tma_shift(int k) { return k == 5 ? -1 : 0; }
    __host__ __device__ static constexpr int tma_extra(int k) { return k == 5 ? 1 : 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.xt;
        ptr[1] = p.uf;
        ptr[2] = p.ur;
        ptr[3] = p.x;
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
                src.ld(rg.xt[r], 0, p.xt, t);
                src.ld(rg.uf[r], 1, p.uf, t);
                src.ld(rg.ur[r], 2, p.ur, t);
                src.ld(rg.x[r], 3, p.x, t);
                src.ld(rg.dh[r], 4, p.dh, t);
                src.ld(rg.c[r], 5, p.c, t);
                if (t > 0) src.ld(rg.cp[r], 5, p.c, t - 1);
                else if (p.c0 != nullptr) rg.cp[r].load(p.c0 + tc.c);
                else rg.cp[r].ident(0.f);
            } else {
                rg.xt[r].ident(0.f);
                rg.uf[r].ident(0.f);
                rg.ur[r].ident(0.f);
                rg.x[r].ident(0.f);
                rg.c[r].ident(0.f);
                rg.cp[r].ident(0.f);
                rg.dh[r].ident(0.f);
            }
        }
    }
    __device__ static void aggregate(const Params& p, const Geom& g, const TileCoord& tc,
                                     const Regs& rg, Work& w, float (&A)[VEC], float (&B)[VEC],
                                     bool side) {
        float bfv[VEC], brv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { bfv[v] = 0.f; brv[v] = 0.f; w.sum_r[v] = 0.f; }
        if (tc.cok) {
            load_param<VEC>(p.bf + tc.cd, bfv);
            load_param<VEC>(p.br + tc.cd, brv);
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            const bool ok = tc.cok && t < g.T;
            float durv[VEC], dxv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float f = act_sigmoid(rg.uf[r].get(v) + bfv[v]);
                const float rg_ = act_sigmoid(rg.ur[r].get(v) + brv[v]);
                float d1;
                const float th = act_tanh_d(rg.c[r].get(v), d1);
                const float gv = rg.dh[r].get(v);
                durv[v] = gv * (th - rg.x[r].get(v)) * rg_ * (1.f - rg_);
                dxv[v] = gv * (1.f - rg_);
                if (ok) w.sum_r[v] += durv[v];
                w.F[r][v] = ok ? f : 1.f;
                w.E[r][v] = ok ? gv * rg_ * d1 : 0.f;
                w.XT[r][v] = rg.xt[r].get(v);
                w.CP[r][v] = rg.cp[r].get(v);
                B[v] = w.F[r][v] * (w.E[r][v] + B[v]);
                A[v] *= w.F[r][v];
            }
            if (ok && side) {
                store_vec<S, VEC>(p.dur + t * g.C + tc.c, durv);
                store_vec<S, VEC>(p.dx + t * g.C + tc.c, dxv);
            }
        }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs&, Work& w, float (&s)[VEC], Smem& xs, Acc& acc) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        float sum_f[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) sum_f[v] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            const bool ok = tc.cok && t < g.T;
            float dxtv[VEC], dufv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float dc = w.E[r][v] + s[v];
                const float f = w.F[r][v];
                dxtv[v] = dc * (1.f - f);
                dufv[v] = dc * (w.CP[r][v] - w.XT[r][v]) * f * (1.f - f);
                s[v] = f * dc;
                if (ok) sum_f[v] += dufv[v];
            }
            if (ok) {
                store_vec<S, VEC>(p.dxt + t * g.C + tc.c, dxtv);
                store_vec<S, VEC>(p.duf + t * g.C + tc.c, dufv);
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
            for (int v = 0; v < VEC; ++v) { acc.sf[v] += sum_f[v]; acc.sr[v] += w.sum_r[v]; }
            if (!tc.acc_flush) {
                if (warp == 0 && tc.cok) {
                    float* pfp = p.partials + tc.tchunk * g.C + tc.c;
                    float* prp = p.partials + (g.n_chunks + tc.tchunk) * g.C + tc.c;
#pragma unroll
                    for (int v = 0; v < VEC; ++v) { pfp[v] = 0.f; prp[v] = 0.f; }
                }
                return;
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sum_f[v] = acc.sf[v];
                w.sum_r[v] = acc.sr[v];
                acc.sf[v] = 0.f;
                acc.sr[v] = 0.f;
            }
        }
        // bias-gradient partials of this tile (or strip): fixed warp order
        csync<NW>();  // every warp is past its reads of the carry smem
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            xs.pf[warp][lane][v] = sum_f[v];
            xs.pr[warp][lane][v] = w.sum_r[v];
        }
        csync<NW>();
        if (warp == 0 && tc.cok) {
            float pf[VEC], pr[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) { pf[v] = 0.f; pr[v] = 0.f; }
#pragma unroll
            for (int ww = 0; ww < NW; ++ww)
#pragma unroll
                for (int v = 0; v < VEC; ++v) { pf[v] += xs.pf[ww][lane][v]; pr[v] += xs.pr[ww][lane][v]; }
            float* pfp = p.partials + tc.tchunk * g.C + tc.c;
            float* prp = p.partials + (g.n_chunks + tc.tchunk) * g.C + tc.c;
#pragma unroll
            for (int v = 0; v < VEC; ++v) { pfp[v] = pf[v]; prp[v] = pr[v]; }
        }
    }
    __device__ static void at_exit(const Params&, Smem&, Acc&) {}
};

// Per-feature parameter gradients (SRU and LSTM biases, DEER's w) from
// per-tile partials, in a fixed order (deterministic): stage 1 sums every
// channel over the time chunks, stage 2 sums the batch rows of each feature.
// partials: [n_arr][n_chunks][C]; colsum: [n_arr][C]; out.o[k]: [D] for
// k < n_arr.  Stage 1: a block owns 32 channels (x) and kColLanes chunk lanes
// (y); lane y sums chunks y, y + kColLanes, ... (each step one coalesced row
// segment), then lane 0 adds the lanes' sums in lane order -- so a channel's
// chain of dependent loads is n_chunks / kColLanes long, not n_chunks.
constexpr int kColLanes = 32;
__global__ void __launch_bounds__(32 * kColLanes)
    k_bias_colsum(const float* __restrict__ partials, int64_t n_chunks, int64_t C,
                  float* __restrict__ colsum) {
    __shared__ float part[kColLanes][33];
    const int64_t c = (int64_t)blockIdx.x * 32 + threadIdx.x;
    const int64_t which = blockIdx.y;
    float acc = 0.f;
    if (c < C) {
        const float* p = partials + which * n_chunks * C + c;
#pragma unroll 4
        for (int64_t k = threadIdx.y; k < n_chunks; k += kColLanes) acc += __ldg(p + k * C);
    }
    part[threadIdx.y][threadIdx.x] = acc;
    __syncthreads();
    if (threadIdx.y == 0 && c < C) {
        float sum = 0.f;
#pragma unroll
        for (int l = 0; l < kColLanes; ++l) sum += part[l][threadIdx.x];
        colsum[which * C + c] = sum;
    }
}

__global__ void __launch_bounds__(256)
    k_bias_batch(const float* __restrict__ colsum, int64_t B, int64_t D, int n_arr, BiasOut out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_arr * D) return;
    const int64_t which = i / D, d = i % D;
    const float* cs = colsum + which * B * D + d;
    float s = 0.f;
    for (int64_t b = 0; b < B; ++b) s += __ldg(cs + b * D);
    out.o[which][d] = s;
}

template <typename S, bool VP, int M>
using SruFwdOpT = SruFwdOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_SRU_FWD, sizeof(S) == 2, M).NW,
                           kcfg(OP_SRU_FWD, sizeof(S) == 2, M).R>;
template <typename S, bool VP, int M>
using SruBwdOpT = SruBwdOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_SRU_BWD, sizeof(S) == 2, M).NW,
                           kcfg(OP_SRU_BWD, sizeof(S) == 2, M).R>;

template <typename S, bool VP>
static cudaError_t sru_fwd_t(const void* xt, const void* uf, const void* ur, const void* x,
                             const float* bf, const float* br, const void* c0, void* h, void* c,
                             const Geom& g, const Carry& cr, cudaStream_t s) {
    return launch_persist<SruFwdOpT<S, VP, CARRY_CHAIN>, SruFwdOpT<S, VP, CARRY_WALK>,
                          SruFwdOpT<S, VP, TILE_TMA>, kcfg(OP_SRU_FWD, sizeof(S) == 2, TILE_TMA).ST>(
        {(const S*)xt, (const S*)uf, (const S*)ur, (const S*)x, bf, br, (const S*)c0, (S*)h, (S*)c},
        g, cr, s);
}

template <typename S, bool VP>
static cudaError_t sru_bwd_t(const void* xt, const void* uf, const void* ur, const void* x,
                             const float* bf, const float* br, const void* c0, const void* c,
                             const void* dh, void* dxt, void* duf, void* dur, void* dx, void* dc0,
                             float* partials, const Geom& g, const Carry& cr, cudaStream_t s) {
    return launch_persist<SruBwdOpT<S, VP, CARRY_CHAIN>, SruBwdOpT<S, VP, CARRY_WALK>,
                          SruBwdOpT<S, VP, TILE_TMA>, kcfg(OP_SRU_BWD, sizeof(S) == 2, TILE_TMA).ST>(
        {(const S*)xt, (const S*)uf, (const S*)ur, (const S*)x, bf, br, (const S*)c0, (const S*)c,
         (const S*)dh, (S*)dxt, (S*)duf, (S*)dur, (S*)dx, (S*)dc0, partials},
        g, cr, s);
}

cudaError_t launch_sru_fwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           void* h, void* c, const Geom& g, const Carry& cr, cudaStream_t s) {
    if (dtype == 0)
        return vec ? sru_fwd_t<float, true>(xt, uf, ur, x, bf, br, c0, h, c, g, cr, s)
                   : sru_fwd_t<float, false>(xt, uf, ur, x, bf, br, c0, h, c, g, cr, s);
    return vec ? sru_fwd_t<__nv_bfloat16, true>(xt, uf, ur, x, bf, br, c0, h, c, g, cr, s)
               : sru_fwd_t<__nv_bfloat16, false>(xt, uf, ur, x, bf, br, c0, h, c, g, cr, s);
}

cudaError_t launch_sru_bwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           const void* c, const void* dh, void* dxt, void* duf, void* dur,
                           void* dx, void* dc0, float* partials, const Geom& g,
                           const Carry& cr, cudaStream_t s) {
    if (dtype == 0)
        return vec ? sru_bwd_t<float, true>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur, dx,
                                            dc0, partials, g, cr, s)
                   : sru_bwd_t<float, false>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur, dx,
                                             dc0, partials, g, cr, s);
    return vec ? sru_bwd_t<__nv_bfloat16, true>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur,
                                                dx, dc0, partials, g, cr, s)
               : sru_bwd_t<__nv_bfloat16, false>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur,
                                                 dx, dc0, partials, g, cr, s);
}

cudaError_t launch_bias_reduce(const float* partials, int64_t n_chunks, int n_arr, int64_t B,
                               int64_t D, BiasOut out, cudaStream_t s) {
    if (n_arr < 1 || n_arr > 4) return cudaErrorInvalidValue;
    const int64_t C = B * D;
    float* colsum = const_cast<float*>(partials) + n_arr * n_chunks * C;
    k_bias_colsum<<<dim3((unsigned)((C + 31) / 32), (unsigned)n_arr), dim3(32, kColLanes), 0, s>>>(
        partials, n_chunks, C, colsum);
    k_bias_batch<<<(unsigned)((n_arr * D + 255) / 256), 256, 0, s>>>(colsum, B, D, n_arr, out);
    return cudaGetLastError();
}

}  // namespace lrs
