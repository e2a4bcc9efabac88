// scan_kernels.cu -- forward and backward diagonal linear scan (rows a1, a2).
//
// Forward: h_t = a_t h_{t-1} + b_t, h_{-1} = h0 -- page [P2] "RNN CUDA内核优化：
// 实现序列长度无关的恒定推理延迟" (LSTM paragraph) and page [P1] "CUDA并行化RNN训练：
// 从O(T)到O(log T)的工程实践与参数调优" (parallel-scan paragraph).
//
// Backward ([P1] parallel-scan paragraph: the same scan serves backward) is
// run in reverse time on u_t = a_t delta_t, the gradient that row t passes to
// row t-1:
//     u_t = a_t (dh_t + u_{t+1}),  u_T = 0,
//     delta_t = dh_t + u_{t+1},  db_t = delta_t,  da_t = delta_t h_{t-1},
//     dh0 = u_0.
// The scan element of row t is the affine map u -> a_t u + a_t dh_t, which
// needs only row-t data, so the carry between tiles is u at the tile edge.
//
// Each element of a, b (resp. a, h, dh) is read once from HBM and each output
// written once: a tile is held in registers between the local scan and the
// output pass while its carry resolves, and the next tile's loads are already
// in flight (lr_persist.cuh).
#include "lr_launch.h"
#include "lr_persist.cuh"

namespace lrs {

template <typename S>
struct ScanFwdParams {
    const S* a;
    const S* b;
    const S* h0;
    S* h;
};

template <typename S_, int VEC_, int NW_, int R_, int RG_ = 1>
struct ScanFwdOp {
    using S = S_;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, RG = RG_, MINB = 2;
    static constexpr bool REV = false;
    static constexpr int IN_ARRAYS = 2;  // a, b
    static constexpr bool STREAM_WS = LR_STREAM_WS != 0;
    static constexpr bool SCRATCH_IN_CARRY = false;
    using Params = ScanFwdParams<S>;
    struct Regs {
        Pack<S, VEC> a[R], b[R];
    };
    struct Work {};
    struct Smem {
        int unused;
    };
    struct Acc {};
    __device__ static void acc_init(Acc&) {}
    __device__ static bool skip(const Params&) { return false; }
    __device__ static const S* init_ptr(const Params& p) { return p.h0; }

    static constexpr int TMA_N = 2;  // staged: a, b
    __host__ __device__ static constexpr int tma_shift(int) { return 0; }
    __host__ __device__ static constexpr int tma_extra(int) { return 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.a;
        ptr[1] = p.b;
    }

    template <class Src>
    __device__ static void load(const Src& src, const Params& p, const Geom& g,
                                const TileCoord& tc, Regs& rg) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
            if (tc.cok && t < g.T) {
                src.ld(rg.a[r], 0, p.a, t);
                src.ld(rg.b[r], 1, p.b, t);
            } else {  // identity element (1, 0) outside the problem
                rg.a[r].ident(1.f);
                rg.b[r].ident(0.f);
            }
        }
    }
    __device__ static void aggregate(const Params&, const Geom&, const TileCoord&, const Regs& rg,
                                     Work&, float (&A)[VEC], float (&B)[VEC], bool) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float av = rg.a[r].get(v);
                B[v] = av * B[v] + rg.b[r].get(v);
                A[v] *= av;
            }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work&, float (&s)[VEC], Smem&, Acc&) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 + r;
#pragma unroll
            for (int v = 0; v < VEC; ++v) s[v] = rg.a[r].get(v) * s[v] + rg.b[r].get(v);
            if (tc.cok && t < g.T) store_vec<S, VEC>(p.h + t * g.C + tc.c, s);
        }
    }
    __device__ static void at_exit(const Params&, Smem&, Acc&) {}
};

template <typename S>
struct ScanBwdParams {
    const S* a;
    const S* h;
    const S* h0;
    const S* dh;
    S* da;
    S* db;
    S* dh0;
};

// RG_: row groups per warp (the lanes of a warp split into RG_ groups of R_
// consecutive rows; 1 everywhere but the cluster kernel's vector path).
template <typename S_, int VEC_, int NW_, int R_, int RG_ = 1>
struct ScanBwdOp {
    using S = S_;
    static constexpr int VEC = VEC_, NW = NW_, R = R_, RG = RG_, MINB = 2;
    static constexpr bool REV = true;
    static constexpr int IN_ARRAYS = 3;  // a, dh, h
    static constexpr bool SCRATCH_IN_CARRY = false;
    using Params = ScanBwdParams<S>;
    struct Regs {
        Pack<S, VEC> a[R], g[R], hp[R];  // a_t, dh_t, h_{t-1}
    };
    struct Work {};
    struct Smem {
        int unused;
    };
    struct Acc {};
    __device__ static void acc_init(Acc&) {}
    __device__ static bool skip(const Params&) { return false; }
    __device__ static const S* init_ptr(const Params&) { return nullptr; }  // u_T = 0

    static constexpr int TMA_N = 3;  // staged: a, dh, h (rows shifted by one: h_{t-1})
    __host__ __device__ static constexpr int tma_shift(int k) { return k == 2 ? -1 : 0; }
    __host__ __device__ static constexpr int tma_extra(int) { return 0; }
    static void tma_arrays(const Params& p, const void** ptr) {
        ptr[0] = p.a;
        ptr[1] = p.dh;
        ptr[2] = p.h;
    }

    template <class Src>
    __device__ static void load(const Src& src, const Params& p, const Geom& g,
                                const TileCoord& tc, Regs& rg) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            if (tc.cok && t < g.T) {
                src.ld(rg.a[r], 0, p.a, t);
                src.ld(rg.g[r], 1, p.dh, t);
                if (t > 0) src.ld(rg.hp[r], 2, p.h, t - 1);
                else if (p.h0 != nullptr) rg.hp[r].load(p.h0 + tc.c);
                else rg.hp[r].ident(0.f);
            } else {
                rg.a[r].ident(1.f);
                rg.g[r].ident(0.f);
                rg.hp[r].ident(0.f);
            }
        }
    }
    __device__ static void aggregate(const Params&, const Geom&, const TileCoord&, const Regs& rg,
                                     Work&, float (&A)[VEC], float (&B)[VEC], bool) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; B[v] = 0.f; }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float av = rg.a[r].get(v);
                B[v] = av * (rg.g[r].get(v) + B[v]);
                A[v] *= av;
            }
    }
    __device__ static void finish(const Params& p, const Geom& g, const TileCoord& tc,
                                  const Regs& rg, Work&, float (&s)[VEC], Smem&, Acc&) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t t = tc.t0 - r;
            float dv[VEC], av[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float d = rg.g[r].get(v) + s[v];
                dv[v] = d;
                av[v] = d * rg.hp[r].get(v);
                s[v] = rg.a[r].get(v) * d;
            }
            if (tc.cok && t < g.T) {
                store_vec<S, VEC>(p.db + t * g.C + tc.c, dv);
                store_vec<S, VEC>(p.da + t * g.C + tc.c, av);
            }
        }
        // row 0 is the last row of the last row group of the last warp of time
        // chunk 0: s = u_0 = dh0
        if (tc.tchunk == 0 && (threadIdx.x >> 5) == NW - 1 && (RG == 1 || (threadIdx.x & 31) >= 32 - 32 / RG) &&
            p.dh0 != nullptr && tc.cok)
            store_vec<S, VEC>(p.dh0 + tc.c, s);
    }
    __device__ static void at_exit(const Params&, Smem&, Acc&) {}
};

template <typename S, bool VP, int M>
using FwdOpT = ScanFwdOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_SCAN_FWD, sizeof(S) == 2, M).NW,
                         kcfg(OP_SCAN_FWD, sizeof(S) == 2, M).R>;
template <typename S, bool VP, int M>
using BwdOpT = ScanBwdOp<S, kvec(sizeof(S) == 2, VP), kcfg(OP_SCAN_BWD, sizeof(S) == 2, M).NW,
                         kcfg(OP_SCAN_BWD, sizeof(S) == 2, M).R>;

// The cluster kernel's instantiations: a warp covers kcfg's R rows of 32
// channels, as V row groups of R / V rows (V channels per lane).
#ifndef LR_CLUSTER_VEC
#define LR_CLUSTER_VEC 2
#endif
constexpr int kClusterVec(bool vp) { return vp ? LR_CLUSTER_VEC : 1; }
template <typename S, bool VP>
using FwdOpK = ScanFwdOp<S, kClusterVec(VP), kcfg(OP_SCAN_FWD, sizeof(S) == 2, TILE_CLUSTER).NW,
                         kcfg(OP_SCAN_FWD, sizeof(S) == 2, TILE_CLUSTER).R / kClusterVec(VP), kClusterVec(VP)>;
template <typename S, bool VP>
using BwdOpK = ScanBwdOp<S, kClusterVec(VP), kcfg(OP_SCAN_BWD, sizeof(S) == 2, TILE_CLUSTER).NW,
                         kcfg(OP_SCAN_BWD, sizeof(S) == 2, TILE_CLUSTER).R / kClusterVec(VP), kClusterVec(VP)>;

template <typename S, bool VP>
static cudaError_t scan_fwd_t(const void* a, const void* b, const void* h0, void* h, const Geom& g,
                              const Carry& cr, cudaStream_t s) {
    return launch_persist<FwdOpT<S, VP, CARRY_CHAIN>, FwdOpT<S, VP, CARRY_WALK>,
                          FwdOpT<S, VP, TILE_TMA>, kcfg(OP_SCAN_FWD, sizeof(S) == 2, TILE_TMA).ST,
                          FwdOpK<S, VP>>(
        {(const S*)a, (const S*)b, (const S*)h0, (S*)h}, g, cr, s);
}

template <typename S, bool VP>
static cudaError_t scan_bwd_t(const void* a, const void* h, const void* h0, const void* dh,
                              void* da, void* db, void* dh0, const Geom& g, const Carry& cr,
                              cudaStream_t s) {
    return launch_persist<BwdOpT<S, VP, CARRY_CHAIN>, BwdOpT<S, VP, CARRY_WALK>,
                          BwdOpT<S, VP, TILE_TMA>, kcfg(OP_SCAN_BWD, sizeof(S) == 2, TILE_TMA).ST,
                          BwdOpK<S, VP>>(
        {(const S*)a, (const S*)h, (const S*)h0, (const S*)dh, (S*)da, (S*)db, (S*)dh0}, g, cr, s);
}

cudaError_t launch_scan_fwd(int dtype, bool vec, const void* a, const void* b, const void* h0,
                            void* h, const Geom& g, const Carry& cr, cudaStream_t s) {
    if (dtype == 0)
        return vec ? scan_fwd_t<float, true>(a, b, h0, h, g, cr, s)
                   : scan_fwd_t<float, false>(a, b, h0, h, g, cr, s);
    return vec ? scan_fwd_t<__nv_bfloat16, true>(a, b, h0, h, g, cr, s)
               : scan_fwd_t<__nv_bfloat16, false>(a, b, h0, h, g, cr, s);
}

cudaError_t launch_scan_bwd(int dtype, bool vec, const void* a, const void* h, const void* h0,
                            const void* dh, void* da, void* db, void* dh0, const Geom& g,
                            const Carry& cr, cudaStream_t s) {
    if (dtype == 0)
        return vec ? scan_bwd_t<float, true>(a, h, h0, dh, da, db, dh0, g, cr, s)
                   : scan_bwd_t<float, false>(a, h, h0, dh, da, db, dh0, g, cr, s);
    return vec ? scan_bwd_t<__nv_bfloat16, true>(a, h, h0, dh, da, db, dh0, g, cr, s)
               : scan_bwd_t<__nv_bfloat16, false>(a, h, h0, dh, da, db, dh0, g, cr, s);
}

}  // namespace lrs
