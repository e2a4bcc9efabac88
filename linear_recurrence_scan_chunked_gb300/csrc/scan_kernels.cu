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
// written once: the tile is held in registers between the local scan and the
// output pass while the look-back resolves the carry.
#include "lr_launch.h"

namespace lrs {

template <typename S, int VEC, int NW, int R>
__global__ void __launch_bounds__(NW * 32, 2)
    k_scan_fwd(const S* __restrict__ a, const S* __restrict__ b, const S* __restrict__ h0,
               S* __restrict__ h, Geom g, Lookback lb) {
    constexpr int L = NW * R, CW = 32 * VEC;
    __shared__ CarrySmem<VEC, NW> sm;
    const uint32_t tile = take_ticket(lb, g);
    const int64_t q = tile / g.n_ct;
    const int j = tile % g.n_ct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = (int64_t)j * CW + lane * VEC;
    const bool cok = c < g.C;
    const int64_t t0 = q * L + warp * R;

    Pack<S, VEC> pa[R], pb[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = t0 + r;
        if (cok && t < g.T) {
            pa[r].load(a + t * g.C + c);
            pb[r].load(b + t * g.C + c);
        } else {  // identity element (1, 0) outside the problem
            pa[r].ident(1.f);
            pb[r].ident(0.f);
        }
    }
    float A[VEC], Bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bs[v] = 0.f; }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const float av = pa[r].get(v);
            Bs[v] = av * Bs[v] + pb[r].get(v);
            A[v] *= av;
        }
    float init[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) init[v] = 0.f;
    if (q == 0 && warp == 0 && h0 != nullptr && cok) load_vec<S, VEC>(h0 + c, init);

    float s[VEC];
    tile_carry<VEC, NW>(sm, A, Bs, init, s, lb, q, j, g.n_ct);

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = t0 + r;
#pragma unroll
        for (int v = 0; v < VEC; ++v) s[v] = pa[r].get(v) * s[v] + pb[r].get(v);
        if (cok && t < g.T) store_vec<S, VEC>(h + t * g.C + c, s);
    }
}

template <typename S, int VEC, int NW, int R>
__global__ void __launch_bounds__(NW * 32, 2)
    k_scan_bwd(const S* __restrict__ a, const S* __restrict__ h, const S* __restrict__ h0,
               const S* __restrict__ dh, S* __restrict__ da, S* __restrict__ db,
               S* __restrict__ dh0, Geom g, Lookback lb) {
    constexpr int L = NW * R, CW = 32 * VEC;
    __shared__ CarrySmem<VEC, NW> sm;
    const uint32_t tile = take_ticket(lb, g);
    const int64_t q = tile / g.n_ct;  // scan order: q = 0 is the last time chunk
    const int j = tile % g.n_ct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = (int64_t)j * CW + lane * VEC;
    const bool cok = c < g.C;
    const int64_t tchunk = g.n_chunks - 1 - q;
    const int64_t tb = tchunk * L + (L - 1) - warp * R;  // time of this thread's first row

    Pack<S, VEC> pa[R], pg[R], ph[R];  // a_t, dh_t, h_{t-1}
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = tb - r;
        if (cok && t < g.T) {
            pa[r].load(a + t * g.C + c);
            pg[r].load(dh + t * g.C + c);
            if (t > 0) ph[r].load(h + (t - 1) * g.C + c);
            else if (h0 != nullptr) ph[r].load(h0 + c);
            else ph[r].ident(0.f);
        } else {
            pa[r].ident(1.f);
            pg[r].ident(0.f);
            ph[r].ident(0.f);
        }
    }
    float A[VEC], Bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bs[v] = 0.f; }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const float av = pa[r].get(v);
            Bs[v] = av * (pg[r].get(v) + Bs[v]);
            A[v] *= av;
        }
    float init[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) init[v] = 0.f;  // u_T = 0

    float s[VEC];
    tile_carry<VEC, NW>(sm, A, Bs, init, s, lb, q, j, g.n_ct);

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = tb - r;
        float dv[VEC], av[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const float d = pg[r].get(v) + s[v];
            dv[v] = d;
            av[v] = d * ph[r].get(v);
            s[v] = pa[r].get(v) * d;
        }
        if (cok && t < g.T) {
            store_vec<S, VEC>(db + t * g.C + c, dv);
            store_vec<S, VEC>(da + t * g.C + c, av);
        }
    }
    // row 0 is the last row of the last warp of time chunk 0: s = u_0 = dh0
    if (tchunk == 0 && warp == NW - 1 && dh0 != nullptr && cok) store_vec<S, VEC>(dh0 + c, s);
}

template <typename S, bool VP>
static cudaError_t scan_fwd_t(const void* a, const void* b, const void* h0, void* h,
                              const Geom& g, const Lookback& lb, cudaStream_t s) {
    constexpr int DT = sizeof(S) == 2 ? 1 : 0;
    constexpr KCfg k = kcfg(OP_SCAN_FWD, DT);
    constexpr int VEC = kvec(DT, VP);
    k_scan_fwd<S, VEC, k.NW, k.R><<<g.n_launch, 32 * k.NW, 0, s>>>(
        (const S*)a, (const S*)b, (const S*)h0, (S*)h, g, lb);
    return cudaGetLastError();
}

template <typename S, bool VP>
static cudaError_t scan_bwd_t(const void* a, const void* h, const void* h0, const void* dh,
                              void* da, void* db, void* dh0, const Geom& g, const Lookback& lb,
                              cudaStream_t s) {
    constexpr int DT = sizeof(S) == 2 ? 1 : 0;
    constexpr KCfg k = kcfg(OP_SCAN_BWD, DT);
    constexpr int VEC = kvec(DT, VP);
    k_scan_bwd<S, VEC, k.NW, k.R><<<g.n_launch, 32 * k.NW, 0, s>>>(
        (const S*)a, (const S*)h, (const S*)h0, (const S*)dh, (S*)da, (S*)db, (S*)dh0, g, lb);
    return cudaGetLastError();
}

cudaError_t launch_scan_fwd(int dtype, bool vec, const void* a, const void* b, const void* h0,
                            void* h, const Geom& g, const Lookback& lb, cudaStream_t s) {
    if (dtype == 0)
        return vec ? scan_fwd_t<float, true>(a, b, h0, h, g, lb, s)
                   : scan_fwd_t<float, false>(a, b, h0, h, g, lb, s);
    return vec ? scan_fwd_t<__nv_bfloat16, true>(a, b, h0, h, g, lb, s)
               : scan_fwd_t<__nv_bfloat16, false>(a, b, h0, h, g, lb, s);
}

cudaError_t launch_scan_bwd(int dtype, bool vec, const void* a, const void* h, const void* h0,
                            const void* dh, void* da, void* db, void* dh0, const Geom& g,
                            const Lookback& lb, cudaStream_t s) {
    if (dtype == 0)
        return vec ? scan_bwd_t<float, true>(a, h, h0, dh, da, db, dh0, g, lb, s)
                   : scan_bwd_t<float, false>(a, h, h0, dh, da, db, dh0, g, lb, s);
    return vec ? scan_bwd_t<__nv_bfloat16, true>(a, h, h0, dh, da, db, dh0, g, lb, s)
               : scan_bwd_t<__nv_bfloat16, false>(a, h, h0, dh, da, db, dh0, g, lb, s);
}

}  // namespace lrs
