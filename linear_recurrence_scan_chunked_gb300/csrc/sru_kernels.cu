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
//   dbf, dbr: per-tile channel sums -> [n_chunks, C] partials -> a fixed-order
//   reduction over chunks and batch (deterministic).
#include "lr_launch.h"

namespace lrs {

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + expf(-z)); }

template <typename S, int VEC, int NW, int R>
__global__ void __launch_bounds__(NW * 32, 2)
    k_sru_fwd(const S* __restrict__ xt, const S* __restrict__ uf, const S* __restrict__ ur,
              const S* __restrict__ x, const float* __restrict__ bf,
              const float* __restrict__ br, const S* __restrict__ c0, S* __restrict__ h,
              S* __restrict__ cst, Geom g, Lookback lb) {
    constexpr int L = NW * R, CW = 32 * VEC;
    __shared__ CarrySmem<VEC, NW> sm;
    const uint32_t tile = take_ticket(lb, g);
    const int64_t q = tile / g.n_ct;
    const int j = tile % g.n_ct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ch = (int64_t)j * CW + lane * VEC;
    const bool cok = ch < g.C;
    const int64_t d = cok ? ch % g.D : 0;
    const int64_t t0 = q * L + warp * R;

    float bfv[VEC], brv[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { bfv[v] = 0.f; brv[v] = 0.f; }
    if (cok) {
        load_param<VEC>(bf + d, bfv);
        load_param<VEC>(br + d, brv);
    }
    float fa[R][VEC], fb[R][VEC];  // scan element (f, (1-f) xt)
    Pack<S, VEC> pur[R], px[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = t0 + r;
        if (cok && t < g.T) {
            Pack<S, VEC> pxt, puf;
            pxt.load(xt + t * g.C + ch);
            puf.load(uf + t * g.C + ch);
            pur[r].load(ur + t * g.C + ch);
            px[r].load(x + t * g.C + ch);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float f = sigmoidf_(puf.get(v) + bfv[v]);
                fa[r][v] = f;
                fb[r][v] = (1.f - f) * pxt.get(v);
            }
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) { fa[r][v] = 1.f; fb[r][v] = 0.f; }
            pur[r].ident(0.f);
            px[r].ident(0.f);
        }
    }
    float A[VEC], Bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bs[v] = 0.f; }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Bs[v] = fa[r][v] * Bs[v] + fb[r][v];
            A[v] *= fa[r][v];
        }
    float init[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) init[v] = 0.f;
    if (q == 0 && warp == 0 && c0 != nullptr && cok) load_vec<S, VEC>(c0 + ch, init);

    float s[VEC];
    tile_carry<VEC, NW>(sm, A, Bs, init, s, lb, q, j, g.n_ct);

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = t0 + r;
        float hv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            s[v] = fa[r][v] * s[v] + fb[r][v];
            const float rg = sigmoidf_(pur[r].get(v) + brv[v]);
            hv[v] = rg * tanhf(s[v]) + (1.f - rg) * px[r].get(v);
        }
        if (cok && t < g.T) {
            store_vec<S, VEC>(cst + t * g.C + ch, s);
            store_vec<S, VEC>(h + t * g.C + ch, hv);
        }
    }
}

template <typename S, int VEC, int NW, int R>
__global__ void __launch_bounds__(NW * 32, 2)
    k_sru_bwd(const S* __restrict__ xt, const S* __restrict__ uf, const S* __restrict__ ur,
              const S* __restrict__ x, const float* __restrict__ bf,
              const float* __restrict__ br, const S* __restrict__ c0,
              const S* __restrict__ cst, const S* __restrict__ dh, S* __restrict__ dxt,
              S* __restrict__ duf, S* __restrict__ dur, S* __restrict__ dx,
              S* __restrict__ dc0, float* __restrict__ partials, Geom g, Lookback lb) {
    constexpr int L = NW * R, CW = 32 * VEC;
    __shared__ CarrySmem<VEC, NW> sm;
    const uint32_t tile = take_ticket(lb, g);
    const int64_t q = tile / g.n_ct;
    const int j = tile % g.n_ct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ch = (int64_t)j * CW + lane * VEC;
    const bool cok = ch < g.C;
    const int64_t d = cok ? ch % g.D : 0;
    const int64_t tchunk = g.n_chunks - 1 - q;
    const int64_t tb = tchunk * L + (L - 1) - warp * R;

    float bfv[VEC], brv[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { bfv[v] = 0.f; brv[v] = 0.f; }
    if (cok) {
        load_param<VEC>(bf + d, bfv);
        load_param<VEC>(br + d, brv);
    }
    float F[R][VEC], E[R][VEC], XT[R][VEC], CP[R][VEC];
    float sum_r[VEC], sum_f[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { sum_r[v] = 0.f; sum_f[v] = 0.f; }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = tb - r;
        if (cok && t < g.T) {
            Pack<S, VEC> pxt, puf, pur, px, pc, pcp, pdh;
            const int64_t o = t * g.C + ch;
            pxt.load(xt + o);
            puf.load(uf + o);
            pur.load(ur + o);
            px.load(x + o);
            pc.load(cst + o);
            pdh.load(dh + o);
            if (t > 0) pcp.load(cst + o - g.C);
            else if (c0 != nullptr) pcp.load(c0 + ch);
            else pcp.ident(0.f);
            float durv[VEC], dxv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float f = sigmoidf_(puf.get(v) + bfv[v]);
                const float rg = sigmoidf_(pur.get(v) + brv[v]);
                const float th = tanhf(pc.get(v));
                const float g_ = pdh.get(v);
                durv[v] = g_ * (th - px.get(v)) * rg * (1.f - rg);
                dxv[v] = g_ * (1.f - rg);
                sum_r[v] += durv[v];
                F[r][v] = f;
                E[r][v] = g_ * rg * (1.f - th * th);
                XT[r][v] = pxt.get(v);
                CP[r][v] = pcp.get(v);
            }
            store_vec<S, VEC>(dur + o, durv);
            store_vec<S, VEC>(dx + o, dxv);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) { F[r][v] = 1.f; E[r][v] = 0.f; XT[r][v] = 0.f; CP[r][v] = 0.f; }
        }
    }
    float A[VEC], Bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bs[v] = 0.f; }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Bs[v] = F[r][v] * (E[r][v] + Bs[v]);
            A[v] *= F[r][v];
        }
    float init[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) init[v] = 0.f;

    float s[VEC];
    tile_carry<VEC, NW>(sm, A, Bs, init, s, lb, q, j, g.n_ct);

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = tb - r;
        const bool ok = cok && t < g.T;
        float dxtv[VEC], dufv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const float dc = E[r][v] + s[v];
            const float f = F[r][v];
            dxtv[v] = dc * (1.f - f);
            dufv[v] = dc * (CP[r][v] - XT[r][v]) * f * (1.f - f);
            s[v] = f * dc;
            if (ok) sum_f[v] += dufv[v];
        }
        if (ok) {
            store_vec<S, VEC>(dxt + t * g.C + ch, dxtv);
            store_vec<S, VEC>(duf + t * g.C + ch, dufv);
        }
    }
    if (tchunk == 0 && warp == NW - 1 && dc0 != nullptr && cok) store_vec<S, VEC>(dc0 + ch, s);

    // bias-gradient partials of this tile: sum over its rows, fixed warp order
    __syncthreads();  // the carry smem is free again
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        sm.a[warp][lane][v] = sum_f[v];
        sm.b[warp][lane][v] = sum_r[v];
    }
    __syncthreads();
    if (warp == 0 && cok) {
        float pf[VEC], pr[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { pf[v] = 0.f; pr[v] = 0.f; }
#pragma unroll
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int v = 0; v < VEC; ++v) { pf[v] += sm.a[w][lane][v]; pr[v] += sm.b[w][lane][v]; }
        float* pfp = partials + tchunk * g.C + ch;
        float* prp = partials + (g.n_chunks + tchunk) * g.C + ch;
#pragma unroll
        for (int v = 0; v < VEC; ++v) { pfp[v] = pf[v]; prp[v] = pr[v]; }
    }
}

// dbf[d] = sum_k sum_b partials_f[k][b*D + d] (likewise dbr), in a fixed order:
// a block owns 32 consecutive features; its 8 warps each sum a fixed slice of
// the (chunk, batch) pairs; the slices are added in warp order.
__global__ void __launch_bounds__(256)
    k_bias_reduce(const float* __restrict__ partials, int64_t n_chunks, int64_t B, int64_t D,
                  float* __restrict__ dbf, float* __restrict__ dbr) {
    __shared__ float sf[8][32], sr[8][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t d = (int64_t)blockIdx.x * 32 + lane;
    const int64_t C = B * D, n = n_chunks * B;
    const int64_t per = (n + 7) / 8, lo = warp * per, hi = lo + per < n ? lo + per : n;
    float af = 0.f, ar = 0.f;
    if (d < D)
        for (int64_t i = lo; i < hi; ++i) {
            const int64_t k = i / B, b = i % B;
            af += partials[k * C + b * D + d];
            ar += partials[(n_chunks + k) * C + b * D + d];
        }
    sf[warp][lane] = af;
    sr[warp][lane] = ar;
    __syncthreads();
    if (warp == 0 && d < D) {
        float tf = 0.f, tr = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) { tf += sf[w][lane]; tr += sr[w][lane]; }
        dbf[d] = tf;
        dbr[d] = tr;
    }
}

template <typename S, bool VP>
static cudaError_t sru_fwd_t(const void* xt, const void* uf, const void* ur, const void* x,
                             const float* bf, const float* br, const void* c0, void* h, void* c,
                             const Geom& g, const Lookback& lb, cudaStream_t s) {
    constexpr int DT = sizeof(S) == 2 ? 1 : 0;
    constexpr KCfg k = kcfg(OP_SRU_FWD, DT);
    constexpr int VEC = kvec(DT, VP);
    k_sru_fwd<S, VEC, k.NW, k.R><<<g.n_launch, 32 * k.NW, 0, s>>>(
        (const S*)xt, (const S*)uf, (const S*)ur, (const S*)x, bf, br, (const S*)c0, (S*)h,
        (S*)c, g, lb);
    return cudaGetLastError();
}

template <typename S, bool VP>
static cudaError_t sru_bwd_t(const void* xt, const void* uf, const void* ur, const void* x,
                             const float* bf, const float* br, const void* c0, const void* c,
                             const void* dh, void* dxt, void* duf, void* dur, void* dx, void* dc0,
                             float* partials, const Geom& g, const Lookback& lb, cudaStream_t s) {
    constexpr int DT = sizeof(S) == 2 ? 1 : 0;
    constexpr KCfg k = kcfg(OP_SRU_BWD, DT);
    constexpr int VEC = kvec(DT, VP);
    k_sru_bwd<S, VEC, k.NW, k.R><<<g.n_launch, 32 * k.NW, 0, s>>>(
        (const S*)xt, (const S*)uf, (const S*)ur, (const S*)x, bf, br, (const S*)c0,
        (const S*)c, (const S*)dh, (S*)dxt, (S*)duf, (S*)dur, (S*)dx, (S*)dc0, partials, g, lb);
    return cudaGetLastError();
}

cudaError_t launch_sru_fwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           void* h, void* c, const Geom& g, const Lookback& lb, cudaStream_t s) {
    if (dtype == 0)
        return vec ? sru_fwd_t<float, true>(xt, uf, ur, x, bf, br, c0, h, c, g, lb, s)
                   : sru_fwd_t<float, false>(xt, uf, ur, x, bf, br, c0, h, c, g, lb, s);
    return vec ? sru_fwd_t<__nv_bfloat16, true>(xt, uf, ur, x, bf, br, c0, h, c, g, lb, s)
               : sru_fwd_t<__nv_bfloat16, false>(xt, uf, ur, x, bf, br, c0, h, c, g, lb, s);
}

cudaError_t launch_sru_bwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           const void* c, const void* dh, void* dxt, void* duf, void* dur,
                           void* dx, void* dc0, float* partials, const Geom& g,
                           const Lookback& lb, cudaStream_t s) {
    if (dtype == 0)
        return vec ? sru_bwd_t<float, true>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur, dx,
                                            dc0, partials, g, lb, s)
                   : sru_bwd_t<float, false>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur, dx,
                                             dc0, partials, g, lb, s);
    return vec ? sru_bwd_t<__nv_bfloat16, true>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur,
                                                dx, dc0, partials, g, lb, s)
               : sru_bwd_t<__nv_bfloat16, false>(xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur,
                                                 dx, dc0, partials, g, lb, s);
}

cudaError_t launch_bias_reduce(const float* partials, int64_t n_chunks, int64_t B, int64_t D,
                               float* dbf, float* dbr, cudaStream_t s) {
    const unsigned blocks = (unsigned)((D + 31) / 32);
    k_bias_reduce<<<blocks, 256, 0, s>>>(partials, n_chunks, B, D, dbf, dbr);
    return cudaGetLastError();
}

}  // namespace lrs
