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
#include "lr_launch.h"

namespace lrs {

template <typename S, int VEC, int NW, int R>
__global__ void __launch_bounds__(NW * 32, 2)
    k_deer_iter(const float* __restrict__ w, const S* __restrict__ u, const S* __restrict__ h0,
                const S* __restrict__ yold, S* __restrict__ ynew, uint32_t* __restrict__ resid,
                Geom g, Lookback lb) {
    constexpr int L = NW * R, CW = 32 * VEC;
    __shared__ CarrySmem<VEC, NW> sm;
    __shared__ uint32_t s_max[NW];
    const uint32_t tile = take_ticket(lb, g);
    const int64_t q = tile / g.n_ct;
    const int j = tile % g.n_ct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ch = (int64_t)j * CW + lane * VEC;
    const bool cok = ch < g.C;
    const int64_t d = cok ? ch % g.D : 0;
    const int64_t t0 = q * L + warp * R;

    float wv[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) wv[v] = 0.f;
    if (cok) load_param<VEC>(w + d, wv);

    // previous iterate at rows t0-1 .. t0+R-1 (row -1 is h0)
    Pack<S, VEC> yo[R + 1];
#pragma unroll
    for (int i = 0; i <= R; ++i) {
        const int64_t t = t0 - 1 + i;
        if (!cok || t >= g.T) yo[i].ident(0.f);
        else if (t < 0) {
            if (h0 != nullptr) yo[i].load(h0 + ch);
            else yo[i].ident(0.f);
        } else if (yold != nullptr) yo[i].load(yold + t * g.C + ch);
        else yo[i].ident(0.f);
    }
    float J[R][VEC], Rh[R][VEC];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = t0 + r;
        if (cok && t < g.T) {
            Pack<S, VEC> pu;
            pu.load(u + t * g.C + ch);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float yt = yo[r].get(v);
                const float th = tanhf(wv[v] * yt + pu.get(v));
                const float jac = wv[v] * (1.f - th * th);
                J[r][v] = jac;
                Rh[r][v] = th - jac * yt;
            }
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) { J[r][v] = 1.f; Rh[r][v] = 0.f; }
        }
    }
    float A[VEC], Bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bs[v] = 0.f; }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Bs[v] = J[r][v] * Bs[v] + Rh[r][v];
            A[v] *= J[r][v];
        }
    float init[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) init[v] = 0.f;
    if (q == 0 && warp == 0 && h0 != nullptr && cok) load_vec<S, VEC>(h0 + ch, init);

    float s[VEC];
    tile_carry<VEC, NW>(sm, A, Bs, init, s, lb, q, j, g.n_ct);

    uint32_t mx = 0;  // max |y - yold| as bits: fp32 order of non-negative values, NaN on top
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t t = t0 + r;
#pragma unroll
        for (int v = 0; v < VEC; ++v) s[v] = J[r][v] * s[v] + Rh[r][v];
        if (cok && t < g.T) {
            store_vec<S, VEC>(ynew + t * g.C + ch, s);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                // the stored (rounded) value is the iterate the next step reads
                float yv = s[v];
                if constexpr (sizeof(S) == 2) yv = bf_lo(bf_bits(yv));
                const uint32_t bits = __float_as_uint(fabsf(yv - yo[r + 1].get(v)));
                mx = bits > mx ? bits : mx;
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, mx, off);
        mx = o > mx ? o : mx;
    }
    if (lane == 0) s_max[warp] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < NW; ++i) m = s_max[i] > m ? s_max[i] : m;
        if (m) atomicMax(resid, m);
    }
}

template <typename S, bool VP>
static cudaError_t deer_t(const float* w, const void* u, const void* h0, const void* yold,
                          void* ynew, uint32_t* resid, const Geom& g, const Lookback& lb,
                          cudaStream_t s) {
    constexpr int DT = sizeof(S) == 2 ? 1 : 0;
    constexpr KCfg k = kcfg(OP_DEER, DT);
    constexpr int VEC = kvec(DT, VP);
    k_deer_iter<S, VEC, k.NW, k.R><<<g.n_launch, 32 * k.NW, 0, s>>>(
        w, (const S*)u, (const S*)h0, (const S*)yold, (S*)ynew, resid, g, lb);
    return cudaGetLastError();
}

cudaError_t launch_deer_iter(int dtype, bool vec, const float* w, const void* u, const void* h0,
                             const void* yold, void* ynew, uint32_t* resid, const Geom& g,
                             const Lookback& lb, cudaStream_t s) {
    if (dtype == 0)
        return vec ? deer_t<float, true>(w, u, h0, yold, ynew, resid, g, lb, s)
                   : deer_t<float, false>(w, u, h0, yold, ynew, resid, g, lb, s);
    return vec ? deer_t<__nv_bfloat16, true>(w, u, h0, yold, ynew, resid, g, lb, s)
               : deer_t<__nv_bfloat16, false>(w, u, h0, yold, ynew, resid, g, lb, s);
}

}  // namespace lrs
