// lr_act.cuh -- the activations of the fused producers and epilogues: the
// logistic sigmoid (SRU gates, page [P1] "CUDA并行化RNN训练：从O(T)到O(log T)的
// 工程实践与参数调优", SRU paragraph; LSTM gates), tanh (SRU output and cell
// gradient; LSTM candidate and output; DEER's diagonal tanh RNN, page [P4],
// section "核心原理") and e^x - 1 (DEER's ODE form, page [P4], section
// "监控与调优").
//
// Both are written from their exponential forms,
//     sigmoid(z) = 1 / (1 + 2^{-z log2 e}),
//     tanh(x)    = 1 - 2 r,  r = 1 / (2^{2 x log2 e} + 1),
// and the derivative of tanh from the same r, 1 - tanh^2 = 4 r (1 - r), free of
// the cancellation of 1 - tanh^2 where tanh saturates;
// with the power of two and the reciprocal taken from the hardware's
// approximate instructions (ex2.approx, rcp.approx) in their flush-to-zero
// forms: one instruction each, with no extra steps for subnormal results,
// which none of these forms needs (a subnormal power of two or reciprocal only
// occurs where the result has saturated to 0 or 1 anyway).  That is a few
// instructions per activation, which matters here: these kernels stream 24-40
// bytes per element, and with two to five activations per element the DEER,
// SRU and LSTM kernels are bound by instruction issue.  Both forms saturate
// correctly (an infinite power gives a reciprocal of 0), keep NaN, and have an
// absolute error of a few 1e-7 on the whole line (no cancellation issue for
// the absolute error near 0), well inside the 1e-5 tolerance the results are
// checked against; lr_test_activations exposes them to the test that bounds
// their error against fp64.
#pragma once

#include <cuda_runtime.h>

namespace lrs {

// 2^x and 1/x, hardware approximations (relative error about 2^-22), with
// subnormal results flushed to zero.
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;       // log2(e)
constexpr float kTwoLog2e = 2.8853900817779268f;    // 2 log2(e)

__device__ __forceinline__ float act_sigmoid(float z) {
    return rcp_ftz(1.f + ex2_ftz(-kLog2e * z));
}

// tanh(x) keeps its sign for x < 0 (r > 1/2 there) and saturates to -1 (the
// power flushes to 0) and +1 (an infinite power gives r = 0).
__device__ __forceinline__ float act_tanh(float x) {
    return fmaf(-2.f, rcp_ftz(ex2_ftz(kTwoLog2e * x) + 1.f), 1.f);
}
// tanh(x), and in d its derivative 1 - tanh(x)^2.
__device__ __forceinline__ float act_tanh_d(float x, float& d) {
    const float r = rcp_ftz(ex2_ftz(kTwoLog2e * x) + 1.f);
    d = 4.f * fmaf(-r, r, r);
    return fmaf(-2.f, r, 1.f);
}
// tanh(x), and in q a quarter of its derivative, r (1 - r) with
// r = 1 / (e^{2x} + 1): a caller that scales the factor it multiplies the
// derivative by with 4 once (exact in fp32) saves a multiply per element and
// gets the same bits as 4 q times that factor.
__device__ __forceinline__ float act_tanh_q(float x, float& q) {
    const float r = rcp_ftz(ex2_ftz(kTwoLog2e * x) + 1.f);
    q = fmaf(-r, r, r);
    return fmaf(-2.f, r, 1.f);
}

// e^x - 1 without the cancellation of e^x - 1 near 0 (DEER's ODE form,
// exp(-G dt) and (1 - exp(-G dt)) / G): below |x| = 1/4 the Taylor series
// x (1 + x/2 (1 + x/3 (... (1 + x/8)))) -- its first omitted term, x^9/9!, is
// under 1e-11 |x| there -- and elsewhere e^x - 1 from the hardware
// exponential, where |e^x - 1| > 0.22 keeps the subtraction exact to a few
// ulp.  NaN stays NaN, -inf gives -1, +inf gives +inf.
__device__ __forceinline__ float act_expm1(float x) {
    if (fabsf(x) < 0.25f) {
        float p = fmaf(x, 0.125f, 1.f);
        p = fmaf(x * (1.f / 7.f), p, 1.f);
        p = fmaf(x * (1.f / 6.f), p, 1.f);
        p = fmaf(x * 0.2f, p, 1.f);
        p = fmaf(x * 0.25f, p, 1.f);
        p = fmaf(x * (1.f / 3.f), p, 1.f);
        p = fmaf(x * 0.5f, p, 1.f);
        return x * p;
    }
    return ex2_ftz(kLog2e * x) - 1.f;
}

}  // namespace lrs
