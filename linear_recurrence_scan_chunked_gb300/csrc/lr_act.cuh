// lr_act.cuh -- the activations of the fused producers and epilogues: the
// logistic sigmoid (SRU gates, page [P1] "CUDA并行化RNN训练：从O(T)到O(log T)的
// 工程实践与参数调优", SRU paragraph; LSTM gates), tanh (SRU output and cell
// gradient; LSTM candidate and output; DEER's diagonal tanh RNN, page [P4],
// section "核心原理") and e^x - 1 (DEER's ODE form, page [P4], section
// "监控与调优").
//
// Both are written from their exponential forms,
//     sigmoid(z) = 1 / (1 + e^{-z}),
//     tanh(x)    = sign(x) (1 - 2 / (e^{2|x|} + 1)),
// with the exponential and the quotient taken from the hardware-approximate
// intrinsics __expf and __fdividef.  That is about a third of the instruction
// count of expf / tanhf with an IEEE division, which matters here: these
// kernels stream 24-40 bytes per element, and three activations per element
// with the accurate routines made the SRU kernels issue-bound.  Both forms
// saturate correctly (an infinite exponential gives a quotient of 0), keep NaN,
// and have an absolute error of a few 1e-7 on the whole line (no cancellation
// issue for the absolute error near 0), well inside the 1e-5 tolerance the
// results are checked against; lr_test_activations exposes them to the test
// that bounds their error against fp64.
#pragma once

#include <cuda_runtime.h>

namespace lrs {

__device__ __forceinline__ float act_sigmoid(float z) {
    return __fdividef(1.f, 1.f + __expf(-z));
}

__device__ __forceinline__ float act_tanh(float x) {
    const float t = 1.f - __fdividef(2.f, __expf(2.f * fabsf(x)) + 1.f);
    return copysignf(t, x);
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
    return __expf(x) - 1.f;
}

}  // namespace lrs
