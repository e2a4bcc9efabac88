// lr_act.cuh -- the activations of the fused producers and epilogues: the
// logistic sigmoid (SRU gates, page [P1] "CUDA并行化RNN训练：从O(T)到O(log T)的
// 工程实践与参数调优", SRU paragraph) and tanh (SRU output and cell gradient;
// DEER's diagonal tanh RNN, page [P4], section "核心原理").
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

}  // namespace lrs
