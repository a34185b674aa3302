// Fused epilogue shared by the GEMM kernels:
//     out = act(alpha * acc + bias[col]) + beta * c
// the bias-add / activation / residual fusion of the "Z-Turbo" tuning page
// (lanjinlin.com.cn), section 2.1 (activation first, residual after), with
// the tanh form of GELU printed there.  Everything is fp32:
//     v   = act(fmaf(alpha, acc, bias))     (alpha * acc without a bias)
//     out = v + (beta * c)                  (beta * c rounded first; c unread
//                                            when beta == 0)
// and the caller converts out to C's type once.  Without bias and
// activation the value is the plain GEMM's fmaf(alpha, acc, beta * c) (alpha
// * acc when beta == 0); with them, the beta term is rounded the same way
// (fmaf(1, v, beta * c) == v + (beta * c) rounded once), so the tensor-core
// kernels can run the activation first and then their plain store path with
// alpha = 1.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace gemm {

struct EpiParams {
    const void *bias;  // nullptr, or N values
    int bias_f32;      // 1: fp32 bias, 0: bf16 bias
    int act;           // GEMM_ACT_NONE / GEMM_ACT_RELU / GEMM_ACT_GELU_TANH
    int on;            // bias != nullptr || act != GEMM_ACT_NONE
};

__device__ __forceinline__ float epi_bias(const EpiParams &e, int col) {
    if (e.bias_f32) return __ldg(static_cast<const float *>(e.bias) + col);
    const uint16_t bits = __ldg(static_cast<const unsigned short *>(e.bias) + col);
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
}

// GELU, tanh form, through the identity 0.5 (1 + tanh(u)) = 1 / (1 + e^-2u):
//     gelu(x) = x / (1 + exp(-2u)),  u = sqrt(2/pi) (x + 0.044715 x^3)
// (no cancellation for negative x, and one exponential instead of a tanh).
// expf is CUDA's (2 ulp); __fdividef returns 0 once 1 + e^-2u passes 2^126,
// where the quotient is below any fp32 value of interest anyway.
__device__ __forceinline__ float gelu_tanh(float x) {
    const float u = 0.7978845608028654f * fmaf(0.044715f * x * x, x, x);
    return __fdividef(x, 1.f + expf(-2.f * u));
}

__device__ __forceinline__ float relu(float v) { return v > 0.f ? v : 0.f; }  // -0, NaN -> +0

__device__ __forceinline__ float epi_act(int act, float v) {
    if (act == 1) return relu(v);
    if (act == 2) return gelu_tanh(v);
    return v;
}

// v = act(alpha * acc + bias[col]), the part of the fused epilogue before
// the beta term.
__device__ __forceinline__ float epi_pre(const EpiParams &e, float alpha, float acc, int col) {
    const float v = e.bias ? fmaf(alpha, acc, epi_bias(e, col)) : alpha * acc;
    return epi_act(e.act, v);
}

// The whole epilogue for one element.  c is read by the caller only when
// beta != 0 (pass 0 otherwise).
__device__ __forceinline__ float epi_finish(const EpiParams &e, float alpha, float beta,
                                            float acc, int col, float c) {
    if (!e.on) return beta != 0.f ? fmaf(alpha, acc, beta * c) : alpha * acc;
    const float v = epi_pre(e, alpha, acc, col);
    return beta != 0.f ? __fadd_rn(v, __fmul_rn(beta, c)) : v;
}

}  // namespace gemm
