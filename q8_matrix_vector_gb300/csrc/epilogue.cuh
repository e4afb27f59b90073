// Fused epilogue: an elementwise statement applied to each output as it is
// written ("dot and tensor cores" page, "The fused epilogue"), instead of
// storing the product and sweeping it again.  For output (m, n) with product x:
//
//     y = alpha * x + beta * C[m, n] (old value, read only if beta != 0) + bias[n]
//     y = act(y)          none, relu, silu = y / (1 + exp(-y)), or the tanh
//                         form of gelu, 0.5 y (1 + tanh(sqrt(2/pi) (y + 0.044715 y^3)))
//     C[m, n] = y + residual[m, n]
//
// f32 throughout; expf and tanhf are CUDA's accurate library functions.  Each
// output is written by exactly one thread, which also reads its old value.
#pragma once

#include <cstdint>

namespace q8epi {

enum : int { kActNone = 0, kActRelu = 1, kActSilu = 2, kActGeluTanh = 3 };

struct Epilogue {
    const float *bias = nullptr;      // [N] or null
    const float *residual = nullptr;  // [M, N] or null
    float alpha = 1.0f;
    float beta = 0.0f;
    int act = kActNone;
    int on = 0;                       // 0: C = x, nothing else is read
};

__device__ __forceinline__ float activate(float y, int act) {
    if (act == kActRelu) return y > 0.0f ? y : 0.0f;
    if (act == kActSilu) return y / (1.0f + expf(-y));
    if (act == kActGeluTanh) {
        const float u = 0.7978845608028654f * (y + 0.044715f * y * y * y);
        return 0.5f * y * (1.0f + tanhf(u));
    }
    return y;
}

// The value to store at C[idx] (idx = m * N + n) for product x.
__device__ __forceinline__ float apply(const Epilogue &e, float x, const float *c, int64_t idx, int64_t n) {
    if (!e.on) return x;
    float y = e.alpha * x;
    if (e.beta != 0.0f) y = fmaf(e.beta, c[idx], y);
    if (e.bias != nullptr) y += __ldg(e.bias + n);
    y = activate(y, e.act);
    if (e.residual != nullptr) y += __ldg(e.residual + idx);
    return y;
}

// The inputs the statement reads for output (idx, n), copied ahead of the
// product into this thread's three shared-memory slots q[0..2] (old C, bias,
// residual) with cp.async, so that their latency hides under the weight stream
// and no register holds them meanwhile.  After cp.async.wait_all, apply_pre
// gives exactly what apply gives.  All pointers 4-byte aligned.
__device__ __forceinline__ void cp_async_f32(float *dst, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

__device__ __forceinline__ void preload_async(const Epilogue &e, const float *c, int64_t idx, int64_t n, float *q) {
    if (e.beta != 0.0f) cp_async_f32(q + 0, c + idx);
    if (e.bias != nullptr) cp_async_f32(q + 1, e.bias + n);
    if (e.residual != nullptr) cp_async_f32(q + 2, e.residual + idx);
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ float apply_pre(const Epilogue &e, float x, const float *q) {
    if (!e.on) return x;
    asm volatile("cp.async.wait_all;" ::: "memory");
    float y = e.alpha * x;
    if (e.beta != 0.0f) y = fmaf(e.beta, q[0], y);
    if (e.bias != nullptr) y += q[1];
    y = activate(y, e.act);
    if (e.residual != nullptr) y += q[2];
    return y;
}

}  // namespace q8epi
