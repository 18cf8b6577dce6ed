// Element-wise epilogue shared by the tensor-core kernel, the CUDA-core
// SGEMM and the split-K reduction:
//     x = act(alpha * acc + beta * C + bias)
// with act the identity, GELU (tanh form or erf form) or ReLU, and the bias
// indexed by column or by row.
// applied once, after accumulation ("Skill: Write a Triton GEMM Kernel",
// Required reasoning process step 6 and Common failure modes on beta*C),
// then rounded once to the output type ("GEMM Kernel Optimization", Common
// Pitfalls).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace dg {

// GELU, tanh form (Hendrycks & Gimpel 2016):
//   gelu(x) = 0.5 x (1 + tanh(y)),  y = sqrt(2/pi) (x + 0.044715 x^3),
// with tanh(y) = 1 - 2 / (exp(2y) + 1), an identity that stays finite for
// every y (exp overflow gives tanh = 1, underflow gives -1).  exp and the
// division use the CUDA fast intrinsics; the absolute error of 1 + tanh(y)
// stays at the fp32 rounding level (~1e-7), so the relative error of the
// result is ~1e-7 wherever the result is not tiny.
__device__ __forceinline__ float gelu_tanh(float x) {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    const float k1 = 0.044715f;
    const float y = k0 * fmaf(k1 * x, x * x, x);
    const float e = __expf(2.0f * y);
    const float t = 1.0f - __fdividef(2.0f, e + 1.0f);
    return 0.5f * x * (1.0f + t);
}

// GELU itself (the same paper): gelu(x) = x Phi(x) = 0.5 x (1 + erf(x / sqrt(2))),
// with CUDA's erff.
__device__ __forceinline__ float gelu_erf(float x) {
    return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

// Rectifier: x for x > 0, else 0 (a NaN gives 0).
__device__ __forceinline__ float relu(float x) { return x > 0.0f ? x : 0.0f; }

__device__ __forceinline__ float apply_act(float x, int act) {
    if (act == ACT_GELU_TANH) return gelu_tanh(x);
    if (act == ACT_RELU) return relu(x);
    if (act == ACT_GELU_ERF) return gelu_erf(x);
    return x;
}

// The activation over NV values held in registers, the branch taken once.
template <int NV>
__device__ __forceinline__ void act_inplace(float* v, int act) {
    if (act == ACT_GELU_TANH) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = gelu_tanh(v[i]);
    } else if (act == ACT_RELU) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = relu(v[i]);
    } else if (act == ACT_GELU_ERF) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = gelu_erf(v[i]);
    }
}

__device__ __forceinline__ float load_elem(const void* p, int dt) {
    if (dt == DT_BF16) return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
    if (dt == DT_F16) return __half2float(*reinterpret_cast<const __half*>(p));
    return *reinterpret_cast<const float*>(p);
}

__device__ __forceinline__ void store_elem(void* p, int dt, float x) {
    if (dt == DT_BF16)
        *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
    else if (dt == DT_F16)
        *reinterpret_cast<__half*>(p) = __float2half_rn(x);
    else
        *reinterpret_cast<float*>(p) = x;
}

__device__ __forceinline__ int dt_size(int dt) { return dt == DT_F32 ? 4 : 2; }

// Element offset of C(b, i, j) from C.
__device__ __forceinline__ int64_t c_off(const Epilogue& e, int64_t b, int64_t i, int64_t j) {
    return b * e.stride_c + (e.c_row_major ? i * e.ldc + j : j * e.ldc + i);
}

// Address of C(b, i, j).
__device__ __forceinline__ char* c_addr(const Epilogue& e, int64_t b, int64_t i, int64_t j) {
    return reinterpret_cast<char*>(e.C) + c_off(e, b, i, j) * dt_size(e.c_dtype);
}

// Debug build: elements [off, off + n) of C lie inside the span the call may
// touch (always true in the product build).
__device__ __forceinline__ bool c_span_ok(const Epilogue& e, int64_t off, int64_t n = 1) {
#if DG_DEBUG
    return DG_CHECK(off >= 0 && off + n <= e.dbg_c_elems, e.dbg_status, STATUS_CHECK_BOUNDS);
#else
    (void)e, (void)off, (void)n;
    return true;
#endif
}

// Debug build: entry k of the bias exists.
__device__ __forceinline__ bool bias_ok(const Epilogue& e, int64_t k) {
#if DG_DEBUG
    return DG_CHECK(k >= 0 && k < e.dbg_bias_len, e.dbg_status, STATUS_CHECK_BOUNDS);
#else
    (void)e, (void)k;
    return true;
#endif
}

// Debug build, count-writes mode: one more write of the final value of
// C(b, i, j) (computed-problem coordinates; transposed back for swap-AB).
__device__ __forceinline__ void count_write(const Epilogue& e, int64_t b, int64_t i, int64_t j) {
#if DG_DEBUG
    if (e.dbg_counts) {
        const int64_t ci = e.dbg_swap ? j : i, cj = e.dbg_swap ? i : j;
        if (DG_CHECK(ci >= 0 && ci < e.dbg_m && cj >= 0 && cj < e.dbg_n, e.dbg_status,
                     STATUS_CHECK_BOUNDS))
            atomicAdd(e.dbg_counts + (b * e.dbg_m + ci) * e.dbg_n + cj, 1u);
    }
#else
    (void)e, (void)b, (void)i, (void)j;
#endif
}

// One element: acc is the fp32 accumulator value of C(b, i, j).
__device__ __forceinline__ void epilogue_store(const Epilogue& e, int64_t b, int64_t i, int64_t j,
                                               float acc) {
    if (!c_span_ok(e, c_off(e, b, i, j))) return;
    char* c = c_addr(e, b, i, j);
    float x = e.alpha * acc;
    if (e.beta != 0.0f) x = fmaf(e.beta, load_elem(c, e.c_dtype), x);
    if (e.bias && bias_ok(e, e.bias_on_rows ? i : j)) x += e.bias_on_rows ? e.bias[i] : e.bias[j];
    x = apply_act(x, e.act);
    store_elem(c, e.c_dtype, x);
    count_write(e, b, i, j);
}

// Four outputs C(b, i, j .. j + 3), j a multiple of 4: one vector access of C
// (16 bytes for fp32, 8 for 16-bit types) when C is row-major with 16-byte
// aligned rows and all four columns are inside N; otherwise one element at a
// time, skipping the columns at or past N.
__device__ __forceinline__ void epilogue_store4(const Epilogue& e, int64_t b, int64_t i,
                                                int64_t j, int64_t N, float4 acc) {
    float v[4] = {acc.x, acc.y, acc.z, acc.w};
    if (!(e.c_row_major && e.c_vec_ok && j + 3 < N)) {
        for (int c = 0; c < 4; ++c)
            if (j + c < N) epilogue_store(e, b, i, j + c, v[c]);
        return;
    }
    if (!c_span_ok(e, c_off(e, b, i, j), 4)) return;
    char* c = c_addr(e, b, i, j);
    if (!DG_CHECK(reinterpret_cast<uintptr_t>(c) % (4 * dt_size(e.c_dtype)) == 0, e.dbg_status,
                  STATUS_CHECK_ALIGN))
        return;
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] *= e.alpha;
    if (e.beta != 0.0f) {
        float o[4];
        if (e.c_dtype == DT_F32) {
            const float4 t = *reinterpret_cast<const float4*>(c);
            o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
        } else {
            const uint2 t = *reinterpret_cast<const uint2*>(c);
            const uint32_t w[2] = {t.x, t.y};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (e.c_dtype == DT_BF16) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
                    o[2 * k] = f.x; o[2 * k + 1] = f.y;
                } else {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
                    o[2 * k] = f.x; o[2 * k + 1] = f.y;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = fmaf(e.beta, o[k], v[k]);
    }
    if (e.bias && bias_ok(e, e.bias_on_rows ? i : j + 3)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] += e.bias_on_rows ? e.bias[i] : e.bias[j + k];
    }
    act_inplace<4>(v, e.act);
    if (e.c_dtype == DT_F32) {
        *reinterpret_cast<float4*>(c) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        uint32_t w[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (e.c_dtype == DT_BF16) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h);
            } else {
                const __half2 h = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }
        *reinterpret_cast<uint2*>(c) = make_uint2(w[0], w[1]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) count_write(e, b, i, j + k);
}

}  // namespace dg
