// gdn_common.cuh -- device helpers shared by the GDN kernels (loads, warp reductions).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// ---------------------------------------------------------------- activation element loads

template <typename T> struct Act;

// one(p), four(p): one element / four consecutive elements (4*sizeof(T)-byte aligned) as f32.
// raw1 / raw4 load the same elements as their stored bits and cvt1 / cvt4 widen them, so a
// load can be issued well before the value is needed.
template <> struct Act<float> {
    using R1 = float;
    using R4 = float4;
    __device__ __forceinline__ static R1 raw1(const float *p) { return *p; }
    __device__ __forceinline__ static R4 raw4(const float *p) {
        return *reinterpret_cast<const float4 *>(p);
    }
    __device__ __forceinline__ static float cvt1(R1 r) { return r; }
    __device__ __forceinline__ static float4 cvt4(R4 r) { return r; }
    __device__ __forceinline__ static float one(const float *p) { return *p; }
    __device__ __forceinline__ static float4 four(const float *p) { return raw4(p); }
};

template <> struct Act<__nv_bfloat16> {
    using R1 = __nv_bfloat16;
    using R4 = uint2;
    __device__ __forceinline__ static R1 raw1(const __nv_bfloat16 *p) { return *p; }
    __device__ __forceinline__ static R4 raw4(const __nv_bfloat16 *p) {
        return *reinterpret_cast<const uint2 *>(p);
    }
    __device__ __forceinline__ static float cvt1(R1 r) { return __bfloat162float(r); }
    __device__ __forceinline__ static float4 cvt4(R4 raw) {
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
        const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
        return make_float4(a.x, a.y, b.x, b.y);
    }
    __device__ __forceinline__ static float one(const __nv_bfloat16 *p) { return cvt1(*p); }
    __device__ __forceinline__ static float4 four(const __nv_bfloat16 *p) { return cvt4(raw4(p)); }
};

template <> struct Act<__half> {
    using R1 = __half;
    using R4 = uint2;
    __device__ __forceinline__ static R1 raw1(const __half *p) { return *p; }
    __device__ __forceinline__ static R4 raw4(const __half *p) {
        return *reinterpret_cast<const uint2 *>(p);
    }
    __device__ __forceinline__ static float cvt1(R1 r) { return __half2float(r); }
    __device__ __forceinline__ static float4 cvt4(R4 raw) {
        const __half2 lo = *reinterpret_cast<const __half2 *>(&raw.x);
        const __half2 hi = *reinterpret_cast<const __half2 *>(&raw.y);
        const float2 a = __half22float2(lo), b = __half22float2(hi);
        return make_float4(a.x, a.y, b.x, b.y);
    }
    __device__ __forceinline__ static float one(const __half *p) { return cvt1(*p); }
    __device__ __forceinline__ static float4 four(const __half *p) { return cvt4(raw4(p)); }
};

// Gate scalars (log_decay, beta) are either f32 or the activation dtype: a runtime switch
// on a warp-uniform value.
__device__ __forceinline__ float load_gate(const void *base, int dtype, int64_t i) {
    if (dtype == GDN_F32) return static_cast<const float *>(base)[i];
    if (dtype == GDN_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]);
    return __half2float(static_cast<const __half *>(base)[i]);
}

// ---------------------------------------------------------------------- warp reductions

// Sum over the `WIDTH` lanes of an aligned lane group (WIDTH a power of two <= 32).
template <int WIDTH>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    acc = fmaf(a.w, b.w, acc);
    return acc;
}

// silu(z) = z * sigmoid(z) = z / (1 + exp(-z)); exp overflow gives z / inf = -0 for z << 0.
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// The same with CUDA's fast exp and divide intrinsics (a few ulp; for z << 0 the quotient
// flushes to 0).  Used where many gates are computed per thread.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

}  // namespace gdn
