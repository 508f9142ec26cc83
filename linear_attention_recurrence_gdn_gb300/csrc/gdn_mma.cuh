// gdn_mma.cuh -- warp-level tensor-core helpers shared by the scan kernels: mma.sync
// m16n8k16 bf16 (f32 accumulate), ldmatrix, bf16 hi / lo operand splits, named barriers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_tma.cuh"

namespace gdn {

// Named barrier `id` over `count` threads (a multiple of 32); bar.arrive does not wait.
__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Every thread of every CTA in the cluster meets here (hardware cluster barrier).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// v -> the same shared-memory location in the cluster's CTA `rank` (distributed shared
// memory), counted as 4 bytes on that CTA's mbarrier `bar` (the local address of it).
__device__ __forceinline__ void st_async_peer(const float *dst, float v, const uint64_t *bar,
                                              int rank) {
    uint32_t rd, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rd) : "r"(smem_u32(dst)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(rd),
                 "f"(v), "r"(rb)
                 : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (hi + lo) . b for an exact bf16 B operand
__device__ __forceinline__ void mma2(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     uint32_t b0, uint32_t b1) {
    mma16816(d, al, b0, b1);
    mma16816(d, ah, b0, b1);
}

// hi.hi + hi.lo + lo.hi
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    mma16816(d, al, bh0, bh1);
    mma16816(d, ah, bl0, bl1);
    mma16816(d, ah, bh0, bh1);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(addr)));
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void *addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(smem_u32(addr)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(addr)));
}

// (x, y) -> bf16x2 hi part and the bf16x2 of the remainders; x in the low half.
__device__ __forceinline__ void split2(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ void split1(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// Eight bf16 (a 16-byte piece) to f32; bf16 -> f32 is a 16-bit shift.
__device__ __forceinline__ void unpack8(const uint4 w, float (&x)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// Squares of a 16-byte piece of raw k or q into ss; for non-bf16 types also its bf16 hi / lo
// parts, written to hi / lo (8 or 4 elements).
template <typename TA> struct Piece;
template <> struct Piece<__nv_bfloat16> {
    __device__ __forceinline__ static void sq(const __nv_bfloat16 *src, float &ss) {
        float x[8];
        unpack8(*reinterpret_cast<const uint4 *>(src), x);
#pragma unroll
        for (int i = 0; i < 8; i++) ss = fmaf(x[i], x[i], ss);
    }
};
template <> struct Piece<__half> {
    static constexpr int E = 8;
    __device__ __forceinline__ static void split(const __half *src, __nv_bfloat16 *hi,
                                                 __nv_bfloat16 *lo, float &ss) {
        const uint4 w = *reinterpret_cast<const uint4 *>(src);
        const __half2 *h = reinterpret_cast<const __half2 *>(&w);
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 f = __half22float2(h[i]);
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
            split2(f.x, f.y, ph[i], pl[i]);
        }
        *reinterpret_cast<uint4 *>(hi) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        *reinterpret_cast<uint4 *>(lo) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
    }
};
template <> struct Piece<float> {
    static constexpr int E = 4;
    __device__ __forceinline__ static void split(const float *src, __nv_bfloat16 *hi,
                                                 __nv_bfloat16 *lo, float &ss) {
        const float4 f = *reinterpret_cast<const float4 *>(src);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
        ss = fmaf(f.z, f.z, ss);
        ss = fmaf(f.w, f.w, ss);
        uint32_t ph[2], pl[2];
        split2(f.x, f.y, ph[0], pl[0]);
        split2(f.z, f.w, ph[1], pl[1]);
        *reinterpret_cast<uint2 *>(hi) = make_uint2(ph[0], ph[1]);
        *reinterpret_cast<uint2 *>(lo) = make_uint2(pl[0], pl[1]);
    }
};

}  // namespace gdn
