// gdn_general.cu -- the recurrence for head dims the tiled kernels do not take (Dk or Dv not a
// multiple of 16 up to 128, nor 256): any Dk, Dv from 1 to 256 whose memory fits in shared
// memory.  Pruned nested-prefix widths (modelopt puzzletron.pruning.gated_delta_net,
// slice_gated_delta_net_state_dict and GDNShape: separate key and value dims) can be any size.
//
// What is computed is the page's per-token step (logicaffeine_compile::codegen_cuda::gdn, module
// description, with the fusion of "The fusion": one pass over a row gives S k^ and S q^):
//     u = S k^,  w = S q^,  coef = beta (v - alpha u),  S <- alpha S + coef k^^T,
//     o = alpha w + coef (k^ . q^),  y = rmsnorm(o * silu(z)) * gn   (or y = o without z).
// One CTA per (b, hv) head keeps the head's f32 memory in shared memory for the whole sequence
// (rows padded to an odd stride, so the row threads' column walks hit distinct banks); thread a
// owns memory row a.  Per token the k, q rows are staged and normalised with one block
// reduction, the rows are updated in place, and the gated RMSNorm reduces over the head's rows.
// A decode step is the same kernel with S = 1.  Plain loads and stores throughout: the operands
// may sit at any element offset (pinned host memory under GDN_FLAG_HOST_IO included).
#include <math.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kGenThreads = 256;          // >= the largest Dv
constexpr int kGenWarps = kGenThreads / 32;
constexpr float kGenMinLogDecay = -80.0f; // exp(-80) ~ 1.8e-35: a full reset in f32

// Row stride of the memory in shared memory: Dk rounded up to odd.
__host__ __device__ constexpr int gen_ld(int dk) { return dk | 1; }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// Sums of a, b, c over the whole CTA (every thread gets them); `red` holds 3 x kGenWarps floats.
__device__ __forceinline__ void block_sum3(float &a, float &b, float &c, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
        c += __shfl_xor_sync(0xffffffffu, c, off);
    }
    __syncthreads();                                       // red free (previous use read)
    if (lane == 0) {
        red[warp] = a;
        red[kGenWarps + warp] = b;
        red[2 * kGenWarps + warp] = c;
    }
    __syncthreads();
    a = b = c = 0.f;
#pragma unroll
    for (int i = 0; i < kGenWarps; i++) {
        a += red[i];
        b += red[kGenWarps + i];
        c += red[2 * kGenWarps + i];
    }
}

template <typename TA>
__global__ void __launch_bounds__(kGenThreads, 1) gdn_general_kernel(const gdn_params p, bool decode) {
    extern __shared__ float gsm[];
    const int Dk = p.Dk, Dv = p.Dv, S = p.S, ld = gen_ld(Dk);
    float *Sm = gsm;                                       // [Dv][ld]
    float *kh = Sm + Dv * ld;                              // [Dk]
    float *qh = kh + Dk;                                   // [Dk]
    float *red = qh + Dk;                                  // [3][kGenWarps]
    const int64_t head = blockIdx.x;                       // b * Hv + hv
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int tid = threadIdx.x;
    const int64_t mem = static_cast<int64_t>(Dv) * Dk;

    // the memory: a decode step updates `state` in place; a scan starts from s0 (or zeros)
    const float *from = decode ? p.state : p.s0;
    for (int64_t i = tid; i < mem; i += kGenThreads) {
        const int r = static_cast<int>(i / Dk), c = static_cast<int>(i - static_cast<int64_t>(r) * Dk);
        Sm[r * ld + c] = from ? from[head * mem + i] : 0.f;
    }
    const TA *q = static_cast<const TA *>(p.q), *k = static_cast<const TA *>(p.k);
    const TA *v = static_cast<const TA *>(p.v), *z = static_cast<const TA *>(p.z);
    const bool gated = z != nullptr;
    const float gna = (gated && tid < Dv) ? p.gn[tid] : 0.f;
    const float qscale = rsqrtf(static_cast<float>(Dk));
    float *row = Sm + tid * ld;

    for (int t = 0; t < S; t++) {
        const int64_t kq_off = p.head_major
            ? ((static_cast<int64_t>(b) * p.Hk + hk) * S + t) * Dk
            : ((static_cast<int64_t>(b) * S + t) * p.Hk + hk) * Dk;
        const int64_t v_off = p.head_major
            ? ((static_cast<int64_t>(b) * p.Hv + hv) * S + t) * Dv
            : ((static_cast<int64_t>(b) * S + t) * p.Hv + hv) * Dv;
        const int64_t g_off = p.head_major ? (static_cast<int64_t>(b) * p.Hv + hv) * S + t
                                           : (static_cast<int64_t>(b) * S + t) * p.Hv + hv;
        // k, q rows and their sums of squares and dot product
        float skk = 0.f, sqq = 0.f, skq = 0.f;
        for (int j = tid; j < Dk; j += kGenThreads) {
            const float kj = to_f32(k[kq_off + j]), qj = to_f32(q[kq_off + j]);
            kh[j] = kj;
            qh[j] = qj;
            skk = fmaf(kj, kj, skk);
            sqq = fmaf(qj, qj, sqq);
            skq = fmaf(kj, qj, skq);
        }
        const float alpha = expf(fmaxf(load_gate(p.log_decay, p.gate_dtype, g_off), kGenMinLogDecay));
        const float beta = load_gate(p.beta, p.gate_dtype, g_off);
        const float va = tid < Dv ? to_f32(v[v_off + tid]) : 0.f;
        const float za = (gated && tid < Dv) ? to_f32(z[v_off + tid]) : 0.f;
        block_sum3(skk, sqq, skq, red);                    // also orders the kh, qh writes
        const float rk = rsqrtf(skk + p.qk_eps);
        const float rq = rsqrtf(sqq + p.qk_eps) * qscale;
        // row a: u, w against the raw rows, then the update with k^ = rk k
        float o = 0.f;
        if (tid < Dv) {
            float u = 0.f, w = 0.f;
            for (int j = 0; j < Dk; j++) {
                const float s = row[j];
                u = fmaf(s, kh[j], u);
                w = fmaf(s, qh[j], w);
            }
            u *= rk;
            w *= rq;
            const float coef = beta * (va - alpha * u);
            const float ck = coef * rk;
            for (int j = 0; j < Dk; j++) row[j] = fmaf(alpha, row[j], ck * kh[j]);
            o = fmaf(alpha, w, coef * (skq * rk * rq));
        }
        float ya = o;
        if (gated) {
            const float g = tid < Dv ? o * silu(za) : 0.f;
            float ss = g * g, unused1 = 0.f, unused2 = 0.f;
            block_sum3(ss, unused1, unused2, red);
            ya = g * rsqrtf(fmaf(ss, 1.0f / static_cast<float>(Dv), p.norm_eps)) * gna;
        }
        if (tid < Dv) p.y[v_off + tid] = ya;
        __syncthreads();                                   // kh, qh are rewritten next token
    }
    // the final memory
    for (int64_t i = tid; i < mem; i += kGenThreads) {
        const int r = static_cast<int>(i / Dk), c = static_cast<int>(i - static_cast<int64_t>(r) * Dk);
        p.state[head * mem + i] = Sm[r * ld + c];
    }
}

template <typename TA>
cudaError_t launch_general_typed(const gdn_params &p, bool decode, cudaStream_t stream) {
    const int bytes = static_cast<int>(general_smem_bytes(p.Dk, p.Dv));
    cudaError_t e = cudaFuncSetAttribute(gdn_general_kernel<TA>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int64_t heads = static_cast<int64_t>(p.B) * p.Hv;
    gdn_general_kernel<TA><<<static_cast<unsigned>(heads), kGenThreads, bytes, stream>>>(p, decode);
    return cudaGetLastError();
}

}  // namespace

size_t general_smem_bytes(int dk, int dv) {
    return sizeof(float) * (static_cast<size_t>(dv) * gen_ld(dk) + 2 * static_cast<size_t>(dk) +
                            3 * kGenWarps);
}

bool general_supported(int dk, int dv) {
    return dk >= 1 && dv >= 1 && dk <= 256 && dv <= kGenThreads &&
           general_smem_bytes(dk, dv) <= kGeneralSmemMax;
}

cudaError_t launch_general(const gdn_params &p, bool decode, cudaStream_t stream) {
    switch (p.act_dtype) {
        case GDN_F32: return launch_general_typed<float>(p, decode, stream);
        case GDN_BF16: return launch_general_typed<__nv_bfloat16>(p, decode, stream);
        case GDN_F16: return launch_general_typed<__half>(p, decode, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
