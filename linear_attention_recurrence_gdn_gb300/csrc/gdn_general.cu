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

    // the memory: a decode step updates `state` in place; a scan starts from s0 (or zeros).
    // A warp per row at a time, lanes along the row (coalesced, no index division), as
    // 4-byte asynchronous copies that are all in flight at once.
    const int warp = tid >> 5, lane = tid & 31;
    const float *from = decode ? p.state : p.s0;
    for (int r = warp; r < Dv; r += kGenWarps) {
        const float *src = from ? from + head * mem + static_cast<int64_t>(r) * Dk : nullptr;
        for (int c = lane; c < Dk; c += 32) {
            if (src) {
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                                 static_cast<uint32_t>(__cvta_generic_to_shared(Sm + r * ld + c))),
                             "l"(src + c)
                             : "memory");
            } else {
                Sm[r * ld + c] = 0.f;
            }
        }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const TA *q = static_cast<const TA *>(p.q), *k = static_cast<const TA *>(p.k);
    const TA *v = static_cast<const TA *>(p.v), *z = static_cast<const TA *>(p.z);
    const bool gated = z != nullptr;
    const float gna = (gated && tid < Dv) ? p.gn[tid] : 0.f;
    const float qscale = rsqrtf(static_cast<float>(Dk));
    float *row = Sm + tid * ld;

    // token t's offsets into q, k / v, z, y / the gates
    auto kq_off = [&](int t) {
        return p.head_major ? ((static_cast<int64_t>(b) * p.Hk + hk) * S + t) * Dk
                            : ((static_cast<int64_t>(b) * S + t) * p.Hk + hk) * Dk;
    };
    auto v_off = [&](int t) {
        return p.head_major ? ((static_cast<int64_t>(b) * p.Hv + hv) * S + t) * Dv
                            : ((static_cast<int64_t>(b) * S + t) * p.Hv + hv) * Dv;
    };
    auto g_off = [&](int t) {
        return p.head_major ? (static_cast<int64_t>(b) * p.Hv + hv) * S + t
                            : (static_cast<int64_t>(b) * S + t) * p.Hv + hv;
    };
    // this thread's inputs of a token (k, q elements tid and tid + 256; v, z row tid; gates),
    // loaded a token ahead so the loads' latency overlaps the current token's work
    float nk0 = 0.f, nq0 = 0.f, nk1 = 0.f, nq1 = 0.f, nv = 0.f, nz = 0.f, ngl = 0.f, ngb = 0.f;
    auto fetch = [&](int t) {
        const int64_t ko = kq_off(t), vo = v_off(t), go = g_off(t);
        nk0 = tid < Dk ? to_f32(k[ko + tid]) : 0.f;
        nq0 = tid < Dk ? to_f32(q[ko + tid]) : 0.f;
        nk1 = tid + kGenThreads < Dk ? to_f32(k[ko + tid + kGenThreads]) : 0.f;
        nq1 = tid + kGenThreads < Dk ? to_f32(q[ko + tid + kGenThreads]) : 0.f;
        nv = tid < Dv ? to_f32(v[vo + tid]) : 0.f;
        nz = (gated && tid < Dv) ? to_f32(z[vo + tid]) : 0.f;
        ngl = load_gate(p.log_decay, p.gate_dtype, go);
        ngb = load_gate(p.beta, p.gate_dtype, go);
    };
    if (S > 0) fetch(0);
    for (int t = 0; t < S; t++) {
        const int64_t y_off = v_off(t);
        // k, q rows and their sums of squares and dot product
        const float k0 = nk0, q0 = nq0, k1 = nk1, q1 = nq1, va = nv, za = nz;
        const float alpha = expf(fmaxf(ngl, kGenMinLogDecay));
        const float beta = ngb;
        if (t + 1 < S) fetch(t + 1);
        if (tid < Dk) {
            kh[tid] = k0;
            qh[tid] = q0;
        }
        if (tid + kGenThreads < Dk) {
            kh[tid + kGenThreads] = k1;
            qh[tid + kGenThreads] = q1;
        }
        float skk = fmaf(k0, k0, k1 * k1), sqq = fmaf(q0, q0, q1 * q1), skq = fmaf(k0, q0, k1 * q1);
        block_sum3(skk, sqq, skq, red);                    // also orders the kh, qh writes
        const float rk = rsqrtf(skk + p.qk_eps);
        const float rq = rsqrtf(sqq + p.qk_eps) * qscale;
        // row a: u, w against the raw rows, then the update with k^ = rk k
        float o = 0.f;
        if (tid < Dv) {
            // four partial sums each, so the shared-memory loads of a row pipeline
            float u4[4] = {0.f, 0.f, 0.f, 0.f}, w4[4] = {0.f, 0.f, 0.f, 0.f};
            int j = 0;
#pragma unroll 2
            for (; j + 4 <= Dk; j += 4) {
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float sj = row[j + e];
                    u4[e] = fmaf(sj, kh[j + e], u4[e]);
                    w4[e] = fmaf(sj, qh[j + e], w4[e]);
                }
            }
            for (; j < Dk; j++) {
                const float sj = row[j];
                u4[0] = fmaf(sj, kh[j], u4[0]);
                w4[0] = fmaf(sj, qh[j], w4[0]);
            }
            const float u = ((u4[0] + u4[1]) + (u4[2] + u4[3])) * rk;
            const float w = ((w4[0] + w4[1]) + (w4[2] + w4[3])) * rq;
            const float coef = beta * (va - alpha * u);
            const float ck = coef * rk;
#pragma unroll 8
            for (int jj = 0; jj < Dk; jj++) row[jj] = fmaf(alpha, row[jj], ck * kh[jj]);
            o = fmaf(alpha, w, coef * (skq * rk * rq));
        }
        float ya = o;
        if (gated) {
            const float g = tid < Dv ? o * silu(za) : 0.f;
            float ss = g * g, unused1 = 0.f, unused2 = 0.f;
            block_sum3(ss, unused1, unused2, red);
            ya = g * rsqrtf(fmaf(ss, 1.0f / static_cast<float>(Dv), p.norm_eps)) * gna;
        }
        if (tid < Dv) p.y[y_off + tid] = ya;
        __syncthreads();                                   // kh, qh are rewritten next token
    }
    // the final memory
    for (int r = warp; r < Dv; r += kGenWarps) {
        float *dst = p.state + head * mem + static_cast<int64_t>(r) * Dk;
        for (int c = lane; c < Dk; c += 32) dst[c] = Sm[r * ld + c];
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
