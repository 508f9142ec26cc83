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
// (rows padded to whole float4s and a bank-spreading stride); 1 to 8 adjacent threads own a
// memory row and split its float4s.  The scan runs in chunks of up to 32 tokens (the chunk's
// k, q norms at once, its tokens' row updates in place back to back, then the gated RMSNorm a
// warp per token); a memory too large for the chunk buffers goes token by token, with block
// reductions for the norms.
// A decode step has its own kernel: the memory streams through shared memory in its dense
// layout (16-byte copies wherever Dv Dk is a multiple of 4), with up to 7 heads per SM in
// flight.  Plain loads and stores of the step's inputs and outputs: they may sit at any
// element offset (pinned host memory under GDN_FLAG_HOST_IO included).
#include <math.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kGenThreads = 256;          // >= the largest Dv
constexpr int kGenWarps = kGenThreads / 32;
constexpr float kGenMinLogDecay = -80.0f; // exp(-80) ~ 1.8e-35: a full reset in f32

// Threads per memory row: the most of 8, 4, 2, 1 with TPR * Dv <= 256 (more threads on the
// row walks of a small head).
__host__ __device__ constexpr int gen_tpr(int dv) { return dv <= 32 ? 8 : dv <= 64 ? 4 : dv <= 128 ? 2 : 1; }
// Dk rounded up to whole float4s (the padding columns stay zero).
__host__ __device__ constexpr int gen_dk4(int dk) { return (dk + 3) & ~3; }
// Row stride of the memory in shared memory (floats): dk4 or a little more, with ld / (4 TPR)
// odd when TPR < 8, so the float4 reads of the 8 / TPR rows one quarter-warp covers fall on
// distinct banks (at most 8 TPR - 4 floats of padding a row).
__host__ __device__ constexpr int gen_ld(int dk, int dv) {
    const int tpr = gen_tpr(dv);
    int ld = gen_dk4(dk);
    if (tpr < 8)
        while (ld % (8 * tpr) != 4 * tpr) ld += 4;
    return ld;
}

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
__global__ void __launch_bounds__(kGenThreads, 1) gdn_general_kernel(const gdn_params p) {
    extern __shared__ __align__(16) float gsm[];
    const int Dk = p.Dk, Dv = p.Dv, S = p.S;
    const int TPR = gen_tpr(Dv), dk4 = gen_dk4(Dk), ld = gen_ld(Dk, Dv), nc = dk4 / 4;
    float *Sm = gsm;                                       // [Dv][ld]
    float *kh = Sm + Dv * ld;                              // [dk4]
    float *qh = kh + dk4;                                  // [dk4]
    float *red = qh + dk4;                                 // [3][kGenWarps]
    const int64_t head = blockIdx.x;                       // b * Hv + hv
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int tid = threadIdx.x;
    const int a = tid / TPR, part = tid - a * TPR;         // this thread's row and column part
    const bool live = a < Dv;
    const int64_t mem = static_cast<int64_t>(Dv) * Dk;

    // the memory from s0 (or zeros): a warp per row at a time, lanes along the row (coalesced),
    // as 4-byte asynchronous copies that are all in flight at once; the padding columns are
    // zeroed
    const int warp = tid >> 5, lane = tid & 31;
    const float *from = p.s0;
    for (int r = warp; r < Dv; r += kGenWarps) {
        const float *src = from ? from + head * mem + static_cast<int64_t>(r) * Dk : nullptr;
        for (int c = lane; c < ld; c += 32) {
            if (src && c < Dk) {
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
    const float gna = (gated && live) ? p.gn[a] : 0.f;
    const float qscale = rsqrtf(static_cast<float>(Dk));
    float4 *row4 = reinterpret_cast<float4 *>(Sm + (live ? a : 0) * ld);
    const float4 *kh4 = reinterpret_cast<const float4 *>(kh);
    const float4 *qh4 = reinterpret_cast<const float4 *>(qh);

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
    // this thread's inputs of a token (k, q element tid; v, z of its row; the gates), loaded a
    // token ahead so the loads' latency overlaps the current token's work
    float nk = 0.f, nq = 0.f, nv = 0.f, nz = 0.f, ngl = 0.f, ngb = 0.f;
    auto fetch = [&](int t) {
        const int64_t ko = kq_off(t), vo = v_off(t), go = g_off(t);
        nk = tid < Dk ? to_f32(k[ko + tid]) : 0.f;
        nq = tid < Dk ? to_f32(q[ko + tid]) : 0.f;
        nv = live ? to_f32(v[vo + a]) : 0.f;
        nz = (gated && live) ? to_f32(z[vo + a]) : 0.f;
        ngl = load_gate(p.log_decay, p.gate_dtype, go);
        ngb = load_gate(p.beta, p.gate_dtype, go);
    };
    if (S > 0) fetch(0);
    for (int t = 0; t < S; t++) {
        const int64_t y_off = v_off(t);
        // k, q rows (zero-padded to whole float4s) and their sums of squares and dot product
        const float kt = nk, qt = nq, va = nv, za = nz;
        const float alpha = expf(fmaxf(ngl, kGenMinLogDecay));
        const float beta = ngb;
        if (t + 1 < S) fetch(t + 1);
        if (tid < dk4) {
            kh[tid] = kt;
            qh[tid] = qt;
        }
        float skk = kt * kt, sqq = qt * qt, skq = kt * qt;
        block_sum3(skk, sqq, skq, red);                    // also orders the kh, qh writes
        const float rk = rsqrtf(skk + p.qk_eps);
        const float rq = rsqrtf(sqq + p.qk_eps) * qscale;
        // row a: u, w against the raw rows (the row's TPR threads take every TPR-th float4),
        // then the update with k^ = rk k
        float uu = 0.f, ww = 0.f;
        if (live) {
#pragma unroll 4
            for (int c = part; c < nc; c += TPR) {
                const float4 s4 = row4[c];
                uu = dot4(s4, kh4[c], uu);
                ww = dot4(s4, qh4[c], ww);
            }
        }
        for (int off = 1; off < TPR; off <<= 1) {          // the row's threads are adjacent lanes
            uu += __shfl_xor_sync(0xffffffffu, uu, off);
            ww += __shfl_xor_sync(0xffffffffu, ww, off);
        }
        float o = 0.f;
        if (live) {
            const float u = uu * rk, w = ww * rq;
            const float coef = beta * (va - alpha * u);
            const float ck = coef * rk;
#pragma unroll 4
            for (int c = part; c < nc; c += TPR) {
                const float4 s4 = row4[c], k4 = kh4[c];
                row4[c] = make_float4(fmaf(alpha, s4.x, ck * k4.x), fmaf(alpha, s4.y, ck * k4.y),
                                      fmaf(alpha, s4.z, ck * k4.z), fmaf(alpha, s4.w, ck * k4.w));
            }
            o = fmaf(alpha, w, coef * (skq * rk * rq));
        }
        float ya = o;
        if (gated) {
            const float g = live ? o * silu(za) : 0.f;
            float ss = part == 0 ? g * g : 0.f, unused1 = 0.f, unused2 = 0.f;
            block_sum3(ss, unused1, unused2, red);
            ya = g * rsqrtf(fmaf(ss, 1.0f / static_cast<float>(Dv), p.norm_eps)) * gna;
        }
        if (live && part == 0) p.y[y_off + a] = ya;
        __syncthreads();                                   // kh, qh are rewritten next token
    }
    // the final memory
    for (int r = warp; r < Dv; r += kGenWarps) {
        float *dst = p.state + head * mem + static_cast<int64_t>(r) * Dk;
        for (int c = lane; c < Dk; c += 32) dst[c] = Sm[r * ld + c];
    }
}

// The scan in chunks of C tokens (C a power of two up to 32, as many as shared memory takes):
// the arithmetic of the kernel above, reordered so that nothing waits per token but the row
// walks.  Per chunk: every token's k, q rows are normalised at once (a warp per token; k^ and
// q^ / sqrt(Dk) into shared memory with k^ . q^, the gates, v and z), then the tokens run one
// after another, each row's threads updating their own row with no barrier between tokens,
// and the outputs o_t of the chunk wait in shared memory for the gated RMSNorm, a warp per
// token, which also stores y.
template <typename TA>
__global__ void __launch_bounds__(kGenThreads, 1) gdn_general_chunk_kernel(const gdn_params p, int C) {
    extern __shared__ __align__(16) float gsm[];
    const int Dk = p.Dk, Dv = p.Dv, S = p.S;
    const int TPR = gen_tpr(Dv), dk4 = gen_dk4(Dk), ld = gen_ld(Dk, Dv), nc = dk4 / 4;
    float *Sm = gsm;                                       // [Dv][ld]
    float *KH = Sm + Dv * ld;                              // [C][dk4]: k_t rk_t
    float *QH = KH + C * dk4;                              // [C][dk4]: q_t rq_t / sqrt(Dk)
    float *VB = QH + C * dk4;                              // [C][Dv]: v
    float *ZB = VB + C * Dv;                               // [C][Dv]: z
    float *OB = ZB + C * Dv;                               // [C][Dv]: o, then o silu(z)
    float *AL = OB + C * Dv;                               // [C]: alpha
    float *BE = AL + C;                                    // [C]: beta
    float *KQ = BE + C;                                    // [C]: k^ . q^
    const int64_t head = blockIdx.x;                       // b * Hv + hv
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int a = tid / TPR, part = tid - a * TPR;         // this thread's row and column part
    const bool live = a < Dv;
    const int64_t mem = static_cast<int64_t>(Dv) * Dk;

    // the memory from s0 (or zeros), as in the kernel above
    for (int r = warp; r < Dv; r += kGenWarps) {
        const float *src = p.s0 ? p.s0 + head * mem + static_cast<int64_t>(r) * Dk : nullptr;
        for (int c = lane; c < ld; c += 32) {
            if (src && c < Dk) {
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
    const float qscale = rsqrtf(static_cast<float>(Dk));
    float4 *row4 = reinterpret_cast<float4 *>(Sm + (live ? a : 0) * ld);
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
    for (int t0 = 0; t0 < S; t0 += C) {
        const int nt = min(C, S - t0);
        // the chunk's k, q rows normalised, a warp per token (Dk <= 256: 8 elements a lane)
        for (int tt = warp; tt < nt; tt += kGenWarps) {
            const int64_t ko = kq_off(t0 + tt);
            float kv[8], qv[8], sk = 0.f, sq = 0.f, skq = 0.f;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int c = lane + 32 * i;
                kv[i] = c < Dk ? to_f32(k[ko + c]) : 0.f;
                qv[i] = c < Dk ? to_f32(q[ko + c]) : 0.f;
                sk = fmaf(kv[i], kv[i], sk);
                sq = fmaf(qv[i], qv[i], sq);
                skq = fmaf(kv[i], qv[i], skq);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                skq += __shfl_xor_sync(0xffffffffu, skq, off);
            }
            const float rk = rsqrtf(sk + p.qk_eps);
            const float rq = rsqrtf(sq + p.qk_eps) * qscale;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int c = lane + 32 * i;
                if (c < dk4) {
                    KH[tt * dk4 + c] = kv[i] * rk;
                    QH[tt * dk4 + c] = qv[i] * rq;
                }
            }
            if (lane == 0) {
                const int64_t go = g_off(t0 + tt);
                KQ[tt] = skq * rk * rq;
                AL[tt] = expf(fmaxf(load_gate(p.log_decay, p.gate_dtype, go), kGenMinLogDecay));
                BE[tt] = load_gate(p.beta, p.gate_dtype, go);
            }
        }
        for (int i = tid; i < nt * Dv; i += kGenThreads) {  // v and z rows of the chunk
            const int tt = i / Dv, r = i - tt * Dv;
            const int64_t vo = v_off(t0 + tt);
            VB[i] = to_f32(v[vo + r]);
            if (gated) ZB[i] = to_f32(z[vo + r]);
        }
        __syncthreads();
        // the tokens in order: each row's TPR threads own it, so no barrier between tokens
        for (int tt = 0; tt < nt; tt++) {
            const float4 *kh4 = reinterpret_cast<const float4 *>(KH + tt * dk4);
            const float4 *qh4 = reinterpret_cast<const float4 *>(QH + tt * dk4);
            float uu = 0.f, ww = 0.f;
            if (live) {
#pragma unroll 4
                for (int c = part; c < nc; c += TPR) {
                    const float4 s4 = row4[c];
                    uu = dot4(s4, kh4[c], uu);
                    ww = dot4(s4, qh4[c], ww);
                }
            }
            for (int off = 1; off < TPR; off <<= 1) {      // the row's threads are adjacent lanes
                uu += __shfl_xor_sync(0xffffffffu, uu, off);
                ww += __shfl_xor_sync(0xffffffffu, ww, off);
            }
            if (live) {
                const float alpha = AL[tt];
                const float coef = BE[tt] * (VB[tt * Dv + a] - alpha * uu);
#pragma unroll 4
                for (int c = part; c < nc; c += TPR) {
                    const float4 s4 = row4[c], k4 = kh4[c];
                    row4[c] = make_float4(fmaf(alpha, s4.x, coef * k4.x), fmaf(alpha, s4.y, coef * k4.y),
                                          fmaf(alpha, s4.z, coef * k4.z), fmaf(alpha, s4.w, coef * k4.w));
                }
                if (part == 0) OB[tt * Dv + a] = fmaf(alpha, ww, coef * KQ[tt]);
            }
        }
        __syncthreads();
        // the gated RMSNorm (or raw o) and the y stores, a warp per token
        for (int tt = warp; tt < nt; tt += kGenWarps) {
            float *yo = p.y + v_off(t0 + tt);
            float *ob = OB + tt * Dv;
            if (gated) {
                const float *zb = ZB + tt * Dv;
                float ss = 0.f;
                for (int r = lane; r < Dv; r += 32) {
                    const float g = ob[r] * silu(zb[r]);
                    ob[r] = g;
                    ss = fmaf(g, g, ss);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float rr = rsqrtf(fmaf(ss, 1.0f / static_cast<float>(Dv), p.norm_eps));
                for (int r = lane; r < Dv; r += 32) yo[r] = ob[r] * rr * p.gn[r];
            } else {
                for (int r = lane; r < Dv; r += 32) yo[r] = ob[r];
            }
        }
        __syncthreads();                                   // the chunk's buffers are rewritten next
    }
    // the final memory
    for (int r = warp; r < Dv; r += kGenWarps) {
        float *dst = p.state + head * mem + static_cast<int64_t>(r) * Dk;
        for (int c = lane; c < Dk; c += 32) dst[c] = Sm[r * ld + c];
    }
}

// One decode step (S = 1) for a head: the same arithmetic as the scan kernel's token, on the
// memory in its dense [Dv][Dk] layout in shared memory.  The memory's copy in is issued first
// and lands while the k, q norms are reduced; the row walks read scalars (a row of odd Dk is
// not float4-aligned); the memory goes back by 16-byte stores where it can.  At most 32
// registers a thread, so up to 7 CTAs share an SM when their memory fits.
template <typename TA>
__global__ void __launch_bounds__(kGenThreads, 7) gdn_general_decode_kernel(const gdn_params p) {
    extern __shared__ __align__(16) float gsm[];
    const int Dk = p.Dk, Dv = p.Dv;
    const int TPR = gen_tpr(Dv), dk4 = gen_dk4(Dk);
    const int64_t mem = static_cast<int64_t>(Dv) * Dk;
    const int mem4 = static_cast<int>((mem + 3) / 4);
    float *Sm = gsm;                                       // [Dv][Dk], dense
    float *kh = Sm + 4 * mem4;                             // [dk4]
    float *qh = kh + dk4;                                  // [dk4]
    float *red = qh + dk4;                                 // [3][kGenWarps]
    const int64_t head = blockIdx.x;                       // b * Hv + hv
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int tid = threadIdx.x;
    const int a = tid / TPR, part = tid - a * TPR;
    const bool live = a < Dv;
    float *gmem = p.state + head * mem;
    // 16-byte copies when every head's memory starts on a 16-byte boundary (state is)
    const bool vec = (mem & 3) == 0;
    if (vec) {
        for (int i = tid; i < mem4; i += kGenThreads)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                             static_cast<uint32_t>(__cvta_generic_to_shared(Sm + 4 * i))),
                         "l"(gmem + 4 * i)
                         : "memory");
    } else {
        for (int i = tid; i < mem; i += kGenThreads)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                             static_cast<uint32_t>(__cvta_generic_to_shared(Sm + i))),
                         "l"(gmem + i)
                         : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    // the step's inputs while the memory lands
    const TA *q = static_cast<const TA *>(p.q), *k = static_cast<const TA *>(p.k);
    const TA *v = static_cast<const TA *>(p.v), *z = static_cast<const TA *>(p.z);
    const bool gated = z != nullptr;
    // with one token both layouts put head (b, h) at b * H + h
    const int64_t ko = (static_cast<int64_t>(b) * p.Hk + hk) * Dk;
    const int64_t vo = (static_cast<int64_t>(b) * p.Hv + hv) * Dv;
    const int64_t go = static_cast<int64_t>(b) * p.Hv + hv;
    const float kt = tid < Dk ? to_f32(k[ko + tid]) : 0.f;
    const float qt = tid < Dk ? to_f32(q[ko + tid]) : 0.f;
    const float va = live ? to_f32(v[vo + a]) : 0.f;
    const float za = (gated && live) ? to_f32(z[vo + a]) : 0.f;
    const float alpha = expf(fmaxf(load_gate(p.log_decay, p.gate_dtype, go), kGenMinLogDecay));
    const float beta = load_gate(p.beta, p.gate_dtype, go);
    const float gna = (gated && live) ? p.gn[a] : 0.f;
    if (tid < dk4) {
        kh[tid] = kt;
        qh[tid] = qt;
    }
    float skk = kt * kt, sqq = qt * qt, skq = kt * qt;
    block_sum3(skk, sqq, skq, red);                        // also orders the kh, qh writes
    const float rk = rsqrtf(skk + p.qk_eps);
    const float rq = rsqrtf(sqq + p.qk_eps) * rsqrtf(static_cast<float>(Dk));
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // row a: u, w against the raw rows (the row's TPR threads take every TPR-th element), then
    // the update with k^ = rk k
    float *row = Sm + static_cast<int64_t>(live ? a : 0) * Dk;
    float uu = 0.f, ww = 0.f;
    if (live) {
#pragma unroll 4
        for (int c = part; c < Dk; c += TPR) {
            const float s = row[c];
            uu = fmaf(s, kh[c], uu);
            ww = fmaf(s, qh[c], ww);
        }
    }
    for (int off = 1; off < TPR; off <<= 1) {              // the row's threads are adjacent lanes
        uu += __shfl_xor_sync(0xffffffffu, uu, off);
        ww += __shfl_xor_sync(0xffffffffu, ww, off);
    }
    float o = 0.f;
    if (live) {
        const float u = uu * rk, w = ww * rq;
        const float coef = beta * (va - alpha * u);
        const float ck = coef * rk;
#pragma unroll 4
        for (int c = part; c < Dk; c += TPR) row[c] = fmaf(alpha, row[c], ck * kh[c]);
        o = fmaf(alpha, w, coef * (skq * rk * rq));
    }
    float ya = o;
    if (gated) {
        const float g = live ? o * silu(za) : 0.f;
        float ss = part == 0 ? g * g : 0.f, unused1 = 0.f, unused2 = 0.f;
        block_sum3(ss, unused1, unused2, red);
        ya = g * rsqrtf(fmaf(ss, 1.0f / static_cast<float>(Dv), p.norm_eps)) * gna;
    }
    if (live && part == 0) p.y[vo + a] = ya;
    __syncthreads();                                       // every row updated
    if (vec) {
        float4 *dst = reinterpret_cast<float4 *>(gmem);
        const float4 *src = reinterpret_cast<const float4 *>(Sm);
        for (int i = tid; i < mem4; i += kGenThreads) dst[i] = src[i];
    } else {
        for (int i = tid; i < mem; i += kGenThreads) gmem[i] = Sm[i];
    }
}

size_t general_chunk_smem_bytes(int dk, int dv, int c) {
    return sizeof(float) * (static_cast<size_t>(dv) * gen_ld(dk, dv) +
                            static_cast<size_t>(c) * (2 * static_cast<size_t>(gen_dk4(dk)) + 3 * static_cast<size_t>(dv) + 3));
}

size_t general_decode_smem_bytes(int dk, int dv) {
    return sizeof(float) * (4 * ((static_cast<size_t>(dv) * dk + 3) / 4) + 2 * static_cast<size_t>(gen_dk4(dk)) +
                            3 * kGenWarps);
}

template <typename TA>
cudaError_t launch_general_typed(const gdn_params &p, bool decode, cudaStream_t stream) {
    const int64_t heads = static_cast<int64_t>(p.B) * p.Hv;
    if (decode) {
        const int bytes = static_cast<int>(general_decode_smem_bytes(p.Dk, p.Dv));
        cudaError_t e = cudaFuncSetAttribute(gdn_general_decode_kernel<TA>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        gdn_general_decode_kernel<TA><<<static_cast<unsigned>(heads), kGenThreads, bytes, stream>>>(p);
        return cudaGetLastError();
    }
    // the chunked scan with the most tokens a chunk (up to 32) that fit; a head whose memory
    // leaves no room even for one token's buffers takes the token-by-token kernel
    int C = 32;
    while (C > 1 && general_chunk_smem_bytes(p.Dk, p.Dv, C) > kGeneralSmemMax) C /= 2;
    if (general_chunk_smem_bytes(p.Dk, p.Dv, C) <= kGeneralSmemMax) {
        const int bytes = static_cast<int>(general_chunk_smem_bytes(p.Dk, p.Dv, C));
        cudaError_t e = cudaFuncSetAttribute(gdn_general_chunk_kernel<TA>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        gdn_general_chunk_kernel<TA><<<static_cast<unsigned>(heads), kGenThreads, bytes, stream>>>(p, C);
        return cudaGetLastError();
    }
    const int bytes = static_cast<int>(general_smem_bytes(p.Dk, p.Dv));
    cudaError_t e = cudaFuncSetAttribute(gdn_general_kernel<TA>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    gdn_general_kernel<TA><<<static_cast<unsigned>(heads), kGenThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t general_smem_bytes(int dk, int dv) {
    return sizeof(float) * (static_cast<size_t>(dv) * gen_ld(dk, dv) + 2 * static_cast<size_t>(gen_dk4(dk)) +
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
