// gdn_scan_tc.cu -- multi-token GDN recurrence on tensor cores, memory resident in registers.
//
// What is computed is the page's per-token recurrence (logicaffeine_compile::codegen_cuda::gdn,
// module description; time loop of torch_to_nnef.op.gated_delta, gated_delta_reference), not
// an approximation of it: blocks of B = 16 tokens are written out exactly.  With S' the
// registers at the block start (true memory lam S') and x_t = S' k^_t, y_t = S' q^_t:
//     u_t = lam D_t x_t + sum_{s<t} d_s KK[s][t]             (u: the page's S k)
//     d_t = beta_t (v_t - alpha_t u_t)                         (d: the page's coef)
//     o_t = alpha_t (lam D_t y_t + sum_{s<t} d_s QX[s][t]) + d_t (k^_t . q^_t)
//     S'  <- S' + sum_s (W_s d_s / lam') k^_s,   lam' = lam Gam
// D_t = prod_{r<t} alpha_r, W_s = prod_{r>s} alpha_r, Gam = prod over the block,
// KK[s][t] = prod_{s<r<t} alpha_r (k^_s . k^_t), QX[s][t] = prod_{s<r<t} alpha_r (k^_s . q^_t);
// every decay product is exp of a non-positive sum of log_decay.  This is the page's update
// expanded the way its "The fusion" section expands o (the update is affine in S).
//
// GB300 mapping:
//   * a warp owns 16 rows of a head's memory; the rows live in registers as the f32
//     accumulator fragments of m16n8k16 tensor-core MMAs (16 x D per warp: D/8 n-tiles);
//   * X = S' K^T and Y = S' Q^T for the block's 16 tokens are MMAs whose A operand is the
//     accumulator itself (an m16n8 accumulator pair has the m16k16 A-fragment layout), and the
//     rank-16 update S' += C K^ is an MMA accumulating into the same registers;
//   * accuracy: every operand is split into bf16 hi + lo parts and a product is formed as
//     hi.hi + hi.lo + lo.hi (relative error about 2^-16 per product, f32 accumulation), so the
//     result tracks the f32 recurrence far inside the tolerance;
//   * the block's coefficients solve a unit-triangular system that is the same for every row:
//     with r_t = beta_t (v_t - alpha_t lam D_t x_t) and N[s][t] = beta_t alpha_t KK[s][t]
//     (s < t), the recurrence d_t + sum_{s<t} N[s][t] d_s = r_t gives d = r (I + N)^-1, and
//     O = lam alpha D Y + d QX' with QX'[s][t] = alpha_t QX[s][t] (s < t), QX'[t][t] =
//     k^_t . q^_t.  Per chunk, one small MMA per block forms KK and QX and one warp per block
//     inverts I + N; every warp then gets d and O of its 16 rows as two more MMAs whose A
//     operands are accumulator fragments (no per-row serial loop, no transposes);
//   * chunks of 32 tokens of q, k, v, z are staged global -> shared with cp.async (double
//     buffer) and normalised once per chunk into the bf16 hi/lo operand arrays;
//   * when a CTA owns a whole head the gated RMSNorm runs in the CTA; otherwise raw o goes to y
//     and gdn_gated_norm_kernel applies the norm afterwards.
#include <math.h>

#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

constexpr int kT = 32;                     // tokens per staged chunk
constexpr int kB = 16;                     // tokens per MMA block
static_assert(kT == 32 && kT % kB == 0, "one lane per chunk token in the decay prefix scan");
constexpr float kMinLogDecay = -80.0f;     // exp(-80) ~ 1.8e-35: a full reset for f32 purposes

template <typename TA, int D, int NW> struct TcCfg {
    static constexpr int RB = 16 * NW;               // rows per CTA
    static constexpr int NRB = D / RB;               // CTAs per head
    static constexpr int NT = 32 * NW;
    static constexpr int NTILE = D / 8;              // n-tiles of a warp's 16 x D memory block
    static constexpr int KST = D / 16;               // k-steps over D
    static constexpr int NBLK = kT / kB;
    static constexpr int LDH = D + 8;                // padded bf16 row stride (conflict-free)
    static constexpr bool WHOLE_HEAD = (RB == D);
    static constexpr int KPIECES = D * (int)sizeof(TA) / 16;
    static constexpr int VPIECES = RB * (int)sizeof(TA) / 16;
    static_assert(D % RB == 0 && D % 16 == 0, "shape");
    static_assert(KPIECES >= 1 && VPIECES >= 1, "16-byte copy granularity");
};

template <typename TA, int D, int NW> struct TcSmem {
    using C = TcCfg<TA, D, NW>;
    TA rawk[2][kT][D];
    TA rawq[2][kT][D];
    TA rawv[2][kT][C::RB];
    TA rawz[2][kT][C::RB];
    __nv_bfloat16 khi[kT][C::LDH], klo[kT][C::LDH];
    __nv_bfloat16 qhi[kT][C::LDH], qlo[kT][C::LDH];
    float vf[kT][C::RB];
    float ob[kT][C::RB];
    float sz[kT][C::RB];
    float4 tok[kT];                  // alpha, beta, k^.q^ (f32), log_decay (clamped)
    float4 dec[kT];                  // D_t, W_t, Gam of the block, block-inclusive log sum
    float nm[C::NBLK][kB][kB];       // N[s][t] = beta_t alpha_t KK[s][t] for s < t, else 0
    // B operands [s][t] (k = s, n = t), bf16 hi/lo, rows padded to 24 (conflict-free ldmatrix):
    __nv_bfloat16 thi[C::NBLK][kB][kB + 8], tlo[C::NBLK][kB][kB + 8];   // T = (I + N)^-1
    __nv_bfloat16 phi[C::NBLK][kB][kB + 8], plo[C::NBLK][kB][kB + 8];   // QX'

};

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

template <typename TA, int D, int NW>
__global__ void __launch_bounds__(TcCfg<TA, D, NW>::NT)
gdn_scan_tc_kernel(const gdn_params p) {
    using C = TcCfg<TA, D, NW>;
    using A = Act<TA>;
    using Sm = TcSmem<TA, D, NW>;
    constexpr int RB = C::RB, NTILE = C::NTILE, KST = C::KST;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);

    const int64_t head = blockIdx.x / C::NRB;              // b * Hv + hv
    const int rblk = blockIdx.x % C::NRB;
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int r0 = rblk * RB;                              // first memory row of this CTA
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;                // MMA fragment coordinates
    const int wrow = warp * 16;                            // first local row of this warp
    const int S = p.S;

    int64_t k_base, k_ts, v_base, v_ts, g_base, g_ts;
    if (p.head_major) {
        k_base = (static_cast<int64_t>(b) * p.Hk + hk) * S * D;  k_ts = D;
        v_base = head * S * D;                                   v_ts = D;
        g_base = head * S;                                       g_ts = 1;
    } else {
        k_base = (static_cast<int64_t>(b) * S * p.Hk + hk) * D;  k_ts = static_cast<int64_t>(p.Hk) * D;
        v_base = (static_cast<int64_t>(b) * S * p.Hv + hv) * D;  v_ts = static_cast<int64_t>(p.Hv) * D;
        g_base = static_cast<int64_t>(b) * S * p.Hv + hv;        g_ts = p.Hv;
    }
    const TA *kg = static_cast<const TA *>(p.k) + k_base;
    const TA *qg = static_cast<const TA *>(p.q) + k_base;
    const TA *vg = static_cast<const TA *>(p.v) + v_base + r0;
    const bool fused_norm = C::WHOLE_HEAD && p.z != nullptr;
    const TA *zg = fused_norm ? static_cast<const TA *>(p.z) + v_base : nullptr;

    auto issue_chunk = [&](int t0, int buf) {
        const int nt = min(kT, S - t0);
        for (int i = tid; i < nt * C::KPIECES; i += C::NT) {
            const int tt = i / C::KPIECES, pc = i % C::KPIECES;
            const int64_t off = (t0 + tt) * k_ts;
            cp_async16(reinterpret_cast<char *>(&sm.rawk[buf][tt][0]) + 16 * pc,
                       reinterpret_cast<const char *>(kg + off) + 16 * pc);
            cp_async16(reinterpret_cast<char *>(&sm.rawq[buf][tt][0]) + 16 * pc,
                       reinterpret_cast<const char *>(qg + off) + 16 * pc);
        }
        for (int i = tid; i < nt * C::VPIECES; i += C::NT) {
            const int tt = i / C::VPIECES, pc = i % C::VPIECES;
            cp_async16(reinterpret_cast<char *>(&sm.rawv[buf][tt][0]) + 16 * pc,
                       reinterpret_cast<const char *>(vg + (t0 + tt) * v_ts) + 16 * pc);
            if (fused_norm)
                cp_async16(reinterpret_cast<char *>(&sm.rawz[buf][tt][0]) + 16 * pc,
                           reinterpret_cast<const char *>(zg + (t0 + tt) * v_ts) + 16 * pc);
        }
        cp_async_commit();
    };

    // the warp's 16 x D block of the memory as accumulator fragments:
    // sacc[j] = S[wrow+g][8j+2tq], S[wrow+g][8j+2tq+1], S[wrow+g+8][8j+2tq], S[wrow+g+8][8j+2tq+1]
    float sacc[NTILE][4];
    {
        const float *s0 = p.s0 ? p.s0 + head * (D * D) + static_cast<int64_t>(r0 + wrow) * D : nullptr;
#pragma unroll
        for (int j = 0; j < NTILE; j++) {
            float2 lo = make_float2(0.f, 0.f), hi = lo;
            if (s0) {
                lo = *reinterpret_cast<const float2 *>(s0 + g * D + 8 * j + 2 * tq);
                hi = *reinterpret_cast<const float2 *>(s0 + (g + 8) * D + 8 * j + 2 * tq);
            }
            sacc[j][0] = lo.x; sacc[j][1] = lo.y; sacc[j][2] = hi.x; sacc[j][3] = hi.y;
        }
    }

    float gl = 0.f, gb = 0.f;
    if (tid < kT && tid < S) {
        gl = load_gate(p.log_decay, p.gate_dtype, g_base + tid * g_ts);
        gb = load_gate(p.beta, p.gate_dtype, g_base + tid * g_ts);
    }
    issue_chunk(0, 0);

    const float inv_sqrt_dk = rsqrtf(static_cast<float>(D));
    const int nchunks = (S + kT - 1) / kT;
    constexpr int EPL_OUT = (D + 31) / 32;
    float gnr[EPL_OUT];                                    // the norm weight, read once
#pragma unroll
    for (int i = 0; i < EPL_OUT; i++) {
        const int j = lane + 32 * i;
        gnr[i] = (fused_norm && j < D) ? p.gn[j] : 0.f;
    }
    float lam = 1.0f;                                      // true memory = lam * registers
    for (int ch = 0; ch < nchunks; ch++) {
        const int t0 = ch * kT;
        const int nt = min(kT, S - t0);
        const int buf = ch & 1;
        if (ch + 1 < nchunks) {
            issue_chunk(t0 + kT, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // ---- stage 1: q^, k^ as bf16 hi/lo operand arrays (rows past the sequence end are
        //      zero so that the block MMAs see exact zeros there); gates; v, silu(z)
#pragma unroll
        for (int it = 0; it < kT / NW; it++) {             // fixed trip count: tokens overlap
            const int tt = warp + it * NW;
            constexpr int EPL = (D + 31) / 32;
            float kx[EPL], qx[EPL];
            float ssk = 0.f, ssq = 0.f, skq = 0.f;
            const bool valid = tt < nt;                    // warp-uniform
#pragma unroll
            for (int i = 0; i < EPL; i++) {
                const int j = lane + 32 * i;
                kx[i] = (valid && j < D) ? A::one(&sm.rawk[buf][tt][j]) : 0.f;
                qx[i] = (valid && j < D) ? A::one(&sm.rawq[buf][tt][j]) : 0.f;
                ssk = fmaf(kx[i], kx[i], ssk);
                ssq = fmaf(qx[i], qx[i], ssq);
                skq = fmaf(kx[i], qx[i], skq);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {       // the three sums reduce together
                ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
                ssq += __shfl_xor_sync(0xffffffffu, ssq, off);
                skq += __shfl_xor_sync(0xffffffffu, skq, off);
            }
            const float rk = rsqrtf(ssk + p.qk_eps);
            const float rq = rsqrtf(ssq + p.qk_eps) * inv_sqrt_dk;
#pragma unroll
            for (int i = 0; i < EPL; i++) {
                const int j = lane + 32 * i;
                if (j < D) {
                    split1(kx[i] * rk, sm.khi[tt][j], sm.klo[tt][j]);
                    split1(qx[i] * rq, sm.qhi[tt][j], sm.qlo[tt][j]);
                }
            }
            if (lane == 0) sm.tok[tt].z = skq * rk * rq;
        }
        static_assert((kT * RB / 4) % C::NT == 0, "4-element groups tile the chunk's v slice");
#pragma unroll
        for (int it = 0; it < kT * RB / 4 / C::NT; it++) {   // 4 consecutive values per thread
            const int i = 4 * (tid + it * C::NT);
            const int tt = i / RB, j = i % RB;
            if (tt < nt) {
                *reinterpret_cast<float4 *>(&sm.vf[tt][j]) = A::four(&sm.rawv[buf][tt][j]);
                if (fused_norm) {
                    const float4 z4 = A::four(&sm.rawz[buf][tt][j]);
                    *reinterpret_cast<float4 *>(&sm.sz[tt][j]) =
                        make_float4(silu_fast(z4.x), silu_fast(z4.y), silu_fast(z4.z), silu_fast(z4.w));
                }
            }
        }
        if (tid < kT) {
            const float gc = (tid < nt) ? fmaxf(gl, kMinLogDecay) : 0.f;
            sm.tok[tid].x = expf(gc);
            sm.tok[tid].y = (tid < nt) ? gb : 0.f;
            sm.tok[tid].w = gc;
        }
        if (tid < kT && t0 + kT + tid < S) {
            const int64_t gi = g_base + static_cast<int64_t>(t0 + kT + tid) * g_ts;
            gl = load_gate(p.log_decay, p.gate_dtype, gi);
            gb = load_gate(p.beta, p.gate_dtype, gi);
        }
        __syncthreads();

        // ---- stage 2: decay products per token; KK, QX by MMA; N and QX' tables
        if (warp == 0) {                                   // kT == 32: one lane per token
            // block-relative inclusive prefix sum of log_decay (invalid tokens hold 0)
            const float gj = sm.tok[lane].w;
            float upto = gj;
#pragma unroll
            for (int off = 1; off < kB; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, upto, off, kB);
                if ((lane & (kB - 1)) >= off) upto += o;
            }
            const float total = __shfl_sync(0xffffffffu, upto, kB - 1, kB);
            sm.dec[lane] = make_float4(expf(upto - gj), expf(total - upto), expf(total), upto);
        }
        __syncthreads();
        for (int task = warp; task < 4 * C::NBLK; task += NW) {
            const int blk = task >> 2;
            const bool isq = (task >> 1) & 1;
            const int nt8 = task & 1;                      // which 8 tokens t
            const int tb = blk * kB;
            float acc2[2][4] = {};                          // even / odd k-steps (shorter chains)
#pragma unroll
            for (int kk = 0; kk < KST; kk++) {
                // A = K^[s = tb..tb+15][cols 16kk..16kk+15]  (hi and lo)
                uint32_t ah[4], al[4];
                const int m = lane >> 3, r = lane & 7;       // matrix, row of ldmatrix
                {
                    const int srow = tb + r + ((m & 1) ? 8 : 0);
                    const int col = 16 * kk + ((m & 2) ? 8 : 0);
                    ldsm_x4(ah, &sm.khi[srow][col]);
                    ldsm_x4(al, &sm.klo[srow][col]);
                }
                // B = (K^ or Q^)^T: rows of the ldmatrix are tokens t, 8 columns each
                uint32_t bb[4];
                const int trow = tb + 8 * nt8 + r;
                const int col = 16 * kk + ((m & 1) ? 8 : 0);
                const __nv_bfloat16 *src = (m & 2) ? (isq ? &sm.qlo[trow][col] : &sm.klo[trow][col])
                                                   : (isq ? &sm.qhi[trow][col] : &sm.khi[trow][col]);
                ldsm_x4(bb, src);
                mma3(acc2[kk & 1], ah, al, bb[0], bb[1], bb[2], bb[3]);
            }
            // epilogue: entry (s, t) with s = g or g + 8, t = 8 nt8 + 2 tq (+1)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int s2 = g + ((e & 2) ? 8 : 0);
                const int t = 8 * nt8 + 2 * tq + (e & 1);
                const float dot = acc2[0][e] + acc2[1][e];
                const float4 tk = sm.tok[tb + t];          // alpha, beta, k^.q^
                float wgt = 0.f;                           // prod_{s<r<t} alpha_r
                if (s2 < t) wgt = expf(sm.dec[tb + t - 1].w - sm.dec[tb + s2].w);
                if (isq) {
                    const float val = (s2 < t) ? tk.x * wgt * dot : (s2 == t ? tk.z : 0.f);
                    split1(val, sm.phi[blk][s2][t], sm.plo[blk][s2][t]);
                } else {
                    sm.nm[blk][s2][t] = (s2 < t) ? tk.y * tk.x * wgt * dot : 0.f;
                }
            }
        }
        __syncthreads();
        // T = (I + N)^-1 (unit upper triangular): lane s of warp blk builds row s by forward
        // accumulation, T[s][t] = -sum_{s<=r<t} T[s][r] N[r][t].
        if (warp < C::NBLK && lane < kB) {
            const int blk = warp, srow = lane;
            float tr[kB], acc[kB];
#pragma unroll
            for (int t = 0; t < kB; t++) { tr[t] = (t == srow) ? 1.f : 0.f; acc[t] = 0.f; }
#pragma unroll
            for (int r = 0; r < kB - 1; r++) {
                if (r > srow) tr[r] = -acc[r];
#pragma unroll
                for (int t = r + 1; t < kB; t++) acc[t] = fmaf(tr[r], sm.nm[blk][r][t], acc[t]);
            }
            if (kB - 1 > srow) tr[kB - 1] = -acc[kB - 1];
#pragma unroll
            for (int t = 0; t < kB; t++) split1(tr[t], sm.thi[blk][srow][t], sm.tlo[blk][srow][t]);
        }
        __syncthreads();

        // ---- stage 3: the blocks; each warp on its own 16 rows, no inter-warp sync
        for (int blk = 0; blk * kB < nt; blk++) {
            const int tb = blk * kB;
            const int nb = min(kB, nt - tb);

            // X = S' K^T, Y = S' Q^T for the block's 16 tokens (two n8 tiles each)
            float xa[2][4] = {}, ya[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < KST; kk++) {
                uint32_t ah[4], al[4];
                split2(sacc[2 * kk][0], sacc[2 * kk][1], ah[0], al[0]);
                split2(sacc[2 * kk][2], sacc[2 * kk][3], ah[1], al[1]);
                split2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], ah[2], al[2]);
                split2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
                for (int nt8 = 0; nt8 < 2; nt8++) {
                    const int m = lane >> 3, r = lane & 7;
                    const int trow = tb + 8 * nt8 + r;
                    const int col = 16 * kk + ((m & 1) ? 8 : 0);
                    uint32_t kb[4], qb[4];
                    ldsm_x4(kb, (m & 2) ? &sm.klo[trow][col] : &sm.khi[trow][col]);
                    ldsm_x4(qb, (m & 2) ? &sm.qlo[trow][col] : &sm.qhi[trow][col]);
                    mma3(xa[nt8], ah, al, kb[0], kb[1], kb[2], kb[3]);
                    mma3(ya[nt8], ah, al, qb[0], qb[1], qb[2], qb[3]);
                }
            }
            // r = beta (v - alpha lam D x), and lam alpha D Y, at this lane's fragment positions
            float ra[2][4], oa[2][4];
#pragma unroll
            for (int nt8 = 0; nt8 < 2; nt8++)
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int rr = g + ((e & 2) ? 8 : 0);
                    const int t = 8 * nt8 + 2 * tq + (e & 1);
                    const float4 tk = sm.tok[tb + t];     // alpha, beta
                    const float lad = lam * tk.x * sm.dec[tb + t].x;
                    // exact zeros past the sequence end: those columns meet every other
                    // token's terms in the d, O and update MMAs
                    ra[nt8][e] = (t < nb) ? tk.y * (sm.vf[tb + t][wrow + rr] - lad * xa[nt8][e]) : 0.f;
                    oa[nt8][e] = lad * ya[nt8][e];
                }
            // d = r T  (A = r, rows x tokens s; B = T[s][t])
            float da[2][4] = {};
            {
                uint32_t rh[4], rl[4];
                split2(ra[0][0], ra[0][1], rh[0], rl[0]);
                split2(ra[0][2], ra[0][3], rh[1], rl[1]);
                split2(ra[1][0], ra[1][1], rh[2], rl[2]);
                split2(ra[1][2], ra[1][3], rh[3], rl[3]);
#pragma unroll
                for (int nt8 = 0; nt8 < 2; nt8++) {
                    uint32_t tbf[4];
                    const int m = lane >> 3, r = lane & 7;
                    const int srow = r + ((m & 1) ? 8 : 0);
                    ldsm_x4_t(tbf, (m & 2) ? &sm.tlo[blk][srow][8 * nt8] : &sm.thi[blk][srow][8 * nt8]);
                    mma3(da[nt8], rh, rl, tbf[0], tbf[1], tbf[2], tbf[3]);
                }
            }
            // O = lam alpha D Y + d QX'
            uint32_t dh[4], dl[4];
            split2(da[0][0], da[0][1], dh[0], dl[0]);
            split2(da[0][2], da[0][3], dh[1], dl[1]);
            split2(da[1][0], da[1][1], dh[2], dl[2]);
            split2(da[1][2], da[1][3], dh[3], dl[3]);
#pragma unroll
            for (int nt8 = 0; nt8 < 2; nt8++) {
                uint32_t pbf[4];
                const int m = lane >> 3, r = lane & 7;
                const int srow = r + ((m & 1) ? 8 : 0);
                ldsm_x4_t(pbf, (m & 2) ? &sm.plo[blk][srow][8 * nt8] : &sm.phi[blk][srow][8 * nt8]);
                mma3(oa[nt8], dh, dl, pbf[0], pbf[1], pbf[2], pbf[3]);
            }
#pragma unroll
            for (int nt8 = 0; nt8 < 2; nt8++) {
                const int t = 8 * nt8 + 2 * tq;
                if (t < nb) {
                    sm.ob[tb + t][wrow + g] = oa[nt8][0];
                    sm.ob[tb + t][wrow + g + 8] = oa[nt8][2];
                }
                if (t + 1 < nb) {
                    sm.ob[tb + t + 1][wrow + g] = oa[nt8][1];
                    sm.ob[tb + t + 1][wrow + g + 8] = oa[nt8][3];
                }
            }
            // the rank-16 update: C = d W / lam' (A fragment), S' += C K^
            const float gam = sm.dec[tb].z;
            const float lam_new = lam * gam;
            const bool fold = !(lam_new >= 0x1p-40f);      // CTA-uniform
            const float scale = fold ? 1.0f : 1.0f / lam_new;
            float cf[2][4];
#pragma unroll
            for (int nt8 = 0; nt8 < 2; nt8++)
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int t = 8 * nt8 + 2 * tq + (e & 1);
                    cf[nt8][e] = da[nt8][e] * sm.dec[tb + t].y * scale;
                }
            // A fragment of the coefficients (rows x tokens, k = token)
            uint32_t ch_[4], cl_[4];
            split2(cf[0][0], cf[0][1], ch_[0], cl_[0]);
            split2(cf[0][2], cf[0][3], ch_[1], cl_[1]);
            split2(cf[1][0], cf[1][1], ch_[2], cl_[2]);
            split2(cf[1][2], cf[1][3], ch_[3], cl_[3]);
            if (fold) {
#pragma unroll
                for (int j = 0; j < NTILE; j++)
#pragma unroll
                    for (int e = 0; e < 4; e++) sacc[j][e] *= lam_new;
            }
            // S' += C K^ : B = K^[tokens][cols 8j..8j+7], k = token (transposed ldmatrix)
#pragma unroll
            for (int j = 0; j < NTILE; j++) {
                uint32_t kb[4];
                const int m = lane >> 3, r = lane & 7;
                const int trow = tb + r + ((m & 1) ? 8 : 0);
                ldsm_x4_t(kb, (m & 2) ? &sm.klo[trow][8 * j] : &sm.khi[trow][8 * j]);
                mma3(sacc[j], ch_, cl_, kb[0], kb[1], kb[2], kb[3]);
            }
            lam = fold ? 1.0f : lam_new;
        }
        __syncthreads();

        // ---- outputs of the chunk
        if (fused_norm) {
            float *yg = p.y + v_base;
#pragma unroll
            for (int it = 0; it < kT / NW; it++) {
                const int tt = warp + it * NW;
                if (tt >= nt) break;                       // warp-uniform
                constexpr int EPL = (D + 31) / 32;
                const int64_t off = static_cast<int64_t>(t0 + tt) * v_ts;
                float x[EPL];
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < EPL; i++) {
                    const int j = lane + 32 * i;
                    x[i] = (j < D) ? sm.ob[tt][j] * sm.sz[tt][j] : 0.f;
                    ss = fmaf(x[i], x[i], ss);
                }
                ss = group_sum<32>(ss);
                const float rr = rsqrtf(ss / static_cast<float>(D) + p.norm_eps);
#pragma unroll
                for (int i = 0; i < EPL; i++) {
                    const int j = lane + 32 * i;
                    if (j < D) yg[off + j] = x[i] * rr * gnr[i];
                }
            }
        } else {
            float *yg = p.y + v_base + r0;
            for (int i = tid; i < nt * RB; i += C::NT) {
                const int tt = i / RB, j = i % RB;
                yg[static_cast<int64_t>(t0 + tt) * v_ts + j] = sm.ob[tt][j];
            }
        }
    }

    // final memory rows (undo the deferred decay)
    float *so = p.state + head * (D * D) + static_cast<int64_t>(r0 + wrow) * D;
#pragma unroll
    for (int j = 0; j < NTILE; j++) {
        *reinterpret_cast<float2 *>(so + g * D + 8 * j + 2 * tq) =
            make_float2(lam * sacc[j][0], lam * sacc[j][1]);
        *reinterpret_cast<float2 *>(so + (g + 8) * D + 8 * j + 2 * tq) =
            make_float2(lam * sacc[j][2], lam * sacc[j][3]);
    }
}

// Occupancy of one variant; a variant whose shared memory exceeds the per-CTA limit of this
// device reports 0 (the caller then uses a variant with fewer rows per CTA).
template <typename TA, int D, int NW>
cudaError_t prepare_tc(int *occupancy) {
    using C = TcCfg<TA, D, NW>;
    auto kern = gdn_scan_tc_kernel<TA, D, NW>;
    const int bytes = static_cast<int>(sizeof(TcSmem<TA, D, NW>));
    *occupancy = 0;
    int dev = 0, limit = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    if (bytes > limit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, kern, C::NT, bytes);
}

template <typename TA, int D, int NW>
cudaError_t launch_tc_cfg(const gdn_params &p, cudaStream_t stream) {
    using C = TcCfg<TA, D, NW>;
    const int bytes = static_cast<int>(sizeof(TcSmem<TA, D, NW>));
    const int64_t ctas = static_cast<int64_t>(p.B) * p.Hv * C::NRB;
    gdn_scan_tc_kernel<TA, D, NW><<<static_cast<unsigned>(ctas), C::NT, bytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!C::WHOLE_HEAD && p.z != nullptr) e = launch_gated_norm(p, stream);
    return e;
}

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Rows per CTA for D = 128: the fewest warps on the busiest SM with every CTA resident at
// once (a sequential scan must not run in waves); ties go to the larger CTA.
template <typename TA>
cudaError_t launch_tc_128(const gdn_params &p, cudaStream_t stream) {
    const int sms = std::max(1, device_sms());
    const int64_t heads = static_cast<int64_t>(p.B) * p.Hv;
    int occ[3] = {0, 0, 0};
    cudaError_t e;
    if ((e = prepare_tc<TA, 128, 8>(&occ[0])) != cudaSuccess) return e;
    if ((e = prepare_tc<TA, 128, 4>(&occ[1])) != cudaSuccess) return e;
    if ((e = prepare_tc<TA, 128, 2>(&occ[2])) != cudaSuccess) return e;
    const int nws[3] = {8, 4, 2};
    int best = -1;
    int64_t best_cost = INT64_MAX;
    for (int i = 0; i < 3; i++) {
        if (occ[i] < 1) continue;
        const int64_t ctas = heads * (8 / nws[i]);
        const int64_t per_sm = (ctas + sms - 1) / sms;
        const int64_t waves = (per_sm + occ[i] - 1) / occ[i];
        const int64_t cost = waves * std::min<int64_t>(per_sm, occ[i]) * nws[i];
        if (cost < best_cost) { best_cost = cost; best = i; }
    }
    if (best < 0) return cudaErrorInvalidConfiguration;
    switch (nws[best]) {
        case 8: return launch_tc_cfg<TA, 128, 8>(p, stream);
        case 4: return launch_tc_cfg<TA, 128, 4>(p, stream);
        default: return launch_tc_cfg<TA, 128, 2>(p, stream);
    }
}

template <typename TA, int D>
cudaError_t launch_tc_small(const gdn_params &p, cudaStream_t stream) {
    int occ = 0;
    cudaError_t e = prepare_tc<TA, D, D / 16>(&occ);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    return launch_tc_cfg<TA, D, D / 16>(p, stream);
}

template <typename TA>
cudaError_t launch_tc_dim(const gdn_params &p, cudaStream_t stream) {
    switch (p.Dk) {
        case 16: return launch_tc_small<TA, 16>(p, stream);
        case 32: return launch_tc_small<TA, 32>(p, stream);
        case 64: return launch_tc_small<TA, 64>(p, stream);
        case 128: return launch_tc_128<TA>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_scan_tc(const gdn_params &p, cudaStream_t stream) {
    switch (p.act_dtype) {
        case GDN_F32: return launch_tc_dim<float>(p, stream);
        case GDN_BF16: return launch_tc_dim<__nv_bfloat16>(p, stream);
        case GDN_F16: return launch_tc_dim<__half>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
