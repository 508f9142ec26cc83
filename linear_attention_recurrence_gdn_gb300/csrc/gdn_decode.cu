// gdn_decode.cu -- single-token GDN step, one HBM read and one HBM write of every state row.
//
// Algorithm: logicaffeine_compile::codegen_cuda::gdn, "The fusion": because the update is
// affine in S, o[a] = alpha (S_old q^)[a] + coef[a] (k^ . q^) with coef[a] = beta (v[a] -
// alpha u[a]), so one pass over a state row gives u[a] = S_old[a,:] k^ and w[a] = S_old[a,:] q^,
// and the updated row alpha S_old[a,:] + coef[a] k^ is written back from the registers that
// already hold it.  The gated RMSNorm (GDN_KERNELS: "needs the whole head") runs in the same
// CTA because one CTA owns a whole head here, so there is no second kernel and o never
// round-trips through memory.
//
// GB300 mapping (differs from the page's one-block-per-(head, row) launch):
//   * one CTA per (b, hv) head; Dv/16 warps; every warp owns 16 rows of the head;
//   * a row is split over L lanes (L = 8 for Dk = 128), each lane holding NV float4 column
//     groups (NV = 4 for Dk = 128); a warp-wide float4 load therefore covers 32/L whole
//     rows, fully coalesced, and every lane issues all of its state loads (R*NV float4,
//     64 KB per CTA for Dk = Dv = 128) before any arithmetic;
//   * row dot products reduce over the L lanes of the row with xor shuffles (log2 L stages);
//   * q^, k^ are normalised in registers (the same lane layout, so the norm sums also reduce
//     over L lanes); k^.q^ is one scalar per head, as the page notes.
#include <math.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

template <int DK> struct DecodeGeom;
template <> struct DecodeGeom<128> { static constexpr int NV = 4; };
template <> struct DecodeGeom<64> { static constexpr int NV = 4; };
template <> struct DecodeGeom<32> { static constexpr int NV = 2; };
template <> struct DecodeGeom<16> { static constexpr int NV = 1; };

template <int DK, int DV> struct DecodeCfg {
    static constexpr int NV = DecodeGeom<DK>::NV;   // float4 per lane per row
    static constexpr int L = DK / (4 * NV);         // lanes per row
    static constexpr int RPS = 32 / L;              // rows covered by one warp-wide load
    static constexpr int R = 16 / RPS;              // row slots per lane (16 rows per warp)
    static constexpr int NWARPS = DV / 16;
    static constexpr int NT = NWARPS * 32;
    static_assert(L * 4 * NV == DK && RPS * L == 32 && R * RPS == 16, "geometry");
    static_assert(DV % 16 == 0 && NWARPS >= 1, "Dv must be a multiple of 16");
};

template <typename TA, int DK, int DV>
__global__ void __launch_bounds__(DecodeCfg<DK, DV>::NT)
gdn_decode_kernel(const gdn_params p) {
    using C = DecodeCfg<DK, DV>;
    using A = Act<TA>;
    constexpr int NV = C::NV, L = C::L, RPS = C::RPS, R = C::R;

    __shared__ float red[C::NWARPS];

    const int64_t head = blockIdx.x;                     // b * Hv + hv
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane / L;                              // row within a warp-wide load
    const int part = lane % L;                           // column part of the row
    const int row0 = warp * 16 + g;                      // rows row0 + r * RPS

    float *S = p.state + head * (DV * DK);

    // 1. every state load of this lane, before anything else (memory-level parallelism)
    float4 s[R][NV];
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
        for (int c = 0; c < NV; c++)
            s[r][c] = *reinterpret_cast<const float4 *>(
                S + (row0 + r * RPS) * DK + 4 * (c * L + part));

    // 2. q, k of the key head (S == 1: both layouts address (b, hk) the same way)
    const TA *kp = static_cast<const TA *>(p.k) + (static_cast<int64_t>(b) * p.Hk + hk) * DK;
    const TA *qp = static_cast<const TA *>(p.q) + (static_cast<int64_t>(b) * p.Hk + hk) * DK;
    float4 kh[NV], qh[NV];
    float ssk = 0.f, ssq = 0.f, skq = 0.f;
#pragma unroll
    for (int c = 0; c < NV; c++) {
        kh[c] = A::four(kp + 4 * (c * L + part));
        qh[c] = A::four(qp + 4 * (c * L + part));
        ssk = dot4(kh[c], kh[c], ssk);
        ssq = dot4(qh[c], qh[c], ssq);
        skq = dot4(kh[c], qh[c], skq);
    }
    ssk = group_sum<L>(ssk);
    ssq = group_sum<L>(ssq);
    skq = group_sum<L>(skq);
    const float rk = rsqrtf(ssk + p.qk_eps);
    const float rq = rsqrtf(ssq + p.qk_eps) * rsqrtf(static_cast<float>(DK));
#pragma unroll
    for (int c = 0; c < NV; c++) {
        kh[c].x *= rk; kh[c].y *= rk; kh[c].z *= rk; kh[c].w *= rk;
        qh[c].x *= rq; qh[c].y *= rq; qh[c].z *= rq; qh[c].w *= rq;
    }
    const float kq = skq * rk * rq;                      // k^ . q^, one scalar per head

    const float alpha = expf(load_gate(p.log_decay, p.gate_dtype, head));
    const float beta = load_gate(p.beta, p.gate_dtype, head);

    const TA *vp = static_cast<const TA *>(p.v) + head * DV;
    float vr[R];
#pragma unroll
    for (int r = 0; r < R; r++) vr[r] = A::one(vp + row0 + r * RPS);

    // 3. fused pass per row: u, w from the registers, write the updated row back
    float o[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
        float pu = 0.f, pw = 0.f;
#pragma unroll
        for (int c = 0; c < NV; c++) {
            pu = dot4(s[r][c], kh[c], pu);
            pw = dot4(s[r][c], qh[c], pw);
        }
        pu = group_sum<L>(pu);
        pw = group_sum<L>(pw);
        const float coef = beta * (vr[r] - alpha * pu);
        float *row = S + (row0 + r * RPS) * DK;
#pragma unroll
        for (int c = 0; c < NV; c++) {
            float4 n;
            n.x = fmaf(alpha, s[r][c].x, coef * kh[c].x);
            n.y = fmaf(alpha, s[r][c].y, coef * kh[c].y);
            n.z = fmaf(alpha, s[r][c].z, coef * kh[c].z);
            n.w = fmaf(alpha, s[r][c].w, coef * kh[c].w);
            *reinterpret_cast<float4 *>(row + 4 * (c * L + part)) = n;
        }
        o[r] = fmaf(alpha, pw, coef * kq);
    }

    // 4. output: gated RMSNorm over the head's Dv rows, or the raw o
    float *yp = p.y + head * DV;
    if (p.z != nullptr) {
        const TA *zp = static_cast<const TA *>(p.z) + head * DV;
        float x[R];
        float ss = 0.f;
#pragma unroll
        for (int r = 0; r < R; r++) {
            x[r] = o[r] * silu(A::one(zp + row0 + r * RPS));
            ss = fmaf(x[r], x[r], ss);
        }
        // every row's x is replicated over its L lanes: count it once (part == 0)
        ss = (part == 0) ? ss : 0.f;
        ss = group_sum<32>(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float total = 0.f;
#pragma unroll
        for (int w = 0; w < C::NWARPS; w++) total += red[w];
        const float rr = rsqrtf(total / static_cast<float>(DV) + p.norm_eps);
        if (part == 0) {
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int a = row0 + r * RPS;
                yp[a] = x[r] * rr * p.gn[a];
            }
        }
    } else if (part == 0) {
#pragma unroll
        for (int r = 0; r < R; r++) yp[row0 + r * RPS] = o[r];
    }
}

template <typename TA, int D>
cudaError_t launch_typed(const gdn_params &p, cudaStream_t stream) {
    using C = DecodeCfg<D, D>;
    const int64_t heads = static_cast<int64_t>(p.B) * p.Hv;
    gdn_decode_kernel<TA, D, D><<<static_cast<unsigned>(heads), C::NT, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_dim(const gdn_params &p, cudaStream_t stream) {
    switch (p.Dk) {
        case 16: return launch_typed<TA, 16>(p, stream);
        case 32: return launch_typed<TA, 32>(p, stream);
        case 64: return launch_typed<TA, 64>(p, stream);
        case 128: return launch_typed<TA, 128>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode(const gdn_params &p, cudaStream_t stream) {
    switch (p.act_dtype) {
        case GDN_F32: return launch_dim<float>(p, stream);
        case GDN_BF16: return launch_dim<__nv_bfloat16>(p, stream);
        case GDN_F16: return launch_dim<__half>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
