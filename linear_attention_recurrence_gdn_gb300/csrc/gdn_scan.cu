// gdn_scan.cu -- multi-token GDN recurrence with the memory resident on chip.
//
// Recurrence: logicaffeine_compile::codegen_cuda::gdn (module description), evaluated per
// token with the single-pass identity of its "The fusion" section; the time loop follows
// torch_to_nnef.op.gated_delta, gated_delta_reference (recurrence over the time axis, s0 in,
// final state out).
//
// GB300 mapping:
//   * the rows of a head are independent given (k^, q^, v[a], alpha, beta): row a only
//     needs its own u[a] for coef[a] and its own w[a] for o[a].  A CTA therefore owns RB
//     rows (a "row block") of one head and keeps them in registers for the whole sequence;
//     the grid is (heads x row blocks), chosen so that every CTA is resident at once;
//   * lane layout as in the decode kernel: a row is split over L lanes holding NV float4
//     column groups each, 16 rows per warp, row dots reduced with xor shuffles;
//   * the time axis is cut into chunks of T tokens.  Raw q, k and the CTA's v slice of the
//     next chunk are copied global -> shared with cp.async while the current chunk runs
//     (double buffer); at the start of a chunk all warps normalise its q, k once into f32
//     shared memory (k^, q^ and the scalar k^.q^ per token), so the per-token loop only
//     reads shared memory;
//   * outputs of a chunk collect in shared memory.  When a CTA owns a whole head the gated
//     RMSNorm runs in the CTA; otherwise raw o goes to y and gdn_gated_norm_kernel applies
//     the norm afterwards (the norm couples all Dv rows of a head).
#include <math.h>

#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

constexpr int kChunk = 32;   // tokens per staged chunk

template <int DK> struct ScanGeom;
template <> struct ScanGeom<128> { static constexpr int NV = 4; };
template <> struct ScanGeom<64> { static constexpr int NV = 4; };
template <> struct ScanGeom<32> { static constexpr int NV = 2; };
template <> struct ScanGeom<16> { static constexpr int NV = 1; };

template <typename TA, int DK, int DV, int NW> struct ScanCfg {
    static constexpr int NV = ScanGeom<DK>::NV;
    static constexpr int L = DK / (4 * NV);
    static constexpr int RPS = 32 / L;
    static constexpr int R = 16 / RPS;
    static constexpr int RB = 16 * NW;               // rows per CTA
    static constexpr int NRB = DV / RB;              // CTAs per head
    static constexpr int NT = 32 * NW;
    static constexpr int T = kChunk;
    static constexpr bool WHOLE_HEAD = (RB == DV);
    static constexpr int KPIECES = DK * (int)sizeof(TA) / 16;   // 16-byte pieces per q/k token
    static constexpr int VPIECES = RB * (int)sizeof(TA) / 16;   // 16-byte pieces per v slice
    static_assert(DV % RB == 0, "row blocks must tile Dv");
    static_assert(KPIECES >= 1 && VPIECES >= 1, "16-byte copy granularity");
    static_assert(2 * R == L, "one reduced value (u or w of a row slot) per lane");
};

// Shared-memory layout of one CTA (dynamic shared memory, 16-byte aligned members).
template <typename TA, int DK, int DV, int NW> struct ScanSmem {
    using C = ScanCfg<TA, DK, DV, NW>;
    TA rawk[2][C::T][DK];
    TA rawq[2][C::T][DK];
    TA rawv[2][C::T][C::RB];
    TA rawz[2][C::T][C::RB];   // only filled when the CTA owns a whole head and z is given
    float kh[C::T][DK];
    float qh[C::T][DK];
    float vf[C::T][C::RB];
    float ob[C::T][C::RB];
    float sz[C::T][C::RB];     // silu(z) of the chunk (whole-head CTAs with z)
    float4 tok[C::T];          // per token: alpha, beta, k^.q^, 1 / alpha
};

// Reduce-scatter over the L lanes of an aligned group: every lane holds L partial values;
// afterwards lane `part` holds the group-wide sum of value number `part`.  L - 1 shuffles
// (L/2 + L/4 + ... + 1) instead of L log2(L) for separate all-reductions.
template <int L>
__device__ __forceinline__ float reduce_scatter(float (&v)[L], int part) {
#pragma unroll
    for (int h = L / 2; h >= 1; h >>= 1) {
        const bool upper = (part & h) != 0;
#pragma unroll
        for (int j = 0; j < h; j++) {
            const float send = upper ? v[j] : v[j + h];
            const float keep = upper ? v[j + h] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, h);
        }
    }
    return v[0];
}

template <typename TA, int DK, int DV, int NW>
__global__ void __launch_bounds__(ScanCfg<TA, DK, DV, NW>::NT)
gdn_scan_kernel(const gdn_params p) {
    using C = ScanCfg<TA, DK, DV, NW>;
    using A = Act<TA>;
    using Sm = ScanSmem<TA, DK, DV, NW>;
    constexpr int NV = C::NV, L = C::L, RPS = C::RPS, R = C::R, T = C::T, RB = C::RB;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);

    const int64_t head = blockIdx.x / C::NRB;              // b * Hv + hv
    const int rblk = blockIdx.x % C::NRB;
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int r0 = rblk * RB;                              // first row of this CTA
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane / L, part = lane % L;
    const int lrow0 = warp * 16 + g;                       // local rows lrow0 + r * RPS
    const int S = p.S;

    // element offsets of token t: base + t * stride, per layout
    int64_t k_base, k_ts, v_base, v_ts, g_base, g_ts;
    if (p.head_major) {
        k_base = (static_cast<int64_t>(b) * p.Hk + hk) * S * DK;  k_ts = DK;
        v_base = head * S * DV;                                   v_ts = DV;
        g_base = head * S;                                        g_ts = 1;
    } else {
        k_base = (static_cast<int64_t>(b) * S * p.Hk + hk) * DK;  k_ts = static_cast<int64_t>(p.Hk) * DK;
        v_base = (static_cast<int64_t>(b) * S * p.Hv + hv) * DV;  v_ts = static_cast<int64_t>(p.Hv) * DV;
        g_base = static_cast<int64_t>(b) * S * p.Hv + hv;         g_ts = p.Hv;
    }
    const TA *kg = static_cast<const TA *>(p.k) + k_base;
    const TA *qg = static_cast<const TA *>(p.q) + k_base;
    const TA *vg = static_cast<const TA *>(p.v) + v_base + r0;
    const bool fused_norm = C::WHOLE_HEAD && p.z != nullptr;
    const TA *zg = fused_norm ? static_cast<const TA *>(p.z) + v_base : nullptr;

    auto issue_chunk = [&](int t0, int buf) {
        const int nt = min(T, S - t0);
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

    // initial memory rows of this lane
    float4 s[R][NV];
    {
        const float *s0 = p.s0 ? p.s0 + head * (DV * DK) + static_cast<int64_t>(r0) * DK : nullptr;
#pragma unroll
        for (int r = 0; r < R; r++)
#pragma unroll
            for (int c = 0; c < NV; c++)
                s[r][c] = s0 ? *reinterpret_cast<const float4 *>(
                                   s0 + (lrow0 + r * RPS) * DK + 4 * (c * L + part))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // gates of the current chunk, one token per thread (tid < T), prefetched a chunk ahead
    float gl = 0.f, gb = 0.f;
    if (tid < T && tid < S) {
        gl = load_gate(p.log_decay, p.gate_dtype, g_base + tid * g_ts);
        gb = load_gate(p.beta, p.gate_dtype, g_base + tid * g_ts);
    }
    issue_chunk(0, 0);

    const float inv_sqrt_dk = rsqrtf(static_cast<float>(DK));
    const int nchunks = (S + T - 1) / T;
    float lam = 1.0f;                                      // S = lam * (registers)
    float rinv = 1.0f;                                     // running product of 1/alpha
    for (int ch = 0; ch < nchunks; ch++) {
        const int t0 = ch * T;
        const int nt = min(T, S - t0);
        const int buf = ch & 1;
        if (ch + 1 < nchunks) {
            issue_chunk(t0 + T, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // ---- normalise q, k of the chunk; gates; v to f32
        for (int tt = warp; tt < nt; tt += NW) {
            constexpr int EPL = (DK + 31) / 32;
            float kx[EPL], qx[EPL];
            float ssk = 0.f, ssq = 0.f, skq = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; i++) {
                const int j = lane + 32 * i;
                kx[i] = (j < DK) ? A::one(&sm.rawk[buf][tt][j]) : 0.f;
                qx[i] = (j < DK) ? A::one(&sm.rawq[buf][tt][j]) : 0.f;
                ssk = fmaf(kx[i], kx[i], ssk);
                ssq = fmaf(qx[i], qx[i], ssq);
                skq = fmaf(kx[i], qx[i], skq);
            }
            ssk = group_sum<32>(ssk);
            ssq = group_sum<32>(ssq);
            skq = group_sum<32>(skq);
            const float rk = rsqrtf(ssk + p.qk_eps);
            const float rq = rsqrtf(ssq + p.qk_eps) * inv_sqrt_dk;
#pragma unroll
            for (int i = 0; i < EPL; i++) {
                const int j = lane + 32 * i;
                if (j < DK) {
                    sm.kh[tt][j] = kx[i] * rk;
                    sm.qh[tt][j] = qx[i] * rq;
                }
            }
            if (lane == 0) sm.tok[tt].z = skq * rk * rq;
        }
        for (int i = tid; i < nt * RB; i += C::NT) {
            const int tt = i / RB, j = i % RB;
            sm.vf[tt][j] = A::one(&sm.rawv[buf][tt][j]);
            if (fused_norm) sm.sz[tt][j] = silu(A::one(&sm.rawz[buf][tt][j]));
        }
        if (tid < nt) {
            const float a = expf(gl);
            sm.tok[tid].x = a;
            sm.tok[tid].y = gb;
            sm.tok[tid].w = 1.0f / a;                 // inf for a == 0: that token folds
        }
        // prefetch the next chunk's gates (latency hidden by the token loop)
        if (tid < T && t0 + T + tid < S) {
            const int64_t gi = g_base + static_cast<int64_t>(t0 + T + tid) * g_ts;
            gl = load_gate(p.log_decay, p.gate_dtype, gi);
            gb = load_gate(p.beta, p.gate_dtype, gi);
        }
        __syncthreads();

        // ---- the recurrence over the chunk's tokens (each warp on its own rows)
        //
        // Deferred decay: the registers hold S' = S / lam, lam the product of the alphas
        // since the last renormalisation, so the per-token update is one FMA per element:
        //   u = lam_old (S' k^),  w = lam_old (S' q^),  lam_new = alpha lam_old,
        //   coef = beta (v - lam_new (S' k^)),  o = lam_new (S' q^) + coef (k^.q^),
        //   S' += (coef / lam_new) k^,           (S = lam_new S' + coef k^ afterwards)
        // which is the page's update with alpha S folded into lam.  When lam_new would fall
        // below 2^-40 (or alpha is 0) the decay is folded into the registers instead:
        //   S' = lam_new S' + coef k^, lam = 1.
        // 1 / lam_new is kept as a running product of 1 / alpha (computed per token while the
        // chunk is staged), so the per-token path has no division.
        float4 k4[NV], q4[NV];
#pragma unroll
        for (int c = 0; c < NV; c++) {
            k4[c] = *reinterpret_cast<const float4 *>(&sm.kh[0][4 * (c * L + part)]);
            q4[c] = *reinterpret_cast<const float4 *>(&sm.qh[0][4 * (c * L + part)]);
        }
        for (int tt = 0; tt < nt; tt++) {
            const float4 tk = sm.tok[tt];                 // alpha, beta, k^.q^
            // this lane's value of v (lanes part < R own the u of row slot `part`)
            const float vrow = sm.vf[tt][lrow0 + (part % R) * RPS];
            // partial dots over this lane's columns, two-wide accumulators
            float red[2 * R];
#pragma unroll
            for (int r = 0; r < R; r++) {
                float2 au = make_float2(0.f, 0.f), aw = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < NV; c++) {
                    au = __ffma2_rn(make_float2(s[r][c].x, s[r][c].y), make_float2(k4[c].x, k4[c].y), au);
                    au = __ffma2_rn(make_float2(s[r][c].z, s[r][c].w), make_float2(k4[c].z, k4[c].w), au);
                    aw = __ffma2_rn(make_float2(s[r][c].x, s[r][c].y), make_float2(q4[c].x, q4[c].y), aw);
                    aw = __ffma2_rn(make_float2(s[r][c].z, s[r][c].w), make_float2(q4[c].z, q4[c].w), aw);
                }
                red[r] = au.x + au.y;
                red[R + r] = aw.x + aw.y;
            }
            // prefetch the next token's k^, q^ (independent of the state)
            float4 kn[NV], qn[NV];
            const int tn = (tt + 1 < nt) ? tt + 1 : tt;
#pragma unroll
            for (int c = 0; c < NV; c++) {
                kn[c] = *reinterpret_cast<const float4 *>(&sm.kh[tn][4 * (c * L + part)]);
                qn[c] = *reinterpret_cast<const float4 *>(&sm.qh[tn][4 * (c * L + part)]);
            }
            // after the reduce-scatter, lane `part` holds value `part`: u' of row slot part
            // (part < R) or w' of row slot part - R
            const float mine = reduce_scatter<L>(red, part);
            const float lam_new = lam * tk.x;
            const float rinv_new = rinv * tk.w;                           // ~ 1 / lam_new
            const bool fold = !(lam_new >= 0x1p-40f);
            const float coef = tk.y * (vrow - lam_new * mine);          // valid in lanes < R
            const float cp = fold ? coef : coef * rinv_new;               // coef / lam_new
            float cr[R];
#pragma unroll
            for (int r = 0; r < R; r++) cr[r] = __shfl_sync(0xffffffffu, cp, (lane & ~(L - 1)) | r);
            const float cw = __shfl_sync(0xffffffffu, cp, (lane & ~(L - 1)) | (part & (R - 1)));
            if (part >= R) {                                              // o of row slot part - R
                const float coef_w = fold ? cw : cw * lam_new;             // coef of that row
                sm.ob[tt][lrow0 + (part - R) * RPS] = fmaf(lam_new, mine, coef_w * tk.z);
            }
            if (fold) {                                                   // rare, CTA-uniform
#pragma unroll
                for (int r = 0; r < R; r++)
#pragma unroll
                    for (int c = 0; c < NV; c++) {
                        s[r][c].x = fmaf(lam_new, s[r][c].x, cr[r] * k4[c].x);
                        s[r][c].y = fmaf(lam_new, s[r][c].y, cr[r] * k4[c].y);
                        s[r][c].z = fmaf(lam_new, s[r][c].z, cr[r] * k4[c].z);
                        s[r][c].w = fmaf(lam_new, s[r][c].w, cr[r] * k4[c].w);
                    }
                lam = 1.0f;
                rinv = 1.0f;
            } else {
#pragma unroll
                for (int r = 0; r < R; r++) {
                    const float2 c2 = make_float2(cr[r], cr[r]);
#pragma unroll
                    for (int c = 0; c < NV; c++) {
                        const float2 lo = __ffma2_rn(c2, make_float2(k4[c].x, k4[c].y),
                                                     make_float2(s[r][c].x, s[r][c].y));
                        const float2 hi = __ffma2_rn(c2, make_float2(k4[c].z, k4[c].w),
                                                     make_float2(s[r][c].z, s[r][c].w));
                        s[r][c] = make_float4(lo.x, lo.y, hi.x, hi.y);
                    }
                }
                lam = lam_new;
                rinv = rinv_new;
            }
#pragma unroll
            for (int c = 0; c < NV; c++) {
                k4[c] = kn[c];
                q4[c] = qn[c];
            }
        }
        __syncthreads();

        // ---- outputs of the chunk
        if (fused_norm) {
            float *yg = p.y + v_base;
            for (int tt = warp; tt < nt; tt += NW) {
                constexpr int EPL = (DV + 31) / 32;
                const int64_t off = static_cast<int64_t>(t0 + tt) * v_ts;
                float x[EPL];
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < EPL; i++) {
                    const int j = lane + 32 * i;
                    x[i] = (j < DV) ? sm.ob[tt][j] * sm.sz[tt][j] : 0.f;
                    ss = fmaf(x[i], x[i], ss);
                }
                ss = group_sum<32>(ss);
                const float rr = rsqrtf(ss / static_cast<float>(DV) + p.norm_eps);
#pragma unroll
                for (int i = 0; i < EPL; i++) {
                    const int j = lane + 32 * i;
                    if (j < DV) yg[off + j] = x[i] * rr * p.gn[j];
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
    float *so = p.state + head * (DV * DK) + static_cast<int64_t>(r0) * DK;
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
        for (int c = 0; c < NV; c++) {
            const float4 v = s[r][c];
            *reinterpret_cast<float4 *>(so + (lrow0 + r * RPS) * DK + 4 * (c * L + part)) =
                make_float4(lam * v.x, lam * v.y, lam * v.z, lam * v.w);
        }
}

// Gated RMSNorm in place on y (raw o -> rmsnorm(o * silu(z)) * gn), one warp per (b, t, hv)
// output row.  z has y's layout, so rows are simply consecutive runs of Dv elements.
template <typename TA, int DV>
__global__ void __launch_bounds__(256) gdn_gated_norm_kernel(const gdn_params p, int64_t rows) {
    using A = Act<TA>;
    constexpr int EPL = (DV + 31) / 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float *y = p.y + row * DV;
    const TA *z = static_cast<const TA *>(p.z) + row * DV;
    float x[EPL];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int j = lane + 32 * i;
        x[i] = (j < DV) ? y[j] * silu(A::one(z + j)) : 0.f;
        ss = fmaf(x[i], x[i], ss);
    }
    ss = group_sum<32>(ss);
    const float rr = rsqrtf(ss / static_cast<float>(DV) + p.norm_eps);
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int j = lane + 32 * i;
        if (j < DV) y[j] = x[i] * rr * p.gn[j];
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <typename TA, int D, int NW>
cudaError_t prepare(int *occupancy) {
    using C = ScanCfg<TA, D, D, NW>;
    auto kern = gdn_scan_kernel<TA, D, D, NW>;
    const int bytes = static_cast<int>(sizeof(ScanSmem<TA, D, D, NW>));
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, kern, C::NT, bytes);
}

template <typename TA, int D, int NW>
cudaError_t launch_scan_cfg(const gdn_params &p, cudaStream_t stream) {
    using C = ScanCfg<TA, D, D, NW>;
    const int bytes = static_cast<int>(sizeof(ScanSmem<TA, D, D, NW>));
    const int64_t ctas = static_cast<int64_t>(p.B) * p.Hv * C::NRB;
    gdn_scan_kernel<TA, D, D, NW><<<static_cast<unsigned>(ctas), C::NT, bytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!C::WHOLE_HEAD && p.z != nullptr) {
        const int64_t rows = static_cast<int64_t>(p.B) * p.S * p.Hv;
        const int64_t blocks = (rows + 7) / 8;
        gdn_gated_norm_kernel<TA, D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p, rows);
        e = cudaGetLastError();
    }
    return e;
}

// Rows-per-CTA choice for Dk = Dv = 128: the fewest warps on the busiest SM (every CTA of the
// grid must be resident at once or the sequential scan would run in waves), ties to the larger
// CTA (less duplicated q/k normalisation per head).
template <typename TA>
cudaError_t launch_scan_128(const gdn_params &p, cudaStream_t stream) {
    const int sms = std::max(1, sm_count());
    const int64_t heads = static_cast<int64_t>(p.B) * p.Hv;
    int occ8 = 0, occ4 = 0, occ2 = 0;
    cudaError_t e;
    if ((e = prepare<TA, 128, 8>(&occ8)) != cudaSuccess) return e;
    if ((e = prepare<TA, 128, 4>(&occ4)) != cudaSuccess) return e;
    if ((e = prepare<TA, 128, 2>(&occ2)) != cudaSuccess) return e;
    const int nws[3] = {8, 4, 2};
    const int occs[3] = {occ8, occ4, occ2};
    int best = 0;
    int64_t best_cost = INT64_MAX;
    for (int i = 0; i < 3; i++) {
        if (occs[i] < 1) continue;
        const int64_t ctas = heads * (8 / nws[i]);
        const int64_t per_sm = (ctas + sms - 1) / sms;
        const int64_t waves = (per_sm + occs[i] - 1) / occs[i];
        const int64_t cost = waves * std::min<int64_t>(per_sm, occs[i]) * nws[i];
        if (cost < best_cost) { best_cost = cost; best = i; }
    }
    switch (nws[best]) {
        case 8: return launch_scan_cfg<TA, 128, 8>(p, stream);
        case 4: return launch_scan_cfg<TA, 128, 4>(p, stream);
        default: return launch_scan_cfg<TA, 128, 2>(p, stream);
    }
}

template <typename TA, int D>
cudaError_t launch_scan_small(const gdn_params &p, cudaStream_t stream) {
    int occ = 0;
    cudaError_t e = prepare<TA, D, D / 16>(&occ);
    if (e != cudaSuccess) return e;
    return launch_scan_cfg<TA, D, D / 16>(p, stream);
}

template <typename TA>
cudaError_t launch_scan_dim(const gdn_params &p, cudaStream_t stream) {
    switch (p.Dk) {
        case 16: return launch_scan_small<TA, 16>(p, stream);
        case 32: return launch_scan_small<TA, 32>(p, stream);
        case 64: return launch_scan_small<TA, 64>(p, stream);
        case 128: return launch_scan_128<TA>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_scan(const gdn_params &p, cudaStream_t stream) {
    switch (p.act_dtype) {
        case GDN_F32: return launch_scan_dim<float>(p, stream);
        case GDN_BF16: return launch_scan_dim<__nv_bfloat16>(p, stream);
        case GDN_F16: return launch_scan_dim<__half>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
