// gdn_scan_umma.cu -- multi-token GDN recurrence with the memory in tensor memory (tcgen05).
//
// What is computed is the page's per-token recurrence (logicaffeine_compile::codegen_cuda::gdn,
// module description; time loop of torch_to_nnef.op.gated_delta, gated_delta_reference),
// written out exactly over chunks of C = 32 tokens.  With S' the memory at the chunk start
// (true memory lam S'), x_t = S' k_t and y_t = S' q_t on the raw k, q (the l2 norms are the
// per-token scalars rk, rq) and cum_t the chunk-inclusive sum of log_decay:
//     r_t = beta_t (v_t - lam e^{cum_t} rk_t x_t),     d = r (I + N)^-1,
//     N[s][t] = beta_t e^{cum_t - cum_s} rk_s rk_t (k_s . k_t)                    (s < t)
//     o_t = lam e^{cum_t} rq_t y_t + sum_{s <= t} d_s e^{cum_t - cum_s} rk_s rq_t (k_s . q_t)
//     S'  <- S' + sum_s (e^{cum_31 - cum_s} rk_s / lam') d_s k_s^T,   lam' = lam e^{cum_31}
// This is the page's update S = alpha S + beta (v - alpha S k) k^T, o = S q unrolled over the
// chunk the way its "The fusion" section unrolls o; every step is exact algebra, so the
// result differs from the sequential loop only by rounding.
//
// GB300 mapping (bf16, Dk = Dv = 128, one CTA per head):
//   * the 128 x 128 f32 memory lives in tensor memory (lanes = memory rows); every product is
//     a tcgen05 MMA with M = 128 issued by one elected lane, A operands in tensor memory (f32 values
//     split into bf16 hi + lo, about 2^-16 relative per product; bf16 k, q exact), B operands in
//     shared memory (k and q as the tensor-map copies land them: 128-byte swizzle, K-major or
//     MN-major; the small per-chunk matrices as 8 x 8 core matrices);
//   * look-ahead: [x | y] of chunk c+1 is S'_c [K;Q]_{c+1}^T (issued while chunk c is still
//     running) plus the correction C_c (K_c [K;Q]_{c+1}^T) once chunk c's update coefficients
//     C_c are known, so the long K = 128 product stays off the serial path; the serial path per
//     chunk is r -> d = R T -> C, D -> O = D QX', S' += C K, correction -> o;
//   * 8 row warps (two per tensor-memory lane quarter, a thread per memory row, each half of
//     the columns and of the tokens) do the element-wise steps; the chunk tables come from
//     one MMA group per chunk, A = [K;Q]_{c+1}, B = [K_c | K_{c+1}]: lanes 0-31 hold
//     K_{c+1} K_c^T and K_{c+1} K_{c+1}^T, lanes 32-63 hold Q_{c+1} K_c^T and Q_{c+1} K_{c+1}^T.
//     Two table warps (lane quarters 0 and 1) turn them into the correction operand, N, the
//     unit-triangular inverse T (16 x 16 diagonal blocks by back substitution, the off-diagonal
//     block as -T11 N12 T22) and QX' (one lane per token column, 16-byte stores of the
//     core-matrix layout); the second of them issues the next chunk's table MMAs.  Six
//     staging warps issue the tensor-map copies, form the decay products one chunk ahead, the
//     q norms, and apply the gated RMSNorm to finished chunks (8 lanes per token).  The
//     operands of a chunk are buffered by chunk % 3, so the producers may run two chunks
//     ahead of the row warps.
//   * MMAs are issued by one elect.sync lane of a converged warp.
//   Only TMA, tcgen05 (mma, ld, st, alloc, commit, fences), plain shared / global accesses,
//   mbarriers and named barriers are used.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_mma.cuh"
#include "gdn_tcgen05.cuh"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

constexpr int uC = 32;                    // tokens per chunk
constexpr int uD = 128;                   // Dk = Dv
constexpr float uMinLogDecay = -80.0f;    // exp(-80) ~ 1.8e-35: a full reset for f32 purposes
constexpr int uRowW = 8;                  // warps 0-7: memory rows (two per lane quarter)
constexpr int uTabW0 = 8;                 // warps 8, 9: table warps (lane quarters 0, 1)
constexpr int uStgW0 = 10, uStgW = 6;     // warps 10-15: staging warps
constexpr int uNT = 32 * (uRowW + 2 + uStgW);
constexpr int uRT = 32 * uRowW;
constexpr int uST = 32 * uStgW;
constexpr int uGateW = uStgW - 1;         // staging warp that forms the decay products
constexpr int uNM = uC + 4;               // padded row of N^T

// Tensor-memory columns (512 allocated).
enum : uint32_t {
    TM_S = 0,                     // S' f32, 128 columns
    TM_SHI = 128, TM_SLO = 192,   // S' bf16 hi / lo (K = 128 in 64 columns of pairs)
    TM_XY = 256,                  // [x | y] of a chunk, two buffers of 64 (d reuses x, o
                                  // accumulates onto the scaled y)
    TM_RH = 384, TM_RL = 400,     // r bf16 hi / lo (K = 32)
    TM_DH = 384, TM_DL = 400,     // d bf16 hi / lo (after the d product has read r)
    TM_CH = 416, TM_CL = 432,     // C bf16 hi / lo
    TM_TAB = 448,                 // chunk tables, 64 columns (lanes 0-63 meaningful)
    TM_COLS = 512
};

constexpr uint32_t kIdN32 = umma_idesc_bf16(128, 32, false);
constexpr uint32_t kIdN64 = umma_idesc_bf16(128, 64, false);
constexpr uint32_t kIdN128Mn = umma_idesc_bf16(128, 128, true);

// A staging slot holds one chunk's k and q rows as four 32-row x 64-column boxes (128-byte
// swizzle, 4 KB each): k[0:64), q[0:64), k[64:128), q[64:128).  Rows 0-31 of a box pair form
// K, rows 32-63 Q, so [K;Q] is one 64-row operand with a uniform 1024-byte group stride.
constexpr uint32_t kBox = 4096;
constexpr uint32_t kSlotKQ = 4 * kBox;

// Byte offset of 16-byte piece pc (0..15) of q row t within a slot.
__device__ __forceinline__ uint32_t q_piece(int t, int pc) {
    return static_cast<uint32_t>(kBox + (pc >> 3) * 2 * kBox + (t >> 3) * 1024 + (t & 7) * 128 +
                                 (((pc & 7) ^ (t & 7)) << 4));
}
// Byte offset of the 16-byte run B[k = 8 kg .. 8 kg + 7][n] of a K-major operand stored as
// 8 x 8 core matrices, K = 32 (4 k-groups per 512-byte n-group row).
__device__ __forceinline__ uint32_t core_run(int n, int kg) {
    return static_cast<uint32_t>((n >> 3) * 512 + kg * 128 + (n & 7) * 16);
}

constexpr int uSlots = 4;                 // staging ring depth (chunks)

struct alignas(1024) U3Smem {
    __nv_bfloat16 kq[uSlots][kSlotKQ / 2];        // k / q staging ring (16 KB per slot)
    alignas(16) __nv_bfloat16 v[uSlots][uC][uD];  // v, z rows (unswizzled boxes)
    alignas(16) __nv_bfloat16 z[uSlots][uC][uD];
    // a chunk's operands for the row warps, by chunk % 3 (the producers may run two chunks ahead)
    alignas(16) __nv_bfloat16 thi[3][uC * uC], tlo[3][uC * uC];   // T = (I + N)^-1, B [s][t]
    alignas(16) __nv_bfloat16 phi[3][uC * uC], plo[3][uC * uC];   // QX', B [s][t]
    alignas(16) __nv_bfloat16 ghi[3][2 * uC * uC], glo[3][2 * uC * uC];   // correction, B [j][n], N = 64
    alignas(16) float ob[2][uC][uD];              // o of a chunk (row warps -> staging warps)
    alignas(16) float cb[3][uC], cx[3][uC], cy[3][uC], cw[3][uC];  // per-token row constants
    alignas(16) float gam[3][4];                  // e^{cum_31} of the chunk
    alignas(16) float4 gts[2][uC];                // beta, e^{cum_t}, e^{cum_31 - cum_t} (by chunk parity)
    alignas(16) float cum[2][uC];
    alignas(16) float gamp[2][4];                 // e^{cum_31}, reference m, factored-exp flag
    alignas(16) float rk[uC], rq[uC], cumk[uC], fk[uC];
    alignas(16) float nT[uC][uNM];                // nT[t][s] = N[s][t]
    alignas(16) float tT[uC][20];                 // column t of the diagonal block of T holding t
    alignas(16) float tR[16][20];                 // T[0:16][0:16] row-major
    alignas(8) uint64_t bar_load[uSlots];         // a slot's copies landed
    alignas(8) uint64_t bar_tab, bar_d, bar_o, bar_pre;   // MMA groups completed
    alignas(8) uint64_t bar_g[3];                 // correction operand written (64 arrivals)
    alignas(8) uint64_t bar_gates[2];             // decay products of a chunk written (32)
    alignas(8) uint64_t bar_drain[2];             // final commits of the two MMA-issuing warps
    alignas(8) uint64_t bar_tabdone;              // table warp 1's MMAs drained
    uint32_t tmem_base;
    int abandon;                                  // a wait ran out twice: stop issuing work
};
static_assert(sizeof(U3Smem) + 1024 <= 227 * 1024, "shared memory");

// Named barriers.  FULL (three, by chunk % 3): row warps sync, table + staging warps arrive
// (chunk operands ready).
// EMPTY: row warps arrive, staging warps sync (o rows of a chunk written).  NORMS: staging
// arrive, table warps sync (the q norms are written; the staging warps have passed the chunk
// before, so the row warps are done with chunk ch-3 and its per-chunk buffers may be rewritten).  TDONE: table warps arrive, staging sync
// (table warps done with the previous chunk's shared buffers).  TBAR: rk and the factored
// exponentials from table warp 0 to table warp 1; TBAR2: the diagonal blocks of T likewise.
// TLD: both table warps have read the chunk tables out of tensor memory, so table warp 1 may
// issue the next chunk's table MMAs into the same columns.
enum {
    uBarFull0 = 1, uBarEmpty0 = 4, uBarRow = 6, uBarStg = 7, uBarT2 = 8, uBarNorms = 9,
    uBarTdone = 10, uBarT = 11, uBarTld = 12
};

__global__ void __launch_bounds__(uNT, 1)
gdn_scan_umma_kernel(const __grid_constant__ gdn_params p, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mv,
                     const __grid_constant__ CUtensorMap mz) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    U3Smem &sm = *reinterpret_cast<U3Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    using A = Act<__nv_bfloat16>;
    constexpr int D = uD;

    const int64_t head = blockIdx.x;                       // b * Hv + hv
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S;
    const int nchunks = (S + uC - 1) / uC;
    const bool gated = p.z != nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < uSlots; i++) mbar_init(&sm.bar_load[i], 1);
        mbar_init(&sm.bar_tab, 1);
        mbar_init(&sm.bar_d, 1);
        mbar_init(&sm.bar_o, 1);
        mbar_init(&sm.bar_pre, 1);
        for (int i = 0; i < 3; i++) mbar_init(&sm.bar_g[i], 64);
        mbar_init(&sm.bar_gates[0], 32);
        mbar_init(&sm.bar_gates[1], 32);
        mbar_init(&sm.bar_drain[0], 1);
        mbar_init(&sm.bar_drain[1], 1);
        mbar_init(&sm.bar_tabdone, 1);
        sm.abandon = 0;
        mbar_init_fence();
    }
    __syncwarp();
    if (warp == 0) tmem_alloc(&sm.tmem_base, TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t kq0 = smem_u32(&sm.kq[0][0]);
    // Bounded wait: if the wait runs out (the watchdog word is set) it is tried once more; if
    // that runs out too the CTA abandons its work: every later wait returns false at once, no
    // MMAs, copies or stores are issued, and what was issued is drained before tensor memory
    // is freed.
    volatile int *abandon = &sm.abandon;
    auto bwait = [&](uint64_t *bar, unsigned parity) -> bool {
        if (*abandon) return false;
        if (mbar_wait_bounded(bar, parity) || mbar_wait_bounded(bar, parity)) return true;
        *abandon = 1;
        return false;
    };
    // MMAs are issued by one elected lane of a converged warp
    bool issued = false;
    auto issue = [&](int by_warp, auto &&body) {
        if (warp == by_warp) {
            if (__all_sync(0xffffffffu, !*abandon)) {
                issued = true;
                if (elect_one()) body();
            }
            __syncwarp();
        }
    };
    // the MMAs this thread's warp issued have completed (bounded)
    auto drain = [&](int i) {
        if (issued) {
            if (elect_one()) {
                umma_commit(&sm.bar_drain[i]);
                mbar_wait_bounded(&sm.bar_drain[i], 0);
            }
            __syncwarp();
        }
    };
    auto kq_slot = [&](int c) { return kq0 + static_cast<uint32_t>(c % uSlots) * kSlotKQ; };
    auto load_parity = [&](int c) { return static_cast<unsigned>((c / uSlots) & 1); };
    // K-major descriptor of rows [K;Q] (or K alone) of a slot, k-step kk (16 features)
    auto kq_desc = [&](uint32_t slot, int kk) {
        return umma_desc(slot + (kk >> 2) * 2 * kBox + (kk & 3) * 32, 16, 1024, true);
    };
    // the chunk tables of chunk c: A = [K;Q]_c, B = K_{c-1} (c >= 1) and K_c
    auto issue_tables = [&](int c) {
        const uint32_t sc = kq_slot(c), sp = kq_slot(c + uSlots - 1);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
            const uint64_t a = kq_desc(sc, kk);
            if (c > 0) umma_ss(tmem + TM_TAB, a, kq_desc(sp, kk), kIdN32, kk > 0);
            umma_ss(tmem + TM_TAB + 32, a, kq_desc(sc, kk), kIdN32, kk > 0);
        }
        umma_commit(&sm.bar_tab);
    };

    if (warp < uRowW) {
        // ================================ row warps =======================================
        // Warps w and w + 4 share lane quarter w & 3 (memory rows 32 (w & 3) + lane); half hr
        // takes S' columns [64 hr, 64 hr + 64) and tokens [16 hr, 16 hr + 16) of each chunk.
        const int quarter = warp & 3, hr = warp >> 2;
        const int row = 32 * quarter + lane;               // memory row = tensor-memory lane
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        // [x | y] of chunk c from the current S' hi / lo into buffer c & 1
        auto issue_pre = [&](int c) {
            const uint32_t sc = kq_slot(c), xy = tmem + TM_XY + 64 * (c & 1);
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                const uint64_t bkq = kq_desc(sc, kk);
                umma_ts(xy, tmem + TM_SLO + 8 * kk, bkq, kIdN64, kk > 0);
                umma_ts(xy, tmem + TM_SHI + 8 * kk, bkq, kIdN64, true);
            }
        };
        // S' -> bf16 hi / lo (this thread's 64 columns)
        auto split_s = [&]() {
            float v[64];
            tm_ld64(tl + TM_S + 64 * hr, v);
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int j = 0; j < 32; j++) split2(v[2 * j], v[2 * j + 1], hi[j], lo[j]);
            tm_st32(tl + TM_SHI + 32 * hr, hi);
            tm_st32(tl + TM_SLO + 32 * hr, lo);
        };
        auto wait_mma = [&](uint64_t *bar, unsigned parity) {
            __syncwarp();
            bwait(bar, parity);
            __syncwarp();
            tc_fence_after();
        };
        auto row_barrier = [&]() {                          // tensor-memory stores -> MMA issue
            tm_wait_st();
            tc_fence_before();
            bar_sync(uBarRow, uRT);
        };

        {
            const float *s0 = p.s0 ? p.s0 + head * (D * D) + static_cast<int64_t>(row) * D + 64 * hr
                                   : nullptr;
#pragma unroll
            for (int i = 0; i < 2; i++) {
                float v[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; j4++) {
                    const float4 f = s0 ? *reinterpret_cast<const float4 *>(s0 + 32 * i + 4 * j4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[4 * j4] = f.x; v[4 * j4 + 1] = f.y; v[4 * j4 + 2] = f.z; v[4 * j4 + 3] = f.w;
                }
                tm_st32f(tl + TM_S + 64 * hr + 32 * i, v);
            }
            tm_wait_st();
        }
        split_s();
        row_barrier();
        issue(0, [&] {                                     // tables and [x | y] of chunk 0
            bwait(&sm.bar_load[0], 0);
            tc_fence_after();
            issue_tables(0);
            issue_pre(0);
            umma_commit(&sm.bar_o);                        // phase 0
        });
        wait_mma(&sm.bar_o, 0);

        float lam = 1.0f;                                  // true memory = lam * S'
        for (int ch = 0; ch < nchunks; ch++) {
            const int hb = ch & 1, tb = ch % 3, slot = ch % uSlots;
            const int nt = min(uC, S - ch * uC);
            const bool more = ch + 1 < nchunks;
            const uint32_t xy = TM_XY + 64 * hb, xyn = TM_XY + 64 * (hb ^ 1);
            bar_sync(uBarFull0 + tb, uNT);                 // chunk ch's operands staged

            // ---- r = beta (v - lam e^cum rk x) (0 past the end); y <- lam e^cum rq y in place
            {                                              // tokens t0r .. t0r + 15
                const int t0r = 16 * hr;
                float xv[16], yv[16];
                tm_ld16(tl + xy + t0r, xv);
                tm_ld16(tl + xy + 32 + t0r, yv);
                uint32_t rh[8], rl[8];
                float ys[16];
#pragma unroll
                for (int t4 = 0; t4 < 4; t4++) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(&sm.cb[tb][t0r + 4 * t4]);
                    const float4 x4 = *reinterpret_cast<const float4 *>(&sm.cx[tb][t0r + 4 * t4]);
                    const float4 y4 = *reinterpret_cast<const float4 *>(&sm.cy[tb][t0r + 4 * t4]);
                    const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
                    const float bx[4] = {x4.x, x4.y, x4.z, x4.w};
                    const float by[4] = {y4.x, y4.y, y4.z, y4.w};
                    float rr[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int j = 4 * t4 + e, t = t0r + j;
                        const float vv = A::one(&sm.v[slot][t][row]);
                        rr[e] = (t < nt) ? bb[e] * fmaf(-lam * bx[e], xv[j], vv) : 0.f;
                        ys[j] = lam * by[e] * yv[j];
                    }
                    split2(rr[0], rr[1], rh[2 * t4], rl[2 * t4]);
                    split2(rr[2], rr[3], rh[2 * t4 + 1], rl[2 * t4 + 1]);
                }
                tm_st8(tl + TM_RH + 8 * hr, rh);
                tm_st8(tl + TM_RL + 8 * hr, rl);
                uint32_t yu[16];
#pragma unroll
                for (int j = 0; j < 16; j++) yu[j] = __float_as_uint(ys[j]);
                tm_st16(tl + xy + 32 + t0r, yu);
            }
            row_barrier();
            issue(0, [&] {                                 // d = R T into x's columns
                tc_fence_after();
                const uint32_t th = smem_u32(&sm.thi[tb][0]), tlw = smem_u32(&sm.tlo[tb][0]);
#pragma unroll
                for (int k2 = 0; k2 < 2; k2++) {
                    const uint64_t bh = umma_desc(th + 256 * k2, 128, 512, false);
                    const uint64_t bl = umma_desc(tlw + 256 * k2, 128, 512, false);
                    umma_ts(tmem + xy, tmem + TM_RL + 8 * k2, bh, kIdN32, k2 > 0);
                    umma_ts(tmem + xy, tmem + TM_RH + 8 * k2, bl, kIdN32, true);
                    umma_ts(tmem + xy, tmem + TM_RH + 8 * k2, bh, kIdN32, true);
                }
                umma_commit(&sm.bar_d);
            });

            // ---- while d runs: S' hi / lo for the next chunk's [x | y] (S' holds S'_ch)
            if (more) {
                split_s();
                row_barrier();
                issue(0, [&] {
                    bwait(&sm.bar_load[(ch + 1) % uSlots], load_parity(ch + 1));
                    tc_fence_after();
                    issue_pre(ch + 1);
                    umma_commit(&sm.bar_pre);
                });
            }
            wait_mma(&sm.bar_d, static_cast<unsigned>(ch & 1));

            // ---- d -> bf16 hi / lo (A of O); C = d W rk / lam' -> hi / lo (A of the update)
            const float lam_new = lam * sm.gam[tb][0];
            const bool fold = !(lam_new >= 0x1p-40f);      // uniform over the CTA
            const float scale = fold ? 1.0f : 1.0f / lam_new;
            {                                              // tokens 16 hr .. 16 hr + 15
                float d[16];
                tm_ld16(tl + xy + 16 * hr, d);
                uint32_t dh[8], dl[8], chh[8], cll[8];
#pragma unroll
                for (int t4 = 0; t4 < 4; t4++) {
                    const float4 w4 = *reinterpret_cast<const float4 *>(&sm.cw[tb][16 * hr + 4 * t4]);
                    const float ww[4] = {w4.x * scale, w4.y * scale, w4.z * scale, w4.w * scale};
#pragma unroll
                    for (int e2 = 0; e2 < 2; e2++) {
                        const int t = 4 * t4 + 2 * e2, j = 2 * t4 + e2;
                        split2(d[t], d[t + 1], dh[j], dl[j]);
                        split2(d[t] * ww[2 * e2], d[t + 1] * ww[2 * e2 + 1], chh[j], cll[j]);
                    }
                }
                tm_st8(tl + TM_DH + 8 * hr, dh);
                tm_st8(tl + TM_DL + 8 * hr, dl);
                tm_st8(tl + TM_CH + 8 * hr, chh);
                tm_st8(tl + TM_CL + 8 * hr, cll);
            }
            if (fold) {                                    // S' <- lam' S', next [x | y] too
                {
                    float v[64];
                    tm_ld64(tl + TM_S + 64 * hr, v);
                    float a[32], c[32];
#pragma unroll
                    for (int j = 0; j < 32; j++) { a[j] = v[j] * lam_new; c[j] = v[32 + j] * lam_new; }
                    tm_st32f(tl + TM_S + 64 * hr, a);
                    tm_st32f(tl + TM_S + 64 * hr + 32, c);
                }
                if (more) {
                    wait_mma(&sm.bar_pre, static_cast<unsigned>(ch & 1));
                    float v[32];
                    tm_ld32(tl + xyn + 32 * hr, v);
#pragma unroll
                    for (int j = 0; j < 32; j++) v[j] *= lam_new;
                    tm_st32f(tl + xyn + 32 * hr, v);
                }
            }
            row_barrier();
            issue(0, [&] {
                tc_fence_after();
                const uint32_t ph_ = smem_u32(&sm.phi[tb][0]), pl_ = smem_u32(&sm.plo[tb][0]);
#pragma unroll
                for (int k2 = 0; k2 < 2; k2++) {           // o += D QX' (onto the scaled y)
                    const uint64_t bh = umma_desc(ph_ + 256 * k2, 128, 512, false);
                    const uint64_t bl = umma_desc(pl_ + 256 * k2, 128, 512, false);
                    umma_ts(tmem + xy + 32, tmem + TM_DL + 8 * k2, bh, kIdN32, true);
                    umma_ts(tmem + xy + 32, tmem + TM_DH + 8 * k2, bl, kIdN32, true);
                    umma_ts(tmem + xy + 32, tmem + TM_DH + 8 * k2, bh, kIdN32, true);
                }
                const uint32_t ks = kq_slot(ch);
#pragma unroll
                for (int k2 = 0; k2 < 2; k2++) {           // S' += C K (K read MN-major)
                    const uint64_t bk = umma_desc(ks + 2048 * k2, 2 * kBox, 1024, true);
                    umma_ts(tmem + TM_S, tmem + TM_CL + 8 * k2, bk, kIdN128Mn, true);
                    umma_ts(tmem + TM_S, tmem + TM_CH + 8 * k2, bk, kIdN128Mn, true);
                }
                if (more) {                                // next [x | y] += C (K_ch [K;Q]_{ch+1}^T)
                    const int gb = (ch + 1) % 3;           // prep ch+1 wrote it, use (ch) / 3 of gb
                    bwait(&sm.bar_g[gb], static_cast<unsigned>((ch / 3) & 1));
                    tc_fence_after();
                    const uint32_t gh = smem_u32(&sm.ghi[gb][0]), gl = smem_u32(&sm.glo[gb][0]);
#pragma unroll
                    for (int k2 = 0; k2 < 2; k2++) {
                        const uint64_t bh = umma_desc(gh + 256 * k2, 128, 512, false);
                        const uint64_t bl = umma_desc(gl + 256 * k2, 128, 512, false);
                        umma_ts(tmem + xyn, tmem + TM_CL + 8 * k2, bh, kIdN64, true);
                        umma_ts(tmem + xyn, tmem + TM_CH + 8 * k2, bl, kIdN64, true);
                        umma_ts(tmem + xyn, tmem + TM_CH + 8 * k2, bh, kIdN64, true);
                    }
                }
                umma_commit(&sm.bar_o);                    // phase ch + 1
            });
            wait_mma(&sm.bar_o, static_cast<unsigned>((ch + 1) & 1));
            {
                float o[16];
                tm_ld16(tl + xy + 32 + 16 * hr, o);
#pragma unroll
                for (int j = 0; j < 16; j++)
                    if (16 * hr + j < nt) sm.ob[hb][16 * hr + j][row] = o[j];
            }
            bar_arrive(uBarEmpty0 + hb, uRT + uST);        // o rows of chunk ch written
            lam = fold ? 1.0f : lam_new;
        }
        // final memory rows (undo the deferred decay)
        float *so = p.state + head * (D * D) + static_cast<int64_t>(row) * D + 64 * hr;
        {
            float v[64];
            tm_ld64(tl + TM_S + 64 * hr, v);
            if (!*abandon) {                               // no stores once abandoned
#pragma unroll
                for (int j4 = 0; j4 < 16; j4++)
                    *reinterpret_cast<float4 *>(so + 4 * j4) =
                        make_float4(lam * v[4 * j4], lam * v[4 * j4 + 1], lam * v[4 * j4 + 2], lam * v[4 * j4 + 3]);
            }
        }
        drain(0);                                          // warp 0's MMAs
        tc_fence_before();
        bar_sync(uBarRow, uRT);
        if (warp == 0) {
            // table warp 1's MMAs too (they are all consumed already unless the CTA abandoned)
            if (lane == 0) mbar_wait_bounded(&sm.bar_tabdone, 0);
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem, TM_COLS);
        }
        return;
    }

    if (warp < uStgW0) {
        // ================================ table warps =====================================
        // Lane t of table warp tq owns token column t of chunk ch: warp 0 (lane quarter 0) the
        // k rows, warp 1 (quarter 1) the q rows of the table product.
        const int tq = warp - uTabW0;
        const int t = lane;
        const uint32_t tabl = tmem + (static_cast<uint32_t>(32 * tq) << 16) + TM_TAB;
        for (int ch = 0; ch < nchunks; ch++) {
            const int hb = ch & 1, tb = ch % 3;
            const int nt = min(uC, S - ch * uC);
            bwait(&sm.bar_tab, static_cast<unsigned>(ch & 1));
            __syncwarp();
            tc_fence_after();
            float tab[64];                                 // [cross (K_{ch-1}) | own chunk]
            tm_ld64(tabl, tab);
            tc_fence_before();
            bar_sync(uBarTld, 64);                         // both table warps hold the tables
            if (ch + 1 < nchunks) {                        // the next chunk's tables, early
                issue(uTabW0 + 1, [&] {
                    tc_fence_after();
                    bwait(&sm.bar_load[ch % uSlots], load_parity(ch));
                    bwait(&sm.bar_load[(ch + 1) % uSlots], load_parity(ch + 1));
                    issue_tables(ch + 1);
                });
            }
            if (ch > 0) {                                  // correction operand, column n
                const int n = 32 * tq + t;
                char *gh = reinterpret_cast<char *>(&sm.ghi[tb][0]);
                char *gl = reinterpret_cast<char *>(&sm.glo[tb][0]);
#pragma unroll
                for (int kg = 0; kg < 4; kg++) {
                    uint32_t h4[4], l4[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) split2(tab[8 * kg + 2 * i], tab[8 * kg + 2 * i + 1], h4[i], l4[i]);
                    *reinterpret_cast<uint4 *>(gh + core_run(n, kg)) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                    *reinterpret_cast<uint4 *>(gl + core_run(n, kg)) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(&sm.bar_g[tb]);
            }
            bwait(&sm.bar_gates[hb], static_cast<unsigned>((ch >> 1) & 1));
            __syncwarp();
            const float4 gt = sm.gts[hb][t];               // beta, e^cum, e^{cum_31 - cum}
            const float cum_t = sm.cum[hb][t];
            const float mref = sm.gamp[hb][1];
            const bool factored = sm.gamp[hb][2] != 0.f;   // e^{cum_t - m}, e^{m - cum_s} finite
            if (tq == 0) {
                // rk from the diagonal of K K^T
                float dg = 0.f;
#pragma unroll
                for (int j = 0; j < uC; j++) dg = (j == t) ? tab[32 + j] : dg;
                const float rk_t = (t < nt) ? rsqrtf(dg + p.qk_eps) : 0.f;
                sm.rk[t] = rk_t;
                sm.cumk[t] = cum_t;
                sm.fk[t] = factored ? rk_t * __expf(mref - cum_t) : 0.f;
                __syncwarp();
                bar_arrive(uBarT, 64);                     // rk, fk ready for the q-row warp
                // N column t: N[s][t] = beta_t e^{cum_t - cum_s} rk_s rk_t (k_s . k_t), s < t
                float col[uC];
                if (factored) {
                    const float g = gt.x * rk_t * __expf(cum_t - mref);
#pragma unroll
                    for (int s4 = 0; s4 < uC / 4; s4++) {
                        const float4 f4 = *reinterpret_cast<const float4 *>(&sm.fk[4 * s4]);
                        const float ff[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int s_ = 4 * s4 + e;
                            col[s_] = ((s_ < t) ? g : 0.f) * ff[e] * tab[32 + s_];
                        }
                    }
                } else {
                    const float bt = gt.x * rk_t;
#pragma unroll
                    for (int s4 = 0; s4 < uC / 4; s4++) {
                        const float4 r4 = *reinterpret_cast<const float4 *>(&sm.rk[4 * s4]);
                        const float4 c4 = *reinterpret_cast<const float4 *>(&sm.cumk[4 * s4]);
                        const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int s_ = 4 * s4 + e;
                            const float m = (s_ < t) ? bt : 0.f;   // exp argument <= 0: finite
                            col[s_] = m * __expf(fminf(cum_t - cc[e], 0.f)) * rr[e] * tab[32 + s_];
                        }
                    }
                }
#pragma unroll
                for (int s4 = 0; s4 < uC / 4; s4++)
                    *reinterpret_cast<float4 *>(&sm.nT[t][4 * s4]) =
                        make_float4(col[4 * s4], col[4 * s4 + 1], col[4 * s4 + 2], col[4 * s4 + 3]);
                __syncwarp();
                // The diagonal 16 x 16 blocks of T = (I + N)^-1 (block upper triangular: T11 =
                // (I + N11)^-1, T22 = (I + N22)^-1, T12 = -T11 N12 T22).  Lane t solves column t
                // of its block by back substitution, T[r][t] = -sum_{r < r' <= t} N[r][r'] T[r'][t].
                const int base = t & 16, tl = t & 15;
                float acc[16], colb[16];
#pragma unroll
                for (int j = 0; j < 16; j++) acc[j] = 0.f;
#pragma unroll
                for (int rr = 15; rr >= 0; rr--) {
                    const float tr = (rr == tl) ? 1.f : ((rr < tl) ? -acc[rr] : 0.f);
                    colb[rr] = tr;
                    if (rr > 0) {
                        const float *nrow = &sm.nT[base + rr][base];
#pragma unroll
                        for (int s4 = 0; s4 < (rr + 3) / 4; s4++) {
                            const float4 n4 = *reinterpret_cast<const float4 *>(nrow + 4 * s4);
                            const float nn[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
                            for (int e = 0; e < 4; e++)
                                if (4 * s4 + e < rr) acc[4 * s4 + e] = fmaf(nn[e], tr, acc[4 * s4 + e]);
                        }
                    }
                }
#pragma unroll
                for (int j4 = 0; j4 < 4; j4++)
                    *reinterpret_cast<float4 *>(&sm.tT[t][4 * j4]) =
                        make_float4(colb[4 * j4], colb[4 * j4 + 1], colb[4 * j4 + 2], colb[4 * j4 + 3]);
                if (t < 16) {
#pragma unroll
                    for (int j = 0; j < 16; j++) sm.tR[j][t] = colb[j];
                }
                __syncwarp();
                bar_arrive(uBarT2, 64);                    // diagonal blocks ready
                bar_sync(uBarNorms, 64 + uST);             // row warps done with chunk ch-3
                // column t of T as B [s][t]: rows of the lane's diagonal block; zeros below
                // the diagonal block for t < 16 (rows 16-31 of T11's columns)
                char *dh = reinterpret_cast<char *>(&sm.thi[tb][0]);
                char *dl = reinterpret_cast<char *>(&sm.tlo[tb][0]);
#pragma unroll
                for (int kk = 0; kk < 2; kk++) {
                    uint32_t h4[4], l4[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) split2(colb[8 * kk + 2 * i], colb[8 * kk + 2 * i + 1], h4[i], l4[i]);
                    const int kg = (base >> 3) + kk;
                    *reinterpret_cast<uint4 *>(dh + core_run(t, kg)) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                    *reinterpret_cast<uint4 *>(dl + core_run(t, kg)) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
                }
                if (t < 16) {
#pragma unroll
                    for (int kg = 2; kg < 4; kg++) {
                        *reinterpret_cast<uint4 *>(dh + core_run(t, kg)) = make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(dl + core_run(t, kg)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            } else {
                bar_sync(uBarNorms, 64 + uST);             // rq of chunk ch
                bar_sync(uBarT, 64);                       // rk, fk of chunk ch
                const float rq_t = sm.rq[t], rk_own = sm.rk[t];
                // QX' column t: e^{cum_t - cum_s} rk_s rq_t (k_s . q_t), s <= t
                float col[uC];
                if (factored) {
                    const float h = rq_t * __expf(cum_t - mref);
#pragma unroll
                    for (int s4 = 0; s4 < uC / 4; s4++) {
                        const float4 f4 = *reinterpret_cast<const float4 *>(&sm.fk[4 * s4]);
                        const float ff[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int s_ = 4 * s4 + e;
                            col[s_] = ((s_ <= t) ? h : 0.f) * ff[e] * tab[32 + s_];
                        }
                    }
                } else {
#pragma unroll
                    for (int s4 = 0; s4 < uC / 4; s4++) {
                        const float4 r4 = *reinterpret_cast<const float4 *>(&sm.rk[4 * s4]);
                        const float4 c4 = *reinterpret_cast<const float4 *>(&sm.cumk[4 * s4]);
                        const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int s_ = 4 * s4 + e;
                            const float m = (s_ <= t) ? rq_t : 0.f;
                            col[s_] = m * __expf(fminf(cum_t - cc[e], 0.f)) * rr[e] * tab[32 + s_];
                        }
                    }
                }
                sm.cb[tb][t] = gt.x;
                sm.cx[tb][t] = gt.y * rk_own;
                sm.cy[tb][t] = gt.y * rq_t;
                sm.cw[tb][t] = gt.z * rk_own;
                if (t == 0) sm.gam[tb][0] = sm.gamp[hb][0];
                char *ph_ = reinterpret_cast<char *>(&sm.phi[tb][0]);
                char *pl_ = reinterpret_cast<char *>(&sm.plo[tb][0]);
#pragma unroll
                for (int kg = 0; kg < 4; kg++) {           // column t as B [s][t], hi / lo
                    uint32_t h4[4], l4[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) split2(col[8 * kg + 2 * i], col[8 * kg + 2 * i + 1], h4[i], l4[i]);
                    *reinterpret_cast<uint4 *>(ph_ + core_run(t, kg)) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                    *reinterpret_cast<uint4 *>(pl_ + core_run(t, kg)) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
                }
                // T12 = -T11 N12 T22: lane -> column tc = 16 + (lane & 15), rows 8 hf .. 8 hf + 7
                bar_sync(uBarT2, 64);
                const int tc = 16 + (t & 15), hf = t >> 4;
                float u[16];                               // u = N12 T22[:, tc]
#pragma unroll
                for (int e = 0; e < 8; e++) u[e] = 0.f;
#pragma unroll
                for (int j4 = 0; j4 < 4; j4++) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(&sm.tT[tc][4 * j4]);
                    const float tj[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                    for (int jj = 0; jj < 4; jj++) {
                        const float *nrow = &sm.nT[16 + 4 * j4 + jj][8 * hf];
                        const float4 a4 = *reinterpret_cast<const float4 *>(nrow);
                        const float4 b4 = *reinterpret_cast<const float4 *>(nrow + 4);
                        const float nn[8] = {a4.x, a4.y, a4.z, a4.w, b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                        for (int e = 0; e < 8; e++) u[e] = fmaf(nn[e], tj[jj], u[e]);
                    }
                }
                // u[0:8] holds rows 8 hf .. 8 hf + 7; the partner lane (t ^ 16) holds the others
                float uo[8];
#pragma unroll
                for (int e = 0; e < 8; e++) uo[e] = __shfl_xor_sync(0xffffffffu, u[e], 16);
                float uf[16];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    uf[e] = hf ? uo[e] : u[e];
                    uf[8 + e] = hf ? u[e] : uo[e];
                }
                float t12[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int srow = 8 * hf + e;
                    float a = 0.f;
#pragma unroll
                    for (int r4 = 0; r4 < 4; r4++) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(&sm.tR[srow][4 * r4]);
                        a = fmaf(w4.x, uf[4 * r4], a);
                        a = fmaf(w4.y, uf[4 * r4 + 1], a);
                        a = fmaf(w4.z, uf[4 * r4 + 2], a);
                        a = fmaf(w4.w, uf[4 * r4 + 3], a);
                    }
                    t12[e] = -a;
                }
                uint32_t h4[4], l4[4];
#pragma unroll
                for (int i = 0; i < 4; i++) split2(t12[2 * i], t12[2 * i + 1], h4[i], l4[i]);
                *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(&sm.thi[tb][0]) + core_run(tc, hf)) =
                    make_uint4(h4[0], h4[1], h4[2], h4[3]);
                *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(&sm.tlo[tb][0]) + core_run(tc, hf)) =
                    make_uint4(l4[0], l4[1], l4[2], l4[3]);
            }
            fence_proxy_async_smem();                      // operands for the tensor core
            if (ch + 1 < nchunks) bar_arrive(uBarTdone, 64 + uST);
            bar_arrive(uBarFull0 + tb, uNT);
        }
        if (warp == uTabW0 + 1) {                          // this warp's table MMAs drained
            drain(1);
            if (lane == 0) mbar_arrive(&sm.bar_tabdone);
            __syncwarp();
        }
        return;
    }

    // ================================ staging warps =======================================
    const int sw = warp - uStgW0;                          // 0 .. 5
    const int stid = threadIdx.x - 32 * uStgW0;            // 0 .. 191
    const unsigned chunk_bytes = (gated ? 4u : 3u) * uC * uD * 2u;   // k, q, v (, z)
    int64_t v_base, v_ts, g_base, g_ts;
    if (p.head_major) {
        v_base = head * S * D;  v_ts = D;
        g_base = head * S;      g_ts = 1;
    } else {
        v_base = (static_cast<int64_t>(b) * S * p.Hv + hv) * D;  v_ts = static_cast<int64_t>(p.Hv) * D;
        g_base = static_cast<int64_t>(b) * S * p.Hv + hv;        g_ts = p.Hv;
    }

    // tensor-map copies of chunk c into slot c % uSlots (one thread); rows past the end read 0
    int last_issued[uSlots] = {-1, -1, -1, -1};           // per slot (thread stid == 0)
    auto issue_chunk = [&](int c) {
        if (*abandon) return;
        const int slot = c % uSlots, t0 = c * uC;
        last_issued[slot] = c;
        uint64_t *bar = &sm.bar_load[slot];
        char *kqs = reinterpret_cast<char *>(&sm.kq[slot][0]);
        mbar_arrive_expect_tx(bar, chunk_bytes);
        for (int half = 0; half < 2; half++) {
            tma_load_4d(kqs + half * 2 * kBox, &mk, 64 * half, hk, t0, b, bar);
            tma_load_4d(kqs + half * 2 * kBox + kBox, &mq, 64 * half, hk, t0, b, bar);
        }
        tma_load_4d(&sm.v[slot][0][0], &mv, 0, hv, t0, b, bar);
        if (gated) tma_load_4d(&sm.z[slot][0][0], &mz, 0, hv, t0, b, bar);
    };

    // y of a finished chunk: 8 lanes per token (4 tokens per warp pass), lane part q holds
    // the float4 column groups q + 8 i; gated RMSNorm or the raw o rows
    const int eq = lane & 7;
    float4 gn4[4];
#pragma unroll
    for (int i = 0; i < 4; i++)
        gn4[i] = gated ? *reinterpret_cast<const float4 *>(p.gn + 4 * (eq + 8 * i))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    const float inv_d = 1.0f / static_cast<float>(D);
    auto emit = [&](int c) {
        if (*abandon) return;                              // no stores once abandoned
        const int hb = c & 1, slot = c % uSlots;
        const int t0 = c * uC, nt = min(uC, S - t0);
        for (int base = 4 * sw; base < nt; base += 4 * uStgW) {
            const int tt = base + (lane >> 3);
            const bool valid = tt < nt;
            const int tr = valid ? tt : base;              // rows past the end: any valid row
            float4 *yr = reinterpret_cast<float4 *>(p.y + v_base + (t0 + tr) * v_ts);
            if (gated) {
                float4 x[4];
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int c4 = eq + 8 * i;
                    const float4 o4 = *reinterpret_cast<const float4 *>(&sm.ob[hb][tr][4 * c4]);
                    const float4 z4 = A::four(&sm.z[slot][tr][4 * c4]);
                    x[i] = make_float4(o4.x * silu_fast(z4.x), o4.y * silu_fast(z4.y),
                                       o4.z * silu_fast(z4.z), o4.w * silu_fast(z4.w));
                    ss = fmaf(x[i].x, x[i].x, fmaf(x[i].y, x[i].y, fmaf(x[i].z, x[i].z, fmaf(x[i].w, x[i].w, ss))));
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                const float rr = rsqrtf(fmaf(ss, inv_d, p.norm_eps));
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        yr[eq + 8 * i] = make_float4(x[i].x * rr * gn4[i].x, x[i].y * rr * gn4[i].y,
                                                     x[i].z * rr * gn4[i].z, x[i].w * rr * gn4[i].w);
                }
            } else if (valid) {
#pragma unroll
                for (int i = 0; i < 4; i++)
                    yr[eq + 8 * i] = *reinterpret_cast<const float4 *>(&sm.ob[hb][tr][4 * (eq + 8 * i)]);
            }
        }
    };

    // decay products of chunk c (the gate warp, one lane per token)
    float gl = 0.f, gbv = 0.f;
    auto load_gates = [&](int c) {
        const int t = c * uC + lane;
        if (t < S) {
            const int64_t gi = g_base + static_cast<int64_t>(t) * g_ts;
            gl = load_gate(p.log_decay, p.gate_dtype, gi);
            gbv = load_gate(p.beta, p.gate_dtype, gi);
        }
    };
    // Written into the buffer of the chunk's parity, announced on bar_gates[parity]; also the
    // reference m = mid-range of cum and whether every e^{+-(cum - m)} stays finite (range <= 120),
    // so the table warps may factor e^{cum_t - cum_s} = e^{cum_t - m} e^{m - cum_s}.
    auto decay_products = [&](int c) {
        const int gb = c & 1;
        const bool valid = c * uC + lane < S;
        const float gc = valid ? fmaxf(gl, uMinLogDecay) : 0.f;
        float upto = gc;                                   // chunk-inclusive prefix sum
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, upto, off);
            if (lane >= off) upto += o;
        }
        const float total = __shfl_sync(0xffffffffu, upto, 31);
        float hi = upto, lo = upto;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        }
        sm.gts[gb][lane] = make_float4(valid ? gbv : 0.f, expf(upto), expf(total - upto), 0.f);
        sm.cum[gb][lane] = upto;
        if (lane == 0) {
            sm.gamp[gb][0] = expf(total);
            sm.gamp[gb][1] = 0.5f * (hi + lo);
            sm.gamp[gb][2] = (hi - lo <= 120.f) ? 1.f : 0.f;
        }
        __syncwarp();
        mbar_arrive(&sm.bar_gates[gb]);
    };

    const float inv_sqrt_dk = rsqrtf(static_cast<float>(D));
    if (sw == uGateW) {                                    // chunk 0's decay products
        load_gates(0);
        decay_products(0);
        if (nchunks > 1) load_gates(1);
    }
    if (stid == 0) {
        issue_chunk(0);
        if (nchunks > 1) issue_chunk(1);
    }
    for (int ch = 0; ch < nchunks; ch++) {
        const int hb = ch & 1, slot = ch % uSlots;
        const int nt = min(uC, S - ch * uC);
        if (ch > 0) bar_sync(uBarTdone, 64 + uST);         // table warps done with chunk ch-1
        if (sw == uGateW && ch + 1 < nchunks) {            // one chunk ahead: the buffer of
            decay_products(ch + 1);                        // parity ch+1 was last read in ch-1
            if (ch + 2 < nchunks) load_gates(ch + 2);
        }
        // q norms of chunk ch (warps 0-3: token 8 w + lane % 8, pieces lane / 8 + 4 i)
        if (sw < 4) {
            bwait(&sm.bar_load[slot], load_parity(ch));
            const int tok = sw * 8 + (lane & 7), nq = lane >> 3;
            const char *kqs = reinterpret_cast<const char *>(&sm.kq[slot][0]);
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                float x[8];
                unpack8(*reinterpret_cast<const uint4 *>(kqs + q_piece(tok, nq + 4 * i)), x);
#pragma unroll
                for (int e = 0; e < 8; e++) ss = fmaf(x[e], x[e], ss);
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            ss += __shfl_xor_sync(0xffffffffu, ss, 16);
            if (nq == 0) sm.rq[tok] = (tok < nt) ? rsqrtf(ss + p.qk_eps) * inv_sqrt_dk : 0.f;
        }
        // the table warps may now write chunk ch's operands: this point comes after the EMPTY
        // wait of the chunk before, so the row warps are done with chunk ch-3
        bar_arrive(uBarNorms, 64 + uST);
        if (ch >= 2) {                                     // chunk ch-2's o rows are written
            bar_sync(uBarEmpty0 + hb, uRT + uST);
            emit(ch - 2);
        }
        bar_sync(uBarStg, uST);                            // its z slot is read: refill it
        if (stid == 0 && ch + 2 < nchunks) issue_chunk(ch + 2);
        bar_arrive(uBarFull0 + ch % 3, uNT);
    }
    for (int ch = max(0, nchunks - 2); ch < nchunks; ch++) {
        bar_sync(uBarEmpty0 + (ch & 1), uRT + uST);
        emit(ch);
    }
    // the copies this thread issued have landed (all consumed already unless the CTA abandoned)
    if (stid == 0) {
        for (int sl = 0; sl < uSlots; sl++)
            if (last_issued[sl] >= 0) mbar_wait_bounded(&sm.bar_load[sl], load_parity(last_issued[sl]));
    }
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// A [B, S, H, W] or [B, H, S, W] bf16 tensor seen with coordinates (w, h, t, b); box of
// `box_w` x 1 x 32 x 1.
bool encode_map(CUtensorMap *m, const void *base, const gdn_params &p, int H, int box_w,
                bool swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t W = uD, S = p.S, B = p.B;
    cuuint64_t dims[4] = {W, static_cast<cuuint64_t>(H), S, B};
    cuuint64_t strides[3];
    if (p.head_major) {
        strides[0] = S * W * 2;                            // h
        strides[1] = W * 2;                                // t
    } else {
        strides[0] = W * 2;                                // h
        strides[1] = static_cast<cuuint64_t>(H) * W * 2;   // t
    }
    strides[2] = static_cast<cuuint64_t>(H) * S * W * 2;   // b
    cuuint32_t box[4] = {static_cast<cuuint32_t>(box_w), 1, static_cast<cuuint32_t>(uC), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool scan_umma_supported(const gdn_params &p) {
    auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    return p.act_dtype == GDN_BF16 && p.Dk == uD && p.Dv == uD && p.S > 0 && p.B > 0 &&
           al16(p.q) && al16(p.k) && al16(p.v) &&
           (p.z == nullptr || al16(p.z)) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_scan_umma(const gdn_params &p, cudaStream_t stream) {
    CUtensorMap mk, mq, mv, mz;
    if (!encode_map(&mk, p.k, p, p.Hk, 64, true) || !encode_map(&mq, p.q, p, p.Hk, 64, true) ||
        !encode_map(&mv, p.v, p, p.Hv, uD, false))
        return cudaErrorInvalidValue;
    if (p.z) {
        if (!encode_map(&mz, p.z, p, p.Hv, uD, false)) return cudaErrorInvalidValue;
    } else {
        mz = mv;                                           // unused
    }
    const int bytes = static_cast<int>(sizeof(U3Smem)) + 1024;
    cudaError_t e = cudaFuncSetAttribute(gdn_scan_umma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int64_t ctas = static_cast<int64_t>(p.B) * p.Hv;
    gdn_scan_umma_kernel<<<static_cast<unsigned>(ctas), uNT, bytes, stream>>>(p, mk, mq, mv, mz);
    return cudaGetLastError();
}

cudaError_t scan_umma_watchdog(unsigned *flag, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_watchdog, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
    const unsigned zero = 0;
    if (*flag) e = cudaMemcpyToSymbolAsync(g_watchdog, &zero, sizeof(unsigned), 0,
                                           cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e;
}

}  // namespace gdn
