// gdn_scan_wy.cu -- multi-token GDN recurrence in chunked (WY) form on tcgen05 tensor cores.
//
// What is computed is the page's per-token recurrence (logicaffeine_compile::codegen_cuda::gdn,
// module description; the time loop of torch_to_nnef.op.gated_delta, gated_delta_reference):
//     S_t = alpha_t S_{t-1} + d_t k^_t^T,   d_t = beta_t (v_t - alpha_t S_{t-1} k^_t),   o_t = S_t q^_t.
// The update is affine in the memory ("The fusion" section of the same page expands o the
// same way), so over a chunk of C = 64 tokens starting from memory S, with G_t the chunk's
// cumulative decay (exp of a running sum of log_decay, clamped at -80 per token), raw k, q and
// their l2 norms as per-token scalars rk, rq (rq carries 1/sqrt(Dk)):
//     A[t][s] = beta_t (G_t / G_s) rk_t rk_s (k_t . k_s)   (s < t),     T = (I + A)^-1,
//     D = U - W S^T,    U = T diag(beta) V,    W = T diag(beta G rk) K,
//     o_t = G_t rq_t (S q_t) + sum_{s <= t} (G_t / G_s) rk_s rq_t (k_s . q_t) d_s,
//     S  <- G_63 S + sum_s rk_s (G_63 / G_s) d_s k_s^T.
// Every decay factor is exp of a non-positive sum, so nothing overflows; every step is exact
// algebra, and the result differs from the sequential loop only by rounding.
//
// GB300 mapping (bf16 or f16 activations, Dk = Dv = 128, one CTA per (b, hv) head):
//   * tensor memory (512 columns) holds the f32 memory S (lanes = memory rows a), its hi part
//     as the A operand of [X | Y], X^T = U^T - S W^T (the corrections d of the chunk, one column
//     per token), Y^T = S Q^T scaled per token and accumulated with the intra-chunk term into
//     o, the corrections as A operands of the update and of the intra-chunk output, and one
//     scratch region for the chunk tables [K;Q] K^T (W^T passes through the update
//     operand's columns between an update and the next chunk's corrections);
//   * every chunk-sized product is a tcgen05 MMA (kind::f16, M = 128, f32 accumulation) issued
//     by one elected lane; f32 values enter as hi + lo pairs of the activation type (hi.hi +
//     hi.lo + lo.hi, about 2^-16 relative per product for bf16), raw k, q, v are exact
//     operands; the 16 x 16 blocks of the triangular inverse's levels are mma.sync tiles;
//   * k, q, v arrive by tensor-map copies (TMA, 64 tokens x 64 features per box, 128-byte
//     swizzle) into shared memory, two chunks of k, q resident; the load warp prefetches their
//     rows (and z's) into L2 two chunks ahead, since a box of 64 strided rows is slow to land;
//   * warp roles: 4 row warps (the serial chain: the corrections, the per-token scale of Y,
//     the next chunk's split of S into hi / lo, -W into shared memory), 4 output warps (o; for
//     the gated RMSNorm o turned through a small shared-memory tile so a lane holds 4 rows of
//     one token; the y stores), 6 table warps (q norms while the chunk tables MMA runs, then tables
//     -> A, rk, P, the unit-triangular inverse T in 16 x 16 blocks, the B operands of U and W;
//     one of them issues the tables and W^T MMAs), one MMA warp (the chain's MMAs), one load
//     warp (the copies and the decay products of each chunk);
//   * the table warps work one chunk ahead, so the chain per chunk is: split S -> X MMAs ->
//     corrections -> update MMAs.
// Every wait is an mbarrier wait: a phase already complete is taken by an inline test, else
// the wait has a time limit; a wait that runs out sets the watchdog word and is retried once
// with the full limit; if that also runs out the CTA abandons its
// work (later waits return at once, no new copies or MMAs, no stores), drains the MMAs and
// copies it issued, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <atomic>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_mma.cuh"
#include "gdn_tcgen05.cuh"
#include "gdn_tma.cuh"

namespace gdn {

// First-attempt time limit of this unit's mbarrier waits in nanoseconds (0: the default
// 2 s).  Only the self-test hook sets it, to make a real wait of the scan run out.
static __device__ unsigned long long g_wy_first_limit_ns;

namespace {

constexpr int kC = 64;                    // tokens per chunk
constexpr int kD = 128;                   // Dk = Dv
constexpr float kMinLogDecay = -80.0f;    // exp(-80) ~ 1.8e-35: a full reset in f32
constexpr uint64_t kLimitNs = 2000000000ull;

// warp roles: three groups of 4 warps (a warp reads tensor-memory lane quarter warp % 4), the
// MMA warp, the load warp and 2 more table warps
constexpr int kRowW0 = 0;                 // 4 row warps
constexpr int kEpiW0 = 4;                 // 4 output warps
constexpr int kTabW0 = 8;                 // 4 table warps; the first issues the table / W MMAs
constexpr int kMmaW = 12;                 // issues the chain's MMAs; warp 13 is the load warp
constexpr int kHelpW0 = 14;               // 2 more table warps (the inverse and B operands)
constexpr int kWarps = 16;
constexpr int kTabT = 192;                // table-role threads
constexpr int kThreads = 32 * kWarps;

// tensor-memory columns (512 allocated)
enum : uint32_t {
    TM_S = 0,        // f32 memory, 128 columns
    TM_SHI = 128,    // hi part of S as packed pairs (K = 128 in 64 columns)
    TM_X = 192,      // U^T - S W^T: the corrections d, one column per token
    TM_YO = 256,     // S Q^T, scaled per token, plus the intra-chunk term: o
    TM_VCH = 320, TM_VCL = 352,   // update operand: d_s rk_s G_63 / G_s, hi / lo (K = 64 tokens);
                                  // between the update and the next corrections: W^T (lanes = j)
    TM_VUH = 384, TM_VUL = 416,   // intra-chunk operand: d_s, hi / lo
    TM_SCR = 448,    // [K;Q] K^T (lanes 0-63: k rows, 64-127: q rows)
    TM_COLS = 512
};

// Shared memory (offsets from a 1024-byte aligned base).  Boxes are 64 rows x 128 bytes with
// the 128-byte swizzle (16-byte piece p of row r at (r / 8) * 1024 + (r % 8) * 128 +
// ((p ^ (r % 8)) * 16)).
constexpr uint32_t kBox = 8192;
constexpr uint32_t OFF_KQ = 0;                        // 2 slots x [K0 | Q0 | K1 | Q1]
constexpr uint32_t kSlot = 4 * kBox;
constexpr uint32_t OFF_V = OFF_KQ + 2 * kSlot;        // [V0 | V1]
constexpr uint32_t OFF_WHI = OFF_V + 2 * kBox;        // -W hi / lo: row j holds 64 tokens
constexpr uint32_t OFF_WLO = OFF_WHI + 2 * kBox;
constexpr uint32_t OFF_SLO = OFF_WLO + 2 * kBox;      // lo part of S: [a][j], two K halves
constexpr uint32_t OFF_P = OFF_SLO + 4 * kBox;        // 2 buffers x [hi | lo], [t][s]
constexpr uint32_t OFF_BU = OFF_P + 4 * kBox;         // T diag(beta): [hi | lo], [t][s]
constexpr int kAS = 68;                               // row stride of A (floats): conflict-free rows
constexpr uint32_t OFF_A = OFF_BU + 2 * kBox;         // f32 A [64][kAS]; later -W's B: [hi | lo]
constexpr uint32_t OFF_TB = OFF_A + 64 * kAS * 4;     // T in 16 x 16 f32 blocks (10 of them)
constexpr uint32_t OFF_SC = OFF_TB + 10 * 1024;       // per-chunk scalars, see Scal
constexpr uint32_t kAlignPad = 1024;

// Arrays by chunk parity are written one chunk ahead by another role; the single ones live
// within one chunk of the table warps.
struct Scal {
    float turn[4][4 * 32];   // output warps: 4 tokens x 32 rows of o per warp (16-byte aligned)
    float cum[2][kC];        // chunk-inclusive sums of clamped log_decay (by chunk parity)
    float beta[2][kC];       // beta (0 past the end)
    float gamma[2][2];       // [0] e^{cum_63}; [1] 1 when every |cum_t - m| <= 80, m = cum_31
    float cvec[2][kC];       // rk_t e^{cum_63 - cum_t}: the update's per-token factor
    float ysc[2][kC];        // e^{cum_t} rq_t: the per-token scale of S q_t (table warps)
    float rk[kC];            // 1 / ||k_t||
    float colk[kC];          // rk_s e^{m - cum_s}: the column factor of A and P ("factored")
    float bws[kC];           // beta_s e^{cum_s} rk_s: W's per-token factor
    float rqs[kC];           // rq_t, handed from the P-row warps to the helpers
    float red[4][kC];        // gated norm: partial sums of squares per output warp
    float rr[kC];            // gated norm: 1 / rms per token
    uint64_t bar[24];        // mbarriers (see enum Bar)
    uint32_t tmem_base;
    int abandon;
};
static_assert(offsetof(Scal, turn) % 16 == 0 && offsetof(Scal, cvec) % 8 == 0 &&
                  offsetof(Scal, colk) % 16 == 0 && offsetof(Scal, bws) % 16 == 0 &&
                  offsetof(Scal, bar) % 8 == 0 && OFF_SC % 16 == 0,
              "vector accesses of the scalars");
constexpr uint32_t kSmemBytes = OFF_SC + static_cast<uint32_t>(sizeof(Scal)) + kAlignPad;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

enum Bar {
    B_LDKQ = 0,      // 2: a slot's k, q boxes landed
    B_LDV = 2,       // v boxes landed
    B_GATES = 3,     // 2: decay products of a chunk written (by chunk parity)
    B_TAB = 5,       // chunk tables MMA done
    B_WT = 6,        // W^T MMA done
    B_X = 7,         // X MMAs done
    B_Y = 8,         // Y MMAs done
    B_UPD = 9,       // update MMAs done
    B_KQFREE = 10,   // 2: the slot's last reader (the update) done
    B_U = 12,        // U^T MMAs done
    B_PFREE = 13,    // 2: intra-chunk output MMAs done (P buffer and o ready)
    B_SPLIT = 15,    // row warps: S split and scaled (4 arrivals)
    B_VP = 16,       // row warps: correction operands written (4)
    B_WRDY = 17,     // row warps: -W in shared memory, W^T read out (4)
    B_BU = 18,       // table warps: U's B operand, the chunk's cvec and Y scales written (4)
    B_YSC = 19,      // output warps: Y scaled (4)
    B_YOFREE = 20,   // output warps: o read out of tensor memory (4)
    B_DRAIN = 21,    // 2: final commits of the two MMA-issuing warps
    B_COUNT = 23
};
static_assert(B_COUNT <= 24, "mbarrier slots");

// named barriers (ids 1-3): table warps, output warps
enum { NB_TAB = 1, NB_EPI = 2 };

// ------------------------------------------------------------------ operand types

template <typename TA> struct Op;
template <> struct Op<__nv_bfloat16> {
    static constexpr uint32_t kFmt = 1;   // kind::f16 operand format: BF16
    __device__ __forceinline__ static void split2(float x, float y, uint32_t &hi, uint32_t &lo) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
        hi = *reinterpret_cast<const uint32_t *>(&h);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
};
template <> struct Op<__half> {
    static constexpr uint32_t kFmt = 0;   // kind::f16 operand format: F16
    __device__ __forceinline__ static void split2(float x, float y, uint32_t &hi, uint32_t &lo) {
        const __half2 h = __floats2half2_rn(x, y);
        const float2 hf = __half22float2(h);
        const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
        hi = *reinterpret_cast<const uint32_t *>(&h);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
};

// Instruction descriptor of kind::f16 with f32 accumulation: operand format, A / B major-ness
// (0 = K-major, 1 = MN-major), N, M.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn, uint32_t fmt) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// Descriptors of the 128-byte swizzled layouts.  K-major: rows of 128 bytes (64 elements of
// K) in 8-row groups of 1024 bytes; a K step of 16 advances 32 bytes inside the row.
// MN-major: rows are K (128 bytes = 64 elements of M or N), 8-row groups of 1024 bytes, a K
// step of 16 rows advances 2048 bytes; `lbo` is the distance between 64-wide M / N blocks.
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) { return umma_desc(saddr, 16, 1024, true); }
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr, uint32_t lbo) {
    return umma_desc(saddr, lbo, 1024, true);
}

__device__ __forceinline__ uint32_t sw_off(int row, int piece) {
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + (((piece ^ row) & 7) << 4));
}

// One 128-byte line of global memory into L2.
__device__ __forceinline__ void prefetch_line_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// silu(z) = z / (1 + e^{-z}) with e^x = 2^{x log2 e}, from the hardware's base-2 exponential
// and reciprocal approximations (ex2.approx, rcp.approx: a few ulp); z -> -inf gives -0.
__device__ __forceinline__ float silu_ex2(float z) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * -1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return z * r;
}

__device__ __forceinline__ void nbar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// One warp's 16 x 8 tile d += L R of f32 operands in shared memory (L 16 x 16 row-major with
// stride ldl, R 16 x 8 row-major with stride ldr), by mma.sync m16n8k16 on bf16 hi + lo parts
// (hi.hi + hi.lo + lo.hi, f32 accumulation).  Fragment layouts of the PTX ISA for m16n8k16:
// lane = 4 g + c holds L rows g, g + 8 at columns 2c, 2c + 1 (+ 8), R rows 2c, 2c + 1 (+ 8) at
// column g, and d rows g, g + 8 at columns 2c, 2c + 1.
__device__ __forceinline__ void tile_mma(float (&d)[4], const float *L, int ldl, const float *R, int ldr,
                                         int lane) {
    const int g = lane >> 2, c = lane & 3;
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const float2 x = *reinterpret_cast<const float2 *>(L + (g + 8 * (e & 1)) * ldl + 2 * c + 8 * (e >> 1));
        split2(x.x, x.y, ah[e], al[e]);
    }
#pragma unroll
    for (int e = 0; e < 2; e++)
        split2(R[(2 * c + 8 * e) * ldr + g], R[(2 * c + 1 + 8 * e) * ldr + g], bh[e], bl[e]);
    mma3(d, ah, al, bh[0], bh[1], bl[0], bl[1]);
}

// s * d of a tile_mma into a 16 x 8 row-major f32 tile with stride ld.
__device__ __forceinline__ void tile_store(float *D, int ld, const float (&d)[4], float s, int lane) {
    const int g = lane >> 2, c = lane & 3;
    *reinterpret_cast<float2 *>(D + g * ld + 2 * c) = make_float2(s * d[0], s * d[1]);
    *reinterpret_cast<float2 *>(D + (g + 8) * ld + 2 * c) = make_float2(s * d[2], s * d[3]);
}

// mbarrier phase test that lets the hardware suspend the warp for up to `hint_ns` while the
// phase is incomplete (it resumes as soon as the phase completes), instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, unsigned parity, unsigned hint_ns) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase (acquire semantics, like the waits).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// One bounded attempt: suspending tests until the phase completes or `limit_ns` has passed.
__device__ __forceinline__ bool wy_wait_for(uint64_t *bar, unsigned parity, uint64_t limit_ns) {
    const unsigned hint = limit_ns < 20000ull ? static_cast<unsigned>(limit_ns) : 20000u;
    if (mbar_try_wait_hint(bar, parity, hint)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_hint(bar, parity, hint))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// Bounded wait (kept out of line: it is called from every role): a first attempt (the test
// hook may shorten it), then, if it ran out (the watchdog word is set), one more with the full
// limit; if that runs out too, the CTA abandons its work and every later wait returns false.
__device__ __noinline__ bool wy_wait(uint64_t *bar, unsigned parity, volatile int *abandon,
                                     unsigned long long first_ns) {
    if (*abandon) return false;
    if (wy_wait_for(bar, parity, first_ns ? first_ns : kLimitNs)) return true;
    atomicOr(&g_watchdog, 1u);
    if (wy_wait_for(bar, parity, kLimitNs)) return true;
    *abandon = 1;
    return false;
}

template <typename TA>
__global__ void __launch_bounds__(kThreads, 1)
gdn_scan_wy_kernel(const __grid_constant__ gdn_params p, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mv) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    Scal &sc = *reinterpret_cast<Scal *>(smem + OFF_SC);
    using O = Op<TA>;
    using A_ = Act<TA>;
    constexpr uint32_t fmt = O::kFmt;
    constexpr uint32_t kIdN64 = idesc(128, 64, false, false, fmt);      // B K-major
    constexpr uint32_t kIdN64Bmn = idesc(128, 64, false, true, fmt);    // B MN-major
    constexpr uint32_t kIdN64Amn = idesc(128, 64, true, false, fmt);    // A MN-major
    constexpr uint32_t kIdN128Bmn = idesc(128, 128, false, true, fmt);

    const int64_t head = blockIdx.x;                       // b * Hv + hv
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S;
    const int nch = (S + kC - 1) / kC;
    const bool gated = p.z != nullptr;
    uint64_t *bar = sc.bar;

    if (threadIdx.x == 0) {
        for (int i = 0; i < B_COUNT; i++) {
            const bool arrivals4 = (i >= B_SPLIT && i <= B_YOFREE);
            mbar_init(&bar[i], arrivals4 ? 4 : 1);
        }
        sc.abandon = 0;
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(&sc.tmem_base, TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sc.tmem_base;
    const unsigned long long first_ns = g_wy_first_limit_ns;
    volatile int *abandon = &sc.abandon;

    // a phase already complete is taken inline (most waits of a steady chunk are); otherwise
    // the out-of-line bounded wait
    auto wait = [&](int i, unsigned parity) -> bool {
        if (mbar_test(&bar[i], parity) && !*abandon) return true;
        return wy_wait(&bar[i], parity, abandon, first_ns);
    };
    auto uniform = [&](bool ok) { return __all_sync(0xffffffffu, ok && !*abandon); };
    auto arrive_warp = [&](int i) {                        // one arrival per warp
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[i]);
    };

    // operand addresses
    auto kq_slot = [&](int c) { return sbase + OFF_KQ + static_cast<uint32_t>(c & 1) * kSlot; };
    const uint32_t a_v = sbase + OFF_V, a_whi = sbase + OFF_WHI, a_wlo = sbase + OFF_WLO;
    const uint32_t a_slo = sbase + OFF_SLO, a_bu = sbase + OFF_BU, a_bw = sbase + OFF_A;
    auto a_p = [&](int c) { return sbase + OFF_P + static_cast<uint32_t>(c & 1) * 2 * kBox; };
    const int64_t v_ts = p.head_major ? kD : static_cast<int64_t>(p.Hv) * kD;   // token stride of v, z, y
    const int64_t v_base = p.head_major ? head * S * kD : (static_cast<int64_t>(b) * S * p.Hv + hv) * kD;
    const int64_t g_ts = p.head_major ? 1 : p.Hv;
    const int64_t g_base = p.head_major ? head * S : static_cast<int64_t>(b) * S * p.Hv + hv;

    const bool tab_warp = warp >= kTabW0 && warp < kTabW0 + 4;
    if (warp >= kRowW0 && warp < kRowW0 + 4) {
        // ================================= row warps ======================================
        const int a = 32 * (warp & 3) + lane;              // memory row = tensor-memory lane
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        // -W of chunk n (row j = this thread's lane of W^T, held in the update operand's columns
        // from the update of n-1 to the corrections of n) into the MN-major B operand of X; the
        // X MMAs of chunk n-1 have read the previous one
        auto w_pass = [&](int n) {
            wait(B_WT, static_cast<unsigned>(n & 1));
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; h++) {
                float w[32];
                tm_ld32(tl + TM_VCH + 32 * h, w);
#pragma unroll
                for (int gg = 0; gg < 4; gg++) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) O::split2(w[8 * gg + 2 * e], w[8 * gg + 2 * e + 1], hi[e], lo[e]);
                    sts128(a_whi + sw_off(a, 4 * h + gg), hi[0], hi[1], hi[2], hi[3]);
                    sts128(a_wlo + sw_off(a, 4 * h + gg), lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            arrive_warp(B_WRDY);
        };
        // the memory at the start of chunk c (after the update of c-1; Y of c-1 has read the
        // hi / lo parts of c-1): split into hi (tensor memory) and lo (shared memory), then
        // gamma S stored back for the update of c
        auto split = [&](int c) {
            const int pb = c & 1;
            wait(B_GATES + pb, static_cast<unsigned>((c >> 1) & 1));
            const float gam = sc.gamma[pb][0];
            if (c > 0) {                                   // S of chunk c; Y of c-1 has read
                wait(B_UPD, static_cast<unsigned>((c - 1) & 1));   // the hi / lo parts of c-1
                wait(B_Y, static_cast<unsigned>((c - 1) & 1));
                tc_fence_after();
            }
            // split S into hi (tensor memory) and lo (shared memory), then store gamma S;
            // 32 columns at a time
#pragma unroll 1
            for (int qc = 0; qc < 4; qc++) {
                float s[32];
                if (c > 0) {
                    tm_ld32(tl + TM_S + 32 * qc, s);
                } else if (p.s0 != nullptr) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.s0 + head * (kD * kD) + static_cast<int64_t>(a) * kD + 32 * qc);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float4 f = src[i];
                        s[4 * i] = f.x; s[4 * i + 1] = f.y; s[4 * i + 2] = f.z; s[4 * i + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++) s[i] = 0.f;
                }
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int j = 0; j < 16; j++) O::split2(s[2 * j], s[2 * j + 1], hi[j], lo[j]);
                tm_st16(tl + TM_SHI + 16 * qc, hi);
                const uint32_t lrow = a_slo + (qc >> 1) * 2 * kBox;   // K half qc / 2
#pragma unroll
                for (int pc = 0; pc < 4; pc++)
                    sts128(lrow + sw_off(a, 4 * (qc & 1) + pc), lo[4 * pc], lo[4 * pc + 1],
                           lo[4 * pc + 2], lo[4 * pc + 3]);
#pragma unroll
                for (int j = 0; j < 32; j++) s[j] *= gam;
                tm_st32f(tl + TM_S + 32 * qc, s);
            }
            tm_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            arrive_warp(B_SPLIT);
        };
        split(0);
        w_pass(0);
        for (int c = 0; c < nch; c++) {
            const int pb = c & 1;
            // corrections d_t = X[a][t] -> intra-chunk operand (d) and update operand (d cvec);
            // cvec and the scales of Y are the table warps', published by their B_BU arrivals
            // of chunk c (complete before U, so before X, of chunk c)
            wait(B_BU, static_cast<unsigned>(c & 1));
            wait(B_X, static_cast<unsigned>(c & 1));
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; h++) {                  // tokens 32 h .. 32 h + 31
                float d[32];
                tm_ld32(tl + TM_X + 32 * h, d);
                uint32_t uh[16], ul[16], ch[16], cl[16];
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const float2 cv = *reinterpret_cast<const float2 *>(&sc.cvec[pb][32 * h + 2 * j]);
                    O::split2(d[2 * j], d[2 * j + 1], uh[j], ul[j]);
                    O::split2(d[2 * j] * cv.x, d[2 * j + 1] * cv.y, ch[j], cl[j]);
                }
                tm_st16(tl + TM_VUH + 16 * h, uh);
                tm_st16(tl + TM_VUL + 16 * h, ul);
                tm_st16(tl + TM_VCH + 16 * h, ch);
                tm_st16(tl + TM_VCL + 16 * h, cl);
            }
            tm_wait_st();
            tc_fence_before();
            arrive_warp(B_VP);

            // S q_t scaled by e^{cum_t} rq_t, in place, before the intra-chunk term is added
            wait(B_Y, static_cast<unsigned>(c & 1));
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; h++) {
                float y[32];
                tm_ld32(tl + TM_YO + 32 * h, y);
#pragma unroll
                for (int j = 0; j < 32; j++) y[j] *= sc.ysc[pb][32 * h + j];
                tm_st32f(tl + TM_YO + 32 * h, y);
            }
            tm_wait_st();
            tc_fence_before();
            arrive_warp(B_YSC);
            if (c + 1 < nch) {
                // the next chunk's split runs here, while the table warps finish its W: only
                // the W pass then stands between them and the next X MMAs
                split(c + 1);
                w_pass(c + 1);                             // X of chunk c is done
            }
        }
        // final memory row a
        const bool ok = wait(B_UPD, static_cast<unsigned>((nch - 1) & 1));
        tc_fence_after();
        float *so = p.state + head * (kD * kD) + static_cast<int64_t>(a) * kD;
        const bool store = ok && !*abandon;
#pragma unroll 1
        for (int qc = 0; qc < 4; qc++) {
            float s[32];
            tm_ld32(tl + TM_S + 32 * qc, s);
            if (store) {
#pragma unroll
                for (int i = 0; i < 8; i++)
                    *reinterpret_cast<float4 *>(so + 32 * qc + 4 * i) =
                        make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
            }
        }
    } else if (warp >= kEpiW0 && warp < kEpiW0 + 4) {
        // ============================== output warps =====================================
        // Tensor memory hands thread a row a of o for the chunk's 64 tokens.  For the gated
        // norm each warp turns its 32 rows through a private shared-memory tile, 4 tokens (one
        // block) at a time, so that lane 4 j + i then holds rows 4 j .. 4 j + 3 of its warp's 32
        // for token 4 b + i: z arrives by one 8-byte load per block, a token's squares add up
        // in the thread and over three shuffles, and y leaves by one 16-byte store per block.
        const int q4 = warp & 3;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        const int etid = 32 * q4 + lane;                   // 0..127
        const int ti = lane & 3;                           // token of the block
        const int r0 = 32 * q4 + 4 * (lane >> 2);          // first of the 4 rows after the turn
        const float4 g4 = gated ? *reinterpret_cast<const float4 *>(p.gn + r0) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float inv_d = 1.0f / static_cast<float>(kD);
        const TA *zr = gated ? static_cast<const TA *>(p.z) + v_base + r0 : nullptr;
        float *tile = sc.turn[q4];                         // 4 tokens x 32 rows
        for (int c = 0; c < nch; c++) {
            const int pb = c & 1;
            const int t0 = c * kC, nt = min(kC, S - t0);
            // z of the chunk in the turned layout (tokens past the end read the last token's,
            // never stored), loaded while o is still being computed
            uint2 zb[16];
            if (gated) {
#pragma unroll
                for (int bk = 0; bk < 16; bk++)
                    zb[bk] = *reinterpret_cast<const uint2 *>(
                        zr + static_cast<int64_t>(t0 + min(4 * bk + ti, nt - 1)) * v_ts);
            }
            // o of the chunk, out of tensor memory at once
            wait(B_PFREE + pb, static_cast<unsigned>((c >> 1) & 1));
            tc_fence_after();
            float o[64];
            tm_ld64(tl + TM_YO, o);
            tc_fence_before();
            arrive_warp(B_YOFREE);
            const bool live = !*abandon;
            if (!gated) {
                // raw o: the natural layout stores it, a warp's 32 rows being 128 contiguous
                // bytes of a token
                if (live) {
                    float *yc = p.y + v_base + static_cast<int64_t>(t0) * v_ts + 32 * q4 + lane;
#pragma unroll
                    for (int t = 0; t < kC; t++)
                        if (t < nt) yc[t * v_ts] = o[t];
                }
                continue;
            }
            // the turn: afterwards o[4 b + e] is row r0 + e of token 4 b + ti.  Row r of token e
            // sits at word 32 e + (r ^ 8 e): the writes of a token cover 32 distinct banks, and
            // the 16-byte reads of any 8 lanes (rows 4 j .. 4 j + 3 at word 32 i + 4 (j ^ 2 i))
            // too.  Only shared-memory traffic here, so that the gating below is one batch of
            // independent work rather than 16 dependent rounds.
#pragma unroll
            for (int bk = 0; bk < 16; bk++) {
#pragma unroll
                for (int e = 0; e < 4; e++) tile[32 * e + (lane ^ (8 * e))] = o[4 * bk + e];
                __syncwarp();
                const float4 v = *reinterpret_cast<const float4 *>(tile + 32 * ti + ((r0 & 31) ^ (8 * ti)));
                __syncwarp();
                o[4 * bk] = v.x; o[4 * bk + 1] = v.y; o[4 * bk + 2] = v.z; o[4 * bk + 3] = v.w;
            }
            // gated RMSNorm over the head's 128 rows: the gate, this lane's 4 squares per token,
            // then the warp's 32 (three shuffles per token), then the 4 warps' partial sums
#pragma unroll
            for (int bk = 0; bk < 16; bk++) {
                const float2 za = O::unpack(zb[bk].x), zc2 = O::unpack(zb[bk].y);
                o[4 * bk] *= silu_ex2(za.x);
                o[4 * bk + 1] *= silu_ex2(za.y);
                o[4 * bk + 2] *= silu_ex2(zc2.x);
                o[4 * bk + 3] *= silu_ex2(zc2.y);
            }
            float ss[16];
#pragma unroll
            for (int bk = 0; bk < 16; bk++) {
                ss[bk] = o[4 * bk] * o[4 * bk];
                ss[bk] = fmaf(o[4 * bk + 1], o[4 * bk + 1], ss[bk]);
                ss[bk] = fmaf(o[4 * bk + 2], o[4 * bk + 2], ss[bk]);
                ss[bk] = fmaf(o[4 * bk + 3], o[4 * bk + 3], ss[bk]);
            }
            // the sums over the 8 lanes of a token class (lane 4 j + ti, j = 0..7) by halving
            // exchanges: after the exchange across lane bit 4 + m a lane keeps the blocks whose
            // bit m matches its own, so lane j ends with blocks 2 j, 2 j + 1 summed (14 shuffles)
            const int rj = lane >> 2;
#pragma unroll
            for (int m = 2, cnt = 8; m >= 0; m--, cnt >>= 1) {
                const bool up = (rj >> m) & 1;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    if (i < cnt) {
                        const float send = up ? ss[i] : ss[i + cnt];
                        const float keep = up ? ss[i + cnt] : ss[i];
                        ss[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4 << m);
                    }
                }
            }
            sc.red[q4][4 * (2 * rj) + ti] = ss[0];
            sc.red[q4][4 * (2 * rj + 1) + ti] = ss[1];
            nbar_sync(NB_EPI, 128);
            if (etid < kC)
                sc.rr[etid] = rsqrtf(fmaf(sc.red[0][etid] + sc.red[1][etid] + sc.red[2][etid] +
                                              sc.red[3][etid], inv_d, p.norm_eps));
            nbar_sync(NB_EPI, 128);
            if (live) {
                float *yc = p.y + v_base + static_cast<int64_t>(t0) * v_ts + r0;
#pragma unroll
                for (int bk = 0; bk < 16; bk++) {
                    const int t = 4 * bk + ti;
                    const float r = sc.rr[t];
                    const float4 v = make_float4(o[4 * bk] * (r * g4.x), o[4 * bk + 1] * (r * g4.y),
                                                 o[4 * bk + 2] * (r * g4.z), o[4 * bk + 3] * (r * g4.w));
                    if (t < nt) *reinterpret_cast<float4 *>(yc + static_cast<int64_t>(t) * v_ts) = v;
                }
            }
        }
    } else if (tab_warp || warp >= kHelpW0) {
        // =============================== table warps =====================================
        // The four table warps (lane quarters 0-3) read the chunk tables out of tensor memory;
        // the two helper warps join them for the triangular inverse and the B operands.
        const bool tabw = tab_warp;
        const int q4 = warp & 3;                           // tensor-memory lane quarter
        const int tt = tabw ? 32 * q4 + lane : 4 * 32 + 32 * (warp - kHelpW0) + lane;   // 0..191
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        float *Am = reinterpret_cast<float *>(smem + OFF_A);        // [64][kAS]
        float *Tb = reinterpret_cast<float *>(smem + OFF_TB);       // 10 blocks [16][16]
        auto blk = [](int i, int j) { return i * (i + 1) / 2 + j; };
        bool issued = false;
        for (int n = 0; n < nch; n++) {
            const int pb = n & 1;
            // the P rows' q norms (rq carries 1 / sqrt(Dk)) from the chunk's q boxes, while
            // the tables MMA runs
            float rq = 0.f;
            if (tt >= kC && tt < 2 * kC && uniform(wait(B_LDKQ + pb, static_cast<unsigned>((n >> 1) & 1)))) {
                const int t = tt - kC;
                const uint32_t qs = kq_slot(n) + kBox;
                float ss = 0.f;
#pragma unroll 4
                for (int pc = 0; pc < 16; pc++) {
                    const uint4 w = lds128(qs + (pc >> 3) * 2 * kBox + sw_off(t, pc));
                    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float2 f = O::unpack(u[e]);
                        ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
                    }
                }
                rq = n * kC + t < S ? rsqrtf(ss + p.qk_eps) * rsqrtf(static_cast<float>(kD)) : 0.f;
            }
            if (warp == kTabW0) {
                // the scratch is free: the table warps read the tables of n-1 before their inverse
                const bool ok = uniform(wait(B_LDKQ + pb, static_cast<unsigned>((n >> 1) & 1)));
                if (ok) {
                    issued = true;
                    if (elect_one()) {
                        tc_fence_after();
                        const uint32_t s = kq_slot(n);
#pragma unroll 1
                        for (int kk = 0; kk < 8; kk++) {
                            const uint32_t off = (kk >> 2) * 2 * kBox + (kk & 3) * 32;
                            umma_ss(tmem + TM_SCR, desc_k(s + off), desc_k(s + off), kIdN64, kk > 0);
                        }
                        umma_commit(&bar[B_TAB]);
                    }
                }
                __syncwarp();
            }
            wait(B_TAB, static_cast<unsigned>(n & 1));
            wait(B_GATES + pb, static_cast<unsigned>((n >> 1) & 1));
            if (n >= 2) wait(B_PFREE + pb, static_cast<unsigned>(((n - 2) >> 1) & 1));
            if (n >= 1) wait(B_WT, static_cast<unsigned>((n - 1) & 1));   // W^T of n-1 read Bw (= A)
            tc_fence_after();
            const uint32_t slot = kq_slot(n);
            const bool fac = sc.gamma[pb][1] != 0.f;       // uniform: factored exponentials
            if (tt < kC) {
                // rk from the diagonal of K K^T: lane t reads column t (this warp's 32 columns)
                const int t = tt;
                float dg = 0.f;
                {
                    float v32[32];
                    tm_ld32(tl + TM_SCR + 32 * q4, v32);
#pragma unroll
                    for (int j = 0; j < 32; j++) dg = (j == lane) ? v32[j] : dg;
                }
                const float rk = rsqrtf(dg + p.qk_eps);
                const float ct = sc.cum[pb][t];
                sc.rk[t] = rk;
                sc.colk[t] = rk * __expf(fminf(sc.cum[pb][kC / 2 - 1] - ct, 80.f));
                sc.cvec[pb][t] = rk * __expf(sc.cum[pb][kC - 1] - ct);
                sc.bws[t] = sc.beta[pb][t] * __expf(ct) * rk;
            } else if (tt < 2 * kC) {
                sc.rqs[tt - kC] = rq;
            }
            nbar_sync(NB_TAB, kTabT);                        // rk of the chunk written
            if (tt < kC) {
                // A[t][s] = beta_t rk_t rk_s e^{cum_t - cum_s} (k_t . k_s), s < t
                const int t = tt;
                const float ct = sc.cum[pb][t], bt = sc.beta[pb][t] * sc.rk[t];
                const float rowf = bt * __expf(fminf(ct - sc.cum[pb][kC / 2 - 1], 80.f));
                if (fac) {                                 // e^{cum_t - cum_s} = ef_t eg_s
#pragma unroll 1
                    for (int h = 0; h < 2; h++) {          // 32 columns at a time
                        float v[32];
                        tm_ld32(tl + TM_SCR + 32 * h, v);
#pragma unroll
                        for (int g4 = 0; g4 < 8; g4++) {
                            const int s0 = 32 * h + 4 * g4;
                            const float4 c4 = *reinterpret_cast<const float4 *>(&sc.colk[s0]);
                            const float cf[4] = {c4.x, c4.y, c4.z, c4.w};
                            float a4[4];
#pragma unroll
                            for (int e = 0; e < 4; e++) a4[e] = s0 + e < t ? rowf * cf[e] * v[4 * g4 + e] : 0.f;
                            *reinterpret_cast<float4 *>(&Am[t * kAS + s0]) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                        }
                    }
                } else {                                   // a chunk of very fast decay: per element
#pragma unroll 1
                    for (int g = 0; g < 8; g++) {
                        float v8[8];
                        tm_ld8(tl + TM_SCR + 8 * g, v8);
#pragma unroll 1
                        for (int j = 0; j < 8; j++) {
                            const int s_ = 8 * g + j;
                            float vj = 0.f;
#pragma unroll
                            for (int jj = 0; jj < 8; jj++) vj = jj == j ? v8[jj] : vj;
                            Am[t * kAS + s_] = s_ < t ? bt * sc.rk[s_] * __expf(ct - sc.cum[pb][s_]) * vj : 0.f;
                        }
                    }
                }
                // ---- T = (I + A)^-1 in 16 x 16 blocks: the diagonal blocks by forward
                // substitution, each from the A rows of its own warp (blocks 0, 1: this warp's
                // rows 0-31; 2, 3: the other's), so a warp barrier suffices
                __syncwarp();
                {
                    const int i = tt >> 4, cs = tt & 15;
                    float x[16];
#pragma unroll
                    for (int r = 0; r < 16; r++) x[r] = r == cs ? 1.f : 0.f;
#pragma unroll
                    for (int r = 1; r < 16; r++) {
                        const float *arow = &Am[(16 * i + r) * kAS + 16 * i];
                        float acc = 0.f;
#pragma unroll
                        for (int u4 = 0; u4 < 4; u4++) {
                            if (4 * u4 < r) {
                                const float4 a4 = *reinterpret_cast<const float4 *>(arow + 4 * u4);
                                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                                for (int e = 0; e < 4; e++)
                                    if (4 * u4 + e < r) acc = fmaf(av[e], x[4 * u4 + e], acc);
                            }
                        }
                        x[r] -= acc;
                    }
                    float *tb = Tb + blk(i, i) * 256;
#pragma unroll
                    for (int r = 0; r < 16; r++) tb[r * 16 + cs] = x[r];
                }
            } else {
                // P[t][s] = e^{cum_t - cum_s} rk_s rq_t (q_t . k_s), s <= t: B of the intra term.
                // The P-row warps take columns 0-31, the helpers (same lane quarters) 32-63.
                const int h = tt >= 2 * kC ? 1 : 0;
                const int t = tt - kC - kC * h;
                const float ct = sc.cum[pb][t];
                const float rqt = h ? sc.rqs[t] : rq;
                if (!h) sc.ysc[pb][t] = __expf(ct) * rq;       // read by the row warps after B_BU
                const float rowf = rqt * __expf(fminf(ct - sc.cum[pb][kC / 2 - 1], 80.f));
                const uint32_t ph = a_p(n), pl = ph + kBox;
                if (fac) {                                 // e^{cum_t - cum_s} = ef_t eg_s
                    float v[32];
                    tm_ld32(tl + TM_SCR + 32 * h, v);
#pragma unroll
                    for (int j = 0; j < 32; j++) {
                        const int s_ = 32 * h + j;
                        v[j] = s_ <= t ? rowf * sc.colk[s_] * v[j] : 0.f;
                    }
#pragma unroll
                    for (int gg = 0; gg < 4; gg++) {
                        const int g = 4 * h + gg;
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) O::split2(v[8 * gg + 2 * e], v[8 * gg + 2 * e + 1], hi[e], lo[e]);
                        sts128(ph + sw_off(t, g), hi[0], hi[1], hi[2], hi[3]);
                        sts128(pl + sw_off(t, g), lo[0], lo[1], lo[2], lo[3]);
                    }
                } else {                                   // a chunk of very fast decay: per element
#pragma unroll 1
                    for (int g = 4 * h; g < 4 * h + 4; g++) {
                        float v8[8];
                        tm_ld8(tl + TM_SCR + 8 * g, v8);
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            const int s_ = 8 * g + j;
                            v8[j] = s_ <= t ? rqt * sc.rk[s_] * __expf(ct - sc.cum[pb][s_]) * v8[j] : 0.f;
                        }
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) O::split2(v8[2 * e], v8[2 * e + 1], hi[e], lo[e]);
                        sts128(ph + sw_off(t, g), hi[0], hi[1], hi[2], hi[3]);
                        sts128(pl + sw_off(t, g), lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            nbar_sync(NB_TAB, kTabT);                        // A, P and T's diagonal blocks complete
            // ---- off-diagonal blocks.  With H_ik = T_ii A_ik (i > k), stored in A's unused
            //      upper block (k, i): T_ij = -sum_{k=j}^{i-1} H_ik T_kj, by levels i - j = 1, 2, 3.
            //      Each 16 x 8 half of an output block is one warp's mma.sync tile (f32 operands
            //      as bf16 hi + lo, f32 accumulation).
            {
                const int tw = tt >> 5;                    // 0..5
                float *Hb = Am;                            // H_ik at Am + 16 k kAS + 16 i, stride kAS
#pragma unroll 1
                for (int task = tw; task < 12; task += 6) {   // (i, k) = (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
                    const int q = task >> 1, n0 = 8 * (task & 1);
                    const int i = q < 1 ? 1 : (q < 3 ? 2 : 3);
                    const int k = q < 1 ? 0 : (q < 3 ? q - 1 : q - 3);
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    tile_mma(d, Tb + blk(i, i) * 256, 16, Am + 16 * i * kAS + 16 * k + n0, kAS, lane);
                    tile_store(Hb + 16 * k * kAS + 16 * i + n0, kAS, d, 1.f, lane);
                }
                nbar_sync(NB_TAB, kTabT);
                // Level 3 (block (3, 0)) has three terms; warps 4 and 5, idle in level 2, sum the
                // first two there (T_00, T_10 are known after level 1) and keep them in
                // registers, so level 3 adds only H_32 T_20.
                float d30[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int L = 1; L < 4; L++) {
                    const int ntask = 2 * (4 - L);         // blocks (j + L, j), two halves each
                    if (L < 3 && tw < ntask) {
                        const int j = tw >> 1, i = j + L, n0 = 8 * (tw & 1);
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                        for (int k = j; k < i; k++)
                            tile_mma(d, Hb + 16 * k * kAS + 16 * i, kAS, Tb + blk(k, j) * 256 + n0, 16, lane);
                        tile_store(Tb + blk(i, j) * 256 + n0, 16, d, -1.f, lane);
                    }
                    if (tw >= 4) {
                        const int n0 = 8 * (tw & 1);
                        if (L == 2) {
#pragma unroll 1
                            for (int k = 0; k < 2; k++)
                                tile_mma(d30, Hb + 16 * k * kAS + 48, kAS, Tb + blk(k, 0) * 256 + n0, 16, lane);
                        } else if (L == 3) {
                            tile_mma(d30, Hb + 32 * kAS + 48, kAS, Tb + blk(2, 0) * 256 + n0, 16, lane);
                            tile_store(Tb + blk(3, 0) * 256 + n0, 16, d30, -1.f, lane);
                        }
                    }
                    nbar_sync(NB_TAB, kTabT);
                }
            }
            // ---- B operands: Bu[t][s] = T[t][s] beta_s, -W's Bw[t][s] = -T[t][s] beta_s G_s rk_s
            if (n >= 1) wait(B_U, static_cast<unsigned>((n - 1) & 1));   // U^T of n-1 read Bu
            {
#pragma unroll 1
                for (int u = tt; u < kC * 8; u += kTabT) { // row t, tokens 8 pc .. 8 pc + 7
                    const int t = u >> 3, pc = u & 7, s0 = 8 * pc;
                    float tv[8];
                    if ((s0 >> 4) <= (t >> 4)) {
                        const float *src = Tb + blk(t >> 4, s0 >> 4) * 256 + (t & 15) * 16 + (s0 & 15);
                        const float4 f0 = *reinterpret_cast<const float4 *>(src);
                        const float4 f1 = *reinterpret_cast<const float4 *>(src + 4);
                        tv[0] = f0.x; tv[1] = f0.y; tv[2] = f0.z; tv[3] = f0.w;
                        tv[4] = f1.x; tv[5] = f1.y; tv[6] = f1.z; tv[7] = f1.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; e++) tv[e] = 0.f;
                    }
                    const float4 b0 = *reinterpret_cast<const float4 *>(&sc.beta[pb][s0]);
                    const float4 b1 = *reinterpret_cast<const float4 *>(&sc.beta[pb][s0 + 4]);
                    const float4 w0 = *reinterpret_cast<const float4 *>(&sc.bws[s0]);
                    const float4 w1 = *reinterpret_cast<const float4 *>(&sc.bws[s0 + 4]);
                    const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                    const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                    uint32_t uh[4], ul[4], wh[4], wl[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        O::split2(tv[2 * e] * bb[2 * e], tv[2 * e + 1] * bb[2 * e + 1], uh[e], ul[e]);
                        O::split2(-tv[2 * e] * ww[2 * e], -tv[2 * e + 1] * ww[2 * e + 1], wh[e], wl[e]);
                    }
                    sts128(a_bu + sw_off(t, pc), uh[0], uh[1], uh[2], uh[3]);
                    sts128(a_bu + kBox + sw_off(t, pc), ul[0], ul[1], ul[2], ul[3]);
                    sts128(a_bw + sw_off(t, pc), wh[0], wh[1], wh[2], wh[3]);
                    sts128(a_bw + kBox + sw_off(t, pc), wl[0], wl[1], wl[2], wl[3]);
                }
            }
            fence_proxy_async_smem();
            nbar_sync(NB_TAB, kTabT);                        // B operands complete (A is dead)
            if (warp == kTabW0) {
                // W^T = K^T Bw^T into the update operand's columns, once the update of n-1 has
                // read them (U^T of n then goes into X without waiting for W's read-out)
                if (uniform(n == 0 || wait(B_UPD, static_cast<unsigned>((n - 1) & 1)))) {
                    issued = true;
                    if (elect_one()) {
                        tc_fence_after();
#pragma unroll 1
                        for (int kt = 0; kt < 4; kt++) {
                            const uint64_t ak = desc_mn(slot + kt * 2048, 2 * kBox);
                            umma_ss(tmem + TM_VCH, ak, desc_k(a_bw + kt * 32), kIdN64Amn, kt > 0);
                            umma_ss(tmem + TM_VCH, ak, desc_k(a_bw + kBox + kt * 32), kIdN64Amn, true);
                        }
                        umma_commit(&bar[B_WT]);
                    }
                }
                __syncwarp();
            }
            if (tabw) arrive_warp(B_BU);
        }
        if (warp == kTabW0 && issued) {                    // drain this warp's MMAs
            if (elect_one()) {
                umma_commit(&bar[B_DRAIN + 1]);
                mbar_wait_bounded(&bar[B_DRAIN + 1], 0, kLimitNs);
            }
            __syncwarp();
        }
    } else if (warp == kMmaW) {
        // ================================ MMA warp =======================================
        bool issued = false;
        // U^T of chunk n into X (the corrections of n-1 were read out before the update of
        // n-1 was issued, earlier on this warp)
        auto issue_u = [&](int n) {
            const bool ok = uniform(wait(B_BU, static_cast<unsigned>(n & 1)) &
                                    wait(B_LDV, static_cast<unsigned>(n & 1)));
            if (ok) {
                issued = true;
                if (elect_one()) {
                    tc_fence_after();
#pragma unroll 1
                    for (int kt = 0; kt < 4; kt++) {
                        const uint64_t av = desc_mn(a_v + kt * 2048, kBox);
                        umma_ss(tmem + TM_X, av, desc_k(a_bu + kt * 32), kIdN64Amn, kt > 0);
                        umma_ss(tmem + TM_X, av, desc_k(a_bu + kBox + kt * 32), kIdN64Amn, true);
                    }
                    umma_commit(&bar[B_U]);
                }
            }
            __syncwarp();
        };
        // X += S (-W)^T of chunk c: hi.hi + hi.lo from tensor memory, lo.hi from shared memory
        auto issue_x = [&](int c) {
            const bool ok = uniform(wait(B_SPLIT, static_cast<unsigned>(c & 1)) &
                                    wait(B_WRDY, static_cast<unsigned>(c & 1)));
            issued |= ok;
            if (ok && elect_one()) {
                tc_fence_after();
#pragma unroll 1
                for (int kk = 0; kk < 8; kk++) {
                    const uint64_t bwh = desc_mn(a_whi + kk * 2048, 2 * kBox);
                    const uint64_t bwl = desc_mn(a_wlo + kk * 2048, 2 * kBox);
                    const uint64_t asl = desc_k(a_slo + (kk >> 2) * 2 * kBox + (kk & 3) * 32);
                    umma_ts(tmem + TM_X, tmem + TM_SHI + 8 * kk, bwh, kIdN64Bmn, true);
                    umma_ts(tmem + TM_X, tmem + TM_SHI + 8 * kk, bwl, kIdN64Bmn, true);
                    umma_ss(tmem + TM_X, asl, bwh, kIdN64Bmn, true);
                }
                umma_commit(&bar[B_X]);
            }
            __syncwarp();
        };
        // o += d P^T of chunk c onto its scaled S q
        auto issue_o = [&](int c) {
            const bool ok = uniform(wait(B_YSC, static_cast<unsigned>(c & 1)));
            issued |= ok;
            if (ok && elect_one()) {
                tc_fence_after();
                const uint32_t ph = a_p(c), pl = ph + kBox;
#pragma unroll 1
                for (int kt = 0; kt < 4; kt++) {
                    const uint64_t bh = desc_k(ph + kt * 32), bl = desc_k(pl + kt * 32);
                    umma_ts(tmem + TM_YO, tmem + TM_VUH + 8 * kt, bh, kIdN64, true);
                    umma_ts(tmem + TM_YO, tmem + TM_VUH + 8 * kt, bl, kIdN64, true);
                    umma_ts(tmem + TM_YO, tmem + TM_VUL + 8 * kt, bh, kIdN64, true);
                }
                umma_commit(&bar[B_PFREE + (c & 1)]);
            }
            __syncwarp();
        };
        // Order per chunk c: Y, update, O of c, then U and X of c+1.  The memory's chain
        // (split -> X -> corrections -> update) waits on the output warps only for the read-out
        // of the previous chunk's o, never for the gated norm itself; O of c completes before X
        // of c+1, so the corrections of c+1 may overwrite its operands.
        issue_u(0);
        issue_x(0);
        for (int c = 0; c < nch; c++) {
            const int pb = c & 1;
            const uint32_t slot = kq_slot(c);
            // Y = S Q^T (q raw): o of the previous chunk has been read out of YO
            bool ok = uniform(c == 0 || wait(B_YOFREE, static_cast<unsigned>((c - 1) & 1)));
            issued |= ok;
            if (ok && elect_one()) {
                tc_fence_after();
#pragma unroll 1
                for (int kk = 0; kk < 8; kk++) {
                    const uint32_t off = kBox + (kk >> 2) * 2 * kBox + (kk & 3) * 32;
                    const uint64_t bq = desc_k(slot + off);
                    const uint64_t asl = desc_k(a_slo + (kk >> 2) * 2 * kBox + (kk & 3) * 32);
                    umma_ts(tmem + TM_YO, tmem + TM_SHI + 8 * kk, bq, kIdN64, kk > 0);
                    umma_ss(tmem + TM_YO, asl, bq, kIdN64, true);
                }
                umma_commit(&bar[B_Y]);
            }
            __syncwarp();
            // S += (d cvec) K: the last reader of the chunk's k, q slot
            ok = uniform(wait(B_VP, static_cast<unsigned>(c & 1)));
            issued |= ok;
            if (ok && elect_one()) {
                tc_fence_after();
#pragma unroll 1
                for (int kt = 0; kt < 4; kt++) {
                    const uint64_t bk = desc_mn(slot + kt * 2048, 2 * kBox);
                    umma_ts(tmem + TM_S, tmem + TM_VCH + 8 * kt, bk, kIdN128Bmn, true);
                    umma_ts(tmem + TM_S, tmem + TM_VCL + 8 * kt, bk, kIdN128Bmn, true);
                }
                umma_commit(&bar[B_UPD]);
                umma_commit(&bar[B_KQFREE + pb]);
            }
            __syncwarp();
            issue_o(c);
            if (c + 1 < nch) {                             // X is free once the corrections are read
                issue_u(c + 1);
                issue_x(c + 1);
            }
        }
        if (issued) {                                      // drain this warp's MMAs
            if (elect_one()) {
                umma_commit(&bar[B_DRAIN]);
                mbar_wait_bounded(&bar[B_DRAIN], 0, kLimitNs);
            }
            __syncwarp();
        }
    } else {
        // ================================= load warp =====================================
        int last_kq[2] = {-1, -1}, last_v = -1;
        auto load_kq = [&](int n) {
            if (*abandon) return;
            if (lane == 0) {
                const int s = n & 1;
                uint64_t *bb = &bar[B_LDKQ + s];
                mbar_arrive_expect_tx(bb, 4 * kBox);
                const uint32_t dst = OFF_KQ + static_cast<uint32_t>(s) * kSlot;
                const int t0 = n * kC;
                tma_load_4d(smem + dst, &mk, 0, hk, t0, b, bb);
                tma_load_4d(smem + dst + kBox, &mq, 0, hk, t0, b, bb);
                tma_load_4d(smem + dst + 2 * kBox, &mk, 64, hk, t0, b, bb);
                tma_load_4d(smem + dst + 3 * kBox, &mq, 64, hk, t0, b, bb);
            }
            last_kq[n & 1] = n;
        };
        auto load_v = [&](int n) {
            if (*abandon) return;
            if (lane == 0) {
                uint64_t *bb = &bar[B_LDV];
                mbar_arrive_expect_tx(bb, 2 * kBox);
                const int t0 = n * kC;
                tma_load_4d(smem + OFF_V, &mv, 0, hv, t0, b, bb);
                tma_load_4d(smem + OFF_V + kBox, &mv, 64, hv, t0, b, bb);
            }
            last_v = n;
        };
        auto gates = [&](int n) {                          // decay products of chunk n
            const int pb = n & 1, t0 = n * kC;
            float g[2], be[2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int t = t0 + lane + 32 * h;
                if (t < S) {
                    const int64_t gi = g_base + static_cast<int64_t>(t) * g_ts;
                    g[h] = fmaxf(load_gate(p.log_decay, p.gate_dtype, gi), kMinLogDecay);
                    be[h] = load_gate(p.beta, p.gate_dtype, gi);
                } else {
                    g[h] = 0.f;
                    be[h] = 0.f;
                }
            }
            float c0 = g[0], c1 = g[1];                    // inclusive prefix sums
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float x0 = __shfl_up_sync(0xffffffffu, c0, off);
                const float x1 = __shfl_up_sync(0xffffffffu, c1, off);
                if (lane >= off) { c0 += x0; c1 += x1; }
            }
            const float m = __shfl_sync(0xffffffffu, c0, 31);       // cum_31: the reference
            c1 += m;
            const float tot = __shfl_sync(0xffffffffu, c1, 31);
            const float first = __shfl_sync(0xffffffffu, c0, 0);
            sc.cum[pb][lane] = c0;
            sc.cum[pb][lane + 32] = c1;
            sc.beta[pb][lane] = be[0];
            sc.beta[pb][lane + 32] = be[1];
            if (lane == 0) {
                sc.gamma[pb][0] = expf(tot);
                sc.gamma[pb][1] = (first - m <= 80.f && m - tot <= 80.f) ? 1.f : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_GATES + pb]);
        };
        // z rows of chunk n into L2 ahead of the output warps' gathers
        // the 64 rows (256 bytes each) of one head's tensor in chunk n into L2, two lanes per
        // row, from the load path (the tensor copy engine's queue stays free for the copies)
        const int64_t k_ts = p.head_major ? kD : static_cast<int64_t>(p.Hk) * kD;
        const int64_t k_base = p.head_major ? (static_cast<int64_t>(b) * p.Hk + hk) * S * kD
                                            : (static_cast<int64_t>(b) * S * p.Hk + hk) * kD;
        auto prefetch_rows = [&](const void *base, int64_t off, int64_t ts, int n) {
            const TA *src = static_cast<const TA *>(base) + off;
#pragma unroll
            for (int i = 0; i < kC / 16; i++) {
                const int t = n * kC + 16 * i + (lane >> 1);
                if (t < S) prefetch_line_l2(src + static_cast<int64_t>(t) * ts + 64 * (lane & 1));
            }
        };
        auto prefetch_z = [&](int n) {
            if (gated) prefetch_rows(p.z, v_base, v_ts, n);
        };
        // k, q and v of chunk n, ahead of their copies
        auto prefetch_kqv = [&](int n) {
            if (n >= nch) return;
            prefetch_rows(p.k, k_base, k_ts, n);
            prefetch_rows(p.q, k_base, k_ts, n);
            prefetch_rows(p.v, v_base, v_ts, n);
        };
        load_kq(0);
        load_v(0);
        if (nch > 1) {
            load_kq(1);
            prefetch_rows(p.v, v_base, v_ts, 1);
        }
        prefetch_kqv(2);
        prefetch_z(0);
        gates(0);
        if (nch > 1) {
            prefetch_z(1);
            gates(1);
        }
        for (int n = 1; n < nch; n++) {
            wait(B_U, static_cast<unsigned>((n - 1) & 1));  // U^T of n-1 has read v
            load_v(n);
            if (n + 1 < nch) {
                // slot (n+1) & 1 was last read by the update of chunk n-1
                wait(B_KQFREE + ((n + 1) & 1), static_cast<unsigned>(((n - 1) >> 1) & 1));
                load_kq(n + 1);
                prefetch_kqv(n + 2);
                prefetch_z(n + 1);
                // the scalars of parity (n+1) & 1 were last read by the output warps' scale
                // pass of chunk n-1, which precedes its intra-chunk MMAs
                wait(B_PFREE + ((n + 1) & 1), static_cast<unsigned>(((n - 1) >> 1) & 1));
                gates(n + 1);
            }
        }
        // drain the copies this warp issued (all consumed already unless the CTA abandoned)
        if (lane == 0) {
            for (int s = 0; s < 2; s++)
                if (last_kq[s] >= 0)
                    mbar_wait_bounded(&bar[B_LDKQ + s], static_cast<unsigned>((last_kq[s] >> 1) & 1), kLimitNs);
            if (last_v >= 0) mbar_wait_bounded(&bar[B_LDV], static_cast<unsigned>(last_v & 1), kLimitNs);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 wy_tensor_map_encoder() {
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

// A [B, S, H, 128] or [B, H, S, 128] 16-bit tensor seen with coordinates (w, h, t, b), boxes of
// 64 features x 1 head x 64 tokens x 1 batch, 128-byte swizzle; tokens past S read as zeros.
bool wy_encode_map(CUtensorMap *m, const void *base, const gdn_params &p, int H) {
    auto enc = wy_tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t W = kD, S = p.S, B = p.B;
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
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kC), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt =
        p.act_dtype == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 4, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename TA>
cudaError_t launch_wy(const gdn_params &p, cudaStream_t stream) {
    CUtensorMap mk, mq, mv;
    if (!wy_encode_map(&mk, p.k, p, p.Hk) || !wy_encode_map(&mq, p.q, p, p.Hk) ||
        !wy_encode_map(&mv, p.v, p, p.Hv))
        return cudaErrorInvalidValue;
    const int bytes = static_cast<int>(kSmemBytes);
    // the shared-memory attribute once per device (it persists in the device's context)
    constexpr int kDevices = 64;
    static std::atomic<bool> attr_set[kDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevices || !attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(gdn_scan_wy_kernel<TA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kDevices) attr_set[dev].store(true, std::memory_order_release);
    }
    const int64_t ctas = static_cast<int64_t>(p.B) * p.Hv;
    gdn_scan_wy_kernel<TA><<<static_cast<unsigned>(ctas), kThreads, bytes, stream>>>(p, mk, mq, mv);
    return cudaGetLastError();
}
}  // namespace

bool scan_wy_supported(const gdn_params &p) {
    auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    return (p.act_dtype == GDN_BF16 || p.act_dtype == GDN_F16) && p.Dk == kD && p.Dv == kD &&
           p.S > 0 && p.B > 0 && al16(p.q) && al16(p.k) && al16(p.v) &&
           wy_tensor_map_encoder() != nullptr;
}

cudaError_t launch_scan_wy(const gdn_params &p, cudaStream_t stream) {
    return p.act_dtype == GDN_BF16 ? launch_wy<__nv_bfloat16>(p, stream) : launch_wy<__half>(p, stream);
}

cudaError_t scan_wy_watchdog(unsigned *flag, cudaStream_t stream) {
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

cudaError_t scan_wy_set_first_wait_limit(unsigned long long ns, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyToSymbolAsync(g_wy_first_limit_ns, &ns, sizeof(ns), 0,
                                            cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e;
}

}  // namespace gdn
