// gdn_api.cu -- the C ABI of libgdn.so: host-side validation, then the kernel launchers.
//
// Validation mirrors the role of torch_to_nnef.op.gated_delta, native_gdn_reject_reason
// (hard constraints checked before anything runs, a short reason string); unlike the page's
// exporter there is no fallback: a rejected call returns its status and enqueues nothing.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

thread_local char g_last_error[256] = "";

struct Range {
    uintptr_t lo, hi;   // [lo, hi) in bytes; empty when lo == hi
};

bool overlaps(Range a, Range b) {
    return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

Range span(const void *ptr, int64_t elems, int64_t elem_bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
    return Range{lo, ptr ? lo + static_cast<uintptr_t>(elems * elem_bytes) : lo};
}

int64_t dtype_bytes(int dt) {
    switch (dt) {
        case GDN_F32: return 4;
        case GDN_BF16:
        case GDN_F16: return 2;
        default: return 0;
    }
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }


// Returns GDN_OK or a status, and sets *why to a static reason.
int check(const gdn_params *p, int is_decode, const char **why) {
    *why = nullptr;
    if (p == nullptr) { *why = "params pointer is NULL"; return GDN_ERR_NULL_PTR; }
    if ((p->flags & ~(GDN_FLAG_SCAN_TMEM | GDN_FLAG_HOST_IO | GDN_FLAG_SCAN_BLOCK16 |
                      GDN_FLAG_SCAN_CHUNKED)) != 0) {
        *why = "unknown flags bit";
        return GDN_ERR_BAD_ARG;
    }
    if (is_decode && (p->flags & GDN_FLAG_SCAN_TMEM)) {
        *why = "flags: GDN_FLAG_SCAN_TMEM applies to gdn_scan only";
        return GDN_ERR_BAD_ARG;
    }
    const int kernel_bits = p->flags & (GDN_FLAG_SCAN_TMEM | GDN_FLAG_SCAN_BLOCK16 | GDN_FLAG_SCAN_CHUNKED);
    if (kernel_bits & (kernel_bits - 1)) {
        *why = "flags: at most one of GDN_FLAG_SCAN_TMEM, GDN_FLAG_SCAN_BLOCK16, GDN_FLAG_SCAN_CHUNKED";
        return GDN_ERR_BAD_ARG;
    }
    if (is_decode && (p->flags & GDN_FLAG_SCAN_CHUNKED)) {
        *why = "flags: GDN_FLAG_SCAN_CHUNKED applies to gdn_scan only";
        return GDN_ERR_BAD_ARG;
    }
    if (is_decode && (p->flags & GDN_FLAG_SCAN_BLOCK16)) {
        *why = "flags: GDN_FLAG_SCAN_BLOCK16 applies to gdn_scan only";
        return GDN_ERR_BAD_ARG;
    }
    if (!is_decode && (p->flags & GDN_FLAG_HOST_IO)) {
        *why = "flags: GDN_FLAG_HOST_IO applies to gdn_decode_step only";
        return GDN_ERR_BAD_ARG;
    }
    if (p->B < 0 || p->S < 0) { *why = "B and S must be >= 0"; return GDN_ERR_BAD_SHAPE; }
    if (p->Hk < 1 || p->Hv < 1) { *why = "Hk and Hv must be >= 1"; return GDN_ERR_BAD_SHAPE; }
    if (p->Hv % p->Hk != 0) {
        *why = "Hv must be a multiple of Hk (value_heads_per_group)";
        return GDN_ERR_BAD_SHAPE;
    }
    if (is_decode && p->S != 1) { *why = "decode step requires S == 1"; return GDN_ERR_BAD_SHAPE; }
    if (p->head_major != 0 && p->head_major != 1) {
        *why = "head_major must be 0 or 1";
        return GDN_ERR_BAD_ARG;
    }
    if (p->Dk < 1 || p->Dv < 1) { *why = "Dk and Dv must be >= 1"; return GDN_ERR_BAD_SHAPE; }
    if (!(gdn::tiled_dim(p->Dk) && gdn::tiled_dim(p->Dv)) && !gdn::general_supported(p->Dk, p->Dv)) {
        *why = "Dk and Dv must be at most 256, with the head's memory (Dv padded rows of Dk "
               "floats) within 226 KB unless both are multiples of 16 up to 128, or 256";
        return GDN_ERR_UNSUPPORTED_DIM;
    }
    const int64_t eact = dtype_bytes(p->act_dtype);
    if (eact == 0) { *why = "act_dtype must be GDN_F32, GDN_BF16 or GDN_F16"; return GDN_ERR_BAD_DTYPE; }
    if (p->gate_dtype != GDN_F32 && p->gate_dtype != p->act_dtype) {
        *why = "gate_dtype must be GDN_F32 or equal to act_dtype";
        return GDN_ERR_BAD_DTYPE;
    }
    const int64_t egate = dtype_bytes(p->gate_dtype);
    if (!(p->qk_eps >= 0.f) || !isfinite(p->qk_eps) || !(p->norm_eps >= 0.f) ||
        !isfinite(p->norm_eps)) {
        *why = "qk_eps and norm_eps must be finite and >= 0";
        return GDN_ERR_BAD_ARG;
    }

    const int64_t B = p->B, S = p->S, Hk = p->Hk, Hv = p->Hv, Dk = p->Dk, Dv = p->Dv;
    // sizes: every element count must stay below 2^40 and the grid below 2^31 CTAs
    const int64_t lim = int64_t(1) << 40;
    if (B * Hv > (int64_t(1) << 30) || B * S > lim / (Hv * Dv) || B * S > lim / (Hk * Dk) ||
        B * Hv > lim / (Dv * Dk)) {
        *why = "tensor too large";
        return GDN_ERR_BAD_ARG;
    }
    if (B == 0) return GDN_OK;   // nothing to do, nothing dereferenced
    // y is untouched (and may be NULL) when S == 0
    if (p->state == nullptr || (p->y == nullptr && S > 0)) {
        *why = "state and y are required";
        return GDN_ERR_NULL_PTR;
    }
    if (S > 0 && (p->z == nullptr) != (p->gn == nullptr)) {
        *why = "z and gn must both be given or both be NULL";
        return GDN_ERR_NULL_PTR;
    }
    if (S > 0 && (p->q == nullptr || p->k == nullptr || p->v == nullptr ||
                  p->log_decay == nullptr || p->beta == nullptr)) {
        *why = "q, k, v, log_decay and beta are required";
        return GDN_ERR_NULL_PTR;
    }
    // alignment: vector loads of 16 bytes on every activation / state operand
    const void *vec[] = {p->q, p->k, p->v, p->z, p->gn, p->s0, p->state, p->y};
    for (const void *ptr : vec)
        if (ptr && !aligned(ptr, 16)) { *why = "operands must be 16-byte aligned"; return GDN_ERR_MISALIGNED; }
    if ((p->log_decay && !aligned(p->log_decay, egate)) || (p->beta && !aligned(p->beta, egate))) {
        *why = "log_decay and beta must be aligned to their element size";
        return GDN_ERR_MISALIGNED;
    }
    // aliasing: y is written while every operand is read
    const int64_t n_qk = B * S * Hk * Dk, n_v = B * S * Hv * Dv, n_g = B * S * Hv;
    const int64_t n_state = B * Hv * Dv * Dk;
    const Range ry = span(p->y, n_v, 4);
    const Range token_reads[] = {span(p->q, n_qk, eact),         span(p->k, n_qk, eact),
                                 span(p->v, n_v, eact),          span(p->z, n_v, eact),
                                 span(p->log_decay, n_g, egate), span(p->beta, n_g, egate),
                                 span(p->gn, Dv, 4)};
    const Range rs = span(p->state, n_state, 4);
    for (const Range &r : token_reads)
        if (overlaps(ry, r)) { *why = "y overlaps an operand"; return GDN_ERR_ALIASING; }
    if (overlaps(ry, rs) || (!is_decode && overlaps(ry, span(p->s0, n_state, 4)))) {
        *why = "y overlaps an operand";
        return GDN_ERR_ALIASING;
    }
    for (const Range &r : token_reads)
        if (overlaps(rs, r)) { *why = "state overlaps an operand"; return GDN_ERR_ALIASING; }
    if (!is_decode && p->s0 && p->s0 != p->state && overlaps(rs, span(p->s0, n_state, 4))) {
        *why = "state partially overlaps s0 (only s0 == state is allowed)";
        return GDN_ERR_ALIASING;
    }
    return GDN_OK;
}

// gdn_scan_split's own arguments (after check(p, 0) passed).
int check_split(const gdn_params *p, int segments, const void *ws, size_t ws_bytes,
                const char **why) {
    *why = nullptr;
    if (segments < 1) { *why = "segments must be >= 1"; return GDN_ERR_BAD_ARG; }
    if (p->flags & GDN_FLAG_SCAN_TMEM) {
        *why = "flags: GDN_FLAG_SCAN_TMEM applies to gdn_scan only";
        return GDN_ERR_BAD_ARG;
    }
    const size_t need = gdn::scan_split_workspace_floats(*p, segments) * sizeof(float);
    if (p->B == 0 || need == 0) return GDN_OK;             // one segment: no workspace used
    if (ws == nullptr) { *why = "workspace is required"; return GDN_ERR_NULL_PTR; }
    if (!aligned(ws, 16)) { *why = "workspace must be 16-byte aligned"; return GDN_ERR_MISALIGNED; }
    if (ws_bytes < need) { *why = "workspace too small (see gdn_scan_split_workspace)"; return GDN_ERR_BAD_ARG; }
    const int64_t B = p->B, S = p->S, Hk = p->Hk, Hv = p->Hv, Dk = p->Dk, Dv = p->Dv;
    const int64_t eact = dtype_bytes(p->act_dtype), egate = dtype_bytes(p->gate_dtype);
    const int64_t n_qk = B * S * Hk * Dk, n_v = B * S * Hv * Dv, n_g = B * S * Hv;
    const int64_t n_state = B * Hv * Dv * Dk;
    const Range rw{reinterpret_cast<uintptr_t>(ws), reinterpret_cast<uintptr_t>(ws) + need};
    const Range all[] = {span(p->q, n_qk, eact),         span(p->k, n_qk, eact),
                         span(p->v, n_v, eact),          span(p->z, n_v, eact),
                         span(p->log_decay, n_g, egate), span(p->beta, n_g, egate),
                         span(p->gn, Dv, 4),             span(p->s0, n_state, 4),
                         span(p->state, n_state, 4),     span(p->y, n_v, 4)};
    for (const Range &r : all)
        if (overlaps(rw, r)) { *why = "workspace overlaps an operand"; return GDN_ERR_ALIASING; }
    return GDN_OK;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int gdn_decode_step(const gdn_params *p, void *stream) {
    const char *why;
    const int st = check(p, 1, &why);
    if (st != GDN_OK) return st;
    if (p->B == 0) return GDN_OK;
    return cuda_status(gdn::launch_decode(*p, static_cast<cudaStream_t>(stream)));
}

int gdn_scan(const gdn_params *p, void *stream) {
    const char *why;
    const int st = check(p, 0, &why);
    if (st != GDN_OK) return st;
    if (p->B == 0) return GDN_OK;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->S == 0) {
        const size_t bytes = sizeof(float) * static_cast<size_t>(p->B) * p->Hv * p->Dv * p->Dk;
        if (p->s0 == p->state) return GDN_OK;
        if (p->s0) return cuda_status(cudaMemcpyAsync(p->state, p->s0, bytes, cudaMemcpyDeviceToDevice, s));
        return cuda_status(cudaMemsetAsync(p->state, 0, bytes, s));
    }
    return cuda_status(gdn::launch_scan(*p, s));
}

size_t gdn_scan_split_workspace(const gdn_params *p, int segments) {
    const char *why;
    if (check(p, 0, &why) != GDN_OK || segments < 1 || p->B == 0) return 0;
    return gdn::scan_split_workspace_floats(*p, segments) * sizeof(float);
}

int gdn_scan_split(const gdn_params *p, int segments, void *workspace, size_t workspace_bytes,
                   void *stream) {
    const char *why;
    int st = check(p, 0, &why);
    if (st != GDN_OK) return st;
    st = check_split(p, segments, workspace, workspace_bytes, &why);
    if (st != GDN_OK) {
        snprintf(g_last_error, sizeof g_last_error, "%s", why);
        return st;
    }
    if (p->B == 0 || p->S == 0) return gdn_scan(p, stream);
    return cuda_status(gdn::launch_scan_split(*p, segments, static_cast<float *>(workspace),
                                              static_cast<cudaStream_t>(stream)));
}

const char *gdn_reject_reason(const gdn_params *p, int is_decode) {
    const char *why;
    return check(p, is_decode, &why) == GDN_OK ? nullptr : why;
}

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL_PTR: return "a required pointer is NULL (or only one of z, gn given)";
        case GDN_ERR_BAD_SHAPE: return "bad shape (dims, Hv % Hk, or S != 1 on decode)";
        case GDN_ERR_UNSUPPORTED_DIM: return "unsupported head dim (above 256, or a memory too large for the general kernel)";
        case GDN_ERR_BAD_DTYPE: return "bad dtype";
        case GDN_ERR_MISALIGNED: return "misaligned pointer";
        case GDN_ERR_ALIASING: return "output overlaps an operand";
        case GDN_ERR_BAD_ARG: return "bad argument (eps, flag, flags bits or size)";
        case GDN_ERR_CUDA: return "CUDA error (see gdn_last_error)";
        case GDN_ERR_TIMEOUT: return "a kernel timed out waiting for its own copies";
        default: return "unknown status";
    }
}

const char *gdn_last_error(void) { return g_last_error; }

int gdn_device_status(void *stream) {
    unsigned flag_decode = 0, flag_scan = 0;
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    int st = cuda_status(gdn::decode_watchdog(&flag_decode, st_));
    if (st != GDN_OK) return st;
    st = cuda_status(gdn::scan_watchdog(&flag_scan, st_));
    if (st != GDN_OK) return st;
    return (flag_decode | flag_scan) ? GDN_ERR_TIMEOUT : GDN_OK;
}

int gdn_selftest_wait_timeout(void *stream, double limit_ms) {
    if (!(limit_ms > 0.0 && limit_ms <= 2000.0)) return GDN_ERR_BAD_ARG;
    const uint64_t ns = static_cast<uint64_t>(limit_ms * 1e6);
    return cuda_status(gdn::launch_wait_timeout(static_cast<cudaStream_t>(stream), ns));
}

int gdn_selftest_scan_wait_limit(void *stream, double limit_us) {
    if (!(limit_us >= 0.0 && limit_us <= 2e6)) return GDN_ERR_BAD_ARG;
    const unsigned long long ns = static_cast<unsigned long long>(limit_us * 1e3);
    return cuda_status(gdn::scan_wy_set_first_wait_limit(limit_us > 0.0 && ns == 0 ? 1 : ns,
                                                         static_cast<cudaStream_t>(stream)));
}

int gdn_version(void) { return GDN_VERSION; }

}  // extern "C"

// ------------------------------------------------------------ gdn_scan_split_noalloc
//
// The split scan for callers that may not allocate device memory: code that runs inside
// another framework's memory pool or arena, or on a path where a cudaMalloc would
// synchronise the device or fail.  Its scratch (transitions, offsets and start memories of
// the segments) is one fixed array of this translation unit; every device that loads the
// library holds it until the process exits.

namespace {

static __device__ __align__(256) unsigned char g_split_scratch[GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];   // device address of g_split_scratch per device ordinal

// The device address of the scratch array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per device (with that
// device current) and kept.
int split_scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(g_last_error, sizeof g_last_error, "device ordinal %d beyond %d", dev, kMaxDevices);
        return GDN_ERR_BAD_ARG;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_split_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        g_scratch_addr[dev] = addr;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_scan_split_noalloc(const gdn_params *p, int segments, void *stream) {
    const char *why;
    int st = check(p, 0, &why);
    if (st != GDN_OK) return st;
    if (segments < 1) {
        snprintf(g_last_error, sizeof g_last_error, "segments must be >= 1");
        return GDN_ERR_BAD_ARG;
    }
    if (p->flags & GDN_FLAG_SCAN_TMEM) {
        snprintf(g_last_error, sizeof g_last_error,
                 "flags: GDN_FLAG_SCAN_TMEM applies to gdn_scan only");
        return GDN_ERR_BAD_ARG;
    }
    if (p->B == 0 || p->S == 0) return gdn_scan(p, stream);
    const size_t need = gdn::scan_split_workspace_floats(*p, segments) * sizeof(float);
    if (need > GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES) {
        snprintf(g_last_error, sizeof g_last_error,
                 "split scratch of %zu bytes exceeds the fixed %zu bytes of "
                 "gdn_scan_split_noalloc (use fewer segments, or gdn_scan_split with a "
                 "workspace)", need, static_cast<size_t>(GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES));
        return GDN_ERR_BAD_ARG;
    }
    void *scratch = nullptr;
    if (need > 0 && (st = split_scratch_address(&scratch)) != GDN_OK) return st;
    // every scratch element is written before it is read: nothing needs clearing
    return cuda_status(gdn::launch_scan_split(*p, segments, static_cast<float *>(scratch),
                                              static_cast<cudaStream_t>(stream)));
}
