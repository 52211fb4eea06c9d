// C-ABI front end: argument checking and kernel dispatch for falcon_fwd.
// The operation, layouts and error contract are documented in include/falcon.h.

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "falcon.h"
#include "falcon_internal.h"

// Scratch of falcon_fwd_static: a file-scope device array (one per device), never allocated.
static __device__ __align__(256) uint8_t g_static_workspace[FALCON_STATIC_WORKSPACE_BYTES];

namespace {

// Its address on the current device, looked up once per device.
void* static_workspace_address() {
    constexpr int kMaxDevices = 64;
    static void* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] && cudaGetSymbolAddress(&addr[dev], g_static_workspace) != cudaSuccess) addr[dev] = nullptr;
    return addr[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool pow2_head(int64_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void* p, size_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + bytes};
}

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

size_t tail_bytes_of(const falcon_dims_t* d) {
    const size_t es = d->dtype == FALCON_BF16 ? 2 : 4;
    const size_t per = (size_t)d->window * (size_t)d->dk + (size_t)(d->window - 1) * (size_t)d->dv;
    return (size_t)d->batch * (size_t)d->heads * per * es;
}

// Workspace bytes a call with these (validated) arguments can use: the scan path's; 0 for the
// single-token, fused and per-column kernels, which need none.
size_t workspace_need(const falcon::Launch& a) {
    if (falcon::decode_supported(a) || falcon::fused_supported(a) || falcon::colw_supported(a)) return 0;
    if (falcon::scan_supported(a)) return falcon::scan_workspace_bytes(a);
    return 0;
}

// Shape/variant/dtype/chunk checks (no pointers). Fills the size fields of `a`.
int validate_shape(int variant, const falcon_dims_t* d, int chunk, bool has_tail, falcon::Launch* a) {
    if (!d) return FALCON_ERR_INVALID_ARG;
    if (variant < FALCON_1 || variant > FALCON_3A) return FALCON_ERR_INVALID_ARG;
    if (d->batch < 0 || d->heads < 0 || d->seqlen < 0 || d->pos < 0) return FALCON_ERR_INVALID_ARG;
    if (d->dk <= 0 || d->dv <= 0) return FALCON_ERR_INVALID_ARG;
    if (!pow2_head(d->dk) || !pow2_head(d->dv)) return FALCON_ERR_UNSUPPORTED;
    if (d->dtype != FALCON_F32 && d->dtype != FALCON_BF16) return FALCON_ERR_UNSUPPORTED;
    if (d->window < 1) return FALCON_ERR_INVALID_ARG;
    const bool win = variant == FALCON_3 || variant == FALCON_3A;
    if (!win && d->window != 1) return FALCON_ERR_INVALID_ARG;
    if (d->window > 8) return FALCON_ERR_UNSUPPORTED;
    if (!(d->eps >= 0.f) || !(d->eps_gamma > 0.f && d->eps_gamma < 1.f)) return FALCON_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64) return chunk <= 0 ? FALCON_ERR_INVALID_ARG : FALCON_ERR_UNSUPPORTED;
    if (win && chunk * d->window > 128) return FALCON_ERR_UNSUPPORTED;
    if ((d->pos > 0) != has_tail) return FALCON_ERR_INVALID_ARG;
    a->variant = variant;
    a->B = d->batch;
    a->H = d->heads;
    a->T = d->seqlen;
    a->dk = d->dk;
    a->dv = d->dv;
    a->pos = d->pos;
    a->W = d->window;
    a->bf16 = d->dtype == FALCON_BF16;
    a->eps = d->eps;
    a->eps_gamma = d->eps_gamma;
    a->chunk = chunk;
    if (falcon::generic_smem_bytes(*a, 16, false) > 200 * 1024 && !falcon::fused_supported(*a) &&
        !falcon::colw_supported(*a))
        return FALCON_ERR_UNSUPPORTED;
    return FALCON_OK;
}

// Full argument check; fills `a` on success.
int validate(int variant, const void* q, const void* k, const void* v, const float* beta, const float* lambda,
             const float* S0, const void* tail, void* out, float* S_final, void* tail_out, const falcon_dims_t* d,
             int chunk, void* ws, size_t ws_bytes, falcon::Launch* a) {
    const int st = validate_shape(variant, d, chunk, tail != nullptr, a);
    if (st != FALCON_OK) return st;
    const int64_t BH = d->batch * d->heads;
    const int64_t tokens = BH * d->seqlen;
    const size_t es = d->dtype == FALCON_BF16 ? 2 : 4;
    if (tokens > 0 && (!q || !k || !v || !beta || !lambda || !out)) return FALCON_ERR_INVALID_ARG;

    const void* al16[] = {q, k, v, out, tail, tail_out, S0, S_final};
    for (const void* p : al16)
        if (p && !aligned(p, 16)) return FALCON_ERR_MISALIGNED;
    if ((beta && !aligned(beta, 4)) || (lambda && !aligned(lambda, 4))) return FALCON_ERR_MISALIGNED;
    if (ws && !aligned(ws, 256)) return FALCON_ERR_MISALIGNED;
    const size_t ws_need = workspace_need(*a);
    if (ws && ws_need > 0 && ws_bytes < ws_need) return FALCON_ERR_INVALID_ARG;

    // Every written buffer (out, S_final, tail_out and a used workspace) overlaps no input and no other
    // written buffer; the one exception is S_final equal to S0 exactly (an in-place state update).
    {
        const size_t bcols = (variant == FALCON_2 || variant == FALCON_2A) ? (size_t)d->dv : 1;
        const size_t sbytes = (size_t)BH * d->dk * d->dv * 4;
        const Range ins[] = {
            range_of(q, (size_t)tokens * d->dk * es), range_of(k, (size_t)tokens * d->dk * es),
            range_of(v, (size_t)tokens * d->dv * es), range_of(beta, (size_t)tokens * bcols * 4),
            range_of(lambda, (size_t)tokens * 4),
            S0 ? range_of(S0, sbytes) : Range{0, 0},
            tail ? range_of(tail, tail_bytes_of(d)) : Range{0, 0},
        };
        const Range outs[] = {
            tokens > 0 ? range_of(out, (size_t)tokens * d->dv * es) : Range{0, 0},
            S_final ? range_of(S_final, sbytes) : Range{0, 0},
            tail_out ? range_of(tail_out, tail_bytes_of(d)) : Range{0, 0},
            ws && ws_need > 0 ? range_of(ws, ws_need) : Range{0, 0},
        };
        const int ni = (int)(sizeof(ins) / sizeof(ins[0])), no = (int)(sizeof(outs) / sizeof(outs[0]));
        for (int o = 0; o < no; ++o) {
            for (int i = 0; i < ni; ++i) {
                const bool in_place = o == 1 && i == 5 && S0 == S_final;
                if (!in_place && overlaps(outs[o], ins[i])) return FALCON_ERR_INVALID_ARG;
            }
            for (int o2 = o + 1; o2 < no; ++o2)
                if (overlaps(outs[o], outs[o2])) return FALCON_ERR_INVALID_ARG;
        }
    }

    a->q = q;
    a->k = k;
    a->v = v;
    a->beta = beta;
    a->lam = lambda;
    a->S0 = S0;
    a->tail = tail;
    a->out = out;
    a->S_final = S_final;
    a->tail_out = tail_out;
    a->ws = ws_need > 0 ? ws : nullptr;
    a->ws_bytes = ws_need > 0 && ws ? ws_bytes : 0;
    return FALCON_OK;
}

// Launch the kernels for validated arguments (a.ws set only when a path uses it).
int dispatch(const falcon::Launch& a, cudaStream_t s) {
    if (a.B * a.H == 0) return FALCON_OK;
    if (falcon::decode_supported(a)) return falcon::launch_decode(a, s);
    if (falcon::fused_supported(a)) return falcon::launch_fused(a, s);
    // the per-column kernel loads beta by TMA (16-byte aligned base); otherwise the CUDA-core kernel
    if (falcon::colw_supported(a) && aligned(a.beta, 16)) return falcon::launch_colw(a, s);
    if (a.ws) return falcon::launch_scan(a, s);
    return falcon::launch_generic(a, s);
}

// Shape checks of falcon_bwd on top of validate_shape.
int validate_bwd_shape(int variant, const falcon_dims_t* d, int chunk, bool has_tail, falcon::Launch* a) {
    const int st = validate_shape(variant, d, chunk, has_tail, a);
    if (st != FALCON_OK) return st;
    return falcon::bwd_supported(*a) ? FALCON_OK : FALCON_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

int falcon_abi_version(void) { return 4; }

size_t falcon_tail_bytes(const falcon_dims_t* d) {
    if (!d || d->batch < 0 || d->heads < 0 || d->dk <= 0 || d->dv <= 0 || d->window < 1) return 0;
    return tail_bytes_of(d);
}

const char* falcon_status_string(int s) {
    switch (s) {
        case FALCON_OK: return "ok";
        case FALCON_ERR_INVALID_ARG: return "invalid argument";
        case FALCON_ERR_UNSUPPORTED: return "unsupported size, dtype, window, chunk or variant";
        case FALCON_ERR_MISALIGNED: return "pointer not aligned as required";
        case FALCON_ERR_CUDA: return "CUDA runtime error";
        case FALCON_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
        default: return "unknown status";
    }
}

int falcon_kernel_for(int variant, const falcon_dims_t* dims, int chunk) {
    falcon::Launch a = {};
    if (validate_shape(variant, dims, chunk, dims && dims->pos > 0, &a) != FALCON_OK) return 0;
    if (falcon::decode_supported(a)) return 4;
    if (falcon::fused_supported(a)) return 6;
    if (falcon::colw_supported(a)) return 7;
    if (falcon::scan_supported(a)) return 5;
    return 1;
}

size_t falcon_workspace_bytes(int variant, const falcon_dims_t* dims, int chunk) {
    falcon::Launch a = {};
    if (validate_shape(variant, dims, chunk, dims && dims->pos > 0, &a) != FALCON_OK) return 0;
    return workspace_need(a);
}

int falcon_fwd(int variant, const void* q, const void* k, const void* v, const float* beta, const float* lambda,
               const float* S0, const void* tail, void* out, float* S_final, void* tail_out,
               const falcon_dims_t* dims, int chunk, void* workspace, size_t workspace_bytes, void* stream) {
    falcon::Launch a = {};
    const int st = validate(variant, q, k, v, beta, lambda, S0, tail, out, S_final, tail_out, dims, chunk, workspace,
                            workspace_bytes, &a);
    if (st != FALCON_OK) return st;
    return dispatch(a, static_cast<cudaStream_t>(stream));
}

int falcon_fwd_static(int variant, const void* q, const void* k, const void* v, const float* beta,
                      const float* lambda, const float* S0, const void* tail, void* out, float* S_final,
                      void* tail_out, const falcon_dims_t* dims, int chunk, void* stream) {
    // Every argument is checked as falcon_fwd checks it (without a caller workspace: the library's array
    // overlaps no caller buffer), before anything touches the device.
    falcon::Launch a = {};
    const int st = validate(variant, q, k, v, beta, lambda, S0, tail, out, S_final, tail_out, dims, chunk, nullptr,
                            0, &a);
    if (st != FALCON_OK) return st;
    // The array's device address is looked up on every call (once per device, then cached), whether or
    // not this call uses it, so that the first call on a device always does the set-up.
    void* const scratch = static_workspace_address();
    if (!scratch) return FALCON_ERR_CUDA;
    const size_t need = workspace_need(a);
    if (need > 0 && need <= FALCON_STATIC_WORKSPACE_BYTES) {  // else the CUDA-core chunk kernel runs
        a.ws = scratch;
        a.ws_bytes = FALCON_STATIC_WORKSPACE_BYTES;
    }
    return dispatch(a, static_cast<cudaStream_t>(stream));
}

size_t falcon_bwd_workspace_bytes(int variant, const falcon_dims_t* dims, int chunk) {
    falcon::Launch a = {};
    if (validate_bwd_shape(variant, dims, chunk, dims && dims->pos > 0, &a) != FALCON_OK) return 0;
    return falcon::bwd_workspace_bytes(a);
}

int falcon_bwd(int variant, const void* q, const void* k, const void* v, const float* beta, const float* lambda,
               const float* S0, const void* tail, const void* dout, const float* dS_final, float* dq, float* dk,
               float* dv, float* dbeta, float* dlambda, float* dS0, float* dtail, const falcon_dims_t* dims,
               int chunk, void* workspace, size_t workspace_bytes, void* stream) {
    falcon::Launch a = {};
    int st = validate_bwd_shape(variant, dims, chunk, tail != nullptr, &a);
    if (st != FALCON_OK) return st;
    const int64_t BH = a.B * a.H;
    const int64_t tokens = BH * a.T;
    const size_t es = a.bf16 ? 2 : 4;
    if (dtail && a.pos == 0) return FALCON_ERR_INVALID_ARG;
    if (tokens > 0 && (!q || !k || !v || !beta || !lambda || !dout || !dq || !dk || !dv || !dbeta || !dlambda))
        return FALCON_ERR_INVALID_ARG;
    const size_t need = falcon::bwd_workspace_bytes(a);
    if (need > 0 && (!workspace || workspace_bytes < need)) return FALCON_ERR_INVALID_ARG;
    const void* al16[] = {q, k, v, tail, dout, S0, dS_final, dq, dk, dv, dS0, dtail};
    for (const void* p : al16)
        if (p && !aligned(p, 16)) return FALCON_ERR_MISALIGNED;
    const void* al4[] = {beta, lambda, dbeta, dlambda};
    for (const void* p : al4)
        if (p && !aligned(p, 4)) return FALCON_ERR_MISALIGNED;
    if (workspace && !aligned(workspace, 256)) return FALCON_ERR_MISALIGNED;
    // every written buffer (the gradients and the workspace) overlaps no other argument
    const size_t sbytes = (size_t)BH * a.dk * a.dv * 4;
    const Range ins[] = {
        range_of(q, (size_t)tokens * a.dk * es), range_of(k, (size_t)tokens * a.dk * es),
        range_of(v, (size_t)tokens * a.dv * es), range_of(beta, (size_t)tokens * 4),
        range_of(lambda, (size_t)tokens * 4), range_of(dout, (size_t)tokens * a.dv * es),
        S0 ? range_of(S0, sbytes) : Range{0, 0}, dS_final ? range_of(dS_final, sbytes) : Range{0, 0},
        tail ? range_of(tail, tail_bytes_of(dims)) : Range{0, 0},
    };
    const Range outs[] = {
        range_of(dq, (size_t)tokens * a.dk * 4), range_of(dk, (size_t)tokens * a.dk * 4),
        range_of(dv, (size_t)tokens * a.dv * 4), range_of(dbeta, (size_t)tokens * 4),
        range_of(dlambda, (size_t)tokens * 4), dS0 ? range_of(dS0, sbytes) : Range{0, 0},
        dtail ? range_of(dtail, (size_t)BH * a.dk * 4) : Range{0, 0},
        need > 0 ? range_of(workspace, need) : Range{0, 0},
    };
    const int no = (int)(sizeof(outs) / sizeof(outs[0]));
    for (int i = 0; i < no; ++i) {
        for (const Range& r : ins)
            if (overlaps(outs[i], r)) return FALCON_ERR_INVALID_ARG;
        for (int j = i + 1; j < no; ++j)
            if (overlaps(outs[i], outs[j])) return FALCON_ERR_INVALID_ARG;
    }
    if (BH == 0) return FALCON_OK;
    a.q = q;
    a.k = k;
    a.v = v;
    a.beta = beta;
    a.lam = lambda;
    a.S0 = S0;
    a.tail = tail;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    falcon::BwdArgs g = {dout, dS_final, dq, dk, dv, dbeta, dlambda, dS0, dtail};
    return falcon::launch_bwd(a, g, static_cast<cudaStream_t>(stream));
}

int falcon_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FALCON_ERR_CUDA;
    int f = 0, g = 0, h = 0, k = 0, b = 0;
    if (falcon::fused_consume_timeout_flag(&f) != 0 || falcon::colw_consume_timeout_flag(&g) != 0 ||
        falcon::f3map_consume_timeout_flag(&h) != 0 || falcon::scan_tc_consume_timeout_flag(&k) != 0 ||
        falcon::bwd_consume_timeout_flag(&b) != 0)
        return FALCON_ERR_CUDA;
    return f || g || h || k || b ? FALCON_ERR_DEVICE_TIMEOUT : FALCON_OK;
}

}  // extern "C"
