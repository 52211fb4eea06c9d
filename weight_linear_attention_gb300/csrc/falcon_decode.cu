// Single-token step (T = 1) for Falcon-1, 1A, 2 and 2A with dk = dv = 64: the recurrent form of the
// update ("Fast Weight Attention for Continual Learning", paperlayer summary §3, Appendix p.34;
// agihunt explainer "Method"), one (batch, head) state per CTA. The state is read once and written
// once, so the step is bound by those 2 x 16 KB per head of HBM traffic.
//
// For the token at global position tau = pos + 1, with x = k_pos (the pending key of the tail; the
// x_1 = 0 sentinel when pos = 0), y = v, q:
//   eta = beta / (|x|^2 + lambda + eps) (0 when the denominator is 0, and at tau = 1)
//   alpha = min(eta lambda, 1 - eps_gamma) (0 at tau = 1), gamma = 1 - alpha
//   Falcon-1:  S' = gamma S + eta x (y - S^T x)^T      Falcon-1A: S' = gamma S + eta x y^T
//   Falcon-2, 2A: Falcon-1, 1A per value column c with beta_c (eta_c, gamma_c)
//   o = S'^T q (read after write), tail_out = k (the next step's x).
// fp32 arithmetic throughout; S_final may be the same buffer as S0 (each element is read and
// written by the same thread).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "falcon_internal.h"
#include "sm103_ptx.cuh"

namespace falcon {
namespace {

constexpr int kD = 64;
constexpr int kThreads = 128;  // thread t: columns 4 (t % 16) .. + 3, rows kRows (t / 16) .. + kRows - 1
constexpr int kRows = kD * 16 / kThreads;
constexpr int kGroups = kThreads / 16;  // row groups

struct DParams {
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    const float* lam;
    const float* S0;
    const void* tail;
    void* out;
    float* S_final;
    void* tail_out;
    long long pos;
    float eps, eps_gamma;
};

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ float get(const float4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; }
__device__ __forceinline__ void set(float4& v, int j, float x) {
    if (j == 0) v.x = x;
    else if (j == 1) v.y = x;
    else if (j == 2) v.z = x;
    else v.w = x;
}

template <typename Tin, int VAR>
__global__ void __launch_bounds__(kThreads) falcon_decode_kernel(const DParams p) {
    __shared__ float xs[kD], qs[kD], ys[kD], rs[kD], eta_s[kD], gam_s[kD];
    __shared__ float part[kGroups][kD];
    __shared__ float nx_s;
    // launched with programmatic stream serialisation: wait until the grid before this one in the
    // stream has finished and its writes are visible (a decode loop's previous step wrote this step's
    // state), then let the next grid start launching while this one runs
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31;
    const long long bh = blockIdx.x;
    const int cq = tid & 15, rg = tid >> 4, c0 = 4 * cq, r0 = kRows * rg;
    const Tin* q = static_cast<const Tin*>(p.q) + bh * kD;
    const Tin* k = static_cast<const Tin*>(p.k) + bh * kD;
    const Tin* v = static_cast<const Tin*>(p.v) + bh * kD;
    const bool first = p.pos == 0;  // tau = 1: x = 0, eta = alpha = 0

    // ---- the state tile of this thread (rows r0 .. r0 + kRows - 1, columns c0 .. c0 + 3)
    float4 sv[kRows];
#pragma unroll
    for (int m = 0; m < kRows; ++m)
        sv[m] = p.S0 ? *reinterpret_cast<const float4*>(p.S0 + (bh * kD + r0 + m) * kD + c0)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < kD) {
        xs[tid] = first ? 0.f : ldf(static_cast<const Tin*>(p.tail) + bh * kD + tid);
        qs[tid] = ldf(q + tid);
        ys[tid] = ldf(v + tid);
        if (p.tail_out) stf(static_cast<Tin*>(p.tail_out) + bh * kD + tid, ldf(k + tid));
    }
    __syncthreads();
    if (tid < 32) {  // |x|^2
        float a = xs[lane] * xs[lane] + xs[lane + 32] * xs[lane + 32];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) nx_s = a;
    }
    __syncthreads();
    if (tid < kD) {  // eta, gamma per value column (one value for Falcon-1 and 1A)
        float eta = 0.f, alpha = 0.f;
        if (!first) {
            const float lm = p.lam[bh];
            const float b = per_column(VAR) ? p.beta[bh * kD + tid] : p.beta[bh];
            const float den = nx_s + lm + p.eps;
            eta = den == 0.f ? 0.f : b / den;
            alpha = fminf(eta * lm, 1.f - p.eps_gamma);
        }
        eta_s[tid] = eta;
        gam_s[tid] = 1.f - alpha;
    }

    // ---- residual r = y - S^T x (Falcon-1, 2) or r = y (Falcon-1A)
    if (!inner_product(VAR)) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float a = 0.f;
#pragma unroll
            for (int m = 0; m < kRows; ++m) a = fmaf(get(sv[m], j), xs[r0 + m], a);
            part[rg][c0 + j] = a;
        }
    }
    __syncthreads();
    if (tid < kD) {
        float a = 0.f;
        if (!inner_product(VAR))
#pragma unroll
            for (int g = 0; g < kGroups; ++g) a += part[g][tid];
        rs[tid] = ys[tid] - a;
    }
    __syncthreads();

    // ---- S' = gamma S + eta x r^T, and this thread's part of o = S'^T q
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = c0 + j;
        const float g = gam_s[c], er = eta_s[c] * rs[c];
        float a = 0.f;
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
            const float s = fmaf(g, get(sv[m], j), er * xs[r0 + m]);
            set(sv[m], j, s);
            a = fmaf(s, qs[r0 + m], a);
        }
        part[rg][c] = a;
    }
    if (p.S_final)
#pragma unroll
        for (int m = 0; m < kRows; ++m) *reinterpret_cast<float4*>(p.S_final + (bh * kD + r0 + m) * kD + c0) = sv[m];
    __syncthreads();
    if (tid < kD) {
        float a = 0.f;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) a += part[g][tid];
        stf(static_cast<Tin*>(p.out) + bh * kD + tid, a);
    }
}

template <typename Tin>
cudaError_t launch_typed(const Launch& a, const DParams& p, cudaStream_t st) {
    void (*fn)(DParams) = nullptr;
    switch (a.variant) {
        case kF1: fn = falcon_decode_kernel<Tin, kF1>; break;
        case kF1A: fn = falcon_decode_kernel<Tin, kF1A>; break;
        case kF2: fn = falcon_decode_kernel<Tin, kF2>; break;
        case kF2A: fn = falcon_decode_kernel<Tin, kF2A>; break;
        default: return cudaErrorInvalidValue;
    }
    // programmatic stream serialisation: consecutive steps overlap one's launch with the other's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * a.H));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace

bool decode_supported(const Launch& a) {
    return a.T == 1 && !windowed(a.variant) && a.W == 1 && a.dk == kD &&
           a.dv == kD && a.B * a.H < (1LL << 31);
}

int launch_decode(const Launch& a, cudaStream_t st) {
    DParams p;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.beta = a.beta;
    p.lam = a.lam;
    p.S0 = a.S0;
    p.tail = a.tail;
    p.out = a.out;
    p.S_final = a.S_final;
    p.tail_out = a.tail_out;
    p.pos = a.pos;
    p.eps = a.eps;
    p.eps_gamma = a.eps_gamma;
    const cudaError_t e = a.bf16 ? launch_typed<__nv_bfloat16>(a, p, st) : launch_typed<float>(a, p, st);
    return e == cudaSuccess ? 0 : 4;
}

}  // namespace falcon
