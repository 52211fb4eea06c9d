// Single-token step (T = 1) for Falcon-1, 1A, 2 and 2A with dk = dv = 64: the recurrent form of the
// update ("Fast Weight Attention for Continual Learning", paperlayer summary §3, Appendix p.34;
// agihunt explainer "Method"), one (batch, head) state per CTA, each of its four warps on 16 value
// columns. The state is read once and written once, so the step is bound by those 2 x 16 KB per head
// of HBM traffic.
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

namespace falcon {
namespace {

constexpr int kD = 64;
constexpr int kThreads = 128;  // four warps; warp w owns value columns 16 w .. 16 w + 15 of one head
constexpr int kHalf = 32;      // rows per lane: lane l holds column 16 w + (l & 15), rows 32 (l >> 4) .. + 31

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

// Each warp works alone on its 16 columns (the columns of the update are independent once |x|^2 is
// known), so the step needs no CTA barrier: a lane's 32 state values are loaded at once, its partial
// sums over its 32 rows meet the other half's by one shuffle.
template <typename Tin, int VAR>
__global__ void __launch_bounds__(kThreads) falcon_decode_kernel(const DParams p) {
    __shared__ float xs[kThreads / 32][kD], qs[kThreads / 32][kD];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long bh = blockIdx.x;
    const int c = 16 * warp + (lane & 15), r0 = kHalf * (lane >> 4);
    const bool first = p.pos == 0;  // tau = 1: x = 0, eta = alpha = 0

    // the lane's state values, all loads issued at once
    float sv[kHalf];
    const float* s0 = p.S0 ? p.S0 + (bh * kD + r0) * kD + c : nullptr;
#pragma unroll
    for (int j = 0; j < kHalf; ++j) sv[j] = s0 ? s0[j * kD] : 0.f;
    // x (the pending key), q, this column's target
    const Tin* q = static_cast<const Tin*>(p.q) + bh * kD;
    float x0 = 0.f, x1 = 0.f;
    if (!first) {
        const Tin* tl = static_cast<const Tin*>(p.tail) + bh * kD;
        x0 = ldf(tl + 2 * lane);
        x1 = ldf(tl + 2 * lane + 1);
    }
    xs[warp][2 * lane] = x0;
    xs[warp][2 * lane + 1] = x1;
    qs[warp][2 * lane] = ldf(q + 2 * lane);
    qs[warp][2 * lane + 1] = ldf(q + 2 * lane + 1);
    const float y = ldf(static_cast<const Tin*>(p.v) + bh * kD + c);
    if (p.tail_out && warp == 0) {
        const Tin* kk = static_cast<const Tin*>(p.k) + bh * kD;
        stf(static_cast<Tin*>(p.tail_out) + bh * kD + 2 * lane, ldf(kk + 2 * lane));
        stf(static_cast<Tin*>(p.tail_out) + bh * kD + 2 * lane + 1, ldf(kk + 2 * lane + 1));
    }
    float nx = x0 * x0 + x1 * x1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nx += __shfl_xor_sync(0xffffffffu, nx, o);
    __syncwarp();
    float eta = 0.f, alpha = 0.f;
    if (!first) {
        const float lm = p.lam[bh];
        const float b = per_column(VAR) ? p.beta[bh * kD + c] : p.beta[bh];
        const float den = nx + lm + p.eps;
        eta = den == 0.f ? 0.f : b / den;
        alpha = fminf(eta * lm, 1.f - p.eps_gamma);
    }
    const float* xw = xs[warp] + r0;
    const float* qw = qs[warp] + r0;
    // r = y - S^T x (Falcon-1, 2) or y (Falcon-1A, 2A)
    float r = y;
    if (!inner_product(VAR)) {
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < kHalf; ++j) a = fmaf(sv[j], xw[j], a);
        a += __shfl_xor_sync(0xffffffffu, a, 16);
        r = y - a;
    }
    // S' = gamma S + eta x r^T, and o = S'^T q
    const float g = 1.f - alpha, er = eta * r;
    float o = 0.f;
#pragma unroll
    for (int j = 0; j < kHalf; ++j) {
        sv[j] = fmaf(g, sv[j], er * xw[j]);
        o = fmaf(sv[j], qw[j], o);
    }
    o += __shfl_xor_sync(0xffffffffu, o, 16);
    if (p.S_final) {
        float* sf = p.S_final + (bh * kD + r0) * kD + c;
#pragma unroll
        for (int j = 0; j < kHalf; ++j) sf[j * kD] = sv[j];
    }
    if (lane < 16) stf(static_cast<Tin*>(p.out) + bh * kD + c, o);
}

template <typename Tin>
cudaError_t launch_typed(const Launch& a, const DParams& p, cudaStream_t st) {
    const unsigned grid = (unsigned)(a.B * a.H);
    switch (a.variant) {
        case kF1: falcon_decode_kernel<Tin, kF1><<<grid, kThreads, 0, st>>>(p); break;
        case kF1A: falcon_decode_kernel<Tin, kF1A><<<grid, kThreads, 0, st>>>(p); break;
        case kF2: falcon_decode_kernel<Tin, kF2><<<grid, kThreads, 0, st>>>(p); break;
        case kF2A: falcon_decode_kernel<Tin, kF2A><<<grid, kThreads, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
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
