// Chunk-parallel backward pass of Falcon-1 and 1A (dk = dv = 64, chunk 64, fp32 or bf16 inputs,
// fp32 arithmetic and gradients). "Fast Weight Attention for Continual Learning", paperlayer summary
// §D.2, §E.3, §G.3: reverse the output materialisation, the inter-chunk recurrence and the local
// structure, backpropagate through the triangular solve, the Gram matrix, the chunk-local decay
// prefixes, the clamp and the step-size normalisation.
//
// Per chunk of C tokens (rows i, j; X the shifted keys, Q, Y = V, dO the output adjoint; eta_j,
// L_i = sum_{u<=i} log(1 - alpha_u) reset at the chunk start, Lx_i = L_{i-1}; S the chunk-start state,
// dS' the adjoint of the chunk-end state):
//   forward   A_ij = eta_j e^{Lx_i - L_j} x_i.x_j (j < i), P_ij = eta_j e^{L_i - L_j} q_i.x_j (j <= i),
//             T = (I + A)^-1, R = T (Y - diag(e^Lx) X S), O = diag(e^L) Q S + P R,
//             S' = e^{L_C} S + X^T diag(w) R with w_j = eta_j e^{L_C - L_j}      (Falcon-1A: R = Y)
//   backward  dR = P^T dO + diag(w) X dS',  dZ = T^T dR,  dV = dZ,
//             dP = dO R^T (j <= i),  dA = -dZ R^T (j < i),
//             dQ = diag(e^L) dO S^T + dSc X,  dX = dSc^T Q + (dG + dG^T) X - diag(e^Lx) dZ S^T
//                  + diag(w) R dS'^T + 2 dden x,  with dSc_ij = dP_ij eta_j e^{L_i - L_j} and
//                  dG_ij = dA_ij eta_j e^{Lx_i - L_j},
//             d eta, d L from every factor, d log(gamma_u) = sum_{i >= u} dL_i inside the chunk,
//             d alpha = -d log(gamma) / gamma where the clamp is inactive (0 where it binds),
//             eta = beta / den: d beta = d eta / den, d den = -d eta eta / den (none where eta is 0
//             by definition: a zero denominator or the first step of a fresh sequence).
// The chunk-start state adjoint is dS = M^T dS' + V with M = e^{L_C} I - X^T diag(w) T diag(e^Lx) X
// and V = Q^T diag(e^L) dO - X^T diag(e^Lx) T^T P^T dO, so three launches do the whole pass:
//   falcon_bwd_prep   every chunk at once: T, the forward transition (M and M^T, U = X^T diag(w) T Y)
//                     and V;
//   falcon_bwd_chain  per sequence (one CTA, the carried matrix in tensor memory, one tcgen05 product
//                     per step): S_{n+1} = M_n S_n + U_n forward, then dS_n = M_n^T dS_{n+1} + V_n
//                     backward, storing S_n and dS_{n+1};
//   falcon_bwd_grad   every chunk at once: all input gradients from S_n and dS_{n+1}.
// The 64 x 64 x 64 products of prep and grad run on the tensor cores as warp-level tf32 MMAs with
// every fp32 operand split into a tf32 head and remainder (fp32-accurate); the scans, the scalars
// and the triangular inverse run on the CUDA cores in fp32.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "falcon_internal.h"
#include "sm103_ptx.cuh"

namespace falcon {

__device__ int g_bwd_timeout_flag = 0;

namespace {

constexpr int kD = 64;        // dk = dv
constexpr int kC = 64;        // chunk length
constexpr int kLd = 68;       // shared-memory row stride (floats): 16-byte rows, tensor-core fragments
constexpr int kMat = kC * kLd;
constexpr int kThreads = 512;       // prep and gradient kernels: 16 warps
constexpr int kWsMat = kD * kD;             // floats per workspace matrix
constexpr int kWsChunk = 7 * kWsMat;        // M, U, V, T, S_n, dS_{n+1}, M^T
enum { kWsM = 0, kWsU = 1, kWsV = 2, kWsT = 3, kWsS = 4, kWsDS = 5, kWsMT = 6 };

struct BParams {
    const void* q;
    const void* k;
    const void* v;
    const void* dout;
    const void* tail;  // pending key k_pos [BH][dk] (pos > 0) or null
    const float* beta;
    const float* lam;
    const float* S0;
    const float* dS_final;
    float* dq;
    float* dk;
    float* dv;
    float* dbeta;
    float* dlam;
    float* dS0;
    float* dtail;
    float* ws;
    long long T, pos, N, BH;  // tokens, position, chunks per sequence, sequences
    float eps, eps_gamma;
};

// Scalars of one chunk, recomputed identically by the prep and gradient kernels.
struct Scal {
    float eta[kC], lam[kC], den[kC], gam[kC], L[kC], Lx[kC], eL[kC], eLx[kC], w[kC];
    int unc[kC], live[kC];  // clamp inactive (alpha differentiable); eta = beta / den differentiable
    float eLC;
};

// Tile loads: every thread issues all of its 16-byte loads of the chunk's tiles before it stores
// any of them to shared memory, so their latencies overlap.
__device__ __forceinline__ void put(float* d, const uint4& v, const float*) {
    d[0] = __uint_as_float(v.x);
    d[1] = __uint_as_float(v.y);
    d[2] = __uint_as_float(v.z);
    d[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void put(float* d, const uint4& v, const __nv_bfloat16*) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        d[2 * h] = __uint_as_float(w[h] << 16);
        d[2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
    }
}

// Rows t0 .. t0 + nr - 1 of the [BH, T, 64] tensors k (shifted: x_t = k_{t-1}, row -1 the tail key or
// zero), q, v and dout into four shared 64 x 64 tiles (zero rows past nr).
template <typename Tin>
__device__ void load_inputs(float* X, float* Q, float* Y, float* dO, const BParams& p, long long bh, long long t0,
                            int nr) {
    constexpr int vw = 16 / sizeof(Tin), nv = kC * kD / vw / kThreads;
    const Tin* src[4] = {static_cast<const Tin*>(p.k), static_cast<const Tin*>(p.q), static_cast<const Tin*>(p.v),
                         static_cast<const Tin*>(p.dout)};
    float* dst[4] = {X, Q, Y, dO};
    const Tin* tail = static_cast<const Tin*>(p.tail);
    uint4 v[4][nv];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int u = 0; u < nv; ++u) {
            const int e = (threadIdx.x + u * kThreads) * vw, r = e >> 6, c = e & 63;
            const long long t = t0 + r - (a == 0 ? 1 : 0);
            const Tin* ptr = nullptr;
            if (r < nr) ptr = t >= 0 ? src[a] + (bh * p.T + t) * kD + c : (tail ? tail + bh * kD + c : nullptr);
            v[a][u] = ptr ? *reinterpret_cast<const uint4*>(ptr) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int u = 0; u < nv; ++u) {
            const int e = (threadIdx.x + u * kThreads) * vw;
            put(dst[a] + (e >> 6) * kLd + (e & 63), v[a][u], (const Tin*)nullptr);
        }
}

// NT dense fp32 64 x 64 workspace matrices into shared tiles.
template <int NT>
__device__ void load_ws(float* const (&dst)[NT], const float* const (&src)[NT]) {
    constexpr int nv = kD * kD / 4 / kThreads;
    uint4 v[NT][nv];
#pragma unroll
    for (int a = 0; a < NT; ++a)
#pragma unroll
        for (int u = 0; u < nv; ++u) v[a][u] = reinterpret_cast<const uint4*>(src[a])[threadIdx.x + u * kThreads];
#pragma unroll
    for (int a = 0; a < NT; ++a)
#pragma unroll
        for (int u = 0; u < nv; ++u) {
            const int e = (threadIdx.x + u * kThreads) * 4;
            put(dst[a] + (e >> 6) * kLd + (e & 63), v[a][u], (const float*)nullptr);
        }
}

// Per-row scalars of the chunk from X (shifted keys), beta and lambda; then the chunk-local log prefixes.
__device__ void chunk_scalars(Scal& s, const float* X, const BParams& p, long long bh, long long t0, int n) {
    const int i = threadIdx.x;
    if (i < kC) {
        float nx = 0.f;
#pragma unroll 8
        for (int c = 0; c < kD; ++c) nx = fmaf(X[i * kLd + c], X[i * kLd + c], nx);
        float eta = 0.f, alpha = 0.f, lm = 0.f, den = 0.f;
        int unc = 0, live = 0;
        if (i < n) {
            const long long t = t0 + i;
            lm = p.lam[bh * p.T + t];
            den = nx + lm + p.eps;
            const bool first = p.pos + t == 0;
            if (!first) {
                eta = den == 0.f ? 0.f : p.beta[bh * p.T + t] / den;
                const float raw = eta * lm, cap = 1.f - p.eps_gamma;
                unc = raw < cap;
                alpha = unc ? raw : cap;
                live = den != 0.f;
            }
        }
        s.eta[i] = eta;
        s.lam[i] = lm;
        s.den[i] = den;
        s.gam[i] = 1.f - alpha;
        s.unc[i] = unc;
        s.live[i] = live;
        s.L[i] = log1pf(-alpha);
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // inclusive prefix over 64 rows: lane l holds rows 2l, 2l + 1
        const int l = threadIdx.x;
        const float a = s.L[2 * l], b = s.L[2 * l + 1];
        float v = a + b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (l >= o) v += u;
        }
        const float ex = v - a - b;  // exclusive prefix of row 2l
        s.L[2 * l] = ex + a;
        s.L[2 * l + 1] = v;
        __syncwarp();
        const float LC = __shfl_sync(0xffffffffu, v, 31);
        if (l == 0) s.eLC = expf(LC);
        s.Lx[2 * l] = ex;
        s.Lx[2 * l + 1] = ex + a;
        s.eL[2 * l] = expf(ex + a);
        s.eL[2 * l + 1] = expf(v);
        s.eLx[2 * l] = expf(ex);
        s.eLx[2 * l + 1] = expf(ex + a);
        s.w[2 * l] = s.eta[2 * l] * expf(LC - (ex + a));
        s.w[2 * l + 1] = s.eta[2 * l + 1] * expf(LC - v);
    }
    __syncthreads();
}

// 64 x 64 x 64 products on the tensor cores: mma.sync m16n8k8 with tf32 operands and fp32
// accumulation, each fp32 operand split into a tf32 head and a tf32 remainder and the product taken
// as head*head + head*rem + rem*head (the remainder products carry the bits tf32 drops, so the
// result has fp32 accuracy). An operand flagged exact (a bf16 input, which tf32 holds without loss)
// has no remainder and skips its pass.
// Warp w (of 16) owns output rows 16 (w >> 2) .. + 15 (one m16 tile) and columns 16 (w & 3) .. + 15
// (two n8 tiles). acc[m][n]: m = the n8 tile, n = the fragment element (2 * row half + column).
__device__ __forceinline__ int tile_row(int m, int n) {
    const int lane = threadIdx.x & 31;
    (void)m;
    return 16 * (threadIdx.x >> 7) + (lane >> 2) + 8 * (n >> 1);
}
__device__ __forceinline__ int tile_col(int m, int n) {
    const int lane = threadIdx.x & 31;
    return 16 * ((threadIdx.x >> 5) & 3) + 8 * m + 2 * (lane & 3) + (n & 1);
}

// x = head + remainder; the remainder goes to the tensor core as its fp32 bits (the unit reads the top
// 19 bits of a tf32 operand, i.e. truncates the remainder, which costs at most 2^-10 of it).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = ptx::tf32_rn(x);
    lo = __float_as_uint(x - __uint_as_float(hi));
}

// acc += A B with A(i, k) = a[i][k] (TA: a[k][i]) and B(k, j) = b[k][j] (TB: b[j][k]).
template <bool TA, bool TB, bool AX = false, bool BX = false>
__device__ __forceinline__ void mm(float (&acc)[2][4], const float* a, const float* b) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int r = 16 * (threadIdx.x >> 7) + g, cb = 16 * ((threadIdx.x >> 5) & 3);
    auto A = [&](int i, int k) { return TA ? a[k * kLd + i] : a[i * kLd + k]; };
    auto B = [&](int k, int j) { return TB ? b[j * kLd + k] : b[k * kLd + j]; };
    float cr[2][4] = {};
#pragma unroll
    for (int k0 = 0; k0 < kD; k0 += 8) {
        uint32_t ah[4], al[4], bh[2][2], bl[2][2];
        {
            const float x[4] = {A(r, k0 + t), A(r + 8, k0 + t), A(r, k0 + t + 4), A(r + 8, k0 + t + 4)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (AX) ah[e] = __float_as_uint(x[e]), al[e] = 0u;
                else split_tf32(x[e], ah[e], al[e]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int c = cb + 8 * nt + g;
            const float y[2] = {B(k0 + t, c), B(k0 + t + 4, c)};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (BX) bh[nt][e] = __float_as_uint(y[e]), bl[nt][e] = 0u;
                else split_tf32(y[e], bh[nt][e], bl[nt][e]);
            }
        }
        // the three passes in turn over the two tiles, remainder terms into their own accumulators
        if (!AX)
#pragma unroll
            for (int q = 0; q < 2; ++q) ptx::mma1688_tf32(cr[q], al[0], al[1], al[2], al[3], bh[q][0], bh[q][1]);
        if (!BX)
#pragma unroll
            for (int q = 0; q < 2; ++q) ptx::mma1688_tf32(cr[q], ah[0], ah[1], ah[2], ah[3], bl[q][0], bl[q][1]);
#pragma unroll
        for (int q = 0; q < 2; ++q) ptx::mma1688_tf32(acc[q], ah[0], ah[1], ah[2], ah[3], bh[q][0], bh[q][1]);
    }
    if (!AX || !BX)
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][e] += cr[q][e];
}

__device__ __forceinline__ void zero(float (&acc)[2][4]) {
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[m][n] = 0.f;
}

// Runs the body for each accumulator element acc[m][n] of this thread, at output (i, j); ri and ci
// index the thread's two rows and four columns (for row_add / col_add).
#define FOR_TILE(...)                                                         \
    _Pragma("unroll") for (int m = 0; m < 2; ++m) {                           \
        _Pragma("unroll") for (int n = 0; n < 4; ++n) {                       \
            const int i = tile_row(m, n), j = tile_col(m, n);                 \
            const int ri = n >> 1, ci = 2 * m + (n & 1);                      \
            (void)ri;                                                         \
            (void)ci;                                                         \
            __VA_ARGS__                                                       \
        }                                                                     \
    }

// arr[i] += sign * scale[i] * (sum over the whole row of this CTA's partial sums v[ri]).
__device__ __forceinline__ void row_add(float* arr, const float (&v)[2], const float* scale = nullptr,
                                        float sign = 1.f) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
        float x = v[ri];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        const int i = tile_row(0, 2 * ri);
        if ((lane & 3) == 0) atomicAdd(&arr[i], sign * (scale ? scale[i] : 1.f) * x);
    }
}
// arr[j] += sign * (sum over the whole column of the partial sums v[ci]).
__device__ __forceinline__ void col_add(float* arr, const float (&v)[4], float sign = 1.f) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
        float x = v[ci];
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        if ((lane >> 2) == 0) atomicAdd(&arr[tile_col(ci >> 1, ci & 1)], sign * x);
    }
}

// T = (I + A)^-1 for a strictly lower 64 x 64 A: the four 16 x 16 diagonal blocks by forward
// substitution (one warp each, a lane per column), then two levels of block combination,
// [L11 0; L21 L22]^-1 = [T11 0; -T22 L21 T11, T22], with 16- and then 32-row blocks.
// W: scratch of 32 rows.
__device__ void unit_lower_inverse(float* Tm, const float* A, float* W) {
    for (int e = threadIdx.x; e < kC * kLd; e += kThreads) Tm[e] = 0.f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < 4 && lane < 16) {
        const int b0 = 16 * warp, c = b0 + lane;
        Tm[c * kLd + c] = 1.f;
        __syncwarp(0xffffu);
        for (int i = b0 + 1; i < b0 + 16; ++i) {
            if (c < i) {
                float a = 0.f;
                for (int j = c; j < i; ++j) a = fmaf(A[i * kLd + j], Tm[j * kLd + c], a);
                Tm[i * kLd + c] = -a;
            }
            __syncwarp(0xffffu);
        }
    }
    __syncthreads();
    for (int h = 16; h < kC; h *= 2) {
        const int nb = kC / (2 * h);
        for (int e = threadIdx.x; e < nb * h * h; e += kThreads) {  // W = L21 T11 (T11 lower: k >= cc)
            const int blk = e / (h * h), rr = (e / h) % h, cc = e % h, r0 = 2 * h * blk;
            float a = 0.f;
            for (int k = cc; k < h; ++k) a = fmaf(A[(r0 + h + rr) * kLd + r0 + k], Tm[(r0 + k) * kLd + r0 + cc], a);
            W[(blk * h + rr) * kLd + cc] = a;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < nb * h * h; e += kThreads) {  // T21 = -T22 W (T22 lower: k <= rr)
            const int blk = e / (h * h), rr = (e / h) % h, cc = e % h, r0 = 2 * h * blk;
            float a = 0.f;
            for (int k = 0; k <= rr; ++k) a = fmaf(Tm[(r0 + h + rr) * kLd + r0 + h + k], W[(blk * h + k) * kLd + cc], a);
            Tm[(r0 + h + rr) * kLd + r0 + cc] = -a;
        }
        __syncthreads();
    }
}

// --------------------------------------------------------------------------------------------------
// falcon_bwd_prep: one CTA per chunk.
template <typename Tin, bool IP>
__global__ void __launch_bounds__(kThreads, 1) falcon_bwd_prep(const BParams p) {
    extern __shared__ __align__(16) float sm[];
    float* X = sm;
    float* Q = X + kMat;
    float* Y = Q + kMat;
    float* dO = Y + kMat;
    float* A = dO + kMat;
    float* Tm = A + kMat;
    float* P = Tm + kMat;
    float* DX = P + kMat;
    float* B1 = DX + kMat;
    float* B2 = B1 + kMat;
    Scal& s = *reinterpret_cast<Scal*>(B2 + kMat);
    constexpr bool EX = sizeof(Tin) == 2;  // bf16 inputs are exact tf32 operands

    const long long cid = blockIdx.x, bh = cid / p.N, nck = cid % p.N;
    const long long t0 = nck * kC;
    const int nr = (int)min((long long)kC, p.T - t0);  // rows of this chunk
    load_inputs<Tin>(X, Q, Y, dO, p, bh, t0, nr);
    __syncthreads();
    chunk_scalars(s, X, p, bh, t0, nr);
    float* ws = p.ws + cid * kWsChunk;
    float acc[2][4], acc2[2][4];

    // Falcon-1: P, A and diag(e^Lx) X
    if (!IP) {
        zero(acc);
        mm<false, true, EX, EX>(acc, Q, X);
        FOR_TILE(P[i * kLd + j] = j <= i ? s.eta[j] * expf(s.L[i] - s.L[j]) * acc[m][n] : 0.f;)
        zero(acc);
        mm<false, true, EX, EX>(acc, X, X);
        FOR_TILE(A[i * kLd + j] = j < i ? s.eta[j] * expf(s.Lx[i] - s.L[j]) * acc[m][n] : 0.f;
                 DX[i * kLd + j] = s.eLx[i] * X[i * kLd + j];)
    }
    __syncthreads();
    if (IP) {
        // M = e^{L_C} I, U = X^T diag(w) Y, V = Q^T diag(e^L) dO
        for (int e = threadIdx.x; e < kC * kD; e += kThreads) {
            const int r = e >> 6, c = e & 63;
            B2[r * kLd + c] = s.w[r] * Y[r * kLd + c];
            dO[r * kLd + c] *= s.eL[r];
        }
        __syncthreads();
        zero(acc);
        mm<true, false, EX, false>(acc, X, B2);
        zero(acc2);
        mm<true, false, EX, false>(acc2, Q, dO);
        FOR_TILE(ws[kWsM * kWsMat + i * kD + j] = i == j ? s.eLC : 0.f;
                 ws[kWsMT * kWsMat + i * kD + j] = i == j ? s.eLC : 0.f;
                 ws[kWsU * kWsMat + i * kD + j] = acc[m][n];
                 ws[kWsV * kWsMat + i * kD + j] = acc2[m][n];)
        return;
    }
    unit_lower_inverse(Tm, A, B1);
    // B1 = diag(w) T diag(e^Lx) X, B2 = diag(w) T Y, A <- P^T dO
    zero(acc);
    mm<false, false>(acc, Tm, DX);
    zero(acc2);
    mm<false, false, false, EX>(acc2, Tm, Y);
    FOR_TILE(B1[i * kLd + j] = s.w[i] * acc[m][n]; B2[i * kLd + j] = s.w[i] * acc2[m][n];)
    zero(acc);
    mm<true, false, false, EX>(acc, P, dO);
    FOR_TILE(A[i * kLd + j] = acc[m][n];)
    __syncthreads();
    // M = e^{L_C} I - X^T B1, U = X^T B2; P <- T^T (P^T dO); dO <- diag(e^L) dO
    zero(acc);
    mm<true, false, EX, false>(acc, X, B1);
    zero(acc2);
    mm<true, false, EX, false>(acc2, X, B2);
    FOR_TILE(const float mij = (i == j ? s.eLC : 0.f) - acc[m][n];
             ws[kWsM * kWsMat + i * kD + j] = mij;
             ws[kWsMT * kWsMat + j * kD + i] = mij;
             ws[kWsU * kWsMat + i * kD + j] = acc2[m][n];
             ws[kWsT * kWsMat + i * kD + j] = Tm[i * kLd + j];)
    zero(acc);
    mm<true, false>(acc, Tm, A);
    __syncthreads();  // every read of P and dO above is done
    FOR_TILE(P[i * kLd + j] = acc[m][n]; dO[i * kLd + j] *= s.eL[i];)
    __syncthreads();
    // V = Q^T diag(e^L) dO - (diag(e^Lx) X)^T T^T P^T dO
    zero(acc);
    mm<true, false, EX, false>(acc, Q, dO);
    zero(acc2);
    mm<true, false>(acc2, DX, P);
    FOR_TILE(ws[kWsV * kWsMat + i * kD + j] = acc[m][n] - acc2[m][n];)
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// falcon_bwd_chain: one CTA of 128 threads per sequence, the two state scans on the tensor cores.
// The carried matrix (S forward, dS backward) is kept transposed in tensor memory, lane c = column c
// (lanes 64-127 zero), as the A operand of one product per step: D = X^T B^T with B = M_n (forward:
// D = (M_n S)^T) or B = M_n^T (backward: D = (M_n^T dS)^T), both K-major as the prep kernel stores them,
// loaded by TMA with the 128-byte swizzle. Each operand x is split into hi = x with its low 13 bits
// cleared (exact in tf32) and lo = x - hi, and D = A_hi B_hi + A_hi B_lo + A_lo B_hi (fp32-accurate).
// U_n / V_n arrive by 16-byte asynchronous copies one step ahead and are added in registers, where
// each thread also stores its column of S_n / dS_{n+1} for the gradient kernel. Every wait is bounded:
// on timeout the CTA raises the device flag, drains what it issued and frees its tensor memory.
constexpr int kChainT = 128;
constexpr uint32_t kCAH = 0, kCAL = 64, kCD = 128;  // TMEM columns: carried hi, lo, product
constexpr long long kTcTimeout = 4000000000LL;     // ~2 s
namespace chl {
constexpr int BHI = 0, BLO = 16384;  // B = M_n or M_n^T: two K halves of 64 rows x 128 bytes each
constexpr int OFS = 32768;           // two offset buffers (U_n or V_n), [64][64] fp32
constexpr int BAR = OFS + 32768;
constexpr int BYTES = BAR + 64;
constexpr int ALLOC = BYTES + 1024;
}  // namespace chl

struct ChainParams {
    CUtensorMap tm_ws;  // the workspace as [rows][64] fp32, 32 x 32 boxes, 128-byte swizzle
    BParams p;
};

__device__ __forceinline__ float hi19(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

__device__ bool chain_wait(uint32_t bar, uint32_t parity) {
    if (ptx::mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    int spins = 0;
    while (!ptx::mbar_try(bar, parity)) {
        if (++spins > 64) __nanosleep(32);
        if (clock64() - t0 > kTcTimeout) {
            atomicExch(&g_bwd_timeout_flag, 1);
            return false;
        }
    }
    return true;
}

// this thread's carried column into the A operand's hi and lo columns of its lane (no wait)
__device__ __forceinline__ void chain_put(uint32_t tq, const float (&x)[kD]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h[16], l[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float v = x[16 * q + e], vh = hi19(v);
            h[e] = __float_as_uint(vh);
            l[e] = __float_as_uint(v - vh);
        }
        ptx::tmem_st16(tq + kCAH + 16 * q, h);
        ptx::tmem_st16(tq + kCAL + 16 * q, l);
    }
}

__global__ void __launch_bounds__(kChainT, 1) falcon_bwd_chain(const __grid_constant__ ChainParams P) {
    using namespace ptx;
    const BParams& p = P.p;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw), base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t bar_full = base + chl::BAR, bar_mma = bar_full + 8, bar_drain = bar_full + 16;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + chl::BAR + 32);
    const long long bh = blockIdx.x, N = p.N;
    if (tid == 0) {
        mbar_init(bar_full, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_drain, 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot, tq = tmem + ((uint32_t)(32 * warp) << 16);
    const int c = tid;            // carried column = TMEM lane
    const bool live = c < kD;     // lanes 64-127 hold zeros
    float* const wsq = p.ws + bh * N * kWsChunk;

    // step k of the 2 N: chunk n, matrix and offset of the pass
    auto chunk_of = [&](long long k) { return k < N ? k : 2 * N - 1 - k; };
    auto issue_b = [&](long long k) {  // thread 0: B of step k by TMA
        const long long n = chunk_of(k);
        const int r = (int)((bh * N + n) * (kWsChunk / kD) + (k < N ? kWsM : kWsMT) * kD);
        mbar_expect_tx(bar_full, 16384u);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t d = base + chl::BHI + h * 8192;
            tma_load_2d(d, &P.tm_ws, 32 * h, r, bar_full);
            tma_load_2d(d + 4096, &P.tm_ws, 32 * h, r + 32, bar_full);
        }
    };
    auto issue_ofs = [&](long long k) {  // every thread: U_n (forward) or V_n (backward) into buffer k & 1
        if (k < 2 * N) {
            const float* src = wsq + chunk_of(k) * kWsChunk + (k < N ? kWsU : kWsV) * kWsMat;
            float* d = reinterpret_cast<float*>(sm + chl::OFS) + (int)(k & 1) * kWsMat;
#pragma unroll
            for (int u = 0; u < kWsMat / 4 / kChainT; ++u) {
                const int e = 4 * (tid + u * kChainT);
                cp_async16(d + e, src + e);
            }
        }
        cp_async_commit();
    };

    float s[kD];
    auto load_start = [&](const float* src) {
#pragma unroll
        for (int r = 0; r < kD; ++r) s[r] = (live && src) ? src[(bh * kD + r) * kD + c] : 0.f;
        chain_put(tq, s);
        tmem_wait_st();
    };
    load_start(p.S0);
    long long pending = 0;  // the step whose B is in flight (-1: none)
    if (tid == 0) issue_b(0);
    issue_ofs(0);
    tc_fence_before();
    __syncthreads();
    bool ok = true;
    constexpr uint32_t id = idesc_tf32(128, kD);
    for (long long k = 0; k < 2 * N; ++k) {
        const long long n = chunk_of(k);
        const bool fwd = k < N;
        if (k == N) {  // the backward scan starts from dS_final
            load_start(p.dS_final);
            tc_fence_before();
            __syncthreads();
        }
        bool bad = false;
        if (tid == 0) bad = !chain_wait(bar_full, (uint32_t)(k & 1));
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (named_bar_or(1, kChainT, bad)) {
            ok = false;
            break;
        }
        pending = -1;
        if (live) {  // S_n (forward) / dS_{n+1} (backward) for the gradient kernel, this thread's column
            float* dst = wsq + n * kWsChunk + (fwd ? kWsS : kWsDS) * kWsMat + c;
#pragma unroll
            for (int r = 0; r < kD; ++r) dst[r * kD] = s[r];
        }
        {  // B: hi (low 13 bits cleared) in place, lo = the rest
            float4* bh4 = reinterpret_cast<float4*>(sm + chl::BHI);
            float4* bl4 = reinterpret_cast<float4*>(sm + chl::BLO);
#pragma unroll 4
            for (int e = tid; e < 16384 / 16; e += kChainT) {
                const float4 v = bh4[e];
                const float4 h = make_float4(hi19(v.x), hi19(v.y), hi19(v.z), hi19(v.w));
                bh4[e] = h;
                bl4[e] = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (uint32_t)((ks >> 2) * 8192 + 32 * (ks & 3));
                const uint64_t dh = desc_k(base + chl::BHI + off), dl = desc_k(base + chl::BLO + off);
                mma_tf32_ta(tmem + kCD, tmem + kCAH + 8 * ks, dh, id, ks > 0);
                mma_tf32_ta(tmem + kCD, tmem + kCAH + 8 * ks, dl, id, 1);
                mma_tf32_ta(tmem + kCD, tmem + kCAL + 8 * ks, dh, id, 1);
            }
            mma_commit(bar_mma);
            bad = !chain_wait(bar_mma, (uint32_t)(k & 1));
            if (!bad && k + 1 < 2 * N) issue_b(k + 1);  // B is free again
        }
        if (named_bar_or(1, kChainT, bad)) {
            ok = false;
            break;
        }
        if (k + 1 < 2 * N) pending = k + 1;
        issue_ofs(k + 1);
        tc_fence_after();
        {
            const float* of = reinterpret_cast<const float*>(sm + chl::OFS) + (int)(k & 1) * kWsMat;
            uint32_t d[4][16];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(tq + kCD + 16 * q, d[q]);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                regs_ready(d[q]);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r = 16 * q + e;
                    s[r] = live ? __uint_as_float(d[q][e]) + of[r * kD + c] : 0.f;
                }
            }
        }
        if (k + 1 < 2 * N && k + 1 != N) chain_put(tq, s);
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
    }
    if (ok && p.dS0 && live) {
#pragma unroll
        for (int r = 0; r < kD; ++r) p.dS0[(bh * kD + r) * kD + c] = s[r];
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (tid == 0 && pending >= 0) mbar_wait_bounded(bar_full, (uint32_t)(pending & 1), kTcTimeout);
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        mma_commit(bar_drain);
        mbar_wait_bounded(bar_drain, 0, kTcTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// --------------------------------------------------------------------------------------------------
// falcon_bwd_grad: one CTA per chunk.
template <typename Tin, bool IP>
__global__ void __launch_bounds__(kThreads, 1) falcon_bwd_grad(const BParams p) {
    extern __shared__ __align__(16) float sm[];
    float* X = sm;
    float* Q = X + kMat;
    float* Y = Q + kMat;   // Y; Falcon-1: Z, then P, then the dX accumulator
    float* dO = Y + kMat;
    float* S = dO + kMat;
    float* dS = S + kMat;
    float* Tm = dS + kMat;  // T (Falcon-1), then dP -> dSc
    float* b0 = Tm + kMat;  // Falcon-1: R; Falcon-1A: P
    float* b1 = b0 + kMat;  // X dS', then dR; Falcon-1: dA -> dG + dG^T
    float* b2 = b1 + kMat;  // Sc
    float* b3 = b2 + kMat;  // G (Falcon-1); Falcon-1A: the dX accumulator
    float* b4 = IP ? b3 : b3 + kMat;  // dZ (Falcon-1)
    Scal& s = *reinterpret_cast<Scal*>(b4 + kMat);
    float* deta = reinterpret_cast<float*>(&s + 1);
    float* dL = deta + kC;
    float* dLx = dL + kC;
    float* dw = dLx + kC;
    float* c2 = dw + kC;
    float* red = c2 + kC;  // [warps] block reduction

    constexpr bool EX = sizeof(Tin) == 2;  // bf16 inputs are exact tf32 operands
    float* R = IP ? Y : b0;
    float* P = IP ? b0 : Y;
    float* DXa = IP ? b3 : Y;

    const long long cid = blockIdx.x, bh = cid / p.N, nck = cid % p.N;
    const long long t0 = nck * kC;
    const int nr = (int)min((long long)kC, p.T - t0);  // rows of this chunk
    const float* ws = p.ws + cid * kWsChunk;
    load_inputs<Tin>(X, Q, Y, dO, p, bh, t0, nr);
    if (IP) {
        float* const d2[2] = {S, dS};
        const float* const s2[2] = {ws + kWsS * kWsMat, ws + kWsDS * kWsMat};
        load_ws<2>(d2, s2);
    } else {
        float* const d3[3] = {S, dS, Tm};
        const float* const s3[3] = {ws + kWsS * kWsMat, ws + kWsDS * kWsMat, ws + kWsT * kWsMat};
        load_ws<3>(d3, s3);
    }
    if (threadIdx.x < kC) {
        deta[threadIdx.x] = 0.f;
        dL[threadIdx.x] = 0.f;
        dLx[threadIdx.x] = 0.f;
    }
    if (threadIdx.x < kThreads / 32) red[threadIdx.x] = 0.f;
    __syncthreads();
    chunk_scalars(s, X, p, bh, t0, nr);
    const int lane = threadIdx.x & 31;
    float acc[2][4], acc2[2][4];

    // <dS', S>
    {
        float a = 0.f;
        for (int e = threadIdx.x; e < kD * kD; e += kThreads) {
            const int rr = e >> 6, cc = e & 63;
            a = fmaf(dS[rr * kLd + cc], S[rr * kLd + cc], a);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) red[threadIdx.x >> 5] = a;
    }
    // Z = Y - diag(e^Lx) X S (Falcon-1); X dS'
    if (!IP) {
        zero(acc);
        mm<false, false, EX, false>(acc, X, S);
        FOR_TILE(Y[i * kLd + j] -= s.eLx[i] * acc[m][n];)
    }
    zero(acc);
    mm<false, false, EX, false>(acc, X, dS);
    FOR_TILE(b1[i * kLd + j] = acc[m][n];)
    __syncthreads();
    // R = T Z (Falcon-1); Sc = Q X^T; G = X X^T (Falcon-1)
    if (!IP) {
        zero(acc);
        mm<false, false>(acc, Tm, Y);
        FOR_TILE(b0[i * kLd + j] = acc[m][n];)
        zero(acc);
        mm<false, true, EX, EX>(acc, X, X);
        FOR_TILE(b3[i * kLd + j] = acc[m][n];)
    }
    zero(acc);
    mm<false, true, EX, EX>(acc, Q, X);
    FOR_TILE(b2[i * kLd + j] = acc[m][n];)
    __syncthreads();
    // dw_j = x_j^T dS' r_j; P
    if (threadIdx.x < kC) {
        const int j = threadIdx.x;
        float a = 0.f;
#pragma unroll 8
        for (int cc = 0; cc < kD; ++cc) a = fmaf(b1[j * kLd + cc], R[j * kLd + cc], a);
        dw[j] = a;
    }
    FOR_TILE(P[i * kLd + j] = j <= i ? s.eta[j] * expf(s.L[i] - s.L[j]) * b2[i * kLd + j] : 0.f;)
    __syncthreads();
    // dR = P^T dO + diag(w) X dS'  (Falcon-1A: dV = dR)
    zero(acc);
    mm<true, false, false, EX>(acc, P, dO);
    FOR_TILE(b1[i * kLd + j] = acc[m][n] + s.w[i] * b1[i * kLd + j];)
    __syncthreads();
    float* dvo = p.dv + (bh * p.T + t0) * kD;
    if (!IP) {  // dZ = T^T dR = dV
        zero(acc);
        mm<true, false>(acc, Tm, b1);
        FOR_TILE(b4[i * kLd + j] = acc[m][n]; if (i < nr) dvo[i * kD + j] = acc[m][n];)
    } else {
        FOR_TILE(if (i < nr) dvo[i * kD + j] = b1[i * kLd + j];)
    }
    __syncthreads();
    // dP = dO R^T (j <= i) -> d eta, dL; dSc = dP eta_j e^{L_i - L_j}, into Tm
    zero(acc);
    mm<false, true, EX, IP && EX>(acc, dO, R);
    if (!IP) {
        zero(acc2);
        mm<false, true>(acc2, b4, R);  // dZ R^T = -dA
    }
    __syncthreads();  // Tm (T) and b1 (dR) are read no more
    {
        float rowL[2] = {0.f, 0.f}, colE[4] = {0.f, 0.f, 0.f, 0.f}, colL[4] = {0.f, 0.f, 0.f, 0.f};
        FOR_TILE({
            float v = 0.f;
            if (j <= i) {
                const float f = expf(s.L[i] - s.L[j]), d = acc[m][n];
                const float pp = P[i * kLd + j];
                colE[ci] = fmaf(d * f, b2[i * kLd + j], colE[ci]);
                rowL[ri] = fmaf(d, pp, rowL[ri]);
                colL[ci] = fmaf(d, pp, colL[ci]);
                v = d * s.eta[j] * f;
            }
            Tm[i * kLd + j] = v;
        })
        row_add(dL, rowL);
        col_add(deta, colE);
        col_add(dL, colL, -1.f);
    }
    if (!IP) {  // dA = -dZ R^T (j < i) -> d eta, dLx, dL; dG = dA eta_j e^{Lx_i - L_j}, into b1
        float rowX[2] = {0.f, 0.f}, colE[4] = {0.f, 0.f, 0.f, 0.f}, colL[4] = {0.f, 0.f, 0.f, 0.f};
        FOR_TILE({
            float v = 0.f;
            if (j < i) {
                const float f = expf(s.Lx[i] - s.L[j]), d = -acc2[m][n];
                const float gv = b3[i * kLd + j];
                const float aa = s.eta[j] * f * gv * d;
                colE[ci] = fmaf(d * f, gv, colE[ci]);
                rowX[ri] += aa;
                colL[ci] += aa;
                v = d * s.eta[j] * f;
            }
            b1[i * kLd + j] = v;
        })
        row_add(dLx, rowX);
        col_add(deta, colE);
        col_add(dL, colL, -1.f);
    }
    __syncthreads();
    if (!IP) {  // dG + dG^T: mirror the strict lower triangle into the upper one
        for (int e = threadIdx.x; e < kC * kC; e += kThreads) {
            const int i = e >> 6, j = e & 63;
            if (j > i) b1[i * kLd + j] = b1[j * kLd + i];
        }
    }
    // dX accumulator: diag(w) R dS'^T  (for Falcon-1 it overwrites P, last read before the barrier above)
    zero(acc);
    mm<false, true, IP && EX, false>(acc, R, dS);
    __syncthreads();
    FOR_TILE(DXa[i * kLd + j] = s.w[i] * acc[m][n];)
    __syncthreads();
    // dX += dSc^T Q (+ (dG + dG^T) X - diag(e^Lx) dZ S^T, with dLx_i -= e^Lx_i x_i . (dZ S^T)_i)
    zero(acc);
    mm<true, false, false, EX>(acc, Tm, Q);
    if (!IP) {
        mm<false, false, false, EX>(acc, b1, X);
        zero(acc2);
        mm<false, true>(acc2, b4, S);
        float rowX[2] = {0.f, 0.f};
        FOR_TILE(DXa[i * kLd + j] += acc[m][n] - s.eLx[i] * acc2[m][n];
                 rowX[ri] = fmaf(X[i * kLd + j], acc2[m][n], rowX[ri]);)
        row_add(dLx, rowX, s.eLx, -1.f);
    } else {
        FOR_TILE(DXa[i * kLd + j] += acc[m][n];)
    }
    // dQ = diag(e^L) dO S^T + dSc X, with dL_i += e^L_i q_i . (dO S^T)_i
    zero(acc);
    mm<false, true, EX, false>(acc, dO, S);
    zero(acc2);
    mm<false, false, false, EX>(acc2, Tm, X);
    {
        float rowL[2] = {0.f, 0.f};
        float* dqo = p.dq + (bh * p.T + t0) * kD;
        FOR_TILE(rowL[ri] = fmaf(Q[i * kLd + j], acc[m][n], rowL[ri]);
                 if (i < nr) dqo[i * kD + j] = s.eL[i] * acc[m][n] + acc2[m][n];)
        row_add(dL, rowL, s.eL);
    }
    __syncthreads();
    // scalars: d eta and dL from w and the chunk-end decay; d log gamma; the clamp; eta = beta / den
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        float dwsum = 0.f;
        float dl[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 2 * l + h;
            const float ww = dw[j] * s.w[j];
            dwsum += ww;
            deta[j] = fmaf(dw[j], expf(s.L[kC - 1] - s.L[j]), deta[j]);
            dl[h] = dL[j] - ww + (j + 1 < kC ? dLx[j + 1] : 0.f);
        }
        dwsum += __shfl_xor_sync(0xffffffffu, dwsum, 16);
        dwsum += __shfl_xor_sync(0xffffffffu, dwsum, 8);
        dwsum += __shfl_xor_sync(0xffffffffu, dwsum, 4);
        dwsum += __shfl_xor_sync(0xffffffffu, dwsum, 2);
        dwsum += __shfl_xor_sync(0xffffffffu, dwsum, 1);
        float dss = 0.f;
#pragma unroll
        for (int u = 0; u < kThreads / 32; ++u) dss += red[u];
        if (l == 31) dl[1] += dwsum + s.eLC * dss;
        // suffix sums: d log gamma_u = sum_{i >= u} dL_i
        float v = dl[0] + dl[1];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_down_sync(0xffffffffu, v, o);
            if (l + o < 32) v += u;
        }
        const float suf[2] = {v, v - dl[0]};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int u = 2 * l + h;
            float db = 0.f, dlm = 0.f, cc = 0.f;
            if (u < nr) {
                float de = deta[u];
                if (s.unc[u]) {
                    const float da = -suf[h] / s.gam[u];
                    de = fmaf(da, s.lam[u], de);
                    dlm = da * s.eta[u];
                }
                if (s.live[u]) {
                    db = de / s.den[u];
                    const float dden = -de * s.eta[u] / s.den[u];
                    dlm += dden;
                    cc = 2.f * dden;
                }
                p.dbeta[bh * p.T + t0 + u] = db;
                p.dlam[bh * p.T + t0 + u] = dlm;
            }
            c2[u] = cc;
        }
    }
    __syncthreads();
    // dX = accumulator + 2 dden x; row i is dk of token t0 + i - 1 (row 0 of the call: the tail key)
    for (int e = threadIdx.x; e < kC * kD; e += kThreads) {
        const int i = e >> 6, j = e & 63;
        if (i >= nr) continue;
        const float g = fmaf(c2[i], X[i * kLd + j], DXa[i * kLd + j]);
        const long long t = t0 + i - 1;
        if (t >= 0) p.dk[(bh * p.T + t) * kD + j] = g;
        else if (p.dtail) p.dtail[bh * kD + j] = g;
    }
    if (t0 + nr == p.T)  // the last key feeds only the next call's tail
        for (int j = threadIdx.x; j < kD; j += kThreads) p.dk[(bh * p.T + p.T - 1) * kD + j] = 0.f;
}

constexpr size_t kScalBytes = sizeof(Scal);
constexpr size_t kPrepSmem = 10 * kMat * sizeof(float) + kScalBytes;
constexpr size_t gradSmem(bool ip) { return (ip ? 11 : 12) * kMat * sizeof(float) + kScalBytes + (5 * kC + kThreads / 32) * sizeof(float); }

template <typename Tin, bool IP>
int launch_typed(const BParams& p, cudaStream_t st) {
    const unsigned chunks = (unsigned)(p.BH * p.N);
    cudaFuncSetAttribute(falcon_bwd_prep<Tin, IP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    cudaFuncSetAttribute(falcon_bwd_grad<Tin, IP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gradSmem(IP));
    falcon_bwd_prep<Tin, IP><<<chunks, kThreads, kPrepSmem, st>>>(p);
    ChainParams cp{};
    cp.p = p;
    const long long rows = p.BH * p.N * (kWsChunk / kD);  // the workspace as rows of 64 floats
    if (rows >= (1LL << 31) || !encode_rows_f32_sw128(&cp.tm_ws, p.ws, rows)) return 4;
    cudaFuncSetAttribute(falcon_bwd_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, chl::ALLOC);
    falcon_bwd_chain<<<(unsigned)p.BH, kChainT, chl::ALLOC, st>>>(cp);
    falcon_bwd_grad<Tin, IP><<<chunks, kThreads, gradSmem(IP), st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

}  // namespace

bool bwd_supported(const Launch& a) {
    return (a.variant == kF1 || a.variant == kF1A) && a.dk == kD && a.dv == kD && a.chunk == kC && a.W == 1;
}

size_t bwd_workspace_bytes(const Launch& a) {
    const long long N = (a.T + kC - 1) / kC;
    return (size_t)(a.B * a.H) * (size_t)N * kWsChunk * sizeof(float);
}

int launch_bwd(const Launch& a, const BwdArgs& g, cudaStream_t st) {
    BParams p;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.dout = g.dout;
    p.tail = a.tail;
    p.beta = a.beta;
    p.lam = a.lam;
    p.S0 = a.S0;
    p.dS_final = g.dS_final;
    p.dq = g.dq;
    p.dk = g.dk;
    p.dv = g.dv;
    p.dbeta = g.dbeta;
    p.dlam = g.dlam;
    p.dS0 = g.dS0;
    p.dtail = g.dtail;
    p.ws = static_cast<float*>(a.ws);
    p.T = a.T;
    p.pos = a.pos;
    p.N = (a.T + kC - 1) / kC;
    p.BH = a.B * a.H;
    p.eps = a.eps;
    p.eps_gamma = a.eps_gamma;
    if (p.BH == 0) return 0;
    if (p.N == 0) {  // no tokens: dS0 = dS_final, nothing else
        if (p.dS0) {
            const size_t bytes = (size_t)p.BH * kD * kD * sizeof(float);
            const cudaError_t e = p.dS_final ? cudaMemcpyAsync(p.dS0, p.dS_final, bytes, cudaMemcpyDeviceToDevice, st)
                                             : cudaMemsetAsync(p.dS0, 0, bytes, st);
            if (e != cudaSuccess) return 4;
        }
        if (p.dtail) return cudaMemsetAsync(p.dtail, 0, (size_t)p.BH * kD * sizeof(float), st) == cudaSuccess ? 0 : 4;
        return 0;
    }
    const bool ip = a.variant == kF1A;
    if (a.bf16) return ip ? launch_typed<__nv_bfloat16, true>(p, st) : launch_typed<__nv_bfloat16, false>(p, st);
    return ip ? launch_typed<float, true>(p, st) : launch_typed<float, false>(p, st);
}

int bwd_consume_timeout_flag(int* flag) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_timeout_flag, sizeof(int)) != cudaSuccess) return 1;
    if (v && cudaMemcpyToSymbol(g_bwd_timeout_flag, &zero, sizeof(int)) != cudaSuccess) return 1;
    *flag = v;
    return 0;
}

}  // namespace falcon
