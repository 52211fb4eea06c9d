// Chunk-parallel split path for Falcon-1 and Falcon-1A (bf16 I/O, dk = dv = 64, chunk 64).
//
// Per chunk of C = 64 tokens (rows i, j) with X the shifted keys (row i = k_{tau_i - 1}), Y the
// values, Q the queries, eta the step sizes, L / Lx the inclusive / exclusive chunk-local log-decay
// prefixes (reset to 0 at every chunk start), w_j = eta_j e^{L_C - L_j} and
//   A_ij = eta_j e^{Lx_i - L_j} x_i.x_j  (j < i),   P_ij = eta_j e^{L_i - L_j} q_i.x_j  (j <= i),
//   T = (I + A)^{-1},
// unrolling the Falcon-1 recurrence over the chunk ("Fast Weight Attention for Continual Learning",
// paperlayer summary: §E.1 WY form of the triangular solve, §E.2 one merged residual solve, §F.2
// read after write, §G.1 chunk-local log prefixes) gives, with S the state at the chunk start,
//   R  = T (Y - diag(e^{Lx}) X S)                    residual targets of the chunk
//   O  = diag(e^{L}) Q S + P R                       the chunk's reads o_i = S_i^T q_i
//   S' = e^{L_C} S + X^T diag(w) R = M S + U,  where
//   M  = e^{L_C} I - X^T diag(w) T diag(e^{Lx}) X,   U = X^T diag(w) T Y.
// M and U do not depend on S, so the work splits into three launches:
//   falcon_prep_kernel   one CTA per chunk, every chunk of every sequence at once: M_n, U_n
//   falcon_chain_kernel  one CTA per sequence: S_{n+1} = M_n S_n + U_n, two 32-column halves pipelined
//   falcon_out_kernel    one CTA per chunk, every chunk at once: R and O from S_n
// Falcon-1A writes the target itself (no residual): T = I, M = e^{L_C} I, U = X^T diag(w) Y.
//
// Precision: tensor-core products of the exact bf16 inputs run in bf16. Every derived operand
// (T, Z = X^T diag(w) T, Y - diag(e^{Lx}) X S, R, P, M, S) is split into bf16 hi and lo parts and
// the products keep hi*hi, hi*lo and lo*hi, so each operand carries ~16 significant bits and every
// sum is fp32. Only factors e^{a - b} with a <= b are formed: when the chunk's total log decay is
// at least -30 they are e^{a} * e^{-b} (both finite, no cancellation), otherwise one exp each.
//
// Every mbarrier wait is bounded: on timeout the kernel raises a device flag, drains what it
// issued (bounded), frees its TMEM and exits; falcon_device_status() reports the flag.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "falcon_internal.h"
#include "sm103_ptx.cuh"

namespace falcon {

__device__ int g_split_timeout_flag = 0;

namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;
constexpr int kTile = 8192;           // 64 x 64 bf16
constexpr int kS = 68;                // fp32 row stride (floats) of A and T in shared memory
constexpr int kFBytes = 64 * kS * 4;  // 17408
constexpr long long kTimeoutCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr float kFastL = 30.f;

struct SplitParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_out, tm_m, tm_s, tm_t, tm_u;
    const float* beta;
    const float* lam;
    const float* S0;
    const bf16* k;
    const bf16* tail;
    bf16* tail_out;
    float* S_final;
    bf16* ws_m;   // [BH][N][2][64][64]: M_n hi, lo
    float* ws_u;  // [BH][N][64][64]:    U_n
    bf16* ws_s;   // [BH][N][2][64][64]: S_n hi, lo (state at the start of chunk n)
    bf16* ws_t;   // [BH][N][2][64][64]: T_n hi, lo
    uint8_t* ws_sc;  // [BH][N] blocks of kScalBytes: the chunk's per-token scalars (a Scal)
    // The chain kernel follows the prep kernel chunk by chunk through a flag per chunk: the prep CTA
    // of the chunk clears it before it lets the chain kernel launch (which cannot happen before every
    // prep CTA has), and sets it to `epoch` once M_n, U_n, T_n and the scalars are in the workspace.
    unsigned long long* fl_prep;  // [BH][N]
    unsigned long long epoch;
    long long BH;
    long long T, pos;
    int N;
    float eps, eps_gamma;
    int variant;
};

__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity) {
    if (mbar_wait_bounded(bar, parity, kTimeoutCycles)) return true;
    atomicExch(&g_split_timeout_flag, 1);
    return false;
}
// CTA-wide wait by thread 0. False (for every thread) on timeout or when thread 0 passes
// `bad` = 1, after thread 0 has given the barrier one more bounded wait so that nothing it tracks
// is still landing when the CTA exits.
__device__ __forceinline__ bool cta_wait(uint32_t bar, uint32_t parity, int tid, int bad = 0) {
    if (tid == 0 && !wait_or_flag(bar, parity)) {
        bad = 1;
        mbar_wait_bounded(bar, parity, kTimeoutCycles);
    }
    return !__syncthreads_or(bad);
}
// Thread 0 of a consumer CTA: wait (bounded) for a producer's flag; on timeout raise the device flag.
__device__ __forceinline__ bool wait_producer(const unsigned long long* flag, unsigned long long epoch) {
    if (wait_flag_bounded(flag, epoch, kTimeoutCycles)) {
        fence_proxy_async_global();  // the TMA loads that follow see what the flag guards
        return true;
    }
    atomicExch(&g_split_timeout_flag, 1);
    return false;
}
// Every thread of a producer CTA calls this after its last global store of the chunk's data;
// thread 0 then publishes `flag`. Contains a CTA barrier.
__device__ __forceinline__ void publish(unsigned long long* flag, unsigned long long epoch, int tid) {
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release_gpu(flag, epoch);
}
__device__ __forceinline__ void release_tmem(uint32_t tmem, int warp, uint32_t cols) {
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, cols);
}
__device__ __forceinline__ void hilo8(const float* v, uint4& h, uint4& l) {
    split2(v[0], v[1], h.x, l.x);
    split2(v[2], v[3], h.y, l.y);
    split2(v[4], v[5], h.z, l.z);
    split2(v[6], v[7], h.w, l.w);
}

// ---------------------------------------------------------------- per-token scalars
struct Scal {
    float eta[64], L[64], Lx[64], eLx[64], eL[64], cA[64], w[64];
    float misc[8];  // [0] e^{L_C}, [1..2] warp totals of the scan, [3] 1 when the fast exp form holds
};
constexpr int kScalBytes = 2048;  // workspace stride of one chunk's Scal
static_assert(sizeof(Scal) % 16 == 0 && sizeof(Scal) <= kScalBytes, "Scal block");

// Threads 0-63 own token i of the chunk; every thread of the CTA takes part in the two barriers.
// tau0 is the global 1-based index of the chunk's first token; token 1 has x = 0 and eta = 0.
__device__ __forceinline__ void chunk_scalars(Scal* s, const uint8_t* Xs, int tid, float beta_i, float lam_i, int nv,
                                              long long tau0, float eps, float eps_gamma) {
    if (tid < 64) {
        const int i = tid, lane = tid & 31;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
            float x[8];
            unpack8(*reinterpret_cast<const uint4*>(Xs + sw128(i, 8 * q8)), x);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(x[e], x[e], acc[e]);
        }
        const float nx = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        float eta = 0.f, alpha = 0.f;
        if (i < nv && tau0 + i >= 2) {
            const float den = nx + lam_i + eps;
            eta = den == 0.f ? 0.f : beta_i / den;
            alpha = fminf(eta * lam_i, 1.f - eps_gamma);
        }
        const float l = log1pf(-alpha);
        float incl = l;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        s->eta[i] = eta;
        s->L[i] = incl;  // warp-local until the carry is added
        s->Lx[i] = l;    // the token's own log-decay until then
        if (lane == 31) s->misc[1 + (i >> 5)] = incl;
    }
    __syncthreads();
    if (tid < 64) {
        const int i = tid;
        const float LC = s->misc[1] + s->misc[2];
        const float Li = s->L[i] + (i >= 32 ? s->misc[1] : 0.f);
        const float Lxi = Li - s->Lx[i];
        const float eta = s->eta[i];
        s->L[i] = Li;
        s->Lx[i] = Lxi;
        s->eLx[i] = expf(Lxi);
        s->eL[i] = expf(Li);
        s->cA[i] = eta * expf(fminf(-Li, kFastL + 1.f));  // read only when L_C >= -kFastL
        s->w[i] = eta * expf(LC - Li);
        if (i == 0) {
            s->misc[0] = expf(LC);
            s->misc[3] = LC >= -kFastL ? 1.f : 0.f;
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- T = (I + A)^{-1}
// In place: on entry M holds A, strictly lower 64 x 64 (fp32, stride kS), with zeros in the 16 x 16
// blocks above the diagonal; on exit M holds T = (I + A)^{-1}. 16 x 16 diagonal blocks by column
// substitution in fp32 (in registers), then two levels of block merges T_ba = -(T_bb A_ba) T_aa as
// warp-level tf32 products (operands rounded to nearest tf32, fp32 accumulation); each merge reads
// the A block it replaces before writing it. Ends with a CTA barrier.
//
// tf32 m16n8k8 fragments: A a0 = (g, t), a1 = (g + 8, t), a2 = (g, t + 4), a3 = (g + 8, t + 4);
// B b0 = (t, g), b1 = (t + 4, g); C c0, c1 = (g, 2t), (g, 2t + 1); c2, c3 = rows g + 8. A product
// whose A operand is a previous accumulator takes it with the k-slots t / t + 4 standing for
// columns 2t / 2t + 1, so its B rows are read in the same order (2t, 2t + 1).
__device__ __forceinline__ void mma_tf_a(float (&d)[4], const float* M, int r0, int k0, int k0b, int n0, int g, int t,
                                         bool permuted_b) {
    // d += M[r0.., k0..k0+7] (A, 16 x 8) x M[k0b.., n0..n0+7] (B, 8 x 8)
    const uint32_t a0 = tf32_rn(M[(r0 + g) * kS + k0 + t]), a1 = tf32_rn(M[(r0 + g + 8) * kS + k0 + t]);
    const uint32_t a2 = tf32_rn(M[(r0 + g) * kS + k0 + t + 4]), a3 = tf32_rn(M[(r0 + g + 8) * kS + k0 + t + 4]);
    const int kb0 = permuted_b ? 2 * t : t, kb1 = permuted_b ? 2 * t + 1 : t + 4;
    const uint32_t b0 = tf32_rn(M[(k0b + kb0) * kS + n0 + g]), b1 = tf32_rn(M[(k0b + kb1) * kS + n0 + g]);
    mma1688_tf32(d, a0, a1, a2, a3, b0, b1);
}
__device__ __forceinline__ void mma_tf_c(float (&d)[4], const float (&c)[4], const float* M, int k0b, int n0, int g,
                                         int t) {
    // d += C (accumulator fragment of a 16 x 8 tile, as the A operand of a k8 step) x M[k0b.., n0..]
    const uint32_t b0 = tf32_rn(M[(k0b + 2 * t) * kS + n0 + g]), b1 = tf32_rn(M[(k0b + 2 * t + 1) * kS + n0 + g]);
    mma1688_tf32(d, tf32_rn(c[0]), tf32_rn(c[2]), tf32_rn(c[1]), tf32_rn(c[3]), b0, b1);
}

__device__ void invert_unit_lower(float* M, int tid) {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    float x[16];
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
        const float* Ab = M + 16 * b * kS + 16 * b;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int j = 0; j + 3 < r; j += 4) {
                const float4 av = *reinterpret_cast<const float4*>(Ab + r * kS + j);
                a0 = fmaf(av.x, x[j], a0);
                a1 = fmaf(av.y, x[j + 1], a1);
                a2 = fmaf(av.z, x[j + 2], a2);
                a3 = fmaf(av.w, x[j + 3], a3);
            }
#pragma unroll
            for (int j = r & ~3; j < r; ++j) a0 = fmaf(Ab[r * kS + j], x[j], a0);
            x[r] = r < c ? 0.f : (r == c ? 1.f : -((a0 + a1) + (a2 + a3)));
        }
    }
    __syncthreads();
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
#pragma unroll
        for (int r = 0; r < 16; ++r) M[(16 * b + r) * kS + 16 * b + c] = x[r];
    }
    __syncthreads();
    if (warp < 2) {  // T_{b+1,b} = -(T_{b+1,b+1} A_{b+1,b}) T_bb for b = 0 (warp 0) and b = 2 (warp 1)
        const int b = 2 * warp, R1 = 16 * (b + 1), C0 = 16 * b;
        float d1[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_tf_a(d1[nt], M, R1, R1 + 8 * ks, R1 + 8 * ks, C0 + 8 * nt, g, t, false);
        float d2[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_tf_c(d2[nt], d1[ks], M, C0 + 8 * ks, C0 + 8 * nt, g, t);
        __syncwarp();
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            *reinterpret_cast<float2*>(M + (R1 + g) * kS + C0 + 8 * nt + 2 * t) = make_float2(-d2[nt][0], -d2[nt][1]);
            *reinterpret_cast<float2*>(M + (R1 + g + 8) * kS + C0 + 8 * nt + 2 * t) = make_float2(-d2[nt][2], -d2[nt][3]);
        }
    }
    __syncthreads();
    if (warp < 4) {  // T[32:64, 0:32] = -(T[32:64, 32:64] A[32:64, 0:32]) T[0:32, 0:32], one 16x16 tile per warp
        const int RB = 32 + 16 * (warp >> 1), CB = 16 * (warp & 1);
        float d1[4][4] = {};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma_tf_a(d1[nt], M, RB, 32 + 8 * ks, 32 + 8 * ks, 8 * nt, g, t, false);
        asm volatile("bar.sync 1, 128;" ::: "memory");  // every warp has read A[32:64, 0:32]
        float d2[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_tf_c(d2[nt], d1[ks], M, 8 * ks, CB + 8 * nt, g, t);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            *reinterpret_cast<float2*>(M + (RB + g) * kS + CB + 8 * nt + 2 * t) = make_float2(-d2[nt][0], -d2[nt][1]);
            *reinterpret_cast<float2*>(M + (RB + g + 8) * kS + CB + 8 * nt + 2 * t) = make_float2(-d2[nt][2], -d2[nt][3]);
        }
    }
    __syncthreads();
}

// One row r of A from 16 columns of G starting at c0 (fp32 to shared memory, stride kS).
__device__ __forceinline__ void a_row16(const Scal* sc, const uint32_t (&u)[16], int r, int c0, bool fast, float* AF) {
    float a[16];
    if (fast) {
        const float ex = sc->eLx[r];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) a[jj] = c0 + jj < r ? ex * sc->cA[c0 + jj] * __uint_as_float(u[jj]) : 0.f;
    } else {
        const float lx = sc->Lx[r];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
            a[jj] = c0 + jj < r ? sc->eta[c0 + jj] * __expf(lx - sc->L[c0 + jj]) * __uint_as_float(u[jj]) : 0.f;
    }
    float4* dst = reinterpret_cast<float4*>(AF + r * kS + c0);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]);
}

// ---------------------------------------------------------------- prep kernel: M_n, U_n, T_n
// The products are M = 128 with the wanted rows in TMEM lanes 64-127 (or in both halves), so that
// every epilogue reads whole 32-lane quadrants; the A operand's first 64 rows are then the tile
// that precedes the wanted one in shared memory (Y before X):
//   [Y; X] X^T            -> G in lanes 64-127
//   [Y^T; X^T] diag(w) T  -> Z = X^T diag(w) T in lanes 64-127 (MN-major A: the tiles are its two atoms)
//   [Z'; Z] [Y | X]       -> Z' X in lanes 0-63 / columns 64-127, Z Y in lanes 64-127 / columns 0-63
// The accumulators take turns in TMEM columns 0-127 (each is read out before the next MMA).
namespace prep {
constexpr int Y = 0, X = kTile;                  // Y first: [Y; X] stacks with X in rows 64-127
constexpr int AF = 2 * kTile;                    // fp32 A, inverted in place into T; then Z' hi, Z hi
constexpr int TT = AF + kFBytes;                 // diag(w) T hi / lo (MN-major B tiles); then Z' lo, Z lo
constexpr int SCAL = TT + 2 * kTile;
constexpr int BAR = SCAL + (int)sizeof(Scal);
constexpr int BYTES = BAR + 32;
constexpr int ALLOC = BYTES + 1024;
constexpr uint32_t kCols = 128;
static_assert(AF % 1024 == 0 && TT % 1024 == 0 && BAR % 8 == 0 && 2 * kTile <= kFBytes, "layout");
}  // namespace prep

__global__ void __launch_bounds__(256, 4) falcon_prep_kernel(const __grid_constant__ SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = (int)(blockIdx.x / p.BH);  // chunk-major: every sequence's chunk n before chunk n + 1
    const long long bh = blockIdx.x - (long long)n * p.BH;
    const long long cid = bh * p.N + n;      // the chunk's workspace slot
    const long long t0 = (long long)n * kC;
    const int nv = (int)min((long long)kC, p.T - t0);
    const bool f1 = p.variant == kF1;
    Scal* sc = reinterpret_cast<Scal*>(sm + prep::SCAL);
    float* AF = reinterpret_cast<float*>(sm + prep::AF);
    const uint32_t bar_tma = base + prep::BAR, bar_mma = base + prep::BAR + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + prep::BAR + 16);

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        mbar_init_fence();
        mbar_expect_tx(bar_tma, 2 * kTile);
        tma_load_3d(base + prep::X, &p.tm_k, 0, (int)t0 - 1, (int)bh, bar_tma);  // row i = k_{t0+i-1}
        tma_load_3d(base + prep::Y, &p.tm_v, 0, (int)t0, (int)bh, bar_tma);
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), prep::kCols);
    if (tid == 32) {  // this call's flag of the chunk starts cleared, visibly before the trigger below
        p.fl_prep[cid] = 0;
        __threadfence();
    }
    float beta_i = 0.f, lam_i = 0.f;
    if (tid < nv) {
        beta_i = p.beta[bh * p.T + t0 + tid];
        lam_i = p.lam[bh * p.T + t0 + tid];
    }
    if (f1)  // A's blocks above the diagonal must read as zero in the block merges
        for (int i = tid; i < kFBytes / 16; i += 256) reinterpret_cast<float4*>(AF)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The chain kernel may launch once every prep CTA is resident; it waits on the chunk flags.
    pdl_launch_dependents();
    const uint32_t tmem = *tslot;
    const int q4 = warp & 3, hw = warp >> 2;
    const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);  // this warp's TMEM lane quadrant
    const int trow = 32 * q4 + lane;                           // this thread's TMEM lane

    if (!cta_wait(bar_tma, 0, tid)) return release_tmem(tmem, warp, prep::kCols);
    if (n == 0 && p.pos > 0 && tid < 8) {  // a continuation's first shifted key is k_pos, from the tail
        const uint4 v = reinterpret_cast<const uint4*>(p.tail + bh * 64)[tid];
        *reinterpret_cast<uint4*>(sm + prep::X + sw128(0, 8 * tid)) = v;
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {  // [Y; X] X^T: G in lanes 64-127
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem, desc_k(base + prep::Y + 32 * ks), desc_k(base + prep::X + 32 * ks), id, ks > 0);
        mma_commit(bar_mma);
    }
    chunk_scalars(sc, sm + prep::X, tid, beta_i, lam_i, nv, p.pos + t0 + 1, p.eps, p.eps_gamma);
    const bool fast = sc->misc[3] != 0.f;
    if (tid < (int)(sizeof(Scal) / 16))  // the scalars, for the output kernel
        reinterpret_cast<uint4*>(p.ws_sc + cid * kScalBytes)[tid] = reinterpret_cast<const uint4*>(sc)[tid];
    if (!cta_wait(bar_mma, 0, tid)) return release_tmem(tmem, warp, prep::kCols);
    tc_fence_after();

    // ---- A (Falcon-1): lanes 64-127 hold G; two threads per row (warps 2, 3, 6, 7), 32 columns each
    if (f1 && trow >= 64) {
        const int r = trow - 64, c0 = 32 * hw;
        uint32_t u0[16], u1[16];
        tmem_ld16(tq + c0, u0);
        tmem_ld16(tq + c0 + 16, u1);
        tmem_wait_ld();
        regs_ready(u0);
        regs_ready(u1);
        if (c0 < r) a_row16(sc, u0, r, c0, fast, AF);
        if (c0 + 16 < r) a_row16(sc, u1, r, c0 + 16, fast, AF);
    }
    tc_fence_before();
    __syncthreads();
    if (f1) invert_unit_lower(AF, tid);

    // ---- T (hi / lo, row-major) to the workspace for the output kernel, and diag(w) T as the
    // MN-major B operand of Z (Falcon-1A: T = I)
    {
        uint8_t* TTh = sm + prep::TT;
        uint4* th = reinterpret_cast<uint4*>(p.ws_t + cid * 2 * 4096);
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            const int task = tid + 256 * k2, i = task >> 3, c8 = 8 * (task & 7);
            const float wi = sc->w[i];
            float v[8];
            if (f1) {
                const float4 a = *reinterpret_cast<const float4*>(AF + i * kS + c8);
                const float4 b = *reinterpret_cast<const float4*>(AF + i * kS + c8 + 4);
                v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = c8 + e == i ? 1.f : 0.f;
            }
            uint4 h, l;
            hilo8(v, h, l);
            th[task] = h;        // row i, columns c8..c8+7 of T_hi
            th[512 + task] = l;  // and of T_lo
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] *= wi;
            st8_hilo(TTh, TTh + kTile, sw128(i, c8), v);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // [Y^T; X^T] (T''_hi + T''_lo): Z in lanes 64-127; A MN-major with atoms Y and X
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, true, true);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem, desc_mn(base + prep::Y + 2048 * ks, kTile), desc_mn(base + prep::TT + 2048 * ks, kTile), id,
                     ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem, desc_mn(base + prep::Y + 2048 * ks, kTile),
                     desc_mn(base + prep::TT + kTile + 2048 * ks, kTile), id, 1);
        mma_commit(bar_mma);
    }
    if (!cta_wait(bar_mma, 1, tid)) return release_tmem(tmem, warp, prep::kCols);
    tc_fence_after();

    // ---- Z (lanes 64-127) -> Z hi / lo and Z' = Z diag(e^{Lx}) hi / lo
    // (K-major A tiles: [Z'h; Zh] at AF, [Z'l; Zl] at TT)
    if (trow >= 64) {
        const int a = trow - 64, c0 = 32 * hw;
        float z[32];
        tmem_ld32(tq + c0, z);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j0 = c0 + 8 * c;
            float zp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) zp[e] = z[8 * c + e] * sc->eLx[j0 + e];
            const uint32_t off = sw128(a, j0);
            st8_hilo(sm + prep::AF + kTile, sm + prep::TT + kTile, off, z + 8 * c);
            st8_hilo(sm + prep::AF, sm + prep::TT, off, zp);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // [Z'; Z] [Y | X]: Y and X are the two 64-column atoms of an MN-major B
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 128, false, true);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem, desc_k(base + prep::AF + 32 * ks), desc_mn(base + prep::Y + 2048 * ks, kTile), id, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem, desc_k(base + prep::TT + 32 * ks), desc_mn(base + prep::Y + 2048 * ks, kTile), id, 1);
        mma_commit(bar_mma);
    }
    if (!cta_wait(bar_mma, 0, tid)) return release_tmem(tmem, warp, prep::kCols);
    tc_fence_after();

    // ---- lanes 0-63: M = e^{L_C} I - Z' X (hi / lo bf16); lanes 64-127: U = Z Y (fp32)
    {
        float v[32];
        const bool mrow = trow < 64;
        const int a = trow & 63;
        tmem_ld32(tq + (mrow ? 64 : 0) + 32 * hw, v);
        if (mrow) {
            const float eLC = sc->misc[0];
            uint4* mh = reinterpret_cast<uint4*>(p.ws_m + (cid * 2 * 64 + a) * 64 + 32 * hw);
            uint4* ml = reinterpret_cast<uint4*>(p.ws_m + ((cid * 2 + 1) * 64 + a) * 64 + 32 * hw);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float m[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int b = 32 * hw + 8 * c + e;
                    m[e] = (b == a ? eLC : 0.f) - (f1 ? v[8 * c + e] : 0.f);
                }
                uint4 h, l;
                hilo8(m, h, l);
                mh[c] = h;
                ml[c] = l;
            }
        } else {
            float4* u = reinterpret_cast<float4*>(p.ws_u + (cid * 64 + a) * 64 + 32 * hw);
#pragma unroll
            for (int c = 0; c < 8; ++c) u[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        }
    }
    tc_fence_before();
    publish(p.fl_prep + cid, p.epoch, tid);  // M, U, T and the scalars of chunk n are in the workspace
    if (warp == 0) tmem_dealloc(tmem, prep::kCols);
}

// ---------------------------------------------------------------- chain kernel: S_{n+1} = M_n S_n + U_n
// One CTA per sequence (one per SM). The state's columns split into two 32-column halves that
// evolve independently (S_{n+1}[:, c] depends only on S_n[:, c]); each half is its own pipeline:
//   warp 10 (loader)   per chunk, waits for the prep kernel's flag, then TMA-loads M_n (hi, lo) and
//                      U_n into a 3-stage ring
//   warp 8 (issuer)    per half and step eight tcgen05 MMAs D_h = (M_hi + M_lo) B_h, where the B
//                      tile of half h is [S_hi | S_lo] of its 32 columns (one 64-column MN-major atom)
//   warps 4h..4h+3     the epilogue of half h: 16x256b TMEM loads of D_h, S_{n+1} = D_h[:, c] +
//                      D_h[:, 32 + c] + U_n in fp32, written as the next B tile (three per half)
//   warp 9 (copier)    each finished B tile to the workspace as the output kernel's S_n
// so that one half's epilogue runs while the other half's MMAs do, and the scan follows the prep
// kernel chunk by chunk instead of waiting for all of it. The barriers that hand a B tile over are
// kept per buffer, so no waiter can fall two phases behind its barrier. All waits are bounded; a
// timeout raises the device flag and every role leaves its loop.
namespace chain {
constexpr int kStages = 3;
constexpr int kUBytes = 64 * 64 * 4;        // U_n, fp32, as two [64][32] halves (128-byte swizzle)
constexpr int kUBytesHalf = kUBytes / 2;
constexpr int kStage = 2 * kTile + kUBytes; // M hi, M lo, U
constexpr int BT = kStages * kStage;        // B tiles [half][buffer]
constexpr int kBuf = 3;                     // B tiles per half: S_n, S_{n+1} and the one being copied
constexpr int kStaging = 2;                 // staging buffers, each S_m hi and lo as standard 64 x 64 tiles
constexpr int SG = BT + 2 * kBuf * kTile;
constexpr int BAR = SG + kStaging * 2 * kTile;
// full[s], empty[s], mma done[h], state ready[h][b], copied[h][b], drain
constexpr int kBars = 2 * kStages + 2 + 4 * kBuf + 1;
constexpr int BYTES = BAR + 8 * kBars + 16;
constexpr int ALLOC = BYTES + 1024;
constexpr int kThreads = 352;
constexpr uint32_t kTmemCols = 128;
static_assert(kStage % 1024 == 0 && BT % 1024 == 0 && SG % 1024 == 0, "stage alignment");
}  // namespace chain

__global__ void __launch_bounds__(chain::kThreads, 1) falcon_chain_kernel(const __grid_constant__ SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, t = lane & 3;
    const long long bh = blockIdx.x;
    const int N = p.N;
    auto bar = [&](int i) -> uint32_t { return base + chain::BAR + 8 * i; };
    auto full = [&](int s) { return bar(s); };
    auto empty = [&](int s) { return bar(chain::kStages + s); };
    auto mmad = [&](int h) { return bar(2 * chain::kStages + h); };
    constexpr int kB = chain::kBuf;
    // phase k of ready(h, b) / copied(h, b): S_{b + kB k} is in tile (h, b) / has been read from it
    auto ready = [&](int h, int b) { return bar(2 * chain::kStages + 2 + kB * h + b); };
    auto copied = [&](int h, int b) { return bar(2 * chain::kStages + 2 + 2 * kB + kB * h + b); };
    const uint32_t drain = bar(2 * chain::kStages + 2 + 4 * kB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + chain::BAR + 8 * chain::kBars);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + chain::BAR + 8 * chain::kBars + 4);
    auto btile = [&](int h, int b) { return chain::BT + (kB * h + b) * kTile; };
    auto fail = [&]() {
        *abort_flag = 1;
        atomicExch(&g_split_timeout_flag, 1);
        return false;
    };
    auto wait = [&](uint32_t br, uint32_t parity) -> bool {  // bounded; gives up early once any role failed
        if (mbar_try(br, parity)) return true;
        const long long c0 = clock64();
        while (!mbar_try(br, parity)) {
            if (*abort_flag) return false;
            __nanosleep(20);
            if (clock64() - c0 > kTimeoutCycles) return fail();
        }
        return true;
    };
    if (tid == 0) {
        for (int s = 0; s < chain::kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 256);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(mmad(h), 1);
            for (int b = 0; b < kB; ++b) {
                mbar_init(ready(h, b), 128);
                mbar_init(copied(h, b), 32);
            }
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), chain::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The output kernel may launch once every chain CTA is resident: its state-independent part runs
    // alongside the scan, and it waits for this kernel's completion before it reads S_n.
    pdl_launch_dependents();
    const uint32_t tmem = *tslot;
    bool ok = true;

    if (warp < 8) {
        // ------------------------------------------------------------ epilogue of half h
        const int h = warp >> 2, q4 = warp & 3;
        const int r0 = 16 * q4 + (lane >> 2);  // rows r0 and r0 + 8 (TMEM quadrant q4)
        const int c0 = 32 * h;                 // this half's first state column
        const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16) + 64 * h;
        float sv[4][4];  // columns c0 + 8j + 2t (+1), j = 0..3; [0..1] row r0, [2..3] row r0 + 8
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 x = make_float2(0.f, 0.f), y = make_float2(0.f, 0.f);
            if (p.S0) {
                x = *reinterpret_cast<const float2*>(p.S0 + (bh * 64 + r0) * 64 + c0 + 8 * j + 2 * t);
                y = *reinterpret_cast<const float2*>(p.S0 + (bh * 64 + r0 + 8) * 64 + c0 + 8 * j + 2 * t);
            }
            sv[j][0] = x.x, sv[j][1] = x.y, sv[j][2] = y.x, sv[j][3] = y.y;
        }
        auto put_state = [&](int b) {  // fragment -> B tile (h, b): hi in columns 0-31, lo in 32-63
            uint8_t* bt = sm + btile(h, b);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int row = r0 + 8 * hf, col = 8 * j + 2 * t;
                    uint32_t hi, lo;
                    split2(sv[j][2 * hf], sv[j][2 * hf + 1], hi, lo);
                    *reinterpret_cast<uint32_t*>(bt + sw128(row, col)) = hi;
                    *reinterpret_cast<uint32_t*>(bt + sw128(row, col + 32)) = lo;
                }
            fence_async_smem();
        };
        // U half tile: [64][32] fp32 rows of 128 bytes, 16-byte chunks swizzled by row % 8
        auto u_at = [&](const uint8_t* uh, int row, int col) {
            return *reinterpret_cast<const float2*>(uh + row * 128 + ((((col >> 2) ^ (row & 7))) << 4) + 4 * (col & 3));
        };
        put_state(0);
        mbar_arrive(ready(h, 0));
        for (int n = 0; n < N; ++n) {
            const int s = n % chain::kStages;
            if (!wait(full(s), (n / chain::kStages) & 1)) {  // U_n in stage s
                ok = false;
                break;
            }
            const uint8_t* uh = sm + s * chain::kStage + 2 * kTile + h * chain::kUBytesHalf;
            float2 ua[4], ub[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                ua[j] = u_at(uh, r0, 8 * j + 2 * t);
                ub[j] = u_at(uh, r0 + 8, 8 * j + 2 * t);
            }
            if (!wait(mmad(h), n & 1)) {
                ok = false;
                break;
            }
            mbar_arrive(empty(s));  // this half's MMAs of step n are done with M_n, and U_n is read
            tc_fence_after();
            uint32_t d0[16], d1[16];
            tmem_ld_16x256b_x4(tq, d0);       // M S_hi part
            tmem_ld_16x256b_x4(tq + 32, d1);  // M S_lo part
            tmem_wait_ld();
            regs_ready(d0);
            regs_ready(d1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sv[j][0] = __uint_as_float(d0[4 * j]) + __uint_as_float(d1[4 * j]) + ua[j].x;
                sv[j][1] = __uint_as_float(d0[4 * j + 1]) + __uint_as_float(d1[4 * j + 1]) + ua[j].y;
                sv[j][2] = __uint_as_float(d0[4 * j + 2]) + __uint_as_float(d1[4 * j + 2]) + ub[j].x;
                sv[j][3] = __uint_as_float(d0[4 * j + 3]) + __uint_as_float(d1[4 * j + 3]) + ub[j].y;
            }
            const int b = (n + 1) % kB;  // the tile that held S_{n+1-kB}: its copy must be done
            if (n + 1 >= kB && !wait(copied(h, b), ((n + 1 - kB) / kB) & 1)) {
                ok = false;
                break;
            }
            put_state(b);
            tc_fence_before();
            mbar_arrive(ready(h, b));  // S_{n+1} written; D_h read
        }
        if (ok && p.S_final) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                *reinterpret_cast<float2*>(p.S_final + (bh * 64 + r0) * 64 + c0 + 8 * j + 2 * t) =
                    make_float2(sv[j][0], sv[j][1]);
                *reinterpret_cast<float2*>(p.S_final + (bh * 64 + r0 + 8) * 64 + c0 + 8 * j + 2 * t) =
                    make_float2(sv[j][2], sv[j][3]);
            }
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------ issuer
        if (lane == 0) {
            int mma_issued = 0;
            for (int n = 0; n < N && ok; ++n) {
                const int s = n % chain::kStages;
                if (!wait(full(s), (n / chain::kStages) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t st = base + s * chain::kStage;
                for (int h = 0; h < 2; ++h) {
                    if (!wait(ready(h, n % kB), (n / kB) & 1)) {  // S_n in tile (h, n % kB); D_h read out
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    constexpr uint32_t id = idesc_bf16(64, 64, false, true);
                    const uint32_t bt = base + btile(h, n % kB);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16(tmem + 64 * h, desc_k(st + part * kTile + 32 * ks),
                                     desc_mn(bt + 2048 * ks, kTile), id, part + ks > 0);
                    mma_commit(mmad(h));
                    mma_issued = 1;
                }
            }
            if (!ok && mma_issued) {  // let the MMAs in flight finish (bounded) before TMEM is freed
                mma_commit(drain);
                mbar_wait_bounded(drain, 0, kTimeoutCycles);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ copier: B tiles -> S_m in the workspace
        // Each half's B tile is regrouped into standard hi and lo tiles in a staging buffer, which lane 0
        // stores with TMA; a staging buffer is reused once its store has read it.
        for (int m = 0; m < N && ok; ++m) {
            const int g = m % chain::kStaging;
            uint8_t* sg = sm + chain::SG + g * 2 * kTile;
            if (lane == 0) bulk_wait_read<chain::kStaging - 1>();  // the store that last used buffer g has read it
            __syncwarp();
            for (int h = 0; h < 2; ++h) {
                if (!wait(ready(h, m % kB), (m / kB) & 1)) {
                    ok = false;
                    break;
                }
                const uint8_t* bt = sm + btile(h, m % kB);
                // all loads before any store: the two areas share one array, so interleaving them
                // would serialise every load behind the store before it
                const int c = lane & 7, cs = 4 * h + (c & 3);  // chunk c: hi 0-3, lo 4-7; its place in the standard tile
                uint4 v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int row = (lane >> 3) + 4 * k;
                    v[k] = *reinterpret_cast<const uint4*>(bt + row * 128 + ((c ^ (row & 7)) << 4));
                }
                mbar_arrive(copied(h, m % kB));  // tile (h, m % kB) has been read
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int row = (lane >> 3) + 4 * k;
                    *reinterpret_cast<uint4*>(sg + (c >> 2) * kTile + row * 128 + ((cs ^ (row & 7)) << 4)) = v[k];
                }
            }
            if (!ok) break;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                const uint32_t sa = base + chain::SG + g * 2 * kTile;
                tma_store_2d(&p.tm_s, sa, 0, (int)((bh * N + m) * 128));
                tma_store_2d(&p.tm_s, sa + kTile, 0, (int)((bh * N + m) * 128 + 64));
                bulk_commit();
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        if (ok && p.tail_out && lane < 8) {  // window 1: the tail is the last key (the next call's x)
            uint4 v = make_uint4(0, 0, 0, 0);
            if (p.T > 0) v = reinterpret_cast<const uint4*>(p.k + (bh * p.T + p.T - 1) * 64)[lane];
            else if (p.pos > 0) v = reinterpret_cast<const uint4*>(p.tail + bh * 64)[lane];
            reinterpret_cast<uint4*>(p.tail_out + bh * 64)[lane] = v;
        }
    } else {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            int last[chain::kStages] = {-1, -1, -1};
            for (int m = 0; m < N && ok; ++m) {
                const int s = m % chain::kStages;
                if (m >= chain::kStages && !wait(empty(s), ((m / chain::kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                if (!wait_flag_bounded(p.fl_prep + bh * N + m, p.epoch, kTimeoutCycles)) {
                    ok = fail();
                    break;
                }
                fence_proxy_async_global();
                const uint32_t st = base + s * chain::kStage;
                const int row = (int)((bh * N + m) * 128);
                mbar_expect_tx(full(s), chain::kStage);
                tma_load_2d(st, &p.tm_m, 0, row, full(s));
                tma_load_2d(st + kTile, &p.tm_m, 0, row + 64, full(s));
                tma_load_2d(st + 2 * kTile, &p.tm_u, 0, (int)((bh * N + m) * 64), full(s));
                tma_load_2d(st + 2 * kTile + chain::kUBytesHalf, &p.tm_u, 32, (int)((bh * N + m) * 64), full(s));
                last[s] = m;
            }
            if (!ok)  // drain the loads in flight (at most one per stage), bounded
                for (int s = 0; s < chain::kStages; ++s)
                    if (last[s] >= 0) mbar_wait_bounded(full(s), (last[s] / chain::kStages) & 1, kTimeoutCycles);
        }
        __syncwarp();
    }
    // Completion of this grid implies completion of the prep grid (the stream's next launch relies on it).
    pdl_wait();
    release_tmem(tmem, warp, chain::kTmemCols);
}

// ---------------------------------------------------------------- output kernel: R and O from S_n
// Every product is M = 128 with the wanted rows in TMEM lanes 64-127 (or 0-63 and 64-127 both
// wanted), so each epilogue reads whole 32-lane quadrants. Where only the second 64 rows are
// wanted, the first 64 rows of the A operand are whatever tile precedes it in shared memory.
namespace outk {
// 8 KB tiles. Loaded: X, Q, Y, S_hi, S_lo, T_hi, T_lo; built: P_hi, P_lo. Later tenants of dead
// tiles: Y' hi / lo in X / Q, R hi / lo in Y / S_hi, the output tile in X. The order makes the
// stacked operands [X; Q], [S_lo; T_hi], [T_hi; T_lo], [T_lo; P_hi] and [P_hi; P_lo] contiguous.
constexpr int X = 0, Q = 1, Y = 2, SH = 3, SL = 4, TH = 5, TL = 6, PH = 7, PL = 8;
constexpr int YH = X, YL = Q, RH = Y, RL = SH, OUT = X;
constexpr int SCAL = 9 * kTile;
constexpr int BAR = SCAL + (int)sizeof(Scal);
constexpr int BYTES = BAR + 32;
constexpr int ALLOC = BYTES + 1024;
constexpr uint32_t kCols = 128;
constexpr uint32_t D1 = 0, DXQ = 64, DR = 0, DO = 0;  // D1 -> DR -> DO take turns in columns 0-63
static_assert(BAR % 8 == 0 && SCAL % 16 == 0, "layout");
}  // namespace outk

__global__ void __launch_bounds__(256, 3) falcon_out_kernel(const __grid_constant__ SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    auto tile = [&](int i) -> uint8_t* { return sm + i * kTile; };
    auto taddr = [&](int i) -> uint32_t { return base + (uint32_t)(i * kTile); };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = (int)(blockIdx.x / p.BH);  // chunk-major, in the order the chain produces S_n
    const long long bh = blockIdx.x - (long long)n * p.BH;
    const long long cid = bh * p.N + n;      // the chunk's workspace slot
    const long long t0 = (long long)n * kC;
    const bool f1 = p.variant == kF1;
    const Scal* sc = reinterpret_cast<const Scal*>(sm + outk::SCAL);
    const uint32_t bar_tma = base + outk::BAR, bar_mma = base + outk::BAR + 8, bar_s = base + outk::BAR + 16;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + outk::BAR + 24);

    int bad = 0;  // thread 0: a producer's flag never came
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_s, 1);
        mbar_init_fence();
        mbar_expect_tx_only(bar_tma, 3 * kTile);  // the inputs first; the phase still needs the arrive below
        tma_load_3d(taddr(outk::X), &p.tm_k, 0, (int)t0 - 1, (int)bh, bar_tma);
        tma_load_3d(taddr(outk::Q), &p.tm_q, 0, (int)t0, (int)bh, bar_tma);
        tma_load_3d(taddr(outk::Y), &p.tm_v, 0, (int)t0, (int)bh, bar_tma);
        if (wait_producer(p.fl_prep + cid, p.epoch)) {  // T and the scalars of the chunk come from the prep kernel
            mbar_expect_tx(bar_tma, 2 * kTile + (uint32_t)sizeof(Scal));
            tma_load_2d(taddr(outk::TH), &p.tm_t, 0, (int)(cid * 128), bar_tma);
            tma_load_2d(taddr(outk::TL), &p.tm_t, 0, (int)(cid * 128 + 64), bar_tma);
            bulk_load(base + outk::SCAL, p.ws_sc + cid * kScalBytes, (uint32_t)sizeof(Scal), bar_tma);
        } else {
            bad = 1;
            mbar_arrive(bar_tma);  // the phase completes once the inputs have landed
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), outk::kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int q4 = warp & 3, hw = warp >> 2;
    const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);
    const int trow = 32 * q4 + lane;
    const bool upper = trow >= 64;  // lanes 64-127: warps 2, 3, 6, 7
    const int r = trow & 63;

    if (!cta_wait(bar_tma, 0, tid, bad)) return release_tmem(tmem, warp, outk::kCols);
    if (n == 0 && p.pos > 0 && tid < 8) {
        const uint4 v = reinterpret_cast<const uint4*>(p.tail + bh * 64)[tid];
        *reinterpret_cast<uint4*>(tile(outk::X) + sw128(0, 8 * tid)) = v;
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idk = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // [G; Sc] = [X; Q] X^T
            mma_bf16(tmem + outk::D1, desc_k(taddr(outk::X) + 32 * ks), desc_k(taddr(outk::X) + 32 * ks), idk, ks > 0);
        mma_commit(bar_mma);
    }
    const bool fast = sc->misc[3] != 0.f;
    if (!cta_wait(bar_mma, 0, tid)) return release_tmem(tmem, warp, outk::kCols);
    tc_fence_after();

    // ---- lanes 64-127: P rows (K-major A tiles)
    if (upper) {
        float v[32];
        tmem_ld32(tq + outk::D1 + 32 * hw, v);
        const int i = r;
        float pv[32];
        if (fast) {
            const float el = sc->eL[i];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = 32 * hw + jj;
                pv[jj] = j <= i ? el * sc->cA[j] * v[jj] : 0.f;
            }
        } else {
            const float li = sc->L[i];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = 32 * hw + jj;
                pv[jj] = j <= i ? sc->eta[j] * __expf(li - sc->L[j]) * v[jj] : 0.f;
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) st8_hilo(tile(outk::PH), tile(outk::PL), sw128(i, 32 * hw + 8 * c), pv + 8 * c);
    }

    // ---- the chunk-start state from the chain kernel: [X S; Q S]
    pdl_wait();  // the chain kernel has completed: every S_n is in the workspace
    if (tid == 0) {
        mbar_expect_tx(bar_s, 2 * kTile);
        tma_load_2d(taddr(outk::SH), &p.tm_s, 0, (int)(cid * 128), bar_s);
        tma_load_2d(taddr(outk::SL), &p.tm_s, 0, (int)(cid * 128 + 64), bar_s);
    }
    if (!cta_wait(bar_s, 0, tid, bad)) return release_tmem(tmem, warp, outk::kCols);
    if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idm = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int part = 0; part < 2; ++part)  // S = S_hi + S_lo (MN-major, K = feature)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + outk::DXQ, desc_k(taddr(outk::X) + 32 * ks),
                         desc_mn(taddr(outk::SH + part) + 2048 * ks, kTile), idm, part + ks > 0);
        mma_commit(bar_mma);
    }
    if (!cta_wait(bar_mma, 1, tid)) return release_tmem(tmem, warp, outk::kCols);
    tc_fence_after();

    // ---- lanes 0-63: Y' = Y - diag(e^{Lx}) X S rows (MN-major B), into the dead X and Q tiles
    if (!upper) {
        float v[32];
        tmem_ld32(tq + outk::DXQ + 32 * hw, v);
        const float ex = f1 ? sc->eLx[r] : 0.f;
        float y[4][8];
#pragma unroll
        for (int c = 0; c < 4; ++c)
            unpack8(*reinterpret_cast<const uint4*>(tile(outk::Y) + sw128(r, 32 * hw + 8 * c)), y[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int e = 0; e < 8; ++e) y[c][e] = fmaf(-ex, v[8 * c + e], y[c][e]);
            st8_hilo(tile(outk::YH), tile(outk::YL), sw128(r, 32 * hw + 8 * c), y[c]);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // R = T Y' in lanes 64-127: A = [S_lo; T_hi] carries T_hi, [T_hi; T_lo] carries T_lo
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + outk::DR, desc_k(taddr(outk::TH - 1) + 32 * ks), desc_mn(taddr(outk::YH) + 2048 * ks, kTile),
                     id, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + outk::DR, desc_k(taddr(outk::TH - 1) + 32 * ks), desc_mn(taddr(outk::YL) + 2048 * ks, kTile),
                     id, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + outk::DR, desc_k(taddr(outk::TL - 1) + 32 * ks), desc_mn(taddr(outk::YH) + 2048 * ks, kTile),
                     id, 1);
        mma_commit(bar_mma);
    }
    if (!cta_wait(bar_mma, 0, tid)) return release_tmem(tmem, warp, outk::kCols);
    tc_fence_after();
    if (upper) {  // R rows -> hi / lo (MN-major B, K = token) in the dead Y and S_hi tiles
        float v[32];
        tmem_ld32(tq + outk::DR + 32 * hw, v);
#pragma unroll
        for (int c = 0; c < 4; ++c) st8_hilo(tile(outk::RH), tile(outk::RL), sw128(r, 32 * hw + 8 * c), v + 8 * c);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // P R in lanes 64-127: A = [T_lo; P_hi] carries P_hi, [P_hi; P_lo] carries P_lo
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + outk::DO, desc_k(taddr(outk::PH - 1) + 32 * ks), desc_mn(taddr(outk::RH) + 2048 * ks, kTile),
                     id, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + outk::DO, desc_k(taddr(outk::PH - 1) + 32 * ks), desc_mn(taddr(outk::RL) + 2048 * ks, kTile),
                     id, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + outk::DO, desc_k(taddr(outk::PL - 1) + 32 * ks), desc_mn(taddr(outk::RH) + 2048 * ks, kTile),
                     id, 1);
        mma_commit(bar_mma);
    }
    if (!cta_wait(bar_mma, 1, tid)) return release_tmem(tmem, warp, outk::kCols);
    tc_fence_after();
    if (upper) {  // O = diag(e^L) Q S + P R -> bf16 output tile
        float qs[32], po[32];
        tmem_ld32x2(tq + outk::DXQ + 32 * hw, tq + outk::DO + 32 * hw, qs, po);
        const float el = sc->eL[r];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = fmaf(el, qs[8 * c + e], po[8 * c + e]);
            *reinterpret_cast<uint4*>(tile(outk::OUT) + sw128(r, 32 * hw + 8 * c)) = pack8(o);
        }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {  // TMA store; rows past T are clipped
        tma_store_3d(&p.tm_out, taddr(outk::OUT), 0, (int)t0, (int)bh);
        tma_store_wait_read();
    }
    release_tmem(tmem, warp, outk::kCols);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(q);
    }
    return fn;
}

// [BH][T][64] bf16, 64 x 64 boxes, 128-byte swizzle
bool encode_bhtd(CUtensorMap* tm, const void* ptr, long long T, long long BH) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {64 * 2, (cuuint64_t)T * 64 * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [rows][64] bf16, 64 x 64 boxes, 128-byte swizzle
bool encode_rows(CUtensorMap* tm, const void* ptr, long long rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    cuuint64_t strides[1] = {64 * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// U: [rows][64] fp32, boxes of 32 columns x 64 rows, 128-byte swizzle
bool encode_u(CUtensorMap* tm, const void* ptr, long long rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    cuuint64_t strides[1] = {64 * 4};
    cuuint32_t box[2] = {32, 64};
    cuuint32_t es[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int smem_optin() {
    static int v = -1;
    if (v < 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            v = 0;
    }
    return v;
}

long long n_chunks(const Launch& a) { return (a.T + kC - 1) / kC; }


}  // namespace

bool split_supported(const Launch& a) {
    const long long BH = a.B * a.H;
    return (a.variant == kF1 || a.variant == kF1A) && a.bf16 && a.dk == 64 && a.dv == 64 && a.chunk == 64 &&
           a.W == 1 && a.T < (1LL << 31) - 64 && BH < 65536 && BH * n_chunks(a) * 128 < (1LL << 31);
}

// Per chunk: M, U, S, T (16 KB each), the scalars (kScalBytes) and an 8-byte flag.
size_t split_workspace_bytes(const Launch& a) {
    return (size_t)(a.B * a.H) * (size_t)n_chunks(a) * (size_t)(4 * 16384 + kScalBytes + 8);
}

int launch_split(const Launch& a, cudaStream_t st) {
    if (smem_optin() < outk::ALLOC) return 2;
    const long long BH = a.B * a.H, N = n_chunks(a);
    SplitParams p;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    const size_t per = (size_t)BH * (size_t)N * 16384;
    p.ws_m = reinterpret_cast<bf16*>(ws);
    p.ws_u = reinterpret_cast<float*>(ws + per);
    p.ws_s = reinterpret_cast<bf16*>(ws + 2 * per);
    p.ws_t = reinterpret_cast<bf16*>(ws + 3 * per);
    p.ws_sc = ws + 4 * per;
    p.fl_prep = reinterpret_cast<unsigned long long*>(ws + 4 * per + (size_t)BH * (size_t)N * kScalBytes);
    p.epoch = 1;
    p.BH = BH;
    if (N > 0) {
        if (!encode_bhtd(&p.tm_q, a.q, a.T, BH) || !encode_bhtd(&p.tm_k, a.k, a.T, BH) ||
            !encode_bhtd(&p.tm_v, a.v, a.T, BH) || !encode_bhtd(&p.tm_out, a.out, a.T, BH) ||
            !encode_rows(&p.tm_m, p.ws_m, BH * N * 128) || !encode_rows(&p.tm_s, p.ws_s, BH * N * 128) ||
            !encode_rows(&p.tm_t, p.ws_t, BH * N * 128) || !encode_u(&p.tm_u, p.ws_u, BH * N * 64))
            return 4;
    }
    p.beta = a.beta;
    p.lam = a.lam;
    p.S0 = a.S0;
    p.k = static_cast<const bf16*>(a.k);
    p.tail = static_cast<const bf16*>(a.tail);
    p.tail_out = static_cast<bf16*>(a.tail_out);
    p.S_final = a.S_final;
    p.T = a.T;
    p.pos = a.pos;
    p.N = (int)N;
    p.eps = a.eps;
    p.eps_gamma = a.eps_gamma;
    p.variant = a.variant;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(falcon_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, prep::ALLOC) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, chain::ALLOC) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, outk::ALLOC) !=
                cudaSuccess)
            return 4;
        attr_set = true;
    }
    // prep: an ordinary launch, after everything that used the workspace before. chain: a programmatic
    // dependent launch that starts once every prep CTA is resident and follows the prep kernel chunk
    // by chunk through the flags. output: a programmatic dependent launch whose state-independent part
    // overlaps the chain and which waits for the chain's completion before it reads S_n. No kernel
    // waits on one launched after it.
    if (N > 0) falcon_prep_kernel<<<(unsigned)(BH * N), 256, prep::ALLOC, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return 4;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)BH);
    cfg.blockDim = dim3(chain::kThreads);
    cfg.dynamicSmemBytes = chain::ALLOC;
    if (cudaLaunchKernelEx(&cfg, falcon_chain_kernel, p) != cudaSuccess) return 4;
    if (N > 0) {
        cfg.gridDim = dim3((unsigned)(BH * N));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = outk::ALLOC;
        if (cudaLaunchKernelEx(&cfg, falcon_out_kernel, p) != cudaSuccess) return 4;
    }
    return 0;
}

int split_consume_timeout_flag(int* flag) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_split_timeout_flag, sizeof(int)) != cudaSuccess) return 1;
    if (v && cudaMemcpyToSymbol(g_split_timeout_flag, &zero, sizeof(int)) != cudaSuccess) return 1;
    *flag = v;
    return 0;
}

}  // namespace falcon
