// Chunk-parallel forward for Falcon-2 and Falcon-2A (bf16 I/O, dk = dv = 64, chunk 64): one
// persistent CTA per (batch, head) sequence with the state on chip, so the only HBM traffic is the
// inputs, the outputs and the final state.
//
// Falcon-2 gives every value column c its own step eta_ic = beta_ic / (||x_i||^2 + lambda_i + eps)
// and decay gamma_ic; the columns of the state never mix ("Fast Weight Attention for Continual
// Learning", paperlayer summary: §1 "Falcon-2", §F "Falcon-2 Parallel Implementation", §F.2
// "Chunk-Parallel Algorithm"). Over a chunk of C = 64 tokens (rows i, j, l), with X the shifted keys,
// Q the queries, y_c the column's targets, G = X X^T (shared by every column), P_ic = prod_{m <= i}
// gamma_mc (P_{-1} = 1), d_ic = P_{i-1,c} and u_ic = eta_ic / P_ic, the column's recurrence
//   s <- gamma_i s + eta_i x_i (y_i - x_i . s),   o_i = q_i . s
// unrolls, with s the column at the chunk start, to
//   v_j = u_j (y_j - d_j a_j),   a_j = (X s)_j + sum_{l<j} G_jl v_l      (one merged residual solve)
//   s'  = P_63 (s + X^T v),   o_i = P_i ((Q s)_i + sum_{l<=i} (q_i . x_l) v_l).
// Per chunk the state-dependent work is the products [Q; X] s and [X^T; masked Q X^T] v for all 64
// columns at once, and the solve, blocked by 32 rows: each diagonal 32 x 32 triangle by forward
// substitution on the CUDA cores, and the first block's contribution G[32:64, 0:32] v_0:32 to the
// later rows' a on tcgen05, accumulated in TMEM onto X s. TMEM lane c holds column c: the products
// are issued with M = 128 and lanes 64-127 carry nothing. Falcon-2A writes the target itself:
// v = u (.) y, no solve.
//
// P_63 >= e^{-30} keeps every u finite; a column whose chunk decays further (the slow case) runs its
// 64 steps of the recurrence directly instead (no factored exponentials) and writes its outputs in
// place of Q s, with its v set to 0 so that the shared products leave it unchanged.
//
// Roles (192 threads):
//   warps 0-1   the state pass, one value column per lane: [Q S | X S] (tcgen05, the state as bf16
//               hi + lo), the blocked solve, V (bf16 hi + lo) into TMEM, [X^T V | Q S + masked(Q X^T)
//               V] (tcgen05), the state update (fp32 registers), and the next chunk's [Q S | X S]
//               at once; warp 0 also loads Y, Q, X (bf16) and beta (fp32) by TMA into a 3-stage ring,
//               lambda by cp.async, with an L2 prefetch
//   warps 2-5   the key side, one chunk ahead: [Q; X] X^T (tcgen05, bf16), the masked scores and G as
//               bf16 hi + lo (B operands), G's diagonal blocks in fp32, the per (token, column)
//               scalars P and u (u over beta in place); and, one chunk behind, the outputs
//               o_i = P_i (...)_i from TMEM to bf16 and a TMA store (warps 4-5, which share the
//               columns' lane quadrants)
// TMEM (512 columns): [0, 64) the state and [64, 128) V as bf16 hi + lo (A operands, 32 columns
// each); [128, 192) X^T V; two product regions [192, 320) and [384, 512), chunk parity, each Q S (then
// + masked(Q X^T) V) and X S (then a); [320, 384) the key side's [Q; X] X^T. The state itself stays in
// fp32 registers.
//
// Precision: products of the exact bf16 inputs are exact with fp32 sums; the state, V, G and the
// masked scores enter the tensor cores as bf16 hi + lo pairs (16 significant bits); every sum and
// the diagonal substitutions are fp32.
//
// Every wait is bounded: on timeout the kernel raises a device flag, both roles leave their loops,
// and the CTA drains what it issued before it frees its TMEM; falcon_device_status() reports it.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "falcon_internal.h"
#include "sm103_f32x2.cuh"
#include "sm103_ptx.cuh"

namespace falcon {

__device__ int g_colw_timeout_flag = 0;

namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;
constexpr int kTile = 8192;  // 64 x 64 bf16
constexpr int kStages = 3;
// a stage's tiles: Y, Q, X (Q directly before X, so that [Q; X] is one 128-row operand)
constexpr int kY = 0, kQ = kTile, kX = 2 * kTile, kTiles = 3 * kTile;
constexpr long long kTimeoutCycles = 4000000000LL;  // ~2 s
constexpr float kFastP = 9.3576230e-14f;            // e^{-30}
constexpr int kThreads = 192;

// The strictly lower part of G's two diagonal 32 x 32 blocks for the substitutions, packed: row t of
// a block holds G_{t t'} for t' from (t + 1) rounded down to a multiple of 4 up to 31 (16-byte groups).
__host__ __device__ constexpr int d_first(int t) { return (t + 1) & ~3; }
__host__ __device__ constexpr int d_row(int t) {
    return 124 * (t >> 2) - 8 * (t >> 2) * ((t >> 2) - 1) + (t & 3) * (32 - 4 * (t >> 2));
}
constexpr int kDBlock = d_row(32);  // 544 floats

struct ColwParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_out, tm_beta;
    const float* lam;
    const float* S0;
    const bf16* k;
    const bf16* tail;
    bf16* tail_out;
    float* S_final;
    long long T, pos;
    int N;
    float eps, eps_gamma;
};

namespace lay {
constexpr int TILES = 0;                  // kStages x (Y, Q, X)
constexpr int PB = kStages * kTiles;      // two chunks' key-side products
// in a key-side buffer: the masked scores Q X^T as bf16 hi and lo (K-major tiles; the hi tile later
// stages the chunk's output tile), G's off-diagonal block G[32:64, 0:32] as bf16 hi and lo (K-major,
// 32 rows), P [i][c], G's diagonal blocks, and per column the fast flag and P_63, per token
// 1 / (||x||^2 + lambda + eps)
constexpr int SCH = 0, SCL = kTile, GH = 2 * kTile, GL = GH + 4096, PP = GL + 4096, GD = PP + 16384,
              MISC = GD + 2 * kDBlock * 4;
constexpr int PB_BYTES = (MISC + 768 + 1023) / 1024 * 1024;
constexpr int BETA = PB + 2 * PB_BYTES;   // kStages x beta [i][c] fp32 (u after the key side)
constexpr int LAM = BETA + kStages * 16384;
constexpr int BAR = LAM + kStages * 256;
constexpr int BYTES = BAR + 256;
constexpr int ALLOC = BYTES + 1024;
static_assert(PB % 1024 == 0 && PB_BYTES % 1024 == 0 && GD % 16 == 0 && BETA % 1024 == 0, "layout");
static_assert(ALLOC <= 232448, "shared memory");
// mbarriers
constexpr int FULL = 0, PM = 3, PREADY = 4, OUTRDY = 6, RFREE = 8, M1 = 10, M2 = 11, M3 = 12, DRAIN = 13,
              NBAR = 15;
constexpr int ABORT = NBAR * 8, TSLOT = ABORT + 4;
static_assert(TSLOT + 4 <= 256, "barrier area");
}  // namespace lay

// TMEM columns
constexpr uint32_t kSV = 0, kVV = 64, kXV = 128, kPD = 320;
__device__ __forceinline__ uint32_t region(int n) { return (n & 1) ? 384u : 192u; }  // Q S at +0, X S at +64

struct Ctx {
    uint8_t* sm;
    uint32_t base;
    uint32_t tmem;
    volatile int* abort;
    long long bh;
    __device__ uint32_t bar(int i) const { return base + lay::BAR + 8 * i; }
    __device__ uint32_t tiles(int n) const { return base + lay::TILES + (n % kStages) * kTiles; }
    __device__ uint8_t* tiles_p(int n) const { return sm + lay::TILES + (n % kStages) * kTiles; }
    __device__ float* beta(int n) const { return reinterpret_cast<float*>(sm + lay::BETA + (n % kStages) * 16384); }
    __device__ float* lam(int n) const { return reinterpret_cast<float*>(sm + lay::LAM + (n % kStages) * 256); }
    __device__ uint8_t* pb(int n) const { return sm + lay::PB + (n & 1) * lay::PB_BYTES; }
    __device__ uint32_t pba(int n) const { return base + lay::PB + (n & 1) * lay::PB_BYTES; }
};

// Bounded wait by one thread; on timeout or when the other role has given up, false.
__device__ bool fwait(const Ctx& c, uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    int spins = 0;
    while (!mbar_try(bar, parity)) {
        if (*c.abort) return false;
        if (++spins > 64) __nanosleep(32);
        if (clock64() - t0 > kTimeoutCycles) {
            *c.abort = 1;
            atomicExch(&g_colw_timeout_flag, 1);
            return false;
        }
    }
    return true;
}

// v[0..63] = 64 consecutive TMEM columns of this thread's lane (one wait).
__device__ __forceinline__ void tld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r0[16], r1[16], r2[16], r3[16];
    tmem_ld16(taddr, r0);
    tmem_ld16(taddr + 16, r1);
    tmem_ld16(taddr + 32, r2);
    tmem_ld16(taddr + 48, r3);
    tmem_wait_ld();
    regs_ready(r0);
    regs_ready(r1);
    regs_ready(r2);
    regs_ready(r3);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        v[e] = __uint_as_float(r0[e]);
        v[16 + e] = __uint_as_float(r1[e]);
        v[32 + e] = __uint_as_float(r2[e]);
        v[48 + e] = __uint_as_float(r3[e]);
    }
}
// 64 fp32 values to 64 consecutive TMEM columns (no wait).
__device__ __forceinline__ void tst64(uint32_t taddr, const float (&x)[64]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(x[16 * q + e]);
        tmem_st16(taddr + 16 * q, r);
    }
}
// x[0..63] as a K = 64 bf16 A operand in TMEM: hi parts in columns [0, 32), lo parts in [32, 64),
// element k in column k / 2 (even k in the low half). No wait.
__device__ __forceinline__ void tst_hilo(uint32_t taddr, const float (&x)[64]) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t h[16], l[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) split2(x[32 * q + 2 * e], x[32 * q + 2 * e + 1], h[e], l[e]);
        tmem_st16(taddr + 16 * q, h);
        tmem_st16(taddr + 32 + 16 * q, l);
    }
}

__device__ __forceinline__ float ld_bf16(const uint8_t* p) { return __bfloat162float(*reinterpret_cast<const bf16*>(p)); }

// ---------------------------------------------------------------- loads
// One warp: TMA of chunk n's Y, Q, X (the box at row t0 - 1: zero above the first token) and beta into
// its ring stage, lambda by cp.async, and an L2 prefetch of the chunk that will next use the stage.
__device__ void issue_load(const ColwParams& p, const Ctx& c, int n, int lane) {
    const int s = n % kStages;
    const uint32_t tiles = c.tiles(n), bar = c.bar(lay::FULL + s);
    const int t0 = n * kC;
    if (lane == 0) {
        mbar_expect_tx(bar, 3 * kTile + 16384);
        tma_load_3d(tiles + kY, &p.tm_v, 0, t0, (int)c.bh, bar);
        tma_load_3d(tiles + kQ, &p.tm_q, 0, t0, (int)c.bh, bar);
        tma_load_3d(tiles + kX, &p.tm_k, 0, t0 - 1, (int)c.bh, bar);  // row i = k_{t0+i-1}
        tma_load_3d(smem_u32(c.beta(n)), &p.tm_beta, 0, t0, (int)c.bh, bar);
        const int np = n + kStages;
        if (np < p.N) {
            tma_prefetch_3d(&p.tm_v, 0, np * kC, (int)c.bh);
            tma_prefetch_3d(&p.tm_q, 0, np * kC, (int)c.bh);
            tma_prefetch_3d(&p.tm_k, 0, np * kC - 1, (int)c.bh);
            tma_prefetch_3d(&p.tm_beta, 0, np * kC, (int)c.bh);
        }
    }
    const long long row0 = c.bh * p.T;
    const uint32_t lam = smem_u32(c.lam(n));
#pragma unroll
    for (int r2 = 0; r2 < 2; ++r2) {
        const int r = lane + 32 * r2;
        const bool in = t0 + r < p.T;
        cp_async4(lam + 4 * r, p.lam + row0 + (in ? t0 + r : 0), in ? 4u : 0u);
    }
    cp_async_arrive(bar);
}

// ---------------------------------------------------------------- key side
// Chunk m's operators and scalars into buffer m & 1. False when a wait gave up.
__device__ bool prepare(const ColwParams& p, const Ctx& c, int pt, int m) {
    const int qd = ((pt >> 5) + 2) & 3, r = 32 * qd + (pt & 31);  // this warp's lane quadrant, this lane's row
    const uint32_t tiles = c.tiles(m);
    uint8_t* tp = c.tiles_p(m);
    uint8_t* pb = c.pb(m);
    const long long t0 = (long long)m * kC;
    const int nv = (int)min((long long)kC, p.T - t0);
    const float cap = 1.f - p.eps_gamma;
    const float* lam = c.lam(m);
    float* ub = c.beta(m);
    float* Pp = reinterpret_cast<float*>(pb + lay::PP);
    float* misc = reinterpret_cast<float*>(pb + lay::MISC);

    bool bad = false;
    if (pt == 0) {
        bad = !fwait(c, c.bar(lay::FULL + m % kStages), (uint32_t)(m / kStages) & 1u);
        bulk_wait_read<0>();  // the output store of chunk m - 2 has read this buffer's score tile
    }
    if (named_bar_or(2, 128, bad)) return false;
    if (m == 0 && p.pos > 0 && pt < 8) {  // a continuation's first shifted key is k_pos, from the tail
        const uint4 v = reinterpret_cast<const uint4*>(p.tail + c.bh * 64)[pt];
        *reinterpret_cast<uint4*>(tp + kX + sw128(0, 8 * pt)) = v;
        fence_async_smem();
    }
    named_bar(2, 128);
    if (pt == 0) {  // [Q; X] X^T: Q X^T in lanes 0-63, G = X X^T in lanes 64-127
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(c.tmem + kPD, desc_k(tiles + kQ + 32 * ks), desc_k(tiles + kX + 32 * ks), id, ks > 0);
        mma_commit(c.bar(lay::PM));
        bad = !fwait(c, c.bar(lay::PM), (uint32_t)m & 1u);
    }
    if (named_bar_or(2, 128, bad)) return false;
    tc_fence_after();
    {
        float v[64];
        tld64(c.tmem + kPD + ((uint32_t)(32 * qd) << 16), v);
        if (r < 64) {  // row i of the scores, masked to l <= i, as bf16 hi + lo
            const int i = r;
#pragma unroll
            for (int e = 0; e < 64; ++e) v[e] = e <= i ? v[e] : 0.f;
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) st8_hilo(pb + lay::SCH, pb + lay::SCL, sw128(i, 8 * q8), v + 8 * q8);
        } else {  // row j of G: the off-diagonal block's row (bf16 hi + lo), its diagonal block's part
                  // (fp32), and 1 / (||x_j||^2 + lambda_j + eps)
            const int j = r - 64, t = j & 31, f = d_first(t);
            float* gd = reinterpret_cast<float*>(pb + lay::GD) + (j >> 5) * kDBlock + d_row(t) - f;
            float gjj = 0.f;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                if ((j >> 5) == b) {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float* x = v + 32 * b + 4 * q4;
                        if (4 * q4 >= f) *reinterpret_cast<float4*>(gd + 4 * q4) = make_float4(x[0], x[1], x[2], x[3]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) gjj = 4 * q4 + e == t ? x[e] : gjj;
                    }
                }
            }
            if (j >= 32) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) st8_hilo(pb + lay::GH, pb + lay::GL, sw128(j - 32, 8 * q8), v + 8 * q8);
            }
            const float den = gjj + lam[j] + p.eps;  // 0 where the step is 0 (the first step, past the end)
            misc[128 + j] = (j < nv && p.pos + t0 + j >= 1 && den != 0.f) ? 1.f / den : 0.f;
        }
    }
    tc_fence_before();
    fence_async_smem();
    named_bar(2, 128);
    {  // thread (column cc, half h = lane parity) walks rows 32h .. 32h + 31; the two halves of a
       // column are neighbouring lanes
        const int cc = pt >> 1, h = pt & 1;
        const float* rd = misc + 128 + 32 * h;
        const float* lm = lam + 32 * h;
        float* ubh = ub + 32 * h * 64 + cc;
        float* Ph = Pp + 32 * h * 64 + cc;
        float eta[32], P[32];
        float prod = 1.f;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            eta[ii] = ubh[ii * 64] * rd[ii];
            prod *= 1.f - fminf(eta[ii] * lm[ii], cap);
            P[ii] = prod;
        }
        const float other = __shfl_xor_sync(0xffffffffu, prod, 1);
        const float p31 = h ? other : prod, pc = p31 * (h ? prod : other);  // P_31, P_63
        const bool fast = pc >= kFastP;
        if (fast) {
            const float sc = h ? p31 : 1.f;
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                const float Pi = P[ii] * sc;
                Ph[ii * 64] = Pi;
                ubh[ii * 64] = __fdividef(eta[ii], Pi);
            }
        } else {  // the direct recurrence reads gamma and eta
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                Ph[ii * 64] = 1.f - fminf(eta[ii] * lm[ii], cap);
                ubh[ii * 64] = eta[ii];
            }
        }
        if (h == 0) {
            misc[cc] = fast ? 1.f : 0.f;
            misc[64 + cc] = pc;
        }
    }
    named_bar(2, 128);
    if (pt == 0) mbar_arrive(c.bar(lay::PREADY + (m & 1)));
    return true;
}

// Chunk m's outputs from its product region, scaled by P_i (a slow column's are final already), to
// bf16 in the buffer's score tile (the products that read it have completed) and a TMA store; then
// the region is free for chunk m + 2. False when a wait gave up.
__device__ bool outputs(const ColwParams& p, const Ctx& c, int pt, int m) {
    const int qd = ((pt >> 5) + 2) & 3, b = m & 1;
    const int col = 32 * qd + (pt & 31);  // lane quadrants 0 and 1 hold the columns
    uint8_t* pb = c.pb(m);
    const float* Pp = reinterpret_cast<const float*>(pb + lay::PP);
    const float* misc = reinterpret_cast<const float*>(pb + lay::MISC);
    uint8_t* ob = pb + lay::SCH;
    bool bad = false;
    if (pt == 0) bad = !fwait(c, c.bar(lay::OUTRDY + b), (uint32_t)(m >> 1) & 1u);
    if (named_bar_or(2, 128, bad)) return false;
    tc_fence_after();
    if (qd < 2) {
        float d[64];
        tld64(c.tmem + region(m) + ((uint32_t)(32 * qd) << 16), d);
        const bool fast = misc[col] != 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 16 loads ahead of 16 stores
            float sc[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) sc[e] = fast ? Pp[(16 * q + e) * 64 + col] : 1.f;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                *reinterpret_cast<bf16*>(ob + sw128(16 * q + e, col)) = __float2bfloat16_rn(sc[e] * d[16 * q + e]);
        }
    }
    tc_fence_before();
    fence_async_smem();
    named_bar(2, 128);
    if (pt == 0) {
        mbar_arrive(c.bar(lay::RFREE + b));
        tma_store_3d(&p.tm_out, c.pba(m) + lay::SCH, 0, m * kC, (int)c.bh);
    }
    return true;
}

__device__ void key_side(const ColwParams& p, const Ctx& c, int pt) {
    for (int m = 0; m <= p.N; ++m) {
        if (m < p.N && !prepare(p, c, pt, m)) break;
        if (m >= 1 && !outputs(p, c, pt, m - 1)) break;
    }
    if (pt == 0) {  // the stores have read shared memory, and no MMA this thread issued is still running
        bulk_wait_all();
        mma_commit(c.bar(lay::DRAIN));
        mbar_wait_bounded(c.bar(lay::DRAIN), 0, kTimeoutCycles);
    }
}

// [Q S | X S] for chunk n (Falcon-2A: Q S only) into its region, committed to M1. One thread.
template <bool f2>
__device__ __forceinline__ void issue_mma1(const Ctx& c, int n) {
    const uint32_t tiles = c.tiles(n);
    tc_fence_after();
    constexpr uint32_t id = idesc_bf16(128, f2 ? 128 : 64, false, false);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        mma_bf16_ta(c.tmem + region(n), c.tmem + kSV + 8 * (ks & 3) + 32 * (ks >> 2), desc_k(tiles + kQ + 32 * (ks & 3)),
                    id, ks > 0);
    mma_commit(c.bar(lay::M1));
}

// ---------------------------------------------------------------- state pass
template <bool f2>
__device__ void state_pass(const ColwParams& p, const Ctx& c, int ct) {
    const int w = ct >> 5, lane = ct & 31;
    const int col = ct;
    const uint32_t tl = c.tmem + ((uint32_t)(32 * w) << 16);  // this warp's lane quadrant
    int issued = 0;
    if (w == 0)
        for (; issued < kStages && issued < p.N; ++issued) issue_load(p, c, issued, lane);
    float S[64];  // column col of the state (fp32)
    if (p.S0) {
        const float* src = p.S0 + c.bh * 4096 + col;
#pragma unroll
        for (int k = 0; k < 64; ++k) S[k] = src[64 * k];
    } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) S[k] = 0.f;
    }
    tst_hilo(tl + kSV, S);
    tmem_wait_st();
    tc_fence_before();
    named_bar(1, 64);
    bool ok = true, pending = false;  // pending: a wait at the end of the previous chunk gave up
    if (ct == 0 && p.N > 0) {  // the first chunk's [Q S | X S]; each later one at the end of the chunk before
        pending = !fwait(c, c.bar(lay::PREADY), 0u);
        if (!pending) issue_mma1<f2>(c, 0);
    }
    for (int n = 0; n < p.N; ++n) {
        const int b = n & 1;
        const uint32_t tiles = c.tiles(n);
        const uint8_t* tp = c.tiles_p(n);
        const uint8_t* pb = c.pb(n);
        const uint32_t pba = c.pba(n);
        const float* misc = reinterpret_cast<const float*>(pb + lay::MISC);
        const float* ub = c.beta(n);                                       // u (eta in the slow case), [i][c]
        const float* Pp = reinterpret_cast<const float*>(pb + lay::PP);  // P (gamma in the slow case)
        const uint32_t R = region(n);

        // ---- [Q S | X S] landed
        bool bad = pending;
        if (ct == 0 && !bad) bad = !fwait(c, c.bar(lay::M1), (uint32_t)n & 1u);
        if (named_bar_or(1, 64, bad)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const bool fast = misc[col] != 0.f;
        const float gC = misc[64 + col];
        if (f2) {
            // ---- v_j = u_j (y_j - d_j a_j) by 32-row blocks: block b's rows take their a from TMEM
            // (X s, plus G[32:64, 0:32] v_0:32 accumulated there for the second block), run the
            // triangle's substitution and write v (bf16 hi + lo) into the A operand
            const float* Gd = reinterpret_cast<const float*>(pb + lay::GD);
#pragma unroll 1
            for (int bk = 0; bk < 2; ++bk) {
                float a[32];
                {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tl + R + 64 + 32 * bk, r0);
                    tmem_ld16(tl + R + 80 + 32 * bk, r1);
                    tmem_wait_ld();
                    regs_ready(r0);
                    regs_ready(r1);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        a[e] = __uint_as_float(r0[e]);
                        a[16 + e] = __uint_as_float(r1[e]);
                    }
                }
                const float* gd = Gd + bk * kDBlock;
                const int j0 = 32 * bk;
                const float* ubj = ub + j0 * 64 + col;
                const float* Pj = Pp + (j0 - 1) * 64 + col;  // P_{j-1}: row j0 - 1 is read only when j0 > 0
                const uint8_t* yj = tp + kY + (j0 >> 3) * 1024;
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float y = ld_bf16(yj + sw128(t, col));
                    const float d = (j0 + t == 0) ? 1.f : Pj[t * 64];
                    const float vj = ubj[t * 64] * fmaf(-d, a[t], y);
                    a[t] = vj;
#pragma unroll
                    for (int t0 = d_first(t); t0 < 32; t0 += 4) {
                        const float4 g4 = *reinterpret_cast<const float4*>(gd + d_row(t) + t0 - d_first(t));
                        // the later rows in pairs (packed fp32 FMAs; every condition is known at compile time)
                        if (t0 > t) fma2(a[t0], a[t0 + 1], g4.x, g4.y, vj);
                        else if (t0 + 1 > t) a[t0 + 1] = fmaf(g4.y, vj, a[t0 + 1]);
                        if (t0 + 2 > t) fma2(a[t0 + 2], a[t0 + 3], g4.z, g4.w, vj);
                        else a[t0 + 3] = fmaf(g4.w, vj, a[t0 + 3]);
                    }
                }
                {
                    uint32_t h[16], l[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        split2(fast ? a[2 * e] : 0.f, fast ? a[2 * e + 1] : 0.f, h[e], l[e]);
                    tmem_st16(tl + kVV + 16 * bk, h);
                    tmem_st16(tl + kVV + 32 + 16 * bk, l);
                }
                if (bk == 0) {  // a[32:64] += G[32:64, 0:32] v_0:32: V_hi G_hi, V_lo G_hi, V_hi G_lo
                    tmem_wait_st();
                    tc_fence_before();
                    named_bar(1, 64);
                    if (ct == 0) {
                        tc_fence_after();
                        constexpr uint32_t id = idesc_bf16(128, 32, false, false);
                        const uint32_t d = c.tmem + R + 96;
#pragma unroll
                        for (int ks = 0; ks < 6; ++ks) {
                            const int kk = ks & 1, part = ks >> 1;
                            mma_bf16_ta(d, c.tmem + kVV + 8 * kk + (part == 1 ? 32 : 0),
                                        desc_k(pba + (part == 2 ? lay::GL : lay::GH) + 32 * kk), id, 1);
                        }
                        mma_commit(c.bar(lay::M3));
                        bad = !fwait(c, c.bar(lay::M3), (uint32_t)n & 1u);
                    }
                    bad = named_bar_or(1, 64, bad);  // every thread takes the same decision
                    if (bad) break;
                    tc_fence_after();
                }
            }
            if (bad) {
                ok = false;
                break;
            }
        } else {  // v = u (.) y
            float a[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) a[j] = fast ? ub[j * 64 + col] * ld_bf16(tp + kY + sw128(j, col)) : 0.f;
            tst_hilo(tl + kVV, a);
        }
        if (__any_sync(0xffffffffu, !fast)) {  // a slow column's 64 steps one by one, its outputs over Q s
            float o[64];
            tld64(tl + R, o);
            if (!fast) {
#pragma unroll 1
                for (int i = 0; i < 64; ++i) {
                    const float eta = ub[i * 64 + col], gam = Pp[i * 64 + col];
                    const uint8_t* xr = tp + kX;
                    float r = ld_bf16(tp + kY + sw128(i, col));
                    if (f2) {  // r = y_i - x_i . s
                        float dot[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int q8 = 0; q8 < 8; ++q8) {
                            float x[8];
                            unpack8(*reinterpret_cast<const uint4*>(xr + sw128(i, 8 * q8)), x);
#pragma unroll
                            for (int e = 0; e < 8; ++e) dot[e & 3] = fmaf(x[e], S[8 * q8 + e], dot[e & 3]);
                        }
                        r -= (dot[0] + dot[1]) + (dot[2] + dot[3]);
                    }
                    const float wv = eta * r;  // s <- gamma s + (eta r) x_i, then o_i = q_i . s
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) {
                        float x[8], qv[8];
                        unpack8(*reinterpret_cast<const uint4*>(xr + sw128(i, 8 * q8)), x);
                        unpack8(*reinterpret_cast<const uint4*>(tp + kQ + sw128(i, 8 * q8)), qv);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            S[8 * q8 + e] = fmaf(wv, x[e], gam * S[8 * q8 + e]);
                            acc[e & 3] = fmaf(qv[e], S[8 * q8 + e], acc[e & 3]);
                        }
                    }
                    const float oi = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
                    for (int e = 0; e < 64; ++e) o[e] = e == i ? oi : o[e];
                }
            }
            tst64(tl + R, o);
        }
        tmem_wait_st();
        tc_fence_before();
        named_bar(1, 64);

        // ---- [X^T V | Q S + masked(Q X^T) V]
        if (ct == 0) {
            tc_fence_after();
            constexpr uint32_t idx = idesc_bf16(128, 64, false, true), idk = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // X^T V: B = X read MN-major, 16 rows (2048 bytes) per K step
                mma_bf16_ta(c.tmem + kXV, c.tmem + kVV + 8 * (ks & 3) + 32 * (ks >> 2),
                            desc_mn(tiles + kX + 2048 * (ks & 3), kTile), idx, ks > 0);
            mma_commit(c.bar(lay::M2));  // the state update needs only X^T V
#pragma unroll
            for (int ks = 0; ks < 12; ++ks) {  // V_hi Sc_hi, V_lo Sc_hi, V_hi Sc_lo onto Q S
                const int kk = ks & 3, part = ks >> 2;
                mma_bf16_ta(c.tmem + R, c.tmem + kVV + 8 * kk + (part == 1 ? 32 : 0),
                            desc_k(pba + (part == 2 ? lay::SCL : lay::SCH) + 32 * kk), idk, 1);
            }
            mma_commit(c.bar(lay::OUTRDY + b));  // the key side forms the outputs from the region
            bad = !fwait(c, c.bar(lay::M2), (uint32_t)n & 1u);
        }
        if (named_bar_or(1, 64, bad)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // the stage is no longer read: refill it
        if (w == 0 && issued < p.N) issue_load(p, c, issued++, lane);

        // ---- s' = P_63 (s + X^T v) (a slow column's is final already) and as the next product's
        // operand; then that product, once the key side has the next chunk and region
        {
            float x[64];
            tld64(tl + kXV, x);
            if (fast) {
#pragma unroll
                for (int k = 0; k < 64; ++k) S[k] = gC * (S[k] + x[k]);
            }
        }
        tst_hilo(tl + kSV, S);
        tmem_wait_st();
        tc_fence_before();
        named_bar(1, 64);
        if (ct == 0 && n + 1 < p.N) {
            pending = !fwait(c, c.bar(lay::PREADY + (b ^ 1)), (uint32_t)((n + 1) >> 1) & 1u);
            if (!pending && n >= 1) pending = !fwait(c, c.bar(lay::RFREE + (b ^ 1)), (uint32_t)((n - 1) >> 1) & 1u);
            if (!pending) issue_mma1<f2>(c, n + 1);
        }
    }
    if (ok && p.S_final) {
        float* dst = p.S_final + c.bh * 4096 + col;
#pragma unroll
        for (int k = 0; k < 64; ++k) dst[64 * k] = S[k];
    }
    if (ok && p.tail_out && ct < 8) {  // window 1: the tail is the last key (the next call's x)
        uint4 v = make_uint4(0, 0, 0, 0);
        if (p.T > 0) v = reinterpret_cast<const uint4*>(p.k + (c.bh * p.T + p.T - 1) * 64)[ct];
        else if (p.pos > 0) v = reinterpret_cast<const uint4*>(p.tail + c.bh * 64)[ct];
        reinterpret_cast<uint4*>(p.tail_out + c.bh * 64)[ct] = v;
    }
    if (w == 0) {  // every load this warp issued has landed before the CTA exits (bounded)
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0)
            for (int n = max(0, issued - kStages); n < issued; ++n)
                mbar_wait_bounded(c.bar(lay::FULL + n % kStages), (uint32_t)(n / kStages) & 1u, kTimeoutCycles);
    }
    if (ct == 0) {
        mma_commit(c.bar(lay::DRAIN + 1));
        mbar_wait_bounded(c.bar(lay::DRAIN + 1), 0, kTimeoutCycles);
    }
}

template <bool f2>
__global__ void __launch_bounds__(kThreads, 1) falcon_colw_kernel(const __grid_constant__ ColwParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    Ctx c;
    c.sm = sm;
    c.base = base;
    c.abort = reinterpret_cast<volatile int*>(sm + lay::BAR + lay::ABORT);
    c.bh = blockIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(c.bar(lay::FULL + s), 1 + 32);  // expect-tx and 32 cp.async arrivals
        mbar_init(c.bar(lay::PM), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(c.bar(lay::PREADY + b), 1);
            mbar_init(c.bar(lay::OUTRDY + b), 1);
            mbar_init(c.bar(lay::RFREE + b), 1);
            mbar_init(c.bar(lay::DRAIN + b), 1);
        }
        mbar_init(c.bar(lay::M1), 1);
        mbar_init(c.bar(lay::M2), 1);
        mbar_init(c.bar(lay::M3), 1);
        *c.abort = 0;
        mbar_init_fence();
    }
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + lay::BAR + lay::TSLOT);
    if (warp == 2) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tslot;

    if (warp < 2) state_pass<f2>(p, c, tid);
    else key_side(p, c, tid - 64);

    tc_fence_before();
    __syncthreads();
    if (warp == 2) tmem_dealloc(c.tmem, 512);
}

// The kernels' dynamic shared-memory attribute, set once per device.
constexpr int kMaxDevices = 64;
bool prepare_device() {
    static bool ready[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (!ready[dev]) {
        int optin = 0;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            optin < lay::ALLOC ||
            cudaFuncSetAttribute(falcon_colw_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay::ALLOC) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_colw_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay::ALLOC) !=
                cudaSuccess)
            return false;
        ready[dev] = true;
    }
    return true;
}

}  // namespace

bool colw_supported(const Launch& a) {
    return (a.variant == kF2 || a.variant == kF2A) && a.bf16 && a.dk == 64 && a.dv == 64 && a.chunk == 64 &&
           a.W == 1 && a.T != 1 && a.T < (1LL << 31) - 64 && a.B * a.H < (1LL << 31);
}

int launch_colw(const Launch& a, cudaStream_t st) {
    if (!prepare_device()) return 4;
    const long long BH = a.B * a.H;
    ColwParams p = {};
    if (a.T > 0 && (!encode_bhtd(&p.tm_q, a.q, a.T, BH) || !encode_bhtd(&p.tm_k, a.k, a.T, BH) ||
                    !encode_bhtd(&p.tm_v, a.v, a.T, BH) || !encode_bhtd(&p.tm_out, a.out, a.T, BH) ||
                    !encode_bhtd_f32(&p.tm_beta, a.beta, a.T, BH)))
        return 4;
    p.lam = a.lam;
    p.S0 = a.S0;
    p.k = static_cast<const bf16*>(a.k);
    p.tail = static_cast<const bf16*>(a.tail);
    p.tail_out = static_cast<bf16*>(a.tail_out);
    p.S_final = a.S_final;
    p.T = a.T;
    p.pos = a.pos;
    p.N = (int)((a.T + kC - 1) / kC);
    p.eps = a.eps;
    p.eps_gamma = a.eps_gamma;
    if (a.variant == kF2) falcon_colw_kernel<true><<<(unsigned)BH, kThreads, lay::ALLOC, st>>>(p);
    else falcon_colw_kernel<false><<<(unsigned)BH, kThreads, lay::ALLOC, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int colw_consume_timeout_flag(int* flag) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_colw_timeout_flag, sizeof(int)) != cudaSuccess) return 1;
    if (v && cudaMemcpyToSymbol(g_colw_timeout_flag, &zero, sizeof(int)) != cudaSuccess) return 1;
    *flag = v;
    return 0;
}

}  // namespace falcon
