// Fused chunk-parallel forward for Falcon-1 and Falcon-1A (bf16 I/O, dk = dv = 64, chunk 64):
// one persistent CTA per (batch, head) sequence, every chunk's operators and the carried state kept
// on chip, so the only HBM traffic is the inputs, the outputs and the final state.
//
// Per chunk of C = 64 tokens (rows i, j), X the shifted keys (row i = k_{tau_i - 1}), Q the queries,
// Y the values, eta the step sizes, L / Lx the inclusive / exclusive log-decay prefixes reset to 0
// at the chunk start, d_i = e^{Lx_i}, u_j = eta_j e^{-L_j}, w_j = eta_j e^{L_C - L_j}, and
//   A_ij = eta_j e^{Lx_i - L_j} x_i.x_j (j < i),   P_ij = eta_j e^{L_i - L_j} q_i.x_j (j <= i),
//   T = (I + A)^{-1},   E = [P ; X^T diag(w)] T   (128 x 64),
// the Falcon-1 recurrence unrolled over the chunk ("Fast Weight Attention for Continual Learning",
// paperlayer summary: §E.1 WY form of the solve, §E.2 one merged residual solve and the three
// phases, §F.2 read after write, §G.1 chunk-local log prefixes) is, with S the state at the chunk
// start,
//   [PW ; K] = E diag(d) X,   [Bo ; U] = E Y,   Ao = diag(e^L) Q - PW,
//   O = Ao S + Bo,            S' = e^{L_C} S - K S + U,
// so the only product that waits for the carried state is [Ao ; -K] S, one 128 x 64 x 64 MMA whose
// top half is the chunk's reads and bottom half the next state's update. Falcon-1A writes the
// target itself: T = I, K = PW = 0.
//
// When the chunk's total log decay L_C is at least -30 the exponentials factor (e^{a - b} =
// e^a e^{-b}, both finite) and the scalings move off the per-element path: E = diag(s) E~ with
// E~ = [Q X^T masked ; X^T] diag(u) T, s_i = e^{L_i} (rows 0-63) and e^{L_C} (rows 64-127); diag(u)
// multiplies T's rows and diag(d) X's rows where those operands are written anyway, and s scales
// the finished products. Otherwise every factor is one exp of a non-positive argument and s = 1.
//
// Roles (384 threads, three warps per SM sub-partition):
//   warps 0-3, 4-7   two key-side groups; group g takes chunks g, g + 2, ...: [Q; X] X^T (tcgen05,
//                    bf16), the scalars, A (shared) and the masked scores (TMEM), T by blocked
//                    substitution, Y^T and X^T read column by column from the staged tiles into
//                    E~'s operands, E~ (tcgen05, tf32, A operand in TMEM), E~ [diag(d) X | Y]
//                    (tcgen05, tf32), then [Ao ; -K] back into TMEM
//   warps 8-11       the state pass: [Ao ; -K] S (tcgen05, tf32), O = Ao S + Bo to bf16 and a TMA
//                    store, S' in fp32 registers and as the next product's operand; its first warp
//                    also loads (TMA of Y, Q and X into a 3-stage ring, beta and lambda by cp.async,
//                    L2 prefetch): a chunk's stage is refilled once the state pass has received the
//                    chunk, since the key side is then done reading it
// TMEM (512 columns): group g owns columns [256g, 256g + 256) as C0 = [0, 64): [Q; X] X^T -> masked
// scores and X^T (E~'s A operand); C1 = [64, 128): E~ -> the state-pass product;
// C2 = [128, 256): [PW | Bo ; K | U] -> [Ao | Bo ; -K | U].
//
// Precision: products of the exact bf16 inputs are bf16 (exact, fp32 sums); E~ and everything after
// it are tf32 with operands rounded to nearest (exact inputs are exact in tf32); the state and every
// sum are fp32.
//
// Every wait is bounded: on timeout the kernel raises a device flag, every role leaves its loop,
// and the CTA drains what it issued before it frees its TMEM; falcon_device_status() reports it.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "falcon_internal.h"
#include "sm103_ptx.cuh"

namespace falcon {

__device__ int g_fused_timeout_flag = 0;

namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;
constexpr int kTile = 8192;            // 64 x 64 bf16
constexpr int kStages = 3;
constexpr int kStage = 25600;          // Y, Q, X (8 KB each), beta and lambda (256 B each); 1024-aligned
constexpr int kQ = kTile, kX = 2 * kTile, kBL = 3 * kTile;  // offsets in a stage
constexpr int kS = 68;                 // row stride (floats) of A / T in shared memory
constexpr long long kTimeoutCycles = 4000000000LL;  // ~2 s
constexpr float kFastL = 30.f;
constexpr int kThreads = 384;

struct FusedParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_out;
    const float* beta;
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

struct FScal {
    float d[64], eL[64], u[64], w[64], eta[64], L[64], Lx[64];
    float misc[8];  // [0] e^{L_C}, [1] 1 when the factored exponentials hold, [2..3] warp totals
};

namespace lay {
constexpr int RING = 0;
// two key-side groups, each: T^T (diag(u) folded in) as E~'s B operand; [(diag(d) X)^T ; Y^T] as the
// B operand of E~'s products, whose first 17 KB hold A / T (fp32) until T^T is written; scalars
constexpr int GRP = kStages * kStage;
constexpr int TOP = 0, B3 = 16384, AT = B3, SCAL = B3 + 32768;
constexpr int GRP_BYTES = SCAL + 3072;
constexpr int SOP = GRP + 2 * GRP_BYTES;  // S^T as the tf32 B operand of the state pass
constexpr int OUTS = SOP + 16384;         // two bf16 output staging tiles
constexpr int CGS = OUTS + 2 * kTile;     // per group: the finished chunk's row scales s (128 floats)
constexpr int BAR = CGS + 1024;
constexpr int BYTES = BAR + 256;
constexpr int ALLOC = BYTES + 1024;
static_assert(GRP % 1024 == 0 && GRP_BYTES % 1024 == 0 && SOP % 1024 == 0 && OUTS % 1024 == 0, "layout");
static_assert(64 * kS * 4 <= 32768 && sizeof(FScal) <= 3072, "group area");
// mbarriers
constexpr int FULL = 0, MMA = 3, CA = 5, CD = 7, CONS = 9, DRAIN = 11, NBAR = 14;
constexpr int ABORT = NBAR * 8, TSLOT = ABORT + 4, GCH = ABORT + 8;  // abort word, TMEM address, e^{L_C} per group
static_assert(GCH + 8 <= 256, "barrier area");
}  // namespace lay

// Offset of element (row r, k) in a K-major tf32 operand of R rows x 64 K: two 128-byte swizzle
// atoms along K, R * 128 bytes apart.
template <int R>
__device__ __forceinline__ uint32_t tf_off(int r, int k) {
    return (uint32_t)((k >> 5) * (R * 128) + (r >> 3) * 1024 + (r & 7) * 128 + ((((k & 31) >> 2) ^ (r & 7)) << 4) +
                      ((k & 3) << 2));
}

struct Ctx {
    uint8_t* sm;
    uint32_t base;
    uint32_t tmem;
    volatile int* abort;
    long long bh;
    __device__ uint32_t bar(int i) const { return base + lay::BAR + 8 * i; }
};

// Bounded wait by one thread; on timeout or when another role has given up, false.
__device__ bool fwait(const Ctx& c, uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    int spins = 0;
    while (!mbar_try(bar, parity)) {
        if (*c.abort) return false;
        if (++spins > 64) __nanosleep(32);
        if (clock64() - t0 > kTimeoutCycles) {
            *c.abort = 1;
            atomicExch(&g_fused_timeout_flag, 1);
            return false;
        }
    }
    return true;
}

// v[0..31] as bits to 32 consecutive TMEM columns (no wait).
__device__ __forceinline__ void tst32(uint32_t taddr, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(v[16 * q + e]);
        tmem_st16(taddr + 16 * q, r);
    }
}
// ---------------------------------------------------------------- T = (I + A)^{-1}, in place
// On entry M holds A (fp32, stride kS), strictly lower with zeros on and above the diagonal; on exit
// M holds T. 16 x 16 diagonal blocks by right-looking column substitution in fp32, then two levels
// of block merges T_ba = -(T_bb A_ba) T_aa as warp-level tf32 products with fp32 accumulation. `gt` is the thread's
// index in its 128-thread group, `bid` the group's named barrier.
// d += C x M[k0.., n0..], C an accumulator fragment used as the A operand (its columns 2t, 2t + 1
// stand in the k-slots t, t + 4, so the B rows are read in that order)
__device__ __forceinline__ void mma_tf_c(float (&d)[4], const float (&c)[4], const float* M, int k0, int n0, int g,
                                         int t) {
    const uint32_t b0 = tf32_rn(M[(k0 + 2 * t) * kS + n0 + g]), b1 = tf32_rn(M[(k0 + 2 * t + 1) * kS + n0 + g]);
    mma1688_tf32(d, tf32_rn(c[0]), tf32_rn(c[2]), tf32_rn(c[1]), tf32_rn(c[3]), b0, b1);
}

__device__ void invert_group(float* M, int gt, int bid) {
    const int warp = gt >> 5, lane = gt & 31, g = lane >> 2, t = lane & 3;
    float x[16];
    if (gt < 64) {  // column c of diagonal block b, right-looking: once x_r is final, update the later rows
        const int b = gt >> 4, c = gt & 15;
        const float* Ab = M + 16 * b * kS + 16 * b;
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r) {
            float col[15];
#pragma unroll
            for (int s2 = r + 1; s2 < 16; ++s2) col[s2 - r - 1] = Ab[s2 * kS + r];
#pragma unroll
            for (int s2 = r + 1; s2 < 16; ++s2) x[s2] = fmaf(-col[s2 - r - 1], x[r], x[s2]);
        }
    }
    named_bar(bid, 128);
    if (gt < 64) {
        const int b = gt >> 4, c = gt & 15;
#pragma unroll
        for (int r = 0; r < 16; ++r) M[(16 * b + r) * kS + 16 * b + c] = x[r];
    }
    named_bar(bid, 128);
    if (warp < 2) {  // T_{b+1,b} = -(T_{b+1,b+1} A_{b+1,b}) T_bb, b = 0 (warp 0) and b = 2 (warp 1)
        const int b = 2 * warp, R1 = 16 * (b + 1), C0 = 16 * b;
        float d1[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {  // T_{b+1,b+1} (rows R1.., k R1 + 8ks) x A (rows R1 + 8ks, cols C0 + 8nt)
            const uint32_t a0 = tf32_rn(M[(R1 + g) * kS + R1 + 8 * ks + t]);
            const uint32_t a1 = tf32_rn(M[(R1 + g + 8) * kS + R1 + 8 * ks + t]);
            const uint32_t a2 = tf32_rn(M[(R1 + g) * kS + R1 + 8 * ks + t + 4]);
            const uint32_t a3 = tf32_rn(M[(R1 + g + 8) * kS + R1 + 8 * ks + t + 4]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const uint32_t b0 = tf32_rn(M[(R1 + 8 * ks + t) * kS + C0 + 8 * nt + g]);
                const uint32_t b1 = tf32_rn(M[(R1 + 8 * ks + t + 4) * kS + C0 + 8 * nt + g]);
                mma1688_tf32(d1[nt], a0, a1, a2, a3, b0, b1);
            }
        }
        float d2[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_tf_c(d2[nt], d1[ks], M, C0 + 8 * ks, C0 + 8 * nt, g, t);
        __syncwarp();
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            *reinterpret_cast<float2*>(M + (R1 + g) * kS + C0 + 8 * nt + 2 * t) = make_float2(-d2[nt][0], -d2[nt][1]);
            *reinterpret_cast<float2*>(M + (R1 + g + 8) * kS + C0 + 8 * nt + 2 * t) =
                make_float2(-d2[nt][2], -d2[nt][3]);
        }
    }
    named_bar(bid, 128);
    {  // T[32:64, 0:32] = -(T[32:64, 32:64] A[32:64, 0:32]) T[0:32, 0:32], one 16 x 16 tile per warp
        const int RB = 32 + 16 * (warp >> 1), CB = 16 * (warp & 1);
        float d1[4][4] = {};
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {
            const uint32_t a0 = tf32_rn(M[(RB + g) * kS + 32 + 8 * ks + t]);
            const uint32_t a1 = tf32_rn(M[(RB + g + 8) * kS + 32 + 8 * ks + t]);
            const uint32_t a2 = tf32_rn(M[(RB + g) * kS + 32 + 8 * ks + t + 4]);
            const uint32_t a3 = tf32_rn(M[(RB + g + 8) * kS + 32 + 8 * ks + t + 4]);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const uint32_t b0 = tf32_rn(M[(32 + 8 * ks + t) * kS + 8 * nt + g]);
                const uint32_t b1 = tf32_rn(M[(32 + 8 * ks + t + 4) * kS + 8 * nt + g]);
                mma1688_tf32(d1[nt], a0, a1, a2, a3, b0, b1);
            }
        }
        named_bar(bid, 128);  // every warp has read A[32:64, 0:32]
        float d2[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_tf_c(d2[nt], d1[ks], M, 8 * ks, CB + 8 * nt, g, t);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            *reinterpret_cast<float2*>(M + (RB + g) * kS + CB + 8 * nt + 2 * t) = make_float2(-d2[nt][0], -d2[nt][1]);
            *reinterpret_cast<float2*>(M + (RB + g + 8) * kS + CB + 8 * nt + 2 * t) =
                make_float2(-d2[nt][2], -d2[nt][3]);
        }
    }
    named_bar(bid, 128);
}

// ---------------------------------------------------------------- key-side group
template <bool f1>
__device__ void key_group(const FusedParams& p, const Ctx& c, int g, int gt) {
    const int warp_in = gt >> 5, lane = gt & 31;
    const int bid = 1 + g, sid = 3 + g;                         // named barriers: group (128), rows 0-63 (64)
    const uint32_t Bg = c.tmem + 256u * g;                      // this group's TMEM columns, lane 0
    const uint32_t tq = Bg + ((uint32_t)(32 * warp_in) << 16);  // ... at this warp's lane quadrant
    const uint32_t C0 = 0, C1 = 64, C2 = 128;
    uint8_t* grp = c.sm + lay::GRP + g * lay::GRP_BYTES;
    float* AT = reinterpret_cast<float*>(grp + lay::AT);
    FScal* sc = reinterpret_cast<FScal*>(grp + lay::SCAL);
    const uint32_t grp_a = c.base + lay::GRP + g * lay::GRP_BYTES;
    float* gch = reinterpret_cast<float*>(c.sm + lay::BAR + lay::GCH);
    float* cgs = reinterpret_cast<float*>(c.sm + lay::CGS) + 128 * g;
    uint32_t mph = 0;  // phases of this group's MMA barrier consumed so far
    // thread 0 issues, commits and waits; every thread learns the outcome at the group barrier
    auto wait_mma = [&]() -> bool {
        bool bad = false;
        if (gt == 0) bad = !fwait(c, c.bar(lay::MMA + g), mph & 1u);
        ++mph;
        return !named_bar_or(bid, 128, bad);
    };
    for (int j = 0;; ++j) {
        const int n = g + 2 * j;
        if (n >= p.N) break;
        const int s = n % kStages;
        const uint32_t stage = c.base + lay::RING + s * kStage;
        uint8_t* stg = c.sm + lay::RING + s * kStage;
        const long long t0 = (long long)n * kC;
        const int nv = (int)min((long long)kC, p.T - t0);

        // ---- inputs landed
        bool bad = false;
        if (gt == 0) bad = !fwait(c, c.bar(lay::FULL + s), (uint32_t)(n / kStages) & 1u) || *c.abort;
        if (named_bar_or(bid, 128, bad)) break;
        if (n == 0 && p.pos > 0 && gt < 8) {  // a continuation's first shifted key is k_pos, from the tail
            const uint4 v = reinterpret_cast<const uint4*>(p.tail + c.bh * 64)[gt];
            *reinterpret_cast<uint4*>(stg + kX + sw128(0, 8 * gt)) = v;
            fence_async_smem();
        }
        named_bar(bid, 128);
        if (gt == 0) {  // [Q; X] X^T: Q X^T in lanes 0-63, G = X X^T in lanes 64-127
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(Bg + C0, desc_k(stage + kQ + 32 * ks), desc_k(stage + kX + 32 * ks), id, ks > 0);
            mma_commit(c.bar(lay::MMA + g));
        }

        // ---- per-token scalars (threads 0-63), while the product runs
        if (gt < 64) {
            const int i = gt;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                float x[8];
                unpack8(*reinterpret_cast<const uint4*>(stg + kX + sw128(i, 8 * q8)), x);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(x[e], x[e], acc[e]);
            }
            const float nx = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            const float bt = reinterpret_cast<const float*>(stg + kBL)[i];
            const float lm = reinterpret_cast<const float*>(stg + kBL + 256)[i];
            float eta = 0.f, alpha = 0.f;
            if (i < nv && p.pos + t0 + i + 1 >= 2) {
                const float den = nx + lm + p.eps;
                eta = den == 0.f ? 0.f : bt / den;
                alpha = fminf(eta * lm, 1.f - p.eps_gamma);
            }
            const float l = log1pf(-alpha);
            float incl = l;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sc->misc[2 + warp_in] = incl;
            named_bar(sid, 64);
            const float LC = sc->misc[2] + sc->misc[3];
            const float Li = incl + (i >= 32 ? sc->misc[2] : 0.f);
            const float Lxi = Li - l;
            const float gC = __expf(LC), wi = eta * __expf(LC - Li);
            sc->eta[i] = eta;
            sc->L[i] = Li;
            sc->Lx[i] = Lxi;
            sc->d[i] = __expf(Lxi);
            sc->eL[i] = __expf(Li);
            sc->w[i] = wi;
            sc->u[i] = LC >= -kFastL ? wi * __frcp_rn(gC) : 0.f;  // eta e^{-L_i}; used only when L_C >= -kFastL
            if (i == 0) {
                sc->misc[0] = gC;
                sc->misc[1] = LC >= -kFastL ? 1.f : 0.f;
            }
        }
        if (!wait_mma()) break;  // also publishes the scalars
        tc_fence_after();
        const bool fast = sc->misc[1] != 0.f;

        // ---- rows 0-63: masked scores (factored: q_i.x_j; otherwise P_ij), written back to C0 as the
        // top of E~'s A operand (Falcon-1A: E~ itself, factored form times u_j);
        //      rows 64-127 (Falcon-1): A_ij in fp32 to shared memory for the inversion
        if (gt < 64) {
            const int i = gt;
            const float li = sc->L[i];
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tq + C0 + 32 * h, v);
                const float* eta = sc->eta + 32 * h;
                const float* L = sc->L + 32 * h;
                const float* u = sc->u + 32 * h;
                if (!fast) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= eta[e] * __expf(fminf(li - L[e], 0.f));
                } else if (!f1) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= u[e];
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(tf32_rn(32 * h + e <= i ? v[e] : 0.f));
                tst32(tq + C0 + 32 * h, v);
            }
        } else if (f1) {
            const int i = gt - 64;
            const float dx = sc->d[i], lx = sc->Lx[i];
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tq + C0 + 32 * h, v);
                const float* eta = sc->eta + 32 * h;
                const float* L = sc->L + 32 * h;
                const float* u = sc->u + 32 * h;
                if (fast) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 32 * h + e < i ? dx * u[e] * v[e] : 0.f;
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = 32 * h + e < i ? eta[e] * __expf(fminf(lx - L[e], 0.f)) * v[e] : 0.f;
                }
                float4* dst = reinterpret_cast<float4*>(AT + i * kS + 32 * h);
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) dst[k4] = make_float4(v[4 * k4], v[4 * k4 + 1], v[4 * k4 + 2], v[4 * k4 + 3]);
            }
        }
        tmem_wait_st();
        tc_fence_before();
        named_bar(bid, 128);

        if (f1) {
            // ---- T = (I + A)^{-1}; diag(u) T (factored) or T as E~'s K-major tf32 B operand
            invert_group(AT, gt, bid);
            const int cc = gt & 63, jh = gt >> 6;
            uint8_t* tb = grp + lay::TOP;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int j0 = 32 * jh + 4 * q;
                const float4 uu = fast ? *reinterpret_cast<const float4*>(sc->u + j0) : make_float4(1.f, 1.f, 1.f, 1.f);
                uint4 v;
                v.x = tf32_rn(AT[(j0 + 0) * kS + cc] * uu.x);
                v.y = tf32_rn(AT[(j0 + 1) * kS + cc] * uu.y);
                v.z = tf32_rn(AT[(j0 + 2) * kS + cc] * uu.z);
                v.w = tf32_rn(AT[(j0 + 3) * kS + cc] * uu.w);
                *reinterpret_cast<uint4*>(tb + tf_off<64>(cc, j0)) = v;
            }
            fence_async_smem();
        }

        // ---- the transposes, each thread its feature's column of the stage's Y or X tile (exact):
        // rows 0-63 (feature c): Y^T row c -> the B operand's rows 64 + c;
        // rows 64-127 (feature a): X^T row a -> diag(d) folded in, B rows a; and to C0 as the bottom
        // of E~'s A operand (factored: as is, Falcon-1A times u_j; otherwise times w_j)
        {
            uint8_t* b3 = grp + lay::B3;
            const int fc = gt & 63;  // the feature
            const uint8_t* colb = stg + (gt < 64 ? 0 : kX) + ((fc & 7) << 1);
            uint32_t xo[8];  // the feature's 16-byte chunk in a swizzled row, per row residue
#pragma unroll
            for (int k = 0; k < 8; ++k) xo[k] = (uint32_t)(((fc >> 3) ^ k) << 4);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {  // token row 32 h + e of the tile
                    const int jr = 32 * h + e;
                    v[e] = __bfloat162float(*reinterpret_cast<const bf16*>(colb + (jr >> 3) * 1024 + (jr & 7) * 128 + xo[jr & 7]));
                }
                if (gt < 64) {
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        *reinterpret_cast<uint4*>(b3 + tf_off<128>(64 + gt, 32 * h + 4 * k4)) =
                            make_uint4(__float_as_uint(v[4 * k4]), __float_as_uint(v[4 * k4 + 1]),
                                       __float_as_uint(v[4 * k4 + 2]), __float_as_uint(v[4 * k4 + 3]));
                } else {
                    const int a = gt - 64;
                    const float* d = sc->d + 32 * h;
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        *reinterpret_cast<uint4*>(b3 + tf_off<128>(a, 32 * h + 4 * k4)) =
                            make_uint4(tf32_rn(v[4 * k4] * d[4 * k4]), tf32_rn(v[4 * k4 + 1] * d[4 * k4 + 1]),
                                       tf32_rn(v[4 * k4 + 2] * d[4 * k4 + 2]), tf32_rn(v[4 * k4 + 3] * d[4 * k4 + 3]));
                    const float* w = (fast ? sc->u : sc->w) + 32 * h;
                    if (!fast || !f1) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(tf32_rn(v[e] * w[e]));
                    }
                    tst32(tq + C0 + 32 * h, v);
                }
            }
        }
        tmem_wait_st();
        fence_async_smem();
        tc_fence_before();
        // C1 and C2 free (the state pass has read chunk n - 2's)
        if (gt == 0 && j > 0) bad = !fwait(c, c.bar(lay::CONS + g), (uint32_t)(j - 1) & 1u);
        if (named_bar_or(bid, 128, bad)) break;

        uint32_t ea = C0;  // TMEM columns of E~ (the A operand of the products with X and Y)
        if (f1) {
            if (gt == 0) {  // E~ = [scores ; X^T] (diag(u) T): into C1
                tc_fence_after();
                constexpr uint32_t id = idesc_tf32(128, 64);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_tf32_ta(Bg + C1, Bg + C0 + 8 * ks, desc_k(grp_a + lay::TOP + (ks >> 2) * 8192 + 32 * (ks & 3)),
                                id, ks > 0);
                mma_commit(c.bar(lay::MMA + g));
            }
            if (!wait_mma()) break;
            tc_fence_after();
            ea = C1;
        }
        if (gt == 0) {  // E~ [diag(d) X | Y] (Falcon-1A: E~ Y): [PW | Bo ; K | U] / s into C2
            tc_fence_after();
            if (f1) {
                constexpr uint32_t id = idesc_tf32(128, 128);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_tf32_ta(Bg + C2, Bg + ea + 8 * ks,
                                desc_k(grp_a + lay::B3 + (ks >> 2) * 16384 + 32 * (ks & 3)), id, ks > 0);
            } else {
                constexpr uint32_t id = idesc_tf32(128, 64);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_tf32_ta(Bg + C2 + 64, Bg + ea + 8 * ks,
                                desc_k(grp_a + lay::B3 + 8192 + (ks >> 2) * 16384 + 32 * (ks & 3)), id, ks > 0);
            }
            mma_commit(c.bar(lay::MMA + g));
        }
        if (!wait_mma()) break;
        tc_fence_after();

        // ---- [Ao ; -K] (tf32) into C2's first 64 columns: the state pass's A operand
        const float sr = fast ? (gt < 64 ? sc->eL[gt] : sc->misc[0]) : 1.f;  // this row's scale s
        if (gt < 64) {
            const int i = gt;
            const float ei = sc->eL[i];
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
                if (f1) tmem_ld32(tq + C2 + 32 * h, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[8];
                    unpack8(*reinterpret_cast<const uint4*>(stg + kQ + sw128(i, 32 * h + 8 * q)), x);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        v[8 * q + e] = __uint_as_float(tf32_rn(f1 ? fmaf(ei, x[e], -sr * v[8 * q + e]) : ei * x[e]));
                }
                tst32(tq + C2 + 32 * h, v);
            }
        } else if (f1) {
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tq + C2 + 32 * h, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(tf32_rn(-sr * v[e]));
                tst32(tq + C2 + 32 * h, v);
            }
        }
        cgs[gt] = sr;
        if (gt == 0) gch[g] = sc->misc[0];  // the chunk's state decay e^{L_C}
        tmem_wait_st();
        tc_fence_before();
        named_bar(bid, 128);
        // the state pass may start chunk n; every read of its stage is done, so it may be refilled
        if (gt == 0) mbar_arrive(c.bar(lay::CA + g));
    }
    if (gt == 0) {  // nothing this thread issued is still running when the CTA frees its TMEM
        mma_commit(c.bar(lay::DRAIN + g));
        mbar_wait_bounded(c.bar(lay::DRAIN + g), 0, kTimeoutCycles);
    }
}

// ---------------------------------------------------------------- loads
// One warp: TMA of chunk n's Y, Q and X (the box at row t0 - 1: zero above the first token) into its
// ring stage, beta and lambda by cp.async, and an L2 prefetch of the chunk that will next use the stage.
__device__ void issue_load(const FusedParams& p, const Ctx& c, int n, int lane) {
    const int s = n % kStages;
    const uint32_t stage = c.base + lay::RING + s * kStage;
    const int t0 = n * kC;
    if (lane == 0) {
        mbar_expect_tx(c.bar(lay::FULL + s), 3 * kTile);
        tma_load_3d(stage, &p.tm_v, 0, t0, (int)c.bh, c.bar(lay::FULL + s));
        tma_load_3d(stage + kQ, &p.tm_q, 0, t0, (int)c.bh, c.bar(lay::FULL + s));
        tma_load_3d(stage + kX, &p.tm_k, 0, t0 - 1, (int)c.bh, c.bar(lay::FULL + s));  // row i = k_{t0+i-1}
        const int np = n + kStages;
        if (np < p.N) {
            tma_prefetch_3d(&p.tm_v, 0, np * kC, (int)c.bh);
            tma_prefetch_3d(&p.tm_q, 0, np * kC, (int)c.bh);
            tma_prefetch_3d(&p.tm_k, 0, np * kC - 1, (int)c.bh);
        }
    }
    const long long row0 = c.bh * p.T;
#pragma unroll
    for (int r2 = 0; r2 < 2; ++r2) {
        const int r = lane + 32 * r2;
        const bool in = t0 + r < p.T;
        const long long idx = row0 + (in ? t0 + r : 0);
        cp_async4(stage + kBL + 4 * r, p.beta + idx, in ? 4u : 0u);
        cp_async4(stage + kBL + 256 + 4 * r, p.lam + idx, in ? 4u : 0u);
    }
    cp_async_arrive(c.bar(lay::FULL + s));
}

// ---------------------------------------------------------------- state pass and outputs
template <bool f1>
__device__ void state_group(const FusedParams& p, const Ctx& c, int ct) {
    const int warp_in = ct >> 5;
    const uint32_t lq = (uint32_t)(32 * warp_in) << 16;
    uint8_t* sop = c.sm + lay::SOP;
    const uint32_t sop_a = c.base + lay::SOP;
    const float* gch = reinterpret_cast<const float*>(c.sm + lay::BAR + lay::GCH);
    for (int n = 0; n < kStages && n < p.N && ct < 32; ++n) issue_load(p, c, n, ct);
    float S[64];  // row a = ct - 64 of the state (threads 64-127)
    if (ct >= 64) {
        const int a = ct - 64;
        if (p.S0) {
            const float4* src = reinterpret_cast<const float4*>(p.S0 + (c.bh * 64 + a) * 64);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 v = src[q];
                S[4 * q] = v.x, S[4 * q + 1] = v.y, S[4 * q + 2] = v.z, S[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) S[e] = 0.f;
        }
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) *reinterpret_cast<uint32_t*>(sop + tf_off<64>(cc, a)) = tf32_rn(S[cc]);
    }
    fence_async_smem();
    named_bar(5, 128);
    bool ok = true;
    for (int n = 0; n < p.N; ++n) {
        const int g = n & 1;
        const uint32_t jj = (uint32_t)(n >> 1) & 1u;
        const uint32_t Bg = c.tmem + 256u * g;
        bool bad = false;
        if (ct == 0) {
            bad = !fwait(c, c.bar(lay::CA + g), jj);
            if (!bad) {
                bulk_wait_read<1>();  // the output store of chunk n - 2 has read its staging tile
                tc_fence_after();
                constexpr uint32_t id = idesc_tf32(128, 64);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_tf32_ta(Bg + 64, Bg + 128 + 8 * ks, desc_k(sop_a + (ks >> 2) * 8192 + 32 * (ks & 3)), id, ks > 0);
                mma_commit(c.bar(lay::CD + g));
                bad = !fwait(c, c.bar(lay::CD + g), jj);
            }
        }
        if (named_bar_or(5, 128, bad)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // the key side has finished with chunk n's stage: refill it with chunk n + kStages
        if (ct < 32 && n + kStages < p.N) issue_load(p, c, n + kStages, ct);
        const float sr = reinterpret_cast<const float*>(c.sm + lay::CGS)[128 * g + ct];
        if (ct < 64) {  // O = Ao S + s Bo~
            const int i = ct;
            uint8_t* ob = c.sm + lay::OUTS + (n & 1) * kTile;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float dv[32], bv[32];
                tmem_ld32x2(Bg + lq + 64 + 32 * h, Bg + lq + 192 + 32 * h, dv, bv);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = fmaf(sr, bv[8 * q + e], dv[8 * q + e]);
                    *reinterpret_cast<uint4*>(ob + sw128(i, 32 * h + 8 * q)) = pack8(o);
                }
            }
        } else {  // S' = e^{L_C} S - K S + s U~
            const int a = ct - 64;
            const float gc = gch[g];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t d0[16], d1[16], u0[16], u1[16];
                tmem_ld16(Bg + lq + 64 + 32 * h, d0);
                tmem_ld16(Bg + lq + 64 + 32 * h + 16, d1);
                tmem_ld16(Bg + lq + 192 + 32 * h, u0);
                tmem_ld16(Bg + lq + 192 + 32 * h + 16, u1);
                tmem_wait_ld();
                regs_ready(d0);
                regs_ready(d1);
                regs_ready(u0);
                regs_ready(u1);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a0 = f1 ? fmaf(sr, __uint_as_float(u0[e]), __uint_as_float(d0[e])) : sr * __uint_as_float(u0[e]);
                    const float a1 = f1 ? fmaf(sr, __uint_as_float(u1[e]), __uint_as_float(d1[e])) : sr * __uint_as_float(u1[e]);
                    S[32 * h + e] = fmaf(gc, S[32 * h + e], a0);
                    S[32 * h + 16 + e] = fmaf(gc, S[32 * h + 16 + e], a1);
                }
            }
#pragma unroll
            for (int cc = 0; cc < 64; ++cc) *reinterpret_cast<uint32_t*>(sop + tf_off<64>(cc, a)) = tf32_rn(S[cc]);
        }
        tc_fence_before();
        fence_async_smem();
        named_bar(5, 128);
        if (ct == 0) {
            mbar_arrive(c.bar(lay::CONS + g));  // this chunk's TMEM has been read
            tma_store_3d(&p.tm_out, c.base + lay::OUTS + (n & 1) * kTile, 0, n * kC, (int)c.bh);
        }
    }
    if (ok && ct >= 64 && p.S_final) {
        float4* dst = reinterpret_cast<float4*>(p.S_final + (c.bh * 64 + ct - 64) * 64);
#pragma unroll
        for (int q = 0; q < 16; ++q) dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
    if (ok && p.tail_out && ct < 8) {  // window 1: the tail is the last key (the next call's x)
        uint4 v = make_uint4(0, 0, 0, 0);
        if (p.T > 0) v = reinterpret_cast<const uint4*>(p.k + (c.bh * p.T + p.T - 1) * 64)[ct];
        else if (p.pos > 0) v = reinterpret_cast<const uint4*>(p.tail + c.bh * 64)[ct];
        reinterpret_cast<uint4*>(p.tail_out + c.bh * 64)[ct] = v;
    }
    if (ct < 32) {  // every load this warp issued has landed before the CTA exits (bounded)
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (ct == 0)
            for (int n = max(0, p.N - kStages); n < p.N; ++n)
                mbar_wait_bounded(c.bar(lay::FULL + n % kStages), (uint32_t)(n / kStages) & 1u, kTimeoutCycles);
    }
    if (ct == 0) {
        bulk_wait_all();
        mma_commit(c.bar(lay::DRAIN + 2));
        mbar_wait_bounded(c.bar(lay::DRAIN + 2), 0, kTimeoutCycles);
    }
}

template <bool f1>
__global__ void __launch_bounds__(kThreads, 1) falcon_fused_kernel(const __grid_constant__ FusedParams p) {
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
        for (int g = 0; g < 2; ++g) {
            mbar_init(c.bar(lay::MMA + g), 1);
            mbar_init(c.bar(lay::CA + g), 1);
            mbar_init(c.bar(lay::CD + g), 1);
            mbar_init(c.bar(lay::CONS + g), 1);
        }
        for (int d = 0; d < 3; ++d) mbar_init(c.bar(lay::DRAIN + d), 1);
        *c.abort = 0;
        mbar_init_fence();
    }
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + lay::BAR + lay::TSLOT);
    if (warp == 8) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tslot;

    if (warp < 8) key_group<f1>(p, c, warp >> 2, tid & 127);
    else state_group<f1>(p, c, tid - 256);

    tc_fence_before();
    __syncthreads();
    if (warp == 8) tmem_dealloc(c.tmem, 512);
}

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

}  // namespace

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
// [BH][T][64] fp32, 64 x 64 boxes (256-byte rows), no swizzle
bool encode_bhtd_f32(CUtensorMap* tm, const void* ptr, long long T, long long BH) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {64 * 4, (cuuint64_t)T * 64 * 4};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
// The opt-in shared-memory limit of the current device, and the kernels' dynamic shared-memory
// attribute set on it, both once per device.
constexpr int kMaxDevices = 64;
bool prepare_device() {
    static int optin[kMaxDevices] = {};
    static bool ready[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (!ready[dev]) {
        if (cudaDeviceGetAttribute(&optin[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            optin[dev] < lay::ALLOC ||
            cudaFuncSetAttribute(falcon_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay::ALLOC) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay::ALLOC) !=
                cudaSuccess)
            return false;
        ready[dev] = true;
    }
    return true;
}

}  // namespace

bool fused_supported(const Launch& a) {
    return (a.variant == kF1 || a.variant == kF1A) && a.bf16 && a.dk == 64 && a.dv == 64 && a.chunk == 64 &&
           a.W == 1 && a.T != 1 && a.T < (1LL << 31) - 64 && a.B * a.H < (1LL << 31);
}

int launch_fused(const Launch& a, cudaStream_t st) {
    if (!prepare_device()) return 4;
    const long long BH = a.B * a.H;
    FusedParams p = {};
    if (a.T > 0 && (!encode_bhtd(&p.tm_q, a.q, a.T, BH) || !encode_bhtd(&p.tm_k, a.k, a.T, BH) ||
                    !encode_bhtd(&p.tm_v, a.v, a.T, BH) || !encode_bhtd(&p.tm_out, a.out, a.T, BH)))
        return 4;
    p.beta = a.beta;
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
    if (a.variant == kF1) falcon_fused_kernel<true><<<(unsigned)BH, kThreads, lay::ALLOC, st>>>(p);
    else falcon_fused_kernel<false><<<(unsigned)BH, kThreads, lay::ALLOC, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int fused_consume_timeout_flag(int* flag) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fused_timeout_flag, sizeof(int)) != cudaSuccess) return 1;
    if (v && cudaMemcpyToSymbol(g_fused_timeout_flag, &zero, sizeof(int)) != cudaSuccess) return 1;
    *flag = v;
    return 0;
}

}  // namespace falcon
