// Chunk maps of Falcon-3 and Falcon-3A on the tensor cores (bf16 I/O, dk = dv = 64, window W = 4,
// chunk C = 32): the map pass of the scan path, one CTA per chunk, two CTAs per SM.
//
// A chunk acts on its start state affinely, S' = M S + U and O = Ao S + Bo ("Fast Weight Attention
// for Continual Learning", paperlayer summary §H.1: chunk maps compose associatively; §H.3 the
// windowed unknowns). Its unknowns are the residuals r_m of every (token i, window slot a) pair,
// m = 4 i + a, whose pair is the extended row e = i - a + 3 (x_e the shifted key, y_e the target).
// With X_w the 128 x 64 matrix of those keys (row m = x_{e(m)}), G = X_w X_w^T, kap_i = eta_i / B_i
// (B_i the window's realised pairs), the chunk-local log-decay prefixes L_i (reset to 0 at the chunk
// start, Lx_i = L_{i-1}), u_m = kap_i e^{-L_i} on realised pairs (0 elsewhere) and d_i = e^{Lx_i}, a
// value column with start column s and targets y satisfies
//   v_m = u_m (y_m - d_i a_m),   a_m = (X_w s)_m + sum_{m' : token(m') < i} G_{m m'} v_{m'}
//   s' = e^{L_C} (s + X_w^T v),  o_i = e^{L_i} ((Q s)_i + sum_{m : token(m) <= i} (q_i . x_m) v_m),
// (Falcon-3A: v_m = u_m y_m, no solve). The maps are these columns for 128 virtual columns at once:
// the unit start columns e_c without targets (the columns of M and Ao) and the zero start with the
// targets (U and Bo). TMEM lane c holds virtual column c; the products are tcgen05 (M = 128).
//
// Per chunk (4 warps; warp w reads TMEM lane quadrant w):
//   loads     TMA of the key tile (from row t0 - 4), the value tile (from t0 - 3) and the query tile,
//             a continuation's first rows from the tail; X_w built from the key tile
//   products  G = X_w X_w^T and Q X_w^T (tcgen05 bf16, exact inputs, fp32 sums); for Falcon-3 then
//             a = X_w s of every virtual column, [I ; 0] X_w^T, beside the scalars
//   operands  G's off-diagonal blocks as bf16 hi + lo K-major tiles, its diagonal 32 x 32 blocks in
//             fp32 (the entries a substitution needs), the masked scores as bf16 hi + lo
//   scalars   per token eta (window normaliser from the scan path's per-token pass, or for Falcon-3A
//             the window's mean key energy), the clamp, log1pf, a warp scan of the prefixes
//   solve     four 32-row blocks (8 tokens): each block's substitution on the CUDA cores, one virtual
//             column per lane, then G[later rows, block] v_block onto the later rows' a in TMEM
//             (tcgen05, bf16 hi/lo products)
//   maps      X_w^T V and masked(Q X_w^T) V (tcgen05), scaled into M, U, Ao, Bo in the workspace
// A chunk whose total log decay is below -30 (the factored exponentials would overflow) is left to
// the CUDA-core map kernel: this kernel marks each chunk it finished in the chunk block's unused state
// slot, and the CUDA-core kernel skips those.
//
// Every wait is bounded: on timeout the kernel raises a device flag, leaves its chunk unmarked and
// drains what it issued before it frees its TMEM; falcon_device_status() reports it.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "falcon_internal.h"
#include "sm103_f32x2.cuh"
#include "sm103_ptx.cuh"

namespace falcon {

__device__ int g_f3map_timeout_flag = 0;

namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kC = 32, kW = 4, kD = 64;
constexpr int kThreads = 128;
constexpr int kTile = 8192;  // 64 x 64 bf16
constexpr long long kTimeoutCycles = 4000000000LL;  // ~2 s
constexpr float kFastL = 30.f;
constexpr long long kMat = 64 * 64, kBlk = 5 * kMat;  // the scan path's chunk block [M | U | S | Ao | Bo]

// G's diagonal 32 x 32 blocks, packed by source row: in-block row r (token t = r / 4) holds G[r2][r]
// for the in-block rows r2 of later tokens, 4 (t + 1) .. 31 (16-byte groups)
__host__ __device__ constexpr int dg_off(int r) {
    return 4 * (28 * (r >> 2) - 2 * (r >> 2) * ((r >> 2) - 1)) + (r & 3) * (28 - 4 * (r >> 2));
}
constexpr int kDBlk = dg_off(32);  // 448 floats

struct MapParams {
    CUtensorMap tm_q, tm_k, tm_v;
    const float* beta;
    const float* lam;
    const float* mu;  // Falcon-3: every token's window normaliser [B*H][T]
    const bf16* k;
    const bf16* v;
    const bf16* tail;
    bf16* tail_out;
    float* ws;
    long long T, pos, N;
    float eps, eps_gamma;
};

namespace lay {
constexpr int KT = 0, VT = kTile, QT = 2 * kTile, XW = 3 * kTile;  // QT directly before XW: [Q; X_w[0:64]]
constexpr int G01H = XW + 16384, G01L = G01H + 12288;  // G[32:128, 0:64], 96 rows
constexpr int G2H = G01L + 12288, G2L = G2H + 4096;    // G[96:128, 64:128], 32 rows
constexpr int SCH = G2L + 4096, SCL = SCH + 8192;      // masked Q X_w^T [i][m], two K-atoms of 32 rows
constexpr int GD = SCL + 8192;                         // four packed diagonal blocks (fp32)
constexpr int U = GD + 4 * kDBlk * 4;                  // u [128]
constexpr int WG = U + 512;                            // G's entries within each token's own window [128][4]
constexpr int DT = WG + 2048, ELT = DT + 128;          // d_i, e^{L_i} [32]
constexpr int MISC = ELT + 128;                        // [0] e^{L_C}, [1] fast, [2..] beta, lambda, mu scratch
constexpr int BAR = MISC + 512;
constexpr int FULL = 0, MMA = 1, DRAIN = 2, NBAR = 3;
constexpr int ABORT = NBAR * 8, TSLOT = ABORT + 4;
constexpr int BYTES = BAR + 64;
constexpr int ALLOC = BYTES + 1024;
static_assert(XW % 1024 == 0 && G01H % 1024 == 0 && G01L % 1024 == 0 && G2H % 1024 == 0 && G2L % 1024 == 0 &&
                  SCH % 1024 == 0 && SCL % 1024 == 0 && GD % 16 == 0, "layout");
static_assert(2 * (ALLOC + 1024) <= 233472, "two CTAs per SM");
}  // namespace lay

// TMEM columns (256 per CTA)
constexpr uint32_t kRA = 0, kRB = 128;

struct Ctx {
    uint8_t* sm;
    uint32_t base;
    uint32_t tmem;
    volatile int* abort;
    __device__ uint32_t bar(int i) const { return base + lay::BAR + 8 * i; }
};

// Bounded wait by one thread; false on timeout.
__device__ bool fwait(const Ctx& c, uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    int spins = 0;
    while (!mbar_try(bar, parity)) {
        if (++spins > 64) __nanosleep(32);
        if (clock64() - t0 > kTimeoutCycles) {
            *c.abort = 1;
            atomicExch(&g_f3map_timeout_flag, 1);
            return false;
        }
    }
    return true;
}

// n consecutive TMEM columns (n = 16 k) of this thread's lane into v (one wait).
template <int NQ>
__device__ __forceinline__ void tld(uint32_t taddr, float* v) {
    uint32_t r[NQ][16];
#pragma unroll
    for (int q = 0; q < NQ; ++q) tmem_ld16(taddr + 16 * q, r[q]);
    tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        regs_ready(r[q]);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[16 * q + e] = __uint_as_float(r[q][e]);
    }
}
// 16 k fp32 values to consecutive TMEM columns (no wait).
template <int NQ>
__device__ __forceinline__ void tst(uint32_t taddr, const float* x) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(x[16 * q + e]);
        tmem_st16(taddr + 16 * q, r);
    }
}

__device__ __forceinline__ float ld_bf16(const uint8_t* p) { return __bfloat162float(*reinterpret_cast<const bf16*>(p)); }

// ---------------------------------------------------------------- the kernel
template <bool F3>
__global__ void __launch_bounds__(kThreads, 2) falcon_f3map_kernel(const __grid_constant__ MapParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx c;
    c.sm = sm;
    c.base = base;
    c.abort = reinterpret_cast<volatile int*>(sm + lay::BAR + lay::ABORT);
    const long long bh = blockIdx.x / p.N, nck = blockIdx.x % p.N, t0 = nck * kC;
    const int n = (int)min((long long)kC, p.T - t0);
    float* blk = p.ws + (bh * p.N + nck) * kBlk;
    float* u = reinterpret_cast<float*>(sm + lay::U);
    float* wg = reinterpret_cast<float*>(sm + lay::WG);
    float* dt = reinterpret_cast<float*>(sm + lay::DT);
    float* elt = reinterpret_cast<float*>(sm + lay::ELT);
    float* misc = reinterpret_cast<float*>(sm + lay::MISC);
    if (tid == 0) {
        mbar_init(c.bar(lay::FULL), 1);
        mbar_init(c.bar(lay::MMA), 1);
        mbar_init(c.bar(lay::DRAIN), 1);
        *c.abort = 0;
        mbar_init_fence();
    }
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + lay::BAR + lay::TSLOT);
    if (warp == 0) tmem_alloc(smem_u32(tslot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tslot;
    const uint32_t tq = c.tmem + ((uint32_t)(32 * warp) << 16);  // this warp's lane quadrant
    uint32_t mph = 0;                                            // MMA barrier phases consumed
    bool ok = true;

    // ---- loads: keys from row t0 - 4 (extended row e = key t0 - 4 + e), values from t0 - 3, queries
    if (tid == 0) {
        mbar_expect_tx(c.bar(lay::FULL), 3 * kTile);
        tma_load_3d(base + lay::KT, &p.tm_k, 0, (int)t0 - 4, (int)bh, c.bar(lay::FULL));
        tma_load_3d(base + lay::VT, &p.tm_v, 0, (int)t0 - 3, (int)bh, c.bar(lay::FULL));
        tma_load_3d(base + lay::QT, &p.tm_q, 0, (int)t0, (int)bh, c.bar(lay::FULL));
    }
    if (tid < kC) {  // the token's inputs (0 past the end)
        const long long g = bh * p.T + t0 + tid;
        misc[32 + tid] = tid < n ? p.beta[g] : 0.f;
        misc[64 + tid] = tid < n ? p.lam[g] : 0.f;
        misc[96 + tid] = (F3 && tid < n) ? p.mu[g] : 0.f;
    }
    {
        bool bad = false;
        if (tid == 0) bad = !fwait(c, c.bar(lay::FULL), 0u);
        ok = !named_bar_or(1, kThreads, bad);
    }
    if (ok) {
        if (nck == 0 && p.pos > 0 && p.tail) {  // a continuation's first rows come from the tail
            const bf16* tl = p.tail + bh * (kW * kD + (kW - 1) * kD);
            if (tid < 32) {  // key rows e = 0..3 (local key e - 4)
                const int e = tid >> 3, q8 = tid & 7;
                if (p.pos + 1 + (e - 4) > 0)
                    *reinterpret_cast<uint4*>(sm + lay::KT + sw128(e, 8 * q8)) =
                        reinterpret_cast<const uint4*>(tl + e * kD)[q8];
            } else if (tid < 56) {  // value rows e = 0..2 (local value e - 3)
                const int e = (tid - 32) >> 3, q8 = tid & 7;
                if (p.pos + 1 + (e - 3) > 0)
                    *reinterpret_cast<uint4*>(sm + lay::VT + sw128(e, 8 * q8)) =
                        reinterpret_cast<const uint4*>(tl + kW * kD + e * kD)[q8];
            }
        }
        __syncthreads();
        // X_w: row m = (i, a) is the key tile's extended row e = i - a + 3
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int idx = tid + kThreads * s, m = idx >> 3, q8 = idx & 7, e = (m >> 2) - (m & 3) + 3;
            *reinterpret_cast<uint4*>(sm + lay::XW + sw128(m, 8 * q8)) =
                *reinterpret_cast<const uint4*>(sm + lay::KT + sw128(e, 8 * q8));
        }
        fence_async_smem();
        __syncthreads();
        bool bad = false;
        if (tid == 0) {  // G = X_w X_w^T into RA; [Q; X_w[0:64]] X_w^T into RB (rows 0-31: the scores)
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(c.tmem + kRA, desc_k(base + lay::XW + 32 * ks), desc_k(base + lay::XW + 32 * ks), id, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(c.tmem + kRB, desc_k(base + lay::QT + 32 * ks), desc_k(base + lay::XW + 32 * ks), id, ks > 0);
            mma_commit(c.bar(lay::MMA));
            bad = !fwait(c, c.bar(lay::MMA), mph & 1u);
        }
        ++mph;
        ok = !named_bar_or(1, kThreads, bad);
    }
    if (ok) {
        tc_fence_after();
        // ---- G row m = tid: the off-diagonal blocks as bf16 hi + lo, this warp's diagonal block (rows
        // 32 w .. 32 w + 31) packed in fp32, and the row's entries within its own token's window
        {
            const int m = tid, r = lane, f = 4 * ((r >> 2) + 1);
            float* gd = reinterpret_cast<float*>(sm + lay::GD) + warp * kDBlk + dg_off(r) - f;
            float g[64];
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                tld<4>(tq + kRA + 64 * h, g);
                if (h == 0 && m >= 32) {
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) st8_hilo(sm + lay::G01H, sm + lay::G01L, sw128(m - 32, 8 * q8), g + 8 * q8);
                }
                if (h == 1 && m >= 96) {
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) st8_hilo(sm + lay::G2H, sm + lay::G2L, sw128(m - 96, 8 * q8), g + 8 * q8);
                }
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {  // this warp's diagonal block, if its columns are in this half
                    if (warp == 2 * h + bb) {
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            const float* x = g + 32 * bb + 4 * q4;
                            if (4 * q4 >= f) *reinterpret_cast<float4*>(gd + 4 * q4) = make_float4(x[0], x[1], x[2], x[3]);
                            if (4 * q4 == f - 4) *reinterpret_cast<float4*>(wg + 4 * m) = make_float4(x[0], x[1], x[2], x[3]);
                        }
                    }
                }
            }
        }
        if (warp == 0) {  // score row i = lane, masked to the pairs of tokens <= i, as bf16 hi + lo
            const int i = lane;
            float s[64];
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                tld<4>(tq + kRB + 64 * h, s);
#pragma unroll
                for (int e = 0; e < 64; ++e) s[e] = ((64 * h + e) >> 2) <= i ? s[e] : 0.f;
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8)
                    st8_hilo(sm + lay::SCH + 4096 * h, sm + lay::SCL + 4096 * h, sw128(i, 8 * q8), s + 8 * q8);
            }
        }
        if (F3) {  // the rows of [I ; 0] (lane c < 64: e_c) as a bf16 A operand in RB's first 32 columns
            // (each warp writes its own lanes, warp 0 after reading its scores there)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t z[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    z[e] = (tid < 64 && (tid >> 1) == 16 * q + e) ? ((tid & 1) ? 0x3F800000u : 0x3F80u) : 0u;
                tmem_st16(tq + kRB + 16 * q, z);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        fence_async_smem();
        __syncthreads();
        // ---- Falcon-3: a = X_w s for every virtual column at once, [I ; 0] X_w^T into RA (a unit
        // column reads X_w's column c, a target column 0), on the tensor cores while warp 0 forms the
        // per-token scalars
        if (F3 && tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ta(c.tmem + kRA, c.tmem + kRB + 8 * ks, desc_k(base + lay::XW + 32 * ks), id, ks > 0);
            mma_commit(c.bar(lay::MMA));
        }
        // ---- per-token scalars (warp 0, token i = lane)
        if (warp == 0) {
            const int i = lane;
            const long long tau = p.pos + t0 + i + 1;
            // the window's realised pairs are the slots a < nb; Falcon-3A's window energy sums their
            // keys' energies G[4 i + a][4 i + a]
            const int nb = (int)min((long long)kW, max(0LL, tau - 1));
            float en = 0.f;
#pragma unroll
            for (int a = 0; a < kW; ++a)
                if (a < nb) en += wg[4 * (4 * i + a) + a];
            float eta = 0.f, alpha = 0.f, kap = 0.f;
            if (i < n && nb > 0) {
                // Falcon-3: the window normaliser from the per-token pass; Falcon-3A: the window's mean
                // key energy
                const float mu = F3 ? misc[96 + i] : en / (float)nb;
                const float lm = misc[64 + i];
                const float den = mu + lm + p.eps;
                eta = den == 0.f ? 0.f : misc[32 + i] / den;
                alpha = fminf(eta * lm, 1.f - p.eps_gamma);
                kap = eta / (float)nb;
            }
            const float l = log1pf(-alpha);
            float incl = l;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const float LC = __shfl_sync(0xffffffffu, incl, 31);
            const float ui = kap * expf(-incl);
#pragma unroll
            for (int a = 0; a < kW; ++a) u[4 * i + a] = (i < n && tau - a >= 2) ? ui : 0.f;
            dt[i] = expf(incl - l);
            elt[i] = expf(incl);
            if (i == 0) {
                misc[0] = expf(LC);
                misc[1] = LC >= -kFastL ? 1.f : 0.f;
            }
        }
        bool bad = false;
        if (F3 && tid == 0) bad = !fwait(c, c.bar(lay::MMA), mph & 1u);
        if (F3) ++mph;
        ok = !named_bar_or(1, kThreads, bad);
    }
    const bool fast = ok && misc[1] != 0.f;
    if (fast) {
        const int col = tid, cc = col & 63;
        const bool unit = col < 64;  // unit start column e_cc without targets (M, Ao), else targets (U, Bo)
        if (F3) {
            tc_fence_after();  // a = X_w s is in RA
            // ---- v_m = u_m (y_m - d_i a_m) by blocks of 32 rows (8 tokens): the block's a from TMEM,
            // its substitution, v (bf16 hi + lo) into the A operand columns, then G[later rows, block]
            // v_block onto the later rows' a
            const float* Gd = reinterpret_cast<const float*>(sm + lay::GD);
#pragma unroll 1
            for (int bk = 0; bk < 4; ++bk) {
                float a[32];
                tld<2>(tq + kRA + 32 * bk, a);
                const float* gd = Gd + bk * kDBlk;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int tok = 8 * bk + t;
                    const float d = dt[tok];
#pragma unroll
                    for (int a4 = 0; a4 < 4; ++a4) {
                        const int r = 4 * t + a4;
                        const float y = unit ? 0.f : ld_bf16(sm + lay::VT + sw128(tok - a4 + 3, cc));
                        a[r] = u[32 * bk + r] * fmaf(-d, a[r], y);
                    }
#pragma unroll
                    for (int a4 = 0; a4 < 4; ++a4) {
                        const int r = 4 * t + a4;
                        const float vr = a[r];
#pragma unroll
                        for (int r2 = 4 * (t + 1); r2 < 32; r2 += 4) {
                            const float4 g4 = *reinterpret_cast<const float4*>(gd + dg_off(r) + r2 - 4 * (t + 1));
                            fma2(a[r2], a[r2 + 1], g4.x, g4.y, vr);  // packed fp32 FMAs
                            fma2(a[r2 + 2], a[r2 + 3], g4.z, g4.w, vr);
                        }
                    }
                }
                {
                    uint32_t hh[16], ll[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) split2(a[2 * e], a[2 * e + 1], hh[e], ll[e]);
                    tmem_st16(tq + kRB + 16 * bk, hh);
                    tmem_st16(tq + kRB + 64 + 16 * bk, ll);
                }
                if (bk < 3) {  // a[rows after the block] += G[those rows, block] v_block: V_hi G_hi, V_lo G_hi, V_hi G_lo
                    tmem_wait_st();
                    tc_fence_before();
                    __syncthreads();
                    bool bad = false;
                    if (tid == 0) {
                        tc_fence_after();
                        const uint32_t id = idesc_bf16(128, (uint32_t)(96 - 32 * bk), false, false);
                        const uint32_t d = c.tmem + kRA + 32 * (bk + 1);
                        // B: the later rows of G at the block's K columns (tile rows at 128 bytes, 8-row
                        // groups 1024 bytes apart; 32 K elements = 64 bytes)
                        const uint32_t off = bk == 1 ? 4096u + 64u : 0u;
                        const uint32_t gh = base + (bk == 2 ? lay::G2H : lay::G01H) + off;
                        const uint32_t gl = base + (bk == 2 ? lay::G2L : lay::G01L) + off;
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
                            mma_bf16_ta(d, c.tmem + kRB + 16 * bk + 8 * ks, desc_k(gh + 32 * ks), id, 1);
                            mma_bf16_ta(d, c.tmem + kRB + 64 + 16 * bk + 8 * ks, desc_k(gh + 32 * ks), id, 1);
                            mma_bf16_ta(d, c.tmem + kRB + 16 * bk + 8 * ks, desc_k(gl + 32 * ks), id, 1);
                        }
                        mma_commit(c.bar(lay::MMA));
                        bad = !fwait(c, c.bar(lay::MMA), mph & 1u);
                    }
                    ++mph;
                    bad = named_bar_or(1, kThreads, bad);  // every thread takes the same decision
                    if (bad) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
            }
        } else {  // Falcon-3A: v_m = u_m y_m (0 for the unit columns)
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float a[64];
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const int m = 64 * h + e;
                    a[e] = unit ? 0.f : u[m] * ld_bf16(sm + lay::VT + sw128((m >> 2) - (m & 3) + 3, cc));
                }
                uint32_t hh[2][16], ll[2][16];
#pragma unroll
                for (int e = 0; e < 32; ++e) split2(a[2 * e], a[2 * e + 1], hh[e >> 4][e & 15], ll[e >> 4][e & 15]);
                tmem_st16(tq + kRB + 32 * h, hh[0]);
                tmem_st16(tq + kRB + 32 * h + 16, hh[1]);
                tmem_st16(tq + kRB + 64 + 32 * h, ll[0]);
                tmem_st16(tq + kRB + 64 + 32 * h + 16, ll[1]);
            }
        }
        if (ok) {
            tmem_wait_st();
            tc_fence_before();
            __syncthreads();
            // ---- X_w^T V into RA[0, 64) and masked(Q X_w^T) V into RA[64, 96)
            bool bad = false;
            if (tid == 0) {
                tc_fence_after();
                constexpr uint32_t idx = idesc_bf16(128, 64, false, true), ido = idesc_bf16(128, 32, false, false);
#pragma unroll
                for (int ks = 0; ks < 16; ++ks)  // B = X_w read MN-major, 16 rows (2048 bytes) per K step
                    mma_bf16_ta(c.tmem + kRA, c.tmem + kRB + 8 * (ks & 7) + 64 * (ks >> 3),
                                desc_mn(base + lay::XW + 2048 * (ks & 7), 16384), idx, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t so = 4096u * (ks >> 2) + 32u * (ks & 3);
                    mma_bf16_ta(c.tmem + kRA + 64, c.tmem + kRB + 8 * ks, desc_k(base + lay::SCH + so), ido, ks > 0);
                    mma_bf16_ta(c.tmem + kRA + 64, c.tmem + kRB + 64 + 8 * ks, desc_k(base + lay::SCH + so), ido, 1);
                    mma_bf16_ta(c.tmem + kRA + 64, c.tmem + kRB + 8 * ks, desc_k(base + lay::SCL + so), ido, 1);
                }
                mma_commit(c.bar(lay::MMA));
                bad = !fwait(c, c.bar(lay::MMA), mph & 1u);
            }
            ++mph;
            ok = !named_bar_or(1, kThreads, bad);
        }
        if (ok) {
            tc_fence_after();
            // ---- the maps: M = e^{L_C} (I + X_w^T V_unit), U = e^{L_C} X_w^T V_targets,
            // Ao_i = e^{L_i} (q_i + (masked Q X_w^T V_unit)_i), Bo_i = e^{L_i} (masked Q X_w^T V_targets)_i
            float x[64];
            tld<4>(tq + kRA, x);
            const float eLC = misc[0];
            float* dst = blk + (unit ? 0 : kMat) + cc;
#pragma unroll
            for (int k = 0; k < 64; ++k) dst[64 * k] = eLC * (x[k] + ((unit && k == cc) ? 1.f : 0.f));
            tld<2>(tq + kRA + 64, x);
            float* od = blk + (unit ? 3 * kMat : 4 * kMat) + cc;
#pragma unroll
            for (int i = 0; i < kC; ++i) {
                const float qv = unit ? ld_bf16(sm + lay::QT + sw128(i, cc)) : 0.f;
                od[64 * i] = elt[i] * (qv + x[i]);
            }
        }
    }
    // the call's tail (the last W keys and W - 1 values) from the last chunk's CTA
    if (ok && p.tail_out && nck == p.N - 1) {
        constexpr int kTailStride = kW * kD + (kW - 1) * kD;
        bf16* to = p.tail_out + bh * kTailStride;
        const bf16* tl = p.tail ? p.tail + bh * kTailStride : nullptr;
        for (int idx = tid; idx < kTailStride; idx += kThreads) {
            const bool key = idx < kW * kD;
            const int j = key ? idx : idx - kW * kD, sl = j >> 6, cc = j & 63;
            const long long uu = key ? p.T - kW + sl : p.T - kW + 1 + sl;  // local index (< 0: the tail)
            bf16 val = __float2bfloat16_rn(0.f);
            if (uu >= 0) val = (key ? p.k : p.v)[(bh * p.T + uu) * kD + cc];
            else if (tl && p.pos + 1 + uu > 0) val = tl[key ? (uu + kW) * kD + cc : kW * kD + (uu + kW - 1) * kD + cc];
            to[idx] = val;
        }
    }
    // mark the chunk: the CUDA-core map kernel takes every chunk left unmarked
    if (tid == 0) reinterpret_cast<int*>(blk + 2 * kMat)[0] = (ok && fast) ? 1 : 0;
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // no MMA this thread issued is still running when the CTA frees its TMEM
        mma_commit(c.bar(lay::DRAIN));
        mbar_wait_bounded(c.bar(lay::DRAIN), 0, kTimeoutCycles);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(c.tmem, 256);
}

bool prepare_device() {
    constexpr int kMaxDevices = 64;
    static bool ready[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (!ready[dev]) {
        if (cudaFuncSetAttribute(falcon_f3map_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay::ALLOC) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_f3map_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay::ALLOC) !=
                cudaSuccess)
            return false;
        ready[dev] = true;
    }
    return true;
}

}  // namespace

bool f3map_supported(const Launch& a) {
    return (a.variant == kF3 || a.variant == kF3A) && a.bf16 && a.dk == kD && a.dv == kD && a.W == kW &&
           a.chunk == kC && a.T < (1LL << 31) - 64 && a.B * a.H < (1LL << 31);
}

int launch_f3map(const Launch& a, float* ws, long long N, const float* mu, cudaStream_t st) {
    if (!prepare_device()) return 4;
    const long long BH = a.B * a.H;
    if (BH == 0 || N == 0) return 0;
    MapParams p = {};
    if (!encode_bhtd(&p.tm_q, a.q, a.T, BH) || !encode_bhtd(&p.tm_k, a.k, a.T, BH) ||
        !encode_bhtd(&p.tm_v, a.v, a.T, BH))
        return 4;
    p.beta = a.beta;
    p.lam = a.lam;
    p.mu = mu;
    p.k = static_cast<const bf16*>(a.k);
    p.v = static_cast<const bf16*>(a.v);
    p.tail = static_cast<const bf16*>(a.tail);
    p.tail_out = static_cast<bf16*>(a.tail_out);
    p.ws = ws;
    p.T = a.T;
    p.pos = a.pos;
    p.N = N;
    p.eps = a.eps;
    p.eps_gamma = a.eps_gamma;
    const unsigned grid = (unsigned)(BH * N);
    if (a.variant == kF3) falcon_f3map_kernel<true><<<grid, kThreads, lay::ALLOC, st>>>(p);
    else falcon_f3map_kernel<false><<<grid, kThreads, lay::ALLOC, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int f3map_consume_timeout_flag(int* flag) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_f3map_timeout_flag, sizeof(int)) != cudaSuccess) return 1;
    if (v && cudaMemcpyToSymbol(g_f3map_timeout_flag, &zero, sizeof(int)) != cudaSuccess) return 1;
    *flag = v;
    return 0;
}

}  // namespace falcon
