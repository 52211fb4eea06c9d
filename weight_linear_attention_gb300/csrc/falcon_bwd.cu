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
//   falcon_bwd_prep   every chunk at once: T, the forward transition (M, U = X^T diag(w) T Y), the
//                     chunk's scalars and V;
//   falcon_bwd_chain  per sequence (two CTAs, one per scan; the carried matrix in tensor memory, one
//                     tcgen05 product per step): S_{n+1} = M_n S_n + U_n forward and dS_n =
//                     M_n^T dS_{n+1} + V_n backward, storing S_n and dS_{n+1};
//   falcon_bwd_grad   every chunk at once: all input gradients from S_n and dS_{n+1}.
// prep and grad run one 256-thread CTA per chunk, two per SM, every 64 x 64 x 64 product a tcgen05
// bf16 product with the fp32 operands split into bf16 hi and lo parts (hi*hi + hi*lo + lo*hi, fp32
// sums in tensor memory); the scalars, the per-element factors and the triangular inverse run on the
// CUDA cores in fp32. With 4 or more sequences a call runs them as 2 or 4 groups, each group's three
// kernels on a stream of its own (its chain on a high-priority one).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "falcon_internal.h"
#include "sm103_ptx.cuh"

namespace falcon {

__device__ int g_bwd_timeout_flag = 0;

namespace {

using namespace ptx;

constexpr int kD = 64;        // dk = dv
constexpr int kC = 64;        // chunk length
constexpr int kWsMat = kD * kD;             // floats per workspace matrix
constexpr int kWsScal = 768;                // floats: the chunk's scalars, as the prep kernel computed them
constexpr int kWsChunk = 6 * kWsMat + kWsScal;  // M, U, V, T, S_n, dS_{n+1}, the scalars: U and V dense
                                            // fp32; M, T, S_n and dS_{n+1} as bf16 hi and lo tiles (8 KB
                                            // each, hi first)
enum { kWsM = 0, kWsU = 1, kWsV = 2, kWsT = 3, kWsS = 4, kWsDS = 5, kWsSC = 6 };

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
    long long T, pos, N, BH;  // tokens, position, chunks per sequence, sequences of this launch
    long long bh0;            // the first of them
    float eps, eps_gamma;
};

// Scalars of one chunk: computed by the prep kernel, which stores them for the gradient kernel.
struct Scal {
    float eta[kC], lam[kC], den[kC], gam[kC], L[kC], Lx[kC], eL[kC], eLx[kC], w[kC];
    int unc[kC], live[kC];  // clamp inactive (alpha differentiable); eta = beta / den differentiable
    float eLC, LC;
};
constexpr int kScal16 = (int)(sizeof(Scal) + 15) / 16 * 16;  // bytes, as copied
static_assert(kScal16 <= kWsScal * 4, "the scalars fit their workspace slot");


// ================================================================================================
// Chunk kernels on the tensor cores: one 256-thread CTA per chunk, two per SM. Thread t reads and
// writes TMEM lane t % 128 (warp w: lanes 32 (w % 4) ..) and takes the columns 32 (t / 128) .. + 31 of
// that lane's rows. Every operand is a 64 x 64 bf16 tile in shared memory (128-byte rows, the 128-byte
// swizzle), usable K-major or MN-major, or a 128-row A operand in TMEM. An fp32 operand x enters as
// two tiles, hi = bf16(x) and lo = bf16(x - hi), and a product as hi*hi + hi*lo + lo*hi with fp32
// sums in TMEM: every operand element keeps ~16 significant bits. The inputs of a bf16 call are exact
// tiles without a lo part. Each product is tcgen05 kind::f16 with M = 128 (two stacked 64-row
// operands, or one whose second half is read and its result rows unused), N = 64 or 128 and K = 64,
// issued by one thread; a tcgen05 instruction costs about the same for every N up to 256, so
// products that share an operand are issued as one where the layout allows.

constexpr int kCT = 256;                        // threads of a chunk CTA
constexpr int kTile = 8192;                     // one 64 x 64 bf16 tile
constexpr int kAS = 68;                         // row stride (floats) of the matrix the inverse works on
constexpr long long kCTimeout = 4000000000LL;   // ~2 s

struct Opd {  // one operand of a 64-deep product
    uint32_t addr, lbo;
    int kind;  // 0: K-major tile(s); 1: MN-major (lbo: bytes to the second 64-wide atom); 2: TMEM A
};
__device__ __forceinline__ Opd kmaj(uint32_t a) { return Opd{a, 0u, 0}; }
__device__ __forceinline__ Opd mnmaj(uint32_t a, uint32_t lbo = kTile) { return Opd{a, lbo, 1}; }
__device__ __forceinline__ Opd tmem_a(uint32_t col) { return Opd{col, 0u, 2}; }

// d (+)= A B, M = 128, K = 64 (four steps of 16), N = n (64 or 128).
__device__ __forceinline__ void mma64(uint32_t d, const Opd& a, const Opd& b, uint32_t n, bool acc) {
    const uint32_t id = idesc_bf16(128, n, a.kind == 1, b.kind == 1);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        const uint64_t bd = b.kind == 1 ? desc_mn(b.addr + 2048 * ks, b.lbo) : desc_k(b.addr + 32 * ks);
        const uint32_t ac = (acc || ks > 0) ? 1u : 0u;
        if (a.kind == 2)
            mma_bf16_ta(d, a.addr + 8 * ks, bd, id, ac);
        else
            mma_bf16(d, a.kind == 1 ? desc_mn(a.addr + 2048 * ks, a.lbo) : desc_k(a.addr + 32 * ks), bd, id, ac);
    }
}

// 32 consecutive TMEM columns of this thread's lane (one wait).
__device__ __forceinline__ void tld32(uint32_t taddr, float* v) {
    uint32_t r[2][16];
    tmem_ld16(taddr, r[0]);
    tmem_ld16(taddr + 16, r[1]);
    tmem_wait_ld();
    regs_ready(r[0]);
    regs_ready(r[1]);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        v[e] = __uint_as_float(r[0][e]);
        v[16 + e] = __uint_as_float(r[1][e]);
    }
}
// v[0..31] (the K elements 32 h .. 32 h + 31 of this lane's row) into a bf16 A operand in TMEM whose
// hi part starts at column hc and lo part at lc (element k in the low half of column k / 2 when k is
// even). No wait.
__device__ __forceinline__ void tst_a32(uint32_t hc, uint32_t lc, int h, const float* v) {
    uint32_t hh[16], ll[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) split2(v[2 * e], v[2 * e + 1], hh[e], ll[e]);
    tmem_st16(hc + 16 * h, hh);
    tmem_st16(lc + 16 * h, ll);
}

// Eight elements of a row (from byte offset `off` of the tile, an sw128 offset) as fp32; for fp32
// inputs hi + lo.
template <bool EX>
__device__ __forceinline__ void row8(const uint8_t* hi, const uint8_t* lo, uint32_t off, float* v) {
    unpack8(*reinterpret_cast<const uint4*>(hi + off), v);
    if (!EX) {
        float w[8];
        unpack8(*reinterpret_cast<const uint4*>(lo + off), w);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] += w[e];
    }
}
template <bool EX>
__device__ __forceinline__ float elem(const uint8_t* hi, const uint8_t* lo, uint32_t off) {
    float x = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(hi + off));
    if (!EX) x += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(lo + off));
    return x;
}
// Four fp32 values as bf16 hi and lo at `off` of two tiles (8 bytes each).
__device__ __forceinline__ void put4_hilo(uint8_t* hi, uint8_t* lo, uint32_t off, float4 v) {
    uint32_t h0, l0, h1, l1;
    split2(v.x, v.y, h0, l0);
    split2(v.z, v.w, h1, l1);
    *reinterpret_cast<uint2*>(hi + off) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(lo + off) = make_uint2(l0, l1);
}
__device__ __forceinline__ void store32(float* dst, const float* v) {
#pragma unroll
    for (int q = 0; q < 8; ++q) reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void cp_async16z(uint32_t dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
// One bulk copy shared -> global (addresses 16-byte aligned, size a multiple of 16) as its own group of
// this thread; the source is free again after bulk_wait_read, the copy complete after bulk_wait_all.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Rows r < nr of q, k, v and dout for the chunk's tokens t0 + r (k shifted: token t0 + r - 1, the
// tail key or zero before the first token) into tiles at byte offsets hi[a] (bf16: asynchronous
// copies, left for the caller to commit and wait on) or hi[a] and lo[a] (fp32: through registers).
// An offset < 0 skips the tensor; rows past nr are zero.
template <typename Tin>
__device__ void load_chunk(const BParams& p, uint8_t* sm, uint32_t base, const int (&hi)[4], const int (&lo)[4],
                           long long bh, long long t0, int nr) {
    const Tin* src[4] = {static_cast<const Tin*>(p.q), static_cast<const Tin*>(p.k), static_cast<const Tin*>(p.v),
                         static_cast<const Tin*>(p.dout)};
    const Tin* tail = static_cast<const Tin*>(p.tail);
    const int tid = threadIdx.x;
    auto row = [&](int a, int r) -> const Tin* {
        if (r >= nr) return nullptr;
        const long long t = t0 + r - (a == 1 ? 1 : 0);
        if (t >= 0) return src[a] + (bh * p.T + t) * kD;
        return tail ? tail + bh * kD : nullptr;
    };
    if constexpr (sizeof(Tin) == 2) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            if (hi[a] < 0) continue;
#pragma unroll
            for (int u = 0; u < 512 / kCT; ++u) {
                const int e = tid + kCT * u, r = e >> 3, q8 = e & 7;
                const Tin* ptr = row(a, r);
                cp_async16z(base + (uint32_t)hi[a] + sw128(r, 8 * q8), ptr ? ptr + 8 * q8 : src[a], ptr ? 16u : 0u);
            }
        }
    } else {
        constexpr int NU = 1024 / kCT;
        float4 v[4][NU];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int e = tid + kCT * u, r = e >> 4, c4 = e & 15;
                const Tin* ptr = hi[a] >= 0 ? row(a, r) : nullptr;
                v[a][u] = ptr ? *reinterpret_cast<const float4*>(ptr + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            if (hi[a] < 0) continue;
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int e = tid + kCT * u, r = e >> 4, c4 = e & 15;
                put4_hilo(sm + hi[a], sm + lo[a], sw128(r, 4 * c4), v[a][u]);
            }
        }
    }
}

// Per-token scalars of the chunk from the key tile(s) (four threads per row share its squared norm),
// beta and lambda; then the chunk-local log prefixes (one warp) and their exponentials (one thread a
// row). All threads call it.
template <bool EX>
__device__ void chunk_scalars(Scal& s, const uint8_t* xh, const uint8_t* xl, const BParams& p, long long bh,
                              long long t0, int n) {
    const int tid = threadIdx.x, r = tid >> 2, q = tid & 3;
    float nx = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float x[8];
        row8<EX>(xh, xl, sw128(r, 16 * q + 8 * h), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) nx = fmaf(x[e], x[e], nx);
    }
    nx += __shfl_xor_sync(0xffffffffu, nx, 1);
    nx += __shfl_xor_sync(0xffffffffu, nx, 2);
    if (q == 0) {
        const int i = r;
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
    if (tid < 32) {  // inclusive prefix over 64 rows: lane l holds rows 2l, 2l + 1
        const int l = tid;
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
        s.Lx[2 * l] = ex;
        s.Lx[2 * l + 1] = ex + a;
        if (l == 31) s.LC = v;
    }
    __syncthreads();
    if (tid < kC) {
        const int i = tid;
        const float L = s.L[i], LC = s.LC;
        s.eL[i] = expf(L);
        s.eLx[i] = expf(s.Lx[i]);
        s.w[i] = s.eta[i] * expf(LC - L);
        if (i == 0) s.eLC = expf(LC);
    }
    fence_async_smem();  // the block may leave by a bulk copy
    __syncthreads();
}

// Column sums of a warp's 32 rows: v[0..31] holds this lane's row over 32 columns; returns the sum of
// column `lane` (each step keeps half of the columns and adds the partner lane's copy of that half).
template <int M, int N>
__device__ __forceinline__ void colsum_step(float* v, bool up) {
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
        const float send = up ? v[k] : v[k + N / 2];
        const float keep = up ? v[k + N / 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, M);
    }
}
__device__ __forceinline__ float warp_colsum32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
    colsum_step<16, 32>(v, lane & 16);
    colsum_step<8, 16>(v, lane & 8);
    colsum_step<4, 8>(v, lane & 4);
    colsum_step<2, 4>(v, lane & 2);
    colsum_step<1, 2>(v, lane & 1);
    return v[0];
}

// T = (I + A)^{-1} in place for the strictly lower 64 x 64 A in M (fp32, stride kAS; zero on and above
// the diagonal on entry, T with its unit diagonal on exit): the four 16 x 16 diagonal blocks by
// right-looking column substitution (one thread per column), then two levels of block merges,
// T_ba = -T_bb (A_ba T_aa) through the scratch W (32 x 33 floats), each thread a column of the block
// over an eighth of its rows. The triangles' zeros stand in for the bounds of the sums, so every
// loop has a fixed length. All threads call it.
template <int H>
__device__ __forceinline__ void merge_level(float* M, float* W) {
    constexpr int RQ = H / 8;  // rows per thread
    const int tid = threadIdx.x;
    static_assert((64 / (2 * H)) * H * 8 == kCT, "one thread per (block, column, eighth of the rows)");
    const int cc = tid % H, rq = (tid / H) % 8, blk = tid / (8 * H), r0 = 2 * H * blk;
    {
        float t[H];
#pragma unroll
        for (int k = 0; k < H; ++k) t[k] = M[(r0 + k) * kAS + r0 + cc];  // T_aa column cc
#pragma unroll 1
        for (int r = 0; r < RQ; ++r) {
            const float* a = M + (r0 + H + RQ * rq + r) * kAS + r0;  // A_ba row
            float x = 0.f;
#pragma unroll
            for (int k = 0; k < H; ++k) x = fmaf(a[k], t[k], x);
            W[(H * blk + RQ * rq + r) * 33 + cc] = x;
        }
    }
    __syncthreads();
    {
        float w[H];
#pragma unroll
        for (int k = 0; k < H; ++k) w[k] = W[(H * blk + k) * 33 + cc];
#pragma unroll 1
        for (int r = 0; r < RQ; ++r) {
            const float* t = M + (r0 + H + RQ * rq + r) * kAS + r0 + H;  // T_bb row
            float x = 0.f;
#pragma unroll
            for (int k = 0; k < H; ++k) x = fmaf(t[k], w[k], x);
            M[(r0 + H + RQ * rq + r) * kAS + r0 + cc] = -x;
        }
    }
    __syncthreads();
}
__device__ void invert128(float* M, float* W) {
    const int tid = threadIdx.x;
    float x[16];
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
        const float* Ab = M + 16 * b * kAS + 16 * b;
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r) {
            float col[15];
#pragma unroll
            for (int s2 = r + 1; s2 < 16; ++s2) col[s2 - r - 1] = Ab[s2 * kAS + r];
#pragma unroll
            for (int s2 = r + 1; s2 < 16; ++s2) x[s2] = fmaf(-col[s2 - r - 1], x[r], x[s2]);
        }
    }
    __syncthreads();
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
#pragma unroll
        for (int r = 0; r < 16; ++r) M[(16 * b + r) * kAS + 16 * b + c] = x[r];
    }
    __syncthreads();
    merge_level<16>(M, W);
    merge_level<32>(M, W);
}

// Waits of the chunk kernels: thread 0 waits for the next phase of the MMA barrier (bounded); every
// thread learns whether it completed.
struct ChunkSync {
    uint32_t bar, mph;
    __device__ bool wait() {
        bool bad = false;
        if (threadIdx.x == 0) {
            bad = !mbar_wait_bounded(bar, mph & 1u, kCTimeout);
            if (bad) atomicExch(&g_bwd_timeout_flag, 1);
        }
        ++mph;
        const bool any = __syncthreads_or(bad) != 0;
        tc_fence_after();
        return !any;
    }
    // shared-memory and TMEM writes of every thread are visible to the tensor cores
    __device__ void publish() {
        fence_async_smem();
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
    }
    // nothing issued is still running (waits at most the timeout), then TMEM is freed
    __device__ void finish(uint32_t tmem, uint32_t cols) {
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x == 0) {
            mma_commit(bar + 8);
            mbar_wait_bounded(bar + 8, 0, kCTimeout);
        }
        __syncthreads();
        tc_fence_after();
        if ((threadIdx.x >> 5) == 0) tmem_dealloc(tmem, cols);
    }
};

// Shared-memory layout of the chunk kernels (bytes from the 1024-aligned base): 8 KB tile slots, then
// (prep, Falcon-1) the fp32 matrix of the inverse, the scalars and the barriers.
template <bool EX, bool IP>
struct PrepLay {
    // Falcon-1:  Q X [QL XL] DO [DOL] DXH YH DXL [YL] TH TL AOH AOL   ([..]: fp32 inputs only)
    // Falcon-1A: WXH Q YH EDH WXL [QL YL] EDL X [XL] DO [DOL]
    enum : int {
        Q = IP ? 1 : 0,
        X = IP ? (EX ? 5 : 8) : 1,
        QL = EX ? -1 : (IP ? 5 : 2),
        XL = EX ? -1 : (IP ? 9 : 3),
        DO = IP ? (EX ? 6 : 10) : (EX ? 2 : 4),
        DOL = EX ? -1 : (IP ? 11 : 5),
        DXH = EX ? 3 : 6,
        YH = IP ? 2 : (EX ? 4 : 7),
        DXL = EX ? 5 : 8,
        YL = EX ? -1 : (IP ? 6 : 9),
        TH = EX ? 6 : 10,
        TL = TH + 1,
        AOH = TH + 2,
        AOL = TH + 3,
        WXH = 0,
        EDH = 3,
        WXL = 4,
        EDL = 7,
        NT = IP ? (EX ? 8 : 12) : (EX ? 10 : 14),
        AT = NT * kTile,                          // Falcon-1: the fp32 matrix of the inverse
        SCAL = AT + (IP ? 0 : 64 * kAS * 4),
        BAR = SCAL + (int)(sizeof(Scal) + 15) / 16 * 16,
        BYTES = BAR + 64,
        ALLOC = BYTES + 1024,
        COLS = IP ? 128 : 256                     // TMEM columns
    };
};
template <bool EX, bool IP>
struct GradLay {
    // Q X [QL XL] DO [DOL] | YZ ZL PRH SH PRL SL TH TL DSH DSL, then the scalars, the gradient
    // accumulators and the barriers. Roles of the shared slots over the kernel:
    //   YZ, ZL   Y (Falcon-1; its lo part in ZL) -> Z -> dR; Falcon-1A: P; then dSc_hi, dG_hi
    //   PRH, PRL P -> R (Falcon-1); Falcon-1A: Y
    //   TH, TL   T (Falcon-1); then dSc_lo, dG_lo
    // Adjacent pairs serve as stacked K-major operands: [Q; X], [YZ; ZL], [PRH; SH], [PRL; SL], [TH; TL].
    enum : int {
        Q = 0,
        X = 1,
        QL = EX ? -1 : 2,
        XL = EX ? -1 : 3,
        DO = EX ? 2 : 4,
        DOL = EX ? -1 : 5,
        YZ = EX ? 3 : 6,
        ZL = YZ + 1,
        PRH = YZ + 2,
        SH = YZ + 3,
        PRL = YZ + 4,
        SL = YZ + 5,
        TH = YZ + 6,
        TL = YZ + 7,
        DSH = YZ + 8,
        DSL = YZ + 9,
        NT = YZ + 10,
        SCAL = NT * kTile,
        ACC = SCAL + (int)(sizeof(Scal) + 15) / 16 * 16,  // deta dL dLx dw c2 [64], red [8]
        BAR = ACC + (5 * kC + 8) * 4,
        BYTES = BAR + 64,
        ALLOC = BYTES + 1024
    };
};

// --------------------------------------------------------------------------------------------------
// falcon_bwd_prep: per chunk T, the forward transition M, U = X^T diag(w) T Y and
// V = Ao^T dO with Ao = diag(e^L) Q - P T diag(e^Lx) X (the chunk's read of its start state).
// Falcon-1, as products: [Sc; G] = [Q; X] X^T; P and A from them; T = (I + A)^{-1} on the CUDA cores;
// E = [P; X^T diag(w)] T; E [diag(e^Lx) X | Y] = [P T diag(e^Lx) X, . ; K, U] with M = e^{L_C} I - K;
// V = Ao^T dO. Falcon-1A (T = I, K = 0): [U, . ; ., V] = [(diag(w) X)^T ; Q^T] [Y | diag(e^L) dO].
// M and T go to the workspace as bf16 hi and lo tiles (the chain's and the gradient kernel's
// operands), U and V as dense fp32 matrices.
template <typename Tin, bool IP>
__global__ void __launch_bounds__(kCT, sizeof(Tin) == 2 ? 2 : 1) falcon_bwd_prep(const BParams p) {
    constexpr bool EX = sizeof(Tin) == 2;
    using L = PrepLay<EX, IP>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw), base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    auto TP = [&](int slot) { return sm + slot * kTile; };
    auto TA = [&](int slot) { return base + (uint32_t)(slot * kTile); };
    const int tid = threadIdx.x, warp = tid >> 5, ln = tid & 127, hf = tid >> 7;  // TMEM lane, column half
    Scal& s = *reinterpret_cast<Scal*>(sm + L::SCAL);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BAR + 16);
    ChunkSync cs{base + L::BAR, 0u};
    const long long bh = p.bh0 + blockIdx.x / p.N, nck = blockIdx.x % p.N, t0 = nck * kC;
    const int nr = (int)min((long long)kC, p.T - t0);
    float* ws = p.ws + (bh * p.N + nck) * kWsChunk;

    if (tid == 0) {
        mbar_init(cs.bar, 1);
        mbar_init(cs.bar + 8, 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), L::COLS);
    {
        const int hi[4] = {L::Q * kTile, L::X * kTile, L::YH * kTile, L::DO * kTile};
        const int lo[4] = {L::QL * kTile, L::XL * kTile, L::YL * kTile, L::DOL * kTile};
        load_chunk<Tin>(p, sm, base, hi, lo, bh, t0, nr);
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    cs.publish();
    tc_fence_after();
    const uint32_t tmem = *tslot, tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint8_t* xl = EX ? nullptr : TP(L::XL);
    const int c0 = 32 * hf;  // this thread's columns
    bool ok = true;

    if constexpr (!IP) {
        if (tid == 0) {  // [Sc; G] = [Q; X] X^T into columns 0-63
            tc_fence_after();
            mma64(tmem, kmaj(TA(L::Q)), kmaj(TA(L::X)), 64, false);
            if constexpr (!EX) {
                mma64(tmem, kmaj(TA(L::Q)), kmaj(TA(L::XL)), 64, true);
                mma64(tmem, kmaj(TA(L::QL)), kmaj(TA(L::X)), 64, true);
            }
            mma_commit(cs.bar);
        }
        chunk_scalars<EX>(s, TP(L::X), xl, p, bh, t0, nr);
        if (tid == 0) bulk_store(ws + kWsSC * kWsMat, base + L::SCAL, kScal16);
        ok = cs.wait();
        float* AT = reinterpret_cast<float*>(sm + L::AT);
        if (ok) {
            float v[32];
            tld32(tq + c0, v);
            {  // rows 0-63: P_ij = eta_j e^{L_i - L_j} Sc_ij (j <= i); rows 64-127: A_ij = eta_j e^{Lx_i - L_j} G_ij
               // (j < i)
                const int side = ln >> 6, i = ln & 63, lim = i + 1 - side;
                const float base = side ? s.Lx[i] : s.L[i];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = c0 + e;
                    v[e] = j < lim ? s.eta[j] * __expf(fminf(base - s.L[j], 0.f)) * v[e] : 0.f;
                }
            }
            if (ln < 64) {  // diag(e^Lx) X row i
                const int i = ln;
                const float di = s.eLx[i];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[8];
                    row8<EX>(TP(L::X), xl, sw128(i, c0 + 8 * q), x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] *= di;
                    st8_hilo(TP(L::DXH), TP(L::DXL), sw128(i, c0 + 8 * q), x);
                }
            } else {  // A row f (fp32, for the inverse), then X^T diag(w) row f in its place
                const int f = ln - 64;
                float4* dst = reinterpret_cast<float4*>(AT + f * kAS + c0);
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) dst[k4] = make_float4(v[4 * k4], v[4 * k4 + 1], v[4 * k4 + 2], v[4 * k4 + 3]);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = elem<EX>(TP(L::X), xl, sw128(c0 + e, f)) * s.w[c0 + e];
            }
            tst_a32(tq + 64, tq + 96, hf, v);  // [P; X^T diag(w)]: E's A operand (columns 64-127)
            cs.publish();
            invert128(AT, reinterpret_cast<float*>(TP(L::TH)));
            {  // T to its hi / lo tiles
                const int r = tid >> 2, cq = 16 * (tid & 3);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = AT[r * kAS + cq + 8 * q + e];
                    st8_hilo(TP(L::TH), TP(L::TL), sw128(r, cq + 8 * q), x);
                }
            }
            cs.publish();
            if (tid == 0) {  // the T tiles to the workspace as they are; E = [P; X^T diag(w)] T into columns 128-191
                bulk_store(ws + kWsT * kWsMat, TA(L::TH), 2 * kTile);
                tc_fence_after();
                mma64(tmem + 128, tmem_a(tmem + 64), mnmaj(TA(L::TH)), 64, false);
                mma64(tmem + 128, tmem_a(tmem + 64), mnmaj(TA(L::TL)), 64, true);
                mma64(tmem + 128, tmem_a(tmem + 96), mnmaj(TA(L::TH)), 64, true);
                mma_commit(cs.bar);
            }
            ok = cs.wait();
        }
        if (ok) {
            {  // E as the next A operand
                float v[32];
                tld32(tq + 128 + c0, v);
                tst_a32(tq + 64, tq + 96, hf, v);
            }
            cs.publish();
            if (tid == 0) {  // E [diag(e^Lx) X | Y] into columns 128-255
                tc_fence_after();
                const Opd bh = mnmaj(TA(L::DXH), (uint32_t)((L::YH - L::DXH) * kTile));
                mma64(tmem + 128, tmem_a(tmem + 64), bh, 128, false);
                if constexpr (EX)
                    mma64(tmem + 128, tmem_a(tmem + 64), mnmaj(TA(L::DXL)), 64, true);
                else
                    mma64(tmem + 128, tmem_a(tmem + 64), mnmaj(TA(L::DXL), (uint32_t)((L::YL - L::DXL) * kTile)), 128, true);
                mma64(tmem + 128, tmem_a(tmem + 96), bh, 128, true);
                mma_commit(cs.bar);
            }
            ok = cs.wait();
        }
        if (ok) {
            if (ln < 64) {  // Ao row i = e^{L_i} q_i - (P T diag(e^Lx) X)_i as hi / lo tiles
                const int i = ln;
                const float ei = s.eL[i];
                const uint8_t* ql = EX ? nullptr : TP(L::QL);
                float v[32];
                tld32(tq + 128 + c0, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[8];
                    row8<EX>(TP(L::Q), ql, sw128(i, c0 + 8 * q), x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = fmaf(ei, x[e], -v[8 * q + e]);
                    st8_hilo(TP(L::AOH), TP(L::AOL), sw128(i, c0 + 8 * q), x);
                }
            } else {  // M row f = e^{L_C} e_f - K_f as hi / lo tiles, U row f: staged in slots read no more
                const int f = ln - 64;
                const float gC = s.eLC;
                float v[32];
                tld32(tq + 128 + c0, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = (c0 + e == f ? gC : 0.f) - v[e];
#pragma unroll
                for (int q = 0; q < 4; ++q) st8_hilo(TP(L::DXL), TP(L::X), sw128(f, c0 + 8 * q), v + 8 * q);
                tld32(tq + 192 + c0, v);
                store32(reinterpret_cast<float*>(TP(L::DXH)) + f * kD + c0, v);  // DXH, YH: 16 KB
            }
            cs.publish();
            if (tid == 0) {  // M and U to the workspace; V = Ao^T dO into columns 0-63
                bulk_store(ws + kWsM * kWsMat, TA(L::DXL), kTile);
                bulk_store(ws + kWsM * kWsMat + kTile / 4, TA(L::X), kTile);
                bulk_store(ws + kWsU * kWsMat, TA(L::DXH), 2 * kTile);
                tc_fence_after();
                mma64(tmem, mnmaj(TA(L::AOH)), mnmaj(TA(L::DO)), 64, false);
                mma64(tmem, mnmaj(TA(L::AOL)), mnmaj(TA(L::DO)), 64, true);
                if constexpr (!EX) mma64(tmem, mnmaj(TA(L::AOH)), mnmaj(TA(L::DOL)), 64, true);
                mma_commit(cs.bar);
            }
            ok = cs.wait();
        }
        if (ok) {  // V through the Ao slots (read no more) to the workspace
            if (ln < 64) {
                float v[32];
                tld32(tq + c0, v);
                store32(reinterpret_cast<float*>(TP(L::AOH)) + ln * kD + c0, v);
            }
            fence_async_smem();
            __syncthreads();
            if (tid == 0) bulk_store(ws + kWsV * kWsMat, TA(L::AOH), 2 * kTile);
        }
    } else {
        chunk_scalars<EX>(s, TP(L::X), xl, p, bh, t0, nr);
        if (tid == 0) bulk_store(ws + kWsSC * kWsMat, base + L::SCAL, kScal16);
        if (ln < 64) {  // diag(w) X and diag(e^L) dO, row j, as hi / lo tiles
            const int j = ln;
            const float wj = s.w[j], ej = s.eL[j];
            const uint8_t* dl = EX ? nullptr : TP(L::DOL);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t off = sw128(j, c0 + 8 * q);
                float x[8], d[8];
                row8<EX>(TP(L::X), xl, off, x);
                row8<EX>(TP(L::DO), dl, off, d);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    x[e] *= wj;
                    d[e] *= ej;
                }
                st8_hilo(TP(L::WXH), TP(L::WXL), off, x);
                st8_hilo(TP(L::EDH), TP(L::EDL), off, d);
            }
        }
        cs.publish();
        if (tid == 0) {  // [U, . ; ., V] = [(diag(w) X)^T ; Q^T] [Y | diag(e^L) dO] into columns 0-127
            tc_fence_after();
            const Opd ah = mnmaj(TA(L::WXH), (uint32_t)((L::Q - L::WXH) * kTile));
            const Opd bh = mnmaj(TA(L::YH), (uint32_t)((L::EDH - L::YH) * kTile));
            mma64(tmem, ah, bh, 128, false);
            if constexpr (EX) {
                mma64(tmem + 64, ah, mnmaj(TA(L::EDL)), 64, true);
                mma64(tmem, mnmaj(TA(L::WXL)), mnmaj(TA(L::YH)), 64, true);
            } else {
                mma64(tmem, ah, mnmaj(TA(L::YL), (uint32_t)((L::EDL - L::YL) * kTile)), 128, true);
                mma64(tmem, mnmaj(TA(L::WXL), (uint32_t)((L::QL - L::WXL) * kTile)), bh, 128, true);
            }
            mma_commit(cs.bar);
        }
        ok = cs.wait();
        if (ok) {  // U (slots 0, 1), V (slots 2, 3) and the tiles of M = e^{L_C} I (slots 4, 5), then out
            const int f = ln & 63;
            float v[32];
            tld32(tq + (ln < 64 ? 0 : 64) + c0, v);
            store32(reinterpret_cast<float*>(TP(ln < 64 ? 0 : 2)) + f * kD + c0, v);
            if (ln < 64) {
                float m[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) m[e] = c0 + e == f ? s.eLC : 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) st8_hilo(TP(4), TP(5), sw128(f, c0 + 8 * q), m + 8 * q);
            }
            fence_async_smem();
            __syncthreads();
            if (tid == 0) {
                bulk_store(ws + kWsU * kWsMat, TA(0), 2 * kTile);
                bulk_store(ws + kWsV * kWsMat, TA(2), 2 * kTile);
                bulk_store(ws + kWsM * kWsMat, TA(4), 2 * kTile);
            }
        }
    }
    if (tid == 0) bulk_wait_all();  // the bulk copies have read their sources before the CTA ends
    cs.finish(tmem, L::COLS);
}

// --------------------------------------------------------------------------------------------------
// falcon_bwd_grad: every input gradient of one chunk from S_n, dS_{n+1} and T. Falcon-1, as products:
//   [X S | X dS'] and [Sc; G] = [Q; X] X^T; Z = Y - diag(e^Lx) X S and P from them;
//   R = T Z and P^T dO, so dR = P^T dO + diag(w) X dS'; dZ = T^T dR (= dV);
//   [dO; dZ] [R^T | S^T] = [dP, dO S^T ; -dA, dZ S^T]; dSc and dG from dP and dA;
//   [dSc; dG] X, dSc^T Q + dG^T X and R dS'^T; then
//   dQ = diag(e^L) dO S^T + dSc X,
//   dX = dSc^T Q + (dG + dG^T) X - diag(e^Lx) dZ S^T + diag(w) R dS'^T + 2 dden x
// and the scalar gradients (eta, the log prefixes, the clamp, beta, lambda). Falcon-1A: R = Y, no
// T, Z, dZ, dA. TMEM columns: [0, 128) X S | X dS' -> R -> dZ -> [dP | dO S^T ; -dA | dZ S^T] ->
// R dS'^T; [128, 192) [Sc; G] -> dSc^T Q + dG^T X; [192, 256) P^T dO -> the [dO; dZ] operand ->
// [dSc; dG] X. S_n, dS_{n+1} and T arrive as bf16 hi / lo tiles from the workspace.
template <typename Tin, bool IP>
__global__ void __launch_bounds__(kCT, sizeof(Tin) == 2 ? 2 : 1) falcon_bwd_grad(const BParams p) {
    constexpr bool EX = sizeof(Tin) == 2;
    using L = GradLay<EX, IP>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw), base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    auto TP = [&](int slot) { return sm + slot * kTile; };
    auto TA = [&](int slot) { return base + (uint32_t)(slot * kTile); };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, ln = tid & 127, hf = tid >> 7;
    const int c0 = 32 * hf;  // this thread's columns of its lane's row
    Scal& s = *reinterpret_cast<Scal*>(sm + L::SCAL);
    float* deta = reinterpret_cast<float*>(sm + L::ACC);
    float* dL = deta + kC;
    float* dLx = dL + kC;
    float* dw = dLx + kC;
    float* c2 = dw + kC;
    float* red = c2 + kC;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BAR + 16);
    ChunkSync cs{base + L::BAR, 0u};
    const long long bh = p.bh0 + blockIdx.x / p.N, nck = blockIdx.x % p.N, t0 = nck * kC;
    const int nr = (int)min((long long)kC, p.T - t0);
    const uint8_t* wsb = reinterpret_cast<const uint8_t*>(p.ws + (bh * p.N + nck) * kWsChunk);
    const uint8_t* xl = EX ? nullptr : TP(L::XL);
    const uint8_t* ql = EX ? nullptr : TP(L::QL);

    if (tid == 0) {
        mbar_init(cs.bar, 1);
        mbar_init(cs.bar + 8, 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), 256);
    {
        const int yh = IP ? L::PRH : L::YZ, yl = IP ? L::PRL : L::ZL;
        const int hi[4] = {L::Q * kTile, L::X * kTile, yh * kTile, L::DO * kTile};
        const int lo[4] = {L::QL * kTile, L::XL * kTile, yl * kTile, L::DOL * kTile};
        load_chunk<Tin>(p, sm, base, hi, lo, bh, t0, nr);
        // S_n, dS_{n+1} (and T): their hi and lo tiles as stored, byte for byte
        constexpr int NM = IP ? 2 : 3;
        const int src[3] = {kWsS, kWsDS, kWsT};
        const int dst[3][2] = {{L::SH, L::SL}, {L::DSH, L::DSL}, {L::TH, L::TL}};
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int u = 0; u < 512 / kCT; ++u) {
                    const int e = tid + kCT * u;
                    cp_async16z(TA(dst[m][h]) + 16 * e, wsb + (size_t)src[m] * kWsMat * 4 + h * kTile + 16 * e, 16u);
                }
        if (tid < kScal16 / 16)  // the chunk's scalars as the prep kernel computed them
            cp_async16z(base + L::SCAL + 16 * tid, wsb + (size_t)kWsSC * kWsMat * 4 + 16 * tid, 16u);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (tid < kC) {
        deta[tid] = 0.f;
        dL[tid] = 0.f;
        dLx[tid] = 0.f;
        dw[tid] = 0.f;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    cs.publish();
    tc_fence_after();
    const uint32_t tmem = *tslot, tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    bool ok = true;

    if (tid == 0) {
        tc_fence_after();
        // A = [Q; X]: the rows of X land in lanes 64-127, beside the rows of G
        if constexpr (!IP) {  // [X S | X dS'] into columns 0-127
            const Opd bh = mnmaj(TA(L::SH), (uint32_t)((L::DSH - L::SH) * kTile));
            mma64(tmem, kmaj(TA(L::Q)), bh, 128, false);
            mma64(tmem, kmaj(TA(L::Q)), mnmaj(TA(L::SL), (uint32_t)((L::DSL - L::SL) * kTile)), 128, true);
            if constexpr (!EX) mma64(tmem, kmaj(TA(L::QL)), bh, 128, true);
        } else {  // X dS' into columns 64-127
            mma64(tmem + 64, kmaj(TA(L::Q)), mnmaj(TA(L::DSH)), 64, false);
            mma64(tmem + 64, kmaj(TA(L::Q)), mnmaj(TA(L::DSL)), 64, true);
            if constexpr (!EX) mma64(tmem + 64, kmaj(TA(L::QL)), mnmaj(TA(L::DSH)), 64, true);
        }
        mma64(tmem + 128, kmaj(TA(L::Q)), kmaj(TA(L::X)), 64, false);  // [Sc; G]
        if constexpr (!EX) {
            mma64(tmem + 128, kmaj(TA(L::Q)), kmaj(TA(L::XL)), 64, true);
            mma64(tmem + 128, kmaj(TA(L::QL)), kmaj(TA(L::X)), 64, true);
        }
        mma_commit(cs.bar);
    }
    {  // <dS_{n+1}, S_n> per warp, from the tiles, while the products run
        const int r = tid >> 2, cq = 16 * (tid & 3);
        float dot = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float a[8], b[8];
            row8<false>(TP(L::SH), TP(L::SL), sw128(r, cq + 8 * q), a);
            row8<false>(TP(L::DSH), TP(L::DSL), sw128(r, cq + 8 * q), b);
#pragma unroll
            for (int e = 0; e < 8; ++e) dot = fmaf(a[e], b[e], dot);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) red[warp] = dot;
    }
    ok = cs.wait();

    // ---- P (rows 0-63 of [Sc; G]) and, beside it, Z (Falcon-1; from X S in lanes 64-127): row i, columns c0 ..
    if (ok) {
        if (ln >= 64 && !IP) {
            const int i = ln - 64;
            const float di = s.eLx[i];
            float v[32];
            tld32(tq + c0, v);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t off = sw128(i, c0 + 8 * q);
                float y[8];
                row8<EX>(TP(L::YZ), TP(L::ZL), off, y);
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = fmaf(-di, v[8 * q + e], y[e]);
                st8_hilo(TP(L::YZ), TP(L::ZL), off, y);
            }
        }
        if (ln < 64) {
            const int i = ln;
            float v[32];
            const int ph = IP ? L::YZ : L::PRH, pl = IP ? L::ZL : L::PRL;
            const float li = s.L[i];
            tld32(tq + 128 + c0, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int j = c0 + e;
                v[e] = j <= i ? s.eta[j] * __expf(fminf(li - s.L[j], 0.f)) * v[e] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) st8_hilo(TP(ph), TP(pl), sw128(i, c0 + 8 * q), v + 8 * q);
        }
        cs.publish();
        if (tid == 0) {
            tc_fence_after();
            // both into lanes 64-127 (the A operands start one slot early: their first halves are unused)
            if constexpr (!IP) {  // R = T Z into columns 0-63
                mma64(tmem, kmaj(TA(L::SL)), mnmaj(TA(L::YZ)), 64, false);
                mma64(tmem, kmaj(TA(L::SL)), mnmaj(TA(L::ZL)), 64, true);
                mma64(tmem, kmaj(TA(L::TH)), mnmaj(TA(L::YZ)), 64, true);
            }
            const int ph = IP ? L::YZ : L::PRH, pl = IP ? L::ZL : L::PRL;  // P^T dO into columns 192-255
            mma64(tmem + 192, mnmaj(TA(ph - 1)), mnmaj(TA(L::DO)), 64, false);
            mma64(tmem + 192, mnmaj(TA(pl - 1)), mnmaj(TA(L::DO)), 64, true);
            if constexpr (!EX) mma64(tmem + 192, mnmaj(TA(ph - 1)), mnmaj(TA(L::DOL)), 64, true);
            mma_commit(cs.bar);
        }
        ok = cs.wait();
    }

    // ---- R (Falcon-1) to tiles; dR = P^T dO + diag(w) X dS' (Falcon-1: tiles; 1A: dV); dw: lanes 64-127
    if (ok) {
        if (ln >= 64) {
            const int i = ln - 64;
            const float wi = s.w[i];
            float xd[32], r[32], d[32];
            tld32(tq + 64 + c0, xd);
            tld32(tq + 192 + c0, d);
            if constexpr (!IP) {
                tld32(tq + c0, r);
#pragma unroll
                for (int q = 0; q < 4; ++q) st8_hilo(TP(L::PRH), TP(L::PRL), sw128(i, c0 + 8 * q), r + 8 * q);
            } else {
                const uint8_t* yl = EX ? nullptr : TP(L::PRL);
#pragma unroll
                for (int q = 0; q < 4; ++q) row8<EX>(TP(L::PRH), yl, sw128(i, c0 + 8 * q), r + 8 * q);
            }
            float dwa = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                dwa = fmaf(xd[e], r[e], dwa);
                d[e] = fmaf(wi, xd[e], d[e]);
            }
            atomicAdd(&dw[i], dwa);
            if constexpr (!IP) {
#pragma unroll
                for (int q = 0; q < 4; ++q) st8_hilo(TP(L::YZ), TP(L::ZL), sw128(i, c0 + 8 * q), d + 8 * q);
            } else {  // dV, staged in the T slots (unused here)
                store32(reinterpret_cast<float*>(TP(L::TH)) + i * kD + c0, d);
            }
        }
        if constexpr (!IP) {
            cs.publish();
            if (tid == 0) {  // dZ = T^T dR into columns 0-63, rows 64-127 (A: [any; T^T], MN-major)
                tc_fence_after();
                const Opd ah = mnmaj(TA(L::SL), (uint32_t)((L::TH - L::SL) * kTile));
                const Opd al = mnmaj(TA(L::TH), (uint32_t)((L::TL - L::TH) * kTile));
                mma64(tmem, ah, mnmaj(TA(L::YZ)), 64, false);
                mma64(tmem, ah, mnmaj(TA(L::ZL)), 64, true);
                mma64(tmem, al, mnmaj(TA(L::YZ)), 64, true);
                mma_commit(cs.bar);
            }
            ok = cs.wait();
        }
    }

    // ---- the A operand [dO; dZ] (columns 192-255: hi, lo); dV = dZ
    if (ok) {
        float v[32];
        if (ln < 64) {
            const uint8_t* dl = EX ? nullptr : TP(L::DOL);
#pragma unroll
            for (int q = 0; q < 4; ++q) row8<EX>(TP(L::DO), dl, sw128(ln, c0 + 8 * q), v + 8 * q);
            tst_a32(tq + 192, tq + 224, hf, v);
        } else if (!IP) {  // dV = dZ, staged in the dR slots (read no more)
            const int i = ln - 64;
            tld32(tq + c0, v);
            store32(reinterpret_cast<float*>(TP(L::YZ)) + i * kD + c0, v);
            tst_a32(tq + 192, tq + 224, hf, v);
        }
        cs.publish();
        if (tid == 0) {  // dV out; [dO; dZ] [R^T | S^T] into columns 0-127 (B: [R; S] K-major, N = 128)
            bulk_store(p.dv + (bh * p.T + t0) * kD, TA(IP ? L::TH : L::YZ), (uint32_t)nr * kD * 4);
            tc_fence_after();
            const Opd ah = tmem_a(tmem + 192), al = tmem_a(tmem + 224);
            mma64(tmem, ah, kmaj(TA(L::PRH)), 128, false);
            if constexpr (IP && EX) {
                mma64(tmem + 64, ah, kmaj(TA(L::SL)), 64, true);
            } else {
                mma64(tmem, ah, kmaj(TA(L::PRL)), 128, true);
                mma64(tmem, al, kmaj(TA(L::PRH)), 128, true);
            }
            mma_commit(cs.bar);
            bulk_wait_read<0>();  // the next phase rewrites the slots dV was staged in
        }
        ok = cs.wait();
    }

    // ---- dP (rows 0-63) and dA (rows 64-127): the score and Gram adjoints, the scalar terms
    if (ok) {
        float d[32], g[32], cE[32], cL[32];
        tld32(tq + c0, d);
        tld32(tq + 128 + c0, g);
        // rows 0-63: dP = dO R^T (j <= i) against Sc, giving dSc; rows 64-127 (Falcon-1): -dA = dZ R^T
        // (j < i) against G, giving dG. One formula with x = dP or dA: the column terms x f g and
        // x eta_j f g, the row sum of the latter, and the adjoint x eta_j f.
        const int side = ln >> 6, i = ln & 63;
        if (!IP || side == 0) {
            const float base = side ? s.Lx[i] : s.L[i], sgn = side ? -1.f : 1.f;
            const int lim = i + 1 - side;
            float rsum = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int j = c0 + e;
                const bool on = j < lim;
                const float f = __expf(fminf(base - s.L[j], 0.f)), x = sgn * d[e], ef = s.eta[j] * f;
                cE[e] = on ? x * f * g[e] : 0.f;
                cL[e] = on ? x * ef * g[e] : 0.f;
                rsum += cL[e];
                d[e] = on ? x * ef : 0.f;
            }
            uint8_t* th = TP(side ? L::ZL : L::YZ);
            uint8_t* tl = TP(side ? L::TL : L::TH);
#pragma unroll
            for (int q = 0; q < 4; ++q) st8_hilo(th, tl, sw128(i, c0 + 8 * q), d + 8 * q);
            atomicAdd(side ? &dLx[i] : &dL[i], rsum);
            const float ce = warp_colsum32(cE);
            const float cl = warp_colsum32(cL);
            atomicAdd(&deta[c0 + lane], ce);
            atomicAdd(&dL[c0 + lane], -cl);
        }
        cs.publish();
        if (tid == 0) {
            tc_fence_after();
            // [dSc; dG] X into columns 192-255
            mma64(tmem + 192, kmaj(TA(L::YZ)), mnmaj(TA(L::X)), 64, false);
            mma64(tmem + 192, kmaj(TA(L::TH)), mnmaj(TA(L::X)), 64, true);
            if constexpr (!EX) mma64(tmem + 192, kmaj(TA(L::YZ)), mnmaj(TA(L::XL)), 64, true);
            // dSc^T Q (+ dG^T X) into columns 128-191, rows 0-63
            mma64(tmem + 128, mnmaj(TA(L::YZ)), mnmaj(TA(L::Q)), 64, false);
            mma64(tmem + 128, mnmaj(TA(L::TH)), mnmaj(TA(L::Q)), 64, true);
            if constexpr (!EX) mma64(tmem + 128, mnmaj(TA(L::YZ)), mnmaj(TA(L::QL)), 64, true);
            if constexpr (!IP) {
                mma64(tmem + 128, mnmaj(TA(L::ZL)), mnmaj(TA(L::X)), 64, true);
                mma64(tmem + 128, mnmaj(TA(L::TL)), mnmaj(TA(L::X)), 64, true);
                if constexpr (!EX) mma64(tmem + 128, mnmaj(TA(L::ZL)), mnmaj(TA(L::XL)), 64, true);
            }
            // R dS'^T into columns 0-63
            mma64(tmem, kmaj(TA(L::PRH)), kmaj(TA(L::DSH)), 64, false);
            mma64(tmem, kmaj(TA(L::PRH)), kmaj(TA(L::DSL)), 64, true);
            if constexpr (!(IP && EX)) mma64(tmem, kmaj(TA(L::PRL)), kmaj(TA(L::DSH)), 64, true);
            mma_commit(cs.bar);
        }
        ok = cs.wait();
    }

    // ---- dQ; the two halves of dX to shared memory; the scalar gradients; dK
    if (ok) {
        float* EA = reinterpret_cast<float*>(TP(L::DSH));  // rows 0-63: dSc^T Q + dG^T X + diag(w) R dS'^T
        float* EB = reinterpret_cast<float*>(TP(L::YZ));   // rows 64-127: dG X - diag(e^Lx) dZ S^T
        // rows 0-63: dQ = e^{L_i} dO S^T + dSc X (staged in the T slots), dL_i += e^{L_i} q_i . (dO S^T)_i;
        // rows 64-127: dG X - e^{Lx_i} dZ S^T (half of dX), dLx_i -= e^{Lx_i} x_i . (dZ S^T)_i
        const int side = ln >> 6, i = ln & 63;
        if (!IP || side == 0) {
            const float sc = side ? -s.eLx[i] : s.eL[i];
            float a[32], b[32], rv[32];
            tld32(tq + 64 + c0, a);   // dO S^T or dZ S^T
            tld32(tq + 192 + c0, b);  // dSc X or dG X
            const uint8_t* rh = TP(side ? L::X : L::Q);
            const uint8_t* rl = side ? xl : ql;
#pragma unroll
            for (int q = 0; q < 4; ++q) row8<EX>(rh, rl, sw128(i, c0 + 8 * q), rv + 8 * q);
            float rsum = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                rsum = fmaf(rv[e], a[e], rsum);
                a[e] = fmaf(sc, a[e], b[e]);
            }
            float4* dst = reinterpret_cast<float4*>(side ? EB : reinterpret_cast<float*>(TP(L::TH))) + 16 * i;
            const int sw = side ? (i & 15) : 0;  // EB's rows are swizzled; dQ's staging is the plain image
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[(8 * hf + q) ^ sw] = make_float4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
            atomicAdd(side ? &dLx[i] : &dL[i], sc * rsum);
            if (side == 0) {  // EA: dSc^T Q + dG^T X + diag(w) R dS'^T
                const float wi = s.w[i];
                tld32(tq + 128 + c0, a);
                tld32(tq + c0, b);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    reinterpret_cast<float4*>(EA + i * kD)[(8 * hf + q) ^ (i & 15)] =
                        make_float4(fmaf(wi, b[4 * q], a[4 * q]), fmaf(wi, b[4 * q + 1], a[4 * q + 1]),
                                    fmaf(wi, b[4 * q + 2], a[4 * q + 2]), fmaf(wi, b[4 * q + 3], a[4 * q + 3]));
            }
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) bulk_store(p.dq + (bh * p.T + t0) * kD, TA(L::TH), (uint32_t)nr * kD * 4);
        // scalars: d eta and dL from w and the chunk-end decay; d log gamma; the clamp; eta = beta / den
        if (tid < 32) {
            const int l = tid;
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
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dwsum += __shfl_xor_sync(0xffffffffu, dwsum, o);
            float dss = 0.f;
#pragma unroll
            for (int u = 0; u < kCT / 32; ++u) dss += red[u];
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
        // dX row r = EA + EB + 2 dden x, 16 columns per thread; row r is dk of token t0 + r - 1 (row 0 of
        // the call: the tail key)
        {
            const int r = tid >> 2, cq = 16 * (tid & 3);
            if (r < nr) {
                const long long t = t0 + r - 1;
                float* dst = t >= 0 ? p.dk + (bh * p.T + t) * kD + cq : (p.dtail ? p.dtail + bh * kD + cq : nullptr);
                if (dst) {
                    const float cr = c2[r];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float x[8];
                        row8<EX>(TP(L::X), xl, sw128(r, cq + 8 * q), x);
#pragma unroll
                        for (int hq = 0; hq < 2; ++hq) {
                            const int f4 = ((cq >> 2) + 2 * q + hq) ^ (r & 15);
                            float4 a = reinterpret_cast<const float4*>(EA + r * kD)[f4];
                            if constexpr (!IP) {
                                const float4 b = reinterpret_cast<const float4*>(EB + r * kD)[f4];
                                a.x += b.x;
                                a.y += b.y;
                                a.z += b.z;
                                a.w += b.w;
                            }
                            reinterpret_cast<float4*>(dst)[2 * q + hq] =
                                make_float4(fmaf(cr, x[4 * hq], a.x), fmaf(cr, x[4 * hq + 1], a.y),
                                            fmaf(cr, x[4 * hq + 2], a.z), fmaf(cr, x[4 * hq + 3], a.w));
                        }
                    }
                }
            }
            if (t0 + nr == p.T && tid < kD / 4)  // the last key feeds only the next call's tail
                reinterpret_cast<float4*>(p.dk + (bh * p.T + p.T - 1) * kD)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (tid == 0) bulk_wait_all();  // the bulk copies have read their sources before the CTA ends
    cs.finish(tmem, 256);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// falcon_bwd_chain: two CTAs of 128 threads per sequence, one per state scan, on the tensor cores:
// the forward scan S_{n+1} = M_n S_n + U_n and the reverse scan dS_n = M_n^T dS_{n+1} + V_n need
// nothing from each other. The carried matrix (S forward, dS backward) is kept transposed in tensor
// memory, lane c = column c (lanes 64-127 zero), as the bf16 A operand of one product per step,
// D = X^T B with B = M_n^T (forward: D = (M_n S)^T; M_n's tile read K-major) or B = M_n (backward:
// D = (M_n^T dS)^T; the same tile read MN-major). Both operands are split into bf16 hi and lo parts and
// D = A_hi B_hi + A_hi B_lo + A_lo B_hi (fp32 sums). M_n's hi and lo tiles, as the prep kernel stores
// them, arrive by one bulk copy two steps ahead into one of two buffers, U_n / V_n by 16-byte
// asynchronous copies one step ahead, added in registers; while the product runs each thread stores
// its column of S_n / dS_{n+1} for the gradient kernel. Every wait is bounded: on timeout the CTA raises
// the device flag, drains what it issued and frees its tensor memory.
constexpr int kChainT = 128;
constexpr uint32_t kCAH = 0, kCAL = 32, kCD = 64;  // TMEM columns: carried hi, lo (bf16 pairs), product
constexpr long long kTcTimeout = 4000000000LL;     // ~2 s
namespace chl {
constexpr int B = 0;                 // two buffers for M_n: hi tile, lo tile
constexpr int BSZ = 2 * kTile;
constexpr int OFS = B + 2 * BSZ;     // two offset buffers (U_n or V_n), [64][64] fp32
constexpr int BAR = OFS + 32768;
constexpr int BYTES = BAR + 64;
constexpr int ALLOC = BYTES + 1024;
}  // namespace chl

__device__ bool chain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    int spins = 0;
    while (!mbar_try(bar, parity)) {
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
    for (int q = 0; q < 2; ++q) {
        uint32_t h[16], l[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) split2(x[32 * q + 2 * e], x[32 * q + 2 * e + 1], h[e], l[e]);
        tmem_st16(tq + kCAH + 16 * q, h);
        tmem_st16(tq + kCAL + 16 * q, l);
    }
}

__global__ void __launch_bounds__(kChainT, 1) falcon_bwd_chain(const BParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw), base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t bar_full0 = base + chl::BAR, bar_mma = bar_full0 + 16, bar_drain = bar_full0 + 24;  // full: two
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + chl::BAR + 32);
    const long long bh = p.bh0 + (blockIdx.x >> 1), N = p.N;
    const bool bwd = (blockIdx.x & 1) != 0;  // this CTA's scan
    const long long k0 = bwd ? N : 0, k1 = k0 + N;  // its steps of the 2 N
    if (tid == 0) {
        mbar_init(bar_full0, 1);
        mbar_init(bar_full0 + 8, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_drain, 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot, tq = tmem + ((uint32_t)(32 * warp) << 16);
    const int c = tid;            // carried column = TMEM lane
    const bool live = c < kD;     // lanes 64-127 hold zeros
    float* const wsq = p.ws + bh * N * kWsChunk;

    // step k: chunk n, matrix and offset of the pass
    auto chunk_of = [&](long long k) { return k < N ? k : 2 * N - 1 - k; };
    auto issue_b = [&](long long k) {  // thread 0: M_n's tiles of step k into buffer (k - k0) & 1
        const uint32_t bar = bar_full0 + 8 * (uint32_t)((k - k0) & 1);
        mbar_expect_tx(bar, (uint32_t)chl::BSZ);
        bulk_load(base + chl::B + (uint32_t)((k - k0) & 1) * chl::BSZ, wsq + chunk_of(k) * kWsChunk + kWsM * kWsMat,
                  (uint32_t)chl::BSZ, bar);
    };
    auto issue_ofs = [&](long long k) {  // every thread: U_n (forward) or V_n (backward) into buffer k & 1
        if (k < k1) {
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
    {
        const float* src = bwd ? p.dS_final : p.S0;
#pragma unroll
        for (int r = 0; r < kD; ++r) s[r] = (live && src) ? src[(bh * kD + r) * kD + c] : 0.f;
        chain_put(tq, s);
        tmem_wait_st();
    }
    if (tid == 0) {
        for (long long k = k0; k < k1 && k < k0 + 2; ++k) issue_b(k);
    }
    long long issued = k1 < k0 + 2 ? k1 : k0 + 2;  // steps whose M has been requested: [k0, issued)
    issue_ofs(k0);
    tc_fence_before();
    __syncthreads();
    bool ok = true;
    long long waited = k0;  // steps whose M has landed: [k0, waited)
    const uint32_t id = idesc_bf16(128, kD, false, bwd);
    for (long long k = k0; k < k1; ++k) {
        const long long n = chunk_of(k), i = k - k0;
        const uint32_t bb = base + chl::B + (uint32_t)(i & 1) * chl::BSZ;
        issue_ofs(k + 1);  // its buffer was last read before the previous step's closing barrier
        bool bad = false;
        if (tid == 0) {
            bad = !chain_wait(bar_full0 + 8 * (uint32_t)(i & 1), (uint32_t)((i >> 1) & 1));
            if (!bad) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t dh = bwd ? desc_mn(bb + 2048 * ks, kTile) : desc_k(bb + 32 * ks);
                    const uint64_t dl = bwd ? desc_mn(bb + kTile + 2048 * ks, kTile) : desc_k(bb + kTile + 32 * ks);
                    mma_bf16_ta(tmem + kCD, tmem + kCAH + 8 * ks, dh, id, ks > 0);
                    mma_bf16_ta(tmem + kCD, tmem + kCAH + 8 * ks, dl, id, 1);
                    mma_bf16_ta(tmem + kCD, tmem + kCAL + 8 * ks, dh, id, 1);
                }
                mma_commit(bar_mma);
            }
        }
        if (live) {  // while the product runs: S_n (forward) / dS_{n+1} (backward) for the gradient kernel,
            // this thread's column of the bf16 hi and lo tiles the gradient kernel copies in as they are
            uint8_t* dst = reinterpret_cast<uint8_t*>(wsq + n * kWsChunk + (bwd ? kWsDS : kWsS) * kWsMat);
#pragma unroll
            for (int r = 0; r < kD; ++r) {
                const __nv_bfloat16 h = __float2bfloat16_rn(s[r]);
                const uint32_t off = sw128(r, c);
                *reinterpret_cast<__nv_bfloat16*>(dst + off) = h;
                *reinterpret_cast<__nv_bfloat16*>(dst + kTile + off) = __float2bfloat16_rn(s[r] - __bfloat162float(h));
            }
        }
        asm volatile("cp.async.wait_group 1;" ::: "memory");  // this step's offsets (the next step's may fly)
        if (tid == 0 && !bad) {
            bad = !chain_wait(bar_mma, (uint32_t)(i & 1));
            if (!bad && k + 2 < k1) issue_b(k + 2);  // the product has read the buffer
        }
        if (named_bar_or(1, kChainT, bad)) {
            ok = false;
            break;
        }
        waited = k + 1;
        if (k + 2 < k1) issued = k + 3;
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
        if (k + 1 < k1) chain_put(tq, s);
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
    }
    if (ok && bwd && p.dS0 && live) {
#pragma unroll
        for (int r = 0; r < kD; ++r) p.dS0[(bh * kD + r) * kD + c] = s[r];
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (tid == 0) {  // copies still in flight after an early exit
        for (long long k = waited; k < issued; ++k) {
            const long long i = k - k0;
            mbar_wait_bounded(bar_full0 + 8 * (uint32_t)(i & 1), (uint32_t)((i >> 1) & 1), kTcTimeout);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        mma_commit(bar_drain);
        mbar_wait_bounded(bar_drain, 0, kTcTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// Streams and events of a split call (created once per device; a mutex orders the calls that use them).
constexpr int kGroups = 4;
struct BwdStreams {
    bool ready = false;
    cudaStream_t group[kGroups], chain[kGroups];
    cudaEvent_t fork, prep[kGroups], chained[kGroups], done[kGroups];
};
std::mutex g_bwd_mu;
BwdStreams g_bwd_streams[64];

bool bwd_streams(BwdStreams*& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    BwdStreams& b = g_bwd_streams[dev];
    if (!b.ready) {
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return false;
        bool ok = cudaEventCreateWithFlags(&b.fork, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kGroups; ++i)
            ok = cudaStreamCreateWithPriority(&b.group[i], cudaStreamNonBlocking, least) == cudaSuccess &&
                 cudaStreamCreateWithPriority(&b.chain[i], cudaStreamNonBlocking, greatest) == cudaSuccess &&
                 cudaEventCreateWithFlags(&b.prep[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&b.chained[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&b.done[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) return false;
        b.ready = true;
    }
    out = &b;
    return true;
}

// Each kernel over the sequences of p, on stream st.
template <typename Tin, bool IP>
bool enqueue_prep(const BParams& p, cudaStream_t st) {
    constexpr bool EX = sizeof(Tin) == 2;
    constexpr int prep_smem = PrepLay<EX, IP>::ALLOC;
    cudaFuncSetAttribute(falcon_bwd_prep<Tin, IP>, cudaFuncAttributeMaxDynamicSharedMemorySize, prep_smem);
    falcon_bwd_prep<Tin, IP><<<(unsigned)(p.BH * p.N), kCT, prep_smem, st>>>(p);
    return cudaGetLastError() == cudaSuccess;
}
bool enqueue_chain(const BParams& p, cudaStream_t st) {
    cudaFuncSetAttribute(falcon_bwd_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, chl::ALLOC);
    falcon_bwd_chain<<<(unsigned)(2 * p.BH), kChainT, chl::ALLOC, st>>>(p);
    return cudaGetLastError() == cudaSuccess;
}
template <typename Tin, bool IP>
bool enqueue_grad(const BParams& p, cudaStream_t st) {
    constexpr bool EX = sizeof(Tin) == 2;
    constexpr int grad_smem = GradLay<EX, IP>::ALLOC;
    cudaFuncSetAttribute(falcon_bwd_grad<Tin, IP>, cudaFuncAttributeMaxDynamicSharedMemorySize, grad_smem);
    falcon_bwd_grad<Tin, IP><<<(unsigned)(p.BH * p.N), kCT, grad_smem, st>>>(p);
    return cudaGetLastError() == cudaSuccess;
}

// One call: with at least 4 sequences, 2 (or with 16 and more, 4) groups of them on streams of their
// own, each group's chain on a high-priority stream, so that a chain launch (a few CTAs per SM) runs
// beside the other groups' chunk kernels; the caller's stream waits for every group.
template <typename Tin, bool IP>
int launch_typed(const BParams& p, cudaStream_t st) {
    if (p.BH < 4) return enqueue_prep<Tin, IP>(p, st) && enqueue_chain(p, st) && enqueue_grad<Tin, IP>(p, st) ? 0 : 4;
    std::lock_guard<std::mutex> lock(g_bwd_mu);
    BwdStreams* b = nullptr;
    if (!bwd_streams(b)) return 4;
    const int G = p.BH >= 16 ? kGroups : 2;
    BParams h[kGroups];
    for (int i = 0; i < G; ++i) {
        h[i] = p;
        h[i].bh0 = p.bh0 + p.BH * i / G;
        h[i].BH = p.BH * (i + 1) / G - p.BH * i / G;
    }
    bool ok = cudaEventRecord(b->fork, st) == cudaSuccess;
    for (int i = 0; ok && i < G; ++i)
        ok = cudaStreamWaitEvent(b->group[i], b->fork, 0) == cudaSuccess && enqueue_prep<Tin, IP>(h[i], b->group[i]) &&
             cudaEventRecord(b->prep[i], b->group[i]) == cudaSuccess;
    for (int i = 0; ok && i < G; ++i)
        ok = cudaStreamWaitEvent(b->chain[i], b->prep[i], 0) == cudaSuccess && enqueue_chain(h[i], b->chain[i]) &&
             cudaEventRecord(b->chained[i], b->chain[i]) == cudaSuccess;
    for (int i = 0; ok && i < G; ++i)
        ok = cudaStreamWaitEvent(b->group[i], b->chained[i], 0) == cudaSuccess &&
             enqueue_grad<Tin, IP>(h[i], b->group[i]) && cudaEventRecord(b->done[i], b->group[i]) == cudaSuccess &&
             cudaStreamWaitEvent(st, b->done[i], 0) == cudaSuccess;
    return ok ? 0 : 4;
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
    p.bh0 = 0;
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
