// CUDA-core chunk-parallel Falcon forward kernel (all variants, fp32 or bf16 I/O).
//
// One CTA owns one (batch, head) sequence and a slice of `dvs` value columns (mode 0), or one chunk
// of one sequence (map mode, used by the scan path: the chunk's affine state and output maps).
// Falcon-1/1A/2/3 value columns evolve independently once the chunk operators
// are known (paperlayer summary §G.1: the shared transition acts on every
// column; Falcon-2 and Falcon-3 only change the per-token scalars or add window
// slots), so slicing the columns across CTAs is exact; each CTA rebuilds the
// key-only operators of its chunk.
//
// Per chunk of C tokens (paperlayer Figure 2 "Chunk-parallel form", §D.1, §E.2,
// §F.2, §H.3):
//   X = shifted keys (row i = k_{tau_i - 1}; the first row comes from the previous
//       chunk, the tail or the x_1 = 0 sentinel), Q, Y = V.
//   per token: eta, alpha = min(eta*lambda, 1 - eps_gamma), l = log1p(-alpha) in
//       fp32 and its prefix L reset to 0 at the chunk start (§G.1; sungsoo post).
//   G = X X^T, Sc = Q X^T.
//   A_ij = eta_j exp(L_{i-1} - L_j) G_ij (j < i), P_ij = eta_j exp(L_i - L_j) Sc_ij (j <= i)
//   Falcon-1: (I + A) R = Y - diag(exp L_{i-1}) X S     (one solve, value and
//       projected-history right-hand sides merged, §E.2, §F.2); Falcon-1A: R = Y.
//   O = diag(exp L) Q S + P R           (read after write, inclusive diagonal, §F.2)
//   S <- exp(L_C) S + X^T diag(eta_j exp(L_C - L_j)) R
// Falcon-2 uses per-column eta, L; Falcon-3 solves over (token, window slot)
// unknowns with a block-strict-lower system (§H, "tensorInv").
// Factors exp(L_a - L_b) have a >= b, so none exceeds 1; Falcon-2 forms them as exp(L_a) exp(-L_b)
// where the column's chunk decay keeps both finite, else one by one.
// With bf16 inputs (whose tiles hold exact bf16 values) G and Sc are warp-level bf16 mma.sync
// products with fp32 sums; fp32 inputs keep fp32 FMA loops throughout.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "falcon_internal.h"

namespace falcon {
namespace {

constexpr int kThreads = 256;
constexpr float kFastL = 30.f;  // Falcon-2: per-column chunk log decay above which e^{a-b} = e^{a} e^{-b}
constexpr int kMaxW = 8;

struct GParams {
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
    long long T, pos;
    int dk, dv, dvs, C, W;
    float eps, eps_gamma;
    // 0: one CTA walks all chunks of its (sequence, column slice);
    // 1 (map, dk = dv = 64): one CTA per (sequence, slice, chunk) computes the chunk's affine maps
    //   S -> M S + U (its end state) and S -> Ao S + Bo (its outputs) over the 2 dk virtual columns:
    //   the first dk those of M and Ao (state e_c, no target), the rest those of U and Bo (zero state,
    //   the targets); the results go to the chunk's workspace block.
    int mode;
    int staged;       // mode 0: the next chunk's inputs are copied ahead into shared memory
    const float* mu;  // Falcon-3, mode 1: every token's window normaliser, precomputed ([B*H][T])
    float* ws;   // per chunk (sequence-major) [M | U | S | Ao | Bo], each 64 x 64 fp32 (Ao, Bo: C rows used)
    long long N; // chunks per sequence (mode 1)
    int skip_marked;  // mode 1: leave the chunks whose block is marked finished (by the tensor-core map kernel)
    long long BH;     // sequences
    int per_cta;      // skip_marked: items per CTA (at most kThreads)
};

__device__ __forceinline__ float ldf(const float* p) { return *p; }
// Eight consecutive elements from a 16-byte aligned address, as fp32.
__device__ __forceinline__ void ld8(const float* p, float (&o)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    o[0] = a.x, o[1] = a.y, o[2] = a.z, o[3] = a.w, o[4] = b.x, o[5] = b.y, o[6] = b.z, o[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&o)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float2 f = __bfloat1622float2(h[m]);
        o[2 * m] = f.x, o[2 * m + 1] = f.y;
    }
}
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Largest eigenvalue of a small symmetric matrix, cyclic Jacobi in fp32 on an N x N matrix held in
// registers (every index a compile-time constant), until the off-diagonal mass is 1e-12 of the
// diagonal's: convergence is quadratic, so a few sweeps; the eigenvalue's error is second order in
// the off-diagonal part, far below fp32 rounding.
template <int N>
__device__ float lambda_max_fixed(float (&a)[N][N]) {
    for (int sweep = 0; sweep < 16; ++sweep) {
        float off = 0.f, dg = 0.f;
#pragma unroll
        for (int p = 0; p < N; ++p) {
            dg += a[p][p] * a[p][p];
#pragma unroll
            for (int r = p + 1; r < N; ++r) off += a[p][r] * a[p][r];
        }
        if (off <= 1e-12f * dg || off == 0.f) break;
#pragma unroll
        for (int p = 0; p < N; ++p)
#pragma unroll
            for (int r = p + 1; r < N; ++r) {
                const float apq = a[p][r];
                if (apq == 0.f) continue;
                const float th = (a[r][r] - a[p][p]) / (2.f * apq);
                const float t = (th >= 0.f ? 1.f : -1.f) / (fabsf(th) + sqrtf(th * th + 1.f));
                const float c = rsqrtf(t * t + 1.f), sn = t * c;
#pragma unroll
                for (int m = 0; m < N; ++m) {
                    const float x = a[m][p], y = a[m][r];
                    a[m][p] = c * x - sn * y;
                    a[m][r] = sn * x + c * y;
                }
#pragma unroll
                for (int m = 0; m < N; ++m) {
                    const float x = a[p][m], y = a[r][m];
                    a[p][m] = c * x - sn * y;
                    a[r][m] = sn * x + c * y;
                }
            }
    }
    float mx = a[0][0];
#pragma unroll
    for (int p = 1; p < N; ++p) mx = fmaxf(mx, a[p][p]);
    return mx;
}

// lambda_max of (1/nb) [G_{slots[x], slots[y]}] (a window's averaged Gram, PSD), zero-padded to N:
// the padding adds zero eigenvalues only.
template <int N>
__device__ float window_lambda_max(const float* G, int ld, const int* slots, int nb) {
    float a[N][N];
    const float inv = 1.f / (float)nb;
#pragma unroll
    for (int x = 0; x < N; ++x)
#pragma unroll
        for (int y = 0; y < N; ++y) a[x][y] = (x < nb && y < nb) ? G[slots[x] * ld + slots[y]] * inv : 0.f;
    return lambda_max_fixed<N>(a);
}

// d += A (16 x 16, row-major bf16) * B (16 x 8, column-major bf16), fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Two fp32 values that are exact bf16 numbers, packed (lo = first) without rounding error.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// G = X X^T (C x C) and Sc = Q X^T (C x C) from fp32 tiles (row stride xs) holding bf16 values, C a
// multiple of 16, dk a multiple of 16: each warp takes one 16-row block of one product across all
// its 8-column tiles. Fragments follow the m16n8k16 layout (g = lane / 4, t = lane % 4).
__device__ void gram_mma(const float* X, const float* Q, float* G, float* Sc, int C, int dk, int xs, int ld, int tid) {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int mbs = C / 16;
    for (int job = warp; job < 2 * mbs; job += kThreads / 32) {
        const float* A = job < mbs ? X : Q;
        float* D = job < mbs ? G : Sc;
        const int r0 = 16 * (job % mbs);
        float acc[8][4] = {};
        for (int k0 = 0; k0 < dk; k0 += 16) {
            const float* ar = A + (r0 + g) * xs + k0 + 2 * t;
            const uint32_t a0 = pack_bf16(ar[0], ar[1]), a1 = pack_bf16(ar[8 * xs], ar[8 * xs + 1]);
            const uint32_t a2 = pack_bf16(ar[8], ar[9]), a3 = pack_bf16(ar[8 * xs + 8], ar[8 * xs + 9]);
#pragma unroll
            for (int nb = 0; nb < 8; ++nb) {
                if (8 * nb >= C) break;
                const float* br = X + (8 * nb + g) * xs + k0 + 2 * t;
                mma_bf16_16816(acc[nb], a0, a1, a2, a3, pack_bf16(br[0], br[1]), pack_bf16(br[8], br[9]));
            }
        }
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            if (8 * nb >= C) break;
            float* dr = D + (r0 + g) * ld + 8 * nb + 2 * t;
            dr[0] = acc[nb][0], dr[1] = acc[nb][1];
            dr[8 * ld] = acc[nb][2], dr[8 * ld + 1] = acc[nb][3];
        }
    }
}

// out[r][c] = sum_{k < K} A(r, k) B(k, c) for r < nr, c < nc on the CUDA cores, A(r, k) = a[r * lda + k],
// B(k, c) = b[k * ldb + c] (BT: b[c * ldb + k]). Each thread takes two rows (r, r + ceil(nr / 2)) by four
// columns, so a k step costs six shared loads (two for a 16-byte-aligned row of B) for eight
// multiply-adds. Columns past nc read a valid neighbour and are not stored.
template <bool BT>
__device__ void mm_tiled(float* out, int ldo, const float* a, int lda, const float* b, int ldb, int nr, int nc, int K,
                         int tid) {
    const int half = (nr + 1) / 2, ncg = (nc + 3) / 4;
    const bool vec = !BT && (ldb % 4 == 0) && (nc % 4 == 0);
    for (int tile = tid; tile < half * ncg; tile += kThreads) {
        const int r0 = tile / ncg, cb = 4 * (tile % ncg), r1 = r0 + half;
        const bool v1 = r1 < nr;
        const float* a0 = a + r0 * lda;
        const float* a1 = a + (v1 ? r1 : r0) * lda;
        int cj[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) cj[jj] = min(cb + jj, nc - 1);
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int k = 0; k < K; ++k) {
            const float x0 = a0[k], x1 = a1[k];
            float y[4];
            if (vec) {
                const float4 v = *reinterpret_cast<const float4*>(b + k * ldb + cb);
                y[0] = v.x, y[1] = v.y, y[2] = v.z, y[3] = v.w;
            } else {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) y[jj] = BT ? b[cj[jj] * ldb + k] : b[k * ldb + cj[jj]];
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                acc0[jj] = fmaf(x0, y[jj], acc0[jj]);
                acc1[jj] = fmaf(x1, y[jj], acc1[jj]);
            }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            if (cb + jj < nc) {
                out[r0 * ldo + cb + jj] = acc0[jj];
                if (v1) out[r1 * ldo + cb + jj] = acc1[jj];
            }
    }
}

// Shared-memory carve-up (floats). NE = C + W - 1 extended pair rows.
struct Smem {
    float *X, *Q, *Y, *S, *G, *Sc, *H, *QS, *R, *A, *P;
    float *eta, *L, *Lx, *kap, *w;
    float* stg;  // mode 0: the next chunk's raw tiles (and per-column gains, ridge terms), copied ahead
};

// es: bytes per input element; staged: room for the next chunk's raw inputs (mode 0).
__host__ __device__ inline size_t smem_floats(int variant, int dk, int dvs, int C, int W, Smem* s, float* base,
                                              int es = 2, bool staged = false) {
    const int NE = C + W - 1;
    const int per_col = per_column(variant) ? dvs : 1;
    size_t off = 0;
    auto take = [&](float** dst, size_t n) {
        if (dst) *dst = base + off;
        off += (n + 3) & ~size_t(3);  // keep 16-byte alignment of every array
    };
    take(s ? &s->X : nullptr, size_t(NE) * (dk + 1));  // rows padded: the Gram reads rows across lanes
    take(s ? &s->Q : nullptr, size_t(C) * (dk + 1));
    // Y doubles as the Falcon-3 block solve's diagonal-block inverses (16 x 16 per block of 16 / W
    // tokens) when a CTA takes all 64 columns, so it is at least that large
    size_t ny = size_t(NE) * dvs;
    if (variant == kF3 && dvs == 64) {
        const int tb = 16 / W, nblk = (C + tb - 1) / tb;
        ny = ny > size_t(nblk) * 256 ? ny : size_t(nblk) * 256;
    }
    take(s ? &s->Y : nullptr, ny);
    take(s ? &s->S : nullptr, size_t(dk) * dvs);
    take(s ? &s->G : nullptr, size_t(NE) * NE);
    take(s ? &s->Sc : nullptr, size_t(C) * NE);
    take(s ? &s->H : nullptr, size_t(NE) * dvs);
    take(s ? &s->QS : nullptr, size_t(C) * dvs);
    take(s ? &s->R : nullptr, size_t(C * W + 1) * dvs);  // column-major, odd stride (see RS)
    take(s ? &s->A : nullptr, size_t(C) * C);
    take(s ? &s->P : nullptr, size_t(C) * C);
    take(s ? &s->eta : nullptr, size_t(C + 1) * per_col);  // Falcon-2: column-major, odd stride (see CS)
    take(s ? &s->L : nullptr, size_t(C + 1) * per_col);
    take(s ? &s->Lx : nullptr, size_t(C + 1) * per_col);
    take(s ? &s->kap : nullptr, size_t(C));
    take(s ? &s->w : nullptr, size_t(C + 1) * per_col);
    if (staged) {
        const size_t vecs = size_t(NE) * (dk / 8) + size_t(C) * (dk / 8) + size_t(NE) * (dvs / 8);
        take(s ? &s->stg : nullptr, vecs * 8 * es / 4 + (per_column(variant) ? size_t(C) * dvs : 0) + size_t(C));
    } else if (s) {
        s->stg = nullptr;
    }
    return off;
}

__device__ __forceinline__ void cp_async16z(void* smem, const void* gmem, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4z(void* smem, const void* gmem, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem), "r"(valid ? 4 : 0)
                 : "memory");
}

// One work item: mode 0 a (sequence, column slice), mode 1 a (chunk, column slice).
template <typename Tin, int VAR>
__device__ __forceinline__ void generic_item(const GParams& p, long long item) {
    extern __shared__ __align__(16) float smem_raw[];
    const int tid = threadIdx.x;
    const int DK = p.dk, DV = p.dv, DVS = p.dvs, C = p.C;
    const int XS = DK + 1;  // row stride of X and Q in shared memory (odd: rows fall in different banks)
    const int W = windowed(VAR) ? p.W : 1;
    // R (and Falcon-2's per-column scalars) are stored column-major with an odd stride, since the
    // forward substitution runs down one column across the lanes of a warp.
    const int RS = C * W + 1, CS = C + 1;
    const int NE = C + W - 1;
    const long long T = p.T, pos = p.pos;
    const int mode = p.mode;  // 0 or 1
    const int slices = (mode == 1 ? DK + DV : DV) / DVS;
    const long long nck = mode == 0 ? 0 : item % p.N;
    const long long rest = mode == 0 ? item : item / p.N;
    const long long bh = rest / slices;
    const int slice = (int)(rest % slices);
    const int c0 = slice * DVS;          // first (virtual) column of this CTA
    // DVS, DK and C are powers of two: index splits by shift and mask
    const int dvs_sh = 31 - __clz(DVS), c_sh = 31 - __clz(C);
    const bool mpart = mode == 1 && c0 < DK;  // map mode, columns of M: unit state, no targets
    const int vc0 = mode == 1 ? (mpart ? 0 : c0 - DK) : c0;  // first value column of the targets
    const long long blk = 5LL * DK * DK;
    float* wsb = mode != 0 ? p.ws + (bh * p.N + nck) * blk : nullptr;  // this chunk's workspace block

    Smem s;
    smem_floats(VAR, DK, DVS, C, W, &s, smem_raw, (int)sizeof(Tin), p.mode == 0 && p.staged);

    const Tin* q = static_cast<const Tin*>(p.q) + bh * T * DK;
    const Tin* k = static_cast<const Tin*>(p.k) + bh * T * DK;
    const Tin* v = static_cast<const Tin*>(p.v) + bh * T * DV;
    const float* beta = p.beta + bh * T * (per_column(VAR) ? DV : 1);
    const float* lam = p.lam + bh * T;
    const long long tail_stride = (long long)W * DK + (long long)(W - 1) * DV;
    const Tin* tail = p.tail ? static_cast<const Tin*>(p.tail) + bh * tail_stride : nullptr;

    // Key with local index u (token u of this call; u < 0 reaches into the tail).
    auto load_key = [&](long long u, int col) -> float {
        if (u >= 0) return ldf(k + u * DK + col);
        if (pos + 1 + u <= 0 || tail == nullptr) return 0.f;
        return ldf(tail + (u + W) * DK + col);
    };
    auto load_val = [&](long long u, int col) -> float {  // col is absolute in [0, DV)
        if (u >= 0) return ldf(v + u * DV + col);
        if (pos + 1 + u <= 0 || tail == nullptr) return 0.f;
        return ldf(tail + (long long)W * DK + (u + W - 1) * DV + col);
    };

    // Initial state slice.
    for (int idx = tid; idx < DK * DVS; idx += kThreads) {
        const int r = (idx >> dvs_sh), c = (idx & (DVS - 1));
        float x;
        if (mode == 1) x = mpart && r == c0 + c ? 1.f : 0.f;
        else x = p.S0 ? p.S0[(bh * DK + r) * DV + c0 + c] : 0.f;
        s.S[idx] = x;
    }

    const long long t_begin = nck * C, t_end = mode == 0 ? T : min(T, t_begin + C);
    for (long long t0 = t_begin; t0 < t_end; t0 += C) {
        const int n = (int)min((long long)C, T - t0);
        __syncthreads();  // previous chunk finished with every buffer
        // ---- (1) tiles. Extended row e <-> pair with global index pos + t0 + 2 - W + e. Eight elements
        // per 16-byte load (rows of q, k, v and the tail are 16-byte aligned), every load of a thread
        // issued before its stores. After the first chunk of a mode-0 walk the tiles were copied ahead
        // into the staging area (during the previous chunk's compute) and are only widened here.
        const int KV = DK / 8, VV = DVS / 8;
        const int nx = NE * KV, nq = C * KV, ny = NE * VV;
        constexpr int kVecF = 8 * (int)sizeof(Tin) / 4;  // floats of staging per 8-element vector
        auto tile_dst = [&](int idx) -> float* {
            if (idx < nx) return s.X + (idx / KV) * XS + 8 * (idx % KV);
            if (idx < nx + nq) return s.Q + ((idx - nx) / KV) * XS + 8 * ((idx - nx) % KV);
            return s.Y + ((idx - nx - nq) / VV) * DVS + 8 * ((idx - nx - nq) % VV);
        };
        const bool staged = mode == 0 && p.staged && t0 > t_begin;
        if (staged) {
            asm volatile("cp.async.wait_all;" ::: "memory");
            __syncthreads();
            for (int idx = tid; idx < nx + nq + ny; idx += kThreads) {
                float v8[8];
                const float* src = s.stg + idx * kVecF;
                if (sizeof(Tin) == 2) {
                    const uint4 u = *reinterpret_cast<const uint4*>(src);
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        v8[2 * h] = __uint_as_float(w4[h] << 16);
                        v8[2 * h + 1] = __uint_as_float(w4[h] & 0xffff0000u);
                    }
                } else {
#pragma unroll
                    for (int e8 = 0; e8 < 8; ++e8) v8[e8] = src[e8];
                }
                float* dst = tile_dst(idx);
#pragma unroll
                for (int e8 = 0; e8 < 8; ++e8) dst[e8] = v8[e8];
            }
            if (per_column(VAR)) {
                const float* sb = s.stg + (nx + nq + ny) * kVecF;
                for (int idx = tid; idx < C * DVS; idx += kThreads) {
                    const int i = (idx >> dvs_sh), c = (idx & (DVS - 1));
                    s.eta[c * CS + i] = sb[idx];
                }
                for (int i = tid; i < C; i += kThreads) s.kap[i] = sb[C * DVS + i];
            }
        } else {
            const int KV = DK / 8, VV = DVS / 8;
            const int nx = NE * KV, nq = C * KV, ny = NE * VV;
            constexpr int kPer = 4;  // vector loads in flight per thread and round
            for (int base = tid; base < nx + nq + ny; base += kPer * kThreads) {
                float buf[kPer][8];
#pragma unroll
                for (int m = 0; m < kPer; ++m) {
                    const int idx = base + m * kThreads;
#pragma unroll
                    for (int e8 = 0; e8 < 8; ++e8) buf[m][e8] = 0.f;
                    if (idx < nx) {  // shifted keys, from k, the tail or the x_1 = 0 sentinel
                        const int e = idx / KV, c8 = 8 * (idx % KV);
                        const long long gpair = pos + t0 + 2 - W + e, u = t0 - W + e;
                        if (e < n + W - 1 && gpair >= 2) {
                            if (u >= 0) ld8(k + u * DK + c8, buf[m]);
                            else if (tail != nullptr && pos + 1 + u > 0) ld8(tail + (u + W) * DK + c8, buf[m]);
                        }
                    } else if (idx < nx + nq) {
                        const int i = (idx - nx) / KV, c8 = 8 * ((idx - nx) % KV);
                        if (i < n) ld8(q + (t0 + i) * DK + c8, buf[m]);
                    } else if (idx < nx + nq + ny) {  // values of the extended rows, this CTA's columns
                        const int e = (idx - nx - nq) / VV, c8 = 8 * ((idx - nx - nq) % VV);
                        const long long gpair = pos + t0 + 2 - W + e, u = t0 + 1 - W + e;
                        if (e < n + W - 1 && gpair >= 2 && !mpart) {
                            if (u >= 0) ld8(v + u * DV + vc0 + c8, buf[m]);
                            else if (tail != nullptr && pos + 1 + u > 0)
                                ld8(tail + (long long)W * DK + (u + W - 1) * DV + vc0 + c8, buf[m]);
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < kPer; ++m) {
                    const int idx = base + m * kThreads;
                    if (idx < nx + nq + ny) {
                        float* dst = tile_dst(idx);
#pragma unroll
                        for (int e8 = 0; e8 < 8; ++e8) dst[e8] = buf[m][e8];
                    }
                }
            }
            if (per_column(VAR)) {  // the chunk's gains (per column, into eta) and ridge coefficients (into kap)
                for (int idx = tid; idx < C * DVS; idx += kThreads) {
                    const int i = (idx >> dvs_sh), c = (idx & (DVS - 1));
                    s.eta[c * CS + i] = i < n ? beta[(t0 + i) * DV + c0 + c] : 0.f;
                }
                for (int i = tid; i < C; i += kThreads) s.kap[i] = i < n ? lam[t0 + i] : 0.f;
            }
        }
        __syncthreads();
        if (mode == 0 && p.staged && t0 + C < t_end) {  // copy the next chunk's inputs ahead (all in k, q, v)
            const long long t1 = t0 + C;
            const int n1 = (int)min((long long)C, T - t1);
            for (int idx = tid; idx < nx + nq + ny; idx += kThreads) {
                const Tin* src;
                bool ok;
                if (idx < nx) {
                    const int e = idx / KV, c8 = 8 * (idx % KV);
                    ok = e < n1 + W - 1;
                    src = k + (t1 - W + e) * DK + c8;
                } else if (idx < nx + nq) {
                    const int i = (idx - nx) / KV, c8 = 8 * ((idx - nx) % KV);
                    ok = i < n1;
                    src = q + (t1 + i) * DK + c8;
                } else {
                    const int e = (idx - nx - nq) / VV, c8 = 8 * ((idx - nx - nq) % VV);
                    ok = e < n1 + W - 1;
                    src = v + (t1 + 1 - W + e) * DV + vc0 + c8;
                }
                if (!ok) src = k;  // not read (zero fill)
                float* dst = s.stg + idx * kVecF;
                cp_async16z(dst, src, ok);
                if (sizeof(Tin) == 4) cp_async16z(dst + 4, reinterpret_cast<const float*>(src) + 4, ok);
            }
            if (per_column(VAR)) {
                float* sb = s.stg + (nx + nq + ny) * kVecF;
                for (int idx = tid; idx < C * DVS; idx += kThreads) {  // 4-byte copies: beta is 4-byte aligned
                    const int i = (idx >> dvs_sh), c = (idx & (DVS - 1));
                    const bool ok = i < n1;
                    cp_async4z(sb + idx, ok ? beta + (t1 + i) * DV + c0 + c : beta, ok);
                }
                for (int i = tid; i < C; i += kThreads) cp_async4z(sb + C * DVS + i, i < n1 ? lam + t1 + i : lam, i < n1);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        // ---- (2) Gram, scores, projected history, Q S
        constexpr bool kMmaGram = std::is_same<Tin, __nv_bfloat16>::value && !windowed(VAR);
        if (kMmaGram && C <= 64 && C % 16 == 0 && DK % 16 == 0) {
            gram_mma(s.X, s.Q, s.G, s.Sc, C, DK, XS, NE, tid);
        } else {
            mm_tiled<true>(s.G, NE, s.X, XS, s.X, XS, NE, NE, DK, tid);
            mm_tiled<true>(s.Sc, NE, s.Q, XS, s.X, XS, C, NE, DK, tid);
        }
        mm_tiled<false>(s.H, DVS, s.X, XS, s.S, DVS, NE, DVS, DK, tid);
        mm_tiled<false>(s.QS, DVS, s.Q, XS, s.S, DVS, C, DVS, DK, tid);
        __syncthreads();
        // ---- (3) per-token scalars and the chunk-local log-decay prefix
        if (per_column(VAR)) {
            // every (token, column) in parallel, then one warp scan of log(gamma) per column
            for (int idx = tid; idx < C * DVS; idx += kThreads) {
                const int i = (idx >> dvs_sh), c = (idx & (DVS - 1));
                float eta = 0.f, alpha = 0.f;
                const long long tau = pos + t0 + i + 1;
                if (i < n && tau >= 2) {
                    const float lm = s.kap[i];
                    const float den = s.G[i * NE + i] + lm + p.eps;
                    eta = den == 0.f ? 0.f : s.eta[c * CS + i] / den;
                    alpha = fminf(eta * lm, 1.f - p.eps_gamma);
                }
                s.eta[c * CS + i] = eta;
                s.L[c * CS + i] = log1pf(-alpha);
            }
            __syncthreads();
            const int wid = tid >> 5, lane = tid & 31, per = (C + 31) / 32;
            for (int c = wid; c < DVS; c += kThreads / 32) {
                float ls[2] = {0.f, 0.f}, lsum = 0.f;
                for (int m = 0; m < per; ++m) {
                    const int i = lane * per + m;
                    ls[m] = i < C ? s.L[c * CS + i] : 0.f;
                    lsum += ls[m];
                }
                float incl = lsum;
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                float run = incl - lsum;
                for (int m = 0; m < per; ++m) {
                    const int i = lane * per + m;
                    if (i < C) {
                        s.Lx[c * CS + i] = run;
                        run += ls[m];
                        s.L[c * CS + i] = run;
                    }
                }
            }
        } else if (tid < 32) {
            const int lane = tid;
            const int per = (C + 31) / 32;
            float lsum = 0.f;
            float ls[2];
            for (int m = 0; m < per; ++m) {
                const int i = lane * per + m;
                float eta = 0.f, alpha = 0.f, kap = 0.f;
                if (i < n) {
                    const long long tau = pos + t0 + i + 1;
                    const float lm = lam[t0 + i];
                    if (windowed(VAR)) {
                        int slots[kMaxW] = {};
                        int nb = 0;
                        for (int sl = 0; sl < W; ++sl)
                            if (tau - sl >= 2) slots[nb++] = i - sl + W - 1;
                        if (nb > 0) {
                            float mu = 0.f;
                            if (VAR == kF3A) {  // the window's mean key energy (trace of the averaged Gram)
                                for (int x = 0; x < nb; ++x) mu += s.G[slots[x] * NE + slots[x]];
                                mu /= (float)nb;
                            } else if (p.mu) {
                                mu = p.mu[bh * T + t0 + i];
                            } else switch (W) {  // the matrix in registers: one instance per window size
                                case 1: mu = s.G[slots[0] * NE + slots[0]]; break;
                                case 2: mu = window_lambda_max<2>(s.G, NE, slots, nb); break;
                                case 3: mu = window_lambda_max<3>(s.G, NE, slots, nb); break;
                                case 4: mu = window_lambda_max<4>(s.G, NE, slots, nb); break;
                                case 5: mu = window_lambda_max<5>(s.G, NE, slots, nb); break;
                                case 6: mu = window_lambda_max<6>(s.G, NE, slots, nb); break;
                                case 7: mu = window_lambda_max<7>(s.G, NE, slots, nb); break;
                                default: mu = window_lambda_max<8>(s.G, NE, slots, nb); break;
                            }
                            const float den = mu + lm + p.eps;
                            eta = den == 0.f ? 0.f : beta[t0 + i] / den;
                            alpha = fminf(eta * lm, 1.f - p.eps_gamma);
                            kap = eta / (float)nb;
                        }
                    } else if (tau >= 2) {
                        const float den = s.G[i * NE + i] + lm + p.eps;
                        eta = den == 0.f ? 0.f : beta[t0 + i] / den;
                        alpha = fminf(eta * lm, 1.f - p.eps_gamma);
                    }
                }
                if (i < C) {
                    s.eta[i] = eta;
                    s.kap[i] = windowed(VAR) ? kap : eta;
                }
                ls[m] = log1pf(-alpha);
                lsum += ls[m];
            }
            // inclusive warp scan of the lane sums
            float incl = lsum;
            for (int o = 1; o < 32; o <<= 1) {
                float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            float run = incl - lsum;
            for (int m = 0; m < per; ++m) {
                const int i = lane * per + m;
                if (i < C) {
                    s.Lx[i] = run;
                    run += ls[m];
                    s.L[i] = run;
                }
            }
        }
        __syncthreads();
        // ---- (4) decay-weighted coefficient matrices (shared by all columns)
        if (!per_column(VAR)) {
            const float LC = s.L[C - 1];
            for (int idx = tid; idx < C * C; idx += kThreads) {
                const int i = idx >> c_sh, j = idx & (C - 1);
                float a = 0.f, pp = 0.f;
                if (j < i) a = s.kap[j] * expf(s.Lx[i] - s.L[j]);
                if (j <= i) pp = s.kap[j] * expf(s.L[i] - s.L[j]);
                if (!windowed(VAR)) {
                    a *= s.G[i * NE + j];
                    pp *= s.Sc[i * NE + j];
                }
                s.A[idx] = a;
                s.P[idx] = pp;
            }
            for (int j = tid; j < C; j += kThreads) s.w[j] = s.kap[j] * expf(LC - s.L[j]);
        } else {
            // Falcon-2, per column c: when the chunk's total log decay is at least -kFastL every factor
            // e^{a - b} (a >= b) is formed as e^{a} e^{-b}, both finite, and w holds eta_j e^{-L_j}
            // ("fast"); otherwise w holds eta_j e^{L_C - L_j} and the factors are formed one by one.
            // Slot C of each column records which.
            for (int idx = tid; idx < C * DVS; idx += kThreads) {
                const int j = (idx >> dvs_sh), c = (idx & (DVS - 1));
                const float LC = s.L[c * CS + C - 1];
                const bool fast = LC >= -kFastL;
                s.w[c * CS + j] = s.eta[c * CS + j] * expf((fast ? 0.f : LC) - s.L[c * CS + j]);
                if (j == 0) s.w[c * CS + C] = fast ? 1.f : 0.f;
            }
        }
        __syncthreads();
        // ---- (5) merged-RHS forward substitution. Falcon-1 and -2: a half-warp per column, 16 rows at a
        // time: each lane owns one row, first sums the earlier blocks' terms, then the block's rows are
        // finished in order, each new r_j handed to the other lanes by a shuffle.
        if (VAR == kF1 || VAR == kF2) {
            const int lane = tid & 31, li = lane & 15;
            for (int cg = 0; cg < DVS; cg += 2 * (kThreads / 32)) {
                const int cl = cg + 2 * (tid >> 5) + (lane >> 4);  // this half-warp's column
                const bool cvalid = cl < DVS;
                // Falcon-2 "fast" columns keep R~_j = eta_j e^{-L_j} r_j, with A_ij R_j = e^{Lx_i} G_ij R~_j
                const bool fast = VAR == kF2 && cvalid && s.w[cl * CS + C] != 0.f;
                auto coef = [&](int i, int j) -> float {  // the factor of the stored R_j (or R~_j) in row i
                    if (VAR == kF1) return s.A[i * C + j];
                    if (fast) return s.G[i * NE + j];
                    return s.eta[cl * CS + j] * expf(s.Lx[cl * CS + i] - s.L[cl * CS + j]) * s.G[i * NE + j];
                };
                for (int b0 = 0; b0 < n; b0 += 16) {
                    const int i = b0 + li;
                    const bool row = cvalid && i < n;
                    float acc = 0.f, dcy = 0.f, yv = 0.f, hv = 0.f, ca = 1.f;
                    float cf[16];
                    if (row) {
                        for (int m = 0; m < b0; ++m) {  // earlier blocks; lanes start apart (no bank clash)
                            int j = m + li;
                            if (j >= b0) j -= b0;
                            acc = fmaf(coef(i, j), s.R[cl * RS + j], acc);
                        }
                        dcy = expf(VAR == kF1 ? s.Lx[i] : s.Lx[cl * CS + i]);
                        yv = s.Y[i * DVS + cl];
                        hv = s.H[i * DVS + cl];
                        if (fast) ca = s.w[cl * CS + i];
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) cf[jj] = (row && b0 + jj < i) ? coef(i, b0 + jj) : 0.f;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        float rv = 0.f;
                        if (li == jj && row) {
                            const float r = fast ? yv - dcy * (hv + acc) : (yv - dcy * hv) - acc;
                            rv = ca * r;
                            s.R[cl * RS + i] = rv;
                        }
                        rv = __shfl_sync(0xffffffffu, rv, jj, 16);
                        acc = fmaf(cf[jj], rv, acc);
                    }
                }
            }
        } else if (VAR == kF3 && DVS == 64) {
            // All 64 columns at once, by blocks of TB = 16 / W tokens (NB = TB W unknowns): per block kb,
            //   r_kb = (I + A_kb,kb)^-1 (rhs_kb - sum_{j < kb} A_kb,j r_j),
            // the 16 x 16 diagonal-block inverses formed once (shared by every column), the earlier
            // blocks' terms as a product over all columns. Invalid unknowns (the sentinel pair's slots,
            // tokens past n) have zero rows and zero right-hand sides, so r = 0 there.
            const int TB = 16 / W, NB = TB * W, nblk = (C + TB - 1) / TB;
            auto valid_u = [&](int i, int a) { return i < n && pos + t0 + i + 1 - a >= 2; };
            // (1) right-hand sides into R
            for (int idx = tid; idx < C * W * DVS; idx += kThreads) {
                const int m = (idx >> dvs_sh), c = (idx & (DVS - 1)), i = m / W, a = m % W, pa = i - a + W - 1;
                s.R[c * RS + m] = valid_u(i, a) ? s.Y[pa * DVS + c] - expf(s.Lx[i]) * s.H[pa * DVS + c] : 0.f;
            }
            __syncthreads();
            // (2) diagonal-block inverses, one warp per block, a lane per column (Y is free now, and sized
            // for them)
            float* Dinv = s.Y;  // [nblk][16][16]
            {
                const int kb = tid >> 5, col = tid & 31;
                if (kb < nblk) {
                    float* D = Dinv + kb * 256;
                    for (int rr = 0; rr < NB; ++rr) {
                        const int i = kb * TB + rr / W, a = rr % W, pa = i - a + W - 1;
                        const bool vr = valid_u(i, a);
                        float x = (rr == col) ? 1.f : 0.f;
                        if (vr && col < NB)
                            for (int r2 = 0; r2 < rr; ++r2) {
                                const int l = kb * TB + r2 / W, b = r2 % W;
                                if (l < i) x = fmaf(-s.A[i * C + l] * s.G[pa * NE + (l - b + W - 1)], D[r2 * 16 + col], x);
                            }
                        if (col < 16) D[rr * 16 + col] = x;
                        __syncwarp();
                    }
                }
            }
            __syncthreads();
            // (3) block by block
            float* Tmp = s.H;  // [16][DVS]: right-hand side minus the earlier blocks' terms
            const int rr = tid >> 4, cb = 4 * (tid & 15);
            for (int kb = 0; kb < nblk; ++kb) {
                if (rr < NB) {
                    const int m = kb * NB + rr, i = kb * TB + rr / W, a = rr % W, pa = i - a + W - 1;
                    float t4[4] = {0.f, 0.f, 0.f, 0.f};
                    if (valid_u(i, a)) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        for (int l = 0; l < kb * TB; ++l) {
                            const float al = s.A[i * C + l];
                            const float* gr = s.G + pa * NE + l + W - 1;  // G[pa][l - b + W - 1] = gr[-b]
                            for (int b = 0; b < W; ++b) {
                                const float cf = al * gr[-b];
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj) acc[jj] = fmaf(cf, s.R[(cb + jj) * RS + l * W + b], acc[jj]);
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) t4[jj] = s.R[(cb + jj) * RS + m] - acc[jj];
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) Tmp[rr * DVS + cb + jj] = t4[jj];
                }
                __syncthreads();
                if (rr < NB && kb * TB + rr / W < C) {  // the last block may reach past the chunk's C tokens
                    const float* D = Dinv + kb * 256 + rr * 16;
                    float o[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int r2 = 0; r2 < NB; ++r2) {
                        const float d = D[r2];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) o[jj] = fmaf(d, Tmp[r2 * DVS + cb + jj], o[jj]);
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) s.R[(cb + jj) * RS + kb * NB + rr] = o[jj];
                }
                __syncthreads();
            }
        } else if (VAR == kF3) {
            // Unknowns r_{i,a} (token i, window slot a) depend only on earlier tokens, so a token's W
            // slots are finished together: a half-warp per column takes 16 / W tokens at a time, one
            // lane per unknown, sums the earlier blocks' terms in parallel, then finishes the block
            // token by token, each token's W values passed to the other lanes by shuffles.
            const int lane = tid & 31, li = lane & 15, TPB = 16 / W, NU = TPB * W;
            for (int cg = 0; cg < DVS; cg += 2 * (kThreads / 32)) {
                const int cl = cg + 2 * (tid >> 5) + (lane >> 4);
                const bool cvalid = cl < DVS;
                for (int b0 = 0; b0 < n; b0 += TPB) {
                    const int i = b0 + li / W, a = li % W;
                    const bool row = cvalid && li < NU && i < n;
                    const int pa = i - a + W - 1;
                    float acc = 0.f, dcy = 0.f, yv = 0.f, hv = 0.f;
                    bool valid = false;
                    if (row) {
                        // the earlier blocks' tokens l, lanes starting apart (no bank clash)
                        const int l0 = b0 > 0 ? li % b0 : 0;
                        for (int ll = 0; ll < b0; ++ll) {
                            int l = ll + l0;
                            if (l >= b0) l -= b0;
                            const float al = s.A[i * C + l];
                            const float* gr = s.G + pa * NE + l + W - 1;  // G[pa][l - bb + W - 1]
                            const float* rr = s.R + cl * RS + l * W;
                            for (int bb = 0; bb < W; ++bb) acc = fmaf(al * gr[-bb], rr[bb], acc);
                        }
                        dcy = expf(s.Lx[i]);
                        yv = s.Y[pa * DVS + cl];
                        hv = s.H[pa * DVS + cl];
                        valid = pos + t0 + i + 1 - a >= 2;
                    }
                    for (int st = 0; st < TPB; ++st) {
                        const int tok = b0 + st;
                        float rv = 0.f;
                        if (row && i == tok) {
                            rv = valid ? (yv - dcy * hv) - acc : 0.f;
                            s.R[cl * RS + i * W + a] = rv;
                        }
                        const float ai = (row && i > tok) ? s.A[i * C + tok] : 0.f;
                        for (int bb = 0; bb < W; ++bb) {
                            const float vb = __shfl_sync(0xffffffffu, rv, st * W + bb, 16);
                            if (row && i > tok) acc = fmaf(ai * s.G[pa * NE + (tok - bb + W - 1)], vb, acc);
                        }
                    }
                }
            }
        } else if (VAR == kF2A) {  // no solve: the targets (Falcon-2A fast columns keep eta_j e^{-L_j} y_j)
            for (int idx = tid; idx < n * DVS; idx += kThreads) {
                const int j = (idx >> dvs_sh), c = (idx & (DVS - 1));
                const float y = s.Y[j * DVS + c];
                s.R[c * RS + j] = s.w[c * CS + C] != 0.f ? s.w[c * CS + j] * y : y;
            }
        } else if (VAR == kF3A) {  // no solve: every window slot's target (zero for the sentinel pair)
            for (int idx = tid; idx < n * W * DVS; idx += kThreads) {
                const int m = (idx >> dvs_sh), c = (idx & (DVS - 1)), i = m / W, a = m % W;
                const bool valid = pos + t0 + i + 1 - a >= 2;
                s.R[c * RS + m] = valid ? s.Y[(i - a + W - 1) * DVS + c] : 0.f;
            }
        }
        __syncthreads();
        // ---- (6) outputs (read after write) and (7) carried state
        Tin* out = static_cast<Tin*>(p.out) + bh * T * DV;
        if (per_column(VAR)) {
            for (int idx = tid; idx < (mode == 1 ? 0 : n * DVS); idx += kThreads) {
                const int i = (idx >> dvs_sh), c = (idx & (DVS - 1));
                float o;
                const float li = s.L[c * CS + i];
                if (s.w[c * CS + C] != 0.f) {  // fast: o = e^{L_i} (QS + sum_j Sc_ij R~_j)
                    o = s.QS[idx];
                    for (int j = 0; j <= i; ++j) o = fmaf(s.Sc[i * NE + j], s.R[c * RS + j], o);
                    o *= expf(li);
                } else {
                    o = expf(li) * s.QS[idx];
                    for (int j = 0; j <= i; ++j)
                        o = fmaf(s.eta[c * CS + j] * expf(li - s.L[c * CS + j]) * s.Sc[i * NE + j], s.R[c * RS + j],
                                 o);
                }
                stf(out + (t0 + i) * DV + c0 + c, o);
            }
        } else {
            // o_i = e^{L_i} QS_i + sum_{l <= i} P_il v_l with v_l = sum_b Sc_{i, l-b+W-1} r_{l,b} (windowed), r_l
            // (Falcon-1) or y_l (Falcon-1A); P is zero above the diagonal, and l < n. Each thread: rows i
            // and i + C/2 by four columns.
            const int half = C / 2, ncg = DVS / 4;
            for (int tile = tid; tile < half * ncg; tile += kThreads) {
                const int i0 = tile / ncg, cb = 4 * (tile % ncg), i1 = i0 + half;
                float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
                const int lmax = min(i1, n - 1);  // rows of R past n were never written
                for (int l = 0; l <= lmax; ++l) {
                    const float f0 = s.P[i0 * C + l], f1 = s.P[i1 * C + l];
                    if (windowed(VAR)) {
                        for (int b = 0; b < W; ++b) {
                            const int e = l - b + W - 1;
                            const float t0v = f0 * s.Sc[i0 * NE + e], t1v = f1 * s.Sc[i1 * NE + e];
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) {
                                const float r = s.R[(cb + jj) * RS + l * W + b];
                                acc0[jj] = fmaf(t0v, r, acc0[jj]);
                                acc1[jj] = fmaf(t1v, r, acc1[jj]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const float r = VAR == kF1A ? s.Y[l * DVS + cb + jj] : s.R[(cb + jj) * RS + l];
                            acc0[jj] = fmaf(f0, r, acc0[jj]);
                            acc1[jj] = fmaf(f1, r, acc1[jj]);
                        }
                    }
                }
                const float e0 = expf(s.L[i0]), e1 = expf(s.L[i1]);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float o0 = fmaf(e0, s.QS[i0 * DVS + cb + jj], acc0[jj]);
                    const float o1 = fmaf(e1, s.QS[i1 * DVS + cb + jj], acc1[jj]);
                    if (mode == 1) {  // the output map: Ao (unit state columns) or Bo (targets)
                        float* ob = wsb + (mpart ? 3LL * DK * DK + c0 : 4LL * DK * DK + vc0) + cb + jj;
                        ob[i0 * DK] = o0;
                        ob[i1 * DK] = o1;
                    } else {
                        if (i0 < n) stf(out + (t0 + i0) * DV + c0 + cb + jj, o0);
                        if (i1 < n) stf(out + (t0 + i1) * DV + c0 + cb + jj, o1);
                    }
                }
            }
        }
        if (windowed(VAR)) {
            // the write sum_l w_l sum_b x_{l-b} r_{l,b}^T gathered by extended row e = l - b + W - 1 first
            // (into H, whose last use was the solve): S' = e^{L_C} S + X_ext^T Rf
            for (int idx = tid; idx < (n + W - 1) * DVS; idx += kThreads) {
                const int e = (idx >> dvs_sh), c = (idx & (DVS - 1));
                float acc = 0.f;
                for (int b = 0; b < W; ++b) {
                    const int l = e + b - (W - 1);
                    if (l >= 0 && l < n) acc = fmaf(s.w[l], s.R[c * RS + l * W + b], acc);
                }
                s.H[idx] = acc;
            }
            __syncthreads();
        }
        for (int idx = tid; idx < DK * DVS; idx += kThreads) {
            const int r = (idx >> dvs_sh), c = (idx & (DVS - 1));
            float acc = 0.f;
            if (windowed(VAR)) {
                for (int e = 0; e < n + W - 1; ++e) acc = fmaf(s.X[e * XS + r], s.H[e * DVS + c], acc);
                s.S[idx] = fmaf(expf(s.L[C - 1]), s.S[idx], acc);
            } else if (per_column(VAR)) {
                const float gC = expf(s.L[c * CS + C - 1]);
                if (s.w[c * CS + C] != 0.f) {  // fast: S' = e^{L_C} (S + sum_j x_j R~_j)
                    for (int j = 0; j < n; ++j) acc = fmaf(s.X[j * XS + r], s.R[c * RS + j], acc);
                    s.S[idx] = gC * (s.S[idx] + acc);
                } else {
                    for (int j = 0; j < n; ++j) acc = fmaf(s.X[j * XS + r] * s.w[c * CS + j], s.R[c * RS + j], acc);
                    s.S[idx] = fmaf(gC, s.S[idx], acc);
                }
            } else if (VAR == kF1A) {
                for (int j = 0; j < n; ++j) acc = fmaf(s.X[j * XS + r] * s.w[j], s.Y[j * DVS + c], acc);
                s.S[idx] = fmaf(expf(s.L[C - 1]), s.S[idx], acc);
            } else {
                for (int j = 0; j < n; ++j) acc = fmaf(s.X[j * XS + r] * s.w[j], s.R[c * RS + j], acc);
                s.S[idx] = fmaf(expf(s.L[C - 1]), s.S[idx], acc);
            }
        }
    }
    __syncthreads();
    if (mode == 1) {  // the chunk's state map: M columns or U columns
        float* dst = mpart ? wsb + c0 : wsb + (long long)DK * DK + vc0;
        const int ld = mpart ? DK : DV;
        for (int idx = tid; idx < DK * DVS; idx += kThreads) {
            const int r = (idx >> dvs_sh), c = (idx & (DVS - 1));
            dst[r * ld + c] = s.S[idx];
        }
    } else if (p.S_final) {
        for (int idx = tid; idx < DK * DVS; idx += kThreads) {
            const int r = (idx >> dvs_sh), c = (idx & (DVS - 1));
            p.S_final[(bh * DK + r) * DV + c0 + c] = s.S[idx];
        }
    }
    if (p.tail_out && (mode == 0 || nck == p.N - 1)) {  // map mode: the last chunk's CTAs
        Tin* to = static_cast<Tin*>(p.tail_out) + bh * tail_stride;
        if (slice == 0)
            for (int idx = tid; idx < W * DK; idx += kThreads) {
                const int sl = idx / DK, cc = idx % DK;
                stf(to + idx, load_key(T - W + sl, cc));
            }
        if (!mpart)
            for (int idx = tid; idx < (W - 1) * DVS; idx += kThreads) {
                const int sl = (idx >> dvs_sh), cc = (idx & (DVS - 1));
                stf(to + (long long)W * DK + sl * DV + vc0 + cc, load_val(T - W + 1 + sl, vc0 + cc));
            }
    }
}

template <typename Tin, int VAR>
__global__ void __launch_bounds__(kThreads, 2) falcon_chunk_generic_kernel(GParams p) {
    generic_item<Tin, VAR>(p, blockIdx.x);
}

template <typename Tin, int VAR>
__global__ void __launch_bounds__(kThreads, 2) falcon_chunk_generic_left_kernel(GParams p) {
    // map mode after the tensor-core map kernel: each CTA takes a range of (chunk, slice) items and runs
    // only those of the chunks that kernel left, so that the launch is about one wave of CTAs when it
    // finished them all, and as many CTAs per item as before when it finished none. A finished chunk is
    // marked with 1 in its block's state slot (only group blocks use theirs); its maps and the tail
    // are written already.
    const int slices = (p.dk + p.dv) / p.dvs;
    const long long items = p.BH * p.N * slices, blk = 5LL * p.dk * p.dk;
    // this CTA's items: a contiguous range of at most kThreads, their marks read by one thread each
    __shared__ int s_list[kThreads];
    __shared__ int s_n;
    const long long first = (long long)blockIdx.x * p.per_cta;
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    const long long me = first + threadIdx.x;
    if (threadIdx.x < p.per_cta && me < items) {
        const long long nck = me % p.N, bh = (me / p.N) / slices;
        if (reinterpret_cast<const int*>(p.ws + (bh * p.N + nck) * blk + 2LL * p.dk * p.dk)[0] != 1)
            s_list[atomicAdd(&s_n, 1)] = threadIdx.x;
    }
    __syncthreads();
    const int n = s_n;
    for (int u = 0; u < n; ++u) {
        generic_item<Tin, VAR>(p, first + s_list[u]);
        __syncthreads();  // the next item reuses the shared memory
    }
}

// Falcon-3: every token's window normaliser mu = lambda_max((1/B) sum_j x_j x_j^T) over the window's
// realised pairs, one thread per token (the same Gram entries, summed in the same order, and the same
// Jacobi as the chunk kernel's own), so that chunk kernels running one chunk per CTA read it instead
// of each recomputing it. A CTA takes 128 consecutive tokens of one sequence and first copies the
// 127 + W key rows they use into shared memory with coalesced 16-byte loads (rows padded by 16 bytes,
// so that neighbouring tokens' rows fall in different banks).
template <typename Tin, int W>
__global__ void __launch_bounds__(128) falcon_window_mu_kernel(const Tin* k, const Tin* tail, float* mu, long long BH,
                                                             long long T, long long pos, int DK,
                                                             long long tail_stride) {
    extern __shared__ __align__(16) unsigned char mu_sm[];
    const long long tiles = (T + 127) / 128;
    const long long bh = blockIdx.x / tiles, t0 = (blockIdx.x % tiles) * 128;
    const int rb = DK * (int)sizeof(Tin), rs = rb + 16, pieces = rb / 16;
    // row r holds the key of local index u = t0 - W + r (a negative u: the tail's key u + W)
    for (int e = threadIdx.x; e < (127 + W) * pieces; e += 128) {
        const int r = e / pieces, q = e % pieces;
        const long long u = t0 - W + r;
        const Tin* src = nullptr;
        if (u >= 0 && u < T) src = k + (bh * T + u) * DK;
        else if (u < 0 && tail) src = tail + bh * tail_stride + (u + W) * DK;
        const uint4 v = src ? reinterpret_cast<const uint4*>(src)[q] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(mu_sm + r * rs + 16 * q) = v;
    }
    __syncthreads();
    const long long t = t0 + threadIdx.x;
    if (t >= T) return;
    const long long tau = pos + t + 1;
    // the window's realised pairs are a = 0 .. nb - 1 (pair tau - a, key k_{tau - a - 1}: row tid + W - a - 1)
    const int nb = (int)min((long long)W, max(0LL, tau - 1));
    const Tin* rows[W];
#pragma unroll
    for (int a = 0; a < W; ++a)
        rows[a] = a >= nb ? nullptr : reinterpret_cast<const Tin*>(mu_sm + (threadIdx.x + W - a - 1) * rs);
    float g[W][W];
#pragma unroll
    for (int x = 0; x < W; ++x)
#pragma unroll
        for (int y = 0; y < W; ++y) g[x][y] = 0.f;
    for (int c8 = 0; c8 < DK; c8 += 8) {
        float v[W][8];
#pragma unroll
        for (int x = 0; x < W; ++x) {
            if (x < nb) ld8(rows[x] + c8, v[x]);
            else
#pragma unroll
                for (int e = 0; e < 8; ++e) v[x][e] = 0.f;
        }
#pragma unroll
        for (int x = 0; x < W; ++x)
#pragma unroll
            for (int y = 0; y <= x; ++y)
#pragma unroll
                for (int e = 0; e < 8; ++e) g[x][y] = fmaf(v[x][e], v[y][e], g[x][y]);
    }
    float m = 0.f;
    if (nb > 0) {
        const float inv = 1.f / (float)nb;
#pragma unroll
        for (int x = 0; x < W; ++x)
#pragma unroll
            for (int y = 0; y < W; ++y) g[x][y] = (x >= y ? g[x][y] : g[y][x]) * inv;
        m = W == 1 ? g[0][0] * (float)nb : lambda_max_fixed<W>(g);
    }
    mu[bh * T + t] = m;
}

template <typename Tin>
cudaError_t launch_typed(const Launch& a, const GParams& gp, dim3 grid, size_t smem, cudaStream_t st) {
    void (*fn)(GParams) = nullptr;
    if (gp.skip_marked) {  // only the tensor-core map kernel's variants leave chunks unmarked
        switch (a.variant) {
            case kF3: fn = falcon_chunk_generic_left_kernel<Tin, kF3>; break;
            case kF3A: fn = falcon_chunk_generic_left_kernel<Tin, kF3A>; break;
            default: return cudaErrorInvalidValue;
        }
    } else switch (a.variant) {
        case kF1: fn = falcon_chunk_generic_kernel<Tin, kF1>; break;
        case kF1A: fn = falcon_chunk_generic_kernel<Tin, kF1A>; break;
        case kF2: fn = falcon_chunk_generic_kernel<Tin, kF2>; break;
        case kF2A: fn = falcon_chunk_generic_kernel<Tin, kF2A>; break;
        case kF3: fn = falcon_chunk_generic_kernel<Tin, kF3>; break;
        case kF3A: fn = falcon_chunk_generic_kernel<Tin, kF3A>; break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(gp);
    return cudaGetLastError();
}

int choose_dvs(const Launch& a) {
    // Enough CTAs to cover the GPU twice over, slices no narrower than 8 columns (one 16-byte
    // load of bf16 values per row), and a shared-memory footprint that fits one CTA.
    int dvs = (int)a.dv;
    const int64_t seqs = a.B * a.H;
    while (dvs > 8 && seqs * (a.dv / dvs) < 2 * 152) dvs /= 2;
    while (dvs > 16 && generic_smem_bytes(a, dvs, false) > 200 * 1024) dvs /= 2;
    return dvs;
}

}  // namespace

size_t generic_smem_bytes(const Launch& a, int dvs, bool staged) {
    const int W = windowed(a.variant) ? a.W : 1;
    return smem_floats(a.variant, (int)a.dk, dvs, a.chunk, W, nullptr, nullptr, a.bf16 ? 2 : 4, staged) * sizeof(float);
}

int launch_generic(const Launch& a, cudaStream_t st) { return launch_generic_mode(a, 0, nullptr, 0, nullptr, st); }

int launch_window_mu(const Launch& a, float* mu, cudaStream_t st) {
    const long long n = a.B * a.H * a.T;
    if (n == 0) return 0;
    const long long ts = (long long)a.W * a.dk + (long long)(a.W - 1) * a.dv;
    const unsigned grid = (unsigned)(a.B * a.H * ((a.T + 127) / 128));
    bool attr_ok = true;
    auto go = [&](auto tin, auto wc) {
        using Tin = decltype(tin);
        constexpr int W = decltype(wc)::value;
        const size_t smem = (size_t)(127 + W) * (size_t)(a.dk * sizeof(Tin) + 16);  // at most 71 KB
        if (cudaFuncSetAttribute(falcon_window_mu_kernel<Tin, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess) {
            attr_ok = false;
            return;
        }
        falcon_window_mu_kernel<Tin, W><<<grid, 128, smem, st>>>(static_cast<const Tin*>(a.k),
                                                                 static_cast<const Tin*>(a.tail), mu, a.B * a.H, a.T,
                                                                 a.pos, (int)a.dk, ts);
    };
    auto by_w = [&](auto tin) {
        switch (a.W) {
            case 1: go(tin, std::integral_constant<int, 1>{}); break;
            case 2: go(tin, std::integral_constant<int, 2>{}); break;
            case 3: go(tin, std::integral_constant<int, 3>{}); break;
            case 4: go(tin, std::integral_constant<int, 4>{}); break;
            case 5: go(tin, std::integral_constant<int, 5>{}); break;
            case 6: go(tin, std::integral_constant<int, 6>{}); break;
            case 7: go(tin, std::integral_constant<int, 7>{}); break;
            default: go(tin, std::integral_constant<int, 8>{}); break;
        }
    };
    if (a.bf16) by_w(__nv_bfloat16{});
    else by_w(float{});
    return attr_ok && cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int launch_generic_mode(const Launch& a, int mode, float* ws, long long N, const float* mu, cudaStream_t st,
                        bool skip_marked) {
    if (a.B * a.H == 0) return 0;
    // map mode: whole 64-column slices (the chunks supply the parallelism, so the key-only work of a
    // chunk is done by two CTAs instead of once per narrow slice)
    const int dvs = mode == 0 ? choose_dvs(a) : (int)a.dv;
    GParams gp;
    gp.q = a.q;
    gp.k = a.k;
    gp.v = a.v;
    gp.beta = a.beta;
    gp.lam = a.lam;
    gp.S0 = a.S0;
    gp.tail = a.tail;
    gp.out = a.out;
    gp.S_final = a.S_final;
    gp.tail_out = a.tail_out;
    gp.T = a.T;
    gp.pos = a.pos;
    gp.dk = (int)a.dk;
    gp.dv = (int)a.dv;
    gp.dvs = dvs;
    gp.C = a.chunk;
    gp.W = windowed(a.variant) ? a.W : 1;
    gp.eps = a.eps;
    gp.eps_gamma = a.eps_gamma;
    gp.mode = mode;
    gp.mu = mu;
    gp.ws = ws;
    gp.N = N;
    gp.skip_marked = skip_marked ? 1 : 0;
    // mode 0 copies each next chunk ahead when the staging area fits beside the tiles
    gp.staged = mode == 0 && generic_smem_bytes(a, dvs, true) <= 200 * 1024;
    const size_t smem = generic_smem_bytes(a, dvs, gp.staged != 0);
    const long long slices = (mode == 1 ? a.dk + a.dv : a.dv) / dvs;
    const long long items = slices * a.B * a.H * (mode == 0 ? 1 : N);
    gp.BH = a.B * a.H;
    gp.per_cta = 1;
    if (skip_marked) {  // about two CTAs per SM, each over a range of items
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 4;
        gp.per_cta = (int)std::min<long long>(kThreads, std::max<long long>(1, (items + 2LL * sms - 1) / (2LL * sms)));
    }
    dim3 grid((unsigned)((items + gp.per_cta - 1) / gp.per_cta));
    cudaError_t e = a.bf16 ? launch_typed<__nv_bfloat16>(a, gp, grid, smem, st)
                           : launch_typed<float>(a, gp, grid, smem, st);
    return e == cudaSuccess ? 0 : 4;
}

}  // namespace falcon
