// CUDA-core chunk-parallel Falcon forward kernel (all variants, fp32 or bf16 I/O).
//
// One CTA owns one (batch, head) sequence and a slice of `dvs` value columns.
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
// Only exp(L_a - L_b) with a >= b is formed, so no factor exceeds 1.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "falcon_internal.h"

namespace falcon {
namespace {

constexpr int kThreads = 256;
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
};

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Largest eigenvalue of a small symmetric matrix (n <= kMaxW), cyclic Jacobi in fp32.
__device__ float lambda_max_small(float (*a)[kMaxW], int n) {
    for (int sweep = 0; sweep < 16; ++sweep) {
        float off = 0.f, dg = 0.f;
        for (int p = 0; p < n; ++p) {
            dg += a[p][p] * a[p][p];
            for (int r = p + 1; r < n; ++r) off += a[p][r] * a[p][r];
        }
        if (off <= 1e-14f * dg || off == 0.f) break;
        for (int p = 0; p < n; ++p)
            for (int r = p + 1; r < n; ++r) {
                float apq = a[p][r];
                if (apq == 0.f) continue;
                float th = (a[r][r] - a[p][p]) / (2.f * apq);
                float t = (th >= 0.f ? 1.f : -1.f) / (fabsf(th) + sqrtf(th * th + 1.f));
                float c = rsqrtf(t * t + 1.f), s = t * c;
                for (int m = 0; m < n; ++m) {
                    float x = a[m][p], y = a[m][r];
                    a[m][p] = c * x - s * y;
                    a[m][r] = s * x + c * y;
                }
                for (int m = 0; m < n; ++m) {
                    float x = a[p][m], y = a[r][m];
                    a[p][m] = c * x - s * y;
                    a[r][m] = s * x + c * y;
                }
            }
    }
    float mx = a[0][0];
    for (int p = 1; p < n; ++p) mx = fmaxf(mx, a[p][p]);
    return mx;
}

// Shared-memory carve-up (floats). NE = C + W - 1 extended pair rows.
struct Smem {
    float *X, *Q, *Y, *S, *G, *Sc, *H, *QS, *R, *A, *P;
    float *eta, *L, *Lx, *kap, *w;
};

__host__ __device__ inline size_t smem_floats(int variant, int dk, int dvs, int C, int W, Smem* s, float* base) {
    const int NE = C + W - 1;
    const int per_col = (variant == kF2) ? dvs : 1;
    size_t off = 0;
    auto take = [&](float** dst, size_t n) {
        if (dst) *dst = base + off;
        off += (n + 3) & ~size_t(3);  // keep 16-byte alignment of every array
    };
    take(s ? &s->X : nullptr, size_t(NE) * (dk + 1));  // rows padded: the Gram reads rows across lanes
    take(s ? &s->Q : nullptr, size_t(C) * (dk + 1));
    take(s ? &s->Y : nullptr, size_t(NE) * dvs);
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
    return off;
}

template <typename Tin, int VAR>
__global__ void __launch_bounds__(kThreads) falcon_chunk_generic_kernel(GParams p) {
    extern __shared__ __align__(16) float smem_raw[];
    const int tid = threadIdx.x;
    const int DK = p.dk, DV = p.dv, DVS = p.dvs, C = p.C;
    const int XS = DK + 1;  // row stride of X and Q in shared memory (odd: rows fall in different banks)
    const int W = (VAR == kF3) ? p.W : 1;
    // R (and Falcon-2's per-column scalars) are stored column-major with an odd stride, since the
    // forward substitution runs down one column across the lanes of a warp.
    const int RS = C * W + 1, CS = C + 1;
    const int NE = C + W - 1;
    const long long T = p.T, pos = p.pos;
    const int slices = DV / DVS;
    const long long bh = blockIdx.x / slices;
    const int slice = blockIdx.x % slices;
    const int c0 = slice * DVS;

    Smem s;
    smem_floats(VAR, DK, DVS, C, W, &s, smem_raw);

    const Tin* q = static_cast<const Tin*>(p.q) + bh * T * DK;
    const Tin* k = static_cast<const Tin*>(p.k) + bh * T * DK;
    const Tin* v = static_cast<const Tin*>(p.v) + bh * T * DV;
    const float* beta = p.beta + bh * T * (VAR == kF2 ? DV : 1);
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
        const int r = idx / DVS, c = idx % DVS;
        s.S[idx] = p.S0 ? p.S0[(bh * DK + r) * DV + c0 + c] : 0.f;
    }

    const int gl = kThreads / DVS;  // lanes cooperating on one column in the solve
    const int col = tid / gl, lg = tid % gl;

    for (long long t0 = 0; t0 < T; t0 += C) {
        const int n = (int)min((long long)C, T - t0);
        __syncthreads();  // previous chunk finished with every buffer
        // ---- (1) tiles. Extended row e <-> pair with global index pos + t0 + 2 - W + e.
        for (int idx = tid; idx < NE * DK; idx += kThreads) {
            const int e = idx / DK, cc = idx % DK;
            const long long gpair = pos + t0 + 2 - W + e;
            float x = 0.f;
            if (e < n + W - 1 && gpair >= 2) x = load_key(t0 - W + e, cc);
            s.X[e * XS + cc] = x;
        }
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int i = idx / DK, cc = idx % DK;
            s.Q[i * XS + cc] = i < n ? ldf(q + (t0 + i) * DK + cc) : 0.f;
        }
        for (int idx = tid; idx < NE * DVS; idx += kThreads) {
            const int e = idx / DVS, cc = idx % DVS;
            const long long gpair = pos + t0 + 2 - W + e;
            float y = 0.f;
            if (e < n + W - 1 && gpair >= 2) y = load_val(t0 + 1 - W + e, c0 + cc);
            s.Y[idx] = y;
        }
        __syncthreads();
        // ---- (2) Gram, scores, projected history, Q S
        for (int idx = tid; idx < NE * NE; idx += kThreads) {
            const int a = idx / NE, b = idx % NE;
            float acc = 0.f;
            for (int cc = 0; cc < DK; ++cc) acc = fmaf(s.X[a * XS + cc], s.X[b * XS + cc], acc);
            s.G[idx] = acc;
        }
        for (int idx = tid; idx < C * NE; idx += kThreads) {
            const int i = idx / NE, b = idx % NE;
            float acc = 0.f;
            for (int cc = 0; cc < DK; ++cc) acc = fmaf(s.Q[i * XS + cc], s.X[b * XS + cc], acc);
            s.Sc[idx] = acc;
        }
        for (int idx = tid; idx < NE * DVS; idx += kThreads) {
            const int e = idx / DVS, c = idx % DVS;
            float acc = 0.f;
            for (int cc = 0; cc < DK; ++cc) acc = fmaf(s.X[e * XS + cc], s.S[cc * DVS + c], acc);
            s.H[idx] = acc;
        }
        for (int idx = tid; idx < C * DVS; idx += kThreads) {
            const int i = idx / DVS, c = idx % DVS;
            float acc = 0.f;
            for (int cc = 0; cc < DK; ++cc) acc = fmaf(s.Q[i * XS + cc], s.S[cc * DVS + c], acc);
            s.QS[idx] = acc;
        }
        __syncthreads();
        // ---- (3) per-token scalars and the chunk-local log-decay prefix
        if (VAR == kF2) {
            if (tid < DVS) {
                const int c = tid;
                float run = 0.f;
                for (int i = 0; i < C; ++i) {
                    float eta = 0.f, alpha = 0.f;
                    const long long tau = pos + t0 + i + 1;
                    if (i < n && tau >= 2) {
                        const float lm = lam[t0 + i];
                        const float den = s.G[i * NE + i] + lm + p.eps;
                        eta = den == 0.f ? 0.f : beta[(t0 + i) * DV + c0 + c] / den;
                        alpha = fminf(eta * lm, 1.f - p.eps_gamma);
                    }
                    s.eta[c * CS + i] = eta;
                    s.Lx[c * CS + i] = run;
                    run += log1pf(-alpha);
                    s.L[c * CS + i] = run;
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
                    if (VAR == kF3) {
                        float a[kMaxW][kMaxW];
                        int slots[kMaxW];
                        int nb = 0;
                        for (int sl = 0; sl < W; ++sl)
                            if (tau - sl >= 2) slots[nb++] = i - sl + W - 1;
                        if (nb > 0) {
                            for (int x = 0; x < nb; ++x)
                                for (int y = 0; y < nb; ++y) a[x][y] = s.G[slots[x] * NE + slots[y]] / (float)nb;
                            const float mu = lambda_max_small(a, nb);
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
                    s.kap[i] = (VAR == kF3) ? kap : eta;
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
        if (VAR != kF2) {
            const float LC = s.L[C - 1];
            for (int idx = tid; idx < C * C; idx += kThreads) {
                const int i = idx / C, j = idx % C;
                float a = 0.f, pp = 0.f;
                if (j < i) a = s.kap[j] * expf(s.Lx[i] - s.L[j]);
                if (j <= i) pp = s.kap[j] * expf(s.L[i] - s.L[j]);
                if (VAR != kF3) {
                    a *= s.G[i * NE + j];
                    pp *= s.Sc[i * NE + j];
                }
                s.A[idx] = a;
                s.P[idx] = pp;
            }
            for (int j = tid; j < C; j += kThreads) s.w[j] = s.kap[j] * expf(LC - s.L[j]);
        } else {
            for (int idx = tid; idx < C * DVS; idx += kThreads) {
                const int j = idx / DVS, c = idx % DVS;
                s.w[c * CS + j] = s.eta[c * CS + j] * expf(s.L[c * CS + C - 1] - s.L[c * CS + j]);
            }
        }
        __syncthreads();
        // ---- (5) merged-RHS forward substitution, column `col`, `gl` lanes per column
        if (VAR == kF1 || VAR == kF2) {
            for (int i = 0; i < n; ++i) {
                float acc = 0.f;
                if (VAR == kF1) {
                    for (int j = lg; j < i; j += gl) acc = fmaf(s.A[i * C + j], s.R[col * RS + j], acc);
                } else {
                    const float lxi = s.Lx[col * CS + i];
                    for (int j = lg; j < i; j += gl)
                        acc = fmaf(s.eta[col * CS + j] * expf(lxi - s.L[col * CS + j]) * s.G[i * NE + j],
                                   s.R[col * RS + j], acc);
                }
                for (int o = gl >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                const float dcy = (VAR == kF1) ? expf(s.Lx[i]) : expf(s.Lx[col * CS + i]);
                const float r = (s.Y[i * DVS + col] - dcy * s.H[i * DVS + col]) - acc;
                if (lg == 0) s.R[col * RS + i] = r;
                __syncwarp();
            }
        } else if (VAR == kF3) {
            for (int i = 0; i < n; ++i) {
                const float dcy = expf(s.Lx[i]);
                for (int a = 0; a < W; ++a) {
                    const int pa = i - a + W - 1;
                    const bool valid = pos + t0 + i + 1 - a >= 2;
                    float acc = 0.f;
                    for (int m = lg; m < i * W; m += gl) {
                        const int l = m / W, b = m % W;
                        acc = fmaf(s.A[i * C + l] * s.G[pa * NE + (l - b + W - 1)], s.R[col * RS + m], acc);
                    }
                    for (int o = gl >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                    const float r = valid ? (s.Y[pa * DVS + col] - dcy * s.H[pa * DVS + col]) - acc : 0.f;
                    if (lg == 0) s.R[col * RS + i * W + a] = r;
                    __syncwarp();
                }
            }
        }
        __syncthreads();
        // ---- (6) outputs (read after write) and (7) carried state
        Tin* out = static_cast<Tin*>(p.out) + bh * T * DV;
        for (int idx = tid; idx < n * DVS; idx += kThreads) {
            const int i = idx / DVS, c = idx % DVS;
            float o;
            if (VAR == kF2) {
                const float li = s.L[c * CS + i];
                o = expf(li) * s.QS[idx];
                for (int j = 0; j <= i; ++j)
                    o = fmaf(s.eta[c * CS + j] * expf(li - s.L[c * CS + j]) * s.Sc[i * NE + j], s.R[c * RS + j], o);
            } else if (VAR == kF3) {
                o = expf(s.L[i]) * s.QS[idx];
                for (int l = 0; l <= i; ++l) {
                    const float f = s.P[i * C + l];
                    float acc = 0.f;
                    for (int b = 0; b < W; ++b) acc = fmaf(s.Sc[i * NE + (l - b + W - 1)], s.R[c * RS + l * W + b], acc);
                    o = fmaf(f, acc, o);
                }
            } else if (VAR == kF1A) {
                o = expf(s.L[i]) * s.QS[idx];
                for (int j = 0; j <= i; ++j) o = fmaf(s.P[i * C + j], s.Y[j * DVS + c], o);
            } else {
                o = expf(s.L[i]) * s.QS[idx];
                for (int j = 0; j <= i; ++j) o = fmaf(s.P[i * C + j], s.R[c * RS + j], o);
            }
            stf(out + (t0 + i) * DV + c0 + c, o);
        }
        for (int idx = tid; idx < DK * DVS; idx += kThreads) {
            const int r = idx / DVS, c = idx % DVS;
            float acc = 0.f;
            if (VAR == kF3) {
                for (int l = 0; l < n; ++l) {
                    float inner = 0.f;
                    for (int b = 0; b < W; ++b) inner = fmaf(s.X[(l - b + W - 1) * XS + r], s.R[c * RS + l * W + b], inner);
                    acc = fmaf(s.w[l], inner, acc);
                }
                s.S[idx] = fmaf(expf(s.L[C - 1]), s.S[idx], acc);
            } else if (VAR == kF2) {
                for (int j = 0; j < n; ++j) acc = fmaf(s.X[j * XS + r] * s.w[c * CS + j], s.R[c * RS + j], acc);
                s.S[idx] = fmaf(expf(s.L[c * CS + C - 1]), s.S[idx], acc);
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
    if (p.S_final)
        for (int idx = tid; idx < DK * DVS; idx += kThreads) {
            const int r = idx / DVS, c = idx % DVS;
            p.S_final[(bh * DK + r) * DV + c0 + c] = s.S[idx];
        }
    if (p.tail_out) {
        Tin* to = static_cast<Tin*>(p.tail_out) + bh * tail_stride;
        if (slice == 0)
            for (int idx = tid; idx < W * DK; idx += kThreads) {
                const int sl = idx / DK, cc = idx % DK;
                stf(to + idx, load_key(T - W + sl, cc));
            }
        for (int idx = tid; idx < (W - 1) * DVS; idx += kThreads) {
            const int sl = idx / DVS, cc = idx % DVS;
            stf(to + (long long)W * DK + sl * DV + c0 + cc, load_val(T - W + 1 + sl, c0 + cc));
        }
    }
}

template <typename Tin>
cudaError_t launch_typed(const Launch& a, const GParams& gp, dim3 grid, size_t smem, cudaStream_t st) {
    void (*fn)(GParams) = nullptr;
    switch (a.variant) {
        case kF1: fn = falcon_chunk_generic_kernel<Tin, kF1>; break;
        case kF1A: fn = falcon_chunk_generic_kernel<Tin, kF1A>; break;
        case kF2: fn = falcon_chunk_generic_kernel<Tin, kF2>; break;
        case kF3: fn = falcon_chunk_generic_kernel<Tin, kF3>; break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(gp);
    return cudaGetLastError();
}

int choose_dvs(const Launch& a) {
    // Enough CTAs to cover the GPU twice over, slices no narrower than 16 columns,
    // and a shared-memory footprint that fits one CTA.
    int dvs = (int)a.dv;
    const int64_t seqs = a.B * a.H;
    while (dvs > 16 && seqs * (a.dv / dvs) < 2 * 152) dvs /= 2;
    while (dvs > 16 && generic_smem_bytes(a, dvs) > 200 * 1024) dvs /= 2;
    return dvs;
}

}  // namespace

size_t generic_smem_bytes(const Launch& a, int dvs) {
    const int W = a.variant == kF3 ? a.W : 1;
    return smem_floats(a.variant, (int)a.dk, dvs, a.chunk, W, nullptr, nullptr) * sizeof(float);
}

int launch_generic(const Launch& a, cudaStream_t st) {
    if (a.B * a.H == 0) return 0;
    const int dvs = choose_dvs(a);
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
    gp.W = a.variant == kF3 ? a.W : 1;
    gp.eps = a.eps;
    gp.eps_gamma = a.eps_gamma;
    const size_t smem = generic_smem_bytes(a, dvs);
    dim3 grid((unsigned)((a.dv / dvs) * a.B * a.H));
    cudaError_t e = a.bf16 ? launch_typed<__nv_bfloat16>(a, gp, grid, smem, st)
                           : launch_typed<float>(a, gp, grid, smem, st);
    return e == cudaSuccess ? 0 : 4;
}

}  // namespace falcon
