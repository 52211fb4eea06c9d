// Scan path for long sequences with few (batch, head) pairs: the chunk-to-chunk state pass as an
// associative scan over the chunks' affine maps ("Fast Weight Attention for Continual Learning",
// paperlayer summary §H.1: chunk maps compose associatively, so the sequential phase can be a scan;
// §H.2; §E.2 for the three-phase structure).
//
// For Falcon-1, 1A, 3 and 3A every chunk acts on the carried state as S -> M_n S + U_n, and its
// outputs are O_n = Ao_n S_n + Bo_n, with M_n, U_n, Ao_n, Bo_n fixed by the chunk's inputs alone (the
// transition is shared by all value columns). With dk = dv = 64:
//   1. map   every chunk's four maps at once: for Falcon-3 and 3A at W = 4, chunk 32, bf16 on the
//            tensor cores (falcon_f3map.cu; a chunk whose decay is too strong for its factored form
//            is left to the CUDA-core kernel), otherwise the CUDA-core chunk kernel in map mode;
//   2. scan  (this file), groups of G = 16 chunks:
//        compose  every group's map (M_g, U_g) = (M_last ... M_first, ...) at once,
//        groups   per sequence, S_{g+1} = M_g S_g + U_g over the groups,
//        apply    every group at once, from the group's start state: O_n = Ao_n S_n + Bo_n, then
//                 S_{n+1} = M_n S_n + U_n (and S_final from the last group);
//      a sequence of N chunks takes 2 G + N / G dependent steps instead of N.
// Workspace: per chunk (sequence-major) and then per group, blocks [M | U | S | Ao | Bo] of 64 x 64 fp32
// (Ao, Bo: C rows used; S: a group's start state); for Falcon-3 then every token's window normaliser
// (computed once by a one-thread-per-token kernel and read by the map pass).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "falcon_internal.h"

namespace falcon {
namespace {

constexpr int kD = 64;
constexpr int kCols = 16;     // state columns per CTA
constexpr int kLdc = 68;      // 16-byte aligned rows
constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr int kGroup = 16;    // chunks per group
constexpr long long kMat = kD * kD;
constexpr long long kBlk = 5 * kMat;  // [M | U | S | Ao | Bo]
// shared floats of one ring stage: M, the offset columns, and (apply) the output maps' rows
__host__ __device__ constexpr int stage_floats(int C) { return kD * kLdc + kD * kCols + C * (kLdc + kCols); }
constexpr size_t smem_bytes(int C) { return ((size_t)kStages * stage_floats(C) + 2 * kCols * kLdc) * sizeof(float); }

struct ScanParams {
    float* ws;
    const float* S0;
    float* S_final;
    void* out;      // apply: [B*H][T][64] in the input dtype
    long long BH, N, NG, T;
    int C;          // chunk length (apply: rows of Ao, Bo)
    int bf16;
    int mode;  // 0 compose, 1 groups, 2 apply
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// Thread (r4, c) owns rows 4 r4 .. 4 r4 + 3 of state column c; the state slice is kept transposed so
// that a thread reads four consecutive k of its column at once. Each step's M (row-major) and offset
// columns arrive through a three-stage ring of 16-byte asynchronous copies issued two steps ahead.
__global__ void __launch_bounds__(kThreads) falcon_scan_kernel(const ScanParams p) {
    extern __shared__ __align__(16) float sm[];
    const int Cr = p.mode == 2 ? p.C : 0;       // output rows fetched per step
    const int SF = stage_floats(Cr);
    // stage st: M [kD][kLdc] | offsets [kD][kCols] | Ao [Cr][kLdc] | Bo [Cr][kCols]
    auto Mst = [&](int st) { return sm + st * SF; };
    auto Ost = [&](int st) { return sm + st * SF + kD * kLdc; };
    auto Ast = [&](int st) { return sm + st * SF + kD * kLdc + kD * kCols; };
    auto Bst = [&](int st) { return sm + st * SF + kD * kLdc + kD * kCols + Cr * kLdc; };
    float (*Sv)[kCols][kLdc] = reinterpret_cast<float (*)[kCols][kLdc]>(sm + kStages * SF);  // [2]
    const int c = threadIdx.x & 15, r0 = 4 * (threadIdx.x >> 4);
    const long long bid = blockIdx.x;
    long long bh, gi = 0;
    int cg, part = 1;  // part 0: the columns of M_g (compose only)
    if (p.mode == 0) {
        const int vs = (int)(bid % 8);
        gi = (bid / 8) % p.NG;
        bh = bid / (8 * p.NG);
        part = vs / 4;
        cg = kCols * (vs % 4);
    } else if (p.mode == 1) {
        cg = kCols * (int)(bid % 4);
        bh = bid / 4;
    } else {
        cg = kCols * (int)(bid % 4);
        gi = (bid / 4) % p.NG;
        bh = bid / (4 * p.NG);
    }
    float* const chunks = p.ws + bh * p.N * kBlk;                      // this sequence's chunk blocks
    float* const groups = p.ws + (p.BH * p.N + bh * p.NG) * kBlk;      // and group blocks
    // steps j = 0 .. nsteps - 1 apply the block blk(j)
    long long first = 0, nsteps;
    if (p.mode == 1) nsteps = p.NG;
    else {
        first = gi * kGroup;
        nsteps = min((long long)kGroup, p.N - first);
    }
    auto blk = [&](long long j) -> float* { return p.mode == 1 ? groups + j * kBlk : chunks + (first + j) * kBlk; };
    const bool has_off = part != 0;

    auto issue = [&](long long j) {
        if (j < nsteps) {
            const int st = (int)(j % kStages);
            const float* b = blk(j);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = 4 * (threadIdx.x + u * kThreads), row = e >> 6, col = e & 63;
                cp_async16(Mst(st) + row * kLdc + col, b + e);
            }
            if (has_off) {
                const int row = threadIdx.x >> 2, q = 4 * (threadIdx.x & 3);
                cp_async16(Ost(st) + row * kCols + q, b + kMat + row * kD + cg + q);
            }
            for (int e = threadIdx.x; e < Cr * 16; e += kThreads) {  // Ao rows, 16-byte pieces
                const int row = e >> 4, col = 4 * (e & 15);
                cp_async16(Ast(st) + row * kLdc + col, b + 3 * kMat + row * kD + col);
            }
            for (int e = threadIdx.x; e < Cr * 4; e += kThreads) {   // Bo rows, this CTA's columns
                const int row = e >> 2, q = 4 * (e & 3);
                cp_async16(Bst(st) + row * kCols + q, b + 4 * kMat + row * kD + cg + q);
            }
        }
        cp_async_commit();
    };

    // initial state slice
    const float* init = nullptr;
    if (p.mode == 1 || (p.mode == 2 && p.NG == 1)) init = p.S0 ? p.S0 + bh * kMat : nullptr;
    else if (p.mode == 2) init = groups + gi * kBlk + 2 * kMat;
#pragma unroll
    for (int z = 0; z < 4; ++z) {
        const int r = r0 + z;
        float x = 0.f;
        if (p.mode == 0) x = (part == 0 && r == cg + c) ? 1.f : 0.f;
        else if (init) x = init[r * kD + cg + c];
        Sv[0][c][r] = x;
    }
    issue(0);
    issue(1);
    int b = 0;
    for (long long j = 0; j < nsteps; ++j, b ^= 1) {
        const int st = (int)(j % kStages);
        issue(j + 2);
        cp_async_wait2();
        __syncthreads();
        const float* Sc = Sv[b][c];
        if (p.mode == 1) {  // the state entering this group
            float* so = blk(j) + 2 * kMat + cg + c;
#pragma unroll
            for (int z = 0; z < 4; ++z) so[(r0 + z) * kD] = Sv[b][c][r0 + z];
        } else if (p.mode == 2) {  // the chunk's outputs from the state entering it: O = Ao S + Bo
            const long long t0 = (first + j) * p.C;
            const int rows = (int)min((long long)p.C, p.T - t0);
            const float* Ak = Ast(st);
            const float* Bk = Bst(st);
            for (int i = threadIdx.x >> 4; i < rows; i += kThreads / 16) {
                float o = Bk[i * kCols + c];
#pragma unroll 4
                for (int k = 0; k < kD; k += 4) {
                    const float4 sv = *reinterpret_cast<const float4*>(Sc + k);
                    const float4 av = *reinterpret_cast<const float4*>(Ak + i * kLdc + k);
                    o = fmaf(av.x, sv.x, fmaf(av.y, sv.y, fmaf(av.z, sv.z, fmaf(av.w, sv.w, o))));
                }
                const long long at = (bh * p.T + t0 + i) * kD + cg + c;
                if (p.bf16) static_cast<__nv_bfloat16*>(p.out)[at] = __float2bfloat16_rn(o);
                else static_cast<float*>(p.out)[at] = o;
            }
        }
        const float* Mk = Mst(st);
        const float* off = Ost(st) + c;
        float acc[4];
#pragma unroll
        for (int z = 0; z < 4; ++z) acc[z] = has_off ? off[(r0 + z) * kCols] : 0.f;
#pragma unroll 4
        for (int k = 0; k < kD; k += 4) {
            const float4 sv = *reinterpret_cast<const float4*>(Sc + k);
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const float4 mv = *reinterpret_cast<const float4*>(Mk + (r0 + z) * kLdc + k);
                acc[z] = fmaf(mv.x, sv.x, fmaf(mv.y, sv.y, fmaf(mv.z, sv.z, fmaf(mv.w, sv.w, acc[z]))));
            }
        }
        *reinterpret_cast<float4*>(Sv[b ^ 1][c] + r0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncthreads();
    }
    // the result is in Sv[b]
    float* dst = nullptr;
    if (p.mode == 0) dst = groups + gi * kBlk + (part == 0 ? 0 : kMat);
    else if (p.mode == 2 && gi == p.NG - 1 && p.S_final) dst = p.S_final + bh * kMat;
    if (dst)
#pragma unroll
        for (int z = 0; z < 4; ++z) dst[(r0 + z) * kD + cg + c] = Sv[b][c][r0 + z];
}


// The same three modes with one CTA per group (mode 1: per sequence) over every state column at once
// (mode 0: the 64 columns of M_g and the 64 of U_g together), so that each chunk's maps are read from
// memory once instead of once per 16-column slice. Thread (rg, cg) owns rows 4 rg .. 4 rg + 3 and
// NCOL / 16 consecutive columns; the state is kept row-major in shared memory; each step's maps arrive
// through a two-stage ring of 16-byte asynchronous copies issued one step ahead.
template <int NCOL>
__global__ void __launch_bounds__(kThreads, 1) falcon_scan_wide_kernel(const ScanParams p) {
    extern __shared__ __align__(16) float sm[];
    constexpr int LD = kLdc, SLD = NCOL + 4, CW = NCOL / 16;
    const int Cr = p.mode == 2 ? p.C : 0;  // output rows fetched per step
    const int MF = kD * LD, AF = Cr * LD, SF = 2 * MF + 2 * AF;
    auto Mst = [&](int st) { return sm + st * SF; };
    auto Ust = [&](int st) { return sm + st * SF + MF; };
    auto Ast = [&](int st) { return sm + st * SF + 2 * MF; };
    auto Bst = [&](int st) { return sm + st * SF + 2 * MF + AF; };
    float* const Sbase = sm + 2 * SF;  // two state buffers [kD][SLD]
    const int tid = threadIdx.x, rg = tid >> 4, c0 = CW * (tid & 15);
    const long long bid = blockIdx.x;
    const long long bh = p.mode == 1 ? bid : bid / p.NG, gi = p.mode == 1 ? 0 : bid % p.NG;
    float* const chunks = p.ws + bh * p.N * kBlk;
    float* const groups = p.ws + (p.BH * p.N + bh * p.NG) * kBlk;
    long long first = 0, nsteps;
    if (p.mode == 1) nsteps = p.NG;
    else {
        first = gi * kGroup;
        nsteps = min((long long)kGroup, p.N - first);
    }
    auto blk = [&](long long j) -> float* { return p.mode == 1 ? groups + j * kBlk : chunks + (first + j) * kBlk; };

    auto issue = [&](long long j) {
        if (j < nsteps) {
            const int st = (int)(j & 1);
            const float* b = blk(j);
            for (int e = tid; e < 2 * kD * 16; e += kThreads) {  // M and U, 16-byte pieces
                const int which = e >> 10, row = (e >> 4) & 63, col = 4 * (e & 15);
                cp_async16((which ? Ust(st) : Mst(st)) + row * LD + col, b + which * kMat + row * kD + col);
            }
            for (int e = tid; e < 2 * Cr * 16; e += kThreads) {  // Ao and Bo rows
                const int which = e / (Cr * 16), r = e % (Cr * 16), row = r >> 4, col = 4 * (r & 15);
                cp_async16((which ? Bst(st) : Ast(st)) + row * LD + col, b + (3 + which) * kMat + row * kD + col);
            }
        }
        cp_async_commit();
    };

    // initial state
    const float* init = nullptr;
    if (p.mode == 1 || (p.mode == 2 && p.NG == 1)) init = p.S0 ? p.S0 + bh * kMat : nullptr;
    else if (p.mode == 2) init = groups + gi * kBlk + 2 * kMat;
    for (int e = tid; e < kD * NCOL; e += kThreads) {
        const int r = e / NCOL, c = e % NCOL;
        float x = 0.f;
        if (p.mode == 0) x = (c < kD && r == c) ? 1.f : 0.f;
        else if (init) x = init[r * kD + c];
        Sbase[r * SLD + c] = x;
    }
    issue(0);
    int b = 0;
    for (long long j = 0; j < nsteps; ++j, b ^= 1) {
        const int st = (int)(j & 1);
        issue(j + 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();
        const float* S = Sbase + b * kD * SLD;
        if (p.mode == 1) {  // the state entering this group
            float* so = blk(j) + 2 * kMat;
            for (int e = tid; e < kD * kD; e += kThreads) so[e] = S[(e >> 6) * SLD + (e & 63)];
        } else if (p.mode == 2) {  // the chunk's outputs from the state entering it: O = Ao S + Bo
            const long long t0 = (first + j) * p.C;
            const int rows = (int)min((long long)p.C, p.T - t0);
            const float* Ak = Ast(st);
            const float* Bk = Bst(st);
            for (int i = rg; i < rows; i += 16) {
                float o[CW];
#pragma unroll
                for (int z = 0; z < CW; ++z) o[z] = Bk[i * LD + c0 + z];
#pragma unroll 4
                for (int k = 0; k < kD; ++k) {
                    const float a = Ak[i * LD + k];
#pragma unroll
                    for (int z = 0; z < CW; ++z) o[z] = fmaf(a, S[k * SLD + c0 + z], o[z]);
                }
                const long long at = (bh * p.T + t0 + i) * kD + c0;
#pragma unroll
                for (int z = 0; z < CW; ++z) {
                    if (p.bf16) static_cast<__nv_bfloat16*>(p.out)[at + z] = __float2bfloat16_rn(o[z]);
                    else static_cast<float*>(p.out)[at + z] = o[z];
                }
            }
        }
        // S' = M S + U (mode 0: + U only on the U part's columns)
        const float* Mk = Mst(st);
        const float* Uk = Ust(st);
        float acc[4][CW];
#pragma unroll
        for (int z = 0; z < 4; ++z)
#pragma unroll
            for (int y = 0; y < CW; ++y) {
                const int c = c0 + y;
                acc[z][y] = p.mode == 0 ? (c >= kD ? Uk[(4 * rg + z) * LD + c - kD] : 0.f) : Uk[(4 * rg + z) * LD + c];
            }
#pragma unroll 2
        for (int k = 0; k < kD; k += 4) {
            float4 mv[4];
#pragma unroll
            for (int z = 0; z < 4; ++z) mv[z] = *reinterpret_cast<const float4*>(Mk + (4 * rg + z) * LD + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float sv[CW];
#pragma unroll
                for (int y = 0; y < CW; y += 4) {
                    const float4 v4 = *reinterpret_cast<const float4*>(S + (k + kk) * SLD + c0 + y);
                    sv[y] = v4.x, sv[y + 1] = v4.y, sv[y + 2] = v4.z, sv[y + 3] = v4.w;
                }
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    const float m = kk == 0 ? mv[z].x : kk == 1 ? mv[z].y : kk == 2 ? mv[z].z : mv[z].w;
#pragma unroll
                    for (int y = 0; y < CW; ++y) acc[z][y] = fmaf(m, sv[y], acc[z][y]);
                }
            }
        }
        float* So = Sbase + (b ^ 1) * kD * SLD;
#pragma unroll
        for (int z = 0; z < 4; ++z)
#pragma unroll
            for (int y = 0; y < CW; y += 4)
                *reinterpret_cast<float4*>(So + (4 * rg + z) * SLD + c0 + y) =
                    make_float4(acc[z][y], acc[z][y + 1], acc[z][y + 2], acc[z][y + 3]);
        __syncthreads();
    }
    const float* S = Sbase + b * kD * SLD;  // the result
    if (p.mode == 0) {
        float* g = groups + gi * kBlk;
        for (int e = tid; e < kD * NCOL; e += kThreads) {
            const int r = e / NCOL, c = e % NCOL;
            g[(c < kD ? 0 : kMat) + r * kD + (c & 63)] = S[r * SLD + c];
        }
    } else if (p.mode == 2 && gi == p.NG - 1 && p.S_final) {
        for (int e = tid; e < kD * kD; e += kThreads) p.S_final[bh * kMat + e] = S[(e >> 6) * SLD + (e & 63)];
    }
}
template <int NCOL>
constexpr size_t wide_smem_bytes(int C) {
    return (size_t)(2 * (2 * kD * kLdc + 2 * C * kLdc) + 2 * kD * (NCOL + 4)) * sizeof(float);
}
}  // namespace

bool scan_supported(const Launch& a) {
    const bool shared = a.variant == kF1 || a.variant == kF1A || a.variant == kF3 || a.variant == kF3A;
    const long long N = (a.T + a.chunk - 1) / a.chunk;
    // few sequences (the one-CTA-per-slice kernel would leave SMs idle) and enough chunks to split
    return shared && a.dk == kD && a.dv == kD && a.B * a.H * (kD / 16) < 2 * 152 && N >= 4 && !fused_supported(a);
}

size_t scan_workspace_bytes(const Launch& a) {
    const long long N = (a.T + a.chunk - 1) / a.chunk, NG = (N + kGroup - 1) / kGroup;
    const size_t mu = a.variant == kF3 ? (size_t)(a.B * a.H * a.T) * sizeof(float) : 0;  // Falcon-3 normalisers
    return (size_t)(a.B * a.H) * (size_t)(N + NG) * (size_t)kBlk * sizeof(float) + mu;
}

int launch_scan(const Launch& a, cudaStream_t st) {
    const long long BH = a.B * a.H, N = (a.T + a.chunk - 1) / a.chunk, NG = (N + kGroup - 1) / kGroup;
    float* ws = static_cast<float*>(a.ws);
    float* mu = nullptr;
    if (a.variant == kF3) {
        mu = ws + BH * (N + NG) * kBlk;
        if (launch_window_mu(a, mu, st)) return 4;
    }
    // chunk maps: on the tensor cores where that kernel applies (the CUDA-core kernel then takes only
    // the chunks it left unmarked), else on the CUDA cores
    const bool tc = f3map_supported(a);
    if (tc && launch_f3map(a, ws, N, mu, st)) return 4;
    int e = launch_generic_mode(a, 1, ws, N, mu, st, tc);
    if (e) return e;
    static_assert(smem_bytes(64) <= 227 * 1024, "scan kernel shared memory");
    if (cudaFuncSetAttribute(falcon_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(a.chunk)) !=
        cudaSuccess)
        return 4;
    ScanParams p{ws, a.S0, a.S_final, a.out, BH, N, NG, a.T, a.chunk, a.bf16, 0};
    if (BH * NG >= 152) {  // enough groups to fill the GPU with one CTA each: every map read once
        static_assert(wide_smem_bytes<128>(0) <= 227 * 1024 && wide_smem_bytes<64>(64) <= 227 * 1024, "wide scan");
        if (cudaFuncSetAttribute(falcon_scan_wide_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)wide_smem_bytes<128>(0)) != cudaSuccess ||
            cudaFuncSetAttribute(falcon_scan_wide_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)wide_smem_bytes<64>(a.chunk)) != cudaSuccess)
            return 4;
        if (NG > 1) {
            p.mode = 0;
            falcon_scan_wide_kernel<128><<<(unsigned)(BH * NG), kThreads, wide_smem_bytes<128>(0), st>>>(p);
            p.mode = 1;
            falcon_scan_wide_kernel<64><<<(unsigned)BH, kThreads, wide_smem_bytes<64>(0), st>>>(p);
        }
        p.mode = 2;
        falcon_scan_wide_kernel<64><<<(unsigned)(BH * NG), kThreads, wide_smem_bytes<64>(a.chunk), st>>>(p);
        return cudaGetLastError() == cudaSuccess ? 0 : 4;
    }
    if (NG > 1) {
        p.mode = 0;
        falcon_scan_kernel<<<(unsigned)(BH * NG * 8), kThreads, smem_bytes(0), st>>>(p);
        p.mode = 1;
        falcon_scan_kernel<<<(unsigned)(BH * 4), kThreads, smem_bytes(0), st>>>(p);
    }
    p.mode = 2;
    falcon_scan_kernel<<<(unsigned)(BH * NG * 4), kThreads, smem_bytes(a.chunk), st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

}  // namespace falcon
