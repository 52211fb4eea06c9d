// Scan path for long sequences with few (batch, head) pairs: the chunk-to-chunk state pass as an
// associative scan over the chunks' affine maps ("Fast Weight Attention for Continual Learning",
// paperlayer summary §H.1: chunk maps compose associatively, so the sequential phase can be a scan;
// §H.2; §E.2 for the three-phase structure).
//
// For Falcon-1, 1A, 3 and 3A every chunk acts on the carried state as S -> M_n S + U_n with M_n, U_n
// fixed by the chunk's inputs alone (the transition is shared by all value columns). With dk = dv = 64:
//   1. map   (CUDA-core chunk kernel, map mode): every chunk's M_n and U_n at once;
//   2. scan  (this file), groups of G = 16 chunks:
//        compose  every group's map (M_g, U_g) = (M_last ... M_first, ...) at once,
//        groups   per sequence, S_{g+1} = M_g S_g + U_g over the groups,
//        apply    every group at once, S_{n+1} = M_n S_n + U_n from the group's start state,
//                 storing each chunk's start state S_n (and S_final from the last group);
//      a sequence of N chunks takes 2 G + N / G dependent steps instead of N;
//   3. read  (CUDA-core chunk kernel, read mode): every chunk's outputs at once from its S_n.
// Workspace: per chunk (sequence-major) and then per group, blocks [M | U | S] of 64 x 64 fp32; for
// Falcon-3 then every token's window normaliser (computed once by a one-thread-per-token kernel and read
// by the map and read passes).

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
constexpr long long kBlk = 3 * kMat;  // [M | U | S]
constexpr size_t kSmem = (size_t)kStages * (kD * kLdc + kD * kCols) * sizeof(float) + 2 * kCols * kLdc * sizeof(float);

struct ScanParams {
    float* ws;
    const float* S0;
    float* S_final;
    long long BH, N, NG;
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
    float* Ms = sm;                              // [kStages][kD * kLdc]
    float* Os = Ms + kStages * kD * kLdc;        // [kStages][kD][kCols]
    float (*Sv)[kCols][kLdc] = reinterpret_cast<float (*)[kCols][kLdc]>(Os + kStages * kD * kCols);  // [2]
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
                cp_async16(Ms + st * kD * kLdc + row * kLdc + col, b + e);
            }
            if (has_off) {
                const int row = threadIdx.x >> 2, q = 4 * (threadIdx.x & 3);
                cp_async16(Os + (st * kD + row) * kCols + q, b + kMat + row * kD + cg + q);
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
        if (p.mode != 0) {  // the state entering this step: a chunk's (apply) or a group's (groups) start state
            float* so = blk(j) + 2 * kMat + cg + c;
#pragma unroll
            for (int z = 0; z < 4; ++z) so[(r0 + z) * kD] = Sv[b][c][r0 + z];
        }
        const float* Mk = Ms + st * kD * kLdc;
        const float* off = Os + st * kD * kCols + c;
        const float* Sc = Sv[b][c];
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

}  // namespace

bool scan_supported(const Launch& a) {
    const bool shared = a.variant == kF1 || a.variant == kF1A || a.variant == kF3 || a.variant == kF3A;
    const long long N = (a.T + a.chunk - 1) / a.chunk;
    // few sequences (the one-CTA-per-slice kernel would leave SMs idle) and enough chunks to split
    return shared && a.dk == kD && a.dv == kD && a.B * a.H * (kD / 16) < 2 * 152 && N >= 4 && !split_supported(a);
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
    int e = launch_generic_mode(a, 1, ws, N, mu, st);
    if (e) return e;
    static_assert(kSmem <= 227 * 1024, "scan kernel shared memory");
    if (cudaFuncSetAttribute(falcon_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) !=
        cudaSuccess)
        return 4;
    ScanParams p{ws, a.S0, a.S_final, BH, N, NG, 0};
    if (NG > 1) {
        p.mode = 0;
        falcon_scan_kernel<<<(unsigned)(BH * NG * 8), kThreads, kSmem, st>>>(p);
        p.mode = 1;
        falcon_scan_kernel<<<(unsigned)(BH * 4), kThreads, kSmem, st>>>(p);
    }
    p.mode = 2;
    falcon_scan_kernel<<<(unsigned)(BH * NG * 4), kThreads, kSmem, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return 4;
    return launch_generic_mode(a, 2, ws, N, mu, st);
}

}  // namespace falcon
