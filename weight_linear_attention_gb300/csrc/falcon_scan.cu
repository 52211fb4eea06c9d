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
//   2. scan  (this file), groups of G = 16 chunks (with many sequences x groups: enough chunks per
//            group that one CTA per group fills two slots of every SM):
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
constexpr int kGroup = 16;    // chunks per group (the workspace holds the group blocks for this size)
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
    long long G;    // chunks per group (compose, apply)
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
        first = gi * p.G;
        nsteps = min(p.G, p.N - first);
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


// The compose and apply passes with one CTA per group over every state column at once, so that each
// chunk's maps are read from memory once. A step is one product of stacked operands:
//   compose  [M_g | U_g] <- M_n [M_g | U_g] + [0 | U_n]      (state 64 x 128, from the group's first map)
//   apply    [S' ; O_n]  <- [M_n ; Ao_n] S + [U_n ; Bo_n]      (state 64 x 64; 64 + C rows)
// Thread (rg, cq) owns rows rg + 16 i and columns 4 cq .. 4 cq + 3 of each 64-column half; a warp spans
// four row groups and eight column quads, so that one read of a state row covers 128 contiguous bytes
// and one read of the stacked operand touches four rows in four different banks. M and Ao arrive
// through a two-stage ring of 16-byte asynchronous copies issued one step ahead; U and Bo go straight
// to registers at the start of the step and are added after the product, which keeps the shared memory
// low enough for two CTAs per SM. CR = C / 16 output rows per thread (0: compose).
template <int CR>
__global__ void __launch_bounds__(kThreads, 2) falcon_scan_wide_kernel(const ScanParams p) {
    extern __shared__ __align__(16) float sm[];
    constexpr int NH = CR == 0 ? 2 : 1;   // 64-column halves of the state
    constexpr int SLD = 64 * NH + 4;      // state row stride (floats)
    constexpr int NR = 4 + CR;            // operand rows per thread
    constexpr int SF = (kD + 16 * CR) * kLdc;  // floats of one ring stage
    float* const S = sm + 2 * SF;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = (lane & 7) + 8 * (warp & 1), rg = (lane >> 3) + 4 * (warp >> 1);
    const long long bh = blockIdx.x / p.NG, gi = blockIdx.x % p.NG;
    const float* const chunks = p.ws + bh * p.N * kBlk;
    float* const groups = p.ws + (p.BH * p.N + bh * p.NG) * kBlk;
    const long long first = gi * p.G, nsteps = min(p.G, p.N - first);

    auto issue = [&](long long j) {
        if (j < nsteps) {
            const float* b = chunks + (first + j) * kBlk;
            float* d = sm + (int)(j & 1) * SF;
#pragma unroll
            for (int u = 0; u < NR; ++u) {  // rows 0..63: M; rows 64..: Ao (the block's fourth matrix)
                const int e = tid + u * kThreads, row = e >> 4, col = 4 * (e & 15);
                cp_async16(d + row * kLdc + col, b + (row < kD ? row * kD : 3 * kMat + (row - kD) * kD) + col);
            }
        }
        cp_async_commit();
    };

    // the state entering the first step: compose starts from the group's first map itself
    {
        const float* src = nullptr;
        if (CR == 0) src = chunks + first * kBlk;
        else if (p.NG > 1) src = groups + gi * kBlk + 2 * kMat;
        else if (p.S0) src = p.S0 + bh * kMat;
        for (int e = tid; e < kD * 64 * NH; e += kThreads) {
            const int r = e / (64 * NH), c = e % (64 * NH);
            S[r * SLD + c] = src ? src[(c < kD ? 0 : kMat) + r * kD + (c & 63)] : 0.f;
        }
    }
    const long long j0 = CR == 0 ? 1 : 0;
    issue(j0);
    for (long long j = j0; j < nsteps; ++j) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();  // this step's operands and the state are in place; the other stage is free
        issue(j + 1);
        const float* bj = chunks + (first + j) * kBlk;
        float4 off[4], bo[CR > 0 ? CR : 1];
#pragma unroll
        for (int i = 0; i < 4; ++i) off[i] = __ldg(reinterpret_cast<const float4*>(bj + kMat + (rg + 16 * i) * kD) + cq);
#pragma unroll
        for (int i = 0; i < CR; ++i) bo[i] = __ldg(reinterpret_cast<const float4*>(bj + 4 * kMat + (rg + 16 * i) * kD) + cq);
        const float* A = sm + (int)(j & 1) * SF;
        float4 acc[NR][NH];
#pragma unroll
        for (int i = 0; i < NR; ++i)
#pragma unroll
            for (int h = 0; h < NH; ++h) acc[i][h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int k = 0; k < kD; k += 4) {
            float4 a[NR];
#pragma unroll
            for (int i = 0; i < NR; ++i) a[i] = *reinterpret_cast<const float4*>(A + (rg + 16 * i) * kLdc + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float4 s[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) s[h] = *reinterpret_cast<const float4*>(S + (k + kk) * SLD + 64 * h + 4 * cq);
#pragma unroll
                for (int i = 0; i < NR; ++i) {
                    const float m = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        acc[i][h].x = fmaf(m, s[h].x, acc[i][h].x);
                        acc[i][h].y = fmaf(m, s[h].y, acc[i][h].y);
                        acc[i][h].z = fmaf(m, s[h].z, acc[i][h].z);
                        acc[i][h].w = fmaf(m, s[h].w, acc[i][h].w);
                    }
                }
            }
        }
        if constexpr (CR > 0) {  // the chunk's outputs O = Ao S + Bo (the ragged last chunk: rows < T)
            const long long t0 = (first + j) * p.C;
#pragma unroll
            for (int i = 0; i < CR; ++i) {
                const int r = rg + 16 * i;
                if (t0 + r >= p.T) continue;
                const float4 o = make_float4(acc[4 + i][0].x + bo[i].x, acc[4 + i][0].y + bo[i].y,
                                             acc[4 + i][0].z + bo[i].z, acc[4 + i][0].w + bo[i].w);
                const long long at = (bh * p.T + t0 + r) * kD + 4 * cq;
                if (p.bf16) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
                    uint2 w;
                    w.x = *reinterpret_cast<uint32_t*>(&lo);
                    w.y = *reinterpret_cast<uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + at) = w;
                } else {
                    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + at) = o;
                }
            }
        }
        __syncthreads();  // every read of the state is done
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                float4 v = acc[i][h];
                if (h == NH - 1) v.x += off[i].x, v.y += off[i].y, v.z += off[i].z, v.w += off[i].w;
                *reinterpret_cast<float4*>(S + (rg + 16 * i) * SLD + 64 * h + 4 * cq) = v;
            }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    if (CR == 0) {  // the group's map [M_g | U_g]
        float* g = groups + gi * kBlk;
        for (int e = tid; e < kD * 128; e += kThreads) {
            const int r = e >> 7, c = e & 127;
            g[(c < kD ? 0 : kMat) + r * kD + (c & 63)] = S[r * SLD + c];
        }
    } else if (gi == p.NG - 1 && p.S_final) {
        for (int e = tid; e < kD * kD; e += kThreads) p.S_final[bh * kMat + e] = S[(e >> 6) * SLD + (e & 63)];
    }
}
template <int CR>
constexpr size_t wide_smem_bytes() {
    return (size_t)(2 * (kD + 16 * CR) * kLdc + kD * (64 * (CR == 0 ? 2 : 1) + 4)) * sizeof(float);
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
    ScanParams p{ws, a.S0, a.S_final, a.out, BH, N, NG, a.T, kGroup, a.chunk, a.bf16, 0};
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 4;
    if (BH * NG >= sms) {  // enough groups for one CTA per SM: each map read once, all columns per CTA
        // the fewest groups that still fill the two CTA slots of every SM (never more groups than the
        // workspace's blocks for groups of 16)
        const long long want = max(1LL, min(NG, 2LL * sms / BH));
        p.G = (N + want - 1) / want;
        p.NG = (N + p.G - 1) / p.G;
        const int C = a.chunk;
        const size_t sm0 = wide_smem_bytes<0>(), sm1 = wide_smem_bytes<1>(), sm2 = wide_smem_bytes<2>(),
                     sm4 = wide_smem_bytes<4>();
        static_assert(wide_smem_bytes<4>() <= 113 * 1024, "two wide-scan CTAs per SM");
        if (cudaFuncSetAttribute(falcon_scan_wide_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm0) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_scan_wide_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_scan_wide_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2) !=
                cudaSuccess ||
            cudaFuncSetAttribute(falcon_scan_wide_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm4) !=
                cudaSuccess)
            return 4;
        const unsigned grid = (unsigned)(BH * p.NG);
        if (p.NG > 1) {
            p.mode = 0;
            falcon_scan_wide_kernel<0><<<grid, kThreads, sm0, st>>>(p);
            p.mode = 1;  // the short pass over the groups: 16-column slices
            falcon_scan_kernel<<<(unsigned)(BH * 4), kThreads, smem_bytes(0), st>>>(p);
        }
        p.mode = 2;
        if (C == 16) falcon_scan_wide_kernel<1><<<grid, kThreads, sm1, st>>>(p);
        else if (C == 32) falcon_scan_wide_kernel<2><<<grid, kThreads, sm2, st>>>(p);
        else falcon_scan_wide_kernel<4><<<grid, kThreads, sm4, st>>>(p);
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
