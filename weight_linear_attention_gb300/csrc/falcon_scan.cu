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
//            group that one CTA per group fills two slots of every SM, and compose and apply on the
//            tensor cores, each map read once):
//        compose  every group's map (M_g, U_g) = (M_last ... M_first, ...) at once,
//        groups   per sequence, S_{g+1} = M_g S_g + U_g over the groups,
//        apply    every group at once, from the group's start state: O_n = Ao_n S_n + Bo_n, then
//                 S_{n+1} = M_n S_n + U_n (and S_final from the last group);
//      a sequence of N chunks takes 2 G + N / G dependent steps instead of N.
// Workspace: per chunk (sequence-major) and then per group, blocks [M | U | S | Ao | Bo] of 64 x 64 fp32
// (Ao, Bo: C rows used; S: a group's start state); for Falcon-3 then every token's window normaliser
// (computed once by a one-thread-per-token kernel and read by the map pass).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "falcon_internal.h"
#include "sm103_ptx.cuh"

namespace falcon {

__device__ int g_scan_tc_timeout_flag = 0;

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



// ---------------------------------------------------------------- the same steps on the tensor cores
// Compose and apply with one CTA of 128 threads per group and the carried state transposed in tensor
// memory: lane c holds state column c (compose: the 128 columns of [M_g | U_g]; apply: 64, the other
// lanes zero), TMEM column k its row k. That is the A operand of one product per step,
//   D = S^T [M_n ; Ao_n]^T   (M = 128, N = 64 + CP, K = 64, kind::tf32),
// whose first 64 columns are (M_n S)^T and the next CP (apply) (Ao_n S)^T, the chunk's outputs
// transposed. B = [M_n ; Ao_n] is K-major as stored (row-major maps), loaded by TMA with the 128-byte
// swizzle, 32 rows x 32 K per load. Each operand x is split into hi = x with its low 13 bits cleared
// (exact in tf32) and lo = x - hi, and D = A_hi B_hi + A_hi B_lo + A_lo B_hi, so the product has
// fp32 accuracy (the dropped A_lo B_lo term is below 2^-22 of it). U_n and Bo_n arrive by 16-byte
// asynchronous copies one step ahead and are added in registers, where each thread also splits its
// new state column for the next step and (apply) writes its column of the chunk's outputs. Every
// wait is bounded: on timeout the CTA raises the device flag, drains what it issued and frees its
// tensor memory.
constexpr int kTcThreads = 128;
constexpr uint32_t kTAH = 0, kTAL = 64, kTD = 128;  // TMEM columns: state hi, state lo, product
constexpr long long kTcTimeout = 4000000000LL;     // ~2 s

template <int CP>  // 0: compose; else apply, output rows rounded up to 32
struct TcLay {
    static constexpr int NB = 64 + CP;             // B rows: M_n, then CP rows of Ao_n
    static constexpr int BHI = 0, BLO = NB * 256;  // each: two K halves of NB rows x 128 bytes
    static constexpr int UF = (64 + CP) * 64;      // floats of one [U_n ; Bo_n] buffer
    static constexpr int UB = 2 * NB * 256;        // two such buffers
    static constexpr int BAR = UB + 2 * UF * 4;
    static constexpr int BYTES = BAR + 64;
    static constexpr int ALLOC = BYTES + 1024;
};

struct ScanTcParams {
    CUtensorMap tm_ws;  // the workspace as [rows][64] fp32
    ScanParams s;
};

__device__ __forceinline__ float hi19(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

__device__ bool tc_wait(uint32_t bar, uint32_t parity) {
    if (ptx::mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    int spins = 0;
    while (!ptx::mbar_try(bar, parity)) {
        if (++spins > 64) __nanosleep(32);
        if (clock64() - t0 > kTcTimeout) {
            atomicExch(&g_scan_tc_timeout_flag, 1);
            return false;
        }
    }
    return true;
}

// NQ x 16 consecutive TMEM columns of this thread's lane (one wait)
template <int NQ>
__device__ __forceinline__ void tc_ld(uint32_t taddr, float* v) {
    uint32_t r[NQ][16];
#pragma unroll
    for (int q = 0; q < NQ; ++q) ptx::tmem_ld16(taddr + 16 * q, r[q]);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        ptx::regs_ready(r[q]);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[16 * q + e] = __uint_as_float(r[q][e]);
    }
}

// this thread's state column into the A operand's hi and lo columns of its lane (no wait)
__device__ __forceinline__ void put_state(uint32_t tq, const float (&x)[kD]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h[16], l[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float v = x[16 * q + e], vh = hi19(v);
            h[e] = __float_as_uint(vh);
            l[e] = __float_as_uint(v - vh);
        }
        ptx::tmem_st16(tq + kTAH + 16 * q, h);
        ptx::tmem_st16(tq + kTAL + 16 * q, l);
    }
}

template <int CP>
__global__ void __launch_bounds__(kTcThreads, 2) falcon_scan_tc_kernel(const __grid_constant__ ScanTcParams P) {
    using L = TcLay<CP>;
    using namespace ptx;
    constexpr bool kCompose = CP == 0;
    const ScanParams& p = P.s;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw), base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t bar_full = base + L::BAR, bar_mma = bar_full + 8, bar_drain = bar_full + 16;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BAR + 32);
    const long long bh = blockIdx.x / p.NG, gi = blockIdx.x % p.NG;
    const long long first = gi * p.G, nsteps = min(p.G, p.N - first);
    const float* const chunks = p.ws + bh * p.N * kBlk;
    float* const groups = p.ws + (p.BH * p.N + bh * p.NG) * kBlk;
    const long long row0 = bh * p.N * (kBlk / kD);  // this sequence's first workspace row of 64 floats
    if (tid == 0) {
        mbar_init(bar_full, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_drain, 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot, tq = tmem + ((uint32_t)(32 * warp) << 16);
    const int c = tid;                     // state column = TMEM lane
    const bool live = kCompose || c < kD;  // apply: lanes 64..127 hold zeros

    auto issue_b = [&](long long j) {  // thread 0: [M_n ; Ao_n] of step j by TMA
        const int r = (int)(row0 + (first + j) * (kBlk / kD));
        mbar_expect_tx(bar_full, (uint32_t)(L::NB * 256));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t d = base + L::BHI + h * L::NB * 128;
            tma_load_2d(d, &P.tm_ws, 32 * h, r, bar_full);
            tma_load_2d(d + 32 * 128, &P.tm_ws, 32 * h, r + 32, bar_full);
#pragma unroll
            for (int q = 0; q < CP / 32; ++q) tma_load_2d(d + (64 + 32 * q) * 128, &P.tm_ws, 32 * h, r + 3 * kD + 32 * q, bar_full);
        }
    };
    auto issue_ub = [&](long long j) {  // every thread: U_n (and Bo_n) rows of step j into buffer j & 1
        if (j < nsteps) {
            const float* b = chunks + (first + j) * kBlk;
            float* d = reinterpret_cast<float*>(sm + L::UB) + (int)(j & 1) * L::UF;
#pragma unroll
            for (int u = 0; u < L::UF / 4 / kTcThreads; ++u) {
                const int e = tid + u * kTcThreads, row = e >> 4, col = 4 * (e & 15);
                cp_async16(d + row * kD + col, b + (row < kD ? kMat + row * kD : 4 * kMat + (row - kD) * kD) + col);
            }
        }
        cp_async_commit();
    };

    // the state entering the first step (compose: the group's first map itself)
    float s[kD];
    {
        const float* src = nullptr;
        if (kCompose) src = chunks + first * kBlk + (c < kD ? 0 : kMat) + (c & 63);
        else if (p.NG > 1) src = groups + gi * kBlk + 2 * kMat + c;
        else if (p.S0) src = p.S0 + bh * kMat + c;
#pragma unroll
        for (int r = 0; r < kD; ++r) s[r] = (live && src) ? src[r * kD] : 0.f;
    }
    put_state(tq, s);
    tmem_wait_st();
    const long long j0 = kCompose ? 1 : 0;
    long long pending = -1;  // the step whose B tile is in flight
    if (j0 < nsteps) {
        if (tid == 0) issue_b(j0);
        pending = j0;
    }
    issue_ub(j0);
    tc_fence_before();
    __syncthreads();
    bool ok = true;
    constexpr uint32_t id = idesc_tf32(128, (uint32_t)L::NB);
    for (long long j = j0; j < nsteps; ++j) {
        const uint32_t ph = (uint32_t)((j - j0) & 1);
        bool bad = false;
        if (tid == 0) bad = !tc_wait(bar_full, ph);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (named_bar_or(1, kTcThreads, bad)) {
            ok = false;
            break;
        }
        pending = -1;
        {  // B: hi (low 13 bits cleared) in place, lo = the rest
            float4* bh4 = reinterpret_cast<float4*>(sm + L::BHI);
            float4* bl4 = reinterpret_cast<float4*>(sm + L::BLO);
#pragma unroll 4
            for (int e = tid; e < L::NB * 16; e += kTcThreads) {
                const float4 v = bh4[e];
                const float4 h = make_float4(hi19(v.x), hi19(v.y), hi19(v.z), hi19(v.w));
                bh4[e] = h;
                bl4[e] = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (uint32_t)((ks >> 2) * (L::NB * 128) + 32 * (ks & 3));
                const uint64_t dh = desc_k(base + L::BHI + off), dl = desc_k(base + L::BLO + off);
                mma_tf32_ta(tmem + kTD, tmem + kTAH + 8 * ks, dh, id, ks > 0);
                mma_tf32_ta(tmem + kTD, tmem + kTAH + 8 * ks, dl, id, 1);
                mma_tf32_ta(tmem + kTD, tmem + kTAL + 8 * ks, dh, id, 1);
            }
            mma_commit(bar_mma);
            bad = !tc_wait(bar_mma, ph);
            if (!bad && j + 1 < nsteps) issue_b(j + 1);  // the B tile is free again
        }
        if (named_bar_or(1, kTcThreads, bad)) {
            ok = false;
            break;
        }
        if (j + 1 < nsteps) pending = j + 1;
        issue_ub(j + 1);
        tc_fence_after();
        const float* ub = reinterpret_cast<const float*>(sm + L::UB) + (int)(j & 1) * L::UF;
        {
            float x[kD];
            tc_ld<4>(tq + kTD, x);
#pragma unroll
            for (int r = 0; r < kD; ++r) {
                float v = x[r];
                if (kCompose) v += c >= kD ? ub[r * kD + c - kD] : 0.f;
                else v = live ? v + ub[r * kD + c] : 0.f;
                s[r] = v;
            }
        }
        if constexpr (!kCompose) {  // the chunk's outputs O = Ao S + Bo, this thread's column
            float o[CP];
            tc_ld<CP / 16>(tq + kTD + kD, o);
            const long long t0 = (first + j) * p.C;
            const int rows = (int)min((long long)p.C, p.T - t0);
            if (live) {
#pragma unroll
                for (int i = 0; i < CP; ++i) {
                    if (i >= rows) break;
                    const float v = o[i] + ub[(kD + i) * kD + c];
                    const long long at = (bh * p.T + t0 + i) * kD + c;
                    if (p.bf16) static_cast<__nv_bfloat16*>(p.out)[at] = __float2bfloat16_rn(v);
                    else static_cast<float*>(p.out)[at] = v;
                }
            }
        }
        if (j + 1 < nsteps) put_state(tq, s);
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
    }
    if (ok) {
        if (kCompose) {  // the group's map [M_g | U_g], column c
            float* g = groups + gi * kBlk + (c < kD ? 0 : kMat) + (c & 63);
#pragma unroll
            for (int r = 0; r < kD; ++r) g[r * kD] = s[r];
        } else if (gi == p.NG - 1 && p.S_final && live) {
#pragma unroll
            for (int r = 0; r < kD; ++r) p.S_final[bh * kMat + r * kD + c] = s[r];
        }
    }
    // drain: copies, a B tile still in flight (only after a timeout), the MMAs; then free TMEM
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (tid == 0 && pending >= 0) mbar_wait_bounded(bar_full, (uint32_t)((pending - j0) & 1), kTcTimeout);
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        mma_commit(bar_drain);
        mbar_wait_bounded(bar_drain, 0, kTcTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

// A workspace as [rows][64] fp32 for TMA: 32 x 32 boxes with the 128-byte swizzle, one 32-element K
// half of 32 rows of a K-major tf32 operand per load (cuTensorMapEncodeTiled through the runtime's
// driver entry point, looked up once).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
bool encode_rows_f32_sw128(CUtensorMap* tm, const void* ptr, long long rows) {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(q);
    }
    if (!fn) return false;
    cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    cuuint64_t strides[1] = {64 * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
    if (BH * NG >= sms) {  // enough groups for a CTA per SM: the tensor-core steps, one CTA per group
        // the fewest groups that still fill the two CTA slots of every SM (never more groups than the
        // workspace's blocks for groups of 16)
        const long long want = max(1LL, min(NG, 2LL * sms / BH));
        p.G = (N + want - 1) / want;
        p.NG = (N + p.G - 1) / p.G;
        const int C = a.chunk;
        const unsigned grid = (unsigned)(BH * p.NG);
        // the workspace as rows of 64 floats for the tensor maps (any workspace that fits in memory has
        // fewer than 2^31)
        const long long rows = BH * (N + NG) * (kBlk / kD);
        ScanTcParams tp{};
        if (rows >= (1LL << 31) || !encode_rows_f32_sw128(&tp.tm_ws, ws, rows)) return 4;
        constexpr int a0 = TcLay<0>::ALLOC, a32 = TcLay<32>::ALLOC, a64 = TcLay<64>::ALLOC;
        static_assert(a64 <= 227 * 1024 && 2 * (a32 + 1024) <= 228 * 1024, "tensor-core scan shared memory");
        if (cudaFuncSetAttribute(falcon_scan_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, a0) != cudaSuccess ||
            cudaFuncSetAttribute(falcon_scan_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, a32) != cudaSuccess ||
            cudaFuncSetAttribute(falcon_scan_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, a64) != cudaSuccess)
            return 4;
        if (p.NG > 1) {
            p.mode = 0;
            tp.s = p;
            falcon_scan_tc_kernel<0><<<grid, kTcThreads, a0, st>>>(tp);
            p.mode = 1;  // the short pass over the groups: 16-column slices
            falcon_scan_kernel<<<(unsigned)(BH * 4), kThreads, smem_bytes(0), st>>>(p);
        }
        p.mode = 2;
        tp.s = p;
        if (C <= 32) falcon_scan_tc_kernel<32><<<grid, kTcThreads, a32, st>>>(tp);
        else falcon_scan_tc_kernel<64><<<grid, kTcThreads, a64, st>>>(tp);
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

int scan_tc_consume_timeout_flag(int* flag) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_scan_tc_timeout_flag, sizeof(int)) != cudaSuccess) return 1;
    if (v && cudaMemcpyToSymbol(g_scan_tc_timeout_flag, &zero, sizeof(int)) != cudaSuccess) return 1;
    *flag = v;
    return 0;
}

}  // namespace falcon
