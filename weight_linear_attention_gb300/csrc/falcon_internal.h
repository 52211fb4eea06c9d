// Internal interface between the C-ABI front end (falcon_api.cu) and the kernels.
// Not installed; the public interface is include/falcon.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace falcon {

enum Variant { kF1 = 1, kF1A = 2, kF2 = 3, kF2A = 4, kF3 = 5, kF3A = 6 };
// per-column gains (2, 2A); a window of W pairs (3, 3A); the target written as is, no solve (1A, 2A, 3A)
__host__ __device__ constexpr bool per_column(int v) { return v == kF2 || v == kF2A; }
__host__ __device__ constexpr bool windowed(int v) { return v == kF3 || v == kF3A; }
__host__ __device__ constexpr bool inner_product(int v) { return v == kF1A || v == kF2A || v == kF3A; }

// Arguments after validation by falcon_fwd: sizes are in range, pointers are
// non-null where required and aligned, tail is present iff pos > 0.
struct Launch {
    int variant;
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    const float* lam;
    const float* S0;      // may be null
    const void* tail;     // null iff pos == 0
    void* out;
    float* S_final;       // may be null
    void* tail_out;       // may be null
    int64_t B, H, T, dk, dv, pos;
    int W;
    int bf16;             // 1: q/k/v/out/tail are bf16, 0: fp32
    float eps, eps_gamma;
    int chunk;
    void* ws;             // caller's workspace, or null
    size_t ws_bytes;
};

// CUDA-core chunk kernel: every variant, both dtypes, all supported sizes.
int launch_generic(const Launch& a, cudaStream_t stream);
// The same kernel one chunk per CTA (mode 1): every chunk's affine state and output maps into `ws`
// (the scan path's layout); mode 0 is launch_generic.
int launch_generic_mode(const Launch& a, int mode, float* ws, long long N, const float* mu, cudaStream_t stream,
                        bool skip_marked = false);
// Falcon-3: every token's window normaliser into mu[B*H][T] (read by modes 1 and 2 instead of recomputed).
int launch_window_mu(const Launch& a, float* mu, cudaStream_t stream);
size_t generic_smem_bytes(const Launch& a, int dvs, bool staged = true);  // staged: mode 0's copy-ahead area

// Fused path (Falcon-1 and 1A, bf16, dk = dv = 64, chunk 64, T != 1): one persistent CTA per
// sequence, TMA + tcgen05, state on chip; no workspace.
bool fused_supported(const Launch& a);
int launch_fused(const Launch& a, cudaStream_t stream);
// Reads and clears the device-side timeout flag of the fused kernel (synchronous).
int fused_consume_timeout_flag(int* flag);
// TMA maps of a [BH][T][64] tensor with 64 x 64 boxes: bf16 with the 128-byte swizzle, or fp32 with
// none. False when the driver entry point is missing or refuses the map.
bool encode_bhtd(CUtensorMap* tm, const void* ptr, long long T, long long BH);
bool encode_bhtd_f32(CUtensorMap* tm, const void* ptr, long long T, long long BH);

// Per-column path (Falcon-2 and 2A, bf16, dk = dv = 64, chunk 64, T != 1): one persistent CTA per
// sequence, the shared Gram and scores on tcgen05 one chunk ahead, each value column's merged
// residual solve on CUDA cores, the state on chip; no workspace.
bool colw_supported(const Launch& a);
int launch_colw(const Launch& a, cudaStream_t stream);
int colw_consume_timeout_flag(int* flag);

// Tensor-core chunk maps for the scan path (Falcon-3 and 3A, bf16, dk = dv = 64, W = 4, chunk 32): every
// chunk's [M | U | . | Ao | Bo] into the scan workspace, each finished chunk marked in its block's
// state slot; chunks whose decay is too strong for the factored form stay unmarked for the CUDA-core
// map kernel (launch_generic_mode with skip_marked).
bool f3map_supported(const Launch& a);
int launch_f3map(const Launch& a, float* ws, long long N, const float* mu, cudaStream_t stream);
int f3map_consume_timeout_flag(int* flag);

// Single-token step (T = 1; Falcon-1, 1A, 2 and 2A; dk = dv = 64): one CTA per (batch, head) state.
bool decode_supported(const Launch& a);
int launch_decode(const Launch& a, cudaStream_t stream);

// Scan path (Falcon-1, 1A, 3, 3A with dk = dv = 64, few sequences, no fused path): chunk maps,
// an associative scan over them, then the chunks' outputs, through a caller workspace.
bool scan_supported(const Launch& a);
size_t scan_workspace_bytes(const Launch& a);
int launch_scan(const Launch& a, cudaStream_t stream);
int scan_tc_consume_timeout_flag(int* flag);
bool encode_rows_f32_sw128(CUtensorMap* tm, const void* ptr, long long rows);  // [rows][64] fp32, 32 x 32 boxes, 128-byte swizzle
int bwd_consume_timeout_flag(int* flag);

// Backward pass (Falcon-1 and 1A, dk = dv = 64, chunk 64): prep, chain and gradient kernels working
// through a caller workspace of bwd_workspace_bytes(a) bytes at a.ws. `a` carries the forward inputs.
struct BwdArgs {
    const void* dout;        // [B,H,T,dv] in the input dtype
    const float* dS_final;   // [B,H,dk,dv] or null (zero)
    float* dq;               // [B,H,T,dk]
    float* dk;               // [B,H,T,dk]
    float* dv;               // [B,H,T,dv]
    float* dbeta;            // [B,H,T]
    float* dlam;             // [B,H,T]
    float* dS0;              // [B,H,dk,dv] or null
    float* dtail;            // [B,H,dk] or null (pos > 0 only)
};
bool bwd_supported(const Launch& a);
size_t bwd_workspace_bytes(const Launch& a);
int launch_bwd(const Launch& a, const BwdArgs& g, cudaStream_t stream);

}  // namespace falcon
