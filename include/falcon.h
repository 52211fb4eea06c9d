/*
 * falcon.h — C ABI of the GB300 (sm_103a) Falcon fast-weight forward pass.
 *
 * The operation ("Fast Weight Attention for Continual Learning", arXiv
 * 2608.27763; paperlayer.ai summary = [PL], agihunt.info explainer = [AH],
 * sungsoo.github.io post = [SG]): for every (batch b, head h) sequence, steps
 * tau = pos+1 .. pos+T update a fast-weight matrix S (dk x dv, fp32) with the
 * prefix-aligned pair x_tau = k_{tau-1} (x_1 = 0), y_tau = v_tau
 * ([PL] abstract, §3, Appendix p.34) and read o_tau = S_tau^T q_tau after the
 * write ([AH] Method). With eta = beta / (||x||^2 + lambda + eps) (0 when the
 * denominator is 0), alpha = min(eta*lambda, 1 - eps_gamma), gamma = 1 - alpha,
 * and eta = alpha = 0 at tau = 1 ([PL] §3.1, §C.3, §4.6; [SG]):
 *   FALCON_1   S = gamma S + eta x (y - S^T x)^T             ([AH] Method)
 *   FALCON_1A  S = gamma S + eta x y^T                        ([AH] Method)
 *   FALCON_2   as FALCON_1 with a per-column gain beta[..., c] ([PL] §1, Figure 5)
 *   FALCON_2A  as FALCON_1A with a per-column gain beta[..., c] ([PL] §4.3, "B. Falcon-2A")
 *   FALCON_3   window of the last `window` pairs (pair 1 excluded), residuals at
 *              the pre-update state, step eta/B_tau, eta normalised by the top
 *              eigenvalue of the window-averaged key covariance ([PL] §4.4, §C.6)
 *   FALCON_3A  the same window written with the targets themselves, eta normalised by
 *              the window's mean key energy (1/B) sum ||x_j||^2 ([PL] §4.5, §4.6, "C. Falcon-3A")
 * The kernels evaluate it in the chunk-parallel form ([PL] Figure 2, §E.2, §F.2,
 * §H.3): per chunk one unit-lower-triangular solve with the value and the
 * projected-history right-hand sides merged, log-prefix decay reset to 0 at
 * every chunk start ([PL] §D.1, §G.1), and a carried state between chunks.
 * A call with T = 1 (Falcon-1, 1A, 2, 2A; dk = dv = 64) runs a single-token kernel instead: the recurrent
 * form of the same update, one (batch, head) state per CTA, so a decoding step costs one read and
 * one write of the state ([PL] §3; [AH] Method).
 * Falcon-1 and 1A at bf16, dk = dv = 64, chunk 64 run a fused tensor-core kernel: one persistent
 * CTA per (batch, head) sequence walks its chunks with the state on chip, the state-independent
 * work of two chunks in flight while the state pass of an earlier one runs ([PL] §E.2: parallel
 * per-chunk work, a short state recurrence, per-chunk reads); it needs no workspace.
 * Falcon-2 and 2A at bf16, dk = dv = 64, chunk 64 run a per-column tensor-core kernel: one
 * persistent CTA per sequence; the chunk's Gram and scores, shared by every value column, are formed
 * one chunk ahead, and each column's merged residual solve runs between two products over all
 * columns ([PL] §F, §F.2); it needs no workspace. It loads beta by TMA, so it runs when beta is
 * 16-byte aligned; with a beta aligned to 4 bytes only, the CUDA-core chunk kernel runs instead.
 * Falcon-1, 1A, 3 and 3A with dk = dv = 64 over few (batch, head) sequences and no fused path have
 * a scan path that uses a caller-provided workspace: every chunk's affine maps of the state and of
 * the outputs, then an associative scan over the chunk maps in groups of chunks ([PL] §H.1, §H.2),
 * whose last step also forms every chunk's outputs. For Falcon-3 and 3A at window 4, chunk 32, bf16
 * the maps are formed on the tensor cores ([PL] §H.3's windowed block system); with enough
 * sequences x groups to fill the GPU, the scan's compose and apply steps run on the tensor cores
 * too (tf32 products of split operands, fp32-accurate).
 *
 * Memory: every pointer argument is DEVICE memory owned by the caller; the
 * library keeps no pointer after a call returns and allocates no device memory.
 * Tensors are dense, row-major, contiguous, outermost dimension first.
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream). Argument checking is synchronous: on any nonzero return nothing was
 * launched and no output was touched.
 */
#ifndef FALCON_H
#define FALCON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FALCON_1 = 1,   /* scalar NLMS regression write                              */
    FALCON_1A = 2,  /* scalar inner-product write                                */
    FALCON_2 = 3,   /* per-column NLMS regression write                          */
    FALCON_2A = 4,  /* per-column inner-product write                            */
    FALCON_3 = 5,   /* sliding-window mini-batch regression write                */
    FALCON_3A = 6   /* sliding-window inner-product write                        */
} falcon_variant_t;

typedef enum { FALCON_F32 = 0, FALCON_BF16 = 1 } falcon_dtype_t;

/* Status codes returned by every entry point that returns int. */
enum {
    FALCON_OK = 0,
    FALCON_ERR_INVALID_ARG = 1,   /* null required pointer, bad variant/window/chunk/dims, tail vs pos, overlap */
    FALCON_ERR_UNSUPPORTED = 2,   /* a head size, dtype, window or chunk with no kernel in the library */
    FALCON_ERR_MISALIGNED = 3,    /* a pointer not aligned as documented below */
    FALCON_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    FALCON_ERR_DEVICE_TIMEOUT = 5 /* a kernel gave up a bounded wait (see falcon_device_status) */
};

/* Problem description. 64 bytes, no implicit padding. */
typedef struct {
    int64_t batch;    /* B >= 0                                                       */
    int64_t heads;    /* H >= 0                                                       */
    int64_t seqlen;   /* T >= 0 tokens in this call                                   */
    int64_t dk;       /* key/query width: 16, 32, 64 or 128                           */
    int64_t dv;       /* value width: 16, 32, 64 or 128                               */
    int32_t window;   /* Falcon-3 / 3A window size 1..8; must be 1 for the other variants */
    int32_t dtype;    /* falcon_dtype_t of q, k, v, out, tail, tail_out                */
    int64_t pos;      /* tokens already consumed by earlier calls; 0 = fresh start    */
    float eps;        /* >= 0, added to the step-size denominator                     */
    float eps_gamma;  /* in (0, 1): alpha is clamped to 1 - eps_gamma                 */
} falcon_dims_t;

/*
 * falcon_fwd — one forward pass over T tokens of B*H sequences.
 *   q, k      [B,H,T,dk] dtype        queries and keys (phi = identity; callers apply
 *                                     QK-RMSNorm upstream, [PL] §5, [AH] Method)
 *   v         [B,H,T,dv] dtype        values (targets y)
 *   beta      fp32 [B,H,T], or [B,H,T,dv] for FALCON_2 and 2A; gains, caller keeps them in (0,2)
 *   lambda    fp32 [B,H,T], >= 0      ridge coefficients
 *   S0        fp32 [B,H,dk,dv] or NULL (zero initial state)
 *   tail      NULL iff pos == 0; else falcon_tail_bytes(dims) bytes in dtype laid out
 *             per (b,h) as keys[window][dk] = k_{pos-window+1..pos} followed by
 *             vals[window-1][dv] = v_{pos-window+2..pos} (entries with global index
 *             <= 0 are zero); this is what tail_out of the previous call holds.
 *             For window 1 it is the pending key k_pos alone ([PL] §C.7, §4.4).
 *   out       [B,H,T,dv] dtype        o_t = S_t^T q_t; must not overlap any input
 *   S_final   fp32 [B,H,dk,dv] or NULL; may be the same pointer as S0, must not overlap any
 *             other argument
 *   tail_out  NULL or falcon_tail_bytes(dims) bytes: the tail for position pos+T;
 *             must not overlap any other argument
 *   dims      problem description (host pointer)
 *   chunk     chunk length C: 16, 32 or 64; FALCON_3 and 3A need chunk*window <= 128.
 *             The result does not depend on C beyond fp32 rounding.
 *   workspace NULL, or scratch device memory of at least
 *             falcon_workspace_bytes(variant, dims, chunk) bytes that overlaps no other
 *             argument. When that size is nonzero and the workspace is given, the scan
 *             path runs; with NULL the CUDA-core chunk kernel runs (same results up to fp32
 *             rounding). Contents on entry are ignored and on return unspecified; calls
 *             that may run at the same time must not share a workspace.
 *   workspace_bytes  size of `workspace` (ignored when workspace is NULL); a given
 *             workspace smaller than falcon_workspace_bytes() is FALCON_ERR_INVALID_ARG
 *   stream    cudaStream_t to launch on
 * Alignment: q, k, v, out, tail, tail_out, S0, S_final 16 bytes; workspace 256 bytes;
 * beta, lambda 4 bytes.
 * Returns FALCON_OK or an error code; see falcon_status_string.
 */
int falcon_fwd(int variant, const void* q, const void* k, const void* v, const float* beta,
               const float* lambda, const float* S0, const void* tail, void* out, float* S_final,
               void* tail_out, const falcon_dims_t* dims, int chunk, void* workspace,
               size_t workspace_bytes, void* stream);

/* Workspace bytes that enable the scan path of falcon_fwd for these arguments
 * (B*H*(N + ceil(N/16)) * 80 KiB with N = ceil(T/chunk), plus 4*B*H*T bytes for Falcon-3;
 * Falcon-1, 1A, 3, 3A with dk = dv = 64, B*H < 76, N >= 4, no fused path); 0 when no path uses a
 * workspace (the fused and single-token kernels need none) or the arguments are invalid. Host only. */
size_t falcon_workspace_bytes(int variant, const falcon_dims_t* dims, int chunk);

/*
 * falcon_fwd_static — falcon_fwd with the library's own scratch instead of a caller workspace.
 * The paper has no counterpart: this entry point is for callers that cannot allocate device memory,
 * for example code running inside another runtime's memory pool (an extra cudaMalloc bypasses the
 * pool's accounting and can fail under memory pressure) or a latency-critical loop that must not pay
 * cudaMalloc's implicit device synchronisation. Same arguments and results as falcon_fwd with a
 * workspace. The scratch is a fixed FALCON_STATIC_WORKSPACE_BYTES device array inside the library
 * (every device that loads the library holds it until the process exits), never allocated or freed
 * per call; every call looks up its device address (cudaGetSymbolAddress, once per device, then
 * cached), whether or not that call uses it, so the first call on a device does that set-up.
 * Nothing in the array needs zeroing: every byte a kernel reads was written earlier in the same call.
 * Only the scan path uses scratch; a shape whose scan path needs more than
 * FALCON_STATIC_WORKSPACE_BYTES runs the CUDA-core chunk kernel instead, and every other shape (the
 * fused and single-token kernels) needs none. Calls that may overlap in time on one device (any
 * streams) race on the scratch and must be serialized by the caller.
 */
#define FALCON_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)
int falcon_fwd_static(int variant, const void* q, const void* k, const void* v, const float* beta,
                      const float* lambda, const float* S0, const void* tail, void* out, float* S_final,
                      void* tail_out, const falcon_dims_t* dims, int chunk, void* stream);

/* Bytes of one tail buffer for `dims` (all B*H sequences); 0 for a NULL or invalid dims. */
size_t falcon_tail_bytes(const falcon_dims_t* dims);

/* Static English text for a status code; never NULL. */
const char* falcon_status_string(int status);

/*
 * Synchronizes `stream`, then reports whether any kernel of this library on the
 * current device gave up a bounded device-side wait since the last call
 * (FALCON_ERR_DEVICE_TIMEOUT), and clears that flag. Returns FALCON_ERR_CUDA if
 * the synchronize fails, else FALCON_OK.
 */
int falcon_device_status(void* stream);

/* Which kernels falcon_fwd launches for these arguments when it is given
 * falcon_workspace_bytes() of workspace (0 = none/invalid, 1 = CUDA-core chunk kernel,
 * 4 = single-token kernel for T = 1, 5 = scan path: chunk maps (tensor-core kernel for Falcon-3 / 3A
 * at window 4, chunk 32, bf16; else the CUDA-core kernel), then the scan over them, 6 = fused
 * tensor-core kernel, 7 = per-column tensor-core kernel (beta 16-byte
 * aligned; else 1); 2 and 3 are retired). Without a workspace, 5 becomes 1. Host only, no launch. */
int falcon_kernel_for(int variant, const falcon_dims_t* dims, int chunk);

/*
 * falcon_bwd — gradients of one falcon_fwd call (Falcon-1 and 1A; dk = dv = 64; chunk 64).
 * Given the adjoints dout of `out` and dS_final of `S_final`, returns the gradients of
 * L = sum(out * dout) + sum(S_final * dS_final) with respect to every input of the call
 * ([PL] §D.2, §E.3, §G.3: the chunk-parallel backward through the triangular solve, the Gram
 * matrix, the chunk-local decay prefixes, the clamp and the step-size normalisation).
 * Conventions of the gradient where the forward pass is not smooth ([PL] §D.2, §E.3, §G.3):
 * where the clamp binds (eta*lambda >= 1 - eps_gamma) alpha is a constant and passes no gradient;
 * where eta is 0 by definition (a zero denominator; the first step of a fresh sequence) beta,
 * lambda and x receive nothing through it.
 *   q, k, v, beta, lambda, S0, tail, dims, chunk   exactly as passed to falcon_fwd (window 1,
 *             so `tail` is the pending key k_pos alone; beta [B,H,T])
 *   dout      [B,H,T,dv] dtype        adjoint of out
 *   dS_final  fp32 [B,H,dk,dv] or NULL (zero adjoint of S_final)
 *   dq, dk    fp32 [B,H,T,dk]         dk[..., T-1, :] is 0: the last key reaches only tail_out,
 *                                     whose gradient (the next call's dtail) the caller adds there
 *   dv        fp32 [B,H,T,dv]
 *   dbeta, dlambda  fp32 [B,H,T]      0 at the first step of a fresh sequence
 *   dS0       fp32 [B,H,dk,dv] or NULL: gradient of S0 (of the zero state when S0 is NULL)
 *   dtail     fp32 [B,H,dk] or NULL: gradient of the tail key; must be NULL when pos == 0
 *   workspace at least falcon_bwd_workspace_bytes() bytes of device scratch (required when it is
 *             nonzero); contents ignored on entry, unspecified on return
 * Every output and the workspace must overlap no other argument. Alignment: q, k, v, tail, dout,
 * S0, dS_final, dq, dk, dv, dS0, dtail 16 bytes; beta, lambda, dbeta, dlambda 4; workspace 256.
 * Shapes other than the above return FALCON_ERR_UNSUPPORTED. Asynchronous on `stream`: with 4 or
 * more sequences (B*H) the call runs them in 2 (16 or more: 4) groups on streams of the library's
 * own (made once per device, non-blocking), which wait for `stream` first and which `stream` waits
 * for at the end, so work ordered on `stream` stays ordered and a CUDA graph capture of `stream`
 * takes them in. Calls from several host threads are serialised while they enqueue.
 */
int falcon_bwd(int variant, const void* q, const void* k, const void* v, const float* beta,
               const float* lambda, const float* S0, const void* tail, const void* dout,
               const float* dS_final, float* dq, float* dk, float* dv, float* dbeta, float* dlambda,
               float* dS0, float* dtail, const falcon_dims_t* dims, int chunk, void* workspace,
               size_t workspace_bytes, void* stream);

/* Workspace bytes falcon_bwd needs: B*H*ceil(T/64) * 99 KiB (per chunk six 16 KiB slots: the
 * transition's offset and the state-free adjoint term in fp32; the transition, the inverse of the
 * chunk's triangular system, the chunk-start state and the chunk-end adjoint, each as two bf16 parts;
 * and 3 KiB of per-token scalars); 0 for invalid or unsupported arguments. */
size_t falcon_bwd_workspace_bytes(int variant, const falcon_dims_t* dims, int chunk);

/* ABI version of this header: 4. */
int falcon_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FALCON_H */
