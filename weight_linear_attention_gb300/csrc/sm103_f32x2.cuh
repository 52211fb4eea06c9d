// Packed fp32 arithmetic of sm_100-class GPUs: two independent single-precision FMAs in one
// instruction (fma.rn.f32x2), each lane rounded exactly as fmaf.
#pragma once

#include <cuda_runtime.h>

namespace falcon {
namespace ptx {

// ---- packed fp32 pair: (x0, x1) += (g0, g1) * v, one fma.rn.f32x2 (each lane rounded exactly as fmaf)
__device__ __forceinline__ void fma2(float& x0, float& x1, float g0, float g1, float v) {
    asm("{\n .reg .b64 a, b, c;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n mov.b64 c, {%4, %4};\n"
        " fma.rn.f32x2 a, b, c, a;\n mov.b64 {%0, %1}, a;\n}\n"
        : "+f"(x0), "+f"(x1)
        : "f"(g0), "f"(g1), "f"(v));
}

}  // namespace ptx
}  // namespace falcon
