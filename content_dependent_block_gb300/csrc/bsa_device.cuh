// Device helpers shared by the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bsa {

// Status codes written by kernels (values match bsa_status in bsa.h).
constexpr int32_t kStatusInvalidArg = 1;
constexpr int32_t kStatusBadIndex = 3;
constexpr int32_t kStatusTimeout = 6;

__device__ __forceinline__ int64_t i64min(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t i64max(int64_t a, int64_t b) { return a > b ? a : b; }

// First error wins; later ones are dropped.
__device__ __forceinline__ void report_status(int32_t *status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

// bf16 bit patterns -> fp32 (exact).
__device__ __forceinline__ float bf16_low_half(uint32_t packed) {
    return __uint_as_float(packed << 16);
}
__device__ __forceinline__ float bf16_high_half(uint32_t packed) {
    return __uint_as_float(packed & 0xFFFF0000u);
}

// fp32 -> bf16 bits, round to nearest even (hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    uint16_t r;
    asm("{ .reg .b16 t; cvt.rn.bf16.f32 t, %1; mov.b16 %0, t; }" : "=h"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Token-level predicate of the static patterns (kinds as in bsa_mask_kind).
__device__ __forceinline__ bool mask_admits(int32_t kind, int32_t window,
                                            int32_t stride, int32_t sliding,
                                            int64_t i, int64_t j) {
    if (kind == 1) {
        int64_t dist = i > j ? i - j : j - i;
        return (window >= 0 && dist <= window) || (stride > 0 && (j % stride) == 0);
    }
    if (kind == 2) return j > i - sliding && j <= i;
    if (kind == 3) return j <= i;
    return true;
}

// Selection options applied to one query's candidates, held as block ids in
// descending score order (INT_MAX = empty): keep the first `kr` (the
// per-head budget of page "sparse-attention-triton-bench", What's next) and,
// with `local`, make sure the query's own block `own` is among them by
// putting it in place of the last one kept (the kept set is then own plus
// the kr - 1 best of the other eligible blocks).
template <int KMAX>
__device__ __forceinline__ void apply_budget(int (&ids)[KMAX], int kr, int own, bool local) {
    bool has_own = false;
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
        if (t >= kr) ids[t] = 0x7fffffff;
        has_own |= ids[t] == own;
    }
    if (local && !has_own) {
#pragma unroll
        for (int t = 0; t < KMAX; ++t)
            if (t == kr - 1) ids[t] = own;
    }
}

}  // namespace bsa
