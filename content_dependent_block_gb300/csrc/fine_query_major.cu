// Stage 2, fine attention, query-major CUDA-core kernel (page
// "sparse-attention-triton-bench", Stage 2 and "The Triton kernel": each
// query attends only the tokens of its listed blocks, with a running max m,
// running sum l and unnormalised accumulator acc updated block by block;
// page "yayme/CUDA-kernel" README: the same loop over a precomputed
// active-tile list with a token-level window/stride predicate).
//
// One warp per query row.  Per 32-key chunk of a listed block, lane t scores
// key j0+t against the query (the query row sits in shared memory and is
// read as a broadcast), the warp folds the chunk into (m, l) and each lane
// updates its D/32 output channels with the chunk's weights, reading every V
// row as one coalesced warp load.  Scores never leave registers.  Works for
// bf16 and fp32 inputs, any key-block size, any list layout.
#include <cmath>

#include "bsa_device.cuh"
#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kWarps = 4;

template <typename T>
struct Elem;
template <>
struct Elem<uint16_t> {   // bf16 bits
    static __device__ __forceinline__ float load(const uint16_t *p) {
        return __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short *>(p))) << 16);
    }
    static __device__ __forceinline__ void store(uint16_t *p, float x) { *p = f32_to_bf16_bits(x); }
};
template <>
struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};

// Dot product of one key row with the query held in shared memory.
template <int D>
__device__ __forceinline__ float dot_row(const uint16_t *krow, const float *qs) {
    const uint4 *src = reinterpret_cast<const uint4 *>(krow);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const uint4 x = __ldg(src + c);
        s = fmaf(bf16_low_half(x.x), qs[8 * c + 0], s);
        s = fmaf(bf16_high_half(x.x), qs[8 * c + 1], s);
        s = fmaf(bf16_low_half(x.y), qs[8 * c + 2], s);
        s = fmaf(bf16_high_half(x.y), qs[8 * c + 3], s);
        s = fmaf(bf16_low_half(x.z), qs[8 * c + 4], s);
        s = fmaf(bf16_high_half(x.z), qs[8 * c + 5], s);
        s = fmaf(bf16_low_half(x.w), qs[8 * c + 6], s);
        s = fmaf(bf16_high_half(x.w), qs[8 * c + 7], s);
    }
    return s;
}
template <int D>
__device__ __forceinline__ float dot_row(const float *krow, const float *qs) {
    const float4 *src = reinterpret_cast<const float4 *>(krow);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < D / 4; ++c) {
        const float4 x = __ldg(src + c);
        s = fmaf(x.x, qs[4 * c + 0], s);
        s = fmaf(x.y, qs[4 * c + 1], s);
        s = fmaf(x.z, qs[4 * c + 2], s);
        s = fmaf(x.w, qs[4 * c + 3], s);
    }
    return s;
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) fine_query_major_kernel(FineArgs a) {
    constexpr int E = D / 32;
    __shared__ float qsm[kWarps][D];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kWarps + warp;
    if (row >= a.bh * a.n) return;
    const int64_t h = row / a.n;
    const int64_t i = row - h * a.n;

    const T *q = static_cast<const T *>(a.q) + row * D;
    const T *kh = static_cast<const T *>(a.k) + h * a.n * D;
    const T *vh = static_cast<const T *>(a.v) + h * a.n * D;
    float *qs = qsm[warp];
#pragma unroll
    for (int e = 0; e < E; ++e) qs[lane * E + e] = Elem<T>::load(q + lane * E + e);
    __syncwarp();

    const int32_t *lp = nullptr;
    int64_t nlist = a.nb;
    if (a.list != nullptr) {
        const int64_t lrow = (a.per_head ? h * a.list_rows : 0) + i / a.q_group;
        lp = a.list + lrow * a.max_blocks;
        nlist = a.max_blocks;
    }

    float m = -INFINITY, l = 0.f;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;

    for (int64_t t = 0; t < nlist; ++t) {
        const int64_t b = lp ? int64_t(__ldg(lp + t)) : t;
        if (b < 0) break;                         // padding only at the tail
        if (b >= a.nb) {
            if (lane == 0) report_status(a.status, kStatusBadIndex);
            continue;
        }
        const int64_t j0 = b * a.kb;
        const int64_t j1 = i64min(a.n, j0 + a.kb);
        for (int64_t jc = j0; jc < j1; jc += 32) {
            const int64_t j = jc + lane;
            const bool ok = j < j1 && mask_admits(a.mask_kind, a.window, a.stride, a.sliding, i, j);
            float s = -INFINITY;
            if (ok) s = dot_row<D>(kh + j * D, qs) * a.scale_log2;
            const float mnew = fmaxf(m, warp_max(s));
            if (mnew == -INFINITY) continue;      // nothing admitted yet
            const float alpha = exp2f(m - mnew);  // m = -inf -> 0
            const float p = ok ? exp2f(s - mnew) : 0.f;
            l = l * alpha + warp_sum(p);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] *= alpha;
            const int nj = int(i64min(32, j1 - jc));
            const T *vr = vh + jc * D + lane * E;
#pragma unroll 4
            for (int u = 0; u < nj; ++u) {
                const float pu = __shfl_sync(0xffffffffu, p, u);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(pu, Elem<T>::load(vr + u * D + e), acc[e]);
            }
            m = mnew;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *o = static_cast<T *>(a.out) + row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) Elem<T>::store(o + e, acc[e] * inv);
}

template <typename T>
cudaError_t launch_t(const FineArgs &a, cudaStream_t st) {
    const int64_t rows = a.bh * a.n;
    const dim3 grid(unsigned((rows + kWarps - 1) / kWarps));
    if (a.d == 64)
        fine_query_major_kernel<T, 64><<<grid, kWarps * 32, 0, st>>>(a);
    else
        fine_query_major_kernel<T, 128><<<grid, kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fine_query_major(const FineArgs &a, int32_t dtype, cudaStream_t st) {
    if (dtype == 0) return launch_t<uint16_t>(a, st);
    return launch_t<float>(a, st);
}

}  // namespace bsa
