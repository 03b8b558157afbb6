// Stage 1, block mean-pool (page "sparse-attention-triton-bench", Two-stage
// block indexer, Stage 1: each B-token key block is represented by the mean
// of its keys).
//
// One warp per (head, block).  Lane l owns the D/32 contiguous channels
// [l*D/32, (l+1)*D/32), so every key row is one fully coalesced 128/256-byte
// warp load; rows are fetched eight at a time to keep loads in flight.
// Accumulation is fp32; the mean divides by the number of valid tokens (a
// ragged last block averages only its own tokens).  Optionally the mean is
// also emitted as a bf16 hi/lo pair (hi = bf16(mean), lo = bf16(mean - hi))
// for the tensor-core scoring stage, whose rows are padded to nb_pad.
//
// HBM-bound: reads K once (bh*n*d*2 bytes), writes bh*nb*d*(4 [+4]) bytes.
#include "bsa_device.cuh"
#include "bsa_internal.h"

namespace bsa {
namespace {

template <int D>
struct RowVec;
template <>
struct RowVec<64> {          // 2 bf16 per lane
    using T = uint32_t;
    static __device__ __forceinline__ void add(float *acc, T x) {
        acc[0] += bf16_low_half(x);
        acc[1] += bf16_high_half(x);
    }
};
template <>
struct RowVec<128> {         // 4 bf16 per lane
    using T = uint2;
    static __device__ __forceinline__ void add(float *acc, T x) {
        acc[0] += bf16_low_half(x.x);
        acc[1] += bf16_high_half(x.x);
        acc[2] += bf16_low_half(x.y);
        acc[3] += bf16_high_half(x.y);
    }
};

template <int D>
__global__ void __launch_bounds__(256) pool_kernel(
    const uint16_t *__restrict__ k, int64_t bh, int64_t n, int32_t kb,
    int64_t nb, float *__restrict__ kbar, uint16_t *__restrict__ hi,
    uint16_t *__restrict__ lo, int64_t nb_pad) {
    constexpr int E = D / 32;
    using V = typename RowVec<D>::T;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= bh * nb) return;
    const int64_t h = warp / nb;
    const int64_t b = warp - h * nb;
    const int64_t j0 = b * kb;
    const int64_t j1 = i64min(n, j0 + kb);
    const V *rows = reinterpret_cast<const V *>(k + (h * n + j0) * D) + lane;
    constexpr int64_t kStride = D / E;   // V elements per key row = 32

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;

    int64_t j = j0;
    for (; j + 8 <= j1; j += 8) {
        V x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = __ldg(rows + (j - j0 + u) * kStride);
#pragma unroll
        for (int u = 0; u < 8; ++u) RowVec<D>::add(acc, x[u]);
    }
    for (; j < j1; ++j) RowVec<D>::add(acc, __ldg(rows + (j - j0) * kStride));

    const float count = float(j1 - j0);
    float *dst = kbar + (h * nb + b) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        acc[e] = __fdiv_rn(acc[e], count);
        dst[e] = acc[e];
    }
    if (hi != nullptr) {
        uint16_t *hd = hi + (h * nb_pad + b) * D + lane * E;
        uint16_t *ld = lo + (h * nb_pad + b) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            uint16_t hb = f32_to_bf16_bits(acc[e]);
            float hf = __uint_as_float(uint32_t(hb) << 16);
            hd[e] = hb;
            ld[e] = f32_to_bf16_bits(acc[e] - hf);
        }
    }
}

// fp32 block means -> bf16 hi/lo pair (hi = bf16(x), lo = bf16(x - hi)).
__global__ void __launch_bounds__(256) split_kernel(const float *__restrict__ x, int64_t count,
                                                    uint16_t *__restrict__ hi,
                                                    uint16_t *__restrict__ lo) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float v = x[i];
    const uint16_t hb = f32_to_bf16_bits(v);
    hi[i] = hb;
    lo[i] = f32_to_bf16_bits(v - __uint_as_float(uint32_t(hb) << 16));
}

}  // namespace

cudaError_t launch_split_kbar(const float *kbar, int64_t count, uint16_t *hi, uint16_t *lo,
                              cudaStream_t st) {
    const int threads = 256;
    const int64_t blocks = (count + threads - 1) / threads;
    split_kernel<<<dim3(unsigned(blocks)), threads, 0, st>>>(kbar, count, hi, lo);
    return cudaGetLastError();
}

cudaError_t launch_pool(const void *k, int64_t bh, int64_t n, int32_t d,
                        int32_t kb, float *kbar, uint16_t *kbar_hi,
                        uint16_t *kbar_lo, int64_t nb_pad, cudaStream_t st) {
    const int64_t nb = (n + kb - 1) / kb;
    const int64_t warps = bh * nb;
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    const uint16_t *kk = static_cast<const uint16_t *>(k);
    if (d == 64)
        pool_kernel<64><<<dim3(unsigned(blocks)), threads, 0, st>>>(
            kk, bh, n, kb, nb, kbar, kbar_hi, kbar_lo, nb_pad);
    else
        pool_kernel<128><<<dim3(unsigned(blocks)), threads, 0, st>>>(
            kk, bh, n, kb, nb, kbar, kbar_hi, kbar_lo, nb_pad);
    return cudaGetLastError();
}

}  // namespace bsa
