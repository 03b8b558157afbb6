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

// One query row i of head h against the listed blocks lp[0 .. nlist) (block
// ids ascending, -1 padding only at the tail; lp may point at global or
// shared memory): running max m, running sum l and the unnormalised
// accumulator, lane t owning channels [E t, E t + E).  qs holds the query
// row in fp32 (shared memory).  Returns l; acc holds the channels.
template <typename T, int D>
__device__ __forceinline__ float row_attention(const FineArgs &a, int64_t h, int64_t i, const float *qs,
                                               const int32_t *lp, int64_t nlist, int lane,
                                               float (&acc)[D / 32], float *m_out = nullptr,
                                               int lstride = 1) {
    constexpr int E = D / 32;
    const T *kh = static_cast<const T *>(a.k) + h * a.n * D;
    const T *vh = static_cast<const T *>(a.v) + h * a.n * D;
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int64_t t = 0; t < nlist; ++t) {
        const int64_t b = lp ? int64_t(lp[t * lstride]) : t;
        if (b < 0) break;                         // padding only at the tail
        if (b >= a.nb) {
            if (lane == 0) report_status(a.status, kStatusBadIndex);
            continue;
        }
        const int64_t j0 = b * a.kb;
        const int64_t j1 = i64min(a.n, j0 + a.kb);
        for (int64_t jc = j0; jc < j1; jc += 32) {
            const int64_t j = jc + lane;
            const int nj = int(i64min(32, j1 - jc));
            const T *vr = vh + jc * D + lane * E;
            // the first 16 keys' values of this lane's channels, loaded before
            // the scores so that the K and V reads overlap
            float va[16][E];
#pragma unroll
            for (int u = 0; u < 16; ++u)
#pragma unroll
                for (int e = 0; e < E; ++e) va[u][e] = u < nj ? Elem<T>::load(vr + u * D + e) : 0.f;
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
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float pu = __shfl_sync(0xffffffffu, p, u);   // 0 past nj
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(pu, va[u][e], acc[e]);
            }
            if (nj > 16) {
#pragma unroll
                for (int u = 0; u < 16; ++u)
#pragma unroll
                    for (int e = 0; e < E; ++e) va[u][e] = 16 + u < nj ? Elem<T>::load(vr + (16 + u) * D + e) : 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float pu = __shfl_sync(0xffffffffu, p, 16 + u);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] = fmaf(pu, va[u][e], acc[e]);
                }
            }
            m = mnew;
        }
    }
    if (m_out != nullptr) *m_out = m;
    return l;
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
    float acc[E];
    const float l = row_attention<T, D>(a, h, i, qs, lp, nlist, lane, acc);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *o = static_cast<T *>(a.out) + row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) Elem<T>::store(o + e, acc[e] * inv);
}

// ------------------------------------------------------------------------
// The whole dynamic forward of a small problem in one launch (page
// "sparse-attention-triton-bench", Key finding: block selection and the
// online softmax fused into a single GPU launch).  One CTA per kSmallQ
// queries of one head: (1) the CTA pools every key block of its head into
// shared memory (fp32 means of the valid keys; the few blocks of a small
// problem make this cheaper than a separate launch), (2) one warp per query
// scores it against every block mean (fp32) and keeps the top-k by k rounds
// of a warp argmax on (score, lower block id first), written ascending to
// the selection, (3) the same warp runs the online-softmax attention over
// the selected blocks (row_attention), each of the query's kSmallWpq warps
// taking every kSmallWpq-th selected block; the warps' running states
// (m, l, acc) are then merged in warp order.  bf16 inputs, no selection
// options.
constexpr int kSmallWarps = 8;
constexpr int kSmallWpq = 1;                      // warps per query
constexpr int kSmallQ = kSmallWarps / kSmallWpq;  // queries per CTA
constexpr int kSmallMaxBlocks = 64;
constexpr int kSmallMaxK = 16;

// order-preserving key of an fp32 score (a larger key is a larger score)
__device__ __forceinline__ uint32_t order_key(float s) {
    const uint32_t u = __float_as_uint(s);
    return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}

template <int D>
__global__ void __launch_bounds__(kSmallWarps * 32) small_forward_kernel(FineArgs a, int32_t topk,
                                                                           int32_t *idx) {
    constexpr int E = D / 32;
    constexpr int KS = D + 1;                     // padded row of the block means
    extern __shared__ float smf[];
    float *kbar = smf;                            // [nb][D + 1]
    float *qsm = smf + kSmallMaxBlocks * KS;      // [kSmallQ][D], then [kSmallWarps][D + 2]
    int32_t *sel = reinterpret_cast<int32_t *>(qsm + kSmallQ * D + kSmallWarps * (D + 2));   // [kSmallQ][kSmallMaxK]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t h = blockIdx.y;
    const uint16_t *kh = static_cast<const uint16_t *>(a.k) + h * a.n * D;
    // (1) block means: thread t sums 8 channels (one 16-byte chunk) of one
    // block at a time over the block's valid keys, loads unrolled so that
    // several are in flight
    for (int64_t w = threadIdx.x; w < a.nb * (D / 8); w += kSmallWarps * 32) {
        const int64_t b = w / (D / 8);
        const int c8 = int(w % (D / 8));
        const int64_t j0 = b * a.kb, j1 = i64min(a.n, j0 + a.kb);
        const uint4 *src = reinterpret_cast<const uint4 *>(kh + j0 * D + c8 * 8);
        float sum[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sum[e] = 0.f;
#pragma unroll 8
        for (int64_t j = 0; j < j1 - j0; ++j) {
            const uint4 x = __ldg(src + j * (D / 8));
            sum[0] += bf16_low_half(x.x);
            sum[1] += bf16_high_half(x.x);
            sum[2] += bf16_low_half(x.y);
            sum[3] += bf16_high_half(x.y);
            sum[4] += bf16_low_half(x.z);
            sum[5] += bf16_high_half(x.z);
            sum[6] += bf16_low_half(x.w);
            sum[7] += bf16_high_half(x.w);
        }
        const float inv = 1.f / float(j1 - j0);
#pragma unroll
        for (int e = 0; e < 8; ++e) kbar[b * KS + c8 * 8 + e] = sum[e] * inv;
    }
    __syncthreads();
    const int qi = warp / kSmallWpq, part = warp % kSmallWpq;
    float *qs = qsm + qi * D;
    int32_t *ws = sel + qi * kSmallMaxK;
    float *pst = qsm + kSmallQ * D;               // per warp: m, l, then D channels
    const int kk = int(i64min(topk, a.nb));
    const int64_t i = int64_t(blockIdx.x) * kSmallQ + qi;
    const bool live = i < a.n;                    // warp-uniform
    const int64_t row = h * a.n + (live ? i : 0);
    if (live && part == 0) {
        const uint16_t *q = static_cast<const uint16_t *>(a.q) + row * D;
#pragma unroll
        for (int e = 0; e < E; ++e) qs[lane * E + e] = Elem<uint16_t>::load(q + lane * E + e);
        __syncwarp();
        // (2) scores of blocks lane and lane + 32; keys: score, then lower id first
        uint64_t key[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int b = lane + 32 * t;
            key[t] = 0;
            if (b < a.nb) {
                float sc = 0.f;
#pragma unroll 8
                for (int c = 0; c < D; ++c) sc = fmaf(qs[c], kbar[b * KS + c], sc);
                key[t] = (uint64_t(order_key(sc)) << 32) | uint32_t(0xFFFFFFFFu - uint32_t(b));
            }
        }
        for (int r = 0; r < kk; ++r) {
            uint64_t best = key[0] > key[1] ? key[0] : key[1];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
                best = other > best ? other : best;
            }
            if (lane == 0) ws[r] = int(0xFFFFFFFFu - uint32_t(best & 0xFFFFFFFFu));
#pragma unroll
            for (int t = 0; t < 2; ++t)
                if (key[t] == best) key[t] = 0;     // taken
        }
        __syncwarp();
        if (lane == 0) {                          // ascending ids (insertion sort, k <= 16)
            for (int x = 1; x < kk; ++x) {
                const int v = ws[x];
                int y = x - 1;
                while (y >= 0 && ws[y] > v) {
                    ws[y + 1] = ws[y];
                    --y;
                }
                ws[y + 1] = v;
            }
        }
        __syncwarp();
        if (lane < topk) idx[row * topk + lane] = lane < kk ? ws[lane] : -1;
    }
    __syncthreads();                              // q rows and selections of the CTA
    // (3) attention: warp `part` of the query takes selected blocks part, part + kSmallWpq, ...
    float acc[E];
    float m = -INFINITY, l = 0.f;
    if (live && part < kk)
        l = row_attention<uint16_t, D>(a, h, i, qs, ws + part, (kk - part + kSmallWpq - 1) / kSmallWpq,
                                       lane, acc, &m, kSmallWpq);
    else {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
    }
    float *mine = pst + warp * (D + 2);
    if (lane == 0) {
        mine[0] = m;
        mine[1] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) mine[2 + lane * E + e] = acc[e];
    __syncthreads();
    if (live && part == 0) {
        // merge the query's warps in order: weights 2^(m_w - M)
        float M = -INFINITY;
        for (int w = 0; w < kSmallWpq; ++w) M = fmaxf(M, pst[(warp + w) * (D + 2)]);
        float L = 0.f, o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = 0.f;
        for (int w = 0; w < kSmallWpq; ++w) {
            const float *pw = pst + (warp + w) * (D + 2);
            const float wt = pw[0] > -INFINITY ? exp2f(pw[0] - M) : 0.f;
            L += wt * pw[1];
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = fmaf(wt, pw[2 + lane * E + e], o[e]);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        uint16_t *dst = static_cast<uint16_t *>(a.out) + row * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) Elem<uint16_t>::store(dst + e, o[e] * inv);
    }
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

bool small_forward_supported(int32_t d, int64_t nb, int32_t topk, int64_t rows) {
    return (d == 64 || d == 128) && nb <= kSmallMaxBlocks && topk <= kSmallMaxK &&
           rows <= kSmallForwardRows;
}

cudaError_t launch_small_forward(const FineArgs &a, int32_t topk, int32_t *idx, cudaStream_t st) {
    const dim3 grid(unsigned((a.n + kSmallQ - 1) / kSmallQ), unsigned(a.bh));
    const size_t smem = (size_t(kSmallMaxBlocks) * (a.d + 1) + size_t(kSmallQ) * a.d +
                         size_t(kSmallWarps) * (a.d + 2)) * sizeof(float) +
                        size_t(kSmallQ) * kSmallMaxK * sizeof(int32_t);
    if (a.d == 64)
        small_forward_kernel<64><<<grid, kSmallWarps * 32, smem, st>>>(a, topk, idx);
    else
        small_forward_kernel<128><<<grid, kSmallWarps * 32, smem, st>>>(a, topk, idx);
    return cudaGetLastError();
}

cudaError_t launch_fine_query_major(const FineArgs &a, int32_t dtype, cudaStream_t st) {
    if (dtype == 0) return launch_t<uint16_t>(a, st);
    return launch_t<float>(a, st);
}

}  // namespace bsa
