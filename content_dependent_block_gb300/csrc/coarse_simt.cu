// Stage 1 scoring + Stage 2 selection, CUDA-core version (page
// "sparse-attention-triton-bench", Two-stage block indexer: score each query
// against every block mean, keep the top-k blocks).
//
// One thread per query; 128 queries of one head per CTA.  The head's block
// means stream through shared memory 32 blocks at a time (each thread reads
// the same Kbar row: a broadcast), the query row lives in registers, and the
// running top-k is a register-resident list kept sorted by (score desc,
// block asc): blocks arrive in ascending order and a candidate displaces an
// entry only when strictly greater, so equal scores keep the lower block id.
// Scores never leave the SM.
//
// This is the portable fallback for shapes the tensor-core kernel does not
// take; fp32 FMA throughout.
#include <climits>

#include "bsa_device.cuh"
#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kQueries = 128;   // threads (queries) per CTA
constexpr int kChunk = 32;      // block means staged per pass

template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&ts)[KMAX], int (&ti)[KMAX],
                                            float s, int b) {
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
        const bool gt = s > ts[t];
        const float ns = gt ? s : ts[t];
        const int ni = gt ? b : ti[t];
        s = gt ? ts[t] : s;
        b = gt ? ti[t] : b;
        ts[t] = ns;
        ti[t] = ni;
    }
}

// Ascending sort of the first `kk` ids (the rest pushed to the end).
template <int KMAX>
__device__ __forceinline__ void sort_ids(int (&ti)[KMAX], int kk) {
#pragma unroll
    for (int t = 0; t < KMAX; ++t)
        if (t >= kk) ti[t] = INT_MAX;
#pragma unroll
    for (int round = 0; round < KMAX; ++round) {
#pragma unroll
        for (int t = round & 1; t + 1 < KMAX; t += 2) {
            const int a = ti[t], c = ti[t + 1];
            ti[t] = min(a, c);
            ti[t + 1] = max(a, c);
        }
    }
}

template <int D, int KMAX>
__global__ void __launch_bounds__(kQueries) coarse_topk_simt_kernel(
    const uint16_t *__restrict__ q, const float *__restrict__ kbar, int64_t n,
    int64_t nb, int32_t topk, const SelectOpts o, int32_t *__restrict__ idx, int32_t *status) {
    __shared__ float ks[kChunk][D];
    const int64_t h = blockIdx.y;
    const int64_t i = int64_t(blockIdx.x) * kQueries + threadIdx.x;
    const bool valid = i < n;
    const int64_t own = i / o.kb;                        // the query's own block
    // eligible blocks: all, or b <= own (causal)
    const int64_t last = o.causal ? own : nb - 1;

    float qr[D];
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(q + (h * n + (valid ? i : 0)) * D);
#pragma unroll
        for (int c = 0; c < D / 2; ++c) {
            const uint32_t x = valid ? __ldg(src + c) : 0u;
            qr[2 * c] = bf16_low_half(x);
            qr[2 * c + 1] = bf16_high_half(x);
        }
    }
    float ts[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
        ts[t] = -INFINITY;
        ti[t] = INT_MAX;
    }

    const float *kh = kbar + h * nb * D;
    for (int64_t c0 = 0; c0 < nb; c0 += kChunk) {
        const int cnt = int(i64min(kChunk, nb - c0));
        __syncthreads();
        for (int e = threadIdx.x; e < cnt * D; e += kQueries)
            ks[e / D][e % D] = kh[c0 * D + e];
        __syncthreads();
        for (int bb = 0; bb < cnt; ++bb) {
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) s = fmaf(qr[c], ks[bb][c], s);
            if (c0 + bb <= last && s > ts[KMAX - 1]) topk_insert<KMAX>(ts, ti, s, int(c0 + bb));
        }
    }
    if (!valid) return;
    int kr = topk;
    if (o.head_k != nullptr) {
        const int32_t hk = __ldg(o.head_k + h);
        kr = min(max(hk, 0), topk);
        if (hk != kr) report_status(status, kStatusInvalidArg);
    }
    apply_budget<KMAX>(ti, kr, int(own), o.local != 0);
    sort_ids<KMAX>(ti, kr);
    int32_t *dst = idx + (h * n + i) * topk;
#pragma unroll
    for (int t = 0; t < KMAX; ++t)
        if (t < topk) dst[t] = (t < kr && ti[t] != INT_MAX) ? ti[t] : -1;
}

template <int D>
cudaError_t launch_d(const void *q, const float *kbar, int64_t bh, int64_t n,
                     int64_t nb, int32_t topk, const SelectOpts &o, int32_t *idx,
                     int32_t *status, cudaStream_t st) {
    const dim3 grid(unsigned((n + kQueries - 1) / kQueries), unsigned(bh));
    const uint16_t *qq = static_cast<const uint16_t *>(q);
    if (topk <= 4)
        coarse_topk_simt_kernel<D, 4><<<grid, kQueries, 0, st>>>(qq, kbar, n, nb, topk, o, idx, status);
    else if (topk <= 8)
        coarse_topk_simt_kernel<D, 8><<<grid, kQueries, 0, st>>>(qq, kbar, n, nb, topk, o, idx, status);
    else if (topk <= 16)
        coarse_topk_simt_kernel<D, 16><<<grid, kQueries, 0, st>>>(qq, kbar, n, nb, topk, o, idx, status);
    else
        coarse_topk_simt_kernel<D, 32><<<grid, kQueries, 0, st>>>(qq, kbar, n, nb, topk, o, idx, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_coarse_topk_simt(const void *q, const float *kbar,
                                    int64_t bh, int64_t n, int32_t d,
                                    int64_t nb, int32_t topk, const SelectOpts &o,
                                    int32_t *idx, int32_t *status, cudaStream_t st) {
    if (d == 64) return launch_d<64>(q, kbar, bh, n, nb, topk, o, idx, status, st);
    return launch_d<128>(q, kbar, bh, n, nb, topk, o, idx, status, st);
}

}  // namespace bsa
