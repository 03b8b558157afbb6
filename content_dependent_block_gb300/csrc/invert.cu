// Inversion of per-query block lists into per-block query lists (CSR), the
// schedule of the block-major fine stage.  Not a step of the method: it
// regroups the selection (page "sparse-attention-triton-bench", Stage 2) so
// that every selected key block is loaded once per group of queries that
// chose it ("Block-Sparse & Linear Attention Kernels", section 4: gather
// through precomputed block indices; dynamic scheduling for balance).
//
// Bins are (head, query range, block): the queries of a head are cut into
// ranges of R queries (R a power of two >= 1024, about two 128-pair tiles
// per bin on average), so that the fine stage finishes one range's partial
// states -- and merges them -- while they are still resident in L2.
//
//   count    per bin: how many (query, slot) pairs selected the block;
//            CTA-local shared-memory histograms, one global atomic per
//            touched bin and CTA
//   scan     exclusive prefix over (head, block) -> CSR offsets, plus the
//            work items (head, block, first pair) of at most kItemPairs
//            pairs each, in head-major order
//   scatter  writes every pair id p = (h*n + i)*k + s into its block's
//            range (order inside a range is arbitrary; results do not
//            depend on it); queries with no valid slot get O = 0 here
//
// Entries outside [0, nb) are skipped and reported (BSA_ERR_BAD_INDEX);
// -1 entries are padding.
#include "bsa_device.cuh"
#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kThreads = 256;
constexpr int kQueriesPerCta = 1024;   // queries of one head per count/scatter CTA

__device__ __forceinline__ bool valid_block(int32_t b, int64_t nb) { return b >= 0 && b < nb; }

// grid: (ceil(n / kQueriesPerCta), bh); dynamic smem: nb ints
__global__ void __launch_bounds__(kThreads) count_kernel(const int32_t *__restrict__ list,
                                                         int64_t n, int64_t nb, int32_t k,
                                                         int64_t range, int64_t nranges,
                                                         int32_t *__restrict__ counts,
                                                         int32_t *status) {
    extern __shared__ int32_t hist[];
    const int64_t h = blockIdx.y;
    const int64_t i0 = int64_t(blockIdx.x) * kQueriesPerCta;
    const int64_t i1 = i64min(n, i0 + kQueriesPerCta);
    for (int64_t b = threadIdx.x; b < nb; b += kThreads) hist[b] = 0;
    __syncthreads();
    const int32_t *base = list + (h * n) * k;
    bool bad = false;
    for (int64_t e = i0 * k + threadIdx.x; e < i1 * k; e += kThreads) {
        const int32_t b = __ldg(base + e);
        if (valid_block(b, nb)) atomicAdd(&hist[b], 1);
        else if (b >= 0 || b < -1) bad = true;
    }
    if (bad) report_status(status, kStatusBadIndex);
    __syncthreads();
    const int64_t bin0 = (h * nranges + i0 / range) * nb;
    for (int64_t b = threadIdx.x; b < nb; b += kThreads)
        if (hist[b] != 0) atomicAdd(counts + bin0 + b, hist[b]);
}

// One CTA of 1024 threads over the nbh bins (head, query range, block):
// offsets[nbh + 1], items[...] = {bin, first pair}
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t *__restrict__ counts,
                                                    int64_t nbh, int32_t item_pairs,
                                                    int32_t *__restrict__ offsets,
                                                    int2 *__restrict__ items,
                                                    int32_t *__restrict__ n_items) {
    __shared__ int64_t warp_pairs[32];
    __shared__ int64_t warp_items[32];
    const int t = threadIdx.x;
    const int64_t per = (nbh + 1023) / 1024;
    const int64_t e0 = i64min(nbh, t * per);
    const int64_t e1 = i64min(nbh, e0 + per);
    int64_t my_pairs = 0, my_items = 0;
    for (int64_t e = e0; e < e1; ++e) {
        const int64_t c = counts[e];
        my_pairs += c;
        my_items += (c + item_pairs - 1) / item_pairs;
    }
    // block-wide exclusive scan of (pairs, items)
    int64_t ip = my_pairs, ii = my_items;
    const int lane = t & 31, warp = t >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t a = __shfl_up_sync(0xffffffffu, ip, o);
        const int64_t b = __shfl_up_sync(0xffffffffu, ii, o);
        if (lane >= o) {
            ip += a;
            ii += b;
        }
    }
    if (lane == 31) {
        warp_pairs[warp] = ip;
        warp_items[warp] = ii;
    }
    __syncthreads();
    if (warp == 0) {
        int64_t wp = warp_pairs[lane], wi = warp_items[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t a = __shfl_up_sync(0xffffffffu, wp, o);
            const int64_t b = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) {
                wp += a;
                wi += b;
            }
        }
        warp_pairs[lane] = wp;   // inclusive over warps
        warp_items[lane] = wi;
    }
    __syncthreads();
    int64_t pair_off = ip - my_pairs + (warp > 0 ? warp_pairs[warp - 1] : 0);
    int64_t item_off = ii - my_items + (warp > 0 ? warp_items[warp - 1] : 0);
    for (int64_t e = e0; e < e1; ++e) {
        const int64_t c = counts[e];
        offsets[e] = int32_t(pair_off);
        for (int64_t f = 0; f < c; f += item_pairs) items[item_off++] = make_int2(int(e), int(f));
        pair_off += c;
    }
    if (t == 1023) {
        offsets[nbh] = int32_t(pair_off);
        *n_items = int32_t(item_off);
    }
}

// grid: (ceil(n / kQueriesPerCta), bh); dynamic smem: 2 * nb ints
template <typename OutT>
__global__ void __launch_bounds__(kThreads) scatter_kernel(
    const int32_t *__restrict__ list, int64_t n, int64_t nb, int32_t k, int64_t range,
    int64_t nranges, const int32_t *__restrict__ offsets, int32_t *__restrict__ cursors,
    int32_t *__restrict__ entries, OutT *__restrict__ out, int32_t d) {
    extern __shared__ int32_t sm[];
    int32_t *hist = sm;          // pairs of this CTA per block
    int32_t *base = sm + nb;     // first slot of this CTA inside the block's range
    const int64_t h = blockIdx.y;
    const int64_t i0 = int64_t(blockIdx.x) * kQueriesPerCta;
    const int64_t i1 = i64min(n, i0 + kQueriesPerCta);
    for (int64_t b = threadIdx.x; b < nb; b += kThreads) hist[b] = 0;
    __syncthreads();
    const int32_t *lh = list + (h * n) * k;
    for (int64_t e = i0 * k + threadIdx.x; e < i1 * k; e += kThreads) {
        const int32_t b = __ldg(lh + e);
        if (valid_block(b, nb)) atomicAdd(&hist[b], 1);
    }
    __syncthreads();
    const int64_t bin0 = (h * nranges + i0 / range) * nb;
    for (int64_t b = threadIdx.x; b < nb; b += kThreads) {
        const int32_t c = hist[b];
        base[b] = c ? offsets[bin0 + b] + atomicAdd(cursors + bin0 + b, c) : 0;
        hist[b] = 0;
    }
    __syncthreads();
    for (int64_t e = i0 * k + threadIdx.x; e < i1 * k; e += kThreads) {
        const int32_t b = __ldg(lh + e);
        if (valid_block(b, nb)) {
            const int32_t r = atomicAdd(&hist[b], 1);
            entries[base[b] + r] = int32_t(h * n * k + e);
        }
    }
    // queries whose list admits nothing: their output is zero
    for (int64_t i = i0 + threadIdx.x; i < i1; i += kThreads) {
        bool any = false;
        for (int s = 0; s < k; ++s) any |= valid_block(__ldg(lh + i * k + s), nb);
        if (!any) {
            OutT *o = out + (h * n + i) * d;
            for (int c = 0; c < d; ++c) o[c] = OutT(0);
        }
    }
}

}  // namespace

int64_t invert_query_range(int64_t n, int64_t nb, int32_t k) {
    // about two full 128-pair tiles per (range, block) on average
    int64_t r = kQueriesPerCta;
    while (r * k < int64_t(256) * nb && r < n) r *= 2;
    return r;
}

int64_t invert_bins(int64_t bh, int64_t n, int64_t nb, int32_t k) {
    const int64_t r = invert_query_range(n, nb, k);
    return bh * ((n + r - 1) / r) * nb;
}

size_t invert_items_capacity(int64_t bh, int64_t n, int64_t nb, int32_t k, int32_t item_pairs) {
    return size_t(invert_bins(bh, n, nb, k)) + size_t((bh * n * k + item_pairs - 1) / item_pairs);
}

cudaError_t launch_invert(const int32_t *list, int64_t bh, int64_t n, int64_t nb, int32_t k,
                          int32_t item_pairs, int32_t *counts, int32_t *cursors,
                          int32_t *offsets, int2 *items, int32_t *n_items, int32_t *entries,
                          uint16_t *out_bf16, int32_t d, int32_t *status, cudaStream_t st) {
    const dim3 grid(unsigned((n + kQueriesPerCta - 1) / kQueriesPerCta), unsigned(bh));
    const size_t smem1 = size_t(nb) * sizeof(int32_t);
    if (smem1 > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem1));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(scatter_kernel<uint16_t>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(2 * smem1));
        if (e != cudaSuccess) return e;
    } else if (2 * smem1 > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(scatter_kernel<uint16_t>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(2 * smem1));
        if (e != cudaSuccess) return e;
    }
    const int64_t range = invert_query_range(n, nb, k);
    const int64_t nranges = (n + range - 1) / range;
    count_kernel<<<grid, kThreads, smem1, st>>>(list, n, nb, k, range, nranges, counts, status);
    scan_kernel<<<1, 1024, 0, st>>>(counts, bh * nranges * nb, item_pairs, offsets, items, n_items);
    scatter_kernel<uint16_t><<<grid, kThreads, 2 * smem1, st>>>(list, n, nb, k, range, nranges,
                                                                offsets, cursors, entries, out_bf16, d);
    return cudaGetLastError();
}

}  // namespace bsa
