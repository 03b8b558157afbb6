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
//   scan     exclusive prefix over the bins -> CSR offsets, plus the work
//            list of the fine stage (fine items per bin, merge items per
//            range, see scan_kernel)
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

// Block-wide exclusive scan of two int64 values per thread (1024 threads).
__device__ __forceinline__ void block_scan2(int64_t &a, int64_t &b, int64_t *wa, int64_t *wb) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t a0 = a, b0 = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t x = __shfl_up_sync(0xffffffffu, a, o);
        const int64_t y = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) {
            a += x;
            b += y;
        }
    }
    if (lane == 31) {
        wa[warp] = a;
        wb[warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        int64_t x = wa[lane], y = wb[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t u = __shfl_up_sync(0xffffffffu, x, o);
            const int64_t v = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) {
                x += u;
                y += v;
            }
        }
        wa[lane] = x;
        wb[lane] = y;
    }
    __syncthreads();
    a = a - a0 + (warp > 0 ? wa[warp - 1] : 0);
    b = b - b0 + (warp > 0 ? wb[warp - 1] : 0);
    __syncthreads();
}

// One CTA of 1024 threads.  Builds the CSR offsets over the bins
// (range-major: bin = range * nb + block, range = head * nranges + r) and
// the two work lists of the fine stage: fine items {bin, first pair} (at
// most item_pairs pairs each) in bin order, and merge items {range, first
// query} (qm queries each) in range order.
__global__ void __launch_bounds__(1024) scan_kernel(
    const int32_t *__restrict__ counts, int64_t nb, int64_t nr, int64_t nranges, int64_t range,
    int64_t n, int32_t item_pairs, int32_t qm, int32_t *__restrict__ offsets,
    int32_t *__restrict__ fitem_off, int32_t *__restrict__ fpre, int32_t *__restrict__ mpre,
    int32_t *__restrict__ range_total, int32_t *__restrict__ range_merges,
    int2 *__restrict__ fine_items, int2 *__restrict__ merge_items, int32_t *__restrict__ n_fine,
    int32_t *__restrict__ n_merge) {
    __shared__ int64_t wa[32], wb[32];
    const int t = threadIdx.x;
    const int64_t nbins = nr * nb;
    // 1. bins: pair offsets and fine-item offsets
    const int64_t per = (nbins + 1023) / 1024;
    const int64_t e0 = i64min(nbins, t * per), e1 = i64min(nbins, e0 + per);
    int64_t pairs = 0, fitems = 0;
    for (int64_t e = e0; e < e1; ++e) {
        const int64_t c = counts[e];
        pairs += c;
        fitems += (c + item_pairs - 1) / item_pairs;
    }
    int64_t poff = pairs, foff = fitems;
    block_scan2(poff, foff, wa, wb);
    for (int64_t e = e0; e < e1; ++e) {
        const int64_t c = counts[e];
        offsets[e] = int32_t(poff);
        fitem_off[e] = int32_t(foff);
        poff += c;
        foff += (c + item_pairs - 1) / item_pairs;
    }
    if (t == 1023) {
        offsets[nbins] = int32_t(poff);
        fitem_off[nbins] = int32_t(foff);
    }
    __syncthreads();
    // 2. ranges: pair totals, fine-item and merge-item prefixes
    const int64_t rper = (nr + 1023) / 1024;
    const int64_t r0 = i64min(nr, t * rper), r1 = i64min(nr, r0 + rper);
    int64_t f_sum = 0, m_sum = 0;
    for (int64_t r = r0; r < r1; ++r) {
        const int64_t rr = r % nranges;
        const int64_t queries = i64min(range, n - rr * range);
        const int64_t m = (queries + qm - 1) / qm;
        range_total[r] = offsets[(r + 1) * nb] - offsets[r * nb];
        range_merges[r] = int32_t(m);
        f_sum += fitem_off[(r + 1) * nb] - fitem_off[r * nb];
        m_sum += m;
    }
    int64_t fo = f_sum, mo = m_sum;
    block_scan2(fo, mo, wa, wb);
    for (int64_t r = r0; r < r1; ++r) {
        fpre[r] = int32_t(fo);
        mpre[r] = int32_t(mo);
        fo += fitem_off[(r + 1) * nb] - fitem_off[r * nb];
        mo += range_merges[r];
    }
    if (t == 1023) {
        fpre[nr] = int32_t(fo);
        fpre[nr + 1] = int32_t(fo);
        mpre[nr] = int32_t(mo);
        *n_fine = int32_t(fo);
        *n_merge = int32_t(mo);
    }
    __syncthreads();
    // 3. the work lists: fine items in bin order, merge items in range order
    for (int64_t e = e0; e < e1; ++e) {
        const int64_t c = counts[e];
        int64_t pos = fitem_off[e];
        for (int64_t f = 0; f < c; f += item_pairs) fine_items[pos++] = make_int2(int(e), int(f));
    }
    for (int64_t r = r0; r < r1; ++r) {
        int64_t pos = mpre[r];
        for (int64_t j = 0; j < range_merges[r]; ++j)
            merge_items[pos++] = make_int2(int(r), int(j * qm));
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
            const int64_t i = e / k;
            entries[base[b] + r] = int32_t(((h * n + i) << 5) | (e - i * k));
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

InvertPlan invert_plan(int64_t bh, int64_t n, int64_t nb, int32_t k) {
    InvertPlan p;
    p.range = invert_query_range(n, nb, k);
    p.nranges = (n + p.range - 1) / p.range;
    p.nr = bh * p.nranges;
    p.nbins = p.nr * nb;
    p.item_pairs = kFineBmItemPairs;
    p.qm = kMergeQueries;
    p.fine_cap = p.nbins + (bh * n * k + p.item_pairs - 1) / p.item_pairs;
    p.merge_cap = p.nr * ((p.range + p.qm - 1) / p.qm);
    p.kpad = (k + 3) / 4 * 4;
    return p;
}

cudaError_t launch_invert(const int32_t *list, int64_t bh, int64_t n, int64_t nb, int32_t k,
                          const InvertPlan &p, const InvertBuffers &w, uint16_t *out_bf16,
                          int32_t d, int32_t *status, cudaStream_t st) {
    const dim3 grid(unsigned((n + kQueriesPerCta - 1) / kQueriesPerCta), unsigned(bh));
    const size_t smem1 = size_t(nb) * sizeof(int32_t);
    cudaError_t e = cudaSuccess;
    if (smem1 > 48 * 1024 &&
        (e = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem1))) != cudaSuccess)
        return e;
    if (2 * smem1 > 48 * 1024 &&
        (e = cudaFuncSetAttribute(scatter_kernel<uint16_t>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, int(2 * smem1))) !=
            cudaSuccess)
        return e;
    count_kernel<<<grid, kThreads, smem1, st>>>(list, n, nb, k, p.range, p.nranges, w.counts,
                                               status);
    scan_kernel<<<1, 1024, 0, st>>>(w.counts, nb, p.nr, p.nranges, p.range, n, p.item_pairs, p.qm,
                                    w.offsets, w.fitem_off, w.fpre, w.mpre, w.range_total,
                                    w.range_merges, w.fine_items, w.merge_items, w.n_fine,
                                    w.n_merge);
    scatter_kernel<uint16_t><<<grid, kThreads, 2 * smem1, st>>>(list, n, nb, k, p.range,
                                                                p.nranges, w.offsets, w.cursors,
                                                                w.entries, out_bf16, d);
    return cudaGetLastError();
}

}  // namespace bsa
