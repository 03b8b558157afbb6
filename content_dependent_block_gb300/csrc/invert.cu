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
//   scatter  writes every pair id p = ((h*n + i) << 5) | s into its block's
//            range (order inside a range is arbitrary; results do not
//            depend on it) and every query's mask of valid slots (for the
//            merge); queries with no valid slot get O = 0 here
//
// Entries outside [0, nb) are skipped and reported (BSA_ERR_BAD_INDEX);
// -1 entries are padding.
#include "bsa_device.cuh"
#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kThreads = 256;
constexpr int kQueriesPerCta = 256;    // queries of one head per count/scatter CTA
constexpr int kScanThreads = 1024;
constexpr int kScanV = 4;              // bins per thread per scan chunk
constexpr int kScanG = 4;              // chunks whose counts are loaded together
constexpr int kScanStage = 8192;       // fine items of a chunk staged in shared memory
static_assert(kFineBmItemPairs == 512, "fine items are cut at 512 pairs (shift below)");

__device__ __forceinline__ bool valid_block(int32_t b, int64_t nb) { return b >= 0 && b < nb; }

// A CTA's list entries, kQueriesPerCta x k <= kThreads x kEntriesMax: thread
// t holds entries t + j * kThreads, all loaded before any is used (the
// shared-memory atomics that follow would otherwise keep the compiler from
// overlapping the loads).
constexpr int kEntriesMax = kQueriesPerCta * 32 / kThreads;
struct CtaEntries {
    int32_t v[kEntriesMax];
    __device__ __forceinline__ void load(const int32_t *__restrict__ base, int32_t m) {
#pragma unroll
        for (int j = 0; j < kEntriesMax; ++j) {
            const int32_t e = int32_t(threadIdx.x) + j * kThreads;
            v[j] = e < m ? __ldg(base + e) : -1;
        }
    }
};

// floor(e / k) for 0 <= e < 2^16 and 1 <= k <= 32: e * ceil(2^32 / k) / 2^32,
// exact because the rounding error (< e / 2^32) stays below 1 / k.
__device__ __forceinline__ uint32_t div_small(uint32_t e, uint32_t magic) { return __umulhi(e, magic); }

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
    const int32_t m = int32_t((i1 - i0) * k);
    CtaEntries ent;
    ent.load(list + (h * n + i0) * k, m);
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kEntriesMax; ++j) {
        const int32_t b = ent.v[j];
        if (valid_block(b, nb)) atomicAdd(&hist[b], 1);
        else if (b >= 0 || b < -1) bad = true;
    }
    if (bad) report_status(status, kStatusBadIndex);
    __syncthreads();
    int32_t *dst = counts + (h * nranges + i0 / range) * nb;
    for (int64_t b = threadIdx.x; b < nb; b += kThreads)
        if (hist[b] != 0) atomicAdd(dst + b, hist[b]);
}

// Block-wide exclusive scan of two int32 values per thread (kScanThreads
// threads); also returns the block totals.
__device__ __forceinline__ void block_scan2(int32_t &a, int32_t &b, int32_t &ta, int32_t &tb,
                                            int32_t *wa, int32_t *wb) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t a0 = a, b0 = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t x = __shfl_up_sync(0xffffffffu, a, o);
        const int32_t y = __shfl_up_sync(0xffffffffu, b, o);
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
        int32_t x = wa[lane], y = wb[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, x, o);
            const int32_t v = __shfl_up_sync(0xffffffffu, y, o);
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
    ta = wa[31];
    tb = wb[31];
    __syncthreads();
}

// One CTA of 1024 threads.  Builds the CSR offsets over the bins
// (range-major: bin = range * nb + block, range = head * nranges + r) and
// the two work lists of the fine stage: fine items {bin, first pair} (at
// most 512 pairs each) in bin order, and merge items {range, first query}
// (qm queries each) in range order.  Bins are scanned in coalesced chunks of
// 4 bins per thread with a running carry; the counts of four chunks are
// loaded at once, and a chunk's offsets are stored 16 bytes per thread and
// its fine items staged in shared memory and copied out contiguously (one
// CTA's scattered small stores would otherwise each cost an L2 transaction).
// Dynamic shared memory: kScanStage int2.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(
    const int32_t *__restrict__ counts, int64_t nb, int64_t nr, int64_t nranges, int64_t range,
    int64_t n, int32_t item_pairs, int32_t qm, int32_t *__restrict__ offsets,
    int32_t *__restrict__ fitem_off, int32_t *__restrict__ fpre, int32_t *__restrict__ mpre,
    int32_t *__restrict__ range_total, int32_t *__restrict__ range_merges,
    int2 *__restrict__ fine_items, int2 *__restrict__ merge_items, int32_t *__restrict__ n_fine,
    int32_t *__restrict__ n_merge) {
    __shared__ int32_t wa[32], wb[32];
    extern __shared__ int2 stage[];
    const int t = threadIdx.x;
    const int32_t nbins = int32_t(nr * nb);
    // 1. bins: pair offsets, fine-item offsets and the fine items themselves
    int32_t carry_p = 0, carry_f = 0;
    for (int32_t base0 = 0; base0 < nbins; base0 += kScanThreads * kScanV * kScanG) {
        int4 cv[kScanG];
#pragma unroll
        for (int g = 0; g < kScanG; ++g) {
            const int32_t e = base0 + g * kScanThreads * kScanV + t * kScanV;
            if (e + kScanV <= nbins) {
                cv[g] = *reinterpret_cast<const int4 *>(counts + e);   // 16-byte aligned
            } else {
                cv[g].x = e < nbins ? counts[e] : 0;
                cv[g].y = e + 1 < nbins ? counts[e + 1] : 0;
                cv[g].z = e + 2 < nbins ? counts[e + 2] : 0;
                cv[g].w = e + 3 < nbins ? counts[e + 3] : 0;
            }
        }
#pragma unroll
        for (int g = 0; g < kScanG; ++g) {
            const int32_t base = base0 + g * kScanThreads * kScanV;
            if (base >= nbins) break;                 // uniform over the CTA
            const int32_t e = base + t * kScanV;
            const int32_t c[kScanV] = {cv[g].x, cv[g].y, cv[g].z, cv[g].w};
            int32_t p = 0, f = 0;
#pragma unroll
            for (int q = 0; q < kScanV; ++q) {
                p += c[q];
                f += (c[q] + 511) >> 9;
            }
            int32_t tp, tf;
            block_scan2(p, f, tp, tf, wa, wb);
            p += carry_p;
            f += carry_f;
            int32_t po[kScanV], fo[kScanV];
#pragma unroll
            for (int q = 0; q < kScanV; ++q) {
                po[q] = p;
                fo[q] = f;
                for (int32_t x = 0; x < c[q]; x += 512, ++f) {
                    const int32_t at = f - carry_f;        // chunk-local item index
                    if (at < kScanStage) stage[at] = make_int2(e + q, x);
                    else fine_items[f] = make_int2(e + q, x);
                }
                p += c[q];
            }
            if (e + kScanV <= nbins) {
                *reinterpret_cast<int4 *>(offsets + e) = make_int4(po[0], po[1], po[2], po[3]);
                *reinterpret_cast<int4 *>(fitem_off + e) = make_int4(fo[0], fo[1], fo[2], fo[3]);
            } else {
                for (int q = 0; q < kScanV && e + q < nbins; ++q) {
                    offsets[e + q] = po[q];
                    fitem_off[e + q] = fo[q];
                }
            }
            __syncthreads();
            for (int32_t i = t; i < min(tf, kScanStage); i += kScanThreads) fine_items[carry_f + i] = stage[i];
            __syncthreads();
            carry_p += tp;
            carry_f += tf;
        }
    }
    if (t == 0) {
        offsets[nbins] = carry_p;
        fitem_off[nbins] = carry_f;
        *n_fine = carry_f;
    }
    __syncthreads();
    // 2. ranges: pair totals, merge-item counts and prefixes
    int32_t carry_m = 0;
    for (int64_t base = 0; base < nr; base += kScanThreads) {
        const int64_t r = base + t;
        int32_t m = 0, dummy = 0;
        if (r < nr) {
            const int64_t rr = r % nranges;
            const int64_t queries = i64min(range, n - rr * range);
            m = int32_t((queries + qm - 1) / qm);
            range_total[r] = offsets[(r + 1) * nb] - offsets[r * nb];
            range_merges[r] = m;
            fpre[r] = fitem_off[r * nb];
        }
        int32_t mo = m, tm, td;
        block_scan2(mo, dummy, tm, td, wa, wb);
        if (r < nr) mpre[r] = carry_m + mo;
        carry_m += tm;
    }
    if (t == 0) {
        fpre[nr] = carry_f;
        fpre[nr + 1] = carry_f;
        mpre[nr] = carry_m;
        *n_merge = carry_m;
    }
    __syncthreads();
    // 3. merge items, one per thread.  Every head has the same ranges: full
    //    ones with range / qm items and a last one with m_last items, so the
    //    range of item mi follows in closed form.
    const int32_t m_full = int32_t(range / qm);
    const int32_t m_last = int32_t((n - (nranges - 1) * range + qm - 1) / qm);
    const int32_t m_head = int32_t(nranges - 1) * m_full + m_last;
    for (int32_t mi = t; mi < carry_m; mi += kScanThreads) {
        const int32_t hh = mi / m_head, rem = mi - hh * m_head;
        const int32_t rr = min(rem / m_full, int32_t(nranges - 1));
        const int32_t j = rem - rr * m_full;
        merge_items[mi] = make_int2(int(hh * nranges + rr), j * qm);
    }
}

// grid: (ceil(n / kQueriesPerCta), bh); dynamic smem: 2 * nb + kQueriesPerCta ints
template <typename OutT>
__global__ void __launch_bounds__(kThreads) scatter_kernel(
    const int32_t *__restrict__ list, int64_t n, int64_t nb, int32_t k, int64_t range,
    int64_t nranges, const int32_t *__restrict__ offsets, int32_t *__restrict__ cursors,
    int32_t *__restrict__ entries, uint32_t *__restrict__ vmask, OutT *__restrict__ out,
    int32_t d) {
    extern __shared__ int32_t sm[];
    int32_t *hist = sm;          // pairs of this CTA per block
    int32_t *base = sm + nb;     // first slot of this CTA inside the block's range
    // per query of the CTA: bit s set when slot s holds a block
    uint32_t *any = reinterpret_cast<uint32_t *>(sm + 2 * nb);
    const int64_t h = blockIdx.y;
    const int64_t i0 = int64_t(blockIdx.x) * kQueriesPerCta;
    const int64_t i1 = i64min(n, i0 + kQueriesPerCta);
    for (int64_t b = threadIdx.x; b < nb; b += kThreads) hist[b] = 0;
    for (int q = threadIdx.x; q < kQueriesPerCta; q += kThreads) any[q] = 0;
    __syncthreads();
    const int32_t *lh = list + (h * n + i0) * k;
    const int32_t m = int32_t((i1 - i0) * k);
    for (int32_t e = threadIdx.x; e < m; e += kThreads) {
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
    const uint32_t magic = 0xFFFFFFFFu / uint32_t(k) + 1u;
    const int32_t row0 = int32_t(h * n + i0);
    for (int32_t e = threadIdx.x; e < m; e += kThreads) {
        const int32_t b = __ldg(lh + e);
        if (valid_block(b, nb)) {
            const int32_t il = int32_t(div_small(uint32_t(e), magic));
            const int32_t r = atomicAdd(&hist[b], 1);
            entries[base[b] + r] = ((row0 + il) << 5) | (e - il * k);
            atomicOr(&any[il], 1u << (e - il * k));
        }
    }
    __syncthreads();
    // the slot masks, for the merge; queries whose list admits nothing:
    // their output is zero
    for (int64_t i = i0 + threadIdx.x; i < i1; i += kThreads) {
        if (vmask != nullptr) vmask[h * n + i] = any[i - i0];
        if (!any[i - i0]) {
            OutT *o = out + (h * n + i) * d;
            for (int c = 0; c < d; ++c) o[c] = OutT(0);
        }
    }
}

}  // namespace

int64_t invert_query_range(int64_t n, int64_t nb, int32_t k) {
    // about two full 128-pair tiles per (range, block) on average; a power
    // of two >= 1024, so a count/scatter CTA never straddles two ranges
    int64_t r = 1024;
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
    if (k < 1 || k > 32) return cudaErrorInvalidValue;   // CtaEntries holds 32 per query
    const dim3 grid(unsigned((n + kQueriesPerCta - 1) / kQueriesPerCta), unsigned(bh));
    const size_t smem1 = size_t(nb) * sizeof(int32_t);
    const size_t smem2 = 2 * smem1 + kQueriesPerCta * sizeof(int32_t);
    cudaError_t e = cudaSuccess;
    if (smem1 > 48 * 1024 &&
        (e = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem1))) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(kScanStage * sizeof(int2)))) != cudaSuccess)
        return e;
    if (smem2 > 48 * 1024 &&
        (e = cudaFuncSetAttribute(scatter_kernel<uint16_t>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem2))) !=
            cudaSuccess)
        return e;
    count_kernel<<<grid, kThreads, smem1, st>>>(list, n, nb, k, p.range, p.nranges, w.counts,
                                               status);
    scan_kernel<<<1, kScanThreads, kScanStage * sizeof(int2), st>>>(
        w.counts, nb, p.nr, p.nranges, p.range, n, p.item_pairs, p.qm, w.offsets, w.fitem_off,
        w.fpre, w.mpre, w.range_total, w.range_merges, w.fine_items, w.merge_items, w.n_fine,
        w.n_merge);
    scatter_kernel<uint16_t><<<grid, kThreads, smem2, st>>>(list, n, nb, k, p.range,
                                                                p.nranges, w.offsets, w.cursors,
                                                                w.entries, w.vmask, out_bf16, d);
    return cudaGetLastError();
}

}  // namespace bsa
