// Stage 1 scoring + Stage 2 selection on the tensor cores (page
// "sparse-attention-triton-bench", Two-stage block indexer: score every
// query against every block mean -- "Q @ K_block_repr.T" -- and keep the
// top-k blocks per query).
//
// The scoring is a dense contraction S = Q . Kbar^T, so it runs as tcgen05
// MMAs into tensor memory; the N x N/B score matrix never reaches HBM.
//
// One CTA owns a 128-query tile of one head (M = 128 TMEM lanes, one query
// per lane) and streams the head's block means through shared memory in
// chunks of kChunk = 128 blocks (MMA N = 128), double-buffered in shared
// memory and in tensor memory:
//   warp 0      TMA producer: Q tile once, then Kbar chunks (hi and lo parts)
//   warp 1      allocates tensor memory; runs the MMA loop warp-uniformly and
//               one elected lane issues
//   warps 2..9  epilogue, two groups of four warps (one per TMEM lane
//               quadrant); group e reads the 32-column slices j = e mod 2 of
//               every chunk, so each thread scans half of its query's scores
//               and keeps a running top-k in registers; the two lists are
//               merged at the end
// Selection: a thread compares each score's key with its current k-th key
// and queues the ones that beat it in shared memory (no branches); when a
// lane of the warp has 16 queued, every lane sorts its first 16 by a bitonic
// network and merges them into its running top-k (element-wise max against
// the reversed batch, then a bitonic merge).  The sorting work follows the
// scores that can still enter the top-k, not all of them.
// Precision: Kbar enters as a bf16 pair (hi = bf16(Kbar), lo = bf16(Kbar -
// hi)); S = Q.hi + Q.lo accumulates in fp32, i.e. about 2^-16 relative to
// the fp32 mean -- far inside the 1e-3 relative tie band of the selection.
// Q is bf16 already, so it is exact.
//
// Top-k keys: each score becomes one order-preserving 32-bit key whose low
// `bits` = ceil(log2 nb) bits hold (mask - block): a larger key is a larger
// score, and equal truncated scores rank the lower block first.  The
// truncation drops `bits` mantissa bits (<= 2^-11 relative for nb <= 4096),
// so two blocks can only swap when their scores agree to that precision.
// The register list is kept sorted by a compare-exchange pass (min/max).
#include <climits>
#include <type_traits>

#include <cudaTypedefs.h>

#include "bsa_device.cuh"
#include "bsa_internal.h"
#include "tc.cuh"

namespace bsa {
namespace {

constexpr int kTileM = 128;        // queries per CTA (TMEM lanes)
constexpr int kChunk = 128;        // blocks per MMA (N)
constexpr int kStages = 2;         // shared-memory stages of Kbar chunks
constexpr int kGroups = 2;         // epilogue warpgroups (column split)
constexpr int kEpi = kGroups * kTileM;
constexpr int kThreads = 64 + kEpi;
constexpr int kTmemCols = 2 * kChunk;
constexpr int kSlice = 8;          // scores filtered between drain checks (divides 32)
constexpr int kQueue = 16 + kSlice;   // queued keys per thread: < 16 after a drain, + one slice
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct CoarseSmem {
    static constexpr int kSub = D / 64;                       // 128-byte K slabs
    static constexpr int kQBytes = kSub * kTileM * 128;
    static constexpr int kKBytes = kSub * kChunk * 128;       // one of hi / lo
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kTiles = kQBytes + kStages * kStageBytes;
    static constexpr int oQueue = kTiles;                     // uint32 [kQueue][kEpi]; after the
                                                              // scan, [KMAX <= 32][kTileM] lists
    static constexpr int kQueueWords = kQueue * kEpi > 32 * kTileM ? kQueue * kEpi : 32 * kTileM;
    static constexpr int oBar = oQueue + kQueueWords * 4;
    static constexpr int kTotal = oBar + 256 /*barriers*/ + 1024 /*align*/;
};

__device__ __forceinline__ uint32_t score_key(float s, uint32_t col, uint32_t mask) {
    uint32_t u = __float_as_uint(s);
    u ^= uint32_t(int32_t(u) >> 31) | 0x80000000u;
    return (u & ~mask) | (mask - col);
}

// Compare-exchange: afterwards a >= b.
__device__ __forceinline__ void cx(uint32_t &a, uint32_t &b) {
    const uint32_t hi = max(a, b), lo = min(a, b);
    a = hi;
    b = lo;
}

// Sort 16 keys in descending order (bitonic network, 80 compare-exchanges).
__device__ __forceinline__ void sort16_desc(uint32_t (&B)[16]) {
#pragma unroll
    for (int k = 2; k <= 16; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    if ((i & k) == 0) cx(B[i], B[l]);
                    else cx(B[l], B[i]);
                }
            }
}

// L (KMAX keys, descending) becomes the top KMAX of L and B (N keys,
// descending).  Against B reversed, the element-wise max of L's last
// min(KMAX, N) slots is a bitonic sequence holding the top KMAX of the union;
// a bitonic merge sorts it descending.  No branches: every lane runs the same
// compare-exchanges.
template <int KMAX, int N>
__device__ __forceinline__ void merge_sorted(uint32_t (&L)[KMAX], const uint32_t (&B)[N]) {
    constexpr int NB = KMAX < N ? KMAX : N;
#pragma unroll
    for (int t = 0; t < NB; ++t) L[KMAX - NB + t] = max(L[KMAX - NB + t], B[NB - 1 - t]);
#pragma unroll
    for (int j = KMAX >> 1; j > 0; j >>= 1)
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            const int l = i ^ j;
            if (l > i) cx(L[i], L[l]);
        }
}

// kOpts: the selection options of `o` are in use (a separate instance, so
// that the plain kernel carries none of their code).
template <int D, int KMAX, bool kOpts>
__global__ void __launch_bounds__(kThreads, 2) coarse_topk_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_hi,
    const __grid_constant__ CUtensorMap tm_lo, int64_t n, int64_t nb, int32_t topk,
    uint32_t key_mask, const SelectOpts o, int32_t *__restrict__ idx, int32_t *status) {
    using S = CoarseSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = tc::align_smem_1024(smem_raw);
    uint8_t *sQ = smem;
    uint8_t *sK = smem + S::kQBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::oBar);
    uint32_t *queue = reinterpret_cast<uint32_t *>(smem + S::oQueue);
    uint32_t *merge = queue;                // reused once every queue is drained
    uint64_t *q_full = bars + 0;
    uint64_t *kv_full = bars + 1;       // [kStages]
    uint64_t *kv_empty = bars + 3;      // [kStages]
    uint64_t *acc_full = bars + 5;      // [2]
    uint64_t *acc_empty = bars + 7;     // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 9);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t h = blockIdx.y;
    const int64_t row0 = int64_t(blockIdx.x) * kTileM;
    const int nchunks = int((nb + kChunk - 1) / kChunk);
    // A wait elsewhere already ran out: do no work (results are invalid anyway).
    // The whole CTA takes the same decision.
    if (__syncthreads_or(status != nullptr &&
                         *reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout))
        return;

    if (threadIdx.x == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(kv_full + s, 1);
            tc::mbar_init(kv_empty + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(acc_full + s, 1);
            tc::mbar_init(acc_empty + s, kEpi);
        }
        tc::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tensormap(&tm_q);
        tc::prefetch_tensormap(&tm_hi);
        tc::prefetch_tensormap(&tm_lo);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------- TMA producer
            tc::mbar_arrive_expect_tx(q_full, S::kQBytes);
#pragma unroll
            for (int sub = 0; sub < S::kSub; ++sub)
                tc::tma_load_3d(sQ + sub * kTileM * 128, &tm_q, q_full, sub * 64, int32_t(row0),
                                int32_t(h));
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kStages;
                const int use = c / kStages;
                if (use > 0 && !tc::mbar_wait(kv_empty + s, (use - 1) & 1, status)) break;
                uint8_t *hi = sK + s * S::kStageBytes;
                uint8_t *lo = hi + S::kKBytes;
                tc::mbar_arrive_expect_tx(kv_full + s, S::kStageBytes);
#pragma unroll
                for (int sub = 0; sub < S::kSub; ++sub) {
                    tc::tma_load_3d(hi + sub * kChunk * 128, &tm_hi, kv_full + s, sub * 64,
                                    c * kChunk, int32_t(h));
                    tc::tma_load_3d(lo + sub * kChunk * 128, &tm_lo, kv_full + s, sub * 64,
                                    c * kChunk, int32_t(h));
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        // warp-uniform loop, one elected lane issues
        constexpr uint32_t idesc = tc::idesc_bf16_f32(kTileM, kChunk);
        bool ok = tc::mbar_wait(q_full, 0, status);
        ok = __all_sync(kFull, ok);
        const uint32_t q_addr = tc::smem_u32(sQ);
        for (int c = 0; ok && c < nchunks; ++c) {
            const int s = c % kStages;
            const int buf = c & 1;
            ok = tc::mbar_wait(kv_full + s, (c / kStages) & 1, status);
            if (ok && c >= 2) ok = tc::mbar_wait(acc_empty + buf, ((c >> 1) - 1) & 1, status);
            if (!__all_sync(kFull, ok)) break;
            tc::tc_fence_after();
            if (tc::elect_one()) {
                const uint32_t hi_addr = tc::smem_u32(sK + s * S::kStageBytes);
                const uint32_t lo_addr = hi_addr + S::kKBytes;
                const uint32_t d_tmem = tmem + uint32_t(buf * kChunk);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = uint32_t((kk >> 2) * kTileM * 128 + (kk & 3) * 32);
                    const uint32_t boff = uint32_t((kk >> 2) * kChunk * 128 + (kk & 3) * 32);
                    tc::mma_bf16(d_tmem, tc::smem_desc_sw128(q_addr + koff, 1024),
                                 tc::smem_desc_sw128(hi_addr + boff, 1024), idesc, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = uint32_t((kk >> 2) * kTileM * 128 + (kk & 3) * 32);
                    const uint32_t boff = uint32_t((kk >> 2) * kChunk * 128 + (kk & 3) * 32);
                    tc::mma_bf16(d_tmem, tc::smem_desc_sw128(q_addr + koff, 1024),
                                 tc::smem_desc_sw128(lo_addr + boff, 1024), idesc, 1);
                }
                tc::mma_commit(kv_empty + s);
                tc::mma_commit(acc_full + buf);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int eg = (warp - 2) >> 2;            // column group
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;            // row inside the tile
        const int64_t own = kOpts ? (row0 + r) / o.kb : 0;   // the query's own block
        uint32_t L[KMAX];
#pragma unroll
        for (int t = 0; t < KMAX; ++t) L[t] = 0u;  // 0 = empty (below every real key)
        // Selection: keys that beat the thread's current k-th key wait in a
        // small shared-memory queue (this thread's column of it); whenever a
        // lane of the warp has 16 queued, every lane sorts its first 16
        // (bitonic, padded with empty keys) and merges them into L.  Most
        // scores stop at one compare; the sort runs on the few that pass.
        uint32_t *qu = queue + eg * kTileM + r;    // [kQueue][kEpi]
        int cnt = 0;
        auto drain = [&]() {
            uint32_t B[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) B[t] = t < cnt ? qu[t * kEpi] : 0u;
            sort16_desc(B);
            merge_sorted<KMAX, 16>(L, B);
#pragma unroll
            for (int t = 0; t < kQueue - 16; ++t)
                if (16 + t < cnt) qu[t * kEpi] = qu[(16 + t) * kEpi];
            cnt = max(cnt - 16, 0);
        };
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const int buf = c & 1;
            if (ok) ok = tc::mbar_wait(acc_full + buf, (c >> 1) & 1, status);
            tc::tc_fence_after();
            if (ok) {
                const int valid = int(i64min(kChunk, nb - int64_t(c) * kChunk));
                for (int j = eg; j < kChunk / 32; j += kGroups) {
                    if (j * 32 >= valid) break;
                    const uint32_t col0 = uint32_t(c * kChunk + j * 32);
                    int lim = valid - j * 32;
                    if (kOpts && o.causal) {
                        // eligible blocks b <= own; skip 32 columns no row of the warp may take
                        lim = int(i64min(lim, i64max(0, own - int64_t(col0) + 1)));
                        if (__all_sync(0xffffffffu, lim == 0)) continue;
                    }
                    uint32_t v[32];
                    tc::tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + uint32_t(buf * kChunk + j * 32), v);
                    tc::tmem_ld_wait();
                    // queue the keys that beat the current k-th key (no branches); a
                    // group of 32 valid columns (the common case) skips the bound check
                    auto filter = [&](auto whole) {
#pragma unroll
                        for (int hf = 0; hf < 32 / kSlice; ++hf) {
                            const uint32_t thr = L[KMAX - 1];
#pragma unroll
                            for (int e = 0; e < kSlice; ++e) {
                                const int x = hf * kSlice + e;
                                const uint32_t key = score_key(__uint_as_float(v[x]), col0 + x, key_mask);
                                qu[cnt * kEpi] = key;
                                cnt += ((decltype(whole)::value || x < lim) && key > thr) ? 1 : 0;
                            }
                            if (__any_sync(kFull, cnt >= 16)) drain();
                        }
                    };
                    if (__all_sync(kFull, lim >= 32)) filter(std::true_type{});
                    else filter(std::false_type{});
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(acc_empty + buf);
        }
        while (__any_sync(kFull, cnt > 0)) drain();
        // group 1 hands its list to group 0, which merges and writes
        static_assert(KMAX * kTileM <= S::kQueueWords, "merge lists fit the queue region");
        tc::named_bar_sync(1, kEpi);               // every queue drained
        if (eg == 1) {
#pragma unroll
            for (int t = 0; t < KMAX; ++t) merge[t * kTileM + r] = L[t];
        }
        tc::named_bar_sync(1, kEpi);
        const int64_t i = row0 + r;
        if (eg == 0 && i < n) {
            uint32_t B[KMAX];
#pragma unroll
            for (int t = 0; t < KMAX; ++t) B[t] = merge[t * kTileM + r];
            merge_sorted<KMAX, KMAX>(L, B);
            int ids[KMAX];
#pragma unroll
            for (int t = 0; t < KMAX; ++t)
                ids[t] = L[t] != 0u ? int(key_mask - (L[t] & key_mask)) : INT_MAX;
            int kr = topk;
            if (kOpts && o.head_k != nullptr) {
                const int32_t hk = __ldg(o.head_k + h);
                kr = min(max(hk, 0), topk);
                if (hk != kr) report_status(status, kStatusInvalidArg);
            }
            apply_budget<KMAX>(ids, kr, int(own), kOpts && o.local != 0);
#pragma unroll
            for (int round = 0; round < KMAX; ++round) {
#pragma unroll
                for (int t = round & 1; t + 1 < KMAX; t += 2) {
                    const int a = ids[t], b = ids[t + 1];
                    ids[t] = min(a, b);
                    ids[t + 1] = max(a, b);
                }
            }
            int32_t *dst = idx + (h * n + i) * topk;
#pragma unroll
            for (int t = 0; t < KMAX; ++t)
                if (t < topk) dst[t] = ids[t] == INT_MAX ? -1 : ids[t];
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// --------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [outer][rows][d] bf16 tensor, box of 64 x box_rows x 1, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int64_t outer, int64_t rows, int d, int box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(rows), cuuint64_t(outer)};
    cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(rows) * d * 2};
    cuuint32_t box[3] = {64, cuuint32_t(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int KMAX>
cudaError_t launch_dk(const CUtensorMap &mq, const CUtensorMap &mh, const CUtensorMap &ml,
                      int64_t bh, int64_t n, int64_t nb, int32_t topk, uint32_t mask,
                      const SelectOpts &o, int32_t *idx, int32_t *status, cudaStream_t st) {
    const int smem = CoarseSmem<D>::kTotal;
    const bool opts = o.head_k != nullptr || o.causal || o.local;
    auto kern = opts ? coarse_topk_tc_kernel<D, KMAX, true> : coarse_topk_tc_kernel<D, KMAX, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(unsigned((n + kTileM - 1) / kTileM), unsigned(bh));
    kern<<<grid, kThreads, smem, st>>>(mq, mh, ml, n, nb, topk, mask, o, idx, status);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const CUtensorMap &mq, const CUtensorMap &mh, const CUtensorMap &ml,
                     int64_t bh, int64_t n, int64_t nb, int32_t topk, uint32_t mask,
                     const SelectOpts &o, int32_t *idx, int32_t *status, cudaStream_t st) {
    if (topk <= 4) return launch_dk<D, 4>(mq, mh, ml, bh, n, nb, topk, mask, o, idx, status, st);
    if (topk <= 8) return launch_dk<D, 8>(mq, mh, ml, bh, n, nb, topk, mask, o, idx, status, st);
    if (topk <= 16) return launch_dk<D, 16>(mq, mh, ml, bh, n, nb, topk, mask, o, idx, status, st);
    return launch_dk<D, 32>(mq, mh, ml, bh, n, nb, topk, mask, o, idx, status, st);
}

}  // namespace

int coarse_tc_key_bits(int64_t nb) {
    int bits = 1;
    while ((int64_t(1) << bits) < nb) ++bits;
    return bits;
}

bool coarse_tc_supported(int64_t nb) { return coarse_tc_key_bits(nb) <= 12; }

cudaError_t launch_coarse_topk_tc(const void *q, const uint16_t *kbar_hi, const uint16_t *kbar_lo,
                                  int64_t bh, int64_t n, int32_t d, int64_t nb, int32_t topk,
                                  const SelectOpts &o, int32_t *idx, int32_t *status,
                                  cudaStream_t st) {
    CUtensorMap mq, mh, ml;
    if (!make_map(&mq, q, bh, n, d, kTileM) || !make_map(&mh, kbar_hi, bh, nb, d, kChunk) ||
        !make_map(&ml, kbar_lo, bh, nb, d, kChunk))
        return cudaErrorInvalidValue;
    const uint32_t mask = (1u << coarse_tc_key_bits(nb)) - 1u;
    if (d == 64) return launch_d<64>(mq, mh, ml, bh, n, nb, topk, mask, o, idx, status, st);
    return launch_d<128>(mq, mh, ml, bh, n, nb, topk, mask, o, idx, status, st);
}

}  // namespace bsa
