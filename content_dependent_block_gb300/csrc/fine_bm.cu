// Stage 2, fine attention, block-major on the tensor cores (page
// "sparse-attention-triton-bench", Stage 2: dense attention over the k*B
// selected tokens; "The Triton kernel": running max m, running sum l and
// accumulator acc merged block by block).
//
// Schedule.  The per-query lists are inverted (invert.cu) so that every
// (head, key block) knows the (query, slot) pairs that selected it.  A work
// item is one key block and up to kItemTiles x 128 of its pairs.  Per item
// the CTA loads K_b and V_b once (TMA, 128-byte swizzle); per tile of 128
// pairs it
//   1. gathers the 128 query rows (cp.async, swizzled by hand),
//   2. S = Q_g . K_b^T            tcgen05 MMA, M = 128, N = B, fp32 in TMEM
//   3. per row (one thread per TMEM lane): m = max s, p = exp2(s - m),
//      l = sum p, P -> shared memory as bf16 (the A operand of step 4)
//   4. O = P . V_b                tcgen05 MMA, M = 128, N = d (V MN-major)
//   5. writes the pair's partial state: o = O / l (bf16) and
//      lse = m + log2 l (fp32, base-2 units of the scaled score)
// and the thread that writes a query's last partial (a per-query counter)
// merges that query's partials in slot order -- the online-softmax merge
// of (m, l, acc) across its blocks -- and writes O.  The merge reads every
// partial in a fixed order, so results do not depend on scheduling.
//
// The grid is persistent (SMs x resident CTAs); items are taken round-robin
// in head-major order so that a head's partials are produced and consumed
// while they are still in L2.  Four 128-thread CTAs share an SM (d = 64),
// which overlaps one CTA's gathers with another's MMAs and exponentials.
#include <cmath>

#include <cudaTypedefs.h>

#include "bsa_device.cuh"
#include "bsa_internal.h"
#include "tc.cuh"

namespace bsa {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 128;
constexpr int kB = 64;                  // key block handled by this kernel

template <int D>
struct BmSmem {
    static constexpr int kSub = D / 64;
    static constexpr int kQBytes = kSub * kTile * 128;   // gathered Q   [128][D]
    static constexpr int kPBytes = kTile * 128;          // P (bf16)     [128][64]
    static constexpr int kKBytes = kSub * kB * 128;      // K_b          [64][D]
    static constexpr int kVBytes = kSub * kB * 128;      // V_b          [64][D]
    static constexpr int kTiles = kQBytes + kPBytes + kKBytes + kVBytes;
    static constexpr int kTotal = kTiles + 1024 + 64;
    static constexpr uint32_t kTmemCols = (kB + D) <= 128 ? 128 : 256;
};

__device__ __forceinline__ int list_valid(const int32_t *row, int32_t k, int64_t nb) {
    int c = 0;
    for (int s = 0; s < k; ++s) {
        const int32_t b = __ldg(row + s);
        c += (b >= 0 && b < nb) ? 1 : 0;
    }
    return c;
}

// Merge the partial states of query row `qrow` (flat h*n + i) into O with
// the whole warp: lane s reads slot s's lse, lane l owns D/32 channels, and
// every partial value of the row is requested before any is used.
template <int D>
__device__ __forceinline__ void merge_query_warp(int64_t qrow, const int32_t *list, int32_t k,
                                                 int64_t nb, int32_t full_valid, int lane,
                                                 const uint16_t *part_o, const float *part_lse,
                                                 uint16_t *out) {
    constexpr int E = D / 32;     // channels per lane: 2 or 4
    bool valid = false;
    if (lane < k) {
        if (full_valid > 0) {
            valid = lane < full_valid;
        } else {
            const int32_t b = __ldg(list + qrow * k + lane);
            valid = b >= 0 && b < nb;
        }
    }
    const float lse = valid ? __ldcg(part_lse + qrow * k + lane) : -INFINITY;
    uint32_t raw[32][E / 2];
#pragma unroll
    for (int s = 0; s < 32; ++s) {
        const bool vs = __shfl_sync(0xffffffffu, valid, s);
        const uint16_t *src = part_o + (qrow * k + s) * D + lane * E;
        if (E == 2) raw[s][0] = vs ? __ldcg(reinterpret_cast<const unsigned int *>(src)) : 0u;
        else {
            const uint2 x = vs ? __ldcg(reinterpret_cast<const uint2 *>(src)) : make_uint2(0u, 0u);
            raw[s][0] = x.x;
            raw[s][E / 2 - 1] = x.y;
        }
    }
    const float M = warp_max(lse);
    const float w = valid ? exp2f(lse - M) : 0.f;
    const float invL = 1.f / warp_sum(w);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int s = 0; s < 32; ++s) {
        const float ws = __shfl_sync(0xffffffffu, w, s);
#pragma unroll
        for (int e2 = 0; e2 < E / 2; ++e2) {
            acc[2 * e2] = fmaf(ws, bf16_low_half(raw[s][e2]), acc[2 * e2]);
            acc[2 * e2 + 1] = fmaf(ws, bf16_high_half(raw[s][e2]), acc[2 * e2 + 1]);
        }
    }
    uint16_t *dst = out + qrow * D + lane * E;
    if (E == 2) {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * invL, acc[1] * invL);
    } else {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc[0] * invL, acc[1] * invL),
                                                     pack_bf16x2(acc[E - 2] * invL, acc[E - 1] * invL));
    }
}

__device__ __forceinline__ int atomic_add_acq_rel(int32_t *p, int32_t v) {
    int32_t old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

template <int D>
__global__ void __launch_bounds__(kThreads) fine_bm_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t *__restrict__ q, const int32_t *__restrict__ list,
    const int32_t *__restrict__ entries, const int32_t *__restrict__ offsets,
    const int2 *__restrict__ items, const int32_t *__restrict__ n_items, int64_t n, int64_t nb,
    int64_t bins_per_head, int32_t k, int32_t full_lists, int32_t item_pairs, float scale_log2,
    uint16_t *__restrict__ part_o, float *__restrict__ part_lse, int32_t *__restrict__ qcount,
    uint16_t *__restrict__ out, int32_t *status) {
    using S = BmSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sP = sQ + S::kQBytes;
    uint8_t *sK = sP + S::kPBytes;
    uint8_t *sV = sK + S::kKBytes;
    uint64_t *bar_kv = reinterpret_cast<uint64_t *>(smem + S::kTiles);
    uint64_t *bar_mma = bar_kv + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_kv + 2);

    const int t = threadIdx.x;
    const int warp = t >> 5;
    if (status != nullptr && *reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout) return;

    if (t == 0) {
        tc::mbar_init(bar_kv, 1);
        tc::mbar_init(bar_mma, 1);
        tc::fence_barrier_init();
        tc::prefetch_tensormap(&tm_k);
        tc::prefetch_tensormap(&tm_v);
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, S::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_s = tmem;                 // S: columns [0, 64)
    const uint32_t tmem_o = tmem + kB;            // O: columns [64, 64 + D)
    const uint32_t lane_off = uint32_t(warp * 32) << 16;

    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kTile, kB);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kTile, D, /*b_mn_major=*/true);
    const uint32_t aq = tc::smem_u32(sQ), ap = tc::smem_u32(sP);
    const uint32_t ak = tc::smem_u32(sK), av = tc::smem_u32(sV);
    const int kvalid_all = int(i64min(k, nb));

    uint32_t kv_phase = 0, mma_phase = 0;
    bool ok = true;
    const int total = *n_items;
    for (int it = blockIdx.x; ok && it < total; it += gridDim.x) {
        const int2 item = items[it];
        const int64_t hb = item.x;                // bin = (head, query range, block)
        const int64_t h = hb / bins_per_head;
        const int64_t b = hb % nb;
        const int32_t cnt = offsets[hb + 1] - offsets[hb];
        const int32_t end = min(cnt, item.y + item_pairs);
        const int32_t *ent = entries + offsets[hb];
        if (t == 0) {
            tc::mbar_arrive_expect_tx(bar_kv, S::kKBytes + S::kVBytes);
#pragma unroll
            for (int sub = 0; sub < S::kSub; ++sub) {
                tc::tma_load_3d(sK + sub * kB * 128, &tm_k, bar_kv, sub * 64, int32_t(b * kB), int32_t(h));
                tc::tma_load_3d(sV + sub * kB * 128, &tm_v, bar_kv, sub * 64, int32_t(b * kB), int32_t(h));
            }
        }
        const int64_t keys_valid = n - b * kB;    // >= 1; < 64 only for a ragged last block
        bool first_tile = true;
        for (int32_t p0 = item.y; ok && p0 < end; p0 += kTile) {
            // 1. gather the tile's query rows
            const int32_t p = p0 + t;
            const bool has = p < end;
            const int32_t pid = has ? __ldg(ent + p) : 0;
            const int64_t qrow = pid / k;
            if (has) {
                const uint16_t *src = q + qrow * D;
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    const int sub = c >> 3, cc = c & 7;
                    tc::cp_async16(sQ + sub * kTile * 128 + t * 128 + ((cc ^ (t & 7)) << 4), src + c * 8);
                }
            }
            tc::cp_async_wait_all();
            tc::fence_proxy_async_smem();
            __syncthreads();
            // 2. S = Q . K_b^T
            if (t == 0) {
                if (first_tile) ok = tc::mbar_wait(bar_kv, kv_phase, status);
                tc::tc_fence_after();
                if (ok) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off_q = uint32_t((kk >> 2) * kTile * 128 + (kk & 3) * 32);
                        const uint32_t off_k = uint32_t((kk >> 2) * kB * 128 + (kk & 3) * 32);
                        tc::mma_bf16(tmem_s, tc::smem_desc_sw128(aq + off_q, 1024),
                                     tc::smem_desc_sw128(ak + off_k, 1024), idesc_s, kk > 0);
                    }
                    tc::mma_commit(bar_mma);
                }
            }
            first_tile = false;
            ok = __syncthreads_and(ok);
            if (!ok) break;
            ok = tc::mbar_wait(bar_mma, mma_phase, status);
            mma_phase ^= 1;
            tc::tc_fence_after();
            // 3. softmax of the row (scores in base-2 units)
            float m2 = -INFINITY, l = 0.f;
            {
                uint32_t sv[2][32];
                tc::tmem_ld32(tmem_s + lane_off, sv[0]);
                tc::tmem_ld32(tmem_s + lane_off + 32, sv[1]);
                tc::tmem_ld_wait();
                float s2[64];
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s2[j] = j < keys_valid ? __uint_as_float(sv[j >> 5][j & 31]) * scale_log2 : -INFINITY;
                    m2 = fmaxf(m2, s2[j]);
                }
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s2[j] = exp2f(s2[j] - m2);
                    l += s2[j];
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = make_uint4(pack_bf16x2(s2[8 * c + 0], s2[8 * c + 1]),
                                               pack_bf16x2(s2[8 * c + 2], s2[8 * c + 3]),
                                               pack_bf16x2(s2[8 * c + 4], s2[8 * c + 5]),
                                               pack_bf16x2(s2[8 * c + 6], s2[8 * c + 7]));
                    *reinterpret_cast<uint4 *>(sP + t * 128 + ((c ^ (t & 7)) << 4)) = v;
                }
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            __syncthreads();
            // 4. O = P . V_b
            if (t == 0 && ok) {
                tc::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kB / 16; ++kk)
                    tc::mma_bf16(tmem_o, tc::smem_desc_sw128(ap + kk * 32, 1024),
                                 tc::smem_desc_sw128_mn(av + kk * 2048, kB * 128, 1024), idesc_o,
                                 kk > 0);
                tc::mma_commit(bar_mma);
            }
            if (ok) ok = tc::mbar_wait(bar_mma, mma_phase, status);
            mma_phase ^= 1;
            tc::tc_fence_after();
            // 5. partial state of the pair, then the last writer merges
            {
                const float inv_l = 1.f / l;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tc::tmem_ld32(tmem_o + lane_off + c0, ov);
                    tc::tmem_ld_wait();
                    if (has) {
                        uint4 *dst = reinterpret_cast<uint4 *>(part_o + int64_t(pid) * D + c0);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(
                                pack_bf16x2(__uint_as_float(ov[8 * v + 0]) * inv_l, __uint_as_float(ov[8 * v + 1]) * inv_l),
                                pack_bf16x2(__uint_as_float(ov[8 * v + 2]) * inv_l, __uint_as_float(ov[8 * v + 3]) * inv_l),
                                pack_bf16x2(__uint_as_float(ov[8 * v + 4]) * inv_l, __uint_as_float(ov[8 * v + 5]) * inv_l),
                                pack_bf16x2(__uint_as_float(ov[8 * v + 6]) * inv_l, __uint_as_float(ov[8 * v + 7]) * inv_l));
                    }
                }
                bool last = false;
                if (has) {
                    part_lse[pid] = m2 + __log2f(l);
                    // release: this pair's partial is visible before the count;
                    // acquire: the last writer sees every other slot's partial
                    const int done = atomic_add_acq_rel(qcount + qrow, 1) + 1;
                    const int need = full_lists ? kvalid_all : list_valid(list + qrow * k, k, nb);
                    last = done == need;
                }
                unsigned todo = __ballot_sync(0xffffffffu, last);
                while (todo != 0u) {
                    const int src_lane = __ffs(todo) - 1;
                    todo &= todo - 1u;
                    const int64_t r = __shfl_sync(0xffffffffu, qrow, src_lane);
                    merge_query_warp<D>(r, list, k, nb, full_lists ? kvalid_all : 0, t & 31, part_o,
                                        part_lse, out);
                }
            }
            tc::tc_fence_before();
            ok = __syncthreads_and(ok);   // keeps the loop conditions uniform
        }
        kv_phase ^= 1;
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, S::kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_rows_map(CUtensorMap *m, const void *base, int64_t bh, int64_t n, int d, int box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(n), cuuint64_t(bh)};
    cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(n) * d * 2};
    cuuint32_t box[3] = {64, cuuint32_t(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const FineBmArgs &a, const CUtensorMap &mk, const CUtensorMap &mv,
                     cudaStream_t st) {
    using S = BmSmem<D>;
    auto kern = fine_bm_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
        return e;
    int dev = 0, sms = 0, smem_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
        return e;
    // resident CTAs per SM: shared memory (+1 KB reserved per CTA) and TMEM
    int per_sm = smem_sm / (S::kTotal + 1024);
    const int tmem_limit = int(512 / S::kTmemCols);
    if (per_sm > tmem_limit) per_sm = tmem_limit;
    if (per_sm < 1) per_sm = 1;
    const int grid = sms * per_sm;
    kern<<<grid, kThreads, S::kTotal, st>>>(mk, mv, a.q, a.list, a.entries, a.offsets, a.items,
                                            a.n_items, a.n, a.nb, a.bins_per_head, a.k,
                                            a.full_lists, a.item_pairs,
                                            a.scale_log2, a.part_o, a.part_lse, a.qcount, a.out,
                                            a.status);
    return cudaGetLastError();
}

}  // namespace

bool fine_bm_supported(int32_t d, int32_t key_block) {
    return (d == 64 || d == 128) && key_block == kB;
}

cudaError_t launch_fine_bm(const FineBmArgs &a, cudaStream_t st) {
    CUtensorMap mk, mv;
    if (!make_rows_map(&mk, a.k_ptr, a.bh, a.n, a.d, kB) || !make_rows_map(&mv, a.v_ptr, a.bh, a.n, a.d, kB))
        return cudaErrorInvalidValue;
    if (a.d == 64) return launch_d<64>(a, mk, mv, st);
    return launch_d<128>(a, mk, mv, st);
}

}  // namespace bsa
