// Stage 2, fine attention, block-major on the tensor cores (page
// "sparse-attention-triton-bench", Stage 2: dense attention over the k*B
// selected tokens; "The Triton kernel": running max m, running sum l and
// accumulator acc merged block by block).
//
// Schedule.  The per-query lists are inverted (invert.cu) into bins
// (head, query range, key block), each listing the (query, slot) pairs
// that selected the block.  A persistent grid pulls work items from one
// queue (an atomic counter) in the order the scan kernel laid out:
//   fine items   one bin and up to 512 of its pairs.  The CTA loads K_b and
//                V_b once (TMA, 128-byte swizzle); per tile of 128 pairs it
//                gathers the query rows (cp.async), S = Q_g . K_b^T
//                (tcgen05, M = 128, N = 64, fp32 in TMEM), per row
//                m = max s, p = exp2(s - m), l = sum p, P -> shared memory
//                (bf16), O = P . V_b (tcgen05, N = d), and stores the pair's
//                partial state o = O / l (bf16) and lse = m + log2 l.
//   merge items  256 queries of a range whose fine items are all done: the
//                k partial states of each query are merged in slot order
//                (online-softmax merge of (m, l, acc)) into O, and the
//                merged partial lines are discarded from L2 so they are
//                never written back to memory.
// Merge items of range r sit after the fine items of range r + 1, so every
// wait is on work taken from the queue earlier (no deadlock), and partial
// states live in a ring of kPartialRing ranges (bounded, L2-sized memory).
// Results do not depend on scheduling: partial states are per pair and the
// merge reads them in slot order.
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

__device__ __forceinline__ int32_t ld_acquire(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *p >= target (acquire).  False on timeout, or when
// another CTA already reported one.
__device__ bool wait_counter(const int32_t *p, int32_t target, int32_t *status) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = tc::global_ns();
    for (;;) {
        __nanosleep(128);
        if (ld_acquire(p) >= target) return true;
        if (*reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout) return false;
        if (tc::global_ns() - t0 > tc::kWaitLimitNs) {
            report_status(status, kStatusTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void discard_l2_line(const void *p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge up to four queries per warp: the warp splits into four 8-lane
// groups, one query each; lane gl of a group owns channels [gl*D/8,
// (gl+1)*D/8).  Slot lse values are spread over the group's lanes; every
// partial row of a chunk of slots is requested before any is used.
// `qrow` / `base` are the group's query row (flat h*n + i) and the index of
// its k partial slots in the ring; `active` false for a group with no query.
template <int D>
__device__ __forceinline__ void merge_group(bool active, int64_t qrow, int64_t base,
                                            const int32_t *list, int32_t k, int64_t nb,
                                            int32_t full_valid, int lane, uint16_t *part_o,
                                            const float *part_lse, uint16_t *out) {
    constexpr int C = D / 8;                   // channels per lane: 8 or 16
    constexpr int V = C / 8;                   // uint4 per partial row chunk: 1 or 2
    constexpr int CH = D == 64 ? 16 : 8;       // slots per load chunk
    const int gl = lane & 7;
    const int gbase = lane & ~7;
    bool vs[4];
    float lse[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int s = gl + 8 * j;
        bool v = active && s < k;
        if (v && full_valid == 0) {
            const int32_t b = __ldg(list + qrow * k + s);
            v = b >= 0 && b < nb;
        } else if (v) {
            v = s < full_valid;
        }
        vs[j] = v;
        lse[j] = v ? __ldcg(part_lse + base + s) : -INFINITY;
    }
    float M = fmaxf(fmaxf(lse[0], lse[1]), fmaxf(lse[2], lse[3]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float w[4], L = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        w[j] = vs[j] ? ex2(lse[j] - M) : 0.f;
        L += w[j];
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
#pragma unroll
    for (int c0 = 0; c0 < 32; c0 += CH) {
        if (c0 >= k) break;
        uint4 x[CH][V];
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int s = c0 + u;
            const bool v = __shfl_sync(0xffffffffu, vs[s >> 3], gbase | (s & 7));
            const uint4 *src = reinterpret_cast<const uint4 *>(part_o + (base + s) * D + gl * C);
#pragma unroll
            for (int e = 0; e < V; ++e) x[u][e] = v ? __ldcg(src + e) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int s = c0 + u;
            const float ws = __shfl_sync(0xffffffffu, w[s >> 3], gbase | (s & 7));
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const uint32_t xw[4] = {x[u][e].x, x[u][e].y, x[u][e].z, x[u][e].w};
#pragma unroll
                for (int h2 = 0; h2 < 4; ++h2) {
                    acc[8 * e + 2 * h2] = fmaf(ws, bf16_low_half(xw[h2]), acc[8 * e + 2 * h2]);
                    acc[8 * e + 2 * h2 + 1] = fmaf(ws, bf16_high_half(xw[h2]), acc[8 * e + 2 * h2 + 1]);
                }
            }
        }
    }
    if (!active || L == 0.f) return;           // nothing listed: O stays 0
    const float invL = 1.f / L;
    uint4 *dst = reinterpret_cast<uint4 *>(out + qrow * D + gl * C);
#pragma unroll
    for (int e = 0; e < V; ++e)
        dst[e] = make_uint4(pack_bf16x2(acc[8 * e + 0] * invL, acc[8 * e + 1] * invL),
                            pack_bf16x2(acc[8 * e + 2] * invL, acc[8 * e + 3] * invL),
                            pack_bf16x2(acc[8 * e + 4] * invL, acc[8 * e + 5] * invL),
                            pack_bf16x2(acc[8 * e + 6] * invL, acc[8 * e + 7] * invL));
    // the merged partial rows are dead: drop them from L2 without write-back
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (vs[j]) {
#pragma unroll
            for (int line = 0; line < D * 2 / 128; ++line)
                discard_l2_line(part_o + (base + gl + 8 * j) * D + line * 64);
        }
}

template <int D>
__global__ void __launch_bounds__(kThreads, D == 64 ? 4 : 2) fine_bm_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const FineBmArgs a) {
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
    int32_t *s_item = reinterpret_cast<int32_t *>(bar_kv + 3);    // [1]
    int32_t *s_ok = s_item + 1;                                     // [1]

    const int t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31;
    int32_t *status = a.status;
    if (*reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout) return;

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
    const int32_t k = a.k;
    const int64_t n = a.n, nb = a.nb, range = a.p.range, nranges = a.p.nranges;
    const int32_t full_valid = a.full_lists ? int32_t(i64min(k, nb)) : 0;
    const int64_t ring_stride = range * k;       // partial slots per ring entry
    const int total = *a.w.n_items;

    uint32_t kv_phase = 0, mma_phase = 0;
    bool ok = true;
    for (;;) {
        if (t == 0) *s_item = atomicAdd(a.queue_head, 1);
        __syncthreads();
        const int it = *s_item;
        __syncthreads();                          // s_item may be rewritten below
        if (it >= total || !ok) break;
        const int2 item = a.w.items[it];

        if (item.x < 0) {
            // -------------------------------------------------- merge item
            const int64_t rg = -int64_t(item.x) - 1;
            const int64_t h = rg / nranges, rr = rg % nranges;
            if (t == 0) {
                const bool got = wait_counter(a.range_done + rg, a.w.range_total[rg], status);
                __threadfence();
                *s_ok = got;
            }
            __syncthreads();
            ok = *s_ok != 0;
            if (ok) {
                const int64_t i_begin = rr * range + item.y;
                const int64_t i_end = i64min(i64min(n, rr * range + range), i_begin + a.p.qm);
                const int64_t slot_base = (rg % kPartialRing) * ring_stride;
                // 16 queries per pass: 4 warps x 4 groups of 8 lanes
                for (int64_t i0 = i_begin; i0 < i_end; i0 += 16) {
                    const int64_t i = i0 + warp * 4 + (lane >> 3);
                    const bool act = i < i_end;
                    const int64_t ic = act ? i : i_begin;
                    merge_group<D>(act, h * n + ic, slot_base + (ic - rr * range) * k, a.list, k,
                                   nb, full_valid, lane, a.part_o, a.part_lse, a.out);
                }
            }
            __threadfence();
            __syncthreads();
            if (t == 0 && ok) atomicAdd(a.merge_done + rg, 1);
            continue;
        }

        // ------------------------------------------------------ fine item
        const int64_t bin = item.x;
        const int64_t rg = bin / nb;              // range = head * nranges + r
        const int64_t h = rg / nranges, rr = rg % nranges;
        const int64_t b = bin % nb;
        const int32_t *ent = a.w.entries + a.w.offsets[bin];
        const int32_t cnt = a.w.offsets[bin + 1] - a.w.offsets[bin];
        const int32_t end = min(cnt, item.y + a.p.item_pairs);
        const int64_t slot_base = (rg % kPartialRing) * ring_stride;
        if (t == 0) {
            bool got = true;
            // the ring entry must have been merged by its previous range
            if (rg >= kPartialRing)
                got = wait_counter(a.merge_done + (rg - kPartialRing),
                                   a.w.range_merges[rg - kPartialRing], status);
            *s_ok = got;
            if (got) {
                tc::mbar_arrive_expect_tx(bar_kv, S::kKBytes + S::kVBytes);
#pragma unroll
                for (int sub = 0; sub < S::kSub; ++sub) {
                    tc::tma_load_3d(sK + sub * kB * 128, &tm_k, bar_kv, sub * 64, int32_t(b * kB),
                                    int32_t(h));
                    tc::tma_load_3d(sV + sub * kB * 128, &tm_v, bar_kv, sub * 64, int32_t(b * kB),
                                    int32_t(h));
                }
            }
        }
        __syncthreads();
        ok = *s_ok != 0;
        if (!ok) break;
        const int64_t keys_valid = n - b * kB;    // >= 1; < 64 only for a ragged last block
        bool first_tile = true;
        for (int32_t p0 = item.y; ok && p0 < end; p0 += kTile) {
            // 1. gather the tile's query rows
            const int32_t p = p0 + t;
            const bool has = p < end;
            const int32_t pid = has ? __ldg(ent + p) : 0;
            const int64_t qrow = pid / k;                       // h * n + i
            const int64_t slot = pid - qrow * k;
            const int64_t part = slot_base + (qrow - h * n - rr * range) * k + slot;
            if (has) {
                const uint16_t *src = a.q + qrow * D;
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
                for (int j = 0; j < 64; ++j) s2[j] = __uint_as_float(sv[j >> 5][j & 31]);
                if (keys_valid < 64) {                    // ragged last block only
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        if (j >= keys_valid) s2[j] = -INFINITY;
                }
                float mraw = s2[0];
#pragma unroll
                for (int j = 1; j < 64; ++j) mraw = fmaxf(mraw, s2[j]);
                m2 = mraw * a.scale_log2;                 // scale > 0 keeps the argmax
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s2[j] = ex2(fmaf(s2[j], a.scale_log2, -m2));
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
            // 5. the pair's partial state
            const float inv_l = 1.f / l;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tc::tmem_ld32(tmem_o + lane_off + c0, ov);
                tc::tmem_ld_wait();
                if (has) {
                    uint4 *dst = reinterpret_cast<uint4 *>(a.part_o + part * D + c0);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(
                            pack_bf16x2(__uint_as_float(ov[8 * v + 0]) * inv_l, __uint_as_float(ov[8 * v + 1]) * inv_l),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 2]) * inv_l, __uint_as_float(ov[8 * v + 3]) * inv_l),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 4]) * inv_l, __uint_as_float(ov[8 * v + 5]) * inv_l),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 6]) * inv_l, __uint_as_float(ov[8 * v + 7]) * inv_l));
                }
            }
            if (has) a.part_lse[part] = m2 + __log2f(l);
            tc::tc_fence_before();
            ok = __syncthreads_and(ok);   // keeps the loop conditions uniform
        }
        kv_phase ^= 1;
        // publish: this item's partial states are written
        __threadfence();
        __syncthreads();
        if (t == 0 && ok) atomicAdd(a.range_done + rg, end - item.y);
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
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    // resident CTAs per SM: shared memory (+1 KB reserved per CTA), TMEM and
    // registers (allocated per warp in units of 256)
    int per_sm = smem_sm / (S::kTotal + 1024);
    const int tmem_limit = int(512 / S::kTmemCols);
    const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;
    const int reg_limit = 65536 / (warp_regs * (kThreads / 32));
    if (per_sm > tmem_limit) per_sm = tmem_limit;
    if (per_sm > reg_limit) per_sm = reg_limit;
    if (per_sm < 1) per_sm = 1;
    kern<<<sms * per_sm, kThreads, S::kTotal, st>>>(mk, mv, a);
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
