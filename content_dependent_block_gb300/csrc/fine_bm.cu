// Stage 2, fine attention, block-major on the tensor cores (page
// "sparse-attention-triton-bench", Stage 2: dense attention over the k*B
// selected tokens; "The Triton kernel": running max m, running sum l and
// accumulator acc merged block by block).
//
// Schedule.  The per-query lists are inverted (invert.cu) into bins
// (head, query range, key block), each listing the (query, slot) pairs that
// selected the block.  One persistent CTA per SM runs five warp roles that
// hand work to each other through mbarrier rings in shared memory:
//
//   prefetch  (warp 14)     takes fine items (one bin, <= 512 pairs) from a
//                           global queue and stages each item's descriptor
//                           and pair ids in a shared-memory ring
//   producer  (warp 0)      per staged item: loads K_b, V_b by TMA (128-byte
//                           swizzle, double-buffered per item) and gathers the
//                           128 query rows of each tile with TMA gather4 (four
//                           rows per instruction) into a ring of Q stages;
//                           publishes per-tile info
//   MMA       (warp 1)      S[j] = Q . K_b^T (tcgen05, M = 128, N = 64) into
//                           one of two TMEM score buffers, then O[j] = P . V_b
//                           (N = d, V MN-major) into one of two TMEM outputs;
//                           tile g's S is issued before tile g-1's P.V
//   softmax   (warps 2-5)   one thread per row: m = max s, p = exp2(s - m),
//                           l = sum p; P (bf16) to shared memory, (m, l) aside
//   epilogue  (warps 6-9)   reads O, stores the pair's partial state
//                           o = O / l (bf16) and lse = m + log2 l into a ring
//                           of query ranges, counts the range's finished pairs
//   merge     (warps 10-13) takes merge items (256 queries of one range) from a
//                           second queue once the range's pairs are all done
//                           and merges each query's k partial states in slot
//                           order (the online-softmax merge of (m, l, acc))
//
// Partial states of a range live in ring entry (range mod kPartialRing); a
// fine item of range r waits until range r - kPartialRing is merged.  Every
// wait is on work taken from a queue earlier, so the schedule cannot
// deadlock, and every wait is bounded.  Results do not depend on scheduling:
// partial states are per pair and merged in slot order.
#include <cmath>

#include <cudaTypedefs.h>

#include "bsa_device.cuh"
#include "bsa_internal.h"
#include "tc.cuh"

namespace bsa {
namespace {

constexpr int kTile = 128;
constexpr int kB = 64;                   // key block handled by this kernel
constexpr int kNT = 8;                   // tile-info ring
constexpr int kNI = 4;                   // staged fine-item ring
constexpr int kItemMax = 512;            // pairs per fine item (kFineBmItemPairs)
constexpr int kWarps = 15;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpEpi = 6, kWarpMerge = 10, kWarpFetch = 14;
constexpr uint32_t kBarEpi = 1, kBarMerge = 2;
constexpr unsigned kFull = 0xffffffffu;

struct TileInfo {
    int32_t bin, p0, count, item, last, rg, end, pad;
};

// A fine item staged by the prefetcher: descriptor plus all its pair ids.
struct StagedItem {
    int32_t bin, first, end, rg, h, b, valid, pad;
    int32_t pid[kItemMax];
};

template <int D>
struct Cfg {
    static constexpr int kSub = D / 64;
    static constexpr int kNQ = D == 64 ? 4 : 3;            // Q stages
    static constexpr int kQBytes = kSub * kTile * 128;
    static constexpr int kPBytes = kTile * 128;
    static constexpr int kKBytes = kSub * kB * 128;        // K or V of one block
    static constexpr int oQ = 0;
    static constexpr int oP = oQ + kNQ * kQBytes;
    static constexpr int kNKV = D == 64 ? 4 : 2;           // K/V buffers (items in flight)
    static constexpr int oK = oP + 2 * kPBytes;
    static constexpr int oV = oK + kNKV * kKBytes;
    static constexpr int oML = oV + kNKV * kKBytes;        // float2 [kNT][128]
    static constexpr int oPid = oML + kNT * kTile * 8;     // int32  [kNT][128]
    static constexpr int oTi = oPid + kNT * kTile * 4;     // TileInfo [kNT]
    static constexpr int oItem = oTi + kNT * 32;           // StagedItem [kNI]
    static constexpr int oBar = oItem + kNI * int(sizeof(StagedItem));
    enum {
        bQFull = 0,
        bQFree = bQFull + kNQ,
        bKvFull = bQFree + kNQ,
        bKvFree = bKvFull + kNKV,
        bSFull = bKvFree + kNKV,
        bSFree = bSFull + 2,
        bPFull = bSFree + 2,
        bPFree = bPFull + 2,
        bOFull = bPFree + 2,
        bOFree = bOFull + 2,
        bMlFull = bOFree + 2,
        bTiFull = bMlFull + kNT,
        bTiFree = bTiFull + kNT,
        bItFull = bTiFree + kNT,
        bItFree = bItFull + kNI,
        bCount = bItFree + kNI
    };
    static constexpr int oMisc = oBar + bCount * 8;
    static constexpr int kTotal = oMisc + 64 + 1024;
    static constexpr uint32_t kTmemCols = D == 64 ? 256 : 512;
    static constexpr uint32_t cO = 2 * kB;                 // O[j] at cO + j*D; S[j] at j*64
};

__device__ __forceinline__ int32_t ld_acquire(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *p >= target (acquire).  False on timeout, or when
// another wait in the grid already timed out.
__device__ bool wait_counter(const int32_t *p, int32_t target, int32_t *status) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = tc::global_ns();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire(p) >= target) return true;
        if (*reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout) return false;
        if (tc::global_ns() - t0 > tc::kWaitLimitNs) {
            report_status(status, kStatusTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void red_add_release(int32_t *p, int32_t v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge up to four queries per warp: four 8-lane groups, one query each;
// lane gl of a group owns channels [gl*D/8, (gl+1)*D/8).  `base` indexes the
// query's partial slots in the ring; `active` false for an idle group.
template <int D>
__device__ __forceinline__ void merge_group(bool active, int64_t qrow, int64_t base,
                                            const int32_t *list, int32_t k, int64_t nb,
                                            int32_t full_valid, int lane, const uint16_t *part_o,
                                            const float *part_lse, uint16_t *out) {
    constexpr int C = D / 8;                   // channels per lane: 8 or 16
    constexpr int V = C / 8;                   // uint4 per partial row chunk: 1 or 2
    constexpr int CH = D == 64 ? 16 : 8;       // slots per load chunk
    const int gl = lane & 7;
    const int gbase = lane & ~7;
    bool vs[4];
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
    }
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    float M = -INFINITY, L = 0.f;
    float w[4];
#pragma unroll
    for (int c0 = 0; c0 < 32; c0 += CH) {
        if (c0 >= k) break;
        // every load of this chunk (and the slot lse values) in flight at once
        uint4 x[CH][V];
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int s = c0 + u;
            const bool v = __shfl_sync(kFull, vs[s >> 3], gbase | (s & 7));
            const uint4 *src = reinterpret_cast<const uint4 *>(part_o + (base + s) * D + gl * C);
#pragma unroll
            for (int e = 0; e < V; ++e) x[u][e] = v ? __ldcg(src + e) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (c0 == 0) {
            float lse[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) lse[j] = vs[j] ? __ldcg(part_lse + base + gl + 8 * j) : -INFINITY;
            M = fmaxf(fmaxf(lse[0], lse[1]), fmaxf(lse[2], lse[3]));
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[j] = vs[j] ? ex2(lse[j] - M) : 0.f;
                L += w[j];
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) L += __shfl_xor_sync(kFull, L, o);
        }
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int s = c0 + u;
            const float ws = __shfl_sync(kFull, w[s >> 3], gbase | (s & 7));
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
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fine_ws_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const FineBmArgs a) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::oBar);
    TileInfo *ti = reinterpret_cast<TileInfo *>(sm + C::oTi);
    StagedItem *items = reinterpret_cast<StagedItem *>(sm + C::oItem);
    int32_t *pids = reinterpret_cast<int32_t *>(sm + C::oPid);
    float2 *ml = reinterpret_cast<float2 *>(sm + C::oML);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::oMisc);
    int32_t *s_merge = reinterpret_cast<int32_t *>(sm + C::oMisc + 16);   // [2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = a.status;
    if (*reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout) return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNQ; ++i) {
            tc::mbar_init(bars + C::bQFull + i, 1);
            tc::mbar_init(bars + C::bQFree + i, 1);
        }
        for (int i = 0; i < C::kNKV; ++i) {
            tc::mbar_init(bars + C::bKvFull + i, 1);
            tc::mbar_init(bars + C::bKvFree + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bars + C::bSFull + i, 1);
            tc::mbar_init(bars + C::bSFree + i, kTile);
            tc::mbar_init(bars + C::bPFull + i, kTile);
            tc::mbar_init(bars + C::bPFree + i, 1);
            tc::mbar_init(bars + C::bOFull + i, 1);
            tc::mbar_init(bars + C::bOFree + i, kTile);
        }
        for (int i = 0; i < kNT; ++i) tc::mbar_init(bars + C::bMlFull + i, kTile);
        for (int i = 0; i < kNT; ++i) {
            tc::mbar_init(bars + C::bTiFull + i, 32);
            tc::mbar_init(bars + C::bTiFree + i, 1);
        }
        for (int i = 0; i < kNI; ++i) {
            tc::mbar_init(bars + C::bItFull + i, 32);
            tc::mbar_init(bars + C::bItFree + i, 32);
        }
        tc::fence_barrier_init();
        tc::prefetch_tensormap(&tm_q);
        tc::prefetch_tensormap(&tm_k);
        tc::prefetch_tensormap(&tm_v);
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(tmem_slot, C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int32_t k = a.k;
    const int64_t n = a.n, nb = a.nb, range = a.p.range, nranges = a.p.nranges;
    const int64_t kpad = a.p.kpad;
    const int64_t ring_stride = range * kpad;

    if (warp == kWarpFetch) {
        // ----------------------------------------------------- prefetcher
        // dequeues fine items and stages descriptor + pair ids in shared memory
        const int n_fine = *a.w.n_fine;
        for (int u = 0;; ++u) {
            const int slot = u % kNI;
            if (u >= kNI && !tc::mbar_wait(bars + C::bItFree + slot, ((u / kNI) - 1) & 1, status)) break;
            int it = 0;
            if (lane == 0) it = atomicAdd(a.fine_head, 1);
            it = __shfl_sync(kFull, it, 0);
            StagedItem *si = items + slot;
            const bool valid = it < n_fine;
            if (valid) {
                const int2 item = a.w.fine_items[it];
                const int64_t bin = item.x;
                const int32_t off = a.w.offsets[bin];
                const int32_t end = min(a.w.offsets[bin + 1] - off, item.y + a.p.item_pairs);
                const int32_t *ent = a.w.entries + off;
                int32_t v[kItemMax / 32];
#pragma unroll
                for (int e = 0; e < kItemMax / 32; ++e) {
                    const int32_t p = item.y + e * 32 + lane;
                    v[e] = p < end ? __ldg(ent + p) : 0;
                }
#pragma unroll
                for (int e = 0; e < kItemMax / 32; ++e) si->pid[e * 32 + lane] = v[e];
                if (lane == 0) {
                    const int64_t rg = bin / nb;
                    si->bin = int32_t(bin);
                    si->first = item.y;
                    si->end = end;
                    si->rg = int32_t(rg);
                    si->h = int32_t(rg / nranges);
                    si->b = int32_t(bin % nb);
                }
            }
            if (lane == 0) si->valid = valid ? 1 : 0;
            __syncwarp();
            tc::mbar_arrive(bars + C::bItFull + slot);
            if (!valid) break;
        }
    } else if (warp == kWarpProducer) {
        // ------------------------------------------------------- producer
        int g = 0, item_idx = 0;
        bool ok = true;
        for (int u = 0;; ++u) {
            const int islot = u % kNI;
            if (!tc::mbar_wait(bars + C::bItFull + islot, (u / kNI) & 1, status)) ok = false;
            ok = __all_sync(kFull, ok);
            const StagedItem *si = items + islot;
            bool done = !ok || !si->valid;
            int64_t bin = 0, rg = 0, h = 0, b = 0;
            int32_t first = 0, end = 0;
            if (!done) {
                bin = si->bin;
                first = si->first;
                end = si->end;
                rg = si->rg;
                h = si->h;
                b = si->b;
                if (rg >= kPartialRing) {
                    // the ring entry must have been merged by its previous range
                    int got = 1;
                    if (lane == 0)
                        got = wait_counter(a.merge_done + (rg - kPartialRing),
                                           a.w.range_merges[rg - kPartialRing], status);
                    if (!__shfl_sync(kFull, got, 0)) {
                        ok = false;
                        done = true;
                    }
                }
            }
            if (done) {
                const int slot = g % kNT;
                bool w = true;
                if (g >= kNT) w = tc::mbar_wait(bars + C::bTiFree + slot, ((g / kNT) - 1) & 1, status);
                w = __all_sync(kFull, w);
                if (w && lane == 0) ti[slot].end = 1;
                __syncwarp();
                if (w) tc::mbar_arrive(bars + C::bTiFull + slot);
                break;
            }
            const int ib = item_idx % C::kNKV;
            if (item_idx >= C::kNKV) {
                ok = tc::mbar_wait(bars + C::bKvFree + ib, ((item_idx / C::kNKV) - 1) & 1, status);
                ok = __all_sync(kFull, ok);
                if (!ok) {
                    tc::mbar_arrive(bars + C::bItFree + islot);
                    continue;                     // publishes the end marker
                }
            }
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(bars + C::bKvFull + ib, 2 * C::kKBytes);
#pragma unroll
                for (int sub = 0; sub < C::kSub; ++sub) {
                    tc::tma_load_3d(sm + C::oK + ib * C::kKBytes + sub * kB * 128, &tm_k,
                                    bars + C::bKvFull + ib, sub * 64, int32_t(b * kB), int32_t(h));
                    tc::tma_load_3d(sm + C::oV + ib * C::kKBytes + sub * kB * 128, &tm_v,
                                    bars + C::bKvFull + ib, sub * 64, int32_t(b * kB), int32_t(h));
                }
            }
            for (int32_t p0 = first; ok && p0 < end; p0 += kTile) {
                const int s = g % C::kNQ, slot = g % kNT;
                if (g >= C::kNQ) ok = tc::mbar_wait(bars + C::bQFree + s, ((g / C::kNQ) - 1) & 1, status);
                if (ok && g >= kNT) ok = tc::mbar_wait(bars + C::bTiFree + slot, ((g / kNT) - 1) & 1, status);
                ok = __all_sync(kFull, ok);
                if (!ok) break;
                const int cnt = min(kTile, end - p0);
                // lane l gathers rows 4l .. 4l+3 (padding rows repeat row 0)
                int32_t qr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = 4 * lane + e;
                    const int32_t pid = si->pid[p0 - first + (r < cnt ? r : 0)];
                    if (r < cnt) pids[slot * kTile + r] = pid;
                    qr[e] = pid / k;                        // flat query row h*n + i
                }
                if (lane == 0) tc::mbar_arrive_expect_tx(bars + C::bQFull + s, C::kQBytes);
                __syncwarp();
                uint8_t *sQ = sm + C::oQ + s * C::kQBytes;
#pragma unroll
                for (int sub = 0; sub < C::kSub; ++sub)
                    tc::tma_gather4(sQ + sub * kTile * 128 + lane * 4 * 128, &tm_q, bars + C::bQFull + s,
                                    sub * 64, qr[0], qr[1], qr[2], qr[3]);
                if (lane == 0) {
                    TileInfo x;
                    x.bin = int32_t(bin);
                    x.p0 = p0;
                    x.count = cnt;
                    x.item = item_idx;
                    x.last = p0 + kTile >= end;
                    x.rg = int32_t(rg);
                    x.end = 0;
                    x.pad = 0;
                    ti[slot] = x;
                }
                __syncwarp();
                tc::mbar_arrive(bars + C::bTiFull + slot);
                ++g;
            }
            __syncwarp();
            tc::mbar_arrive(bars + C::bItFree + islot);
            ++item_idx;
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA
        // One thread, run as an event loop: issue whichever is ready first,
        // the S of the next tile or the P.V of the oldest tile whose P is in
        // shared memory (both in tile order), so no P.V is ever held back.
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kTile, kB);
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kTile, D, /*b_mn_major=*/true);
            int g1 = 0, g2 = 0;                   // next tile for S, next tile for P.V
            int cur_item = -1, x_item = 0, x_last = 0;
            int t_ib[4] = {0, 0, 0, 0}, t_last[4] = {0, 0, 0, 0};
            bool end_seen = false, have_info = false;
            uint64_t idle_since = 0;
            for (uint32_t spin = 0;; ++spin) {
                bool progressed = false;
                if (g2 < g1) {
                    const int j = g2 & 1;
                    if (tc::mbar_try_wait(bars + C::bPFull + j, (g2 >> 1) & 1) &&
                        (g2 < 2 || tc::mbar_try_wait(bars + C::bOFree + j, ((g2 >> 1) - 1) & 1))) {
                        tc::tc_fence_after();
                        const int ib = t_ib[g2 & 3];
                        const uint32_t ap = tc::smem_u32(sm + C::oP + j * C::kPBytes);
                        const uint32_t av = tc::smem_u32(sm + C::oV + ib * C::kKBytes);
#pragma unroll
                        for (int kk = 0; kk < kB / 16; ++kk)
                            tc::mma_bf16(tmem + C::cO + uint32_t(j * D), tc::smem_desc_sw128(ap + kk * 32, 1024),
                                         tc::smem_desc_sw128_mn(av + kk * 2048, kB * 128, 1024), idesc_o,
                                         kk > 0);
                        tc::mma_commit(bars + C::bOFull + j);
                        tc::mma_commit(bars + C::bPFree + j);
                        if (t_last[g2 & 3]) tc::mma_commit(bars + C::bKvFree + ib);
                        ++g2;
                        progressed = true;
                    }
                }
                if (!end_seen && g1 - g2 < 3) {
                    const int slot = g1 % kNT;
                    if (!have_info && tc::mbar_try_wait(bars + C::bTiFull + slot, (g1 / kNT) & 1)) {
                        const volatile TileInfo *xi = ti + slot;
                        if (xi->end) {
                            end_seen = true;
                        } else {
                            have_info = true;
                            x_item = xi->item;
                            x_last = xi->last;
                        }
                        progressed = true;
                    }
                    if (have_info) {
                        const int s = g1 % C::kNQ, j = g1 & 1, ib = x_item % C::kNKV;
                        bool ready = x_item == cur_item ||
                                     tc::mbar_try_wait(bars + C::bKvFull + ib, (x_item / C::kNKV) & 1);
                        ready = ready && tc::mbar_try_wait(bars + C::bQFull + s, (g1 / C::kNQ) & 1);
                        ready = ready && (g1 < 2 || tc::mbar_try_wait(bars + C::bSFree + j, ((g1 >> 1) - 1) & 1));
                        if (ready) {
                            cur_item = x_item;
                            tc::tc_fence_after();
                            const uint32_t aq = tc::smem_u32(sm + C::oQ + s * C::kQBytes);
                            const uint32_t ak = tc::smem_u32(sm + C::oK + ib * C::kKBytes);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off_q = uint32_t((kk >> 2) * kTile * 128 + (kk & 3) * 32);
                                const uint32_t off_k = uint32_t((kk >> 2) * kB * 128 + (kk & 3) * 32);
                                tc::mma_bf16(tmem + uint32_t(j * kB), tc::smem_desc_sw128(aq + off_q, 1024),
                                             tc::smem_desc_sw128(ak + off_k, 1024), idesc_s, kk > 0);
                            }
                            tc::mma_commit(bars + C::bSFull + j);
                            tc::mma_commit(bars + C::bQFree + s);
                            t_ib[g1 & 3] = ib;
                            t_last[g1 & 3] = x_last;
                            ++g1;
                            have_info = false;
                            progressed = true;
                        }
                    }
                }
                if (end_seen && g2 == g1) break;
                if (progressed) {
                    idle_since = 0;
                } else if ((spin & 63u) == 0) {
                    if (*reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout) break;
                    const uint64_t now = tc::global_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > tc::kWaitLimitNs) {
                        report_status(status, kStatusTimeout);
                        break;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < kWarpEpi) {
        // -------------------------------------------------------- softmax
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        for (int g = 0;; ++g) {
            const int slot = g % kNT, j = g & 1;
            if (!tc::mbar_wait(bars + C::bTiFull + slot, (g / kNT) & 1, status)) break;
            const int32_t end_flag = reinterpret_cast<volatile TileInfo *>(ti + slot)->end;
            if (end_flag) break;
            const int64_t bin = reinterpret_cast<volatile TileInfo *>(ti + slot)->bin;
            if (!tc::mbar_wait(bars + C::bSFull + j, (g >> 1) & 1, status)) break;
            tc::tc_fence_after();
            uint32_t sv[2][32];
            tc::tmem_ld32(tmem + uint32_t(j * kB) + lane_off, sv[0]);
            tc::tmem_ld32(tmem + uint32_t(j * kB + 32) + lane_off, sv[1]);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            tc::mbar_arrive(bars + C::bSFree + j);
            const int64_t keys_valid = n - (bin % nb) * kB;
            float s2[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) s2[c] = __uint_as_float(sv[c >> 5][c & 31]);
            if (keys_valid < 64) {                    // ragged last block only
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c >= keys_valid) s2[c] = -INFINITY;
            }
            float mraw = s2[0];
#pragma unroll
            for (int c = 1; c < 64; ++c) mraw = fmaxf(mraw, s2[c]);
            const float m2 = mraw * a.scale_log2;     // scale > 0 keeps the argmax
            float l = 0.f;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                s2[c] = ex2(fmaf(s2[c], a.scale_log2, -m2));
                l += s2[c];
            }
            // (m, l) live with the tile slot, which the producer reuses only
            // after this tile's epilogue is done
            ml[slot * kTile + row] = make_float2(m2, l);
            tc::mbar_arrive(bars + C::bMlFull + slot);
            if (g >= 2 && !tc::mbar_wait(bars + C::bPFree + j, ((g >> 1) - 1) & 1, status)) break;
            uint8_t *sP = sm + C::oP + j * C::kPBytes;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = make_uint4(pack_bf16x2(s2[8 * c + 0], s2[8 * c + 1]),
                                           pack_bf16x2(s2[8 * c + 2], s2[8 * c + 3]),
                                           pack_bf16x2(s2[8 * c + 4], s2[8 * c + 5]),
                                           pack_bf16x2(s2[8 * c + 6], s2[8 * c + 7]));
                *reinterpret_cast<uint4 *>(sP + row * 128 + ((c ^ (row & 7)) << 4)) = v;
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(bars + C::bPFull + j);
        }
    } else if (warp < kWarpMerge) {
        // ------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int et = (warp - kWarpEpi) * 32 + lane;
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        for (int g = 0;; ++g) {
            const int slot = g % kNT, j = g & 1;
            if (!tc::mbar_wait(bars + C::bTiFull + slot, (g / kNT) & 1, status)) break;
            const int32_t x_end = reinterpret_cast<volatile TileInfo *>(ti + slot)->end;
            if (x_end) break;
            const int32_t x_count = reinterpret_cast<volatile TileInfo *>(ti + slot)->count;
            const int32_t x_rg = reinterpret_cast<volatile TileInfo *>(ti + slot)->rg;
            if (!tc::mbar_wait(bars + C::bOFull + j, (g >> 1) & 1, status)) break;
            if (!tc::mbar_wait(bars + C::bMlFull + slot, (g / kNT) & 1, status)) break;
            tc::tc_fence_after();
            const float2 mlv = ml[slot * kTile + row];
            const bool has = row < x_count;
            int64_t part = 0;
            if (has) {
                const int32_t pid = pids[slot * kTile + row];
                const int64_t qrow = pid / k;
                const int64_t s = pid - qrow * k;
                const int64_t h = x_rg / nranges, rr = x_rg % nranges;
                part = (x_rg % kPartialRing) * ring_stride + (qrow - h * n - rr * range) * kpad + s;
            }
            const float inv_l = 1.f / mlv.y;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tc::tmem_ld32(tmem + C::cO + uint32_t(j * D + c0) + lane_off, ov);
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
            tc::tc_fence_before();
            tc::mbar_arrive(bars + C::bOFree + j);
            if (has) a.part_lse[part] = mlv.x + __log2f(mlv.y);
            // the group's partial stores happen before one release-add
            tc::named_bar_sync(kBarEpi, 128);
            if (et == 0) {
                red_add_release(a.range_done + x_rg, x_count);
                tc::mbar_arrive(bars + C::bTiFree + slot);
            }
        }
    } else {
        // ---------------------------------------------------------- merge
        const int mt = (warp - kWarpMerge) * 32 + lane;
        const int mw = warp - kWarpMerge;
        const int n_merge = *a.w.n_merge;
        const int32_t full_valid = a.full_lists ? int32_t(i64min(k, nb)) : 0;
        for (;;) {
            if (mt == 0) s_merge[0] = atomicAdd(a.merge_head, 1);
            tc::named_bar_sync(kBarMerge, 128);
            const int it = s_merge[0];
            tc::named_bar_sync(kBarMerge, 128);
            if (it >= n_merge) break;
            const int2 item = a.w.merge_items[it];
            const int64_t rg = item.x;
            if (mt == 0) {
                const bool got = wait_counter(a.range_done + rg, a.w.range_total[rg], status);
                __threadfence();
                s_merge[1] = got;
            }
            tc::named_bar_sync(kBarMerge, 128);
            if (!s_merge[1]) break;
            const int64_t h = rg / nranges, rr = rg % nranges;
            const int64_t i_begin = rr * range + item.y;
            const int64_t i_end = i64min(i64min(n, rr * range + range), i_begin + a.p.qm);
            const int64_t slot_base = (rg % kPartialRing) * ring_stride;
            // 16 queries per pass: 4 warps x 4 groups of 8 lanes
            for (int64_t i0 = i_begin; i0 < i_end; i0 += 16) {
                const int64_t i = i0 + mw * 4 + (lane >> 3);
                const bool act = i < i_end;
                const int64_t ic = act ? i : i_begin;
                merge_group<D>(act, h * n + ic, slot_base + (ic - rr * range) * kpad, a.list, k, nb,
                               full_valid, lane, a.part_o, a.part_lse, a.out);
            }
            __threadfence();
            tc::named_bar_sync(kBarMerge, 128);
            if (mt == 0) atomicAdd(a.merge_done + rg, 1);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, C::kTmemCols);
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

// [rows][d] bf16 viewed as 2-D, box 64 x 1 (one row per gathered row).
bool make_gather_map(CUtensorMap *m, const void *base, int64_t rows, int d) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {cuuint64_t(d), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(d) * 2};
    cuuint32_t box[2] = {64, 1};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const FineBmArgs &a, const CUtensorMap &mq, const CUtensorMap &mk,
                     const CUtensorMap &mv, cudaStream_t st) {
    using C = Cfg<D>;
    auto kern = fine_ws_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kTotal);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    kern<<<sms, kThreads, C::kTotal, st>>>(mq, mk, mv, a);   // one CTA per SM
    return cudaGetLastError();
}

}  // namespace

bool fine_bm_supported(int32_t d, int32_t key_block) {
    return (d == 64 || d == 128) && key_block == kB;
}

cudaError_t launch_fine_bm(const FineBmArgs &a, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!make_gather_map(&mq, a.q, a.bh * a.n, a.d) ||
        !make_rows_map(&mk, a.k_ptr, a.bh, a.n, a.d, kB) || !make_rows_map(&mv, a.v_ptr, a.bh, a.n, a.d, kB))
        return cudaErrorInvalidValue;
    if (a.d == 64) return launch_d<64>(a, mq, mk, mv, st);
    return launch_d<128>(a, mq, mk, mv, st);
}

}  // namespace bsa
