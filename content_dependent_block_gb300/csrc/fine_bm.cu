// Stage 2, fine attention, block-major on the tensor cores (page
// "sparse-attention-triton-bench", Stage 2: dense attention over the k*B
// selected tokens; "The Triton kernel": running max m, running sum l and
// accumulator acc merged block by block).
//
// Schedule.  The per-query lists are inverted (invert.cu) into bins
// (head, query range, key block), each listing the (query, slot) pairs that
// selected the block.  One persistent CTA per SM runs these warp roles,
// handing work over mbarriers in shared memory:
//
//   prefetch  (warp 12)     takes fine items (one bin, <= 512 pairs) from a
//                           global queue (claiming the next while it stages
//                           the current one), stages each item's descriptor and
//                           pair ids in a shared-memory ring and starts the
//                           TMA loads of its K_b and V_b (128-byte swizzle,
//                           one buffer per item in flight)
//   gather    (warps 8-11)  per tile of 128 pairs of a staged item, 128
//                           threads copy the query rows with cp.async
//                           straight into the swizzled operand layout; the
//                           hardware arrives on the stage's barrier when the
//                           copies land (no thread waits for them)
//   owners    (warps 0-3,   fine items alternate between the two owner
//              4-7)         warpgroups, and a group runs each tile of its
//                           items from start to end: its first warp issues
//                           S = Q . K_b^T (tcgen05, M = 128, N = 64) into the
//                           group's TMEM columns; one thread per pair row
//                           turns its row into P (bf16, back into TMEM) and
//                           (m, l); the first warp issues O = P . V_b (A = P
//                           from TMEM, N = d, V MN-major); every thread stores
//                           its pair's unnormalised O (bf16) and (m, l) into
//                           a ring of query ranges.  One group's softmax or
//                           stores run while the other's MMAs do.  One
//                           thread of the group counts finished pairs per
//                           range, up to four tiles under one GPU-scope fence
//   merge     (warps 13-15) each takes merge items (32 queries of one range)
//                           from a second queue once the range's pairs are all
//                           done, pulls the queries' partial states into
//                           shared-memory stages with bulk copies and merges
//                           each query's k states in slot order (the
//                           online-softmax merge of (m, l, acc)); the valid
//                           slots come from the inversion's per-query masks
//                           (padded lists); at d = 128 one query per warp
//
// Partial states of a range live in ring entry (range mod R), R the ring
// depth (4, 8 or 16 ranges: as many as fit about 72 MB of partial states); a
// fine item of range r waits until range r - R is merged.  Every
// wait is on work taken from a queue earlier or on this CTA's own progress,
// and a group counts its finished pairs before it waits for a tile that may
// depend on other CTAs, so the schedule cannot deadlock; every wait is
// bounded.  Results do not depend on scheduling: a row's arithmetic does not
// depend on the other rows of its tile, and partial states are per pair and
// merged in slot order.
#include <cmath>
#include <type_traits>

#include <cudaTypedefs.h>

#include "bsa_device.cuh"
#include "bsa_internal.h"
#include "tc.cuh"

namespace bsa {
namespace {

constexpr int kTile = 128;
constexpr int kB = 64;                   // key block handled by this kernel
constexpr int kNTW = 4;                  // tile-info ring of each owner warpgroup
constexpr int kNI = 2;                   // staged fine-item ring
constexpr int kItemMax = 512;            // pairs per fine item (kFineBmItemPairs)
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
// Warp w runs on SM sub-partition w % 4, and a warp reaches only the TMEM lane
// quadrant w % 4.  Two owner warpgroups (warps 0-3 and 4-7) each run whole
// tiles; the other roles spread over the four sub-partitions:
//   0-3, 4-7   owner warpgroups (fine items alternate between them)
//   8-11       gather
//   12         prefetch
//   13-15      merge
constexpr int kWarpFetch = 12;
__device__ __forceinline__ int gather_index(int w) { return w >= 8 && w < 12 ? w - 8 : -1; }
__device__ __forceinline__ int merge_index(int w) { return w >= 13 ? w - 13 : -1; }
constexpr int kGather = 128;             // gather threads (warps 8-11)
constexpr int kMergeWarps = 3;
constexpr unsigned kFull = 0xffffffffu;

// Per-tile constants, computed once by the gather group: keys in the block
// (kv < 64 only for a ragged last block), flat row of the range's first
// query (qbase), the range's offset in the partial-state ring (roff), the
// range's first query index (ibase) and the block's first key (j0).
struct TileInfo {
    int32_t bin, p0, count, item, last, rg, end, kv, qbase, roff, ibase, j0, g;
};

// A fine item staged by the prefetcher: descriptor plus all its pair ids
// ((flat query row << 5) | slot).
struct StagedItem {
    int32_t bin, first, end, rg, h, b, valid, kv, qbase, roff, ibase, j0;
    int32_t pid[kItemMax];
};

template <int D>
struct Cfg {
    static constexpr int kSub = D / 64;
    static constexpr int kNQ = D == 64 ? 3 : 2;            // Q stages
    static constexpr int kNKV = D == 64 ? 3 : 2;           // K/V buffers (items in flight)
    static constexpr int kMS = 2;                          // merge stages per merge warp
    // one merge stage: >= 4 queries at d = 64, >= 1 at d = 128 (k <= 32)
    static constexpr int kStageBytes = D == 64 ? 17408 : 8704;
    static constexpr int kQBytes = kSub * kTile * 128;
    static constexpr int kKBytes = kSub * kB * 128;        // K or V of one block
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + kNQ * kQBytes;
    static constexpr int oV = oK + kNKV * kKBytes;
    static constexpr int oMs = oV + kNKV * kKBytes;        // merge stages
    static constexpr int oEpi = oMs + kMergeWarps * kMS * kStageBytes;  // 8 owner warps x 2 KB
    static constexpr int oPid = oEpi + 8 * 2048;           // int32  [2][kNTW][128]
    static constexpr int oTi = oPid + 2 * kNTW * kTile * 4;     // TileInfo [2][kNTW]
    static constexpr int oItem = oTi + 2 * kNTW * int(sizeof(TileInfo));   // StagedItem [kNI]
    static constexpr int oBar = oItem + kNI * int(sizeof(StagedItem));
    enum {
        bQFull = 0,
        bQFree = bQFull + kNQ,
        bKvFull = bQFree + kNQ,
        bKvFree = bKvFull + kNKV,
        bTiFull = bKvFree + kNKV,          // [2][kNTW]
        bTiFree = bTiFull + 2 * kNTW,      // [2][kNTW]
        bSDone = bTiFree + 2 * kNTW,       // [2]
        bODone = bSDone + 2,               // [2]
        bItFull = bODone + 2,
        bItFree = bItFull + kNI,
        bMsFull = bItFree + kNI,
        bCount = bMsFull + kMergeWarps * kMS
    };
    static constexpr int oMisc = oBar + bCount * 8;
    static constexpr int kTotal = oMisc + 64 + 1024;
    static constexpr uint32_t kTmemCols = 512;
    // each owner warpgroup: S (64 columns), P (bf16 pairs, 32), O (D)
    static constexpr uint32_t kWgCols = 64 + 32 + D;
    static_assert(2 * kWgCols <= kTmemCols, "tensor memory");
};
static_assert(Cfg<64>::kTotal <= 227 * 1024, "shared memory (d = 64)");
static_assert(Cfg<128>::kTotal <= 227 * 1024, "shared memory (d = 128)");

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void red_add_release(int32_t *p, int32_t v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge one query's partial states from a shared-memory stage.  Slot s
// holds the unnormalised output O_s = sum_j 2^(s_j - m_s) v_j of its block
// (bf16) and (m_s, l_s); the query's output is sum_s w_s O_s / sum_s w_s l_s
// with w_s = 2^(m_s - M), M the largest m_s (the online-softmax merge of
// (m, l, acc)).  The query is owned by a group of LPQ = D/16 lanes; lane gl
// owns channels [16 gl, 16 gl + 16), read as two 16-byte chunks per slot.
// `po` points at this lane's channels of slot 0 (slots D channels apart),
// `pml` at the query's (m, l) pairs, `vm` has bit s set for every listed
// slot s.  Slot s's (m, l) is read by lane s mod LPQ and the weights are
// shared by shuffles.  Neighbouring queries read their two chunks in
// opposite order, so that a quarter warp touches all 32 banks once.  The
// slot loop is rolled (four slots per trip) to keep the code small.  Returns
// false when nothing is listed; else acc holds the merged channels and lse
// the query's log2-sum-exp, M + log2 sum_s w_s l_s.  kOpts:
// a listed slot may hold a partial that admitted no key (m = -inf, under the
// causal mask); it weighs 0.
template <int D, bool kOpts>
__device__ __forceinline__ bool merge_query(const uint16_t *po, const float *pml, uint32_t vm, int k,
                                            int lane, float (&acc)[16], float &lse) {
    constexpr int LPQ = D / 16;
    constexpr int SPL = 32 / LPQ;              // slots per lane (k <= 32)
    const int gl = lane % LPQ, gbase = lane - gl;
    const int c0 = (lane / LPQ) & 1;           // chunk read first
    float w[SPL], lv[SPL];
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < SPL; ++t) {
        const int s = gl + LPQ * t;
        const bool listed = ((vm >> s) & 1u) != 0;
        w[t] = listed ? pml[2 * s] : -INFINITY;
        lv[t] = listed ? pml[2 * s + 1] : 0.f;
        M = fmaxf(M, w[t]);
    }
#pragma unroll
    for (int o = 1; o < LPQ; o <<= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float L = 0.f;
#pragma unroll
    for (int t = 0; t < SPL; ++t) {
        const int s = gl + LPQ * t;
        // unlisted slots hold -inf, and so does a partial that admitted no key
        const bool use = kOpts ? w[t] > -INFINITY : ((vm >> s) & 1u) != 0;
        w[t] = use ? ex2(w[t] - M) : 0.f;
        L += w[t] * lv[t];
    }
#pragma unroll
    for (int o = 1; o < LPQ; o <<= 1) L += __shfl_xor_sync(kFull, L, o);
    float a0[8], a1[8];                        // chunk c0, chunk 1 - c0
#pragma unroll
    for (int c = 0; c < 8; ++c) a0[c] = a1[c] = 0.f;
#pragma unroll 1
    for (int s0 = 0; s0 < k; s0 += 4) {
        const int u0 = s0 % LPQ;               // w[0] holds slots gl + s0 - u0 .. of the group
        float ws[4];
        uint4 x[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            ws[u] = __shfl_sync(kFull, w[0], gbase + u0 + u);
            const uint16_t *src = po + (s0 + u) * D;
            x[u][0] = ws[u] != 0.f ? *reinterpret_cast<const uint4 *>(src + c0 * 8) : make_uint4(0u, 0u, 0u, 0u);
            x[u][1] = ws[u] != 0.f ? *reinterpret_cast<const uint4 *>(src + (1 - c0) * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t xa[4] = {x[u][0].x, x[u][0].y, x[u][0].z, x[u][0].w};
            const uint32_t xb[4] = {x[u][1].x, x[u][1].y, x[u][1].z, x[u][1].w};
#pragma unroll
            for (int h2 = 0; h2 < 4; ++h2) {
                a0[2 * h2] = fmaf(ws[u], bf16_low_half(xa[h2]), a0[2 * h2]);
                a0[2 * h2 + 1] = fmaf(ws[u], bf16_high_half(xa[h2]), a0[2 * h2 + 1]);
                a1[2 * h2] = fmaf(ws[u], bf16_low_half(xb[h2]), a1[2 * h2]);
                a1[2 * h2 + 1] = fmaf(ws[u], bf16_high_half(xb[h2]), a1[2 * h2 + 1]);
            }
        }
        if (u0 + 4 == LPQ) {                   // this lane's next slot group
#pragma unroll
            for (int t = 0; t + 1 < SPL; ++t) w[t] = w[t + 1];
        }
    }
    lse = L > 0.f ? M + __log2f(L) : -INFINITY;
    if (L == 0.f) return false;
    const float invL = 1.f / L;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        acc[c] = (c0 == 0 ? a0[c] : a1[c]) * invL;
        acc[8 + c] = (c0 == 0 ? a1[c] : a0[c]) * invL;
    }
    return true;
}

// The same merge at d = 128, one query per warp: lane l owns channels
// [4 l, 4 l + 4) (one 8-byte chunk per slot; a slot's row is 256 contiguous
// bytes, so the lanes read it without bank conflicts) and slot l's (m, l).
// A stage of such queries is small, so that two fit per merge warp.  The
// weights and chunks of eight slots are fetched before their FMAs (the loop
// is latency-bound: one shuffle and one shared load per slot).
template <bool kOpts>
__device__ __forceinline__ bool merge_query_w(const uint16_t *po, const float *pml, uint32_t vm, int k,
                                              int lane, float (&acc)[4], float &lse) {
    const bool listed = ((vm >> lane) & 1u) != 0;
    const float m = listed ? pml[2 * lane] : -INFINITY;
    const float lv = listed ? pml[2 * lane + 1] : 0.f;
    const float M = warp_max(m);
    // unlisted slots hold -inf, and so does a partial that admitted no key
    const bool use = kOpts ? m > -INFINITY : listed;
    const float w = use ? ex2(m - M) : 0.f;
    const float L = warp_sum(w * lv);
    float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int s0 = 0; s0 < k; s0 += 8) {
        float ws[8];
        uint2 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            ws[u] = __shfl_sync(kFull, w, (s0 + u) & 31);
            ws[u] = s0 + u < k ? ws[u] : 0.f;
            x[u] = ws[u] != 0.f ? *reinterpret_cast<const uint2 *>(po + (s0 + u) * 128) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            a4[0] = fmaf(ws[u], bf16_low_half(x[u].x), a4[0]);
            a4[1] = fmaf(ws[u], bf16_high_half(x[u].x), a4[1]);
            a4[2] = fmaf(ws[u], bf16_low_half(x[u].y), a4[2]);
            a4[3] = fmaf(ws[u], bf16_high_half(x[u].y), a4[3]);
        }
    }
    lse = L > 0.f ? M + __log2f(L) : -INFINITY;
    if (L == 0.f) return false;
    const float invL = 1.f / L;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = a4[c] * invL;
    return true;
}

// kOpts: the causal key limit (a.causal) and selection-derived slot masks
// (a.sel_lists) may be in use; a separate instance, so that the plain kernel
// carries none of their code.
template <int D, bool kOpts>
__global__ void __launch_bounds__(kThreads, 1) fine_ws_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const FineBmArgs a) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = tc::align_smem_1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::oBar);
    TileInfo *ti = reinterpret_cast<TileInfo *>(sm + C::oTi);
    StagedItem *items = reinterpret_cast<StagedItem *>(sm + C::oItem);
    int32_t *pids = reinterpret_cast<int32_t *>(sm + C::oPid);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::oMisc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = a.status;
    // A wait elsewhere already ran out: the whole CTA leaves together.
    if (__syncthreads_or(*reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout)) return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNQ; ++i) {
            tc::mbar_init(bars + C::bQFull + i, kGather);
            tc::mbar_init(bars + C::bQFree + i, 1);
        }
        for (int i = 0; i < C::kNKV; ++i) {
            tc::mbar_init(bars + C::bKvFull + i, 1);
            tc::mbar_init(bars + C::bKvFree + i, 1);
        }
        for (int i = 0; i < 2 * kNTW; ++i) {
            tc::mbar_init(bars + C::bTiFull + i, kGather);
            tc::mbar_init(bars + C::bTiFree + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bars + C::bSDone + i, 1);
            tc::mbar_init(bars + C::bODone + i, 1);
        }
        for (int i = 0; i < kNI; ++i) {
            tc::mbar_init(bars + C::bItFull + i, 32);
            tc::mbar_init(bars + C::bItFree + i, kGather);
        }
        for (int i = 0; i < kMergeWarps * C::kMS; ++i) tc::mbar_init(bars + C::bMsFull + i, 1);
        tc::fence_barrier_init();
        tc::prefetch_tensormap(&tm_k);
        tc::prefetch_tensormap(&tm_v);
    }
    if (warp == 0) {
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
    const int32_t ring = a.p.ring, ring_mask = ring - 1;   // a power of two

    if (warp == kWarpFetch) {
        // ----------------------------------------------------- prefetcher
        // dequeues fine items and stages descriptor + pair ids in shared memory
        const int n_fine = *a.w.n_fine;
        // the next item is claimed, and its descriptor loaded, while the
        // current one is staged (claims stay in queue order, and every CTA
        // stages its items in the order it claimed them)
        int it = 0;
        if (lane == 0) it = atomicAdd(a.fine_head, 1);
        it = __shfl_sync(kFull, it, 0);
        int2 item = make_int2(0, 0);
        int32_t off = 0, off1 = 0;
        if (it < n_fine) {
            item = a.w.fine_items[it];
            off = a.w.offsets[item.x];
            off1 = a.w.offsets[item.x + 1];
        }
        for (int u = 0;; ++u) {
            const int slot = u % kNI;
            const bool valid = it < n_fine;
            int it_next = n_fine;
            if (valid && lane == 0) it_next = atomicAdd(a.fine_head, 1);
            if (u >= kNI && !tc::mbar_wait(bars + C::bItFree + slot, ((u / kNI) - 1) & 1, status)) break;
            StagedItem *si = items + slot;
            if (valid) {
                const int64_t bin = item.x;
                const int32_t end = min(off1 - off, item.y + a.p.item_pairs);
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
                    const int64_t rg = bin / nb, b = bin - rg * nb;
                    const int64_t h = rg / nranges, rr = rg - h * nranges;
                    si->bin = int32_t(bin);
                    si->first = item.y;
                    si->end = end;
                    si->rg = int32_t(rg);
                    si->h = int32_t(h);
                    si->b = int32_t(b);
                    si->kv = int32_t(i64min(kB, n - b * kB));
                    si->qbase = int32_t(h * n + rr * range);
                    si->roff = int32_t((int32_t(rg) & ring_mask) * ring_stride);
                    si->ibase = int32_t(rr * range);
                    si->j0 = int32_t(b * kB);
                }
            }
            if (lane == 0) si->valid = valid ? 1 : 0;
            if (valid) {
                // K_b and V_b into the item's buffer once the item three back is done
                // with it (u counts valid items, as the gather's and owners' do)
                const int ib = u % C::kNKV;
                bool free_ok = true;
                if (u >= C::kNKV)
                    free_ok = __all_sync(kFull, tc::mbar_wait(bars + C::bKvFree + ib,
                                                              ((u / C::kNKV) - 1) & 1, status));
                if (!free_ok) {
                    if (lane == 0) si->valid = 0;
                    __syncwarp();
                    tc::mbar_arrive(bars + C::bItFull + slot);
                    break;
                }
                if (lane == 0) {
                    const int32_t h = si->h, b = si->b;
                    tc::mbar_arrive_expect_tx(bars + C::bKvFull + ib, 2 * C::kKBytes);
#pragma unroll
                    for (int sub = 0; sub < C::kSub; ++sub) {
                        tc::tma_load_3d(sm + C::oK + ib * C::kKBytes + sub * kB * 128, &tm_k,
                                        bars + C::bKvFull + ib, sub * 64, b * kB, h);
                        tc::tma_load_3d(sm + C::oV + ib * C::kKBytes + sub * kB * 128, &tm_v,
                                        bars + C::bKvFull + ib, sub * 64, b * kB, h);
                    }
                }
            }
            __syncwarp();
            tc::mbar_arrive(bars + C::bItFull + slot);
            if (!valid) break;
            it = __shfl_sync(kFull, it_next, 0);
            if (it < n_fine) {
                item = a.w.fine_items[it];
                off = a.w.offsets[item.x];
                off1 = a.w.offsets[item.x + 1];
            }
        }
    } else if (gather_index(warp) >= 0) {
        // --------------------------------------------------------- gather
        // Thread gt owns pair row gt of each tile (its pid and query row);
        // for the copies, lane l of warp gw moves 16-byte chunk (l & 7) of
        // rows gw*32 + 4*i + (l >> 3), i < 8, taking the query row from the
        // owning lane.  Each thread then arrives on the stage's barrier
        // asynchronously: the arrival happens when its copies have landed,
        // so a tile's Q rows are ready as soon as they are in shared memory
        // and the gather never waits for its own copies.  (The K and V of an
        // item are loaded by the prefetcher when it stages the item.)
        const int gw = gather_index(warp), gt = gw * 32 + lane;
        const int chunk = lane & 7, rsub = lane >> 3;
        int g = 0, item_idx = 0;
        int gx[2] = {0, 0};                      // tiles handed to each owner warpgroup
        bool ok = true;
        auto wait = [&](uint64_t *bar, uint32_t par) -> bool {
            return __all_sync(kFull, tc::mbar_wait(bar, par, status));
        };
        for (int u = 0;; ++u) {
            const int islot = u % kNI;
            if (!wait(bars + C::bItFull + islot, (u / kNI) & 1)) {
                ok = false;
                break;
            }
            const StagedItem *si = items + islot;
            if (!si->valid) break;
            const int32_t first = si->first, end = si->end, bin = si->bin, rg = si->rg;
            const int32_t kv = si->kv, qbase = si->qbase, roff = si->roff;
            const int32_t ibase = si->ibase, j0 = si->j0;
            if (gw == 0 && rg >= ring) {
                // the ring entry must have been merged by its previous range
                int got = 1;
                if (lane == 0)
                    got = tc::wait_counter(a.merge_done + (rg - ring), a.w.range_merges[rg - ring],
                                           status);
                if (!__shfl_sync(kFull, got, 0)) {
                    ok = false;
                    break;
                }
            }
            // every tile of an item goes to one owner warpgroup, items alternate
            const int X = item_idx & 1;
            for (int32_t p0 = first; p0 < end; p0 += kTile) {
                const int s = g % C::kNQ, tx = gx[X], slot = X * kNTW + tx % kNTW;
                if (g >= C::kNQ && !wait(bars + C::bQFree + s, ((g / C::kNQ) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (tx >= kNTW && !wait(bars + C::bTiFree + slot, ((tx / kNTW) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int cnt = min(kTile, end - p0);
                const int32_t *pp = si->pid + (p0 - first);
                const int32_t my_pid = pp[gt < cnt ? gt : 0];
                if (gt < cnt) pids[slot * kTile + gt] = my_pid;
                const int32_t my_q = my_pid >> 5;            // flat query row h*n + i
                uint8_t *sQ = sm + C::oQ + s * C::kQBytes;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rl = i * 4 + rsub, r = gw * 32 + rl;
                    const int64_t qrow = __shfl_sync(kFull, my_q, rl);
                    const uint16_t *src = a.q + qrow * D + chunk * 8;
                    uint8_t *dst = sQ + r * 128 + ((chunk ^ (r & 7)) << 4);
#pragma unroll
                    for (int sub = 0; sub < C::kSub; ++sub)   // rows past the pairs read as zeros
                        tc::cp_async16_zfill(dst + sub * kTile * 128, src + sub * 64, r < cnt);
                }
                cp_async_arrive_noinc(bars + C::bQFull + s);
                if (gt == 0) {
                    TileInfo x;
                    x.bin = bin;
                    x.p0 = p0;
                    x.count = cnt;
                    x.item = item_idx;
                    x.last = p0 + kTile >= end;
                    x.rg = rg;
                    x.end = 0;
                    x.kv = kv;
                    x.qbase = qbase;
                    x.roff = roff;
                    x.ibase = ibase;
                    x.j0 = j0;
                    x.g = g;
                    ti[slot] = x;
                }
                tc::mbar_arrive(bars + C::bTiFull + slot);
                ++g;
                ++gx[X];
            }
            if (!ok) break;
            tc::mbar_arrive(bars + C::bItFree + islot);
            ++item_idx;
        }
        if (ok) {
            // an end marker for each owner warpgroup
            for (int X = 0; X < 2; ++X) {
                const int tx = gx[X], slot = X * kNTW + tx % kNTW;
                if (tx < kNTW || wait(bars + C::bTiFree + slot, ((tx / kNTW) - 1) & 1)) {
                    if (gt == 0) ti[slot].end = 1;
                    tc::mbar_arrive(bars + C::bTiFull + slot);
                }
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------ owner warpgroups
        // Warpgroup X (warps 4X .. 4X+3) runs every tile of its fine items
        // from start to end, one thread per pair row: the issuing warp
        // (the first of the group) waits for the tile's Q rows and its
        // item's K_b, V_b and issues S = Q K_b^T into the group's S columns;
        // every thread turns its row of S into P (bf16, into tensor memory)
        // and (m, l); the issuing warp issues O = P V_b; every thread then
        // stores its pair's partial state o = O / l (bf16) and
        // lse = m + log2 l.  With two groups one runs its softmax or stores
        // while the other's MMAs run.  Every wait's outcome is combined over
        // the group at its named barriers, so the group leaves together.
        // One thread counts the group's finished pairs per query range for
        // the merges, up to four tiles under one GPU-scope fence; it counts
        // at once whenever the group's next tile is not there yet, so that no
        // count is held back while this CTA waits on others.
        const int X = warp >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int wt = threadIdx.x & 127;        // thread within the group
        const uint32_t bid = 2 + uint32_t(X);    // the group's named barrier
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        const uint32_t tS = tmem + uint32_t(X) * C::kWgCols, tP = tS + 64, tO = tS + 96;
        uint64_t *b_tifull = bars + C::bTiFull + X * kNTW, *b_tifree = bars + C::bTiFree + X * kNTW;
        uint64_t *b_sdone = bars + C::bSDone + X, *b_odone = bars + C::bODone + X;
        uint8_t *eb = sm + C::oEpi + warp * 2048;
        const int srow = lane >> 2, spiece = lane & 3;      // store phase: rows 8i + srow
        constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kTile, kB);
        constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kTile, D, /*b_mn_major=*/true);
        int cur_item = -1;                       // item whose K/V buffer is known to be full
        int32_t pend_rg = -1, pend_cnt = 0, pend_rg2 = -1, pend_cnt2 = 0, pend_tiles = 0;
        auto publish = [&]() {                   // thread wt == 32 only
            if (pend_tiles > 0) {
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                if (pend_rg2 >= 0) atomicAdd(a.range_done + pend_rg2, pend_cnt2);
                atomicAdd(a.range_done + pend_rg, pend_cnt);
                pend_rg = pend_rg2 = -1;
                pend_cnt = pend_cnt2 = pend_tiles = 0;
            }
        };
        for (int t = 0;; ++t) {
            const int slot = t % kNTW;
            const uint32_t par = (t / kNTW) & 1;
            if (wt == 32 && pend_tiles > 0 && !tc::mbar_test_wait(b_tifull + slot, par)) publish();
            bool ok = tc::mbar_wait(b_tifull + slot, par, status);
            if (!tc::named_bar_and(bid, 128, ok)) break;
            const volatile TileInfo *xi = ti + X * kNTW + slot;
            if (xi->end) break;
            const int32_t x_item = xi->item, x_g = xi->g, x_count = xi->count, x_last = xi->last;
            const int32_t x_rg = xi->rg, x_qbase = xi->qbase, x_roff = xi->roff;
            const int32_t *tpid = pids + (X * kNTW + slot) * kTile;
            int keys_valid = xi->kv;                    // < 64: ragged last block
            if (kOpts && a.causal && row < x_count) {
                // causal: query i admits the keys j <= i of the block
                const int32_t i = (tpid[row] >> 5) - x_qbase + xi->ibase;
                keys_valid = min(keys_valid, i - xi->j0 + 1);   // <= 0: nothing admitted
            }
            const int s = x_g % C::kNQ, ib = x_item % C::kNKV;
            // ---- S = Q K_b^T
            bool issued = true;
            if (quad == 0) {
                if (x_item != cur_item)
                    issued = tc::mbar_wait(bars + C::bKvFull + ib, (x_item / C::kNKV) & 1, status);
                cur_item = x_item;
                issued = issued && tc::mbar_wait(bars + C::bQFull + s, (x_g / C::kNQ) & 1, status);
                issued = __all_sync(kFull, issued);
                if (issued) {
                    // the Q rows were written by cp.async (generic proxy); the MMA
                    // reads them through the async proxy
                    tc::fence_proxy_async_smem();
                    tc::tc_fence_after();
                    if (tc::elect_one()) {
                        const uint32_t aq = tc::smem_u32(sm + C::oQ + s * C::kQBytes);
                        const uint32_t ak = tc::smem_u32(sm + C::oK + ib * C::kKBytes);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off_q = uint32_t((kk >> 2) * kTile * 128 + (kk & 3) * 32);
                            const uint32_t off_k = uint32_t((kk >> 2) * kB * 128 + (kk & 3) * 32);
                            tc::mma_bf16(tS, tc::smem_desc_sw128(aq + off_q, 1024),
                                         tc::smem_desc_sw128(ak + off_k, 1024), idesc_s, kk > 0);
                        }
                        tc::mma_commit(b_sdone);
                        tc::mma_commit(bars + C::bQFree + s);
                    }
                    __syncwarp();
                }
            }
            // if the S was not issued, this wait runs out too
            ok = tc::mbar_wait(b_sdone, uint32_t(t) & 1, status);
            float m2 = -INFINITY, lrow = 0.f;
            if (ok) {
                // ---- softmax: all 64 scores of the row in one load.  Keys past
                // `keys_valid` (a ragged last block, or the causal limit) are
                // masked out; a warp whose rows are all full skips the masks.
                // Both forms do the same arithmetic in the same order (a masked
                // key adds an exact zero), so a row's result does not depend on
                // which other rows share its tile.
                tc::tc_fence_after();
                uint32_t s0[32], s1[32];
                tc::tmem_ld32(tS + lane_off, s0);
                tc::tmem_ld32(tS + 32 + lane_off, s1);
                tc::tmem_ld_wait();
                const bool full = __all_sync(kFull, keys_valid == kB);
                auto row_softmax = [&](auto masked) {
                    constexpr bool kMasked = decltype(masked)::value;
                    auto sc = [&](int c) -> float {       // score of key c, -inf when masked
                        const float x = __uint_as_float(c < 32 ? s0[c] : s1[c - 32]);
                        return (!kMasked || c < keys_valid) ? x : -INFINITY;
                    };
                    float mx[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        // 16 scores per chain, four independent chains
                        float x[16];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            x[e] = sc(8 * u + e);
                            x[8 + e] = sc(32 + 8 * u + e);
                        }
                        float m = fmax3(x[0], x[1], x[2]);
#pragma unroll
                        for (int e = 3; e < 15; e += 2) m = fmax3(m, x[e], x[e + 1]);
                        mx[u] = fmaxf(m, x[15]);
                    }
                    m2 = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
                    auto pr = [&](int c) -> float {       // p of key c, exactly 0 when masked
                        const float x = __uint_as_float(c < 32 ? s0[c] : s1[c - 32]);
                        return (!kMasked || c < keys_valid) ? ex2(fmaf(x, a.scale_log2, -m2)) : 0.f;
                    };
                    float lsum[4] = {0.f, 0.f, 0.f, 0.f};
                    uint32_t pk0[16], pk1[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float p0 = pr(c), p1 = pr(c + 1), p2 = pr(c + 32), p3 = pr(c + 33);
                        lsum[(c >> 1) & 3] += (p0 + p1) + (p2 + p3);
                        pk0[c >> 1] = pack_bf16x2(p0, p1);
                        pk1[c >> 1] = pack_bf16x2(p2, p3);
                    }
                    tc::tmem_st16(tP + lane_off, pk0);
                    tc::tmem_st16(tP + 16 + lane_off, pk1);
                    lrow = (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
                };
                if (full) row_softmax(std::false_type{});
                else row_softmax(std::true_type{});
                tc::tmem_st_wait();
                tc::tc_fence_before();
            }
            // every row's P is in tensor memory
            if (!tc::named_bar_and(bid, 128, ok && issued)) break;
            // ---- O = P V_b
            if (quad == 0) {
                tc::tc_fence_after();
                if (tc::elect_one()) {
                    const uint32_t av = tc::smem_u32(sm + C::oV + ib * C::kKBytes);
#pragma unroll
                    for (int kk = 0; kk < kB / 16; ++kk)
                        tc::mma_bf16_ts(tO, tP + uint32_t(kk * 8),
                                        tc::smem_desc_sw128_mn(av + kk * 2048, kB * 128, 1024), idesc_o,
                                        kk > 0);
                    tc::mma_commit(b_odone);
                    if (x_last) tc::mma_commit(bars + C::bKvFree + ib);
                }
                __syncwarp();
            }
            ok = tc::mbar_wait(b_odone, uint32_t(t) & 1, status);
            if (ok) {
                // ---- epilogue: this row's pair state, the unnormalised O (bf16)
                // and (m, l); the merge divides once per query.  O is read from
                // TMEM 64 columns at a time and goes through a small swizzled
                // shared buffer per warp, so that a store instruction writes
                // whole row segments: at d = 64 each 32-column half as 64
                // contiguous bytes of 8 rows; at d = 128 each 64-column chunk
                // as 128 bytes of 4 rows, staged 16 rows at a time (measured:
                // the first form is faster at d = 64, the second at d = 128;
                // one 16-byte store per row per instruction is far slower).
                tc::tc_fence_after();
                const bool has = row < x_count;
                int32_t part = 0;                               // < ring * range * kpad
                if (has) {
                    const int32_t pid = tpid[row];
                    part = x_roff + ((pid >> 5) - x_qbase) * int32_t(kpad) + (pid & 31);
                }
                if constexpr (D == 64) {
                    int32_t sp[4];                                  // part of rows 8i + srow
                    bool sh[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        sp[i] = __shfl_sync(kFull, part, 8 * i + srow);
                        sh[i] = quad * 32 + 8 * i + srow < x_count;
                    }
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 64) {
                        uint32_t ov[2][32];
                        tc::tmem_ld32(tO + uint32_t(c0) + lane_off, ov[0]);
                        tc::tmem_ld32(tO + uint32_t(c0 + 32) + lane_off, ov[1]);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const uint4 val = make_uint4(
                                    pack_bf16x2(__uint_as_float(ov[hf][8 * v + 0]), __uint_as_float(ov[hf][8 * v + 1])),
                                    pack_bf16x2(__uint_as_float(ov[hf][8 * v + 2]), __uint_as_float(ov[hf][8 * v + 3])),
                                    pack_bf16x2(__uint_as_float(ov[hf][8 * v + 4]), __uint_as_float(ov[hf][8 * v + 5])),
                                    pack_bf16x2(__uint_as_float(ov[hf][8 * v + 6]), __uint_as_float(ov[hf][8 * v + 7])));
                                *reinterpret_cast<uint4 *>(eb + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) = val;
                            }
                            __syncwarp();
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int r = 8 * i + srow;
                                const uint4 val =
                                    *reinterpret_cast<const uint4 *>(eb + r * 64 + ((spiece ^ ((r >> 1) & 3)) << 4));
                                if (sh[i])
                                    *reinterpret_cast<uint4 *>(a.part_o + int64_t(sp[i]) * D + c0 + hf * 32 + spiece * 8) = val;
                            }
                            __syncwarp();
                        }
                    }
                } else {
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 64) {
                        uint32_t ov[2][32];
                        tc::tmem_ld32(tO + uint32_t(c0) + lane_off, ov[0]);
                        tc::tmem_ld32(tO + uint32_t(c0 + 32) + lane_off, ov[1]);
                        tc::tmem_ld_wait();
                        // two passes of 16 rows: lanes 16p .. 16p + 15 put their 128-byte
                        // row segment into the buffer (row r, chunk c at c ^ (r & 7)),
                        // then every store instruction writes four whole rows
#pragma unroll
                        for (int ps = 0; ps < 2; ++ps) {
                            if ((lane >> 4) == ps) {
                                const int r = lane & 15;
#pragma unroll
                                for (int v = 0; v < 8; ++v) {
                                    const int hf = v >> 2, vv = v & 3;
                                    const uint4 val = make_uint4(
                                        pack_bf16x2(__uint_as_float(ov[hf][8 * vv + 0]), __uint_as_float(ov[hf][8 * vv + 1])),
                                        pack_bf16x2(__uint_as_float(ov[hf][8 * vv + 2]), __uint_as_float(ov[hf][8 * vv + 3])),
                                        pack_bf16x2(__uint_as_float(ov[hf][8 * vv + 4]), __uint_as_float(ov[hf][8 * vv + 5])),
                                        pack_bf16x2(__uint_as_float(ov[hf][8 * vv + 6]), __uint_as_float(ov[hf][8 * vv + 7])));
                                    *reinterpret_cast<uint4 *>(eb + r * 128 + ((v ^ (r & 7)) << 4)) = val;
                                }
                            }
                            __syncwarp();
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int r = 4 * i + (lane >> 3), ch = lane & 7;   // buffer row, chunk
                                const int src = 16 * ps + r;                         // lane of the row
                                const int32_t pr = __shfl_sync(kFull, part, src);
                                const uint4 val = *reinterpret_cast<const uint4 *>(eb + r * 128 + ((ch ^ (r & 7)) << 4));
                                if (quad * 32 + src < x_count)
                                    *reinterpret_cast<uint4 *>(a.part_o + int64_t(pr) * D + c0 + ch * 8) = val;
                            }
                            __syncwarp();
                        }
                    }
                }
                if (has) a.part_ml[part] = make_float2(m2, lrow);
                tc::tc_fence_before();
            }
            // the group's stores are done and its tile slot is no longer read
            if (!tc::named_bar_and(bid, 128, ok)) break;
            if (wt == 0) tc::mbar_arrive(b_tifree + slot);
            if (wt == 32) {
                if (pend_tiles > 0 && x_rg != pend_rg && pend_rg2 >= 0) publish();
                if (pend_tiles > 0 && x_rg != pend_rg) {
                    pend_rg2 = pend_rg;
                    pend_cnt2 = pend_cnt;
                    pend_cnt = 0;
                }
                pend_rg = x_rg;
                pend_cnt += x_count;
                if (++pend_tiles >= 4) publish();
            }
        }
        if (wt == 32) publish();
    } else if (merge_index(warp) >= 0) {
        // ---------------------------------------------------------- merge
        // Each merge warp runs on its own: it takes a merge item, waits for
        // the range's pairs, then streams the item's queries through its
        // shared-memory stages (one bulk copy for the partial o block and one
        // for the lse values of up to qs consecutive queries).  A group of
        // D/16 lanes merges one query, each lane owning 16 channels.
        constexpr bool kWide = D == 128;             // one query per warp (merge_query_w)
        constexpr int LPQ = kWide ? 32 : D / 16;     // lanes per query
        constexpr int CPL = D / LPQ;                 // channels per lane
        constexpr int QP = 32 / LPQ;                 // queries per pass
        const int mw = merge_index(warp);
        const int gq = lane / LPQ, gl = lane % LPQ;
        const int n_merge = *a.w.n_merge;
        const int32_t full_valid = a.full_lists ? int32_t(i64min(k, nb)) : 0;
        const uint32_t full_mask = full_valid >= 32 ? kFull : ((1u << full_valid) - 1u);
        const int64_t per_q = kpad * D * 2 + kpad * 8;
        const int qs = int(C::kStageBytes / per_q);               // queries per stage (>= QP)
        const int64_t o_cap = int64_t(qs) * kpad * D * 2;         // lse offset within a stage
        uint8_t *stage0 = sm + C::oMs + mw * C::kMS * C::kStageBytes;
        uint64_t *msbar = bars + C::bMsFull + mw * C::kMS;
        uint32_t sc = 0;                                          // stages used so far
        for (;;) {
            int it = 0;
            if (lane == 0) it = atomicAdd(a.merge_head, 1);
            it = __shfl_sync(kFull, it, 0);
            if (it >= n_merge) break;
            const int2 item = a.w.merge_items[it];
            const int64_t rg = item.x;
            const int64_t h = rg / nranges, rr = rg % nranges;
            const int64_t i_begin = rr * range + item.y;
            const int64_t i_end = i64min(i64min(n, rr * range + range), i_begin + a.p.qm);
            const int nq = int(i_end - i_begin);
            // lists with padding: the slot mask of query (i_begin + lane), loaded
            // while the range's pairs are still being finished
            uint32_t vml = 0u;
            if (full_valid == 0 && !(kOpts && a.sel_lists) && lane < nq)
                vml = __ldg(a.w.vmask + h * n + i_begin + lane);
            int got = 1;
            if (lane == 0) {
                got = tc::wait_counter(a.range_done + rg, a.w.range_total[rg], status);
                tc::fence_proxy_async_global();      // partials were written by generic stores
            }
            if (!__shfl_sync(kFull, got, 0)) break;
            // lists from the selection: the valid slots follow from the budget
            const int kr_h = kOpts && a.head_k != nullptr ? min(max(__ldg(a.head_k + h), 0), k) : k;
            const int nch = (nq + qs - 1) / qs;
            const int64_t slot0 = (int32_t(rg) & ring_mask) * ring_stride + (i_begin - rr * range) * kpad;
            auto issue = [&](int c) {                // lane 0: chunk c into its stage
                const uint32_t b = (sc + uint32_t(c)) % C::kMS;
                const int qn = min(qs, nq - c * qs);
                const uint32_t bo = uint32_t(qn * kpad * D * 2), bl = uint32_t(qn * kpad * 8);
                const int64_t sl = slot0 + int64_t(c) * qs * kpad;
                uint8_t *st = stage0 + b * C::kStageBytes;
                tc::mbar_arrive_expect_tx(msbar + b, bo + bl);
                tc::bulk_g2s(st, a.part_o + sl * D, bo, msbar + b);
                tc::bulk_g2s(st + o_cap, a.part_ml + sl, bl, msbar + b);
            };
            if (lane == 0)
                for (int c = 0; c < min(C::kMS, nch); ++c) issue(c);
            bool ok = true;
            for (int c = 0; c < nch; ++c) {
                const uint32_t u = sc + uint32_t(c), b = u % C::kMS;
                const int q0 = c * qs, qn = min(qs, nq - q0);
                const uint8_t *st = stage0 + b * C::kStageBytes;
                if (!tc::mbar_wait(msbar + b, (u / C::kMS) & 1, status)) {
                    ok = false;
                    break;
                }
                for (int q = 0; q < qn; q += QP) {
                    const int jq = q + gq;                // groups past qn read nothing
                    const bool act = jq < qn;
                    const int64_t qrow = h * n + i_begin + q0 + (act ? jq : 0);
                    uint32_t vm = act ? full_mask : 0u;
                    if (kOpts && full_valid == 0 && a.sel_lists) {
                        // the first min(k_h, eligible) slots hold ids
                        const int64_t i = i_begin + q0 + jq;
                        const int cnt = int(i64min(i64min(kr_h, nb), a.causal ? i / kB + 1 : nb));
                        vm = act ? (cnt >= 32 ? kFull : (1u << cnt) - 1u) : 0u;
                    } else if (full_valid == 0) {
                        // lists with padding: a slot counts only if its id is a block
                        vm = __shfl_sync(kFull, vml, (q0 + jq) & 31);
                        if (!act) vm = 0u;
                    }
                    float acc[CPL];
                    const uint16_t *po = reinterpret_cast<const uint16_t *>(st) + jq * kpad * D + gl * CPL;
                    const float *pl = reinterpret_cast<const float *>(st + o_cap) + 2 * jq * kpad;
                    // every lane takes part (the merge shuffles across the warp); a
                    // query with nothing listed was zeroed by the inversion, one
                    // whose listed blocks admit nothing (causal mask) is zeroed here
                    float lse = -INFINITY;
                    bool any;
                    if constexpr (kWide) any = merge_query_w<kOpts>(po, pl, vm, k, lane, acc, lse);
                    else any = merge_query<D, kOpts>(po, pl, vm, k, lane, acc, lse);
                    if (a.lse_out != nullptr && act && gl == 0) a.lse_out[qrow] = lse;
                    if (act && (any || kOpts)) {
                        if (!any) {
#pragma unroll
                            for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
                        }
                        if constexpr (CPL == 16) {
                            uint4 *dst = reinterpret_cast<uint4 *>(a.out + qrow * D + gl * 16);
                            dst[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
                            dst[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                                                pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
                        } else {
                            *reinterpret_cast<uint2 *>(a.out + qrow * D + gl * 4) =
                                make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
                        }
                    }
                }
                __syncwarp();                             // stage read by every lane
                if (lane == 0 && c + C::kMS < nch) issue(c + C::kMS);
            }
            if (!ok) break;
            sc += uint32_t(nch);
            if (lane == 0) red_add_release(a.merge_done + rg, 1);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
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

template <int D, bool kOpts>
cudaError_t launch_d(const FineBmArgs &a, const CUtensorMap &mk, const CUtensorMap &mv,
                     cudaStream_t st) {
    using C = Cfg<D>;
    auto kern = fine_ws_kernel<D, kOpts>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kTotal);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    kern<<<sms, kThreads, C::kTotal, st>>>(mk, mv, a);   // one CTA per SM
    return cudaGetLastError();
}

}  // namespace

bool fine_bm_supported(int32_t d, int32_t key_block) {
    return (d == 64 || d == 128) && key_block == kB;
}

cudaError_t launch_fine_bm(const FineBmArgs &a, cudaStream_t st) {
    if (a.k < 1 || a.k > 32) return cudaErrorInvalidValue;   // slot masks are 32 bits wide
    CUtensorMap mk, mv;
    if (!make_rows_map(&mk, a.k_ptr, a.bh, a.n, a.d, kB) || !make_rows_map(&mv, a.v_ptr, a.bh, a.n, a.d, kB))
        return cudaErrorInvalidValue;
    if (a.causal || a.sel_lists)
        return a.d == 64 ? launch_d<64, true>(a, mk, mv, st) : launch_d<128, true>(a, mk, mv, st);
    return a.d == 64 ? launch_d<64, false>(a, mk, mv, st) : launch_d<128, false>(a, mk, mv, st);
}

}  // namespace bsa
