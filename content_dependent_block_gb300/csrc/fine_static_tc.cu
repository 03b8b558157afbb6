// Stage 2 over static block lists on the tensor cores: every query of a
// 128-query tile attends the tokens of the tile's listed 64-key blocks,
// restricted by a token-level predicate (page "yayme/CUDA-kernel" README:
// local window |i - j| <= w or global stride j % s == 0 over a precomputed
// active-tile list; page "Block-Sparse & Linear Attention Kernels",
// section 2: sliding window over the nearest W tokens), with softmax scaled
// by 1/sqrt(d) (same page, sliding-window formula).  A NULL list means every
// block.
//
// Query-tile-major: one CTA per (head, 128-query tile).  The list is shared
// by the tile, so K_b and V_b are loaded once per tile.  Listed blocks are
// taken two at a time ("superblocks" of 128 keys; an odd list ends with a
// half made of keys past the sequence, loaded as zeros and masked out), so
// that every score tile is a 128 x 128 x d contraction and every P.V one of
// 128 keys: an N = 64 MMA costs nearly as long as an N = 128 one.  The
// softmax is exact and two-pass: pass 0 computes the row maxima over all
// listed blocks, pass 1 recomputes the scores, forms p = exp2(s * scale *
// log2 e - m) once, accumulates l and O += P V in tensor memory.  O is never
// rescaled, at the price of computing Q K^T twice.
//
// With a workspace the first pass is skipped: any m >= the row maximum gives
// the same softmax, so each row takes the bound m = |q_i| max_j |k_j| scale
// log2 e over the tile's listed blocks (the key norms come from a small
// kernel run first) and does pass 1 only.  That is exact up to rounding while
// the bound exceeds the true maximum by less than ~100 (p stays far above
// the smallest fp32 and bf16 normals); a tile with a row beyond that is
// flagged and recomputed by the two-pass kernel in a second launch whose
// other CTAs return at once.  Stage-use u runs over
// u < ns (pass 0, superblock u) and ns <= u < 2 ns (pass 1, superblock
// u - ns), ns = ceil(listed / 2).
//
//   warp 0     producer of Q (once) and of K for every stage-use, into a
//              ring of three 128-key stages
//   warp 1     MMA, warp-uniform loop, one elected lane issues:
//              S_u = Q K^T (M 128, N 128) into TMEM buffer u mod 3; the P.V
//              of a pass-1 superblock (A = P from TMEM, N = d, V MN-major)
//              two stage-uses later
//   warp 2     producer of V for every pass-1 superblock, into a ring of two
//   warps 3-14 three softmax warpgroups; group g takes the stage-uses
//              u = g mod 3 (TMEM buffer g), one thread per query row: masked
//              row max (pass 0), combined over the groups through shared
//              memory; masked p, l, and P (bf16) written over the scores
//              already read (pass 1); then O / l, 32-column chunks dealt
//              round-robin to the groups
#include <cmath>

#include <cudaTypedefs.h>

#include "bsa_device.cuh"
#include "bsa_internal.h"
#include "tc.cuh"

namespace bsa {
namespace {

constexpr int kTile = 128;             // queries per CTA (TMEM lanes)
constexpr int kB = 64;                 // keys per block
constexpr int kSB = 2 * kB;            // keys per superblock (two listed blocks)
constexpr int kGroups = 3;             // softmax warpgroups = S buffers in TMEM
constexpr int kLag = 2;                // P.V of a superblock this many stage-uses behind its scores
constexpr int kWarpSoftmax = 3;        // first softmax warp
constexpr int kThreads = 32 * kWarpSoftmax + kGroups * 128;
constexpr int kMaxList = 512;          // listed blocks held in shared memory per chunk
constexpr uint32_t kBarGroups = 1;     // named barrier of the softmax warpgroups
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct SCfg {
    static constexpr int kSub = D / 64;
    static constexpr int kKStages = 3;                      // K ring
    static constexpr int kVStages = 2;                      // V ring
    static constexpr int kS = kGroups;                      // S (and P) buffers in TMEM
    static constexpr int kQBytes = kSub * kTile * 128;
    static constexpr int kPanel = kSB * 128;                // 128 keys x 64 channels
    static constexpr int kStageBytes = kSub * kPanel;       // K or V of one superblock
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + kQBytes;
    static constexpr int oV = oK + kKStages * kStageBytes;
    static constexpr int oList = oV + kVStages * kStageBytes;   // int32 [kMaxList]
    static constexpr int oRed = oList + kMaxList * 4;       // float [2][kGroups][kTile]
    static constexpr int oBar = oRed + 2 * kGroups * kTile * 4;
    enum {
        bQFull = 0,
        bKFull = 1,
        bKEmpty = bKFull + kKStages,
        bVFull = bKEmpty + kKStages,
        bVEmpty = bVFull + kVStages,
        bSFull = bVEmpty + kVStages,
        bSFree = bSFull + kS,           // pass-0 scores read
        bPFull = bSFree + kS,           // pass-1 P written over its scores
        bPvDone = bPFull + kS,          // pass-1 P.V done: the buffer is free
        bOFull = bPvDone + kS,
        bCount = bOFull + 1
    };
    static constexpr int oMisc = oBar + bCount * 8;
    static constexpr int kTotal = oMisc + 64 + 1024;
    static constexpr uint32_t kTmemCols = 512;              // S[3] (P in the first 64 columns) from 0; O after them
    static constexpr uint32_t cO = kS * kSB;
};
static_assert(SCfg<128>::kTotal <= 227 * 1024, "shared memory (d = 128)");
static_assert(SCfg<128>::cO + 128 <= SCfg<128>::kTmemCols, "tensor memory (d = 128)");
static_assert(kLag < kGroups, "an S buffer is reused only after its P.V was issued");

// Pass-0 stage-uses (u < ns) that fall on S buffer j of ks.
__device__ __forceinline__ int pass0_uses(int ns, int j, int ks) { return (ns - j + ks - 1) / ks; }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Every (row, key) pair of the tile and block admitted by the predicate?
__device__ __forceinline__ bool block_full(const FineArgs &a, int64_t i0, int64_t j0) {
    const int64_t i1 = i64min(a.n, i0 + kTile) - 1, j1 = i64min(a.n, j0 + kB) - 1;
    if (j0 + kB > a.n) return false;                     // ragged last block: mask the tail
    if (a.mask_kind == 0) return true;
    if (a.mask_kind == 2) return j1 <= i0 && j0 > i1 - a.sliding;
    if (a.mask_kind == 3) return j1 <= i0;
    // local + global: every pair within the window
    return a.window >= 0 && i1 - j0 <= a.window && j1 - i0 <= a.window;
}

// Bits [lo, hi) of a 32-bit word, the bounds clamped to [0, 32].
__device__ __forceinline__ uint32_t bits_between(int64_t lo, int64_t hi) {
    const int l = int(lo < 0 ? 0 : (lo > 32 ? 32 : lo));
    const int h = int(hi < 0 ? 0 : (hi > 32 ? 32 : hi));
    if (l >= h) return 0u;
    return (h == 32 ? 0xffffffffu : (1u << h) - 1u) & ~((1u << l) - 1u);
}

// Bit c set iff key jc + c (c < 32) lies in the sequence and the predicate
// admits it for query i: the same sets as mask_admits, built once per 32 keys
// from the ranges they form (|i - j| <= w, i - W < j <= i and j <= i are
// intervals of j; j mod s == 0 is every s-th column).
__device__ __forceinline__ uint32_t admitted_bits(const FineArgs &a, int64_t i, int64_t jc) {
    const uint32_t inside = bits_between(0, a.n - jc);
    const int64_t d0 = i - jc;                           // key jc + c has i - j = d0 - c
    if (a.mask_kind == 2) return inside & bits_between(d0 - a.sliding + 1, d0 + 1);
    if (a.mask_kind == 3) return inside & bits_between(0, d0 + 1);
    if (a.mask_kind != 1) return inside;
    uint32_t m = a.window >= 0 ? bits_between(d0 - a.window, d0 + int64_t(a.window) + 1) : 0u;
    if (a.stride > 0) {
        const int64_t r0 = jc % a.stride;
        for (int64_t c = r0 == 0 ? 0 : a.stride - r0; c < 32; c += a.stride) m |= 1u << int(c);
    }
    return inside & m;
}

// Row maximum of 32 raw scores; kMasked keeps only the columns set in `adm`.
template <bool kMasked>
__device__ __forceinline__ float chunk_max(const uint32_t (&sv)[32], uint32_t adm) {
    float m[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = -INFINITY;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const float x = __uint_as_float(sv[c]);
        m[c & 7] = fmaxf(m[c & 7], (!kMasked || ((adm >> c) & 1u)) ? x : -INFINITY);
    }
#pragma unroll
    for (int w = 4; w > 0; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e) m[e] = fmaxf(m[e], m[e + w]);
    return m[0];
}

// p = 2^(s * scale_log2 - mm) of 32 raw scores (0 where not admitted), packed
// to bf16 pairs; returns their fp32 sum.
template <bool kMasked>
__device__ __forceinline__ float chunk_exp(const uint32_t (&sv)[32], uint32_t adm, float scale_log2,
                                           float mm, uint32_t (&pk)[16]) {
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
        float p[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            p[e] = ex2(fmaf(__uint_as_float(sv[c + e]), scale_log2, -mm));
            if (kMasked && !((adm >> (c + e)) & 1u)) p[e] = 0.f;
        }
        ls[(c >> 1) & 3] += p[0] + p[1];
        pk[c >> 1] = pack_bf16x2(p[0], p[1]);
    }
    return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// Largest key norm of each 64-key block: one CTA of 64 threads per (block, head).
template <int D>
__global__ void __launch_bounds__(64) key_norm_kernel(const uint16_t *__restrict__ k, int64_t n,
                                                       int64_t nb, float *__restrict__ kmax) {
    const int64_t h = blockIdx.y, b = blockIdx.x, j = b * kB + threadIdx.x;
    float s = 0.f;
    if (j < n) {
        const uint4 *row = reinterpret_cast<const uint4 *>(k + (h * n + j) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 u = __ldg(row + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
                s = fmaf(lo, lo, fmaf(hi, hi, s));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = fmaxf(s, __shfl_xor_sync(kFull, s, o));
    __shared__ float wmax[2];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) kmax[h * nb + b] = sqrtf(fmaxf(wmax[0], wmax[1]));
}

template <int D, bool kOnePass>
__global__ void __launch_bounds__(kThreads, 1) fine_static_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const FineArgs a) {
    using C = SCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = tc::align_smem_1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::oBar);
    int32_t *list_s = reinterpret_cast<int32_t *>(sm + C::oList);
    float *m_part = reinterpret_cast<float *>(sm + C::oRed);           // [kGroups][kTile]
    float *l_part = m_part + kGroups * kTile;                           // [kGroups][kTile]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::oMisc);
    int32_t *nlist_s = reinterpret_cast<int32_t *>(sm + C::oMisc + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = a.status;
    const int64_t tile = int64_t(blockIdx.y) * gridDim.x + blockIdx.x;
    // A wait elsewhere already ran out, or (second launch) the one-pass launch
    // served this tile: the whole CTA leaves together.
    if (__syncthreads_or(*reinterpret_cast<volatile int32_t *>(status) == kStatusTimeout ||
                         (!kOnePass && a.flags != nullptr && a.flags[tile] == 0)))
        return;
    const int64_t h = blockIdx.y;
    const int64_t i0 = int64_t(blockIdx.x) * kTile;
    float *kmax_s = reinterpret_cast<float *>(sm + C::oMisc + 32);   // largest key norm of the list

    // the tile's list, compacted to valid ids (padding and bad ids dropped)
    if (warp == 0) {
        int cnt = 0;
        if (a.list == nullptr) {
            for (int64_t b = lane; b < a.nb && b < kMaxList; b += 32) list_s[b] = int32_t(b);
            cnt = int(i64min(a.nb, kMaxList));
        } else {
            const int64_t row = i0 / a.q_group;
            const int32_t *lr = a.list + ((a.per_head ? h * a.list_rows : 0) + row) * a.max_blocks;
            bool bad = false;
            for (int base = 0; base < a.max_blocks; base += 32) {
                const int e = base + lane;
                const int32_t b = e < a.max_blocks ? __ldg(lr + e) : -1;
                const bool ok = b >= 0 && b < a.nb;
                bad |= e < a.max_blocks && !ok && b != -1;
                const unsigned m = __ballot_sync(kFull, ok);
                if (ok) {
                    const int pos = cnt + __popc(m & ((1u << lane) - 1u));
                    if (pos < kMaxList) list_s[pos] = b;
                }
                cnt += __popc(m);
            }
            if (__any_sync(kFull, bad) && lane == 0) report_status(status, kStatusBadIndex);
            cnt = min(cnt, kMaxList);
        }
        if (lane == 0) *nlist_s = cnt;
        if (kOnePass) {
            __syncwarp();
            float km = 0.f;
            for (int t = lane; t < cnt; t += 32) km = fmaxf(km, __ldg(a.kmax + h * a.nb + list_s[t]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) km = fmaxf(km, __shfl_xor_sync(kFull, km, o));
            if (lane == 0) *kmax_s = km;
        }
    }
    if (threadIdx.x == 0) {
        tc::mbar_init(bars + C::bQFull, 1);
        for (int s = 0; s < C::kKStages; ++s) {
            tc::mbar_init(bars + C::bKFull + s, 1);
            tc::mbar_init(bars + C::bKEmpty + s, 1);
        }
        for (int r = 0; r < C::kVStages; ++r) {
            tc::mbar_init(bars + C::bVFull + r, 1);
            tc::mbar_init(bars + C::bVEmpty + r, 1);
        }
        for (int j = 0; j < C::kS; ++j) {
            tc::mbar_init(bars + C::bSFull + j, 1);
            tc::mbar_init(bars + C::bSFree + j, kTile);     // one warpgroup per stage-use
            tc::mbar_init(bars + C::bPFull + j, kTile);
            tc::mbar_init(bars + C::bPvDone + j, 1);
        }
        tc::mbar_init(bars + C::bOFull, 1);
        tc::fence_barrier_init();
        tc::prefetch_tensormap(&tm_q);
        tc::prefetch_tensormap(&tm_k);
        tc::prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int nl = *nlist_s;
    const int ns = (nl + 1) >> 1;                     // superblocks
    const int np0 = kOnePass ? 0 : ns;                // pass-0 stage-uses
    // first key of block `blk` of the list; past the end: keys beyond the
    // sequence (loaded as zeros, never admitted)
    auto block_key0 = [&](int blk) -> int64_t {
        return blk < nl ? int64_t(list_s[blk]) * kB : a.nb * kB;
    };

    if (warp == 0) {
        // ------------------------------------------------- producer of Q, K
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(bars + C::bQFull, C::kQBytes);
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
                tc::tma_load_3d(sm + C::oQ + sub * kTile * 128, &tm_q, bars + C::bQFull, sub * 64,
                                int32_t(i0), int32_t(h));
            for (int u = 0; u < np0 + ns; ++u) {
                const int sb = u >= np0 ? u - np0 : u, s = u % C::kKStages;
                if (u >= C::kKStages &&
                    !tc::mbar_wait(bars + C::bKEmpty + s, ((u / C::kKStages) - 1) & 1, status))
                    break;
                tc::mbar_arrive_expect_tx(bars + C::bKFull + s, C::kStageBytes);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int32_t key0 = int32_t(block_key0(2 * sb + half));
#pragma unroll
                    for (int sub = 0; sub < C::kSub; ++sub)
                        tc::tma_load_3d(sm + C::oK + s * C::kStageBytes + sub * C::kPanel + half * kB * 128,
                                        &tm_k, bars + C::bKFull + s, sub * 64, key0, int32_t(h));
                }
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ producer of V
        if (lane == 0) {
            for (int sb = 0; sb < ns; ++sb) {
                const int r = sb % C::kVStages;
                if (sb >= C::kVStages &&
                    !tc::mbar_wait(bars + C::bVEmpty + r, ((sb / C::kVStages) - 1) & 1, status))
                    break;
                tc::mbar_arrive_expect_tx(bars + C::bVFull + r, C::kStageBytes);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int32_t key0 = int32_t(block_key0(2 * sb + half));
#pragma unroll
                    for (int sub = 0; sub < C::kSub; ++sub)
                        tc::tma_load_3d(sm + C::oV + r * C::kStageBytes + sub * C::kPanel + half * kB * 128,
                                        &tm_v, bars + C::bVFull + r, sub * 64, key0, int32_t(h));
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kTile, kSB);
        constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kTile, D, /*b_mn_major=*/true);
        bool ok = __all_sync(kFull, tc::mbar_wait(bars + C::bQFull, 0, status));
        const uint32_t aq = tc::smem_u32(sm + C::oQ);
        // O += P_sb V_sb, P (bf16) in the first 64 columns of the superblock's S buffer
        auto issue_pv = [&](int sb) {
            const int u = sb + np0, j = u % C::kS, r = sb % C::kVStages;
            bool w = tc::mbar_wait(bars + C::bVFull + r, (sb / C::kVStages) & 1, status);
            w = w && tc::mbar_wait(bars + C::bPFull + j, (u / C::kS - pass0_uses(np0, j, C::kS)) & 1,
                                   status);
            ok = __all_sync(kFull, w);
            if (!ok) return;
            tc::tc_fence_after();
            if (tc::elect_one()) {
                const uint32_t av = tc::smem_u32(sm + C::oV + r * C::kStageBytes);
#pragma unroll
                for (int kk = 0; kk < kSB / 16; ++kk)
                    tc::mma_bf16_ts(tmem + C::cO, tmem + uint32_t(j * kSB + kk * 8),
                                    tc::smem_desc_sw128_mn(av + kk * 2048, C::kPanel, 1024), idesc_o,
                                    (sb > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit(bars + C::bPvDone + j);
                tc::mma_commit(bars + C::bVEmpty + r);
                if (sb == ns - 1) tc::mma_commit(bars + C::bOFull);
            }
            __syncwarp();
        };
        for (int u = 0; ok && u < np0 + ns + kLag; ++u) {
            if (u < np0 + ns) {
                const int s = u % C::kKStages, j = u % C::kS, prev = u - C::kS;
                bool w = tc::mbar_wait(bars + C::bKFull + s, (u / C::kKStages) & 1, status);
                // the buffer's last use: pass-0 scores read, or the P.V of its P done
                if (w && prev >= 0)
                    w = prev < np0 ? tc::mbar_wait(bars + C::bSFree + j, (prev / C::kS) & 1, status)
                                   : tc::mbar_wait(bars + C::bPvDone + j,
                                                   (prev / C::kS - pass0_uses(np0, j, C::kS)) & 1, status);
                ok = __all_sync(kFull, w);
                if (!ok) break;
                tc::tc_fence_after();
                if (tc::elect_one()) {
                    const uint32_t ak = tc::smem_u32(sm + C::oK + s * C::kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off_q = uint32_t((kk >> 2) * kTile * 128 + (kk & 3) * 32);
                        const uint32_t off_k = uint32_t((kk >> 2) * C::kPanel + (kk & 3) * 32);
                        tc::mma_bf16(tmem + uint32_t(j * kSB), tc::smem_desc_sw128(aq + off_q, 1024),
                                     tc::smem_desc_sw128(ak + off_k, 1024), idesc_s, kk > 0);
                    }
                    tc::mma_commit(bars + C::bSFull + j);
                    tc::mma_commit(bars + C::bKEmpty + s);             // K is read by S only
                }
                __syncwarp();
            }
            // P.V kLag stage-uses behind the scores
            if (u - kLag >= np0) issue_pv(u - kLag - np0);
        }
    } else {
        // ----------------------------------------- softmax and epilogue
        const int g = (warp - kWarpSoftmax) >> 2;      // warpgroup: stage-uses u = g mod kGroups
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int64_t i = i0 + row;
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        float m2 = -INFINITY, l = 0.f;
        bool ok = true;
        // pass 0: masked row maxima of this group's superblocks
        for (int u = g; ok && u < np0; u += kGroups) {
            const int j = u % C::kS;
            if (!tc::mbar_wait(bars + C::bSFull + j, (u / C::kS) & 1, status)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const int64_t j0a = block_key0(2 * u), j0b = block_key0(2 * u + 1);
            const bool fa = 2 * u < nl && block_full(a, i0, j0a);
            const bool fb = 2 * u + 1 < nl && block_full(a, i0, j0b);
            float mraw = -INFINITY;
#pragma unroll 1
            for (int c = 0; c < kSB / 32; ++c) {
                uint32_t sv[32];
                tc::tmem_ld32(tmem + uint32_t(j * kSB + c * 32) + lane_off, sv);
                tc::tmem_ld_wait();
                const bool full = c < 2 ? fa : fb;
                const int64_t jc = (c < 2 ? j0a : j0b) + (c & 1) * 32;
                mraw = fmaxf(mraw, full ? chunk_max<false>(sv, 0u)
                                        : chunk_max<true>(sv, admitted_bits(a, i, jc)));
            }
            tc::tc_fence_before();
            tc::mbar_arrive(bars + C::bSFree + j);
            m2 = fmaxf(m2, mraw * a.scale_log2);                     // scale > 0 keeps the order
        }
        float mm;
        if (kOnePass) {
            // the row's bound |q_i| max |k| scale log2 e on every admitted score
            float qq = 0.f;
            if (i < a.n) {
                const uint4 *qr = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.q) +
                                                                  (h * a.n + i) * D);
#pragma unroll 4
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 u = __ldg(qr + c);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
                        qq = fmaf(lo, lo, fmaf(hi, hi, qq));
                    }
                }
            }
            mm = sqrtf(qq) * *kmax_s * a.scale_log2;
        } else {
            // the row maximum over the groups (every group thread passes here once)
            m_part[g * kTile + row] = m2;
            tc::named_bar_sync(kBarGroups, kGroups * 128);
#pragma unroll
            for (int o = 0; o < kGroups; ++o) m2 = fmaxf(m2, m_part[o * kTile + row]);
            mm = m2 == -INFINITY ? 0.f : m2;                          // a row with no admitted key
        }
        float mtrue = -INFINITY;                                      // one pass: the actual maximum (raw)
        // pass 1: p, l and P of this group's superblocks
        for (int u = np0 + (g + kGroups - np0 % kGroups) % kGroups; ok && u < np0 + ns; u += kGroups) {
            const int sb = u - np0, j = u % C::kS;
            if (!tc::mbar_wait(bars + C::bSFull + j, (u / C::kS) & 1, status)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const int64_t j0a = block_key0(2 * sb), j0b = block_key0(2 * sb + 1);
            const bool fa = 2 * sb < nl && block_full(a, i0, j0a);
            const bool fb = 2 * sb + 1 < nl && block_full(a, i0, j0b);
#pragma unroll 1
            for (int c = 0; c < kSB / 32; ++c) {
                uint32_t sv[32];
                tc::tmem_ld32(tmem + uint32_t(j * kSB + c * 32) + lane_off, sv);
                tc::tmem_ld_wait();
                const bool full = c < 2 ? fa : fb;
                const int64_t jc = (c < 2 ? j0a : j0b) + (c & 1) * 32;
                uint32_t pk[16];
                const uint32_t adm = full ? 0xffffffffu : admitted_bits(a, i, jc);
                if (kOnePass)
                    mtrue = fmaxf(mtrue, full ? chunk_max<false>(sv, 0u) : chunk_max<true>(sv, adm));
                l += full ? chunk_exp<false>(sv, 0u, a.scale_log2, mm, pk)
                          : chunk_exp<true>(sv, adm, a.scale_log2, mm, pk);
                // P over scores already read: columns [16 c, 16 c + 16) of the buffer
                tc::tmem_st16(tmem + uint32_t(j * kSB + c * 16) + lane_off, pk);
            }
            tc::tmem_st_wait();
            tc::tc_fence_before();
            tc::mbar_arrive(bars + C::bPFull + j);
        }
        // the row sum over the groups
        l_part[g * kTile + row] = l;
        tc::named_bar_sync(kBarGroups, kGroups * 128);
        l = 0.f;
#pragma unroll
        for (int o = 0; o < kGroups; ++o) l += l_part[o * kTile + row];
        if (kOnePass) {
            // did the bound serve every row?  Else the second launch redoes the tile.
            m_part[g * kTile + row] = mtrue;
            tc::named_bar_sync(kBarGroups, kGroups * 128);
#pragma unroll
            for (int o = 0; o < kGroups; ++o) mtrue = fmaxf(mtrue, m_part[o * kTile + row]);
            const float gap = mm - mtrue * a.scale_log2;
            const bool bad_row = i < a.n && mtrue > -INFINITY && !(gap <= 100.f && l > 0.f && l < INFINITY);
            if (g == 0 && __any_sync(kFull, bad_row) && lane == 0) a.flags[tile] = 1;
        }
        // epilogue: O / l; group g writes the 32-column chunks c = g mod kGroups
        if (ok && nl > 0 && tc::mbar_wait(bars + C::bOFull, 0, status)) {
            tc::tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            uint16_t *dst = static_cast<uint16_t *>(a.out) + (h * a.n + i) * D;
#pragma unroll 1
            for (int c0 = g * 32; c0 < D; c0 += kGroups * 32) {
                uint32_t ov[32];
                tc::tmem_ld32(tmem + C::cO + uint32_t(c0) + lane_off, ov);
                tc::tmem_ld_wait();
                if (i < a.n) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        reinterpret_cast<uint4 *>(dst + c0)[v] = make_uint4(
                            pack_bf16x2(__uint_as_float(ov[8 * v + 0]) * inv_l, __uint_as_float(ov[8 * v + 1]) * inv_l),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 2]) * inv_l, __uint_as_float(ov[8 * v + 3]) * inv_l),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 4]) * inv_l, __uint_as_float(ov[8 * v + 5]) * inv_l),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 6]) * inv_l, __uint_as_float(ov[8 * v + 7]) * inv_l));
                }
            }
        } else if (nl == 0 && i < a.n) {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + (h * a.n + i) * D);
            for (int v = g * 4; v < D / 8; v += kGroups * 4) {               // nothing listed
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[v + e] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

// [bh][n][d] bf16 viewed as a 3-D tensor, box 64 x rows x 1, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int64_t bh, int64_t n, int d, int rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(n), cuuint64_t(bh)};
    cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(n) * d * 2};
    cuuint32_t box[3] = {64, cuuint32_t(rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kOnePass>
cudaError_t launch_kernel(const FineArgs &a, const CUtensorMap &mq, const CUtensorMap &mk,
                          const CUtensorMap &mv, cudaStream_t st) {
    using C = SCfg<D>;
    auto kern = fine_static_tc_kernel<D, kOnePass>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kTotal);
    if (e != cudaSuccess) return e;
    const dim3 grid(unsigned((a.n + kTile - 1) / kTile), unsigned(a.bh));
    kern<<<grid, kThreads, C::kTotal, st>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FineArgs &a, const CUtensorMap &mq, const CUtensorMap &mk,
                     const CUtensorMap &mv, cudaStream_t st) {
    if (a.kmax == nullptr || a.flags == nullptr) {
        FineArgs b = a;
        b.flags = nullptr;                   // every tile, two passes
        return launch_kernel<D, false>(b, mq, mk, mv, st);
    }
    key_norm_kernel<D><<<dim3(unsigned(a.nb), unsigned(a.bh)), kB, 0, st>>>(
        static_cast<const uint16_t *>(a.k), a.n, a.nb, a.kmax);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t tiles = a.bh * ((a.n + kTile - 1) / kTile);
    if ((e = cudaMemsetAsync(a.flags, 0, size_t(tiles) * sizeof(int32_t), st)) != cudaSuccess) return e;
    if ((e = launch_kernel<D, true>(a, mq, mk, mv, st)) != cudaSuccess) return e;
    return launch_kernel<D, false>(a, mq, mk, mv, st);      // flagged tiles only
}

}  // namespace

bool fine_static_tc_supported(const FineArgs &a, int32_t dtype) {
    return dtype == 0 /*bf16*/ && (a.d == 64 || a.d == 128) && a.kb == kB &&
           (a.list == nullptr || a.q_group == kTile) && a.bh <= 65535 &&
           (a.list == nullptr ? a.nb <= kMaxList : a.max_blocks <= kMaxList);
}

size_t fine_static_tc_workspace(int64_t bh, int64_t n, int32_t kb) {
    const int64_t nb = (n + kb - 1) / kb, tiles = (n + kTile - 1) / kTile;
    return size_t(bh) * size_t(nb) * 4 + 256 + size_t(bh) * size_t(tiles) * 4;
}

cudaError_t launch_fine_static_tc(const FineArgs &a, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, a.bh, a.n, a.d, kTile) || !make_map(&mk, a.k, a.bh, a.n, a.d, kB) ||
        !make_map(&mv, a.v, a.bh, a.n, a.d, kB))
        return cudaErrorInvalidValue;
    if (a.d == 64) return launch_d<64>(a, mq, mk, mv, st);
    return launch_d<128>(a, mq, mk, mv, st);
}

}  // namespace bsa
