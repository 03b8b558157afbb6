// Backward pass of the fine stage over per-query block lists (page
// "sparse-attention-triton-bench", What's next: a backward pass through the
// sparse softmax-weighted sum over the selected blocks; the selection is a
// discrete choice and is held fixed).  For query i with token set T_i (the
// listed blocks' keys; only j <= i under the causal mask), s_ij = scale
// q_i.k_j, p_ij = softmax over T_i, and the output gradient dO:
//   D_i   = dO_i . O_i                 (= sum_j p_ij dO_i . v_j)
//   dS_ij = p_ij (dO_i . v_j - D_i)
//   dQ_i  = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
//   dV_j  = sum_i p_ij dO_i.
// CUDA cores, fp32 throughout, three steps:
//   bwd_query_kernel  one warp per query, lanes over keys: the log-sum-exp
//                     of the row (online, recomputed), D_i, then dQ_i
//   count/scan/scatter  the lists inverted to (head, block) -> queries
//   bwd_kv_kernel     one CTA per (head, block): each thread owns 16
//                     channels of one key and accumulates dK, dV over the
//                     queries that listed the block (32 at a time in shared
//                     memory)
// No atomics on the gradients: every output element has one writer.
#include <cmath>

#include "bsa_device.cuh"
#include "bsa_internal.h"
#include "tc.cuh"

namespace bsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kQWarps = 8;          // queries per CTA of the per-query kernel
constexpr int kBatch = 32;          // queries staged per round of the (head, block) kernel
constexpr int kScanThreads = 1024;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf(uint16_t x) { return __uint_as_float(uint32_t(x) << 16); }

// q . row for a bf16 row of D channels (16-byte loads) against fp32 q in
// shared memory, read four channels at a time (every lane reads the same q:
// broadcast).
template <int D>
__device__ __forceinline__ float dot_row(const float *q, const uint16_t *row) {
    float s = 0.f;
    const float4 *q4 = reinterpret_cast<const float4 *>(q);
#pragma unroll
    for (int c = 0; c < D; c += 8) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(row + c));
        const float4 qa = q4[c / 4], qb = q4[c / 4 + 1];
        s = fmaf(qa.x, bf16_low_half(u.x), s);
        s = fmaf(qa.y, bf16_high_half(u.x), s);
        s = fmaf(qa.z, bf16_low_half(u.y), s);
        s = fmaf(qa.w, bf16_high_half(u.y), s);
        s = fmaf(qb.x, bf16_low_half(u.z), s);
        s = fmaf(qb.y, bf16_high_half(u.z), s);
        s = fmaf(qb.z, bf16_low_half(u.w), s);
        s = fmaf(qb.w, bf16_high_half(u.w), s);
    }
    return s;
}

// The keys of listed block b that query i attends: [j0, jend).
__device__ __forceinline__ void block_keys(const BwdArgs &a, int32_t b, int64_t i, int64_t &j0,
                                           int64_t &jend) {
    j0 = int64_t(b) * a.kb;
    jend = i64min(a.n, j0 + a.kb);
    if (a.causal) jend = i64min(jend, i + 1);
}

template <int D>
__global__ void __launch_bounds__(kQWarps * 32) bwd_query_kernel(const BwdArgs a) {
    __shared__ __align__(16) float sq[kQWarps][D];
    __shared__ __align__(16) float sdo[kQWarps][D];
    constexpr int CPL = D / 32;                        // channels per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t h = blockIdx.y;
    const int64_t i = int64_t(blockIdx.x) * kQWarps + warp;
    if (i >= a.n) return;                              // whole warp; no CTA barrier follows
    const int64_t row = h * a.n + i;
    float dsum = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        const int c = lane + 32 * e;
        const float dov = bf(a.dout[row * D + c]);
        sq[warp][c] = bf(a.q[row * D + c]);
        sdo[warp][c] = dov;
        dsum = fmaf(dov, bf(a.out[row * D + c]), dsum);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(kFull, dsum, o);
    __syncwarp();
    const int32_t *lst = a.list + row * a.k;
    const uint16_t *kh = a.kp + h * a.n * D, *vh = a.vp + h * a.n * D;
    // pass 1: online (max, sum) of exp2(s * scale_log2) per lane, then over the warp
    float m = -INFINITY, l = 0.f;
    bool bad = false;
    for (int t = 0; t < a.k; ++t) {
        const int32_t b = __ldg(lst + t);
        if (b < 0 || b >= a.nb) {
            bad |= b >= 0 || b < -1;
            continue;
        }
        int64_t j0, jend;
        block_keys(a, b, i, j0, jend);
        for (int64_t jb = j0; jb < jend; jb += 32) {
            const int64_t j = jb + lane;
            if (j < jend) {
                const float s = dot_row<D>(sq[warp], kh + j * D) * a.scale_log2;
                const float mn = fmaxf(m, s);
                l = l * ex2(m - mn) + ex2(s - mn);
                m = mn;
            }
        }
    }
    if (bad && lane == 0) report_status(a.status, kStatusBadIndex);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(kFull, m, o), lo = __shfl_xor_sync(kFull, l, o);
        const float mn = fmaxf(m, mo);
        l = (l > 0.f ? l * ex2(m - mn) : 0.f) + (lo > 0.f ? lo * ex2(mo - mn) : 0.f);
        m = mn;
    }
    const float lse = l > 0.f ? m + __log2f(l) : -INFINITY;
    if (lane == 0) {
        a.lse[row] = lse;
        a.dsum[row] = dsum;
    }
    // pass 2: dS per key (lanes over keys), dQ accumulated with lanes over
    // channels: lane owns channels [CPL lane, CPL lane + CPL)
    float dq[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) dq[e] = 0.f;
    if (l > 0.f) {
        for (int t = 0; t < a.k; ++t) {
            const int32_t b = __ldg(lst + t);
            if (b < 0 || b >= a.nb) continue;
            int64_t j0, jend;
            block_keys(a, b, i, j0, jend);
            for (int64_t jb = j0; jb < jend; jb += 32) {
                const int64_t j = jb + lane;
                float ds = 0.f;
                if (j < jend) {
                    const float p = ex2(dot_row<D>(sq[warp], kh + j * D) * a.scale_log2 - lse);
                    ds = p * (dot_row<D>(sdo[warp], vh + j * D) - dsum);
                }
                const int cnt = int(i64min(32, jend - jb));
                for (int u = 0; u < cnt; ++u) {
                    const float dsu = __shfl_sync(kFull, ds, u);
                    const uint32_t *kr = reinterpret_cast<const uint32_t *>(kh + (jb + u) * D) +
                                         lane * (CPL / 2);
#pragma unroll
                    for (int e = 0; e < CPL / 2; ++e) {
                        const uint32_t w = __ldg(kr + e);
                        dq[2 * e] = fmaf(dsu, bf16_low_half(w), dq[2 * e]);
                        dq[2 * e + 1] = fmaf(dsu, bf16_high_half(w), dq[2 * e + 1]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < CPL; ++e) a.dq[row * D + lane * CPL + e] = dq[e] * a.scale;
}

// grid: (ceil(n * k / 256), bh)
__global__ void __launch_bounds__(256) bwd_count_kernel(const BwdArgs a) {
    const int64_t h = blockIdx.y;
    const int64_t e = int64_t(blockIdx.x) * 256 + threadIdx.x;
    if (e >= a.n * a.k) return;
    const int32_t b = __ldg(a.list + h * a.n * a.k + e);
    if (b >= 0 && b < a.nb) atomicAdd(a.counts + h * a.nb + b, 1);
}

// one CTA: offsets = exclusive scan of counts over bh * nb bins (+ the total)
__global__ void __launch_bounds__(kScanThreads) bwd_scan_kernel(const BwdArgs a) {
    __shared__ int32_t warp_tot[kScanThreads / 32];
    __shared__ int32_t carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t m = a.bh * a.nb;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < m; base += kScanThreads) {
        const int64_t e = base + threadIdx.x;
        const int32_t v = e < m ? a.counts[e] : 0;
        int32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(kFull, w, o);
                if (lane >= o) w += y;
            }
            warp_tot[lane] = w;                        // inclusive over warps
        }
        __syncthreads();
        const int32_t before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
        if (e < m) a.offsets[e] = before;
        __syncthreads();
        if (threadIdx.x == 0) carry += warp_tot[kScanThreads / 32 - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) a.offsets[m] = carry;
}

__global__ void __launch_bounds__(256) bwd_scatter_kernel(const BwdArgs a) {
    const int64_t h = blockIdx.y;
    const int64_t e = int64_t(blockIdx.x) * 256 + threadIdx.x;
    if (e >= a.n * a.k) return;
    const int32_t b = __ldg(a.list + h * a.n * a.k + e);
    if (b < 0 || b >= a.nb) return;
    const int64_t bin = h * a.nb + b;
    const int32_t pos = atomicAdd(a.cursors + bin, 1);
    a.qlist[a.offsets[bin] + pos] = int32_t(e / a.k);
}

// grid: (nb, bh); kb * D / 16 threads: thread (key tok, part) owns channels
// [16 part, 16 part + 16) of key j = b * kb + tok.
template <int D>
__global__ void __launch_bounds__(512) bwd_kv_kernel(const BwdArgs a) {
    constexpr int G = D / 16;                          // threads per key
    __shared__ float sq[kBatch][D], sdo[kBatch][D];
    __shared__ float slse[kBatch], sds[kBatch];
    __shared__ int32_t si[kBatch];
    const int64_t h = blockIdx.y, b = blockIdx.x;
    const int tok = threadIdx.x / G, part = threadIdx.x % G;
    const int64_t j = b * a.kb + tok;
    const bool live = j < a.n;                         // tok < kb by the launch shape
    float kr[16], vr[16], dk[16], dv[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        kr[c] = live ? bf(a.kp[(h * a.n + j) * D + part * 16 + c]) : 0.f;
        vr[c] = live ? bf(a.vp[(h * a.n + j) * D + part * 16 + c]) : 0.f;
        dk[c] = dv[c] = 0.f;
    }
    const int64_t bin = h * a.nb + b;
    const int32_t q0 = a.offsets[bin], q1 = a.offsets[bin + 1];
    for (int32_t base = q0; base < q1; base += kBatch) {
        const int cnt = min(kBatch, q1 - base);
        __syncthreads();                               // the previous round is read
        for (int e = threadIdx.x; e < cnt * D; e += blockDim.x) {
            const int qi = e / D, c = e % D;
            const int64_t r = h * a.n + a.qlist[base + qi];
            sq[qi][c] = bf(a.q[r * D + c]);
            sdo[qi][c] = bf(a.dout[r * D + c]);
        }
        for (int e = threadIdx.x; e < cnt; e += blockDim.x) {
            const int32_t i = a.qlist[base + e];
            si[e] = i;
            slse[e] = a.lse[h * a.n + i];
            sds[e] = a.dsum[h * a.n + i];
        }
        __syncthreads();
        for (int qi = 0; qi < cnt; ++qi) {
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                s = fmaf(sq[qi][part * 16 + c], kr[c], s);
                dp = fmaf(sdo[qi][part * 16 + c], vr[c], dp);
            }
#pragma unroll
            for (int o = 1; o < G; o <<= 1) {
                s += __shfl_xor_sync(kFull, s, o);
                dp += __shfl_xor_sync(kFull, dp, o);
            }
            const bool adm = live && (!a.causal || j <= si[qi]) && slse[qi] > -INFINITY;
            const float p = adm ? ex2(s * a.scale_log2 - slse[qi]) : 0.f;
            const float ds = p * (dp - sds[qi]);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                dv[c] = fmaf(p, sdo[qi][part * 16 + c], dv[c]);
                dk[c] = fmaf(ds, sq[qi][part * 16 + c], dk[c]);
            }
        }
    }
    if (live) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            a.dk[(h * a.n + j) * D + part * 16 + c] = dk[c] * a.scale;
            a.dv[(h * a.n + j) * D + part * 16 + c] = dv[c];
        }
    }
}

// D_i = dO_i . O_i, one warp per query row (the forward's bf16 output).
template <int D>
__global__ void __launch_bounds__(256) bwd_dsum_kernel(const BwdArgs a) {
    const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= a.bh * a.n) return;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
        const int c = lane + 32 * e;
        s = fmaf(bf(a.dout[row * D + c]), bf(a.out[row * D + c]), s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if (lane == 0) a.dsum[row] = s;
}

// ------------------------------------------------------------------------
// Tensor-core backward for 64-key blocks: one CTA of 128 threads per (head,
// block) -- the queries that listed the block, read from the forward fine
// stage's inversion (one bin per query range), in tiles of 128 rows, one
// thread per row.  Per tile (every product on the tensor cores, bf16 operands
// in 128-byte-swizzled shared memory, fp32 accumulators in tensor memory):
//   S  = Q K_b^T, dP = dO V_b^T                     (M 128, N 64, K d)
//   P  = 2^(S scale log2e - lse_i), dS = scale P (dP - D_i)   (one thread per row)
//   dV_b += P^T dO, dK_b += dS^T Q                  (M 64 keys, N d, K 128 queries:
//                                                    P, dS and dO, Q read MN-major)
//   dQ_i += dS K_b                                   (M 128, N d, K 64; added into dQ
//                                                    with vector atomics, since a
//                                                    query's blocks are different bins)
// dK_b and dV_b stay in tensor memory across the bin's tiles and are written
// once (their rows of an M = 64 accumulator sit in the first 16 lanes of each
// warp's lane quadrant).  lse_i comes from the forward's merge, D_i from
// bwd_dsum_kernel.  Every wait is bounded, and its outcome is combined over
// the CTA at the next barrier so that all threads leave together.
template <int D>
struct BwdTc {
    static constexpr int kSub = D / 64;
    static constexpr int kKB = 64;                       // keys per block
    static constexpr int kRows = 128;
    static constexpr int kKvBytes = kSub * kKB * 128;    // K_b or V_b
    static constexpr int kRowBytes = kSub * kRows * 128; // Q or dO tile
    static constexpr int kPBytes = kRows * 128;          // P or dS tile (64 keys)
    static constexpr int oK = 0, oV = oK + kKvBytes, oQ = oV + kKvBytes, oDo = oQ + kRowBytes;
    static constexpr int oP = oDo + kRowBytes, oDs = oP + kPBytes, oBar = oDs + kPBytes;
    static constexpr int kSmem = oBar + 64 + 1024;
    // tensor memory: S and dP, dQ over them once they are read; dK and dV
    static constexpr uint32_t cS = 0, cDp = 64, cDq = 0, cDk = 128, cDv = 128 + D;
    static constexpr uint32_t kCols = D == 64 ? 256 : 512;
    static_assert(cDv + D <= kCols, "tensor memory");
};

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// Row r of a [rows][64-column sub-tiles] bf16 tile in the 128-byte-swizzled
// K-major layout: 16-byte chunk c of row r at chunk c ^ (r & 7).
__device__ __forceinline__ uint8_t *swz(uint8_t *tile, int r, int c) {
    return tile + r * 128 + ((c ^ (r & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(128) bwd_tc_kernel(const BwdArgs a) {
    using C = BwdTc<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = tc::align_smem_1024(smem_raw);
    uint64_t *bar_s = reinterpret_cast<uint64_t *>(sm + C::oBar);
    uint64_t *bar_g = bar_s + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_s + 2);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t h = blockIdx.y, b = blockIdx.x;
    int32_t nq = 0;                                      // pairs over all query ranges
    for (int64_t r = 0; r < a.nranges; ++r) {
        const int64_t bin = (h * a.nranges + r) * a.nb + b;
        nq += a.bin_offsets[bin + 1] - a.bin_offsets[bin];
    }
    const int64_t j0 = b * C::kKB;
    const int kv_all = int(i64min(C::kKB, a.n - j0));    // keys of the block inside the sequence
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    if (nq == 0) {
        // no query listed the block: its gradients are zero
        const int kr = t >> 1, half = t & 1;
        if (kr < kv_all) {
            float *dk = a.dk + (h * a.n + j0 + kr) * D + half * (D / 2);
            float *dv = a.dv + (h * a.n + j0 + kr) * D + half * (D / 2);
            for (int c = 0; c < D / 2; c += 4) {
                *reinterpret_cast<float4 *>(dk + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(dv + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        return;
    }
    if (t == 0) {
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_g, 1);
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, C::kCols);
        tc::tmem_relinquish();
    }
    // K_b and V_b rows (threads 0-63 and 64-127); keys past the sequence read as zeros
    {
        const int r = t & 63;
        const bool is_v = t >= 64;
        const bool ok = r < kv_all;
        const uint16_t *src = (is_v ? a.vp : a.kp) + (h * a.n + j0 + (ok ? r : 0)) * D;
        uint8_t *dst = sm + (is_v ? C::oV : C::oK);
#pragma unroll
        for (int sub = 0; sub < C::kSub; ++sub)
#pragma unroll
            for (int c = 0; c < 8; ++c)
                tc::cp_async16_zfill(swz(dst + sub * C::kKB * 128, r, c), src + sub * 64 + c * 8, ok);
    }
    tc::cp_async_commit();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t aK = tc::smem_u32(sm + C::oK), aV = tc::smem_u32(sm + C::oV);
    const uint32_t aQ = tc::smem_u32(sm + C::oQ), aDo = tc::smem_u32(sm + C::oDo);
    const uint32_t aP = tc::smem_u32(sm + C::oP), aDs = tc::smem_u32(sm + C::oDs);
    constexpr uint32_t id_sdp = tc::idesc_bf16_f32(C::kRows, C::kKB);
    // dV, dK: A (P or dS transposed) and B (dO or Q) both stored N- / M-contiguous
    constexpr uint32_t id_kv = tc::idesc_bf16_f32(C::kKB, D, /*b_mn_major=*/true) | (1u << 15);
    constexpr uint32_t id_q = tc::idesc_bf16_f32(C::kRows, D, /*b_mn_major=*/true);
    bool ok = true;
    int tile = 0;
    int64_t r = 0;
    int32_t e0 = 0, cnt_r = 0, base = 0;                 // current bin and its next tile
    for (;; ++tile, base += C::kRows) {
        while (base >= cnt_r && r < a.nranges) {         // next bin with pairs left
            const int64_t bin = (h * a.nranges + r) * a.nb + b;
            e0 = a.bin_offsets[bin];
            cnt_r = a.bin_offsets[bin + 1] - e0;
            base = 0;
            ++r;
        }
        if (base >= cnt_r) break;
        // ---- this row's query, its Q and dO rows, lse and D
        const int rr = base + t;
        const bool live = rr < cnt_r;
        const int64_t qrow = live ? int64_t(a.entries[e0 + rr] >> 5) : h * a.n;   // flat row
        const int32_t i = int32_t(qrow - h * a.n);
        {
            const uint16_t *sq = a.q + qrow * D, *sdo = a.dout + qrow * D;
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    tc::cp_async16_zfill(swz(sm + C::oQ + sub * C::kRows * 128, t, c), sq + sub * 64 + c * 8, live);
                    tc::cp_async16_zfill(swz(sm + C::oDo + sub * C::kRows * 128, t, c), sdo + sub * 64 + c * 8, live);
                }
        }
        const float lse = live ? a.lse[qrow] : -INFINITY;
        const float dsum = live ? a.dsum[qrow] : 0.f;
        int kv = kv_all;
        if (a.causal) kv = int(i64min(kv, int64_t(i) - j0 + 1));   // keys j <= i
        if (!live || !(lse > -INFINITY)) kv = 0;                      // the row adds nothing
        tc::cp_async_wait_all();
        tc::fence_proxy_async_smem();            // cp.async writes -> the MMAs' reads
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
        // ---- S and dP
        if (t == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t oq = uint32_t((kk >> 2) * C::kRows * 128 + (kk & 3) * 32);
                const uint32_t ok_ = uint32_t((kk >> 2) * C::kKB * 128 + (kk & 3) * 32);
                tc::mma_bf16(tmem + C::cS, tc::smem_desc_sw128(aQ + oq, 1024), tc::smem_desc_sw128(aK + ok_, 1024),
                             id_sdp, kk > 0);
                tc::mma_bf16(tmem + C::cDp, tc::smem_desc_sw128(aDo + oq, 1024), tc::smem_desc_sw128(aV + ok_, 1024),
                             id_sdp, kk > 0);
            }
            tc::mma_commit(bar_s);
        }
        ok = tc::mbar_wait(bar_s, uint32_t(tile) & 1, a.status);
        // ---- P and dS, one row per thread
        if (ok) {
            tc::tc_fence_after();
            uint32_t sv[2][32], dpv[2][32];
            tc::tmem_ld32(tmem + C::cS + lane_off, sv[0]);
            tc::tmem_ld32(tmem + C::cS + 32 + lane_off, sv[1]);
            tc::tmem_ld32(tmem + C::cDp + lane_off, dpv[0]);
            tc::tmem_ld32(tmem + C::cDp + 32 + lane_off, dpv[1]);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t pk[4], dk[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float p2[2], d2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c = c8 * 8 + e + u;
                        const float sc = __uint_as_float(sv[c >> 5][c & 31]);
                        const float dp = __uint_as_float(dpv[c >> 5][c & 31]);
                        const float p = c < kv ? ex2(fmaf(sc, a.scale_log2, -lse)) : 0.f;
                        p2[u] = p;
                        d2[u] = p * (dp - dsum) * a.scale;
                    }
                    pk[e >> 1] = pack_bf16x2(p2[0], p2[1]);
                    dk[e >> 1] = pack_bf16x2(d2[0], d2[1]);
                }
                *reinterpret_cast<uint4 *>(swz(sm + C::oP, t, c8)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(swz(sm + C::oDs, t, c8)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
            }
        }
        tc::fence_proxy_async_smem();            // P, dS stores -> the MMAs' reads
        tc::tc_fence_before();
        if (!__syncthreads_and(ok)) {            // S and dP read; P and dS written
            ok = false;
            break;
        }
        tc::tc_fence_after();
        // ---- dV += P^T dO, dK += dS^T Q, dQ = dS K_b
        if (t == 0) {
#pragma unroll
            for (int kq = 0; kq < C::kRows / 16; ++kq) {
                const uint32_t off = uint32_t(kq * 2048);       // 16 query rows
                const uint32_t acc = (tile > 0 || kq > 0) ? 1u : 0u;
                tc::mma_bf16(tmem + C::cDv, tc::smem_desc_sw128_mn(aP + off, 8192, 1024),
                             tc::smem_desc_sw128_mn(aDo + off, C::kRows * 128, 1024), id_kv, acc);
                tc::mma_bf16(tmem + C::cDk, tc::smem_desc_sw128_mn(aDs + off, 8192, 1024),
                             tc::smem_desc_sw128_mn(aQ + off, C::kRows * 128, 1024), id_kv, acc);
            }
#pragma unroll
            for (int kk = 0; kk < C::kKB / 16; ++kk)
                tc::mma_bf16(tmem + C::cDq, tc::smem_desc_sw128(aDs + uint32_t(kk * 32), 1024),
                             tc::smem_desc_sw128_mn(aK + uint32_t(kk * 2048), C::kKB * 128, 1024), id_q, kk > 0);
            tc::mma_commit(bar_g);
        }
        ok = tc::mbar_wait(bar_g, uint32_t(tile) & 1, a.status);
        // ---- dQ of this row into the global sum
        if (ok) {
            tc::tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + C::cDq + uint32_t(c0) + lane_off, v);
                tc::tmem_ld_wait();
                if (kv > 0) {
                    float *dst = a.dq + qrow * D + c0;
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        red_add_v4(dst + c, __uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                                   __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
                }
            }
        }
        tc::tc_fence_before();
        if (!__syncthreads_and(ok)) {            // dQ read; next tile may overwrite
            ok = false;
            break;
        }
    }
    // ---- dK_b and dV_b: row kr of the M = 64 accumulators is lane 32 (kr / 16) + kr % 16
    if (ok) {
        tc::tc_fence_after();
        const int kr = warp * 16 + lane;
        const bool mine = lane < 16 && kr < kv_all;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t vk[32], vv[32];
            tc::tmem_ld32(tmem + C::cDk + uint32_t(c0) + lane_off, vk);
            tc::tmem_ld32(tmem + C::cDv + uint32_t(c0) + lane_off, vv);
            tc::tmem_ld_wait();
            if (mine) {
                float *dk = a.dk + (h * a.n + j0 + kr) * D + c0;
                float *dv = a.dv + (h * a.n + j0 + kr) * D + c0;
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    *reinterpret_cast<float4 *>(dk + c) = make_float4(
                        __uint_as_float(vk[c]), __uint_as_float(vk[c + 1]), __uint_as_float(vk[c + 2]),
                        __uint_as_float(vk[c + 3]));
                    *reinterpret_cast<float4 *>(dv + c) = make_float4(
                        __uint_as_float(vv[c]), __uint_as_float(vv[c + 1]), __uint_as_float(vv[c + 2]),
                        __uint_as_float(vv[c + 3]));
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, C::kCols);
    }
}

template <int D>
cudaError_t launch_tc_d(const BwdArgs &a, cudaStream_t st) {
    const int64_t rows = a.bh * a.n;
    bwd_dsum_kernel<D><<<unsigned((rows + 7) / 8), 256, 0, st>>>(a);
    cudaError_t e = cudaMemsetAsync(a.dq, 0, size_t(rows) * D * sizeof(float), st);
    if (e != cudaSuccess) return e;
    auto kern = bwd_tc_kernel<D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdTc<D>::kSmem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(unsigned(a.nb), unsigned(a.bh)), 128, BwdTc<D>::kSmem, st>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const BwdArgs &a, cudaStream_t st) {
    const dim3 gq(unsigned((a.n + kQWarps - 1) / kQWarps), unsigned(a.bh));
    bwd_query_kernel<D><<<gq, kQWarps * 32, 0, st>>>(a);
    const dim3 ge(unsigned((a.n * a.k + 255) / 256), unsigned(a.bh));
    bwd_count_kernel<<<ge, 256, 0, st>>>(a);
    bwd_scan_kernel<<<1, kScanThreads, 0, st>>>(a);
    bwd_scatter_kernel<<<ge, 256, 0, st>>>(a);
    bwd_kv_kernel<D><<<dim3(unsigned(a.nb), unsigned(a.bh)), unsigned(a.kb * (D / 16)), 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool fine_backward_supported(int32_t d, int32_t kb) {
    return (d == 64 || d == 128) && kb * (d / 16) <= 512;
}

bool fine_backward_tc_supported(int32_t d, int32_t kb, int32_t k) {
    return (d == 64 || d == 128) && kb == 64 && k >= 1 && k <= 32;
}

cudaError_t launch_fine_backward_tc(const BwdArgs &a, cudaStream_t st) {
    if (!fine_backward_tc_supported(a.d, a.kb, a.k)) return cudaErrorInvalidValue;
    return a.d == 64 ? launch_tc_d<64>(a, st) : launch_tc_d<128>(a, st);
}

cudaError_t launch_fine_backward(const BwdArgs &a, cudaStream_t st) {
    if (!fine_backward_supported(a.d, a.kb)) return cudaErrorInvalidValue;
    if (a.d == 64) return launch_d<64>(a, st);
    if (a.d == 128) return launch_d<128>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace bsa
