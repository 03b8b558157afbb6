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

cudaError_t launch_fine_backward(const BwdArgs &a, cudaStream_t st) {
    if (!fine_backward_supported(a.d, a.kb)) return cudaErrorInvalidValue;
    if (a.d == 64) return launch_d<64>(a, st);
    if (a.d == 128) return launch_d<128>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace bsa
