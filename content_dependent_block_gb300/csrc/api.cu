// C-ABI layer of libbsa.so: argument validation, workspace carving and the
// launch sequence of every entry point declared in include/bsa.h.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

constexpr int32_t kVersion = 100;   // 0.1.0
constexpr int kMaxDevices = 64;

thread_local char g_last_error[256] = "";

bsa_status fail(bsa_status code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

bsa_status ok() {
    g_last_error[0] = '\0';
    return BSA_OK;
}

// Device status word: first kernel-detected error since the last read.
__device__ int32_t g_device_status = 0;

int32_t *device_status_ptr() {
    static std::mutex mu;
    static int32_t *cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int32_t *>(p);
    }
    return cache[dev];
}

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bsa_status check_shape(const bsa_shape &s) {
    if (s.bh < 1 || s.n < 1) return fail(BSA_ERR_INVALID_ARG, "bh and n must be >= 1");
    if (s.bh > 65535) return fail(BSA_ERR_UNSUPPORTED, "bh must be <= 65535");
    if (s.n > (int64_t(1) << 31) - 1) return fail(BSA_ERR_UNSUPPORTED, "n must fit in int32");
    if (s.d != 64 && s.d != 128) return fail(BSA_ERR_UNSUPPORTED, "d must be 64 or 128 (got %d)", s.d);
    if (s.dtype != BSA_BF16 && s.dtype != BSA_FP32) return fail(BSA_ERR_INVALID_ARG, "bad dtype %d", s.dtype);
    return BSA_OK;
}

bsa_status check_key_block(int32_t kb) {
    if (kb != 16 && kb != 32 && kb != 64 && kb != 128)
        return fail(BSA_ERR_UNSUPPORTED, "key_block must be 16, 32, 64 or 128 (got %d)", kb);
    return BSA_OK;
}

bsa_status check_ptr(const void *p, const char *name) {
    if (p == nullptr) return fail(BSA_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, 16)) return fail(BSA_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
    return BSA_OK;
}

bsa_status check_ws(const void *ws, size_t have, size_t need) {
    if (need == 0) return BSA_OK;
    if (ws == nullptr || have < need)
        return fail(BSA_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, ws ? have : size_t(0));
    if (!aligned(ws, 256)) return fail(BSA_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
    return BSA_OK;
}

bsa_status launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

#define BSA_TRY(expr)                      \
    do {                                   \
        bsa_status st_ = (expr);           \
        if (st_ != BSA_OK) return st_;     \
    } while (0)

// Workspace of the whole forward: fp32 block means, their bf16 hi/lo pair
// (tensor-core scoring), then the selection.
struct ForwardLayout {
    size_t kbar = 0, hi = 0, lo = 0, idx = 0, total = 0;
};

ForwardLayout forward_layout(const bsa_shape &s, int32_t kb, int32_t topk) {
    ForwardLayout L;
    const int64_t nb = ceil_div(s.n, kb);
    const size_t means = size_t(s.bh) * nb * s.d;
    size_t off = 0;
    L.kbar = off;
    off = round_up(off + means * sizeof(float), 256);
    L.hi = off;
    off = round_up(off + means * sizeof(uint16_t), 256);
    L.lo = off;
    off = round_up(off + means * sizeof(uint16_t), 256);
    L.idx = off;
    off = round_up(off + size_t(s.bh) * s.n * topk * sizeof(int32_t), 256);
    L.total = off;
    return L;
}

// Scoring + selection from fp32 means (and their bf16 pair when present).
cudaError_t run_coarse(const bsa_shape &s, const void *q, const float *kbar, const uint16_t *hi,
                       const uint16_t *lo, int64_t nb, int32_t topk, const bsa::SelectOpts &o,
                       int32_t *idx, int32_t *status, cudaStream_t st) {
    if (hi != nullptr && bsa::coarse_tc_supported(nb))
        return bsa::launch_coarse_topk_tc(q, hi, lo, s.bh, s.n, s.d, nb, topk, o, idx, status, st);
    return bsa::launch_coarse_topk_simt(q, kbar, s.bh, s.n, s.d, nb, topk, o, idx, status, st);
}

// The selection options of `sel` (NULL: none) for blocks of kb tokens.
bsa::SelectOpts select_opts(const bsa_select *sel, int32_t kb) {
    bsa::SelectOpts o;
    o.kb = kb;
    if (sel != nullptr) {
        o.head_k = sel->head_topk;
        o.causal = sel->causal ? 1 : 0;
        o.local = sel->local_block ? 1 : 0;
    }
    return o;
}

bool has_options(const bsa::SelectOpts &o) { return o.head_k != nullptr || o.causal || o.local; }

bsa_status check_select(const bsa_select *sel) {
    if (sel != nullptr && sel->head_topk != nullptr && !aligned(sel->head_topk, 4))
        return fail(BSA_ERR_ALIGNMENT, "head_topk is not 4-byte aligned");
    return BSA_OK;
}

// Workspace of the block-major fine stage over per-query lists [bh][n][k].
struct BmLayout {
    bsa::InvertPlan plan;
    size_t zero = 0, zero_bytes = 0;     // counts, cursors, queue heads, range counters
    size_t counts = 0, cursors = 0, fine_head = 0, merge_head = 0, range_done = 0, merge_done = 0;
    size_t offsets = 0, fitem_off = 0, fpre = 0, mpre = 0, range_total = 0, range_merges = 0;
    size_t n_fine = 0, n_merge = 0, fine_items = 0, merge_items = 0, entries = 0, vmask = 0;
    size_t part_o = 0, part_lse = 0, total = 0;
};

BmLayout bm_layout(const bsa_shape &s, int32_t kb, int32_t k, size_t base) {
    BmLayout L;
    const int64_t nb = ceil_div(s.n, kb);
    L.plan = bsa::invert_plan(s.bh, s.n, nb, k);
    const size_t nbins = size_t(L.plan.nbins), nr = size_t(L.plan.nr);
    // as many query ranges in flight as fit the byte budget (a range's
    // partial states: range x kpad x (2d + 8) bytes): a power of two in
    // [4, 16], so that the kernel finds a range's entry with a mask
    const int64_t range_bytes = L.plan.range * L.plan.kpad * (2 * int64_t(s.d) + 8);
    int32_t ring = bsa::kPartialRing;
    while (ring < bsa::kPartialRingMax && 2 * ring * range_bytes <= bsa::kPartialRingBytes &&
           ring < L.plan.nr)
        ring *= 2;
    L.plan.ring = ring;
    const size_t ring_slots = size_t(L.plan.ring) * size_t(L.plan.range) * size_t(L.plan.kpad);
    size_t off = base;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 16);
        return at;
    };
    L.zero = off;
    L.counts = take(nbins * 4);
    L.cursors = take(nbins * 4);
    L.fine_head = take(4);
    L.merge_head = take(4);
    L.range_done = take(nr * 4);
    L.merge_done = take(nr * 4);
    L.zero_bytes = off - L.zero;
    off = round_up(off, 256);
    L.offsets = take((nbins + 1) * 4);
    L.fitem_off = take((nbins + 1) * 4);
    L.fpre = take((nr + 2) * 4);
    L.mpre = take((nr + 1) * 4);
    L.range_total = take(nr * 4);
    L.range_merges = take(nr * 4);
    L.n_fine = take(4);
    L.n_merge = take(4);
    L.fine_items = take(size_t(L.plan.fine_cap) * sizeof(int2));
    L.merge_items = take(size_t(L.plan.merge_cap) * sizeof(int2));
    L.entries = take(size_t(s.bh) * s.n * k * 4);
    L.vmask = take(size_t(s.bh) * s.n * 4);
    off = round_up(off, 256);
    L.part_o = take(ring_slots * s.d * 2);
    off = round_up(off, 256);
    L.part_lse = take(ring_slots * 8);
    L.total = round_up(off, 256);
    return L;
}

bool bm_path(const bsa_shape &s, int32_t kb, int64_t nb) {
    return s.dtype == BSA_BF16 && bsa::fine_bm_supported(s.d, kb) && nb <= 16384 &&
           s.bh * s.n * int64_t(32) < (int64_t(1) << 31);
}

// The lists' inversion and the block-major stage's work lists (count ->
// scan -> scatter) into the workspace at L; rows whose list admits nothing
// get zeros in out.
cudaError_t run_invert_bm(const bsa_shape &s, const int32_t *list, int32_t kb, int32_t topk,
                          void *out, char *ws, const BmLayout &L, int32_t *status,
                          cudaStream_t st, bsa::InvertBuffers &w) {
    const int64_t nb = ceil_div(s.n, kb);
    cudaError_t e = cudaMemsetAsync(ws + L.zero, 0, L.zero_bytes, st);
    if (e != cudaSuccess) return e;
    w = bsa::InvertBuffers{};
    w.counts = reinterpret_cast<int32_t *>(ws + L.counts);
    w.cursors = reinterpret_cast<int32_t *>(ws + L.cursors);
    w.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    w.fitem_off = reinterpret_cast<int32_t *>(ws + L.fitem_off);
    w.fpre = reinterpret_cast<int32_t *>(ws + L.fpre);
    w.mpre = reinterpret_cast<int32_t *>(ws + L.mpre);
    w.range_total = reinterpret_cast<int32_t *>(ws + L.range_total);
    w.range_merges = reinterpret_cast<int32_t *>(ws + L.range_merges);
    w.fine_items = reinterpret_cast<int2 *>(ws + L.fine_items);
    w.merge_items = reinterpret_cast<int2 *>(ws + L.merge_items);
    w.n_fine = reinterpret_cast<int32_t *>(ws + L.n_fine);
    w.n_merge = reinterpret_cast<int32_t *>(ws + L.n_merge);
    w.entries = reinterpret_cast<int32_t *>(ws + L.entries);
    w.vmask = reinterpret_cast<uint32_t *>(ws + L.vmask);
    return bsa::launch_invert(list, s.bh, s.n, nb, topk, L.plan, w, static_cast<uint16_t *>(out),
                              s.d, status, st);
}

// Invert the lists and run the block-major fine stage; ws points at L.
cudaError_t run_fine_bm(const bsa_shape &s, const void *q, const void *k, const void *v,
                        const int32_t *list, int32_t kb, int32_t topk, bool full_lists,
                        bool causal, const bsa::SelectOpts *sel, float scale_log2, void *out,
                        char *ws, const BmLayout &L, int32_t *status, cudaStream_t st,
                        float *lse_out = nullptr) {
    const int64_t nb = ceil_div(s.n, kb);
    bsa::InvertBuffers w{};
    cudaError_t e = run_invert_bm(s, list, kb, topk, out, ws, L, status, st, w);
    if (e != cudaSuccess) return e;
    bsa::FineBmArgs a{};
    a.k_ptr = k;
    a.v_ptr = v;
    a.q = static_cast<const uint16_t *>(q);
    a.list = list;
    a.w = w;
    a.p = L.plan;
    a.fine_head = reinterpret_cast<int32_t *>(ws + L.fine_head);
    a.merge_head = reinterpret_cast<int32_t *>(ws + L.merge_head);
    a.range_done = reinterpret_cast<int32_t *>(ws + L.range_done);
    a.merge_done = reinterpret_cast<int32_t *>(ws + L.merge_done);
    a.bh = s.bh;
    a.n = s.n;
    a.nb = nb;
    a.d = s.d;
    a.k = topk;
    a.full_lists = full_lists ? 1 : 0;
    a.causal = causal ? 1 : 0;
    a.sel_lists = sel != nullptr ? 1 : 0;
    a.head_k = sel != nullptr ? sel->head_k : nullptr;
    a.scale_log2 = scale_log2;
    a.part_o = reinterpret_cast<uint16_t *>(ws + L.part_o);
    a.part_ml = reinterpret_cast<float2 *>(ws + L.part_lse);
    a.out = static_cast<uint16_t *>(out);
    a.lse_out = lse_out;
    a.status = status;
    return bsa::launch_fine_bm(a, st);
}

float softmax_scale_log2(float scale, int32_t d) {
    const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(float(d));
    return sc * 1.4426950408889634f;   // log2(e)
}

}  // namespace

namespace bsa {
void set_last_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }
}  // namespace bsa

extern "C" {

int32_t bsa_version(void) { return kVersion; }

const char *bsa_last_error(void) { return g_last_error; }

const char *bsa_status_string(int32_t status) {
    switch (status) {
        case BSA_OK: return "ok";
        case BSA_ERR_INVALID_ARG: return "invalid argument";
        case BSA_ERR_UNSUPPORTED: return "unsupported configuration";
        case BSA_ERR_BAD_INDEX: return "block index out of range";
        case BSA_ERR_WORKSPACE: return "workspace missing or too small";
        case BSA_ERR_CUDA: return "CUDA runtime error";
        case BSA_ERR_TIMEOUT: return "device wait timed out";
        case BSA_ERR_ALIGNMENT: return "misaligned pointer";
        default: return "unknown status";
    }
}

bsa_status bsa_get_device_status(int32_t *status, void *stream) {
    if (status == nullptr) return fail(BSA_ERR_INVALID_ARG, "status is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
    int32_t *p = device_status_ptr();
    if (p == nullptr) return fail(BSA_ERR_CUDA, "status word unavailable");
    int32_t v = 0;
    e = cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof v);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
    *status = v;
    return ok();
}

bsa_status bsa_pool_blocks(bsa_shape shape, const void *k, int32_t key_block, float *kbar,
                           void *stream) {
    BSA_TRY(check_shape(shape));
    if (shape.dtype != BSA_BF16) return fail(BSA_ERR_UNSUPPORTED, "pooling takes bf16 keys");
    BSA_TRY(check_key_block(key_block));
    BSA_TRY(check_ptr(k, "k"));
    BSA_TRY(check_ptr(kbar, "kbar"));
    return launched(bsa::launch_pool(k, shape.bh, shape.n, shape.d, key_block, kbar, nullptr,
                                     nullptr, 0, static_cast<cudaStream_t>(stream)),
                    "pool launch");
}

size_t bsa_coarse_topk_workspace_size(bsa_shape shape, int32_t key_block, int32_t) {
    if (check_shape(shape) != BSA_OK || check_key_block(key_block) != BSA_OK) return 0;
    const int64_t nb = ceil_div(shape.n, key_block);
    if (!bsa::coarse_tc_supported(nb)) return 0;
    const size_t half = round_up(size_t(shape.bh) * nb * shape.d * sizeof(uint16_t), 256);
    return 2 * half;   // bf16 hi / lo copies of the block means
}

bsa_status bsa_coarse_topk(bsa_shape shape, const void *q, const float *kbar, int32_t key_block,
                           int32_t topk, int32_t *idx, void *ws, size_t ws_bytes, void *stream) {
    return bsa_coarse_topk_ex(shape, q, kbar, key_block, topk, nullptr, idx, ws, ws_bytes, stream);
}

bsa_status bsa_coarse_topk_ex(bsa_shape shape, const void *q, const float *kbar, int32_t key_block,
                              int32_t topk, const bsa_select *sel, int32_t *idx, void *ws,
                              size_t ws_bytes, void *stream) {
    BSA_TRY(check_shape(shape));
    if (shape.dtype != BSA_BF16) return fail(BSA_ERR_UNSUPPORTED, "scoring takes bf16 queries");
    BSA_TRY(check_key_block(key_block));
    if (topk < 1 || topk > 32) return fail(BSA_ERR_UNSUPPORTED, "topk must be in [1, 32] (got %d)", topk);
    BSA_TRY(check_ptr(q, "q"));
    BSA_TRY(check_ptr(kbar, "kbar"));
    BSA_TRY(check_ptr(idx, "idx"));
    BSA_TRY(check_select(sel));
    const size_t need = bsa_coarse_topk_workspace_size(shape, key_block, topk);
    BSA_TRY(check_ws(ws, ws_bytes, need));
    const int64_t nb = ceil_div(shape.n, key_block);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *status = device_status_ptr();
    if (status == nullptr) return fail(BSA_ERR_CUDA, "status word unavailable");
    uint16_t *hi = nullptr, *lo = nullptr;
    if (need > 0) {
        hi = static_cast<uint16_t *>(ws);
        lo = reinterpret_cast<uint16_t *>(static_cast<char *>(ws) + need / 2);
        BSA_TRY(launched(bsa::launch_split_kbar(kbar, shape.bh * nb * shape.d, hi, lo, st),
                         "split launch"));
    }
    return launched(run_coarse(shape, q, kbar, hi, lo, nb, topk, select_opts(sel, key_block), idx,
                               status, st),
                    "coarse top-k launch");
}

// Per-query lists (q_group = 1, one list per head, no mask or the causal
// one) of bf16 inputs with 64-token blocks take the block-major tensor-core
// schedule; everything else (static tile lists, fp32, other block sizes) the
// query-major kernel.
bool bm_lists(const bsa_shape &shape, const bsa_list_desc &ld, const bsa_mask &mask) {
    return ld.q_group == 1 && ld.per_head &&
           (mask.kind == BSA_MASK_NONE || mask.kind == BSA_MASK_CAUSAL) && ld.max_blocks >= 1 &&
           ld.max_blocks <= 32 && bm_path(shape, ld.key_block, ceil_div(shape.n, ld.key_block));
}

bool fine_uses_bm(const bsa_shape &shape, const int32_t *list, const bsa_list_desc &ld,
                  const bsa_mask &mask) {
    return list != nullptr && bm_lists(shape, ld, mask);
}

size_t bsa_fine_attention_workspace_size(bsa_shape shape, bsa_list_desc ld, bsa_mask mask) {
    if (check_shape(shape) != BSA_OK || check_key_block(ld.key_block) != BSA_OK) return 0;
    // a non-null list is assumed (max_blocks 0 stands for no list)
    if (bm_lists(shape, ld, mask)) return bm_layout(shape, ld.key_block, ld.max_blocks, 0).total;
    // static tile lists on the tensor cores: optional, lets them run one pass
    if (shape.dtype == BSA_BF16 && (shape.d == 64 || shape.d == 128) && ld.key_block == 64 &&
        (ld.q_group == 128 || ld.max_blocks == 0) && ld.max_blocks <= 512 && shape.bh <= 65535)
        return bsa::fine_static_tc_workspace(shape.bh, shape.n, ld.key_block);
    return 0;   // the query-major path needs none
}

namespace {

// bsa_fine_attention, with each row's log2-sum-exp into lse_out (non-NULL
// only on the block-major path)
bsa_status fine_attention_impl(bsa_shape shape, const void *q, const void *k, const void *v,
                               const int32_t *list, bsa_list_desc ld, bsa_mask mask, float scale,
                               void *out, float *lse_out, void *ws, size_t ws_bytes, void *stream) {
    BSA_TRY(check_shape(shape));
    BSA_TRY(check_key_block(ld.key_block));
    BSA_TRY(check_ptr(q, "q"));
    BSA_TRY(check_ptr(k, "k"));
    BSA_TRY(check_ptr(v, "v"));
    BSA_TRY(check_ptr(out, "out"));
    if (list != nullptr) {
        if (!aligned(list, 4)) return fail(BSA_ERR_ALIGNMENT, "list is not 4-byte aligned");
        if (ld.q_group < 1 || ld.max_blocks < 1)
            return fail(BSA_ERR_INVALID_ARG, "list needs q_group >= 1 and max_blocks >= 1");
    }
    if (mask.kind < BSA_MASK_NONE || mask.kind > BSA_MASK_CAUSAL)
        return fail(BSA_ERR_INVALID_ARG, "bad mask kind %d", mask.kind);
    if (mask.kind == BSA_MASK_SLIDING && mask.sliding < 1)
        return fail(BSA_ERR_INVALID_ARG, "sliding window needs W >= 1");
    const bool bm = fine_uses_bm(shape, list, ld, mask);
    const size_t need = bm ? bsa_fine_attention_workspace_size(shape, ld, mask) : 0;
    BSA_TRY(check_ws(ws, ws_bytes, need));
    int32_t *status = device_status_ptr();
    if (status == nullptr) return fail(BSA_ERR_CUDA, "status word unavailable");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const float sl2 = softmax_scale_log2(scale, shape.d);
    if (bm) {
        const BmLayout L = bm_layout(shape, ld.key_block, ld.max_blocks, 0);
        return launched(run_fine_bm(shape, q, k, v, list, ld.key_block, ld.max_blocks, false,
                                    mask.kind == BSA_MASK_CAUSAL, nullptr, sl2, out,
                                    static_cast<char *>(ws), L, status, st, lse_out),
                        "fine attention (block-major) launch");
    }
    bsa::FineArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.list = list;
    a.bh = shape.bh;
    a.n = shape.n;
    a.kb = ld.key_block;
    a.nb = ceil_div(shape.n, ld.key_block);
    a.d = shape.d;
    a.q_group = list ? ld.q_group : 1;
    a.max_blocks = list ? ld.max_blocks : 0;
    a.per_head = ld.per_head ? 1 : 0;
    a.list_rows = ceil_div(shape.n, a.q_group);
    a.mask_kind = mask.kind;
    a.window = mask.window;
    a.stride = mask.stride;
    a.sliding = mask.sliding;
    a.scale_log2 = sl2;
    a.status = status;
    if (bsa::fine_static_tc_supported(a, shape.dtype)) {
        // with the optional workspace: block key norms, then one pass with a score bound
        const size_t need_s = bsa::fine_static_tc_workspace(shape.bh, shape.n, ld.key_block);
        if (ws != nullptr && ws_bytes >= need_s && aligned(ws, 256)) {
            a.kmax = static_cast<float *>(ws);
            a.flags = reinterpret_cast<int32_t *>(static_cast<char *>(ws) +
                                                  round_up(size_t(shape.bh) * size_t(a.nb) * 4, 256));
        }
        return launched(bsa::launch_fine_static_tc(a, st), "fine attention (tensor-core tiles) launch");
    }
    return launched(bsa::launch_fine_query_major(a, shape.dtype, st), "fine attention launch");
}

}  // namespace

bsa_status bsa_fine_attention(bsa_shape shape, const void *q, const void *k, const void *v,
                              const int32_t *list, bsa_list_desc ld, bsa_mask mask, float scale,
                              void *out, void *ws, size_t ws_bytes, void *stream) {
    return fine_attention_impl(shape, q, k, v, list, ld, mask, scale, out, nullptr, ws, ws_bytes,
                               stream);
}

bsa_status bsa_fine_attention_lse(bsa_shape shape, const void *q, const void *k, const void *v,
                                  const int32_t *list, bsa_list_desc ld, bsa_mask mask,
                                  float scale, void *out, float *lse_out, void *ws,
                                  size_t ws_bytes, void *stream) {
    BSA_TRY(check_shape(shape));
    BSA_TRY(check_key_block(ld.key_block));
    if (lse_out == nullptr) return fail(BSA_ERR_INVALID_ARG, "lse_out is NULL");
    if (!aligned(lse_out, 4)) return fail(BSA_ERR_ALIGNMENT, "lse_out is not 4-byte aligned");
    if (!fine_uses_bm(shape, list, ld, mask))
        return fail(BSA_ERR_UNSUPPORTED,
                    "the log2-sum-exp output needs the block-major path (per-query lists, bf16, "
                    "key_block 64, max_blocks <= 32, no mask or the causal one)");
    return fine_attention_impl(shape, q, k, v, list, ld, mask, scale, out, lse_out, ws, ws_bytes,
                               stream);
}

size_t bsa_forward_workspace_size(bsa_shape shape, int32_t key_block, int32_t topk) {
    if (check_shape(shape) != BSA_OK || check_key_block(key_block) != BSA_OK || topk < 1 ||
        topk > 32)
        return 0;
    const ForwardLayout F = forward_layout(shape, key_block, topk);
    if (!bm_path(shape, key_block, ceil_div(shape.n, key_block))) return F.total;
    return bm_layout(shape, key_block, topk, F.total).total;
}

int32_t bsa_forward_launches(bsa_shape shape, int32_t key_block, int32_t topk) {
    if (check_shape(shape) != BSA_OK || check_key_block(key_block) != BSA_OK || topk < 1 || topk > 32)
        return -int32_t(BSA_ERR_INVALID_ARG);
    // a small problem: one fused launch; else pool (+ hi/lo), score + top-k,
    // then either the query-major fine kernel or count + scan + scatter +
    // block-major fine
    const int64_t nb = ceil_div(shape.n, key_block);
    if (shape.dtype == BSA_BF16 && bsa::small_forward_supported(shape.d, nb, topk, shape.bh * shape.n))
        return 1;
    return bm_path(shape, key_block, nb) ? 6 : 3;
}

bsa_status bsa_forward(bsa_shape shape, const void *q, const void *k, const void *v,
                       int32_t key_block, int32_t topk, float scale, void *out, int32_t *idx_out,
                       void *ws, size_t ws_bytes, void *stream) {
    return bsa_forward_ex(shape, q, k, v, key_block, topk, nullptr, scale, out, idx_out, ws,
                          ws_bytes, stream);
}

namespace {

// bsa_forward_ex; with lse_out the rows' log2-sum-exp too (block-major path)
bsa_status forward_impl(bsa_shape shape, const void *q, const void *k, const void *v,
                        int32_t key_block, int32_t topk, const bsa_select *sel, float scale,
                        void *out, int32_t *idx_out, float *lse_out, void *ws, size_t ws_bytes,
                        void *stream) {
    BSA_TRY(check_shape(shape));
    if (shape.dtype != BSA_BF16) return fail(BSA_ERR_UNSUPPORTED, "the dynamic forward takes bf16");
    BSA_TRY(check_key_block(key_block));
    if (topk < 1 || topk > 32) return fail(BSA_ERR_UNSUPPORTED, "topk must be in [1, 32] (got %d)", topk);
    BSA_TRY(check_ptr(q, "q"));
    BSA_TRY(check_ptr(k, "k"));
    BSA_TRY(check_ptr(v, "v"));
    BSA_TRY(check_ptr(out, "out"));
    if (idx_out != nullptr) BSA_TRY(check_ptr(idx_out, "idx_out"));
    BSA_TRY(check_select(sel));
    if (lse_out != nullptr && !bm_path(shape, key_block, ceil_div(shape.n, key_block)))
        return fail(BSA_ERR_UNSUPPORTED,
                    "the log2-sum-exp output needs the block-major fine stage (key_block 64)");
    const bsa::SelectOpts opts = select_opts(sel, key_block);
    const ForwardLayout L = forward_layout(shape, key_block, topk);
    BSA_TRY(check_ws(ws, ws_bytes, bsa_forward_workspace_size(shape, key_block, topk)));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    float *kbar = reinterpret_cast<float *>(base + L.kbar);
    uint16_t *hi = reinterpret_cast<uint16_t *>(base + L.hi);
    uint16_t *lo = reinterpret_cast<uint16_t *>(base + L.lo);
    int32_t *idx = idx_out ? idx_out : reinterpret_cast<int32_t *>(base + L.idx);
    const int64_t nb = ceil_div(shape.n, key_block);
    int32_t *status = device_status_ptr();
    if (status == nullptr) return fail(BSA_ERR_CUDA, "status word unavailable");
    if (lse_out == nullptr && !has_options(opts) &&
        bsa::small_forward_supported(shape.d, nb, topk, shape.bh * shape.n)) {
        // a small problem: pooling, selection and the fine stage in one launch
        bsa::FineArgs a{};
        a.q = q;
        a.k = k;
        a.v = v;
        a.out = out;
        a.bh = shape.bh;
        a.n = shape.n;
        a.nb = nb;
        a.kb = key_block;
        a.d = shape.d;
        a.mask_kind = BSA_MASK_NONE;
        a.scale_log2 = softmax_scale_log2(scale, shape.d);
        a.status = status;
        return launched(bsa::launch_small_forward(a, topk, idx, st), "fused forward launch");
    }

    BSA_TRY(launched(bsa::launch_pool(k, shape.bh, shape.n, shape.d, key_block, kbar, hi, lo, nb,
                                      st), "pool launch"));
    BSA_TRY(launched(run_coarse(shape, q, kbar, hi, lo, nb, topk, opts, idx, status, st),
                     "coarse top-k launch"));
    const float sl2 = softmax_scale_log2(scale, shape.d);
    if (bm_path(shape, key_block, nb)) {
        const BmLayout B = bm_layout(shape, key_block, topk, L.total);
        // options leave -1 padding (budgets, early causal queries): lists are not full
        return launched(run_fine_bm(shape, q, k, v, idx, key_block, topk, !has_options(opts),
                                    opts.causal != 0, has_options(opts) ? &opts : nullptr, sl2,
                                    out, base, B, status, st, lse_out),
                        "fine attention (block-major) launch");
    }
    bsa::FineArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.list = idx;
    a.bh = shape.bh;
    a.n = shape.n;
    a.kb = key_block;
    a.nb = nb;
    a.d = shape.d;
    a.q_group = 1;
    a.max_blocks = topk;
    a.per_head = 1;
    a.list_rows = shape.n;
    a.mask_kind = opts.causal ? BSA_MASK_CAUSAL : BSA_MASK_NONE;
    a.scale_log2 = sl2;
    a.status = status;
    if (bsa::fine_static_tc_supported(a, shape.dtype))
        return launched(bsa::launch_fine_static_tc(a, st), "fine attention (tensor-core tiles) launch");
    return launched(bsa::launch_fine_query_major(a, shape.dtype, st), "fine attention launch");
}

}  // namespace

bsa_status bsa_forward_ex(bsa_shape shape, const void *q, const void *k, const void *v,
                          int32_t key_block, int32_t topk, const bsa_select *sel, float scale,
                          void *out, int32_t *idx_out, void *ws, size_t ws_bytes, void *stream) {
    return forward_impl(shape, q, k, v, key_block, topk, sel, scale, out, idx_out, nullptr, ws,
                        ws_bytes, stream);
}

bsa_status bsa_forward_lse(bsa_shape shape, const void *q, const void *k, const void *v,
                           int32_t key_block, int32_t topk, const bsa_select *sel, float scale,
                           void *out, int32_t *idx_out, float *lse_out, void *ws, size_t ws_bytes,
                           void *stream) {
    if (lse_out == nullptr) return fail(BSA_ERR_INVALID_ARG, "lse_out is NULL");
    if (!aligned(lse_out, 4)) return fail(BSA_ERR_ALIGNMENT, "lse_out is not 4-byte aligned");
    return forward_impl(shape, q, k, v, key_block, topk, sel, scale, out, idx_out, lse_out, ws,
                        ws_bytes, stream);
}

// ---------------------------------------------------------- backward pass
struct BwdLayout {
    size_t lse = 0, dsum = 0, counts = 0, cursors = 0, offsets = 0, qlist = 0, total = 0;
    size_t o_scratch = 0, fwd = 0;     // tensor-core path only
};

// The tensor-core backward (64-key blocks, at most 32 per query) also runs
// one block-major forward fine stage for the rows' log2-sum-exp: its
// workspace and a scratch output follow the backward's own buffers.
bool bwd_tc_path(const bsa_shape &s, int32_t kb, int32_t k) {
    return bsa::fine_backward_tc_supported(s.d, kb, k) && bm_path(s, kb, ceil_div(s.n, kb));
}

BwdLayout bwd_layout(const bsa_shape &s, int32_t kb, int32_t k) {
    BwdLayout L;
    const size_t rows = size_t(s.bh) * size_t(s.n), bins = size_t(s.bh) * size_t(ceil_div(s.n, kb));
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t o = at;
        at += round_up(bytes, 256);
        return o;
    };
    L.lse = take(rows * 4);
    L.dsum = take(rows * 4);
    if (bwd_tc_path(s, kb, k)) {
        // the forward fine stage's workspace holds the lists' inversion
        L.o_scratch = take(rows * size_t(s.d) * 2);
        L.fwd = at;
        L.total = bm_layout(s, kb, k, at).total;
        return L;
    }
    L.counts = take(bins * 4);
    L.cursors = take(bins * 4);
    L.offsets = take((bins + 1) * 4);
    L.qlist = take(rows * size_t(k) * 4);
    L.total = at;
    return L;
}

bool bwd_lists_ok(const bsa_list_desc &ld) {
    return ld.q_group == 1 && ld.per_head && ld.max_blocks >= 1 && ld.max_blocks <= 64;
}

size_t bsa_fine_backward_workspace_size(bsa_shape shape, bsa_list_desc ld) {
    if (check_shape(shape) != BSA_OK || check_key_block(ld.key_block) != BSA_OK || !bwd_lists_ok(ld))
        return 0;
    return bwd_layout(shape, ld.key_block, ld.max_blocks).total;
}

namespace {

// bsa_fine_backward; with lse_in (the forward's log2-sum-exp per row) the
// tensor-core path inverts the lists and skips the statistics pass
bsa_status fine_backward_impl(bsa_shape shape, const void *q, const void *k, const void *v,
                              const void *out, const void *dout, const int32_t *list,
                              bsa_list_desc ld, bsa_mask mask, float scale, const float *lse_in,
                              float *dq, float *dk, float *dv, void *ws, size_t ws_bytes,
                              void *stream) {
    BSA_TRY(check_shape(shape));
    if (shape.dtype != BSA_BF16) return fail(BSA_ERR_UNSUPPORTED, "the backward pass takes bf16");
    BSA_TRY(check_key_block(ld.key_block));
    if (!bwd_lists_ok(ld))
        return fail(BSA_ERR_UNSUPPORTED,
                    "the backward pass takes per-query lists (q_group 1, per head, 1..64 blocks)");
    if (mask.kind != BSA_MASK_NONE && mask.kind != BSA_MASK_CAUSAL)
        return fail(BSA_ERR_UNSUPPORTED, "the backward pass takes no mask or the causal one");
    if (!bsa::fine_backward_supported(shape.d, ld.key_block))
        return fail(BSA_ERR_UNSUPPORTED, "the backward pass takes d 64 or 128 and key_block * d <= 8192");
    BSA_TRY(check_ptr(q, "q"));
    BSA_TRY(check_ptr(k, "k"));
    BSA_TRY(check_ptr(v, "v"));
    BSA_TRY(check_ptr(out, "out"));
    BSA_TRY(check_ptr(dout, "dout"));
    BSA_TRY(check_ptr(dq, "dq"));
    BSA_TRY(check_ptr(dk, "dk"));
    BSA_TRY(check_ptr(dv, "dv"));
    if (list == nullptr) return fail(BSA_ERR_INVALID_ARG, "list is NULL");
    if (!aligned(list, 4)) return fail(BSA_ERR_ALIGNMENT, "list is not 4-byte aligned");
    const BwdLayout L = bwd_layout(shape, ld.key_block, ld.max_blocks);
    BSA_TRY(check_ws(ws, ws_bytes, L.total));
    int32_t *status = device_status_ptr();
    if (status == nullptr) return fail(BSA_ERR_CUDA, "status word unavailable");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    const bool tc_path = bwd_tc_path(shape, ld.key_block, ld.max_blocks);
    cudaError_t e = cudaSuccess;
    if (!tc_path) {
        // counts and cursors are adjacent: one memset
        e = cudaMemsetAsync(base + L.counts, 0, L.offsets - L.counts, st);
        if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
    }
    bsa::BwdArgs a{};
    a.q = static_cast<const uint16_t *>(q);
    a.kp = static_cast<const uint16_t *>(k);
    a.vp = static_cast<const uint16_t *>(v);
    a.out = static_cast<const uint16_t *>(out);
    a.dout = static_cast<const uint16_t *>(dout);
    a.list = list;
    a.bh = shape.bh;
    a.n = shape.n;
    a.nb = ceil_div(shape.n, ld.key_block);
    a.d = shape.d;
    a.k = ld.max_blocks;
    a.kb = ld.key_block;
    a.causal = mask.kind == BSA_MASK_CAUSAL ? 1 : 0;
    a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(float(shape.d));
    a.scale_log2 = softmax_scale_log2(scale, shape.d);
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.lse = reinterpret_cast<float *>(base + L.lse);
    a.dsum = reinterpret_cast<float *>(base + L.dsum);
    a.counts = reinterpret_cast<int32_t *>(base + L.counts);
    a.cursors = reinterpret_cast<int32_t *>(base + L.cursors);
    a.offsets = reinterpret_cast<int32_t *>(base + L.offsets);
    a.qlist = reinterpret_cast<int32_t *>(base + L.qlist);
    a.status = status;
    if (tc_path) {
        const BmLayout F = bm_layout(shape, ld.key_block, ld.max_blocks, L.fwd);
        if (lse_in != nullptr) {
            // the lists inverted by (head, query range, block); the row
            // statistics are the forward's (read only by the gradient kernel)
            bsa::InvertBuffers w{};
            e = run_invert_bm(shape, list, ld.key_block, ld.max_blocks, base + L.o_scratch, base, F,
                              status, st, w);
            a.lse = const_cast<float *>(lse_in);
        } else {
            // the forward fine stage once more: every row's log2-sum-exp, and
            // the lists inverted by (head, query range, block)
            e = run_fine_bm(shape, q, k, v, list, ld.key_block, ld.max_blocks, false,
                            a.causal != 0, nullptr, a.scale_log2, base + L.o_scratch, base, F,
                            status, st, a.lse);
        }
        if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "backward (statistics): %s", cudaGetErrorString(e));
        a.bin_offsets = reinterpret_cast<const int32_t *>(base + F.offsets);
        a.entries = reinterpret_cast<const int32_t *>(base + F.entries);
        a.nranges = F.plan.nranges;
        return launched(bsa::launch_fine_backward_tc(a, st), "backward launch");
    }
    return launched(bsa::launch_fine_backward(a, st), "backward launch");
}

}  // namespace

bsa_status bsa_fine_backward(bsa_shape shape, const void *q, const void *k, const void *v,
                             const void *out, const void *dout, const int32_t *list,
                             bsa_list_desc ld, bsa_mask mask, float scale, float *dq, float *dk,
                             float *dv, void *ws, size_t ws_bytes, void *stream) {
    return fine_backward_impl(shape, q, k, v, out, dout, list, ld, mask, scale, nullptr, dq, dk,
                              dv, ws, ws_bytes, stream);
}

bsa_status bsa_fine_backward_lse(bsa_shape shape, const void *q, const void *k, const void *v,
                                 const void *out, const void *dout, const int32_t *list,
                                 bsa_list_desc ld, bsa_mask mask, float scale, const float *lse,
                                 float *dq, float *dk, float *dv, void *ws, size_t ws_bytes,
                                 void *stream) {
    if (lse == nullptr) return fail(BSA_ERR_INVALID_ARG, "lse is NULL");
    if (!aligned(lse, 4)) return fail(BSA_ERR_ALIGNMENT, "lse is not 4-byte aligned");
    return fine_backward_impl(shape, q, k, v, out, dout, list, ld, mask, scale, lse, dq, dk, dv,
                              ws, ws_bytes, stream);
}

// ------------------------------------------------------- failure path
bsa_status bsa_selftest_wait_timeout(int32_t kind, uint64_t limit_ns, void *stream) {
    if (kind != 0 && kind != 1) return fail(BSA_ERR_INVALID_ARG, "kind must be 0 or 1 (got %d)", kind);
    if (limit_ns < 1000 || limit_ns > 2000000000ull)
        return fail(BSA_ERR_INVALID_ARG, "limit_ns must be in [1e3, 2e9]");
    int32_t *status = device_status_ptr();
    if (status == nullptr) return fail(BSA_ERR_CUDA, "status word unavailable");
    return launched(bsa::launch_wait_selftest(kind, limit_ns, status, static_cast<cudaStream_t>(stream)),
                    "self-test launch");
}

// ------------------------------------------------------------ CUDA graphs
struct bsa_graph_s {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

bsa_status bsa_forward_graph_create(bsa_shape shape, const void *q, const void *k, const void *v,
                                    int32_t key_block, int32_t topk, const bsa_select *sel,
                                    float scale, void *out, int32_t *idx_out, void *ws,
                                    size_t ws_bytes, bsa_graph *graph) {
    if (graph == nullptr) return fail(BSA_ERR_INVALID_ARG, "graph is NULL");
    *graph = nullptr;
    if (device_status_ptr() == nullptr) return fail(BSA_ERR_CUDA, "status word unavailable");
    cudaStream_t cs = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "capture stream: %s", cudaGetErrorString(e));
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) {
        cudaStreamDestroy(cs);
        return fail(BSA_ERR_CUDA, "begin capture: %s", cudaGetErrorString(e));
    }
    const bsa_status st = bsa_forward_ex(shape, q, k, v, key_block, topk, sel, scale, out, idx_out,
                                         ws, ws_bytes, cs);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (st != BSA_OK) {                       // the reason is already recorded
        if (g != nullptr) cudaGraphDestroy(g);
        return st;
    }
    if (e != cudaSuccess || g == nullptr)
        return fail(BSA_ERR_CUDA, "end capture: %s", cudaGetErrorString(e));
    cudaGraphExec_t x = nullptr;
    e = cudaGraphInstantiate(&x, g, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(g);
        return fail(BSA_ERR_CUDA, "instantiate: %s", cudaGetErrorString(e));
    }
    bsa_graph h = new (std::nothrow) bsa_graph_s{g, x};
    if (h == nullptr) {
        cudaGraphExecDestroy(x);
        cudaGraphDestroy(g);
        return fail(BSA_ERR_CUDA, "out of host memory");
    }
    *graph = h;
    return ok();
}

bsa_status bsa_graph_launch(bsa_graph graph, void *stream) {
    if (graph == nullptr) return fail(BSA_ERR_INVALID_ARG, "graph is NULL");
    const cudaError_t e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "graph launch: %s", cudaGetErrorString(e));
    return ok();
}

bsa_status bsa_graph_destroy(bsa_graph graph) {
    if (graph == nullptr) return ok();
    cudaGraphExecDestroy(graph->exec);
    cudaGraphDestroy(graph->graph);
    delete graph;
    return ok();
}

}  // extern "C"
