// Static block lists on the host (page "yayme/CUDA-kernel" README: the
// local-window + global-stride pattern, with the active (row_tile, col_tile)
// pairs precomputed on the CPU so the kernel walks a list instead of
// scanning a mask; page "Block-Sparse & Linear Attention Kernels", section
// 2: block-level masks for the sliding window).
//
// Lists are derived in closed form per query tile [i0, i1]:
//   local window  keys within [i0 - w, i1 + w]: every key of that interval
//                 is within w of some query of the tile;
//   global stride the key blocks that contain a multiple of s (below n);
//   sliding       keys within [i0 - W + 1, i1] (causal, W keys incl. self);
//   causal        keys within [0, i1] (page "Block-Sparse & Linear
//                 Attention Kernels", section 1, the lower triangle);
// intersected with [0, n).  A block is listed iff the pattern admits at
// least one (query, key) pair inside the tile x block rectangle.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "bsa.h"

namespace {

bool valid_args(int64_t n, int32_t q_group, int32_t key_block, const bsa_mask &m) {
    if (n < 1 || q_group < 1 || key_block < 1) return false;
    if (m.kind == BSA_MASK_SLIDING) return m.sliding >= 1;
    if (m.kind == BSA_MASK_LOCAL_GLOBAL || m.kind == BSA_MASK_CAUSAL) return true;
    return m.kind == BSA_MASK_NONE;
}

// Ascending, de-duplicated list of key blocks holding a global-stride key.
std::vector<int64_t> stride_blocks(int64_t n, int32_t key_block, int32_t s) {
    std::vector<int64_t> out;
    if (s <= 0) return out;
    for (int64_t j = 0; j < n; j += s) {
        const int64_t b = j / key_block;
        if (out.empty() || out.back() != b) out.push_back(b);
    }
    return out;
}

// Calls emit(b) for each listed block of tile row r, in ascending order.
template <typename F>
void for_each_block(int64_t n, int32_t q_group, int32_t key_block, const bsa_mask &m,
                    const std::vector<int64_t> &sblocks, int64_t r, F emit) {
    const int64_t nb = (n + key_block - 1) / key_block;
    const int64_t i0 = r * q_group;
    const int64_t i1 = std::min(n, i0 + q_group) - 1;
    if (m.kind == BSA_MASK_NONE) {
        for (int64_t b = 0; b < nb; ++b) emit(b);
        return;
    }
    int64_t lo_key = 0, hi_key = -1;   // empty band by default
    if (m.kind == BSA_MASK_SLIDING) {
        lo_key = std::max<int64_t>(0, i0 - int64_t(m.sliding) + 1);
        hi_key = i1;
    } else if (m.kind == BSA_MASK_CAUSAL) {
        lo_key = 0;
        hi_key = i1;
    } else if (m.window >= 0) {
        lo_key = std::max<int64_t>(0, i0 - m.window);
        hi_key = std::min<int64_t>(n - 1, i1 + m.window);
    }
    const int64_t blo = hi_key >= lo_key ? lo_key / key_block : 1;
    const int64_t bhi = hi_key >= lo_key ? hi_key / key_block : 0;
    // merge the band interval [blo, bhi] with the stride blocks
    size_t k = 0;
    int64_t last = -1;
    auto put = [&](int64_t b) {
        if (b != last) {
            emit(b);
            last = b;
        }
    };
    const bool strided = m.kind == BSA_MASK_LOCAL_GLOBAL;
    for (int64_t b = blo; b <= bhi; ++b) {
        while (strided && k < sblocks.size() && sblocks[k] < b) put(sblocks[k++]);
        put(b);
    }
    while (strided && k < sblocks.size()) {
        if (sblocks[k] > last) put(sblocks[k]);
        ++k;
    }
}

// Keys admitted for query i (closed form), summed over the sequence.
int64_t count_pairs(int64_t n, const bsa_mask &m) {
    int64_t total = 0;
    if (m.kind == BSA_MASK_NONE) return n * n;
    if (m.kind == BSA_MASK_CAUSAL) return n * (n + 1) / 2;
    if (m.kind == BSA_MASK_SLIDING) {
        for (int64_t i = 0; i < n; ++i) total += std::min<int64_t>(i + 1, m.sliding);
        return total;
    }
    const int64_t s = m.stride;
    const int64_t globals = s > 0 ? (n - 1) / s + 1 : 0;
    for (int64_t i = 0; i < n; ++i) {
        if (m.window < 0) {
            total += globals;
            continue;
        }
        const int64_t lo = std::max<int64_t>(0, i - m.window);
        const int64_t hi = std::min<int64_t>(n - 1, i + m.window);
        int64_t in_band = 0;
        if (s > 0) in_band = hi / s - (lo == 0 ? -1 : (lo - 1) / s);
        total += (hi - lo + 1) + globals - in_band;
    }
    return total;
}

}  // namespace

extern "C" int32_t bsa_static_max_blocks(int64_t n, int32_t q_group, int32_t key_block,
                                         bsa_mask mask) {
    if (!valid_args(n, q_group, key_block, mask)) return -int32_t(BSA_ERR_INVALID_ARG);
    const std::vector<int64_t> sb = stride_blocks(n, key_block, mask.kind == BSA_MASK_LOCAL_GLOBAL ? mask.stride : 0);
    const int64_t rows = (n + q_group - 1) / q_group;
    int64_t best = 0;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t c = 0;
        for_each_block(n, q_group, key_block, mask, sb, r, [&](int64_t) { ++c; });
        best = std::max(best, c);
    }
    return int32_t(best);
}

extern "C" bsa_status bsa_static_blocks(int64_t n, int32_t q_group, int32_t key_block,
                                        bsa_mask mask, int32_t *list, int32_t max_blocks,
                                        int32_t *counts, int64_t *active_pairs) {
    if (!valid_args(n, q_group, key_block, mask) || list == nullptr || max_blocks < 1)
        return BSA_ERR_INVALID_ARG;
    const std::vector<int64_t> sb = stride_blocks(n, key_block, mask.kind == BSA_MASK_LOCAL_GLOBAL ? mask.stride : 0);
    const int64_t rows = (n + q_group - 1) / q_group;
    for (int64_t r = 0; r < rows; ++r) {
        int32_t *dst = list + r * max_blocks;
        int64_t c = 0;
        bool overflow = false;
        for_each_block(n, q_group, key_block, mask, sb, r, [&](int64_t b) {
            if (c < max_blocks) dst[c] = int32_t(b);
            else overflow = true;
            ++c;
        });
        if (overflow) return BSA_ERR_INVALID_ARG;   // max_blocks too small
        for (int64_t t = c; t < max_blocks; ++t) dst[t] = -1;
        if (counts) counts[r] = int32_t(c);
    }
    if (active_pairs) *active_pairs = count_pairs(n, mask);
    return BSA_OK;
}
