// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed, not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bsa {

// Everything a fine-attention launch needs; plain values and pointers.
struct FineArgs {
    const void *q;
    const void *k;
    const void *v;
    void *out;
    const int32_t *list;   // nullptr: every block
    int64_t bh;
    int64_t n;
    int64_t nb;            // key blocks of size kb
    int32_t kb;
    int32_t d;
    int32_t q_group;
    int32_t max_blocks;
    int32_t per_head;
    int64_t list_rows;     // list rows per head = ceil(n / q_group)
    int32_t mask_kind;
    int32_t window;
    int32_t stride;
    int32_t sliding;
    float scale_log2;      // softmax scale * log2(e)
    int32_t *status;       // device status word
    // tensor-core static path, optional workspace: with both set, one pass
    // with a per-row bound on the scores, then the exact two passes only for
    // the tiles the bound did not serve
    float *kmax;           // [bh][nb] largest key norm of each block
    int32_t *flags;        // [bh][ceil(n / 128)] tiles to redo
};

// Options of the dynamic selection (bsa_select in bsa.h).
struct SelectOpts {
    const int32_t *head_k = nullptr;   // [bh] budgets in [0, topk], or null: topk
    int32_t kb = 1;                    // key block: the query's own block is i / kb
    int32_t causal = 0;                // eligible blocks b <= i / kb
    int32_t local = 0;                 // the own block is always selected
};

// Backward pass of the fine stage over per-query lists (bf16 in, fp32 out).
struct BwdArgs {
    const uint16_t *q, *kp, *vp, *out, *dout;
    const int32_t *list;          // [bh][n][k]
    int64_t bh, n, nb;
    int32_t d, k, kb, causal;
    float scale, scale_log2;      // softmax scale, and times log2(e)
    float *dq, *dk, *dv;          // [bh][n][d]
    float *lse, *dsum;            // [bh * n] workspace: log2-sum-exp, dO . O
    int32_t *counts, *cursors;    // [bh * nb] workspace, zeroed
    int32_t *offsets;             // [bh * nb + 1] workspace
    int32_t *qlist;               // [bh * n * k] workspace: queries by (head, block)
    // tensor-core path: the forward fine stage's inversion -- pair ids
    // ((h * n + i) << 5 | slot) grouped by bin (head, query range, block)
    const int32_t *bin_offsets;   // [bh * nranges * nb + 1]
    const int32_t *entries;
    int64_t nranges;
    int32_t *status;
};
bool fine_backward_supported(int32_t d, int32_t kb);   // one CTA of kb * d / 16 <= 512 threads
cudaError_t launch_fine_backward(const BwdArgs &a, cudaStream_t st);
// Tensor-core backward (64-key blocks, at most 32 per query): a.lse must hold
// every query's log2-sum-exp and a.bin_offsets / a.entries the inversion of
// the lists, both from the forward fine stage; a.dsum is filled here; dq is
// zeroed and accumulated.
bool fine_backward_tc_supported(int32_t d, int32_t kb, int32_t k);
cudaError_t launch_fine_backward_tc(const BwdArgs &a, cudaStream_t st);

// One small kernel whose bounded wait nothing completes (kind 0: an mbarrier,
// 1: a global counter); it records BSA_ERR_TIMEOUT after about limit_ns.
cudaError_t launch_wait_selftest(int32_t kind, uint64_t limit_ns, int32_t *status,
                                 cudaStream_t st);

// Records the one-line reason bsa_last_error() reports on this thread.
void set_last_error(const char *msg);

// Launchers return the cudaError_t of the launch.
cudaError_t launch_pool(const void *k, int64_t bh, int64_t n, int32_t d,
                        int32_t kb, float *kbar, uint16_t *kbar_hi,
                        uint16_t *kbar_lo, int64_t nb_pad, cudaStream_t st);

cudaError_t launch_coarse_topk_simt(const void *q, const float *kbar,
                                    int64_t bh, int64_t n, int32_t d,
                                    int64_t nb, int32_t topk, const SelectOpts &o,
                                    int32_t *idx, int32_t *status, cudaStream_t st);

// fp32 block means -> bf16 (hi, lo) pair for the tensor-core scoring.
cudaError_t launch_split_kbar(const float *kbar, int64_t count, uint16_t *hi, uint16_t *lo,
                              cudaStream_t st);

// Tensor-core scoring + top-k.  Needs ceil(log2 nb) <= 12 (nb <= 4096).
bool coarse_tc_supported(int64_t nb);
cudaError_t launch_coarse_topk_tc(const void *q, const uint16_t *kbar_hi, const uint16_t *kbar_lo,
                                  int64_t bh, int64_t n, int32_t d, int64_t nb, int32_t topk,
                                  const SelectOpts &o, int32_t *idx, int32_t *status,
                                  cudaStream_t st);

// ---- block-major fine stage over per-query lists [bh][n][k] ----------
constexpr int32_t kFineBmItemPairs = 512;   // pairs per fine work item (<= 4 tiles)
constexpr int32_t kMergeQueries = 32;       // queries per merge work item
constexpr int32_t kPartialRing = 4;         // query ranges whose partials coexist, at least
constexpr int32_t kPartialRingMax = 16;     // and at most
constexpr int64_t kPartialRingBytes = int64_t(72) << 20;   // partial-state bytes aimed at

// Bins are (head, query range of `range` queries, key block).
struct InvertPlan {
    int64_t range = 0, nranges = 0, nr = 0, nbins = 0, fine_cap = 0, merge_cap = 0;
    int32_t item_pairs = 0, qm = 0;
    int32_t kpad = 0;       // partial slots per query in the ring (k rounded up to 4)
    int32_t ring = 0;       // query ranges whose partial states coexist, a power of two (set by the fine stage)
};
InvertPlan invert_plan(int64_t bh, int64_t n, int64_t nb, int32_t k);

struct InvertBuffers {
    int32_t *counts;        // [nbins], zeroed
    int32_t *cursors;       // [nbins], zeroed
    int32_t *offsets;       // [nbins + 1]
    int32_t *fitem_off;     // [nbins + 1]
    int32_t *fpre;          // [nr + 2]
    int32_t *mpre;          // [nr + 1]
    int32_t *range_total;   // [nr] pairs per range
    int32_t *range_merges;  // [nr] merge items per range
    int2 *fine_items;       // [fine_cap]  {bin, first pair}
    int2 *merge_items;      // [merge_cap] {range, first query}
    int32_t *n_fine;
    int32_t *n_merge;
    int32_t *entries;       // [bh * n * k] pair ids (flat query row << 5) | slot, by bin
    uint32_t *vmask;        // [bh * n] per query: bit s set when slot s holds a block (nullable)
};
// count + scan + scatter launches
cudaError_t launch_invert(const int32_t *list, int64_t bh, int64_t n, int64_t nb, int32_t k,
                          const InvertPlan &p, const InvertBuffers &w, uint16_t *out_bf16,
                          int32_t d, int32_t *status, cudaStream_t st);

struct FineBmArgs {
    const void *k_ptr;
    const void *v_ptr;
    const uint16_t *q;
    const int32_t *list;          // [bh][n][k]
    InvertBuffers w;
    InvertPlan p;
    int32_t *fine_head;           // zeroed queue heads
    int32_t *merge_head;
    int32_t *range_done;          // [nr] zeroed: pairs with partials written
    int32_t *merge_done;          // [nr] zeroed: merge items finished
    int64_t bh, n, nb;
    int32_t d, k;
    int32_t full_lists;           // every row holds min(k, nb) valid ids, first
    int32_t causal;               // query i attends only keys j <= i
    // Lists written by the selection with options: row i of head h holds
    // min(k_h, eligible) ids first (k_h = head_k[h] clamped to [0, k], or k;
    // eligible = i / 64 + 1 when causal, else nb), -1 after them.
    int32_t sel_lists;
    const int32_t *head_k;
    float scale_log2;
    uint16_t *part_o;             // [ring][range * kpad][d] bf16
    float2 *part_ml;              // [ring][range * kpad] (m, l) of each pair, log2 units
    uint16_t *out;
    float *lse_out;               // optional [bh * n]: each query's log2-sum-exp over
                                  // its admitted keys (-inf when none), for the backward
    int32_t *status;
};
bool fine_bm_supported(int32_t d, int32_t key_block);
cudaError_t launch_fine_bm(const FineBmArgs &a, cudaStream_t st);

cudaError_t launch_fine_query_major(const FineArgs &a, int32_t dtype,
                                    cudaStream_t st);
// The whole forward of a small problem (bf16, d in {64, 128}, at most 64
// blocks, top-k <= 16, at most kSmallForwardRows rows of bh * n, no
// selection options) in one launch: pooling, scores, top-k and the fine
// stage (query-major, CUDA cores).  Writes out and idx [bh][n][topk].
constexpr int64_t kSmallForwardRows = 16384;
bool small_forward_supported(int32_t d, int64_t nb, int32_t topk, int64_t rows);
cudaError_t launch_small_forward(const FineArgs &a, int32_t topk, int32_t *idx, cudaStream_t st);
// Static or dense lists of bf16 inputs on the tensor cores: d in {64, 128},
// 64-key blocks, one list row per 128-query tile (or no list), at most 512
// listed blocks per row.
bool fine_static_tc_supported(const FineArgs &a, int32_t dtype);
// Workspace (bytes) that lets the static tensor-core path run one pass.
size_t fine_static_tc_workspace(int64_t bh, int64_t n, int32_t kb);
cudaError_t launch_fine_static_tc(const FineArgs &a, cudaStream_t st);

}  // namespace bsa
