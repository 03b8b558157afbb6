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
};

// Records the one-line reason bsa_last_error() reports on this thread.
void set_last_error(const char *msg);

// Launchers return the cudaError_t of the launch.
cudaError_t launch_pool(const void *k, int64_t bh, int64_t n, int32_t d,
                        int32_t kb, float *kbar, uint16_t *kbar_hi,
                        uint16_t *kbar_lo, int64_t nb_pad, cudaStream_t st);

cudaError_t launch_coarse_topk_simt(const void *q, const float *kbar,
                                    int64_t bh, int64_t n, int32_t d,
                                    int64_t nb, int32_t topk, int32_t *idx,
                                    cudaStream_t st);

// fp32 block means -> bf16 (hi, lo) pair for the tensor-core scoring.
cudaError_t launch_split_kbar(const float *kbar, int64_t count, uint16_t *hi, uint16_t *lo,
                              cudaStream_t st);

// Tensor-core scoring + top-k.  Needs ceil(log2 nb) <= 12 (nb <= 4096).
bool coarse_tc_supported(int64_t nb);
cudaError_t launch_coarse_topk_tc(const void *q, const uint16_t *kbar_hi, const uint16_t *kbar_lo,
                                  int64_t bh, int64_t n, int32_t d, int64_t nb, int32_t topk,
                                  int32_t *idx, int32_t *status, cudaStream_t st);

// Per-query list -> per-block pair lists (count, scan, scatter launches).
int64_t invert_query_range(int64_t n, int64_t nb, int32_t k);
int64_t invert_bins(int64_t bh, int64_t n, int64_t nb, int32_t k);
size_t invert_items_capacity(int64_t bh, int64_t n, int64_t nb, int32_t k, int32_t item_pairs);
cudaError_t launch_invert(const int32_t *list, int64_t bh, int64_t n, int64_t nb, int32_t k,
                          int32_t item_pairs, int32_t *counts, int32_t *cursors,
                          int32_t *offsets, int2 *items, int32_t *n_items, int32_t *entries,
                          uint16_t *out_bf16, int32_t d, int32_t *status, cudaStream_t st);

// Block-major tensor-core fine stage over inverted lists (bf16, B = 64).
struct FineBmArgs {
    const void *k_ptr;
    const void *v_ptr;
    const uint16_t *q;
    const int32_t *list;       // [bh][n][k] per-query lists
    const int32_t *entries;
    const int32_t *offsets;
    const int2 *items;
    const int32_t *n_items;
    int64_t bh, n, nb;
    int64_t bins_per_head;     // query ranges per head * nb
    int32_t d, k;
    int32_t full_lists;        // every row holds min(k, nb) valid ids
    int32_t item_pairs;
    float scale_log2;
    uint16_t *part_o;          // [bh*n*k][d] bf16
    float *part_lse;           // [bh*n*k]
    int32_t *qcount;           // [bh*n], zeroed
    uint16_t *out;
    int32_t *status;
};
constexpr int32_t kFineBmItemPairs = 512;
bool fine_bm_supported(int32_t d, int32_t key_block);
cudaError_t launch_fine_bm(const FineBmArgs &a, cudaStream_t st);

cudaError_t launch_fine_query_major(const FineArgs &a, int32_t dtype,
                                    cudaStream_t st);

}  // namespace bsa
