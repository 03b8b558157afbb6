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

cudaError_t launch_fine_query_major(const FineArgs &a, int32_t dtype,
                                    cudaStream_t st);

}  // namespace bsa
