/*
 * bsa.h -- C ABI of libbsa.so: content-dependent block-sparse attention
 * (forward) on one NVIDIA GB300 (sm_103a).
 *
 * The method (page "sparse-attention-triton-bench", section "Two-stage
 * block indexer"):
 *   Stage 1  mean-pool every B-token key block into a representative Kbar_b,
 *            score every query against every block (q . Kbar_b) and keep the
 *            k best blocks per query, ties to the lower block index;
 *   Stage 2  softmax attention, scale 1/sqrt(d) by default, over only the
 *            k*B tokens of the selected blocks, accumulated with an online
 *            softmax state (running max m, running sum l, accumulator acc;
 *            same page, section "The Triton kernel").
 * The fine stage also runs over static block lists (page "yayme/CUDA-kernel"
 * README: local window |i-j| <= w plus global stride j % s == 0, walked as a
 * precomputed active-tile list; page "Block-Sparse & Linear Attention
 * Kernels", section 2: block-sparse loop and the causal sliding window).
 *
 * Conventions shared by every entry point
 *   - Tensors Q, K, V, O are [bh][n][d] row-major (d fastest), contiguous,
 *     element type given by bsa_shape.dtype.  bh = batch * heads.
 *   - Every tensor pointer is a DEVICE pointer unless the parameter says
 *     host.  Device pointers must be 16-byte aligned; workspaces 256-byte.
 *   - The caller owns every buffer.  The library never allocates memory and
 *     keeps no per-call state; calls only enqueue work on `stream` (a
 *     cudaStream_t passed as void*, NULL = legacy default stream) and return
 *     at once.  Results are ready when the stream reaches that point.
 *   - Argument errors are detected on the host and returned synchronously;
 *     nothing is enqueued then.  bsa_last_error() gives a one-line reason.
 *   - Errors found by a kernel (a listed block index outside [0, nb), a
 *     bounded wait that ran out) never trap: the kernel skips the offending
 *     work, records the first such code in a device status word and
 *     returns.  bsa_get_device_status() reads and clears that word.
 *   - Supported: d in {64, 128}; key_block B in {16, 32, 64, 128};
 *     dtype bf16 everywhere, fp32 for the fine stage.
 */
#ifndef BSA_H_
#define BSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSA_OK = 0,
    BSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum value      */
    BSA_ERR_UNSUPPORTED = 2,   /* valid request outside the supported set     */
    BSA_ERR_BAD_INDEX = 3,     /* (device) a listed block id outside [0, nb)  */
    BSA_ERR_WORKSPACE = 4,     /* workspace null or smaller than required     */
    BSA_ERR_CUDA = 5,          /* a CUDA runtime call failed                  */
    BSA_ERR_TIMEOUT = 6,       /* (device) a bounded barrier wait ran out     */
    BSA_ERR_ALIGNMENT = 7      /* pointer not 16-byte (workspace: 256) aligned */
} bsa_status;

typedef enum { BSA_BF16 = 0, BSA_FP32 = 1 } bsa_dtype;

/* Shape of Q, K, V and O: [bh][n][d], element type `dtype` (bsa_dtype). */
typedef struct {
    int64_t bh;
    int64_t n;
    int32_t d;
    int32_t dtype;
} bsa_shape;

typedef enum {
    BSA_MASK_NONE = 0,          /* every token of a listed block is attended   */
    BSA_MASK_LOCAL_GLOBAL = 1,  /* |i-j| <= window  or  j % stride == 0        */
    BSA_MASK_SLIDING = 2,       /* causal window: i - sliding < j <= i         */
    BSA_MASK_CAUSAL = 3         /* causal: j <= i                              */
} bsa_mask_kind;

/*
 * Token-level predicate applied inside the listed blocks (page
 * "yayme/CUDA-kernel" README, sparsity pattern; page "Block-Sparse & Linear
 * Attention Kernels", section 2, sliding window, and section 1, the causal
 * lower triangle).  LOCAL_GLOBAL: window < 0 disables the band, stride <= 0
 * disables the global columns.  SLIDING: sliding >= 1 is W, the number of
 * keys up to and including the query.  CAUSAL takes no parameter; with
 * per-query lists (q_group = 1) it is what a causal selection needs inside
 * the query's own block.
 */
typedef struct {
    int32_t kind;
    int32_t window;
    int32_t stride;
    int32_t sliding;
} bsa_mask;

/*
 * Layout of a block-index list.  The list is int32
 *   [per_head ? bh : 1][ceil(n / q_group)][max_blocks]:
 * row r serves queries [r*q_group, (r+1)*q_group); each row holds key-block
 * ids (block b = tokens [b*key_block, min(n, (b+1)*key_block))) in strictly
 * ascending order, padded with -1 at the tail only.
 *   dynamic lists (stage 2):  q_group = 1, max_blocks = k, per_head = 1;
 *   static lists:             q_group = the query-tile height, per_head = 0.
 */
typedef struct {
    int32_t q_group;
    int32_t key_block;
    int32_t max_blocks;
    int32_t per_head;
} bsa_list_desc;

/*
 * Stage 1, pooling (page "sparse-attention-triton-bench", Two-stage block
 * indexer, Stage 1: "mean-pooling the keys within" each block).
 *   k     [bh][n][d] bf16 keys (device).
 *   kbar  [bh][nb][d] fp32 output, nb = ceil(n / key_block) (device);
 *         kbar[h][b] = mean of the valid keys of block b (a ragged last
 *         block averages its n - b*key_block tokens).
 */
bsa_status bsa_pool_blocks(bsa_shape shape, const void *k, int32_t key_block,
                           float *kbar, void *stream);

/*
 * Stage 1 scoring + Stage 2 selection (same page and section: score every
 * query against every block representative, "take the top-k
 * highest-scoring blocks").  Scores are q . Kbar_b (unscaled: a positive
 * scale cannot change the ranking) and are never written to memory.
 *   q     [bh][n][d] bf16 queries (device).
 *   kbar  [bh][nb][d] fp32 block means, as written by bsa_pool_blocks.
 *   idx   [bh][n][topk] int32 output (device): the min(topk, nb) selected
 *         block ids of each query in ascending order, ties in score going to
 *         the lower block id; entries past nb are -1.
 *   ws    device workspace of bsa_coarse_topk_workspace_size() bytes.
 * topk in [1, 32].
 */
size_t bsa_coarse_topk_workspace_size(bsa_shape shape, int32_t key_block,
                                      int32_t topk);
bsa_status bsa_coarse_topk(bsa_shape shape, const void *q, const float *kbar,
                           int32_t key_block, int32_t topk, int32_t *idx,
                           void *ws, size_t ws_bytes, void *stream);

/*
 * Options of the selection (NULL = none, which is bsa_coarse_topk).
 *   head_topk    optional DEVICE int32 [bh]: the budget k_h of each
 *                (batch * head) row, in [0, topk] (page
 *                "sparse-attention-triton-bench", What's next: per-head
 *                sparsity budgets chosen at run time on the per-head stage-1
 *                scores).  Row h of idx then holds min(k_h, eligible) ids and
 *                -1 after them.  A value outside [0, topk] is clamped into it
 *                and reported as BSA_ERR_INVALID_ARG through
 *                bsa_get_device_status().  NULL: topk for every row.
 *   causal       nonzero: query i may select only blocks b <= i / key_block
 *                (blocks holding some key j <= i; page "Block-Sparse &
 *                Linear Attention Kernels", section 1, the causal pattern),
 *                and the fine stage of bsa_forward_ex attends only keys
 *                j <= i.
 *   local_block  nonzero: the query's own block i / key_block is always
 *                selected (when its budget is >= 1); the other k_h - 1 are
 *                the best-scoring eligible blocks except it.
 * Ties and output order as bsa_coarse_topk.
 */
typedef struct {
    const int32_t *head_topk;
    int32_t causal;
    int32_t local_block;
} bsa_select;

bsa_status bsa_coarse_topk_ex(bsa_shape shape, const void *q, const float *kbar,
                              int32_t key_block, int32_t topk,
                              const bsa_select *sel, int32_t *idx, void *ws,
                              size_t ws_bytes, void *stream);

/*
 * Stage 2, fine attention over a block list (page
 * "sparse-attention-triton-bench", Stage 2 and "The Triton kernel": dense
 * softmax attention over the listed blocks' tokens with an online-softmax
 * state; page "Block-Sparse & Linear Attention Kernels", section 2: skip
 * every unlisted block).
 *   q, k, v  [bh][n][d] of shape.dtype (bf16 or fp32), device.
 *   list     int32 block list laid out as `ld` says (device), or NULL for
 *            every block of the sequence.
 *   mask     token-level predicate inside listed blocks.
 *   scale    softmax scale; <= 0 selects 1/sqrt(d).
 *   out      [bh][n][d] of shape.dtype (device); a query whose list admits
 *            no key gets zeros.
 *   ws       device workspace of bsa_fine_attention_workspace_size() bytes.
 *            Per-query lists need it.  For static tile lists (and no list)
 *            of bf16 inputs on the tensor-core path it is optional: with it
 *            the kernel first takes each block's largest key norm and runs
 *            one pass with a per-row bound on the scores (the exact two-pass
 *            kernel redoes only the tiles the bound does not serve); without
 *            it (NULL) every tile runs two passes.  The results agree to
 *            rounding.
 * A listed id outside [0, nb) is skipped and reported as BSA_ERR_BAD_INDEX
 * through bsa_get_device_status().
 */
size_t bsa_fine_attention_workspace_size(bsa_shape shape, bsa_list_desc ld,
                                         bsa_mask mask);
bsa_status bsa_fine_attention(bsa_shape shape, const void *q, const void *k,
                              const void *v, const int32_t *list,
                              bsa_list_desc ld, bsa_mask mask, float scale,
                              void *out, void *ws, size_t ws_bytes,
                              void *stream);

/*
 * bsa_fine_attention that also returns each query's log2-sum-exp
 * lse_i = log2 sum_{j in T_i} 2^(s_ij * scale * log2 e), the softmax's
 * normaliser in base 2 ("The Triton kernel": the row statistics m and l of
 * the online softmax, lse = m + log2 l), for a backward pass to reuse
 * (bsa_fine_backward_lse).  A query whose list admits no key gets -inf.
 *   lse_out  [bh][n] fp32 (device), 4-byte aligned.
 * Only where bsa_fine_attention takes its block-major path: per-query lists
 * (q_group 1, per_head 1, max_blocks <= 32), bf16, d in {64, 128},
 * key_block 64, at most 16384 blocks, no mask or the causal one; other calls
 * return BSA_ERR_UNSUPPORTED.  Workspace and everything else as
 * bsa_fine_attention.
 */
bsa_status bsa_fine_attention_lse(bsa_shape shape, const void *q, const void *k,
                                  const void *v, const int32_t *list,
                                  bsa_list_desc ld, bsa_mask mask, float scale,
                                  void *out, float *lse_out, void *ws,
                                  size_t ws_bytes, void *stream);

/*
 * Backward pass of the fine stage (page "sparse-attention-triton-bench",
 * What's next: a backward pass through the sparse softmax-weighted sum over
 * the selected blocks).  The selection is a discrete choice and is held
 * fixed: the gradients flow through the fine stage only.  For query i with
 * token set T_i (its listed blocks' keys; only j <= i under
 * BSA_MASK_CAUSAL) and the output gradient dO:
 *   D_i = dO_i . O_i,  dS_ij = p_ij (dO_i . v_j - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 *   dV_j = sum_i p_ij dO_i.
 * The row statistics of the softmax are recomputed from q, k and the list.
 *   q, k, v   [bh][n][d] bf16 (device), as given to the forward.
 *   out       [bh][n][d] bf16: the forward's output O for this list.
 *   dout      [bh][n][d] bf16: dO.
 *   list, ld  per-query lists as the forward took them (q_group 1,
 *             per_head 1, max_blocks <= 64; ascending ids, -1 padding).
 *   mask      BSA_MASK_NONE or BSA_MASK_CAUSAL.
 *   scale     softmax scale; <= 0 selects 1/sqrt(d).
 *   dq, dk, dv  [bh][n][d] fp32 outputs (device); every element is written
 *             (keys no query listed get zeros).
 *   ws        device workspace of bsa_fine_backward_workspace_size() bytes.
 * d in {64, 128}, key_block * d <= 8192; bf16 only.  Listed ids outside
 * [0, nb) are skipped and
 * reported as BSA_ERR_BAD_INDEX through bsa_get_device_status().
 */
size_t bsa_fine_backward_workspace_size(bsa_shape shape, bsa_list_desc ld);
bsa_status bsa_fine_backward(bsa_shape shape, const void *q, const void *k,
                             const void *v, const void *out, const void *dout,
                             const int32_t *list, bsa_list_desc ld,
                             bsa_mask mask, float scale, float *dq, float *dk,
                             float *dv, void *ws, size_t ws_bytes,
                             void *stream);

/*
 * bsa_fine_backward given the forward's log2-sum-exp per query (as
 * bsa_fine_attention_lse writes it, for the same inputs, lists, mask and
 * scale), so that the softmax statistics are not recomputed: on the
 * tensor-core path (key_block 64, max_blocks <= 32) the call inverts the
 * lists and runs the gradient kernels only.  Other shapes recompute the
 * statistics as bsa_fine_backward does and ignore lse.
 *   lse  [bh][n] fp32 (device), 4-byte aligned; not modified.
 * Same workspace (bsa_fine_backward_workspace_size) and outputs as
 * bsa_fine_backward.
 */
bsa_status bsa_fine_backward_lse(bsa_shape shape, const void *q, const void *k,
                                 const void *v, const void *out, const void *dout,
                                 const int32_t *list, bsa_list_desc ld,
                                 bsa_mask mask, float scale, const float *lse,
                                 float *dq, float *dk, float *dv, void *ws,
                                 size_t ws_bytes, void *stream);

/*
 * The whole dynamic forward: pool -> score + top-k -> fine attention, all
 * enqueued on `stream` (page "sparse-attention-triton-bench", Two-stage
 * block indexer).  bf16 only, non-causal (bsa_forward_ex below takes the causal and
 * per-head options).
 *   idx_out  optional [bh][n][topk] int32 (device) receiving the selection;
 *            NULL keeps it in the workspace.
 *   ws       device workspace of bsa_forward_workspace_size() bytes.
 */
size_t bsa_forward_workspace_size(bsa_shape shape, int32_t key_block,
                                  int32_t topk);
bsa_status bsa_forward(bsa_shape shape, const void *q, const void *k,
                       const void *v, int32_t key_block, int32_t topk,
                       float scale, void *out, int32_t *idx_out, void *ws,
                       size_t ws_bytes, void *stream);

/*
 * bsa_forward with selection options (bsa_select above; NULL = none).  With
 * `causal` the fine stage attends, for query i, only the keys j <= i of its
 * selected blocks.  Same workspace as bsa_forward (its size does not depend
 * on the options); same errors.
 */
bsa_status bsa_forward_ex(bsa_shape shape, const void *q, const void *k,
                          const void *v, int32_t key_block, int32_t topk,
                          const bsa_select *sel, float scale, void *out,
                          int32_t *idx_out, void *ws, size_t ws_bytes,
                          void *stream);

/*
 * bsa_forward_ex that also writes each query's log2-sum-exp (as
 * bsa_fine_attention_lse defines it) for a backward pass over the same
 * selection (bsa_fine_backward_lse with idx_out as the list), so that a
 * training step computes the softmax statistics once.  The forward then
 * always runs as separate launches (the one-launch form for small problems
 * keeps no statistics).
 *   lse_out  [bh][n] fp32 (device), 4-byte aligned.
 * Only where the fine stage takes its block-major path (key_block 64, at most
 * 16384 blocks); other shapes return BSA_ERR_UNSUPPORTED.  Workspace and
 * everything else as bsa_forward_ex.
 */
bsa_status bsa_forward_lse(bsa_shape shape, const void *q, const void *k,
                           const void *v, int32_t key_block, int32_t topk,
                           const bsa_select *sel, float scale, void *out,
                           int32_t *idx_out, float *lse_out, void *ws,
                           size_t ws_bytes, void *stream);

/*
 * The whole forward as one CUDA graph (page "sparse-attention-triton-bench",
 * The Triton kernel: the forward as a few fused launches instead of the
 * hundreds of a Python loop; here every launch of bsa_forward_ex is captured
 * once and the caller replays them with one host call).
 *   bsa_forward_graph_create  captures bsa_forward_ex for these exact
 *       pointers and arguments (same validation and errors) on a private
 *       stream and instantiates it; *graph receives the handle (NULL on
 *       error).  Nothing runs at creation.
 *   bsa_graph_launch  enqueues one replay on `stream`: it reads whatever the
 *       captured q, k, v (and head_topk) buffers hold at that time and writes
 *       out (and idx_out); the workspace must stay allocated and unshared
 *       while replays can run.
 *   bsa_graph_destroy  releases the handle (NULL is a no-op); replays already
 *       enqueued complete.
 */
typedef struct bsa_graph_s *bsa_graph;
bsa_status bsa_forward_graph_create(bsa_shape shape, const void *q,
                                    const void *k, const void *v,
                                    int32_t key_block, int32_t topk,
                                    const bsa_select *sel, float scale,
                                    void *out, int32_t *idx_out, void *ws,
                                    size_t ws_bytes, bsa_graph *graph);
bsa_status bsa_graph_launch(bsa_graph graph, void *stream);
bsa_status bsa_graph_destroy(bsa_graph graph);

/*
 * bsa_forward without a workspace argument, for callers that must not
 * allocate device memory at call time (e.g. a plugin inside an application
 * whose memory manager owns the device, or a latency-bound loop that cannot
 * afford cudaMalloc).  The pages have no counterpart: this is a packaging
 * variant of bsa_forward, same kernels, same results.
 *   - Scratch is a static device array of 32 MiB inside the library; every
 *     device that loads the library holds it until the process exits.  A
 *     problem whose bsa_forward_workspace_size() exceeds 32 MiB is rejected
 *     with BSA_ERR_WORKSPACE (2 heads x 1024 tokens, top-4 needs about
 *     2.1 MiB and fits; 8 heads x 8192 tokens, top-16 needs about 25 MiB
 *     and fits; 8 heads x 32768 tokens, top-16 needs about 100 MiB and is
 *     rejected; the workspace grows with heads * n * k).
 *   - Allocates nothing: no cudaMalloc/cudaFree and no allocating library
 *     call.  The first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current; make that
 *     first call before any stream capture.  The address is kept for the
 *     life of the process (like the status word's, see
 *     bsa_get_device_status): calls after a cudaDeviceReset of that device
 *     are not supported.
 *   - Every call on a device shares the one array: calls whose work can
 *     overlap on the GPU (different streams, or different host threads)
 *     race on it and must be serialised by the caller.
 * Other arguments and errors as bsa_forward.
 */
bsa_status bsa_forward_noalloc(bsa_shape shape, const void *q, const void *k,
                               const void *v, int32_t key_block, int32_t topk,
                               float scale, void *out, int32_t *idx_out,
                               void *stream);

/* Number of kernel launches one bsa_forward call enqueues for this problem
 * (for launch accounting by callers); negative bsa_status on bad arguments. */
int32_t bsa_forward_launches(bsa_shape shape, int32_t key_block, int32_t topk);

/*
 * Static block lists, built on the host, synchronously (page
 * "yayme/CUDA-kernel" README: "precompute the list of active (row_tile,
 * col_tile) pairs on the CPU and pass it in").  A key block is listed for a
 * query tile iff at least one (query, key) pair inside it satisfies `mask`
 * (BSA_MASK_NONE lists every block).
 *   list          HOST int32 [ceil(n/q_group)][max_blocks], -1 padded.
 *   counts        optional HOST int32 [ceil(n/q_group)]: blocks per row.
 *   active_pairs  optional HOST int64: number of (i, j) pairs the mask
 *                 admits over the whole sequence (one head).
 * bsa_static_max_blocks() returns the smallest max_blocks that fits, or a
 * negative bsa_status on invalid arguments.
 */
int32_t bsa_static_max_blocks(int64_t n, int32_t q_group, int32_t key_block,
                              bsa_mask mask);
bsa_status bsa_static_blocks(int64_t n, int32_t q_group, int32_t key_block,
                             bsa_mask mask, int32_t *list, int32_t max_blocks,
                             int32_t *counts, int64_t *active_pairs);

/*
 * Reads the device status word into *status (a bsa_status value), then
 * clears it.  Synchronises `stream` first.  The word is a static device
 * variable of the library, one per device; its address is looked up on the
 * first call that needs it on a device and kept for the life of the process
 * (a cudaDeviceReset of that device is not supported afterwards).
 */
bsa_status bsa_get_device_status(int32_t *status, void *stream);

/*
 * Failure-path self-test (the pages have no counterpart; it tests this
 * library's own error handling).  Enqueues one small kernel that runs the
 * library's bounded wait on something nothing will ever complete -- kind 0:
 * an mbarrier no thread arrives on (the wait every TMA / MMA hand-off of the
 * tensor-core kernels uses); kind 1: a counter in global memory no thread
 * raises (the wait the block-major fine stage uses between its query ranges
 * and merges).  After about limit_ns (1e3 .. 2e9 ns; the kernels use 2e9)
 * the wait gives up, records BSA_ERR_TIMEOUT in the device status word and
 * the kernel returns; the CUDA context stays usable.  If the status word
 * already holds BSA_ERR_TIMEOUT the wait gives up at once.  Read (and clear)
 * the result with bsa_get_device_status().  BSA_ERR_INVALID_ARG for another
 * kind or a limit outside the range.
 */
bsa_status bsa_selftest_wait_timeout(int32_t kind, uint64_t limit_ns, void *stream);

/* Static description of a status code. */
const char *bsa_status_string(int32_t status);

/* One-line reason for the last error returned on the calling thread. */
const char *bsa_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t bsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H_ */
