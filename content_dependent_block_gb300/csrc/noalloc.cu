// bsa_forward_noalloc: the dynamic forward without a caller-supplied
// workspace.  Its scratch memory is one file-scope device array that the
// library brings with it, so the call itself never allocates.
//
// Who needs this: callers that are not allowed to allocate device memory
// at call time -- for example a plugin living inside a host application
// whose memory manager owns the whole device and forbids stray
// cudaMalloc calls, or a latency-bound loop in which cudaMalloc (which can
// synchronise the device and may fail under a memory cap) is not an
// option.  They still own their inputs and outputs; only the forward's
// intermediate buffers (block means, their bf16 pair, the selection) move
// into the static array.
#include <cstdio>
#include <mutex>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

// Lives on every device that loads the library, until the process exits.
// In host code `g_scratch` names only a host-side stand-in: its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch on the current device; looked up once per
// device (on that device's first call) and cached.
bsa_status scratch_address(void **out) {
    static std::mutex mu;
    static void *cache[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        bsa::set_last_error("no usable current CUDA device");
        return BSA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[160];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress(static scratch): %s",
                     cudaGetErrorString(e));
            bsa::set_last_error(msg);
            return BSA_ERR_CUDA;
        }
        cache[dev] = p;
    }
    *out = cache[dev];
    return BSA_OK;
}

}  // namespace

extern "C" bsa_status bsa_forward_noalloc(bsa_shape shape, const void *q, const void *k,
                                          const void *v, int32_t key_block, int32_t topk,
                                          float scale, void *out, int32_t *idx_out,
                                          void *stream) {
    const size_t need = bsa_forward_workspace_size(shape, key_block, topk);
    if (need == 0)   // invalid arguments: let the forward report which one
        return bsa_forward(shape, q, k, v, key_block, topk, scale, out, idx_out, nullptr, 0,
                           stream);
    if (need > kScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "problem needs %zu bytes of scratch; the static scratch holds %zu bytes "
                 "(use bsa_forward with a caller workspace)",
                 need, kScratchBytes);
        bsa::set_last_error(msg);
        return BSA_ERR_WORKSPACE;
    }
    void *ws = nullptr;
    const bsa_status st = scratch_address(&ws);
    if (st != BSA_OK) return st;
    // Every workspace byte the forward reads it first writes in the same
    // call, so the previous call's leftovers need no clearing.
    return bsa_forward(shape, q, k, v, key_block, topk, scale, out, idx_out, ws, kScratchBytes,
                       stream);
}
