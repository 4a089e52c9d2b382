// attention_noalloc.cu -- pf_paged_decode_attention_noalloc: the decode
// attention call for callers that cannot allocate device memory.
//
// pf_paged_decode_attention needs a caller-provided workspace.  Some callers
// have no way to provide one: code that may only touch the buffers it is
// handed (a plugin inside another runtime, an operator whose framework owns
// every allocation) cannot call cudaMalloc or an allocating library routine.
// This variant keeps its workspace in a fixed array of this file instead,
// sized kNoAllocScratchBytes, which every GPU that loads the library holds
// until the process exits.  Nothing here allocates.
#include <mutex>

#include "internal.h"

namespace pkv {
namespace {

// Scratch of the no-allocation variant: reserved bytes, partial records and
// merge jobs of one call (the same layout as a caller's workspace).
constexpr size_t kNoAllocScratchBytes = 8u << 20;   // 8 MiB per device
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// In host code g_noalloc_scratch names a host-side stand-in, not device
// memory: the device address is looked up once per device, with that device
// current, and cached.
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

int scratch_for_current_device(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_decode_attention_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(PF_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch);
        if (e != cudaSuccess)
            return cuda_error(e, "pf_paged_decode_attention_noalloc: cudaGetSymbolAddress of the scratch array");
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return PF_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pf_paged_decode_attention_noalloc(const pf_pool *pool, int layer, const void *q,
                                                 const int32_t *block_tables, int max_blocks_per_seq,
                                                 const int32_t *context_lens, int n_seqs, int n_q_heads, float scale,
                                                 void *out, int out_dtype, int split_tokens, void *stream) {
    pkv::clear_error();
    if (n_seqs == 0) return PF_OK;
    if (!pool) return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention_noalloc: pool is null");
    const size_t need = pf_decode_workspace_bytes(pool, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens);
    if (need == 0) return PF_ERR_INVALID;   // message set by pf_decode_workspace_bytes
    if (need > pkv::kNoAllocScratchBytes)
        return pkv::set_error(PF_ERR_INVALID,
                              "pf_paged_decode_attention_noalloc: this batch needs " + std::to_string(need) +
                                  " bytes of scratch but the built-in scratch holds " +
                                  std::to_string(pkv::kNoAllocScratchBytes) +
                                  "; split the batch or call pf_paged_decode_attention with a workspace");
    void *ws = nullptr;
    int rc = pkv::scratch_for_current_device(&ws);
    if (rc) return rc;
    // The scratch is zero when the library loads.  Every word a call reads
    // back (merge jobs, span records) carries the epoch of the launch that
    // wrote it, so nothing left by an earlier call -- one that timed out
    // included -- is taken for this call's data, and nothing needs resetting.
    return pf_paged_decode_attention(pool, layer, q, block_tables, max_blocks_per_seq, context_lens, n_seqs,
                                     n_q_heads, scale, out, out_dtype, split_tokens, ws, pkv::kNoAllocScratchBytes,
                                     stream);
}
