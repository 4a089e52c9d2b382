// internal.h -- declarations shared by the host C++ and the CUDA launchers of
// libpagedkv.so.  Not part of the public ABI (include/pagedkv.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>

#include "../../include/pagedkv.h"

namespace pkv {

// Thread-local last-error message; set_error returns the status it is given.
int set_error(int status, const std::string &msg);
int cuda_error(cudaError_t err, const char *what);
void clear_error();

// Maximum devices a pool caches descriptors for.
constexpr int kMaxDevices = 64;

// Tile height (tokens) the attention kernel stages per TMA transaction.
constexpr int kTileTokens = 16;

// pf_paged_prefill_attention without the decode kernel: at least this many
// query rows (new tokens x q-heads per kv-head) per (sequence, kv-head) take
// the tcgen05 kernel, fewer the warp-level MMA kernel.
constexpr int kTcMinRows = 128;

}  // namespace pkv

// Non-owning description of caller-owned K and V pools.
struct pf_pool {
    void *k_base;
    void *v_base;
    int n_layers;
    int n_blocks;
    int block_size;
    int n_kv_heads;
    int head_dim;
    int dtype;
    // TMA descriptors over K and V viewed as [rows][n_kv_heads][head_dim]
    // with rows = n_layers * n_blocks * block_size, encoded lazily per device.
    std::mutex mu;
    // per device: boxes of 1, 2, 4 kv-heads (CUDA-core consumers), then the
    // tensor-core layout for 1, 2, 4 kv-heads per item
    bool tmap_ready[pkv::kMaxDevices][6];
    CUtensorMap tmap_k[pkv::kMaxDevices][6];
    CUtensorMap tmap_v[pkv::kMaxDevices][6];
    // per device: the prompt kernel's boxes (one 64-element half of up to a
    // page of rows of one kv-head, swizzled)
    bool tmap_pf_ready[pkv::kMaxDevices];
    CUtensorMap tmap_pf_k[pkv::kMaxDevices];
    CUtensorMap tmap_pf_v[pkv::kMaxDevices];
};

namespace pkv {

// Device status word of the current device (a __device__ variable of this
// library); kernels OR pf_device_flag bits into it.
int *device_status_ptr();

// TMA descriptors of the pool for boxes of hg (1, 2 or 4) kv-heads, or (hg
// = 0) the tensor-core layout, on `device`, encoded on first use; *index
// receives their slot.
int encode_pool_tmaps(pf_pool *pool, int device, int hg, int *index);

struct WriteArgs {
    const pf_pool *pool;
    int layer;
    const void *k_new;
    const void *v_new;
    const int32_t *block_tables;
    int n_table_rows;
    int max_blocks;
    const int32_t *seq_idx;
    const int32_t *pos;
    int n_tokens;
};
int launch_write_kv(const WriteArgs &a, cudaStream_t stream);

// Whole-block copies: pool -> pool (both id arrays set), pool -> image
// (dst_ids null: destination i is image i of `image`), image -> pool
// (src_ids null).  Ids are device int32 arrays of n entries.
struct BlockCopyArgs {
    const pf_pool *pool;
    const int32_t *src_ids;
    const int32_t *dst_ids;
    const void *image;   // device-accessible address of the host images
    int n;
};
int launch_block_copy(const BlockCopyArgs &a, cudaStream_t stream);

// Multi-token append attention (pf_paged_prefill_attention).
struct PrefillArgs {
    const pf_pool *pool;
    int layer;
    const void *q;
    const int32_t *block_tables;
    int max_blocks;
    const int32_t *context_lens;
    const int32_t *cu_q;
    int n_seqs;
    int max_new;
    int n_q_heads;
    float scale;
    void *out;
    int out_dtype;
};
int launch_prefill(const PrefillArgs &a, cudaStream_t stream);   // prefill_mma.cu
int launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream);   // prefill_tc.cu

struct GatherArgs {
    const pf_pool *pool;
    int layer;
    const int32_t *block_tables;
    int max_blocks;
    const int32_t *context_lens;
    const int64_t *cu_off;
    int n_seqs;
    void *k_out;
    void *v_out;
};
int launch_gather_kv(const GatherArgs &a, cudaStream_t stream);

// How an attention call is scheduled and what workspace it needs.
struct AttnPlan {
    bool spans;            // balanced spans (split_tokens 0 or -2) or fixed chunks
    bool cuda_cores;       // CUDA-core consumers (split_tokens != 0): fp32 scores and weights
    int chunk;             // chunk schedule: tokens per chunk
    int grid;              // persistent grid (0 when planned without a device)
    size_t counter_bytes;  // reserved bytes at the front of the workspace (256 B)
    size_t partial_bytes;  // partial records (spans: epoch-tagged 64-bit words; chunks: fp32), then merge jobs
    size_t n_jobs;         // chunk schedule: merge job slots (0: no merge kernel)
};
int attention_plan(const pf_pool *pool, int n_seqs, int n_q_heads, int max_blocks, int split_tokens,
                   bool need_device, AttnPlan *plan);

struct AttnArgs {
    pf_pool *pool;
    int layer;
    const void *q;
    const void *k_new;   // fused decode step: new token rows (null: attention only)
    const void *v_new;
    bool overlap_previous;   // launch as a programmatic dependent of the previous kernel
    const int32_t *block_tables;
    int max_blocks;
    const int32_t *context_lens;
    int n_seqs;
    int n_q_heads;
    // rows per kv-head: its q-heads for decode; for an append (cu_q set),
    // the most query tokens of a sequence x its q-heads (at most 8)
    int rows;
    const int32_t *cu_q;   // append: query rows of sequence s are cu_q[s] .. cu_q[s + 1] - 1
    float scale;
    void *out;
    int out_dtype;
    AttnPlan plan;
    void *workspace;
    size_t ws_bytes;
};
int launch_attention(const AttnArgs &a, cudaStream_t stream);

}  // namespace pkv
