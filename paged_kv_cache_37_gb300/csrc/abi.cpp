// abi.cpp -- C ABI entry points of libpagedkv.so that are not the allocator:
// error reporting, pool descriptors, host-side argument validation and the
// dispatch of the device calls to their launchers.
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "internal.h"

namespace pkv {

namespace {
thread_local std::string g_last_error;
}

int set_error(int status, const std::string &msg) {
    g_last_error = msg;
    return status;
}

int cuda_error(cudaError_t err, const char *what) {
    return set_error(PF_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(err) + " (" +
                                      cudaGetErrorString(err) + ")");
}

void clear_error() { g_last_error.clear(); }

}  // namespace pkv

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_block_size(int b) { return b == 1 || b == 16 || b == 64 || b == 256; }

bool valid_head_dim(int d) { return d == 64 || d == 128; }

int check_pool(const pf_pool *pool, int layer, const char *fn) {
    if (!pool) return pkv::set_error(PF_ERR_INVALID, std::string(fn) + ": pool is null");
    if (layer < 0 || layer >= pool->n_layers)
        return pkv::set_error(PF_ERR_INVALID, std::string(fn) + ": layer " + std::to_string(layer) +
                                                  " outside [0, " + std::to_string(pool->n_layers) + ")");
    return PF_OK;
}

}  // namespace

extern "C" {

const char *pf_last_error(void) { return pkv::g_last_error.c_str(); }

int pf_abi_version(void) { return PF_ABI_VERSION; }

size_t pf_pool_bytes(int n_layers, int n_blocks, int block_size, int n_kv_heads, int head_dim,
                     int dtype) {
    if (n_layers <= 0 || n_blocks <= 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0 ||
        dtype != PF_F16)
        return 0;
    return (size_t)n_layers * (size_t)n_blocks * (size_t)block_size * (size_t)n_kv_heads *
           (size_t)head_dim * 2u;
}

int pf_pool_create(pf_pool **out, void *k_base, void *v_base, int n_layers, int n_blocks,
                   int block_size, int n_kv_heads, int head_dim, int dtype) {
    pkv::clear_error();
    if (!out) return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: out is null");
    *out = nullptr;
    if (!k_base || !v_base) return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: null pool pointer");
    if (!aligned16(k_base) || !aligned16(v_base))
        return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: pool pointers must be 16-byte aligned");
    if (dtype != PF_F16) return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: dtype must be PF_F16");
    if (!valid_head_dim(head_dim))
        return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: head_dim must be 64 or 128");
    if (!valid_block_size(block_size))
        return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: block_size must be 1, 16, 64 or 256");
    if (n_layers <= 0 || n_blocks <= 0 || n_kv_heads <= 0 || n_kv_heads > 256)
        return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: n_layers, n_blocks must be positive and "
                                              "n_kv_heads in [1, 256]");
    uint64_t rows = (uint64_t)n_layers * (uint64_t)n_blocks * (uint64_t)block_size;
    if (rows >= (1ull << 31))
        return pkv::set_error(PF_ERR_INVALID, "pf_pool_create: n_layers * n_blocks * block_size must be "
                                              "below 2^31 token rows");
    pf_pool *p = new (std::nothrow) pf_pool;
    if (!p) return pkv::set_error(PF_ERR_OOM, "pf_pool_create: host allocation failed");
    p->k_base = k_base;
    p->v_base = v_base;
    p->n_layers = n_layers;
    p->n_blocks = n_blocks;
    p->block_size = block_size;
    p->n_kv_heads = n_kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    for (int i = 0; i < pkv::kMaxDevices; ++i) {
        for (int j = 0; j < 6; ++j) p->tmap_ready[i][j] = false;
        p->tmap_pf_ready[i] = false;
    }
    *out = p;
    return PF_OK;
}

int pf_pool_destroy(pf_pool *pool) {
    pkv::clear_error();
    delete pool;
    return PF_OK;
}

int pf_write_kv(const pf_pool *pool, int layer, const void *k_new, const void *v_new,
                const int32_t *block_tables, int n_table_rows, int max_blocks_per_seq,
                const int32_t *seq_idx, const int32_t *pos, int n_tokens, void *stream) {
    pkv::clear_error();
    int rc = check_pool(pool, layer, "pf_write_kv");
    if (rc) return rc;
    if (n_tokens < 0) return pkv::set_error(PF_ERR_INVALID, "pf_write_kv: negative n_tokens");
    if (n_tokens == 0) return PF_OK;
    if (!k_new || !v_new || !block_tables || !seq_idx || !pos)
        return pkv::set_error(PF_ERR_INVALID, "pf_write_kv: null pointer");
    if (!aligned16(k_new) || !aligned16(v_new))
        return pkv::set_error(PF_ERR_INVALID, "pf_write_kv: k_new / v_new must be 16-byte aligned");
    if (max_blocks_per_seq <= 0 || n_table_rows <= 0)
        return pkv::set_error(PF_ERR_INVALID,
                              "pf_write_kv: n_table_rows and max_blocks_per_seq must be positive");
    pkv::WriteArgs a{pool, layer, k_new, v_new, block_tables, n_table_rows, max_blocks_per_seq,
                     seq_idx, pos, n_tokens};
    return pkv::launch_write_kv(a, static_cast<cudaStream_t>(stream));
}

int pf_gather_kv(const pf_pool *pool, int layer, const int32_t *block_tables, int max_blocks_per_seq,
                 const int32_t *context_lens, const int64_t *cu_off, int n_seqs, void *k_out,
                 void *v_out, void *stream) {
    pkv::clear_error();
    int rc = check_pool(pool, layer, "pf_gather_kv");
    if (rc) return rc;
    if (n_seqs < 0) return pkv::set_error(PF_ERR_INVALID, "pf_gather_kv: negative n_seqs");
    if (n_seqs == 0) return PF_OK;
    if (!block_tables || !context_lens || !cu_off || !k_out || !v_out)
        return pkv::set_error(PF_ERR_INVALID, "pf_gather_kv: null pointer");
    if (!aligned16(k_out) || !aligned16(v_out))
        return pkv::set_error(PF_ERR_INVALID, "pf_gather_kv: k_out / v_out must be 16-byte aligned");
    if (max_blocks_per_seq <= 0)
        return pkv::set_error(PF_ERR_INVALID, "pf_gather_kv: max_blocks_per_seq must be positive");
    pkv::GatherArgs a{pool, layer, block_tables, max_blocks_per_seq, context_lens, cu_off,
                      n_seqs, k_out, v_out};
    return pkv::launch_gather_kv(a, static_cast<cudaStream_t>(stream));
}

size_t pf_block_image_bytes(const pf_pool *pool) {
    if (!pool) return 0;
    return (size_t)pool->n_layers * 2 * pool->block_size * pool->n_kv_heads * pool->head_dim * sizeof(uint16_t);
}

int pf_copy_blocks(const pf_pool *pool, const int32_t *src_ids, const int32_t *dst_ids, int n, void *stream) {
    pkv::clear_error();
    if (!pool) return pkv::set_error(PF_ERR_INVALID, "pf_copy_blocks: pool is null");
    if (n < 0) return pkv::set_error(PF_ERR_INVALID, "pf_copy_blocks: negative count");
    if (n == 0) return PF_OK;
    if (!src_ids || !dst_ids) return pkv::set_error(PF_ERR_INVALID, "pf_copy_blocks: null id array");
    pkv::BlockCopyArgs a{pool, src_ids, dst_ids, nullptr, n};
    return pkv::launch_block_copy(a, static_cast<cudaStream_t>(stream));
}

// Device address of a page-locked host buffer (its mapping), or an error.
static int host_image_ptr(const void *host, void **dev_out, const char *what) {
    if (!host) return pkv::set_error(PF_ERR_INVALID, std::string(what) + ": host buffer is null");
    if (!aligned16(host)) return pkv::set_error(PF_ERR_INVALID, std::string(what) + ": host buffer must be 16-byte aligned");
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, host);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return pkv::cuda_error(e, (std::string(what) + ": cudaPointerGetAttributes").c_str());
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr)
        return pkv::set_error(PF_ERR_INVALID, std::string(what) +
                                                  ": host buffer must be page-locked host memory "
                                                  "(cudaHostAlloc, cudaHostRegister or a pinned tensor)");
    *dev_out = attr.devicePointer;
    return PF_OK;
}

int pf_swap_out(const pf_pool *pool, const int32_t *ids, int n, void *host_dst, void *stream) {
    pkv::clear_error();
    if (!pool) return pkv::set_error(PF_ERR_INVALID, "pf_swap_out: pool is null");
    if (n < 0) return pkv::set_error(PF_ERR_INVALID, "pf_swap_out: negative count");
    if (n == 0) return PF_OK;
    if (!ids) return pkv::set_error(PF_ERR_INVALID, "pf_swap_out: ids is null");
    void *img = nullptr;
    int rc = host_image_ptr(host_dst, &img, "pf_swap_out");
    if (rc) return rc;
    pkv::BlockCopyArgs a{pool, ids, nullptr, img, n};
    return pkv::launch_block_copy(a, static_cast<cudaStream_t>(stream));
}

int pf_swap_in(const pf_pool *pool, const void *host_src, const int32_t *ids, int n, void *stream) {
    pkv::clear_error();
    if (!pool) return pkv::set_error(PF_ERR_INVALID, "pf_swap_in: pool is null");
    if (n < 0) return pkv::set_error(PF_ERR_INVALID, "pf_swap_in: negative count");
    if (n == 0) return PF_OK;
    if (!ids) return pkv::set_error(PF_ERR_INVALID, "pf_swap_in: ids is null");
    void *img = nullptr;
    int rc = host_image_ptr(host_src, &img, "pf_swap_in");
    if (rc) return rc;
    pkv::BlockCopyArgs a{pool, nullptr, ids, img, n};
    return pkv::launch_block_copy(a, static_cast<cudaStream_t>(stream));
}

size_t pf_decode_workspace_bytes(const pf_pool *pool, int n_seqs, int n_q_heads, int max_blocks_per_seq,
                                 int split_tokens) {
    pkv::clear_error();
    if (!pool || n_seqs <= 0 || n_q_heads <= 0 || max_blocks_per_seq <= 0 ||
        n_q_heads % pool->n_kv_heads) {
        pkv::set_error(PF_ERR_INVALID, "pf_decode_workspace_bytes: bad arguments");
        return 0;
    }
    pkv::AttnPlan plan;
    if (pkv::attention_plan(pool, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens, false, &plan)) return 0;
    return plan.counter_bytes + plan.partial_bytes;
}

int pf_decode_workspace_init(void *workspace, size_t ws_bytes, void *stream) {
    pkv::clear_error();
    if (!workspace || ws_bytes == 0)
        return pkv::set_error(PF_ERR_INVALID, "pf_decode_workspace_init: null or empty workspace");
    cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv::cuda_error(e, "pf_decode_workspace_init: cudaMemsetAsync");
    return PF_OK;
}

// Checks and launch shared by pf_paged_decode_attention (k_new = v_new =
// null) and pf_decode_step (the fused write of the new token rows).
static int decode_call(const pf_pool *pool, int layer, const void *q, const void *k_new, const void *v_new,
                       bool overlap_previous, const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                       int n_seqs, int n_q_heads, float scale, void *out, int out_dtype, int split_tokens,
                       void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_pool(pool, layer, "pf_paged_decode_attention");
    if (rc) return rc;
    if (n_seqs < 0) return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention: negative n_seqs");
    if (n_seqs == 0) return PF_OK;
    if (!q || !block_tables || !context_lens || !out || !workspace)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention: null pointer");
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace))
        return pkv::set_error(PF_ERR_INVALID,
                              "pf_paged_decode_attention: q, out and workspace must be 16-byte aligned");
    if (out_dtype != PF_F16 && out_dtype != PF_F32)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention: out_dtype must be PF_F16 or PF_F32");
    if (n_q_heads <= 0 || n_q_heads % pool->n_kv_heads)
        return pkv::set_error(PF_ERR_INVALID,
                              "pf_paged_decode_attention: n_q_heads must be a positive multiple of n_kv_heads");
    int group = n_q_heads / pool->n_kv_heads;
    if (group > 16 || (group > 8 && (split_tokens != 0 || pool->block_size < 16)))
        return pkv::set_error(PF_ERR_UNSUPPORTED,
                              "pf_paged_decode_attention: at most 8 q-heads per kv-head are built (16 with "
                              "split_tokens = 0 and pages of at least 16 tokens)");
    if (max_blocks_per_seq <= 0)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention: max_blocks_per_seq must be positive");
    if (!(scale > 0.0f) || scale != scale)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention: scale must be a positive number");
    pkv::AttnPlan plan;
    // host-only checks first (no device query), then the device-sized plan
    rc = pkv::attention_plan(pool, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens, false, &plan);
    if (rc) return rc;
    if (ws_bytes < plan.counter_bytes)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention: workspace has " +
                                                  std::to_string(ws_bytes) + " bytes, needs at least " +
                                                  std::to_string(plan.counter_bytes));
    rc = pkv::attention_plan(pool, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens, true, &plan);
    if (rc) return rc;
    const size_t need = plan.counter_bytes + plan.partial_bytes;
    if (ws_bytes < need)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_decode_attention: workspace has " +
                                                  std::to_string(ws_bytes) + " bytes, needs " +
                                                  std::to_string(need));
    pkv::AttnArgs a{const_cast<pf_pool *>(pool), layer, q, k_new, v_new, overlap_previous, block_tables,
                    max_blocks_per_seq, context_lens, n_seqs, n_q_heads, n_q_heads / pool->n_kv_heads, nullptr,
                    scale, out, out_dtype, plan, workspace, ws_bytes};
    return pkv::launch_attention(a, static_cast<cudaStream_t>(stream));
}

int pf_paged_decode_attention(const pf_pool *pool, int layer, const void *q, const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *context_lens, int n_seqs, int n_q_heads,
                              float scale, void *out, int out_dtype, int split_tokens, void *workspace,
                              size_t ws_bytes, void *stream) {
    pkv::clear_error();
    return decode_call(pool, layer, q, nullptr, nullptr, false, block_tables, max_blocks_per_seq, context_lens, n_seqs,
                       n_q_heads, scale, out, out_dtype, split_tokens, workspace, ws_bytes, stream);
}

int pf_decode_step(const pf_pool *pool, int layer, const void *q, const void *k_new, const void *v_new,
                   const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens, int n_seqs,
                   int n_q_heads, float scale, void *out, int out_dtype, int split_tokens, void *workspace,
                   size_t ws_bytes, int flags, void *stream) {
    pkv::clear_error();
    if (flags & ~PF_STEP_OVERLAP_PREVIOUS)
        return pkv::set_error(PF_ERR_INVALID, "pf_decode_step: unknown flags " + std::to_string(flags));
    if (n_seqs > 0) {
        if (!k_new || !v_new) return pkv::set_error(PF_ERR_INVALID, "pf_decode_step: null k_new / v_new");
        if (!aligned16(k_new) || !aligned16(v_new))
            return pkv::set_error(PF_ERR_INVALID, "pf_decode_step: k_new / v_new must be 16-byte aligned");
    }
    // the same checks as pf_paged_decode_attention, then the fused launch
    return decode_call(pool, layer, q, k_new, v_new, (flags & PF_STEP_OVERLAP_PREVIOUS) != 0, block_tables,
                       max_blocks_per_seq, context_lens, n_seqs,
                       n_q_heads, scale, out, out_dtype, split_tokens, workspace, ws_bytes, stream);
}

// Rows per kv-head when an append takes the decode kernel (its query tokens
// x its q-heads), or 0 when they do not fit (the standalone kernel then).
// Rows per kv-head of an append on the decode kernel (query tokens x
// q-heads): up to 16 on pages of at least 16 tokens (the tensor-core
// consumers take 9 and more), up to 8 otherwise; 0 = too many.
static int append_rows(const pf_pool *pool, int n_q_heads, int max_new_tokens) {
    if (n_q_heads <= 0 || n_q_heads % pool->n_kv_heads) return 0;
    const long long rows = (long long)max_new_tokens * (n_q_heads / pool->n_kv_heads);
    const int cap = pool->block_size >= 16 ? 16 : 8;
    return rows >= 1 && rows <= cap ? (int)rows : 0;
}

size_t pf_prefill_workspace_bytes(const pf_pool *pool, int n_seqs, int n_q_heads, int max_blocks_per_seq,
                                  int max_new_tokens) {
    pkv::clear_error();
    if (!pool || n_seqs < 0 || max_blocks_per_seq <= 0 || max_new_tokens < 0) {
        pkv::set_error(PF_ERR_INVALID, "pf_prefill_workspace_bytes: bad arguments");
        return 0;
    }
    const int rows = append_rows(pool, n_q_heads, max_new_tokens);
    if (rows == 0) return 0;   // the call takes the kernel that needs no workspace
    pkv::AttnPlan plan;
    // sized like pf_decode_workspace_bytes: by the resident grid, or by a
    // bound on it when no device can be queried
    if (pkv::attention_plan(pool, n_seqs, rows * pool->n_kv_heads, max_blocks_per_seq, 0, false, &plan) != PF_OK)
        return 0;
    return plan.counter_bytes + plan.partial_bytes;
}

int pf_paged_prefill_attention(const pf_pool *pool, int layer, const void *q, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens, const int32_t *cu_q, int n_seqs,
                               int max_new_tokens, int n_q_heads, float scale, void *out, int out_dtype,
                               void *workspace, size_t ws_bytes, void *stream) {
    pkv::clear_error();
    int rc = check_pool(pool, layer, "pf_paged_prefill_attention");
    if (rc) return rc;
    if (n_seqs < 0 || max_new_tokens < 0)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: negative n_seqs or max_new_tokens");
    if (n_seqs == 0 || max_new_tokens == 0) return PF_OK;
    if (!q || !block_tables || !context_lens || !cu_q || !out)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: null pointer");
    if (!aligned16(q) || !aligned16(out))
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: q and out must be 16-byte aligned");
    if (out_dtype != PF_F16 && out_dtype != PF_F32)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: out_dtype must be PF_F16 or PF_F32");
    if (n_q_heads <= 0 || n_q_heads % pool->n_kv_heads)
        return pkv::set_error(PF_ERR_INVALID,
                              "pf_paged_prefill_attention: n_q_heads must be a positive multiple of n_kv_heads");
    if (n_q_heads / pool->n_kv_heads > 16)
        return pkv::set_error(PF_ERR_UNSUPPORTED, "pf_paged_prefill_attention: at most 16 q-heads per kv-head are built");
    if (max_blocks_per_seq <= 0 || (long long)max_blocks_per_seq * pool->block_size > (1ll << 30))
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: bad max_blocks_per_seq");
    if (!(scale > 0.0f) || scale != scale)
        return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: scale must be a positive number");
    const int rows = append_rows(pool, n_q_heads, max_new_tokens);
    if (workspace != nullptr && rows > 0) {
        // The decode kernel, its G rows per kv-head being the query tokens x
        // q-heads: balanced spans over the contexts, merged in the kernel.
        if (!aligned16(workspace))
            return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: workspace must be 16-byte aligned");
        pkv::AttnPlan plan;
        rc = pkv::attention_plan(pool, n_seqs, rows * pool->n_kv_heads, max_blocks_per_seq, 0, true, &plan);
        if (rc) return rc;
        const size_t need = plan.counter_bytes + plan.partial_bytes;
        if (ws_bytes < need)
            return pkv::set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: workspace has " +
                                                      std::to_string(ws_bytes) + " bytes, needs " +
                                                      std::to_string(need));
        pkv::AttnArgs a{const_cast<pf_pool *>(pool), layer, q, nullptr, nullptr, false, block_tables,
                        max_blocks_per_seq, context_lens, n_seqs, n_q_heads, rows, cu_q, scale, out, out_dtype, plan,
                        workspace, ws_bytes};
        return pkv::launch_attention(a, static_cast<cudaStream_t>(stream));
    }
    pkv::PrefillArgs a{pool, layer, q, block_tables, max_blocks_per_seq, context_lens, cu_q, n_seqs, max_new_tokens,
                       n_q_heads, scale, out, out_dtype};
    return pkv::launch_prefill(a, static_cast<cudaStream_t>(stream));
}

int pf_device_status(int *status_out, int reset, void *stream) {
    pkv::clear_error();
    if (!status_out) return pkv::set_error(PF_ERR_INVALID, "pf_device_status: status_out is null");
    int *dev = pkv::device_status_ptr();
    if (!dev) return PF_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, dev, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return pkv::cuda_error(e, "pf_device_status: read");
    *status_out = host;
    if (reset) {
        e = cudaMemsetAsync(dev, 0, sizeof(int), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return pkv::cuda_error(e, "pf_device_status: reset");
    }
    return PF_OK;
}

}  // extern "C"
