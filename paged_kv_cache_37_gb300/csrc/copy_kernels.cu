// copy_kernels.cu -- scatter (pf_write_kv) and gather (pf_gather_kv) of token
// rows between dense buffers and the paged pool, plus the device status word.
//
// A token row of one layer is n_kv_heads * head_dim fp16 values, contiguous in
// the pool at slot table[t / B] * B + t % B ("Why Naive KV-Caches Waste >60%
// VRAM", section 1), and contiguous in the dense buffers.  Both kernels move
// whole rows with 16-byte streaming loads/stores; a page of B rows is itself
// contiguous, so every access is fully coalesced.  Pure copies: bit-exact.
#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {

__device__ int g_device_status;

int *device_status_ptr() {
    static std::mutex mu;
    static int *cache[kMaxDevices] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cuda_error(e, "cudaGetDevice");
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error(PF_ERR_UNSUPPORTED, "device index out of range");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) {
            cuda_error(e, "cudaGetSymbolAddress(device status)");
            return nullptr;
        }
        cache[dev] = static_cast<int *>(p);
    }
    return cache[dev];
}

namespace {

constexpr int kCopyThreads = 256;
constexpr int kGatherRows = 64;     // token rows per gather CTA
constexpr int kUnroll = 4;          // 16-byte vectors in flight per thread

// ---------------------------------------------------------------- scatter

struct WriteParams {
    uint4 *k_pool;
    uint4 *v_pool;
    const uint4 *k_new;
    const uint4 *v_new;
    const int32_t *bt;
    const int32_t *seq_idx;
    const int32_t *pos;
    int *status;
    int n_rows_table;   // rows of the block table
    int max_blocks;
    int n_blocks;
    int block_size;
    int64_t layer_row0; // layer * n_blocks * block_size
    int vecs_per_row;   // n_kv_heads * head_dim / 8
    int n_tokens;
};

// One CTA per token (grid-stride): K and V rows of the token, 16 B per thread.
__global__ void __launch_bounds__(kCopyThreads) write_kv_kernel(const WriteParams p) {
    for (int i = blockIdx.x; i < p.n_tokens; i += gridDim.x) {
        const int s = p.seq_idx[i];
        const int t = p.pos[i];
        if (s < 0 || s >= p.n_rows_table || t < 0 || t / p.block_size >= p.max_blocks) {
            if (threadIdx.x == 0) atomicOr(p.status, PF_DEV_BAD_POSITION);
            continue;
        }
        const int blk = p.bt[(int64_t)s * p.max_blocks + t / p.block_size];
        if (blk < 0 || blk >= p.n_blocks) {
            if (threadIdx.x == 0) atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
            continue;
        }
        const int64_t dst = (p.layer_row0 + (int64_t)blk * p.block_size + t % p.block_size) * p.vecs_per_row;
        const int64_t src = (int64_t)i * p.vecs_per_row;
        for (int c = threadIdx.x; c < 2 * p.vecs_per_row; c += blockDim.x) {
            if (c < p.vecs_per_row) {
                st_stream(p.k_pool + dst + c, ld_stream(p.k_new + src + c));
            } else {
                const int cc = c - p.vecs_per_row;
                st_stream(p.v_pool + dst + cc, ld_stream(p.v_new + src + cc));
            }
        }
    }
}

// ----------------------------------------------------------------- gather

struct GatherParams {
    const uint4 *k_pool;
    const uint4 *v_pool;
    uint4 *k_out;
    uint4 *v_out;
    const int32_t *bt;
    const int32_t *lens;
    const int64_t *cu_off;
    int *status;
    int max_blocks;
    int n_blocks;
    int block_size;
    int64_t layer_row0;
    int vecs_per_row;
};

// CTA (y, s) copies rows [y * kGatherRows, ...) of sequence s; CTAs past the
// end of a sequence exit at once.  Each warp moves whole rows, kUnroll
// vectors per lane in flight.
__global__ void __launch_bounds__(kCopyThreads) gather_kv_kernel(const GatherParams p) {
    __shared__ int64_t src_row[kGatherRows];   // pool row of each token of this CTA
    __shared__ int n_rows_sh;
    __shared__ int64_t out_row0_sh;
    const int s = blockIdx.y;
    const int r0 = blockIdx.x * kGatherRows;
    if (threadIdx.x == 0) {
        int L = p.lens[s];
        const int maxctx = p.max_blocks * p.block_size;
        if (L < 0 || L > maxctx) {
            atomicOr(p.status, PF_DEV_BAD_LENGTH);
            L = L < 0 ? 0 : maxctx;
        }
        n_rows_sh = max(0, min(kGatherRows, L - r0));
        out_row0_sh = n_rows_sh > 0 ? p.cu_off[s] + r0 : 0;
    }
    __syncthreads();
    const int n_rows = n_rows_sh;
    if (n_rows == 0) return;
    if (threadIdx.x < n_rows) {
        const int t = r0 + threadIdx.x;
        int blk = p.bt[(int64_t)s * p.max_blocks + t / p.block_size];
        if (blk < 0 || blk >= p.n_blocks) {
            atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
            blk = -1;
        }
        src_row[threadIdx.x] = blk < 0 ? -1 : p.layer_row0 + (int64_t)blk * p.block_size + t % p.block_size;
    }
    __syncthreads();
    const int64_t out_row0 = out_row0_sh;
    const int vpr = p.vecs_per_row;
    const int total = n_rows * vpr;     // vectors this CTA moves for K (same for V)
    // Flattened (row, vector) index; kUnroll vectors per thread per round.
    for (int base = threadIdx.x; base < 2 * total; base += kCopyThreads * kUnroll) {
        uint4 v[kUnroll];
        int64_t dst[kUnroll];
        bool ok[kUnroll], is_v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int idx = base + u * kCopyThreads;
            ok[u] = false;
            is_v[u] = idx >= total;
            if (idx < 2 * total) {
                const int j = is_v[u] ? idx - total : idx;
                const int r = j / vpr;
                const int c = j - r * vpr;
                const int64_t sr = src_row[r];
                if (sr >= 0) {
                    v[u] = ld_stream((is_v[u] ? p.v_pool : p.k_pool) + sr * vpr + c);
                    dst[u] = (out_row0 + r) * vpr + c;
                    ok[u] = true;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (ok[u]) st_stream((is_v[u] ? p.v_out : p.k_out) + dst[u], v[u]);
    }
}

}  // namespace

int launch_write_kv(const WriteArgs &a, cudaStream_t stream) {
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;
    const pf_pool *pool = a.pool;
    WriteParams p;
    p.k_pool = static_cast<uint4 *>(pool->k_base);
    p.v_pool = static_cast<uint4 *>(pool->v_base);
    p.k_new = static_cast<const uint4 *>(a.k_new);
    p.v_new = static_cast<const uint4 *>(a.v_new);
    p.bt = a.block_tables;
    p.seq_idx = a.seq_idx;
    p.pos = a.pos;
    p.status = status;
    p.n_rows_table = a.n_table_rows;
    p.max_blocks = a.max_blocks;
    p.n_blocks = pool->n_blocks;
    p.block_size = pool->block_size;
    p.layer_row0 = (int64_t)a.layer * pool->n_blocks * pool->block_size;
    p.vecs_per_row = pool->n_kv_heads * pool->head_dim / 8;
    p.n_tokens = a.n_tokens;
    const int grid = a.n_tokens < 65535 ? a.n_tokens : 65535;
    write_kv_kernel<<<grid, kCopyThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "pf_write_kv: launch");
    return PF_OK;
}

int launch_gather_kv(const GatherArgs &a, cudaStream_t stream) {
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;
    const pf_pool *pool = a.pool;
    if (a.n_seqs > 65535)
        return set_error(PF_ERR_INVALID, "pf_gather_kv: at most 65535 sequences per call");
    GatherParams p;
    p.k_pool = static_cast<const uint4 *>(pool->k_base);
    p.v_pool = static_cast<const uint4 *>(pool->v_base);
    p.k_out = static_cast<uint4 *>(a.k_out);
    p.v_out = static_cast<uint4 *>(a.v_out);
    p.bt = a.block_tables;
    p.lens = a.context_lens;
    p.cu_off = a.cu_off;
    p.status = status;
    p.max_blocks = a.max_blocks;
    p.n_blocks = pool->n_blocks;
    p.block_size = pool->block_size;
    p.layer_row0 = (int64_t)a.layer * pool->n_blocks * pool->block_size;
    p.vecs_per_row = pool->n_kv_heads * pool->head_dim / 8;
    const int64_t maxctx = (int64_t)a.max_blocks * pool->block_size;
    const int64_t gx = (maxctx + kGatherRows - 1) / kGatherRows;
    if (gx > 0x7fffffff) return set_error(PF_ERR_INVALID, "pf_gather_kv: table too wide");
    dim3 grid((unsigned)gx, (unsigned)a.n_seqs);
    gather_kv_kernel<<<grid, kCopyThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "pf_gather_kv: launch");
    return PF_OK;
}

}  // namespace pkv
