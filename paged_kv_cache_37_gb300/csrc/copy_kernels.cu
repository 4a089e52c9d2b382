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

// Gather with bulk copies: the tokens of every sequence are cut into chunks
// of CR consecutive rows (a power of two, at most the page size for pages of
// 16 tokens or more, so a chunk lies inside one page), and chunk u = (sequence, chunk)
// goes to CTA u mod grid (grid = one CTA per SM).  A chunk's K and V rows are
// each one contiguous run in the pool (a row per page for 1-token pages) and
// in the output, so they move by bulk copies through a ring of shared-memory
// stages: one thread loads pool -> stage (completing on the stage's full
// mbarrier), another stores stage -> output (a bulk group) and, once the
// store has read the stage, hands it back on its empty mbarrier.  Every CTA first scans the lengths into the
// chunk counts' prefix (at most kBulkGatherMaxSeqs sequences).
constexpr int kBulkGatherMaxStages = 16;
constexpr int kBulkGatherMaxSeqs = 4096;
constexpr int kBulkGatherThreads = 128;
constexpr uint32_t kBulkGatherRingBytes = 192 * 1024;   // all stages (K and V of a chunk each)
constexpr int kBulkGatherMaxRows = 64;                  // rows per chunk, at most

struct BulkGatherParams {
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    uint8_t *k_out;
    uint8_t *v_out;
    const int32_t *bt;
    const int32_t *lens;
    const int64_t *cu_off;
    int *status;
    int n_seqs;
    int max_blocks;
    int n_blocks;
    int block_size;
    int64_t layer_row0;
    uint32_t row_bytes;   // n_kv_heads * head_dim * 2
    int chunk_rows;       // CR
    int stages;           // kBulkGatherRingBytes / (2 * CR * row_bytes), at most kBulkGatherMaxStages
};

__global__ void __launch_bounds__(kBulkGatherThreads, 1) gather_kv_bulk_kernel(const BulkGatherParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int NST = p.stages;
    const uint32_t chunk_bytes = (uint32_t)p.chunk_rows * p.row_bytes;
    uint8_t *stage = smem_raw;   // [NST][K, V][chunk_bytes]
    int *pre = reinterpret_cast<int *>(smem_raw + (size_t)NST * 2 * chunk_bytes);   // [n_seqs + 1]
    __shared__ uint64_t full[kBulkGatherMaxStages];
    __shared__ uint64_t empty[kBulkGatherMaxStages];
    __shared__ int warp_tot[kBulkGatherThreads / 32];
    const int S = p.n_seqs;
    const int CR = p.chunk_rows;
    const int maxctx = p.max_blocks * p.block_size;
    const int lane = threadIdx.x % 32;
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), 1);
        }
        mbar_init_fence();
    }
    // chunks of every sequence (clamped lengths), then their exclusive prefix
    for (int s = threadIdx.x; s < S; s += kBulkGatherThreads) {
        int L = p.lens[s];
        if (L < 0 || L > maxctx) {
            if (blockIdx.x == 0) atomicOr(p.status, PF_DEV_BAD_LENGTH);
            L = L < 0 ? 0 : maxctx;
        }
        pre[s + 1] = (L + CR - 1) / CR;
    }
    __syncthreads();
    const int per = (S + kBulkGatherThreads - 1) / kBulkGatherThreads;
    const int lo = 1 + threadIdx.x * per;
    const int hi = min(S + 1, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += pre[i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += warp_tot[w];
    for (int i = lo; i < hi; ++i) {
        run += pre[i];
        pre[i] = run;
    }
    if (threadIdx.x == 0) pre[0] = 0;
    __syncthreads();
    // thread 0 of warp 0 loads chunks into free stages; thread 0 of warp 1
    // stores the landed ones and hands their stages back
    if (lane != 0 || warp > 1) return;

    const int total = pre[S];
    const int n_local = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    // Chunk u: its sequence s (largest s with pre[s] <= u), first row r0 and
    // rows n; ok = false when one of its pages is not in the pool (flagged
    // by the loader, skipped by both).
    auto chunk_of = [&](int u, int &s, int &r0, int &n, bool &ok) {
        int a = 0, b = S - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (pre[mid] <= u) a = mid;
            else b = mid - 1;
        }
        s = a;
        int L = p.lens[s];
        L = L < 0 ? 0 : (L > maxctx ? maxctx : L);
        r0 = (u - pre[s]) * CR;
        n = min(CR, L - r0);
        const int32_t *row = p.bt + (size_t)s * p.max_blocks;
        ok = true;
        const int pages = p.block_size >= CR ? 1 : n;
        for (int j = 0; j < pages; ++j) {
            const int blk = row[(r0 + j) / p.block_size];
            if (blk < 0 || blk >= p.n_blocks) ok = false;
        }
    };
    if (warp == 0) {
        // loader
        int issued = 0;
        for (int i = 0; i < n_local; ++i) {
            const int st = i % NST;
            if (i >= NST && !mbar_wait(smem_addr(&empty[st]), ((i / NST) - 1) & 1, p.status)) break;
            const uint32_t bar = smem_addr(&full[st]);
            uint8_t *dk = stage + (size_t)st * 2 * chunk_bytes;
            uint8_t *dv = dk + chunk_bytes;
            int s, r0, n;
            bool ok;
            chunk_of((int)blockIdx.x + i * (int)gridDim.x, s, r0, n, ok);
            ++issued;
            if (!ok) {
                atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
                mbar_arrive(bar);   // completes the phase with no bytes
                continue;
            }
            const int32_t *row = p.bt + (size_t)s * p.max_blocks;
            mbar_arrive_expect_tx(bar, 2u * (uint32_t)n * p.row_bytes);
            if (p.block_size >= CR) {
                const int64_t src = p.layer_row0 + (int64_t)row[r0 / p.block_size] * p.block_size + r0 % p.block_size;
                bulk_load(smem_addr(dk), p.k_pool + src * p.row_bytes, (uint32_t)n * p.row_bytes, bar);
                bulk_load(smem_addr(dv), p.v_pool + src * p.row_bytes, (uint32_t)n * p.row_bytes, bar);
            } else {   // one row per page
                for (int j = 0; j < n; ++j) {
                    const int64_t src = p.layer_row0 + (int64_t)row[r0 + j] * p.block_size;
                    bulk_load(smem_addr(dk + j * p.row_bytes), p.k_pool + src * p.row_bytes, p.row_bytes, bar);
                    bulk_load(smem_addr(dv + j * p.row_bytes), p.v_pool + src * p.row_bytes, p.row_bytes, bar);
                }
            }
        }
        // the loads still in flight land before the CTA ends (bounded; only
        // after a wait gave up are there any the storer did not wait for)
        for (int i = issued - NST > 0 ? issued - NST : 0; i < issued; ++i)
            mbar_wait(smem_addr(&full[i % NST]), (i / NST) & 1, p.status);
    } else {
        // storer: up to two stores in flight; a stage goes back to the loader
        // once the store from it has read it
        int stored = 0;
        for (int i = 0; i < n_local; ++i) {
            const int st = i % NST;
            if (!mbar_wait(smem_addr(&full[st]), (i / NST) & 1, p.status)) break;
            int s, r0, n;
            bool ok;
            chunk_of((int)blockIdx.x + i * (int)gridDim.x, s, r0, n, ok);
            if (ok) {
                uint8_t *dk = stage + (size_t)st * 2 * chunk_bytes;
                const int64_t dst = (p.cu_off[s] + r0) * (int64_t)p.row_bytes;
                bulk_store(p.k_out + dst, smem_addr(dk), (uint32_t)n * p.row_bytes);
                bulk_store(p.v_out + dst, smem_addr(dk + chunk_bytes), (uint32_t)n * p.row_bytes);
            }
            bulk_commit();
            stored = i + 1;
            if (i >= 1) {
                bulk_wait_read<1>();   // the store of chunk i - 1 has read its stage
                mbar_arrive(smem_addr(&empty[(i - 1) % NST]));
            }
        }
        bulk_wait<0>();   // every store has reached global memory
        if (stored > 0) mbar_arrive(smem_addr(&empty[(stored - 1) % NST]));
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
    // bulk-copy path: chunks of CR rows (a power of two, within a page on
    // pages of 16 tokens or more, at most 64 rows) whose K and V take at most
    // 48 KB, at least 4 stages in the 192 KB ring; a length scan that fits
    // the CTA's shared memory
    const uint32_t row_bytes = (uint32_t)pool->n_kv_heads * pool->head_dim * 2;
    int cr = pool->block_size >= 16 ? pool->block_size : kBulkGatherMaxRows;
    if (cr > kBulkGatherMaxRows) cr = kBulkGatherMaxRows;
    while (cr > 1 && 2u * (uint32_t)cr * row_bytes > kBulkGatherRingBytes / 4) cr >>= 1;
    int stages = (int)(kBulkGatherRingBytes / (2u * (uint32_t)cr * row_bytes));
    if (stages > kBulkGatherMaxStages) stages = kBulkGatherMaxStages;
    const int64_t maxctx_b = (int64_t)a.max_blocks * pool->block_size;
    if (stages >= 4 && a.n_seqs <= kBulkGatherMaxSeqs && maxctx_b <= (1 << 30)) {
        BulkGatherParams b;
        b.k_pool = static_cast<const uint8_t *>(pool->k_base);
        b.v_pool = static_cast<const uint8_t *>(pool->v_base);
        b.k_out = static_cast<uint8_t *>(a.k_out);
        b.v_out = static_cast<uint8_t *>(a.v_out);
        b.bt = a.block_tables;
        b.lens = a.context_lens;
        b.cu_off = a.cu_off;
        b.status = status;
        b.n_seqs = a.n_seqs;
        b.max_blocks = a.max_blocks;
        b.n_blocks = pool->n_blocks;
        b.block_size = pool->block_size;
        b.layer_row0 = p.layer_row0;
        b.row_bytes = row_bytes;
        b.chunk_rows = cr;
        b.stages = stages;
        const size_t smem = (size_t)stages * 2 * cr * row_bytes + ((size_t)a.n_seqs + 1) * 4;
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gather_kv_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_error(e, "pf_gather_kv: set-up");
        gather_kv_bulk_kernel<<<sms, kBulkGatherThreads, smem, stream>>>(b);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_error(e, "pf_gather_kv: launch");
        return PF_OK;
    }
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
