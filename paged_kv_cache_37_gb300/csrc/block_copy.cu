// block_copy.cu -- whole-block copies: copy-on-write copies inside the pool
// (pf_copy_blocks) and swapping blocks to and from host memory (pf_swap_out,
// pf_swap_in).
//
// A block of one layer is B * Hkv * D fp16 values, contiguous in the pool
// (PageForge, "Four layers, one pointer": one page holds all heads of its
// tokens).  A copy-on-write gives a diverging sequence its own copy of a
// shared block in every layer (PagedAttention blog, "Copy-on-Write for
// Parallel Sampling"); swapping moves a block's contents, every layer, K and
// V, to CPU memory and back (same blog, "Preemption and Swapping").  The host
// side is a sequence of block images [n_layers][2][B][Hkv][D].
//
// One CTA moves one (block, layer, K or V) with 16-byte vectors, several in
// flight per thread.  For swapping, the kernel reads or writes the
// page-locked host buffer directly through its device mapping (on GB300 the
// Grace memory is reached over NVLink-C2C), so no staging buffer and no
// per-block memcpy is needed.  Pure copies: bit-exact.
#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // 16-byte vectors in flight per thread

struct BlockCopyParams {
    // pool bases, or (when the ids on that side are null) the image array in
    // the *_k pointer
    const uint4 *src_k;
    const uint4 *src_v;
    uint4 *dst_k;
    uint4 *dst_v;
    const int32_t *src_ids;   // null: source i is image i
    const int32_t *dst_ids;   // null: destination i is image i
    int *status;
    int n_layers;
    int n_blocks;
    int64_t vecs;             // 16-byte vectors per block of one layer
};

// Address of (item i, layer, kv) on one side, or null for a bad block id.
__device__ __forceinline__ const uint4 *side_addr(const uint4 *pool_k, const uint4 *pool_v, const int32_t *ids,
                                                  int i, int layer, int kv, const BlockCopyParams &p) {
    if (ids == nullptr) return pool_k + (((int64_t)i * p.n_layers + layer) * 2 + kv) * p.vecs;
    const int b = ids[i];
    if (b < 0 || b >= p.n_blocks) return nullptr;
    return (kv ? pool_v : pool_k) + ((int64_t)layer * p.n_blocks + b) * p.vecs;
}

__global__ void __launch_bounds__(kThreads) block_copy_kernel(const BlockCopyParams p) {
    const int i = blockIdx.x;
    const int layer = blockIdx.y >> 1;
    const int kv = blockIdx.y & 1;
    const uint4 *src = side_addr(p.src_k, p.src_v, p.src_ids, i, layer, kv, p);
    uint4 *dst = const_cast<uint4 *>(side_addr(p.dst_k, p.dst_v, p.dst_ids, i, layer, kv, p));
    if (src == nullptr || dst == nullptr) {
        if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
        return;   // the pair is skipped in every layer
    }
    for (int64_t v0 = threadIdx.x; v0 < p.vecs; v0 += (int64_t)kThreads * kUnroll) {
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            if (v < p.vecs) x[u] = ld_stream(src + v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            if (v < p.vecs) st_stream(dst + v, x[u]);
        }
    }
}

}  // namespace

int launch_block_copy(const BlockCopyArgs &a, cudaStream_t stream) {
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;
    const pf_pool *pool = a.pool;
    if (pool->n_layers > 65535 / 2) return set_error(PF_ERR_INVALID, "block copy: too many layers for one launch");
    BlockCopyParams p;
    const uint4 *pk = static_cast<const uint4 *>(pool->k_base);
    const uint4 *pv = static_cast<const uint4 *>(pool->v_base);
    if (a.src_ids) {
        p.src_k = pk;
        p.src_v = pv;
    } else {
        p.src_k = static_cast<const uint4 *>(a.image);
        p.src_v = nullptr;
    }
    if (a.dst_ids) {
        p.dst_k = const_cast<uint4 *>(pk);
        p.dst_v = const_cast<uint4 *>(pv);
    } else {
        p.dst_k = static_cast<uint4 *>(const_cast<void *>(a.image));
        p.dst_v = nullptr;
    }
    p.src_ids = a.src_ids;
    p.dst_ids = a.dst_ids;
    p.status = status;
    p.n_layers = pool->n_layers;
    p.n_blocks = pool->n_blocks;
    p.vecs = (int64_t)pool->block_size * pool->n_kv_heads * pool->head_dim / 8;
    dim3 grid((unsigned)a.n, (unsigned)(pool->n_layers * 2));
    block_copy_kernel<<<grid, kThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "block copy: launch");
    return PF_OK;
}

}  // namespace pkv
