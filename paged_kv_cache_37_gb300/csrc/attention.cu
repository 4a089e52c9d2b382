// attention.cu -- host side of pf_paged_decode_attention: TMA descriptors
// over the pool, the split heuristic, workspace layout and the launch of the
// persistent kernel (device code in attention_kernel.cuh).
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "attention_kernel.cuh"
#include "internal.h"

namespace pkv {
namespace {

using attn::KernelFn;
using attn::KernelInfo;
using attn::TB;

struct LaunchShape {
    bool ready = false;
    int grid = 0;
};

std::mutex g_shape_mu;
LaunchShape g_shapes[kMaxDevices][2][17][5][2];

// Kv-heads with at least this many rows (q-heads, or query tokens x
// q-heads) take the tensor-core consumers when the call runs the span
// schedule (the CUDA-core consumers serve fixed chunks).  Measured (256 sequences of U[32, 4096]
// tokens, GB/s, CUDA-core vs tensor-core consumers with their heads per
// item): head_dim 64, 1 row 5593 vs 6358, 2 rows 4105 vs 6111, 3 rows 2402
// vs 6044, 8 rows 1132 vs 3324; head_dim 128, 1 row 4180 vs 6123, 8 rows 867
// vs 5248.
#ifndef PKV_MMA_MIN_ROWS_D64
#define PKV_MMA_MIN_ROWS_D64 1
#endif
#ifndef PKV_MMA_MIN_ROWS_D128
#define PKV_MMA_MIN_ROWS_D128 1
#endif
constexpr int kMmaMaxRows = 16;
int mma_min_rows(int head_dim) { return head_dim == 64 ? PKV_MMA_MIN_ROWS_D64 : PKV_MMA_MIN_ROWS_D128; }

// kv-heads per item of the tensor-core consumers: as many as the pool has,
// up to PKV_MMA_MAX_HEADS (the boxes of a token's heads are issued back to
// back, so more heads read longer runs of each page row), 2 at head_dim 128
// above 8 rows (shared memory).
#ifndef PKV_MMA_MAX_HEADS
#define PKV_MMA_MAX_HEADS 4
#endif
int mma_heads(int n_kv_heads, int rows, int head_dim) {
    int hg = n_kv_heads >= 4 ? 4 : (n_kv_heads >= 2 ? 2 : 1);
    if (hg > PKV_MMA_MAX_HEADS) hg = PKV_MMA_MAX_HEADS;
    if (head_dim == 128 && rows > 8 && hg > 2) hg = 2;
    return hg;
}

KernelInfo kernel_mma(int head_dim, int rows, int hg) {
    if (head_dim == 64) return rows <= 8 ? attn::kernel_mma_d64_s(rows, hg) : attn::kernel_mma_d64_l(rows, hg);
    return rows <= 8 ? attn::kernel_mma_d128_s(rows, hg) : attn::kernel_mma_d128_l(rows, hg);
}

// kv-heads per work item: 4 (a 512 B run per token at head_dim 64), fewer
// when the pool has fewer heads or a kv-head has many rows (q-heads, or
// query tokens x q-heads): the consumer warps of a head then split its rows,
// 2 each from 5 rows up and from 3 up with 2 heads.
int heads_per_item(int n_kv_heads, int rows) {
    int hg = n_kv_heads >= 4 ? 4 : (n_kv_heads >= 2 ? 2 : 1);
    if (rows >= 5) hg = 1;
    else if (rows >= 3 && hg > 2) hg = 2;
    return hg;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// hg > 0: boxes {D, hg heads, TB rows}, unswizzled.  hg < 0: the
// tensor-core layout for -hg kv-heads, 64-element halves of a row swizzled
// in 128-byte rows, one box per tile with the heads outermost: the map's
// dimensions are ordered (64 elements, rows, heads) at head_dim 64 and (64,
// rows, halves, heads) at 128 (strides need not grow with the dimension), so
// a box {64, TB, (2,) -hg} lands as [head][half][row][64] -- each head's
// 16-row, 128-byte-row blocks contiguous, swizzled by row mod 8.
int encode_one(CUtensorMap *map, void *base, const pf_pool *pool, int hg) {
    auto encode = get_encode_fn();
    if (!encode) return set_error(PF_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const uint64_t rows = (uint64_t)pool->n_layers * pool->n_blocks * pool->block_size;
    const cuuint64_t D = (cuuint64_t)pool->head_dim;
    const cuuint64_t H = (cuuint64_t)pool->n_kv_heads;
    const int box_rows = pool->block_size < TB ? pool->block_size : TB;
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r;
    if (hg > 0) {
        cuuint64_t dims[3] = {D, H, (cuuint64_t)rows};
        cuuint64_t strides[2] = {D * 2, H * D * 2};
        cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)hg, (cuuint32_t)box_rows};
        r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (D == 64) {
        cuuint64_t dims[3] = {64, (cuuint64_t)rows, H};
        cuuint64_t strides[2] = {H * D * 2, D * 2};
        cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, (cuuint32_t)(-hg)};
        r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[4] = {64, (cuuint64_t)rows, D / 64, H};
        cuuint64_t strides[3] = {H * D * 2, 128, D * 2};
        cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, (cuuint32_t)(D / 64), (cuuint32_t)(-hg)};
        r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS)
        return set_error(PF_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r));
    return PF_OK;
}

}  // namespace

int encode_pool_tmaps(pf_pool *pool, int device, int hg, int *index) {
    const int a = hg < 0 ? -hg : hg;
    const int i = (hg < 0 ? 3 : 0) + (a == 1 ? 0 : (a == 2 ? 1 : 2));
    *index = i;
    std::lock_guard<std::mutex> lock(pool->mu);
    if (pool->tmap_ready[device][i]) return PF_OK;
    int rc = encode_one(&pool->tmap_k[device][i], pool->k_base, pool, hg);
    if (rc) return rc;
    rc = encode_one(&pool->tmap_v[device][i], pool->v_base, pool, hg);
    if (rc) return rc;
    pool->tmap_ready[device][i] = true;
    return PF_OK;
}

namespace {

// The kernel for G = n_q_heads / n_kv_heads rows per kv-head: *hg its
// kv-heads per item, *mma whether it has the tensor-core consumers (one
// kv-head per item, its tensor map the swizzled one).  The tensor-core
// consumers serve the balanced schedule unless the call asks for the CUDA
// cores.
int kernel_for(const pf_pool *pool, int n_q_heads, bool spans, bool cuda_cores, KernelInfo *ki, int *hg,
               bool *mma) {
    const int G = n_q_heads / pool->n_kv_heads;
    *mma = spans && !cuda_cores && G >= mma_min_rows(pool->head_dim) && G <= kMmaMaxRows;
    if (*mma) {
        *hg = mma_heads(pool->n_kv_heads, G, pool->head_dim);
        *ki = kernel_mma(pool->head_dim, G, *hg);
    } else {
        *hg = heads_per_item(pool->n_kv_heads, G);
        *ki = pool->head_dim == 64 ? attn::kernel_d64(G, *hg) : attn::kernel_d128(G, *hg);
    }
    if (!ki->fn || ki->smem == 0) return set_error(PF_ERR_UNSUPPORTED, "attention: unsupported head_dim / group");
    return PF_OK;
}

// Persistent grid of the kernel on the current device: SMs x resident CTAs.
int resident_grid(const pf_pool *pool, int n_q_heads, bool spans, bool cuda_cores, int *grid) {
    KernelInfo ki;
    int HG = 0;
    bool mma = false;
    int rc = kernel_for(pool, n_q_heads, spans, cuda_cores, &ki, &HG, &mma);
    if (rc) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "attention: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(PF_ERR_UNSUPPORTED, "device index out of range");
    const int D = pool->head_dim;
    const int G = n_q_heads / pool->n_kv_heads;
    std::lock_guard<std::mutex> lock(g_shape_mu);
    LaunchShape &sh = g_shapes[dev][D == 64 ? 0 : 1][G][HG][mma ? 1 : 0];
    if (!sh.ready) {
        const void *fn_ptr = reinterpret_cast<const void *>(ki.fn);
        for (KernelFn f : {ki.fn, ki.fn32}) {   // fp16 and fp32 output instances
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(f), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)ki.smem);
            if (e != cudaSuccess) return cuda_error(e, "attention: cudaFuncSetAttribute");
        }
        int occ = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn_ptr, attn::NTHREADS, ki.smem);
        if (e != cudaSuccess) return cuda_error(e, "attention: occupancy query");
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_error(e, "attention: SM count");
        if (occ < 1) return set_error(PF_ERR_UNSUPPORTED, "attention: kernel does not fit on an SM");
        sh.grid = sms * occ;
        sh.ready = true;
    }
    *grid = sh.grid;
    return PF_OK;
}

// Merge-job stamp of each main-kernel launch (never 0, so a zeroed
// workspace holds no job of any launch).
std::atomic<unsigned> g_epoch{0};
unsigned next_epoch() {
    unsigned e = ++g_epoch;
    if (e == 0) e = ++g_epoch;
    return e;
}

// Grid bound used to size span records when no device can be queried.
constexpr int kGridBoundNoDevice = 4096;

// pf_test_inject_wait_timeout: block 0 of the next launch leaves its first
// ring stage unfilled.
std::atomic<int> g_inject_timeout{0};



}  // namespace

int attention_plan(const pf_pool *pool, int n_seqs, int n_q_heads, int max_blocks, int split_tokens,
                   bool need_device, AttnPlan *plan) {
    const long long maxctx = (long long)max_blocks * pool->block_size;
    const long long cap = (maxctx + TB - 1) / TB * TB;
    if (cap > (1ll << 30))
        return set_error(PF_ERR_INVALID, "attention: max_blocks_per_seq * block_size is too large");
    if (split_tokens < -2)
        return set_error(PF_ERR_INVALID, "attention: split_tokens must be -2, -1, 0 or positive");
    KernelInfo ki;
    int HG = 0;
    bool mma = false;
    plan->spans = split_tokens == 0 || split_tokens == -2;
    plan->cuda_cores = split_tokens != 0;
    int rc = kernel_for(pool, n_q_heads, plan->spans, plan->cuda_cores, &ki, &HG, &mma);
    if (rc) return rc;
    // a record: the rows of the kernel instance x (D + 2) words (acc, m, l);
    // fp32 for fixed chunks, 64-bit (value, epoch) for spans
    const size_t rec_words = (size_t)ki.rows * (size_t)(pool->head_dim + 2);
    const int per_launch = n_seqs < attn::kMaxSeqsPerLaunch ? n_seqs : attn::kMaxSeqsPerLaunch;
    plan->grid = 0;
    if (need_device) {
        rc = resident_grid(pool, n_q_heads, plan->spans, plan->cuda_cores, &plan->grid);
        if (rc) return rc;
    }
    // [reserved: 256 B][records][merge jobs]
    plan->counter_bytes = 256;
    const int ng = (pool->n_kv_heads + HG - 1) / HG;
    if (plan->spans) {
        plan->chunk = TB;
        int grid = plan->grid;
        if (!need_device && resident_grid(pool, n_q_heads, true, plan->cuda_cores, &grid) != PF_OK) {
            clear_error();
            grid = kGridBoundNoDevice;
        }
        // two records (first and last segment of a span) per span and head
        // of the group.  Cut pairs are merged inside the kernel, so there
        // are no jobs.
        const size_t spans = (size_t)grid;
        plan->n_jobs = 0;
        plan->partial_bytes = spans * 2 * (size_t)HG * rec_words * sizeof(unsigned long long);
    } else {
        long long c = split_tokens == -1 ? cap : ((long long)split_tokens + TB - 1) / TB * TB;
        if (c > cap) c = cap;
        if (c < TB) c = TB;
        plan->chunk = (int)c;
        const long long per_seq = (maxctx + c - 1) / c;
        if (per_seq <= 1) {
            plan->n_jobs = 0;   // no sequence is ever cut: nothing to merge
            plan->partial_bytes = 0;
        } else {
            const size_t units = (size_t)per_launch * (size_t)per_seq;
            plan->n_jobs = units * ng;
            plan->partial_bytes =
                units * (size_t)pool->n_kv_heads * rec_words * sizeof(float) + plan->n_jobs * sizeof(attn::Job);
        }
    }
    return PF_OK;
}

int launch_attention(const AttnArgs &a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_decode_attention: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(PF_ERR_UNSUPPORTED, "device index out of range");
    pf_pool *pool = a.pool;
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;
    const AttnPlan &plan = a.plan;
    KernelInfo ki;
    int HG = 0;
    bool mma = false;
    int rc = kernel_for(pool, a.rows * pool->n_kv_heads, plan.spans, plan.cuda_cores, &ki, &HG, &mma);
    if (rc) return rc;
    int tmi = 0;
    rc = encode_pool_tmaps(pool, dev, mma ? -HG : HG, &tmi);
    if (rc) return rc;

    attn::Params p;
    p.k_pool = static_cast<__half *>(pool->k_base);
    p.v_pool = static_cast<__half *>(pool->v_base);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    const size_t rec_bytes = plan.partial_bytes - plan.n_jobs * sizeof(attn::Job);
    p.partials = reinterpret_cast<float *>(ws + plan.counter_bytes);
    p.span_recs = reinterpret_cast<unsigned long long *>(ws + plan.counter_bytes);
    p.jobs = reinterpret_cast<attn::Job *>(ws + plan.counter_bytes + rec_bytes);
    p.status = status;
    p.max_blocks = a.max_blocks;
    p.n_q_heads = a.n_q_heads;
    p.n_kv_heads = pool->n_kv_heads;
    p.n_groups = (pool->n_kv_heads + HG - 1) / HG;
    p.n_blocks = pool->n_blocks;
    p.block_size = pool->block_size;
    p.layer_row0 = a.layer * pool->n_blocks * pool->block_size;
    p.chunk = plan.chunk;
    p.spans = plan.spans ? 1 : 0;
    p.out_f32 = a.out_dtype == PF_F32;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    // L2 prefetch of each CTA's first tiles before the dependency wait (one
    // TMA prefetch per K or V tile).  Measured on the mixed workload: back to
    // back (the launch overlaps the previous kernel's tail), 16 tiles 32.56
    // us, 20: 32.63, 24: 32.43, 32: 32.88; a call on its own, 6 tiles 39.1 us,
    // 8: 39.4, 10: 40.2, 16: 42.7 (and 0 tiles 0.5-1 us slower than 6).  The
    // prefetches reach DRAM ahead of the ring's loads, which then find their
    // lines on the way in.
    p.prefetch_tiles = a.overlap_previous ? 24 : 6;
    p.gh = a.n_q_heads / pool->n_kv_heads;
    p.rows = a.rows;
    p.test_skip = g_inject_timeout.exchange(0) != 0 ? 1 : 0;
    const KernelFn fn = a.out_dtype == PF_F32 ? ki.fn32 : ki.fn;
    const size_t out_elem = a.out_dtype == PF_F32 ? 4 : 2;
    const size_t row = (size_t)a.n_q_heads * pool->head_dim;   // q / out elements per sequence

    // Sequences are independent: batches larger than one launch's share of
    // shared memory run as consecutive launches on the stream; each launch
    // stamps its merge jobs with a fresh epoch.
    for (int s0 = 0; s0 < a.n_seqs; s0 += attn::kMaxSeqsPerLaunch) {
        const int n = a.n_seqs - s0 < attn::kMaxSeqsPerLaunch ? a.n_seqs - s0 : attn::kMaxSeqsPerLaunch;
        // decode: q and out rows are the sequences; append: cu_q holds
        // absolute rows, so only it moves with the launch
        const size_t qoff = a.cu_q ? 0 : (size_t)s0 * row;
        p.cu_q = a.cu_q ? a.cu_q + s0 : nullptr;
        p.q = static_cast<const __half *>(a.q) + qoff;
        const size_t kv_row = (size_t)pool->n_kv_heads * pool->head_dim;
        p.k_new = a.k_new ? static_cast<const __half *>(a.k_new) + (size_t)s0 * kv_row : nullptr;
        p.v_new = a.v_new ? static_cast<const __half *>(a.v_new) + (size_t)s0 * kv_row : nullptr;
        p.out = static_cast<uint8_t *>(a.out) + qoff * out_elem;
        p.bt = a.block_tables + (size_t)s0 * a.max_blocks;
        p.lens = a.context_lens + s0;
        p.n_seqs = n;
        p.epoch = next_epoch();
        if (a.overlap_previous) {
            // A programmatic dependent of the previous kernel on the stream:
            // resident while that kernel drains; the kernel waits for it
            // (griddepcontrol.wait) before it touches anything but the
            // lengths and the tables.
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(plan.grid);
            cfg.blockDim = dim3(attn::NTHREADS);
            cfg.dynamicSmemBytes = ki.smem;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, fn, pool->tmap_k[dev][tmi], pool->tmap_v[dev][tmi], p);
        } else {
            fn<<<plan.grid, attn::NTHREADS, ki.smem, stream>>>(pool->tmap_k[dev][tmi], pool->tmap_v[dev][tmi], p);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return cuda_error(e, "pf_paged_decode_attention: launch");
        if (plan.n_jobs == 0) continue;
        // merge grid: a programmatic dependent of the main grid (it launches
        // while the main grid drains and waits for it before reading)
        const int n_jobs = (int)plan.n_jobs;
        // one warp per (job slot, head), at most one resident wave of CTAs
        unsigned long long warps = (unsigned long long)plan.n_jobs * HG;
        unsigned blocks = (unsigned)((warps + 3) / 4);
        const unsigned wave = (unsigned)plan.grid * 4u;
        if (blocks > wave) blocks = wave;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(blocks);
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, ki.merge, p, n_jobs);
        if (e != cudaSuccess) return cuda_error(e, "pf_paged_decode_attention: merge launch");
    }
    return PF_OK;
}

}  // namespace pkv

extern "C" int pf_test_inject_wait_timeout(void) {
    pkv::clear_error();
    pkv::g_inject_timeout.store(1);
    return PF_OK;
}
