// prefill.cu -- multi-token append attention through the block tables
// (pf_paged_prefill_attention): a prompt, or a chunk of one, whose K/V rows
// are already in the sequence's last pages (PagedAttention blog,
// "Architecture": append into the last block, then attend).
//
// Sequence s has L_s tokens, the last n_s of them new; the query of new token
// i sits at position p = L_s - n_s + i and attends causally to tokens 0 .. p
// (a decode step is the case n_s = 1).  out row = softmax(scale q K^T) V over
// those tokens, fp32 accumulation.
//
// One CTA serves one (chunk of new tokens, sequence, kv-head): up to 8 query
// rows (4 at head_dim 128) -- the chunk's tokens x the G q-heads of the
// kv-head -- so every K/V tile it stages in shared memory serves all of them.
// Its 4 warps all hold those rows and split each tile's tokens; their
// softmax states merge through shared memory at the end.
// Tiles are 16 tokens of one kv-head, fetched with 16-byte cp.async through
// the block table into a ring of stages (several tiles in flight per CTA).
// The warp math is that of the decode kernel: D/8 lanes hold one token row,
// q . k reduces over them with xor shuffles, an fp32 online softmax in the
// log2 domain raises its reference maximum only when a score passes it by
// more than 2^8, and the token groups merge at the end.  The causal limit is
// per row.  Every thread runs the same tile loop, so plain CTA barriers are
// used.
#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace prefill {
namespace {

constexpr int TB = 16;          // tokens per staged tile
constexpr int NW = 4;           // warps per CTA
constexpr int NTHREADS = 32 * NW;
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned FULL = 0xffffffffu;

struct Params {
    const __half *q;
    const __half *k_pool;
    const __half *v_pool;
    void *out;
    const int32_t *bt;
    const int32_t *lens;
    const int32_t *cu_q;
    int *status;
    int n_q_heads;
    int n_kv_heads;
    int max_blocks;
    int max_new;
    int n_blocks;
    int block_size;
    long long layer_row0;
    int out_f32;
    float scale_log2;
};

template <int D, int G>
struct Shape {
    static constexpr int ROWS_MAX = D == 64 ? 8 : 4;                 // query rows the warps hold
    static constexpr int QC = G >= ROWS_MAX ? 1 : ROWS_MAX / G;      // new tokens per CTA
    static constexpr int R = QC * G;                                 // query rows per CTA
    static constexpr int LPT = D / 8;                                // lanes per token row
    static constexpr int TPW = 32 / LPT;                             // token rows per warp-step
    static constexpr int STEPS = TB / TPW;                           // warp-steps per tile
    static constexpr int SPW = STEPS / NW;                           // of which each warp takes
    static_assert(SPW * NW == STEPS, "a tile splits evenly over the warps");
    static constexpr int VECS = TB * D / 8;                          // 16-byte vectors per tile (K or V)
    static constexpr int NST = D == 64 ? 12 : 6;                     // tile stages (48 KB of K and V)
    static constexpr int SMEM = 2 * NST * TB * D * 2;
    static_assert(NW * R * (D + 2) * 4 <= SMEM, "the merge area fits in the ring");
};

__device__ __forceinline__ void cp_async16(uint32_t smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int D, int G>
__global__ void __launch_bounds__(NTHREADS) prefill_kernel(const Params p) {
    using S = Shape<D, G>;
    __shared__ __align__(16) uint8_t smem[S::SMEM];
    __half (*kt)[TB * D] = reinterpret_cast<__half (*)[TB * D]>(smem);
    __half (*vt)[TB * D] = reinterpret_cast<__half (*)[TB * D]>(smem + S::SMEM / 2);

    const int s = blockIdx.y;
    const int h = blockIdx.z;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int maxctx = p.max_blocks * p.block_size;

    // lengths: clamped (and flagged) to what the table and the call allow
    int L = p.lens[s];
    if (L < 0 || L > maxctx) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.status, PF_DEV_BAD_LENGTH);
        L = L < 0 ? 0 : maxctx;
    }
    const int q0 = p.cu_q[s];
    int n = p.cu_q[s + 1] - q0;
    if (n < 0 || n > L || n > p.max_new) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.status, PF_DEV_BAD_LENGTH);
        n = n < 0 ? 0 : min(min(n, L), p.max_new);
    }
    const int i0 = blockIdx.x * S::QC;
    if (i0 >= n) return;                                   // the whole CTA: no new token here
    const int i_end = min(i0 + S::QC, n);
    const int p_max = L - n + i_end - 1;                   // last position any query of the CTA sees
    const int n_tiles = p_max / TB + 1;

    // Every warp holds all R rows (row r = new token i0 + r / G, q-head r % G)
    // and takes SPW of each tile's warp-steps.
    const int grp = lane / S::LPT;
    const int sub = lane % S::LPT;
    float qf[S::R][8];
    int pos[S::R];
#pragma unroll
    for (int r = 0; r < S::R; ++r) {
        const int i = i0 + r / G;
        const bool valid = i < i_end;
        pos[r] = valid ? L - n + i : -1;                   // -1: every token is masked
        if (valid) {
            const size_t row = ((size_t)(q0 + i) * p.n_q_heads + (size_t)h * G + r % G) * D;
            const uint4 raw = *reinterpret_cast<const uint4 *>(p.q + row + sub * 8);
            half8_to_float(raw, qf[r]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[r][e] = valid ? qf[r][e] * p.scale_log2 : 0.0f;
    }
    float m[S::R], l[S::R], acc[S::R][8];
#pragma unroll
    for (int r = 0; r < S::R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[r][e] = 0.0f;
    }

    // Stage tile t: K and V rows of tokens t*16 .. t*16+15 that are <= p_max.
    auto stage_tile = [&](int t, int stage) {
        for (int c = threadIdx.x; c < 2 * S::VECS; c += NTHREADS) {
            const int kv = c / S::VECS;
            const int rem = c - kv * S::VECS;
            const int row = rem / (D / 8);
            const int col = rem - row * (D / 8);
            const int tok = t * TB + row;
            if (tok > p_max) continue;                     // never read into a result
            int id = p.bt[(size_t)s * p.max_blocks + tok / p.block_size];
            if (id < 0 || id >= p.n_blocks) {
                atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
                id = 0;                                    // stay inside the pool
            }
            const size_t src =
                ((size_t)(p.layer_row0 + (long long)id * p.block_size + tok % p.block_size) * p.n_kv_heads + h) * D +
                col * 8;
            __half *dst = (kv ? vt[stage] : kt[stage]) + row * D + col * 8;
            cp_async16(smem_addr(dst), (kv ? p.v_pool : p.k_pool) + src);
        }
        cp_async_commit();
    };

    // NST - 1 tiles in flight ahead of the one being used; one commit group
    // per tile (empty past the end), so wait_group NST - 1 means "tile t done".
#pragma unroll 1
    for (int t = 0; t < S::NST - 1; ++t) {
        if (t < n_tiles) stage_tile(t, t);
        else cp_async_commit();
    }
    for (int t = 0; t < n_tiles; ++t) {
        const int stage = t % S::NST;
        const int ahead = t + S::NST - 1;
        if (ahead < n_tiles) stage_tile(ahead, ahead % S::NST);
        else cp_async_commit();
        cp_async_wait<S::NST - 1>();                       // tile t has landed (this thread's part)
        __syncthreads();                                   // ... and every thread's part
        const int tile0 = t * TB;
        float z[S::SPW][S::R];
#pragma unroll
        for (int k = 0; k < S::SPW; ++k) {
            const int row = (warp + k * NW) * S::TPW + grp;
            float kf[8];
            half8_to_float(*reinterpret_cast<const uint4 *>(&kt[stage][row * D + sub * 8]), kf);
#pragma unroll
            for (int r = 0; r < S::R; ++r) {
                float a = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) a = fmaf(qf[r][e], kf[e], a);
                z[k][r] = a;
            }
        }
#pragma unroll
        for (int o = S::LPT / 2; o > 0; o >>= 1) {
#pragma unroll
            for (int k = 0; k < S::SPW; ++k) {
#pragma unroll
                for (int r = 0; r < S::R; ++r) z[k][r] += __shfl_xor_sync(FULL, z[k][r], o);
            }
        }
        // causal mask per row (also hides tokens past p_max, never staged)
#pragma unroll
        for (int k = 0; k < S::SPW; ++k) {
            const int tok = tile0 + (warp + k * NW) * S::TPW + grp;
#pragma unroll
            for (int r = 0; r < S::R; ++r)
                if (tok > pos[r]) z[k][r] = -INFINITY;
        }
#pragma unroll
        for (int r = 0; r < S::R; ++r) {
            float mt = z[0][r];
#pragma unroll
            for (int k = 1; k < S::SPW; ++k) mt = fmaxf(mt, z[k][r]);
#pragma unroll
            for (int o = S::LPT; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, o));
            if (mt > m[r] + kRescaleLog2) {
                const float sc = exp2f(m[r] - mt);         // m = -inf gives 0
                l[r] *= sc;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r][e] *= sc;
                m[r] = mt;
            }
        }
#pragma unroll
        for (int k = 0; k < S::SPW; ++k) {
            const int row = (warp + k * NW) * S::TPW + grp;
            float vf[8];
            half8_to_float(*reinterpret_cast<const uint4 *>(&vt[stage][row * D + sub * 8]), vf);
            if (tile0 + row > p_max) {
#pragma unroll
                for (int e = 0; e < 8; ++e) vf[e] = 0.0f;          // not staged: may hold anything
            }
#pragma unroll
            for (int r = 0; r < S::R; ++r) {
                const float pz = z[k][r] == -INFINITY ? 0.0f : exp2f(z[k][r] - m[r]);
                l[r] += pz;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pz, vf[e], acc[r][e]);
            }
        }
        __syncthreads();                                   // the stage is refilled NST - 1 tiles later
    }

    // Merge: the warp's token groups first (they share its reference
    // maximum), then the four warps through shared memory (the ring is idle
    // now), each warp finishing rows r = warp, warp + NW, ...
#pragma unroll
    for (int o = S::LPT; o < 32; o <<= 1) {
#pragma unroll
        for (int r = 0; r < S::R; ++r) {
            l[r] += __shfl_xor_sync(FULL, l[r], o);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[r][e] += __shfl_xor_sync(FULL, acc[r][e], o);
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    float *red = reinterpret_cast<float *>(smem);          // [NW][R][D + 2]
#pragma unroll
    for (int r = 0; r < S::R; ++r) {
        float *dst = red + ((size_t)warp * S::R + r) * (D + 2);
        if (lane < S::LPT) {
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[sub * 8 + e] = acc[r][e];
        }
        if (lane == 0) {
            dst[D] = m[r];
            dst[D + 1] = l[r];
        }
    }
    __syncthreads();
    constexpr int DPL = D / 32;                            // output dims per lane
    for (int r = warp; r < S::R; r += NW) {
        if (i0 + r / G >= i_end) continue;                 // a row past the chunk's last token
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) mx = fmaxf(mx, red[((size_t)w * S::R + r) * (D + 2) + D]);
        float ls = 0.0f, a[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) a[e] = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float *src = red + ((size_t)w * S::R + r) * (D + 2);
            const float f = src[D] == -INFINITY ? 0.0f : exp2f(src[D] - mx);
            ls = fmaf(src[D + 1], f, ls);
#pragma unroll
            for (int e = 0; e < DPL; ++e) a[e] = fmaf(src[lane + 32 * e], f, a[e]);
        }
        const float inv = 1.0f / ls;
        const size_t o = ((size_t)(q0 + i0 + r / G) * p.n_q_heads + (size_t)h * G + r % G) * D;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            if (p.out_f32) static_cast<float *>(p.out)[o + lane + 32 * e] = a[e] * inv;
            else static_cast<__half *>(p.out)[o + lane + 32 * e] = __float2half_rn(a[e] * inv);
        }
    }
}

using PrefillFn = void (*)(Params);

template <int D>
PrefillFn kernel_for(int g) {
    switch (g) {
        case 1: return prefill_kernel<D, 1>;
        case 2: return prefill_kernel<D, 2>;
        case 3: return prefill_kernel<D, 3>;
        case 4: return prefill_kernel<D, 4>;
        case 5: return prefill_kernel<D, 5>;
        case 6: return prefill_kernel<D, 6>;
        case 7: return prefill_kernel<D, 7>;
        case 8: return prefill_kernel<D, 8>;
        default: return nullptr;
    }
}

template <int D>
int tokens_per_cta(int g) {
    switch (g) {
        case 1: return Shape<D, 1>::QC;
        case 2: return Shape<D, 2>::QC;
        case 3: return Shape<D, 3>::QC;
        case 4: return Shape<D, 4>::QC;
        case 5: return Shape<D, 5>::QC;
        case 6: return Shape<D, 6>::QC;
        case 7: return Shape<D, 7>::QC;
        case 8: return Shape<D, 8>::QC;
        default: return 0;
    }
}

}  // namespace
}  // namespace prefill

int launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;
    const pf_pool *pool = a.pool;
    const int G = a.n_q_heads / pool->n_kv_heads;
    prefill::PrefillFn fn = pool->head_dim == 64 ? prefill::kernel_for<64>(G) : prefill::kernel_for<128>(G);
    const int qc = pool->head_dim == 64 ? prefill::tokens_per_cta<64>(G) : prefill::tokens_per_cta<128>(G);
    if (!fn || qc <= 0) return set_error(PF_ERR_UNSUPPORTED, "pf_paged_prefill_attention: unsupported head_dim / group");
    if (a.n_seqs > 65535 || pool->n_kv_heads > 65535)
        return set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: at most 65535 sequences and kv-heads per call");
    prefill::Params p;
    p.q = static_cast<const __half *>(a.q);
    p.k_pool = static_cast<const __half *>(pool->k_base);
    p.v_pool = static_cast<const __half *>(pool->v_base);
    p.out = a.out;
    p.bt = a.block_tables;
    p.lens = a.context_lens;
    p.cu_q = a.cu_q;
    p.status = status;
    p.n_q_heads = a.n_q_heads;
    p.n_kv_heads = pool->n_kv_heads;
    p.max_blocks = a.max_blocks;
    p.max_new = a.max_new;
    p.n_blocks = pool->n_blocks;
    p.block_size = pool->block_size;
    p.layer_row0 = (long long)a.layer * pool->n_blocks * pool->block_size;
    p.out_f32 = a.out_dtype == PF_F32;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const unsigned gx = (unsigned)((a.max_new + qc - 1) / qc);
    dim3 grid(gx, (unsigned)a.n_seqs, (unsigned)pool->n_kv_heads);
    fn<<<grid, prefill::NTHREADS, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_prefill_attention: launch");
    return PF_OK;
}

}  // namespace pkv
