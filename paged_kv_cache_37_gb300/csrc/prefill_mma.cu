// prefill_mma.cu -- multi-token append and prompt attention through the block
// tables on tensor cores (pf_paged_prefill_attention without a workspace, or
// with more rows per kv-head than the decode kernel takes).
//
// Sequence s has L_s tokens, the last n_s of them new (PagedAttention blog,
// "Architecture": append into the last block, then attend); the query of new
// token i sits at position p = L_s - n_s + i and attends causally to tokens
// 0 .. p.  A kv-head's query rows are its new tokens x its gh q-heads, row
// r = i * gh + g.
//
// One CTA serves 64 consecutive rows of one (sequence, kv-head): 4 warps of
// 16 rows, each row set one m16 fragment of warp-level MMA (fp16 in, fp32
// accumulate).  K/V tiles of 16 tokens come through the block table by
// 16-byte cp.async into a ring of stages, stored in the 128-byte swizzled
// layout (16-byte chunk c of a 128-byte row t at c ^ (t mod 8)) so that
// ldmatrix reads them without bank conflicts; every tile serves all 64 rows.
// Per tile a warp computes S = Q K^T (m16n8k16), applies the causal limit
// per row, runs the online softmax on the score fragments (reference maximum
// raised only past 2^8, log2 domain) and adds P V with the weights rounded
// to fp16; l sums those rounded weights.  CTAs walk their tiles in order up
// to the last position any of their rows sees; the grid takes the q-tiles of
// a head longest first.
#include <type_traits>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace prefill_mma {
namespace {

constexpr int TB = 16;           // tokens per K/V tile
constexpr int NW = 4;            // warps, 16 query rows each
constexpr int QR = 16 * NW;      // query rows per CTA
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
    int gh;           // q-heads per kv-head
    int max_blocks;
    int max_new;
    int n_blocks;
    int block_size;
    int n_qt;         // 64-row tiles of the longest (sequence, kv-head)
    long long layer_row0;
    int out_f32;
    float scale_log2;
};

template <int D>
struct Shape {
    static constexpr int NST = D == 64 ? 9 : 6;       // K/V stages
    static constexpr int TILE_BYTES = TB * D * 2;     // K or V of one tile
    static constexpr int SMEM = QR * D * 2 + 2 * NST * TILE_BYTES;
};

// Byte offset of 16-byte chunk c (dims 8c .. 8c + 7) of row t in a block of
// `rows` rows: per 64-dim half, rows of 128 bytes, chunk c % 8 of row t at
// position (c % 8) ^ (t % 8).
__device__ __forceinline__ uint32_t swz(int t, int c, int rows) {
    return (uint32_t)((((c >> 3) * rows + t) << 7) + ((((c & 7) ^ (t & 7))) << 4));
}

// 16-byte cp.async that reads `bytes` (16 or 0) and zero-fills the rest.
__device__ __forceinline__ void cp_async16(uint32_t smem, const void *gmem, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem), "l"(gmem), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int D>
__global__ void __launch_bounds__(NTHREADS) prefill_mma_kernel(const Params p) {
    using S = Shape<D>;
    constexpr int CH = D / 8;     // 16-byte chunks of a row
    constexpr int NKS = D / 16;   // k-steps of the score product
    constexpr int NNB = D / 8;    // 8-dim column blocks of O
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *qs = smem;                                  // QR swizzled q rows
    uint8_t *ks = smem + QR * D * 2;                     // NST K tiles
    uint8_t *vs = ks + S::NST * S::TILE_BYTES;           // NST V tiles

    const int qt = p.n_qt - 1 - (int)blockIdx.x;         // longest first
    const int h = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int maxctx = p.max_blocks * p.block_size;

    // lengths and new-token counts, clamped (and flagged) to what the table
    // and the call allow
    int L = p.lens[s];
    const bool flagger = threadIdx.x == 0 && qt == 0 && h == 0;
    if (L < 0 || L > maxctx) {
        if (flagger) atomicOr(p.status, PF_DEV_BAD_LENGTH);
        L = L < 0 ? 0 : maxctx;
    }
    const int q0 = p.cu_q[s];
    int n = p.cu_q[s + 1] - q0;
    if (n < 0 || n > L || n > p.max_new) {
        if (flagger) atomicOr(p.status, PF_DEV_BAD_LENGTH);
        n = n < 0 ? 0 : min(min(n, L), p.max_new);
    }
    const int rows = n * p.gh;
    const int r0 = qt * QR;
    if (r0 >= rows) return;                              // the whole CTA: no row here
    const int r_end = min(r0 + QR, rows);
    const int base = L - n;                              // position of new token 0
    const int p_max = base + (r_end - 1) / p.gh;         // last position any row of the CTA sees
    const int n_tiles = p_max / TB + 1;

    // q rows r0 .. r_end - 1 (zeros past them; their results are dropped)
    for (int c = threadIdx.x; c < QR * CH; c += NTHREADS) {
        const int row = c / CH, col = c - (c / CH) * CH;
        const int r = r0 + row;
        const bool ok = r < r_end;
        const int i = ok ? r / p.gh : 0;
        const __half *src = p.q + ((size_t)(q0 + i) * p.n_q_heads + (size_t)h * p.gh + (r - i * p.gh)) * D + col * 8;
        cp_async16(smem_addr(qs + swz(row, col, QR)), ok ? src : p.q, ok ? 16u : 0u);
    }
    // Stage tile t: K and V rows of tokens t*16 .. t*16+15 up to p_max
    // (zeros past it: never part of a result, and finite).  Thread x copies
    // chunk x % CH of rows x / CH + j * (NTHREADS / CH) of K and of V, so it
    // needs RPT block ids per tile; they are loaded LOOK tiles ahead of use
    // (a block-table load waited for at issue would serialise the ring).
    constexpr int RPT = TB * CH / NTHREADS;             // rows per thread and tile (1 at D = 64, 2 at 128)
    constexpr int LOOK = 3;
    static_assert(RPT * NTHREADS == TB * CH, "a tile's chunks split evenly over the threads");
    const int my_col = threadIdx.x % CH;
    const int my_row = threadIdx.x / CH;                  // rows my_row + j * (NTHREADS / CH)
    auto load_ids = [&](int t, int (&ids)[RPT]) {
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int tok = t * TB + my_row + j * (NTHREADS / CH);
            ids[j] = tok <= p_max ? p.bt[(size_t)s * p.max_blocks + tok / p.block_size] : 0;
        }
    };
    auto stage_tile = [&](int t, int stage, const int (&ids)[RPT]) {
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int row = my_row + j * (NTHREADS / CH);
            const int tok = t * TB + row;
            int id = ids[j];
            bool ok = tok <= p_max;
            if (ok && (id < 0 || id >= p.n_blocks)) {
                atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
                ok = false;
            }
            const size_t src =
                ok ? ((size_t)(p.layer_row0 + (long long)id * p.block_size + tok % p.block_size) * p.n_kv_heads + h) *
                             D + my_col * 8
                   : 0;
            const uint32_t off = stage * S::TILE_BYTES + swz(row, my_col, TB);
            cp_async16(smem_addr(ks + off), p.k_pool + src, ok ? 16u : 0u);
            cp_async16(smem_addr(vs + off), p.v_pool + src, ok ? 16u : 0u);
        }
        cp_async_commit();
    };

    // This warp's rows: fragment rows gq and gq + 8 of rows wr0 .. wr0 + 15;
    // a row past r_end takes the CTA's last limit (its results are dropped).
    const int wr0 = r0 + 16 * warp;
    const bool warp_rows = wr0 < r_end;
    int lim[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = wr0 + gq + 8 * r;
        lim[r] = row < r_end ? base + row / p.gh : p_max;
    }
    const int wlim_lo = base + min(wr0, r_end - 1) / p.gh;                    // smallest limit of the warp
    const int wlim_hi = base + (min(wr0 + 15, r_end - 1)) / p.gh;             // largest

    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.0f, 0.0f};
    float o[NNB][4];
#pragma unroll
    for (int b = 0; b < NNB; ++b) o[b][0] = o[b][1] = o[b][2] = o[b][3] = 0.0f;
    uint32_t qa[NKS][4];

    // Tiles are used two at a time, as one 32-token softmax step.  NST - 2
    // tiles are in flight ahead of the pair in use; one commit group per tile
    // (empty past the end; q rides with tile 0), so wait_group NST - 2 after
    // staging the pair's successors means "tiles t and t + 1 done".  ids[k]
    // hold the block ids of tile (next tile to stage) + k.
    constexpr int LOOK2 = 2 * LOOK;
    int ids[LOOK2][RPT];
#pragma unroll 1
    for (int t = 0; t < S::NST - 2; ++t) {
        int id_now[RPT];
        load_ids(t, id_now);
        if (t < n_tiles) stage_tile(t, t, id_now);
        else cp_async_commit();
    }
#pragma unroll
    for (int k = 0; k < LOOK2; ++k) load_ids(S::NST - 2 + k, ids[k]);

    // One softmax step over NT consecutive staged tiles (sub-tile u at stage
    // (t + u) % NST, tokens tile0 + 16 u ..).
    auto step = [&](int t, auto nt_c) {
        constexpr int NT = decltype(nt_c)::value;
        const int tile0 = t * TB;
        const bool masked = tile0 + NT * TB - 1 > wlim_lo;
        // S = Q K^T: K rows are the B fragments' columns (tokens)
        float sc[2 * NT][4];
#pragma unroll
        for (int u = 0; u < NT; ++u) {
            const uint32_t kb = smem_addr(ks + ((t + u) % S::NST) * S::TILE_BYTES);
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                float *c = sc[2 * u + nb];
                c[0] = c[1] = c[2] = c[3] = 0.0f;
#pragma unroll
                for (int kp = 0; kp < NKS / 2; ++kp) {
                    uint32_t b[4];
                    ldmatrix_x4(b, kb + swz(nb * 8 + (lane & 7), kp * 4 + (lane >> 3), TB));
                    mma_f16_16816(sc[2 * u + nb], qa[2 * kp], b[0], b[1]);
                    mma_f16_16816(sc[2 * u + nb], qa[2 * kp + 1], b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int cb = 0; cb < 2 * NT; ++cb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sc[cb][e] *= p.scale_log2;
                if (masked && tile0 + cb * 8 + 2 * tq + (e & 1) > lim[e >> 1]) sc[cb][e] = -INFINITY;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float mt = -INFINITY;
#pragma unroll
            for (int cb = 0; cb < 2 * NT; ++cb) mt = fmaxf(mt, fmaxf(sc[cb][2 * r], sc[cb][2 * r + 1]));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
            if (mt > m[r] + kRescaleLog2) {
                const float f = exp2f(m[r] - mt);         // m = -inf gives 0
                l[r] *= f;
#pragma unroll
                for (int b = 0; b < NNB; ++b) {
                    o[b][2 * r] *= f;
                    o[b][2 * r + 1] *= f;
                }
                m[r] = mt;
            }
        }
        // weights of sub-tile u as the A fragment of P V: register 2 nb + r
        // holds row g + 8 r, tokens 8 nb + 2t, 8 nb + 2t + 1 of the sub-tile
        uint32_t pa[NT][4];
#pragma unroll
        for (int u = 0; u < NT; ++u) {
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float z0 = sc[2 * u + nb][2 * r], z1 = sc[2 * u + nb][2 * r + 1];
                    const float p0 = z0 == -INFINITY ? 0.0f : exp2f(z0 - m[r]);
                    const float p1 = z1 == -INFINITY ? 0.0f : exp2f(z1 - m[r]);
                    const __half2 w = __floats2half2_rn(p0, p1);
                    const float2 wf = __half22float2(w);
                    l[r] += wf.x + wf.y;
                    pa[u][2 * nb + r] = *reinterpret_cast<const uint32_t *>(&w);
                }
            }
        }
        // O += P V: V rows (tokens) are the B fragments' k
#pragma unroll
        for (int u = 0; u < NT; ++u) {
            const uint32_t vb = smem_addr(vs + ((t + u) % S::NST) * S::TILE_BYTES);
#pragma unroll
            for (int np = 0; np < NNB / 2; ++np) {
                uint32_t b[4];
                ldmatrix_x4_trans(b, vb + swz((lane & 7) + ((lane >> 3) & 1) * 8, np * 2 + (lane >> 4), TB));
                mma_f16_16816(o[2 * np], pa[u], b[0], b[1]);
                mma_f16_16816(o[2 * np + 1], pa[u], b[2], b[3]);
            }
        }
    };

    for (int t = 0; t < n_tiles; t += 2) {
        // the pair's successors go into the stages of the previous pair
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int a = t + S::NST - 2 + u;
            if (a < n_tiles) stage_tile(a, a % S::NST, ids[u]);
            else cp_async_commit();
        }
#pragma unroll
        for (int k = 0; k + 2 < LOOK2; ++k) {
#pragma unroll
            for (int j = 0; j < RPT; ++j) ids[k][j] = ids[k + 2][j];
        }
        load_ids(t + S::NST - 2 + LOOK2, ids[LOOK2 - 2]);
        load_ids(t + S::NST - 1 + LOOK2, ids[LOOK2 - 1]);
        cp_async_wait<S::NST - 2>();                     // tiles t, t + 1 have landed (this thread's part)
        __syncthreads();                                 // ... and every thread's part
        if (t == 0) {
            // q as A fragments: lanes 0-7 / 8-15 / 16-23 / 24-31 give rows
            // 0-7 / 8-15 / 0-7 / 8-15 of the warp's 16 at dims +0 / +0 / +8 / +8
            const int lrow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < NKS; ++kk)
                ldmatrix_x4(qa[kk], smem_addr(qs + swz(lrow, 2 * kk + (lane >> 4), QR)));
        }
        if (warp_rows && t * TB <= wlim_hi) {
            // a pair, or the last tile alone (its partner was never staged)
            if (t + 1 < n_tiles && (t + 1) * TB <= wlim_hi) step(t, std::integral_constant<int, 2>());
            else step(t, std::integral_constant<int, 1>());
        }
        __syncthreads();                                 // the pair's stages are refilled next iteration
    }
    cp_async_wait<0>();

    if (!warp_rows) return;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(FULL, l[r], 1);
        l[r] += __shfl_xor_sync(FULL, l[r], 2);
        const int row = wr0 + gq + 8 * r;
        if (row >= r_end) continue;
        const int i = row / p.gh;
        const float inv = 1.0f / l[r];
        const size_t ob = ((size_t)(q0 + i) * p.n_q_heads + (size_t)h * p.gh + (row - i * p.gh)) * D + 2 * tq;
#pragma unroll
        for (int b = 0; b < NNB; ++b) {
            const float x0 = o[b][2 * r] * inv, x1 = o[b][2 * r + 1] * inv;
            if (p.out_f32) *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + ob + b * 8) = make_float2(x0, x1);
            else *reinterpret_cast<__half2 *>(static_cast<__half *>(p.out) + ob + b * 8) = __floats2half2_rn(x0, x1);
        }
    }
}

}  // namespace
}  // namespace prefill_mma

int launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;
    const pf_pool *pool = a.pool;
    if (a.n_seqs > 65535 || pool->n_kv_heads > 65535)
        return set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: at most 65535 sequences and kv-heads per call");
    const int gh = a.n_q_heads / pool->n_kv_heads;
    // 128 rows or more per (sequence, kv-head): the tcgen05 kernel
    if ((long long)a.max_new * gh >= kTcMinRows) return launch_prefill_tc(a, stream);
    const long long n_qt = ((long long)a.max_new * gh + prefill_mma::QR - 1) / prefill_mma::QR;
    if (n_qt > 0x7fffffffll)
        return set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: too many new tokens for one launch");
    prefill_mma::Params p;
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
    p.gh = gh;
    p.max_blocks = a.max_blocks;
    p.max_new = a.max_new;
    p.n_blocks = pool->n_blocks;
    p.block_size = pool->block_size;
    p.n_qt = (int)n_qt;
    p.layer_row0 = (long long)a.layer * pool->n_blocks * pool->block_size;
    p.out_f32 = a.out_dtype == PF_F32;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    void (*fn)(prefill_mma::Params) =
        pool->head_dim == 64 ? prefill_mma::prefill_mma_kernel<64> : prefill_mma::prefill_mma_kernel<128>;
    const int smem = pool->head_dim == 64 ? prefill_mma::Shape<64>::SMEM : prefill_mma::Shape<128>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_prefill_attention: cudaFuncSetAttribute");
    dim3 grid((unsigned)n_qt, (unsigned)pool->n_kv_heads, (unsigned)a.n_seqs);
    fn<<<grid, prefill_mma::NTHREADS, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_prefill_attention: launch");
    return PF_OK;
}

}  // namespace pkv
