// prefill_tc.cu -- prompt attention through the block tables on the
// fifth-generation tensor cores: tcgen05.mma with fp32 accumulators in
// tensor memory (pf_paged_prefill_attention calls with 128 or more query
// rows per (sequence, kv-head)).
//
// Sequence s has L_s tokens, the last n_s of them new (PagedAttention blog,
// "Architecture": append into the last block, then attend); the query of new
// token i sits at position p = L_s - n_s + i and attends causally to tokens
// 0 .. p.  A kv-head's query rows are its new tokens x its gh q-heads, row
// r = i * gh + g.
//
// A CTA serves 256 consecutive rows of one (sequence, kv-head) as two query
// tiles of 128 rows (the MMA's M), with sixteen warps:
//   warps 0-3 and 4-7  the softmax of query tile 0 and 1: thread t owns row t
//                      of its tile, which is lane t of tensor memory;
//   warps 8-11         the loaders, two for K and two for V: tiles of BN
//                      tokens (128 at head_dim 64, 64 at 128) through the
//                      block table into a ring of four stages in the
//                      128-byte swizzle, by TMA boxes of up to a page (block
//                      size 16 and up; each warp every other box) or 16-byte
//                      cp.async per token (block size 1);
//   warp 12            issues the scores S_g = Q_g K_j^T (A and B in shared
//                      memory) and owns the tensor memory;
//   warp 13            issues the products O_g += P_g V_j (P in tensor
//                      memory, V in shared memory); warps 14-15 idle.
// The softmax warpgroups run with 200 registers a thread, the others with
// 56 (setmaxnreg after the setup barrier).
// The softmax threads read their row of S, apply the causal limit, keep a
// running maximum per row (raised only past 2^8, log2 domain, so O is
// rescaled rarely), add their weights to the row sum in fp32 and write them,
// rounded to fp16, back to tensor memory as P_g.  Scores and products are
// issued by separate warps so that one's waits leave the tensor pipe to the
// other; with four stages the scores of the next tiles are computed while
// the softmax threads exponentiate.
//
// Measured bounds (GB300, clock64 traces and single-CTA microbenchmarks of
// tcgen05.mma kind::f16, M = 128, K = 16): one MMA costs about 100 cycles
// with A and B in shared memory at N = 128 and about 71 with A in tensor
// memory at N = 64 or 128 -- so P lives in tensor memory and the row sums
// are summed on the CUDA cores rather than by another MMA over P.  A K/V
// step of head_dim 64 (24 MMAs) then takes about 2,400 cycles.  TMA boxes
// issued from one warp arrive at a few hundred cycles each whatever their
// size, and the rate grows with the number of issuing warps (measured: 1, 2,
// 4 warps -> 11.8, 23.4, 44 bytes a cycle per SM on 8 KB boxes), hence two
// loader warps per tensor; 16-byte cp.async from the loader warps was several
// times slower than TMA.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <string>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace prefill_tc {
namespace {

constexpr int QT = 128;          // rows per query tile (the MMA's M)
constexpr int SOFTMAX_WARPS = 8;  // warpgroups 0 and 1
constexpr int LOAD_WARP0 = 8;     // warpgroup 2: K loaders (warps 8, 9), V loaders (10, 11)
constexpr int MMA_S_WARP = 12;    // warpgroup 3: issues the scores; owns the tensor memory
constexpr int MMA_PV_WARP = 13;   // issues the products (warps 14 and 15 idle)
constexpr int NTHREADS = 512;
// Registers: launched at 128 a thread (512 threads, one CTA per SM); the
// loader and MMA warpgroups then give theirs down to REG_OTHER and the
// softmax warpgroups take REG_SOFTMAX.  Each SM sub-partition holds one warp
// of every warpgroup, so the split must also fit its 16K registers.
constexpr int REG_SOFTMAX = 200;
constexpr int REG_OTHER = 56;
static_assert(2 * 128 * REG_SOFTMAX + 2 * 128 * REG_OTHER == NTHREADS * 128, "the split is the launch's registers");
static_assert(32 * (2 * REG_SOFTMAX + 2 * REG_OTHER) <= 16384, "a sub-partition's registers");
constexpr int NS = 4;            // K/V stages
constexpr int TMEM_COLS = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned FULL = 0xffffffffu;

template <int D>
struct Cfg {
    static constexpr int BN = D == 64 ? 128 : 64;       // tokens per K/V tile (the scores' N)
    static constexpr int HALVES = D / 64;               // 64-element halves of a row
    static constexpr int Q_BYTES = QT * D * 2;          // one query tile
    static constexpr int KV_BYTES = BN * D * 2;         // one K or V tile
    static constexpr int OFF_K = 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + NS * KV_BYTES;
    static constexpr int DATA = OFF_V + NS * KV_BYTES;
    static constexpr int SMEM = DATA + 1024;            // slack to align the base to 1024 bytes
    // tensor memory (fp32 columns): S of query tile g at g BN, O of tile g at
    // 2 BN + g D, and the fp16 weights P of tile g, two per column (token 2c
    // in the low half of column c), at 2 BN + 2 D + g BN / 2
    static constexpr int COL_O = 2 * BN;
    static constexpr int COL_P = COL_O + 2 * D;
    static_assert(COL_P + BN <= TMEM_COLS, "tensor memory columns");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

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
    int gh;
    int max_blocks;
    int max_new;
    int n_blocks;
    int block_size;
    int box_rows;     // rows of one TMA box (block size 16 and up)
    int n_items;      // sequences x kv-heads
    int n_qp;         // 256-row tiles of the longest (sequence, kv-head)
    long long layer_row0;
    int out_f32;
    float scale_log2;
};

struct Bars {
    unsigned long long k_full[NS];
    unsigned long long v_full[NS];
    unsigned long long k_empty[NS];
    unsigned long long v_empty[NS];
    unsigned long long s_full[2];
    unsigned long long s_free[2];
    unsigned long long p_full[2];
    unsigned long long o_done[2];
    unsigned long long mma_done[2];
    uint32_t tmem_base;
};

// ---- tcgen05 ---------------------------------------------------------------

// Shared-memory operand descriptor of the 128-byte swizzled layout: rows of
// 128 bytes, 8-row groups 1024 bytes apart (the stride field), 16-byte chunk
// c of row t stored at chunk c ^ (t mod 8).  The start address advances by
// 32 bytes per 16-element K step inside a 64-element half; every block
// starts on a 1024-byte boundary, so the base-offset field stays 0.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, fp16 A and B, A
// K-major, B K-major or (mn_major) MN-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (b_mn_major ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
        : "memory");
}

// The same with A in tensor memory: row m of A in lane m, 16-bit elements
// two per column from a_tmem on.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
        : "memory");
}

// The mbarrier gets one arrival when every MMA this thread issued so far has
// completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define PKV_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), \
                  "=r"(v[i + 6]), "=r"(v[i + 7])
#define PKV_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), "r"(v[i + 4]), "r"(v[i + 5]), \
                  "r"(v[i + 6]), "r"(v[i + 7])

// Lane l of the warp reads lane (32 (warp mod 4) + l) of tensor memory,
// columns col .. col + 31 (resp. 15); complete with tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : PKV_R8(0), PKV_R8(8)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        PKV_W8(0), PKV_W8(8)
        : "memory");
}
#undef PKV_R8
#undef PKV_W8
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait on an mbarrier phase by every lane of the warp (each lane
// observes the completion itself; cheaper than one lane polling and a
// broadcast when the phase has already completed); true on every lane only
// if it completed for all of them, so the warp leaves its loops together.
__device__ __forceinline__ bool wait_lanes(uint32_t bar, uint32_t parity, int *status) {
    return __all_sync(FULL, mbar_wait(bar, parity, status));
}

// Packed pairs of fp32 for Blackwell's two-wide add.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 4-D tiled TMA load (no cache hint): K/V tiles are read again by the other
// query tiles of the same head, so they keep the default L2 policy.
__device__ __forceinline__ void tma_load_4d_plain(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                                  int c3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Byte offset of 16-byte chunk c (elements 8c .. 8c + 7) of row t in a block
// of `rows` rows stored as 64-element halves, each half [rows][128 bytes]
// swizzled.
__device__ __forceinline__ uint32_t swz(int t, int c, int rows) {
    return (uint32_t)((((c >> 3) * rows + t) << 7) + (((c & 7) ^ (t & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const Params p) {
    using C = Cfg<D>;
    constexpr int BN = C::BN;
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    uint8_t *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

    // work item: the longest query tiles first
    const int b = (int)blockIdx.x;
    const int qp = p.n_qp - 1 - b / p.n_items;
    const int item = b - (b / p.n_items) * p.n_items;
    const int s = item / p.n_kv_heads;
    const int h = item - s * p.n_kv_heads;
    const int warp = (int)threadIdx.x / 32;
    const int lane = (int)threadIdx.x % 32;
    const int maxctx = p.max_blocks * p.block_size;

    // lengths and new-token counts, clamped (and flagged) to what the table
    // and the call allow
    int L = p.lens[s];
    const bool flagger = threadIdx.x == 0 && qp == 0 && h == 0;
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
    const int r0 = qp * 2 * QT;
    if (r0 >= rows) return;                  // the whole CTA: no row here
    const int r_end = min(r0 + 2 * QT, rows);
    const int base = L - n;                  // position of new token 0
    // per query tile: its last position and its number of K/V tiles
    int nt[2], pmax[2];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int gr0 = r0 + g * QT;
        if (gr0 >= r_end) {
            nt[g] = 0;
            pmax[g] = 0;
        } else {
            pmax[g] = base + (min(gr0 + QT, r_end) - 1) / p.gh;
            nt[g] = pmax[g] / BN + 1;
        }
    }
    const int p_max = max(pmax[0], pmax[1]);
    const int ntt = max(nt[0], nt[1]);

    const uint32_t s_k = smem_addr(sm + C::OFF_K);
    const uint32_t s_v = smem_addr(sm + C::OFF_V);
    auto bar = [](unsigned long long &x) { return smem_addr(&x); };

    // Softmax threads: their row, and the query row into shared memory
    // (zeros past the last row) before the setup barrier, which then orders
    // it before the first MMA.
    const int g = (warp / 4) & 1;
    const int t = (int)threadIdx.x % 128;                    // row of the tile = tensor-memory lane
    const int r = r0 + g * QT + t;
    const bool valid = warp < SOFTMAX_WARPS && r < r_end;
    const int i = valid ? r / p.gh : 0;
    const int lim = valid ? base + i : pmax[g];                // last position this row sees
    const size_t ob = valid ? ((size_t)(q0 + i) * p.n_q_heads + (size_t)h * p.gh + (r - i * p.gh)) * D : 0;
    if (warp < SOFTMAX_WARPS) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ob);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 x = valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(sm + g * C::Q_BYTES + swz(t, c, QT)) = x;
        }
        fence_proxy_async_shared();
    }
    // Loaders: block id of box `lane` of tile j (pages of 16 tokens and
    // more; boxes past the CTA's last position are not loaded), read two
    // tiles ahead of its use and range-checked only when used.
    const int32_t *bt_row = p.bt + (size_t)s * p.max_blocks;
    const int box = p.box_rows;
    auto n_boxes = [&](int j) { return min(BN / box, (p_max - j * BN) / box + 1); };
    auto raw_id = [&](int j) {
        return (p.block_size >= 16 && j < ntt && lane < n_boxes(j)) ? bt_row[(j * BN + lane * box) / p.block_size] : 0;
    };
    // Loaders (two warps for K, two for V, each issuing every other page
    // box of a tile; a stage is refilled once the MMAs of the tile that used
    // it -- the scores for K, the products for V -- are done).  They set up
    // their barriers and stage tile 0 before the setup barrier, so the first
    // tiles arrive while the query rows load.
    const bool loader = warp >= LOAD_WARP0 && warp < LOAD_WARP0 + 4;
    const bool is_v = warp >= LOAD_WARP0 + 2;
    const int li = (warp - LOAD_WARP0) & 1;                  // this warp's boxes: lane % 2 == li
    const CUtensorMap *map = is_v ? &tmv : &tmk;
    unsigned long long *full = is_v ? bars.v_full : bars.k_full;
    unsigned long long *empty = is_v ? bars.v_empty : bars.k_empty;
    const uint32_t s_base = is_v ? s_v : s_k;
    const __half *pool_base = is_v ? p.v_pool : p.k_pool;
    const int B = p.block_size;
    int issued = 0;
    // tile j into its stage (box `lane` from block id `id`); false if a wait ran out
    auto load_tile = [&](int j, int id) -> bool {
        const int st = j % NS;
        const uint32_t dst = s_base + st * C::KV_BYTES;
        if (j >= NS && !wait_lanes(bar(empty[st]), ((j / NS) - 1) & 1, p.status)) return false;
        if (B >= 16) {
            const int nb = n_boxes(j);
            const bool mine = lane < nb && (lane & 1) == li;
            if (mine && (id < 0 || id >= p.n_blocks)) {
                atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
                id = 0;
            }
            if (lane == 0) mbar_arrive_expect_tx(bar(full[st]), (uint32_t)((nb + 1 - li) / 2) * box * D * 2);
            __syncwarp();
            if (mine) {
                const int row = (int)(p.layer_row0 + (long long)id * B + (j * BN + lane * box) % B);
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf)
                    tma_load_4d_plain(dst + (uint32_t)(hf * BN + lane * box) * 128u, map, 0, row, hf, h, bar(full[st]));
            }
        } else {
            // one token per page: 16-byte cp.async per chunk into its
            // swizzled place, then a proxy fence before the arrival
            for (int tk = lane + 32 * li; tk < BN; tk += 64) {
                const int tok = j * BN + tk;
                if (tok > p_max) break;
                int bid = bt_row[tok];
                if (bid < 0 || bid >= p.n_blocks) {
                    atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
                    bid = 0;
                }
                const __half *src = pool_base + ((size_t)(p.layer_row0 + bid) * p.n_kv_heads + h) * D;
#pragma unroll
                for (int c = 0; c < D / 8; ++c) cp_async16_cg(dst + swz(tk, c, BN), src + c * 8);
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            fence_proxy_async_shared();
            mbar_arrive(bar(full[st]));
        }
        ++issued;
        return true;
    };
    int id0 = 0, id1 = 0;
    if (loader) {
        if (warp == LOAD_WARP0 && lane == 0) {
            // two loader warps arrive on each full barrier
            for (int k = 0; k < NS; ++k) {
                mbar_init(bar(bars.k_full[k]), B >= 16 ? 2u : 64u);
                mbar_init(bar(bars.v_full[k]), B >= 16 ? 2u : 64u);
                mbar_init(bar(bars.k_empty[k]), 1);
                mbar_init(bar(bars.v_empty[k]), 1);
            }
            mbar_init_fence();
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");   // the loader warps: barriers initialised
        prefetch_tensormap(map);
        id0 = raw_id(0);
        id1 = raw_id(1);
        if (B >= 16) {
            const int id = id0;
            id0 = id1;
            id1 = raw_id(2);
            load_tile(0, id);
        }
    }

    if (warp == MMA_S_WARP) {
        if (lane == 0) {
            for (int u = 0; u < 2; ++u) {
                mbar_init(bar(bars.s_full[u]), 1);
                mbar_init(bar(bars.s_free[u]), 128);
                mbar_init(bar(bars.p_full[u]), 128);
                mbar_init(bar(bars.o_done[u]), 1);
            }
            mbar_init(bar(bars.mma_done[0]), 1);
            mbar_init(bar(bars.mma_done[1]), 1);
            mbar_init_fence();
        }
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&bars.tmem_base)),
                     "n"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = bars.tmem_base;
    if (warp >= SOFTMAX_WARPS) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_OTHER));
    else asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_SOFTMAX));

    if (warp < SOFTMAX_WARPS) {
        // ---------------------------------------------------------- softmax
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t t_s = tmem + lane_off + (uint32_t)(g * BN);
        const uint32_t t_o = tmem + lane_off + (uint32_t)(C::COL_O + g * D);
        const uint32_t t_p = tmem + lane_off + (uint32_t)(C::COL_P + g * (BN / 2));
        const float sl = p.scale_log2;
        float m = -INFINITY;                                   // reference maximum, log2 units
        float l = 0.0f;                                        // sum of the weights
        bool ok = true;
        for (int j = 0; j < nt[g]; ++j) {
            if (!wait_lanes(bar(bars.s_full[g]), j & 1, p.status)) {
                ok = false;
                break;
            }
            tc_after_sync();
            uint32_t x[BN];                                    // raw scores (fp32 bits)
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) tmem_ld32(t_s + q * 32, x + q * 32);
            tmem_ld_wait();
            tc_before_sync();
            mbar_arrive(bar(bars.s_free[g]));                 // the MMA warp may overwrite S

            // causal limit: columns past it never count
            const int cl = lim - j * BN;
            if (cl < BN - 1) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c > cl) x[c] = 0xff800000u;             // -inf
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < BN; c += 8) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    mx[e] = max3(mx[e], __uint_as_float(x[c + 2 * e]), __uint_as_float(x[c + 2 * e + 1]));
            }
            const float mt = max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl;   // scale > 0
            float f = 1.0f;
            const bool resc = mt > m + kRescaleLog2;
            if (resc) {
                f = ex2(m - mt);                                // m = -inf gives 0
                m = mt;
                l *= f;
            }
            // weights 2^(s sl - m); their sum two at a time
            const float nm = -m;
            uint64_t ls[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
                const float w0 = ex2(fmaf(__uint_as_float(x[2 * c]), sl, nm));
                const float w1 = ex2(fmaf(__uint_as_float(x[2 * c + 1]), sl, nm));
                ls[c & 1] = f2_add(ls[c & 1], f2_pack(w0, w1));
                pk[c] = pack_half2(w0, w1);
            }
            {
                float a0, a1, b0, b1;
                f2_unpack(ls[0], a0, a1);
                f2_unpack(ls[1], b0, b1);
                l += (a0 + a1) + (b0 + b1);
            }

            // the previous product has finished reading P and adding to O
            if (j > 0) {
                if (!wait_lanes(bar(bars.o_done[g]), (j - 1) & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_after_sync();
                if (__any_sync(FULL, resc)) {
                    // rescale O (lanes without a new maximum scale by 1)
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 16) {
                        uint32_t o[16];
                        tmem_ld16(t_o + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st16(t_o + c0, o);
                    }
                    tmem_st_wait();
                }
            }
            // P row t into tensor memory
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) tmem_st32(t_p + q * 32, pk + q * 32);
            tmem_st_wait();
            tc_before_sync();
            mbar_arrive(bar(bars.p_full[g]));
        }
        if (ok && nt[g] > 0 && wait_lanes(bar(bars.o_done[g]), (nt[g] - 1) & 1, p.status)) {
            tc_after_sync();
            const float inv = 1.0f / l;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
                uint32_t o[16];
                tmem_ld16(t_o + c0, o);
                tmem_ld_wait();
                if (valid) {
                    if (p.out_f32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + ob + c0);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                                 __uint_as_float(o[4 * e + 2]) * inv,
                                                 __uint_as_float(o[4 * e + 3]) * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(p.out) + ob + c0);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            dst[e] = make_uint4(
                                pack_half2(__uint_as_float(o[8 * e]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                                pack_half2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv),
                                pack_half2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv),
                                pack_half2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv));
                        }
                    }
                }
            }
        }
    } else if (loader) {
        // ---------------------------------------------------------- loaders
        for (int j = issued; j < ntt; ++j) {
            int id = id0;
            id0 = id1;
            id1 = raw_id(j + 2);
            if (!load_tile(j, id)) break;
        }
        // copies still in flight (only after a wait ran out) land before the CTA exits
        if (B >= 16) {
            for (int j = max(0, issued - NS); j < issued; ++j) wait_lanes(bar(full[j % NS]), (j / NS) & 1, p.status);
        }
    } else if (warp == MMA_S_WARP) {
        // ------------------------------------------------- MMA: S = Q K^T
        constexpr uint32_t ID_S = idesc_f16(QT, BN, false);
        const uint32_t s_q = smem_addr(sm);
        bool ok = true;
        for (int j = 0; ok && j < ntt; ++j) {
            const int st = j % NS;
            if (!wait_lanes(bar(bars.k_full[st]), (j / NS) & 1, p.status)) break;
            for (int g = 0; g < 2; ++g) {
                if (j >= nt[g]) continue;
                // S of this query tile has been read (its previous tile)
                if (j > 0 && !wait_lanes(bar(bars.s_free[g]), (j - 1) & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_after_sync();
                if (lane == 0) {
                    const uint32_t a0 = s_q + g * C::Q_BYTES;
                    const uint32_t b0 = s_k + st * C::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma(tmem + g * BN, sdesc(a0 + (kk / 4) * QT * 128 + (kk % 4) * 32),
                             sdesc(b0 + (kk / 4) * BN * 128 + (kk % 4) * 32), ID_S, kk > 0);
                    umma_commit(bar(bars.s_full[g]));
                }
            }
            if (ok && lane == 0) umma_commit(bar(bars.k_empty[st]));
        }
        // every MMA issued has completed before tensor memory is released
        if (lane == 0) umma_commit(bar(bars.mma_done[0]));
        wait_lanes(bar(bars.mma_done[0]), 0, p.status);
    } else if (warp == MMA_PV_WARP) {
        // ------------------------------------------------ MMA: O += P V
        constexpr uint32_t ID_PV = idesc_f16(QT, 64, true);
        bool ok = true;
        for (int j = 0; ok && j < ntt; ++j) {
            const int st = j % NS;
            if (!wait_lanes(bar(bars.v_full[st]), (j / NS) & 1, p.status)) break;
            if (j == ntt - 1 && p_max - j * BN < BN - 1) {
                // V rows past the CTA's last position: zeros (a zero weight
                // times a non-finite value would not vanish)
                uint8_t *vt = sm + C::OFF_V + st * C::KV_BYTES;
                const int first = p_max - j * BN + 1;
                for (int e = lane; e < (BN - first) * 8 * C::HALVES; e += 32) {
                    const int row = first + e / (8 * C::HALVES);
                    const int rest = e % (8 * C::HALVES);
                    *reinterpret_cast<uint4 *>(vt + ((rest / 8) * BN + row) * 128 + (rest % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_shared();
                __syncwarp();
            }
            for (int g = 0; g < 2; ++g) {
                if (j >= nt[g]) continue;
                if (!wait_lanes(bar(bars.p_full[g]), j & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_after_sync();
                if (lane == 0) {
                    const uint32_t a0 = tmem + C::COL_P + g * (BN / 2);
                    const uint32_t v0 = s_v + st * C::KV_BYTES;
                    const uint32_t to = tmem + C::COL_O + g * D;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
#pragma unroll
                        for (int hf = 0; hf < C::HALVES; ++hf)
                            umma_ts(to + hf * 64, a0 + kk * 8, sdesc(v0 + hf * BN * 128 + kk * 2048), ID_PV,
                                    j > 0 || kk > 0);
                    }
                    umma_commit(bar(bars.o_done[g]));
                }
            }
            if (ok && lane == 0) umma_commit(bar(bars.v_empty[st]));
        }
        if (lane == 0) umma_commit(bar(bars.mma_done[1]));
        wait_lanes(bar(bars.mma_done[1]), 0, p.status);
    }

    tc_before_sync();
    __syncthreads();
    if (warp == MMA_S_WARP) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TMEM_COLS)
                     : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// K or V viewed as (64 elements, rows, halves, kv-heads) with strides (row,
// 128 bytes, head): a box {64, box_rows, 1, 1} is one 64-element half of
// box_rows consecutive rows of one kv-head, landing as [box_rows][128 bytes]
// in the 128-byte swizzle.
int encode(CUtensorMap *map, void *base, const pf_pool *pool, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return set_error(PF_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t rows = (cuuint64_t)pool->n_layers * pool->n_blocks * pool->block_size;
    const cuuint64_t D = (cuuint64_t)pool->head_dim;
    const cuuint64_t H = (cuuint64_t)pool->n_kv_heads;
    cuuint64_t dims[4] = {64, rows, D / 64, H};
    cuuint64_t strides[3] = {H * D * 2, 128, D * 2};
    cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, 1u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(PF_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r));
    return PF_OK;
}

}  // namespace
}  // namespace prefill_tc

int launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream) {
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;
    pf_pool *pool = const_cast<pf_pool *>(a.pool);
    const int D = pool->head_dim;
    const int BN = D == 64 ? prefill_tc::Cfg<64>::BN : prefill_tc::Cfg<128>::BN;
    const int gh = a.n_q_heads / pool->n_kv_heads;
    const long long n_items = (long long)a.n_seqs * pool->n_kv_heads;
    const long long n_qp = ((long long)a.max_new * gh + 2 * prefill_tc::QT - 1) / (2 * prefill_tc::QT);
    if (n_items * n_qp > 0x7fffffffll)
        return set_error(PF_ERR_INVALID, "pf_paged_prefill_attention: too many query tiles for one launch");
    const int box_rows = pool->block_size >= 16 ? (pool->block_size < BN ? pool->block_size : BN) : 1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_prefill_attention: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(PF_ERR_UNSUPPORTED, "device index out of range");
    {
        std::lock_guard<std::mutex> lock(pool->mu);
        if (!pool->tmap_pf_ready[dev]) {
            int rc = prefill_tc::encode(&pool->tmap_pf_k[dev], pool->k_base, pool, box_rows);
            if (rc) return rc;
            rc = prefill_tc::encode(&pool->tmap_pf_v[dev], pool->v_base, pool, box_rows);
            if (rc) return rc;
            pool->tmap_pf_ready[dev] = true;
        }
    }
    prefill_tc::Params p;
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
    p.box_rows = box_rows;
    p.n_items = (int)n_items;
    p.n_qp = (int)n_qp;
    p.layer_row0 = (long long)a.layer * pool->n_blocks * pool->block_size;
    p.out_f32 = a.out_dtype == PF_F32;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    void (*fn)(CUtensorMap, CUtensorMap, prefill_tc::Params) =
        D == 64 ? prefill_tc::prefill_tc_kernel<64> : prefill_tc::prefill_tc_kernel<128>;
    const int smem = D == 64 ? prefill_tc::Cfg<64>::SMEM : prefill_tc::Cfg<128>::SMEM;
    e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_prefill_attention: cudaFuncSetAttribute");
    fn<<<(unsigned)(n_items * n_qp), prefill_tc::NTHREADS, smem, stream>>>(pool->tmap_pf_k[dev], pool->tmap_pf_v[dev],
                                                                           p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_prefill_attention: launch");
    return PF_OK;
}

}  // namespace pkv
