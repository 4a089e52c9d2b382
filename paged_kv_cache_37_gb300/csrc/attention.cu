// attention.cu -- single-query paged decode attention (pf_paged_decode_attention).
//
// What it computes (PagedAttention blog, "The Attention Kernel"): for each
// sequence s and query head hq, softmax(scale * q K^T) V over the sequence's
// L tokens, reading K/V through the block table; kv-head h = hq / G serves
// the G query heads of its group.  Long sequences are cut into chunks whose
// partial results (running max m, sum l, unnormalised acc) are combined with
// the log-sum-exp rule (same section: a reduction across thread blocks).
//
// How, on sm_103a:
// * Work item = (chunk of C tokens of one sequence, kv-head h).  Items are
//   numbered unit-major, head-minor, and a persistent grid of
//   (SMs x resident CTAs) takes them with a static stride, so the CTAs
//   working at the same moment read all heads of the same pages together.
//   The unit numbering is computed on the device from context_lens by a
//   warp-wide prefix scan over 32-sequence windows (no host knowledge of the
//   lengths, no planning kernel).
// * Warp 0 is the producer.  It walks the block table, 32 entries per load
//   with the next window prefetched, and stages each 16-token tile of K and
//   of V for head h into a ring of shared-memory stages with 3-D TMA
//   (cp.async.bulk.tensor over the pool viewed as [rows][Hkv][D]; box
//   D x 1 x min(B, 16) rows).  The q rows of the item arrive by a 1-D bulk
//   copy.  mbarrier full/empty pairs hand stages to the consumers.
// * Warps 1..4 are consumers.  8 lanes hold one token row (16 B each: 8 dims
//   as fp16 -> fp32), so a warp covers 4 tokens (D = 64) or 2 (D = 128) per
//   step; q . k is a 3- or 4-step xor-shuffle reduction; the softmax is an
//   fp32 online softmax in the log2 domain whose reference maximum is only
//   raised when a score exceeds it by more than 2^8 (exact up to rounding:
//   every term is scaled by the same reference); then acc += p * v.
// * End of item: token groups merge by shuffles, warps through shared memory.
//   A whole sequence writes `out` directly; a chunk writes its partial
//   (acc[D], m, l) to the workspace, and the last chunk of (s, h) to arrive
//   -- found by an atomic counter, no waiting -- merges all partials and
//   writes `out`, then resets the counter to 0.
// * Every mbarrier wait is bounded (1 s); a timeout sets
//   PF_DEV_WAIT_TIMEOUT in the device status word and the CTA returns after
//   waiting (bounded) for its own copies in flight.
#include <cudaTypedefs.h>

#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int TB = kTileTokens;       // tokens per staged tile
constexpr int NCW = 4;                // consumer warps
constexpr int NTHREADS = 32 * (NCW + 1);
constexpr int NS = 8;                 // K/V ring stages
constexpr int NQ = 2;                 // item (q) slots
constexpr float kRescaleLog2 = 8.0f;  // raise the reference max past 2^8
constexpr unsigned FULL = 0xffffffffu;

struct ItemDesc {
    int s;      // sequence; -1 = no more items
    int h;      // kv-head
    int tok0;   // first token of the chunk
    int ntok;   // tokens in the chunk (>= 1)
    int unit;   // global chunk index (partials are stored per unit)
    int chunk;  // chunk index within the sequence
    int nch;    // chunks of this sequence
    int pad;
};

struct AttnParams {
    const __half *q;
    void *out;
    const int32_t *bt;
    const int32_t *lens;
    float *partials;
    int *counters;
    int *status;
    int n_seqs;
    int max_blocks;
    int n_q_heads;
    int n_kv_heads;
    int n_blocks;
    int block_size;
    int layer_row0;   // layer * n_blocks * block_size (< 2^31, checked at pool creation)
    int chunk;        // tokens per unit, multiple of TB
    int out_f32;
    float scale_log2; // scale * log2(e)
};

template <int D, int G>
struct __align__(128) Smem {
    __half k[NS][TB * D];
    __half v[NS][TB * D];
    __half q[NQ][G * D];
    float red[NCW][G][D + 2];   // per consumer warp: acc[D], m, l
    ItemDesc desc[NQ];
    uint64_t full[NS];
    uint64_t empty[NS];
    uint64_t qfull[NQ];
    uint64_t qempty[NQ];
    uint64_t cbar;              // consumer-warps barrier (count NCW)
    int is_last;
};

// ------------------------------------------------------------ producer

template <int D, int G>
__device__ __forceinline__ void producer(const CUtensorMap *tmk, const CUtensorMap *tmv, const AttnParams &p,
                                         Smem<D, G> &sm, int lane) {
    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }
    const uint64_t pol = policy_evict_first();
    const int Hkv = p.n_kv_heads;
    const int B = p.block_size;
    const int C = p.chunk;
    const int maxctx = p.max_blocks * B;

    // 32-sequence window of the unit numbering: per lane its length, unit
    // count and inclusive prefix of unit counts inside the window.
    int win = 0, wl = 0, wu = 0, wincl = 0, wtotal = 0;
    long long before = 0;
    auto load_window = [&](int base) {
        const int s = base + lane;
        int L = 0;
        if (s < p.n_seqs) {
            L = p.lens[s];
            if (L < 0 || L > maxctx) {
                atomicOr(p.status, PF_DEV_BAD_LENGTH);
                L = L < 0 ? 0 : maxctx;
            }
        }
        wl = L;
        wu = (L + C - 1) / C;
        int x = wu;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        wincl = x;
        wtotal = __shfl_sync(FULL, x, 31);
    };
    load_window(0);

    uint32_t st = 0;   // tiles issued
    int posted = 0;    // item slots posted (including the final sentinel)
    bool ok = true;
    for (int k = 0;; ++k) {
        const long long item = (long long)blockIdx.x + (long long)k * gridDim.x;
        const long long u = item / Hkv;
        const int h = (int)(item - u * Hkv);
        bool done = false;
        while (u >= before + wtotal) {
            if (win + 32 >= p.n_seqs) {
                done = true;
                break;
            }
            before += wtotal;
            win += 32;
            load_window(win);
        }
        const int slot = k % NQ;
        if (done) {
            if (!warp_wait(smem_addr(&sm.qempty[slot]), ((k / NQ) & 1) ^ 1, p.status, lane)) break;
            if (lane == 0) {
                sm.desc[slot].s = -1;
                mbar_arrive(smem_addr(&sm.qfull[slot]));
            }
            ++posted;
            break;
        }
        const int rel = (int)(u - before);
        const unsigned hit = __ballot_sync(FULL, wincl > rel);
        const int ls = __ffs(hit) - 1;
        const int s = win + ls;
        const int L = __shfl_sync(FULL, wl, ls);
        const int nch = __shfl_sync(FULL, wu, ls);
        const int chunk = rel - __shfl_sync(FULL, wincl - wu, ls);
        const int tok0 = chunk * C;
        const int ntok = min(C, L - tok0);
        const int ntiles = (ntok + TB - 1) / TB;

        // Block-table entries of the item's pages, 32 per window, next
        // window prefetched.  Ids outside the pool are flagged and replaced
        // by block 0 so every copy stays inside the pool.
        const int pg0 = tok0 / B;
        const int npg = (tok0 + ntok - 1) / B - pg0 + 1;
        const int32_t *row = p.bt + (size_t)s * p.max_blocks + pg0;
        auto load_ids = [&](int off) {
            int id = 0;
            if (off + lane < npg) {
                id = row[off + lane];
                if (id < 0 || id >= p.n_blocks) {
                    atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
                    id = 0;
                }
            }
            return id;
        };
        int wbase = 0;
        int cur = load_ids(0);
        int nxt = load_ids(32);

        if (!warp_wait(smem_addr(&sm.qempty[slot]), ((k / NQ) & 1) ^ 1, p.status, lane)) break;
        if (lane == 0) {
            ItemDesc d;
            d.s = s;
            d.h = h;
            d.tok0 = tok0;
            d.ntok = ntok;
            d.unit = (int)u;
            d.chunk = chunk;
            d.nch = nch;
            d.pad = 0;
            sm.desc[slot] = d;
            const uint32_t qbytes = G * D * 2;
            mbar_arrive_expect_tx(smem_addr(&sm.qfull[slot]), qbytes);
            bulk_load(smem_addr(sm.q[slot]), p.q + ((size_t)s * p.n_q_heads + (size_t)h * G) * D, qbytes,
                      smem_addr(&sm.qfull[slot]));
        }
        ++posted;

        for (int j = 0; j < ntiles; ++j, ++st) {
            const int t = tok0 + j * TB;
            const int nt = min(TB, tok0 + ntok - t);
            const int pa = t / B - pg0;               // first page of the tile, item-relative
            if (pa - wbase >= 32) {                    // move to the prefetched window
                wbase += 32;
                cur = nxt;
                nxt = load_ids(wbase + 32);
            }
            const int stage = st % NS;
            if (!warp_wait(smem_addr(&sm.empty[stage]), ((st / NS) & 1) ^ 1, p.status, lane)) {
                ok = false;
                break;
            }
            const uint32_t full_bar = smem_addr(&sm.full[stage]);
            if (B >= TB) {
                // the tile is rows [t % B, t % B + TB) of one page
                const int id = __shfl_sync(FULL, cur, pa - wbase);
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar, 2u * TB * D * 2);
                    const int r = p.layer_row0 + id * B + (t % B);
                    tma_load_3d(smem_addr(sm.k[stage]), tmk, 0, h, r, full_bar, pol);
                    tma_load_3d(smem_addr(sm.v[stage]), tmv, 0, h, r, full_bar, pol);
                }
            } else {
                // B < TB (B = 1): TB / B pages per tile, one box of B rows each
                const int pb = (t + nt - 1) / B - pg0;
                const int np = pb - pa + 1;
                const int id = __shfl_sync(FULL, cur, (pa - wbase + lane) & 31);
                if (lane == 0) mbar_arrive_expect_tx(full_bar, 2u * np * B * D * 2);
                __syncwarp();
                if (lane < np) {
                    const int r = p.layer_row0 + id * B;
                    tma_load_3d(smem_addr(sm.k[stage] + lane * B * D), tmk, 0, h, r, full_bar, pol);
                    tma_load_3d(smem_addr(sm.v[stage] + lane * B * D), tmv, 0, h, r, full_bar, pol);
                }
            }
        }
        if (!ok) break;
    }

    // Wait (bounded) for this CTA's last copies so none is in flight when the
    // CTA retires, whatever happened above.
    const uint32_t last = st < (uint32_t)NS ? st : (uint32_t)NS;
    for (uint32_t i = 0; i < last; ++i) {
        const uint32_t x = st - 1 - i;
        warp_wait(smem_addr(&sm.full[x % NS]), (x / NS) & 1, p.status, lane);
    }
    for (int i = 0; i < NQ && i < posted; ++i) {
        const int x = posted - 1 - i;
        warp_wait(smem_addr(&sm.qfull[x % NQ]), (x / NQ) & 1, p.status, lane);
    }
}

// ------------------------------------------------------------ consumers

template <int D, int G>
__device__ __forceinline__ void consumers(const AttnParams &p, Smem<D, G> &sm, int cw, int lane) {
    constexpr int LPT = D / 8;        // lanes per token row
    constexpr int TPW = 32 / LPT;     // tokens per warp-step
    constexpr int TPS = NCW * TPW;    // tokens per CTA-step
    constexpr int STEPS = TB / TPS;
    static_assert(STEPS * TPS == TB, "tile must be a whole number of steps");
    const int grp = lane / LPT;
    const int sub = lane % LPT;
    const int ctid = cw * 32 + lane;
    const int Hkv = p.n_kv_heads;
    const int Hq = p.n_q_heads;

    // Empty (or invalid, clamped to empty) sequences get a zero output.
    for (int s = blockIdx.x; s < p.n_seqs; s += gridDim.x) {
        if (p.lens[s] <= 0) {
            for (int e = ctid; e < Hq * D; e += NCW * 32) {
                const size_t o = (size_t)s * Hq * D + e;
                if (p.out_f32) static_cast<float *>(p.out)[o] = 0.0f;
                else static_cast<__half *>(p.out)[o] = __float2half_rn(0.0f);
            }
        }
    }

    uint32_t st = 0;
    uint32_t cphase = 0;   // uses of the consumer barrier
    const uint32_t cbar = smem_addr(&sm.cbar);
    for (int k = 0;; ++k) {
        const int slot = k % NQ;
        if (!warp_wait(smem_addr(&sm.qfull[slot]), (k / NQ) & 1, p.status, lane)) return;
        const ItemDesc d = sm.desc[slot];
        if (d.s < 0) return;

        float qf[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(&sm.q[slot][g * D + sub * 8]);
            half8_to_float(raw, qf[g]);
#pragma unroll
            for (int i = 0; i < 8; ++i) qf[g][i] *= p.scale_log2;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.qempty[slot]));

        float m[G], l[G], acc[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[g][i] = 0.0f;
        }

        const int ntiles = (d.ntok + TB - 1) / TB;
        const int tend = d.tok0 + d.ntok;
        for (int j = 0; j < ntiles; ++j, ++st) {
            const int stage = st % NS;
            if (!warp_wait(smem_addr(&sm.full[stage]), (st / NS) & 1, p.status, lane)) return;
            const __half *kt = sm.k[stage];
            const __half *vt = sm.v[stage];
#pragma unroll
            for (int step = 0; step < STEPS; ++step) {
                const int tl = step * TPS + cw * TPW + grp;
                const bool valid = d.tok0 + j * TB + tl < tend;
                const uint4 kraw = *reinterpret_cast<const uint4 *>(kt + tl * D + sub * 8);
                const uint4 vraw = *reinterpret_cast<const uint4 *>(vt + tl * D + sub * 8);
                float kf[8];
                half8_to_float(kraw, kf);
                float z[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) a = fmaf(qf[g][i], kf[i], a);
                    z[g] = a;
                }
#pragma unroll
                for (int o = LPT / 2; o > 0; o >>= 1) {
#pragma unroll
                    for (int g = 0; g < G; ++g) z[g] += __shfl_xor_sync(FULL, z[g], o);
                }
                bool need = false;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (!valid) z[g] = -INFINITY;
                    need |= z[g] > m[g] + kRescaleLog2;
                }
                if (__any_sync(FULL, need)) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float mn = fmaxf(m[g], z[g]);
                        const float sc = (mn == -INFINITY) ? 1.0f : exp2f(m[g] - mn);
                        l[g] *= sc;
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[g][i] *= sc;
                        m[g] = mn;
                    }
                }
                if (valid) {
                    float vf[8];
                    half8_to_float(vraw, vf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float pz = exp2f(z[g] - m[g]);
                        l[g] += pz;
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(pz, vf[i], acc[g][i]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&sm.empty[stage]));
        }

        // Merge the token groups of this warp (lanes with the same `sub`).
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mo = __shfl_xor_sync(FULL, m[g], o);
                const float lo = __shfl_xor_sync(FULL, l[g], o);
                const float mn = fmaxf(m[g], mo);
                const float a = (m[g] == -INFINITY) ? 0.0f : exp2f(m[g] - mn);
                const float b = (mo == -INFINITY) ? 0.0f : exp2f(mo - mn);
                l[g] = l[g] * a + lo * b;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float ao = __shfl_xor_sync(FULL, acc[g][i], o);
                    acc[g][i] = acc[g][i] * a + ao * b;
                }
                m[g] = mn;
            }
        }
        if (grp == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int i = 0; i < 8; ++i) sm.red[cw][g][sub * 8 + i] = acc[g][i];
                if (sub == 0) {
                    sm.red[cw][g][D] = m[g];
                    sm.red[cw][g][D + 1] = l[g];
                }
            }
        }
        if (!warps_sync(cbar, cphase, p.status, lane)) return;

        const bool split = d.nch > 1;
        float *part = p.partials + ((size_t)d.unit * Hkv + d.h) * (size_t)(G * (D + 2));
        for (int e = ctid; e < G * D; e += NCW * 32) {
            const int g = e / D;
            const int dd = e - g * D;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCW; ++w) mx = fmaxf(mx, sm.red[w][g][D]);
            float ls = 0.0f, a = 0.0f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float mw = sm.red[w][g][D];
                const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - mx);
                ls = fmaf(sm.red[w][g][D + 1], f, ls);
                a = fmaf(sm.red[w][g][dd], f, a);
            }
            if (!split) {
                const size_t o = ((size_t)d.s * Hq + (size_t)d.h * G + g) * D + dd;
                const float val = a / ls;
                if (p.out_f32) static_cast<float *>(p.out)[o] = val;
                else static_cast<__half *>(p.out)[o] = __float2half_rn(val);
            } else {
                part[g * (D + 2) + dd] = a;
                if (dd == 0) {
                    part[g * (D + 2) + D] = mx;
                    part[g * (D + 2) + D + 1] = ls;
                }
            }
        }

        if (split) {
            __threadfence();
            if (!warps_sync(cbar, cphase, p.status, lane)) return;
            if (ctid == 0) {
                const int old = atomicAdd(&p.counters[(size_t)d.s * Hkv + d.h], 1);
                sm.is_last = (old == d.nch - 1);
            }
            if (!warps_sync(cbar, cphase, p.status, lane)) return;
            if (sm.is_last) {
                __threadfence();
                const int u0 = d.unit - d.chunk;
                for (int e = ctid; e < G * D; e += NCW * 32) {
                    const int g = e / D;
                    const int dd = e - g * D;
                    float mx = -INFINITY;
                    for (int c = 0; c < d.nch; ++c) {
                        const float *pc = p.partials + ((size_t)(u0 + c) * Hkv + d.h) * (size_t)(G * (D + 2)) +
                                          g * (D + 2);
                        mx = fmaxf(mx, __ldcg(pc + D));
                    }
                    float ls = 0.0f, a = 0.0f;
                    for (int c = 0; c < d.nch; ++c) {
                        const float *pc = p.partials + ((size_t)(u0 + c) * Hkv + d.h) * (size_t)(G * (D + 2)) +
                                          g * (D + 2);
                        const float f = exp2f(__ldcg(pc + D) - mx);
                        ls = fmaf(__ldcg(pc + D + 1), f, ls);
                        a = fmaf(__ldcg(pc + dd), f, a);
                    }
                    const size_t o = ((size_t)d.s * Hq + (size_t)d.h * G + g) * D + dd;
                    const float val = a / ls;
                    if (p.out_f32) static_cast<float *>(p.out)[o] = val;
                    else static_cast<__half *>(p.out)[o] = __float2half_rn(val);
                }
                if (ctid == 0) p.counters[(size_t)d.s * Hkv + d.h] = 0;
            }
        }
        if (!warps_sync(cbar, cphase, p.status, lane)) return;   // red[] / is_last reused next item
    }
}

template <int D, int G>
__global__ void __launch_bounds__(NTHREADS) paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                 const __grid_constant__ CUtensorMap tmv,
                                                                 const AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem<D, G> &sm = *reinterpret_cast<Smem<D, G> *>(smem_raw);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_addr(&sm.full[i]), 1);
            mbar_init(smem_addr(&sm.empty[i]), NCW);
        }
        for (int i = 0; i < NQ; ++i) {
            mbar_init(smem_addr(&sm.qfull[i]), 1);
            mbar_init(smem_addr(&sm.qempty[i]), NCW);
        }
        mbar_init(smem_addr(&sm.cbar), NCW);
        mbar_init_fence();
    }
    __syncthreads();
    if (warp == 0) producer<D, G>(&tmk, &tmv, p, sm, lane);
    else consumers<D, G>(p, sm, warp - 1, lane);
}

// ------------------------------------------------------------ host side

using KernelFn = void (*)(CUtensorMap, CUtensorMap, AttnParams);

template <int D, int G>
KernelFn kernel_for() {
    return paged_decode_kernel<D, G>;
}

template <int D>
KernelFn pick_group(int g) {
    switch (g) {
        case 1: return kernel_for<D, 1>();
        case 2: return kernel_for<D, 2>();
        case 3: return kernel_for<D, 3>();
        case 4: return kernel_for<D, 4>();
        case 5: return kernel_for<D, 5>();
        case 6: return kernel_for<D, 6>();
        case 7: return kernel_for<D, 7>();
        case 8: return kernel_for<D, 8>();
        default: return nullptr;
    }
}

template <int D>
size_t smem_bytes_for(int g) {
    switch (g) {
        case 1: return sizeof(Smem<D, 1>);
        case 2: return sizeof(Smem<D, 2>);
        case 3: return sizeof(Smem<D, 3>);
        case 4: return sizeof(Smem<D, 4>);
        case 5: return sizeof(Smem<D, 5>);
        case 6: return sizeof(Smem<D, 6>);
        case 7: return sizeof(Smem<D, 7>);
        case 8: return sizeof(Smem<D, 8>);
        default: return 0;
    }
}

struct LaunchShape {
    bool ready = false;
    int grid = 0;
};

std::mutex g_shape_mu;
LaunchShape g_shapes[kMaxDevices][2][9];

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

int encode_one(CUtensorMap *map, void *base, const pf_pool *pool) {
    auto encode = get_encode_fn();
    if (!encode) return set_error(PF_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const uint64_t rows = (uint64_t)pool->n_layers * pool->n_blocks * pool->block_size;
    cuuint64_t dims[3] = {(cuuint64_t)pool->head_dim, (cuuint64_t)pool->n_kv_heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)pool->head_dim * 2, (cuuint64_t)pool->n_kv_heads * pool->head_dim * 2};
    const int box_rows = pool->block_size < TB ? pool->block_size : TB;
    cuuint32_t box[3] = {(cuuint32_t)pool->head_dim, 1u, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(PF_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r));
    return PF_OK;
}

}  // namespace

int encode_pool_tmaps(pf_pool *pool, int device) {
    std::lock_guard<std::mutex> lock(pool->mu);
    if (pool->tmap_ready[device]) return PF_OK;
    int rc = encode_one(&pool->tmap_k[device], pool->k_base, pool);
    if (rc) return rc;
    rc = encode_one(&pool->tmap_v[device], pool->v_base, pool);
    if (rc) return rc;
    pool->tmap_ready[device] = true;
    return PF_OK;
}

int attention_chunk_tokens(const pf_pool *pool, int max_blocks, int split_tokens) {
    const long long maxctx = (long long)max_blocks * pool->block_size;
    const long long cap = (maxctx + TB - 1) / TB * TB;
    if (cap > (1ll << 30)) {
        set_error(PF_ERR_INVALID, "attention: max_blocks_per_seq * block_size is too large");
        return 0;
    }
    long long c;
    if (split_tokens == -1) {
        c = cap;
    } else if (split_tokens > 0) {
        c = ((long long)split_tokens + TB - 1) / TB * TB;
    } else if (split_tokens == 0) {
        c = pool->head_dim == 64 ? 128 : 64;
    } else {
        set_error(PF_ERR_INVALID, "attention: split_tokens must be -1, 0 or positive");
        return 0;
    }
    if (c > cap) c = cap;
    if (c < TB) c = TB;
    return (int)c;
}

size_t attention_counter_bytes(int n_seqs, int n_kv_heads) {
    const size_t b = (size_t)n_seqs * (size_t)n_kv_heads * sizeof(int);
    return (b + 255) / 256 * 256;
}

size_t attention_partial_bytes(const pf_pool *pool, int n_seqs, int n_q_heads, int max_blocks, int chunk) {
    const long long maxctx = (long long)max_blocks * pool->block_size;
    const long long per_seq = (maxctx + chunk - 1) / chunk;
    if (per_seq <= 1) return 0;   // no sequence is ever split
    return (size_t)n_seqs * (size_t)per_seq * (size_t)n_q_heads * (size_t)(pool->head_dim + 2) * sizeof(float);
}

int launch_attention(const AttnArgs &a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_decode_attention: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(PF_ERR_UNSUPPORTED, "device index out of range");
    pf_pool *pool = a.pool;
    int rc = encode_pool_tmaps(pool, dev);
    if (rc) return rc;
    int *status = device_status_ptr();
    if (!status) return PF_ERR_CUDA;

    const int D = pool->head_dim;
    const int G = a.n_q_heads / pool->n_kv_heads;
    KernelFn fn = D == 64 ? pick_group<64>(G) : pick_group<128>(G);
    const size_t smem = D == 64 ? smem_bytes_for<64>(G) : smem_bytes_for<128>(G);
    if (!fn || smem == 0) return set_error(PF_ERR_UNSUPPORTED, "attention: unsupported head_dim / group");

    int grid = 0;
    {
        std::lock_guard<std::mutex> lock(g_shape_mu);
        LaunchShape &sh = g_shapes[dev][D == 64 ? 0 : 1][G];
        if (!sh.ready) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
            if (e != cudaSuccess) return cuda_error(e, "attention: cudaFuncSetAttribute");
            int occ = 0, sms = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, reinterpret_cast<const void *>(fn), NTHREADS,
                                                              smem);
            if (e != cudaSuccess) return cuda_error(e, "attention: occupancy query");
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_error(e, "attention: SM count");
            if (occ < 1) return set_error(PF_ERR_UNSUPPORTED, "attention: kernel does not fit on an SM");
            sh.grid = sms * occ;
            sh.ready = true;
        }
        grid = sh.grid;
    }

    AttnParams p;
    p.q = static_cast<const __half *>(a.q);
    p.out = a.out;
    p.bt = a.block_tables;
    p.lens = a.context_lens;
    const size_t cnt_bytes = attention_counter_bytes(a.n_seqs, pool->n_kv_heads);
    p.counters = static_cast<int *>(a.workspace);
    p.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + cnt_bytes);
    p.status = status;
    p.n_seqs = a.n_seqs;
    p.max_blocks = a.max_blocks;
    p.n_q_heads = a.n_q_heads;
    p.n_kv_heads = pool->n_kv_heads;
    p.n_blocks = pool->n_blocks;
    p.block_size = pool->block_size;
    p.layer_row0 = a.layer * pool->n_blocks * pool->block_size;
    p.chunk = a.chunk_tokens;
    p.out_f32 = a.out_dtype == PF_F32;
    p.scale_log2 = a.scale * 1.4426950408889634f;

    fn<<<grid, NTHREADS, smem, stream>>>(pool->tmap_k[dev], pool->tmap_v[dev], p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "pf_paged_decode_attention: launch");
    return PF_OK;
}

}  // namespace pkv
