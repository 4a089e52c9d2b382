// attention_kernel.cuh -- device code of single-query paged decode attention.
//
// What it computes (PagedAttention blog, "The Attention Kernel"): for each
// sequence s and query head hq, softmax(scale * q K^T) V over the sequence's
// L tokens, reading K/V through the block table; kv-head h = hq / G serves
// the G query heads of its group.  Long sequences are cut into chunks whose
// partial results (reference max m, sum l, unnormalised acc) are combined
// with the log-sum-exp rule (same section: a reduction across thread blocks
// combines partial softmax results).
//
// How, on sm_103a:
// * Work is counted in tiles of 16 tokens of one (sequence, group of HG
//   kv-heads) pair.  The pool stores a token's heads next to each other, so a
//   group's rows are one contiguous run of HG * D * 2 bytes (512 B for 4 heads
//   of 64): each TMA box {D, HG, 16 rows} moves 16 such runs.  A ragged last
//   group reads past n_kv_heads, which TMA fills with zeros without touching
//   memory.
// * Schedule "spans" (the default): the tiles of all pairs, in (sequence,
//   group, tile) order, are cut into one equal contiguous span per CTA of a
//   persistent grid (SMs x resident CTAs).  Every CTA reads the lengths,
//   scans the tile counts into shared memory and walks its own span: whole
//   pairs inside it are finished directly, and only the pairs cut by a span
//   boundary (at most two per CTA) leave partial results to merge.  The cut
//   points depend on the lengths alone, so results are bit-identical for any
//   placement of the pages.
// * Schedule "chunks" (split_tokens > 0, or -1 for one chunk per sequence):
//   fixed C-token chunks numbered chunk-major, group-minor, taken by the CTAs
//   with a static stride; the numbering comes from a warp prefix scan over
//   32-sequence windows of the lengths.
// * Warp 0 is the producer: it decodes items (the next one while the current
//   one's tiles are issued, so its block-table loads overlap), posts q by a
//   1-D bulk copy and streams 16-token K and V tiles into a ring of shared
//   memory stages with 3-D TMA; mbarrier full/empty pairs hand stages over.
// * Warps 1..4 are consumers; warp w serves head w / WPH of the group and
//   1/WPH of each tile's tokens (WPH = 4 / HG).  D/8 lanes hold one token row
//   (8 dims each, fp16 -> fp32); q . k reduces over those lanes with xor
//   shuffles; the softmax is an fp32 online softmax in the log2 domain whose
//   reference maximum is only raised when a score passes it by more than 2^8
//   (exact up to rounding: all terms share the reference); acc += p v.
// * End of item: token groups merge by shuffles (and the WPH warps of a head
//   through shared memory).  A whole sequence writes `out`; a chunk writes
//   its partial (acc[D], m, l) to the workspace, and the warp whose acq_rel
//   counter increment completes the count for (s, h) merges the partials of
//   that head and writes `out`, then resets the counter.  Nobody waits.
// * Every wait is bounded (1 s) and parks the thread in hardware while it
//   waits; a timeout sets PF_DEV_WAIT_TIMEOUT and the CTA returns after
//   waiting (bounded) for its own copies in flight.
#pragma once

#include "device_common.cuh"

namespace pkv {
namespace attn {

constexpr int TB = 16;                // tokens per staged tile
constexpr int NCW = 4;                // consumer warps
constexpr int NTHREADS = 32 * (NCW + 1);
constexpr int NQ = 2;                 // item (q) slots
constexpr float kRescaleLog2 = 8.0f;  // raise the reference max past 2^8
constexpr unsigned FULL = 0xffffffffu;

enum ItemKind { kWhole = 0, kChunk = 1, kSpanPart = 2 };

struct ItemDesc {
    int s;      // sequence; -1 = no more items
    int h0;     // first kv-head of the group
    int tok0;   // first token
    int ntok;   // tokens (>= 1)
    int kind;   // ItemKind
    int a;      // kChunk: global chunk index; kSpanPart: flattened first tile of the pair
    int b;      // kChunk: chunk index in the sequence; kSpanPart: tiles of the pair
    int c;      // kChunk: chunks of the sequence; kSpanPart: this CTA's record slot (0/1)
};

constexpr int kMaxSeqsPerLaunch = 1024;   // the span schedule keeps lengths in shared memory
constexpr int kSeqSmemInts = 2 * kMaxSeqsPerLaunch + 4;

struct Params {
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
    int n_groups;     // ceil(n_kv_heads / HG)
    int n_blocks;
    int block_size;
    int layer_row0;   // layer * n_blocks * block_size (< 2^31, checked at pool creation)
    int chunk;        // chunk schedule: tokens per chunk, multiple of TB
    int spans;        // 1 = span schedule, 0 = chunk schedule
    int out_f32;
    float scale_log2; // scale * log2(e)
};

// Span schedule over W flattened tiles and n = min(grid, W) CTAs (so no span
// is empty): CTA b < n owns tiles [span_start(b), span_start(b+1)).
__device__ __forceinline__ long long span_start(long long b, long long W, long long n) { return b * W / n; }
__device__ __forceinline__ long long span_ctas(long long W) { return W < (long long)gridDim.x ? W : gridDim.x; }
// The CTA whose span holds flattened tile x.
__device__ __forceinline__ long long span_owner(long long x, long long W, long long n) {
    return ((x + 1) * n - 1) / W;
}

template <int D, int HG>
struct Shape {
    static constexpr int STAGE_HALVES = TB * HG * D;                 // one of K or V
    static constexpr int STAGE_BYTES = 2 * STAGE_HALVES * 2;          // K + V
    static constexpr int RING_TARGET = D == 64 ? 64 * 1024 : 96 * 1024;
    static constexpr int NS_RAW = RING_TARGET / STAGE_BYTES;
    static constexpr int NS = NS_RAW < 3 ? 3 : (NS_RAW > 16 ? 16 : NS_RAW);
    static constexpr int WPH = NCW / HG;      // consumer warps per head
};

template <int D, int G, int HG>
struct __align__(128) Smem {
    static constexpr int NS = Shape<D, HG>::NS;
    __half k[NS][Shape<D, HG>::STAGE_HALVES];
    __half v[NS][Shape<D, HG>::STAGE_HALVES];
    __half q[NQ][HG * G * D];
    float red[Shape<D, HG>::WPH > 1 ? NCW : 1][G][D + 2];   // per consumer warp: acc[D], m, l
    ItemDesc desc[NQ];
    uint64_t full[NS];
    uint64_t empty[NS];
    uint64_t qfull[NQ];
    uint64_t qempty[NQ];
    uint64_t cbar;   // consumer-warps barrier (count NCW), used when WPH > 1
    int warp_tot[NTHREADS / 32];
    // span schedule: pre[s] = tiles (per group) of sequences before s, for
    // s = 0..S; len[s] = clamped length of sequence s
    int pre[kMaxSeqsPerLaunch + 1];
    int len[kMaxSeqsPerLaunch];
};

// ------------------------------------------------------------ producer

struct ProdItem {
    bool done;
    int s, h0, tok0, ntok, kind, a, b, c, pg0, npg;
    int ids0, ids1;   // raw block ids of pages pg0 + lane and pg0 + 32 + lane
};

template <int D, int G, int HG>
__device__ __forceinline__ void producer(const CUtensorMap *tmk, const CUtensorMap *tmv, const Params &p,
                                         Smem<D, G, HG> &sm, int lane) {
    constexpr int NS = Shape<D, HG>::NS;
    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }
    const uint64_t pol = policy_evict_first();
    const int B = p.block_size;
    const int C = p.chunk;
    const int ng = p.n_groups;
    const int maxctx = p.max_blocks * B;

    // Raw block id of page pg0 + off + lane (0 past the item).  Checked
    // where it is used, so the load's latency is not waited for here.
    auto load_id = [&](int s, int pg0, int npg, int off) {
        return (off + lane < npg) ? p.bt[(size_t)s * p.max_blocks + pg0 + off + lane] : 0;
    };
    auto checked = [&](int id) {
        if (id < 0 || id >= p.n_blocks) {
            atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);
            id = 0;   // stay inside the pool
        }
        return id;
    };
    auto finish_decode = [&](ProdItem &it, int L) {
        it.ntok = min(it.ntok, L - it.tok0);
        it.pg0 = it.tok0 / B;
        it.npg = (it.tok0 + it.ntok - 1) / B - it.pg0 + 1;
        it.ids0 = load_id(it.s, it.pg0, it.npg, 0);
        it.ids1 = load_id(it.s, it.pg0, it.npg, 32);
    };

    // ---- chunk schedule: 32-sequence window of the chunk numbering: per lane
    // its length, chunk count and inclusive prefix of chunk counts.
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
    auto decode_chunk = [&](int k) {
        ProdItem it;
        const long long item = (long long)blockIdx.x + (long long)k * gridDim.x;
        const long long u = item / ng;
        it.h0 = (int)(item - u * ng) * HG;
        it.done = false;
        while (u >= before + wtotal) {
            if (win + 32 >= p.n_seqs) {
                it.done = true;
                return it;
            }
            before += wtotal;
            win += 32;
            load_window(win);
        }
        const int rel = (int)(u - before);
        const unsigned hit = __ballot_sync(FULL, wincl > rel);
        const int ls = __ffs(hit) - 1;
        it.s = win + ls;
        const int L = __shfl_sync(FULL, wl, ls);
        const int nch = __shfl_sync(FULL, wu, ls);
        const int chunk = rel - __shfl_sync(FULL, wincl - wu, ls);
        it.kind = nch == 1 ? kWhole : kChunk;
        it.a = (int)u;
        it.b = chunk;
        it.c = nch;
        it.tok0 = chunk * C;
        it.ntok = C;
        finish_decode(it, L);
        return it;
    };

    // ---- span schedule: this CTA's flattened tiles [x, xend)
    const int S = p.n_seqs;
    long long W = 0, x = 0, xend = 0;
    long long n_span = 0;
    if (p.spans) {
        W = (long long)sm.pre[S] * ng;
        n_span = span_ctas(W);
        if (blockIdx.x < n_span) {
            x = span_start(blockIdx.x, W, n_span);
            xend = span_start(blockIdx.x + 1, W, n_span);
        }
    } else {
        load_window(0);
    }
    auto decode_span = [&]() {
        ProdItem it;
        it.done = x >= xend;
        if (it.done) return it;
        // largest s with pre[s] * ng <= x (it has tiles: pre[s + 1] * ng > x)
        int lo = 0, hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)sm.pre[mid] * ng <= x) lo = mid;
            else hi = mid - 1;
        }
        const int s = lo;
        const int nt = sm.pre[s + 1] - sm.pre[s];
        const long long pair0 = (long long)sm.pre[s] * ng;
        const int grp = (int)((x - pair0) / nt);
        const int t0 = (int)(x - pair0 - (long long)grp * nt);
        const int len = (int)min((long long)(nt - t0), xend - x);
        it.s = s;
        it.h0 = grp * HG;
        it.tok0 = t0 * TB;
        it.ntok = len * TB;
        const bool whole = t0 == 0 && len == nt;
        it.kind = whole ? kWhole : kSpanPart;
        it.a = (int)(pair0 + (long long)grp * nt);       // flattened first tile of the pair
        it.b = nt;
        it.c = (x == span_start(blockIdx.x, W, n_span)) ? 0 : 1;
        x += len;
        finish_decode(it, sm.len[s]);
        return it;
    };
    auto decode = [&](int k) { return p.spans ? decode_span() : decode_chunk(k); };

    constexpr uint32_t kTileBytes = 2u * TB * HG * D * 2;   // K + V boxes of a tile
    uint32_t st = 0;   // tiles issued
    int posted = 0;    // item slots posted (including the final sentinel)
    bool ok = true;
    ProdItem it = decode(0);
    for (int k = 0;; ++k) {
        const int slot = k % NQ;
        if (!warp_wait(smem_addr(&sm.qempty[slot]), ((k / NQ) & 1) ^ 1, p.status, lane)) break;
        if (it.done) {
            if (lane == 0) {
                sm.desc[slot].s = -1;
                mbar_arrive(smem_addr(&sm.qfull[slot]));
            }
            ++posted;
            break;
        }
        if (lane == 0) {
            ItemDesc d;
            d.s = it.s;
            d.h0 = it.h0;
            d.tok0 = it.tok0;
            d.ntok = it.ntok;
            d.kind = it.kind;
            d.a = it.a;
            d.b = it.b;
            d.c = it.c;
            sm.desc[slot] = d;
            const int nv = min(HG, p.n_kv_heads - it.h0);           // heads that exist
            const uint32_t qbytes = (uint32_t)nv * G * D * 2;
            mbar_arrive_expect_tx(smem_addr(&sm.qfull[slot]), qbytes);
            bulk_load(smem_addr(sm.q[slot]), p.q + ((size_t)it.s * p.n_q_heads + (size_t)it.h0 * G) * D, qbytes,
                      smem_addr(&sm.qfull[slot]));
        }
        ++posted;

        // The next item's numbering and block ids are requested now; their
        // latency overlaps with issuing this item's tiles.
        const ProdItem nx = decode(k + 1);

        int wbase = 0;
        int cur = it.ids0;
        int nxt = it.ids1;
        const int ntiles = (it.ntok + TB - 1) / TB;
        for (int j = 0; j < ntiles; ++j, ++st) {
            const int t = it.tok0 + j * TB;
            const int nt = min(TB, it.tok0 + it.ntok - t);
            const int pa = t / B - it.pg0;            // first page of the tile, item-relative
            if (pa - wbase >= 32) {                    // move to the prefetched window
                wbase += 32;
                cur = nxt;
                nxt = load_id(it.s, it.pg0, it.npg, wbase + 32);
            }
            const int stage = st % NS;
            if (!warp_wait(smem_addr(&sm.empty[stage]), ((st / NS) & 1) ^ 1, p.status, lane)) {
                ok = false;
                break;
            }
            const uint32_t full_bar = smem_addr(&sm.full[stage]);
            if (B >= TB) {
                // the tile is rows [t % B, t % B + TB) of one page
                const int id = checked(__shfl_sync(FULL, cur, pa - wbase));
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar, kTileBytes);
                    const int r = p.layer_row0 + id * B + (t % B);
                    tma_load_3d(smem_addr(sm.k[stage]), tmk, 0, it.h0, r, full_bar, pol);
                    tma_load_3d(smem_addr(sm.v[stage]), tmv, 0, it.h0, r, full_bar, pol);
                }
            } else {
                // B < TB (B = 1): one box of B rows per page
                const int pb = (t + nt - 1) / B - it.pg0;
                const int np = pb - pa + 1;
                const int raw = __shfl_sync(FULL, cur, (pa - wbase + lane) & 31);
                if (lane == 0) mbar_arrive_expect_tx(full_bar, (uint32_t)np * B * HG * D * 2 * 2);
                __syncwarp();
                if (lane < np) {
                    const int r = p.layer_row0 + checked(raw) * B;
                    const int off = lane * B * HG * D;
                    tma_load_3d(smem_addr(sm.k[stage] + off), tmk, 0, it.h0, r, full_bar, pol);
                    tma_load_3d(smem_addr(sm.v[stage] + off), tmv, 0, it.h0, r, full_bar, pol);
                }
            }
        }
        if (!ok) break;
        it = nx;
    }

    // Wait (bounded) for this CTA's last copies so none is in flight when the
    // CTA retires, whatever happened above.
    const uint32_t last = st < (uint32_t)NS ? st : (uint32_t)NS;
    for (uint32_t i = 0; i < last; ++i) {
        const uint32_t xs = st - 1 - i;
        warp_wait(smem_addr(&sm.full[xs % NS]), (xs / NS) & 1, p.status, lane);
    }
    for (int i = 0; i < NQ && i < posted; ++i) {
        const int xq = posted - 1 - i;
        warp_wait(smem_addr(&sm.qfull[xq % NQ]), (xq / NQ) & 1, p.status, lane);
    }
}

// ------------------------------------------------------------ consumers

// Store 8 consecutive output values (dims d0 .. d0 + 7) of one q-head row.
__device__ __forceinline__ void store8(const Params &p, size_t o, const float (&x)[8]) {
    if (p.out_f32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o);
        dst[0] = make_float4(x[0], x[1], x[2], x[3]);
        dst[1] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
        uint4 v;
        __half2 *h = reinterpret_cast<__half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
        *reinterpret_cast<uint4 *>(static_cast<__half *>(p.out) + o) = v;
    }
}

// Finish one (item, head) from the state a warp holds: lanes 0 .. D/8 - 1
// hold dims [8 * lane, 8 * lane + 8) of acc; m and l are the same in every
// lane.  A whole pair writes out.  A part writes its partial record, counts
// it, and if this warp's count completes the head, merges every record of the
// head (chunk records, or the span records of the CTAs that share the pair).
template <int D, int G, int HG>
__device__ __forceinline__ void finish_head(const Params &p, const Smem<D, G, HG> &sm, const ItemDesc &d, int h,
                                            int hl, int lane, const float (&m)[G], const float (&l)[G],
                                            const float (&acc)[G][8]) {
    constexpr int LPT = D / 8;
    constexpr int REC = G * (D + 2);   // floats per record: per q-head acc[D], m, l
    const int Hq = p.n_q_heads;
    if (d.kind == kWhole) {
        if (lane < LPT) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float x[8];
                const float inv = 1.0f / l[g];
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = acc[g][i] * inv;
                store8(p, ((size_t)d.s * Hq + (size_t)h * G + g) * D + lane * 8, x);
            }
        }
        return;
    }
    const int Hkv = p.n_kv_heads;
    // record of this part, and how to find every record of the head
    long long W = 0, n_cta = 0;
    int b_first = 0, n_parts;
    size_t rec;
    if (d.kind == kChunk) {
        rec = (size_t)d.a * Hkv + h;
        n_parts = d.c;
    } else {
        W = (long long)sm.pre[p.n_seqs] * p.n_groups;
        n_cta = span_ctas(W);
        b_first = (int)span_owner(d.a, W, n_cta);
        n_parts = (int)span_owner((long long)d.a + d.b - 1, W, n_cta) - b_first + 1;
        rec = ((size_t)blockIdx.x * 2 + d.c) * HG + hl;
    }
    float *part = p.partials + rec * REC;
    if (lane < LPT) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            // rows of D + 2 floats keep 8-float runs 8-byte (not 16-byte) aligned
            float2 *d2 = reinterpret_cast<float2 *>(part + g * (D + 2) + lane * 8);
#pragma unroll
            for (int i = 0; i < 4; ++i) d2[i] = make_float2(acc[g][2 * i], acc[g][2 * i + 1]);
            if (lane == 0) {
                part[g * (D + 2) + D] = m[g];
                part[g * (D + 2) + D + 1] = l[g];
            }
        }
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        const int old = atomic_add_acq_rel_gpu(&p.counters[(size_t)d.s * Hkv + h], 1);
        last = (old == n_parts - 1);
    }
    last = __shfl_sync(FULL, last, 0);
    if (!last) return;
    for (int e = lane; e < G * D; e += 32) {
        const int g = e / D;
        const int dd = e - g * D;
        float mx = -INFINITY, ls = 0.0f, a = 0.0f;
#pragma unroll 4
        for (int i = 0; i < n_parts; ++i) {
            size_t r;
            if (d.kind == kChunk) {
                r = (size_t)(d.a - d.b + i) * Hkv + h;
            } else {
                const long long b = b_first + i;
                const int z = span_start(b, W, n_cta) >= d.a ? 0 : 1;
                r = ((size_t)b * 2 + z) * HG + hl;
            }
            const float *pc = p.partials + r * REC + g * (D + 2);
            const float mc = __ldcg(pc + D);
            const float lc = __ldcg(pc + D + 1);
            const float ac = __ldcg(pc + dd);
            const float mn = fmaxf(mx, mc);
            const float fo = (mx == -INFINITY) ? 0.0f : exp2f(mx - mn);
            const float fc = exp2f(mc - mn);
            ls = ls * fo + lc * fc;
            a = a * fo + ac * fc;
            mx = mn;
        }
        const size_t o = ((size_t)d.s * Hq + (size_t)h * G + g) * D + dd;
        const float val = a / ls;
        if (p.out_f32) static_cast<float *>(p.out)[o] = val;
        else static_cast<__half *>(p.out)[o] = __float2half_rn(val);
    }
    if (lane == 0) p.counters[(size_t)d.s * Hkv + h] = 0;
}

template <int D, int G, int HG>
__device__ __forceinline__ void consumers(const Params &p, Smem<D, G, HG> &sm, int cw, int lane) {
    constexpr int NS = Shape<D, HG>::NS;
    constexpr int WPH = Shape<D, HG>::WPH;
    constexpr int LPT = D / 8;        // lanes per token row
    constexpr int TPW = 32 / LPT;     // tokens per warp-step
    constexpr int TPT = TB / WPH;     // tokens of a tile this warp serves
    constexpr int STEPS = TPT / TPW;
    static_assert(STEPS * TPW == TPT, "tile must split into whole warp-steps");
    const int grp = lane / LPT;
    const int sub = lane % LPT;
    const int hl = cw / WPH;          // head within the group
    const int part = cw % WPH;        // which share of each tile's tokens
    const int Hq = p.n_q_heads;

    // Empty (or invalid, clamped to empty) sequences get a zero output.
    for (int s = blockIdx.x; s < p.n_seqs; s += gridDim.x) {
        if (p.lens[s] <= 0) {
            for (int e = cw * 32 + lane; e < Hq * D; e += NCW * 32) {
                const size_t o = (size_t)s * Hq * D + e;
                if (p.out_f32) static_cast<float *>(p.out)[o] = 0.0f;
                else static_cast<__half *>(p.out)[o] = __float2half_rn(0.0f);
            }
        }
    }

    uint32_t st = 0;
    uint32_t cphase = 0;
    const uint32_t cbar = smem_addr(&sm.cbar);
    for (int k = 0;; ++k) {
        const int slot = k % NQ;
        if (!warp_wait(smem_addr(&sm.qfull[slot]), (k / NQ) & 1, p.status, lane)) return;
        const ItemDesc d = sm.desc[slot];
        if (d.s < 0) return;
        const int h = d.h0 + hl;
        const bool active = h < p.n_kv_heads;   // ragged last group: idle warps keep the protocol

        float qf[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (active) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(&sm.q[slot][(hl * G + g) * D + sub * 8]);
                half8_to_float(raw, qf[g]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) qf[g][i] = active ? qf[g][i] * p.scale_log2 : 0.0f;
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
            if (active) {
                const __half *kt = sm.k[stage];
                const __half *vt = sm.v[stage];
#pragma unroll
                for (int step = 0; step < STEPS; ++step) {
                    const int tl = part * TPT + step * TPW + grp;
                    const bool valid = d.tok0 + j * TB + tl < tend;
                    const int row = (tl * HG + hl) * D + sub * 8;
                    const uint4 kraw = *reinterpret_cast<const uint4 *>(kt + row);
                    const uint4 vraw = *reinterpret_cast<const uint4 *>(vt + row);
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

        if constexpr (WPH == 1) {
            if (active) finish_head<D, G, HG>(p, sm, d, h, hl, lane, m, l, acc);
        } else {
            // The WPH warps of a head meet in shared memory; the first of
            // them finishes the head.
            if (lane < LPT) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) sm.red[cw][g][lane * 8 + i] = acc[g][i];
                    if (lane == 0) {
                        sm.red[cw][g][D] = m[g];
                        sm.red[cw][g][D + 1] = l[g];
                    }
                }
            }
            if (!warps_sync(cbar, cphase, p.status, lane)) return;
            if (part == 0 && active) {
                const int w0 = cw;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int w = 0; w < WPH; ++w) mx = fmaxf(mx, sm.red[w0 + w][g][D]);
                    float ls = 0.0f;
                    float a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = 0.0f;
#pragma unroll
                    for (int w = 0; w < WPH; ++w) {
                        const float mw = sm.red[w0 + w][g][D];
                        const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - mx);
                        ls = fmaf(sm.red[w0 + w][g][D + 1], f, ls);
                        if (lane < LPT) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) a[i] = fmaf(sm.red[w0 + w][g][lane * 8 + i], f, a[i]);
                        }
                    }
                    m[g] = mx;
                    l[g] = ls;
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[g][i] = a[i];
                }
                finish_head<D, G, HG>(p, sm, d, h, hl, lane, m, l, acc);
            }
            if (!warps_sync(cbar, cphase, p.status, lane)) return;   // red[] is reused next item
        }
    }
}

template <int D, int G, int HG>
__global__ void __launch_bounds__(NTHREADS) paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                 const __grid_constant__ CUtensorMap tmv,
                                                                 const Params p) {
    constexpr int NS = Shape<D, HG>::NS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem<D, G, HG> &sm = *reinterpret_cast<Smem<D, G, HG> *>(smem_raw);
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
    if (p.spans) {
        // Clamped lengths and tile counts of every sequence, then an
        // exclusive prefix of the tile counts (all threads, in place).
        const int S = p.n_seqs;
        const int maxctx = p.max_blocks * p.block_size;
#pragma unroll 4
        for (int s = threadIdx.x; s < S; s += NTHREADS) {
            int L = p.lens[s];
            if (L < 0 || L > maxctx) {
                atomicOr(p.status, PF_DEV_BAD_LENGTH);
                L = L < 0 ? 0 : maxctx;
            }
            sm.len[s] = L;
            sm.pre[s + 1] = (L + TB - 1) / TB;
        }
        __syncthreads();
        const int per = (S + NTHREADS - 1) / NTHREADS;
        const int lo = 1 + threadIdx.x * per;
        const int hi = min(S + 1, lo + per);
        int local = 0;
        for (int i = lo; i < hi; ++i) local += sm.pre[i];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) sm.warp_tot[warp] = incl;
        __syncthreads();
        int run = incl - local;
        for (int w = 0; w < warp; ++w) run += sm.warp_tot[w];
        for (int i = lo; i < hi; ++i) {
            run += sm.pre[i];
            sm.pre[i] = run;
        }
        if (threadIdx.x == 0) sm.pre[0] = 0;
    }
    __syncthreads();
    if (warp == 0) producer<D, G, HG>(&tmk, &tmv, p, sm, lane);
    else consumers<D, G, HG>(p, sm, warp - 1, lane);
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);

struct KernelInfo {
    KernelFn fn;
    size_t smem;
};

// Defined in attention_d64.cu / attention_d128.cu.
KernelInfo kernel_d64(int g, int hg);
KernelInfo kernel_d128(int g, int hg);

}  // namespace attn
}  // namespace pkv
