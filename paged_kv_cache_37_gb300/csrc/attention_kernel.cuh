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
// * Fused decode step (k_new != null): the item that holds a sequence's
//   token L - 1 also bulk-copies that token's new K and V rows next to q.
//   The consumers use them in place of the tile's row L - 1 and write them
//   into the token's pool slot with plain stores; no other block reads that
//   slot in the launch, so nothing waits for the write.
// * End of item: token groups merge by shuffles (and the WPH warps of a head
//   through shared memory).  A whole pair writes `out`.  A part of a cut pair
//   writes its record (acc[D], m, l per q-head).
//   - Span schedule: every word of the record carries the launch's epoch
//     (one indivisible 64-bit store per value, no fence).  The pair's last
//     span merges it: when its CTA has no items left, the head's warp loads
//     the pair's records, polls until every word carries this launch's
//     epoch (the other parts belong to earlier spans, whose CTAs never wait
//     for anyone), combines them with the log-sum-exp rule and writes
//     `out`.  Nothing needs resetting between calls.
//   - Chunk schedule: chunk 0 of the pair also writes a merge job stamped
//     with the call's epoch; merge_kernel, launched next on the stream as a
//     programmatic dependent of this grid, merges every job of this epoch.
//   Only a merging warp waits for other CTAs, and only for parts that need
//   nothing from it.
// * Every wait is bounded (1 s) and parks the thread in hardware while it
//   waits; a timeout sets PF_DEV_WAIT_TIMEOUT and the CTA returns after
//   waiting (bounded) for its own copies in flight.
#pragma once

#include "device_common.cuh"

namespace pkv {
namespace attn {

constexpr int TB = 16;                // tokens per staged tile
constexpr int NCW = 4;                // consumer warps
constexpr int NTHREADS = 32 * (NCW + 1);  // producer, consumers
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
    int a;      // kChunk: global chunk index; kSpanPart: flattened first unit of the pair
    int b;      // kChunk: chunk index in the sequence; kSpanPart: units of the pair
    int c;      // kChunk: chunks of the sequence; kSpanPart: record slot (0/1) in the span
    int span;   // kSpanPart: span index
    int newrow;   // fused step: token L - 1 when this item holds it, else -1
    int newslot;  // fused step: pool row of token L - 1 (-1: bad block id, not written)
    int L;        // the sequence's (clamped) length
    int nq;       // its query tokens (1 for decode; the new tokens of an append)
    int qrow0;    // q / out row of its first query token
    int pad0;
};

// A cut pair to merge: records first .. first + n_parts - 1 (chunk records
// (unit * Hkv + h), or span records ((span * 2 + slot) * HG + hl) where only
// the first span can use slot 1).
struct Job {
    int s, h0, kind, first, z_first, n_parts;
    unsigned epoch;
    int pad;
};

// A part of a cut pair that a consumer warp finished (span schedule): the
// pair's output location and the span records that hold its parts.
struct PendPart {
    int s, h0, first, z_first, n_parts, qrow0, nq;
};

constexpr int kMaxSeqsPerLaunch = 512;

// Span schedule: a (sequence, head-group) pair costs its tiles plus
// kPairCost "cost units" (tiles' worth) in the partition, so spans of many
// short pairs get fewer tiles.  The cost units sit at the pair's start and
// carry no work.  Measured on the mixed workload: a CTA's last tile comes
// about 0.6 us later per tile and 0.9 us later per item of its span; per
// call (per call / back to back) with a cost of 1: 39.5 / 35.3 us, 2: 39.1 /
// 34.6, 3: 39.0 / 34.5, 4: 39.3 / 34.5, 5: 40.4 / 35.0, 6: 40.8 / 35.2.
constexpr int kPairCost = 3;

struct Params {
    const __half *q;
    // fused decode step (pf_decode_step): the new token of each sequence,
    // [n_seqs][n_kv_heads][D]: attended to as token L - 1 and written to
    // that token's pool slot; null for plain attention
    const __half *k_new;
    const __half *v_new;
    __half *k_pool;   // pool bases (for the fused write)
    __half *v_pool;
    void *out;
    const int32_t *bt;
    const int32_t *lens;
    float *partials;         // chunk schedule: fp32 records of the chunks of cut pairs
    struct Job *jobs;        // chunk schedule: merge jobs for merge_kernel
    // span schedule: records of the parts of cut pairs, 64-bit words
    // (value, epoch) per float (see st_tagged)
    unsigned long long *span_recs;
    unsigned epoch;   // this launch's stamp for merge jobs and span records (never 0)
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
    int prefetch_tiles;   // tiles of the first item pulled into L2 before the dependency wait (<= 32)
    // Append (multi-token) attention: sequence s's query tokens are q rows
    // cu_q[s] .. cu_q[s + 1] - 1, the last positions of its L tokens, each
    // attending causally.  Null for decode (one query per sequence, row s).
    // A kv-head's G rows are its query tokens x its gh q-heads.
    const int32_t *cu_q;
    int gh;               // q-heads per kv-head
    int rows;             // rows per kv-head the call allows (gh for decode; <= the instance's G)
    // Testing hook (0 normally): block 0 never fills its first ring stage,
    // so the waits for it run out and the launch reports PF_DEV_WAIT_TIMEOUT.
    int test_skip;
};

// Span map of the span schedule: the W flattened tiles cut into
// n = min(W, grid) equal spans (none empty); CTA b takes span b.  Measured on
// the 128-sequence mixed workload, one static span per CTA beat every
// dynamic scheme tried (ticketed spans of equal or decreasing size): small
// spans pay per-segment costs and cut more pairs, and the merges of the cut
// pairs cost more than the balance gains.
struct SpanMap {
    long long W;   // tiles in all
    long long n;   // spans
    bool narrow;   // W * n < 2^32: the products and quotients fit 32-bit unsigned arithmetic
    __device__ __forceinline__ SpanMap(long long W_, int grid)
        : W(W_), n(W_ < grid ? W_ : grid), narrow(W_ * (W_ < grid ? W_ : grid) < (1ll << 32)) {}
    // first tile of span j (W for j = n)
    __device__ __forceinline__ long long start(long long j) const {
        if (j >= n) return W;
        return narrow ? (long long)((unsigned)W * (unsigned)j / (unsigned)n) : W * j / n;
    }
    // the span that holds tile x
    __device__ __forceinline__ long long owner(long long x) const {
        return narrow ? (long long)((((unsigned)x + 1u) * (unsigned)n - 1u) / (unsigned)W) : ((x + 1) * n - 1) / W;
    }
};

template <int D, int HG>
struct Shape {
    static constexpr int STAGE_HALVES = TB * HG * D;                 // one of K or V
    static constexpr int STAGE_BYTES = 2 * STAGE_HALVES * 2;          // K + V
    static constexpr int RING_TARGET = D == 64 ? 64 * 1024 : 96 * 1024;
    static constexpr int NS_RAW = RING_TARGET / STAGE_BYTES;
    static constexpr int NS = NS_RAW < 3 ? 3 : (NS_RAW > 16 ? 16 : NS_RAW);
    static constexpr int WPH = NCW / HG;      // consumer warps per head
};

// Tensor-core consumers (HG kv-heads per item, each head's tiles dealt
// round-robin to its NCW / HG consumer warps): a stage holds SUB consecutive
// 16-token tiles of one item behind one full/empty barrier pair, so that a
// stage is at least kMmaStageMinBytes (with few kv-heads per item a tile is
// small, and a barrier round trip and a producer turn per tile would bound
// the rate).  The ring takes what is left of a CTA's share of the SM's
// 228 KB -- 3 CTAs per SM at head_dim 64, 2 at 128 -- after the fixed part
// (q slots, new rows, the warps' merge area, the span tables, barriers),
// between 2 and 16 stages.
#ifndef PKV_MMA_STAGE_MIN_BYTES
#define PKV_MMA_STAGE_MIN_BYTES 16384
#endif
constexpr int kMmaStageMinBytes = PKV_MMA_STAGE_MIN_BYTES;
template <int D, int G, int HG>
struct MmaShape {
    static constexpr int TILE_BYTES = 2 * TB * HG * D * 2;   // K and V of one tile
    static constexpr int BUDGET = (D == 64 ? 228 * 1024 / 3 : 228 * 1024 / 2) - 2048;   // reserved + alignment slack
    static constexpr bool MERGE = NCW / HG > 1;   // several warps per head meet in shared memory
    static constexpr int REDW = MERGE ? HG * (NCW / HG - 1) : 1;   // merge slots: a head's warps but its first
    static constexpr int FIXED = NQ * HG * G * D * 2 + NQ * 2 * HG * D * 2 + REDW * G * (D + 2) * 4 +
                                 (kMaxSeqsPerLaunch + 1) * 4 + kMaxSeqsPerLaunch + 1024;   // + barriers, items
    static constexpr int SUB_WANT = TILE_BYTES >= kMmaStageMinBytes ? 1 : kMmaStageMinBytes / TILE_BYTES;
    static constexpr int SUB_FIT = (BUDGET - FIXED) / (2 * TILE_BYTES);   // at least two stages
    static constexpr int SUB = SUB_WANT < SUB_FIT ? SUB_WANT : (SUB_FIT < 1 ? 1 : SUB_FIT);
    static constexpr int STAGE_BYTES = SUB * TILE_BYTES;
    static constexpr int NS_RAW = (BUDGET - FIXED) / STAGE_BYTES;
    static constexpr int NS = NS_RAW < 2 ? 2 : (NS_RAW > 16 ? 16 : NS_RAW);
};

// MMA: the stages hold swizzled tiles (128-byte rows, 16-byte chunks XORed
// with the row index mod 8) and must sit at 1024-byte boundaries; the kernel
// places the struct there at run time.
template <int D, int G, int HG, bool MMA = false>
struct __align__(128) Smem {
    static constexpr int NS = MMA ? MmaShape<D, G, HG>::NS : Shape<D, HG>::NS;
    static constexpr int SUB = MMA ? MmaShape<D, G, HG>::SUB : 1;   // tiles per stage
    __half k[NS][SUB * Shape<D, HG>::STAGE_HALVES];
    __half v[NS][SUB * Shape<D, HG>::STAGE_HALVES];
    __half q[NQ][HG * G * D];
    __half knew[NQ][2][HG * D];   // fused step: the new token's K and V rows of the item's heads
    // acc[D], m, l per merging warp: every consumer warp (CUDA cores), a head's
    // warps but its first (tensor cores)
    float red[MMA ? MmaShape<D, G, HG>::REDW : (Shape<D, HG>::WPH > 1 ? NCW : 1)][G][D + 2];
    ItemDesc desc[NQ];
    uint64_t full[NS];
    uint64_t empty[NS];
    uint64_t qfull[NQ];
    uint64_t qempty[NQ];
    uint64_t cbar;   // consumer-warps barrier (count NCW), used when WPH > 1
    PendPart pend[NCW][2];   // span schedule: this warp's cut parts (record slot 0 / 1)
    int warp_tot[NTHREADS / 32];
    // span schedule: pre[s] = units (per group: tiles + kPairCost, 0 for an
    // empty sequence) of sequences before s, for
    // s = 0..S; rem[s] = tokens of sequence s in its last tile (1..16), so
    // its clamped length is (pre[s + 1] - pre[s] - kPairCost - 1) * 16 + rem[s]
    int pre[kMaxSeqsPerLaunch + 1];
    uint8_t rem[kMaxSeqsPerLaunch];
    int s_first;   // span schedule: the sequence that holds this CTA's first unit
};

// L2 prefetch of the first min(row, max(128, kTablePrefetchBytes / S)) bytes
// of each block-table row, the 128-byte lines shared out over all threads
// of the grid.  Only addresses inside the table are touched.
constexpr long long kTablePrefetchBytes = 1 << 20;

__device__ __forceinline__ void prefetch_table_rows(const Params &p) {
    const long long row_bytes = (long long)p.max_blocks * 4;
    long long per_row = kTablePrefetchBytes / (p.n_seqs > 0 ? p.n_seqs : 1);
    if (per_row < 128) per_row = 128;
    if (per_row > row_bytes) per_row = row_bytes;
    const long long lines = (per_row + 127) / 128;
    const long long total = lines * p.n_seqs;
    const char *base = reinterpret_cast<const char *>(p.bt);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long s = i / lines;
        const long long off = (i - s * lines) * 128;
        prefetch_l2(base + s * row_bytes + off);
    }
}

// Append: a sequence without query tokens has no work (length 0); more
// query tokens than its length or than the call's rows hold is flagged (and
// clamped where the tokens are read).  Decode: the length as is.
__device__ __forceinline__ int append_length(const Params &p, int s, int L) {
    if (p.cu_q == nullptr) return L;
    const int nq = p.cu_q[s + 1] - p.cu_q[s];
    if (nq < 0 || nq > L || nq * p.gh > p.rows) atomicOr(p.status, PF_DEV_BAD_LENGTH);
    return nq > 0 ? L : 0;
}

// ------------------------------------------------------------ producer

struct ProdItem {
    bool done;
    int s, h0, tok0, ntok, kind, a, b, c, span, pg0, npg, L;
    int last_id;      // fused step: raw block id of token L - 1 when the item holds it
    int ids0, ids1;   // raw block ids of pages pg0 + lane and pg0 + 32 + lane
    int qrow0, nq;    // q row of the sequence's first query token; its query tokens
};

// Byte offset, in an MMA stage (one kv-head), of 16-byte chunk c (dims
// 8c .. 8c + 7) of tile row t: per 64-dim half, TB rows of 128 bytes, chunk
// c % 8 of row t stored at position (c % 8) ^ (t % 8) -- the layout a TMA
// copy with 128-byte swizzling writes at a 1024-byte aligned stage.
__device__ __forceinline__ uint32_t swz(int t, int c) {
    return (uint32_t)((((c >> 3) * TB + t) << 7) + ((((c & 7) ^ (t & 7))) << 4));
}

// Issue one K or V tile (pool rows r .. r + TB - 1 of heads h0 ..) into a
// stage.  Plain: one box {D, HG, TB}.  MMA: one swizzled box {64, TB, (D /
// 64,) HG} of the heads-outermost map, landing as [head][half][row][64]:
// head hl's half hf at stage offset (hl * D / 64 + hf) * TB * 64.
template <int D, int HG, bool MMA>
__device__ __forceinline__ void tile_load(__half *dst, const CUtensorMap *map, int h0, int r, uint32_t bar,
                                          uint64_t pol) {
    if constexpr (!MMA) tma_load_3d(smem_addr(dst), map, 0, h0, r, bar, pol);
    else if constexpr (D == 64) tma_load_3d(smem_addr(dst), map, 0, r, h0, bar, pol);
    else tma_load_4d(smem_addr(dst), map, 0, r, 0, h0, bar, pol);
}

template <int D, int HG, bool MMA>
__device__ __forceinline__ void tile_prefetch(const CUtensorMap *map, int h0, int r) {
    if constexpr (!MMA) tma_prefetch_3d(map, 0, h0, r);
    else if constexpr (D == 64) tma_prefetch_3d(map, 0, r, h0);
    else tma_prefetch_4d(map, 0, r, 0, h0);
}

template <int D, int G, int HG, bool MMA = false>
__device__ __forceinline__ void producer(const CUtensorMap *tmk, const CUtensorMap *tmv, const Params &p,
                                         Smem<D, G, HG, MMA> &sm, int lane) {
    constexpr int NS = Smem<D, G, HG, MMA>::NS;
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
        it.L = L;
        it.ntok = min(it.ntok, L - it.tok0);
        it.pg0 = it.tok0 / B;
        it.npg = (it.tok0 + it.ntok - 1) / B - it.pg0 + 1;
        it.ids0 = load_id(it.s, it.pg0, it.npg, 0);
        it.ids1 = load_id(it.s, it.pg0, it.npg, 32);
        // Fused decode step: the item that ends at the sequence's end holds
        // its newest token; its page's block id is needed when it is posted.
        it.last_id = (p.k_new != nullptr && it.tok0 + it.ntok == L)
                         ? p.bt[(size_t)it.s * p.max_blocks + (L - 1) / B] : 0;
        // Append: the sequence's query tokens (clamped as the length scan
        // flagged them); decode: one, at row s.
        if (p.cu_q != nullptr) {
            it.qrow0 = p.cu_q[it.s];
            it.nq = max(1, min(min(p.cu_q[it.s + 1] - it.qrow0, L), p.rows / p.gh));
        } else {
            it.qrow0 = it.s;
            it.nq = 1;
        }
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
            L = append_length(p, s, L);
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

    // ---- span schedule: this CTA's span, walked segment by segment
    const int S = p.n_seqs;
    const SpanMap map(p.spans ? (long long)sm.pre[S] * ng : 0, gridDim.x);
    const long long span = blockIdx.x;
    long long x = 0, xend = 0;
    if (p.spans) {
        x = map.start(span);
        xend = map.start(span + 1);
    } else {
        load_window(0);
    }
    const long long sstart = x;
    auto decode_span = [&]() {
        ProdItem it;
        for (;;) {
            it.done = x >= xend;
            if (it.done) return it;
            // largest s with pre[s] * ng <= x (it has units: pre[s + 1] * ng > x);
            // the prologue found it for the span's first unit
            int lo = 0, hi = S - 1;
            if (x == sstart) lo = hi = sm.s_first;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if ((long long)sm.pre[mid] * ng <= x) lo = mid;
                else hi = mid - 1;
            }
            const int s = lo;
            const int u = sm.pre[s + 1] - sm.pre[s];          // units of each of its pairs
            const int nt = u - kPairCost;                     // tiles of each of its pairs
            const long long pair0 = (long long)sm.pre[s] * ng;
            const int grp = map.narrow ? (int)((unsigned)(x - pair0) / (unsigned)u) : (int)((x - pair0) / u);
            const long long a = pair0 + (long long)grp * u;    // the pair's first unit (its cost unit)
            const int off = (int)(x - a);
            const int len = (int)min((long long)(u - off), xend - x);
            const int t0 = max(off - kPairCost, 0);           // the pair's tiles in this span
            const int t1 = min(off + len - kPairCost, nt);
            const bool first_segment = x == sstart;
            x += len;
            if (t1 <= t0) continue;                           // only the pair's cost unit: no work
            it.s = s;
            it.h0 = grp * HG;
            it.tok0 = t0 * TB;
            it.ntok = (t1 - t0) * TB;
            it.kind = (t0 == 0 && t1 == nt) ? kWhole : kSpanPart;
            it.a = (int)a;
            it.b = u;
            it.c = first_segment ? 0 : 1;
            it.span = (int)span;
            finish_decode(it, (nt - 1) * TB + sm.rem[s]);
            return it;
        }
    };
    auto decode = [&](int k) { return p.spans ? decode_span() : decode_chunk(k); };

    constexpr uint32_t kTileBytes = 2u * TB * HG * D * 2;   // K + V boxes of a tile
    uint32_t st = 0;   // tiles issued
    int posted = 0;    // item slots posted (including the final sentinel)
    bool ok = true;
    ProdItem it = decode(0);
    // Pull the first tiles into L2 before waiting for the previous kernel
    // (prefetch_tiles of them: deeper when this launch overlaps one).  A
    // prefetch brings nothing into this CTA: the copies after the wait read
    // the lines as they are then, with whatever the previous kernel wrote,
    // but from L2 instead of DRAM.
    if (!it.done && B >= TB) {
        const int j = lane;                                // this lane's tile of item 0
        const int tiles0 = (it.ntok + TB - 1) / TB;
        const int t = it.tok0 + j * TB;
        const int pa = j < tiles0 ? t / B - it.pg0 : 0;    // <= j < 32: inside the id window
        const int id = __shfl_sync(FULL, it.ids0, pa);
        if (j < p.prefetch_tiles && j < tiles0 && id >= 0 && id < p.n_blocks) {
            const int r = p.layer_row0 + id * B + (t % B);
            tile_prefetch<D, HG, MMA>(tmk, it.h0, r);
            tile_prefetch<D, HG, MMA>(tmv, it.h0, r);
        }
    }
    // Launched as a programmatic dependent: wait for the previous kernel on
    // the stream before the first read of q or the pool (a no-op otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Block ids of the current item: pages wbase .. wbase + 31 (lane l holds
    // page wbase + l in cur) and the next 32 (nxt), item-relative.
    int wbase = 0;
    int cur = it.ids0;
    int nxt = it.ids1;
    // Issue tiles j0 .. j0 + SUB - 1 of the current item (those it has) into
    // the next stage (st), at SUBH halves apart; false when the wait for the
    // stage gave up.
    constexpr int SUB = Smem<D, G, HG, MMA>::SUB;
    constexpr int SUBH = Shape<D, HG>::STAGE_HALVES;
    auto issue_stage = [&](int j0) -> bool {
        const int nsub = min(SUB, (it.ntok + TB - 1) / TB - j0);
        const int stage = st % NS;
        if (!warp_wait(smem_addr(&sm.empty[stage]), ((st / NS) & 1) ^ 1, p.status, lane)) return false;
        const uint32_t full_bar = smem_addr(&sm.full[stage]);
        if (st == 0 && p.test_skip && blockIdx.x == 0) {   // testing hook: nothing will fill this stage
            ++st;
            return true;
        }
        if (B >= TB) {
            if (lane == 0) mbar_arrive_expect_tx(full_bar, (uint32_t)nsub * kTileBytes);
        }
        for (int u = 0; u < nsub; ++u) {
            const int t = it.tok0 + (j0 + u) * TB;
            const int nt = min(TB, it.tok0 + it.ntok - t);
            const int pa = t / B - it.pg0;            // first page of the tile, item-relative
            if (pa - wbase >= 32) {                    // move to the prefetched window
                wbase += 32;
                cur = nxt;
                nxt = load_id(it.s, it.pg0, it.npg, wbase + 32);
            }
            if (B >= TB) {
                // the tile is rows [t % B, t % B + TB) of one page
                const int id = checked(__shfl_sync(FULL, cur, pa - wbase));
                if (lane == 0) {
                    const int r = p.layer_row0 + id * B + (t % B);
                    tile_load<D, HG, MMA>(sm.k[stage] + u * SUBH, tmk, it.h0, r, full_bar, pol);
                    tile_load<D, HG, MMA>(sm.v[stage] + u * SUBH, tmv, it.h0, r, full_bar, pol);
                }
            } else if constexpr (!MMA) {
                // B < TB (B = 1): one box of B rows per page (one tile per stage)
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
            } else {
                // B < TB (B = 1) in the tensor-core layout: each token row
                // goes by cp.async to its swizzled place (a TMA box of one
                // row could not follow the swizzle).  Lanes 0-15 copy K and
                // 16-31 V of token lane % 16.
                const int tk = lane & 15;
                const int raw = __shfl_sync(FULL, cur, (pa - wbase + tk) & 31);   // page of token t + tk
                if (tk < nt) {
                    const int id = checked(raw);
                    const size_t row = (size_t)(p.layer_row0 + id * B + (t + tk) % B);
                    const __half *src = (lane < 16 ? p.k_pool : p.v_pool) + (row * p.n_kv_heads + it.h0) * D;
                    uint8_t *dst = reinterpret_cast<uint8_t *>((lane < 16 ? sm.k[stage] : sm.v[stage]) + u * SUBH);
#pragma unroll
                    for (int hl = 0; hl < HG; ++hl) {
                        if (it.h0 + hl < p.n_kv_heads) {
#pragma unroll
                            for (int c = 0; c < D / 8; ++c)
                                cp_async16_cg(smem_addr(dst + hl * (D / 64) * TB * 128 + swz(tk, c)), src + hl * D + c * 8);
                        }
                    }
                }
            }
        }
        // cp.async stages: every lane's copies complete on the stage's full
        // barrier (32 arrivals for these stages)
        if constexpr (MMA) {
            if (B < TB) cp_async_mbar_arrive_noinc(full_bar);
        }
        ++st;
        return true;
    };

    for (int k = 0; ok; ++k) {
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
            d.span = it.span;
            // Fused decode step: the item holding token L - 1 also brings
            // that token's K and V rows (with q, on the same barrier); the
            // consumers use them for row L - 1 and write them to the pool.
            const bool writes_new = p.k_new != nullptr && it.tok0 + it.ntok == it.L;
            d.newrow = writes_new ? it.L - 1 : -1;
            d.newslot = -1;
            if (writes_new) {
                if (it.last_id >= 0 && it.last_id < p.n_blocks)
                    d.newslot = p.layer_row0 + it.last_id * B + (it.L - 1) % B;
                else
                    atomicOr(p.status, PF_DEV_BAD_BLOCK_ID);   // attended to, not written
            }
            d.L = it.L;
            d.nq = it.nq;
            d.qrow0 = it.qrow0;
            d.pad0 = 0;
            sm.desc[slot] = d;
            // q: one bulk copy per query token, its nv heads x gh q-heads
            // (contiguous in q) to rows (i * HG + hl) * gh + g of the slot
            const int nv = min(HG, p.n_kv_heads - it.h0);           // heads that exist
            const uint32_t tokbytes = (uint32_t)nv * p.gh * D * 2;
            const uint32_t rowbytes = (uint32_t)nv * D * 2;
            const uint32_t qfull = smem_addr(&sm.qfull[slot]);
            mbar_arrive_expect_tx(qfull, (uint32_t)it.nq * tokbytes + (writes_new ? 2 * rowbytes : 0));
            if (writes_new) {
                const size_t src = ((size_t)it.s * p.n_kv_heads + it.h0) * D;
                bulk_load(smem_addr(sm.knew[slot][0]), p.k_new + src, rowbytes, qfull);
                bulk_load(smem_addr(sm.knew[slot][1]), p.v_new + src, rowbytes, qfull);
            }
        }
        __syncwarp();   // the expected bytes are set before any copy can complete
        if (lane < it.nq) {
            bulk_load(smem_addr(sm.q[slot] + (size_t)lane * HG * p.gh * D),
                      p.q + ((size_t)(it.qrow0 + lane) * p.n_q_heads + (size_t)it.h0 * p.gh) * D,
                      (uint32_t)min(HG, p.n_kv_heads - it.h0) * p.gh * D * 2, smem_addr(&sm.qfull[slot]));
        }
        ++posted;

        // The next item's numbering and block ids are requested now; their
        // latency overlaps with issuing this item's tiles.
        const ProdItem nx = decode(k + 1);
        const int ntiles = (it.ntok + TB - 1) / TB;
        for (int j = 0; j < ntiles && ok; j += SUB) ok = issue_stage(j);
        if (!ok) break;
        it = nx;
        wbase = 0;
        cur = it.ids0;
        nxt = it.ids1;
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

// Normalise and store the rows row0 .. row0 + R - 1 of a whole pair's head
// from the state a warp holds: lanes 0 .. D/8 - 1 hold dims
// [8 * lane, 8 * lane + 8) of acc.
template <int D, int G, int R>
__device__ __forceinline__ void store_whole(const Params &p, const ItemDesc &d, int h, int lane, int row0,
                                            const float (&l)[R], const float (&acc)[R][8]) {
    constexpr int LPT = D / 8;
    if (lane < LPT) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int g = row0 + r;
            const int i = g / p.gh;               // query token of row g
            if (g >= G || i >= d.nq) continue;
            float x[8];
            const float inv = 1.0f / l[r];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = acc[r][e] * inv;
            store8(p, ((size_t)(d.qrow0 + i) * p.n_q_heads + (size_t)h * p.gh + g - i * p.gh) * D + lane * 8, x);
        }
    }
}

// Rows row0 .. row0 + R - 1 of the record of one part of a cut pair for head
// hl (state as in store_whole, m and l the same in every lane).  Chunk
// schedule: fp32 words, and the first part also writes the pair's job.  Span
// schedule: words tagged with the launch's epoch, record ((span * 2 + slot)
// * HG + hl).
template <int D, int G, int HG, int R>
__device__ __forceinline__ void write_part(const Params &p, const Smem<D, G, HG> &sm, const ItemDesc &d, int hl,
                                           int lane, int row0, bool write_job, const float (&m)[R],
                                           const float (&l)[R], const float (&acc)[R][8]) {
    constexpr int LPT = D / 8;
    constexpr int REC = G * (D + 2);
    const int Hkv = p.n_kv_heads;
    if (d.kind == kSpanPart) {
        unsigned long long *part = p.span_recs + (((size_t)d.span * 2 + d.c) * HG + hl) * REC;
        if (lane < LPT) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int g = row0 + r;
                if (g >= G) continue;
                unsigned long long *w = part + g * (D + 2);
#pragma unroll
                for (int i = 0; i < 8; ++i) st_tagged(w + lane * 8 + i, acc[r][i], p.epoch);
                if (lane == 0) {
                    st_tagged(w + D, m[r], p.epoch);
                    st_tagged(w + D + 1, l[r], p.epoch);
                }
            }
        }
        return;
    }
    const size_t rec = (size_t)d.a * Hkv + d.h0 + hl;
    float *part = p.partials + rec * REC;
    if (lane < LPT) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int g = row0 + r;
            if (g >= G) continue;
            // rows of D + 2 floats keep 8-float runs 8-byte (not 16-byte) aligned
            float2 *d2 = reinterpret_cast<float2 *>(part + g * (D + 2) + lane * 8);
#pragma unroll
            for (int i = 0; i < 4; ++i) d2[i] = make_float2(acc[r][2 * i], acc[r][2 * i + 1]);
            if (lane == 0) {
                part[g * (D + 2) + D] = m[r];
                part[g * (D + 2) + D + 1] = l[r];
            }
        }
    }
    if (write_job && lane == 0) {   // chunk schedule: the pair's merge job
        Job jb;
        jb.s = d.s;
        jb.h0 = d.h0;
        jb.kind = d.kind;
        jb.pad = 0;
        jb.first = d.a;          // chunk 0 of the sequence
        jb.z_first = 0;
        jb.n_parts = d.c;
        jb.epoch = p.epoch;
        p.jobs[(size_t)d.a * p.n_groups + d.h0 / HG] = jb;
    }
}

// Merge the n_parts records of one cut pair for kv-head h with the
// log-sum-exp rule and write its G output rows (chunk schedule: records
// (first + i) * Hkv + h, complete when the merge kernel runs).  Each lane
// loads one part's (m, l) and, in the same round trip, every part's acc
// values of its own dims (D / 32 of them), PB parts at a time.
template <int D, int G, int HG>
__device__ __forceinline__ void merge_pair(const Params &p, int first, int n, int qrow0, int nq, int h, int lane) {
    constexpr int REC = G * (D + 2);
    constexpr int DPL = D / 32;   // dims per lane
    constexpr int PB = 8;         // parts whose acc loads are in flight together
    const int Hkv = p.n_kv_heads;
    const int Hq = p.n_q_heads;
    auto rec_of = [&](int i) -> size_t { return (size_t)(first + i) * Hkv + h; };
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        const int qi = g / p.gh;                  // query token of row g
        if (qi >= nq) break;
        float mx = -INFINITY, ls = 0.0f;
        float a[DPL];
#pragma unroll
        for (int q = 0; q < DPL; ++q) a[q] = 0.0f;
        for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            float mi = -INFINITY, li = 0.0f;
            if (i < n) {
                const float *pc = p.partials + rec_of(i) * REC + g * (D + 2);
                mi = __ldcg(pc + D);
                li = __ldcg(pc + D + 1);
            }
            const int nb = min(32, n - i0);
            for (int j0 = 0; j0 < nb; j0 += PB) {
                float v[PB][DPL];
#pragma unroll
                for (int jj = 0; jj < PB; ++jj) {
                    if (j0 + jj < nb) {
                        const float *pc = p.partials + rec_of(i0 + j0 + jj) * REC + g * (D + 2);
#pragma unroll
                        for (int q = 0; q < DPL; ++q) v[jj][q] = __ldcg(pc + lane + 32 * q);
                    }
                }
                // running reference over the batches of 32 parts
                float bm = mi;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, o));
                const float mn = fmaxf(mx, bm);
                if (mn > mx) {
                    const float sc = (mx == -INFINITY) ? 0.0f : exp2f(mx - mn);
                    ls *= sc;
#pragma unroll
                    for (int q = 0; q < DPL; ++q) a[q] *= sc;
                    mx = mn;
                }
                const float w = (i < n && j0 == 0) ? exp2f(mi - mx) : 0.0f;
                if (j0 == 0) ls = fmaf(w, li, ls);
#pragma unroll
                for (int jj = 0; jj < PB; ++jj) {
                    const float wj = __shfl_sync(FULL, exp2f(mi - mx), j0 + jj);
                    if (j0 + jj < nb) {
#pragma unroll
                        for (int q = 0; q < DPL; ++q) a[q] = fmaf(wj, v[jj][q], a[q]);
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(FULL, ls, o);
        const float inv = 1.0f / ls;
#pragma unroll
        for (int q = 0; q < DPL; ++q) {
            const size_t o = ((size_t)(qrow0 + qi) * Hq + (size_t)h * p.gh + g - qi * p.gh) * D + lane + 32 * q;
            if (p.out_f32) static_cast<float *>(p.out)[o] = a[q] * inv;
            else static_cast<__half *>(p.out)[o] = __float2half_rn(a[q] * inv);
        }
    }
}

// Consumer start: wait for the previous kernel on the stream (as in the
// producer: it may still be writing `out`), then give empty (or invalid,
// clamped to empty) sequences a zero output (decode: row s; append: its
// query rows, when it has any).
template <int D>
__device__ __forceinline__ void zero_empty_outputs(const Params &p, int cw, int lane) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int Hq = p.n_q_heads;
    for (int s = blockIdx.x; s < p.n_seqs; s += gridDim.x) {
        if (p.lens[s] <= 0) {
            const int r0 = p.cu_q != nullptr ? p.cu_q[s] : s;
            const int nr = p.cu_q != nullptr ? p.cu_q[s + 1] - r0 : 1;
            for (long long e = cw * 32 + lane; e < (long long)nr * Hq * D; e += NCW * 32) {
                const size_t o = (size_t)r0 * Hq * D + e;
                if (p.out_f32) static_cast<float *>(p.out)[o] = 0.0f;
                else static_cast<__half *>(p.out)[o] = __float2half_rn(0.0f);
            }
        }
    }
}

// Span schedule: merge the n parts of a cut pair for kv-head h (head hl of
// its group) and write its G output rows.  Part i is record ((first + i) * 2
// + slot) * HG + hl, slot z_first for i = 0 (the pair may start inside its
// first span, after that span's first segment) and 0 for the others.  Each
// lane loads one part's (m, l) and, in the same round trip, every part's acc
// values of its own dims (D / 32 of them), PB parts at a time; a batch is
// loaded again (after a short sleep) until every word carries this launch's
// epoch.  The parts are written by CTAs of earlier spans (and this warp),
// which wait for no one, so the words arrive; the wait is bounded all the
// same and gives up with PF_DEV_WAIT_TIMEOUT.
template <int D, int G, int HG>
__device__ __forceinline__ bool merge_span_pair(const Params &p, int first, int z_first, int n, int qrow0, int nq,
                                                int h, int hl, int lane) {
    constexpr int REC = G * (D + 2);
    constexpr int DPL = D / 32;   // dims per lane
    constexpr int PB = 8;         // parts whose acc loads are in flight together
    const int Hq = p.n_q_heads;
    auto rec_of = [&](int i) -> const unsigned long long * {
        return p.span_recs + (((size_t)(first + i) * 2 + (i == 0 ? z_first : 0)) * HG + hl) * REC;
    };
    unsigned long long t_wait = 0;   // when polling began (0: not yet)
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        const int qi = g / p.gh;                  // query token of row g
        if (qi >= nq) break;
        float mx = -INFINITY, ls = 0.0f;
        float a[DPL];
#pragma unroll
        for (int q = 0; q < DPL; ++q) a[q] = 0.0f;
        for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            const int nb = min(32, n - i0);
            float mi = -INFINITY, li = 0.0f;
            for (int j0 = 0; j0 < nb; j0 += PB) {
                float v[PB][DPL];
                for (;;) {
                    bool have = true;
                    if (j0 == 0 && i < n) {
                        const unsigned long long *pc = rec_of(i) + g * (D + 2);
                        const unsigned long long wm = ld_tagged(pc + D), wl = ld_tagged(pc + D + 1);
                        have = tagged_epoch(wm) == p.epoch && tagged_epoch(wl) == p.epoch;
                        mi = tagged_value(wm);
                        li = tagged_value(wl);
                    }
#pragma unroll
                    for (int jj = 0; jj < PB; ++jj) {
                        if (j0 + jj < nb) {
                            const unsigned long long *pc = rec_of(i0 + j0 + jj) + g * (D + 2);
#pragma unroll
                            for (int q = 0; q < DPL; ++q) {
                                const unsigned long long w = ld_tagged(pc + lane + 32 * q);
                                have = have && tagged_epoch(w) == p.epoch;
                                v[jj][q] = tagged_value(w);
                            }
                        }
                    }
                    if (__all_sync(FULL, have)) break;
                    const unsigned long long now = global_timer_ns();
                    if (t_wait == 0) {
                        t_wait = now;
                    } else if (now - t_wait > kWaitLimitNs) {
                        if (lane == 0) atomicOr(p.status, PF_DEV_WAIT_TIMEOUT);
                        return false;
                    }
                    __nanosleep(256);
                }
                // running reference over the batches of 32 parts
                float bm = mi;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, o));
                const float mn = fmaxf(mx, bm);
                if (mn > mx) {
                    const float sc = (mx == -INFINITY) ? 0.0f : exp2f(mx - mn);
                    ls *= sc;
#pragma unroll
                    for (int q = 0; q < DPL; ++q) a[q] *= sc;
                    mx = mn;
                }
                const float w = (i < n && j0 == 0) ? exp2f(mi - mx) : 0.0f;
                if (j0 == 0) ls = fmaf(w, li, ls);
#pragma unroll
                for (int jj = 0; jj < PB; ++jj) {
                    const float wj = __shfl_sync(FULL, exp2f(mi - mx), j0 + jj);
                    if (j0 + jj < nb) {
#pragma unroll
                        for (int q = 0; q < DPL; ++q) a[q] = fmaf(wj, v[jj][q], a[q]);
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(FULL, ls, o);
        const float inv = 1.0f / ls;
#pragma unroll
        for (int q = 0; q < DPL; ++q) {
            const size_t o = ((size_t)(qrow0 + qi) * Hq + (size_t)h * p.gh + g - qi * p.gh) * D + lane + 32 * q;
            if (p.out_f32) static_cast<float *>(p.out)[o] = a[q] * inv;
            else static_cast<__half *>(p.out)[o] = __float2half_rn(a[q] * inv);
        }
    }
    return true;
}

// Span schedule, when a consumer warp has no items left: its CTA merges the
// cut pair whose last part is its span's first segment (record slot 0, bit 0
// of `pending`).  A part in slot 1 (a pair that starts inside the span and
// runs past its end) is merged by a later span.
template <int D, int G, int HG>
__device__ __forceinline__ void merge_if_last(const Params &p, const PendPart &pp, int pending, int hl, int lane) {
    if (!(pending & 1) || pp.first + pp.n_parts - 1 != (int)blockIdx.x) return;
    __syncwarp();
    merge_span_pair<D, G, HG>(p, pp.first, pp.z_first, pp.n_parts, pp.qrow0, pp.nq, pp.h0 + hl, hl, lane);
}

// Span schedule: note a finished cut part (lane 0; written to the warp's
// pend slot d.c).  Units a .. a + b - 1 of the pair are the cost unit, then
// the tiles; its parts are spans owner(a) .. owner(a + b - 1), and the
// first uses slot 1 when the pair starts inside it.
__device__ __forceinline__ PendPart pending_part(const Params &p, const int *pre, const ItemDesc &d) {
    const SpanMap map((long long)pre[p.n_seqs] * p.n_groups, gridDim.x);
    const long long first = map.owner((long long)d.a + kPairCost);
    PendPart pp;
    pp.s = d.s;
    pp.h0 = d.h0;
    pp.first = (int)first;
    pp.z_first = (long long)d.a <= map.start(first) ? 0 : 1;   // the span's first segment?
    pp.n_parts = (int)(map.owner((long long)d.a + d.b - 1) - first + 1);
    pp.qrow0 = d.qrow0;
    pp.nq = d.nq;
    return pp;
}

template <int D, int G, int HG>
__device__ __forceinline__ void consumers(const Params &p, Smem<D, G, HG> &sm, int cw, int lane) {
    constexpr int NS = Shape<D, HG>::NS;
    constexpr int WPH = Shape<D, HG>::WPH;
    constexpr int LPT = D / 8;        // lanes per token row
    constexpr int TPW = 32 / LPT;     // tokens per warp-step
    // Several warps of a head split its rows when it has at least as many
    // rows as warps (each then holds fewer of them: registers, occupancy);
    // otherwise they split each tile's tokens and merge at the end.
    constexpr bool RSPLIT = WPH > 1 && G >= WPH;
    constexpr int R = RSPLIT ? (G + WPH - 1) / WPH : G;   // rows this warp holds
    constexpr int TPT = RSPLIT ? TB : TB / WPH;          // tokens of a tile this warp serves
    constexpr int STEPS = TPT / TPW;
    static_assert(STEPS * TPW == TPT, "tile must split into whole warp-steps");
    const int grp = lane / LPT;
    const int sub = lane % LPT;
    const int hl = cw / WPH;          // head within the group
    const int part = cw % WPH;        // which share of the head's rows, or of each tile's tokens
    const int row0 = RSPLIT ? part * R : 0;
    const int tok_base = RSPLIT ? 0 : part * TPT;

    zero_empty_outputs<D>(p, cw, lane);

    uint32_t st = 0;
    uint32_t cphase = 0;
    const uint32_t cbar = smem_addr(&sm.cbar);
    int pending = 0;   // span schedule: bit c = this warp wrote a cut part's record in slot c
    for (int k = 0;; ++k) {
        const int slot = k % NQ;
        if (!warp_wait(smem_addr(&sm.qfull[slot]), (k / NQ) & 1, p.status, lane)) return;
        const ItemDesc d = sm.desc[slot];
        if (d.s < 0) {
            if (part == 0) merge_if_last<D, G, HG>(p, sm.pend[cw][0], pending, hl, lane);
            return;
        }
        const int h = d.h0 + hl;
        const bool active = h < p.n_kv_heads;   // ragged last group: idle warps keep the protocol

        // This warp holds rows row0 .. row0 + R - 1 of the head.  Row g:
        // query token g / gh, q-head g % gh; it sees tokens 0 .. lim (L - 1
        // for decode; causal for an append).
        float qf[R][8];
        int lim[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int g = row0 + r;
            const int i = g / p.gh;
            const bool valid = active && g < G && i < d.nq;
            lim[r] = valid ? d.L - d.nq + i : -1;
            if (valid) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(
                    &sm.q[slot][((i * HG + hl) * p.gh + g - i * p.gh) * D + sub * 8]);
                half8_to_float(raw, qf[r]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[r][e] = valid ? qf[r][e] * p.scale_log2 : 0.0f;
        }
        // Fused decode step: the new token's rows stand in for the tile's row
        // L - 1 (whatever the tile read there), and the first warp of each
        // head writes them into the pool slot.  No other block reads that
        // slot in this launch, so the write needs no ordering here.
        uint4 nk = make_uint4(0u, 0u, 0u, 0u), nvv = nk;
        if (d.newrow >= 0 && active) {
            nk = *reinterpret_cast<const uint4 *>(&sm.knew[slot][0][hl * D + sub * 8]);
            nvv = *reinterpret_cast<const uint4 *>(&sm.knew[slot][1][hl * D + sub * 8]);
            if (part == 0 && grp == 0 && d.newslot >= 0) {
                const size_t dst = ((size_t)d.newslot * p.n_kv_heads + h) * D + sub * 8;
                *reinterpret_cast<uint4 *>(p.k_pool + dst) = nk;
                *reinterpret_cast<uint4 *>(p.v_pool + dst) = nvv;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.qempty[slot]));

        float m[R], l[R], acc[R][8];
#pragma unroll
        for (int g = 0; g < R; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[g][i] = 0.0f;
        }

        const int ntiles = (d.ntok + TB - 1) / TB;
        for (int j = 0; j < ntiles; ++j, ++st) {
            const int stage = st % NS;
            if (!warp_wait(smem_addr(&sm.full[stage]), (st / NS) & 1, p.status, lane)) return;
            if (active) {
                const __half *kt = sm.k[stage];
                const __half *vt = sm.v[stage];
                const int tile0 = d.tok0 + j * TB;
                // tiles that reach a row's limit or the sequence's end
                const bool masked = tile0 + TB > d.L - d.nq;
                const int newr = (d.newrow >= 0 && j == ntiles - 1) ? d.newrow - tile0 : -1;   // row of token L - 1
                // phase 1: this lane group's scores for all of the warp's steps
                // (independent chains: loads, dots and shuffles interleave)
                uint4 kraw[STEPS];
#pragma unroll
                for (int step = 0; step < STEPS; ++step) {
                    kraw[step] = *reinterpret_cast<const uint4 *>(
                        kt + ((tok_base + step * TPW + grp) * HG + hl) * D + sub * 8);
                    if (tok_base + step * TPW + grp == newr) kraw[step] = nk;
                }
                float z[STEPS][R];
#pragma unroll
                for (int step = 0; step < STEPS; ++step) {
                    float kf[8];
                    half8_to_float(kraw[step], kf);
#pragma unroll
                    for (int g = 0; g < R; ++g) {
                        float a = 0.0f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) a = fmaf(qf[g][i], kf[i], a);
                        z[step][g] = a;
                    }
                }
#pragma unroll
                for (int o = LPT / 2; o > 0; o >>= 1) {
#pragma unroll
                    for (int step = 0; step < STEPS; ++step) {
#pragma unroll
                        for (int g = 0; g < R; ++g) z[step][g] += __shfl_xor_sync(FULL, z[step][g], o);
                    }
                }
                if (masked) {
#pragma unroll
                    for (int step = 0; step < STEPS; ++step) {
                        const int tok = tile0 + tok_base + step * TPW + grp;
#pragma unroll
                        for (int g = 0; g < R; ++g)
                            if (tok > lim[g]) z[step][g] = -INFINITY;
                    }
                }
                // phase 2: the warp's maximum over the tile; the reference
                // maximum m (the same in every lane) is raised only when the
                // tile passes it by more than 2^8
#pragma unroll
                for (int g = 0; g < R; ++g) {
                    float mt = z[0][g];
#pragma unroll
                    for (int step = 1; step < STEPS; ++step) mt = fmaxf(mt, z[step][g]);
#pragma unroll
                    for (int o = LPT; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, o));
                    if (mt > m[g] + kRescaleLog2) {
                        const float sc = exp2f(m[g] - mt);   // m = -inf gives 0
                        l[g] *= sc;
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[g][i] *= sc;
                        m[g] = mt;
                    }
                }
                // phase 3: weights and the weighted sum of V
                uint4 vraw[STEPS];
#pragma unroll
                for (int step = 0; step < STEPS; ++step) {
                    vraw[step] = *reinterpret_cast<const uint4 *>(
                        vt + ((tok_base + step * TPW + grp) * HG + hl) * D + sub * 8);
                    if (tok_base + step * TPW + grp == newr) vraw[step] = nvv;
                }
#pragma unroll
                for (int step = 0; step < STEPS; ++step) {
                    float vf[8];
                    half8_to_float(vraw[step], vf);
                    if (masked && tile0 + tok_base + step * TPW + grp >= d.L) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) vf[i] = 0.0f;   // tail rows may hold anything
                    }
#pragma unroll
                    for (int g = 0; g < R; ++g) {
                        // a masked score has weight 0 (also when m is still -inf)
                        const float pz = (masked && z[step][g] == -INFINITY) ? 0.0f : exp2f(z[step][g] - m[g]);
                        l[g] += pz;
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(pz, vf[i], acc[g][i]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&sm.empty[stage]));
        }

        // Sum the token groups of this warp (they share the reference m).
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) {
#pragma unroll
            for (int g = 0; g < R; ++g) {
                l[g] += __shfl_xor_sync(FULL, l[g], o);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[g][i] += __shfl_xor_sync(FULL, acc[g][i], o);
            }
        }

        if constexpr (WPH > 1 && !RSPLIT) {
            // The WPH warps of a head meet in shared memory; the first of
            // them carries the merged state on.
            if (lane < LPT) {
#pragma unroll
                for (int g = 0; g < R; ++g) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) sm.red[cw][g][lane * 8 + i] = acc[g][i];
                    if (lane == 0) {
                        sm.red[cw][g][D] = m[g];
                        sm.red[cw][g][D + 1] = l[g];
                    }
                }
            }
            if (!warps_sync(cbar, cphase, p.status, lane)) return;
            if (part == 0) {
#pragma unroll
                for (int g = 0; g < R; ++g) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int w = 0; w < WPH; ++w) mx = fmaxf(mx, sm.red[cw + w][g][D]);
                    float ls = 0.0f;
                    float a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = 0.0f;
#pragma unroll
                    for (int w = 0; w < WPH; ++w) {
                        const float mw = sm.red[cw + w][g][D];
                        const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - mx);
                        ls = fmaf(sm.red[cw + w][g][D + 1], f, ls);
                        if (lane < LPT) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) a[i] = fmaf(sm.red[cw + w][g][lane * 8 + i], f, a[i]);
                        }
                    }
                    m[g] = mx;
                    l[g] = ls;
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[g][i] = a[i];
                }
            }
            if (!warps_sync(cbar, cphase, p.status, lane)) return;   // red[] is reused next item
        }
        const bool leader = (RSPLIT || part == 0) && active;
        if (d.kind == kWhole) {
            if (leader) store_whole<D, G, R>(p, d, h, lane, row0, l, acc);
        } else if (leader) {
            if (d.kind == kChunk) {
                // chunk 0 of the sequence also writes the merge job
                write_part<D, G, HG, R>(p, sm, d, hl, lane, row0, d.b == 0 && hl == 0 && part == 0, m, l, acc);
            } else {
                // Span part: write the record and note the pair; the CTA
                // of its last span merges it.
                write_part<D, G, HG, R>(p, sm, d, hl, lane, row0, false, m, l, acc);
                if (lane == 0) sm.pend[cw][d.c] = pending_part(p, sm.pre, d);
                pending |= 1 << d.c;
            }
        }
    }
}

// ------------------------------------------------------------ tensor-core consumers

// Two consecutive output values of one row.
__device__ __forceinline__ void store2(const Params &p, size_t o, float x0, float x1) {
    if (p.out_f32) *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + o) = make_float2(x0, x1);
    else *reinterpret_cast<__half2 *>(static_cast<__half *>(p.out) + o) = __floats2half2_rn(x0, x1);
}

// Consumers for kv-heads with many rows (q-heads, or query tokens x
// q-heads), HG kv-heads per item.  A head's rows (at most 16) form the M side
// of warp-level tensor-core products, fp16 in, fp32 accumulate: scores
// S = Q K^T over a 16-token tile (m16n8k16, two 8-token column blocks), then
// O += P V (m16n8k16 per 8 dims).  The online softmax runs on the score
// fragments: lane (g, t) = (lane / 4, lane % 4) holds rows g and g + 8,
// tokens 2t, 2t + 1 of each column block, and the same rows of O at dims
// 8b + 2t, 8b + 2t + 1.  fp16 output: P is the tile's weights rounded to
// fp16 and the row sums l are the sums of those rounded weights, so the
// normalised output is an exact weighted mean of V under them.  fp32 output:
// P V is taken twice, with the weights' fp16 part and with its rounding
// error (also fp16), and l sums the fp32 weights, so the weights keep about
// 22 bits (the fp32-output path carries no fp16 rounding of the weights).
//
// Each head has WPH = NCW / HG consumer warps; its tiles are dealt
// round-robin (warp part p computes tiles j = p mod WPH, whole).  With
// several warps per head their states meet in shared memory at the end and
// the head's first warp carries the merged state on.
template <int D, int G, int HG, bool HILO>
__device__ __forceinline__ void consumers_mma(const Params &p, Smem<D, G, HG, true> &sm, int cw, int lane) {
    constexpr int NS = Smem<D, G, HG, true>::NS;
    constexpr int SUB = Smem<D, G, HG, true>::SUB;   // tiles per stage
    constexpr int SUBH = Shape<D, HG>::STAGE_HALVES;   // halves of one tile's K (or V)
    constexpr int WPH = NCW / HG;   // consumer warps per head
    constexpr int NKS = D / 16;     // k-steps of the score product
    constexpr int NNB = D / 8;      // 8-dim column blocks of O
    constexpr int CH = D / 8;       // 16-byte chunks of a row
    static_assert(G <= 16, "the rows of a kv-head fill at most one m16 fragment");
    static_assert(WPH * HG == NCW, "heads per item divide the consumer warps");
    const int gq = lane >> 2;
    const int tq = lane & 3;
    const int hl = cw / WPH;        // head within the item
    const int part = cw % WPH;      // which of the head's tiles this warp computes
    const uint32_t hoff = (uint32_t)hl * (D / 64) * TB * 128;   // the head's bytes in a stage
    const int Hq = p.n_q_heads;
    constexpr bool hilo = HILO;   // fp32 output: weights as fp16 hi + lo parts

    zero_empty_outputs<D>(p, cw, lane);

    uint32_t st = 0;
    uint32_t cphase = 0;
    const uint32_t cbar = smem_addr(&sm.cbar);
    int pending = 0;   // span schedule: bit c = this warp wrote a cut part's record in slot c
    for (int k = 0;; ++k) {
        const int slot = k % NQ;
        if (!warp_wait(smem_addr(&sm.qfull[slot]), (k / NQ) & 1, p.status, lane)) return;
        const ItemDesc d = sm.desc[slot];
        if (d.s < 0) {
            merge_if_last<D, G, HG>(p, sm.pend[cw][0], pending, hl, lane);
            return;
        }
        const int h = d.h0 + hl;
        const bool active = h < p.n_kv_heads;   // ragged last group: idle warps keep the protocol

        // Fragment rows gq and gq + 8.  Row g: query token g / gh, q-head
        // g % gh, sees tokens 0 .. lim; a row past the item's rows repeats
        // row 0 (its results are dropped).
        int lim[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int g = gq + 8 * r;
            const int i = g / p.gh;
            lim[r] = d.L - d.nq + ((g < G && i < d.nq) ? i : 0);
        }
        // q as A fragments, one ldmatrix.x4 per k-step: lanes 0-7 / 8-15 /
        // 16-23 / 24-31 give rows 0-7 / 8-15 / 0-7 / 8-15 at dims +0 / +0 /
        // +8 / +8.  Row g of head hl is at ((i * HG + hl) * gh + g % gh) * D.
        uint32_t qa[NKS][4];
        {
            const int g = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int gg = (g < G && g / p.gh < d.nq) ? g : 0;
            const int i = gg / p.gh;
            const uint32_t qrow = smem_addr(&sm.q[slot][((i * HG + hl) * p.gh + gg - i * p.gh) * D]) +
                                  (uint32_t)(lane >> 4) * 16u;
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) ldmatrix_x4(qa[ks], qrow + ks * 32);
        }
        // Fused decode step: lanes 0 .. 2 CH - 1 keep one 16-byte chunk of
        // the new token's K (lanes < CH) or V row of the head; the head's
        // first warp writes the rows to the pool slot, and the warp that
        // computes the item's last tile puts them in place of its row L - 1.
        uint4 nrow = make_uint4(0u, 0u, 0u, 0u);
        if (d.newrow >= 0 && active && lane < 2 * CH) {
            nrow = *reinterpret_cast<const uint4 *>(&sm.knew[slot][lane / CH][hl * D + (lane % CH) * 8]);
            if (part == 0 && d.newslot >= 0) {
                const size_t dst = ((size_t)d.newslot * p.n_kv_heads + h) * D + (lane % CH) * 8;
                *reinterpret_cast<uint4 *>((lane < CH ? p.k_pool : p.v_pool) + dst) = nrow;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.qempty[slot]));

        float m[2] = {-INFINITY, -INFINITY};
        float l[2] = {0.0f, 0.0f};
        float o[NNB][4];
#pragma unroll
        for (int b = 0; b < NNB; ++b) o[b][0] = o[b][1] = o[b][2] = o[b][3] = 0.0f;

        const int ntiles = (d.ntok + TB - 1) / TB;
        for (int j0 = 0; j0 < ntiles; j0 += SUB, ++st) {
            const int stage = st % NS;
            if (!warp_wait(smem_addr(&sm.full[stage]), (st / NS) & 1, p.status, lane)) return;
            const int nsub = min(SUB, ntiles - j0);
            for (int u = 0; u < nsub; ++u) {
            const int j = j0 + u;   // tile of the item; the stage holds tile j at u * SUBH halves
            if (active && (j % WPH) == part) {
                uint8_t *kt = reinterpret_cast<uint8_t *>(sm.k[stage] + u * SUBH) + hoff;
                uint8_t *vt = reinterpret_cast<uint8_t *>(sm.v[stage] + u * SUBH) + hoff;
                const uint32_t kb = smem_addr(kt);
                const uint32_t vb = smem_addr(vt);
                const int tile0 = d.tok0 + j * TB;
                // tiles that reach a row's limit or the sequence's end
                const bool masked = tile0 + TB > d.L - d.nq;
                const int newr = (d.newrow >= 0 && j == ntiles - 1) ? d.newrow - tile0 : -1;
                if (newr >= 0 || masked) {
                    // patch the head's part of the stage: the new token's
                    // rows, and zeros over V rows past the sequence's end
                    // (they may hold anything; a zero weight times a
                    // non-finite value would not vanish)
                    if (newr >= 0 && lane < 2 * CH)
                        *reinterpret_cast<uint4 *>((lane < CH ? kt : vt) + swz(newr, lane % CH)) = nrow;
                    if (masked) {
                        const int nvalid = d.L - tile0;
                        for (int e = lane; e < TB * CH; e += 32) {
                            const int t = e / CH;
                            if (t >= nvalid) *reinterpret_cast<uint4 *>(vt + swz(t, e % CH)) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    // the stage is refilled by TMA (async proxy) later
                    fence_proxy_async_shared();
                    __syncwarp();
                }
                // S = Q K^T: K rows are the B fragments' columns (tokens);
                // one ldmatrix.x4 gives two k-steps of one column block
                float sc[2][4];
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
                    sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.0f;
#pragma unroll
                    for (int kp = 0; kp < NKS / 2; ++kp) {
                        uint32_t b[4];
                        ldmatrix_x4(b, kb + swz(nb * 8 + (lane & 7), kp * 4 + (lane >> 3)));
                        mma_f16_16816(sc[nb], qa[2 * kp], b[0], b[1]);
                        mma_f16_16816(sc[nb], qa[2 * kp + 1], b[2], b[3]);
                    }
                }
                // scaled scores (log2 domain) with the limits applied
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        sc[nb][e] *= p.scale_log2;
                        if (masked && tile0 + nb * 8 + 2 * tq + (e & 1) > lim[e >> 1]) sc[nb][e] = -INFINITY;
                    }
                }
                // the rows' maxima over the tile (the 4 lanes of a row
                // group); the reference m is raised only when the tile passes
                // it by more than 2^8
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float mt = fmaxf(fmaxf(sc[0][2 * r], sc[0][2 * r + 1]), fmaxf(sc[1][2 * r], sc[1][2 * r + 1]));
                    mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
                    mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
                    if (mt > m[r] + kRescaleLog2) {
                        const float f = exp2f(m[r] - mt);   // m = -inf gives 0
                        l[r] *= f;
#pragma unroll
                        for (int b = 0; b < NNB; ++b) {
                            o[b][2 * r] *= f;
                            o[b][2 * r + 1] *= f;
                        }
                        m[r] = mt;
                    }
                }
                // weights as the A fragment of P V: register 2 nb + r holds
                // row g + 8 r, tokens 8 nb + 2t, 8 nb + 2t + 1.  fp16 output:
                // the weights rounded to fp16, l their sum.  fp32 output: P
                // = P_hi + P_lo, both fp16 (P_lo the rounding error of P_hi),
                // and P V as two products, so the weights carry about 22
                // bits; l sums the fp32 weights.
                uint32_t pa[4], pl[4];
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float z0 = sc[nb][2 * r], z1 = sc[nb][2 * r + 1];
                        const float p0 = z0 == -INFINITY ? 0.0f : exp2f(z0 - m[r]);
                        const float p1 = z1 == -INFINITY ? 0.0f : exp2f(z1 - m[r]);
                        const __half2 w = __floats2half2_rn(p0, p1);
                        const float2 wf = __half22float2(w);
                        pa[2 * nb + r] = *reinterpret_cast<const uint32_t *>(&w);
                        if (hilo) {
                            const __half2 wl = __floats2half2_rn(p0 - wf.x, p1 - wf.y);
                            pl[2 * nb + r] = *reinterpret_cast<const uint32_t *>(&wl);
                            l[r] += p0 + p1;
                        } else {
                            l[r] += wf.x + wf.y;
                        }
                    }
                }
                // O += P V: V rows (tokens) are the B fragments' k; one
                // ldmatrix.x4.trans gives two 8-dim column blocks
#pragma unroll
                for (int np = 0; np < NNB / 2; ++np) {
                    uint32_t b[4];
                    ldmatrix_x4_trans(b, vb + swz((lane & 7) + ((lane >> 3) & 1) * 8, np * 2 + (lane >> 4)));
                    mma_f16_16816(o[2 * np], pa, b[0], b[1]);
                    mma_f16_16816(o[2 * np + 1], pa, b[2], b[3]);
                    if (hilo) {
                        mma_f16_16816(o[2 * np], pl, b[0], b[1]);
                        mma_f16_16816(o[2 * np + 1], pl, b[2], b[3]);
                    }
                }
            }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&sm.empty[stage]));
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l[r] += __shfl_xor_sync(FULL, l[r], 1);
            l[r] += __shfl_xor_sync(FULL, l[r], 2);
        }

        if (WPH > 1 && ntiles > 1) {
            // The head's warps' states meet in shared memory (rows < G): its
            // other warps leave theirs there, and its first warp merges them
            // into its own with the log-sum-exp rule.
            const int w1 = hl * (WPH - 1);   // the head's merge slots
            if (part != 0) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int g = gq + 8 * r;
                    if (g < G) {
                        float *rw = sm.red[w1 + part - 1][g];
#pragma unroll
                        for (int b = 0; b < NNB; ++b)
                            *reinterpret_cast<float2 *>(rw + b * 8 + 2 * tq) = make_float2(o[b][2 * r], o[b][2 * r + 1]);
                        if (tq == 0) {
                            rw[D] = m[r];
                            rw[D + 1] = l[r];
                        }
                    }
                }
            }
            if (!warps_sync(cbar, cphase, p.status, lane)) return;
            if (part == 0) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int g = gq + 8 * r;
                    if (g >= G) continue;
                    float mx = m[r];
#pragma unroll
                    for (int w = 1; w < WPH; ++w) mx = fmaxf(mx, sm.red[w1 + w - 1][g][D]);
                    const float f0 = m[r] == -INFINITY ? 0.0f : exp2f(m[r] - mx);
                    float ls = l[r] * f0;
                    float a[NNB][2];
#pragma unroll
                    for (int b = 0; b < NNB; ++b) {
                        a[b][0] = o[b][2 * r] * f0;
                        a[b][1] = o[b][2 * r + 1] * f0;
                    }
#pragma unroll
                    for (int w = 1; w < WPH; ++w) {
                        const float mw = sm.red[w1 + w - 1][g][D];
                        const float f = mw == -INFINITY ? 0.0f : exp2f(mw - mx);
                        ls = fmaf(sm.red[w1 + w - 1][g][D + 1], f, ls);
#pragma unroll
                        for (int b = 0; b < NNB; ++b) {
                            const float2 v = *reinterpret_cast<const float2 *>(&sm.red[w1 + w - 1][g][b * 8 + 2 * tq]);
                            a[b][0] = fmaf(v.x, f, a[b][0]);
                            a[b][1] = fmaf(v.y, f, a[b][1]);
                        }
                    }
                    m[r] = mx;
                    l[r] = ls;
#pragma unroll
                    for (int b = 0; b < NNB; ++b) {
                        o[b][2 * r] = a[b][0];
                        o[b][2 * r + 1] = a[b][1];
                    }
                }
            }
            if (!warps_sync(cbar, cphase, p.status, lane)) return;   // red[] is reused next item
        }
        if (part != 0 || !active) continue;
        if (d.kind == kWhole) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int g = gq + 8 * r;
                const int i = g / p.gh;
                if (g >= G || i >= d.nq) continue;
                const float inv = 1.0f / l[r];
                const size_t ob = ((size_t)(d.qrow0 + i) * Hq + (size_t)h * p.gh + g - i * p.gh) * D + 2 * tq;
#pragma unroll
                for (int b = 0; b < NNB; ++b) store2(p, ob + b * 8, o[b][2 * r] * inv, o[b][2 * r + 1] * inv);
            }
        } else {
            // Span part: write the record ((span * 2 + slot) * HG + head),
            // every word tagged with the launch's epoch, and note the pair;
            // the CTA of its last span merges it.
            unsigned long long *part_rec =
                p.span_recs + (((size_t)d.span * 2 + d.c) * HG + hl) * (size_t)(G * (D + 2));
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int g = gq + 8 * r;
                if (g >= G) continue;
                unsigned long long *rw = part_rec + g * (D + 2);
#pragma unroll
                for (int b = 0; b < NNB; ++b) {
                    st_tagged(rw + b * 8 + 2 * tq, o[b][2 * r], p.epoch);
                    st_tagged(rw + b * 8 + 2 * tq + 1, o[b][2 * r + 1], p.epoch);
                }
                if (tq == 0) {
                    st_tagged(rw + D, m[r], p.epoch);
                    st_tagged(rw + D + 1, l[r], p.epoch);
                }
            }
            if (lane == 0) sm.pend[cw][d.c] = pending_part(p, sm.pre, d);
            pending |= 1 << d.c;
        }
    }
}

template <int D, int G, int HG, bool MMA = false, bool HILO = false>
__device__ __forceinline__ void decode_attention(const CUtensorMap &tmk, const CUtensorMap &tmv, const Params &p) {
    using SM = Smem<D, G, HG, MMA>;
    constexpr int NS = SM::NS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw;
    // MMA: the swizzled stages need a 1024-byte aligned struct (the launch
    // adds 1 KB of slack for this)
    if constexpr (MMA) base += (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    SM &sm = *reinterpret_cast<SM *>(base);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // The merge grid that follows may start launching now; it waits for
    // this grid's completion before it reads anything.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Start-up is a chain of dependent memory round trips (lengths, then
    // block ids, then the first tile).  Fetch the descriptors and the leading
    // part of every block-table row now, so the block-id loads that follow
    // the length scan find their lines in L2.
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    prefetch_table_rows(p);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            // tensor-core layout on pages of fewer than TB tokens: the
            // producer's 32 lanes arrive (cp.async); otherwise one arrival
            // with the TMA byte count
            mbar_init(smem_addr(&sm.full[i]), (MMA && p.block_size < TB) ? 32 : 1);
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
            L = append_length(p, s, L);
            sm.rem[s] = (uint8_t)(L - (L - 1) / TB * TB);   // unused when L = 0
            sm.pre[s + 1] = L > 0 ? (L + TB - 1) / TB + kPairCost : 0;
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
        long long units = 0;   // per group, all sequences
#pragma unroll
        for (int w = 0; w < NTHREADS / 32; ++w) {
            if (w < warp) run += sm.warp_tot[w];
            units += sm.warp_tot[w];
        }
        // Each thread finds whether its sequences hold this CTA's first unit
        // (x0), so the producer starts without a search.
        const long long ng = p.n_groups;
        const long long x0 = SpanMap(units * ng, gridDim.x).start(blockIdx.x);
        for (int i = lo; i < hi; ++i) {
            const int before = run;
            run += sm.pre[i];
            sm.pre[i] = run;
            if (before * ng <= x0 && x0 < run * ng) sm.s_first = i - 1;   // sequence i - 1: units [before, run)
        }
        if (threadIdx.x == 0) sm.pre[0] = 0;
    }
    __syncthreads();
    if (warp == 0) producer<D, G, HG, MMA>(&tmk, &tmv, p, sm, lane);
    else if constexpr (MMA) consumers_mma<D, G, HG, HILO>(p, sm, warp - 1, lane);
    else consumers<D, G, HG>(p, sm, warp - 1, lane);
}

// Resident CTAs per SM are set by shared memory (3 at head_dim 64 with the
// 64 KB ring, 2 at 128) and by registers.  The register file is split over
// the SM's four sub-partitions, so 3 CTAs of 5 warps (4 warps on one
// sub-partition) need at most 128 registers a thread.  The instances whose
// state fits that without spilling are compiled under that cap; the others
// get all the registers they ask for.
template <int D, int G, int HG>
struct RegisterCap {
    static constexpr int WPH = Shape<D, HG>::WPH;
    static constexpr int ROWS = (WPH > 1 && G >= WPH) ? (G + WPH - 1) / WPH : G;   // rows per consumer warp
    static constexpr bool k128 = D == 64 && (ROWS <= 2 || (HG <= 2 && G <= 3));
};

template <int D, int G, int HG>
__global__ void __launch_bounds__(NTHREADS, 1) paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                 const __grid_constant__ CUtensorMap tmv,
                                                                 const Params p) {
    decode_attention<D, G, HG>(tmk, tmv, p);
}

template <int D, int G, int HG>
__global__ void __maxnreg__(128) paged_decode_kernel_r128(const __grid_constant__ CUtensorMap tmk,
                                                          const __grid_constant__ CUtensorMap tmv, const Params p) {
    decode_attention<D, G, HG>(tmk, tmv, p);
}

// Tensor-core consumers, HG kv-heads per item (span schedule, block size
// >= TB).  At head_dim 64 the state fits 128 registers (3 CTAs per SM); at
// 128, 2 CTAs put up to 3 warps on a sub-partition: 168 registers.
// HILO: the fp32-output instance (weights as fp16 hi + lo parts), a kernel
// of its own so that the fp16 path's tile loop carries none of it.
template <int D, int G, int HG, bool HILO>
__global__ void __maxnreg__(168) paged_decode_kernel_mma(const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv, const Params p) {
    decode_attention<D, G, HG, true, HILO>(tmk, tmv, p);
}

template <int D, int G, int HG, bool HILO>
__global__ void __maxnreg__(128) paged_decode_kernel_mma_r128(const __grid_constant__ CUtensorMap tmk,
                                                              const __grid_constant__ CUtensorMap tmv,
                                                              const Params p) {
    decode_attention<D, G, HG, true, HILO>(tmk, tmv, p);
}

// Chunk schedule: merge the records of every job of this launch's epoch, one
// warp per (job slot, head).  A head costs about two dependent memory round
// trips (the job, then its records).
template <int D, int G, int HG>
__global__ void __launch_bounds__(128, 1) merge_kernel(const Params p, int n_jobs) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the main grid has finished
    const int lane = threadIdx.x % 32;
    const long long n_warps = (long long)gridDim.x * blockDim.x / 32;
    for (long long wi = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32; wi < (long long)n_jobs * HG;
         wi += n_warps) {
        const int j = (int)(wi / HG);
        const int hl = (int)(wi - (long long)j * HG);
        const Job jb = p.jobs[j];
        if (jb.epoch != p.epoch || jb.h0 + hl >= p.n_kv_heads) continue;
        int qrow0 = jb.s, nq = 1;
        if (p.cu_q != nullptr) {
            qrow0 = p.cu_q[jb.s];
            nq = max(1, min(p.cu_q[jb.s + 1] - qrow0, p.rows / p.gh));
        }
        merge_pair<D, G, HG>(p, jb.first, jb.n_parts, qrow0, nq, jb.h0 + hl, lane);
    }
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);
using MergeFn = void (*)(Params, int);

struct KernelInfo {
    KernelFn fn;
    size_t smem;
    MergeFn merge;
    int rows;      // rows per kv-head of the instance (its G): the size of a record's rows
    KernelFn fn32; // the instance for fp32 output (the same as fn except on the tensor-core path)
};

// Defined in attention_d64.cu / attention_d128.cu / attention_mma.cu (the
// tensor-core instances: span schedule only, no merge kernel; smem includes
// 1 KB of alignment slack).
KernelInfo kernel_d64(int g, int hg);
KernelInfo kernel_d128(int g, int hg);
// Tensor-core instances: rows per kv-head rounded up to 1, 4, 8 (the "_s"
// files) or 12, 16; hg 1, 2 or 4 (not 4 at head_dim 128 above 8 rows).
KernelInfo kernel_mma_d64_s(int g, int hg);
KernelInfo kernel_mma_d64_l(int g, int hg);
KernelInfo kernel_mma_d128_s(int g, int hg);
KernelInfo kernel_mma_d128_l(int g, int hg);

template <int D, int G, int HG>
KernelInfo mma_info() {
    constexpr size_t smem = sizeof(Smem<D, G, HG, true>) + 1024;
    // with the 1 KB each CTA reserves: 3 CTAs per SM (228 KB) at head_dim 64, 2 at 128
    static_assert(smem + 1024 <= (D == 64 ? 228 * 1024 / 3 : 228 * 1024 / 2), "shared memory per CTA");
    if constexpr (D == 64)
        return {paged_decode_kernel_mma_r128<D, G, HG, false>, smem, nullptr, G, paged_decode_kernel_mma_r128<D, G, HG, true>};
    else return {paged_decode_kernel_mma<D, G, HG, false>, smem, nullptr, G, paged_decode_kernel_mma<D, G, HG, true>};
}

template <int D, int G>
KernelInfo mma_by_heads(int hg) {
    switch (hg) {
        case 1: return mma_info<D, G, 1>();
        case 2: return mma_info<D, G, 2>();
        case 4:
            if constexpr (D == 64 || G <= 8) return mma_info<D, G, 4>();
            else return {nullptr, 0, nullptr, 0, nullptr};
        default: return {nullptr, 0, nullptr, 0, nullptr};
    }
}

}  // namespace attn
}  // namespace pkv
