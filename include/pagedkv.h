/*
 * pagedkv.h -- C ABI of libpagedkv.so: the paged KV-cache decode hot path on
 * one GB300 (sm_103a).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every call returns an int status: PF_OK (0) or one of PF_ERR_*.  On
 *   failure pf_last_error() gives a message (per calling thread) and nothing
 *   was launched or changed.
 * - Device pointers are owned by the caller (e.g. PyTorch tensors); the
 *   library makes no device allocation and frees none.  Its only device
 *   memory is static, per device, for the life of the process: a status
 *   word (pf_device_status) and the fixed 8 MiB scratch of
 *   pf_paged_decode_attention_noalloc.  Host handles (pf_pool, pf_alloc)
 *   are allocated by *_create and released by *_destroy.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Device calls are asynchronous on that stream; the caller keeps
 *   the buffers alive until the work completes.
 * - Host-visible arguments (null pointers, sizes, 16-byte alignment of
 *   device buffers, head_dim in {64, 128}, block_size in {1, 16, 64, 256},
 *   layer in range) are checked before any launch and rejected with
 *   PF_ERR_INVALID.  Device-resident data (block ids, context lengths,
 *   positions) cannot be checked on the host: kernels that find a value out
 *   of range skip that access and record a flag readable with
 *   pf_device_status(); results for the affected rows are then undefined.
 * - fp16 is IEEE binary16 (PF_F16); fp32 (PF_F32) is only an output option.
 *
 * Pool layout
 * -----------
 * K and V are separate pools, each [n_layers][n_blocks][block_size]
 * [n_kv_heads][head_dim] fp16, row-major ("Why Naive KV-Caches Waste >60%
 * VRAM", "Implementation Walkthrough": the cache is sized to the physical
 * pool [N_blocks, block_size, N_heads, D_head]; PageForge, "Five techniques",
 * 04: all layers stacked in one pool tensor share the block ids).  Token t of
 * a sequence whose block-table row is `row` lives at slot
 *     row[t / block_size] * block_size + t % block_size
 * ("Why Naive KV-Caches Waste >60% VRAM", section 1 "Physical Block Pool &
 * Block Tables"; PageFault README, "The OS analogy").
 *
 * Block tables are int32 [n_seqs][max_blocks_per_seq], row-major; entries
 * past a sequence's ceil(L / block_size) used blocks are never read.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PF_API __attribute__((visibility("default")))
#else
#define PF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum pf_status {
    PF_OK = 0,
    PF_ERR_INVALID = 1,     /* bad argument; nothing launched */
    PF_ERR_OOM = 2,         /* allocator has fewer free blocks than asked */
    PF_ERR_DOUBLE_FREE = 3, /* freeing a block that is not allocated */
    PF_ERR_CUDA = 4,        /* a CUDA runtime call failed (message says which) */
    PF_ERR_UNSUPPORTED = 5  /* valid but not built (e.g. no sm_103a device) */
};

enum pf_dtype { PF_F16 = 1, PF_F32 = 2 };

/* Flags in the device status word (pf_device_status). */
enum pf_device_flag {
    PF_DEV_BAD_BLOCK_ID = 1,  /* a block id outside [0, n_blocks) was met */
    PF_DEV_BAD_LENGTH = 2,    /* a context length < 0 or > max_blocks * B */
    PF_DEV_BAD_POSITION = 4,  /* a write position < 0 or past the table row */
    PF_DEV_WAIT_TIMEOUT = 8   /* a bounded on-chip wait gave up (kernel bug) */
};

typedef struct pf_pool pf_pool;
typedef struct pf_alloc pf_alloc;

/* Message of the last failing call on this thread ("" if none). */
PF_API const char *pf_last_error(void);

/* ABI version of this header (PF_ABI_VERSION). */
#define PF_ABI_VERSION 3
PF_API int pf_abi_version(void);

/* ------------------------------------------------------------- pool ---- */

/* Bytes of ONE of the two pools (K or V) for these dimensions; 0 if a
 * dimension is not positive or dtype is not PF_F16.  An implementation
 * call with no counterpart on the pages: the size of the pool layout below,
 * for the caller who allocates it. */
PF_API size_t pf_pool_bytes(int n_layers, int n_blocks, int block_size,
                     int n_kv_heads, int head_dim, int dtype);

/* Describe caller-owned K and V pools (each pf_pool_bytes() bytes of device
 * memory, 16-byte aligned) as a pool.  Non-owning: destroying the handle
 * does not free the memory.  The handle caches TMA descriptors for the
 * current device.  dtype must be PF_F16; head_dim 64 or 128; block_size 1,
 * 16, 64 or 256.  Source: PageForge "Four layers, one pointer" (one pool
 * tensor of shape (N_pages, page_size, n_layers x n_heads, d_head)). */
PF_API int pf_pool_create(pf_pool **out, void *k_base, void *v_base, int n_layers,
                   int n_blocks, int block_size, int n_kv_heads, int head_dim,
                   int dtype);
PF_API int pf_pool_destroy(pf_pool *pool);

/* -------------------------------------------------- host allocator ---- */
/* O(1) free-list allocator over block ids [0, n_blocks).  A LIFO stack
 * ("Why Naive KV-Caches Waste >60% VRAM", "Implementation Walkthrough":
 * stack initialised so block 0 comes out first; pop to allocate, append to
 * free).  shuffle_seed != 0 permutes the initial hand-out order with a
 * Fisher-Yates shuffle driven by SplitMix64 (what a pool looks like after
 * churn, PageFault README "Four stages"); 0 keeps 0, 1, 2, ...
 * Host memory only; not thread-safe (one owner thread). */
PF_API int pf_alloc_create(pf_alloc **out, int n_blocks, uint64_t shuffle_seed);
PF_API int pf_alloc_destroy(pf_alloc *a);
/* Pop n block ids into ids_out[0..n).  All-or-nothing: PF_ERR_OOM and no
 * change if fewer than n are free (PageFault README "Test"). */
PF_API int pf_alloc_blocks(pf_alloc *a, int n, int32_t *ids_out);
/* Drop one reference per listed id; a block whose last reference goes is
 * pushed back, in list order (ids[0] first, so the last one pushed is handed
 * out next).  Every id is checked first: one that is out of range, free, or
 * listed more often than it is referenced gives PF_ERR_DOUBLE_FREE and no
 * change.  An unshared block has one reference, so this is a plain free. */
PF_API int pf_free_blocks(pf_alloc *a, const int32_t *ids, int n);
/* Shared blocks (PagedAttention blog, "Copy-on-Write for Parallel
 * Sampling": sequences that share a prefix point at the same physical
 * blocks, and a reference count tracks the sharing).  Add one reference to
 * each listed block; all-or-nothing, PF_ERR_INVALID if one is free or out of
 * range. */
PF_API int pf_alloc_share(pf_alloc *a, const int32_t *ids, int n);
/* References of block id (0 = free), or -1 for a null handle or bad id. */
PF_API int pf_alloc_refcount(const pf_alloc *a, int32_t id);
/* Copy-on-write, before a write into the block *entry (one host table
 * entry): if that block has other references, pop a fresh block, move one
 * reference to it, store it in *entry and return *src_out = old block,
 * *dst_out = new block -- the caller copies the contents with
 * pf_copy_blocks before writing (same section: allocate a new block, copy,
 * update only that sequence's table).  A block with one reference is the
 * writer's own: *src_out = *entry, *dst_out = -1, nothing changes.
 * PF_ERR_OOM (no change) if no block is free; PF_ERR_INVALID if *entry is
 * free or out of range. */
PF_API int pf_alloc_cow(pf_alloc *a, int32_t *entry, int32_t *src_out, int32_t *dst_out);
/* Fork a sequence (same section: parent and child share pages until one
 * writes): child_row[0..ceil(len/B)) = parent_row's entries, each with one
 * more reference.  Host int32 rows; PF_ERR_INVALID if the child row
 * (max_blocks entries) is too short. */
PF_API int pf_seq_fork(pf_alloc *a, int block_size, const int32_t *parent_row,
                       int len, int32_t *child_row, int max_blocks);
/* Number of free blocks, or -1 for a null handle. */
PF_API int pf_alloc_free_count(const pf_alloc *a);
/* Demand paging (PagedAttention blog, "Architecture"): grow one sequence
 * from cur_len to new_len tokens, appending ceil(new_len/B) - ceil(cur_len/B)
 * fresh blocks to table_row (host int32, max_blocks entries).  Tokens go into
 * the last block while it has room.  All-or-nothing (PF_ERR_OOM, row and
 * allocator unchanged); PF_ERR_INVALID if the row is too short or
 * new_len < cur_len. */
PF_API int pf_seq_reserve(pf_alloc *a, int block_size, int32_t *table_row,
                   int max_blocks, int cur_len, int new_len);
/* Free the ceil(len/B) blocks of a finished sequence (PageForge: pages are
 * returned the moment a sequence finishes). */
PF_API int pf_seq_release(pf_alloc *a, int block_size, const int32_t *table_row,
                   int len);

/* ---------------------------------------------------- device calls ---- */

/* Scatter (PageForge, "Four layers, one pointer": scatter_kv_layer writes
 * new tokens back into their pages).  Token i of the batch belongs to
 * sequence seq_idx[i] (a row of block_tables, which has n_table_rows rows of
 * max_blocks_per_seq entries) at logical position pos[i]; its rows
 * k_new[i][0..Hkv)[0..D) and v_new[i][..] (fp16, [n_tokens][Hkv][D],
 * contiguous, device) are copied to its slot of layer `layer`.  One launch
 * covers all tokens and heads.  block_tables, seq_idx, pos: device int32.
 * Two tokens of one call must not target the same slot.  Bit-exact copy.
 * n_tokens == 0 is a no-op. */
PF_API int pf_write_kv(const pf_pool *pool, int layer, const void *k_new,
                const void *v_new, const int32_t *block_tables,
                int n_table_rows, int max_blocks_per_seq,
                const int32_t *seq_idx, const int32_t *pos, int n_tokens,
                void *stream);

/* Gather (PageForge, "Four layers, one pointer": gather_kv assembles a
 * sequence's scattered pages into a contiguous buffer).  For every sequence
 * s and t < context_lens[s], row cu_off[s] + t of k_out / v_out
 * ([rows][Hkv][D] fp16, device) receives token t of layer `layer`.
 * context_lens: device int32 [n_seqs]; cu_off: device int64 [n_seqs]
 * (row offsets; the caller sizes the outputs).  Bit-exact copy. */
PF_API int pf_gather_kv(const pf_pool *pool, int layer, const int32_t *block_tables,
                 int max_blocks_per_seq, const int32_t *context_lens,
                 const int64_t *cu_off, int n_seqs, void *k_out, void *v_out,
                 void *stream);

/* ------------------------------------------- whole-block copies ---- */

/* Bytes of one block image: block b's K then V rows of layer 0, then of
 * layer 1, ...: [n_layers][2][B][Hkv][D] fp16.  0 for a null pool. */
PF_API size_t pf_block_image_bytes(const pf_pool *pool);
/* Copy-on-write copies (PagedAttention blog, "Copy-on-Write for Parallel
 * Sampling"): for i < n, block dst_ids[i] takes the contents of block
 * src_ids[i] in every layer, K and V.  src_ids, dst_ids: device int32 [n].
 * A destination must not also be a source or another pair's destination.
 * Ids outside [0, n_blocks) set PF_DEV_BAD_BLOCK_ID and that pair is
 * skipped.  Bit-exact.  n == 0 is a no-op. */
PF_API int pf_copy_blocks(const pf_pool *pool, const int32_t *src_ids,
                          const int32_t *dst_ids, int n, void *stream);
/* Swap out (same blog, "Preemption and Swapping": under memory pressure a
 * sequence's blocks are evicted to CPU memory, per block): the images of
 * blocks ids[0..n) (device int32) are written to host_dst[i] (n images of
 * pf_block_image_bytes each).  host_dst must be page-locked host memory
 * (cudaHostAlloc, cudaHostRegister, a pinned torch tensor); the kernel
 * writes it directly through its device mapping, with no staging copy.
 * PF_ERR_INVALID otherwise.  Bad ids are flagged and skipped as above. */
PF_API int pf_swap_out(const pf_pool *pool, const int32_t *ids, int n,
                       void *host_dst, void *stream);
/* Swap in: blocks ids[0..n) take the contents of the host images
 * host_src[0..n) (page-locked, as above; any block ids, so a sequence can
 * come back into other physical blocks -- patch its table to match). */
PF_API int pf_swap_in(const pf_pool *pool, const void *host_src,
                      const int32_t *ids, int n, void *stream);

/* Workspace bytes pf_paged_decode_attention needs for a batch of n_seqs
 * sequences of at most max_blocks_per_seq * block_size tokens with
 * n_q_heads query heads and this split setting.  0 on bad arguments.  An
 * implementation call with no counterpart on the pages (the workspace holds
 * the partial results of split sequences, the reduction of the
 * PagedAttention blog's "The Attention Kernel"). */
PF_API size_t pf_decode_workspace_bytes(const pf_pool *pool, int n_seqs,
                                 int n_q_heads, int max_blocks_per_seq,
                                 int split_tokens);

/* Prepare a workspace for first use (zero it); an implementation call with
 * no counterpart on the pages.  Needed once after the
 * workspace is allocated: everything a call reads back from the workspace
 * (merge jobs, the partial records of split sequences) carries a stamp of
 * the launch that wrote it, and zeroed memory holds no stamp of any launch.
 * Nothing else needs resetting, so every call -- one that set
 * PF_DEV_WAIT_TIMEOUT included -- leaves the workspace ready for the next.
 * Stamps count launches in the process (2^32 of them before they repeat). */
PF_API int pf_decode_workspace_init(void *workspace, size_t ws_bytes, void *stream);

/* Single-query decode attention through the block tables (PagedAttention
 * blog, "The Attention Kernel").  For each sequence s and q-head hq, with
 * L = context_lens[s] and kv-head h = hq / (n_q_heads / Hkv):
 *   z_t = scale * sum_d q[s][hq][d] * K[slot(s, t)][h][d],  t < L
 *   out[s][hq][d] = sum_t softmax(z)_t * V[slot(s, t)][h][d]
 * fp32 accumulation; L = 0 gives zeros.  q: fp16 [n_seqs][n_q_heads][D];
 * out: [n_seqs][n_q_heads][D] of out_dtype (PF_F16, rounded to nearest even,
 * or PF_F32); n_q_heads must be a multiple of Hkv (grouped heads share one
 * page load): 1 to 8 q-heads per kv-head under any split setting, up to 16
 * with split_tokens = 0 on pages of at least 16 tokens (PF_ERR_UNSUPPORTED
 * otherwise).  Schedules: split_tokens 0 = balanced spans (the work of all
 * sequences cut into equal shares, one per resident block; a sequence cut
 * by a share boundary has its partial results combined with the log-sum-exp
 * rule -- same section: reduction across thread blocks); -2 = the same
 * spans on the CUDA cores; -1 = never split; > 0 = fixed chunks of that
 * many tokens (rounded up to a multiple of 16), combined the same way.
 * Arithmetic: fp32 throughout, inputs fp16.  split_tokens 0 computes the
 * score and weighted-sum products on tensor cores (fp16 operands, fp32
 * accumulation); for fp16 output the softmax weights enter the weighted sum
 * rounded to fp16 (within the attention tolerance of the exact result), for
 * fp32 output as an fp16 part plus its fp16 rounding error (about 22 bits,
 * like the other schedules).  Every other schedule uses CUDA-core fp32
 * arithmetic (warp-shuffle dot products, fp32 weights) and no tensor
 * cores.
 * workspace: device memory of at least pf_decode_workspace_bytes(...) bytes,
 * initialised once with pf_decode_workspace_init; calls sharing a workspace
 * must not overlap on the GPU. */
PF_API int pf_paged_decode_attention(const pf_pool *pool, int layer, const void *q,
                              const int32_t *block_tables,
                              int max_blocks_per_seq,
                              const int32_t *context_lens, int n_seqs,
                              int n_q_heads, float scale, void *out,
                              int out_dtype, int split_tokens,
                              void *workspace, size_t ws_bytes, void *stream);

/* One decode step of one layer, fused (the scatter of PageForge, "Four
 * layers, one pointer", and the attention of the PagedAttention blog, "The
 * Attention Kernel", in one pass): for every sequence s with
 * L = context_lens[s] >= 1, the new token's rows k_new[s] and v_new[s]
 * (fp16 [n_seqs][Hkv][D], device) are written to slot(s, L - 1) of layer
 * `layer`, and then single-query attention runs over the L tokens exactly as
 * pf_paged_decode_attention does.  Results are those of pf_write_kv with
 * seq_idx[i] = i, pos[i] = L_i - 1 followed by pf_paged_decode_attention.
 * The write happens inside the attention kernel, by the block that reads
 * that slot, so a step costs one launch (plus a merge launch when
 * split_tokens > 0 cuts a sequence).  Same workspace as
 * pf_paged_decode_attention.
 * flags: 0, or PF_STEP_OVERLAP_PREVIOUS: the step's kernel is launched as a
 * programmatic dependent of the kernel issued just before it on the stream.
 * It then becomes resident while that kernel drains and reads only
 * context_lens and block_tables (to plan its work) before waiting for it to
 * finish; q, k_new, v_new, the pool, out and the workspace are touched only
 * after that.  Set the flag only when the kernel issued just before this call
 * does not write context_lens or block_tables (for instance when it is the
 * previous layer's or step's pf_decode_step).  If the previous operation on
 * the stream is not a kernel, the flag changes nothing.  Unknown bits give
 * PF_ERR_INVALID. */
enum pf_step_flags { PF_STEP_OVERLAP_PREVIOUS = 1 };
PF_API int pf_decode_step(const pf_pool *pool, int layer, const void *q,
                          const void *k_new, const void *v_new,
                          const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int n_seqs,
                          int n_q_heads, float scale, void *out,
                          int out_dtype, int split_tokens, void *workspace,
                          size_t ws_bytes, int flags, void *stream);

/* Multi-token append attention: a prompt, or a chunk of one, whose K/V rows
 * were already written into the sequence's last pages (pf_write_kv), then
 * attended to (PagedAttention blog, "Architecture": append, then attend;
 * PageFault README, "Four stages": the prompt is reserved up front).
 * Sequence s has L = context_lens[s] tokens, the last n_s = cu_q[s + 1] -
 * cu_q[s] of them new; their queries are rows cu_q[s] .. cu_q[s + 1] - 1 of
 * q (fp16 [T_q][n_q_heads][D], T_q = cu_q[n_seqs]).  The query of new token
 * i sits at position p = L - n_s + i and attends causally to tokens 0 .. p:
 *   out[row][hq][d] = sum_{t <= p} softmax_t(scale * q . K[slot(s, t)][h]) V[..][h][d]
 * with h = hq / (n_q_heads / Hkv); fp32 accumulation; out has q's shape, of
 * out_dtype.  A decode step is the case n_s = 1.  cu_q: device int32
 * [n_seqs + 1], non-decreasing; max_new_tokens bounds every n_s (it sizes
 * the grid).  On the device, n_s > L or > max_new_tokens, or a length
 * outside the table, sets PF_DEV_BAD_LENGTH and is clamped; bad block ids set
 * PF_DEV_BAD_BLOCK_ID.
 * Three kernels, chosen by rows = max_new_tokens x (n_q_heads / Hkv):
 * - with a workspace (of pf_prefill_workspace_bytes bytes, initialised once
 *   with pf_decode_workspace_init, not shared by overlapping calls) and
 *   rows <= 8 (16 on pages of at least 16 tokens), the decode kernel serves
 *   the new tokens as extra rows of each kv-head -- balanced spans over the
 *   contexts, every K/V byte read once per kv-head (a chunked append);
 * - otherwise, with rows >= 128 (prompts, long appends), a kernel on the
 *   fifth-generation tensor cores (tcgen05.mma, fp32 accumulators in tensor
 *   memory) takes 256 query rows of one (sequence, kv-head) per block and
 *   walks the context up to their last position; it needs no workspace;
 * - otherwise a warp-level MMA kernel does the same with 64 rows per block.
 * All compute the products on tensor cores with the softmax weights rounded
 * to fp16 (within the attention tolerance).
 * Up to 16 q-heads per kv-head; the tcgen05 kernel holds one block per SM
 * (165 KB of shared memory at head_dim 64, 197 KB at 128, and all 512
 * tensor-memory columns). */
PF_API int pf_paged_prefill_attention(const pf_pool *pool, int layer,
                                      const void *q,
                                      const int32_t *block_tables,
                                      int max_blocks_per_seq,
                                      const int32_t *context_lens,
                                      const int32_t *cu_q, int n_seqs,
                                      int max_new_tokens, int n_q_heads,
                                      float scale, void *out, int out_dtype,
                                      void *workspace, size_t ws_bytes,
                                      void *stream);
/* Workspace bytes of pf_paged_prefill_attention's decode-kernel path for
 * these sizes, or 0 when that path does not apply (more than 16 rows per
 * kv-head, or 8 on pages of fewer than 16 tokens; the call then needs no
 * workspace) or on bad arguments. */
PF_API size_t pf_prefill_workspace_bytes(const pf_pool *pool, int n_seqs,
                                         int n_q_heads, int max_blocks_per_seq,
                                         int max_new_tokens);

/* The decode attention call for callers that cannot allocate device memory.
 * No counterpart on the pages: it exists for code that may only touch the
 * buffers it is handed -- for instance an operator inside another runtime
 * or framework that owns every allocation -- and so cannot call cudaMalloc
 * or any allocating routine to provide the workspace that
 * pf_paged_decode_attention needs.  Same arguments and results as that call,
 * without workspace / ws_bytes: the scratch is a fixed 8 MiB array inside
 * the library (held by every GPU that loads the library until the process
 * exits).  Nothing is allocated.
 * - A batch whose scratch need (pf_decode_workspace_bytes) exceeds 8 MiB is
 *   rejected with PF_ERR_INVALID; split the batch or pass a workspace to
 *   pf_paged_decode_attention.
 * - The first call on a device looks up the array's device address (once
 *   per device, with that device current); make that first call before any
 *   stream capture.
 * - Every call on a device uses the same array, and each call leaves it
 *   ready for the next one (a call that set PF_DEV_WAIT_TIMEOUT included:
 *   what a call reads back carries its own launch's stamp).  Calls that
 *   overlap on the GPU (other streams, other threads) race on the scratch:
 *   order them on one stream.
 * - The device address is kept for the life of the process; after
 *   cudaDeviceReset (or anything else that tears down the device's primary
 *   context) this call must not be used again in that process. */
PF_API int pf_paged_decode_attention_noalloc(const pf_pool *pool, int layer,
                                             const void *q,
                                             const int32_t *block_tables,
                                             int max_blocks_per_seq,
                                             const int32_t *context_lens,
                                             int n_seqs, int n_q_heads,
                                             float scale, void *out,
                                             int out_dtype, int split_tokens,
                                             void *stream);

/* Testing hook for the bounded waits (no counterpart on the pages): block 0
 * of the next decode-attention launch in this process
 * (pf_paged_decode_attention, pf_decode_step, the noalloc variant, or the
 * decode-kernel path of pf_paged_prefill_attention) leaves the first stage of
 * its copy ring unfilled.  Every wait in the library gives up after 1 s: the
 * waits for that stage, and the merge of any split sequence with a part in
 * block 0, run out (the launch takes a few seconds), the kernel sets
 * PF_DEV_WAIT_TIMEOUT, every block returns (after its own copies in flight
 * have landed), and the context stays usable.  That launch's output is
 * undefined; the next launch with the same workspace computes normally.
 * Nothing is faulted and no memory is touched out of bounds.  Always PF_OK. */
PF_API int pf_test_inject_wait_timeout(void);

/* Read the device status word (OR of pf_device_flag bits set by kernels of
 * this library on the current device since the last reset) into *status_out.
 * Synchronises `stream`.  reset != 0 clears the word afterwards. */
PF_API int pf_device_status(int *status_out, int reset, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
