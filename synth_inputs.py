"""Seeded synthetic inputs for the paged KV-cache hot path.

This module is the one place both sides of a parity check get their inputs
from: the fp64 oracle (``oracle/``) and the CUDA library are fed the same
arrays.  It holds none of the method's arithmetic -- no slot translation, no
attention -- only random draws and the shape of each workload:

* values: fp16 N(0, 1) (float32 normal draws rounded to fp16), seed 1234;
* context lengths: uniform integer draws, seed 42;
* physical block ids: each sequence owns ``pages(L)`` distinct pool blocks.
  "ordered" hands out 0, 1, 2, ... sequence by sequence; "shuffled" hands out
  a seeded random permutation of the pool (seed 7), which is what a pool looks
  like after churn.  Unused table entries are 0.

Workload shapes (the pages' own workloads, restated):

* ``tiny``   1 layer, 4 seqs, 12 heads x 64, B = 16, 64-page pool, L ~ U[1, 100].
* ``gpt2``   GPT-2 124M shape: 12 layers x 12 heads x 64, 32 seqs, prompt
             U[16, 64] then 50 decode steps, pool of 512 tokens per sequence.
* ``mixed``  1 layer, 12 x 64, 4096 blocks of 16, 128 seqs: 64 with
             L ~ U[32, 128], 38 with U[256, 512], 26 with U[1024, 2048]
             (50 % / 30 % / 20 %), in a seeded random order.
* ``13b``    40 heads x 128, one layer, batch 1..64 at 2048 tokens.
* ``gqa``    14 q-heads / 2 kv-heads x 64, 256 seqs, L ~ U[32, 4096],
             block sizes 1 / 16 / 64 / 256 over the same lengths.
"""
import numpy as np

SEED_LENGTHS = 42
SEED_VALUES = 1234
SEED_SHUFFLE = 7

WORKLOADS = {
    "tiny": dict(n_layers=1, n_seqs=4, n_q_heads=12, n_kv_heads=12, head_dim=64,
                 block_size=16, n_blocks=64, len_lo=1, len_hi=100, scale=1.0 / 8),
    "gpt2": dict(n_layers=12, n_seqs=32, n_q_heads=12, n_kv_heads=12, head_dim=64,
                 block_size=16, prompt_lo=16, prompt_hi=64, decode_steps=50,
                 tokens_per_seq=512, scale=1.0 / 8),
    "mixed": dict(n_layers=1, n_seqs=128, n_q_heads=12, n_kv_heads=12, head_dim=64,
                  block_size=16, n_blocks=4096,
                  bands=((64, 32, 128), (38, 256, 512), (26, 1024, 2048)),
                  scale=1.0 / 8),
    "13b": dict(n_layers=1, n_q_heads=40, n_kv_heads=40, head_dim=128, block_size=16,
                context_len=2048, batches=(1, 2, 4, 8, 16, 32, 64),
                scale=float(np.float32(1.0 / np.sqrt(128.0)))),
    "gqa": dict(n_layers=24, n_seqs=256, n_q_heads=14, n_kv_heads=2, head_dim=64,
                len_lo=32, len_hi=4096, block_sizes=(1, 16, 64, 256), scale=1.0 / 8),
}


def fp16_normal(shape, seed):
    """fp16 N(0, 1) values from a seeded PCG64 stream."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def uniform_lengths(n, lo, hi, seed=SEED_LENGTHS):
    """n integer lengths uniform in [lo, hi] (both ends included)."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def band_lengths(bands, seed=SEED_LENGTHS):
    """Lengths from (count, lo, hi) bands, in a seeded random order."""
    rng = np.random.default_rng(seed)
    parts = [rng.integers(lo, hi + 1, size=c, dtype=np.int64) for c, lo, hi in bands]
    lens = np.concatenate(parts)
    rng.shuffle(lens)
    return lens.astype(np.int32)


def pages_for(length, block_size):
    """Pages a sequence of `length` tokens occupies (input structure only)."""
    return -(-int(length) // int(block_size))


def block_tables(lens, block_size, n_blocks, shuffle_seed=SEED_SHUFFLE, max_blocks=None):
    """Per-sequence physical block ids, [n_seqs, max_blocks] int32.

    shuffle_seed = 0 gives ordered frames (sequence s owns a contiguous,
    ascending run); any other seed draws ids from a seeded permutation of the
    pool.  Raises if the pool is too small for the lengths."""
    lens = np.asarray(lens)
    need = [pages_for(L, block_size) for L in lens]
    total = int(sum(need))
    if total > n_blocks:
        raise ValueError(f"workload needs {total} blocks, pool has {n_blocks}")
    if max_blocks is None:
        max_blocks = max(need) if need else 1
    max_blocks = max(int(max_blocks), 1)
    if shuffle_seed:
        ids = np.random.default_rng(shuffle_seed).permutation(n_blocks)
    else:
        ids = np.arange(n_blocks)
    table = np.zeros((len(lens), max_blocks), dtype=np.int32)
    cur = 0
    for s, n in enumerate(need):
        table[s, :n] = ids[cur:cur + n]
        cur += n
    return table


def cu_offsets(lens):
    """Packed-row offsets [n_seqs + 1] int64 for a varlen buffer."""
    off = np.zeros(len(lens) + 1, dtype=np.int64)
    off[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return off


def pool(n_layers, n_blocks, block_size, n_heads, head_dim, seed):
    """A K or V pool [n_layers, N, B, H, D] of fp16 N(0, 1)."""
    return fp16_normal((n_layers, n_blocks, block_size, n_heads, head_dim), seed)


def mixed_workload(shuffled=True):
    """Lengths and block tables of the 128-sequence mixed-length workload."""
    w = WORKLOADS["mixed"]
    lens = band_lengths(w["bands"])
    bt = block_tables(lens, w["block_size"], w["n_blocks"],
                      SEED_SHUFFLE if shuffled else 0,
                      max_blocks=2048 // w["block_size"])
    return lens, bt
