"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formula: each checks it against a
value the pages print, a closed form, a library routine (numpy's fp16 decoder,
torch's fp64 scaled-dot-product attention) or an invariant that a plausible
mistake (a wrong slot index, a transposed operand, a dropped scale or
normaliser, a wrong grouped-head mapping) would break.
"""
import math

import numpy as np
import pytest

import synth_inputs as si
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------- fp16

def test_fp16_decode_all_patterns(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.half_array_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero survives
    assert math.copysign(1.0, oracle_mod.half_to_double(0x8000)) == -1.0


# ----------------------------------------------------------- slot math

def test_slot_translation_golden(oracle_mod):
    g = {r[0]: r[1:] for r in read_golden("slot_translation.txt") if r[0] != "range"}
    ranges = [tuple(map(int, r[1:])) for r in read_golden("slot_translation.txt") if r[0] == "range"]
    B, L = int(g["block_size"][0]), int(g["length"][0])
    table = np.array([int(x) for x in g["table"]], dtype=np.int32)
    assert oracle_mod.blocks_needed(L, B) == int(g["blocks_needed"][0]) == len(table)
    assert oracle_mod.tail_waste(L, B) == int(g["tail_free"][0])
    for lo, hi, blk in ranges:
        for t in range(lo, hi + 1):
            # token t sits in physical block `blk`, row t - lo of that block
            assert oracle_mod.slot(table, B, t) == blk * B + (t - lo)


def test_tail_waste_bound(oracle_mod):
    for B in (1, 16, 64, 256):
        for L in range(1, 4 * B + 3):
            w = oracle_mod.tail_waste(L, B)
            assert 0 <= w <= B - 1
            assert oracle_mod.blocks_needed(L, B) * B == L + w


@pytest.mark.parametrize("name,shuffled", [("tiny", True), ("mixed", True), ("mixed", False)])
def test_no_two_tokens_share_a_slot(oracle_mod, name, shuffled):
    w = si.WORKLOADS[name]
    if name == "tiny":
        lens = si.uniform_lengths(w["n_seqs"], w["len_lo"], w["len_hi"])
        bt = si.block_tables(lens, w["block_size"], w["n_blocks"], si.SEED_SHUFFLE if shuffled else 0)
    else:
        lens, bt = si.mixed_workload(shuffled)
    seen = set()
    B = w["block_size"]
    for s, L in enumerate(lens):
        for t in range(int(L)):
            sl = oracle_mod.slot(bt[s], B, t)
            assert 0 <= sl < w["n_blocks"] * B
            assert sl not in seen
            seen.add(sl)
    assert len(seen) == int(np.sum(lens))


# ---------------------------------------------------- memory accounting

def _mb(x):
    return round(x / 1e6, 2)


def test_memory_accounting_golden(oracle_mod):
    rows = read_golden("memory_accounting.txt")
    seen = set()
    worked = {}
    for r in rows:
        key, vals = r[0], r[1:]
        seen.add(key)
        if key.startswith("worked_"):
            worked[key] = vals
        elif key == "pagefault_bytes_per_token":
            layers, heads, dim, dbytes, want = map(int, vals)
            assert oracle_mod.kv_bytes_per_token(layers, heads, dim, dbytes) == want
        elif key == "pagefault_naive_capacity":
            n, b, maxlen, want = map(int, vals)
            assert (n * b) // maxlen == want
        elif key == "naive_mb":
            n, maxlen, bpt, want = int(vals[0]), int(vals[1]), int(vals[2]), float(vals[3])
            assert _mb(oracle_mod.naive_reserved_bytes(n, maxlen, bpt)) == want
        elif key == "paged_mb":
            blocks, b, bpt, want, ratio = int(vals[0]), int(vals[1]), int(vals[2]), float(vals[3]), float(vals[4])
            lens = np.full(blocks, b, dtype=np.int32)   # any lengths filling `blocks` pages
            paged = oracle_mod.paged_reserved_bytes(lens, b, bpt)
            assert _mb(paged) == want
            naive = oracle_mod.naive_reserved_bytes(32, 2048, 512)
            assert round(naive / paged, 2) == ratio
        elif key == "sweep":
            b, blocks, res_mb, frag_mb, util, entries = (int(vals[0]), int(vals[1]), float(vals[2]),
                                                         float(vals[3]), float(vals[4]), int(vals[5]))
            stored = 20500
            # a 32-sequence length mix with `stored` tokens in exactly `blocks` pages:
            # all but one sequence fill whole pages; the remainder sits in the last.
            lens = _lens_with(blocks, b, stored)
            assert oracle_mod.paged_blocks(lens, b) == blocks
            assert _mb(oracle_mod.paged_reserved_bytes(lens, b, 512)) == res_mb
            assert _mb(oracle_mod.internal_fragmentation_tokens(lens, b) * 512) == frag_mb
            assert round(100 * oracle_mod.paged_utilization(lens, b), 1) == util
            assert 2048 // b == entries
        elif key == "naive_util":
            stored, n, maxlen, want = int(vals[0]), int(vals[1]), int(vals[2]), float(vals[3])
            assert round(100 * stored / (n * maxlen), 1) == want
        elif key == "seed7_util":
            blocks, b, frag, n, maxlen, paged_util, naive_util = (int(vals[0]), int(vals[1]), float(vals[2]),
                                                                   int(vals[3]), int(vals[4]),
                                                                   float(vals[5]), float(vals[6]))
            stored = blocks * b - round(frag * n)
            lens = _lens_with(blocks, b, stored)
            assert round(100 * oracle_mod.paged_utilization(lens, b), 1) == paged_util
            assert round(100 * stored / (n * maxlen), 1) == naive_util
        elif key == "stored_tokens":
            assert int(vals[0]) == 1298 * 16 - round(8.38 * 32)
        elif key == "llama3_70b":
            assert oracle_mod.kv_bytes_per_token(*map(int, vals[:4])) == int(vals[4]) == 320 * 1024
        elif key == "llama3_70b_capacity":
            budget, naive_len, naive_n, mean_len, paged_n, ratio = (float(vals[0]), int(vals[1]), int(vals[2]),
                                                                     int(vals[3]), int(vals[4]), float(vals[5]))
            bpt = oracle_mod.kv_bytes_per_token(80, 8, 128, 2)
            assert int(budget // (bpt * naive_len)) == naive_n
            assert int(budget // (bpt * mean_len)) == paged_n
            assert round(paged_n / naive_n, 1) == ratio
        elif key.startswith("gpt2"):
            bpt = oracle_mod.kv_bytes_per_token(12, 12, 64, 2)
            page = 16 * bpt
            if key == "gpt2":
                assert bpt == oracle_mod.kv_bytes_per_token(*map(int, vals))
            elif key == "gpt2_page_mb":
                assert _mb(oracle_mod.paged_reserved_bytes([int(vals[0])], 16, bpt)) == float(vals[1])
            elif key == "gpt2_naive_seq_mb":
                assert _mb(oracle_mod.naive_reserved_bytes(1, int(vals[0]), bpt)) == float(vals[1])
            elif key == "gpt2_naive_total_mb":
                assert _mb(oracle_mod.naive_reserved_bytes(int(vals[0]), 512, bpt)) == float(vals[1])
            elif key == "gpt2_paged_total_mb":
                assert _mb(int(vals[0]) * page) == float(vals[1])
            elif key == "gpt2_per_seq_pages":
                lens = [16 * int(vals[0])]
                assert _mb(oracle_mod.paged_reserved_bytes(lens, 16, bpt)) == float(vals[1])
            elif key == "gpt2_pool_capacity":
                pool_pages, naive_n, paged_lo, paged_hi = map(int, vals)
                naive_pages = oracle_mod.blocks_needed(512, 16)
                assert pool_pages // naive_pages == naive_n
                assert pool_pages // 4 == paged_lo and pool_pages // 1 == paged_hi
            elif key == "gpt2_seqs_per_gb":
                naive_n, paged_n = map(int, vals)
                assert round(1e9 / oracle_mod.naive_reserved_bytes(1, 512, bpt)) == naive_n
                assert round(1e9 / oracle_mod.paged_reserved_bytes([60], 16, bpt)) == paged_n
            elif key == "gpt2_savings":
                prompt, step, ratio = int(vals[0]), int(vals[1]), float(vals[2])
                paged = oracle_mod.blocks_needed(prompt + step, 16)
                assert round(oracle_mod.blocks_needed(512, 16) / paged, 1) == ratio
            elif key == "gpt2_recovery":
                n, naive_mb, peak_pages, peak_mb, pct = (int(vals[0]), int(vals[1]), int(vals[2]),
                                                         float(vals[3]), float(vals[4]))
                naive = oracle_mod.naive_reserved_bytes(n, 512, bpt)
                assert round(naive / 1e6) == naive_mb
                assert _mb(peak_pages * page) == peak_mb
                assert round(100 * peak_pages * page / naive, 1) == pct
        elif key.startswith("thirteen_b"):
            if key == "thirteen_b":
                assert oracle_mod.kv_bytes_per_token(*map(int, vals[:4])) == int(vals[4]) == 800 * 1024
            elif key == "thirteen_b_seq":
                assert round(int(vals[0]) * 800e3 / 1e9, 1) == float(vals[1])
            elif key == "thirteen_b_used":
                assert int(int(vals[0]) * 800e3 / 1e6) == int(vals[1])
            elif key == "thirteen_b_capacity":
                assert (int(vals[0]) * 10) // 16 == int(vals[1])   # 24 GB / 1.6 GB per sequence
        else:
            raise AssertionError(f"unhandled golden key {key}")
    lens = [int(x) for x in worked["worked_lengths"]]
    B = int(worked["worked_block_size"][0])
    assert oracle_mod.paged_blocks(lens, B) == int(worked["worked_blocks"][0])
    assert oracle_mod.internal_fragmentation_tokens(lens, B) == int(worked["worked_fragmentation"][0])
    assert {"sweep", "gpt2_savings", "thirteen_b", "llama3_70b", "paged_mb"} <= seen


def _lens_with(blocks, b, stored, n=32):
    """n lengths occupying exactly `blocks` pages of size b and holding
    `stored` tokens (used only to feed the accounting formulas)."""
    per = [blocks // n + (1 if i < blocks % n else 0) for i in range(n)]
    lens = [p * b for p in per]
    excess = sum(lens) - stored
    i = 0
    while excess > 0:
        cut = min(excess, b - 1, lens[i] - 1 - (per[i] - 1) * b) if per[i] > 0 else 0
        cut = max(cut, 0)
        lens[i] -= cut
        excess -= cut
        i += 1
    assert excess == 0
    return np.array(lens, dtype=np.int32)


def test_mean_tail_waste_matches_half_block(oracle_mod):
    # PageFault README, "Stage 2: memory": expected internal fragmentation of
    # (B - 1) / 2 tokens per sequence for uniformly distributed lengths.
    lens = si.uniform_lengths(200_000, 1, 4096, seed=3)
    mean = oracle_mod.internal_fragmentation_tokens(lens, 16) / len(lens)
    assert abs(mean - 7.5) < 0.05


# ------------------------------------------------------------ attention

def _contig_case(seed, lens, hq, hkv, d):
    q = si.fp16_normal((len(lens), hq, d), seed)
    T = int(np.sum(lens))
    k = si.fp16_normal((T, hkv, d), seed + 1)
    v = si.fp16_normal((T, hkv, d), seed + 2)
    return q, k, v, si.cu_offsets(lens)


@pytest.mark.parametrize("hq,hkv,d", [(12, 12, 64), (14, 2, 64), (8, 2, 128), (4, 1, 32)])
def test_attention_matches_torch_sdpa_fp64(oracle_mod, hq, hkv, d):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    lens = np.array([1, 2, 7, 16, 17, 100, 333], dtype=np.int32)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    q, k, v, off = _contig_case(11, lens, hq, hkv, d)
    ours = oracle_mod.attention_contiguous(q, k, v, off, lens, scale)
    for s, L in enumerate(lens):
        qs = torch.from_numpy(q[s].astype(np.float64))[None, :, None, :]          # [1, Hq, 1, D]
        ks = torch.from_numpy(k[off[s]:off[s] + L].astype(np.float64)).permute(1, 0, 2)[None]
        vs = torch.from_numpy(v[off[s]:off[s] + L].astype(np.float64)).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(qs, ks, vs, scale=scale, enable_gqa=(hq != hkv))
        np.testing.assert_allclose(ours[s], ref[0, :, 0, :].numpy(), rtol=0, atol=1e-12)


def test_attention_uniform_keys_give_mean_of_values(oracle_mod):
    # PageFault README, "Test": uniform keys -> mean of values.
    L, h, d = 37, 3, 64
    q = si.fp16_normal((1, h, d), 5)
    krow = si.fp16_normal((1, h, d), 6)
    k = np.repeat(krow, L, axis=0)
    v = si.fp16_normal((L, h, d), 7)
    out = oracle_mod.attention_contiguous(q, k, v, si.cu_offsets([L]), np.array([L]), 0.125)
    np.testing.assert_allclose(out[0], v.astype(np.float64).mean(axis=0), rtol=0, atol=1e-14)


def test_attention_one_hot_key_selects_its_value(oracle_mod):
    # PageFault README, "Test": one-hot key -> that value.
    L, h, d, j = 50, 2, 64, 17
    q = si.fp16_normal((1, h, d), 8)
    k = np.zeros((L, h, d), dtype=np.float16)
    k[j] = (q[0] * 8).astype(np.float16)     # z_j = scale * 8 |q|^2 ~ 64, others 0
    v = si.fp16_normal((L, h, d), 9)
    out = oracle_mod.attention_contiguous(q, k, v, si.cu_offsets([L]), np.array([L]), 0.125)
    np.testing.assert_allclose(out[0], v[j].astype(np.float64), rtol=0, atol=1e-12)


def test_attention_single_token_is_exact_value(oracle_mod):
    q = si.fp16_normal((3, 4, 64), 10)
    k = si.fp16_normal((3, 4, 64), 11)
    v = si.fp16_normal((3, 4, 64), 12)
    lens = np.array([1, 1, 1], dtype=np.int32)
    out = oracle_mod.attention_contiguous(q, k, v, si.cu_offsets(lens), lens, 0.125)
    assert np.array_equal(out, v.astype(np.float64))


def test_attention_two_tokens_logistic_closed_form(oracle_mod):
    # softmax of two scores is the logistic function of their difference
    q = si.fp16_normal((1, 1, 64), 13).astype(np.float64)[0, 0]
    k = si.fp16_normal((2, 1, 64), 14)
    v = si.fp16_normal((2, 1, 64), 15)
    out = oracle_mod.attention_contiguous(q.astype(np.float16)[None, None], k, v,
                                          si.cu_offsets([2]), np.array([2]), 0.125)
    z0 = 0.125 * float(np.dot(q, k[0, 0].astype(np.float64)))
    z1 = 0.125 * float(np.dot(q, k[1, 0].astype(np.float64)))
    w0 = 1.0 / (1.0 + math.exp(z1 - z0))
    ref = w0 * v[0, 0].astype(np.float64) + (1.0 - w0) * v[1, 0].astype(np.float64)
    np.testing.assert_allclose(out[0, 0], ref, rtol=0, atol=1e-14)


def test_attention_empty_sequence_is_zero(oracle_mod):
    q = si.fp16_normal((2, 2, 64), 16)
    k = si.fp16_normal((5, 2, 64), 17)
    v = si.fp16_normal((5, 2, 64), 18)
    lens = np.array([0, 5], dtype=np.int32)
    out = oracle_mod.attention_contiguous(q, k, v, si.cu_offsets(lens), lens, 0.125)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out[1]))


def test_grouped_heads_read_their_own_kv_head(oracle_mod):
    # q-head hq reads kv-head hq // G: give each kv-head a constant V so the
    # output identifies which kv-head a q-head attended to.
    hq, hkv, d, L = 14, 2, 64, 9
    q = si.fp16_normal((1, hq, d), 19)
    k = si.fp16_normal((L, hkv, d), 20)
    v = np.zeros((L, hkv, d), dtype=np.float16)
    v[:, 0, :] = 1.0
    v[:, 1, :] = 2.0
    out = oracle_mod.attention_contiguous(q, k, v, si.cu_offsets([L]), np.array([L]), 0.125)
    for h in range(hq):
        assert np.allclose(out[0, h], 1.0 + (h // 7), atol=1e-14)


def test_paged_readback_equals_contiguous_bitwise(oracle_mod):
    # PageFault README, "Test": paged == contiguous bitwise on a shuffled pool.
    w = si.WORKLOADS["tiny"]
    lens = si.uniform_lengths(w["n_seqs"], w["len_lo"], w["len_hi"])
    H, D, B, N = w["n_kv_heads"], w["head_dim"], w["block_size"], w["n_blocks"]
    bt = si.block_tables(lens, B, N, si.SEED_SHUFFLE)
    q, kc, vc, off = _contig_case(21, lens, w["n_q_heads"], H, D)
    kp = si.pool(1, N, B, H, D, 22)
    vp = si.pool(1, N, B, H, D, 23)
    seq_idx = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    oracle_mod.scatter(kp, vp, 0, kc, vc, bt, seq_idx, pos)
    kg, vg = oracle_mod.gather(kp, vp, 0, bt, lens, off)
    assert np.array_equal(kg.view(np.uint16), kc.view(np.uint16))
    assert np.array_equal(vg.view(np.uint16), vc.view(np.uint16))
    paged = oracle_mod.attention_paged(q, kp, vp, 0, bt, lens, w["scale"])
    contig = oracle_mod.attention_contiguous(q, kc, vc, off, lens, w["scale"])
    assert np.array_equal(paged, contig)


def test_scatter_touches_only_its_slots(oracle_mod):
    N, B, H, D = 8, 4, 2, 8
    kp = si.pool(2, N, B, H, D, 24)
    vp = si.pool(2, N, B, H, D, 25)
    k0, v0 = kp.copy(), vp.copy()
    bt = np.array([[5, 2], [7, 0]], dtype=np.int32)
    kn = si.fp16_normal((2, H, D), 26)
    vn = si.fp16_normal((2, H, D), 27)
    oracle_mod.scatter(kp, vp, 1, kn, vn, bt, np.array([0, 1]), np.array([6, 1]))
    # token 6 of seq 0 -> block bt[0][1] = 2, row 2; token 1 of seq 1 -> block 7, row 1
    assert np.array_equal(kp[1, 2, 2], kn[0]) and np.array_equal(vp[1, 7, 1], vn[1])
    kp[1, 2, 2] = k0[1, 2, 2]
    kp[1, 7, 1] = k0[1, 7, 1]
    vp[1, 2, 2] = v0[1, 2, 2]
    vp[1, 7, 1] = v0[1, 7, 1]
    assert np.array_equal(kp.view(np.uint16), k0.view(np.uint16))
    assert np.array_equal(vp.view(np.uint16), v0.view(np.uint16))


@pytest.mark.parametrize("cuts", [[0, 300], [0, 1, 300], [0, 16, 32, 250, 300], [0, 0, 128, 300, 300]])
def test_split_partials_merge_to_unsplit(oracle_mod, cuts):
    # PagedAttention blog, "The Attention Kernel": partial softmax results over
    # disjoint token ranges combine with the log-sum-exp rule.
    L, H, D = 300, 3, 64
    q = si.fp16_normal((H, D), 28)
    k = si.fp16_normal((L, H, D), 29)
    v = si.fp16_normal((L, H, D), 30)
    full = oracle_mod.attention_contiguous(q[None], k, v, si.cu_offsets([L]), np.array([L]), 0.125)
    for h in range(H):
        parts = [oracle_mod.attention_partial(q[h], k, v, h, a, b, 0.125) for a, b in zip(cuts, cuts[1:])]
        ms = [p[0] for p in parts]
        ls = [p[1] for p in parts]
        accs = np.stack([p[2] for p in parts])
        merged = oracle_mod.lse_merge(ms, ls, accs)
        np.testing.assert_allclose(merged, full[0, h], rtol=0, atol=1e-13)


def _marked_pools(n_layers, n_blocks, block_size, heads, dim):
    """Pools whose every (layer, block, K/V) image holds one distinct fp16
    bit pattern, so an image's origin can be read off its contents."""
    k = np.zeros((n_layers, n_blocks, block_size, heads, dim), dtype=np.uint16)
    v = np.zeros_like(k)
    for layer in range(n_layers):
        for b in range(n_blocks):
            k[layer, b] = 0x1000 + 64 * layer + 2 * b
            v[layer, b] = 0x1000 + 64 * layer + 2 * b + 1
    return k.view(np.float16), v.view(np.float16)


def test_block_copies_move_whole_images_and_nothing_else(oracle_mod):
    # PagedAttention blog, "Copy-on-Write for Parallel Sampling": the new
    # block receives the shared block's contents; other blocks are untouched.
    k, v = _marked_pools(3, 10, 16, 2, 8)
    k0, v0 = k.copy(), v.copy()
    oracle_mod.copy_blocks(k, v, [4, 7], [9, 1])
    for layer in range(3):
        assert np.array_equal(k[layer, 9], k0[layer, 4]) and np.array_equal(v[layer, 9], v0[layer, 4])
        assert np.array_equal(k[layer, 1], k0[layer, 7]) and np.array_equal(v[layer, 1], v0[layer, 7])
    untouched = [b for b in range(10) if b not in (9, 1)]
    assert np.array_equal(k[:, untouched], k0[:, untouched]) and np.array_equal(v[:, untouched], v0[:, untouched])


def test_swap_images_layout_and_round_trip(oracle_mod):
    # Same blog, "Preemption and Swapping": blocks go to host memory one by
    # one and come back later, possibly into other physical blocks.
    k, v = _marked_pools(3, 10, 16, 2, 8)
    ids = [6, 0, 3]
    img = oracle_mod.swap_out(k, v, ids).view(np.uint16)
    assert img.shape == (3, 3, 2, 16, 2, 8)
    for i, b in enumerate(ids):
        for layer in range(3):
            assert np.all(img[i, layer, 0] == 0x1000 + 64 * layer + 2 * b)       # K
            assert np.all(img[i, layer, 1] == 0x1000 + 64 * layer + 2 * b + 1)   # V
    k2, v2 = np.zeros_like(k), np.zeros_like(v)
    oracle_mod.swap_in(k2, v2, img.view(np.float16), [2, 8, 5])
    for src, dst in zip(ids, [2, 8, 5]):
        assert np.array_equal(k2[:, dst], k[:, src]) and np.array_equal(v2[:, dst], v[:, src])
    others = [b for b in range(10) if b not in (2, 8, 5)]
    assert not k2[:, others].view(np.uint16).any() and not v2[:, others].view(np.uint16).any()


def _prompt_pool(tokens, heads, dim, seed):
    """One-layer pool holding a `tokens`-token prompt in shuffled 16-token
    pages, plus its table row."""
    B = 16
    n_pages = -(-tokens // B)
    table = np.array(np.random.default_rng(seed).permutation(n_pages + 3)[:n_pages], dtype=np.int32)
    k = si.fp16_normal((1, n_pages + 3, B, heads, dim), seed + 1)
    v = si.fp16_normal((1, n_pages + 3, B, heads, dim), seed + 2)
    return k, v, table[None, :]


def test_prefill_of_a_two_token_prompt_closed_form(oracle_mod):
    # Prompt of two tokens, both new: query 0 sees token 0 only (its output
    # is V0 exactly); query 1 sees both (the two-term softmax).
    heads, dim, scale = 3, 64, 0.125
    k, v, bt = _prompt_pool(2, heads, dim, 31)
    q = si.fp16_normal((2, heads, dim), 34)
    out = oracle_mod.prefill_attention(q, k, v, 0, bt, [2], [0, 2], scale)
    K = k.astype(np.float64)[0][bt[0]].reshape(-1, heads, dim)
    V = v.astype(np.float64)[0][bt[0]].reshape(-1, heads, dim)
    Q = q.astype(np.float64)
    for h in range(heads):
        assert np.array_equal(out[0, h], V[0, h])
        z0 = scale * Q[1, h] @ K[0, h]
        z1 = scale * Q[1, h] @ K[1, h]
        w0 = 1.0 / (1.0 + math.exp(z1 - z0))
        assert np.allclose(out[1, h], w0 * V[0, h] + (1.0 - w0) * V[1, h], rtol=0, atol=1e-12)


def test_prefill_is_causal(oracle_mod):
    # A later token's keys and values never reach an earlier query; an
    # earlier token's do.
    heads, dim, L, n = 2, 64, 40, 6
    k, v, bt = _prompt_pool(L, heads, dim, 41)
    q = si.fp16_normal((n, heads, dim), 44)
    base = oracle_mod.prefill_attention(q, k, v, 0, bt, [L], [0, n], 0.125)
    page, off = divmod(L - 1, 16)              # the last token, position L - 1
    k2 = k.copy()
    k2[0, bt[0, page], off] = np.float16(7.0)
    out = oracle_mod.prefill_attention(q, k2, v, 0, bt, [L], [0, n], 0.125)
    assert np.array_equal(out[: n - 1], base[: n - 1])      # queries at L - 6 .. L - 2
    assert not np.array_equal(out[n - 1], base[n - 1])      # the query at L - 1 sees it
    page, off = divmod(L - n, 16)               # the first new token
    k3 = k.copy()
    k3[0, bt[0, page], off] = np.float16(7.0)
    out = oracle_mod.prefill_attention(q, k3, v, 0, bt, [L], [0, n], 0.125)
    assert all(not np.array_equal(out[i], base[i]) for i in range(n))


@pytest.mark.parametrize("hq,hkv,d,B", [(4, 2, 64, 16), (6, 6, 32, 1), (8, 1, 128, 4)])
def test_prefill_matches_torch_sdpa_with_a_causal_mask(oracle_mod, hq, hkv, d, B):
    """The multi-token append against torch's fp64 scaled-dot-product
    attention with an explicit mask: new token i of a sequence of L tokens (n
    of them new) sits at position L - n + i and attends to positions 0 .. L - n
    + i, through the block table; whole prompts, appends and a sequence with
    no new token."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    lens = np.array([1, 9, 40, 23, 17], dtype=np.int32)
    n_new = np.array([1, 9, 6, 0, 17], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    n_blocks = int(sum(-(-int(L) // B) for L in lens)) + 5
    bt = si.block_tables(lens, B, n_blocks, 61)
    k = si.pool(1, n_blocks, B, hkv, d, 62)
    v = si.pool(1, n_blocks, B, hkv, d, 63)
    q = si.fp16_normal((int(cu[-1]), hq, d), 64)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    ours = oracle_mod.prefill_attention(q, k, v, 0, bt, lens, cu, scale)
    K = k.astype(np.float64)[0].reshape(-1, hkv, d)
    V = v.astype(np.float64)[0].reshape(-1, hkv, d)
    for s, (L, n) in enumerate(zip(lens, n_new)):
        if n == 0:
            continue
        t = np.arange(L)
        slots = bt[s, t // B].astype(np.int64) * B + t % B
        ks = torch.from_numpy(K[slots]).permute(1, 0, 2)[None]                     # [1, Hkv, L, D]
        vs = torch.from_numpy(V[slots]).permute(1, 0, 2)[None]
        qs = torch.from_numpy(q[cu[s]:cu[s + 1]].astype(np.float64)).permute(1, 0, 2)[None]   # [1, Hq, n, D]
        pos = L - n + np.arange(n)
        mask = torch.from_numpy(t[None, :] <= pos[:, None])                        # [n, L], True = attended
        ref = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=scale, enable_gqa=(hq != hkv))
        np.testing.assert_allclose(ours[cu[s]:cu[s + 1]], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
