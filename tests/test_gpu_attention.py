"""Paged decode attention on the GPU against the fp64 oracle.

Tolerance (the stated target): max abs err <= 2e-3 and mean abs err <= 2e-4
against the unrounded fp64 result, fp16 inputs ~ N(0, 1)."""
import math

import numpy as np
import pytest

import synth_inputs as si
from gpu_util import PagedCase, assert_close_to_oracle, dev, host

pytestmark = pytest.mark.gpu


def _tiny(pkv, cuda_dev, shuffled=True):
    w = si.WORKLOADS["tiny"]
    lens = si.uniform_lengths(w["n_seqs"], w["len_lo"], w["len_hi"])
    return PagedCase(pkv, cuda_dev, lens, w["n_q_heads"], w["n_kv_heads"], w["head_dim"], w["block_size"],
                     n_blocks=w["n_blocks"], shuffle_seed=si.SEED_SHUFFLE if shuffled else 0), w["scale"]


# fp32 output carries no fp16 rounding of the softmax weights on any path
# (the CUDA-core consumers keep fp32 weights; the tensor-core consumers take
# P V with the weights' fp16 part and its fp16 rounding error): it is held to
# 1e-5 max / 1e-6 mean against the fp64 oracle, far inside the fp16 bound.
TIGHT = dict(max_abs=1e-5, mean_abs=1e-6)


@pytest.mark.parametrize("split", [0, -2, -1, 16, 48])
@pytest.mark.parametrize("out_f32", [False, True])
def test_tiny_matches_oracle(pkv, cuda_dev, oracle_mod, split, out_f32):
    import torch
    c, scale = _tiny(pkv, cuda_dev)
    out = c.attention(scale, split=split, out_dtype=torch.float32 if out_f32 else torch.float16)
    ref = c.oracle(oracle_mod, scale)
    assert_close_to_oracle(host(out), ref, what=f"tiny split={split}")
    if out_f32:
        assert_close_to_oracle(host(out), ref, what="tiny fp32", **TIGHT)
    assert pkv.pf_device_status(reset=True) == 0


def test_tiny_brute_force_edge_lengths(pkv, cuda_dev, oracle_mod):
    # every length from 1 to 70 (one to five pages, ragged tails), plus 0
    import torch
    lens = np.array([0] + list(range(1, 71)), dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 4, 2, 64, 16)
    for split in (0, -2, 16, 32, -1):
        out = c.attention(0.125, split=split, out_dtype=torch.float32)
        ref = c.oracle(oracle_mod, 0.125)
        assert np.all(host(out)[0] == 0.0)
        assert_close_to_oracle(host(out), ref, what=f"edge split={split}", **TIGHT)


def test_single_token_is_exact_value(pkv, cuda_dev):
    lens = np.ones(9, dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    out = host(c.attention(0.125))
    for s in range(9):
        blk = c.bt[s, 0]
        assert np.array_equal(out[s].view(np.uint16), c.v_host[0, blk, 0].view(np.uint16))


def test_tail_slots_are_never_read(pkv, cuda_dev, oracle_mod):
    lens = np.array([1, 7, 16, 17, 30, 100], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    # poison every slot a sequence does not use, including whole unused blocks
    k, v = c.k_host.copy(), c.v_host.copy()
    used = np.zeros((c.n_blocks, 16), dtype=bool)
    for s, L in enumerate(lens):
        for t in range(L):
            used[c.bt[s, t // 16], t % 16] = True
    k[0][~used] = np.float16(np.nan)
    v[0][~used] = np.float16(np.nan)
    c.k_dev.copy_(dev(k, cuda_dev))
    c.v_dev.copy_(dev(v, cuda_dev))
    for split in (0, 16, -1):
        out = host(c.attention(0.125, split=split))
        ref = oracle_mod.attention_paged(c.q, k, v, 0, c.bt, lens, 0.125)
        assert_close_to_oracle(out, ref, what=f"poisoned tails split={split}")


def test_mixed_full_size_shuffled_and_ordered(pkv, cuda_dev, oracle_mod):
    """The 128-sequence mixed-length workload at full size (4096 blocks of 16),
    in the launch configuration the benchmark times (auto split), every output
    checked.  The same token rows are written by the library's scatter into
    ordered and into shuffled frames; both give bit-identical results (the
    reduction order never depends on block ids)."""
    w = si.WORKLOADS["mixed"]
    lens = si.band_lengths(w["bands"])
    off = si.cu_offsets(lens)
    T = int(off[-1])
    kc = si.fp16_normal((T, 12, 64), 301)
    vc = si.fp16_normal((T, 12, 64), 302)
    q = si.fp16_normal((len(lens), 12, 64), 303)
    ref = oracle_mod.attention_contiguous(q, kc, vc, off, lens, w["scale"])
    seq_idx = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    outs = {}
    for shuffled in (True, False):
        c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16, n_blocks=w["n_blocks"],
                      shuffle_seed=si.SEED_SHUFFLE if shuffled else 0, max_blocks=128)
        pkv.pf_write_kv(c.pool, 0, dev(kc, cuda_dev), dev(vc, cuda_dev), c.bt_dev,
                        dev(seq_idx, cuda_dev), dev(pos, cuda_dev))
        # the tensor-core consumers (the default) and the CUDA-core ones
        for split in (0, -2):
            out = host(c.attention(w["scale"], split=split, q_dev=dev(q, cuda_dev)))
            assert_close_to_oracle(out, ref, what=f"mixed shuffled={shuffled} split={split}")
            outs[(shuffled, split)] = out
    for split in (0, -2):
        assert np.array_equal(outs[(True, split)].view(np.uint16), outs[(False, split)].view(np.uint16))


@pytest.mark.parametrize("batch", [1, 4])
def test_13b_like_split_and_no_split(pkv, cuda_dev, oracle_mod, batch):
    w = si.WORKLOADS["13b"]
    lens = np.full(batch, w["context_len"], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, w["n_q_heads"], w["n_kv_heads"], w["head_dim"], w["block_size"])
    ref = c.oracle(oracle_mod, w["scale"])
    for split in (-1, 0, 256):
        out = host(c.attention(w["scale"], split=split))
        assert_close_to_oracle(out, ref, what=f"13b batch={batch} split={split}")


def test_gqa_block_size_sweep_same_tokens(pkv, cuda_dev, oracle_mod):
    """14 q-heads / 2 kv-heads; the same token stream stored with block sizes
    1, 16, 64, 256 gives the oracle's result, and bit-identical outputs across
    block sizes (tiles are 16 tokens whatever the page size: 1-token pages are
    staged row by row into the same tile layout)."""
    w = si.WORKLOADS["gqa"]
    lens = si.uniform_lengths(48, w["len_lo"], w["len_hi"])
    Hq, Hkv, D = w["n_q_heads"], w["n_kv_heads"], w["head_dim"]
    off = si.cu_offsets(lens)
    T = int(off[-1])
    kc = si.fp16_normal((T, Hkv, D), 201)
    vc = si.fp16_normal((T, Hkv, D), 202)
    q = si.fp16_normal((len(lens), Hq, D), 203)
    ref = oracle_mod.attention_contiguous(q, kc, vc, off, lens, w["scale"])
    seq_idx = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    results = []
    for B in w["block_sizes"]:
        c = PagedCase(pkv, cuda_dev, lens, Hq, Hkv, D, B)
        # write the token stream through the library's own scatter
        pkv.pf_write_kv(c.pool, 0, dev(kc, cuda_dev), dev(vc, cuda_dev), c.bt_dev,
                        dev(seq_idx, cuda_dev), dev(pos, cuda_dev))
        out = host(c.attention(w["scale"], q_dev=dev(q, cuda_dev)))
        assert_close_to_oracle(out, ref, what=f"gqa B={B}")
        results.append(out)
    for r in results[1:]:
        assert np.array_equal(r.view(np.uint16), results[0].view(np.uint16))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4)])
def test_one_token_pages_head_dim_128(pkv, cuda_dev, oracle_mod, hq, hkv):
    """head_dim 128 on 1-token pages (rows staged by cp.async into the
    two-half tile layout): the oracle's result, and bit-identical to the same
    tokens on 16-token pages."""
    lens = si.uniform_lengths(9, 1, 300, seed=31)
    D = 128
    off = si.cu_offsets(lens)
    T = int(off[-1])
    kc = si.fp16_normal((T, hkv, D), 311)
    vc = si.fp16_normal((T, hkv, D), 312)
    q = si.fp16_normal((len(lens), hq, D), 313)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    ref = oracle_mod.attention_contiguous(q, kc, vc, off, lens, scale)
    seq_idx = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    outs = []
    for B in (1, 16):
        c = PagedCase(pkv, cuda_dev, lens, hq, hkv, D, B)
        pkv.pf_write_kv(c.pool, 0, dev(kc, cuda_dev), dev(vc, cuda_dev), c.bt_dev,
                        dev(seq_idx, cuda_dev), dev(pos, cuda_dev))
        out = host(c.attention(scale, q_dev=dev(q, cuda_dev)))
        assert_close_to_oracle(out, ref, what=f"{hq}/{hkv}x128 B={B}")
        outs.append(out)
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0


def test_gqa_full_size_every_output(pkv, cuda_dev, oracle_mod):
    """The grouped-heads workload at full size (256 sequences of U[32, 4096]
    tokens, 14/2 x 64, pages of 16, shuffled frames) in the launch
    configuration the benchmark times (balanced schedule): every output
    against the oracle."""
    w = si.WORKLOADS["gqa"]
    lens = si.uniform_lengths(w["n_seqs"], w["len_lo"], w["len_hi"], seed=12)
    c = PagedCase(pkv, cuda_dev, lens, w["n_q_heads"], w["n_kv_heads"], w["head_dim"], 16)
    out = host(c.attention(w["scale"], split=0))
    assert_close_to_oracle(out, c.oracle(oracle_mod, w["scale"]), what="gqa full size")
    assert pkv.pf_device_status(reset=True) == 0


def test_13b_like_full_batch_sampled(pkv, cuda_dev, oracle_mod):
    """The 13B-like shape at its largest batch (64 sequences of 2048 tokens,
    40 x 128, 2.7 GB of K/V), balanced schedule and no split.  The pool is
    filled on the device; the pages of four sampled sequences are overwritten
    with seeded host values, and those sequences' outputs (which read only
    their own pages) are checked against the oracle."""
    import torch
    w = si.WORKLOADS["13b"]
    S, L, H, D, B = 64, w["context_len"], w["n_q_heads"], w["head_dim"], w["block_size"]
    pages = L // B
    N = S * pages
    bt = si.block_tables(np.full(S, L, dtype=np.int32), B, N, si.SEED_SHUFFLE, max_blocks=pages)
    gen = torch.Generator(device=cuda_dev)
    gen.manual_seed(77)
    k = torch.randn((1, N, B, H, D), generator=gen, device=cuda_dev, dtype=torch.float32).half()
    v = torch.randn((1, N, B, H, D), generator=gen, device=cuda_dev, dtype=torch.float32).half()
    sample = np.array([0, 17, 40, 63])
    kh = si.fp16_normal((len(sample), pages, B, H, D), 78)
    vh = si.fp16_normal((len(sample), pages, B, H, D), 79)
    for j, s in enumerate(sample):
        ids = torch.from_numpy(bt[s].astype(np.int64)).to(cuda_dev)
        k[0, ids] = dev(kh[j], cuda_dev)
        v[0, ids] = dev(vh[j], cuda_dev)
    q = si.fp16_normal((S, H, D), 80)
    pool = pkv.pf_pool_create(k, v)
    bt_dev, lens_dev = dev(bt, cuda_dev), dev(np.full(S, L, dtype=np.int32), cuda_dev)
    # the oracle over the sampled sequences: contiguous K/V of each, pages in table order
    kc = kh.reshape(len(sample), L, H, D).reshape(-1, H, D)
    vc = vh.reshape(len(sample), L, H, D).reshape(-1, H, D)
    off = np.arange(len(sample) + 1, dtype=np.int64) * L
    ref = oracle_mod.attention_contiguous(q[sample], kc, vc, off, np.full(len(sample), L, dtype=np.int32), w["scale"])
    for split in (0, -1):
        out = torch.empty((S, H, D), dtype=torch.float16, device=cuda_dev)
        ws = pkv.make_workspace(pool, S, H, pages, split)
        pkv.pf_paged_decode_attention(pool, 0, dev(q, cuda_dev), bt_dev, lens_dev, w["scale"], out, split, ws)
        torch.cuda.synchronize()
        assert_close_to_oracle(host(out)[sample], ref, what=f"13b batch 64 split={split}")
    assert pkv.pf_device_status(reset=True) == 0
    del k, v


# q-heads per kv-head from 1 to 16 at both head sizes: 4 and more take the
# tensor-core consumers under the balanced schedule; up to 8 also run under
# fixed chunks (CUDA-core consumers), more than 8 only under the balanced one
@pytest.mark.parametrize("hq,hkv,d", [(8, 1, 64), (6, 2, 128), (5, 5, 128), (16, 2, 64), (24, 8, 128), (32, 8, 64),
                                      (32, 4, 128), (12, 1, 64), (64, 4, 64), (16, 1, 128), (20, 2, 128)])
def test_head_layouts(pkv, cuda_dev, oracle_mod, hq, hkv, d):
    lens = si.uniform_lengths(11, 1, 600, seed=9)
    c = PagedCase(pkv, cuda_dev, lens, hq, hkv, d, 16)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    ref = c.oracle(oracle_mod, scale)
    for split in ((0, -2, 32) if hq // hkv <= 8 else (0,)):
        assert_close_to_oracle(host(c.attention(scale, split=split)), ref, what=f"{hq}/{hkv}x{d} split={split}")


def test_workspace_is_reusable_and_results_repeat(pkv, cuda_dev, oracle_mod):
    lens = si.uniform_lengths(40, 1, 3000, seed=10)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    ws = pkv.make_workspace(c.pool, len(lens), 12, c.bt.shape[1], 64)
    a = host(c.attention(0.125, split=64, ws=ws))
    b = host(c.attention(0.125, split=64, ws=ws))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert_close_to_oracle(a, c.oracle(oracle_mod, 0.125), what="reuse")
    # the scheduler words at the front of the workspace are back at zero
    import torch
    assert np.all(host(ws[:256].view(torch.int32)) == 0)
    for split in (0, -1, 16):   # every schedule leaves them at zero
        ws2 = pkv.make_workspace(c.pool, len(lens), 12, c.bt.shape[1], split)
        a2 = host(c.attention(0.125, split=split, ws=ws2))
        b2 = host(c.attention(0.125, split=split, ws=ws2))
        assert np.array_equal(a2.view(np.uint16), b2.view(np.uint16))
        assert np.all(host(ws2[:256].view(torch.int32)) == 0)


def test_many_short_sequences_and_large_batch(pkv, cuda_dev, oracle_mod):
    lens = si.uniform_lengths(3000, 0, 40, seed=11)
    c = PagedCase(pkv, cuda_dev, lens, 4, 4, 64, 16)
    out = host(c.attention(0.125))
    ref = c.oracle(oracle_mod, 0.125)
    assert np.all(out[lens == 0] == 0)
    assert_close_to_oracle(out, ref, what="3000 short seqs")


def test_bad_block_id_is_flagged(pkv, cuda_dev):
    lens = np.array([40, 40], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    bad = c.bt.copy()
    bad[1, 2] = c.n_blocks + 100
    c.bt_dev = dev(bad, cuda_dev)
    pkv.pf_device_status(reset=True)
    c.attention(0.125)
    assert pkv.pf_device_status(reset=True) == pkv.PF_DEV_BAD_BLOCK_ID


@pytest.mark.parametrize("split", [0, -2])
def test_peaked_softmax_long_contexts(pkv, cuda_dev, oracle_mod, split):
    """4096-token contexts where a few tokens dominate the softmax (q aligned
    with three of the sequence's keys, scaled up), so a handful of weights
    near 1 sit beside thousands near 0: the case where rounding the weights
    would show.  fp16 output within the attention tolerance; fp32 output
    within 1e-5 / 1e-6 of the fp64 oracle on both consumer paths."""
    import torch
    lens = np.array([4096, 4096, 4095, 3001, 2048, 1], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 8, 2, 64, 16)
    rng = np.random.default_rng(55)
    q = c.q.astype(np.float32).copy()
    for s, L in enumerate(lens):
        hot = rng.choice(int(L), size=min(3, int(L)), replace=False)
        for h in range(2):
            # the mean of the hot keys of kv-head h, scaled so its scores stand
            # out by ~10-20 logits over the N(0, 1) background
            keys = np.stack([c.k_host[0, c.bt[s, t // 16], t % 16, h].astype(np.float32) for t in hot])
            d = keys.mean(axis=0)
            q[s, h * 4:(h + 1) * 4] = d / max(np.linalg.norm(d), 1e-3) * 2.2 + 0.1 * q[s, h * 4:(h + 1) * 4]
    q16 = q.astype(np.float16)
    ref = c.oracle(oracle_mod, 1.0, q=q16)
    out16 = host(c.attention(1.0, split=split, q_dev=dev(q16, cuda_dev)))
    assert_close_to_oracle(out16, ref, what=f"peaked fp16 split={split}")
    out32 = host(c.attention(1.0, split=split, out_dtype=torch.float32, q_dev=dev(q16, cuda_dev)))
    assert_close_to_oracle(out32, ref, what=f"peaked fp32 split={split}", **TIGHT)
    assert pkv.pf_device_status(reset=True) == 0


@pytest.mark.parametrize("split", [0, -2])
def test_wait_that_runs_out_reports_and_recovers(pkv, cuda_dev, oracle_mod, split):
    """The bounded waits, made to run out on purpose: the testing hook makes
    block 0 leave one stage of its copy ring unfilled (a barrier that nothing
    completes); every wait gives up after 1 s.  The launch must come back
    with PF_DEV_WAIT_TIMEOUT and a usable context, and the next call on the
    same workspace must match the oracle again (partial records carry their
    launch's stamp, so nothing the timed-out launch left behind is read)."""
    w = si.WORKLOADS["mixed"]
    lens = si.band_lengths(w["bands"])
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16, n_blocks=w["n_blocks"], max_blocks=128)
    ref = c.oracle(oracle_mod, w["scale"])
    ws = pkv.make_workspace(c.pool, len(lens), 12, 128, split)
    assert pkv.pf_device_status(reset=True) == 0
    pkv.pf_test_inject_wait_timeout()
    c.attention(w["scale"], split=split, ws=ws)
    assert pkv.pf_device_status(reset=True) & pkv.PF_DEV_WAIT_TIMEOUT
    for _ in range(2):
        out = host(c.attention(w["scale"], split=split, ws=ws))
        assert_close_to_oracle(out, ref, what=f"after a timeout split={split}")
        assert pkv.pf_device_status(reset=True) == 0
