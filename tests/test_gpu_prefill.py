"""pf_paged_prefill_attention (multi-token append: each sequence's last n_s
tokens attend causally over its context) against the oracle, on mixed
lengths, grouped heads, block sizes 1..256 and head_dim 64/128, including
whole prompts and the write-then-attend flow."""
import numpy as np
import pytest

import synth_inputs as si
from gpu_util import MAX_ABS, MEAN_ABS, PagedCase, assert_close_to_oracle, dev, host

pytestmark = pytest.mark.gpu


def _run(pkv, cuda_dev, c, n_new, scale, out_f32=False, seed=500):
    import torch
    cu = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    q = si.fp16_normal((int(cu[-1]), c.Hq, c.D), seed)
    out = torch.full((int(cu[-1]), c.Hq, c.D), float("nan"),
                     dtype=torch.float32 if out_f32 else torch.float16, device=cuda_dev)
    pkv.pf_paged_prefill_attention(c.pool, 0, dev(q, cuda_dev), c.bt_dev, c.lens_dev, dev(cu, cuda_dev),
                                   int(max(n_new.max(), 1)), scale, out)
    torch.cuda.synchronize()
    return q, cu, host(out)


@pytest.mark.parametrize("hq,hkv,d,b", [(12, 12, 64, 16), (14, 2, 64, 1), (14, 2, 64, 256), (8, 4, 128, 64),
                                        (40, 40, 128, 16), (16, 2, 64, 16)])
def test_chunked_append_mixed_lengths(pkv, cuda_dev, oracle_mod, hq, hkv, d, b):
    lens = si.uniform_lengths(24, 1, 700, seed=21)
    rng = np.random.default_rng(5)
    n_new = np.minimum(lens, rng.integers(0, 40, size=lens.size)).astype(np.int32)   # some 0, some all of L
    n_new[3] = lens[3]
    c = PagedCase(pkv, cuda_dev, lens, hq, hkv, d, b)
    q, cu, got = _run(pkv, cuda_dev, c, n_new, 1.0 / np.sqrt(d))
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, np.float32(1.0 / np.sqrt(d)))
    assert_close_to_oracle(got, ref, what=f"prefill {hq}/{hkv}x{d} B={b}")
    assert pkv.pf_device_status(reset=True) == 0


def test_whole_prompts_fp32(pkv, cuda_dev, oracle_mod):
    """Tensor-core products with fp16 weights: fp32 output within the
    attention tolerance (the weights, not the output rounding, set the error)."""
    lens = np.array([1, 2, 15, 16, 17, 33, 100, 64], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 6, 3, 64, 16)
    q, cu, got = _run(pkv, cuda_dev, c, lens.copy(), 0.125, out_f32=True)
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, 0.125)
    assert_close_to_oracle(got, ref, what="whole prompts")
    # the first token of a prompt sees only itself: its output is V0
    v0 = c.v_host[0, c.bt[0, 0], 0].astype(np.float32)          # sequence 0, token 0, all kv-heads
    assert np.array_equal(got[0].reshape(3, 2, 64), np.repeat(v0[:, None, :], 2, axis=1))


@pytest.mark.parametrize("hq,hkv,d,b,lens", [(16, 1, 64, 16, (1000, 700, 333)), (8, 4, 128, 64, (600, 257, 1)),
                                             (12, 12, 64, 1, (129, 64)), (20, 2, 128, 16, (300, 65))])
def test_long_prompts(pkv, cuda_dev, oracle_mod, hq, hkv, d, b, lens):
    """Whole prompts: many 64-row query tiles per kv-head (rows = tokens x
    q-heads), each walking its causal range; up to 16 q-heads per kv-head."""
    lens = np.array(lens, dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, hq, hkv, d, b)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    q, cu, got = _run(pkv, cuda_dev, c, lens.copy(), scale)
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, np.float32(scale))
    assert_close_to_oracle(got, ref, what=f"prompts {hq}/{hkv}x{d} B={b}")
    assert pkv.pf_device_status(reset=True) == 0


def test_write_prompt_then_attend(pkv, cuda_dev, oracle_mod):
    """The prompt's K/V rows go into the pages with pf_write_kv, then its
    queries attend: the pool and the outputs match the oracle doing the same."""
    import torch
    lens = si.uniform_lengths(10, 1, 200, seed=23)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    seq_idx = np.repeat(np.arange(lens.size), lens).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    kn = si.fp16_normal((seq_idx.size, 12, 64), 60)
    vn = si.fp16_normal((seq_idx.size, 12, 64), 61)
    pkv.pf_write_kv(c.pool, 0, dev(kn, cuda_dev), dev(vn, cuda_dev), c.bt_dev, dev(seq_idx, cuda_dev),
                    dev(pos, cuda_dev))
    oracle_mod.scatter(c.k_host, c.v_host, 0, kn, vn, c.bt, seq_idx, pos)
    q, cu, got = _run(pkv, cuda_dev, c, lens.copy(), 0.125)
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, 0.125)
    assert_close_to_oracle(got, ref, what="write then attend")
    assert np.array_equal(host(c.k_dev).view(np.uint16), c.k_host.view(np.uint16))


def test_one_new_token_is_decode_attention(pkv, cuda_dev, oracle_mod):
    lens = si.uniform_lengths(40, 1, 1500, seed=24)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    n_new = np.ones(lens.size, dtype=np.int32)
    q, cu, got = _run(pkv, cuda_dev, c, n_new, 0.125)
    assert_close_to_oracle(got, c.oracle(oracle_mod, 0.125, q=q), what="n_s = 1")


def test_too_many_new_tokens_is_flagged(pkv, cuda_dev):
    import torch
    lens = np.array([5, 20], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 4, 4, 64, 16)
    cu = np.array([0, 9, 11], dtype=np.int32)                # 9 new tokens in a 5-token sequence
    q = dev(si.fp16_normal((11, 4, 64), 70), cuda_dev)
    out = torch.zeros((11, 4, 64), dtype=torch.float16, device=cuda_dev)
    pkv.pf_device_status(reset=True)
    pkv.pf_paged_prefill_attention(c.pool, 0, q, c.bt_dev, c.lens_dev, dev(cu, cuda_dev), 9, 0.125, out)
    torch.cuda.synchronize()
    assert pkv.pf_device_status(reset=True) & pkv.PF_DEV_BAD_LENGTH
    assert np.all(np.isfinite(host(out)))


def _run_ws(pkv, cuda_dev, c, n_new, scale, seed=500):
    """The decode-kernel path: a workspace, at most 16 rows per kv-head (8 on
    pages of fewer than 16 tokens)."""
    import torch
    cu = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    mx = int(max(n_new.max(), 1))
    ws = pkv.make_prefill_workspace(c.pool, len(n_new), c.Hq, c.bt.shape[1], mx)
    assert ws is not None
    q = si.fp16_normal((int(cu[-1]), c.Hq, c.D), seed)
    out = torch.full((int(cu[-1]), c.Hq, c.D), float("nan"), dtype=torch.float16, device=cuda_dev)
    pkv.pf_paged_prefill_attention(c.pool, 0, dev(q, cuda_dev), c.bt_dev, c.lens_dev, dev(cu, cuda_dev), mx, scale,
                                   out, workspace=ws)
    torch.cuda.synchronize()
    return q, cu, host(out)


@pytest.mark.parametrize("hq,hkv,d,b,mx", [(12, 12, 64, 16, 8), (14, 2, 64, 1, 1), (8, 4, 128, 64, 4),
                                           (40, 40, 128, 16, 8), (16, 2, 64, 256, 1), (6, 3, 64, 16, 4),
                                           (12, 12, 64, 16, 16), (8, 4, 128, 64, 8), (4, 1, 64, 16, 4),
                                           (4, 4, 64, 1, 8)])
def test_short_append_on_the_decode_kernel(pkv, cuda_dev, oracle_mod, hq, hkv, d, b, mx):
    lens = si.uniform_lengths(30, 1, 1500, seed=26)
    rng = np.random.default_rng(7)
    n_new = np.minimum(lens, rng.integers(0, mx + 1, size=lens.size)).astype(np.int32)
    n_new[0] = min(mx, lens[0])
    c = PagedCase(pkv, cuda_dev, lens, hq, hkv, d, b)
    scale = 1.0 / np.sqrt(d)
    q, cu, got = _run_ws(pkv, cuda_dev, c, n_new, scale)
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, np.float32(scale))
    assert_close_to_oracle(got, ref, what=f"append on the decode kernel {hq}/{hkv}x{d} B={b}")
    # the same inputs through the kernel without a workspace
    q2, cu2, got2 = _run(pkv, cuda_dev, c, n_new, scale)
    assert_close_to_oracle(got2, ref, what="append on the prefill kernel")
    assert pkv.pf_device_status(reset=True) == 0


def test_one_new_token_on_the_decode_kernel_is_decode_bit_for_bit(pkv, cuda_dev):
    lens = si.uniform_lengths(50, 1, 2000, seed=27)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    q, cu, got = _run_ws(pkv, cuda_dev, c, np.ones(lens.size, dtype=np.int32), 0.125)
    dec = host(c.attention(0.125, q_dev=dev(q, cuda_dev)))
    assert np.array_equal(got.view(np.uint16), dec.view(np.uint16))


def test_short_append_large_batch(pkv, cuda_dev, oracle_mod):
    """More than 1024 sequences: the kernel runs in two launches, and the
    query rows are absolute in cu_q."""
    lens = si.uniform_lengths(1500, 1, 120, seed=28)
    rng = np.random.default_rng(8)
    n_new = np.minimum(lens, rng.integers(0, 5, size=lens.size)).astype(np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 4, 4, 64, 16)
    q, cu, got = _run_ws(pkv, cuda_dev, c, n_new, 0.125)
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, 0.125)
    assert_close_to_oracle(got, ref, what="append, 1500 sequences")


@pytest.mark.parametrize("d,b", [(64, 16), (128, 64)])
def test_prompt_with_growing_scores_rescales(pkv, cuda_dev, oracle_mod, d, b):
    """Keys that grow along the prompt in the queries' direction raise every
    row's running maximum by far more than 2^8 from one K/V tile to the next,
    so the accumulated output in tensor memory is rescaled at nearly every
    tile; the result still matches the oracle."""
    import torch
    lens = np.array([900, 513, 130], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 4, 2, d, b)
    u = np.full(d, 1.0 / np.sqrt(d), dtype=np.float32)          # unit direction
    for s, L in enumerate(lens):
        for t in range(L):
            blk, row = c.bt[s, t // b], t % b
            k = c.k_host[0, blk, row].astype(np.float32) * 0.1 + u * (t / 4.0)
            c.k_host[0, blk, row] = k.astype(np.float16)
    c.k_dev.copy_(torch.from_numpy(c.k_host))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = (si.fp16_normal((int(cu[-1]), 4, d), 501).astype(np.float32) * 0.1 + 4.0 * u).astype(np.float16)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    out = torch.full((int(cu[-1]), 4, d), float("nan"), dtype=torch.float16, device=cuda_dev)
    pkv.pf_paged_prefill_attention(c.pool, 0, dev(q, cuda_dev), c.bt_dev, c.lens_dev, dev(cu, cuda_dev),
                                   int(lens.max()), scale, out)
    torch.cuda.synchronize()
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, np.float32(scale))
    assert_close_to_oracle(host(out), ref, what=f"growing scores d={d}")
    assert pkv.pf_device_status(reset=True) == 0


def test_prompt_kernel_flags_a_bad_block_id(pkv, cuda_dev, oracle_mod):
    """A block id outside the pool in one prompt's table (on the tcgen05
    kernel: 128+ rows per kv-head) is flagged and read as page 0: that
    prompt's output stays finite, and the other prompt still matches the
    oracle."""
    import torch
    lens = np.array([300, 200], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 4, 2, 64, 16)
    bt_bad = c.bt.copy()
    bt_bad[0, 3] = c.n_blocks + 7
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = si.fp16_normal((int(cu[-1]), 4, 64), 502)
    out = torch.full((int(cu[-1]), 4, 64), float("nan"), dtype=torch.float16, device=cuda_dev)
    pkv.pf_device_status(reset=True)
    pkv.pf_paged_prefill_attention(c.pool, 0, dev(q, cuda_dev), dev(bt_bad, cuda_dev), c.lens_dev, dev(cu, cuda_dev),
                                   int(lens.max()), 0.125, out)
    torch.cuda.synchronize()
    assert pkv.pf_device_status(reset=True) & pkv.PF_DEV_BAD_BLOCK_ID
    got = host(out)
    assert np.all(np.isfinite(got))
    ref = oracle_mod.prefill_attention(q, c.k_host, c.v_host, 0, c.bt, lens, cu, 0.125)
    assert_close_to_oracle(got[cu[1]:], ref[cu[1]:], what="the other prompt")


def test_prompt_kernel_flags_too_many_new_tokens(pkv, cuda_dev):
    """More new tokens than a sequence holds, on the tcgen05 kernel: flagged,
    clamped, and every output finite."""
    import torch
    lens = np.array([100, 300], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 4, 4, 64, 16)
    cu = np.array([0, 150, 450], dtype=np.int32)            # 150 new tokens in a 100-token sequence
    q = dev(si.fp16_normal((450, 4, 64), 503), cuda_dev)
    out = torch.zeros((450, 4, 64), dtype=torch.float16, device=cuda_dev)
    pkv.pf_device_status(reset=True)
    pkv.pf_paged_prefill_attention(c.pool, 0, q, c.bt_dev, c.lens_dev, dev(cu, cuda_dev), 300, 0.125, out)
    torch.cuda.synchronize()
    assert pkv.pf_device_status(reset=True) & pkv.PF_DEV_BAD_LENGTH
    assert np.all(np.isfinite(host(out)))
