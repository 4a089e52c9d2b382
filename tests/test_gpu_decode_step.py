"""pf_decode_step (the new token's K/V written by the attention kernel, then
attention over the grown context) against the oracle's scatter + attention,
and bit-for-bit against the unfused pf_write_kv + pf_paged_decode_attention."""
import numpy as np
import pytest

import synth_inputs as si
from gpu_util import PagedCase, assert_close_to_oracle, dev, host

pytestmark = pytest.mark.gpu


def _run_both(pkv, cuda_dev, oracle_mod, c, scale, split=0, out_f32=False, seed=400):
    """Fused step on case c; unfused on a copy of the same pool; oracle on
    host copies.  Returns (fused out, unfused out, oracle)."""
    import torch
    n = len(c.lens)
    kn = si.fp16_normal((n, c.Hkv, c.D), seed)
    vn = si.fp16_normal((n, c.Hkv, c.D), seed + 1)
    q = si.fp16_normal((n, c.Hq, c.D), seed + 2)
    odt = torch.float32 if out_f32 else torch.float16
    # unfused on a copy of the pool
    k2, v2 = c.k_dev.clone(), c.v_dev.clone()
    pool2 = pkv.pf_pool_create(k2, v2)
    live = np.flatnonzero(c.lens > 0).astype(np.int32)
    pkv.pf_write_kv(pool2, 0, dev(kn[live], cuda_dev), dev(vn[live], cuda_dev), c.bt_dev, dev(live, cuda_dev),
                    dev((c.lens[live] - 1).astype(np.int32), cuda_dev))
    out2 = torch.empty((n, c.Hq, c.D), dtype=odt, device=cuda_dev)
    ws2 = pkv.make_workspace(pool2, n, c.Hq, c.bt.shape[1], split)
    pkv.pf_paged_decode_attention(pool2, 0, dev(q, cuda_dev), c.bt_dev, c.lens_dev, scale, out2, split, ws2)
    # fused
    out = torch.empty((n, c.Hq, c.D), dtype=odt, device=cuda_dev)
    ws = pkv.make_workspace(c.pool, n, c.Hq, c.bt.shape[1], split)
    pkv.pf_decode_step(c.pool, 0, dev(q, cuda_dev), dev(kn, cuda_dev), dev(vn, cuda_dev), c.bt_dev, c.lens_dev,
                       scale, out, split, ws)
    torch.cuda.synchronize()
    # oracle
    kh, vh = c.k_host.copy(), c.v_host.copy()
    oracle_mod.scatter(kh, vh, 0, kn[live], vn[live], c.bt, live, c.lens[live] - 1)
    ref = oracle_mod.attention_paged(q, kh, vh, 0, c.bt, c.lens, scale)
    assert np.array_equal(host(c.k_dev).view(np.uint16), kh.view(np.uint16)), "fused write: K pool differs"
    assert np.array_equal(host(c.v_dev).view(np.uint16), vh.view(np.uint16)), "fused write: V pool differs"
    return host(out), host(out2), ref


@pytest.mark.parametrize("shuffled", [True, False])
@pytest.mark.parametrize("split", [0, 128, -1])
def test_step_mixed(pkv, cuda_dev, oracle_mod, shuffled, split):
    w = si.WORKLOADS["mixed"]
    lens = si.band_lengths(w["bands"])
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16, n_blocks=w["n_blocks"],
                  shuffle_seed=si.SEED_SHUFFLE if shuffled else 0, max_blocks=128)
    fused, unfused, ref = _run_both(pkv, cuda_dev, oracle_mod, c, w["scale"], split)
    assert_close_to_oracle(fused, ref, what=f"step mixed split={split}")
    assert np.array_equal(fused.view(np.uint16), unfused.view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0


@pytest.mark.parametrize("block_size", [1, 16, 64, 256])
def test_step_gqa_block_sizes(pkv, cuda_dev, oracle_mod, block_size):
    w = si.WORKLOADS["gqa"]
    lens = si.uniform_lengths(40, w["len_lo"], w["len_hi"], seed=12)
    c = PagedCase(pkv, cuda_dev, lens, 14, 2, 64, block_size)
    fused, unfused, ref = _run_both(pkv, cuda_dev, oracle_mod, c, w["scale"])
    assert_close_to_oracle(fused, ref, what=f"step gqa B={block_size}")
    assert np.array_equal(fused.view(np.uint16), unfused.view(np.uint16))


@pytest.mark.parametrize("split", [0, -2, 16, -1])
def test_step_edge_lengths_fp32(pkv, cuda_dev, oracle_mod, split):
    lens = np.array([0] + list(range(1, 71)), dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 6, 3, 64, 16)
    fused, unfused, ref = _run_both(pkv, cuda_dev, oracle_mod, c, 0.125, split, out_f32=True)
    assert np.all(fused[0] == 0)
    # fp32 output keeps fp32-accurate weights on every path
    assert_close_to_oracle(fused, ref, what=f"step edges split={split}", max_abs=1e-5, mean_abs=1e-6)
    assert np.array_equal(fused.view(np.uint32), unfused.view(np.uint32))


@pytest.mark.parametrize("hq,hkv,d,b", [(32, 4, 128, 16), (16, 1, 64, 64), (12, 1, 128, 16), (8, 2, 64, 16)])
def test_step_many_rows(pkv, cuda_dev, oracle_mod, hq, hkv, d, b):
    """4 to 16 q-heads per kv-head (the tensor-core consumers), the new row
    substituted in the tile, ragged tails and empty sequences, fp32 out."""
    lens = np.array([0] + list(range(1, 40)) + list(si.uniform_lengths(20, 40, 900, seed=14)), dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, hq, hkv, d, b)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    fused, unfused, ref = _run_both(pkv, cuda_dev, oracle_mod, c, scale, out_f32=True)
    assert np.all(fused[0] == 0)
    assert_close_to_oracle(fused, ref, what=f"step {hq}/{hkv}x{d} B={b}", max_abs=1e-5, mean_abs=1e-6)
    assert np.array_equal(fused.view(np.uint32), unfused.view(np.uint32))
    assert pkv.pf_device_status(reset=True) == 0


def test_step_13b_like(pkv, cuda_dev, oracle_mod):
    w = si.WORKLOADS["13b"]
    lens = np.array([2048, 2000, 17, 1], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 40, 40, 128, 16)
    fused, unfused, ref = _run_both(pkv, cuda_dev, oracle_mod, c, w["scale"])
    assert_close_to_oracle(fused, ref, what="step 13b")
    assert np.array_equal(fused.view(np.uint16), unfused.view(np.uint16))


def test_step_bad_block_id_is_flagged_and_not_written(pkv, cuda_dev):
    import torch
    lens = np.array([40, 40], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    bad = c.bt.copy()
    bad[1, 2] = c.n_blocks + 7      # the page of token 39 of sequence 1
    bt_dev = dev(bad, cuda_dev)
    k0 = host(c.k_dev).copy()
    pkv.pf_device_status(reset=True)
    out = torch.empty((2, 12, 64), dtype=torch.float16, device=cuda_dev)
    ws = pkv.make_workspace(c.pool, 2, 12, c.bt.shape[1], 0)
    kn = dev(si.fp16_normal((2, 12, 64), 50), cuda_dev)
    pkv.pf_decode_step(c.pool, 0, c.q_dev, kn, kn, bt_dev, c.lens_dev, 0.125, out, 0, ws)
    torch.cuda.synchronize()
    assert pkv.pf_device_status(reset=True) & pkv.PF_DEV_BAD_BLOCK_ID
    k1 = host(c.k_dev)
    # sequence 0's new row was written; nothing was written for sequence 1
    changed = np.argwhere(np.any(k1.view(np.uint16) != k0.view(np.uint16), axis=(3, 4)))
    slot0 = (c.bt[0, 39 // 16], 39 % 16)
    assert {(int(b), int(r)) for _, b, r in changed} == {(int(slot0[0]), int(slot0[1]))}


@pytest.mark.parametrize("flags", [0, 1])
def test_back_to_back_steps_read_what_the_previous_step_wrote(pkv, cuda_dev, oracle_mod, flags):
    """Ten steps of two layers, the layers' calls back to back on the stream
    (with flags=PF_STEP_OVERLAP_PREVIOUS the second launch overlaps the
    first), sharing one workspace.  Each step reads the rows the previous
    step wrote; lengths change between steps by host copies; sequence 5 stays
    empty, so its output rows must stay zero."""
    import torch
    S, Hq, Hkv, D = 24, 8, 4, 64
    lens = si.uniform_lengths(S, 1, 300, seed=13)
    lens[5] = 0
    grow = np.ones(S, dtype=np.int32)
    grow[5] = 0
    maxb = -(-(int(lens.max()) + 10) // 16)
    c = PagedCase(pkv, cuda_dev, lens + 10 * grow, Hq, Hkv, D, 16, max_blocks=maxb, n_layers=2)
    kh, vh = c.k_host.copy(), c.v_host.copy()
    ws = pkv.make_workspace(c.pool, S, Hq, maxb, 0)
    outs = [torch.full((S, Hq, D), float("nan"), dtype=torch.float16, device=cuda_dev) for _ in range(2)]
    cur = lens.copy()
    live = np.flatnonzero(grow).astype(np.int32)
    for step in range(10):
        cur = cur + grow
        lens_dev = dev(cur.astype(np.int32), cuda_dev)
        ins = []
        for layer in range(2):
            seed = 600 + 10 * step + 5 * layer
            kn = si.fp16_normal((S, Hkv, D), seed)
            vn = si.fp16_normal((S, Hkv, D), seed + 1)
            q = si.fp16_normal((S, Hq, D), seed + 2)
            ins.append((kn, vn, q, dev(kn, cuda_dev), dev(vn, cuda_dev), dev(q, cuda_dev)))
        for layer in range(2):
            kn, vn, q, kn_d, vn_d, q_d = ins[layer]
            pkv.pf_decode_step(c.pool, layer, q_d, kn_d, vn_d, c.bt_dev, lens_dev, 0.125, outs[layer], 0, ws,
                               flags=flags)
        for layer in range(2):
            kn, vn, q, *_ = ins[layer]
            oracle_mod.scatter(kh, vh, layer, kn[live], vn[live], c.bt, live, (cur[live] - 1).astype(np.int32))
            ref = oracle_mod.attention_paged(q, kh, vh, layer, c.bt, cur, 0.125)
            got = host(outs[layer])
            assert np.all(got[5] == 0)
            assert_close_to_oracle(got, ref, what=f"step {step} layer {layer} flags {flags}")
    assert np.array_equal(host(c.k_dev).view(np.uint16), kh.view(np.uint16))
    assert np.array_equal(host(c.v_dev).view(np.uint16), vh.view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0
