"""Scatter (pf_write_kv) and gather (pf_gather_kv) on the GPU against the
oracle: bit-exact, every byte of the pool / output compared."""
import numpy as np
import pytest

import synth_inputs as si
from gpu_util import PagedCase, dev, host

pytestmark = pytest.mark.gpu


def _tokens_for_write(lens, seed, per_seq=1):
    """Distinct (seq, pos) pairs: the last token of each sequence plus
    per_seq - 1 other positions."""
    rng = np.random.default_rng(seed)
    si_, ps = [], []
    for s, L in enumerate(lens):
        if L <= 0:
            continue
        pos = {int(L) - 1}
        while len(pos) < min(per_seq, int(L)):
            pos.add(int(rng.integers(0, L)))
        for t in sorted(pos):
            si_.append(s)
            ps.append(t)
    return np.array(si_, dtype=np.int32), np.array(ps, dtype=np.int32)


@pytest.mark.parametrize("name,shuffled,per_seq", [("tiny", True, 1), ("tiny", False, 5),
                                                   ("mixed", True, 1), ("mixed", False, 3)])
def test_write_kv_bit_exact(pkv, cuda_dev, oracle_mod, name, shuffled, per_seq):
    w = si.WORKLOADS[name]
    if name == "tiny":
        lens = si.uniform_lengths(w["n_seqs"], w["len_lo"], w["len_hi"])
        n_blocks = w["n_blocks"]
    else:
        lens = si.band_lengths(w["bands"])
        n_blocks = w["n_blocks"]
    c = PagedCase(pkv, cuda_dev, lens, w["n_q_heads"], w["n_kv_heads"], w["head_dim"], w["block_size"],
                  n_blocks=n_blocks, shuffle_seed=si.SEED_SHUFFLE if shuffled else 0)
    seq_idx, pos = _tokens_for_write(lens, 3, per_seq)
    kn = si.fp16_normal((len(seq_idx), c.Hkv, c.D), 101)
    vn = si.fp16_normal((len(seq_idx), c.Hkv, c.D), 102)
    pkv.pf_write_kv(c.pool, 0, dev(kn, cuda_dev), dev(vn, cuda_dev), c.bt_dev,
                    dev(seq_idx, cuda_dev), dev(pos, cuda_dev))
    kref, vref = c.k_host.copy(), c.v_host.copy()
    oracle_mod.scatter(kref, vref, 0, kn, vn, c.bt, seq_idx, pos)
    assert np.array_equal(host(c.k_dev).view(np.uint16), kref.view(np.uint16))
    assert np.array_equal(host(c.v_dev).view(np.uint16), vref.view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0


def test_write_kv_multilayer_touches_only_its_layer(pkv, cuda_dev, oracle_mod):
    lens = np.array([5, 17, 33], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16, n_layers=3)
    seq_idx, pos = _tokens_for_write(lens, 4, 4)
    kn = si.fp16_normal((len(seq_idx), 12, 64), 103)
    vn = si.fp16_normal((len(seq_idx), 12, 64), 104)
    pkv.pf_write_kv(c.pool, 1, dev(kn, cuda_dev), dev(vn, cuda_dev), c.bt_dev,
                    dev(seq_idx, cuda_dev), dev(pos, cuda_dev))
    kref, vref = c.k_host.copy(), c.v_host.copy()
    oracle_mod.scatter(kref, vref, 1, kn, vn, c.bt, seq_idx, pos)
    assert np.array_equal(host(c.k_dev).view(np.uint16), kref.view(np.uint16))
    assert np.array_equal(host(c.v_dev).view(np.uint16), vref.view(np.uint16))


@pytest.mark.parametrize("block_size", [1, 16, 64, 256])
@pytest.mark.parametrize("head_dim,hkv", [(64, 12), (128, 2)])
def test_gather_bit_exact(pkv, cuda_dev, oracle_mod, block_size, head_dim, hkv):
    lens = np.array([0, 1, 15, 16, 17, 64, 65, 255, 256, 257, 700], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, hkv, hkv, head_dim, block_size, n_layers=2)
    off = si.cu_offsets(lens)
    T = int(off[-1])
    for layer in (0, 1):
        k_out = pkv_empty(cuda_dev, (T + 3, hkv, head_dim))
        v_out = pkv_empty(cuda_dev, (T + 3, hkv, head_dim))
        pkv.pf_gather_kv(c.pool, layer, c.bt_dev, c.lens_dev, dev(off[:-1], cuda_dev), k_out, v_out)
        kg, vg = oracle_mod.gather(c.k_host, c.v_host, layer, c.bt, lens, off)
        got_k, got_v = host(k_out), host(v_out)
        assert np.array_equal(got_k[:T].view(np.uint16), kg.view(np.uint16))
        assert np.array_equal(got_v[:T].view(np.uint16), vg.view(np.uint16))
        # rows past the packed output are untouched (canary)
        assert np.all(got_k[T:].view(np.uint16) == 0x7E00) and np.all(got_v[T:].view(np.uint16) == 0x7E00)


def pkv_empty(device, shape):
    import torch
    t = torch.empty(shape, dtype=torch.float16, device=device)
    t.view(torch.int16).fill_(0x7E00)   # NaN canary
    return t


@pytest.mark.parametrize("shuffled", [True, False])
def test_gather_then_scatter_roundtrip_mixed(pkv, cuda_dev, oracle_mod, shuffled):
    lens, bt = si.mixed_workload(shuffled)
    w = si.WORKLOADS["mixed"]
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16, n_blocks=w["n_blocks"],
                  shuffle_seed=si.SEED_SHUFFLE if shuffled else 0, max_blocks=bt.shape[1])
    assert np.array_equal(c.bt, bt)
    off = si.cu_offsets(lens)
    T = int(off[-1])
    k_out = pkv_empty(cuda_dev, (T, 12, 64))
    v_out = pkv_empty(cuda_dev, (T, 12, 64))
    pkv.pf_gather_kv(c.pool, 0, c.bt_dev, c.lens_dev, dev(off[:-1], cuda_dev), k_out, v_out)
    kg, vg = oracle_mod.gather(c.k_host, c.v_host, 0, c.bt, lens, off)
    assert np.array_equal(host(k_out).view(np.uint16), kg.view(np.uint16))
    assert np.array_equal(host(v_out).view(np.uint16), vg.view(np.uint16))
    # scatter the gathered rows into a fresh pool with the same tables: the
    # used slots come back bit for bit
    import torch
    kp2 = torch.zeros_like(c.k_dev)
    vp2 = torch.zeros_like(c.v_dev)
    pool2 = pkv.pf_pool_create(kp2, vp2)
    seq_idx = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    pkv.pf_write_kv(pool2, 0, k_out, v_out, c.bt_dev, dev(seq_idx, cuda_dev), dev(pos, cuda_dev))
    k2 = host(kp2)
    kref = np.zeros_like(c.k_host)
    vref = np.zeros_like(c.v_host)
    oracle_mod.scatter(kref, vref, 0, kg, vg, c.bt, seq_idx, pos)
    assert np.array_equal(k2.view(np.uint16), kref.view(np.uint16))
    assert np.array_equal(host(vp2).view(np.uint16), vref.view(np.uint16))


def test_bad_device_data_is_flagged_not_faulted(pkv, cuda_dev):
    """Out-of-range block ids, positions and lengths are skipped by the
    kernels' own checks and reported through the device status word."""
    lens = np.array([20, 40], dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16)
    pkv.pf_device_status(reset=True)
    kn = dev(si.fp16_normal((2, 12, 64), 105), cuda_dev)
    vn = dev(si.fp16_normal((2, 12, 64), 106), cuda_dev)
    # position past the table row
    pkv.pf_write_kv(c.pool, 0, kn, vn, c.bt_dev, dev(np.array([0, 1], np.int32), cuda_dev),
                    dev(np.array([5, 16 * c.bt.shape[1] + 3], np.int32), cuda_dev))
    assert pkv.pf_device_status(reset=True) == pkv.PF_DEV_BAD_POSITION
    # block id outside the pool
    bad_bt = c.bt.copy()
    bad_bt[1, 1] = c.n_blocks + 5
    bad_bt_dev = dev(bad_bt, cuda_dev)
    pkv.pf_write_kv(c.pool, 0, kn, vn, bad_bt_dev, dev(np.array([0, 1], np.int32), cuda_dev),
                    dev(np.array([5, 20], np.int32), cuda_dev))
    assert pkv.pf_device_status(reset=True) == pkv.PF_DEV_BAD_BLOCK_ID
    off = si.cu_offsets(lens)
    k_out = pkv_empty(cuda_dev, (int(off[-1]), 12, 64))
    v_out = pkv_empty(cuda_dev, (int(off[-1]), 12, 64))
    pkv.pf_gather_kv(c.pool, 0, bad_bt_dev, c.lens_dev, dev(off[:-1], cuda_dev), k_out, v_out)
    assert pkv.pf_device_status(reset=True) == pkv.PF_DEV_BAD_BLOCK_ID
    # a length beyond the table is clamped and flagged
    big = dev(np.array([20, 16 * c.bt.shape[1] + 1], np.int32), cuda_dev)
    k_out2 = pkv_empty(cuda_dev, (20 + 16 * c.bt.shape[1], 12, 64))
    v_out2 = pkv_empty(cuda_dev, (20 + 16 * c.bt.shape[1], 12, 64))
    pkv.pf_gather_kv(c.pool, 0, c.bt_dev, big, dev(np.array([0, 20], np.int64), cuda_dev), k_out2, v_out2)
    assert pkv.pf_device_status(reset=True) & pkv.PF_DEV_BAD_LENGTH
