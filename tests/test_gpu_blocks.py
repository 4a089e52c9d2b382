"""Whole-block copies on the GPU against the oracle, byte for byte:
copy-on-write copies inside the pool (pf_copy_blocks) and swapping blocks to
and from page-locked host memory (pf_swap_out / pf_swap_in), PagedAttention
blog, "Copy-on-Write for Parallel Sampling" and "Preemption and Swapping".
The last test runs forked sequences through decode steps with copy-on-write
and checks attention and the pool against the oracle doing the same."""
import ctypes

import numpy as np
import pytest

import synth_inputs as si
from gpu_util import assert_close_to_oracle, dev, host

pytestmark = pytest.mark.gpu


def _pools(pkv, cuda_dev, n_layers, n_blocks, block_size, heads, dim, seed):
    k = si.pool(n_layers, n_blocks, block_size, heads, dim, seed)
    v = si.pool(n_layers, n_blocks, block_size, heads, dim, seed + 1)
    kd, vd = dev(k, cuda_dev), dev(v, cuda_dev)
    return k, v, kd, vd, pkv.pf_pool_create(kd, vd)


@pytest.mark.parametrize("block_size,heads,dim", [(16, 12, 64), (1, 4, 128), (256, 2, 64)])
def test_copy_blocks_bit_exact(pkv, cuda_dev, oracle_mod, block_size, heads, dim):
    n_layers, n_blocks = 3, 40
    k, v, kd, vd, pool = _pools(pkv, cuda_dev, n_layers, n_blocks, block_size, heads, dim, 70)
    rng = np.random.default_rng(4)
    perm = rng.permutation(n_blocks).astype(np.int32)
    src, dst = perm[:12], perm[12:24]          # destinations are neither sources nor repeated
    pkv.pf_copy_blocks(pool, dev(src, cuda_dev), dev(dst, cuda_dev))
    oracle_mod.copy_blocks(k, v, src, dst)
    assert np.array_equal(host(kd).view(np.uint16), k.view(np.uint16))
    assert np.array_equal(host(vd).view(np.uint16), v.view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0


def test_copy_blocks_bad_ids_are_flagged_and_skipped(pkv, cuda_dev):
    k, v, kd, vd, pool = _pools(pkv, cuda_dev, 2, 16, 16, 4, 64, 71)
    pkv.pf_device_status(reset=True)
    src = np.array([1, 99, 3], dtype=np.int32)
    dst = np.array([5, 6, -2], dtype=np.int32)
    pkv.pf_copy_blocks(pool, dev(src, cuda_dev), dev(dst, cuda_dev))
    assert pkv.pf_device_status(reset=True) & pkv.PF_DEV_BAD_BLOCK_ID
    kh = host(kd)
    assert np.array_equal(kh[:, 5].view(np.uint16), k[:, 1].view(np.uint16))        # the good pair
    untouched = [b for b in range(16) if b != 5]
    assert np.array_equal(kh[:, untouched].view(np.uint16), k[:, untouched].view(np.uint16))


@pytest.mark.parametrize("block_size", [16, 64])
def test_swap_out_and_in_bit_exact(pkv, cuda_dev, oracle_mod, block_size):
    import torch
    n_layers, n_blocks, heads, dim = 2, 48, 12, 64
    k, v, kd, vd, pool = _pools(pkv, cuda_dev, n_layers, n_blocks, block_size, heads, dim, 72)
    ids = np.array([7, 0, 31, 12, 47], dtype=np.int32)
    nbytes = pkv.pf_block_image_bytes(pool)
    assert nbytes == n_layers * 2 * block_size * heads * dim * 2
    buf = torch.zeros(len(ids) * nbytes // 2, dtype=torch.float16).pin_memory()
    pkv.pf_swap_out(pool, dev(ids, cuda_dev), buf)
    torch.cuda.synchronize()
    want = oracle_mod.swap_out(k, v, ids)
    assert np.array_equal(buf.numpy().view(np.uint16), want.view(np.uint16).ravel())
    # back into other physical blocks
    back = np.array([3, 44, 20, 8, 9], dtype=np.int32)
    pkv.pf_swap_in(pool, buf, dev(back, cuda_dev))
    torch.cuda.synchronize()
    oracle_mod.swap_in(k, v, want, back)
    assert np.array_equal(host(kd).view(np.uint16), k.view(np.uint16))
    assert np.array_equal(host(vd).view(np.uint16), v.view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0


def test_swap_rejects_pageable_host_memory(pkv, cuda_dev):
    import torch
    k, v, kd, vd, pool = _pools(pkv, cuda_dev, 1, 8, 16, 4, 64, 73)
    ids = dev(np.array([1], dtype=np.int32), cuda_dev)
    with pytest.raises(pkv.PagedKVError):
        pkv.pf_swap_out(pool, ids, torch.zeros(pkv.pf_block_image_bytes(pool), dtype=torch.uint8))
    # through the C ABI: a pageable numpy buffer is refused before any launch
    buf = np.zeros(pkv.pf_block_image_bytes(pool) + 16, dtype=np.uint8)
    addr = buf.ctypes.data + (-buf.ctypes.data) % 16
    rc = pkv.lib().pf_swap_out(pool.handle, ctypes.c_void_p(ids.data_ptr()), 1, ctypes.c_void_p(addr), None)
    assert rc == pkv.PF_ERR_INVALID and "page-locked" in pkv.pf_last_error()


def test_forked_sequences_decode_with_copy_on_write(pkv, cuda_dev, oracle_mod):
    """A parent prompt, forked into three samples that share its blocks
    (the last one partly filled).  Each decode step first makes the block
    that receives the new token private (pf_alloc_cow + pf_copy_blocks), then
    runs the fused step.  Attention, tables and pool match the oracle doing
    the same on host copies; the parent's blocks keep their contents."""
    import torch
    B, H, D, NL = 16, 4, 64, 2
    N = 64
    MAXB = 8
    alloc = pkv.pf_alloc_create(N, 11)
    model_k = si.pool(NL, N, B, H, D, 80)
    model_v = si.pool(NL, N, B, H, D, 81)
    kd, vd = dev(model_k, cuda_dev), dev(model_v, cuda_dev)
    pool = pkv.pf_pool_create(kd, vd)
    prompt = 37                                     # 3 blocks, the last with 5 tokens
    parent = np.zeros(MAXB, dtype=np.int32)
    pkv.pf_seq_reserve(alloc, B, parent, 0, prompt)
    parent_blocks = parent[:3].copy()
    kids = [np.zeros(MAXB, dtype=np.int32) for _ in range(3)]
    for kid in kids:
        pkv.pf_seq_fork(alloc, B, parent, prompt, kid)
    assert [pkv.pf_alloc_refcount(alloc, b) for b in parent_blocks] == [4, 4, 4]
    parent_k = model_k[:, parent_blocks].copy()
    lens = np.full(3, prompt, dtype=np.int32)
    ws = pkv.make_workspace(pool, 3, 8, MAXB, 0)
    out = torch.empty((3, 8, D), dtype=torch.float16, device=cuda_dev)
    for step in range(20):
        src, dst = [], []
        for s, kid in enumerate(kids):
            L = int(lens[s])
            if L % B == 0:                          # the new token opens a fresh block
                pkv.pf_seq_reserve(alloc, B, kid, L, L + 1)
            else:                                   # it lands in the current last block
                pair = pkv.pf_alloc_cow(alloc, kid, L // B)
                if pair is not None:
                    src.append(pair[0])
                    dst.append(pair[1])
        if src:
            pkv.pf_copy_blocks(pool, dev(np.array(src, np.int32), cuda_dev), dev(np.array(dst, np.int32), cuda_dev))
            oracle_mod.copy_blocks(model_k, model_v, src, dst)
        lens = lens + 1
        bt = np.stack(kids)
        for layer in range(NL):
            rng = np.random.default_rng(900 + 10 * step + layer)
            kn = rng.standard_normal((3, H, D), dtype=np.float32).astype(np.float16)
            vn = rng.standard_normal((3, H, D), dtype=np.float32).astype(np.float16)
            q = rng.standard_normal((3, 8, D), dtype=np.float32).astype(np.float16)
            pkv.pf_decode_step(pool, layer, dev(q, cuda_dev), dev(kn, cuda_dev), dev(vn, cuda_dev), dev(bt, cuda_dev),
                               dev(lens, cuda_dev), 0.125, out, 0, ws)
            oracle_mod.scatter(model_k, model_v, layer, kn, vn, bt, np.arange(3, dtype=np.int32),
                               (lens - 1).astype(np.int32))
            ref = oracle_mod.attention_paged(q, model_k, model_v, layer, bt, lens, 0.125)
            assert_close_to_oracle(host(out), ref, what=f"step {step} layer {layer}")
    torch.cuda.synchronize()
    assert np.array_equal(host(kd).view(np.uint16), model_k.view(np.uint16))
    assert np.array_equal(host(vd).view(np.uint16), model_v.view(np.uint16))
    # nobody wrote into the parent's blocks: the samples diverged on copies
    assert np.array_equal(host(kd)[:, parent_blocks].view(np.uint16), parent_k.view(np.uint16))
    assert pkv.pf_alloc_refcount(alloc, parent_blocks[2]) == 1     # every sample copied the shared tail
    assert pkv.pf_device_status(reset=True) == 0
