"""GPT-2 124M shape (12 layers x 12 heads x 64, 32 sequences, prompts of
16..64 tokens then 50 decode steps, pool of 512 tokens per sequence): the
whole demand-paged decode loop on the GPU against the oracle.

Each step every sequence grows by one token: the product allocator appends a
block when the last one is full (and must hand out exactly the ids the
oracle's free-list model does), then per layer the new K/V token is scattered
and decode attention runs over the grown context (two calls on even layers,
the fused pf_decode_step on odd ones).  Attention is checked
against the oracle at several steps; at the end the whole pool must equal the
oracle's scatter of the same tokens, byte for byte, and every block returns to
the free list."""
import numpy as np
import pytest

import synth_inputs as si
from gpu_util import assert_close_to_oracle, dev, host
from oracle.free_list import FreeListModel

pytestmark = pytest.mark.gpu

CHECK_STEPS = (0, 1, 15, 49)


def test_gpt2_shape_demand_paged_decode(pkv, cuda_dev, oracle_mod):
    import torch
    w = si.WORKLOADS["gpt2"]
    S, NL, H, D, B = w["n_seqs"], w["n_layers"], w["n_kv_heads"], w["head_dim"], w["block_size"]
    maxb = w["tokens_per_seq"] // B
    N = S * maxb
    prompts = si.uniform_lengths(S, w["prompt_lo"], w["prompt_hi"])

    alloc = pkv.pf_alloc_create(N, si.SEED_SHUFFLE)
    model = FreeListModel(N, si.SEED_SHUFFLE)
    bt = np.zeros((S, maxb), dtype=np.int32)
    mbt = [[0] * maxb for _ in range(S)]

    k_dev = torch.zeros((NL, N, B, H, D), dtype=torch.float16, device=cuda_dev)
    v_dev = torch.zeros_like(k_dev)
    k_host = np.zeros((NL, N, B, H, D), dtype=np.float16)
    v_host = np.zeros_like(k_host)
    pool = pkv.pf_pool_create(k_dev, v_dev)

    # prompt phase: reserve the prompt's blocks, scatter its tokens per layer
    for s in range(S):
        pkv.pf_seq_reserve(alloc, B, bt[s], 0, int(prompts[s]))
        model.seq_reserve(mbt[s], B, 0, int(prompts[s]))
    assert bt.tolist() == mbt
    seq_idx = np.repeat(np.arange(S), prompts).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in prompts]).astype(np.int32)
    bt_dev = dev(bt, cuda_dev)
    for layer in range(NL):
        kn = si.fp16_normal((len(seq_idx), H, D), 500 + 2 * layer)
        vn = si.fp16_normal((len(seq_idx), H, D), 501 + 2 * layer)
        pkv.pf_write_kv(pool, layer, dev(kn, cuda_dev), dev(vn, cuda_dev), bt_dev,
                        dev(seq_idx, cuda_dev), dev(pos, cuda_dev))
        oracle_mod.scatter(k_host, v_host, layer, kn, vn, bt, seq_idx, pos)

    lens = prompts.copy()
    ws = pkv.make_workspace(pool, S, H, maxb, 0)
    out = torch.empty((S, H, D), dtype=torch.float16, device=cuda_dev)
    all_seq = dev(np.arange(S, dtype=np.int32), cuda_dev)
    for step in range(w["decode_steps"]):
        for s in range(S):
            pkv.pf_seq_reserve(alloc, B, bt[s], int(lens[s]), int(lens[s]) + 1)
            model.seq_reserve(mbt[s], B, int(lens[s]), int(lens[s]) + 1)
        assert bt.tolist() == mbt
        new_pos = lens.copy()            # the new token's position
        lens = lens + 1
        bt_dev = dev(bt, cuda_dev)
        lens_dev = dev(lens, cuda_dev)
        pos_dev = dev(new_pos, cuda_dev)
        rng = np.random.default_rng(10_000 + step)
        for layer in range(NL):
            kn = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
            vn = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
            q = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
            if layer % 2 == 0:   # two calls: scatter, then attention
                pkv.pf_write_kv(pool, layer, dev(kn, cuda_dev), dev(vn, cuda_dev), bt_dev, all_seq, pos_dev)
                pkv.pf_paged_decode_attention(pool, layer, dev(q, cuda_dev), bt_dev, lens_dev, w["scale"], out, 0, ws)
            else:                # the fused decode step
                pkv.pf_decode_step(pool, layer, dev(q, cuda_dev), dev(kn, cuda_dev), dev(vn, cuda_dev), bt_dev,
                                   lens_dev, w["scale"], out, 0, ws, flags=pkv.PF_STEP_OVERLAP_PREVIOUS)
            oracle_mod.scatter(k_host, v_host, layer, kn, vn, bt, np.arange(S, dtype=np.int32), new_pos)
            if step in CHECK_STEPS:
                ref = oracle_mod.attention_paged(q, k_host, v_host, layer, bt, lens, w["scale"])
                assert_close_to_oracle(host(out), ref, what=f"step {step} layer {layer}")
    torch.cuda.synchronize()
    assert np.array_equal(host(k_dev).view(np.uint16), k_host.view(np.uint16))
    assert np.array_equal(host(v_dev).view(np.uint16), v_host.view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0

    # every sequence finishes: all blocks return to the pool
    used = sum(si.pages_for(L, B) for L in lens)
    assert pkv.pf_alloc_free_count(alloc) == N - used
    for s in range(S):
        pkv.pf_seq_release(alloc, B, bt[s], int(lens[s]))
    assert pkv.pf_alloc_free_count(alloc) == N
