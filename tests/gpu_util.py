"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the library through its binding, and compare with the oracle."""
import numpy as np

import synth_inputs as si

# Attention tolerance against the unrounded fp64 oracle on N(0,1) fp16 inputs.
MAX_ABS = 2e-3
MEAN_ABS = 2e-4


def dev(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t):
    return t.detach().cpu().numpy()


def assert_close_to_oracle(out, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    """out: GPU result (fp16 or fp32 array); ref: fp64 oracle."""
    got = np.asarray(out, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= max_abs, f"{what}: max abs err {mx:.3e} > {max_abs:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert mean <= mean_abs, f"{what}: mean abs err {mean:.3e} > {mean_abs:.1e}"
    return mx, mean


class PagedCase:
    """A single-layer (or multi-layer) pool with seeded contents and tables."""

    def __init__(self, pkv, device, lens, n_q_heads, n_kv_heads, head_dim, block_size, n_blocks=None,
                 shuffle_seed=si.SEED_SHUFFLE, n_layers=1, seed=si.SEED_VALUES, max_blocks=None):
        import torch
        self.pkv = pkv
        self.device = device
        self.lens = np.asarray(lens, dtype=np.int32)
        need = sum(si.pages_for(L, block_size) for L in self.lens)
        self.n_blocks = n_blocks or max(need + 8, 16)
        self.bt = si.block_tables(self.lens, block_size, self.n_blocks, shuffle_seed, max_blocks=max_blocks)
        self.Hq, self.Hkv, self.D, self.B, self.L = n_q_heads, n_kv_heads, head_dim, block_size, n_layers
        self.k_host = si.pool(n_layers, self.n_blocks, block_size, n_kv_heads, head_dim, seed)
        self.v_host = si.pool(n_layers, self.n_blocks, block_size, n_kv_heads, head_dim, seed + 1)
        self.q = si.fp16_normal((len(self.lens), n_q_heads, head_dim), seed + 2)
        self.k_dev = dev(self.k_host, device)
        self.v_dev = dev(self.v_host, device)
        self.pool = pkv.pf_pool_create(self.k_dev, self.v_dev)
        self.bt_dev = dev(self.bt, device)
        self.lens_dev = dev(self.lens, device)
        self.q_dev = dev(self.q, device)
        self.torch = torch

    def attention(self, scale, split=0, out_dtype=None, layer=0, ws=None, q_dev=None):
        torch = self.torch
        out_dtype = out_dtype or torch.float16
        n = len(self.lens)
        out = torch.empty((n, self.Hq, self.D), dtype=out_dtype, device=self.device)
        if ws is None:
            ws = self.pkv.make_workspace(self.pool, n, self.Hq, self.bt.shape[1], split)
        self.pkv.pf_paged_decode_attention(self.pool, layer, self.q_dev if q_dev is None else q_dev,
                                           self.bt_dev, self.lens_dev, scale, out, split, ws)
        torch.cuda.synchronize()
        return out

    def oracle(self, oracle_mod, scale, layer=0, q=None):
        return oracle_mod.attention_paged(self.q if q is None else q, self.k_host, self.v_host, layer,
                                          self.bt, self.lens, scale)
