"""pf_paged_decode_attention_noalloc: decode attention for callers that
cannot allocate device memory (code that may only touch the buffers it is
handed, e.g. an operator inside a framework that owns every allocation).  Its
scratch is a fixed array inside the library.  Through the C ABI, two calls in
a row must give pf_paged_decode_attention's result with a caller workspace
bit for bit: both run the same kernel and schedule on the same inputs, and
nothing the first call (or a call on another batch in between) leaves in the
shared scratch may leak into the second.

This file is named to be collected last, so a run that stops at the first
failure has run every other test first; it also passes on its own in a fresh
process."""
import ctypes

import numpy as np
import pytest

import synth_inputs as si
from gpu_util import PagedCase, dev, host

pytestmark = pytest.mark.gpu


def _call_noalloc(pkv, c, out, scale, split, q_dev):
    lib = pkv.lib()
    import torch
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    n, hq, _ = q_dev.shape
    return lib.pf_paged_decode_attention_noalloc(
        c.pool.handle, 0, P(q_dev), P(c.bt_dev), c.bt.shape[1], P(c.lens_dev), n, hq, ctypes.c_float(scale),
        P(out), pkv.PF_F16 if out.dtype == torch.float16 else pkv.PF_F32, split, stream)


@pytest.mark.parametrize("split", [0, 128])
def test_noalloc_matches_workspace_entry_point_twice(pkv, cuda_dev, split):
    import torch
    w = si.WORKLOADS["mixed"]
    lens = si.band_lengths(w["bands"])
    c = PagedCase(pkv, cuda_dev, lens, 12, 12, 64, 16, n_blocks=w["n_blocks"], max_blocks=128)
    ref = host(c.attention(w["scale"], split=split))
    # another batch (its own pool, lengths and queries)
    other = PagedCase(pkv, cuda_dev, si.uniform_lengths(37, 1, 2048, seed=41), 12, 12, 64, 16, max_blocks=128)
    outs = []
    for i in range(2):
        out = torch.full_like(c.q_dev, float("nan"))
        rc = _call_noalloc(pkv, c, out, w["scale"], split, c.q_dev)
        assert rc == pkv.PF_OK, pkv.pf_last_error()
        torch.cuda.synchronize()
        outs.append(host(out))
        if i == 0:
            # leave another launch's records in the scratch before the second call
            o2 = torch.empty_like(other.q_dev)
            assert _call_noalloc(pkv, other, o2, w["scale"], split, other.q_dev) == pkv.PF_OK
            torch.cuda.synchronize()
    for got in outs:
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    assert pkv.pf_device_status(reset=True) == 0


def test_noalloc_rejects_batches_beyond_its_scratch(pkv, cuda_dev):
    import torch
    lens = np.full(1024, 4096, dtype=np.int32)
    c = PagedCase(pkv, cuda_dev, lens[:2], 40, 40, 128, 16, max_blocks=256)
    # 1024 sequences of 4096 tokens in 16-token chunks need far more than the
    # built-in scratch; the call must refuse before launching anything
    q = torch.zeros((1024, 40, 128), dtype=torch.float16, device=cuda_dev)
    bt = torch.zeros((1024, 256), dtype=torch.int32, device=cuda_dev)
    ln = torch.full((1024,), 16, dtype=torch.int32, device=cuda_dev)
    out = torch.zeros_like(q)
    lib = pkv.lib()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.pf_paged_decode_attention_noalloc(c.pool.handle, 0, P(q), P(bt), 256, P(ln), 1024, 40,
                                               ctypes.c_float(0.1), P(out), pkv.PF_F16, 16, None)
    assert rc == pkv.PF_ERR_INVALID
    assert "built-in scratch" in pkv.pf_last_error()
