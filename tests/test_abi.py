"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad host-visible arguments before launching anything (no GPU needed)."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"^PF_API\s+[\w\s\*]+?\b(pf_\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("pf_pool_create", "pf_write_kv", "pf_gather_kv", "pf_paged_decode_attention",
                     "pf_alloc_create", "pf_alloc_blocks", "pf_free_blocks"):
        assert required in names


def test_library_exports_every_declared_symbol(pkv):
    lib = ctypes.CDLL(pkv.build())
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_version(pkv):
    assert pkv.pf_abi_version() == 3


def test_pool_bytes(pkv):
    assert pkv.pf_pool_bytes(1, 4096, 16, 12, 64) == 4096 * 16 * 12 * 64 * 2
    assert pkv.pf_pool_bytes(0, 4096, 16, 12, 64) == 0
    assert pkv.pf_pool_bytes(1, 4096, 16, 12, 64, dtype=2) == 0


def _raw_pool(lib, k=0x10000, v=0x20000, L=1, N=64, B=16, H=12, D=64, dtype=1):
    h = ctypes.c_void_p()
    rc = lib.pf_pool_create(ctypes.byref(h), ctypes.c_void_p(k), ctypes.c_void_p(v), L, N, B, H, D, dtype)
    return rc, h


def test_pool_create_validation(pkv):
    lib = pkv.lib()
    assert _raw_pool(lib, k=0)[0] == pkv.PF_ERR_INVALID
    assert _raw_pool(lib, k=0x10008)[0] == pkv.PF_ERR_INVALID          # not 16-byte aligned
    assert "aligned" in pkv.pf_last_error()
    assert _raw_pool(lib, B=8)[0] == pkv.PF_ERR_INVALID
    assert _raw_pool(lib, D=96)[0] == pkv.PF_ERR_INVALID
    assert _raw_pool(lib, dtype=2)[0] == pkv.PF_ERR_INVALID
    assert _raw_pool(lib, N=0)[0] == pkv.PF_ERR_INVALID
    assert _raw_pool(lib, L=4096, N=65536, B=16)[0] == pkv.PF_ERR_INVALID  # >= 2^31 rows
    rc, h = _raw_pool(lib)
    assert rc == pkv.PF_OK and h.value
    assert lib.pf_pool_destroy(h) == pkv.PF_OK


def test_device_calls_reject_bad_arguments_before_launch(pkv):
    lib = pkv.lib()
    rc, pool = _raw_pool(lib)
    assert rc == 0
    P = ctypes.c_void_p
    ok = P(0x30000)
    # null pool / bad layer
    assert lib.pf_write_kv(None, 0, ok, ok, ok, 4, 7, ok, ok, 1, None) == pkv.PF_ERR_INVALID
    assert lib.pf_write_kv(pool, 1, ok, ok, ok, 4, 7, ok, ok, 1, None) == pkv.PF_ERR_INVALID
    assert "layer" in pkv.pf_last_error()
    # unaligned token rows
    assert lib.pf_write_kv(pool, 0, P(0x30002), ok, ok, 4, 7, ok, ok, 1, None) == pkv.PF_ERR_INVALID
    # zero tokens is a no-op
    assert lib.pf_write_kv(pool, 0, None, None, None, 0, 0, None, None, 0, None) == pkv.PF_OK
    assert lib.pf_gather_kv(pool, 0, ok, 7, ok, ok, 4, None, ok, None) == pkv.PF_ERR_INVALID
    assert lib.pf_gather_kv(pool, 0, ok, 7, ok, ok, 0, None, None, None) == pkv.PF_OK
    # attention: q-heads not a multiple of kv-heads, group > 16 (> 8 unless balanced), bad dtype, bad scale, small workspace
    args = lambda hq=12, dt=1, scale=0.125, ws=1 << 20, split=0: (
        pool, 0, ok, ok, 7, ok, 4, hq, ctypes.c_float(scale), ok, dt, split, ok, ws, None)
    assert lib.pf_paged_decode_attention(*args(hq=13)) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_decode_attention(*args(hq=12 * 17)) == pkv.PF_ERR_UNSUPPORTED
    assert lib.pf_paged_decode_attention(*args(hq=12 * 9, split=-1)) == pkv.PF_ERR_UNSUPPORTED
    assert lib.pf_paged_decode_attention(*args(hq=12 * 9, split=64)) == pkv.PF_ERR_UNSUPPORTED
    assert lib.pf_decode_workspace_bytes(pool, 4, 12 * 16, 7, 0) > 0    # 16 rows: balanced schedule only
    assert lib.pf_decode_workspace_bytes(pool, 4, 12 * 16, 7, -1) == 0
    # balanced schedule: records hold the rows of the tensor-core instance
    # (rows rounded up to 1, 4, 8, 12, 16), so sizes step with the instance
    ws = {g: lib.pf_decode_workspace_bytes(pool, 4, 12 * g, 7, 0) for g in range(1, 17)}
    assert ws[2] == ws[3] == ws[4] and ws[5] == ws[8] and ws[9] == ws[12] and ws[13] == ws[16]
    assert ws[1] < ws[4] < ws[8] < ws[12] < ws[16]
    # fixed chunks: CUDA-core instances, records of exactly G rows
    wc = {g: lib.pf_decode_workspace_bytes(pool, 4, 12 * g, 7, 16) for g in range(1, 9)}
    assert all(wc[g] < wc[g + 1] for g in range(1, 8))
    assert lib.pf_paged_decode_attention(*args(dt=3)) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_decode_attention(*args(scale=0.0)) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_decode_attention(*args(scale=float("nan"))) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_decode_attention(*args(ws=16)) == pkv.PF_ERR_INVALID
    assert "workspace" in pkv.pf_last_error()
    assert lib.pf_paged_decode_attention(*args(split=-7)) == pkv.PF_ERR_INVALID
    assert lib.pf_decode_workspace_bytes(pool, 4, 13, 7, 0) == 0
    assert lib.pf_decode_workspace_bytes(pool, 4, 12, 7, 0) > 0
    # decode step: unknown flag bits, null new-token rows
    step = lambda flags=0, kn=ok: (pool, 0, ok, kn, kn, ok, 7, ok, 4, 12, ctypes.c_float(0.125), ok, 1, 0, ok,
                                   1 << 20, flags, None)
    assert lib.pf_decode_step(*step(flags=2)) == pkv.PF_ERR_INVALID
    assert "flags" in pkv.pf_last_error()
    assert lib.pf_decode_step(*step(flags=pkv.PF_STEP_OVERLAP_PREVIOUS | 4)) == pkv.PF_ERR_INVALID
    assert lib.pf_decode_step(*step(kn=None)) == pkv.PF_ERR_INVALID
    # whole-block copies and swapping: null pool / ids / buffer, negative counts; 0 is a no-op
    assert lib.pf_block_image_bytes(pool) == 1 * 2 * 16 * 12 * 64 * 2
    assert lib.pf_block_image_bytes(None) == 0
    assert lib.pf_copy_blocks(None, ok, ok, 1, None) == pkv.PF_ERR_INVALID
    assert lib.pf_copy_blocks(pool, ok, None, 1, None) == pkv.PF_ERR_INVALID
    assert lib.pf_copy_blocks(pool, ok, ok, -1, None) == pkv.PF_ERR_INVALID
    assert lib.pf_copy_blocks(pool, None, None, 0, None) == pkv.PF_OK
    assert lib.pf_swap_out(pool, None, 2, ok, None) == pkv.PF_ERR_INVALID
    assert lib.pf_swap_out(pool, ok, 2, None, None) == pkv.PF_ERR_INVALID
    assert lib.pf_swap_out(pool, ok, 2, P(0x30008), None) == pkv.PF_ERR_INVALID      # not 16-byte aligned
    assert lib.pf_swap_in(pool, ok, ok, -3, None) == pkv.PF_ERR_INVALID
    assert lib.pf_swap_in(pool, None, None, 0, None) == pkv.PF_OK
    # prefill: q-heads not a multiple, group > 16, unaligned q, negative counts; no new token is a no-op
    pre = lambda hq=12, qp=ok, n=4, mx=3, dt=1: (pool, 0, qp, ok, 7, ok, ok, n, mx, hq, ctypes.c_float(0.125), ok,
                                                 dt, None, 0, None)
    assert lib.pf_paged_prefill_attention(*pre(hq=13)) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_prefill_attention(*pre(hq=12 * 17)) == pkv.PF_ERR_UNSUPPORTED
    assert lib.pf_paged_prefill_attention(*pre(qp=P(0x30004))) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_prefill_attention(*pre(n=-1)) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_prefill_attention(*pre(dt=7)) == pkv.PF_ERR_INVALID
    assert lib.pf_paged_prefill_attention(*pre(mx=0)) == pkv.PF_OK
    assert lib.pf_prefill_workspace_bytes(pool, 4, 12, 7, 17) == 0       # 17 rows per kv-head: no workspace path
    assert lib.pf_prefill_workspace_bytes(pool, 4, 12, 7, 16) > 0        # 16 rows on 16-token pages
    assert lib.pf_prefill_workspace_bytes(pool, 4, 12, 0, 2) == 0        # bad table width
    lib.pf_pool_destroy(pool)


def test_workspace_size_grows_with_split(pkv):
    lib = pkv.lib()
    rc, pool = _raw_pool(lib, N=4096)
    never = lib.pf_decode_workspace_bytes(pool, 128, 12, 128, -1)
    auto = lib.pf_decode_workspace_bytes(pool, 128, 12, 128, 0)
    fine = lib.pf_decode_workspace_bytes(pool, 128, 12, 128, 16)
    assert 0 < never < auto < fine
    # balanced spans on the CUDA cores: span records like the default schedule
    assert never < lib.pf_decode_workspace_bytes(pool, 128, 12, 128, -2)
    assert lib.pf_decode_workspace_bytes(pool, 128, 12, 128, -3) == 0
    lib.pf_pool_destroy(pool)
