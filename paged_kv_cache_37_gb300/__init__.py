"""Paged KV-cache decode path for one GB300 (sm_103a).

The product is ``libpagedkv.so`` (C ABI in ``include/pagedkv.h``): the scatter
of new K/V tokens into their page slots, the gather of pages back into
contiguous rows, and single-query paged decode attention with split-K and
grouped heads, plus a host O(1) free-list allocator.  This package is its thin
ctypes binding: the functions keep the C names and take torch CUDA tensors.
Nothing here computes on the CPU and nothing falls back: a call whose library
is missing or whose CUDA launch fails raises.
"""
from ._native import (  # noqa: F401
    PF_DEV_BAD_BLOCK_ID, PF_DEV_BAD_LENGTH, PF_DEV_BAD_POSITION, PF_DEV_WAIT_TIMEOUT, PF_STEP_OVERLAP_PREVIOUS,
    PF_ERR_CUDA, PF_ERR_DOUBLE_FREE, PF_ERR_INVALID, PF_ERR_OOM, PF_ERR_UNSUPPORTED,
    PF_F16, PF_F32, PF_OK,
    Allocator, DoubleFree, OutOfBlocks, PagedKVError, Pool,
    build, lib,
    pf_abi_version, pf_alloc_blocks, pf_alloc_cow, pf_alloc_create, pf_alloc_destroy, pf_alloc_free_count,
    pf_alloc_refcount, pf_alloc_share, pf_block_image_bytes, pf_copy_blocks, pf_seq_fork, pf_swap_in,
    pf_swap_out,
    pf_decode_step, pf_decode_workspace_bytes, pf_decode_workspace_init, pf_device_status, pf_free_blocks,
    pf_test_inject_wait_timeout,
    pf_gather_kv, pf_last_error, pf_paged_decode_attention, pf_paged_decode_attention_noalloc,
    pf_paged_prefill_attention, pf_prefill_workspace_bytes,
    pf_pool_bytes, pf_pool_create,
    pf_pool_destroy, pf_seq_release, pf_seq_reserve, pf_write_kv,
)


def make_prefill_workspace(pool, n_seqs, n_q_heads, max_blocks_per_seq, max_new_tokens, device=None):
    """Allocate (with torch) and initialise a workspace for the decode-kernel
    path of pf_paged_prefill_attention; None when that path does not apply."""
    import torch
    nbytes = pf_prefill_workspace_bytes(pool, n_seqs, n_q_heads, max_blocks_per_seq, max_new_tokens)
    if nbytes == 0:
        return None
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or pool.k_pool.device)
    pf_decode_workspace_init(ws)
    return ws


def make_workspace(pool, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens=0, device=None):
    """Allocate (with torch) and initialise an attention workspace."""
    import torch
    nbytes = pf_decode_workspace_bytes(pool, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or pool.k_pool.device)
    pf_decode_workspace_init(ws)
    return ws
