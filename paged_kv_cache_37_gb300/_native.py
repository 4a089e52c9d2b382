"""ctypes binding of libpagedkv.so (the C ABI declared in include/pagedkv.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Functions keep the C names; device buffers are torch CUDA tensors
(their data pointers are passed through), block tables and lengths are int32
CUDA tensors, and the stream defaults to torch's current stream.  A failing
call raises PagedKVError carrying the library's status and message.  There is
no fallback: if the library is not built, or a device call fails, the call
raises.
"""
import ctypes
import os

from . import build as _build_mod

PF_OK = 0
PF_ERR_INVALID = 1
PF_ERR_OOM = 2
PF_ERR_DOUBLE_FREE = 3
PF_ERR_CUDA = 4
PF_ERR_UNSUPPORTED = 5

PF_F16 = 1
PF_F32 = 2

PF_DEV_BAD_BLOCK_ID = 1
PF_DEV_BAD_LENGTH = 2
PF_DEV_BAD_POSITION = 4
PF_DEV_WAIT_TIMEOUT = 8
PF_STEP_OVERLAP_PREVIOUS = 1

_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"[status {status}] {message}")
        self.status = status


class OutOfBlocks(PagedKVError):
    pass


class DoubleFree(PagedKVError):
    pass


def build(force=False, verbose=False):
    """Compile the library in-tree for sm_103a (see build.py)."""
    return _build_mod.build(force=force, verbose=verbose)


def lib():
    """Load libpagedkv.so (it must have been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build_mod.LIB
    if not os.path.exists(path):
        raise PagedKVError(PF_ERR_UNSUPPORTED,
                           f"{path} is not built; call paged_kv_cache_37_gb300.build() first")
    L = ctypes.CDLL(path)
    P, I, Z, F, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_uint64
    sigs = {
        "pf_last_error": (ctypes.c_char_p, []),
        "pf_abi_version": (I, []),
        "pf_pool_bytes": (Z, [I, I, I, I, I, I]),
        "pf_pool_create": (I, [ctypes.POINTER(P), P, P, I, I, I, I, I, I]),
        "pf_pool_destroy": (I, [P]),
        "pf_alloc_create": (I, [ctypes.POINTER(P), I, U64]),
        "pf_alloc_destroy": (I, [P]),
        "pf_alloc_blocks": (I, [P, I, P]),
        "pf_free_blocks": (I, [P, P, I]),
        "pf_alloc_free_count": (I, [P]),
        "pf_seq_reserve": (I, [P, I, P, I, I, I]),
        "pf_seq_release": (I, [P, I, P, I]),
        "pf_alloc_share": (I, [P, P, I]),
        "pf_alloc_refcount": (I, [P, ctypes.c_int32]),
        "pf_alloc_cow": (I, [P, P, P, P]),
        "pf_seq_fork": (I, [P, I, P, I, P, I]),
        "pf_block_image_bytes": (Z, [P]),
        "pf_paged_prefill_attention": (I, [P, I, P, P, I, P, P, I, I, I, F, P, I, P, Z, P]),
        "pf_prefill_workspace_bytes": (Z, [P, I, I, I, I]),
        "pf_copy_blocks": (I, [P, P, P, I, P]),
        "pf_swap_out": (I, [P, P, I, P, P]),
        "pf_swap_in": (I, [P, P, P, I, P]),
        "pf_write_kv": (I, [P, I, P, P, P, I, I, P, P, I, P]),
        "pf_gather_kv": (I, [P, I, P, I, P, P, I, P, P, P]),
        "pf_decode_workspace_bytes": (Z, [P, I, I, I, I]),
        "pf_decode_workspace_init": (I, [P, Z, P]),
        "pf_paged_decode_attention": (I, [P, I, P, P, I, P, I, I, F, P, I, I, P, Z, P]),
        "pf_device_status": (I, [ctypes.POINTER(I), I, P]),
        "pf_test_inject_wait_timeout": (I, []),
        "pf_paged_decode_attention_noalloc": (I, [P, I, P, P, I, P, I, I, F, P, I, I, P]),
        "pf_decode_step": (I, [P, I, P, P, P, P, I, P, I, I, F, P, I, I, P, Z, I, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(rc):
    if rc != PF_OK:
        msg = lib().pf_last_error().decode(errors="replace")
        cls = {PF_ERR_OOM: OutOfBlocks, PF_ERR_DOUBLE_FREE: DoubleFree}.get(rc, PagedKVError)
        raise cls(rc, msg)


# --------------------------------------------------------------- helpers

def _dev_ptr(t, name, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise PagedKVError(PF_ERR_INVALID, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PagedKVError(PF_ERR_INVALID, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PagedKVError(PF_ERR_INVALID, f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _host_i32(a, name):
    import numpy as np
    if not isinstance(a, np.ndarray) or a.dtype != np.int32 or not a.flags.c_contiguous:
        raise TypeError(f"{name} must be a C-contiguous numpy int32 array")
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ ABI

def pf_last_error():
    return lib().pf_last_error().decode(errors="replace")


def pf_abi_version():
    return lib().pf_abi_version()


def pf_pool_bytes(n_layers, n_blocks, block_size, n_kv_heads, head_dim, dtype=PF_F16):
    return lib().pf_pool_bytes(n_layers, n_blocks, block_size, n_kv_heads, head_dim, dtype)


class Pool:
    """Handle of a pf_pool over two caller-owned [L, N, B, Hkv, D] fp16 tensors
    (kept referenced here so they outlive the handle)."""

    def __init__(self, handle, k_pool, v_pool):
        self.handle = handle
        self.k_pool = k_pool
        self.v_pool = v_pool
        self.n_layers, self.n_blocks, self.block_size, self.n_kv_heads, self.head_dim = k_pool.shape

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.pf_pool_destroy(self.handle)
            self.handle = None


def pf_pool_create(k_pool, v_pool):
    import torch
    if k_pool.dim() != 5 or k_pool.shape != v_pool.shape:
        raise PagedKVError(PF_ERR_INVALID, "pools must both be [n_layers, n_blocks, block_size, n_kv_heads, head_dim]")
    kp = _dev_ptr(k_pool, "k_pool", torch.float16)
    vp = _dev_ptr(v_pool, "v_pool", torch.float16)
    h = ctypes.c_void_p()
    L, N, B, H, D = k_pool.shape
    _check(lib().pf_pool_create(ctypes.byref(h), kp, vp, L, N, B, H, D, PF_F16))
    return Pool(h, k_pool, v_pool)


def pf_pool_destroy(pool):
    if pool.handle:
        _check(lib().pf_pool_destroy(pool.handle))
        pool.handle = None


class Allocator:
    """Handle of a pf_alloc (host free list)."""

    def __init__(self, handle, n_blocks):
        self.handle = handle
        self.n_blocks = n_blocks

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.pf_alloc_destroy(self.handle)
            self.handle = None


def pf_alloc_create(n_blocks, shuffle_seed=0):
    h = ctypes.c_void_p()
    _check(lib().pf_alloc_create(ctypes.byref(h), n_blocks, shuffle_seed))
    return Allocator(h, n_blocks)


def pf_alloc_destroy(alloc):
    if alloc.handle:
        _check(lib().pf_alloc_destroy(alloc.handle))
        alloc.handle = None


def pf_alloc_blocks(alloc, n):
    import numpy as np
    ids = np.zeros(max(n, 1), dtype=np.int32)
    _check(lib().pf_alloc_blocks(alloc.handle, n, ids.ctypes.data_as(ctypes.c_void_p)))
    return ids[:n]


def pf_free_blocks(alloc, ids):
    import numpy as np
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    _check(lib().pf_free_blocks(alloc.handle, ids.ctypes.data_as(ctypes.c_void_p), ids.size))


def pf_alloc_free_count(alloc):
    return lib().pf_alloc_free_count(alloc.handle)


def pf_seq_reserve(alloc, block_size, table_row, cur_len, new_len):
    """Grow one sequence; table_row is a host int32 numpy row, updated in place."""
    _check(lib().pf_seq_reserve(alloc.handle, block_size, _host_i32(table_row, "table_row"),
                                table_row.size, cur_len, new_len))


def pf_seq_release(alloc, block_size, table_row, length):
    _check(lib().pf_seq_release(alloc.handle, block_size, _host_i32(table_row, "table_row"), length))


def pf_alloc_share(alloc, ids):
    """One more reference on each listed block (a fork's shared prefix)."""
    import numpy as np
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    _check(lib().pf_alloc_share(alloc.handle, ids.ctypes.data_as(ctypes.c_void_p), ids.size))


def pf_alloc_refcount(alloc, block):
    return lib().pf_alloc_refcount(alloc.handle, int(block))


def pf_alloc_cow(alloc, table_row, j):
    """Copy-on-write of table_row[j] (host int32 numpy row, patched in place)
    before a write into that block.  Returns None when the block is the
    writer's own, else (old block, new block) for pf_copy_blocks."""
    import numpy as np
    if not isinstance(table_row, np.ndarray) or table_row.dtype != np.int32:
        raise TypeError("table_row must be a numpy int32 array")
    entry = table_row[j:j + 1]
    src, dst = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().pf_alloc_cow(alloc.handle, entry.ctypes.data_as(ctypes.c_void_p), ctypes.byref(src),
                              ctypes.byref(dst)))
    return None if dst.value < 0 else (src.value, dst.value)


def pf_seq_fork(alloc, block_size, parent_row, length, child_row):
    """child_row[:ceil(length/B)] = parent_row's blocks, shared (host int32 rows)."""
    _check(lib().pf_seq_fork(alloc.handle, block_size, _host_i32(parent_row, "parent_row"), length,
                             _host_i32(child_row, "child_row"), child_row.size))


def pf_block_image_bytes(pool):
    return lib().pf_block_image_bytes(pool.handle)


def pf_copy_blocks(pool, src_ids, dst_ids, stream=None):
    """Block dst_ids[i] := block src_ids[i], every layer, K and V (device int32)."""
    import torch
    n = src_ids.numel()
    if dst_ids.numel() != n:
        raise PagedKVError(PF_ERR_INVALID, "src_ids and dst_ids must have the same length")
    _check(lib().pf_copy_blocks(pool.handle, _dev_ptr(src_ids, "src_ids", torch.int32),
                                _dev_ptr(dst_ids, "dst_ids", torch.int32), n, _stream_ptr(stream)))


def _pinned_ptr(t, name, nbytes):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned() or not t.is_contiguous():
        raise PagedKVError(PF_ERR_INVALID, f"{name} must be a contiguous pinned host tensor")
    if t.numel() * t.element_size() < nbytes:
        raise PagedKVError(PF_ERR_INVALID, f"{name} holds {t.numel() * t.element_size()} bytes, needs {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


def pf_swap_out(pool, ids, host_dst, stream=None):
    """Images of blocks ids (device int32) into the pinned host tensor host_dst."""
    import torch
    n = ids.numel()
    ptr = _pinned_ptr(host_dst, "host_dst", n * pf_block_image_bytes(pool))
    _check(lib().pf_swap_out(pool.handle, _dev_ptr(ids, "ids", torch.int32), n, ptr, _stream_ptr(stream)))


def pf_swap_in(pool, host_src, ids, stream=None):
    """Blocks ids (device int32) take the images in the pinned host tensor host_src."""
    import torch
    n = ids.numel()
    ptr = _pinned_ptr(host_src, "host_src", n * pf_block_image_bytes(pool))
    _check(lib().pf_swap_in(pool.handle, ptr, _dev_ptr(ids, "ids", torch.int32), n, _stream_ptr(stream)))


def pf_prefill_workspace_bytes(pool, n_seqs, n_q_heads, max_blocks_per_seq, max_new_tokens):
    """Workspace bytes of the decode-kernel path of pf_paged_prefill_attention
    (0: that path does not apply, no workspace needed)."""
    return lib().pf_prefill_workspace_bytes(pool.handle, n_seqs, n_q_heads, max_blocks_per_seq, max_new_tokens)


def pf_paged_prefill_attention(pool, layer, q, block_tables, context_lens, cu_q, max_new_tokens, scale, out,
                               workspace=None, stream=None):
    """Causal attention of each sequence's last n_s = cu_q[s+1] - cu_q[s]
    tokens (q rows cu_q[s]..cu_q[s+1]-1) over its context (device tensors).
    With a workspace, short appends run on the decode kernel."""
    import torch
    n = context_lens.numel()
    if block_tables.dim() != 2 or block_tables.shape[0] != n or cu_q.numel() != n + 1:
        raise PagedKVError(PF_ERR_INVALID, "block_tables must be [n_seqs, max_blocks]; cu_q [n_seqs + 1]")
    if tuple(out.shape) != tuple(q.shape):
        raise PagedKVError(PF_ERR_INVALID, "out must have the shape of q")
    out_dtype = {torch.float16: PF_F16, torch.float32: PF_F32}.get(out.dtype)
    if out_dtype is None:
        raise PagedKVError(PF_ERR_INVALID, "out must be float16 or float32")
    _check(lib().pf_paged_prefill_attention(
        pool.handle, layer, _dev_ptr(q, "q", torch.float16), _dev_ptr(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev_ptr(context_lens, "context_lens", torch.int32),
        _dev_ptr(cu_q, "cu_q", torch.int32), n, int(max_new_tokens), q.shape[1], float(scale),
        _dev_ptr(out, "out"), out_dtype,
        None if workspace is None else _dev_ptr(workspace, "workspace"),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream_ptr(stream)))


def pf_write_kv(pool, layer, k_new, v_new, block_tables, seq_idx, pos, stream=None):
    import torch
    n = k_new.shape[0]
    if tuple(k_new.shape) != (n, pool.n_kv_heads, pool.head_dim) or tuple(v_new.shape) != tuple(k_new.shape):
        raise PagedKVError(PF_ERR_INVALID, "k_new / v_new must be [n_tokens, n_kv_heads, head_dim]")
    if seq_idx.numel() != n or pos.numel() != n or block_tables.dim() != 2:
        raise PagedKVError(PF_ERR_INVALID, "seq_idx / pos must have n_tokens entries; block_tables is 2-D")
    _check(lib().pf_write_kv(pool.handle, layer, _dev_ptr(k_new, "k_new", torch.float16),
                             _dev_ptr(v_new, "v_new", torch.float16),
                             _dev_ptr(block_tables, "block_tables", torch.int32),
                             block_tables.shape[0], block_tables.shape[1],
                             _dev_ptr(seq_idx, "seq_idx", torch.int32), _dev_ptr(pos, "pos", torch.int32),
                             n, _stream_ptr(stream)))


def pf_gather_kv(pool, layer, block_tables, context_lens, cu_off, k_out, v_out, stream=None):
    import torch
    n = context_lens.numel()
    if block_tables.dim() != 2 or block_tables.shape[0] != n or cu_off.numel() < n:
        raise PagedKVError(PF_ERR_INVALID, "block_tables must be [n_seqs, max_blocks]; cu_off needs n_seqs entries")
    _check(lib().pf_gather_kv(pool.handle, layer, _dev_ptr(block_tables, "block_tables", torch.int32),
                              block_tables.shape[1], _dev_ptr(context_lens, "context_lens", torch.int32),
                              _dev_ptr(cu_off, "cu_off", torch.int64), n,
                              _dev_ptr(k_out, "k_out", torch.float16), _dev_ptr(v_out, "v_out", torch.float16),
                              _stream_ptr(stream)))


def pf_decode_workspace_bytes(pool, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens=0):
    b = lib().pf_decode_workspace_bytes(pool.handle, n_seqs, n_q_heads, max_blocks_per_seq, split_tokens)
    if b == 0:
        raise PagedKVError(PF_ERR_INVALID, pf_last_error())
    return b


def pf_decode_workspace_init(workspace, stream=None):
    _check(lib().pf_decode_workspace_init(_dev_ptr(workspace, "workspace"),
                                          workspace.numel() * workspace.element_size(), _stream_ptr(stream)))


def pf_paged_decode_attention(pool, layer, q, block_tables, context_lens, scale, out, split_tokens,
                              workspace, stream=None):
    import torch
    n, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != n or context_lens.numel() != n:
        raise PagedKVError(PF_ERR_INVALID, "block_tables must be [n_seqs, max_blocks]; context_lens [n_seqs]")
    if tuple(out.shape) != (n, hq, d):
        raise PagedKVError(PF_ERR_INVALID, "out must have the shape of q")
    if out.dtype == torch.float16:
        out_dtype = PF_F16
    elif out.dtype == torch.float32:
        out_dtype = PF_F32
    else:
        raise PagedKVError(PF_ERR_INVALID, "out must be float16 or float32")
    _check(lib().pf_paged_decode_attention(
        pool.handle, layer, _dev_ptr(q, "q", torch.float16), _dev_ptr(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev_ptr(context_lens, "context_lens", torch.int32), n, hq, float(scale),
        _dev_ptr(out, "out"), out_dtype, split_tokens, _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))


def pf_decode_step(pool, layer, q, k_new, v_new, block_tables, context_lens, scale, out, split_tokens, workspace,
                   flags=0, stream=None):
    """Fused decode step: write each sequence's new K/V row at position
    context_lens[s] - 1, then decode attention over the grown context.
    flags=PF_STEP_OVERLAP_PREVIOUS overlaps the launch with the previous
    kernel on the stream, which must not write context_lens or block_tables."""
    import torch
    n, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != n or context_lens.numel() != n:
        raise PagedKVError(PF_ERR_INVALID, "block_tables must be [n_seqs, max_blocks]; context_lens [n_seqs]")
    if tuple(k_new.shape) != (n, pool.n_kv_heads, d) or tuple(v_new.shape) != tuple(k_new.shape):
        raise PagedKVError(PF_ERR_INVALID, "k_new / v_new must be [n_seqs, n_kv_heads, head_dim]")
    if tuple(out.shape) != (n, hq, d):
        raise PagedKVError(PF_ERR_INVALID, "out must have the shape of q")
    out_dtype = {torch.float16: PF_F16, torch.float32: PF_F32}.get(out.dtype)
    if out_dtype is None:
        raise PagedKVError(PF_ERR_INVALID, "out must be float16 or float32")
    _check(lib().pf_decode_step(
        pool.handle, layer, _dev_ptr(q, "q", torch.float16), _dev_ptr(k_new, "k_new", torch.float16),
        _dev_ptr(v_new, "v_new", torch.float16), _dev_ptr(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev_ptr(context_lens, "context_lens", torch.int32), n, hq, float(scale),
        _dev_ptr(out, "out"), out_dtype, split_tokens, _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), int(flags), _stream_ptr(stream)))


def pf_paged_decode_attention_noalloc(pool, layer, q, block_tables, context_lens, scale, out, split_tokens,
                                      stream=None):
    """pf_paged_decode_attention without a workspace argument: the scratch is
    a fixed array inside the library, for callers that cannot allocate."""
    import torch
    n, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != n or context_lens.numel() != n:
        raise PagedKVError(PF_ERR_INVALID, "block_tables must be [n_seqs, max_blocks]; context_lens [n_seqs]")
    if tuple(out.shape) != (n, hq, d):
        raise PagedKVError(PF_ERR_INVALID, "out must have the shape of q")
    out_dtype = {torch.float16: PF_F16, torch.float32: PF_F32}.get(out.dtype)
    if out_dtype is None:
        raise PagedKVError(PF_ERR_INVALID, "out must be float16 or float32")
    _check(lib().pf_paged_decode_attention_noalloc(
        pool.handle, layer, _dev_ptr(q, "q", torch.float16), _dev_ptr(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev_ptr(context_lens, "context_lens", torch.int32), n, hq, float(scale),
        _dev_ptr(out, "out"), out_dtype, split_tokens, _stream_ptr(stream)))


def pf_test_inject_wait_timeout():
    """Testing hook: block 0 of the next decode-attention launch leaves one
    stage of its copy ring unfilled; the waits for it give up after 1 s (see
    the C header)."""
    _check(lib().pf_test_inject_wait_timeout())


def pf_device_status(reset=False, stream=None):
    st = ctypes.c_int(0)
    _check(lib().pf_device_status(ctypes.byref(st), 1 if reset else 0, _stream_ptr(stream)))
    return st.value
