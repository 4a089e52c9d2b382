"""fp64 CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  It shares
no code with the CUDA path and imports nothing from the product package.

The arithmetic lives in ``pagedkv_oracle.c`` (plain C99, fp64, compiled with
floating-point contraction off so x86 and Arm hosts give identical results);
this module only builds it and marshals numpy arrays.  fp16 arrays are passed
as their raw 16-bit patterns and decoded inside the C code.

``free_list.py`` is the plain-Python model of the host block allocator.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pagedkv_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

_lib = None


def build(force=False):
    """Compile the C oracle into ``liboracle.so`` next to its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(LIB)
    P = ctypes.c_void_p
    i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    sig = {
        "or_half_to_double": (f64, [ctypes.c_uint16]),
        "or_half_to_double_array": (None, [P, P, i64]),
        "or_blocks_needed": (i64, [i64, i64]),
        "or_tail_waste": (i64, [i64, i64]),
        "or_slot": (i64, [P, i64, i64]),
        "or_scatter": (None, [P, P, i32, i32, i32, i32, i32, P, P, P, i32, P, P, i32]),
        "or_gather": (None, [P, P, i32, i32, i32, i32, i32, P, i32, P, P, i32, P, P]),
        "or_copy_blocks": (None, [P, P, i32, i32, i64, P, P, i32]),
        "or_swap_out": (None, [P, P, i32, i32, i64, P, i32, P]),
        "or_swap_in": (None, [P, P, i32, i32, i64, P, P, i32]),
        "or_attention_contiguous": (i32, [P, P, P, P, P, i32, i32, i32, i32, f32, P]),
        "or_attention_paged": (i32, [P, P, P, i32, i32, i32, i32, i32, P, i32, P, i32, i32, f32, P]),
        "or_attention_partial": (None, [P, P, P, i64, i64, i32, f32, i64, i64, P, P, P]),
        "or_lse_merge": (None, [P, P, P, i32, i32, P]),
        "or_kv_bytes_per_token": (i64, [i64, i64, i64, i64]),
        "or_naive_reserved_bytes": (i64, [i64, i64, i64]),
        "or_paged_blocks": (i64, [P, i32, i64]),
        "or_paged_reserved_bytes": (i64, [P, i32, i64, i64]),
        "or_internal_fragmentation_tokens": (i64, [P, i32, i64]),
        "or_paged_utilization": (f64, [P, i32, i64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    """Raw fp16 bit patterns of an fp16 (or uint16) array, C-contiguous."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 bits, got {a.dtype}")


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


# ---------------------------------------------------------------- scalars

def half_to_double(bits):
    return _load().or_half_to_double(int(bits) & 0xFFFF)


def half_array_to_double(a):
    a = _u16(a)
    out = np.empty(a.shape, dtype=np.float64)
    _load().or_half_to_double_array(_ptr(a), _ptr(out), a.size)
    return out


def blocks_needed(length, block_size):
    return _load().or_blocks_needed(int(length), int(block_size))


def tail_waste(length, block_size):
    return _load().or_tail_waste(int(length), int(block_size))


def slot(table_row, block_size, t):
    row = _i32(table_row)
    return _load().or_slot(_ptr(row), int(block_size), int(t))


# ------------------------------------------------------ scatter / gather

def scatter(k_pool, v_pool, layer, k_new, v_new, block_tables, seq_idx, pos):
    """In-place scatter into host pools [n_layers, N, B, H, D] (fp16)."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    _, n_blocks, block_size, n_heads, head_dim = k_pool.shape
    kp, vp = _u16(k_pool), _u16(v_pool)
    kn, vn = _u16(k_new), _u16(v_new)
    bt, si, ps = _i32(block_tables), _i32(seq_idx), _i32(pos)
    _load().or_scatter(_ptr(kp), _ptr(vp), n_blocks, block_size, n_heads, head_dim,
                       layer, _ptr(kn), _ptr(vn), _ptr(bt), bt.shape[1],
                       _ptr(si), _ptr(ps), si.size)


def gather(k_pool, v_pool, layer, block_tables, context_lens, cu_off):
    _, n_blocks, block_size, n_heads, head_dim = k_pool.shape
    kp, vp = _u16(k_pool), _u16(v_pool)
    bt, lens, off = _i32(block_tables), _i32(context_lens), _i64(cu_off)
    total = int(off[-1]) if off.size else 0
    k_out = np.zeros((total, n_heads, head_dim), dtype=np.uint16)
    v_out = np.zeros((total, n_heads, head_dim), dtype=np.uint16)
    _load().or_gather(_ptr(kp), _ptr(vp), n_blocks, block_size, n_heads, head_dim,
                      layer, _ptr(bt), bt.shape[1], _ptr(lens), _ptr(off), lens.size,
                      _ptr(k_out), _ptr(v_out))
    return k_out.view(np.float16), v_out.view(np.float16)


# ------------------------------------------------- block copies, swap

def copy_blocks(k_pool, v_pool, src, dst):
    """In place: block dst[i] := block src[i] in every layer of host pools
    [n_layers, N, B, H, D] (fp16)."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    n_layers, n_blocks = k_pool.shape[:2]
    block_elems = int(np.prod(k_pool.shape[2:]))
    s, d = _i32(src), _i32(dst)
    _load().or_copy_blocks(_ptr(_u16(k_pool)), _ptr(_u16(v_pool)), n_layers, n_blocks, block_elems,
                           _ptr(s), _ptr(d), s.size)


def swap_out(k_pool, v_pool, ids):
    """Host images [n, n_layers, 2, B, H, D] (fp16) of blocks ids."""
    n_layers, n_blocks = k_pool.shape[:2]
    block_elems = int(np.prod(k_pool.shape[2:]))
    i = _i32(ids)
    images = np.zeros((i.size, n_layers, 2) + tuple(k_pool.shape[2:]), dtype=np.uint16)
    _load().or_swap_out(_ptr(_u16(k_pool)), _ptr(_u16(v_pool)), n_layers, n_blocks, block_elems,
                        _ptr(i), i.size, _ptr(images))
    return images.view(np.float16)


def swap_in(k_pool, v_pool, images, ids):
    """In place: blocks ids take the contents of host images [n, n_layers, 2, ...]."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    n_layers, n_blocks = k_pool.shape[:2]
    block_elems = int(np.prod(k_pool.shape[2:]))
    i = _i32(ids)
    img = _u16(images)
    _load().or_swap_in(_ptr(_u16(k_pool)), _ptr(_u16(v_pool)), n_layers, n_blocks, block_elems,
                       _ptr(img), _ptr(i), i.size)


# ------------------------------------------------------------ attention

def attention_contiguous(q, kc, vc, cu_off, context_lens, scale):
    """q [S, Hq, D] fp16; kc/vc [T, Hkv, D] fp16 packed rows -> fp64 [S, Hq, D]."""
    qq, kk, vv = _u16(q), _u16(kc), _u16(vc)
    off, lens = _i64(cu_off), _i32(context_lens)
    n_seqs, n_q_heads, head_dim = qq.shape
    n_kv_heads = kk.shape[1]
    out = np.zeros((n_seqs, n_q_heads, head_dim), dtype=np.float64)
    rc = _load().or_attention_contiguous(_ptr(qq), _ptr(kk), _ptr(vv), _ptr(off), _ptr(lens),
                                         n_seqs, n_q_heads, n_kv_heads, head_dim,
                                         float(scale), _ptr(out))
    if rc:
        raise ValueError("or_attention_contiguous: bad arguments")
    return out


def attention_paged(q, k_pool, v_pool, layer, block_tables, context_lens, scale):
    """q [S, Hq, D] fp16; pools [n_layers, N, B, Hkv, D] fp16 -> fp64 [S, Hq, D]."""
    qq, kp, vp = _u16(q), _u16(k_pool), _u16(v_pool)
    bt, lens = _i32(block_tables), _i32(context_lens)
    _, n_blocks, block_size, n_kv_heads, head_dim = kp.shape
    n_seqs, n_q_heads, _ = qq.shape
    out = np.zeros((n_seqs, n_q_heads, head_dim), dtype=np.float64)
    rc = _load().or_attention_paged(_ptr(qq), _ptr(kp), _ptr(vp), n_blocks, block_size,
                                    n_kv_heads, head_dim, layer, _ptr(bt), bt.shape[1],
                                    _ptr(lens), n_seqs, n_q_heads, float(scale), _ptr(out))
    if rc:
        raise ValueError("or_attention_paged: bad arguments")
    return out


def prefill_attention(q, k_pool, v_pool, layer, block_tables, context_lens, cu_q, scale):
    """Multi-token append (a prompt, or a chunk of one, written into the
    sequence's last pages: PagedAttention blog, "Architecture", append then
    attend).  Sequence s's new tokens are q rows cu_q[s] .. cu_q[s + 1] - 1,
    its last n_s = cu_q[s + 1] - cu_q[s] positions of L_s = context_lens[s];
    the query at position p = L_s - n_s + i attends causally to tokens
    0 .. p, which is single-query attention over those p + 1 tokens.
    q [T_q, Hq, D] fp16 -> fp64 [T_q, Hq, D]."""
    bt = _i32(block_tables)
    lens = _i32(context_lens)
    cu = np.asarray(cu_q, dtype=np.int64)
    rows, qlen = [], []
    for s in range(lens.size):
        n = int(cu[s + 1] - cu[s])
        for i in range(n):
            rows.append(s)
            qlen.append(int(lens[s]) - n + i + 1)
    if not rows:
        return np.zeros((0,) + tuple(q.shape[1:]), dtype=np.float64)
    return attention_paged(q, k_pool, v_pool, layer, bt[np.asarray(rows)], np.asarray(qlen, dtype=np.int32), scale)


def attention_partial(q_row, k, v, head, t0, t1, scale):
    """Partial (m, l, acc) of one query row over tokens [t0, t1) of a contiguous
    sequence k/v [L, Hkv, D]."""
    qq, kk, vv = _u16(q_row), _u16(k), _u16(v)
    _, n_kv_heads, head_dim = kk.shape
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(head_dim)
    _load().or_attention_partial(_ptr(qq), _ptr(kk), _ptr(vv), n_kv_heads * head_dim,
                                 head * head_dim, head_dim, float(scale), int(t0), int(t1),
                                 _ptr(m), _ptr(l), _ptr(acc))
    return m[0], l[0], acc


def lse_merge(ms, ls, accs):
    ms, ls = np.ascontiguousarray(ms, dtype=np.float64), np.ascontiguousarray(ls, dtype=np.float64)
    accs = np.ascontiguousarray(accs, dtype=np.float64)
    n, head_dim = accs.shape
    out = np.zeros(head_dim)
    _load().or_lse_merge(_ptr(ms), _ptr(ls), _ptr(accs), n, head_dim, _ptr(out))
    return out


# ---------------------------------------------------- memory accounting

def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, dtype_bytes):
    return _load().or_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, dtype_bytes)


def naive_reserved_bytes(n_seqs, max_seq_len, bytes_per_token):
    return _load().or_naive_reserved_bytes(n_seqs, max_seq_len, bytes_per_token)


def paged_blocks(lens, block_size):
    a = _i32(lens)
    return _load().or_paged_blocks(_ptr(a), a.size, block_size)


def paged_reserved_bytes(lens, block_size, bytes_per_token):
    a = _i32(lens)
    return _load().or_paged_reserved_bytes(_ptr(a), a.size, block_size, bytes_per_token)


def internal_fragmentation_tokens(lens, block_size):
    a = _i32(lens)
    return _load().or_internal_fragmentation_tokens(_ptr(a), a.size, block_size)


def paged_utilization(lens, block_size):
    a = _i32(lens)
    return _load().or_paged_utilization(_ptr(a), a.size, block_size)
