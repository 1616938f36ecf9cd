"""fp64 CPU oracle for paged grouped-query attention.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library; the only common module is the seeded input
generator (``paged_kv_gqa_02_gb300.inputs``), which holds none of the
attention arithmetic.

``pa_oracle.c`` is the oracle proper (two-pass softmax in double over keys
gathered through the block table); ``dense.py`` is an independently written
second path (materialise dense K/V, then numpy) used to pin it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
OK, BAD_LEN, BAD_PAGE, BAD_ARG = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Problem(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("window", ctypes.c_int32),
                ("page_stride", ctypes.c_int64), ("token_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64), ("scale", ctypes.c_double),
                ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("q", ctypes.c_void_p), ("cu_q_lens", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.POINTER(Problem)
            L.or_attention.argtypes = [P, ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]
            L.or_attention.restype = ctypes.c_int
            L.or_attention_one.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.POINTER(ctypes.c_int64)]
            L.or_attention_one.restype = ctypes.c_int
            L.or_split_partial.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            L.or_split_partial.restype = ctypes.c_int
            L.or_combine.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p]
            L.or_combine.restype = None
            L.or_set_mutation.argtypes = [ctypes.c_int]
            L.or_max_threads.restype = ctypes.c_int
            L.or_upcast.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64]
            L.or_upcast.restype = ctypes.c_double
            _lib = L
    return _lib


def max_threads() -> int:
    return lib().or_max_threads()


def set_mutation(m: int) -> None:
    lib().or_set_mutation(int(m))


class _Bound:
    """Keeps the numpy arrays behind a Problem alive."""

    def __init__(self, inp, *, num_q_heads, num_kv_heads, head_dim, page_size, scale,
                 q_dtype, kv_dtype, strides=None, window=0):
        q = np.ascontiguousarray(inp["q"])
        k = np.ascontiguousarray(inp["k_cache"])
        v = np.ascontiguousarray(inp["v_cache"])
        bt = np.ascontiguousarray(inp["block_tables"], dtype=np.int32)
        cl = np.ascontiguousarray(inp["context_lens"], dtype=np.int32)
        cu = np.ascontiguousarray(inp["cu_q_lens"], dtype=np.int32)
        self.arrays = (q, k, v, bt, cl, cu)
        if strides is None:  # contiguous [pages][P][Hkv][D]
            strides = (page_size * num_kv_heads * head_dim, num_kv_heads * head_dim, head_dim)
        self.total_q = int(cu[-1])
        self.Hq, self.D = num_q_heads, head_dim
        self.p = Problem(num_seqs=len(cl), num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                         head_dim=head_dim, page_size=page_size, num_pages=int(inp["num_pages"]),
                         max_blocks_per_seq=bt.shape[1], window=int(window),
                         page_stride=strides[0], token_stride=strides[1], head_stride=strides[2],
                         scale=float(scale), q_dtype=DTYPE_CODE[q_dtype],
                         kv_dtype=DTYPE_CODE[kv_dtype], q=q.ctypes.data, cu_q_lens=cu.ctypes.data,
                         k_cache=k.ctypes.data, v_cache=v.ctypes.data,
                         block_tables=bt.ctypes.data, context_lens=cl.ctypes.data)


def bind(inp, wl=None, **kw):
    """Bind an input dict to problem fields (from a Workload or keywords)."""
    if wl is not None:
        kw = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                  head_dim=wl.head_dim, page_size=wl.page_size, scale=wl.scale,
                  q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype, **kw)
    return _Bound(inp, **kw)


def attention(inp, wl=None, threads: int = 1, return_keys: bool = False, **kw):
    """Whole problem -> float64 [total_q][Hq][D]."""
    b = bind(inp, wl, **kw)
    out = np.zeros((b.total_q, b.Hq, b.D), dtype=np.float64)
    keys = ctypes.c_int64(0)
    err = lib().or_attention(ctypes.byref(b.p), out.ctypes.data, int(threads), ctypes.byref(keys))
    if err != OK:
        raise ValueError(f"oracle rejected the problem (code {err})")
    return (out, keys.value) if return_keys else out


def attention_one(inp, row: int, head: int, wl=None, **kw):
    b = bind(inp, wl, **kw)
    out = np.zeros(b.D, dtype=np.float64)
    keys = ctypes.c_int64(0)
    err = lib().or_attention_one(ctypes.byref(b.p), int(row), int(head), out.ctypes.data,
                                 ctypes.byref(keys))
    if err != OK:
        raise ValueError(f"oracle rejected the problem (code {err})")
    return out


def attention_rows(inp, rows_heads, wl=None, **kw):
    """Sampled distributions: list of (row, head) -> float64 [n][D]."""
    b = bind(inp, wl, **kw)
    out = np.zeros((len(rows_heads), b.D), dtype=np.float64)
    keys = ctypes.c_int64(0)
    for i, (r, h) in enumerate(rows_heads):
        err = lib().or_attention_one(ctypes.byref(b.p), int(r), int(h),
                                     out[i].ctypes.data, ctypes.byref(keys))
        if err != OK:
            raise ValueError(f"oracle rejected row {r} head {h} (code {err})")
    return out


def split_partial(inp, seq: int, head: int, t0: int, t1: int, wl=None, **kw):
    """(m_log2, l, acc[D]) of keys [t0, t1) for the last row of ``seq``."""
    b = bind(inp, wl, **kw)
    m = ctypes.c_double(0.0)
    l = ctypes.c_double(0.0)
    acc = np.zeros(b.D, dtype=np.float64)
    err = lib().or_split_partial(ctypes.byref(b.p), int(seq), int(head), int(t0), int(t1),
                                 ctypes.addressof(m), ctypes.addressof(l), acc.ctypes.data)
    if err != OK:
        raise ValueError(f"oracle rejected the split (code {err})")
    return m.value, l.value, acc


def combine(m_log2, l, acc):
    """Combine n splits of one distribution (m in base-2 units) -> out[D]."""
    m_log2 = np.ascontiguousarray(m_log2, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    n, D = acc.shape
    out = np.zeros(D, dtype=np.float64)
    lib().or_combine(n, D, m_log2.ctypes.data, l.ctypes.data, acc.ctypes.data, out.ctypes.data)
    return out


def upcast(dtype: str, arr: np.ndarray, i: int) -> float:
    arr = np.ascontiguousarray(arr)
    return lib().or_upcast(DTYPE_CODE[dtype], arr.ctypes.data, int(i))
