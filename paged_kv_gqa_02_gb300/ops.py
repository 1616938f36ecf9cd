"""ctypes binding of libpaged_gqa.so (see ``include/paged_gqa.h``).

Argument marshalling only: every step of the attention runs in the CUDA
library.  torch supplies device memory and the current stream.  There is no
fallback: if the library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
# PA_GQA_LIB names another build of the library (e.g. the checked build)
LIB_PATH = os.environ.get("PA_GQA_LIB") or os.path.join(PKG, "libpaged_gqa.so")

PA_F32, PA_F16, PA_BF16 = 0, 1, 2
DTYPE_CODE = {"f32": PA_F32, "f16": PA_F16, "bf16": PA_BF16}
PA_DEV_BAD_PAGE, PA_DEV_BAD_LEN, PA_DEV_TIMEOUT, PA_DEV_OOB = 1, 2, 4, 8
PA_FORM_AUTO, PA_FORM_PAIR, PA_FORM_COUNTED = 0, 1, 2
STATUS = {0: "PA_OK", 1: "PA_ERR_NULL", 2: "PA_ERR_SHAPE", 3: "PA_ERR_DTYPE",
          4: "PA_ERR_ALIGN", 5: "PA_ERR_WORKSPACE", 6: "PA_ERR_UNSUPPORTED", 7: "PA_ERR_CUDA"}

EXPORTS = ("pa_params_init", "pa_status_string", "pa_decode_plan", "pa_decode_workspace_size",
           "pa_decode", "pa_decode_partial", "pa_combine", "pa_prefill_workspace_size",
           "pa_prefill_chunk", "pa_version", "pa_decode_append", "pa_decode_noalloc",
           "pa_build_flags", "pa_decode_kernels")


class PaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class Params(ctypes.Structure):
    """Mirror of ``pa_params``."""
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
                ("page_stride", ctypes.c_int64), ("token_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64), ("scale", ctypes.c_float),
                ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("deterministic", ctypes.c_int32),
                ("num_splits", ctypes.c_int32), ("decode_phases", ctypes.c_int32),
                ("decode_q_rows", ctypes.c_int32), ("sliding_window", ctypes.c_int32),
                ("decode_form", ctypes.c_int32), ("debug_timeout", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Loads the library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: run paged_kv_gqa_02_gb300.build.build()")
            L = ctypes.CDLL(path)
            P = ctypes.POINTER(Params)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            L.pa_params_init.argtypes = [P]
            L.pa_params_init.restype = P
            L.pa_status_string.argtypes = [ctypes.c_int]
            L.pa_status_string.restype = ctypes.c_char_p
            L.pa_decode_plan.argtypes = [P, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.pa_decode_workspace_size.argtypes = [P]
            L.pa_decode_workspace_size.restype = sz
            L.pa_decode.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
            L.pa_decode_partial.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp]
            L.pa_decode_append.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
            L.pa_combine.argtypes = [P, vp, vp, i32, vp, vp, vp]
            L.pa_prefill_workspace_size.argtypes = [P, i32, i32]
            L.pa_prefill_workspace_size.restype = sz
            L.pa_prefill_chunk.argtypes = [P, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]
            L.pa_decode_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
            if hasattr(L, "pa_decode_kernels"):
                L.pa_decode_kernels.argtypes = [P, i32]
                L.pa_decode_kernels.restype = i32
            for name in ("pa_decode_plan", "pa_decode", "pa_decode_append", "pa_decode_partial",
                         "pa_combine", "pa_prefill_chunk", "pa_decode_noalloc"):
                getattr(L, name).restype = ctypes.c_int
            L.pa_version.restype = i32
            if hasattr(L, "pa_build_flags"):
                L.pa_build_flags.restype = i32
            _lib = L
    return _lib


def make_params(*, num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                max_blocks_per_seq, max_context_len, scale=None, dtype="bf16", kv_dtype=None,
                deterministic=1, num_splits=0, strides=(0, 0, 0), decode_phases=0,
                decode_q_rows=0, sliding_window=0, decode_form=0, debug_timeout=0) -> Params:
    p = Params()
    load().pa_params_init(ctypes.byref(p))
    p.num_seqs, p.num_q_heads, p.num_kv_heads = num_seqs, num_q_heads, num_kv_heads
    p.head_dim, p.page_size, p.num_pages = head_dim, page_size, num_pages
    p.max_blocks_per_seq, p.max_context_len = max_blocks_per_seq, max_context_len
    p.page_stride, p.token_stride, p.head_stride = strides
    p.scale = (1.0 / math.sqrt(head_dim)) if scale is None else scale
    p.q_dtype = DTYPE_CODE[dtype]
    p.kv_dtype = DTYPE_CODE[kv_dtype or dtype]
    p.out_dtype = PA_F32
    p.deterministic, p.num_splits = deterministic, num_splits
    p.decode_phases = decode_phases
    p.decode_q_rows = decode_q_rows
    p.sliding_window = sliding_window
    p.decode_form = decode_form
    p.debug_timeout = debug_timeout
    return p


def params_for(wl, num_pages=None, **kw) -> Params:
    """Params of a ``workloads.Workload``."""
    args = dict(num_seqs=wl.num_seqs, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                head_dim=wl.head_dim, page_size=wl.page_size,
                num_pages=num_pages or wl.num_pages, max_blocks_per_seq=wl.max_blocks_per_seq,
                max_context_len=wl.max_blocks_per_seq * wl.page_size, scale=wl.scale,
                dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    args.update(kw)
    return make_params(**args)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code, what):
    if code != 0:
        raise PaError(code, what)


def decode_plan(p: Params):
    S, tok = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load().pa_decode_plan(ctypes.byref(p), ctypes.byref(S), ctypes.byref(tok)),
           "pa_decode_plan")
    return S.value, tok.value


def decode_kernels(p: Params, with_append: bool = False) -> int:
    """Kernels one pa_decode (or pa_decode_append) call launches (-1: invalid)."""
    return int(load().pa_decode_kernels(ctypes.byref(p), int(with_append)))


def decode_workspace_size(p: Params) -> int:
    return int(load().pa_decode_workspace_size(ctypes.byref(p)))


def prefill_workspace_size(p: Params, total_q: int, max_q_len: int) -> int:
    return int(load().pa_prefill_workspace_size(ctypes.byref(p), total_q, max_q_len))


def _empty_out(q, p):
    import torch
    return torch.empty((q.shape[0], p.num_q_heads, p.head_dim), dtype=torch.float32,
                       device=q.device)


def decode(p: Params, q, k_cache, v_cache, block_tables, context_lens, out=None,
           workspace=None, dev_status=None, stream=None):
    """Decode attention; q [B][Hq][D] -> out [B][Hq][D] f32 (torch CUDA tensors)."""
    import torch
    if out is None:
        out = _empty_out(q, p)
    if workspace is None:
        n = decode_workspace_size(p)
        workspace = torch.zeros(max(n, 1), dtype=torch.uint8, device=q.device) if n else None
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_decode(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                            _ptr(block_tables), _ptr(context_lens), _ptr(out), _ptr(workspace),
                            nbytes, _ptr(dev_status), _stream(stream)), "pa_decode")
    return out


def decode_append(p: Params, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out=None,
                  workspace=None, dev_status=None, stream=None):
    """Decode with the new token's K/V ([B][Hkv][D]) written to row L-1 of each
    sequence's last page first; k_cache / v_cache are updated in place."""
    import torch
    if out is None:
        out = _empty_out(q, p)
    if workspace is None:
        n = decode_workspace_size(p)
        workspace = torch.zeros(max(n, 1), dtype=torch.uint8, device=q.device) if n else None
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_decode_append(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), _ptr(out),
                                   _ptr(workspace), nbytes, _ptr(dev_status), _stream(stream)),
           "pa_decode_append")
    return out


def decode_partial(p: Params, q, k_cache, v_cache, block_tables, context_lens, partial_ml,
                   partial_acc, num_splits, dev_status=None, stream=None):
    _check(load().pa_decode_partial(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_tables), _ptr(context_lens), _ptr(partial_ml),
                                    _ptr(partial_acc), num_splits, _ptr(dev_status),
                                    _stream(stream)), "pa_decode_partial")


def combine(p: Params, partial_ml, partial_acc, num_splits, out, stream=None, splits_per_seq=None):
    """pa_combine: num_splits is the partials' split stride (max_splits);
    splits_per_seq (device int32 [B], optional) limits each sequence."""
    _check(load().pa_combine(ctypes.byref(p), _ptr(partial_ml), _ptr(partial_acc), num_splits,
                             _ptr(splits_per_seq), _ptr(out), _stream(stream)), "pa_combine")
    return out


def prefill_chunk(p: Params, q, cu_q_lens, total_q, max_q_len, k_cache, v_cache, block_tables,
                  context_lens, out=None, workspace=None, dev_status=None, stream=None):
    """Chunked causal prefill; q [total_q][Hq][D] -> out [total_q][Hq][D] f32."""
    import torch
    if out is None:
        out = _empty_out(q, p)
    if workspace is None:
        n = prefill_workspace_size(p, total_q, max_q_len)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_prefill_chunk(ctypes.byref(p), _ptr(q), _ptr(cu_q_lens), total_q, max_q_len,
                                   _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), _ptr(out), _ptr(workspace), nbytes,
                                   _ptr(dev_status), _stream(stream)), "pa_prefill_chunk")
    return out


# ---- numpy inputs -> torch device tensors ----------------------------------

def to_device(arr, dtype: str | None = None, device="cuda"):
    """numpy array (bf16 given as uint16 bits when dtype == 'bf16') -> torch."""
    import numpy as np
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.to(device)


def device_inputs(inp, wl_or_dtype, device="cuda"):
    """Input dict from ``inputs.make_paged_inputs`` -> dict of device tensors."""
    q_dt = getattr(wl_or_dtype, "q_dtype", wl_or_dtype)
    kv_dt = getattr(wl_or_dtype, "kv_dtype", wl_or_dtype)
    return dict(q=to_device(inp["q"], q_dt, device), k_cache=to_device(inp["k_cache"], kv_dt, device),
                v_cache=to_device(inp["v_cache"], kv_dt, device),
                block_tables=to_device(inp["block_tables"], None, device),
                context_lens=to_device(inp["context_lens"], None, device),
                cu_q_lens=to_device(inp["cu_q_lens"], None, device))


def decode_noalloc(p: Params, q, k_cache, v_cache, block_tables, context_lens, out=None,
                   dev_status=None, stream=None):
    """pa_decode_noalloc: decode with the split partials in the library's
    static device scratch (for callers that cannot allocate at call time).
    Raises PaError(PA_ERR_WORKSPACE) when the partials exceed the scratch."""
    fn = load().pa_decode_noalloc
    if out is None:
        out = _empty_out(q, p)
    _check(fn(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
              _ptr(context_lens), _ptr(out), _ptr(dev_status), _stream(stream)),
           "pa_decode_noalloc")
    return out
