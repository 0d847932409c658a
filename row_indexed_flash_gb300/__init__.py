"""Python binding of libfa_rows: row-indexed flash attention over a unified KV pool.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of ``libfa_rows.so``; torch supplies device memory, streams and
pointers.  If the library has not been built the calls raise instead of
computing anything another way.

The operation ("llama.cpp 0.9.0 inference boundaries", section 1): K/V rows of
all sequences share one pool; each query slice passes an int32 ``kv_rows``
list of the pool rows it attends to; a negative index is padding (mask minus
infinity); the result is exact attention over the listed rows.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = [
    "FaRowsError", "lib", "library_path", "fa_rows_args", "fa_rows_workspace_size", "fa_rows_workspace_init",
    "fa_rows_status", "fa_set_wait_limit_ns", "default_workspace", "FA_WS_WAIT_EXPIRED",
    "fa_rows_decode", "fa_rows_prefill", "fa_rows_validate", "fa_kv_page_table_to_rows", "fa_kv_quantize_int8",
    "fa_kv_dequantize_int8", "fa_kv_quantize_int4", "fa_kv_dequantize_int4", "fa_kv_quantize_fp8", "fa_kv_dequantize_fp8", "fa_kv_sparse_rows_workspace_size", "fa_kv_sparse_rows", "fa_kv_append", "fa_status_string", "fa_last_error", "fa_version",
    "FA_F16", "FA_BF16", "FA_F32", "FA_I8", "FA_I4", "FA_F8E4M3", "FA_MASK_NONE", "FA_MASK_DENSE", "FA_MASK_CAUSAL",
]

FA_F16, FA_BF16, FA_F32, FA_I8, FA_I4, FA_F8E4M3 = 0, 1, 2, 3, 4, 5
FA_MASK_NONE, FA_MASK_DENSE, FA_MASK_CAUSAL = 0, 1, 2
_STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_WORKSPACE",
           4: "FA_ERR_INDEX_OOB", 5: "FA_ERR_CUDA", 6: "FA_ERR_WAIT_EXPIRED"}
FA_ERR_WAIT_EXPIRED = 6
FA_WS_WAIT_EXPIRED = 1   # bit of the workspace status word (first uint32 of a workspace)

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libfa_rows.so")


class FaRowsError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


class fa_rows_args(ctypes.Structure):
    """Mirror of ``fa_rows_args`` in include/fa_rows.h."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_dtype", ctypes.c_int),
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("kv_dtype", ctypes.c_int),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("n_pool_rows", ctypes.c_int64),
        ("kv_rows", ctypes.c_void_p), ("list_len", ctypes.c_int32),
        ("kv_len", ctypes.c_void_p),
        ("mask_kind", ctypes.c_int), ("mask", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int), ("lse", ctypes.c_void_p),
        ("S", ctypes.c_int32), ("Nq", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("n_valid_hint", ctypes.c_int64),
    ]


_lib = None
_lib_lock = threading.Lock()

_P = ctypes.c_void_p
_SIGS = {
    "fa_rows_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(fa_rows_args), ctypes.c_int]),
    "fa_rows_decode_launches": (ctypes.c_int, [ctypes.POINTER(fa_rows_args)]),
    "fa_rows_workspace_init": (ctypes.c_int, [_P, ctypes.c_size_t, _P]),
    "fa_rows_status": (ctypes.c_int, [_P, ctypes.c_size_t, _P, ctypes.c_int, _P]),
    "fa_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "fa_rows_decode": (ctypes.c_int, [ctypes.POINTER(fa_rows_args), _P, ctypes.c_size_t, _P]),
    "fa_rows_prefill": (ctypes.c_int, [ctypes.POINTER(fa_rows_args), _P, ctypes.c_size_t, _P]),
    "fa_rows_decode_static": (ctypes.c_int, [ctypes.POINTER(fa_rows_args), _P]),
    "fa_rows_validate": (ctypes.c_int, [ctypes.POINTER(fa_rows_args), _P, _P]),
    "fa_kv_page_table_to_rows": (ctypes.c_int, [_P, ctypes.c_int32, _P, ctypes.c_int32, ctypes.c_int32, _P,
                                                ctypes.c_int32, _P]),
    "fa_kv_quantize_int8": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                           _P, ctypes.c_int64, _P]),
    "fa_kv_dequantize_int8": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P]),
    "fa_kv_quantize_int4": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                           _P, ctypes.c_int64, _P]),
    "fa_kv_dequantize_int4": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P]),
    "fa_kv_quantize_fp8": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                          _P, ctypes.c_int64, _P]),
    "fa_kv_dequantize_fp8": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P]),
    "fa_kv_sparse_rows_workspace_size": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32]),
    "fa_kv_sparse_rows": (ctypes.c_int, [_P, ctypes.c_int32, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, _P, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "fa_kv_append": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                    ctypes.c_int64, _P]),
    "fa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_last_error": (ctypes.c_char_p, []),
    "fa_version": (ctypes.c_char_p, []),
}


def lib() -> ctypes.CDLL:
    """The loaded libfa_rows.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                if not os.path.exists(library_path):
                    raise RuntimeError(f"libfa_rows.so is not built ({library_path}); "
                                       "run `python -m row_indexed_flash_gb300.build`")
                h = ctypes.CDLL(library_path)
                for name, (res, args) in _SIGS.items():
                    fn = getattr(h, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = h
    return _lib


def fa_status_string(s: int) -> str:
    return lib().fa_status_string(s).decode()


def fa_last_error() -> str:
    return lib().fa_last_error().decode()


def fa_version() -> str:
    return lib().fa_version().decode()


def _check(status: int):
    if status != 0:
        raise FaRowsError(status, fa_last_error())


# ---------------------------------------------------------------------------
# marshalling helpers

_DT = {torch.float16: FA_F16, torch.bfloat16: FA_BF16, torch.float32: FA_F32, torch.int8: FA_I8, torch.uint8: FA_I4,
       torch.float8_e4m3fn: FA_F8E4M3}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class _Workspace:
    """Caller-side scratch (status word, split counters, partials): grown on demand, zeroed once."""

    def __init__(self):
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int, device, stream_handle: int) -> Tuple[int, int]:
        if nbytes == 0:
            return 0, 0
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
            _check(lib().fa_rows_workspace_init(self.buf.data_ptr(), self.buf.numel(), stream_handle))
        return self.buf.data_ptr(), self.buf.numel()


_workspaces = {}


def _default_ws(device, stream_handle, is_prefill: bool) -> _Workspace:
    """The binding's own workspace for calls without one: one per (device, stream, decode or prefill)."""
    key = (str(device), stream_handle, bool(is_prefill))
    if key not in _workspaces:
        _workspaces[key] = _Workspace()
    return _workspaces[key]


def default_workspace(device=None, stream=None, is_prefill: bool = False) -> Optional[torch.Tensor]:
    """The workspace tensor the binding uses for calls made without one (None before the first such call)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return _default_ws(device, _stream(stream, device), is_prefill).buf


def make_args(q, k, v, kv_rows, scale, *, kv_len=None, mask=None, causal=False, k_scale=None, v_scale=None,
              out=None, lse=None, out_dtype=torch.float32, want_lse=False, n_valid_hint=0):
    """Builds fa_rows_args from torch tensors; allocates ``out``/``lse`` if not given."""
    S, Nq, Hq, D = q.shape
    R, Hkv, Dk = k.shape
    packed = k.dtype == torch.uint8   # INT4 pool: two codes per byte
    if tuple(v.shape) != (R, Hkv, Dk) or Dk * (2 if packed else 1) != D:
        raise ValueError(f"k {tuple(k.shape)} / v {tuple(v.shape)} do not match q {tuple(q.shape)}")
    if kv_rows.dtype != torch.int32 or kv_rows.dim() != 2 or kv_rows.shape[0] != S:
        raise ValueError("kv_rows must be int32 [S, L]")
    if k.dtype != v.dtype:
        raise ValueError("k and v must share a dtype")
    if k.dtype in (torch.int8, torch.uint8, torch.float8_e4m3fn) and (k_scale is None or v_scale is None):
        raise ValueError("a quantised pool needs k_scale and v_scale")
    if kv_len is not None and (kv_len.dtype != torch.int32 or kv_len.shape != (S,)):
        raise ValueError("kv_len must be int32 [S]")
    if mask is not None and (mask.dtype != torch.float32 or tuple(mask.shape) != (S, Nq, kv_rows.shape[1])):
        raise ValueError("mask must be float32 [S, Nq, L]")
    if out is None:
        out = torch.empty((S, Nq, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((S, Nq, Hq), dtype=torch.float32, device=q.device)
    a = fa_rows_args()
    a.q, a.q_dtype = _ptr(q), _DT[q.dtype]
    a.k, a.v, a.kv_dtype = _ptr(k), _ptr(v), _DT[k.dtype]
    a.k_scale, a.v_scale = _ptr(k_scale), _ptr(v_scale)
    a.n_pool_rows = R
    a.kv_rows, a.list_len = _ptr(kv_rows), kv_rows.shape[1]
    a.kv_len = _ptr(kv_len)
    if mask is not None:
        a.mask_kind, a.mask = FA_MASK_DENSE, _ptr(mask)
    else:
        a.mask_kind = FA_MASK_CAUSAL if causal else FA_MASK_NONE
    a.scale = float(scale)
    a.out, a.out_dtype, a.lse = _ptr(out), _DT[out.dtype], _ptr(lse)
    a.S, a.Nq, a.Hq, a.Hkv, a.D = S, Nq, Hq, Hkv, D
    a.n_valid_hint = int(n_valid_hint)
    return a, out, lse


def fa_rows_workspace_size(args: fa_rows_args, is_prefill: bool = False) -> int:
    n = lib().fa_rows_workspace_size(ctypes.byref(args), int(is_prefill))
    err = fa_last_error()
    if err:
        raise FaRowsError(1, err)
    return n


def fa_rows_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().fa_rows_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream, ws.device)))


def fa_rows_status(ws: torch.Tensor, clear: bool = False, stream=None) -> int:
    """The workspace's status word (FA_WS_WAIT_EXPIRED set: a call on it had a
    pipeline wait run out).  Synchronises the stream to read it."""
    sh = _stream(stream, ws.device)
    word = torch.empty(1, dtype=torch.int32, device=ws.device)
    _check(lib().fa_rows_status(_ptr(ws), ws.numel() * ws.element_size(), word.data_ptr(), int(clear), sh))
    return int(word.item()) & 0xffffffff


def fa_set_wait_limit_ns(limit_ns: int):
    """Limit of every bounded pipeline wait in kernels launched afterwards (0 = the 1 s default)."""
    _check(lib().fa_set_wait_limit_ns(int(limit_ns)))


def _attend(entry: str, is_prefill: bool, q, k, v, kv_rows, scale, *, workspace=None, stream=None,
            check_status=False, **kw):
    a, out, lse = make_args(q, k, v, kv_rows, scale, **kw)
    sh = _stream(stream, q.device)
    need = fa_rows_workspace_size(a, is_prefill)
    if workspace is None:
        wsobj = _default_ws(q.device, sh, is_prefill)
        wptr, wbytes = wsobj.get(need, q.device, sh)
        wtensor = wsobj.buf
    else:
        wptr, wbytes = _ptr(workspace), workspace.numel() * workspace.element_size()
        wtensor = workspace
    _check(getattr(lib(), entry)(ctypes.byref(a), wptr, wbytes, sh))
    if check_status and wtensor is not None:
        word = fa_rows_status(wtensor, clear=True, stream=stream)
        if word & FA_WS_WAIT_EXPIRED:
            raise FaRowsError(FA_ERR_WAIT_EXPIRED, f"{entry}: a pipeline wait ran out; the outputs are invalid")
    return out, lse


def fa_rows_decode(q, k, v, kv_rows, scale, **kw):
    """Decode (few query rows per slice).  Returns (out, lse or None).

    Keyword args: kv_len, mask (fp32 [S,Nq,L]), causal, k_scale/v_scale (int8
    pool, fp16 [R/64,Hkv,64]), out, lse, out_dtype, want_lse, n_valid_hint,
    workspace (zero-initialised uint8 tensor), stream, check_status (read the
    workspace status word after the call -- this synchronises -- and raise
    FA_ERR_WAIT_EXPIRED if a pipeline wait ran out, clearing the word).
    """
    return _attend("fa_rows_decode", False, q, k, v, kv_rows, scale, **kw)


def fa_rows_prefill(q, k, v, kv_rows, scale, **kw):
    """Prefill (many query rows per slice), tensor-core path.  Same arguments as decode."""
    return _attend("fa_rows_prefill", True, q, k, v, kv_rows, scale, **kw)


def fa_rows_validate(kv_rows: torch.Tensor, n_pool_rows: int, kv_len=None, stream=None) -> Tuple[int, int]:
    """Range check of the lists; returns (entries >= n_pool_rows, first flat index or -1).  Synchronises."""
    a = fa_rows_args()
    a.kv_rows, a.list_len, a.S = _ptr(kv_rows), kv_rows.shape[1], kv_rows.shape[0]
    a.kv_len = _ptr(kv_len)
    a.n_pool_rows = int(n_pool_rows)
    status = torch.empty(2, dtype=torch.int64, device=kv_rows.device)
    _check(lib().fa_rows_validate(ctypes.byref(a), status.data_ptr(), _stream(stream, kv_rows.device)))
    c, f = status.tolist()
    return int(c), int(f)


def fa_kv_page_table_to_rows(page_table: torch.Tensor, seq_len: torch.Tensor, list_len: int, page_size: int = 64,
                             out=None, stream=None) -> torch.Tensor:
    n_seq, max_pages = page_table.shape
    if out is None:
        out = torch.empty((n_seq, list_len), dtype=torch.int32, device=page_table.device)
    _check(lib().fa_kv_page_table_to_rows(_ptr(page_table), max_pages, _ptr(seq_len), n_seq, page_size, _ptr(out),
                                          list_len, _stream(stream, page_table.device)))
    return out


def fa_kv_quantize_int8(x: torch.Tensor, n_pool_rows: Optional[int] = None, dst_rows=None, q=None, scale=None,
                        stream=None):
    """Quantises x [n, Hkv, D] (bf16/f16) into an INT8 pool; returns (q [R,Hkv,D] int8, scale fp16 [R/64,Hkv,64])."""
    n, Hkv, D = x.shape
    R = n if n_pool_rows is None else int(n_pool_rows)
    if q is None:
        q = torch.zeros((R, Hkv, D), dtype=torch.int8, device=x.device)
    if scale is None:
        scale = torch.zeros((R // 64, Hkv, 64), dtype=torch.float16, device=x.device)
    _check(lib().fa_kv_quantize_int8(_ptr(x), _DT[x.dtype], n, Hkv, D, _ptr(dst_rows), _ptr(q), _ptr(scale),
                                     q.shape[0], _stream(stream, x.device)))
    return q, scale


def fa_kv_dequantize_int8(q: torch.Tensor, scale: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    R, Hkv, D = q.shape
    if out is None:
        out = torch.empty((R, Hkv, D), dtype=torch.float32, device=q.device)
    _check(lib().fa_kv_dequantize_int8(_ptr(q), _ptr(scale), R, Hkv, D, _ptr(out), _stream(stream, q.device)))
    return out


def fa_kv_quantize_int4(x: torch.Tensor, n_pool_rows: Optional[int] = None, dst_rows=None, q=None, scale=None,
                        stream=None):
    """Quantises x [n, Hkv, D] (bf16/f16) into an INT4 pool; returns (q [R,Hkv,D/2] uint8, scale fp16 [R/64,Hkv,64])."""
    n, Hkv, D = x.shape
    R = n if n_pool_rows is None else int(n_pool_rows)
    if q is None:
        q = torch.zeros((R, Hkv, D // 2), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.zeros((R // 64, Hkv, 64), dtype=torch.float16, device=x.device)
    _check(lib().fa_kv_quantize_int4(_ptr(x), _DT[x.dtype], n, Hkv, D, _ptr(dst_rows), _ptr(q), _ptr(scale),
                                     q.shape[0], _stream(stream, x.device)))
    return q, scale


def fa_kv_dequantize_int4(q: torch.Tensor, scale: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    R, Hkv, Dh = q.shape
    if out is None:
        out = torch.empty((R, Hkv, 2 * Dh), dtype=torch.float32, device=q.device)
    _check(lib().fa_kv_dequantize_int4(_ptr(q), _ptr(scale), R, Hkv, 2 * Dh, _ptr(out), _stream(stream, q.device)))
    return out


def fa_kv_quantize_fp8(x: torch.Tensor, n_pool_rows: Optional[int] = None, dst_rows=None, q=None, scale=None,
                       stream=None):
    """Quantises x [n, Hkv, D] (bf16/f16) into an FP8 E4M3 pool; returns (q [R,Hkv,D] float8_e4m3fn, scale fp16)."""
    n, Hkv, D = x.shape
    R = n if n_pool_rows is None else int(n_pool_rows)
    if q is None:
        q = torch.zeros((R, Hkv, D), dtype=torch.float8_e4m3fn, device=x.device)
    if scale is None:
        scale = torch.zeros((R // 64, Hkv, 64), dtype=torch.float16, device=x.device)
    _check(lib().fa_kv_quantize_fp8(_ptr(x), _DT[x.dtype], n, Hkv, D, _ptr(dst_rows), _ptr(q), _ptr(scale),
                                    q.shape[0], _stream(stream, x.device)))
    return q, scale


def fa_kv_dequantize_fp8(q: torch.Tensor, scale: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    R, Hkv, D = q.shape
    if out is None:
        out = torch.empty((R, Hkv, D), dtype=torch.float32, device=q.device)
    _check(lib().fa_kv_dequantize_fp8(_ptr(q), _ptr(scale), R, Hkv, D, _ptr(out), _stream(stream, q.device)))
    return out


def fa_kv_sparse_rows(score: torch.Tensor, sinks: int, recent: int, k: int, list_len: Optional[int] = None,
                      n_len=None, row_map=None, out=None, workspace="auto", stream=None) -> torch.Tensor:
    """Sorted kv_rows [S, list_len] of sinks + top-k(score) + recent per slice (score fp32 [S, n_max]).

    workspace: "auto" allocates the multi-block scratch, None runs one block
    per slice without scratch, or a uint8 tensor of at least
    fa_kv_sparse_rows_workspace_size(S, n_max) bytes.
    """
    if score.dtype != torch.float32 or score.dim() != 2:
        raise ValueError("score must be float32 [S, n_max]")
    S, n_max = score.shape
    L = sinks + recent + k if list_len is None else int(list_len)
    if out is None:
        out = torch.empty((S, L), dtype=torch.int32, device=score.device)
    if isinstance(workspace, str):
        nbytes = lib().fa_kv_sparse_rows_workspace_size(S, n_max)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=score.device)
    wptr = _ptr(workspace)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fa_kv_sparse_rows(_ptr(score), n_max, _ptr(n_len), S, sinks, recent, k, _ptr(row_map), _ptr(out),
                                   L, wptr, wbytes, _stream(stream, score.device)))
    return out


def fa_kv_append(x: torch.Tensor, dst_rows: torch.Tensor, pool: torch.Tensor, stream=None) -> torch.Tensor:
    n, Hkv, D = x.shape
    if pool.dtype != x.dtype or tuple(pool.shape[1:]) != (Hkv, D):
        raise ValueError("pool must be [R, Hkv, D] of x's dtype")
    _check(lib().fa_kv_append(_ptr(x), _DT[x.dtype], n, Hkv, D, _ptr(dst_rows), _ptr(pool), pool.shape[0],
                              _stream(stream, x.device)))
    return pool
