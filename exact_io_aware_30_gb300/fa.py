"""ctypes binding of libfa.so (include/fa.h) -- argument marshalling only.

Every step of the attention forward, backward and paged decoding runs inside
the library's CUDA kernels; this module checks tensor metadata, allocates
outputs (and workspaces) with torch and passes raw pointers and sizes through
the C ABI.  If the library is missing or
refuses a request, it raises: there is no other code path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_CUDA = 4
FA_ERR_DEVICE_TIMEOUT = 5

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_SLIDING_WINDOW = 2
MASKS = {"none": MASK_NONE, "causal": MASK_CAUSAL, "window": MASK_SLIDING_WINDOW,
         "sliding_window": MASK_SLIDING_WINDOW}

DTYPE_BF16 = 0
DTYPE_FP16 = 1
DECODE_AUTO = 0            # fa_decode_paged kernel choice
DECODE_TENSOR_CORES = 1
DECODE_CUDA_CORES = 2
_DECODE_KERNELS = {"auto": DECODE_AUTO, "tensor_cores": DECODE_TENSOR_CORES,
                   "cuda_cores": DECODE_CUDA_CORES}

# Every entry point declared in include/fa.h.
EXPORTS = ("fa_fwd", "fa_fwd_fp16", "fa_fwd_gqa", "fa_fwd_fp8", "fa_bwd", "fa_bwd_noalloc",
           "fa_bwd_workspace_query", "fa_decode_paged", "fa_decode_workspace_query",
           "fa_workspace_query", "fa_status_string", "fa_describe", "fa_get_device_error",
           "fa_fwd_host", "fa_fwd_host_workspace_query", "fa_set_debug_stall_ms")


class FAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i = ctypes.c_int


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load libfa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise FAError(-1, f"{p} is missing: build it with exact_io_aware_30_gb300.build.build()")
        lib = ctypes.CDLL(p)
        fwd_args = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _vp]
        for name in ("fa_fwd", "fa_fwd_fp16"):
            fn = getattr(lib, name)
            fn.restype = _i
            fn.argtypes = fwd_args
        lib.fa_fwd_gqa.restype = _i
        lib.fa_fwd_gqa.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                   ctypes.c_float, _i, _i, _i, _vp]
        lib.fa_bwd.restype = _i
        lib.fa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                               _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _i, _vp]
        lib.fa_bwd_noalloc.restype = _i
        lib.fa_bwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _i, _vp]
        lib.fa_fwd_fp8.restype = _i
        lib.fa_fwd_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_float,
                                   ctypes.c_float, ctypes.c_float, ctypes.c_float, _i, _i, _vp]
        lib.fa_decode_paged.restype = _i
        lib.fa_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                        _i, _i, _i, _i, _i, _i, _i, _i, _i, ctypes.c_float, _i,
                                        _i, _i, _vp]
        lib.fa_decode_workspace_query.restype = _i
        lib.fa_decode_workspace_query.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                                  ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_set_debug_stall_ms.restype = _i
        lib.fa_set_debug_stall_ms.argtypes = [_i]
        lib.fa_bwd_workspace_query.restype = _i
        lib.fa_bwd_workspace_query.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _i,
                                               ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_fwd_host.restype = _i
        lib.fa_fwd_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i, _i, _i,
                                    _i, _i, _i, ctypes.c_float, _i, _i, _i, _vp]
        lib.fa_fwd_host_workspace_query.restype = _i
        lib.fa_fwd_host_workspace_query.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _i,
                                                    ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_workspace_query.restype = _i
        lib.fa_workspace_query.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i,
                                           ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_status_string.argtypes = [_i]
        lib.fa_describe.restype = _i
        lib.fa_describe.argtypes = [_i, _i, _i, ctypes.c_char_p, ctypes.c_size_t]
        lib.fa_get_device_error.restype = _i
        lib.fa_get_device_error.argtypes = []
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != FA_OK:
        raise FAError(status, f"{what}: {status_string(status)}")


def mask_code(mask) -> int:
    return MASKS[mask] if isinstance(mask, str) else int(mask)


def fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
            Sq: int, Sk: int, d: int, scale: float, mask_kind: int, window: int,
            stream: int, dtype: int = DTYPE_BF16) -> int:
    """Call fa_fwd / fa_fwd_fp16 with raw device pointers; returns the status."""
    lib = load()
    fn = lib.fa_fwd if dtype == DTYPE_BF16 else lib.fa_fwd_fp16
    return fn(_vp(q_ptr), _vp(k_ptr), _vp(v_ptr), _vp(o_ptr), _vp(lse_ptr), int(B), int(H),
              int(Sq), int(Sk), int(d), ctypes.c_float(scale), int(mask_kind), int(window),
              _vp(stream))


def fwd_gqa_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
                H_kv: int, Sq: int, Sk: int, d: int, scale: float, mask_kind: int, window: int,
                stream: int, dtype: int = DTYPE_BF16) -> int:
    """Call fa_fwd_gqa (K/V with H_kv heads) with raw device pointers; returns the status."""
    return load().fa_fwd_gqa(_vp(q_ptr), _vp(k_ptr), _vp(v_ptr), _vp(o_ptr), _vp(lse_ptr),
                             int(B), int(H), int(H_kv), int(Sq), int(Sk), int(d),
                             ctypes.c_float(scale), int(mask_kind), int(window), int(dtype),
                             _vp(stream))


def bwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, do_ptr: int,
            dq_ptr: int, dk_ptr: int, dv_ptr: int, ws_ptr: int, ws_bytes: int, B: int, H: int,
            H_kv: int, Sq: int, Sk: int, d: int, scale: float, mask_kind: int, window: int,
            stream: int, dtype: int = DTYPE_BF16) -> int:
    """Call fa_bwd with raw device pointers; returns the status."""
    return load().fa_bwd(_vp(q_ptr), _vp(k_ptr), _vp(v_ptr), _vp(o_ptr), _vp(lse_ptr),
                         _vp(do_ptr), _vp(dq_ptr), _vp(dk_ptr), _vp(dv_ptr), _vp(ws_ptr),
                         ctypes.c_size_t(ws_bytes), int(B), int(H), int(H_kv), int(Sq), int(Sk),
                         int(d), ctypes.c_float(scale), int(mask_kind), int(window), int(dtype),
                         _vp(stream))


def bwd_noalloc_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, do_ptr: int,
                    dq_ptr: int, dk_ptr: int, dv_ptr: int, B: int, H: int, H_kv: int, Sq: int,
                    Sk: int, d: int, scale: float, mask_kind: int, window: int, stream: int,
                    dtype: int = DTYPE_BF16) -> int:
    """Call fa_bwd_noalloc (the library's fixed workspace) with raw device pointers."""
    return load().fa_bwd_noalloc(_vp(q_ptr), _vp(k_ptr), _vp(v_ptr), _vp(o_ptr), _vp(lse_ptr),
                                 _vp(do_ptr), _vp(dq_ptr), _vp(dk_ptr), _vp(dv_ptr), int(B),
                                 int(H), int(H_kv), int(Sq), int(Sk), int(d),
                                 ctypes.c_float(scale), int(mask_kind), int(window), int(dtype),
                                 _vp(stream))


def fwd_fp8_raw(q_ptr, k_ptr, vt_ptr, o_ptr, lse_ptr, B, H, H_kv, Sq, Sk, d, scale, q_descale,
                k_descale, v_descale, mask_kind, window, stream) -> int:
    """Call fa_fwd_fp8 with raw device pointers; returns the status."""
    return load().fa_fwd_fp8(_vp(q_ptr), _vp(k_ptr), _vp(vt_ptr), _vp(o_ptr), _vp(lse_ptr), int(B),
                             int(H), int(H_kv), int(Sq), int(Sk), int(d), ctypes.c_float(scale),
                             ctypes.c_float(q_descale), ctypes.c_float(k_descale),
                             ctypes.c_float(v_descale), int(mask_kind), int(window), _vp(stream))


def forward_fp8(q, k, vt, q_descale: float, k_descale: float, v_descale: float,
                scale: float | None = None, mask="none", window: int = 0, out=None, lse=None,
                stream=None):
    """8-bit forward (fa_fwd_fp8) on CUDA uint8 tensors of e4m3 codes.

    q [B, H, Sq, d]; k [B, H_kv, Sk, d]; vt = V transposed [B, H_kv, d, Sk].
    Returns (o bf16 [B, H, Sq, d], lse fp32 [B, H, Sq]).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("vt", vt)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 4 or t.element_size() != 1:
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 4-D CUDA tensor of bytes")
    B, H, Sq, d = q.shape
    H_kv, Sk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, H_kv, Sk, d) or tuple(vt.shape) != (B, H_kv, d, Sk):
        raise FAError(FA_ERR_INVALID_ARG, "k must be [B,H_kv,Sk,d] and vt [B,H_kv,d,Sk]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Sq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = fwd_fp8_raw(q.data_ptr(), k.data_ptr(), vt.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H,
                     H_kv, Sq, Sk, d, float(scale), float(q_descale), float(k_descale),
                     float(v_descale), mask_code(mask), int(window), sp)
    _check(st, "fa_fwd_fp8")
    return out, lse


def decode_raw(q_ptr, k_ptr, v_ptr, table_ptr, lens_ptr, o_ptr, lse_ptr, ws_ptr, ws_bytes, B, H,
               H_kv, Sq, d, block_size, max_blocks, num_blocks, max_seq_len, scale, mask_kind,
               dtype, stream, kernel=DECODE_AUTO) -> int:
    """Call fa_decode_paged with raw device pointers; returns the status."""
    return load().fa_decode_paged(_vp(q_ptr), _vp(k_ptr), _vp(v_ptr), _vp(table_ptr),
                                  _vp(lens_ptr), _vp(o_ptr), _vp(lse_ptr), _vp(ws_ptr),
                                  ctypes.c_size_t(ws_bytes), int(B), int(H), int(H_kv), int(Sq),
                                  int(d), int(block_size), int(max_blocks), int(num_blocks),
                                  int(max_seq_len), ctypes.c_float(scale), int(mask_kind),
                                  int(dtype), int(kernel), _vp(stream))


def decode_kernel_code(kernel) -> int:
    """"auto", "tensor_cores", "cuda_cores" (or the FA_DECODE_* code)."""
    if isinstance(kernel, str):
        if kernel not in _DECODE_KERNELS:
            raise FAError(FA_ERR_UNSUPPORTED, f"decode kernel {kernel!r}: one of {list(_DECODE_KERNELS)}")
        return _DECODE_KERNELS[kernel]
    return int(kernel)


def decode_workspace_query(B, H, H_kv, Sq, d, block_size, max_blocks, num_blocks, max_seq_len,
                           mask="none", dtype=DTYPE_BF16, kernel=DECODE_AUTO):
    """(status, bytes) of fa_decode_workspace_query."""
    n = ctypes.c_size_t(12345)
    st = load().fa_decode_workspace_query(int(B), int(H), int(H_kv), int(Sq), int(d),
                                          int(block_size), int(max_blocks), int(num_blocks),
                                          int(max_seq_len), mask_code(mask), int(dtype),
                                          decode_kernel_code(kernel), ctypes.byref(n))
    return st, n.value


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int,
                 scale: float | None = None, mask="none", out=None, lse=None, workspace=None,
                 stream=None, kernel="auto"):
    """Attention of q's new rows over a paged K/V cache (fa_decode_paged).

    q [B, H, Sq, d]; k_cache, v_cache [num_blocks, H_kv, block_size, d] (one
    16-bit dtype); block_table int32 [B, max_blocks] and seq_lens int32 [B] on
    the same CUDA device.  kernel: "auto" (the library's choice by rows per
    K/V head), "tensor_cores" or "cuda_cores".  Returns (o, lse).
    """
    import torch
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_table", block_table), ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous CUDA tensor")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise FAError(FA_ERR_INVALID_ARG, "q and the caches must share one dtype")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise FAError(FA_ERR_INVALID_ARG, "block_table and seq_lens must be int32")
    dt = _dtype_code(q)
    B, H, Sq, d = q.shape
    nb, H_kv, bs, d2 = k_cache.shape
    if (tuple(v_cache.shape) != tuple(k_cache.shape) or d2 != d or block_table.dim() != 2
            or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,)):
        raise FAError(FA_ERR_INVALID_ARG, "shapes: q [B,H,Sq,d]; caches [blocks,H_kv,bs,d]; "
                      "block_table [B,n]; seq_lens [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    mb = block_table.shape[1]
    kc = decode_kernel_code(kernel)
    st, ws_bytes = decode_workspace_query(B, H, H_kv, Sq, d, bs, mb, nb, max_seq_len, mask, dt, kc)
    _check(st, "fa_decode_workspace_query")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = decode_raw(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
                    seq_lens.data_ptr(), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                    workspace.numel(), B, H, H_kv, Sq, d, bs, mb, nb, max_seq_len, float(scale),
                    mask_code(mask), dt, sp, kc)
    _check(st, "fa_decode_paged")
    return out, lse


def bwd_workspace_query(B, H, H_kv, Sq, Sk, d, mask="none", window=0, dtype=DTYPE_BF16):
    """(status, bytes) of fa_bwd_workspace_query."""
    n = ctypes.c_size_t(12345)
    st = load().fa_bwd_workspace_query(int(B), int(H), int(H_kv), int(Sq), int(Sk), int(d),
                                       mask_code(mask), int(window), int(dtype), ctypes.byref(n))
    return st, n.value


def workspace_query(B, H, Sq, Sk, d, mask="none", window=0, dtype=DTYPE_BF16):
    """(status, bytes) of fa_workspace_query."""
    n = ctypes.c_size_t(12345)
    st = load().fa_workspace_query(int(B), int(H), int(Sq), int(Sk), int(d), mask_code(mask),
                                   int(window), int(dtype), ctypes.byref(n))
    return st, n.value


def describe(d: int, mask="none", dtype=DTYPE_BF16) -> str:
    buf = ctypes.create_string_buffer(256)
    st = load().fa_describe(int(d), mask_code(mask), int(dtype), buf, 256)
    _check(st, "fa_describe")
    return buf.value.decode()


def device_error() -> int:
    return load().fa_get_device_error()


def set_debug_stall_ms(ms: int) -> None:
    """Test hook (fa_set_debug_stall_ms): with ms > 0 every later launch's
    first pipeline wait runs out after ms; 0 turns it off."""
    _check(load().fa_set_debug_stall_ms(int(ms)), "fa_set_debug_stall_ms")


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float16:
        return DTYPE_FP16
    raise FAError(FA_ERR_UNSUPPORTED, f"dtype {t.dtype} is not supported (bf16 / fp16 only)")


def forward(q, k, v, scale: float | None = None, mask="none", window: int = 0,
            out=None, lse=None, stream=None):
    """Fused attention forward on CUDA tensors [B, H, S, d] (bf16 or fp16).

    k and v may carry fewer heads than q (grouped-query attention: [B, H_kv,
    Sk, d] with H_kv dividing H, query head h reading K/V head h // (H //
    H_kv)); that case goes through fa_fwd_gqa, the rest through fa_fwd /
    fa_fwd_fp16.
    Returns (o, lse): o like q, lse fp32 [B, H, Sq].  Enqueued on ``stream``
    (default: torch's current stream of q's device); raises FAError if the
    library rejects the call.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous [B,H,S,d] tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise FAError(FA_ERR_INVALID_ARG, "q, k, v must share one dtype")
    dt = _dtype_code(q)
    B, H, Sq, d = q.shape
    H_kv, Sk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, H_kv, Sk, d) or tuple(v.shape) != (B, H_kv, Sk, d):
        raise FAError(FA_ERR_INVALID_ARG, "k and v must be [B,H_kv,Sk,d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if H_kv == H:
        st = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                     B, H, Sq, Sk, d, float(scale), mask_code(mask), int(window), sp, dt)
        _check(st, "fa_fwd")
    else:
        st = fwd_gqa_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr(), B, H, H_kv, Sq, Sk, d, float(scale), mask_code(mask),
                         int(window), sp, dt)
        _check(st, "fa_fwd_gqa")
    return out, lse


def backward(q, k, v, o, lse, dout, scale: float | None = None, mask="none", window: int = 0,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Attention backward on CUDA tensors (fa_bwd): returns (dq, dk, dv).

    q, o, dout [B, H, Sq, d]; k, v [B, H_kv, Sk, d] (bf16 or fp16, one dtype);
    lse fp32 [B, H, Sq] from ``forward`` with the same scale, mask and window.
    The workspace (a uint8 CUDA tensor) is allocated here unless given.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("lse", lse)):
        if not t.is_cuda:
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be contiguous")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise FAError(FA_ERR_INVALID_ARG, "q, k, v, o, dout must share one dtype")
    if lse.dtype != torch.float32:
        raise FAError(FA_ERR_INVALID_ARG, "lse must be float32")
    dt = _dtype_code(q)
    B, H, Sq, d = q.shape
    H_kv, Sk = k.shape[1], k.shape[2]
    if (tuple(k.shape) != (B, H_kv, Sk, d) or tuple(v.shape) != (B, H_kv, Sk, d)
            or tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape)
            or tuple(lse.shape) != (B, H, Sq)):
        raise FAError(FA_ERR_INVALID_ARG, "shapes: q, o, dout [B,H,Sq,d]; k, v [B,H_kv,Sk,d]; lse [B,H,Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st, ws_bytes = bwd_workspace_query(B, H, H_kv, Sq, Sk, d, mask, window, dt)
    _check(st, "fa_bwd_workspace_query")
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                 dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                 workspace.numel(), B, H, H_kv, Sq, Sk, d, float(scale), mask_code(mask),
                 int(window), sp, dt)
    _check(st, "fa_bwd")
    return dq, dk, dv


def fwd_host_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, ws_ptr, ws_bytes, B, H, H_kv, Sq, Sk, d,
                 scale, mask_code_, window, dtype, stream_ptr) -> int:
    """fa_fwd_host with raw pointers (host buffers, device workspace)."""
    return load().fa_fwd_host(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, ws_ptr, ws_bytes, B, H, H_kv,
                              Sq, Sk, d, scale, mask_code_, window, dtype, stream_ptr)


def host_workspace_query(B, H, H_kv, Sq, Sk, d, mask="none", window=0, dtype=DTYPE_BF16):
    n = ctypes.c_size_t(0)
    st = load().fa_fwd_host_workspace_query(B, H, H_kv, Sq, Sk, d, mask_code(mask), int(window),
                                            dtype, ctypes.byref(n))
    return st, n.value


def forward_host(q, k, v, scale: float | None = None, mask="none", window: int = 0,
                 out=None, lse=None, workspace=None, device=None, stream=None, sync: bool = True):
    """End to end from host (CPU) tensors through fa_fwd_host: the library
    copies Q, K, V in, runs the forward and copies O and lse out, chunk by
    chunk with the copies overlapping the kernels.

    q [B, H, Sq, d], k and v [B, H_kv, Sk, d] CPU tensors (bf16 or fp16;
    pinned memory for asynchronous copies).  ``out`` / ``lse``: CPU tensors to
    write (allocated pinned here if not given); ``workspace``: a uint8 CUDA
    tensor of at least ``host_workspace_query`` bytes (allocated here if not
    given).  With sync=False the call returns once enqueued on ``stream``.
    Returns (out, lse).
    """
    import torch
    dev = torch.device(device or "cuda")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda:
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be a host tensor (use forward)")
        if t.dim() != 4 or not t.is_contiguous():
            raise FAError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous [B,H,S,d] tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise FAError(FA_ERR_INVALID_ARG, "q, k, v must share one dtype")
    dt = _dtype_code(q)
    B, H, Sq, d = q.shape
    H_kv, Sk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, H_kv, Sk, d) or tuple(v.shape) != (B, H_kv, Sk, d):
        raise FAError(FA_ERR_INVALID_ARG, "k and v must be [B,H_kv,Sk,d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, pin_memory=True)
    if out.is_cuda or lse.is_cuda or tuple(out.shape) != tuple(q.shape) or \
            tuple(lse.shape) != (B, H, Sq) or out.dtype != q.dtype or lse.dtype != torch.float32:
        raise FAError(FA_ERR_INVALID_ARG, "out / lse must be host tensors like q / [B,H,Sq] fp32")
    st, ws_bytes = host_workspace_query(B, H, H_kv, Sq, Sk, d, mask, window, dt)
    _check(st, "fa_fwd_host_workspace_query")
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      workspace.data_ptr(), workspace.numel(), B, H, H_kv, Sq, Sk, d, float(scale),
                      mask_code(mask), int(window), dt, sp)
    _check(st, "fa_fwd_host")
    if sync:
        stream.synchronize()
    return out, lse
