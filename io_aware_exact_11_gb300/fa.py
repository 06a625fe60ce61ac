"""ctypes binding for libfa.so (the C ABI in include/fa.h).

Argument marshalling only: tensors are passed as raw device pointers plus
sizes and strides, on the caller's current CUDA stream.  PyTorch provides
device memory and streams; every step of the computation runs in the
library's CUDA kernels.  If libfa.so has not been built this module raises,
there is no fallback path.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT = range(5)
FA_BF16, FA_FP32 = 0, 1
FA_MASK_NONE, FA_MASK_CAUSAL = 0, 1

EXPORTED = (
    "fa_abi_version",
    "fa_forward",
    "fa_forward_masked",
    "fa_forward_fp8",
    "fa_forward_host_workspace_size",
    "fa_forward_host",
    "fa_decode_choose_splits",
    "fa_decode_workspace_size",
    "fa_decode_splitkv",
    "fa_decode_splitkv_gqa",
    "fa_decode_paged",
    "fa_decode_splitkv_noalloc",
    "fa_backward_workspace_size",
    "fa_backward",
    "fa_backward_masked",
    "fa_device_status",
    "fa_watchdog_selftest",
    "fa_status_string",
    "fa_get_last_error",
    "fa_launch_count",
)


class FAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[status {status}] {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Open libfa.so once (raises FileNotFoundError if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FileNotFoundError(
                f"{LIB_PATH} is missing: build it with `python -m io_aware_exact_11_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.fa_abi_version.restype = i32
        L.fa_forward.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, vp]
        L.fa_forward.restype = i32
        L.fa_forward_masked.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, i32, vp]
        L.fa_forward_masked.restype = i32
        L.fa_forward_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, f32, f32, f32, i32, vp]
        L.fa_forward_fp8.restype = i32
        L.fa_forward_host_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        L.fa_forward_host_workspace_size.restype = sz
        L.fa_forward_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, i32, vp, sz, vp]
        L.fa_forward_host.restype = i32
        L.fa_decode_choose_splits.argtypes = [i32, i32, i32, i32]
        L.fa_decode_choose_splits.restype = i32
        L.fa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        L.fa_decode_workspace_size.restype = sz
        L.fa_decode_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
        L.fa_decode_splitkv.restype = i32
        L.fa_decode_splitkv_gqa.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
        L.fa_decode_splitkv_gqa.restype = i32
        L.fa_decode_paged.argtypes = [vp] * 7 + [i32] * 8 + [f32, i32, vp, sz, vp]
        L.fa_decode_paged.restype = i32
        L.fa_backward_workspace_size.argtypes = [i32, i32, i32, i32]
        L.fa_backward_workspace_size.restype = sz
        L.fa_backward.argtypes = [vp] * 9 + [i32, i32, i32, i32, i32, f32, vp, sz, vp]
        L.fa_backward.restype = i32
        L.fa_backward_masked.argtypes = [vp] * 9 + [i32, i32, i32, i32, i32, f32, vp, sz, i32, vp]
        L.fa_backward_masked.restype = i32
        L.fa_device_status.argtypes = [vp]
        L.fa_device_status.restype = i32
        L.fa_watchdog_selftest.argtypes = [vp]
        L.fa_watchdog_selftest.restype = i32
        L.fa_status_string.argtypes = [i32]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_get_last_error.restype = ctypes.c_char_p
        L.fa_launch_count.restype = ctypes.c_uint64
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != FA_OK:
        msg = lib().fa_get_last_error().decode(errors="replace")
        raise FAError(status, msg or lib().fa_status_string(status).decode())


def _torch():
    import torch
    return torch


def _stream_ptr(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must live on a CUDA device")


def launch_count() -> int:
    """Kernels the library has enqueued since it was loaded."""
    return int(lib().fa_launch_count())


def device_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel's bounded wait gave up."""
    _check(lib().fa_device_status(_stream_ptr(stream)))


def watchdog_selftest(stream=None) -> None:
    """Enqueue a kernel whose bounded wait runs out (~1 s); the next
    device_status() raises FAError with FA_ERR_DEVICE_TIMEOUT."""
    _check(lib().fa_watchdog_selftest(_stream_ptr(stream)))


def forward(q, k, v, scale: float | None = None, out=None, lse=None, return_lse: bool = True, stream=None,
            causal: bool = False):
    """Exact attention forward.  q [B,H,Nq,d], k/v [B,H,Nkv,d] (bf16 or fp32).

    Returns (O, LSE) with O like q and LSE fp32 [B,H,Nq].  Non-contiguous
    inputs are passed by stride (d must be the contiguous dim).  ``causal``
    masks keys j > i + Nkv − Nq for query row i.
    """
    torch = _torch()
    _check_cuda(q, k, v)
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    if k.shape != (B, H, Nkv, d) or v.shape != (B, H, Nkv, d):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    strides = None
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous() and out.is_contiguous()):
        for t in (q, k, v, out):
            if t.stride(3) != 1:
                raise ValueError("the head dim must be contiguous")
        arr = (ctypes.c_int64 * 12)(*[int(t.stride(i)) for t in (q, k, v, out) for i in range(3)])
        strides = ctypes.cast(arr, ctypes.c_void_p)
    if causal:
        _check(lib().fa_forward_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nkv, d,
                                       _dtype_code(q), float(scale), strides, FA_MASK_CAUSAL, _stream_ptr(stream)))
    else:
        _check(lib().fa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nkv, d,
                                _dtype_code(q), float(scale), strides, _stream_ptr(stream)))
    return out, lse


_host_ws = {}
_host_ws_lock = threading.Lock()


def forward_host(q, k, v, scale: float | None = None, out=None, lse=None, causal: bool = False,
                 heads_per_chunk: int = 0, device=None, stream=None):
    """Forward on host tensors: q [B,H,Nq,d], k/v [B,H,Nkv,d] contiguous CPU
    tensors (bf16 or fp32; page-locked ones let the copies overlap).  The
    library streams (b, h) chunks through a device workspace, overlapping the
    copies in and out with the forward.  Returns (O, LSE) as CPU tensors
    (page-locked when allocated here); they are valid once ``stream`` (default:
    the device's current stream) has been synchronised.  The workspace is cached
    per device and shared: eager calls from several threads or streams are
    ordered by the library, while a call captured in a CUDA graph is not, so
    replays must not overlap other calls on that device."""
    torch = _torch()
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("forward_host takes contiguous CPU tensors")
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    if k.shape != (B, H, Nkv, d) or v.shape != (B, H, Nkv, d):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=True)
    for t in (out, lse):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("out and lse must be contiguous CPU tensors")
    code = _dtype_code(q)
    with torch.cuda.device(dev):
        need = int(lib().fa_forward_host_workspace_size(B, H, Nq, Nkv, d, code, int(heads_per_chunk)))
        if need == 0:
            raise FAError(FA_ERR_INVALID_ARG, "fa_forward_host_workspace_size rejected the arguments")
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        # One cached workspace per device, shared by all threads and streams:
        # the library orders the calls that use it, and record_stream keeps the
        # caching allocator from handing it out again while a call on another
        # stream may still read it after it has been replaced by a larger one.
        with _host_ws_lock:
            ws = _host_ws.get(dev.index)
            if ws is None or ws.numel() < need:
                ws = torch.empty(need, dtype=torch.uint8, device=dev)
                _host_ws[dev.index] = ws
            _check(lib().fa_forward_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nkv, d, code,
                                         float(scale), FA_MASK_CAUSAL if causal else FA_MASK_NONE,
                                         int(heads_per_chunk), _ptr(ws), ws.numel(), _stream_ptr(s)))
            ws.record_stream(s)
    return out, lse


def forward_fp8(q8, k8, v8, q_descale: float = 1.0, k_descale: float = 1.0, v_descale: float = 1.0,
                scale: float | None = None, out=None, lse=None, causal: bool = False, stream=None):
    """FP8 forward.  q8/k8/v8: uint8 tensors of E4M3 codes [B,H,N,d] (or torch
    float8_e4m3fn); true values are descale × code value.  Returns (O bf16, LSE)."""
    torch = _torch()
    _check_cuda(q8, k8, v8)
    B, H, Nq, d = q8.shape
    Nkv = k8.shape[2]
    for t in (q8, k8, v8):
        if t.element_size() != 1 or not t.is_contiguous():
            raise ValueError("fp8 inputs must be contiguous one-byte tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device)
    _check(lib().fa_forward_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(out), _ptr(lse), B, H, Nq, Nkv, d, float(scale),
                                float(q_descale), float(k_descale), float(v_descale),
                                FA_MASK_CAUSAL if causal else FA_MASK_NONE, _stream_ptr(stream)))
    return out, lse


def decode_workspace_size(B: int, H: int, d: int, n_splits: int) -> int:
    return int(lib().fa_decode_workspace_size(B, H, d, n_splits))


def choose_splits(B: int, Hq: int, Hkv: int, Nkv: int) -> int:
    """The library's split count for a decode shape (fa_decode_choose_splits)."""
    s = int(lib().fa_decode_choose_splits(B, Hq, Hkv, Nkv))
    if s <= 0:
        raise FAError(FA_ERR_INVALID_ARG, f"no split count for B={B} Hq={Hq} Hkv={Hkv} Nkv={Nkv}")
    return s


def _check_decode_kv(q, k, v) -> int:
    """k and v must be [B, H, N_kv, d] like q's B, H, d and share its dtype; returns N_kv."""
    B, H, _, d = q.shape
    if k.dim() != 4 or tuple(k.shape[:2]) != (B, H) or k.shape[3] != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("decode inputs must be contiguous")
    return int(k.shape[2])


def decode_splitkv(q, k, v, n_splits: int | None = None, scale: float | None = None, out=None, lse=None,
                   workspace=None, stream=None):
    """Split-KV decode: q [B,H,1,d] against k/v [B,H,Nkv,d]; returns (O, LSE).
    n_splits=None takes the library's choice for the shape."""
    torch = _torch()
    _check_cuda(q, k, v)
    B, H, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query row per head")
    Nkv = _check_decode_kv(q, k, v)
    if n_splits is None:
        n_splits = choose_splits(B, H, H, Nkv)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, 1, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    need = decode_workspace_size(B, H, d, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib().fa_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nkv, d,
                                   _dtype_code(q), float(scale), int(n_splits), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def decode_splitkv_gqa(q, k, v, n_splits: int | None = None, scale: float | None = None, out=None, lse=None,
                       workspace=None, stream=None):
    """Grouped-query split-KV decode: q [B,Hq,1,d], k/v [B,Hkv,Nkv,d], Hq = G·Hkv (G <= 128).
    n_splits=None takes the library's choice for the shape."""
    torch = _torch()
    _check_cuda(q, k, v)
    B, Hq, one, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    if one != 1:
        raise ValueError("decode takes one query row per head")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("decode inputs must be contiguous")
    if n_splits is None:
        n_splits = choose_splits(B, Hq, Hkv, Nkv)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, 1, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = decode_workspace_size(B, Hq, d, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib().fa_decode_splitkv_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nkv, d,
                                       _dtype_code(q), float(scale), int(n_splits), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, n_splits: int | None = None,
                 scale: float | None = None, out=None, lse=None, workspace=None, stream=None):
    """Split-KV decode over a paged cache.

    q [B,Hq,1,d]; k_cache/v_cache [num_blocks, Hkv, block_size, d]; block_table
    [B, max_blocks] int32; seq_lens [B] int32 (device tensors).  n_splits=None
    takes the library's choice for the longest sequence the table can hold.
    """
    torch = _torch()
    _check_cuda(q, k_cache, v_cache, block_table, seq_lens)
    B, Hq, one, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if one != 1 or d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        if not t.is_contiguous():
            raise ValueError("paged decode inputs must be contiguous")
    if n_splits is None:
        n_splits = choose_splits(B, Hq, Hkv, block_table.shape[1] * bs)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, 1, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = decode_workspace_size(B, Hq, d, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib().fa_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(out),
                                 _ptr(lse), B, Hq, Hkv, NB, bs, block_table.shape[1], d, _dtype_code(q), float(scale),
                                 int(n_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)))
    return out, lse


DECODE_STATIC_SCRATCH_BYTES = 36 << 20


def decode_splitkv_noalloc(q, k, v, n_splits: int = 32, scale: float | None = None, out=None, lse=None,
                           return_lse: bool = True, stream=None):
    """Split-KV decode whose scratch is the library's fixed 36 MiB buffer.

    For callers that cannot provide device workspace (no allocator at decode
    time).  The library allocates nothing; `out` and `lse` are allocated here
    only when not given (with ``return_lse=False`` and no `lse`, the library
    writes no LSE and None is returned for it).  Calls overlapping on the GPU
    race on the buffer.
    """
    torch = _torch()
    _check_cuda(q, k, v)
    L = lib()
    fn = L.fa_decode_splitkv_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
    fn.restype = i32
    B, H, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query row per head")
    Nkv = _check_decode_kv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, 1, d), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nkv, d, _dtype_code(q), float(scale),
              int(n_splits), _stream_ptr(stream)))
    return out, lse


def backward_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(lib().fa_backward_workspace_size(B, H, N, d))


def backward(q, k, v, o, lse, do, scale: float | None = None, dq=None, dk=None, dv=None,
             workspace=None, stream=None, causal: bool = False):
    """Gradients (dQ, dK, dV) from the saved O and LSE; all [B,H,N,d] contiguous.

    ``causal`` must match the forward that produced O and LSE.
    """
    torch = _torch()
    _check_cuda(q, k, v, o, lse, do)
    B, H, N, d = q.shape
    for t in (q, k, v, o, do):
        if tuple(t.shape) != (B, H, N, d) or not t.is_contiguous():
            raise ValueError("backward tensors must be contiguous [B,H,N,d]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = backward_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
            _dtype_code(q), float(scale), _ptr(workspace), workspace.numel() * workspace.element_size())
    if causal:
        _check(lib().fa_backward_masked(*args, FA_MASK_CAUSAL, _stream_ptr(stream)))
    else:
        _check(lib().fa_backward(*args, _stream_ptr(stream)))
    return dq, dk, dv
