"""Exact IO-aware attention for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in ``include/fa.h`` (``libfa_gb300.so``,
built in-tree by ``build.py``). The functions ``fa_fwd``, ``fa_fwd_splitkv``,
``fa_fwd_splitkv_workspace_size``, ``fa_bwd``, ``fa_bwd_workspace_size``,
``fa_dropout_mask``, ``fa_check_device_status``, ``fa_status_string``,
``fa_set_kernel_path`` and ``fa_fwd_bwd_host`` take the same arguments as
their C counterparts (pointers as integers, sizes, a stream handle) and only
marshal them. ``attention_fwd`` / ``attention_bwd``, ``attention_fwd_bwd_host``
(a step on host tensors) and ``FlashAttention`` add the tensor plumbing:
PyTorch allocates the outputs and the workspace and supplies the current
stream; every step of the computation runs in the library's CUDA kernels.

There is no CPU fallback: if the library cannot be loaded, importing the
binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "FA_BF16", "FA_FP32", "FA_FP16", "FaError", "load_library", "library_path",
    "fa_fwd", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size", "fa_bwd", "fa_bwd_workspace_size", "fa_dropout_mask",
    "fa_check_device_status", "fa_status_string", "fa_set_kernel_path", "fa_launch_count",
    "fa_set_main_kernel_events", "fa_bwd_noalloc", "fa_fwd_fp8", "attention_fwd_fp8", "fa_ex2_probe", "FA_BWD_NOALLOC_SCRATCH_BYTES", "attention_fwd", "attention_bwd", "dropout_mask", "FlashAttention", "attention",
    "fa_fwd_bwd_host", "fa_fwd_bwd_host_workspace_size", "fa_fwd_bwd_host_chunks", "attention_fwd_bwd_host",
]

FA_BF16 = 0
FA_FP32 = 1
FA_FP16 = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "libfa_gb300.so")
_lib = None
_lock = threading.Lock()

EXPORTED = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_dropout_mask",
            "fa_check_device_status", "fa_status_string", "fa_set_kernel_path", "fa_launch_count",
            "fa_bwd_noalloc", "fa_test_wait_timeout", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size",
            "fa_set_main_kernel_events", "fa_fwd_fp8", "fa_ex2_probe", "fa_fwd_bwd_host",
            "fa_fwd_bwd_host_workspace_size", "fa_fwd_bwd_host_chunks")

# Size of the fixed device array fa_bwd_noalloc takes its workspace from.
FA_BWD_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def load_library(build_if_missing: bool = True):
    """Loads libfa_gb300.so (building it with nvcc if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            if not build_if_missing:
                raise RuntimeError(f"attention library not built: {_LIB_PATH}")
            from . import build as _build
            _build.build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
        lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, F, I, P, F, U64, I, P, P]
        lib.fa_fwd.restype = I
        lib.fa_fwd_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, P, P]
        lib.fa_fwd_fp8.restype = I
        lib.fa_fwd_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, F, I, P, F, U64, I, P, I, P, SZ, P]
        lib.fa_fwd_splitkv.restype = I
        lib.fa_fwd_splitkv_workspace_size.argtypes = [I, I, I, I, I]
        lib.fa_fwd_splitkv_workspace_size.restype = SZ
        lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, F, U64, I, P, P, SZ, P]
        lib.fa_bwd.restype = I
        lib.fa_bwd_workspace_size.argtypes = [I, I, I, I]
        lib.fa_bwd_workspace_size.restype = SZ
        lib.fa_dropout_mask.argtypes = [P, I, I, I, F, U64, P]
        lib.fa_dropout_mask.restype = I
        lib.fa_check_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        lib.fa_check_device_status.restype = I
        lib.fa_status_string.argtypes = [I]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_set_kernel_path.argtypes = [I]
        lib.fa_set_kernel_path.restype = I
        lib.fa_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, F, U64, I, P, P]
        lib.fa_bwd_noalloc.restype = I
        lib.fa_fwd_bwd_host.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, F, U64, I, P, I, P, SZ, P]
        lib.fa_fwd_bwd_host.restype = I
        lib.fa_fwd_bwd_host_workspace_size.argtypes = [I, I, I, I, I, P, F, P, I]
        lib.fa_fwd_bwd_host_workspace_size.restype = SZ
        lib.fa_fwd_bwd_host_chunks.argtypes = [I, I, I, P, F, I, P, I]
        lib.fa_fwd_bwd_host_chunks.restype = I
        lib.fa_test_wait_timeout.argtypes = [U64, P]
        lib.fa_test_wait_timeout.restype = I
        lib.fa_ex2_probe.argtypes = [P, I, I, P]
        lib.fa_ex2_probe.restype = I
        lib.fa_set_main_kernel_events.argtypes = [P, P]
        lib.fa_set_main_kernel_events.restype = I
        lib.fa_launch_count.argtypes = []
        lib.fa_launch_count.restype = ctypes.c_uint64
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# C ABI, same names and argument order as include/fa.h.
# ---------------------------------------------------------------------------

def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, block_mask, dropout_p, seed, dtype, kv_len, stream):
    return load_library().fa_fwd(q, k, v, o, lse, B, H, N, d, scale, int(causal), block_mask, dropout_p,
                                 seed & 0xFFFFFFFFFFFFFFFF, dtype, kv_len, stream)


def fa_fwd_fp8(q, k, vt, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale, causal, block_mask, kv_len,
               stream):
    return load_library().fa_fwd_fp8(q, k, vt, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale,
                                     int(causal), block_mask, kv_len, stream)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, block_mask, dropout_p, seed, dtype, kv_len,
                   n_splits, workspace, workspace_bytes, stream):
    return load_library().fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, int(causal), block_mask, dropout_p,
                                         seed & 0xFFFFFFFFFFFFFFFF, dtype, kv_len, n_splits, workspace,
                                         workspace_bytes, stream)


def fa_fwd_splitkv_workspace_size(B, H, N, d, n_splits):
    return load_library().fa_fwd_splitkv_workspace_size(B, H, N, d, n_splits)


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, block_mask, dropout_p, seed, dtype,
           kv_len, workspace, workspace_bytes, stream):
    return load_library().fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, int(causal), block_mask,
                                 dropout_p, seed & 0xFFFFFFFFFFFFFFFF, dtype, kv_len, workspace,
                                 workspace_bytes, stream)


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, block_mask, dropout_p, seed,
                   dtype, kv_len, stream):
    """fa_bwd without a caller-provided workspace: for callers that cannot
    allocate device memory (their framework's allocator owns the device, or
    allocation is not allowed on their path). The workspace is a fixed
    FA_BWD_NOALLOC_SCRATCH_BYTES array inside the library; larger problems
    are refused with FA_ERR_WORKSPACE, and overlapping calls race on it."""
    return load_library().fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, int(causal),
                                         block_mask, dropout_p, seed & 0xFFFFFFFFFFFFFFFF, dtype, kv_len, stream)


def fa_bwd_workspace_size(B, H, N, d):
    return load_library().fa_bwd_workspace_size(B, H, N, d)


def fa_fwd_bwd_host(q, k, v, dO, o, lse, dq, dk, dv, B, H, N, d, scale, causal, block_mask, dropout_p, seed,
                    dtype, kv_len, chunk_heads, workspace, workspace_bytes, stream):
    """Forward and backward on HOST buffers (addresses as integers), the
    copies overlapped with the kernels chunk by chunk; see include/fa.h."""
    return load_library().fa_fwd_bwd_host(q, k, v, dO, o, lse, dq, dk, dv, B, H, N, d, scale, int(causal),
                                          block_mask, dropout_p, seed & 0xFFFFFFFFFFFFFFFF, dtype, kv_len,
                                          int(chunk_heads), workspace, workspace_bytes, stream)


def fa_fwd_bwd_host_workspace_size(B, H, N, d, dtype, block_mask, dropout_p, kv_len, chunk_heads):
    return load_library().fa_fwd_bwd_host_workspace_size(B, H, N, d, dtype, block_mask, float(dropout_p), kv_len,
                                                         int(chunk_heads))


def fa_fwd_bwd_host_chunks(B, H, N, kv_len, dropout_p, chunk_heads):
    """The chunks fa_fwd_bwd_host uses: a list of (first head, B, H, first
    batch). kv_len only matters through being None or not."""
    lib = load_library()
    n = lib.fa_fwd_bwd_host_chunks(B, H, N, kv_len, float(dropout_p), int(chunk_heads), None, 0)
    if n < 0:
        raise FaError(n, "fa_fwd_bwd_host_chunks")
    buf = (ctypes.c_int * (4 * max(n, 1)))()
    lib.fa_fwd_bwd_host_chunks(B, H, N, kv_len, float(dropout_p), int(chunk_heads), buf, n)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]


def fa_dropout_mask(keep, B, H, N, p, seed, stream):
    return load_library().fa_dropout_mask(keep, B, H, N, p, seed & 0xFFFFFFFFFFFFFFFF, stream)


def fa_check_device_status(stream):
    """Returns (status, site)."""
    site = ctypes.c_int(0)
    st = load_library().fa_check_device_status(stream, ctypes.byref(site))
    return st, site.value


def fa_status_string(status):
    return load_library().fa_status_string(int(status)).decode()


def fa_set_kernel_path(path):
    return load_library().fa_set_kernel_path(int(path))


def fa_test_wait_timeout(limit_ns, stream):
    """Runs the bounded-wait failure path once (see include/fa.h)."""
    return load_library().fa_test_wait_timeout(int(limit_ns), stream)


def fa_launch_count():
    return int(load_library().fa_launch_count())


def fa_ex2_probe(out, n_blocks, iters, stream):
    """Launches the exponential-throughput probe (see include/fa.h)."""
    return load_library().fa_ex2_probe(out, int(n_blocks), int(iters), stream)


def fa_set_main_kernel_events(ev_start, ev_stop):
    """Events (cudaEvent_t handles as integers, or None) recorded around the
    main kernel of the following calls; see include/fa.h."""
    return load_library().fa_set_main_kernel_events(ev_start, ev_stop)


# ---------------------------------------------------------------------------
# Tensor plumbing (PyTorch for device memory and streams only).
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_FP32
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16, float16 or float32")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t, name, like=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B,H,N,d]")
    if like is not None and (t.shape != like.shape or t.dtype != like.dtype):
        raise ValueError(f"{name} must match q in shape and dtype")


def _check_masks(block_mask, kv_len, B, N, device):
    """The optional masks must be what the kernels read: block_mask uint8
    [ceil(N/128)^2] and kv_len int32 [B], contiguous, on q's device."""
    torch = _torch()
    nb = (N + 127) // 128
    for name, t, dt, numel in (("block_mask", block_mask, torch.uint8, nb * nb), ("kv_len", kv_len, torch.int32, B)):
        if t is None:
            continue
        if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device or not t.is_contiguous() or
                t.dtype != dt or t.numel() != numel):
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor of {numel} elements on {device}")


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def attention_fwd(q, k, v, scale=None, causal=False, block_mask=None, dropout_p=0.0, seed=0, kv_len=None,
                  out=None, lse=None, stream=None, num_splits=1):
    """O, LSE = attention(q, k, v) for [B,H,N,d] CUDA tensors (bf16, fp16 or fp32).

    num_splits > 1 runs the split-KV forward (fa_fwd_splitkv) with a
    workspace allocated here."""
    torch = _torch()
    _check(q, "q")
    _check(k, "k", q)
    _check(v, "v", q)
    B, H, N, d = q.shape
    _check_masks(block_mask, kv_len, B, N, q.device)
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if num_splits > 1:
        wsb = fa_fwd_splitkv_workspace_size(B, H, N, d, int(num_splits))
        if wsb == 0 and N > 0:
            raise FaError(-1, "fa_fwd_splitkv_workspace_size")
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=q.device)
        rc = fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, scale, causal,
                            _ptr(block_mask), float(dropout_p), int(seed), _dtype_code(q), _ptr(kv_len),
                            int(num_splits), ws.data_ptr(), wsb, _stream(stream))
        if rc != 0:
            raise FaError(rc, "fa_fwd_splitkv")
        return o, l
    rc = fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, scale, causal, _ptr(block_mask),
                float(dropout_p), int(seed), _dtype_code(q), _ptr(kv_len), _stream(stream))
    if rc != 0:
        raise FaError(rc, "fa_fwd")
    return o, l


def attention_fwd_fp8(q8, k8, vt8, descale_q, descale_k, descale_v, scale=None, causal=False, block_mask=None,
                      kv_len=None, stream=None):
    """O (bf16), LSE = attention on E4M3 inputs (fa_fwd_fp8).

    q8, k8: uint8 E4M3 codes [B,H,N,128]; vt8: V's codes transposed,
    [B,H,128,N]; descale_*: fp32 [B*H] per-head factors (real value =
    code * factor). All CUDA tensors."""
    torch = _torch()
    for name, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous() or t.dtype != torch.uint8:
            raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor of E4M3 codes")
    for name, t in (("descale_q", descale_q), ("descale_k", descale_k), ("descale_v", descale_v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
            raise ValueError(f"{name} must be a float32 CUDA tensor [B*H]")
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or tuple(vt8.shape) != (B, H, d, N):
        raise ValueError("k8 must match q8 and vt8 must be [B,H,d,N]")
    _check_masks(block_mask, kv_len, B, N, q8.device)
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    l = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    rc = fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(descale_q), _ptr(descale_k), _ptr(descale_v), _ptr(o),
                    _ptr(l), B, H, N, d, scale, causal, _ptr(block_mask), _ptr(kv_len), _stream(stream))
    if rc != 0:
        raise FaError(rc, "fa_fwd_fp8")
    return o, l


def attention_bwd(q, k, v, o, lse, do, scale=None, causal=False, block_mask=None, dropout_p=0.0, seed=0,
                  kv_len=None, workspace=None, stream=None, dq=None, dk=None, dv=None):
    """dQ, dK, dV for the forward above (same masks, scale and dropout)."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check(t, name, q)
    B, H, N, d = q.shape
    _check_masks(block_mask, kv_len, B, N, q.device)
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    need = fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device) if workspace is None else workspace
    rc = fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                B, H, N, d, scale, causal, _ptr(block_mask), float(dropout_p), int(seed), _dtype_code(q),
                _ptr(kv_len), _ptr(ws), ws.numel(), _stream(stream))
    if rc != 0:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def attention_fwd_bwd_host(q, k, v, do, scale=None, causal=False, block_mask=None, dropout_p=0.0, seed=0,
                           kv_len=None, chunk_heads=0, out=None, workspace=None, device=None, stream=None):
    """O, LSE, dQ, dK, dV for [B,H,N,d] tensors in HOST memory (fa_fwd_bwd_host).

    q, k, v, do: contiguous CPU tensors (page-locked, e.g. .pin_memory(),
    for the copies to overlap the kernels); block_mask (uint8) and kv_len
    (int32) are CPU tensors too. out: optional (o, lse, dq, dk, dv) CPU
    tensors to write; by default they are allocated page-locked. The
    workspace is device memory on `device` (default: the current CUDA
    device), allocated here unless given. Returns (o, lse, dq, dk, dv); they
    are ready once `stream` (default: the current stream) has caught up."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor [B,H,N,d]")
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    B, H, N, d = q.shape
    nb = (N + 127) // 128
    for name, t, dt, numel in (("block_mask", block_mask, torch.uint8, nb * nb), ("kv_len", kv_len, torch.int32, B)):
        if t is not None and (not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous() or
                              t.dtype != dt or t.numel() != numel):
            raise ValueError(f"{name} must be a contiguous CPU {dt} tensor of {numel} elements")
    dt = _dtype_code(q)
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if out is None:
        pin = q.is_pinned()
        mk = lambda shape, dtype: torch.empty(shape, dtype=dtype, pin_memory=pin)
        out = (mk(q.shape, q.dtype), mk((B, H, N), torch.float32), mk(q.shape, q.dtype), mk(q.shape, q.dtype),
               mk(q.shape, q.dtype))
    o, l, dq, dk, dv = out
    need = fa_fwd_bwd_host_workspace_size(B, H, N, d, dt, _ptr(block_mask), dropout_p, _ptr(kv_len),
                                          chunk_heads)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev) if workspace is None else workspace
    with torch.cuda.device(dev):
        rc = fa_fwd_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(o), _ptr(l), _ptr(dq), _ptr(dk), _ptr(dv),
                             B, H, N, d, scale, causal, _ptr(block_mask), float(dropout_p), int(seed), dt,
                             _ptr(kv_len), int(chunk_heads), _ptr(ws), ws.numel(), _stream(stream))
    if rc != 0:
        raise FaError(rc, "fa_fwd_bwd_host")
    return o, l, dq, dk, dv


def dropout_mask(B, H, N, p, seed, device="cuda", stream=None):
    """The keep mask Z (uint8 [B,H,N,N]) the kernels apply for (p, seed)."""
    torch = _torch()
    z = torch.empty((B, H, N, N), dtype=torch.uint8, device=device)
    rc = fa_dropout_mask(_ptr(z), B, H, N, float(p), int(seed), _stream(stream))
    if rc != 0:
        raise FaError(rc, "fa_dropout_mask")
    return z


def _make_autograd():
    torch = _torch()

    class FlashAttention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, scale, causal, block_mask, dropout_p, seed, kv_len):
            o, lse = attention_fwd(q, k, v, scale, causal, block_mask, dropout_p, seed, kv_len)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.args = (scale, causal, block_mask, dropout_p, seed, kv_len)
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            scale, causal, block_mask, dropout_p, seed, kv_len = ctx.args
            dq, dk, dv = attention_bwd(q, k, v, o, lse, do.contiguous(), scale, causal, block_mask, dropout_p,
                                       seed, kv_len)
            return dq, dk, dv, None, None, None, None, None, None

    return FlashAttention


_autograd_cls = None


def __getattr__(name):
    global _autograd_cls
    if name == "FlashAttention":
        if _autograd_cls is None:
            _autograd_cls = _make_autograd()
        return _autograd_cls
    raise AttributeError(name)


def attention(q, k, v, scale=None, causal=False, block_mask=None, dropout_p=0.0, seed=0, kv_len=None):
    """Differentiable exact attention (autograd over the library's kernels)."""
    B, H, N, d = q.shape
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    return __getattr__("FlashAttention").apply(q, k, v, scale, causal, block_mask, dropout_p, seed, kv_len)
