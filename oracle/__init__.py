"""fp64 CPU oracle for exact attention (forward, backward, dropout mask).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the CPU-baseline leg of ``bench.py``; never by the product library. The
arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over rows); this
module builds it with gcc and marshals numpy arrays into it.

Everything here states the plain definition of attention (standard attention:
S = scale*Q K^T with masks, P = softmax(S), O = P V) and its closed-form
gradients; see the header of ``oracle.c`` for the readings of open points.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        U64 = ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_keep_threshold.argtypes = [D]
        lib.oracle_keep_threshold.restype = U64
        lib.oracle_dropout_keep.argtypes = [P, I, I, I, D, U64]
        lib.oracle_dropout_keep.restype = None
        common = [I, I, I, I, D, I, P, I, P, D, U64, P, I, I]
        lib.oracle_fwd.argtypes = [P, P, P, P, P] + common
        lib.oracle_fwd.restype = I
        lib.oracle_bwd.argtypes = [P, P, P, P, P, P, P] + common
        lib.oracle_bwd.restype = I
        lib.oracle_probs.argtypes = [P, P, P, P, I, I, I, I, D, I, P, I, P, I]
        lib.oracle_probs.restype = I
        lib.oracle_e4m3_dequantize.argtypes = [P, P, ctypes.c_long, ctypes.c_long, ctypes.c_long, P]
        lib.oracle_e4m3_dequantize.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = I
        _lib = lib
        return lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().to(dtype=__import__("torch").float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _u8(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint8))


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _load().oracle_max_threads()


def philox4x32_10(counter, key):
    """Philox4x32-10 of one 4-word counter and 2-word key (uint32 each)."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def keep_threshold(p: float) -> int:
    return int(_load().oracle_keep_threshold(float(p)))


def dropout_keep(B, H, N, p, seed):
    """Keep mask Z (uint8 [B,H,N,N]) of the dropout contract."""
    z = np.zeros((B, H, N, N), dtype=np.uint8)
    _load().oracle_dropout_keep(_ptr(z), B, H, N, float(p), int(seed))
    return z


def _common(shape, scale, causal, block_mask, block, kv_len, dropout_p, seed, heads, nthreads):
    B, H, N, d = shape
    bm = _u8(block_mask)
    kl = _i32(kv_len)
    hd = None if heads is None else _i32(heads)
    nh = 0 if hd is None else int(hd.size)
    args = [B, H, N, d, float(scale), int(bool(causal)), _ptr(bm), int(block), _ptr(kl),
            float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(hd), nh, int(nthreads)]
    return args, (bm, kl, hd)


def attention_fwd(q, k, v, scale, causal=False, block_mask=None, block=128, kv_len=None,
                  dropout_p=0.0, seed=0, heads=None, nthreads=0):
    """Returns (O, LSE) in fp64: O [B,H,N,d], LSE [B,H,N].

    ``heads`` (flat indices b*H+h) restricts the work to those heads; the
    other entries of the outputs are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    o = np.full(q.shape, np.nan)
    lse = np.full(q.shape[:3], np.nan)
    args, keep = _common(q.shape, scale, causal, block_mask, block, kv_len, dropout_p, seed, heads, nthreads)
    rc = _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), *args)
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed ({rc})")
    return o, lse


def attention_bwd(q, k, v, do, scale, causal=False, block_mask=None, block=128, kv_len=None,
                  dropout_p=0.0, seed=0, heads=None, nthreads=0):
    """Returns (dQ, dK, dV) in fp64, each [B,H,N,d]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq = np.full(q.shape, np.nan)
    dk = np.full(q.shape, np.nan)
    dv = np.full(q.shape, np.nan)
    args, keep = _common(q.shape, scale, causal, block_mask, block, kv_len, dropout_p, seed, heads, nthreads)
    rc = _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), *args)
    if rc != 0:
        raise RuntimeError(f"oracle_bwd failed ({rc})")
    return dq, dk, dv


def attention_probs(q, k, scale, head=0, causal=False, block_mask=None, block=128, kv_len=None):
    """Scores S and probabilities P (pre-dropout) of one head, each [N,N]."""
    q, k = _f64(q), _f64(k)
    B, H, N, d = q.shape
    s = np.zeros((N, N))
    p = np.zeros((N, N))
    bm = _u8(block_mask)
    kl = _i32(kv_len)
    _load().oracle_probs(_ptr(q), _ptr(k), _ptr(s), _ptr(p), B, H, N, d, float(scale),
                         int(bool(causal)), _ptr(bm), int(block), _ptr(kl), int(head))
    return s, p


def e4m3_dequantize(codes, descale=None, rows_per_scale=None):
    """Decodes E4M3 bytes (uint8 array of shape [..., n]) to fp64, each block
    of ``rows_per_scale`` rows multiplied by its factor in ``descale``
    (one factor per head for [B,H,N,d]: rows_per_scale = N). Without
    ``descale`` the plain decoded values are returned."""
    u = _u8(codes)
    shape = u.shape
    row_len = shape[-1] if u.ndim else 1
    rows = u.size // max(row_len, 1)
    if descale is None:
        ds = np.ones(1)
        rows_per_scale = rows
    else:
        ds = _f64(descale).reshape(-1)
        rows_per_scale = rows // ds.size if rows_per_scale is None else int(rows_per_scale)
        assert rows_per_scale * ds.size == rows, "descale does not divide the rows"
    out = np.empty(shape, dtype=np.float64)
    _load().oracle_e4m3_dequantize(_ptr(u), _ptr(out), int(ds.size), int(rows_per_scale), int(row_len), _ptr(ds))
    return out


def attention_fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, scale, causal=False, block_mask=None,
                      block=128, kv_len=None, heads=None, nthreads=0):
    """Forward attention on E4M3 inputs: q8, k8, v8 are uint8 codes
    [B,H,N,d] (V in its natural layout) with one dequantisation factor per
    head (fp32 or fp64 arrays of B*H). The inputs are decoded exactly and
    scaled, then the fp64 definition runs on them: (O, LSE) in fp64."""
    q8, k8, v8 = _u8(q8), _u8(k8), _u8(v8)
    N = q8.shape[2]
    q = e4m3_dequantize(q8, descale_q, N)
    k = e4m3_dequantize(k8, descale_k, N)
    v = e4m3_dequantize(v8, descale_v, N)
    return attention_fwd(q, k, v, scale, causal=causal, block_mask=block_mask, block=block, kv_len=kv_len,
                         heads=heads, nthreads=nthreads)
