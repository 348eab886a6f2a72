"""Pins for the oracle's Philox4x32-10 and dropout keep rule.

The oracle implements Philox4x32-10 from Salmon et al. (SC'11). Here it is
compared with an independent library implementation, Triton's Philox, run on
the CPU through Triton's interpreter, over many counters and keys. The keep
rule (keep iff u >= floor(p * 2^32)) is checked for its closed-form threshold
and its keep rate.
"""
import os

import numpy as np
import pytest

import oracle


def _triton_philox(counters, seed):
    os.environ["TRITON_INTERPRET"] = "1"
    triton = pytest.importorskip("triton")
    import torch
    import triton.language
    import triton.language.random
    globals()["tl"] = triton.language

    @triton.jit
    def kern(c_ptr, out_ptr, seed, n, BLOCK: tl.constexpr):
        offs = tl.program_id(0) * BLOCK + tl.arange(0, BLOCK)
        msk = offs < n
        c0 = tl.load(c_ptr + offs * 4 + 0, mask=msk).to(tl.uint32)
        c1 = tl.load(c_ptr + offs * 4 + 1, mask=msk).to(tl.uint32)
        c2 = tl.load(c_ptr + offs * 4 + 2, mask=msk).to(tl.uint32)
        c3 = tl.load(c_ptr + offs * 4 + 3, mask=msk).to(tl.uint32)
        r0, r1, r2, r3 = tl.random.philox(seed, c0, c1, c2, c3, 10)
        tl.store(out_ptr + offs * 4 + 0, r0.to(tl.int64), mask=msk)
        tl.store(out_ptr + offs * 4 + 1, r1.to(tl.int64), mask=msk)
        tl.store(out_ptr + offs * 4 + 2, r2.to(tl.int64), mask=msk)
        tl.store(out_ptr + offs * 4 + 3, r3.to(tl.int64), mask=msk)

    n = counters.shape[0]
    c = torch.from_numpy(counters.astype(np.int64))
    out = torch.zeros((n, 4), dtype=torch.int64)
    kern[(triton.cdiv(n, 256),)](c, out, seed, n, BLOCK=256)
    return (out.numpy() & 0xFFFFFFFF).astype(np.uint32)


@pytest.mark.parametrize("seed", [0, 1003, 0x123456789ABCDEF0, 2**64 - 1])
def test_philox_matches_triton_library(seed):
    rng = np.random.default_rng(seed % 1000)
    counters = rng.integers(0, 2**32, size=(512, 4), dtype=np.uint64)
    counters[:8] = [[0, 0, 0, 0], [1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0],
                    [0, 0, 0, 1], [2**32 - 1] * 4, [5, 7, 3, 1], [127, 511, 15, 31]]
    ref = _triton_philox(counters, seed)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint32)
    got = np.stack([oracle.philox4x32_10(c, key) for c in counters.astype(np.uint32)])
    assert np.array_equal(got, ref)


def test_keep_threshold_closed_form():
    assert oracle.keep_threshold(0.0) == 0
    assert oracle.keep_threshold(0.1) == 429496729
    assert oracle.keep_threshold(0.5) == 2**31
    assert oracle.keep_threshold(0.9999999999999999) == 2**32 - 1


def test_keep_mask_uses_counter_layout():
    """Z[b,h,i,j] is word j%4 of Philox((j//4, i, h, b), (lo32, hi32)) >= T."""
    B, H, N, p, seed = 2, 3, 10, 0.37, 0xDEADBEEF12345
    z = oracle.dropout_keep(B, H, N, p, seed)
    thr = oracle.keep_threshold(p)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                for j in range(N):
                    r = oracle.philox4x32_10([j // 4, i, h, b], key)
                    assert z[b, h, i, j] == (int(r[j % 4]) >= thr)


@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_keep_rate(p):
    z = oracle.dropout_keep(2, 2, 256, p, 42)
    rate = z.mean()
    assert abs(rate - (1 - p)) < 5 * np.sqrt(p * (1 - p) / z.size) + 1e-12
    if p == 0.0:
        assert z.all()
