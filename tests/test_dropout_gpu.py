"""Dropout masks are bit-exact against the oracle's independent Philox.

1. fa_dropout_mask equals the oracle's keep mask Z.
2. The production forward reveals Z: with Q = 0 the probabilities are uniform
   over visible keys, a block mask leaves one key block per query block, and
   V_j = e_(j mod 128) (d = 128) makes O[i, c] = Z[i, j(c)] / (n (1 - p)),
   where j(c) is the key of that block with j mod 128 = c. Cycling the
   selected block covers every (query block, key block) pair.
3. The backward reveals Z^T the same way through dV with dO_i = e_(i mod 128).
"""
import numpy as np
import pytest
import torch

import io_aware_exact_08_gb300 as fa
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,p,seed", [(2, 2, 512, 0.1, 1003), (1, 3, 77, 0.5, 2**63 + 5),
                                          (2, 1, 130, 0.0, 1), (1, 1, 256, 0.9, 42)])
def test_mask_hook_bit_exact(cuda_device, B, H, N, p, seed):
    z_gpu = fa.dropout_mask(B, H, N, p, seed).cpu().numpy()
    z_ref = oracle.dropout_keep(B, H, N, p, seed)
    assert np.array_equal(z_gpu, z_ref)


def _reveal_inputs(B, H, N, d, shift, dt=torch.bfloat16):
    nb = N // 128
    q = torch.zeros(B, H, N, d, dtype=dt)
    k = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(3)).to(dt)
    v = torch.zeros(B, H, N, d, dtype=dt)
    for j in range(N):
        v[:, :, j, j % d] = 1.0
    bm = torch.zeros(nb, nb, dtype=torch.uint8)
    for i in range(nb):
        bm[i, (i + shift) % nb] = 1
    return q, k, v, bm


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("shift", [0, 1, 2, 3])
def test_forward_applies_the_same_mask(cuda_device, shift, dt):
    B, H, N, d, p, seed = 2, 2, 512, 128, 0.1, 1003
    q, k, v, bm = _reveal_inputs(B, H, N, d, shift, dt)
    dev = lambda t: t.cuda().contiguous()
    o, lse = fa.attention_fwd(dev(q), dev(k), dev(v), scale=0.125, block_mask=dev(bm), dropout_p=p, seed=seed)
    o = o.float().cpu().numpy()
    z = oracle.dropout_keep(B, H, N, p, seed)
    nb = N // 128
    for ib in range(nb):
        jb = (ib + shift) % nb
        rows = slice(ib * 128, ib * 128 + 128)
        keys = slice(jb * 128, jb * 128 + 128)
        got = o[:, :, rows, :] != 0  # column c <-> key jb*128 + c
        assert np.array_equal(got, z[:, :, rows, keys].astype(bool))
        kept = o[:, :, rows, :][got]
        assert np.allclose(kept, 1.0 / (128 * (1 - p)), rtol=1e-2)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("shift", [0, 3])
def test_backward_applies_the_same_mask(cuda_device, shift, dt):
    B, H, N, d, p, seed = 2, 2, 512, 128, 0.1, 77
    q, k, v, bm = _reveal_inputs(B, H, N, d, shift, dt)
    do = torch.zeros(B, H, N, d, dtype=dt)
    for i in range(N):
        do[:, :, i, i % d] = 1.0
    dev = lambda t: t.cuda().contiguous()
    q, k, v, bm, do = dev(q), dev(k), dev(v), dev(bm), dev(do)
    o, lse = fa.attention_fwd(q, k, v, scale=0.125, block_mask=bm, dropout_p=p, seed=seed)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, do, scale=0.125, block_mask=bm, dropout_p=p, seed=seed)
    dv = dv.float().cpu().numpy()
    z = oracle.dropout_keep(B, H, N, p, seed)
    nb = N // 128
    for ib in range(nb):
        jb = (ib + shift) % nb
        rows = slice(ib * 128, ib * 128 + 128)
        keys = slice(jb * 128, jb * 128 + 128)
        # dV[j, c] = P^[i(c), j] with i(c) = ib*128 + c
        got = dv[:, :, keys, :] != 0
        assert np.array_equal(got, np.swapaxes(z[:, :, rows, keys], 2, 3).astype(bool))
