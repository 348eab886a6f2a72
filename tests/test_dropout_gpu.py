"""Dropout masks are bit-exact against the oracle's independent Philox, in
every kernel instance that applies them.

A wrong keep bit moves O by about 1e-3, well inside the value tolerances, so
the mask is revealed structurally instead. The oracle computes the expected
outputs on the same inputs; the zero / non-zero (or sign) pattern of the GPU
result must equal the oracle's entry for entry.

With Q = 0 (or K = 0) every score is 0, so P is uniform over the visible keys
of a row: P_ij = 1 / n_i. One-hot "selector" tensors then route one entry of
Z to one output element:

* forward: V_j = e_(j - j0) for the keys j of one d-wide block j0 .. j0+d-1
  and 0 elsewhere, so O[i, c] = Z[i, j0 + c] / (n_i (1 - p)) on visible keys;
  cycling j0 over the key range reveals all of Z. No block mask is needed,
  so the instances without one (key padding, causal) are covered too.
* dV: dO_i = e_(i - i0) on one query block, so dV[j, c] = P^[i0 + c, j].
* dQ: K = selector on a key block, V_j = dO_i = e_0. Then dP_ij =
  Z_ij / (1 - p), D_i = rowsum(dO o O) = kept_i / (n_i (1 - p)) and
  dS_ij = (Z_ij / (1 - p) - D_i) / n_i, which is > 0 for a kept entry and
  < 0 for a dropped one (when 0 < kept_i < n_i); dQ[i, c] = scale dS[i, j0+c].
  This reveals the Z applied to dP.
* dK: Q = selector on a query block (K = 0), the rest as for dQ:
  dK[j, c] = scale dS[i0 + c, j].

The d = 256 backward runs three kernels (dV, dK and dQ passes), each with its
own keep-bit indexing; the three reveals check each of them. The split-KV
forward draws its bits per key range, so it gets the forward reveal too.
"""
import numpy as np
import pytest
import torch

import io_aware_exact_08_gb300 as fa
import oracle
from workloads import random_block_mask

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@pytest.mark.parametrize("B,H,N,p,seed", [(2, 2, 512, 0.1, 1003), (1, 3, 77, 0.5, 2**63 + 5),
                                          (2, 1, 130, 0.0, 1), (1, 1, 256, 0.9, 42)])
def test_mask_hook_bit_exact(cuda_device, B, H, N, p, seed):
    z_gpu = fa.dropout_mask(B, H, N, p, seed).cpu().numpy()
    z_ref = oracle.dropout_keep(B, H, N, p, seed)
    assert np.array_equal(z_gpu, z_ref)


def _masks(B, N, variant, seed):
    """(causal, kv_len, block_mask) of a reveal case."""
    g = torch.Generator().manual_seed(seed)
    causal, kv_len, bm = False, None, None
    if variant == "kvlen":  # key padding as in the BERT-shaped workload
        kv_len = torch.randint(N // 2, N + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    elif variant == "causal":
        causal = True
    elif variant == "block":
        nb = (N + 127) // 128
        bm = random_block_mask(nb, 0.5, seed)
        if nb > 2:
            bm[1, :] = 0  # a query block that sees nothing
    else:
        raise ValueError(variant)
    return causal, kv_len, bm


def _selector(B, H, N, d, s, dt):
    """[B,H,N,d] with rows s*d .. s*d+d-1 set to e_0 .. e_(d-1), zeros elsewhere."""
    t = torch.zeros(B, H, N, d, dtype=dt)
    r0, r1 = s * d, min(N, s * d + d)
    t[:, :, r0:r1, : r1 - r0] = torch.eye(r1 - r0, dtype=dt)
    return t


def _e0(B, H, N, d, dt):
    t = torch.zeros(B, H, N, d, dtype=dt)
    t[..., 0] = 1
    return t


def _dev(t):
    return None if t is None else t.cuda().contiguous()


def _status_ok():
    torch.cuda.synchronize()
    st, site = fa.fa_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"device status {st} at site {site}"


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


FWD_CASES = [
    # d, N, variant, dtype, splits, p
    (64, 384, "kvlen", "bf16", 1, 0.1),     # the BERT-shaped workload's instance (d = 64, no block mask)
    (64, 300, "causal", "fp16", 1, 0.1),
    (64, 384, "block", "bf16", 1, 0.1),
    (128, 384, "kvlen", "bf16", 1, 0.1),
    (128, 300, "block", "fp16", 1, 0.2),
    (128, 256, "causal", "bf16", 1, 0.5),
    (256, 384, "kvlen", "bf16", 1, 0.1),
    (256, 300, "causal", "bf16", 1, 0.1),
    (256, 384, "block", "fp16", 1, 0.1),
    # split-KV forward
    (64, 640, "kvlen", "bf16", 3, 0.1),
    (64, 512, "causal", "bf16", 4, 0.1),
    (64, 512, "block", "bf16", 2, 0.1),
    (128, 512, "block", "bf16", 2, 0.1),
    (256, 384, "causal", "bf16", 2, 0.1),
    (256, 384, "block", "bf16", 3, 0.1),
    # fp32 runs on the CUDA-core kernels
    (64, 300, "kvlen", "fp32", 1, 0.1),
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: f"d{c[0]}-N{c[1]}-{c[2]}-{c[3]}-s{c[4]}-p{c[5]}")
def test_forward_reveals_the_mask(cuda_device, case):
    d, N, variant, dname, splits, p = case
    B, H, seed, scale = 2, 2, 4242 + d + N, 0.125
    dt = TORCH_DT[dname]
    causal, kv_len, bm = _masks(B, N, variant, seed)
    q = torch.zeros(B, H, N, d, dtype=dt)
    k = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(seed)).to(dt)
    kw = dict(causal=causal, block_mask=bm, block=128, kv_len=kv_len, dropout_p=p, seed=seed)
    n_kept = 0
    for s in range((N + d - 1) // d):
        v = _selector(B, H, N, d, s, dt)
        o, lse = fa.attention_fwd(_dev(q), _dev(k), _dev(v), scale=scale, causal=causal, block_mask=_dev(bm),
                                  dropout_p=p, seed=seed, kv_len=_dev(kv_len), num_splits=splits)
        _status_ok()
        o = _np(o)
        o_ref, _ = oracle.attention_fwd(q, k, v, scale, **kw)
        assert np.array_equal(o != 0, o_ref != 0), f"keep pattern differs for key block {s}"
        nz = o_ref != 0
        np.testing.assert_allclose(o[nz], o_ref[nz], rtol=1e-2)
        n_kept += int(nz.sum())
    assert n_kept > 0


BWD_CASES = [
    # d, N, variant, dtype, p
    (64, 384, "kvlen", "bf16", 0.1),    # the BERT-shaped workload's instance
    (64, 300, "causal", "fp16", 0.3),
    (64, 384, "block", "bf16", 0.1),
    (128, 384, "kvlen", "bf16", 0.1),
    (128, 300, "block", "fp16", 0.2),
    (128, 256, "causal", "bf16", 0.5),
    (256, 384, "kvlen", "bf16", 0.1),
    (256, 300, "causal", "bf16", 0.3),
    (256, 384, "block", "fp16", 0.1),
    (64, 300, "causal", "fp32", 0.3),   # CUDA-core kernels
]


def _run_bwd(q, k, v, do, scale, causal, bm, kv_len, p, seed):
    q, k, v, do = _dev(q), _dev(k), _dev(v), _dev(do)
    bm, kl = _dev(bm), _dev(kv_len)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal, block_mask=bm, dropout_p=p, seed=seed,
                              kv_len=kl)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, do, scale=scale, causal=causal, block_mask=bm, dropout_p=p,
                                  seed=seed, kv_len=kl)
    _status_ok()
    return _np(dq), _np(dk), _np(dv)


def _visible(B, H, N, kw):
    """Visible (unmasked) entries [B,H,N,N], from the oracle's probabilities."""
    z = torch.zeros(B, H, N, 1)
    vis = np.zeros((B, H, N, N), dtype=bool)
    for b in range(B):
        for h in range(H):
            _, prob = oracle.attention_probs(z, z, 1.0, head=b * H + h, causal=kw["causal"],
                                             block_mask=kw["block_mask"], block=128, kv_len=kw["kv_len"])
            vis[b, h] = prob > 0
    return vis


@pytest.mark.parametrize("grad", ["dv", "dq", "dk"])
@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"d{c[0]}-N{c[1]}-{c[2]}-{c[3]}-p{c[4]}")
def test_backward_reveals_the_mask(cuda_device, case, grad):
    d, N, variant, dname, p = case
    B, H, seed, scale = 2, 2, 777 + d + N, 0.125
    dt = TORCH_DT[dname]
    causal, kv_len, bm = _masks(B, N, variant, seed)
    kw = dict(causal=causal, block_mask=bm, block=128, kv_len=kv_len, dropout_p=p, seed=seed)
    zeros = torch.zeros(B, H, N, d, dtype=dt)
    vis = _visible(B, H, N, kw)
    n_row = vis.sum(-1)                                                     # visible keys per row
    kept_row = (vis & oracle.dropout_keep(B, H, N, p, seed).astype(bool)).sum(-1)
    checked = skipped = kept = dropped = 0
    for s in range((N + d - 1) // d):
        r0, r1 = s * d, min(N, s * d + d)
        sel = _selector(B, H, N, d, s, dt)
        e0 = _e0(B, H, N, d, dt)
        if grad == "dv":
            q, k, v, do = zeros, zeros, zeros, sel
        elif grad == "dq":
            q, k, v, do = zeros, sel, e0, e0
        else:
            q, k, v, do = sel, zeros, e0, e0
        got = dict(zip(("dq", "dk", "dv"), _run_bwd(q, k, v, do, scale, causal, bm, kv_len, p, seed)))[grad]
        ref = dict(zip(("dq", "dk", "dv"), oracle.attention_bwd(q, k, v, do, scale, **kw)))[grad]
        if grad == "dv":
            # dV[j, c] = P^[s*d + c, j]: non-zero exactly where the entry is kept and visible
            assert np.array_equal(got != 0, ref != 0), f"keep pattern differs for query block {s}"
            kept += int((ref != 0).sum())
            continue
        # per output entry: is its (i, j) visible, and the counts of row i
        # dQ[i, c] <-> (i, j = r0 + c); dK[j, c] <-> (i = r0 + c, j)
        vis_e = np.zeros((B, H, N, d), dtype=bool)
        n_e = np.zeros((B, H, N, d))
        kept_e = np.zeros((B, H, N, d))
        if grad == "dq":
            vis_e[..., : r1 - r0] = vis[..., :, r0:r1]
            n_e[:] = n_row[..., :, None]
            kept_e[:] = kept_row[..., :, None]
        else:
            vis_e[..., : r1 - r0] = np.swapaxes(vis[..., r0:r1, :], 2, 3)
            n_e[..., : r1 - r0] = n_row[..., None, r0:r1]
            kept_e[..., : r1 - r0] = kept_row[..., None, r0:r1]
        # masked entries, and rows that keep nothing (dP = 0 and D = 0), give
        # exactly 0
        zero = ~vis_e | (kept_e == 0)
        assert not got[zero].any(), f"masked entries not zero for block {s}"
        # the sign of dS: positive kept, negative dropped. The kernels form D
        # from the stored O, so entries whose oracle value is within
        # scale * 2^-6 / n_i of 0 (rows that keep all or almost all of their
        # keys) are not decided by the sign.
        with np.errstate(divide="ignore"):
            margin = scale * 2.0 ** -6 / n_e
        decide = ~zero & (np.abs(ref) >= margin)
        assert np.array_equal(np.sign(got[decide]), np.sign(ref[decide])), f"keep pattern differs for block {s}"
        checked += int(decide.sum())
        skipped += int((~zero & ~decide).sum())
        kept += int((decide & (ref > 0)).sum())
        dropped += int((decide & (ref < 0)).sum())
    assert kept > 0
    if grad != "dv":
        assert dropped > 0
        assert skipped <= 0.02 * (checked + skipped), (checked, skipped)
