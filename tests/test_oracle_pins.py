"""Pins for the fp64 oracle: facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the pages'
block-update rule and two-block merge identity written out here, row sums,
finite differences of its own forward, closed-form special cases, and
PyTorch's fp64 CPU attention with autograd (a library reduction).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import band_butterfly_block_mask, random_block_mask


def _rand(shape, seed, dtype=np.float64):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape).astype(dtype)


def _mask_bruteforce(N, causal, kv_len_b, block_mask, block):
    """Boolean [N,N], True where the key is visible, from the set definitions."""
    vis = np.ones((N, N), dtype=bool)
    for i in range(N):
        for j in range(N):
            if causal and j > i:
                vis[i, j] = False
            if kv_len_b is not None and j >= kv_len_b:
                vis[i, j] = False
            if block_mask is not None and not block_mask[i // block, j // block]:
                vis[i, j] = False
    return vis


# --------------------------------------------------------------------------
# Online softmax: the pages' merge identity and block update, written here.
# --------------------------------------------------------------------------

def _stats(x):
    m = np.max(x)
    return m, np.sum(np.exp(x - m))


def test_two_block_merge_identity():
    """m(x) = max(m1, m2); l(x) = e^{m1-m} l1 + e^{m2-m} l2 equals the direct
    statistics ("FlashAttention: Fast and Memory-Efficient Exact Attention
    with IO-Awareness", section "Pelacakan Softmax Inkremental")."""
    rng = np.random.default_rng(7)
    for n1, n2 in [(1, 1), (5, 11), (64, 64), (3, 200)]:
        x = rng.standard_normal(n1 + n2) * 6
        m1, l1 = _stats(x[:n1])
        m2, l2 = _stats(x[n1:])
        m = max(m1, m2)
        l = math.exp(m1 - m) * l1 + math.exp(m2 - m) * l2
        md, ld = _stats(x)
        assert m == md
        assert abs(l - ld) <= 1e-12 * ld
        # softmax = f(x)/l(x) with f rescaled per block ("FlashAttention" blog
        # post, section "Tiling")
        f = np.concatenate([math.exp(m1 - m) * np.exp(x[:n1] - m1),
                            math.exp(m2 - m) * np.exp(x[n1:] - m2)])
        ref = np.exp(x - md) / ld
        assert np.max(np.abs(f / l - ref)) <= 1e-14


def _tiled_forward(q, k, v, scale, Bc, vis=None):
    """The pages' per-block update (steps 1-4 of "Metode"), one head, fp64."""
    N, d = q.shape
    O = np.zeros((N, d))
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    for j0 in range(0, N, Bc):
        S = scale * q @ k[j0:j0 + Bc].T
        if vis is not None:
            S = np.where(vis[:, j0:j0 + Bc], S, -np.inf)
        mt = S.max(axis=1)
        with np.errstate(invalid="ignore"):
            Pt = np.where(np.isfinite(S), np.exp(S - mt[:, None]), 0.0)
        lt = Pt.sum(axis=1)
        mn = np.maximum(m, mt)
        with np.errstate(invalid="ignore"):
            a = np.where(np.isfinite(m), np.exp(m - mn), 0.0)
            bb = np.where(np.isfinite(mt), np.exp(mt - mn), 0.0)
        ln = a * l + bb * lt
        with np.errstate(invalid="ignore", divide="ignore"):
            O = np.where(ln[:, None] > 0,
                         (l * a)[:, None] * O + bb[:, None] * (Pt @ v[j0:j0 + Bc]),
                         0.0)
            O = np.where(ln[:, None] > 0, O / np.where(ln > 0, ln, 1.0)[:, None], 0.0)
        m, l = mn, ln
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, lse


@pytest.mark.parametrize("N,d,Bc,causal", [(64, 16, 32, False), (100, 8, 16, True),
                                           (37, 5, 8, False), (130, 16, 64, True)])
def test_block_update_matches_oracle(N, d, Bc, causal):
    q, k, v = (_rand((1, 1, N, d), s) for s in (1, 2, 3))
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, scale, causal=causal)
    vis = _mask_bruteforce(N, causal, None, None, 1) if causal else None
    ot, lt = _tiled_forward(q[0, 0], k[0, 0], v[0, 0], scale, Bc, vis)
    assert np.max(np.abs(o[0, 0] - ot)) <= 1e-12
    assert np.max(np.abs(lse[0, 0] - lt)) <= 1e-12


# --------------------------------------------------------------------------
# Row sums and masks.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal,kv,blocky", [(False, None, False), (True, None, False),
                                              (False, 9, False), (True, 11, True),
                                              (False, None, True)])
def test_rows_sum_to_one_and_masks_zero(causal, kv, blocky):
    B, H, N, d, block = 2, 2, 17, 4, 4
    q, k = _rand((B, H, N, d), 11), _rand((B, H, N, d), 12)
    kv_len = np.array([kv if kv else N, N], dtype=np.int32) if kv else None
    nb = (N + block - 1) // block
    bm = random_block_mask(nb, 0.5, 3).numpy() if blocky else None
    for head in range(B * H):
        b = head // H
        s, p = oracle.attention_probs(q, k, 0.5, head=head, causal=causal, block_mask=bm,
                                      block=block, kv_len=kv_len)
        vis = _mask_bruteforce(N, causal, None if kv_len is None else kv_len[b], bm, block)
        assert np.all(p[~vis] == 0.0)
        assert np.all(np.isneginf(s[~vis]))
        rows = vis.any(axis=1)
        assert np.max(np.abs(p[rows].sum(axis=1) - 1.0)) <= 1e-12
        assert np.all(p[~rows] == 0.0)
        assert np.all(p[vis] > 0.0)


def test_block_mask_builder_against_sets():
    """Band |i-j| <= 2 plus butterfly partners j = i XOR 2^k, by set union."""
    for nb in (1, 2, 5, 8, 128):
        m = band_butterfly_block_mask(nb).numpy().astype(bool)
        ref = set()
        for i in range(nb):
            ref |= {(i, j) for j in range(nb) if abs(i - j) <= 2}
            ref |= {(i, i ^ (1 << kk)) for kk in range(nb.bit_length() + 1) if (i ^ (1 << kk)) < nb}
        got = {(i, j) for i in range(nb) for j in range(nb) if m[i, j]}
        assert got == ref
    m = band_butterfly_block_mask(128).numpy()
    assert (m == m.T).all()
    assert int(m.sum()) == 1274  # 128 blocks: 634 band + 640 butterfly off-band
    assert abs(m.mean() - 1274 / 16384) < 1e-15


# --------------------------------------------------------------------------
# Special cases with closed forms.
# --------------------------------------------------------------------------

def test_single_key_gives_v_and_lse_is_score():
    q, k, v = (_rand((2, 3, 1, 8), s) for s in (4, 5, 6))
    o, lse = oracle.attention_fwd(q, k, v, 0.3)
    assert np.max(np.abs(o - v)) <= 1e-15
    assert np.max(np.abs(lse - 0.3 * np.sum(q * k, axis=-1))) <= 1e-13


def test_zero_queries_give_uniform_average():
    B, H, N, d = 2, 2, 23, 6
    q = np.zeros((B, H, N, d))
    k, v = _rand((B, H, N, d), 8), _rand((B, H, N, d), 9)
    kv_len = np.array([23, 7], dtype=np.int32)
    o, lse = oracle.attention_fwd(q, k, v, 1.0, kv_len=kv_len)
    for b in range(B):
        n = kv_len[b]
        assert np.max(np.abs(o[b] - v[b, :, :n].mean(axis=1, keepdims=True))) <= 1e-14
        assert np.max(np.abs(lse[b] - math.log(n))) <= 1e-14


def test_causal_first_row_is_v0():
    q, k, v = (_rand((1, 2, 9, 4), s) for s in (10, 11, 12))
    o, lse = oracle.attention_fwd(q, k, v, 0.7, causal=True)
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0])) <= 1e-15
    assert np.max(np.abs(lse[:, :, 0] - 0.7 * np.sum(q[:, :, 0] * k[:, :, 0], axis=-1))) <= 1e-14


@pytest.mark.parametrize("p", [0.0, 0.3])
def test_identity_values_expose_dropped_probabilities(p):
    """With V = I (N = d), O = P o Z / (1-p) exactly."""
    B, H, N = 2, 2, 12
    q, k = _rand((B, H, N, N), 13), _rand((B, H, N, N), 14)
    v = np.broadcast_to(np.eye(N), (B, H, N, N)).copy()
    o, _ = oracle.attention_fwd(q, k, v, 0.4, causal=True, dropout_p=p, seed=99)
    z = oracle.dropout_keep(B, H, N, p, 99)
    for head in range(B * H):
        b, h = divmod(head, H)
        _, P = oracle.attention_probs(q, k, 0.4, head=head, causal=True)
        ref = P * z[b, h] / (1.0 - p)
        assert np.max(np.abs(o[b, h] - ref)) <= 1e-15
        assert np.array_equal(o[b, h] != 0, (P != 0) & (z[b, h] != 0))


def test_fully_masked_row_is_zero():
    N, d, block = 8, 4, 4
    bm = np.array([[1, 0], [0, 0]], dtype=np.uint8)  # rows 4..7 see nothing
    q, k, v, do = (_rand((1, 1, N, d), s) for s in (15, 16, 17, 18))
    o, lse = oracle.attention_fwd(q, k, v, 1.0, block_mask=bm, block=block)
    assert np.all(o[0, 0, 4:] == 0.0) and np.all(np.isneginf(lse[0, 0, 4:]))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 1.0, block_mask=bm, block=block)
    assert np.all(dq[0, 0, 4:] == 0.0)
    assert np.all(dk[0, 0, 4:] == 0.0) and np.all(dv[0, 0, 4:] == 0.0)


# --------------------------------------------------------------------------
# Backward: finite differences of the oracle's own forward.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,d,causal,kv,blocky,p", [
    (4, 3, False, None, False, 0.0),
    (8, 4, True, None, False, 0.0),
    (13, 3, False, 9, False, 0.0),
    (13, 4, True, None, True, 0.0),
    (8, 4, False, None, False, 0.25),
    (13, 3, True, 10, True, 0.4),
])
def test_gradients_match_finite_differences(N, d, causal, kv, blocky, p):
    B, H, block = 1, 1, 4
    q, k, v, do = (_rand((B, H, N, d), s) for s in (21, 22, 23, 24))
    kv_len = np.array([kv], dtype=np.int32) if kv else None
    nb = (N + block - 1) // block
    bm = random_block_mask(nb, 0.6, 5).numpy() if blocky else None
    kw = dict(causal=causal, block_mask=bm, block=block, kv_len=kv_len, dropout_p=p, seed=1234)
    scale = 0.8

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, **kw)
        return float(np.sum(o * do))

    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, **kw)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                        - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
        err = np.max(np.abs(num - g))
        assert err <= 1e-7 * max(1.0, np.max(np.abs(g))), (name, err)


def test_rowsum_identity_for_backward_preprocess():
    """sum_c dO_ic O_ic = sum_j P^_ij dP^_ij, with dP^ = dO V^T."""
    B, H, N, d, p = 1, 2, 19, 5, 0.2
    q, k, v, do = (_rand((B, H, N, d), s) for s in (31, 32, 33, 34))
    o, _ = oracle.attention_fwd(q, k, v, 0.5, causal=True, dropout_p=p, seed=5)
    z = oracle.dropout_keep(B, H, N, p, 5)
    for h in range(H):
        _, P = oracle.attention_probs(q, k, 0.5, head=h, causal=True)
        Ph = P * z[0, h] / (1 - p)
        lhs = np.sum(do[0, h] * o[0, h], axis=1)
        rhs = np.sum(Ph * (do[0, h] @ v[0, h].T), axis=1)
        assert np.max(np.abs(lhs - rhs)) <= 1e-13


# --------------------------------------------------------------------------
# Library reduction: PyTorch fp64 CPU attention + autograd.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,d,causal,kv,blocky", [
    (33, 8, False, None, False), (64, 16, True, None, False),
    (50, 8, False, 31, False), (40, 8, True, None, True), (48, 4, False, 29, True),
    (20, 256, True, None, False), (24, 128, False, 17, True)])
def test_matches_torch_fp64_sdpa(N, d, causal, kv, blocky):
    B, H, block = 2, 3, 8
    q, k, v, do = (torch.from_numpy(_rand((B, H, N, d), s)) for s in (41, 42, 43, 44))
    kv_len = np.array([kv, N], dtype=np.int32) if kv else None
    nb = (N + block - 1) // block
    bm = random_block_mask(nb, 0.5, 8).numpy() if blocky else None
    scale = 1.0 / math.sqrt(d)
    mask = torch.ones(B, 1, N, N, dtype=torch.bool)
    for b in range(B):
        vis = _mask_bruteforce(N, causal, None if kv_len is None else kv_len[b], bm, block)
        mask[b, 0] = torch.from_numpy(vis)
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    ref.backward(do)
    o, lse = oracle.attention_fwd(q, k, v, scale, causal=causal, block_mask=bm, block=block,
                                  kv_len=kv_len)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal=causal, block_mask=bm,
                                      block=block, kv_len=kv_len)
    # rows with no visible key are undefined for the library (NaN); the oracle
    # defines them as zero, which test_fully_masked_row_is_zero pins
    live = mask.any(dim=-1).expand(B, H, N).numpy()
    assert live.any()
    assert np.max(np.abs(o - ref.detach().numpy())[live]) <= 1e-12
    assert np.max(np.abs(dq - qt.grad.numpy())[live]) <= 1e-12
    s = scale * (q @ k.transpose(-1, -2)).masked_fill(~mask, float("-inf"))
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())[live]) <= 1e-12
    if live.all():
        assert np.max(np.abs(dk - kt.grad.numpy())) <= 1e-12
        assert np.max(np.abs(dv - vt.grad.numpy())) <= 1e-12
