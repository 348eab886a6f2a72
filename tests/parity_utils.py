"""Shared helpers for the GPU parity tests: run the library through its C ABI
and the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import io_aware_exact_08_gb300 as fa
import oracle

# Tolerances (max-abs), for bf16 inputs with fp32 accumulation and for fp32.
# fp16 carries three more mantissa bits than bf16 (unit roundoff 2^-11 vs
# 2^-8), and the kernels' only roundings beyond fp32 are those of P, dS and the
# stored outputs to the input type, so its O and gradient bars are the bf16
# ones divided by 4 (rather than the full factor 8, to leave room for the fp32
# accumulation and ex2 errors that do not shrink with the input type); LSE is
# fp32 arithmetic on the same inputs and keeps the bf16 bar.
TOL = {
    "bf16": dict(o=1e-2, lse=1e-3, dq=3e-2, dk=3e-2, dv=3e-2),
    "fp16": dict(o=2.5e-3, lse=1e-3, dq=7.5e-3, dk=7.5e-3, dv=7.5e-3),
    "fp32": dict(o=1e-4, lse=1e-4, dq=1e-4, dk=1e-4, dv=1e-4),
}


def to_dev(x, device="cuda"):
    return None if x is None else x.to(device).contiguous()


def gpu_forward(inp, device="cuda"):
    q, k, v = (to_dev(inp[n], device) for n in ("q", "k", "v"))
    o, lse = fa.attention_fwd(q, k, v, scale=inp["scale"], causal=inp["causal"],
                              block_mask=to_dev(inp["block_mask"], device), dropout_p=inp["dropout_p"],
                              seed=inp["seed"], kv_len=to_dev(inp["kv_len"], device))
    return q, k, v, o, lse


def gpu_fwd_bwd(inp, device="cuda"):
    q, k, v, o, lse = gpu_forward(inp, device)
    do = to_dev(inp["do"], device)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, do, scale=inp["scale"], causal=inp["causal"],
                                  block_mask=to_dev(inp["block_mask"], device), dropout_p=inp["dropout_p"],
                                  seed=inp["seed"], kv_len=to_dev(inp["kv_len"], device))
    torch.cuda.synchronize()
    st, site = fa.fa_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"device status {st} at site {site}"
    return {n: t.float().cpu().numpy().astype(np.float64)
            for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}


def oracle_fwd_bwd(inp, heads=None, backward=True):
    kw = dict(causal=inp["causal"], block_mask=inp["block_mask"], block=128, kv_len=inp["kv_len"],
              dropout_p=inp["dropout_p"], seed=inp["seed"], heads=heads)
    o, lse = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], inp["scale"], **kw)
    out = dict(o=o, lse=lse)
    if backward:
        dq, dk, dv = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["do"], inp["scale"], **kw)
        out.update(dq=dq, dk=dk, dv=dv)
    return out


def half_ulp(ref, dtype):
    """Half a unit in the last place of the stored type at |ref| (0 at 0)."""
    mant = {"bf16": 7, "fp16": 10}.get(dtype, 23)
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - mant - 1), 0.0)


def max_err(got, ref, heads=None, H=None, allowance=None):
    """Max-abs error; -inf entries (fully masked rows' LSE) must match exactly.

    With ``allowance`` (a dtype name), the rounding of the stored output is
    taken off first: the error is max(|got - ref| - half_ulp(ref), 0), i.e.
    the error of the kernel's fp32 result before its final store.
    """
    if heads is not None:
        B = got.shape[0]
        g = got.reshape((-1,) + got.shape[2:])[list(heads)]
        r = ref.reshape((-1,) + ref.shape[2:])[list(heads)]
    else:
        g, r = got, ref
    inf_r = np.isneginf(r)
    if inf_r.any():
        assert np.array_equal(np.isneginf(g), inf_r), "masked-row -inf pattern differs"
        g = np.where(inf_r, 0.0, g)
        r = np.where(inf_r, 0.0, r)
    assert np.all(np.isfinite(g)), "non-finite values in GPU output"
    if not g.size:
        return 0.0
    d = np.abs(g - r)
    if allowance is not None:
        d = np.maximum(d - half_ulp(r, allowance), 0.0)
    return float(np.max(d))


def _select(got, ref, heads):
    if heads is None:
        return got, ref
    g = got.reshape((-1,) + got.shape[2:])[list(heads)]
    r = ref.reshape((-1,) + ref.shape[2:])[list(heads)]
    return g, r


def compare(got, ref, dtype, keys=("o", "lse", "dq", "dk", "dv"), heads=None):
    """Checks every output against its tolerance, on the raw error first.

    O, dQ, dK, dV are stored in the input dtype. Where half an ulp of the
    stored type at the reference value is at most a quarter of the bar
    (bf16: |O| < 1 and gradients below 2 in magnitude; fp16: |x| < 2), the
    raw max-abs error must be within the bar. Only the remaining entries,
    where the storage rounding alone is a sizeable part of the bar (large
    values of early causal rows, or scaled by dropout's 1/(1-p)), are
    compared after that rounding is taken off; they are counted
    (key + "_n_allow"). LSE is fp32 and is always compared raw. Returned: per key the error used for the
    check, the raw max-abs error over all entries (key + "_raw") and the
    count of entries that needed the rounding allowance.
    """
    tol = TOL[dtype]
    errs = {}
    bad = {}
    for key in keys:
        if key not in ref:
            continue
        t = tol[key]
        raw = max_err(got[key], ref[key], heads)
        errs[key + "_raw"] = raw
        if key == "lse" or dtype == "fp32":
            errs[key] = raw
            errs[key + "_n_allow"] = 0
            if not raw <= t:
                bad[key] = (raw, t)
            continue
        g, r = _select(got[key], ref[key], heads)
        hu = half_ulp(r, dtype)
        strict = hu <= t / 4
        d = np.abs(g - r)
        strict_err = float(d[strict].max()) if strict.any() else 0.0
        loose = ~strict
        allow_err = float(np.maximum(d[loose] - hu[loose], 0.0).max()) if loose.any() else 0.0
        errs[key] = max(strict_err, allow_err)
        errs[key + "_strict"] = strict_err
        errs[key + "_n_allow"] = int(loose.sum())
        if not strict_err <= t:
            bad[key + "_strict"] = (strict_err, t)
        if not allow_err <= t:
            bad[key + "_allow"] = (allow_err, t)
    assert not bad, f"tolerance exceeded: {bad} (all errors: {errs})"
    return errs
