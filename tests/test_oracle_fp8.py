"""Pins of the oracle's E4M3 decoding and of its FP8 forward (fp64 on the
dequantised inputs), against a library's E4M3 conversion, closed forms of
the format, and properties of attention that fix how the dequantisation
factors enter."""
import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, make_fp8_inputs, quantize_e4m3


def test_every_code_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_dequantize(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])


def test_closed_forms_of_the_format():
    v = oracle.e4m3_dequantize(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0                       # exponent 7 = bias, mantissa 0
    assert v[0x7E] == 448.0                     # 1.75 * 2^8, the largest finite value
    assert v[0x08] == 2.0 ** -6                 # smallest normal
    assert v[0x01] == 2.0 ** -9                 # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9             # largest subnormal
    assert v[0x00] == 0.0 and v[0x80] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])  # no infinities
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)             # codes 0..0x7E increase
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F])  # sign bit only flips the sign


def test_per_head_factors_scale_each_head():
    codes = np.full((2, 3, 4, 8), 0x38, dtype=np.uint8)  # all 1.0
    ds = np.arange(1, 7, dtype=np.float64)
    out = oracle.e4m3_dequantize(codes, ds, 4)
    for bh in range(6):
        assert np.all(out.reshape(6, 4, 8)[bh] == ds[bh])


def test_fp8_forward_is_the_definition_on_dequantised_inputs():
    w = Workload("fp8_pin", 0, B=1, H=2, N=40, d=16, dtype="fp32", causal=True)
    inp = make_fp8_inputs(w, seed=5)
    o, lse = oracle.attention_fwd_fp8(inp["q8"], inp["k8"], inp["v8"], inp["descale_q"], inp["descale_k"],
                                      inp["descale_v"], 0.25, causal=True)
    deq = {}
    for n in ("q", "k", "v"):
        x = inp[n + "8"].view(torch.float8_e4m3fn).double()
        deq[n] = x * inp["descale_" + n].double().reshape(1, 2, 1, 1)
    o2, lse2 = oracle.attention_fwd(deq["q"], deq["k"], deq["v"], 0.25, causal=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_factors_enter_as_the_definition_says():
    """O is linear in V's factor; Q's and K's factors multiply the scores,
    which is the same as multiplying the softmax scale."""
    w = Workload("fp8_pin", 0, B=1, H=1, N=33, d=16, dtype="fp32")
    inp = make_fp8_inputs(w, seed=9)
    one = np.ones(1)
    o1, l1 = oracle.attention_fwd_fp8(inp["q8"], inp["k8"], inp["v8"], one, one, one, 0.3)
    o2, _ = oracle.attention_fwd_fp8(inp["q8"], inp["k8"], inp["v8"], one, one, 2 * one, 0.3)
    assert np.allclose(o2, 2 * o1, rtol=0, atol=1e-12)
    o3, l3 = oracle.attention_fwd_fp8(inp["q8"], inp["k8"], inp["v8"], 0.5 * one, 4 * one, one, 0.3)
    o4, l4 = oracle.attention_fwd_fp8(inp["q8"], inp["k8"], inp["v8"], one, one, one, 0.6)
    assert np.allclose(o3, o4, rtol=0, atol=1e-12) and np.allclose(l3, l4, rtol=0, atol=1e-12)


def test_quantiser_round_trip_error_is_within_half_a_unit():
    x = torch.randn(2, 2, 64, 32, generator=torch.Generator().manual_seed(3))
    codes, ds = quantize_e4m3(x)
    back = oracle.e4m3_dequantize(codes, ds, 64)
    rel = np.abs(back - x.double().numpy()) / ds.double().numpy().repeat(64 * 32).reshape(2, 2, 64, 32)
    # relative half-unit 2^-4 for normals, absolute 2^-10 (in code units) for subnormals
    mag = np.abs(x.double().numpy()) / ds.double().numpy().repeat(64 * 32).reshape(2, 2, 64, 32)
    assert np.all(rel <= np.maximum(mag * 2.0 ** -4, 2.0 ** -10) + 1e-12)
