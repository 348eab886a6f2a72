"""Host-side helpers of bench.py: the FLOP/byte models and the recorded DRAM
traffic, which is reported only for the kernel sources it was measured on."""
import json

import bench
from workloads import WORKLOADS


def test_flop_model_matches_formula():
    w = WORKLOADS["long_causal"]
    fwd, bwd = bench.flops(w)
    assert fwd == 4 * w.B * w.H * w.N * w.N * w.d / 2
    assert bwd == 2.5 * fwd


def test_recorded_traffic_requires_matching_sources(tmp_path, monkeypatch):
    rec = {"kernels": {"gpt2_causal": {"bwd_tc_kernel": {"dram_bytes": 1234,
                                                         "source_sha256": bench.kernel_source_hash("bwd_tc_kernel")}}}}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the hash is taken from the package sources under ROOT: point it back
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k=None: rec["kernels"]["gpt2_causal"]["bwd_tc_kernel"]
                        ["source_sha256"] if k == "bwd_tc_kernel" else "x")
    assert bench.recorded_traffic("gpt2_causal", "bwd_tc_kernel") == 1234
    assert bench.recorded_traffic("gpt2_causal", "fwd_pp_kernel") is None
    assert bench.recorded_traffic("long_causal", "bwd_tc_kernel") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k=None: "0" * 64)
    assert bench.recorded_traffic("gpt2_causal", "bwd_tc_kernel") is None


def test_each_kernel_hashes_its_own_sources():
    assert bench.kernel_source_hash("bwd_tc_kernel") != bench.kernel_source_hash("fwd_pp_kernel")
    assert bench.kernel_source_hash("fwd_pp_kernel") == bench.kernel_source_hash("fwd_d256_kernel")


def test_source_hash_tracks_kernel_files():
    h1 = bench.kernel_source_hash()
    assert len(h1) == 64 and h1 == bench.kernel_source_hash()


def test_traffic_key_separates_dtype_and_splits():
    w = WORKLOADS["long_causal"]
    assert bench.traffic_key(w) == "long_causal"
    assert bench.traffic_key(w.with_(dtype="fp16")) == "long_causal/fp16"
    assert bench.traffic_key(w, 2) == "long_causal/splits=2"
    assert bench.traffic_key(w.with_(dtype="fp16"), 4) == "long_causal/fp16/splits=4"


def test_byte_model_uses_the_element_size():
    w = WORKLOADS["gpt2_causal"]
    f16, b16 = bench.algorithmic_bytes(w.with_(dtype="fp16"))
    assert (f16, b16) == bench.algorithmic_bytes(w)  # bf16 and fp16 are both 2 bytes
    f32, _ = bench.algorithmic_bytes(w.with_(dtype="fp32"))
    bhn = w.B * w.H * w.N
    assert f32 - f16 == 4 * bhn * w.d * (4 - 2)


def test_main_kernel_names_and_bytes():
    w = WORKLOADS["long_causal"]
    assert bench.main_kernel_names(w) == ("fwd_pp_kernel", "bwd_tc_kernel")
    assert bench.main_kernel_names(w.with_(d=256))[0] == "fwd_d256_kernel"
    assert bench.main_kernel_names(w.with_(d=64))[0] == "fwd_1t_kernel"
    assert bench.main_kernel_names(w.with_(d=64), splits=2)[0] == "fwd_pp_kernel"
    assert bench.main_kernel_names(WORKLOADS["single_head_fp32"])[0] == "fwd_simt_kernel"
    # the backward's main kernel reads Q, K, V, dO, LSE, delta and writes dQ, dK, dV
    bhnd, bhn = w.B * w.H * w.N * w.d, w.B * w.H * w.N
    assert bench.bwd_main_bytes(w) == 7 * bhnd * 2 + 8 * bhn
    assert bench.bwd_main_bytes(w) < bench.algorithmic_bytes(w)[1]


def test_visible_pairs_closed_forms():
    from workloads import Workload, make_inputs
    w = Workload("t", 0, B=2, H=3, N=300, d=64, dtype="bf16", causal=True)
    inp = make_inputs(w, with_grad_out=False)
    assert bench.visible_pairs(w, inp) == 2 * 3 * 300 * 301 // 2
    w2 = w.with_(causal=False, kv_len_range=(100, 200))
    inp2 = make_inputs(w2, with_grad_out=False)
    assert bench.visible_pairs(w2, inp2) == 3 * 300 * int(inp2["kv_len"].sum())
    w3 = Workload("t", 0, B=1, H=2, N=16384, d=64, dtype="bf16", block_sparse=True)
    inp3 = make_inputs(w3, with_grad_out=False)
    dens = float(inp3["block_mask"].double().mean())
    assert bench.visible_pairs(w3, inp3) == round(2 * 16384 * 16384 * dens)
