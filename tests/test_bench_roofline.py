"""bench.py's roofline arithmetic on made-up measurements (no GPU): the
algorithmic bytes and FLOPs per launch, the achieved rate and its fraction of
the peak, and the rule that a committed traffic record counts only while the
hash of its kernel's sources still matches."""
import json

import pytest

import bench
import synthetic

PK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def test_decode_stack_is_bytes_over_launch_time():
    wl = synthetic.WORKLOADS["decode80b"]
    blob = 1_769_472                                  # 80B blob: 3 I H weights at half a byte + 4 bytes of (s, b) per 64
    m = {"blob": blob, "uniq": [10] * wl.n_layers, "stacked": True, "kern_ms": 0.64, "ms": 0.64, "steps": 1}
    r = bench.roofline_of(wl, m, PK, "measured")
    alg = 11 * blob * wl.n_layers                     # 10 routed + the shared expert per layer
    assert r["bound"] == "hbm" and r["bytes_per_launch"] == alg
    assert r["achieved"] == pytest.approx(alg / 0.64e-3 / 1e9, abs=0.05)
    assert r["frac"] == pytest.approx(r["achieved"] / PK["hbm_gbs"], abs=1e-4)
    assert r["us_per_launch"] == pytest.approx(640.0)


def test_zipf_layer_uses_the_whole_layer_time():
    wl = synthetic.WORKLOADS["zipf80b_t64"]
    m = {"blob": 1000, "uniq": [55], "stacked": False, "kern_ms": None, "ms": 0.086 * 30, "steps": 30}
    r = bench.roofline_of(wl, m, PK, "measured")
    assert r["bytes_per_launch"] == 56 * 1000
    assert r["us_per_launch"] == pytest.approx(86.0)


def test_prefill_counts_both_gemms_flops():
    wl = synthetic.WORKLOADS["prefill80b"]
    m = {"blob": 1, "uniq": [512], "stacked": False, "kern_ms": 0.394, "down_ms": 0.221, "ms": 0.777, "steps": 1}
    r = bench.roofline_of(wl, m, PK, "measured")
    pairs = wl.T * (wl.k + 1)                          # routed pairs and one shared row per token
    f_gu, f_dn = 2.0 * pairs * 2 * wl.I * wl.H, 2.0 * pairs * wl.I * wl.H
    assert r["bound"] == "tensor" and r["flops_per_launch"] == f_gu + f_dn
    assert r["achieved"] == pytest.approx((f_gu + f_dn) / 0.615e-3 / 1e12, abs=0.05)
    assert r["frac"] == pytest.approx(r["achieved"] / PK["bf16_tflops"], abs=1e-4)
    assert r["gate_up_tflops"] == pytest.approx(f_gu / 0.394e-3 / 1e12, abs=0.05)
    assert r["layer_us"] == pytest.approx(777.0)
    assert bench.roofline_of(wl, dict(m, kern_ms=None), PK, "measured") is None


def test_traffic_record_needs_matching_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text("kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"source_sha256": bench.src_hash(["k.cu"]), "records": {"w": {"dram_bytes_per_launch": 123}}}
    (tmp_path / "profiles" / "t.json").write_text(json.dumps(rec))
    assert bench._traffic_record("t.json", ["k.cu"], "w", "dram_bytes_per_launch") == 123
    assert bench._traffic_record("t.json", ["k.cu"], "other", "dram_bytes_per_launch") is None
    (tmp_path / "k.cu").write_text("kernel v2")        # the kernel changed since the capture
    assert bench._traffic_record("t.json", ["k.cu"], "w", "dram_bytes_per_launch") is None
    assert bench._traffic_record("missing.json", ["k.cu"], "w", "dram_bytes_per_launch") is None
