"""Host-side checks of the benchmark's accounting (no GPU).

The roofline figures divide algorithmic work by measured time, so the work
must be the method's own count: 6 R D H FLOPs for the two expert GEMMs, and
for the permute and the combine the activation-width rows of x, x_perm,
y_perm and out (page "Expert Parallelism (EP)", section 1: the routed rows
are copied to the permuted buffer and reduced back, each once).  These tests
recompute those counts from the shapes alone and compare.
"""
import json
import os

import pytest

import moe_inputs


def _bench():
    import bench
    return bench


@pytest.mark.parametrize("name", ["fine-grained-bf16", "deepseek-v3-shaped", "zipf-skewed",
                                  "decode-masked", "tiny-fp32"])
def test_algorithmic_counts(name):
    bench = _bench()
    w = moe_inputs.WORKLOADS[name]
    b = 4 if w.dtype == "f32" else 2
    R = w.T * w.k
    alg = bench.algorithmic(w)
    assert alg["ffn_flops"] == 6.0 * R * w.D * w.H
    assert alg["permute_bytes"] == w.T * w.D * b + R * w.D * b
    # y rows at the activation width, out once, a row index and a weight per slot
    assert alg["combine_bytes"] == R * w.D * b + w.T * w.D * b + R * 8
    assert alg["weight_bytes"] == w.E * 3 * w.D * w.H * b


def test_fine_grained_figures():
    """The fine-grained layer's headline figures: 425.2 GFLOP per call,
    117.4 MB permuted, 117.6 MB combined, 1.1 GB of expert weights."""
    bench = _bench()
    alg = bench.algorithmic(moe_inputs.WORKLOADS["fine-grained-bf16"])
    assert alg["ffn_flops"] == 425_201_762_304
    assert alg["permute_bytes"] == 117_440_512
    assert alg["combine_bytes"] == 117_637_120
    assert alg["weight_bytes"] == 1_107_296_256


def test_decode_bytes_count_touched_experts_only():
    bench = _bench()
    w = moe_inputs.WORKLOADS["decode-masked"]
    R = w.T * w.k
    full = bench.algorithmic(w, R, w.E)["grouped_bytes"]
    part = bench.algorithmic(w, R, 250)["grouped_bytes"]
    assert full - part == 6 * 3 * w.D * w.H * 2


def test_recorded_traffic_needs_the_current_source(monkeypatch):
    """A DRAM-traffic record is reported only while the kernel source it was
    taken on is unchanged."""
    bench = _bench()
    path = os.path.join(bench.ROOT, "profiles", "grouped_swiglu_traffic.json")
    rec = json.load(open(path))
    for wl, entry in rec.items():
        assert entry["dram_bytes_per_call"] > 0
        got = bench.recorded_traffic(wl)
        if entry["kernel_source_hash"] == bench.kernel_source_hash(wl):
            assert got == entry["dram_bytes_per_call"]
        else:
            assert got is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda wl=None: "0" * 16)
    assert all(bench.recorded_traffic(wl) is None for wl in rec)


def test_recorded_traffic_is_near_the_algorithmic_bytes():
    """The recorded DRAM bytes of a grouped call are the algorithmic bytes
    within a few percent (no operand re-read from DRAM) where the weights
    dominate: the fine-grained call and the decode call."""
    bench = _bench()
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "grouped_swiglu_traffic.json")))
    w = moe_inputs.WORKLOADS["fine-grained-bf16"]
    R = w.T * w.k
    # x_perm rows, w1, w3, w2 read once; h written and read; y (fp16) written
    alg = R * w.D * 2 + w.E * 3 * w.D * w.H * 2 + 2 * R * w.H * 2 + R * w.D * 2
    assert 0.98 < rec["fine-grained-bf16"]["dram_bytes_per_call"] / alg < 1.05
    d = moe_inputs.WORKLOADS["decode-masked"]
    dec = bench.algorithmic(d, d.T * d.k, 250)["grouped_bytes"]
    assert 0.98 < rec["decode-masked"]["dram_bytes_per_call"] / dec < 1.05


def test_binding_roof_per_workload():
    """The roof the grouped call is reported against is the larger of its two
    floors: FLOPs at the tensor peak, algorithmic bytes at the copy rate.  The
    fine-grained call sits at the ridge (221 against 216 us at the measured
    peaks); the 256-expert layer (about 256 rows per expert) is byte-bound."""
    bench = _bench()
    peaks = {"hbm_gbs": 6687.5, "bf16_tflops": 1927.1}
    W = moe_inputs.WORKLOADS
    want = {"fine-grained-bf16": "tensor", "zipf-skewed": "tensor", "deepseek-v3-shaped": "hbm",
            "decode-masked": "hbm", "tiny-fp32": "alu"}
    for name, bound in want.items():
        w = W[name]
        assert bench.grouped_bound(w, w.T * w.k, w.E, peaks) == bound, name
    w = W["fine-grained-bf16"]
    compute_ms, hbm_ms = bench.floors(w, w.T * w.k, w.E, peaks)
    assert abs(compute_ms - 425_201_762_304 / 1927.1e12 * 1e3) < 1e-9
    assert 0.215 < hbm_ms < 0.218 and 0.220 < compute_ms < 0.221
    d = W["deepseek-v3-shaped"]
    compute_ms, hbm_ms = bench.floors(d, d.T * d.k, d.E, peaks)
    assert hbm_ms > 1.2 * compute_ms


def test_backward_floors():
    """The backward's floor is the sum over its kernels of the larger of FLOPs
    at the tensor peak and algorithmic bytes at the copy rate.  With fp32
    weight gradients every expert GEMM is byte-bound (dgrad2 reads the saved
    gate/up and writes dg/du, dgrad1 writes fp32 dx_perm, the wgrads write 0.74
    and 1.48 GB); with bf16 ones wgrad13 becomes tensor-bound."""
    bench = _bench()
    peaks = {"hbm_gbs": 6687.5, "bf16_tflops": 1927.1}
    w = moe_inputs.WORKLOADS["fine-grained-bf16"]
    R, D, H, E = w.T * w.k, w.D, w.H, w.E
    f32 = bench.backward_floors(w, peaks, 4)
    f16 = bench.backward_floors(w, peaks, 2)
    gemms = ("dgrad2_swiglu_bwd", "dgrad1", "wgrad2", "wgrad13")
    assert sum(f32[g]["flops"] for g in gemms) == 12.0 * R * D * H
    assert all(f32[g]["bound"] == "hbm" for g in gemms)
    assert f16["wgrad13"]["bound"] == "tensor"
    assert f32["wgrad13"]["bytes"] - f16["wgrad13"]["bytes"] == 2 * E * H * D * 2
    assert f32["wgrad2"]["bytes"] == R * D * 2 + R * H * 2 + E * D * H * 4
    assert 0.73 < f32["total_floor_ms"] < 0.74
    assert 0.56 < f16["total_floor_ms"] < 0.58
