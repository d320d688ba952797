"""CPU checks of bench.py's bookkeeping: the roofline object of the grouped
expert GEMMs, the traffic records under profiles/, and the algorithmic work
of every stage the layer reports."""
import json
import os

import pytest

import bench
import qb_inputs as QI

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PEAKS = {"hbm_gbs": 6789.3, "bf16_tflops": 1889.5}


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_roofline_object_has_both_roofs(name):
    shape = bench.WORKLOADS[name]
    stages = {"expert_gate_up": 3.3, "expert_down": 1.9}
    mx = (2.0, {"mxf8f6f4": 4800.0, "bf16": 2400.0}) if shape.wfmt == "mxfp4" else None
    r = bench.expert_gemm_roofline(shape, stages, PEAKS, "measured", mx)
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic", "tensor_frac", "hbm_frac"):
        assert key in r, key
    assert r["bound"] in ("hbm", "tensor")
    # frac is the roof that binds
    assert r["frac"] == pytest.approx(r["hbm_frac"] if r["bound"] == "hbm" else r["tensor_frac"])
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])


def test_prefill_is_bound_by_hbm_by_its_arithmetic_intensity():
    # 5.772 TFLOP against 22.8 GB: 253 flop/B, below the 278 flop/B ridge of the measured peaks
    r = bench.expert_gemm_roofline(QI.PREFILL, {"expert_gate_up": 3.3, "expert_down": 1.9}, PEAKS, "measured")
    assert r["bound"] == "hbm"
    assert r["tensor_frac"] == pytest.approx(5.772e12 / 5.2e-3 / 1889.5e12, rel=1e-3)


def test_traffic_records_parse_and_cover_the_k3_workloads():
    sha = bench.kernel_source_sha256()
    found = {}
    for fn in os.listdir(os.path.join(ROOT, "profiles")):
        if not fn.endswith(".md"):
            continue
        file_sha = None
        for line in open(os.path.join(ROOT, "profiles", fn)):
            if line.startswith("kernel_source_sha256:"):
                file_sha = line.split(":", 1)[1].strip()
            elif line.startswith("traffic:"):
                k, w, b = line.split(":", 1)[1].split()
                found[(k, w)] = (int(b), file_sha)
    for w in ("k3_prefill_T16384", "k3_decode_T256", "k3_prefill_mxfp4_T16384", "k3_decode_mxfp4_T256"):
        for k in ("expert_gate_up", "expert_down"):
            assert (k, w) in found
            b, file_sha = found[(k, w)]
            assert b > 0
            if file_sha == sha:
                assert bench.recorded_traffic(k, w) == b


def test_every_reported_stage_has_algorithmic_work():
    # the layer's stage names (tensor-core and CUDA-core paths) that carry work
    for shape in (QI.PREFILL, QI.DECODE, QI.PREFILL_MXFP4, QI.DECODE_MXFP4):
        work = bench.stage_work(shape, shape.T)
        for nm in ("router", "expert_gate_up", "expert_down", "xside_gemm", "down_proj", "shared_gate_up",
                   "combine_rmsnorm", "up_proj_shared"):
            assert nm in work, nm
            b, f = work[nm]
            assert b > 0 and f >= 0, nm


def test_measured_peaks_file_is_read_when_present():
    pk, src = bench.peaks()
    assert pk["hbm_gbs"] > 0 and pk["bf16_tflops"] > 0
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            assert pk["hbm_gbs"] == json.load(f)["hbm_gbs"]
