"""Host-side logic of bench.py on CPU: the algorithmic bytes and flops behind
the roofline, the clock-sample summary, and the guard that keeps ncu traffic
taken on other kernel sources out of the JSON line."""
from __future__ import annotations

import importlib.util
import json
import os

import pytest

from workloads import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_expert_bytes_match_the_format(bench):
    # group 32 along K, fp16 scales, two int4 per byte: 21,233,664 B per
    # GLM-shaped expert (H 6144, I 2048) and 55,296 B for the tiny layer
    for name, per_expert in (("glm_decode", 21_233_664), ("tiny", 55_296)):
        sh = CONFIGS[name].shape
        assert bench.expert_gate_up_bytes(sh) + bench.expert_down_bytes(sh) == per_expert
    # one fp16 scale a row: 3 x 6144 x 2048 / 2 B of nibbles + (2 x 2048 +
    # 6144) scales x 2 B = 18,874,368 + 20,480
    sh = CONFIGS["glm_decode_rowscale"].shape
    assert bench.expert_gate_up_bytes(sh) + bench.expert_down_bytes(sh) == 18_894_848
    # int8, grouped: twice the weight bytes, the same scales
    from workloads.configs import LayerShape
    sh8 = LayerShape(6144, 2048, 256, 8, 8, 4, 2.5, weight_format="int8")
    assert bench.expert_gate_up_bytes(sh8) + bench.expert_down_bytes(sh8) == \
        2 * 18_874_368 + 21_233_664 - 18_874_368


def test_single_token_bytes_are_the_per_token_figure(bench):
    # 9 experts (8 routed + shared) + fp32 router weight and bias + bf16 x +
    # fp32 y: 9 * 21,233,664 + 6,291,456 + 1,024 + 12,288 + 24,576
    sh = CONFIGS["glm_decode"].shape
    want = 9 * 21_233_664 + 6_291_456 + 1_024 + 12_288 + 24_576
    assert bench.phase_bytes("decode_fused", sh, 1, 8, 2) == want == 197_432_320


def test_grouped_gemm_flops(bench):
    # 2 flops per multiply-add; gate and up are two H x I products per row,
    # down one; 512 tokens x 8 routed rows + 512 shared rows
    sh = CONFIGS["glm_prefill"].shape
    rows = 512 * 8 + 512
    assert bench.phase_flops("tc_gate_up", sh, 512) == 2 * 2 * 6144 * 2048 * rows
    assert bench.phase_flops("tc_down", sh, 512) == 2 * 6144 * 2048 * rows
    assert bench.phase_flops("decode_fused", sh, 1) is None


def test_clock_summary_uses_only_the_timed_window(bench):
    s = bench.ClockSampler(0)
    row = lambda mhz, *r: [str(mhz), "2070", "900.0", *r]  # noqa: E731
    ok = ("Not Active",) * 4
    s.samples = [(0.5, row(900, *ok)),                       # before the window
                 (1.0, row(2070, *ok)), (1.2, row(2055, "Active", *ok[1:])),
                 (1.4, row(2040, *ok)),
                 (3.0, row(600, "Not Active", "Active", "Not Active", "Not Active"))]
    c = s.summary(1.0, 2.0)
    assert c["sm_mhz"] == 2055 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies after the window
    assert s.summary(5.0, 6.0)["reasons"] == ["no samples"]
    # each record of a run summarises its own window
    assert s.summary(2.5, 3.5)["reasons"] == ["hw_slowdown"]


def test_ncu_traffic_needs_the_profiled_sources(bench, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        t = json.load(f)
    for key, nbytes in t["per_launch_bytes"].items():
        workload, kernel = key.split(":")
        if bench.kernel_source_hash(kernel) == t["source_hash"][kernel]:
            assert bench.ncu_traffic(kernel, workload) == nbytes
        monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
        assert bench.ncu_traffic(kernel, workload) is None  # sources changed
        monkeypatch.undo()
    assert bench.ncu_traffic("no_such_kernel", "glm_decode") is None


def test_job_throughput_counts_every_rank(bench):
    # tokens of all ranks over the slowest rank's time
    assert bench.job_tokens_per_s(4, 256, 10, 500.0) == pytest.approx(4 * 256 * 10 / 0.5)


def test_verify_union_bytes(bench):
    """A verify call streams its distinct experts and the shared one once:
    14.5 experts on average give (14.5 + 1) x 21,233,664 B of experts plus the
    router (256 x 6144 fp32 weights and 256 biases), 4 rows of x and y."""
    from workloads import CONFIGS
    wl = CONFIGS["glm_verify"]
    per_expert = 21_233_664
    router = 256 * 6144 * 4 + 256 * 4
    want = 15.5 * per_expert + router + 4 * 6144 * 2 + 4 * 6144 * 4
    assert bench.union_bytes_per_call(wl, 14.5, 2) == pytest.approx(want)
    # the accepted-token rates of the MTP A/B the per-emitted-token figures use
    assert dict(bench.ACCEPTED_PER_VERIFY) == {"G4": 2.065, "G5": 2.286}


def test_host_cpu_is_described(bench):
    n, model = bench.host_cpu()
    assert n == os.cpu_count() and n >= 1
    assert isinstance(model, str) and model
