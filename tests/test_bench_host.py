"""Host-side arithmetic of bench.py on CPU: the roofline numerators, the traffic lookup and
the peak denominators.

The expected work figures are worked by hand from the method's shapes: a d -> d_g gate MLP
over every input row (deep dive section 3.1, Eq. (3)), and causal attention over the kept
rows of each sequence (Eq. (5)). They are not read back from bench.py.
"""
import json
import os

import pytest

import bench
from learned_token_pruning_07_b300 import inputs as I

pytestmark = pytest.mark.cpu


def test_stage_work_at_the_32k_workload_with_4096_kept_documents():
    wl = I.WORKLOADS["sweep_32k"]
    M = 4096 + 256
    w = bench.stage_work(wl, 4096, [M])
    # gate MLP: 2 * 33,024 rows * 2,048 * 512 multiply-adds
    assert w["gate_score"]["flops"] == 2 * 33024 * 2048 * 512 == 69_256_347_648
    # causal attention: 4 d_h H_q flops per visible (query, key) pair, M (M + 1) / 2 pairs
    assert M * (M + 1) // 2 == 9_472_128
    assert w["gated_attention"]["flops"] == 4 * 128 * 16 * 9_472_128 == 77_595_672_576
    # gather: every kept row of h read once and written once in bf16 (4 KB each way at d = 2048)
    assert w["gather_kept"]["bytes"] >= 2 * M * 2048 * 2 == 35_651_584
    assert w["gather_kept"]["bytes"] - 35_651_584 < 64 * M   # plus the few int/float columns
    # select reads the fp32 scores and the byte mask once
    assert w["topk_select"]["bytes"] >= 33024 * 5
    assert w["gate_score"]["bound"] == w["gated_attention"]["bound"] == "tensor"
    assert w["topk_select"]["bound"] == w["gather_kept"]["bound"] == "hbm"


def test_attention_work_counts_pairs_per_sequence():
    # three sequences of 1, 2 and 3 kept rows: 1 + 3 + 6 visible pairs, none across sequences
    wl = I.WORKLOADS["tiny"]
    w = bench.stage_work(wl, 1, [1, 2, 3])
    assert w["gated_attention"]["flops"] == 4 * wl.d_h * wl.H_q * 10
    one = bench.stage_work(wl, 1, [6])
    assert one["gated_attention"]["flops"] == 4 * wl.d_h * wl.H_q * 21


def test_traffic_lookup_needs_the_same_source_workload_and_budget(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("gated_attention")
    f = tmp_path / "traffic.txt"
    f.write_text("# kernel workload K source-hash bytes\n"
                 f"gated_attention sweep_32k 4096 {h} 123456\n"
                 "gated_attention sweep_32k 1024 0123456789abcdef 999\n"
                 f"gate_score sweep_32k 4096 {h} 777\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(f))
    assert bench.measured_traffic("gated_attention", "sweep_32k", 4096) == 123456.0
    assert bench.measured_traffic("gated_attention", "sweep_32k", 1024) is None   # another source
    assert bench.measured_traffic("gated_attention", "long_128k", 4096) is None   # another workload
    assert bench.measured_traffic("gate_score", "sweep_32k", 4096) is None        # its own hash differs
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "absent.txt"))
    assert bench.measured_traffic("gated_attention", "sweep_32k", 4096) is None


def test_each_kernel_has_its_own_source_hash():
    hashes = {k: bench.kernel_source_hash(k) for k in ("gate_score", "topk_select", "gather_kept", "gated_attention")}
    assert len(set(hashes.values())) == 4 and all(len(v) == 16 for v in hashes.values())


def test_source_hash_ignores_comments_but_not_code():
    src = 'int a = 1; // one\n/* a block\n   comment */\nint b = a + 2;\n\n  // indented note\n'
    same = 'int a = 1;\nint b = a + 2; /* trailing */\n'
    changed = 'int a = 1;\nint b = a + 3;\n'
    assert bench.strip_comments(src) == bench.strip_comments(same)
    assert bench.strip_comments(src) != bench.strip_comments(changed)
    assert "//" not in bench.strip_comments(src) and "/*" not in bench.strip_comments(src)


def test_peaks_come_from_the_measured_file_when_present():
    p = bench.load_peaks()
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        assert p["source"] == "fallback" and p["hbm_gbs"] == 6400.0 and p["bf16_tflops"] == 1800.0
        return
    with open(path) as fh:
        j = json.load(fh)
    assert p["source"] == "measured"
    assert p["hbm_gbs"] == float(j["hbm_gbs"]) and p["bf16_tflops"] == float(j["bf16_tflops"])


def _run_bench(*args, env_extra=None):
    import subprocess
    import sys
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), *args], capture_output=True,
                       text=True, env=env, timeout=300, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_arm_prints_the_contract_line():
    # the reference arm times the oracle on the host cores; the tiny workload keeps this quick
    line = json.loads(_run_bench("--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "tiny")[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 1
    assert line["steps"] == 2 and line["warmup"] >= 3
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["ms_per_step"] == pytest.approx(1000.0 * 512 / line["value"], rel=1e-9)
    assert line["config"]["workload"].startswith("tiny") and line["vs_baseline"] is None
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"] and cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_prints_only_on_rank_zero():
    out = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "tiny",
                     env_extra={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out == []


def test_cpu_baseline_times_whole_unsampled_oracle_steps():
    # the tiny workload: every row scored, every kept row attended; stage times add up to the step
    wl = I.WORKLOADS["tiny"]
    cache = {}
    t = bench.oracle_step(wl, wl.K, cache)
    assert set(t) == {"score", "select", "gather", "attention", "step"}
    parts = t["score"] + t["select"] + t["gather"] + t["attention"]
    assert 0.0 < parts <= t["step"] * 1.0001 + 1e-6
    cpu = bench.cpu_baseline(wl, wl.K, min_s=0.0, max_steps=1)
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1
    assert cpu["value"] == pytest.approx(wl.T_total / (cpu["ms_per_step"] / 1000.0))
    assert "unsampled" in cpu["sample"] and "1 whole" in cpu["sample"]
    thr = cpu["front_stages_by_threads"]
    assert thr["single_thread"] is not None and thr["threads_all_cores"] >= 1
    assert set(thr["single_thread"]) == set(thr["all_cores"]) == {"score", "select", "gather"}


def test_stage_summary_fractions_use_the_measured_peaks():
    import numpy as np
    wl = I.WORKLOADS["sweep_32k"]
    work = bench.stage_work(wl, 4096, [4352])
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1500.0}
    per_stage = np.array([[0.05, 0.01, 0.01, 0.1]])          # ms per stage
    st = bench.stage_summary(work, per_stage, peaks)
    assert st["gate_score"]["frac"] == pytest.approx(work["gate_score"]["flops"] / 50e-6 / 1e12 / 1500.0)
    assert st["gather_kept"]["frac"] == pytest.approx(work["gather_kept"]["bytes"] / 10e-6 / 1e9 / 6000.0)
    sg = bench.select_gather_summary(work, st, peaks)
    assert sg["us"] == pytest.approx(20.0)
    assert sg["frac"] == pytest.approx((work["topk_select"]["bytes"] + work["gather_kept"]["bytes"]) / 20e-6 / 1e9
                                       / 6000.0)
