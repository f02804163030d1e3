"""Host-side checks of bench.py: the algorithmic byte counts behind the roofline, the whole-job rate,
and the reference arm's JSON line (the oracle on the host cores, on a small sample)."""
import argparse
import os

import numpy as np

import bench


def test_algorithmic_bytes_per_layer():
    # 102,400 tokens, 8 kv / 32 q heads: 102,080 history tokens x 8 heads x 80 B, 320 BF16 tokens x 8 x 512 B,
    # and q + o in bf16
    assert bench.layer_bytes(np.array([102400]), 8, 32) == 102080 * 8 * 80 + 320 * 8 * 512 + 2 * 32 * 128 * 2
    assert bench.layer_bytes(np.array([300]), 8, 32) == 300 * 8 * 512 + 2 * 32 * 128 * 2     # BF16 segments only
    # a shared prefix counts its history and sink pages once
    lens = np.array([102400] * 4)
    full = bench.layer_bytes(lens, 8, 32)
    uniq = bench.shared_unique_bytes(lens, 92160, 8, 32)
    assert full - uniq == 3 * ((92160 - 64) * 8 * 80 + 64 * 8 * 512)


def test_whole_job_rate_and_single_rank_reductions():
    assert bench.whole_job_rate(1000.0, 2.0, 4) == 1000.0 * 4 / 2e-3
    assert bench.max_over_ranks(3.5, 1, None) == 3.5


def test_reference_arm_line(monkeypatch):
    monkeypatch.setattr(bench, "REFERENCE_SAMPLE_TOKENS", 1024)
    args = argparse.Namespace(workload="qwen3_8b_l1", steps=1, warmup=3, meta_format="f16")
    res = bench.run_reference(args, 0, 1)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in res, key
    assert res["impl"] == "reference" and res["metric"] == bench.METRIC and res["unit"] == bench.UNIT
    assert res["value"] > 0 and res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["cores"] >= 1
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["value"] == res["value"]
    assert "first 1024 tokens" in res["cpu_baseline"]["sample"]
    # the measured CPU seconds per wall second cover every thread of the process (numpy's BLAS pool and any
    # other library's), so they are bounded by the machine's cores, not by the BLAS pool alone; over a
    # sample this short the process clock's granularity (and a container whose quota exceeds the cores it
    # reports) allow a generous margin
    assert 0 < res["cpu_baseline"]["cpu_s_per_wall_s"] <= (os.cpu_count() or 1) * 2.0 + 1.0
    assert bench.run_reference(args, 1, 2) is None            # other ranks print nothing


def test_cpu_baseline_sampler_cycles_heads_until_min_time():
    import time
    seen = []

    def fake(hd):
        seen.append(hd)
        time.sleep(0.01)

    n, dt, busy = bench.time_head_decodes(fake, 3, 0.08, 5.0)
    assert n == len(seen) and n >= 4 and dt >= 0.08
    assert seen == [i % 3 for i in range(n)]            # the layer's kv heads in turn
    assert busy >= 0.0                                   # (a BLAS pool left spinning by earlier work counts)
    seen.clear()
    n, dt, _ = bench.time_head_decodes(fake, 3, 10.0, 0.03)
    assert 1 <= n <= 10 and dt < 1.0                     # the budget ends it long before the minimum time
