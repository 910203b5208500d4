"""The per-step roofline arithmetic of bench.py, checked against hand-computed
algorithmic work for the measured workloads: forward 2 G D^2 flops and
(G + S) D e bytes per (b, n, t); backward 4 G D^2 flops and (2S + 2G) D e
bytes."""
import pytest

import bench
from recurrent_networks_gb300.synth import WORKLOADS


def per_step(k, fn, esize):
    w = WORKLOADS[k]
    a = bench.algorithmic(w, fn, esize)
    return {key: v / w["T"] for key, v in a.items() if key != "units"}


def test_lstm_d256_bench_workload():
    # B = 8, N = 3, D = 256, G = 4, S = 2, bf16: 24 sequences per step
    s = per_step(2, "lstm", 2)
    assert s["fwd_bytes"] == 24 * (4 + 2) * 256 * 2 == 73728
    assert s["fwd_flops"] == 24 * 2 * 4 * 256 * 256 == pytest.approx(12.58e6, rel=1e-3)
    assert s["bwd_bytes"] == 24 * (2 * 2 + 2 * 4) * 256 * 2
    assert s["bwd_flops"] == 2 * s["fwd_flops"]
    # at the measured 6789.3 GB/s the forward step's HBM time is 10.86 ns
    assert s["fwd_bytes"] / 6789.3e9 == pytest.approx(10.86e-9, rel=1e-3)


def test_lstm_d1024_is_tensor_bound():
    # B = 32, N = 1, D = 1024: 268 MFLOP per forward step, 140 ns at 1.91 PFLOP/s
    s = per_step(5, "lstm", 2)
    assert s["fwd_flops"] == 32 * 2 * 4 * 1024 * 1024 == pytest.approx(268.4e6, rel=1e-3)
    assert s["fwd_flops"] / 1.9125e15 > s["fwd_bytes"] / 6789.3e9


def test_slstm_counts_four_states():
    s = per_step(4, "slstm", 2)
    assert s["fwd_bytes"] == 16 * 4 * (4 + 4) * 192 * 2
    assert s["bwd_bytes"] == 16 * 4 * (2 * 4 + 2 * 4) * 192 * 2


def test_traffic_record_follows_the_kernel_sources(monkeypatch, tmp_path):
    """A traffic record's DRAM bytes are reported only while the kernel's
    sources hash to what they were when the counters were taken."""
    import json
    rec = tmp_path / "traffic.json"
    key = "fused_bwd_kernel@lstm_bf16_B8_T1024_N3_D256"
    rec.write_text(json.dumps({key: {"dram_bytes_per_launch": 2.0e8,
                                     "sources_sha256": bench.kernel_sources_sha("fused_bwd_kernel")}}))
    got = bench.measured_traffic("fused_bwd_kernel", "lstm_bf16_B8_T1024_N3_D256", path=str(rec))
    assert got == 2.0e8
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda kernel: "0" * 64)
    assert bench.measured_traffic("fused_bwd_kernel", "lstm_bf16_B8_T1024_N3_D256", path=str(rec)) is None
    assert bench.measured_traffic("fused_fwd_kernel", "no_such_workload", path=str(rec)) is None


def test_oracle_sample_is_bounded():
    # the bench workload fits whole; the D = 1024 workload takes a time prefix
    # over at least as many sequences as cores
    w2, w5 = WORKLOADS[2], WORKLOADS[5]
    assert bench.oracle_sample(w2, "lstm", 16) == (w2["B"], w2["T"])
    for budget in (bench.ORACLE_BUDGET_BASELINE, bench.ORACLE_BUDGET_REFERENCE_STEP):
        rows, steps = bench.oracle_sample(w5, "lstm", 16, budget)
        assert rows >= 16 and 8 <= steps < w5["T"]
        assert 3 * 2 * 4 * 1024 * 1024 * rows * steps <= budget


@pytest.mark.parametrize("kernel,main", [("fused_fwd_kernel", "fused_fwd.cuh"), ("fused_bwd_kernel", "fused_bwd.cuh"),
                                         ("grid_bwd_kernel", "grid_bwd.cuh")])
def test_traffic_record_hashes_every_source_of_its_kernel(kernel, main):
    """A DRAM-traffic record counts as current only while the hash of its
    kernel's sources is unchanged: that list must hold every local header the
    kernel's code includes, directly or not, or an edit could leave a stale
    record looking current."""
    import os
    import re
    csrc = os.path.join(bench.ROOT, "recurrent_networks_gb300", "csrc")
    seen, todo = set(), [main]
    while todo:
        f = todo.pop()
        path = os.path.join(csrc, f)
        if f in seen or not os.path.exists(path):
            continue
        seen.add(f)
        todo += re.findall(r'#include\s+"([^"]+)"', open(path).read())
    assert seen <= set(bench.KERNEL_SOURCES[kernel]), sorted(seen - set(bench.KERNEL_SOURCES[kernel]))
