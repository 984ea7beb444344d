"""Host-side logic of bench.py (no GPU): algorithmic bytes, the traffic
record lookup, and the JSON line of the reference arm (the CPU oracle)."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_algorithmic_bytes_of_the_workloads():
    W = workloads.WORKLOADS
    # Q, K, V read once and Y written once: 4 d bf16 values a head-token
    dit = W["dit"]
    assert bench.tokens_per_step(dit) == 8 * 6 * 4096
    assert bench.workload_bytes(dit) == 196_608 * 512 + 6 * 16 * 16 * 4  # + the mixing matrix
    assert bench.workload_bytes(W["causal"]) == 524_288 * 512
    # RALA, d = 32: Q, K, V, Y 4 x 32 x 2 bytes a head-token, X once per token, W once
    rala = W["rala"]
    assert bench.workload_bytes(rala) == 401_408 * 256 + 64 * 3136 * 64 * 2 + 64 * 32 * 2
    # decode: the fp32 state (S and z) read and written, q, k, v, out in bf16
    dec = W["decode"]
    assert bench.tokens_per_step(dec) == 256 * 16
    assert bench.workload_bytes(dec) == 4096 * (2 * (64 * 64 + 64) * 4 + 4 * 64 * 2)
    # fused decode: the state once in and out, 1024 steps of q, k, v, out (bf16) and den (fp32)
    fused = W["decode_fused"]
    assert bench.tokens_per_step(fused) == 4096 * 1024
    assert bench.workload_bytes(fused) == 4096 * (2 * (64 * 64 + 64) * 4 + 1024 * (4 * 64 * 2 + 4))
    assert bench.workload_flops(fused) == 4096 * 1024 * (4 * 64 * 64 + 3 * 64)
    assert abs(bench.fp32_peak_tflops(152) - 80.548) < 0.001
    # causal MHLA inference of 1024 tokens after 2048 (16 frozen blocks of 128, 8 blocks touched):
    # tokens' q, k, v, out and den; the 16 frozen slots read once; the 8 touched slots written once;
    # 3 d^2 + 3 d FMAs a token, and blocks 16 .. 23 each mix the i slots before them
    st = W["stream"]
    slot = (64 * 64 + 64) * 4
    assert bench.tokens_per_step(st) == 4096 * 1024
    assert bench.workload_bytes(st) == 4096 * (1024 * (4 * 64 * 2 + 4) + 16 * slot + 8 * slot)
    assert bench.workload_flops(st) == 4096 * (1024 * (6 * 64 * 64 + 5 * 64) + 156 * 2 * (64 * 64 + 64))
    # backward on the DiT inputs: Q, K, V, dY in, dQ, dK, dV out (bf16), the mixing in and dM out (fp32)
    bw = W["dit_backward"]
    assert bench.workload_bytes(bw) == 196_608 * 64 * 2 * 7 + 2 * 6 * 16 * 16 * 4
    assert bench.workload_flops(bw) == 48 * (4096 * (12 * 64 * 64 + 13 * 64) + 6 * 16 * 16 * (64 * 64 + 64))


def test_traffic_record_needs_matching_sources(monkeypatch):
    records = []
    for path in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        text = open(os.path.join(ROOT, "profiles", path)).read()
        fields = dict(l.split(":", 1) for l in text.splitlines() if ":" in l and l.split(":")[0] in
                      ("bench_kernel", "workload", "traffic_bytes_per_launch", "source_sha256"))
        if "bench_kernel" in fields:
            records.append((fields["bench_kernel"].strip(), fields["workload"].strip(),
                            float(fields["traffic_bytes_per_launch"]), fields["source_sha256"].strip()))
    assert records, "no profile names a bench kernel"
    monkeypatch.setattr(bench, "source_digest", lambda *a: "0" * 16)
    for kname, wname, _, _ in records:
        assert bench.parse_traffic(kname, wname) is None  # counters of other sources are not reported
    for kname, wname, traffic, digest in records:
        monkeypatch.setattr(bench, "source_digest", lambda *a, d=digest: d)
        assert bench.parse_traffic(kname, wname) == traffic
        assert bench.parse_traffic(kname, "no-such-workload") is None
    # each record is keyed on its own family's sources
    monkeypatch.undo()
    assert bench.source_digest("mhla_tcgen05") != bench.source_digest("causal_tcgen05")


def test_hbm_peak_is_positive():
    peak, src = bench.hbm_peak()
    assert peak > 1000.0 and src


@pytest.mark.timeout(300)
def test_reference_arm_json_line(capsys):
    bench.main(["--impl", "reference", "--workload", "causal", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("causal")


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "2"])
