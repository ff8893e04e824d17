"""Host-side logic of bench.py that needs no GPU: the per-sequence-length
workload stays inside its capacities and its byte count reduces to the
uniform one when every sequence has the batch-wide counts."""

import bench
from visual_token_sparsity_gb300 import synth


def test_varlen_counts_within_capacities():
    shape = synth.llava_next_decode(batch=16, keep=0.5, layers=32)
    nv, nt, k = bench.varlen_counts(shape)
    assert len(nv) == len(nt) == len(k) == 16
    for v, t, kk in zip(nv, nt, k):
        assert shape.n_vis // 2 <= v <= shape.n_vis
        assert shape.n_text // 2 <= t <= shape.n_text
        assert 0 <= kk <= min(v, shape.k)
    assert bench.varlen_counts(shape) == (nv, nt, k), "counts must be seeded"


def test_varlen_bytes_reduce_to_uniform():
    shape = synth.llava_next_decode(batch=4, keep=0.5, layers=3)
    B = shape.batch
    rb, ab = bench.decode_bytes(shape)
    assert bench.varlen_bytes(shape, [shape.n_vis] * B, [shape.n_text] * B, [shape.k] * B) == rb + ab


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle timed on host cores) prints one
    JSON line with the keys the base contract and the reference arm need."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("llava-next-7b-decode")


def test_cpu_baseline_reports_single_thread_and_all_cores():
    """The oracle leg of the bench line: single-threaded and on every host
    core (spawned workers), with the core count and CPU model recorded."""
    d = bench.cpu_baseline(synth.tiny_decode(), budget_s=0.2)
    assert d["kind"] == "oracle" and d["unit"] == "GB/s"
    assert d["single_thread_gbs"] > 0 and d["all_cores_gbs"] > 0 and d["value"] == d["all_cores_gbs"]
    assert d["cores"] == bench.host_cores() >= 1
    assert isinstance(d["cpu_model"], str) and d["cpu_model"]
