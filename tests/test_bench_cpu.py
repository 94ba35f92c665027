"""The benchmark's own arithmetic (CPU only): the algorithmic FLOP and byte
counts it divides by, against a brute-force count over every query token, and
the rule that a stored DRAM-traffic figure is used only for the workload and
kernel sources it was captured on."""
import json
import os

import numpy as np
import pytest

import bench
import oracle
import workloads as W


def _brute(spec):
    """Per query token: it attends keys [0, pos] of its request (pos = its
    absolute position). Prefill tokens contribute 4 D Hq FLOP per key; decode
    tokens (N == 1 with a cached prefix) are counted apart, with their K/V bytes."""
    bt, _ = W.block_tables(spec)
    rows = oracle.row_plan(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size, spec.num_shards,
                           spec.split_mode)["rows"]
    pre_pairs = dec_keys = n_dec = 0
    for r in rows:
        q_len, kv_end, is_dec = int(r[3]), int(r[5]), int(r[7])
        for j in range(q_len):
            keys = kv_end - q_len + j + 1
            if is_dec:
                dec_keys += keys
                n_dec += 1
            else:
                pre_pairs += keys
    return rows, pre_pairs, dec_keys, n_dec


@pytest.mark.parametrize("kv_bytes", [2, 1])
@pytest.mark.parametrize("case", [
    dict(q=[300, 1, 77, 1], p=[0, 500, 13, 9], hq=8, hkv=2, d=128),
    dict(q=[129, 1], p=[0, 4000], hq=32, hkv=8, d=128, mode=1),
    dict(q=[64, 64, 1], p=[1, 2, 3], hq=4, hkv=4, d=64, s=4),
])
def test_plan_work_matches_brute_force(case, kv_bytes):
    spec = W.custom_spec(case["q"], case["p"], num_q_heads=case["hq"], num_kv_heads=case["hkv"],
                         head_dim=case["d"], num_shards=case.get("s", 2), split_mode=case.get("mode", 0))
    rows, pre_pairs, dec_keys, n_dec = _brute(spec)
    w = bench.plan_work(rows, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, kv_bytes)
    D, hq, hkv = spec.head_dim, spec.num_q_heads, spec.num_kv_heads
    assert w["prefill_flop"] == 4.0 * D * hq * pre_pairs
    assert w["decode_flop"] == 4.0 * D * hq * dec_keys
    assert w["decode_bytes"] == dec_keys * hkv * D * kv_bytes * 2 + n_dec * (hq * D * 2 * 2 + hq * 4)
    # cache write: each new token's K and V read as bf16 and written at kv_bytes, plus its slot
    assert w["write_bytes"] == sum(case["q"]) * (2 * hkv * D * (2 + kv_bytes) + 8)


def test_plan_work_on_the_bench_workload():
    spec = W.workload_spec(4)
    rows, pre_pairs, dec_keys, n_dec = _brute(spec)
    w = bench.plan_work(rows, spec.num_q_heads, spec.num_kv_heads, spec.head_dim)
    assert n_dec == 56 and w["prefill_flop"] == 4.0 * 128 * 32 * pre_pairs
    assert w["decode_bytes"] == dec_keys * 8 * 128 * 2 * 2 + 56 * (32 * 128 * 4 + 32 * 4)


def test_stored_traffic_only_for_its_workload_and_sources(monkeypatch):
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        entry = json.load(f)["prefill_kernel"]
    assert entry["bytes_per_launch"] == entry["dram_read_bytes"] + entry["dram_write_bytes"]
    assert bench.measured_traffic("some-other-workload") is None
    if entry["source_hash"] == bench.kernel_source_hash():
        assert bench.measured_traffic(entry["workload"]) == entry["bytes_per_launch"]
    # once the kernel sources change, the stored figure is no longer reported
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.measured_traffic(entry["workload"]) is None


def test_merge_bytes_counts_both_partials_and_the_result():
    T, hq, d = 37, 4, 128
    read = 2 * (T * hq * d * 4) + 2 * (hq * T * 4)     # out_a, out_b fp32; lse_a, lse_b fp32
    written = T * hq * d * 2 + hq * T * 4              # out bf16, lse fp32
    assert bench.merge_bytes(T, hq, d) == read + written


def _run_bench(args, env_extra=None):
    import subprocess
    import sys
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py")] + args, capture_output=True,
                          text=True, timeout=300, env=env, cwd=bench.ROOT)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_reference_arm_prints_one_contract_line(kv):
    """The reference arm (the oracle on the host cores) prints one JSON line with
    the contract's keys, on the same metric and workload naming as the native arm."""
    r = _run_bench(["--impl", "reference", "--workload", "1", "--steps", "1", "--warmup", "0",
                    "--ref-seconds", "0.5", "--kv-cache", kv])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["value"] > 0
    assert line["config"]["workload"].endswith("-fp8kv") == (kv == "fp8")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _run_bench(["--impl", "reference", "--workload", "1", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and not r.stdout.strip()
