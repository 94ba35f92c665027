"""Seeded random batches through the whole call, against the oracle.

Each case draws every axis of a step at once: the head layout (1 to 16 q heads
per kv head, head_dim 64 or 128), the page size, the number of PCP shards and
the split mode of the row plan ("[MRv2][PCP] Carry the row plan in attention
metadata", sections 1-2), the attention flags (fused, separate context pass,
row-start split, n key shards merged by LSE), the cache type (bf16, or FP8
codes with a different descale per request and kv head), and a mix of request
kinds: decode rows (one new token over a cached context), short and long new
token runs with or without a cached prefix, and requests with no new tokens;
every other case lets the step run its decode rows beside its prefill rows.
Every token of every head is compared with the oracle at the fixed bounds
(max |out - oracle| <= 1e-2, max |lse - oracle| <= 1e-3). The caches start out
NaN-filled, so a read of a slot the step should not touch poisons the result.
"""
import numpy as np
import pytest

import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case

SEP = 1
ROWSTART = 2
NUM_CASES = 32


def draw(i: int) -> dict:
    """Case i: a plain dict of the drawn axes (seeded, the same on every machine)."""
    rng = np.random.default_rng(20_000 + i)
    hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 12, 16]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([8, 16, 32, 64, 128]))
    shards = int(rng.choice([1, 2, 3, 4]))
    mode = int(rng.choice([0, 1]))
    R = int(rng.integers(1, 7))
    q_len, ctx = [], []
    for _ in range(R):
        kind = rng.choice(["decode", "short", "long", "none"], p=[0.35, 0.25, 0.3, 0.1])
        if kind == "decode":
            q_len.append(1)
            ctx.append(int(rng.integers(1, 4200)))
        elif kind == "short":
            q_len.append(int(rng.integers(2, 65)))
            ctx.append(int(rng.integers(0, 600)) if rng.random() < 0.5 else 0)
        elif kind == "long":
            q_len.append(int(rng.integers(65, 520)))
            ctx.append(int(rng.integers(0, 2500)) if rng.random() < 0.5 else 0)
        else:
            q_len.append(0)
            ctx.append(int(rng.integers(1, 300)))
    if sum(q_len) == 0:
        q_len[0] = 1
        ctx[0] = max(ctx[0], 1)
    flags = [0, SEP, SEP | ROWSTART, None][int(rng.integers(0, 4))]
    n_kv = int(rng.integers(2, 6)) if flags is None else 0
    kv_fp8 = bool(rng.random() < 0.3)
    return dict(hq=hkv * G, hkv=hkv, d=d, bs=bs, shards=shards, mode=mode, q_len=q_len, ctx=ctx, flags=flags,
                n_kv=n_kv, kv_fp8=kv_fp8, seed=30_000 + i)


def test_draws_cover_every_axis():
    """The fixed seeds reach every value of the axes that pick a kernel path."""
    cases = [draw(i) for i in range(NUM_CASES)]
    assert {c["d"] for c in cases} == {64, 128}
    assert {c["bs"] for c in cases} == {8, 16, 32, 64, 128}
    assert {c["flags"] for c in cases} == {0, SEP, SEP | ROWSTART, None}
    assert {c["kv_fp8"] for c in cases} == {False, True}
    assert {c["mode"] for c in cases} == {0, 1}
    assert any(c["hq"] // c["hkv"] > 8 for c in cases)
    assert any(c["hq"] // c["hkv"] % 2 == 1 for c in cases)
    assert any(0 in c["q_len"] for c in cases)
    assert any(any(q == 1 and p > 0 for q, p in zip(c["q_len"], c["ctx"])) for c in cases)


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(NUM_CASES), ids=[f"case{i:02d}" for i in range(NUM_CASES)])
def test_random_batch_matches_oracle(i):
    import context_prefill_attention_gb300 as P
    c = draw(i)
    flags = P.PCP_ATTN_KV_SHARDS(c["n_kv"]) if c["flags"] is None else c["flags"]
    spec = W.custom_spec(c["q_len"], c["ctx"], num_q_heads=c["hq"], num_kv_heads=c["hkv"], head_dim=c["d"],
                         block_size=c["bs"], num_shards=c["shards"], split_mode=c["mode"], seed=c["seed"])
    # odd cases let the step run decode rows beside the prefill rows where it picks a split
    case = Case(spec, flags=flags, kv_fp8=c["kv_fp8"], descales="varied", decode_beside=bool(i % 2))
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (c, eo, el)
