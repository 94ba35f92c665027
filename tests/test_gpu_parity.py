"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact: cache contents. Floating point: max |out - oracle| <= 1e-2 and
max |lse - oracle| <= 1e-3 over every compared (token, head).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case, shard_segments

pytestmark = pytest.mark.gpu

SEP = 1
ROWSTART = 2


def _P():
    import context_prefill_attention_gb300 as P
    P.load()
    return P


def test_cache_write_bit_exact_with_pad_slots():
    P = _P()
    spec = W.custom_spec([37, 1, 200, 5], [0, 19, 40, 3], num_q_heads=4, num_kv_heads=2, head_dim=128,
                         block_size=16, num_shards=2)
    bt, nb = W.block_tables(spec)
    plan = P.pcp_build_row_plan(spec.query_len, spec.num_computed, bt, 16, 2)
    k = W.packed_new_tokens(spec, W.KIND_K)
    v = W.packed_new_tokens(spec, W.KIND_V)
    for shard in (0, 1):
        slot = P.pcp_mask_slots_for_shard(plan["slot_mapping"], plan["owner_shard"], shard)
        kc = torch.full((nb, 16, 2, 128), 7.0, dtype=torch.bfloat16)
        vc = torch.full((nb, 16, 2, 128), -3.0, dtype=torch.bfloat16)
        ref_k = kc.view(torch.int16).numpy().view(np.uint16).copy()
        ref_v = vc.view(torch.int16).numpy().view(np.uint16).copy()
        assert oracle.cache_write(k, slot, ref_k) == 0
        assert oracle.cache_write(v, slot, ref_v) == 0
        kd, vd = kc.cuda(), vc.cuda()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        P.pcp_kv_cache_write(k.cuda(), v.cuda(), torch.from_numpy(slot).cuda(), kd, vd, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        np.testing.assert_array_equal(kd.cpu().view(torch.int16).numpy().view(np.uint16), ref_k)
        np.testing.assert_array_equal(vd.cpu().view(torch.int16).numpy().view(np.uint16), ref_v)


def test_cache_write_reports_slot_past_end():
    P = _P()
    kc = torch.zeros((4, 16, 1, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones((3, 1, 64), dtype=torch.bfloat16, device="cuda")
    slot = torch.tensor([0, 64, -1], dtype=torch.int64, device="cuda")   # 64 = one past the end
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pcp_kv_cache_write(k, k, slot, kc, vc, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == P.PCP_ERR_RANGE
    assert float(kc[0, 0, 0, 0]) == 1.0 and float(kc.float().sum()) == 64.0


SMALL = {
    "ragged_d128": dict(q=[300], p=[0], hq=4, hkv=2, d=128),
    "d64_two_reqs": dict(q=[200, 77], p=[0, 0], hq=4, hkv=2, d=64),
    "prefix": dict(q=[150, 40], p=[333, 17], hq=8, hkv=2, d=128),
    "mha_single_slot": dict(q=[260], p=[5], hq=2, hkv=2, d=128),
    "gqa8": dict(q=[129], p=[64], hq=16, hkv=2, d=128),
    "gqa3_odd": dict(q=[140], p=[10], hq=6, hkv=2, d=64),
    "mixed_decode": dict(q=[257, 1, 1, 1], p=[0, 700, 31, 1], hq=4, hkv=1, d=128),
    "decode_g8": dict(q=[1, 1, 33], p=[1500, 2, 0], hq=8, hkv=1, d=128),
    "one_token_prompt": dict(q=[1, 50], p=[0, 0], hq=4, hkv=2, d=128),
    "bs32": dict(q=[333, 90], p=[41, 0], hq=4, hkv=2, d=128, bs=32),
    "bs128": dict(q=[400], p=[130], hq=4, hkv=2, d=64, bs=128),
    "bs8": dict(q=[150], p=[21], hq=4, hkv=2, d=128, bs=8),
    "dual_chunk": dict(q=[1000, 333], p=[0, 100], hq=4, hkv=2, d=128, mode=1),
    "four_shards": dict(q=[777], p=[0], hq=4, hkv=1, d=128, s=4),
    "many_reqs": dict(q=[3, 64, 129, 1, 17, 256, 2, 90, 1, 500], p=[0, 5, 0, 44, 130, 0, 1, 7, 300, 0],
                      hq=8, hkv=4, d=128),
}


@pytest.mark.parametrize("flags", [0, SEP, SEP | ROWSTART], ids=["fused", "separate", "split_at_row_start"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_cases_match_oracle(name, flags):
    c = SMALL[name]
    spec = W.custom_spec(c["q"], c["p"], num_q_heads=c["hq"], num_kv_heads=c["hkv"], head_dim=c["d"],
                         block_size=c.get("bs", 16), num_shards=c.get("s", 2), split_mode=c.get("mode", 0),
                         seed=zlib.crc32(name.encode()) % 100000)
    case = Case(spec, flags=flags)
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("shards", [2, 3, 5])
@pytest.mark.parametrize("name", ["ragged_d128", "prefix", "mixed_decode", "gqa3_odd", "many_reqs", "bs32"])
def test_kv_shard_partials_match_oracle(name, shards):
    """Decode-context-parallel emulation: every row's keys in `shards` contiguous
    shards, one partial each, merged by LSE — the same attention."""
    import context_prefill_attention_gb300 as P
    c = SMALL[name]
    spec = W.custom_spec(c["q"], c["p"], num_q_heads=c["hq"], num_kv_heads=c["hkv"], head_dim=c["d"],
                         block_size=c.get("bs", 16), num_shards=c.get("s", 2), split_mode=c.get("mode", 0),
                         seed=zlib.crc32(name.encode()) % 100000 + shards)
    case = Case(spec, flags=P.PCP_ATTN_KV_SHARDS(shards))
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_workload3_kv_shards_matches_oracle():
    import context_prefill_attention_gb300 as P
    spec = W.workload_spec(3)
    case = Case(spec, flags=P.PCP_ATTN_KV_SHARDS(4))
    out, lse = case.run()
    segs = shard_segments(case.plan["rows"])
    tokens = W.sample_segments(segs, 48, spec.seed + 13).numpy()
    eo, el = case.compare(out, lse, tokens)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_separate_context_with_empty_prefix_merges_to_new_part():
    """Rows without a cached prefix have an empty context pass (lse = -inf);
    the merge must return the new-token part unchanged (the 'context pass
    skipped when the max context length is 0' trap)."""
    spec = W.custom_spec([300, 64], [0, 200], num_q_heads=4, num_kv_heads=2, head_dim=128)
    a = Case(spec, flags=SEP)
    out_a, lse_a = a.run()
    b = Case(spec, flags=0)
    out_b, lse_b = b.run()
    eo, el = a.compare(out_a, lse_a)
    assert eo <= OUT_TOL and el <= LSE_TOL
    assert (out_a.float() - out_b.float()).abs().max().item() <= 2 * OUT_TOL


def test_deterministic_bits():
    spec = W.custom_spec([513, 1, 70], [0, 900, 64], num_q_heads=8, num_kv_heads=2, head_dim=128)
    case = Case(spec)
    o1, l1 = case.run()
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = case.run()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_untouched_tokens_stay_untouched():
    """Output rows of tokens no plan row covers are never written."""
    P = _P()
    spec = W.custom_spec([200, 100], [0, 0], num_q_heads=4, num_kv_heads=2, head_dim=128)
    case = Case(spec)
    case.step.out.fill_(5.0)
    case.step.lse_buf.fill_(5.0)
    n = case.plan["rows"].shape[0]
    keep = [i for i in range(n) if case.plan["rows"][i][0] == 0]
    rows = torch.from_numpy(case.plan["rows"][keep]).cuda()
    case.step.upload_plan()
    case.step.write_cache(case.k_dev, case.v_dev, case.kc, case.vc)
    out, lse = P.pcp_attn_varlen(case.q_dev, case.kc, case.vc, case.bt_dev, rows, spec.scale,
                                 out=case.step.out[:spec.total_q],
                                 lse=case.step.lse_buf[:spec.total_q * 4].view(4, spec.total_q),
                                 workspace=case.step.workspace, status=case.step.status)
    torch.cuda.synchronize()
    assert torch.all(out[200:].float() == 5.0) and torch.all(lse[:, 200:] == 5.0)
    eo, el = case.compare(out, lse, np.arange(200))
    assert eo <= OUT_TOL and el <= LSE_TOL


def test_lse_merge_kernel_matches_oracle():
    P = _P()
    g = torch.Generator().manual_seed(5)
    T, H, D = 300, 4, 128
    # partial outputs are convex combinations of value rows; keep them in [-2, 2]
    # so that the bf16 rounding of the merged output stays inside the tolerance
    oa = torch.rand((T, H, D), generator=g) * 4 - 2
    ob = torch.rand((T, H, D), generator=g) * 4 - 2
    la = torch.randn((H, T), generator=g) * 4
    lb = torch.randn((H, T), generator=g) * 4
    la[0, :10] = float("-inf")
    lb[0, 5:15] = float("-inf")
    out, lse = P.pcp_lse_merge(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.lse_merge(oa.double().numpy(), la.t().double().numpy(),
                              ob.double().numpy(), lb.t().double().numpy())
    np.testing.assert_allclose(out.double().cpu().numpy(), ro, atol=OUT_TOL)
    got_l = lse.t().double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_l), np.isneginf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(got_l[fin], rl[fin], atol=LSE_TOL)


# ------------------------------------------------------------ full workloads

# None: every token; n: a seeded sample of n query tokens per shard row plus its
# first and last (the 131072-token prompt: 4096 of each shard's 32768)
SAMPLES = {1: None, 2: None, 3: None, 4: None, 5: 4096}


@pytest.mark.parametrize("workload", [1, 2, 3, 4, 5])
def test_workload_matches_oracle(workload):
    """The five workloads at full size, in the launch configuration the
    benchmark times. Workloads 1-4 compare every output (all heads of every
    token, decode rows included); workload 5 compares 4096 seeded query tokens
    of each of its four shards plus each shard's first and last token."""
    spec = W.workload_spec(workload)
    case = Case(spec)
    out, lse = case.run()
    k = SAMPLES[workload]
    if k is None:
        tokens = None
    else:
        rows = case.plan["rows"]
        segs = [(int(r[2]), int(r[3])) for r in rows]
        tokens = W.sample_segments(segs, k, spec.seed + 11).numpy()
    eo, el = case.compare(out, lse, tokens)
    print(f"workload {workload}: max|out err| {eo:.3e}  max|lse err| {el:.3e}")
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_workload2_dual_chunk_matches_oracle():
    spec = W.workload_spec(2, split_mode=W.SPLIT_DUAL_CHUNK)
    case = Case(spec)
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_workload3_separate_context_matches_oracle():
    spec = W.workload_spec(3)
    case = Case(spec, flags=SEP)
    out, lse = case.run()
    segs = shard_segments(case.plan["rows"])
    tokens = W.sample_segments(segs, 64, spec.seed + 12).numpy()
    eo, el = case.compare(out, lse, tokens)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


# ------------------------------------------------------------ edge cases

EDGE = {
    "all_decode": dict(q=[1, 1, 1, 1, 1], p=[5, 900, 33, 1, 2048], hq=8, hkv=2, d=128),
    "one_shard": dict(q=[300, 1, 77], p=[0, 40, 200], hq=4, hkv=2, d=128, s=1),
    "request_without_new_tokens": dict(q=[0, 150, 0, 1], p=[64, 10, 30, 99], hq=4, hkv=2, d=128),
    "gqa16": dict(q=[140, 1], p=[9, 300], hq=16, hkv=1, d=128),
    "gqa16_d64": dict(q=[140, 1], p=[9, 300], hq=32, hkv=2, d=64),
    "eight_shards_dual": dict(q=[1000], p=[3], hq=4, hkv=2, d=64, s=8, mode=1),
    "tile_exact": dict(q=[256, 128], p=[128, 0], hq=4, hkv=2, d=128),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_cases_match_oracle(name):
    c = EDGE[name]
    spec = W.custom_spec(c["q"], c["p"], num_q_heads=c["hq"], num_kv_heads=c["hkv"], head_dim=c["d"],
                         block_size=c.get("bs", 16), num_shards=c.get("s", 2), split_mode=c.get("mode", 0),
                         seed=zlib.crc32(name.encode()) % 100000)
    case = Case(spec)
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_empty_plan_and_empty_batch_launch_nothing():
    P = _P()
    q = torch.zeros((4, 2, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((2, 16, 1, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    rows = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    lse = torch.full((2, 4), 7.0, device="cuda")
    P.pcp_attn_varlen(q, kc, kc, bt, rows, 0.1, out=out, lse=lse,
                      workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(out.float() == 7.0) and torch.all(lse == 7.0)
    plan = P.pcp_build_row_plan([0, 0], [3, 0], np.zeros((2, 1), np.int32), 16, 2)
    assert plan["rows"].shape[0] == 0 and plan["slot_mapping"].shape[0] == 0


# ------------------------------------------------------------ rising scores

def _rising_keys(step: float):
    """Inputs whose scores rise by about `step` (natural-log units) per 128-key
    tile: positive queries and keys shifted by step-proportional offsets, so
    the kernel's running reference max is overtaken again and again (the
    path that falls back from the max-free exponentials). The softmax is then
    peaked (a few keys carry almost all the weight), where rounding P to bf16
    costs up to ~2^-8 |v| (a CPU emulation of exactly that rounding gives
    1.14e-2 with N(0, 1) values on the 700-token case); V is halved to keep
    |v| within the range the 1e-2 bound assumes."""
    def hook(case):
        case.q = case.q.float().abs().to(torch.bfloat16)
        D = case.spec.head_dim
        per_unit = float(case.q.float().abs().sum(-1).mean()) * case.spec.scale
        for r, k in enumerate(case.kfull):
            idx = torch.arange(k.shape[0], dtype=torch.float32)
            shift = (idx // 128) * step / per_unit
            case.kfull[r] = (k.float() * 0.1 + shift[:, None, None]).to(torch.bfloat16)
            case.vfull[r] = (case.vfull[r].float() * 0.5).to(torch.bfloat16)
    return hook


@pytest.mark.parametrize("step", [20.0, 60.0])
@pytest.mark.parametrize("name,q,p,hq,hkv,d", [
    ("prefill", [700], [0], 4, 2, 128),
    ("prefix_decode", [300, 1], [400, 900], 8, 2, 128),
    ("d64", [520], [0], 4, 2, 64),
])
def test_rising_scores_match_oracle(name, q, p, hq, hkv, d, step):
    spec = W.custom_spec(q, p, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                         seed=zlib.crc32(f"rise{name}{step}".encode()) % 100000)
    case = Case(spec, inputs_hook=_rising_keys(step))
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
