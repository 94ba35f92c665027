"""GPU parity of the FP8 (e4m3) KV-cache path against the CPU oracle.

Bit-exact: the FP8 cache write (codes) against the oracle's encoder, including
hand-picked ties, subnormals, signed zero and saturation. Floating point: the
attention over the codes with per-(request, kv head) descales, max |out -
oracle| <= 1e-2 and max |lse - oracle| <= 1e-3, in every prefill / decode /
split mode.
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


def _write_and_compare(P, k, v, slot, nb, bs, H, D, k_scale, v_scale):
    kc = torch.full((nb, bs, H, D), 0x7F, dtype=torch.uint8)
    vc = torch.full((nb, bs, H, D), 0x7F, dtype=torch.uint8)
    ref_k, ref_v = kc.numpy().copy(), vc.numpy().copy()
    assert oracle.cache_write_fp8(k, slot, ref_k, k_scale) == 0
    assert oracle.cache_write_fp8(v, slot, ref_v, v_scale) == 0
    kd, vd = kc.cuda(), vc.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pcp_kv_cache_write_fp8(k.cuda(), v.cuda(), torch.from_numpy(slot).cuda(), kd, vd, k_scale, v_scale,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(kd.cpu().numpy(), ref_k)
    np.testing.assert_array_equal(vd.cpu().numpy(), ref_v)


def test_fp8_cache_write_bit_exact_with_pad_slots():
    P = _P()
    spec = W.custom_spec([37, 1, 200, 5], [0, 19, 40, 3], num_q_heads=4, num_kv_heads=2, head_dim=128,
                         block_size=16, num_shards=2)
    bt, nb = W.block_tables(spec)
    plan = P.pcp_build_row_plan(spec.query_len, spec.num_computed, bt, 16, 2)
    k = W.packed_new_tokens(spec, W.KIND_K) * 3
    v = W.packed_new_tokens(spec, W.KIND_V)
    for shard in (0, 1):
        slot = P.pcp_mask_slots_for_shard(plan["slot_mapping"], plan["owner_shard"], shard)
        _write_and_compare(P, k, v, slot, nb, 16, 2, 128, W.FP8_K_SCALE, W.FP8_V_SCALE)


def test_fp8_cache_write_ties_subnormals_zero_and_saturation():
    """Power-of-two scales make x / scale exact, so the values below reach the
    encoder as they are: halfway cases (ties to even), the subnormal range,
    signed zeros and values far past 448 (saturation)."""
    P = _P()
    special = [1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, -(2.0 ** -11), 0.0, -0.0, 448.0, 464.0,
               1.0e4, -1.0e4, 2.0 ** -9, 7 * 2.0 ** -9, 0.0146484375, 240.0, 248.0, -232.0, 2.0 ** -7 * 1.5]
    T, H, D = 5, 2, 64
    g = torch.Generator().manual_seed(3)
    x = torch.randn((T, H, D), generator=g) * 50
    flat = x.view(-1)
    flat[:len(special)] = torch.tensor(special)
    for scale in (1.0, 0.5, 0.125):
        k = (x * scale).to(torch.bfloat16)        # exact: every value above has <= 8 significant bits
        v = (-x * scale).to(torch.bfloat16)
        slot = np.array([3, 0, -1, 7, 5], dtype=np.int64)
        _write_and_compare(P, k, v, slot, 2, 4, H, D, scale, scale)


def test_fp8_cache_write_reports_slot_past_end():
    P = _P()
    kc = torch.zeros((4, 16, 1, 64), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones((3, 1, 64), dtype=torch.bfloat16, device="cuda")
    slot = torch.tensor([0, 64, -1], dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pcp_kv_cache_write_fp8(k, k, slot, kc, vc, 1.0, 1.0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == P.PCP_ERR_RANGE
    assert int(kc[0, 0, 0, 0]) == 0x38 and int(kc.sum()) == 64 * 0x38


def test_fp8_cache_write_rejects_bad_scales():
    P = _P()
    kc = torch.zeros((1, 16, 1, 64), dtype=torch.uint8, device="cuda")
    k = torch.ones((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    slot = torch.zeros(1, dtype=torch.int64, device="cuda")
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        with pytest.raises(P.PcpError) as e:
            P.pcp_kv_cache_write_fp8(k, k, slot, kc, kc.clone(), ks, vs)
        assert e.value.code == P.PCP_ERR_ARG


FP8_CASES = {
    "ragged_d128": dict(q=[300], p=[0], hq=4, hkv=2, d=128),
    "d64_two_reqs": dict(q=[200, 77], p=[0, 0], hq=4, hkv=2, d=64),
    "prefix": dict(q=[150, 40], p=[333, 17], hq=8, hkv=2, d=128),
    "gqa3_odd": dict(q=[140], p=[10], hq=6, hkv=2, d=64),
    "mixed_decode": dict(q=[257, 1, 1, 1], p=[0, 700, 31, 1], hq=4, hkv=1, d=128),
    "decode_g8_d64": dict(q=[1, 1, 33], p=[1500, 2, 0], hq=16, hkv=2, d=64),
    "bs32": dict(q=[333, 90], p=[41, 0], hq=4, hkv=2, d=128, bs=32),
    "bs8": dict(q=[150], p=[21], hq=4, hkv=2, d=128, bs=8),
    "bs128": dict(q=[400], p=[130], hq=4, hkv=2, d=64, bs=128),
    "dual_chunk": dict(q=[1000, 333], p=[0, 100], hq=4, hkv=2, d=128, mode=1),
    "many_reqs": dict(q=[3, 64, 129, 1, 17, 256, 2, 90, 1, 500], p=[0, 5, 0, 44, 130, 0, 1, 7, 300, 0],
                      hq=8, hkv=4, d=128),
    "gqa16": dict(q=[140, 1], p=[9, 300], hq=16, hkv=1, d=128),
    "tile_exact": dict(q=[256, 128], p=[128, 0], hq=4, hkv=2, d=128),
    "bs64": dict(q=[200, 1], p=[77, 300], hq=8, hkv=2, d=128, bs=64),
    "gqa16_d64": dict(q=[140, 1, 1], p=[9, 300, 1200], hq=32, hkv=2, d=64),
    # head_dim 128 with an odd group (one head slot per item: one warpgroup splits q
    # into its e4m3 terms and frees Q alone) and a decode row of that group
    "gqa3_odd_d128": dict(q=[140, 1], p=[10, 700], hq=6, hkv=2, d=128),
    "gqa5_d128": dict(q=[200, 1, 1], p=[30, 1025, 9], hq=10, hkv=2, d=128),
    "request_without_new_tokens": dict(q=[0, 150, 0, 1], p=[64, 10, 30, 99], hq=4, hkv=2, d=128),
    "all_decode": dict(q=[1, 1, 1, 1, 1], p=[5, 900, 33, 1, 2048], hq=8, hkv=2, d=128),
}


def _spec(name, extra_seed=0):
    c = FP8_CASES[name]
    return W.custom_spec(c["q"], c["p"], num_q_heads=c["hq"], num_kv_heads=c["hkv"], head_dim=c["d"],
                         block_size=c.get("bs", 16), num_shards=c.get("s", 2), split_mode=c.get("mode", 0),
                         seed=zlib.crc32(("fp8" + name).encode()) % 100000 + extra_seed)


@pytest.mark.parametrize("descales", ["layer", "varied"])
@pytest.mark.parametrize("name", list(FP8_CASES))
def test_fp8_small_cases_match_oracle(name, descales):
    case = Case(_spec(name), kv_fp8=True, descales=descales)
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("mode", ["separate", "split_at_row_start", "kv_shards3"])
@pytest.mark.parametrize("name", ["prefix", "mixed_decode", "many_reqs", "gqa3_odd"])
def test_fp8_split_modes_match_oracle(name, mode):
    import context_prefill_attention_gb300 as P
    flags = {"separate": SEP, "split_at_row_start": SEP | ROWSTART, "kv_shards3": P.PCP_ATTN_KV_SHARDS(3)}[mode]
    case = Case(_spec(name, 1), flags=flags, kv_fp8=True, descales="varied")
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_fp8_descale_doubles_output():
    """Doubling every V descale doubles the output (exactly, up to the bf16
    rounding of out) and leaves lse bit-identical."""
    case = Case(_spec("mixed_decode", 2), kv_fp8=True)
    o1, l1 = case.run()
    o1, l1 = o1.clone(), l1.clone()
    case.step.v_descale.mul_(2.0)
    o2, l2 = case.step.attend(case.q_dev, case.kc, case.vc, case.bt_dev, case.spec.scale)
    torch.cuda.synchronize()
    assert torch.equal(l1, l2)
    assert torch.equal(o2.float(), 2 * o1.float())


def test_fp8_workload4_matches_oracle():
    """The mixed benchmark workload over an FP8 cache (sampled prefill rows,
    every decode row)."""
    spec = W.workload_spec(4)
    case = Case(spec, kv_fp8=True, descales="varied")
    out, lse = case.run()
    segs = shard_segments(case.plan["rows"])
    tokens = W.sample_segments(segs, 128, spec.seed + 17).numpy()
    eo, el = case.compare(out, lse, tokens)
    print(f"fp8 workload 4: max|out err| {eo:.3e}  max|lse err| {el:.3e}")
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_fp8_workload2_matches_oracle():
    spec = W.workload_spec(2)
    case = Case(spec, kv_fp8=True)
    out, lse = case.run()
    segs = shard_segments(case.plan["rows"])
    tokens = W.sample_segments(segs, 128, spec.seed + 18).numpy()
    eo, el = case.compare(out, lse, tokens)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_fp8_q_beyond_f16_range_is_reported():
    """An element of q beyond +-65504 on the FP8 path is reported as
    PCP_ERR_RANGE (head_dim 128 writes q as two e4m3 terms after a per-row
    scale, head_dim 64 converts it to f16 and saturates there); every other
    row's output still matches the oracle."""
    P = _P()
    spec = W.custom_spec([200, 150], [0, 40], num_q_heads=4, num_kv_heads=2, head_dim=128, seed=6550)

    def hook(case):
        case.q = case.q.clone()
        case.q[5, 1, 7] = 1.0e5          # token 5 of the first request, q head 1
    case = Case(spec, kv_fp8=True, inputs_hook=hook)
    out, lse = case.step.run(case.q_dev, case.k_dev, case.v_dev, case.kc, case.vc, case.bt_dev, spec.scale)
    torch.cuda.synchronize()
    assert int(case.step.status.item()) == P.PCP_ERR_RANGE
    others = np.array([t for t in range(spec.total_q) if t != 5])
    eo, el = case.compare(out, lse, others)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
