"""Decode rows beside the prefill rows (PCP_ATTN_DECODE_SMS).

Mixed prefill + decode batches in one attention call are the pages' case
("[MRv2] FlashAttention PCP support for GQA on MRv2", overview). With the flag
the library runs the decode rows on a few SMs of a stream of its own while the
prefill rows take the rest. A prefill work item's result does not depend on
the grid, so the prefill rows must keep every bit. A decode item shares its key
tiles between two softmax warpgroups by a count that runs on across the CTA's
items, so another split sums the same terms in another order: the decode rows
agree with the sequence up to fp32 rounding. These tests check both at several
SM counts with both caches, check the split against the oracle, and replay a
step with the split from a CUDA graph.
"""
import numpy as np
import pytest
import torch

import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case

pytestmark = pytest.mark.gpu


def _P():
    import context_prefill_attention_gb300 as P
    P.load()
    return P


def _mixed_spec(seed, hq=16, hkv=4, prompts=(700, 300, 129, 1000)):
    """Long and short prompts, prompts with a cached prefix, and decode rows of
    1 to 9000 keys (partial and whole 2048-key splits)."""
    rng = np.random.default_rng(seed)
    q = list(prompts) + [1] * 24
    p = [0, 2000, 40, 0][:len(prompts)] + rng.integers(1, 9000, size=24).tolist()
    return W.custom_spec(q, p, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, seed=seed)


def _attend(case, flags):
    P = _P()
    st = case.step
    T = case.spec.total_q
    n = int(st.plan["rows"].shape[0])
    out = torch.empty_like(case.q_dev)
    lse = torch.empty((case.spec.num_q_heads, T), dtype=torch.float32, device="cuda")
    if case.kv_fp8:
        R = case.spec.num_reqs
        P.pcp_attn_varlen_fp8kv(case.q_dev, case.kc, case.vc, st.k_descale[:R], st.v_descale[:R], case.bt_dev,
                                st.rows_dev[:n], case.spec.scale, out=out, lse=lse, workspace=st.workspace,
                                flags=flags, status=st.status)
    else:
        P.pcp_attn_varlen(case.q_dev, case.kc, case.vc, case.bt_dev, st.rows_dev[:n], case.spec.scale, out=out,
                          lse=lse, workspace=st.workspace, flags=flags, status=st.status)
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return out, lse


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16", "fp8"])
def test_split_against_the_sequence(kv_fp8):
    """1, 7, 19 and 75 decode SMs against none: prefill tokens bit for bit;
    decode tokens within a few fp32 rounding steps of lse (and one bf16 step of
    out); every split within the oracle's bounds; a split repeated gives its
    own bits again."""
    P = _P()
    case = Case(_mixed_spec(71), kv_fp8=kv_fp8, descales="varied")
    case.run()                                   # writes the new tokens' K/V
    rows = case.plan["rows"]
    dec = torch.tensor([int(r[2]) for r in rows if int(r[7])], device="cuda")
    pre = torch.tensor(sorted(set(range(case.spec.total_q)) - set(dec.tolist())), device="cuda")
    assert len(dec) == 24 and len(pre) > 0
    ref_o, ref_l = _attend(case, 0)
    for k in (1, 7, 19, 75):
        o, l = _attend(case, P.PCP_ATTN_DECODE_SMS(k))
        assert torch.equal(o[pre], ref_o[pre]) and torch.equal(l[:, pre], ref_l[:, pre]), k
        d_l = (l[:, dec] - ref_l[:, dec]).abs().max().item()
        d_o = (o[dec].float() - ref_o[dec].float()).abs() / ref_o[dec].float().abs().clamp_min(2.0 ** -8)
        assert d_l <= 1e-5 and d_o.max().item() <= 2.0 ** -7, (k, d_l, d_o.max().item())
        eo, el = case.compare(o, l)
        assert eo <= OUT_TOL and el <= LSE_TOL, (k, eo, el)
        o2, l2 = _attend(case, P.PCP_ATTN_DECODE_SMS(k))
        assert torch.equal(o2, o) and torch.equal(l2, l), k


def test_split_matches_oracle_and_the_step_picks_it():
    """PcpStep, asked to, picks a split for a mixed bf16 batch (none for an FP8
    cache, none unless asked); the step's result matches the oracle."""
    spec = _mixed_spec(72, hq=32, hkv=8, prompts=(6000, 5000, 3000, 7000))
    case = Case(spec, decode_beside=True)
    assert case.step.decode_sms > 0
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert Case(spec, kv_fp8=True, decode_beside=True).step.decode_sms == 0
    assert Case(spec).step.decode_sms == 0


def test_split_inside_a_cuda_graph():
    """The fork to the library's stream and the join back are captured with the
    caller's stream; a replay gives the bits of a direct call with the same split."""
    P = _P()
    case = Case(_mixed_spec(73))
    case.run()
    k = P.PCP_ATTN_DECODE_SMS(19)
    ref_o, ref_l = _attend(case, k)              # first call: the internal stream exists before capture
    st = case.step
    n = int(st.plan["rows"].shape[0])
    out = torch.zeros_like(case.q_dev)
    lse = torch.zeros((case.spec.num_q_heads, case.spec.total_q), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        P.pcp_attn_varlen(case.q_dev, case.kc, case.vc, case.bt_dev, st.rows_dev[:n], case.spec.scale, out=out,
                          lse=lse, workspace=st.workspace, flags=k, status=st.status)
    torch.cuda.synchronize()
    for _ in range(2):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
