"""pcp_attn_varlen_noalloc: the attention call for callers that cannot
allocate device memory (a framework that owns all device memory, or a serving
loop that may not call cudaMalloc after start-up). Instead of a caller-provided
workspace it uses the library's fixed per-GPU scratch array.

The array keeps each call's contents for the next one, so the main test makes
calls in a row whose scratch contents differ: first a larger batch (more rows,
longer contexts and so more decode splits, separate context/new-token partials),
then a smaller batch with other row and split counts, fused and then separate.
A stale byte read from an earlier call would show up in a later one. Each call
is checked through the C ABI against the workspace entry point pcp_attn_varlen
run on a workspace filled with NaN bytes, within the parity tolerance, and the
smaller batch also against the oracle.

This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case

pytestmark = pytest.mark.gpu


def _lib():
    import context_prefill_attention_gb300 as P
    return P, P.load()


def _noalloc(lib, case: Case, flags: int):
    spec = case.spec
    n = int(case.plan["rows"].shape[0])
    rows = case.step.rows_dev[:n]
    T, hq = spec.total_q, spec.num_q_heads
    out = torch.full((T, hq, spec.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((hq, T), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.pcp_attn_varlen_noalloc(
        ctypes.c_void_p(case.q_dev.data_ptr()), ctypes.c_void_p(case.kc.data_ptr()),
        ctypes.c_void_p(case.vc.data_ptr()), ctypes.c_void_p(case.bt_dev.data_ptr()), int(case.bt.shape[0]),
        int(case.bt.shape[1]), int(case.kc.shape[0]), spec.block_size, ctypes.c_void_p(rows.data_ptr()), n,
        T, hq, spec.num_kv_heads, spec.head_dim, float(spec.scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), flags, ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, int(status.item()), out, lse


def _reference(case: Case):
    """pcp_attn_varlen on a workspace whose bytes are all 0xFF (NaN as fp32)."""
    case.step.workspace.fill_(0xFF)
    out, lse = case.run()
    return out.clone(), lse.clone()


LARGE = dict(q=[1500, 1, 1, 1, 900, 1, 600], p=[0, 6000, 4000, 3000, 2000, 5000, 100])
SMALL = dict(q=[300, 1, 1], p=[0, 2100, 900])


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row():
    P, lib = _lib()
    large = W.custom_spec(LARGE["q"], LARGE["p"], num_q_heads=8, num_kv_heads=2, head_dim=128, seed=778)
    small = W.custom_spec(SMALL["q"], SMALL["p"], num_q_heads=8, num_kv_heads=2, head_dim=128, seed=779)
    calls = [(large, 1), (small, 0), (small, 1)]
    for i, (spec, flags) in enumerate(calls):
        case = Case(spec, flags=flags)
        ref_out, ref_lse = _reference(case)
        rc, st, out, lse = _noalloc(lib, case, flags)
        assert rc == P.PCP_OK and st == 0, (i, rc, st)
        assert torch.isfinite(out.float()).all(), i
        assert (out.float() - ref_out.float()).abs().max().item() <= OUT_TOL, i
        assert (lse - ref_lse).abs().max().item() <= LSE_TOL, i
        if spec is small:
            eo, el = case.compare(out, lse)
            assert eo <= OUT_TOL and el <= LSE_TOL, (i, eo, el)


def test_noalloc_empty_call_is_ok():
    """No rows: nothing to do, PCP_OK, as for pcp_attn_varlen."""
    P, lib = _lib()
    rc = lib.pcp_attn_varlen_noalloc(None, None, None, None, 1, 1 << 28, 1, 16, None, 0, 0, 64, 8, 128, 0.1,
                                     None, None, 1, None, None)
    assert rc == P.PCP_OK


def test_noalloc_rejects_oversized_batch():
    """Valid buffers, but a key capacity per request whose decode partials need
    far more than the fixed scratch: PCP_ERR_WORKSPACE, nothing written."""
    P, lib = _lib()
    q = torch.zeros((64, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 16, 2, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    rows = torch.zeros((64, 8), dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    lse = torch.full((8, 64), 3.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    # 64 rows x 8 heads x (2^26 keys / 2048 per split) x 2 partials x 128 dims of fp32: 16 GiB
    rc = lib.pcp_attn_varlen_noalloc(ptr(q), ptr(kc), ptr(kc), ptr(bt), 1, 1 << 22, 4, 16, ptr(rows), 64, 64, 8,
                                     2, 128, 0.1, ptr(out), ptr(lse), 0, ptr(status), None)
    torch.cuda.synchronize()
    assert rc == P.PCP_ERR_WORKSPACE
    assert torch.all(out.float() == 3.0) and torch.all(lse == 3.0) and int(status.item()) == 0
