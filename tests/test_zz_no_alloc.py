"""pcp_attn_varlen_noalloc: the attention call for callers that cannot
allocate device memory (a framework that owns all device memory, or a serving
loop that may not call cudaMalloc after start-up). Instead of a caller-provided
workspace it uses the library's fixed per-GPU scratch array.

The test calls it through the C ABI twice in a row (the array keeps the first
call's contents, which must not leak into the second) and checks each output
against the workspace entry point pcp_attn_varlen on the same inputs, within
the parity tolerance. The batch has decode rows (the split-KV decode kernel
keeps its per-split partials in the scratch) and runs with and without the
separate context/new-token partials (also kept in the scratch).

This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("flags", [0, 1], ids=["fused", "separate"])
def test_noalloc_matches_workspace_entry_point_twice(flags):
    import context_prefill_attention_gb300 as P
    lib = P.load()
    spec = W.custom_spec([700, 1, 1, 300, 1], [0, 2100, 5, 900, 777], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, block_size=16, num_shards=2, seed=777)
    case = Case(spec, flags=flags)
    ref_out, ref_lse = case.run()
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    n = int(case.plan["rows"].shape[0])
    rows = case.step.rows_dev[:n]
    T, hq = spec.total_q, spec.num_q_heads
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = lib.pcp_attn_varlen_noalloc(
            ctypes.c_void_p(case.q_dev.data_ptr()), ctypes.c_void_p(case.kc.data_ptr()),
            ctypes.c_void_p(case.vc.data_ptr()), ctypes.c_void_p(case.bt_dev.data_ptr()), int(case.bt.shape[0]),
            int(case.bt.shape[1]), int(case.kc.shape[0]), spec.block_size, ctypes.c_void_p(rows.data_ptr()), n,
            T, hq, spec.num_kv_heads, spec.head_dim, float(spec.scale), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), flags, ctypes.c_void_p(status.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == P.PCP_OK, rc
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isfinite(out.float()).all()
        assert (out.float() - ref_out.float()).abs().max().item() <= OUT_TOL, call
        assert (lse - ref_lse).abs().max().item() <= LSE_TOL, call
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL


def test_noalloc_rejects_oversized_batch():
    import context_prefill_attention_gb300 as P
    lib = P.load()
    # 1M query tokens x 64 heads of separate fp32 partials need far more than the fixed scratch
    rc = lib.pcp_attn_varlen_noalloc(None, None, None, None, 1, 1, 1, 16, None, 1, 1 << 20, 64, 8, 128, 0.1,
                                     None, None, 1, None, None)
    assert rc == P.PCP_ERR_WORKSPACE
