"""Failure detection on the GPU without a GPU fault.

* A stuck pipeline: the bounded mbarrier wait gives up and reports
  PCP_ERR_TIMEOUT through the status word; the context stays usable.
* Bad inputs that only the device can see (a block-table entry past the cache,
  plan rows out of range) are caught by the kernels' own bounds checks: they
  report PCP_ERR_RANGE, skip the bad accesses and leave the rest correct.
Every access in these tests stays inside its buffer by construction of those
checks; nothing traps, faults or hangs.
"""
import ctypes
import time

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


def test_bounded_wait_reports_timeout_and_context_survives():
    P = _P()
    lib = P.load()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    rc = lib.pcp_selftest_bounded_wait(ctypes.c_void_p(status.data_ptr()), 2000,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == P.PCP_OK
    torch.cuda.synchronize()
    assert int(status.item()) == P.PCP_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    # the device still computes correctly afterwards
    spec = W.custom_spec([130, 1], [0, 77], num_q_heads=4, num_kv_heads=2, head_dim=128, seed=9)
    case = Case(spec)
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL
    assert lib.pcp_selftest_bounded_wait(None, 10, None) == P.PCP_ERR_ARG


def test_block_table_entry_past_the_cache_is_reported():
    P = _P()
    spec = W.custom_spec([300, 1], [40, 500], num_q_heads=4, num_kv_heads=2, head_dim=128, seed=10)
    case = Case(spec)
    case.run()                                  # plan + cache write with the good table
    bad = case.bt.clone()
    bad[0, 1] = case.num_blocks + 7             # a page of request 0 (prefill) past the cache
    bad[1, 3] = 1 << 30                         # a page of request 1 (decode) far past it
    case.step.status.zero_()
    out, lse = case.step.attend(case.q_dev, case.kc, case.vc, bad.cuda(), spec.scale)
    torch.cuda.synchronize()
    assert int(case.step.status.item()) == P.PCP_ERR_RANGE
    assert torch.isfinite(out[:spec.total_q].float()).all()


def test_invalid_plan_rows_are_skipped_and_reported():
    P = _P()
    spec = W.custom_spec([200, 100], [0, 30], num_q_heads=4, num_kv_heads=2, head_dim=128, seed=11)
    case = Case(spec)
    case.run()
    rows = case.plan["rows"].copy()
    keep = rows[:, 0] == 0                      # request 0's rows stay valid
    rows[rows[:, 0] == 1, 0] = 5                # request index past the batch
    extra = rows[0:1].copy()
    extra[0, 2] = spec.total_q - 10             # q range running past the packed tokens
    extra[0, 3] = 50
    rows = np.concatenate([rows, extra])
    out = torch.full((spec.total_q, 4, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((4, spec.total_q), 3.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pcp_attn_varlen(case.q_dev, case.kc, case.vc, case.bt_dev, torch.from_numpy(rows).cuda(), spec.scale,
                      out=out, lse=lse, workspace=case.step.workspace, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == P.PCP_ERR_RANGE
    assert torch.all(out[200:].float() == 3.0) and torch.all(lse[:, 200:] == 3.0)   # skipped rows untouched
    eo, el = case.compare(out, lse, np.arange(200))                                   # valid rows still right
    assert eo <= OUT_TOL and el <= LSE_TOL
    assert keep.sum() > 0


@pytest.mark.parametrize("kv_fp8,hq", [(False, 8), (True, 8), (True, 32)],
                         ids=["tc_bf16", "tc_fp8", "cuda_core_fp8_g16"])
def test_decode_page_past_the_cache_is_reported(kv_fp8, hq):
    """A decode-only batch with one bad page in one row's context: the decode
    kernel that runs (tensor cores for G = 4; CUDA cores for FP8 at G = 16)
    reports PCP_ERR_RANGE, reads a zero-filled page instead, and the other row
    still matches the oracle."""
    P = _P()
    spec = W.custom_spec([1, 1], [500, 3000], num_q_heads=hq, num_kv_heads=2, head_dim=128, seed=12)
    case = Case(spec, kv_fp8=kv_fp8)
    case.run()
    bad = case.bt.clone()
    bad[0, 5] = case.num_blocks + 3             # a page inside request 0's context, past the cache
    case.step.status.zero_()
    out, lse = case.step.attend(case.q_dev, case.kc, case.vc, bad.cuda(), spec.scale)
    torch.cuda.synchronize()
    assert int(case.step.status.item()) == P.PCP_ERR_RANGE
    assert torch.isfinite(out[:spec.total_q].float()).all()
    eo, el = case.compare(out, lse, np.array([1]))
    assert eo <= OUT_TOL and el <= LSE_TOL
