"""The multi-GPU PCP step (context_prefill_attention_gb300/ranks.py) through
the real kernels, with W ranks played in one process on one GPU: each rank has
its own paged cache, the collective is replaced by the ranks' own send buffers
(the same bytes an all-gather delivers), and the ranks run one after another
(no kernel of one waits on another's). Each rank's cache must equal the
single-rank cache bit for bit, and each rank's output rows must match the
oracle at its own tokens."""
import numpy as np
import pytest
import torch

import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world,mode", [(2, 0), (3, 1)], ids=["2_ranks_contiguous", "3_ranks_dual_chunk"])
def test_ranks_match_oracle_and_single_rank_cache(world, mode):
    import context_prefill_attention_gb300 as P
    from context_prefill_attention_gb300 import ranks as R
    P.load()
    spec = W.custom_spec([700, 1, 300, 1, 129], [0, 900, 64, 40, 0], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, block_size=16, num_shards=world, split_mode=mode, seed=4100 + world)
    ref = Case(spec)                      # the single-rank step: its cache is the reference
    ref.run()
    k, v, q = ref.k_new, ref.v_new, ref.q
    plan = P.pcp_build_row_plan(spec.query_len, spec.num_computed, ref.bt, spec.block_size, world, mode)
    counts = R.token_counts(plan, world)
    owns = [R.own_tokens(plan, r) for r in range(world)]
    sends = [R.send_buffer(k[o].cuda(), v[o].cuda(), max(counts)) for o in owns]
    bt_dev = ref.bt.cuda()
    max_kv = ref.bt.shape[1] * spec.block_size
    for r in range(world):
        case = Case(spec)                 # fresh caches holding only the cached prefixes
        rank = R.PcpRank(r, world, num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                         head_dim=spec.head_dim, block_size=spec.block_size, split_mode=mode,
                         max_tokens=spec.total_q, max_reqs=spec.num_reqs, max_kv_len=max_kv,
                         gather=lambda x: sends)
        rank.build_plan(spec.query_len, spec.num_computed, ref.bt)
        own = owns[r]
        out, lse = rank.step(q[own].cuda(), k[own].cuda(), v[own].cuda(), case.kc, case.vc, bt_dev, spec.scale)
        torch.cuda.synchronize()
        rank.check_status()
        assert torch.equal(case.kc.view(torch.int16), ref.kc.view(torch.int16)), r
        assert torch.equal(case.vc.view(torch.int16), ref.vc.view(torch.int16)), r
        # the rank's compact outputs against the oracle at its own (packed) tokens
        ro, rl = ref.oracle(own)
        got_o = out.double().cpu().numpy()
        got_l = lse.t().double().cpu().numpy()
        assert np.abs(got_o - ro).max() <= OUT_TOL, r
        assert np.abs(got_l - rl).max() <= LSE_TOL, r
