"""The multi-rank host path on CPU (gloo, world size 2).

Each rank plays one PCP shard: it builds the same row plan, keeps the
PAD-masked slot mapping of its own shard ("[MRv2][PCP] Carry the row plan
...", commit "drop pcp_has_prefill": every entry a rank must not write is
PAD, decode rows are written by rank 0 only), and the ranks all-gather their
views: together they write every token exactly once. The benchmark's
max-over-ranks timing reduction is checked the same way.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import bench
        import workloads as W
        import context_prefill_attention_gb300 as P
        spec = W.custom_spec([300, 1, 77, 1, 500], [0, 40, 12, 999, 3], num_q_heads=4, num_kv_heads=2,
                             head_dim=64, block_size=16, num_shards=world, split_mode=W.SPLIT_DUAL_CHUNK)
        bt, _ = W.block_tables(spec)
        plan = P.pcp_build_row_plan(spec.query_len, spec.num_computed, bt, 16, world, W.SPLIT_DUAL_CHUNK)
        mine = P.pcp_mask_slots_for_shard(plan["slot_mapping"], plan["owner_shard"], rank)
        views = [torch.zeros(len(mine), dtype=torch.int64) for _ in range(world)]
        dist.all_gather(views, torch.from_numpy(mine))
        stacked = torch.stack(views).numpy()
        written = (stacked >= 0).sum(0)
        ok_once = bool(np.all(written == 1))
        union = stacked.max(0)
        ok_union = bool(np.array_equal(union, plan["slot_mapping"]))
        decode_tokens = [int(r[2]) for r in plan["rows"] if r[7] == 1]
        ok_decode = all(stacked[0][t] >= 0 and all(stacked[k][t] < 0 for k in range(1, world))
                        for t in decode_tokens)
        own_rows = int((plan["rows"][:, 1] == rank).sum())
        t_max = bench.max_over_ranks(float(rank + 1) * 1.5, world)
        q.put((rank, ok_once, ok_union, ok_decode, own_rows, t_max))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, "error", repr(e)))


def test_two_ranks_write_every_token_once_and_agree_on_max_time():
    from context_prefill_attention_gb300 import build
    build.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    assert all(r[1] != "error" for r in results), results
    for rank, ok_once, ok_union, ok_decode, own_rows, t_max in results:
        assert ok_once and ok_union and ok_decode
        assert own_rows <= 2 * 5
        assert t_max == pytest.approx(3.0)
