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


def _pcp_worker(rank, world, port, q):
    """One PCP rank: its own tokens' K/V, the all-gather, and both cache writes
    (the oracle's cache write stands in for the device writer on the CPU)."""
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        import workloads as W
        import context_prefill_attention_gb300 as P
        from context_prefill_attention_gb300 import ranks as R
        spec = W.custom_spec([300, 1, 77, 1, 500, 2], [0, 40, 12, 999, 3, 0], num_q_heads=4, num_kv_heads=2,
                             head_dim=64, block_size=16, num_shards=world, split_mode=W.SPLIT_DUAL_CHUNK)
        bt, nb = W.block_tables(spec)
        plan = P.pcp_build_row_plan(spec.query_len, spec.num_computed, bt, 16, world, W.SPLIT_DUAL_CHUNK)
        k = W.packed_new_tokens(spec, W.KIND_K)
        v = W.packed_new_tokens(spec, W.KIND_V)
        own = R.own_tokens(plan, rank)
        k_all, v_all = R.gather_new_kv(k[own], v[own], plan, world, R.dist_all_gather())
        ok_gather = bool(torch.equal(k_all.view(torch.int16), k.view(torch.int16)) and
                         torch.equal(v_all.view(torch.int16), v.view(torch.int16)))
        # this rank's cache: own tokens through the PAD view, then the others' tokens
        shape = (nb, 16, spec.num_kv_heads, spec.head_dim)
        kc = np.full(shape, 0x7FC1, dtype=np.uint16)
        vc = np.full(shape, 0x7FC1, dtype=np.uint16)
        slot = plan["slot_mapping"]
        assert oracle.cache_write(k[own], slot[own], kc) == 0 and oracle.cache_write(v[own], slot[own], vc) == 0
        other = R.other_slots(plan, rank)
        assert oracle.cache_write(k_all, other, kc) == 0 and oracle.cache_write(v_all, other, vc) == 0
        ref_k = np.full(shape, 0x7FC1, dtype=np.uint16)
        ref_v = np.full(shape, 0x7FC1, dtype=np.uint16)
        assert oracle.cache_write(k, slot, ref_k) == 0 and oracle.cache_write(v, slot, ref_v) == 0
        ok_cache = bool(np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v))
        # own rows: contiguous runs of the compact buffer that map back to the plan's tokens
        rows = R.rank_rows(plan, rank)
        covered = np.zeros(own.shape[0], dtype=np.int64)
        ok_rows = True
        orig = plan["rows"][plan["rows"][:, 1] == rank]
        for r, o in zip(rows, orig):
            s0, n = int(r[2]), int(r[3])
            covered[s0:s0 + n] += 1
            ok_rows &= bool(np.array_equal(own[s0:s0 + n], np.arange(int(o[2]), int(o[2]) + n)))
        ok_rows &= bool(np.all(covered == 1))
        q.put((rank, ok_gather, ok_cache, ok_rows, int(own.shape[0]), int(rows.shape[0])))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, "error", repr(e)))


def test_two_pcp_ranks_gather_kv_into_identical_caches():
    """The multi-GPU PCP step's host and collective logic on two gloo ranks:
    the all-gathered new K/V equal the single-rank tensors bit for bit, each
    rank's cache after its two PAD-masked writes equals the single-rank cache,
    and each rank's rows cover its compact token buffer exactly once; together
    the ranks own every token."""
    from context_prefill_attention_gb300 import build
    build.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_pcp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    assert all(r[1] != "error" for r in results), results
    assert all(r[1] and r[2] and r[3] for r in results), results
    assert sum(r[4] for r in results) == 300 + 1 + 77 + 1 + 500 + 2
