"""Pins of the CPU oracle against things other than itself (CPU only).

* dense brute force: per request, a full L x L causal softmax built with numpy
  matrix operations, compared with the oracle's row-decomposed result;
* closed forms: one key, all keys equal, a zero query;
* invariants the pages fix: sharded + LSE-merged attention equals unsharded
  causal attention, the last shard's end-aligned rows equal the tail rows of
  full causal attention, both context/new splits give the same result;
* merge algebra;
* row plan: hand-worked golden fixture, the 14-row mixed batch, partition,
  ownership, per-shard row bound, balance and slot-inversion invariants;
* cache write: read back through the block table.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _random_batch(rng, R, Hq, Hkv, D, bs, max_new=9, max_prefix=7):
    ql = [int(rng.integers(0, max_new + 1)) for _ in range(R)]
    if sum(ql) == 0:
        ql[0] = 3
    nc = [int(rng.integers(0, max_prefix + 1)) for _ in range(R)]
    need = [-(-(p + n) // bs) for p, n in zip(nc, ql)]
    pool = rng.permutation(sum(need) + 3)
    mb = max(1, max(need))
    bt = np.full((R, mb), -1, dtype=np.int32)
    o = 0
    for r, k in enumerate(need):
        bt[r, :k] = pool[o:o + k]
        o += k
    L = [p + n for p, n in zip(nc, ql)]
    kfull = [_bf16(rng.standard_normal((l, Hkv, D))) for l in L]
    vfull = [_bf16(rng.standard_normal((l, Hkv, D))) for l in L]
    q = _bf16(rng.standard_normal((sum(ql), Hq, D)))
    return ql, nc, bt, kfull, vfull, q


def _dense_reference(ql, nc, kfull, vfull, q, Hq, Hkv, scale):
    """Plain causal attention of each request's new tokens over its whole
    sequence: dense score matrix, boolean causal mask, numpy softmax."""
    G = Hq // Hkv
    outs, lses = [], []
    off = 0
    for r, (n, p) in enumerate(zip(ql, nc)):
        if n == 0:
            continue
        L = p + n
        K, V, Q = _f64(kfull[r]), _f64(vfull[r]), _f64(q[off:off + n])
        o_r = np.zeros((n, Hq, Q.shape[-1]))
        l_r = np.zeros((n, Hq))
        qpos = np.arange(p, L)[:, None]
        kpos = np.arange(L)[None, :]
        mask = kpos <= qpos                       # [n, L]
        for h in range(Hq):
            s = scale * (Q[:, h, :] @ K[:, h // G, :].T)    # [n, L]
            s = np.where(mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            z = e.sum(axis=1, keepdims=True)
            o_r[:, h, :] = (e / z) @ V[:, h // G, :]
            l_r[:, h] = (m + np.log(z))[:, 0]
        outs.append(o_r)
        lses.append(l_r)
        off += n
    return np.concatenate(outs, 0), np.concatenate(lses, 0)


def _oracle_all(ql, nc, bt, bs, S, mode, kfull, vfull, q, Hq, Hkv, D, scale, part="fused"):
    plan = oracle.row_plan(ql, nc, bt, bs, S, mode)
    kv_off = np.cumsum([0] + [k.shape[0] for k in kfull[:-1]])
    kk = torch.cat(kfull, 0)
    vv = torch.cat(vfull, 0)
    tokens = np.arange(sum(ql), dtype=np.int64)
    out, lse = oracle.attention(plan["rows"], q, kk, vv, kv_off, Hq, Hkv, D, scale, tokens, part=part)
    return plan, out, lse


@pytest.mark.parametrize("bs", [1, 2, 16])
@pytest.mark.parametrize("S,mode", [(1, 0), (2, 0), (3, 0), (2, 1), (3, 1)])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (2, 1), (4, 2)])
def test_oracle_matches_dense_brute_force(bs, S, mode, Hq, Hkv):
    rng = np.random.default_rng(1000 * bs + 10 * S + mode + Hq * 7 + Hkv)
    D = 8
    scale = 1.0 / math.sqrt(D)
    ql, nc, bt, kf, vf, q = _random_batch(rng, 3, Hq, Hkv, D, bs)
    _, out, lse = _oracle_all(ql, nc, bt, bs, S, mode, kf, vf, q, Hq, Hkv, D, scale)
    ref_o, ref_l = _dense_reference(ql, nc, kf, vf, q, Hq, Hkv, scale)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_brute_force_catches_a_wrong_key_range():
    """The dense comparison would fail for a row that sees one key too many
    (the first query of a shard seeing its own successor)."""
    rng = np.random.default_rng(5)
    D, Hq, Hkv = 8, 2, 1
    ql, nc, bt, kf, vf, q = _random_batch(rng, 2, Hq, Hkv, D, 2)
    plan = oracle.row_plan(ql, nc, bt, 2, 2, 0)
    lo, hi = oracle.key_ranges(plan["rows"], "fused")
    rows = plan["rows"].copy()
    rows[:, 5] += 1                      # kv_end one past the row end
    kv_off = np.cumsum([0] + [k.shape[0] for k in kf[:-1]])
    kk = torch.cat([torch.cat([k, k[-1:]], 0) for k in kf], 0)   # pad so the extra key exists
    vv = torch.cat([torch.cat([v, v[-1:] + 1], 0) for v in vf], 0)
    kv_off = np.cumsum([0] + [k.shape[0] + 1 for k in kf[:-1]])
    tokens = np.arange(sum(ql))
    out, _ = oracle.attention(rows, q, kk, vv, kv_off, Hq, Hkv, D, 0.3, tokens, key_lo=lo, key_hi=hi + 1)
    ref_o, _ = _dense_reference(ql, nc, kf, vf, q, Hq, Hkv, 0.3)
    assert np.abs(out - ref_o).max() > 1e-3


@pytest.mark.parametrize("split", [("context", "new"), ("before_row", "own")])
@pytest.mark.parametrize("S,mode", [(2, 0), (2, 1), (4, 0)])
def test_context_plus_new_merged_equals_fused(split, S, mode):
    """Context pass over the cached prefix merged by LSE with the causal pass
    over the new tokens equals the single fused pass, for both ways of
    splitting a row ("Carry the row plan ...", "What made it removable")."""
    rng = np.random.default_rng(77 + S + 10 * mode + len(split[0]))
    D, Hq, Hkv = 8, 4, 2
    ql, nc, bt, kf, vf, q = _random_batch(rng, 4, Hq, Hkv, D, 2, max_new=11, max_prefix=13)
    _, fo, fl = _oracle_all(ql, nc, bt, 2, S, mode, kf, vf, q, Hq, Hkv, D, 0.4)
    _, ao, al = _oracle_all(ql, nc, bt, 2, S, mode, kf, vf, q, Hq, Hkv, D, 0.4, part=split[0])
    _, bo, bl = _oracle_all(ql, nc, bt, 2, S, mode, kf, vf, q, Hq, Hkv, D, 0.4, part=split[1])
    mo, ml = oracle.lse_merge(ao, al, bo, bl)
    np.testing.assert_allclose(mo, fo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, fl, rtol=0, atol=1e-12)


@pytest.mark.parametrize("nshards", [2, 3, 5])
def test_kv_sharded_partials_merged_equal_full(nshards):
    """Splitting every row's keys into contiguous shards (the DCP-style split)
    and merging the partials by LSE gives the full causal result."""
    rng = np.random.default_rng(300 + nshards)
    D, Hq, Hkv = 8, 2, 1
    ql, nc, bt, kf, vf, q = _random_batch(rng, 3, Hq, Hkv, D, 4, max_new=12, max_prefix=9)
    plan, fo, fl = _oracle_all(ql, nc, bt, 4, 2, 0, kf, vf, q, Hq, Hkv, D, 0.5)
    rows = plan["rows"]
    kv_off = np.cumsum([0] + [k.shape[0] for k in kf[:-1]])
    kk, vv = torch.cat(kf, 0), torch.cat(vf, 0)
    tokens = np.arange(sum(ql))
    acc_o = acc_l = None
    for i in range(nshards):
        lo = (rows[:, 5].astype(np.int64) * i) // nshards
        hi = (rows[:, 5].astype(np.int64) * (i + 1)) // nshards
        o, l = oracle.attention(rows, q, kk, vv, kv_off, Hq, Hkv, D, 0.5, tokens, key_lo=lo, key_hi=hi)
        if acc_o is None:
            acc_o, acc_l = o, l
        else:
            acc_o, acc_l = oracle.lse_merge(acc_o, acc_l, o, l)
    np.testing.assert_allclose(acc_o, fo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(acc_l, fl, rtol=0, atol=1e-12)


def test_last_shard_end_aligned_equals_tail_of_full_causal():
    """The last shard of a prompt is end-aligned: its rows reproduce the last
    q_len rows of unsharded causal attention ("Feat/pcp qwen36 hybrid",
    "Changes")."""
    rng = np.random.default_rng(9)
    D, Hq, Hkv = 8, 4, 2
    n = 23
    ql, nc = [n], [0]
    bt = np.arange(-(-n // 4), dtype=np.int32)[None, :]
    kf = [_bf16(rng.standard_normal((n, Hkv, D)))]
    vf = [_bf16(rng.standard_normal((n, Hkv, D)))]
    q = _bf16(rng.standard_normal((n, Hq, D)))
    _, full_o, full_l = _oracle_all(ql, nc, bt, 4, 1, 0, kf, vf, q, Hq, Hkv, D, 0.35)
    plan, sh_o, sh_l = _oracle_all(ql, nc, bt, 4, 4, 0, kf, vf, q, Hq, Hkv, D, 0.35)
    last = plan["rows"][-1]
    assert last[1] == 3 and last[5] == n
    tail = slice(n - last[3], n)
    np.testing.assert_allclose(sh_o[tail], full_o[tail], rtol=0, atol=1e-13)
    np.testing.assert_allclose(sh_l[tail], full_l[tail], rtol=0, atol=1e-13)
    # and the dense definition agrees
    ref_o, ref_l = _dense_reference(ql, nc, kf, vf, q, Hq, Hkv, 0.35)
    np.testing.assert_allclose(sh_o, ref_o, rtol=0, atol=1e-12)


def test_closed_form_single_key():
    """One visible key: out = v_0, lse = scale * q . k_0."""
    rng = np.random.default_rng(3)
    D, Hq, Hkv = 16, 2, 1
    k = _bf16(rng.standard_normal((1, Hkv, D)))
    v = _bf16(rng.standard_normal((1, Hkv, D)))
    q = _bf16(rng.standard_normal((1, Hq, D)))
    _, out, lse = _oracle_all([1], [0], np.array([[0]], np.int32), 16, 1, 0, [k], [v], q, Hq, Hkv, D, 0.25)
    for h in range(Hq):
        np.testing.assert_array_equal(out[0, h], _f64(v[0, 0]))
        assert lse[0, h] == pytest.approx(0.25 * float(_f64(q[0, h]) @ _f64(k[0, 0])), abs=1e-12)


def test_closed_form_equal_keys_and_zero_query():
    """All keys equal: uniform weights, out = mean of the visible values,
    lse = s + ln(n_visible). A zero query: lse = ln(n_visible)."""
    rng = np.random.default_rng(4)
    D, Hq, Hkv, n, p = 8, 2, 1, 6, 5
    k = _bf16(np.repeat(rng.standard_normal((1, Hkv, D)), n + p, axis=0))
    v = _bf16(rng.standard_normal((n + p, Hkv, D)))
    q = _bf16(rng.standard_normal((n, Hq, D)))
    q[:, 1, :] = 0
    bt = np.arange(-(-(n + p) // 2), dtype=np.int32)[None, :]
    _, out, lse = _oracle_all([n], [p], bt, 2, 2, 0, [k], [v], q, Hq, Hkv, D, 0.3)
    V = _f64(v)[:, 0, :]
    for j in range(n):
        vis = p + j + 1
        np.testing.assert_allclose(out[j, 0], V[:vis].mean(0), atol=1e-12)
        s = 0.3 * float(_f64(q[j, 0]) @ _f64(k[0, 0]))
        assert lse[j, 0] == pytest.approx(s + math.log(vis), abs=1e-12)
        assert lse[j, 1] == pytest.approx(math.log(vis), abs=1e-12)
        np.testing.assert_allclose(out[j, 1], V[:vis].mean(0), atol=1e-12)


def test_decode_row_is_last_row_of_full_causal():
    """A decode row (one new token after C-1 cached ones) equals the last row
    of a full causal pass over the C tokens."""
    rng = np.random.default_rng(12)
    D, Hq, Hkv, C = 8, 4, 1, 19
    k = _bf16(rng.standard_normal((C, Hkv, D)))
    v = _bf16(rng.standard_normal((C, Hkv, D)))
    qall = _bf16(rng.standard_normal((C, Hq, D)))
    bt = np.arange(-(-C // 4), dtype=np.int32)[None, :]
    _, full_o, full_l = _oracle_all([C], [0], bt, 4, 1, 0, [k], [v], qall, Hq, Hkv, D, 0.3)
    plan, dec_o, dec_l = _oracle_all([1], [C - 1], bt, 4, 2, 0, [k], [v], qall[C - 1:], Hq, Hkv, D, 0.3)
    assert plan["rows"].shape[0] == 1 and plan["rows"][0, 7] == 1
    np.testing.assert_allclose(dec_o[0], full_o[-1], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dec_l[0], full_l[-1], rtol=0, atol=1e-13)


def test_empty_key_range_gives_minus_inf_and_zero():
    """A pass with no visible key (an empty context) yields lse = -inf and
    out = 0 ("Carry the row plan ...", the max_dcp_context_kv_len == 0 trap)."""
    rng = np.random.default_rng(13)
    D, Hq, Hkv = 8, 2, 2
    k = _bf16(rng.standard_normal((5, Hkv, D)))
    v = _bf16(rng.standard_normal((5, Hkv, D)))
    q = _bf16(rng.standard_normal((5, Hq, D)))
    _, o, l = _oracle_all([5], [0], np.array([[0, 1, 2]], np.int32), 2, 2, 0, [k], [v], q, Hq, Hkv, D, 0.3,
                          part="context")
    assert np.all(np.isneginf(l)) and np.all(o == 0)


def test_merge_algebra():
    rng = np.random.default_rng(21)
    n, D = 50, 7
    parts = [(rng.standard_normal((n, D)), rng.standard_normal(n) * 3) for _ in range(3)]
    (a, la), (b, lb), (c, lc) = parts
    ab, lab = oracle.lse_merge(a, la, b, lb)
    ba, lba = oracle.lse_merge(b, lb, a, la)
    np.testing.assert_allclose(ab, ba, atol=1e-14)
    np.testing.assert_allclose(lab, lba, atol=1e-14)
    abc1, l1 = oracle.lse_merge(ab, lab, c, lc)
    bc, lbc = oracle.lse_merge(b, lb, c, lc)
    abc2, l2 = oracle.lse_merge(a, la, bc, lbc)
    np.testing.assert_allclose(abc1, abc2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)
    # lse of the merge is log(exp(la) + exp(lb)); weights follow the softmax definition
    np.testing.assert_allclose(lab, np.logaddexp(la, lb), atol=1e-12)
    wa = 1.0 / (1.0 + np.exp(lb - la))
    np.testing.assert_allclose(ab, wa[:, None] * a + (1 - wa)[:, None] * b, atol=1e-12)
    # an empty partial is the identity; two empty partials give (0, -inf)
    e_o, e_l = np.full((n, D), 5.0), np.full(n, -np.inf)
    io, il = oracle.lse_merge(a, la, e_o, e_l)
    np.testing.assert_array_equal(io, a)
    np.testing.assert_array_equal(il, la)
    zo, zl = oracle.lse_merge(e_o, e_l, e_o, e_l)
    assert np.all(zo == 0) and np.all(np.isneginf(zl))


# ----------------------------------------------------------------- row plan

def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_plan_hand_worked_fixture():
    g = _load("plan_small_handworked.json")
    plan = oracle.row_plan(g["query_len"], g["num_computed"], g["block_table"], g["block_size"],
                           g["num_shards"], g["split_mode"])
    assert plan["rows"].tolist() == g["rows"]
    assert plan["cu_q"].tolist() == g["cu_q"]
    assert plan["slot"].tolist() == g["slot_mapping"]
    assert plan["owner"].tolist() == g["owner_shard"]


def test_plan_mixed_batch_has_14_rows_on_shard0():
    g = _load("plan_mixed_batch_14_rows.json")
    spec = W.custom_spec(g["query_len"], g["num_computed"], num_q_heads=2, num_kv_heads=1, head_dim=8,
                         block_size=g["block_size"], num_shards=g["num_shards"], split_mode=g["split_mode"])
    bt, _ = W.block_tables(spec)
    plan = oracle.row_plan(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size,
                           spec.num_shards, spec.split_mode)
    per = np.bincount(plan["rows"][:, 1], minlength=spec.num_shards).tolist()
    assert per == g["rows_per_shard"]
    assert plan["rows"].shape[0] == g["rows_total"]
    # a buffer sized by the number of requests would have overflowed
    assert max(per) > len(g["query_len"])
    with pytest.raises(oracle.OracleError):
        oracle.row_plan(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size,
                        spec.num_shards, spec.split_mode, rows_cap=len(g["query_len"]))


def _check_plan_invariants(ql, nc, bt, bs, S, mode, plan):
    rows, slot, owner, cu = plan["rows"], plan["slot"], plan["owner"], plan["cu_q"]
    R = len(ql)
    offs = np.concatenate([[0], np.cumsum(ql)])
    covered = np.zeros(int(offs[-1]), dtype=np.int64)
    assert cu[0] == 0 and np.all(np.diff(cu) == rows[:, 3])
    # shard-major row order
    assert np.all(np.diff(rows[:, 1]) >= 0)
    for row in rows:
        req, shard, qs, qn, ctx, end, coff, dec = [int(x) for x in row]
        assert qn > 0
        assert offs[req] <= qs and qs + qn <= offs[req + 1]
        assert ctx == nc[req]
        start = nc[req] + (qs - offs[req])          # absolute position of the row's first token
        assert end - qn == start                    # seq_len - query_len is the row start
        assert coff == end - ctx - qn
        assert dec == int(ql[req] == 1 and nc[req] > 0)
        if ql[req] == 1:
            assert shard == 0
        covered[qs:qs + qn] += 1
        assert np.all(owner[qs:qs + qn] == shard)
    assert np.all(covered == 1)                     # each token in exactly one row
    for s in range(S):
        assert np.sum(rows[:, 1] == s) <= 2 * R     # up to two rows per request per shard
    for r in range(R):
        for j in range(ql[r]):
            t, pos = offs[r] + j, nc[r] + j
            blk, off = divmod(int(slot[t]), bs)
            assert blk == bt[r][pos // bs] and off == pos % bs
    if mode == 0:
        for r in range(R):
            if ql[r] <= 1:
                continue
            sizes = [int(x[3]) for x in rows if x[0] == r]
            sizes += [0] * (S - len(sizes))
            assert max(sizes) - min(sizes) <= 1
    else:
        for r in range(R):
            if ql[r] < 2 * S:
                continue
            pairs = np.zeros(S)
            for x in rows:
                if x[0] == r:
                    pairs[x[1]] += sum(x[5] - x[3] + j + 1 for j in range(x[3]))
            assert pairs.max() - pairs.min() <= 4 * (ql[r] + nc[r])


@pytest.mark.parametrize("seed", range(12))
def test_plan_invariants_random(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 9))
    S = int(rng.integers(1, 5))
    mode = int(rng.integers(0, 2))
    bs = int(rng.choice([1, 2, 4, 16]))
    ql = [int(rng.choice([0, 1, 1, 2, 3, 7, 40, 123])) for _ in range(R)]
    nc = [int(rng.integers(0, 50)) for _ in range(R)]
    need = [-(-(p + n) // bs) for p, n in zip(nc, ql)]
    pool = rng.permutation(sum(need) + 2)
    bt = np.full((R, max(1, max(need))), -1, dtype=np.int32)
    o = 0
    for r, k in enumerate(need):
        bt[r, :k] = pool[o:o + k]
        o += k
    plan = oracle.row_plan(ql, nc, bt, bs, S, mode)
    _check_plan_invariants(ql, nc, bt, bs, S, mode, plan)


@pytest.mark.parametrize("workload", [1, 2, 3, 4, 5])
def test_plan_invariants_workloads(workload):
    spec = W.workload_spec(workload)
    bt, _ = W.block_tables(spec)
    plan = oracle.row_plan(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size,
                           spec.num_shards, spec.split_mode)
    expected_rows = {1: 2, 2: 16, 3: 8, 4: 72, 5: 4}[workload]
    assert plan["rows"].shape[0] == expected_rows
    if workload == 5:   # the only workload cheap enough for the per-token loop is skipped
        rows = plan["rows"]
        assert rows[:, 3].tolist() == [32768] * 4
        assert rows[:, 5].tolist() == [32768, 65536, 98304, 131072]
        return
    _check_plan_invariants(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size,
                           spec.num_shards, spec.split_mode, plan)


def test_plan_dual_chunk_workload2_has_32_rows():
    spec = W.workload_spec(2, split_mode=W.SPLIT_DUAL_CHUNK)
    bt, _ = W.block_tables(spec)
    plan = oracle.row_plan(spec.query_len, spec.num_computed, bt.numpy(), 16, 2, 1)
    assert plan["rows"].shape[0] == 32
    assert np.bincount(plan["rows"][:, 1]).tolist() == [16, 16]


def test_plan_rejects_missing_page():
    with pytest.raises(oracle.OracleError) as e:
        oracle.row_plan([5], [0], np.array([[3, -1, -1]], np.int32), 2, 1, 0)
    assert e.value.code == -2


# -------------------------------------------------------------- cache write

def test_cache_write_read_back_through_block_table():
    rng = np.random.default_rng(31)
    bs, Hkv, D = 4, 2, 8
    ql, nc = [6, 1, 9], [0, 5, 2]
    need = [-(-(p + n) // bs) for p, n in zip(nc, ql)]
    nb = sum(need) + 2
    pool = rng.permutation(nb)
    bt = np.full((3, max(need)), -1, np.int32)
    o = 0
    for r, k in enumerate(need):
        bt[r, :k] = pool[o:o + k]
        o += k
    plan = oracle.row_plan(ql, nc, bt, bs, 2, 0)
    T = sum(ql)
    src = rng.integers(0, 2 ** 16, size=(T, Hkv, D), dtype=np.uint16)
    sentinel = np.uint16(0x7BCD)
    cache = np.full((nb, bs, Hkv, D), sentinel, dtype=np.uint16)
    slot = plan["slot"].copy()
    slot[plan["owner"] == 1] = -1          # shard 0's PAD-masked view
    assert oracle.cache_write(src, slot, cache) == 0
    offs = np.concatenate([[0], np.cumsum(ql)])
    written = np.zeros((nb, bs), bool)
    for r in range(3):
        for j in range(ql[r]):
            t, pos = offs[r] + j, nc[r] + j
            b, off = bt[r][pos // bs], pos % bs
            if plan["owner"][t] == 0:
                np.testing.assert_array_equal(cache[b, off], src[t])
                written[b, off] = True
    assert np.all(cache[~written] == sentinel)
    # a slot past the end is reported
    bad = np.array([nb * bs], np.int64)
    assert oracle.cache_write(src[:1], bad, cache) == -2
