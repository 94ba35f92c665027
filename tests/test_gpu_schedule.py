"""The prefill work list for long lists: more than 4096 work units.

The scheduler sorts up to 4096 units exactly in shared memory and longer lists
by a counting sort over cost classes. These tests run batches on both sides of
that limit through the C ABI, compare the attention with the oracle, and read
back from the workspace the unit count and the sorted unit list that the
scheduler wrote. The list must hold every expected unit exactly once, and its
costs (key tiles walked) must not increase along the list.
"""
import zlib

import numpy as np
import pytest
import torch

import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case

pytestmark = pytest.mark.gpu

BLOCK_M = BLOCK_N = 128
SORT_CAP = 4096
COST_CLASSES = 8192


def _P():
    import context_prefill_attention_gb300 as P
    P.load()
    return P


def _align256(x: int) -> int:
    return (x + 255) & ~255


def _nparts(flags: int) -> int:
    """Partial passes per row: n key shards, 2 for separate context, 0 fused."""
    shards = (flags >> 8) & 0xFF
    return shards if shards else (2 if flags & 1 else 0)


def _passes(flags: int) -> int:
    return max(1, _nparts(flags))


def _key_range(row, flags: int, p: int):
    kv_end, ctx, ql = int(row[5]), int(row[4]), int(row[3])
    shards = (flags >> 8) & 0xFF
    if shards:
        return kv_end * (p - 1) // shards, kv_end * p // shards
    if flags & 1:
        split = kv_end - ql if flags & 2 else ctx
        return (0, split) if p == 1 else (split, kv_end)
    return 0, kv_end


def _cost(row, mt: int, k_lo: int, k_hi: int, bs: int) -> int:
    """Key tiles walked by the item of tile mt of a row over keys [k_lo, k_hi)."""
    ql, kv_end = int(row[3]), int(row[5])
    pos0 = kv_end - ql + mt * BLOCK_M
    rv = min(BLOCK_M, ql - mt * BLOCK_M)
    k_end = min(k_hi, pos0 + rv)
    if k_end <= k_lo:
        return 0
    kb = (k_lo // bs) * bs
    return (k_end - kb + BLOCK_N - 1) // BLOCK_N


def expected_units(rows: np.ndarray, flags: int, bs: int):
    passes, nparts = _passes(flags), _nparts(flags)
    out = []
    for ri, row in enumerate(rows):
        if int(row[7]):
            continue
        for mt in range(-(-int(row[3]) // BLOCK_M)):
            for i in range(passes):
                p = i + 1 if nparts else 0
                lo, hi = _key_range(row, flags, max(p, 1))
                out.append((ri, mt | (p << 24), lo, hi))
    return out


DECODE_CHUNK = 2048


def read_schedule(case: Case):
    """Unit count and sorted units from the workspace of the last call. The
    offsets follow pcp_attn_varlen's workspace layout: a 64-entry int32 header
    (the unit count first), the row flags, the decode-item layout (2 num_rows + 1
    int32), the unsorted units, then the sorted units (16 bytes each), every
    part 256-byte aligned."""
    spec, flags = case.spec, case.flags
    n_rows = int(case.plan["rows"].shape[0])
    max_units = _passes(flags) * (-(-spec.total_q // BLOCK_M) + n_rows)
    off_units = 256 + _align256(n_rows * 4) + _align256((2 * n_rows + 1) * 4)
    off_sorted = off_units + _align256(max_units * 16)
    ws = case.step.workspace[:off_sorted + max_units * 16].cpu().numpy()
    n = int(ws[:4].view(np.int32)[0])
    units = ws[off_sorted:off_sorted + 16 * n].view(np.int32).reshape(n, 4)
    return n, units


def read_decode_items(case: Case):
    """header[1], the full-split prefix (num_rows + 1 int32) and the list of rows
    with a partial last split, as the last call left them."""
    n_rows = int(case.plan["rows"].shape[0])
    off = 256 + _align256(n_rows * 4)
    ws = case.step.workspace[:off + (2 * n_rows + 1) * 4].cpu().numpy()
    region = ws[off:off + (2 * n_rows + 1) * 4].view(np.int32).copy()
    return int(ws[4:8].view(np.int32)[0]), region[:n_rows + 1], region[n_rows + 1:]


def expected_full_prefix(rows: np.ndarray, num_kv_heads: int) -> np.ndarray:
    """Full-split items of the rows before each row: kv heads x whole 2048-key
    splits of every decode row, none for prefill rows."""
    cnt = [num_kv_heads * (int(r[5]) // DECODE_CHUNK) if int(r[7]) else 0 for r in rows]
    return np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)


def check_decode_items(case: Case) -> int:
    """The decode work list: the full splits' prefix, then every decode row with
    a partial last split exactly once, in non-increasing order of that split's
    128-key tiles; header[1] counts kv heads x (full splits + partial splits)."""
    rows = case.plan["rows"]
    hkv = case.spec.num_kv_heads
    total, pre, tail_area = read_decode_items(case)
    np.testing.assert_array_equal(pre, expected_full_prefix(rows, hkv))
    tail_rows = [i for i, r in enumerate(rows) if int(r[7]) and int(r[5]) % DECODE_CHUNK]
    listed = [int(x) for x in tail_area[:len(tail_rows)]]
    assert sorted(listed) == tail_rows, "every row with a partial split once"
    tiles = [-(-(int(rows[i][5]) % DECODE_CHUNK) // 128) for i in listed]
    assert all(x >= y for x, y in zip(tiles, tiles[1:])), "partial splits longest first"
    assert total == int(pre[-1]) + hkv * len(tail_rows)
    return total


def check_schedule(case: Case):
    rows = case.plan["rows"]
    bs = case.spec.block_size
    want = expected_units(rows, case.flags, bs)
    n, units = read_schedule(case)
    assert n == len(want)
    got = [tuple(int(x) for x in u) for u in units]
    assert sorted(got) == sorted(want), "the sorted list is not a permutation of the units"
    costs = [_cost(rows[u[0]], u[1] & 0xFFFFFF, u[2], u[3], bs) for u in got]
    if n > SORT_CAP:
        costs = [min(c, COST_CLASSES - 1) for c in costs]
    assert all(a >= b for a, b in zip(costs, costs[1:])), "costs rise along the list"
    return n


def _run(spec, flags, tokens=None):
    case = Case(spec, flags=flags)
    out, lse = case.run()
    eo, el = case.compare(out, lse, tokens)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    return case


def test_bitonic_path_order_and_parity():
    """A list under the limit: exact longest-first order. The decode rows'
    work list is checked too."""
    spec = W.custom_spec([3, 64, 129, 1, 17, 256, 2, 90, 1, 500], [0, 5, 0, 44, 130, 0, 1, 7, 300, 0],
                         num_q_heads=8, num_kv_heads=4, head_dim=128, seed=31)
    case = _run(spec, 0)
    assert 0 < check_schedule(case) <= SORT_CAP
    assert check_decode_items(case) > 0


def test_decode_items_full_splits_then_partials_longest_first():
    """Decode rows whose keys (cached context + the new token) end on, before
    and after split boundaries (2048 keys: one full split, no partial; 2049: a
    one-key partial; 6000: two full splits and a 1904-key partial; ...), beside
    a prefill row: the work list holds the full splits first and the partial
    ones longest first, and the result matches the oracle."""
    keys = [2048, 2049, 2047, 6000, 2, 130, 4096, 5000, 128, 4200]
    spec = W.custom_spec([1] * len(keys) + [70], [k - 1 for k in keys] + [300], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, seed=47)
    case = _run(spec, 0)
    rows = case.plan["rows"]
    n_partial = sum(1 for r in rows if int(r[7]) and int(r[5]) % DECODE_CHUNK)
    assert n_partial == 8
    assert check_decode_items(case) == 2 * (int(sum(int(r[5]) // DECODE_CHUNK for r in rows if int(r[7]))) +
                                            n_partial)


def test_kv_shards_64_over_limit():
    """64 key shards per row: 76 query tiles x 64 passes = 4864 units."""
    P = _P()
    spec = W.custom_spec([4000, 3000, 2500, 1], [0, 700, 0, 3000], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, seed=zlib.crc32(b"kv64") % 100000)
    case = _run(spec, P.PCP_ATTN_KV_SHARDS(64))
    assert check_schedule(case) > SORT_CAP


def test_many_short_rows_over_limit():
    """2100 requests of 2 to 4 new tokens in 2 shards: over 4096 one-tile rows in
    one fused call."""
    g = np.random.default_rng(2100)
    ql = g.integers(2, 5, size=2100).tolist()
    pre = g.integers(0, 41, size=2100).tolist()
    spec = W.custom_spec(ql, pre, num_q_heads=4, num_kv_heads=2, head_dim=64, seed=2100)
    case = _run(spec, 0)
    assert check_schedule(case) > SORT_CAP


def test_workload5_kv_shards_5_over_limit():
    """The 131072-token prompt in 4 shard rows with 5 key shards each: 5120 units,
    a valid batch that reaches the counting sort. Compared on a seeded sample of
    each row's tokens (plus its first and last)."""
    P = _P()
    spec = W.workload_spec(5)
    case = Case(spec, flags=P.PCP_ATTN_KV_SHARDS(5))
    out, lse = case.run()
    segs = [(int(r[2]), int(r[3])) for r in case.plan["rows"]]
    tokens = W.sample_segments(segs, 24, spec.seed + 21).numpy()
    eo, el = case.compare(out, lse, tokens)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert check_schedule(case) > SORT_CAP
    del case
    torch.cuda.empty_cache()
