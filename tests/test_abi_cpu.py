"""The C-ABI library on the host (no GPU needed): it loads, exports every
function include/pcp.h declares, its host row plan matches the oracle bit for
bit, and invalid arguments are refused before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def P():
    from context_prefill_attention_gb300 import build
    build.build()
    import context_prefill_attention_gb300 as P
    P.load()
    return P


def _declared():
    with open(os.path.join(ROOT, "include", "pcp.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pcp_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(P):
    lib = P.load()
    names = _declared()
    assert "pcp_attn_varlen" in names and "pcp_build_row_plan" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(P.EXPORTS)


@pytest.mark.parametrize("seed", range(20))
def test_host_plan_matches_oracle_random(P, seed):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.integers(1, 12))
    S = int(rng.integers(1, 6))
    mode = int(rng.integers(0, 2))
    bs = int(rng.choice([1, 4, 16, 32]))
    ql = [int(rng.choice([0, 1, 1, 2, 5, 31, 128, 1000])) for _ in range(R)]
    nc = [int(rng.integers(0, 3000)) for _ in range(R)]
    need = [-(-(p + n) // bs) for p, n in zip(nc, ql)]
    pool = rng.permutation(sum(need) + 3)
    bt = np.full((R, max(1, max(need))), -1, dtype=np.int32)
    o = 0
    for r, k in enumerate(need):
        bt[r, :k] = pool[o:o + k]
        o += k
    a = P.pcp_build_row_plan(ql, nc, bt, bs, S, mode)
    b = oracle.row_plan(ql, nc, bt, bs, S, mode)
    np.testing.assert_array_equal(a["rows"], b["rows"])
    np.testing.assert_array_equal(a["cu_q"], b["cu_q"])
    np.testing.assert_array_equal(a["slot_mapping"], b["slot"])
    np.testing.assert_array_equal(a["owner_shard"], b["owner"])


@pytest.mark.parametrize("workload,mode", [(1, 0), (2, 0), (2, 1), (3, 0), (4, 0), (5, 0)])
def test_host_plan_matches_oracle_workloads(P, workload, mode):
    spec = W.workload_spec(workload, split_mode=mode)
    bt, _ = W.block_tables(spec)
    a = P.pcp_build_row_plan(spec.query_len, spec.num_computed, bt, spec.block_size, spec.num_shards, mode)
    b = oracle.row_plan(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size, spec.num_shards, mode)
    np.testing.assert_array_equal(a["rows"], b["rows"])
    np.testing.assert_array_equal(a["slot_mapping"], b["slot"])
    np.testing.assert_array_equal(a["owner_shard"], b["owner"])


def test_host_plan_errors(P):
    with pytest.raises(P.PcpError) as e:
        P.pcp_build_row_plan([5], [0], np.array([[1, -1, -1]], np.int32), 2, 1)
    assert e.value.code == P.PCP_ERR_RANGE
    with pytest.raises(P.PcpError) as e:
        P.pcp_build_row_plan([5, 5], [0, 0], np.array([[0, 1, 2], [3, 4, 5]], np.int32), 2, 2, rows_capacity=3)
    assert e.value.code == P.PCP_ERR_RANGE
    with pytest.raises(P.PcpError) as e:
        P.pcp_build_row_plan([5], [0], np.array([[0, 1, 2]], np.int32), 2, 0)
    assert e.value.code == P.PCP_ERR_ARG
    with pytest.raises(P.PcpError) as e:
        P.pcp_build_row_plan([-1], [0], np.array([[0]], np.int32), 2, 1)
    assert e.value.code == P.PCP_ERR_ARG


def test_mask_slots_for_shard(P):
    spec = W.custom_spec([10, 1, 7], [0, 5, 2], num_q_heads=2, num_kv_heads=1, head_dim=8, block_size=4,
                         num_shards=3)
    bt, _ = W.block_tables(spec)
    plan = P.pcp_build_row_plan(spec.query_len, spec.num_computed, bt, 4, 3)
    seen = np.zeros(spec.total_q, dtype=int)
    for s in range(3):
        m = P.pcp_mask_slots_for_shard(plan["slot_mapping"], plan["owner_shard"], s)
        own = plan["owner_shard"] == s
        np.testing.assert_array_equal(m[own], plan["slot_mapping"][own])
        assert np.all(m[~own] == -1)
        seen += own
    assert np.all(seen == 1)
    # the decode token (request 1) is written by shard 0 only
    assert plan["owner_shard"][10] == 0


FAKE = 0x10000  # a 256-byte aligned address that is never dereferenced


def _attn(lib, **kw):
    args = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, nreq=1, mb=4, nb=64, bs=16, rows=FAKE, nrows=2, T=100,
                hq=8, hkv=2, d=128, scale=0.1, out=FAKE, lse=FAKE, ws=FAKE, wsb=1 << 30, flags=0, status=None)
    args.update(kw)
    P_ = ctypes.c_void_p
    return lib.pcp_attn_varlen(P_(args["q"]), P_(args["kc"]), P_(args["vc"]), P_(args["bt"]), args["nreq"],
                               args["mb"], args["nb"], args["bs"], P_(args["rows"]), args["nrows"], args["T"],
                               args["hq"], args["hkv"], args["d"], args["scale"], P_(args["out"]), P_(args["lse"]),
                               P_(args["ws"]), args["wsb"], args["flags"], args["status"], None)


def test_attn_varlen_validates_before_launch(P):
    lib = P.load()
    assert _attn(lib, d=96) == P.PCP_ERR_UNSUPPORTED
    assert _attn(lib, hq=6, hkv=4) == P.PCP_ERR_UNSUPPORTED
    assert _attn(lib, bs=12) == P.PCP_ERR_UNSUPPORTED
    assert _attn(lib, hq=64, hkv=2) == P.PCP_ERR_UNSUPPORTED
    assert _attn(lib, q=None) == P.PCP_ERR_ARG
    assert _attn(lib, nrows=-1) == P.PCP_ERR_ARG
    assert _attn(lib, flags=8) == P.PCP_ERR_ARG
    assert _attn(lib, flags=P.PCP_ATTN_KV_SHARDS(1)) == P.PCP_ERR_ARG
    assert _attn(lib, flags=P.PCP_ATTN_KV_SHARDS(65)) == P.PCP_ERR_ARG
    assert _attn(lib, flags=P.PCP_ATTN_SEPARATE_CONTEXT | P.PCP_ATTN_KV_SHARDS(2)) == P.PCP_ERR_ARG
    assert _attn(lib, flags=1 << 24) == P.PCP_ERR_ARG
    assert _attn(lib, nrows=0, flags=P.PCP_ATTN_DECODE_SMS(18)) == P.PCP_OK
    assert P.pcp_attn_workspace_size(2, 100, 8, 128, 64, P.PCP_ATTN_DECODE_SMS(18)) == \
        P.pcp_attn_workspace_size(2, 100, 8, 128, 64, 0)
    assert P.pcp_attn_workspace_size(2, 100, 8, 128, 64, P.PCP_ATTN_KV_SHARDS(4)) > \
        P.pcp_attn_workspace_size(2, 100, 8, 128, 64, P.PCP_ATTN_KV_SHARDS(2))
    assert _attn(lib, q=FAKE + 8) == P.PCP_ERR_ALIGN
    assert _attn(lib, ws=FAKE + 16) == P.PCP_ERR_ALIGN
    assert _attn(lib, wsb=100) == P.PCP_ERR_WORKSPACE
    assert _attn(lib, nb=1 << 28) == P.PCP_ERR_ARG
    assert _attn(lib, nrows=0) == P.PCP_OK          # nothing to do, nothing launched
    need = P.pcp_attn_workspace_size(2, 100, 8, 128, 64, 0)
    assert need > 0 and P.pcp_attn_workspace_size(2, 100, 8, 128, 64, 1) > need
    assert P.pcp_attn_workspace_size(-1, 100, 8, 128, 64, 0) == 0


def test_cache_write_and_merge_validate_before_launch(P):
    lib = P.load()
    V = ctypes.c_void_p
    # every call below fails a host check, so nothing is launched on a fake pointer
    assert lib.pcp_kv_cache_write(V(FAKE + 4), V(FAKE), V(FAKE), 10, V(FAKE), V(FAKE), 8, 16, 2, 128, None,
                                  None) == P.PCP_ERR_ALIGN
    assert lib.pcp_kv_cache_write(None, V(FAKE), V(FAKE), 10, V(FAKE), V(FAKE), 8, 16, 2, 128, None,
                                  None) == P.PCP_ERR_ARG
    assert lib.pcp_kv_cache_write(V(FAKE), V(FAKE), V(FAKE), 10, V(FAKE), V(FAKE), 8, 16, 1, 3, None,
                                  None) == P.PCP_ERR_UNSUPPORTED
    assert lib.pcp_kv_cache_write(V(FAKE), V(FAKE), V(FAKE), 0, V(FAKE), V(FAKE), 8, 16, 2, 128, None,
                                  None) == P.PCP_OK
    assert lib.pcp_lse_merge(V(FAKE), V(FAKE), V(FAKE), V(FAKE), V(FAKE), V(FAKE), 4, 2, 12, None) \
        == P.PCP_ERR_UNSUPPORTED
    assert lib.pcp_lse_merge(V(FAKE), V(FAKE), V(FAKE), V(FAKE), V(FAKE), V(FAKE), 4, 2, 128, None) \
        == P.PCP_ERR_ARG   # lse aliases lse_a
    assert lib.pcp_lse_merge(V(FAKE + 4), V(FAKE), V(FAKE), V(FAKE + 512), V(FAKE), V(FAKE + 1024), 4, 2, 128,
                             None) == P.PCP_ERR_ALIGN
    assert lib.pcp_status_string(P.PCP_ERR_TIMEOUT) == b"device wait timed out"


def _attn_fp8(lib, kd=FAKE, vd=FAKE, **kw):
    args = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, nreq=1, mb=4, nb=64, bs=16, rows=FAKE, nrows=2, T=100,
                hq=8, hkv=2, d=128, scale=0.1, out=FAKE, lse=FAKE, ws=FAKE, wsb=1 << 30, flags=0, status=None)
    args.update(kw)
    P_ = ctypes.c_void_p
    return lib.pcp_attn_varlen_fp8kv(P_(args["q"]), P_(args["kc"]), P_(args["vc"]), P_(kd), P_(vd), P_(args["bt"]),
                                     args["nreq"], args["mb"], args["nb"], args["bs"], P_(args["rows"]), args["nrows"],
                                     args["T"], args["hq"], args["hkv"], args["d"], args["scale"], P_(args["out"]),
                                     P_(args["lse"]), P_(args["ws"]), args["wsb"], args["flags"], args["status"],
                                     None)


def test_fp8_entry_points_validate_before_launch(P):
    """Every call below fails a host check (or has nothing to do), so nothing
    is launched on a fake pointer."""
    lib = P.load()
    V = ctypes.c_void_p
    assert _attn_fp8(lib, kd=None) == P.PCP_ERR_ARG
    assert _attn_fp8(lib, vd=None) == P.PCP_ERR_ARG
    assert _attn_fp8(lib, kd=FAKE + 2) == P.PCP_ERR_ALIGN
    assert _attn_fp8(lib, vd=FAKE + 1) == P.PCP_ERR_ALIGN
    assert _attn_fp8(lib, d=96) == P.PCP_ERR_UNSUPPORTED
    assert _attn_fp8(lib, flags=8) == P.PCP_ERR_ARG
    assert _attn_fp8(lib, wsb=100) == P.PCP_ERR_WORKSPACE
    assert _attn_fp8(lib, nrows=0, kd=None, vd=None) == P.PCP_OK
    w = lib.pcp_kv_cache_write_fp8
    args = (V(FAKE), V(FAKE), V(FAKE), 10, V(FAKE), V(FAKE), 8, 16, 2, 128)
    for ks, vs in ((0.0, 1.0), (1.0, -2.0), (float("nan"), 1.0), (1.0, float("inf"))):
        assert w(*args, ks, vs, None, None) == P.PCP_ERR_ARG
    assert w(V(FAKE), V(FAKE), V(FAKE), 10, V(FAKE), V(FAKE), 8, 16, 1, 8, 1.0, 1.0, None, None) \
        == P.PCP_ERR_UNSUPPORTED      # Hkv * D = 8 is not a multiple of 16
    assert w(V(FAKE + 4), V(FAKE), V(FAKE), 10, V(FAKE), V(FAKE), 8, 16, 2, 128, 1.0, 1.0, None, None) \
        == P.PCP_ERR_ALIGN
    assert w(V(FAKE), V(FAKE), V(FAKE), 0, V(FAKE), V(FAKE), 8, 16, 2, 128, 1.0, 1.0, None, None) == P.PCP_OK


GiB = 1 << 30
BASE = 1 << 40          # distinct fake buffers, 1 GiB apart, never dereferenced


def _distinct(**kw):
    names = ["q", "kc", "vc", "bt", "rows", "out", "lse", "ws"]
    d = {n: BASE + i * GiB for i, n in enumerate(names)}
    d.update(kw)
    return d


def test_overlapping_outputs_and_non_finite_scale_are_refused(P):
    """Every call below fails a host check, so nothing is launched on a fake
    pointer. With distinct buffers a too-small workspace (the check just
    before the overlap checks) is what fails; moving one output onto an input
    turns that into PCP_ERR_ARG."""
    lib = P.load()
    V = ctypes.c_void_p
    assert _attn(lib, wsb=100, **_distinct()) == P.PCP_ERR_WORKSPACE
    for scale in (float("nan"), float("inf"), float("-inf")):
        assert _attn(lib, scale=scale, **_distinct()) == P.PCP_ERR_ARG
    out_bytes = 100 * 8 * 128 * 2
    for kw in (dict(out=BASE), dict(out=BASE + 3 * GiB - 256),          # onto q; across the block table
               dict(lse=BASE + 4 * GiB + 32), dict(out=BASE + 7 * GiB + 256),   # into rows; into the workspace
               dict(lse=BASE + 5 * GiB + out_bytes - 4), dict(kc=BASE + 6 * GiB)):  # out/lse; lse on a cache
        assert _attn(lib, **_distinct(**kw)) == P.PCP_ERR_ARG, kw
    # the FP8 descales are inputs too
    d = _distinct()
    assert _attn_fp8(lib, kd=d["out"] + 64, **{k: v for k, v in d.items()}) == P.PCP_ERR_ARG
    # cache write: the caches overlap neither each other nor k, v, slot_mapping
    tok = 10 * 2 * 128 * 2

    def write(k, v, slot, kc, vc):
        return lib.pcp_kv_cache_write(V(k), V(v), V(slot), 10, V(kc), V(vc), 8, 16, 2, 128, None, None)
    assert write(BASE, BASE + GiB, BASE + 2 * GiB, BASE + 3 * GiB, BASE + 3 * GiB) == P.PCP_ERR_ARG
    assert write(BASE, BASE + GiB, BASE + 2 * GiB, BASE + tok - 16, BASE + 4 * GiB) == P.PCP_ERR_ARG
    assert write(BASE, BASE + GiB, BASE + 2 * GiB, BASE + 3 * GiB, BASE + 2 * GiB + 64) == P.PCP_ERR_ARG
    w8 = lib.pcp_kv_cache_write_fp8
    assert w8(V(BASE), V(BASE + GiB), V(BASE + 2 * GiB), 10, V(BASE + 3 * GiB), V(BASE + 3 * GiB + 16), 8, 16, 2,
              128, 1.0, 1.0, None, None) == P.PCP_ERR_ARG
    # LSE merge: no in-place merge, no partial overlap of the lse arrays
    T, H, D = 4, 2, 128
    part, lse_b = T * H * D * 4, T * H * 4

    def merge(oa, la, ob, lb, o, l):
        return lib.pcp_lse_merge(V(oa), V(la), V(ob), V(lb), V(o), V(l), T, H, D, None)
    a = [BASE + i * GiB for i in range(6)]
    assert merge(a[0], a[1], a[2], a[3], a[0], a[5]) == P.PCP_ERR_ARG            # out onto out_a
    assert merge(a[0], a[1], a[2], a[3], a[2] + part - 16, a[5]) == P.PCP_ERR_ARG  # out runs into out_b
    assert merge(a[0], a[1], a[2], a[3], a[4], a[1] + 4) == P.PCP_ERR_ARG         # lse shifted onto lse_a
    assert merge(a[0], a[1], a[2], a[3], a[4], a[4] + part // 2 - lse_b // 2) == P.PCP_ERR_ARG  # out / lse


def test_debug_plan_summary(P, monkeypatch, capsys):
    """PCP_DEBUG=1 prints the plan summary (rows and tokens per shard, decode
    rows, PAD slots) to stderr; without it nothing is printed."""
    bt = np.arange(200, dtype=np.int32).reshape(4, 50)
    plan = P.pcp_build_row_plan([300, 1, 77, 0], [0, 500, 13, 4], bt, 16, 2)
    text = P.plan_summary(plan, 2)
    assert "5 rows (4 prefill, 1 decode), 378 tokens, 2 shards" in text
    assert "shard 0: 3 rows, 189 tokens" in text and "shard 1: 2 rows, 189 tokens" in text
    assert "378 (0 PAD)" in text
    masked = dict(plan, slot_mapping=P.pcp_mask_slots_for_shard(plan["slot_mapping"], plan["owner_shard"], 1))
    assert "378 (189 PAD)" in P.plan_summary(masked, 2)
    monkeypatch.delenv("PCP_DEBUG", raising=False)
    P.debug_plan(plan, 2)
    assert capsys.readouterr().err == ""
    monkeypatch.setenv("PCP_DEBUG", "1")
    P.debug_plan(plan, 2)
    assert capsys.readouterr().err.strip() == text


def test_binding_refuses_host_and_malformed_tensors(P):
    """The binding checks every tensor before its pointer crosses the ABI: a
    host tensor (which the kernels would read as a device address), a wrong
    dtype, a non-contiguous view or a wrong shape raises, and nothing is
    called. (CUDA tensors are not available here: each check is reached with
    host tensors, the device check last.)"""
    import torch
    from context_prefill_attention_gb300 import _lib as L
    q = torch.zeros((10, 4, 128), dtype=torch.bfloat16)
    kc = torch.zeros((2, 16, 2, 128), dtype=torch.bfloat16)
    bt = torch.zeros((1, 2), dtype=torch.int32)
    rows = torch.zeros((1, 8), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        P.pcp_attn_varlen(q, kc, kc, bt, rows, 0.1)
    with pytest.raises(TypeError, match="dtype"):
        P.pcp_attn_varlen(q.float(), kc, kc, bt, rows, 0.1)
    with pytest.raises(ValueError, match="contiguous"):
        P.pcp_attn_varlen(q.transpose(0, 1), kc, kc, bt, rows, 0.1)
    with pytest.raises(ValueError, match="shape"):
        P.pcp_attn_varlen(q[0], kc, kc, bt, rows, 0.1)
    with pytest.raises(ValueError, match="CUDA"):
        P.pcp_attn_varlen_fp8kv(q, kc.view(torch.uint8)[..., :128], kc, None, None, bt, rows, 0.1)
    with pytest.raises(ValueError, match="CUDA"):
        P.pcp_attn_varlen_noalloc(q, kc, kc, bt, rows, 0.1, q, torch.zeros((4, 10)))
    k = torch.zeros((5, 2, 128), dtype=torch.bfloat16)
    slot = torch.zeros(5, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA"):
        P.pcp_kv_cache_write(k, k, slot, kc, kc.clone())
    with pytest.raises(TypeError, match="dtype"):
        P.pcp_kv_cache_write_fp8(k, k, slot, kc, kc.clone(), 1.0, 1.0)      # a bf16 cache for the FP8 writer
    with pytest.raises(ValueError, match="CUDA"):
        P.pcp_lse_merge(torch.zeros((10, 4, 128)), torch.zeros((4, 10)), torch.zeros((10, 4, 128)),
                        torch.zeros((4, 10)))
    with pytest.raises(TypeError, match="torch.Tensor"):
        P.pcp_lse_merge(np.zeros((10, 4, 128), np.float32), None, None, None)
    # the shape rule: exact sizes, -1 free, the rank must match
    t = torch.zeros((3, 8))
    for shape in ((3, 9), (3,), (3, 8, 1), (-1, 7)):
        with pytest.raises(ValueError, match="shape"):
            L._dev(t, "t", shape=shape)
    with pytest.raises(ValueError, match="CUDA"):
        L._dev(t, "t", (torch.float32,), shape=(-1, 8))          # every other check passes


class _FakeLib:
    """Stands in for libpcp: records each call's arguments and returns PCP_OK
    (so the binding's marshalling runs to the end with nothing launched)."""

    def __init__(self, real):
        self.calls = {}
        self.real = real

    def pcp_attn_workspace_size(self, *a):
        return self.real.pcp_attn_workspace_size(*a)

    def pcp_status_string(self, code):
        return self.real.pcp_status_string(code)

    def pcp_last_cuda_error(self):
        return 0

    def __getattr__(self, name):
        def f(*args):
            self.calls[name] = args
            return 0
        return f


def test_binding_marshals_consistent_tensors_and_checks_every_argument(P, monkeypatch):
    """Host tensors stand in for device ones (the device test is switched off
    and the library replaced by a recorder, so nothing reaches a kernel): the
    wrappers accept consistent arguments, pass the right sizes across the ABI,
    and refuse each inconsistent one."""
    import torch
    from context_prefill_attention_gb300 import _lib as L
    fake = _FakeLib(L.load())
    monkeypatch.setattr(L, "_lib", fake)
    monkeypatch.setattr(L, "_is_device_tensor", lambda t: True)
    T, hq, hkv, D, nb, bs, R, mb, n = 10, 8, 2, 128, 6, 16, 3, 2, 4
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q = torch.zeros((T, hq, D), dtype=bf)
    kc, vc = torch.zeros((nb, bs, hkv, D), dtype=bf), torch.zeros((nb, bs, hkv, D), dtype=bf)
    bt = torch.zeros((R, mb), dtype=i32)
    rows = torch.zeros((n, 8), dtype=i32)
    out, lse = torch.zeros((T, hq, D), dtype=bf), torch.zeros((hq, T), dtype=f32)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    st = torch.zeros(1, dtype=i32)
    P.pcp_attn_varlen(q, kc, vc, bt, rows, 0.1, out=out, lse=lse, workspace=ws, flags=1, status=st, stream=0)
    a = fake.calls["pcp_attn_varlen"]
    assert a[4:14] == (R, mb, nb, bs) + a[8:9] + (n, T, hq, hkv, D) and a[18] == ws.numel() and a[19] == 1
    bad = [dict(out=torch.zeros((T, hq, 64), dtype=bf)), dict(lse=torch.zeros((T, hq), dtype=f32)),
           dict(lse=torch.zeros((hq, T), dtype=bf)), dict(status=torch.zeros(1, dtype=torch.int64)),
           dict(status=torch.zeros(0, dtype=i32))]
    for kw in bad:
        args = dict(out=out, lse=lse, workspace=ws, status=st, stream=0)
        args.update(kw)
        with pytest.raises((TypeError, ValueError)):
            P.pcp_attn_varlen(q, kc, vc, bt, rows, 0.1, **args)
    for k2, v2, b2, r2 in ((kc, vc[:, :8], bt, rows), (kc[..., :64].contiguous(), vc, bt, rows),
                           (kc, vc, bt.long(), rows), (kc, vc, bt, rows[:, :7].contiguous()),
                           (kc.view(torch.uint8)[..., :D].contiguous(), vc, bt, rows)):
        with pytest.raises((TypeError, ValueError)):
            P.pcp_attn_varlen(q, k2, v2, b2, r2, 0.1, stream=0)
    # FP8 cache: uint8 codes and fp32 descales [R, Hkv]
    kc8, vc8 = torch.zeros((nb, bs, hkv, D), dtype=torch.uint8), torch.zeros((nb, bs, hkv, D), dtype=torch.uint8)
    kd, vd = torch.ones((R, hkv)), torch.ones((R, hkv))
    P.pcp_attn_varlen_fp8kv(q, kc8, vc8, kd, vd, bt, rows, 0.1, stream=0)
    a = fake.calls["pcp_attn_varlen_fp8kv"]
    assert a[6:16] == (R, mb, nb, bs) + a[10:11] + (n, T, hq, hkv, D)
    for kd2, vd2, c2 in ((kd[:2], vd, kc8), (kd, vd.double(), kc8), (kd, vd, kc)):
        with pytest.raises((TypeError, ValueError)):
            P.pcp_attn_varlen_fp8kv(q, c2, vc8, kd2, vd2, bt, rows, 0.1, stream=0)
    # no-allocation entry point: out and lse required
    P.pcp_attn_varlen_noalloc(q, kc, vc, bt, rows, 0.1, out, lse, stream=0)
    assert fake.calls["pcp_attn_varlen_noalloc"][4:6] == (R, mb)
    with pytest.raises(ValueError):
        P.pcp_attn_varlen_noalloc(q, kc, vc, bt, rows, 0.1, None, lse, stream=0)
    # cache writes
    k, v = torch.zeros((T, hkv, D), dtype=bf), torch.zeros((T, hkv, D), dtype=bf)
    slot = torch.zeros(T, dtype=torch.int64)
    P.pcp_kv_cache_write(k, v, slot, kc, vc, status=st, stream=0)
    assert fake.calls["pcp_kv_cache_write"][3:4] + fake.calls["pcp_kv_cache_write"][6:10] == (T, nb, bs, hkv, D)
    P.pcp_kv_cache_write_fp8(k, v, slot, kc8, vc8, 0.5, 0.25, stream=0)
    assert fake.calls["pcp_kv_cache_write_fp8"][10:12] == (0.5, 0.25)
    for k2, v2, s2 in ((k[:, :1].contiguous(), v, slot), (k, v[:5], slot), (k, v, slot[:5]), (k, v, slot.int()),
                       (k.float(), v, slot)):
        with pytest.raises((TypeError, ValueError)):
            P.pcp_kv_cache_write(k2, v2, s2, kc, vc, stream=0)
    # LSE merge
    oa, ob = torch.zeros((T, hq, D)), torch.zeros((T, hq, D))
    la, lb = torch.zeros((hq, T)), torch.zeros((hq, T))
    o, l_ = P.pcp_lse_merge(oa, la, ob, lb, stream=0)
    assert o.dtype == bf and o.shape == (T, hq, D) and l_.shape == (hq, T)
    assert fake.calls["pcp_lse_merge"][6:9] == (T, hq, D)
    for args in ((oa, la, ob[:5], lb), (oa, la.t(), ob, lb), (oa, la, ob, lb.double()), (oa.bfloat16(), la, ob, lb)):
        with pytest.raises((TypeError, ValueError)):
            P.pcp_lse_merge(*args, stream=0)


def _plan_rows(P, spec):
    bt, _ = W.block_tables(spec)
    return P.pcp_build_row_plan(spec.query_len, spec.num_computed, bt, spec.block_size, spec.num_shards,
                                spec.split_mode)["rows"]


def test_decode_sms_on_the_mixed_workload(P):
    """The mixed benchmark batch (8 prompts + 56 decode rows, 32 q / 8 kv heads)
    on 152 SMs: measured on GB300, 18 decode SMs gave the shortest step (20:
    1 % longer, 16: 12 % longer); the function may round up, not down."""
    rows = _plan_rows(P, W.workload_spec(4))
    k = P.pcp_decode_sms(rows, 32, 8, 128, False, 152)
    assert 18 <= k <= 20, k


def test_decode_sms_hand_worked():
    """One prefill row of 128 tokens without context (one 128-key tile, 4 two-head
    items at 8 q / 2 kv heads: 4 x (3.65 + 1.68) us = 21.32 us of SM time) and one
    decode row of 256 keys (256 x 2 kv heads x 128 dims x 2 bytes x 2 (K, V) =
    262144 bytes at 78.6 GB/s = 3.335 us, plus 2 items x 1 us = 5.335 us).
    Decode side rounded up by 5 %: 5.602 us; ceil(152 x 5.602 / 26.92) = 32."""
    import context_prefill_attention_gb300 as P
    P.load()
    rows = np.array([[0, 0, 0, 128, 0, 128, 0, 0],
                     [1, 0, 128, 1, 255, 256, 0, 1]], dtype=np.int32)
    assert P.pcp_decode_sms(rows, 8, 2, 128, False, 152) == 32


def test_decode_sms_zero_cases(P):
    """0 (decode rows in sequence) whenever the split does not apply."""
    mixed = _plan_rows(P, W.workload_spec(4))
    assert P.pcp_decode_sms(_plan_rows(P, W.workload_spec(2)), 16, 8, 128, False, 152) == 0  # no decode rows
    decode_only = mixed[mixed[:, 7] == 1]
    assert len(decode_only) == 56 and P.pcp_decode_sms(decode_only, 32, 8, 128, False, 152) == 0
    assert P.pcp_decode_sms(mixed, 32, 8, 128, True, 152) == 0     # FP8 cache
    assert P.pcp_decode_sms(mixed, 32, 8, 64, False, 152) == 0     # head_dim 64: CUDA-core decode
    assert P.pcp_decode_sms(mixed, 32, 1, 128, False, 152) == 0    # 32 q heads per kv head
    assert P.pcp_decode_sms(mixed, 32, 8, 128, False, 1) == 0
    assert P.pcp_decode_sms(mixed[:0], 32, 8, 128, False, 152) == 0
    many = np.concatenate([mixed] * 20)                              # more rows than the kernel takes
    assert len(many) > 1024 and P.pcp_decode_sms(many, 32, 8, 128, False, 152) == 0
    # decode-heavy: one short prompt beside the 56 long decode rows needs half the SMs or more
    short = np.concatenate([decode_only, [[0, 0, 0, 16, 0, 16, 0, 0]]]).astype(np.int32)
    assert P.pcp_decode_sms(short, 32, 8, 128, False, 152) == 0


def test_decode_sms_grows_with_decode_work(P):
    mixed = _plan_rows(P, W.workload_spec(4))
    prefill, decode = mixed[mixed[:, 7] == 0], mixed[mixed[:, 7] == 1]
    ks = [P.pcp_decode_sms(np.concatenate([prefill, decode[:n]]), 32, 8, 128, False, 152) for n in (4, 14, 28, 56)]
    assert all(a <= b for a, b in zip(ks, ks[1:])) and ks[0] >= 1 and ks[-1] > ks[0], ks
