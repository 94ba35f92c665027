"""Pins of the oracle's FP8 (e4m3) KV-cache functions against things other
than itself (CPU only).

* the e4m3 code table against PyTorch's own ``float8_e4m3fn`` dtype (a library
  routine) for all 256 codes, and against the format's printed landmarks
  (largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9);
* rounding: PyTorch's float -> e4m3 conversion on random values inside the
  finite range, hand-worked ties (to even), the subnormal boundary, signed
  zero, and saturation at +-448 outside it (the saturating reading);
* the FP8 cache write read back through the block table;
* attention over codes with per-(request, kv-head) descales against a dense
  numpy softmax over the codes' values (decoded by PyTorch) times the
  descales, and the descales' algebra.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero is kept
    assert math.copysign(1.0, ours[0x80]) == -1.0 and math.copysign(1.0, ours[0x00]) == 1.0


def test_decode_landmarks():
    d = oracle.e4m3_decode(np.array([0x7E, 0xFE, 0x08, 0x01, 0x07, 0x38, 0x39, 0x3F], dtype=np.uint8))
    assert d[0] == 448.0 and d[1] == -448.0          # largest finite magnitude
    assert d[2] == 2.0 ** -6                          # smallest normal
    assert d[3] == 2.0 ** -9                          # smallest subnormal
    assert d[4] == 7 * 2.0 ** -9                      # largest subnormal
    assert d[5] == 1.0 and d[6] == 1.125 and d[7] == 1.875


def test_encode_matches_torch_inside_the_range():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 1e-2, 0.3, 3.0, 60.0)])
    x = np.concatenate([x, rng.uniform(-463.9, 463.9, 2000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),        # halfway 1.0 (even) / 1.125 -> 1.0
    (1.1875, 0x3A),        # halfway 1.125 / 1.25 (even) -> 1.25
    (-1.0625, 0xB8),
    (2.0 ** -10, 0x00),    # halfway 0 / 2^-9 -> +0
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 / 2^-8 (even) -> 2^-8
    (-(2.0 ** -11), 0x80),  # rounds to -0
    (0.0, 0x00),
    (-0.0, 0x80),
    (448.0, 0x7E),
    (463.9, 0x7E),
    (464.0, 0x7E),         # saturates (no infinity in e4m3)
    (1.0e6, 0x7E),
    (-1.0e6, 0xFE),
    (float("inf"), 0x7E),
])
def test_encode_hand_worked(x, code):
    assert oracle.e4m3_encode(x) == code


def test_encode_round_trips_every_finite_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = oracle.e4m3_decode(np.array([c], dtype=np.uint8))[0]
        assert oracle.e4m3_encode(v) == c


def test_cache_write_fp8_reads_back_through_the_block_table():
    rng = np.random.default_rng(5)
    T, H, D, bs, nb = 37, 2, 16, 4, 16
    src = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32) * 3).to(torch.bfloat16)
    slot = rng.permutation(nb * bs)[:T].astype(np.int64)
    slot[5] = -1                                     # PAD-masked token: skipped
    cache = np.full((nb, bs, H, D), 0x7F, dtype=np.uint8)
    scale = 0.37
    assert oracle.cache_write_fp8(src, slot, cache, scale) == 0
    flat = cache.reshape(nb * bs, H, D)
    x32 = src.to(torch.float32)
    q = (x32 / torch.tensor(scale, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t in range(T):
        if slot[t] < 0:
            continue
        assert np.array_equal(flat[slot[t]], q[t])
    untouched = np.ones(nb * bs, dtype=bool)
    untouched[slot[slot >= 0]] = False
    assert (flat[untouched] == 0x7F).all()
    # a slot past the end is reported
    bad = slot.copy()
    bad[0] = nb * bs
    assert oracle.cache_write_fp8(src, bad, cache, scale) == -2


def _dense(Q, K, V, lo, hi, pos, scale, G):
    """Dense softmax of one request's query rows over keys [lo, min(hi, pos + 1))."""
    n, Hq, D = Q.shape
    L = K.shape[0]
    out = np.zeros((n, Hq, D))
    lse = np.full((n, Hq), -np.inf)
    kpos = np.arange(L)[None, :]
    mask = (kpos >= lo) & (kpos < np.minimum(hi, pos[:, None] + 1))
    for h in range(Hq):
        s = scale * (Q[:, h, :] @ K[:, h // G, :].T)
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        ok = np.isfinite(m[:, 0])
        e = np.exp(s - np.where(np.isfinite(m), m, 0.0))
        z = e.sum(axis=1, keepdims=True)
        out[ok, h, :] = ((e / np.where(z > 0, z, 1.0)) @ V[:, h // G, :])[ok]
        lse[ok, h] = (m + np.log(np.where(z > 0, z, 1.0)))[ok, 0]
    return out, lse


def _torch_decode(codes: np.ndarray) -> np.ndarray:
    """e4m3 values through PyTorch's float8_e4m3fn (independent of the oracle)."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _random_codes(rng, shape):
    c = rng.integers(0, 0x7F, size=shape, dtype=np.uint8)          # 0 .. 126: finite magnitudes
    return c | (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_attention_fp8kv_matches_dense(G):
    """Two requests (one with a cached prefix), random codes and a different
    descale per (request, kv head): every token of every part (fused, context,
    new) against a dense softmax over the codes' values (decoded by PyTorch)
    times the descales."""
    rng = np.random.default_rng(40 + G)
    Hkv, D = 2, 8
    Hq = G * Hkv
    lens = [(9, 7), (0, 11)]
    ql = [n for _, n in lens]
    nc = [p for p, _ in lens]
    ck = [_random_codes(rng, (p + n, Hkv, D)) for p, n in lens]
    cv = [_random_codes(rng, (p + n, Hkv, D)) for p, n in lens]
    kd = rng.uniform(0.001, 0.02, size=(2, Hkv)).astype(np.float32)
    vd = rng.uniform(0.001, 0.02, size=(2, Hkv)).astype(np.float32)
    Lmax = max(p + n for p, n in lens)
    bt = np.stack([np.arange(Lmax, dtype=np.int32) + r * Lmax for r in range(2)])
    rows = oracle.row_plan(ql, nc, bt, 1, 2, 0)["rows"]
    q = torch.from_numpy(rng.standard_normal((sum(ql), Hq, D)).astype(np.float32)).to(torch.bfloat16)
    off = [0, lens[0][0] + lens[0][1]]
    K = [_torch_decode(c) * kd[r][None, :, None].astype(np.float64) for r, c in enumerate(ck)]
    V = [_torch_decode(c) * vd[r][None, :, None].astype(np.float64) for r, c in enumerate(cv)]
    tokens = np.arange(sum(ql))
    for part in ("fused", "context", "new"):
        lo, hi = oracle.key_ranges(rows, part)
        out, lse = oracle.attention_fp8kv(rows, q, np.concatenate(ck), np.concatenate(cv), off, kd, vd, Hq, Hkv, D,
                                          0.3, tokens, key_lo=lo, key_hi=hi)
        for ri, r in enumerate(rows):
            j = np.arange(r[3])
            t = r[2] + j
            pos = r[5] - r[3] + j
            ro, rl = _dense(q.to(torch.float64).numpy()[t], K[r[0]], V[r[0]], lo[ri], hi[ri], pos, 0.3, G)
            np.testing.assert_allclose(out[t], ro, rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[t], rl, rtol=0, atol=1e-12)


def test_descale_algebra():
    """A V descale of 2x doubles the output and leaves the LSE alone; a K
    descale of 2x equals a softmax scale of 2x (factors of two: exact in fp32)."""
    rng = np.random.default_rng(77)
    Hkv, G, D = 2, 2, 16
    Hq = G * Hkv
    n = 13
    ck = _random_codes(rng, (n, Hkv, D))
    cv = _random_codes(rng, (n, Hkv, D))
    kd = rng.uniform(0.001, 0.02, size=(1, Hkv)).astype(np.float32)
    vd = rng.uniform(0.001, 0.02, size=(1, Hkv)).astype(np.float32)
    rows = oracle.row_plan([n], [0], np.arange(n, dtype=np.int32)[None, :], 1, 1, 0)["rows"]
    q = torch.from_numpy(rng.standard_normal((n, Hq, D)).astype(np.float32)).to(torch.bfloat16)
    tok = np.arange(n)
    o1, l1 = oracle.attention_fp8kv(rows, q, ck, cv, [0], kd, vd, Hq, Hkv, D, 0.25, tok)
    o2, l2 = oracle.attention_fp8kv(rows, q, ck, cv, [0], kd, 2 * vd, Hq, Hkv, D, 0.25, tok)
    np.testing.assert_allclose(o2, 2 * o1, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(l2, l1)
    o3, l3 = oracle.attention_fp8kv(rows, q, ck, cv, [0], 2 * kd, vd, Hq, Hkv, D, 0.25, tok)
    o4, l4 = oracle.attention_fp8kv(rows, q, ck, cv, [0], kd, vd, Hq, Hkv, D, 0.5, tok)
    np.testing.assert_allclose(o3, o4, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l3, l4, rtol=0, atol=1e-12)


def test_finite_codes_increase_with_the_code():
    """The premise of the encoder's bisection: codes 0..126 are the
    non-negative finite values in increasing order (PyTorch's table)."""
    v = _torch_decode(np.arange(127, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)
