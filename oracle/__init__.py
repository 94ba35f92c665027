"""CPU oracle for PCP attention — TEST INFRASTRUCTURE, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It wraps ``oracle.c`` (plain fp64 C,
OpenMP over query tokens) through ctypes and shares no code with the CUDA
library: the two meet only in the seeded inputs of ``workloads.py``.

What each function follows is stated in ``oracle.c``. Every function is pinned
by the CPU tests in ``tests/test_oracle_pins.py`` (dense brute force, closed
forms, shard/merge invariants and the golden fixtures in ``tests/golden/``) and
``tests/test_oracle_fp8_pins.py`` (the e4m3 codec against PyTorch's
``float8_e4m3fn`` and hand-worked cases, FP8-cache attention against a dense
softmax); no function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

ROW_FIELDS = ("req", "shard", "q_start", "q_len", "ctx_len", "kv_end", "causal_off", "is_decode")


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, fp64, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_row_plan.argtypes = [i32, P, P, P, i32, i32, i32, i32, P, i32, P, P, P, P]
        lib.oracle_row_plan.restype = i32
        lib.oracle_cache_write.argtypes = [P, P, i64, P, i64, i32]
        lib.oracle_cache_write.restype = i32
        lib.oracle_attention.argtypes = [i32, P, P, P, P, P, P, P, i32, i32, i32, dbl, P, i64, P, P]
        lib.oracle_attention.restype = i32
        lib.oracle_lse_merge.argtypes = [P, P, P, P, i64, i32, P, P]
        lib.oracle_lse_merge.restype = None
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = dbl
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode_array.argtypes = [P, i64, P]
        lib.oracle_e4m3_decode_array.restype = None
        lib.oracle_cache_write_fp8.argtypes = [P, P, i64, P, i64, i32, ctypes.c_float]
        lib.oracle_cache_write_fp8.restype = i32
        lib.oracle_attention_fp8kv.argtypes = [i32, P, P, P, P, P, P, P, P, P, i32, i32, i32, dbl, P, i64, P, P]
        lib.oracle_attention_fp8kv.restype = i32
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 numpy array."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint16))


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} returned {code}")
        self.code = code


def row_plan(query_len: Sequence[int], num_computed: Sequence[int], block_table, block_size: int,
             num_shards: int, split_mode: int, rows_cap: Optional[int] = None):
    """Row plan and slot mapping (see ``oracle_row_plan`` in oracle.c).

    Returns ``dict(rows=int32[n, 8], cu_q=int32[n+1], slot=int64[T], owner=int8[T])``.
    Raises ``OracleError`` with the C status on failure.
    """
    lib = _load()
    ql = np.ascontiguousarray(np.asarray(query_len, dtype=np.int32))
    nc = np.ascontiguousarray(np.asarray(num_computed, dtype=np.int32))
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    R = int(ql.shape[0])
    max_blocks = int(bt.shape[1]) if bt.ndim == 2 else 0
    T = int(ql.sum())
    cap = rows_cap if rows_cap is not None else max(1, 2 * num_shards * R)
    rows = np.zeros((max(cap, 1), 8), dtype=np.int32)
    cu = np.zeros(max(cap, 1) + 1, dtype=np.int32)
    slot = np.full(max(T, 1), -7, dtype=np.int64)
    owner = np.full(max(T, 1), -7, dtype=np.int8)
    n = np.zeros(1, dtype=np.int32)
    rc = lib.oracle_row_plan(R, _ptr(ql), _ptr(nc), _ptr(bt), max_blocks, block_size, num_shards,
                             split_mode, _ptr(rows), cap, _ptr(n), _ptr(cu), _ptr(slot), _ptr(owner))
    if rc != 0:
        raise OracleError(rc, "oracle_row_plan")
    k = int(n[0])
    return dict(rows=rows[:k].copy(), cu_q=cu[:k + 1].copy(), slot=slot[:T].copy(), owner=owner[:T].copy())


def cache_write(src, slot, cache: np.ndarray) -> int:
    """Scatter ``src[t]`` to ``cache[slot[t]]`` for ``slot[t] >= 0`` (in place).

    ``src`` is ``[T, H, D]`` bf16 (torch) or uint16; ``cache`` is a uint16 numpy
    array ``[num_blocks, bs, H, D]``. Returns the C status (0, or -2 when a slot
    is past the end)."""
    lib = _load()
    s = _u16(src)
    sl = np.ascontiguousarray(np.asarray(slot, dtype=np.int64))
    assert cache.dtype == np.uint16 and cache.flags.c_contiguous
    row = int(np.prod(s.shape[1:])) if s.ndim > 1 else 1
    num_slots = cache.size // row
    return int(lib.oracle_cache_write(_ptr(s), _ptr(sl), int(sl.shape[0]), _ptr(cache), num_slots, row))


def key_ranges(rows: np.ndarray, part: str = "fused"):
    """Key range each row attends, per pass.

    ``fused``   [0, kv_end): the whole causal result;
    ``context`` [0, ctx_len): the non-causal pass over the cached prefix;
    ``new``     [ctx_len, kv_end): the causal pass over the new tokens
                (the "before" split of "Carry the row plan ...", "What made it removable");
    ``before_row`` [0, kv_end - q_len) and ``own`` [kv_end - q_len, kv_end): the
                "now" split of the same section (context up to the row start, then the
                row's own tokens).
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 8)
    kv_end, ctx, ql = rows[:, 5], rows[:, 4], rows[:, 3]
    zero = np.zeros_like(kv_end)
    if part == "fused":
        lo, hi = zero, kv_end
    elif part == "context":
        lo, hi = zero, ctx
    elif part == "new":
        lo, hi = ctx, kv_end
    elif part == "before_row":
        lo, hi = zero, kv_end - ql
    elif part == "own":
        lo, hi = kv_end - ql, kv_end
    else:
        raise ValueError(part)
    return np.ascontiguousarray(lo, dtype=np.int64), np.ascontiguousarray(hi, dtype=np.int64)


def attention(rows, q, kv_k, kv_v, kv_off, num_q_heads: int, num_kv_heads: int, head_dim: int,
              scale: float, tokens, key_lo=None, key_hi=None, part: str = "fused"):
    """fp64 attention of the packed tokens ``tokens`` (see ``oracle_attention``).

    ``q`` is ``[T, Hq, D]`` bf16; ``kv_k``/``kv_v`` hold every request's
    contiguous keys back to back (request r from token ``kv_off[r]``).
    Returns ``(out float64[n, Hq, D], lse float64[n, Hq])``.
    """
    lib = _load()
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 8))
    if key_lo is None or key_hi is None:
        key_lo, key_hi = key_ranges(rows, part)
    key_lo = np.ascontiguousarray(np.asarray(key_lo, dtype=np.int64))
    key_hi = np.ascontiguousarray(np.asarray(key_hi, dtype=np.int64))
    qa, ka, va = _u16(q), _u16(kv_k), _u16(kv_v)
    off = np.ascontiguousarray(np.asarray(kv_off, dtype=np.int64))
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = int(tok.shape[0])
    out = np.zeros((max(n, 1), num_q_heads, head_dim), dtype=np.float64)
    lse = np.zeros((max(n, 1), num_q_heads), dtype=np.float64)
    rc = lib.oracle_attention(int(rows.shape[0]), _ptr(rows), _ptr(key_lo), _ptr(key_hi), _ptr(qa),
                              _ptr(ka), _ptr(va), _ptr(off), num_q_heads, num_kv_heads, head_dim,
                              float(scale), _ptr(tok), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise OracleError(rc, "oracle_attention")
    return out[:n], lse[:n]


def lse_merge(out_a, lse_a, out_b, lse_b):
    """Log-sum-exp merge of two partials (see ``oracle_lse_merge``).

    ``out_*`` has shape ``[..., D]`` and ``lse_*`` the leading shape ``[...]``.
    """
    lib = _load()
    oa = np.ascontiguousarray(out_a, dtype=np.float64)
    ob = np.ascontiguousarray(out_b, dtype=np.float64)
    la = np.ascontiguousarray(lse_a, dtype=np.float64)
    lb = np.ascontiguousarray(lse_b, dtype=np.float64)
    D = oa.shape[-1]
    n = la.size
    out = np.zeros(oa.shape, dtype=np.float64)
    lse = np.zeros(la.shape, dtype=np.float64)
    lib.oracle_lse_merge(_ptr(oa), _ptr(la), _ptr(ob), _ptr(lb), n, D, _ptr(out), _ptr(lse))
    return out, lse


def e4m3_decode(codes) -> np.ndarray:
    """Values of e4m3 codes (uint8 array, any shape) as float64; NaN codes give NaN."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(c.shape, dtype=np.float64)
    lib.oracle_e4m3_decode_array(_ptr(c), int(c.size), _ptr(out))
    return out


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code of a float32 (ties to even, saturating at 448)."""
    return int(_load().oracle_e4m3_encode(float(x)))


def cache_write_fp8(src, slot, cache: np.ndarray, scale: float) -> int:
    """FP8 cache write (see ``oracle_cache_write_fp8``): ``cache[slot[t]] =
    e4m3(src[t] / scale)`` for ``slot[t] >= 0``, in place. ``cache`` is a uint8
    numpy array ``[num_blocks, bs, H, D]``. Returns the C status."""
    lib = _load()
    s = _u16(src)
    sl = np.ascontiguousarray(np.asarray(slot, dtype=np.int64))
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    row = int(np.prod(s.shape[1:])) if s.ndim > 1 else 1
    num_slots = cache.size // row
    return int(lib.oracle_cache_write_fp8(_ptr(s), _ptr(sl), int(sl.shape[0]), _ptr(cache), num_slots, row,
                                          float(scale)))


def attention_fp8kv(rows, q, codes_k, codes_v, kv_off, k_descale, v_descale, num_q_heads: int,
                    num_kv_heads: int, head_dim: int, scale: float, tokens, key_lo=None, key_hi=None,
                    part: str = "fused"):
    """``attention`` over an FP8 cache (see ``oracle_attention_fp8kv``): every
    request's e4m3 key/value codes back to back (uint8 ``[L_total, Hkv, D]``,
    request r from token ``kv_off[r]``) and float32 descales ``[num_reqs, Hkv]``;
    key k of head g is value(code) * k_descale[r][g]."""
    lib = _load()
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 8))
    if key_lo is None or key_hi is None:
        key_lo, key_hi = key_ranges(rows, part)
    key_lo = np.ascontiguousarray(np.asarray(key_lo, dtype=np.int64))
    key_hi = np.ascontiguousarray(np.asarray(key_hi, dtype=np.int64))
    qa = _u16(q)
    ka = np.ascontiguousarray(np.asarray(codes_k, dtype=np.uint8))
    va = np.ascontiguousarray(np.asarray(codes_v, dtype=np.uint8))
    kd = np.ascontiguousarray(np.asarray(k_descale, dtype=np.float32))
    vd = np.ascontiguousarray(np.asarray(v_descale, dtype=np.float32))
    off = np.ascontiguousarray(np.asarray(kv_off, dtype=np.int64))
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = int(tok.shape[0])
    out = np.zeros((max(n, 1), num_q_heads, head_dim), dtype=np.float64)
    lse = np.zeros((max(n, 1), num_q_heads), dtype=np.float64)
    rc = lib.oracle_attention_fp8kv(int(rows.shape[0]), _ptr(rows), _ptr(key_lo), _ptr(key_hi), _ptr(qa),
                                    _ptr(ka), _ptr(va), _ptr(off), _ptr(kd), _ptr(vd), num_q_heads, num_kv_heads,
                                    head_dim, float(scale), _ptr(tok), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise OracleError(rc, "oracle_attention_fp8kv")
    return out[:n], lse[:n]


def workload_kv(spec, device: str = "cpu"):
    """Contiguous K and V of every request of a workload, back to back, and
    each request's start token: ``(kv_k, kv_v, kv_off)``."""
    import torch
    import workloads as W
    ks, vs, off, o = [], [], [], 0
    for r in range(spec.num_reqs):
        k, v = W.full_kv(spec, r, device)
        ks.append(k)
        vs.append(v)
        off.append(o)
        o += k.shape[0]
    return torch.cat(ks, 0), torch.cat(vs, 0), np.asarray(off, dtype=np.int64)
