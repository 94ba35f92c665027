"""ctypes binding of libpcp (include/pcp.h). Argument marshalling only: every
step of the path runs in the library. The binding refuses to work without the
compiled library; there is no fallback of any kind."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpcp.so")

PCP_OK = 0
PCP_ERR_ARG = -1
PCP_ERR_RANGE = -2
PCP_ERR_UNSUPPORTED = -3
PCP_ERR_ALIGN = -4
PCP_ERR_CUDA = -5
PCP_ERR_TIMEOUT = -6
PCP_ERR_WORKSPACE = -7

PCP_SPLIT_CONTIGUOUS = 0
PCP_SPLIT_DUAL_CHUNK = 1

PCP_ATTN_SEPARATE_CONTEXT = 1
PCP_ATTN_SPLIT_AT_ROW_START = 2


def PCP_ATTN_KV_SHARDS(n: int) -> int:
    """Flag: compute each prefill row as n partials over n contiguous key shards
    (decode-context-parallel emulation) and merge them by LSE."""
    return (int(n) & 0xFF) << 8


def PCP_ATTN_DECODE_SMS(n: int) -> int:
    """Flag: run the decode rows on n SMs beside the prefill rows (see
    :func:`pcp_decode_sms`)."""
    return (int(n) & 0xFF) << 16

ROW_FIELDS = ("req", "shard", "q_start", "q_len", "ctx_len", "kv_end", "causal_off", "is_decode")

# every symbol include/pcp.h declares
EXPORTS = ("pcp_build_row_plan", "pcp_mask_slots_for_shard", "pcp_decode_sms", "pcp_kv_cache_write",
           "pcp_kv_cache_write_fp8", "pcp_attn_workspace_size", "pcp_attn_varlen", "pcp_attn_varlen_noalloc",
           "pcp_attn_varlen_fp8kv", "pcp_lse_merge",
           "pcp_set_profile_events", "pcp_selftest_bounded_wait",
           "pcp_last_cuda_error", "pcp_status_string")

_lib = None


class PcpError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = "?"
        if _lib is not None:
            msg = _lib.pcp_status_string(code).decode()
        extra = ""
        if code == PCP_ERR_CUDA and _lib is not None:
            extra = f" (cudaError {_lib.pcp_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [{code}]{extra}")
        self.code = code


def load(path: Optional[str] = None):
    """Load libpcp.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with context_prefill_attention_gb300.build.build() "
                           "(nvcc, sm_103a); there is no fallback path")
    lib = ctypes.CDLL(path)
    P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    lib.pcp_build_row_plan.argtypes = [i32, P, P, P, i32, i32, i32, i32, P, i32, P, P, P, P]
    lib.pcp_build_row_plan.restype = ctypes.c_int
    lib.pcp_mask_slots_for_shard.argtypes = [P, P, i32, i32, P]
    lib.pcp_mask_slots_for_shard.restype = ctypes.c_int
    lib.pcp_decode_sms.argtypes = [P, i32, i32, i32, i32, i32, i32]
    lib.pcp_decode_sms.restype = i32
    lib.pcp_kv_cache_write.argtypes = [P, P, P, i32, P, P, i64, i32, i32, i32, P, P]
    lib.pcp_kv_cache_write.restype = ctypes.c_int
    lib.pcp_kv_cache_write_fp8.argtypes = [P, P, P, i32, P, P, i64, i32, i32, i32, f32, f32, P, P]
    lib.pcp_kv_cache_write_fp8.restype = ctypes.c_int
    lib.pcp_attn_varlen_fp8kv.argtypes = [P, P, P, P, P, P, i32, i32, i64, i32, P, i32, i32, i32, i32, i32, f32,
                                          P, P, P, sz, i32, P, P]
    lib.pcp_attn_varlen_fp8kv.restype = ctypes.c_int
    lib.pcp_attn_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pcp_attn_workspace_size.restype = sz
    lib.pcp_attn_varlen.argtypes = [P, P, P, P, i32, i32, i64, i32, P, i32, i32, i32, i32, i32, f32, P, P, P,
                                    sz, i32, P, P]
    lib.pcp_attn_varlen.restype = ctypes.c_int
    lib.pcp_lse_merge.argtypes = [P, P, P, P, P, P, i32, i32, i32, P]
    lib.pcp_lse_merge.restype = ctypes.c_int
    lib.pcp_attn_varlen_noalloc.argtypes = [P, P, P, P, i32, i32, i64, i32, P, i32, i32, i32, i32, i32, f32,
                                            P, P, i32, P, P]
    lib.pcp_attn_varlen_noalloc.restype = ctypes.c_int
    lib.pcp_selftest_bounded_wait.argtypes = [P, ctypes.c_uint32, P]
    lib.pcp_selftest_bounded_wait.restype = ctypes.c_int
    lib.pcp_set_profile_events.argtypes = [P, P, P, P]
    lib.pcp_set_profile_events.restype = ctypes.c_int
    lib.pcp_last_cuda_error.argtypes = []
    lib.pcp_last_cuda_error.restype = ctypes.c_int
    lib.pcp_status_string.argtypes = [ctypes.c_int]
    lib.pcp_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _np_ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _t_ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, what: str):
    if rc != PCP_OK:
        raise PcpError(rc, what)


BF16 = (torch.bfloat16,)
F32 = (torch.float32,)
I32 = (torch.int32,)
I64 = (torch.int64,)
# an FP8 cache holds one e4m3 code per byte: raw bytes or PyTorch's e4m3 "fn" type
FP8_CACHE = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def _is_device_tensor(t: torch.Tensor) -> bool:
    return t.device.type == "cuda"


def _dev(t, name: str, dtypes=None, shape=None, device=None) -> torch.Tensor:
    """``t`` checked before its pointer crosses the ABI: a contiguous CUDA tensor
    (the library takes device pointers), of one of ``dtypes``, of ``shape``
    where given (-1 leaves a dimension free) and on ``device`` where given.
    Raises TypeError / ValueError; nothing is launched."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {' or '.join(str(d) for d in dtypes)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and (t.dim() != len(shape) or
                              any(want != -1 and want != got for want, got in zip(shape, t.shape))):
        want = tuple("*" if x == -1 else x for x in shape)
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {want}")
    if not _is_device_tensor(t):
        raise ValueError(f"{name}: must be a CUDA tensor (the library takes device pointers), got {t.device}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, the other arguments are on {device}")
    return t


def _status(status, device) -> Optional[torch.Tensor]:
    if status is None:
        return None
    _dev(status, "status", I32, device=device)
    if status.numel() < 1:
        raise ValueError("status: needs one int32 element")
    return status


def _check_write(k, v, slot_mapping, key_cache, value_cache, status, cache_dtypes):
    _dev(key_cache, "key_cache", cache_dtypes, shape=(-1, -1, -1, -1))
    dev = key_cache.device
    nb, bs, hkv, d = (int(x) for x in key_cache.shape)
    _dev(value_cache, "value_cache", cache_dtypes, shape=(nb, bs, hkv, d), device=dev)
    _dev(k, "k", BF16, shape=(-1, hkv, d), device=dev)
    T = int(k.shape[0])
    _dev(v, "v", BF16, shape=(T, hkv, d), device=dev)
    _dev(slot_mapping, "slot_mapping", I64, shape=(T,), device=dev)
    _status(status, dev)
    return T, nb, bs, hkv, d


def _check_attn(q, key_cache, value_cache, block_table, rows, out, lse, workspace, status, cache_dtypes):
    _dev(q, "q", BF16, shape=(-1, -1, -1))
    dev = q.device
    T, hq, d = (int(x) for x in q.shape)
    _dev(key_cache, "key_cache", cache_dtypes, shape=(-1, -1, -1, d), device=dev)
    nb, bs, hkv, _ = (int(x) for x in key_cache.shape)
    _dev(value_cache, "value_cache", cache_dtypes, shape=(nb, bs, hkv, d), device=dev)
    _dev(block_table, "block_table", I32, shape=(-1, -1), device=dev)
    _dev(rows, "rows", I32, shape=(-1, len(ROW_FIELDS)), device=dev)
    if out is not None:
        _dev(out, "out", BF16, shape=(T, hq, d), device=dev)
    if lse is not None:
        _dev(lse, "lse", F32, shape=(hq, T), device=dev)
    if workspace is not None:
        _dev(workspace, "workspace", device=dev)
    _status(status, dev)
    return T, hq, d, nb, bs, hkv


def pcp_build_row_plan(query_len, num_computed, block_table, block_size: int, num_shards: int,
                       split_mode: int = PCP_SPLIT_CONTIGUOUS, rows_capacity: Optional[int] = None):
    """Host row plan and slot mapping. Returns a dict of numpy arrays:
    ``rows`` int32[n, 8], ``cu_q`` int32[n+1], ``slot_mapping`` int64[T],
    ``owner_shard`` int8[T]."""
    lib = load()
    ql = np.ascontiguousarray(np.asarray(query_len, dtype=np.int32))
    nc = np.ascontiguousarray(np.asarray(num_computed, dtype=np.int32))
    bt = block_table.numpy() if isinstance(block_table, torch.Tensor) else block_table
    bt = np.ascontiguousarray(np.asarray(bt, dtype=np.int32))
    R = int(ql.shape[0])
    mb = int(bt.shape[1]) if bt.ndim == 2 else 0
    T = int(ql.sum())
    cap = rows_capacity if rows_capacity is not None else max(1, 2 * num_shards * R)
    rows = np.zeros((max(cap, 1), 8), dtype=np.int32)
    cu = np.zeros(max(cap, 1) + 1, dtype=np.int32)
    slot = np.zeros(max(T, 1), dtype=np.int64)
    owner = np.zeros(max(T, 1), dtype=np.int8)
    n = np.zeros(1, dtype=np.int32)
    rc = lib.pcp_build_row_plan(R, _np_ptr(ql), _np_ptr(nc), _np_ptr(bt), mb, block_size, num_shards,
                                split_mode, _np_ptr(rows), cap, _np_ptr(n), _np_ptr(cu), _np_ptr(slot),
                                _np_ptr(owner))
    _check(rc, "pcp_build_row_plan")
    k = int(n[0])
    return dict(rows=rows[:k], cu_q=cu[:k + 1], slot_mapping=slot[:T], owner_shard=owner[:T])


def pcp_mask_slots_for_shard(slot_mapping: np.ndarray, owner_shard: np.ndarray, shard: int) -> np.ndarray:
    """PAD-masked slot mapping of one shard (host arrays)."""
    lib = load()
    s = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    o = np.ascontiguousarray(owner_shard, dtype=np.int8)
    out = np.empty_like(s)
    _check(lib.pcp_mask_slots_for_shard(_np_ptr(s), _np_ptr(o), int(s.shape[0]), shard, _np_ptr(out)),
           "pcp_mask_slots_for_shard")
    return out


def pcp_decode_sms(rows: np.ndarray, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   kv_cache_fp8: bool, num_sms: int) -> int:
    """SMs for the decode rows of a host row plan (int32 ``[n, 8]``) beside its
    prefill rows, or 0 to run them in sequence (host function, no GPU)."""
    lib = load()
    r = np.ascontiguousarray(rows, dtype=np.int32)
    if r.ndim != 2 or (r.shape[0] and r.shape[1] != 8):
        raise ValueError(f"rows: shape {r.shape}, expected [n, 8]")
    return int(lib.pcp_decode_sms(_np_ptr(r), int(r.shape[0]), int(num_q_heads), int(num_kv_heads),
                                  int(head_dim), 1 if kv_cache_fp8 else 0, int(num_sms)))


def pcp_kv_cache_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                       key_cache: torch.Tensor, value_cache: torch.Tensor,
                       status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Scatter new K/V ``[T, Hkv, D]`` into the paged caches ``[num_blocks, bs, Hkv, D]``."""
    lib = load()
    T, nb, bs, hkv, d = _check_write(k, v, slot_mapping, key_cache, value_cache, status, BF16)
    rc = lib.pcp_kv_cache_write(_t_ptr(k), _t_ptr(v), _t_ptr(slot_mapping), T, _t_ptr(key_cache),
                                _t_ptr(value_cache), nb, bs, hkv, d, _t_ptr(status), _stream(stream))
    _check(rc, "pcp_kv_cache_write")


def pcp_kv_cache_write_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                           key_cache: torch.Tensor, value_cache: torch.Tensor, k_scale: float, v_scale: float,
                           status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Scatter new bf16 K/V ``[T, Hkv, D]`` into FP8 (e4m3) caches ``[num_blocks, bs,
    Hkv, D]`` (uint8) as e4m3(x / k_scale) and e4m3(x / v_scale)."""
    lib = load()
    T, nb, bs, hkv, d = _check_write(k, v, slot_mapping, key_cache, value_cache, status, FP8_CACHE)
    rc = lib.pcp_kv_cache_write_fp8(_t_ptr(k), _t_ptr(v), _t_ptr(slot_mapping), T, _t_ptr(key_cache),
                                    _t_ptr(value_cache), nb, bs, hkv, d, float(k_scale), float(v_scale),
                                    _t_ptr(status), _stream(stream))
    _check(rc, "pcp_kv_cache_write_fp8")


def pcp_attn_workspace_size(num_rows: int, total_q: int, num_q_heads: int, head_dim: int,
                            max_kv_len: int, flags: int = 0) -> int:
    return int(load().pcp_attn_workspace_size(num_rows, total_q, num_q_heads, head_dim, max_kv_len, flags))


def pcp_attn_varlen(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                    block_table: torch.Tensor, rows: torch.Tensor, scale: float,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, flags: int = 0,
                    status: Optional[torch.Tensor] = None, stream=None):
    """Attention of every planned row. ``q`` ``[T, Hq, D]`` bf16; ``rows`` int32
    ``[n, 8]`` on the device; returns ``(out [T, Hq, D] bf16, lse [Hq, T] fp32)``.
    Pass ``out``/``lse``/``workspace`` to avoid allocating per call."""
    lib = load()
    T, hq, d, nb, bs, hkv = _check_attn(q, key_cache, value_cache, block_table, rows, out, lse, workspace, status,
                                        BF16)
    n_rows = int(rows.shape[0])
    mb = int(block_table.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    need = pcp_attn_workspace_size(n_rows, T, hq, d, mb * bs, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.pcp_attn_varlen(_t_ptr(q), _t_ptr(key_cache), _t_ptr(value_cache), _t_ptr(block_table),
                             int(block_table.shape[0]), mb, nb,
                             bs, _t_ptr(rows), n_rows, T, hq, hkv, d, float(scale), _t_ptr(out), _t_ptr(lse),
                             _t_ptr(workspace), int(workspace.numel() * workspace.element_size()), flags,
                             _t_ptr(status), _stream(stream))
    _check(rc, "pcp_attn_varlen")
    return out, lse


def pcp_attn_varlen_fp8kv(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                          k_descale: torch.Tensor, v_descale: torch.Tensor, block_table: torch.Tensor,
                          rows: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          flags: int = 0, status: Optional[torch.Tensor] = None, stream=None):
    """:func:`pcp_attn_varlen` over FP8 (e4m3, uint8) caches with fp32 descales
    ``[num_reqs, Hkv]`` on the device."""
    lib = load()
    T, hq, d, nb, bs, hkv = _check_attn(q, key_cache, value_cache, block_table, rows, out, lse, workspace, status,
                                        FP8_CACHE)
    R = int(block_table.shape[0])
    _dev(k_descale, "k_descale", F32, shape=(R, hkv), device=q.device)
    _dev(v_descale, "v_descale", F32, shape=(R, hkv), device=q.device)
    n_rows = int(rows.shape[0])
    mb = int(block_table.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    need = pcp_attn_workspace_size(n_rows, T, hq, d, mb * bs, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.pcp_attn_varlen_fp8kv(_t_ptr(q), _t_ptr(key_cache), _t_ptr(value_cache), _t_ptr(k_descale),
                                   _t_ptr(v_descale), _t_ptr(block_table), int(block_table.shape[0]), mb, nb, bs,
                                   _t_ptr(rows), n_rows, T, hq, hkv, d, float(scale), _t_ptr(out), _t_ptr(lse),
                                   _t_ptr(workspace), int(workspace.numel() * workspace.element_size()), flags,
                                   _t_ptr(status), _stream(stream))
    _check(rc, "pcp_attn_varlen_fp8kv")
    return out, lse


def pcp_attn_varlen_noalloc(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                            block_table: torch.Tensor, rows: torch.Tensor, scale: float, out: torch.Tensor,
                            lse: torch.Tensor, flags: int = 0, status: Optional[torch.Tensor] = None,
                            stream=None):
    """:func:`pcp_attn_varlen` for callers that cannot allocate device memory:
    the caller passes ``out`` and ``lse``, and the library's own fixed 64 MiB
    scratch array (reserved on each GPU that loads the library) replaces the
    workspace. Calls on one device share that array: keep them on one stream."""
    lib = load()
    if out is None or lse is None:
        raise ValueError("pcp_attn_varlen_noalloc: out and lse are required")
    T, hq, d, nb, bs, hkv = _check_attn(q, key_cache, value_cache, block_table, rows, out, lse, None, status,
                                        BF16)
    rc = lib.pcp_attn_varlen_noalloc(_t_ptr(q), _t_ptr(key_cache), _t_ptr(value_cache), _t_ptr(block_table),
                                     int(block_table.shape[0]), int(block_table.shape[1]), nb, bs, _t_ptr(rows),
                                     int(rows.shape[0]), T, hq, hkv, d, float(scale), _t_ptr(out), _t_ptr(lse),
                                     flags, _t_ptr(status), _stream(stream))
    _check(rc, "pcp_attn_varlen_noalloc")
    return out, lse


def pcp_lse_merge(out_a: torch.Tensor, lse_a: torch.Tensor, out_b: torch.Tensor, lse_b: torch.Tensor,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, stream=None):
    """LSE merge of two fp32 partials ``[T, Hq, D]`` / ``[Hq, T]`` into bf16 out and fp32 lse."""
    lib = load()
    _dev(out_a, "out_a", F32, shape=(-1, -1, -1))
    dev = out_a.device
    T, hq, d = (int(x) for x in out_a.shape)
    _dev(out_b, "out_b", F32, shape=(T, hq, d), device=dev)
    _dev(lse_a, "lse_a", F32, shape=(hq, T), device=dev)
    _dev(lse_b, "lse_b", F32, shape=(hq, T), device=dev)
    if out is None:
        out = torch.empty(out_a.shape, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty_like(lse_a)
    _dev(out, "out", BF16, shape=(T, hq, d), device=dev)
    _dev(lse, "lse", F32, shape=(hq, T), device=dev)
    rc = lib.pcp_lse_merge(_t_ptr(out_a), _t_ptr(lse_a), _t_ptr(out_b), _t_ptr(lse_b), _t_ptr(out), _t_ptr(lse),
                           T, hq, d, _stream(stream))
    _check(rc, "pcp_lse_merge")
    return out, lse


def pcp_set_profile_events(prefill_begin=None, prefill_end=None, decode_begin=None, decode_end=None) -> None:
    """Register ``torch.cuda.Event`` objects (already recorded once, so that they
    exist) to be recorded around the prefill and decode kernels of later
    :func:`pcp_attn_varlen` calls in this thread; no arguments unregisters."""
    def h(e):
        return None if e is None else ctypes.c_void_p(int(e.cuda_event))
    load().pcp_set_profile_events(h(prefill_begin), h(prefill_end), h(decode_begin), h(decode_end))
