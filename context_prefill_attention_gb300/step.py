"""One PCP attention step through the C ABI, with every buffer preallocated.

A step ("Feat/pcp qwen36 hybrid", "Changes"; "[MRv2][PCP] Carry the row plan
...", sections 1-2 and "What made it removable") is:

1. ``pcp_build_row_plan`` on the host: shard rows and the slot mapping;
2. the plan (rows, slots) copied to the device from pinned staging buffers;
3. ``pcp_kv_cache_write``: the new tokens' K/V into the paged cache, ordered
   before attention on the same stream;
4. ``pcp_attn_varlen``: prefill, context and decode rows in one call. With
   ``decode_beside_prefill=True`` (and a bf16 cache) the decode rows run on the
   SMs ``pcp_decode_sms`` picks from the host plan, beside the prefill rows
   (``PCP_ATTN_DECODE_SMS``): a shorter step, with each kernel on part of the GPU.

With ``kv_cache_dtype="fp8"`` the cache holds e4m3 codes: step 3 is
``pcp_kv_cache_write_fp8`` with the layer's k/v scales and step 4
``pcp_attn_varlen_fp8kv`` with descales of shape (num_reqs, num_kv_heads),
by default those scales broadcast ("[MRv2] FlashAttention PCP support ...",
the context-pass call).

This module only sequences those calls and owns the buffers (the reviewer's
"use the workspace and pass out so we aren't allocating each step").
"""
from __future__ import annotations

import os
import sys
from typing import Optional, Sequence

import numpy as np
import torch

from . import _lib as L


class PcpStep:
    """Preallocated buffers and the call sequence of one PCP step on one GPU."""

    def __init__(self, *, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                 num_shards: int, split_mode: int, max_tokens: int, max_reqs: int, max_kv_len: int,
                 flags: int = 0, device: str = "cuda", kv_cache_dtype: str = "bf16", k_scale: float = 1.0,
                 v_scale: float = 1.0, decode_beside_prefill: bool = False):
        if kv_cache_dtype not in ("bf16", "fp8"):
            raise ValueError(f"kv_cache_dtype {kv_cache_dtype!r}: 'bf16' or 'fp8'")
        self.kv_fp8 = kv_cache_dtype == "fp8"
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        self.hq, self.hkv, self.d = num_q_heads, num_kv_heads, head_dim
        self.bs, self.shards, self.split_mode, self.flags = block_size, num_shards, split_mode, flags
        self.device = torch.device(device)
        # decode rows beside the prefill rows, on request, unless the caller's flags
        # already say how many SMs they take
        self.decode_beside = decode_beside_prefill and ((flags >> 16) & 0xFF) == 0
        self.num_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.decode_sms = 0
        self.max_rows = max(1, 2 * num_shards * max_reqs)
        self.max_tokens = max_tokens
        ws = L.pcp_attn_workspace_size(self.max_rows, max_tokens, num_q_heads, head_dim, max_kv_len, flags)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device)
        self.out = torch.empty((max(max_tokens, 1), num_q_heads, head_dim), dtype=torch.bfloat16,
                               device=self.device)
        self.lse_buf = torch.empty(max(max_tokens, 1) * num_q_heads, dtype=torch.float32, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.rows_dev = torch.empty((self.max_rows, 8), dtype=torch.int32, device=self.device)
        self.slot_dev = torch.empty(max(max_tokens, 1), dtype=torch.int64, device=self.device)
        self.rows_host = torch.empty((self.max_rows, 8), dtype=torch.int32, pin_memory=True)
        self.slot_host = torch.empty(max(max_tokens, 1), dtype=torch.int64, pin_memory=True)
        # FP8 descales [max_reqs, Hkv]: the layer scales broadcast; a caller may overwrite them
        self.k_descale = self.v_descale = None
        if self.kv_fp8:
            self.k_descale = torch.full((max(max_reqs, 1), num_kv_heads), self.k_scale, dtype=torch.float32,
                                        device=self.device)
            self.v_descale = torch.full((max(max_reqs, 1), num_kv_heads), self.v_scale, dtype=torch.float32,
                                        device=self.device)
        self.plan = None

    def build_plan(self, query_len: Sequence[int], num_computed: Sequence[int], block_table_host) -> dict:
        """Step 1. With ``PCP_DEBUG=1`` in the environment a summary of the plan
        (:func:`plan_summary`) goes to stderr."""
        self.plan = L.pcp_build_row_plan(query_len, num_computed, block_table_host, self.bs, self.shards,
                                         self.split_mode, rows_capacity=self.max_rows)
        self.decode_sms = (L.pcp_decode_sms(self.plan["rows"], self.hq, self.hkv, self.d, self.kv_fp8,
                                            self.num_sms) if self.decode_beside else 0)
        debug_plan(self.plan, self.shards)
        return self.plan

    def upload_plan(self, stream=None) -> None:
        p = self.plan
        n, T = p["rows"].shape[0], p["slot_mapping"].shape[0]
        self.rows_host[:n].numpy()[...] = p["rows"]
        self.slot_host[:T].numpy()[...] = p["slot_mapping"]
        self.rows_dev[:n].copy_(self.rows_host[:n], non_blocking=True)
        self.slot_dev[:T].copy_(self.slot_host[:T], non_blocking=True)

    def write_cache(self, k_new: torch.Tensor, v_new: torch.Tensor, key_cache: torch.Tensor,
                    value_cache: torch.Tensor, stream=None) -> None:
        T = int(k_new.shape[0])
        if self.kv_fp8:
            L.pcp_kv_cache_write_fp8(k_new, v_new, self.slot_dev[:T], key_cache, value_cache, self.k_scale,
                                     self.v_scale, status=self.status, stream=stream)
        else:
            L.pcp_kv_cache_write(k_new, v_new, self.slot_dev[:T], key_cache, value_cache, status=self.status,
                                 stream=stream)

    def attend(self, q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
               block_table_dev: torch.Tensor, scale: float, stream=None):
        T = int(q.shape[0])
        n = int(self.plan["rows"].shape[0])
        out = self.out[:T]
        lse = self.lse_buf[:T * self.hq].view(self.hq, T)
        flags = self.flags | L.PCP_ATTN_DECODE_SMS(self.decode_sms)
        if self.kv_fp8:
            R = int(block_table_dev.shape[0])
            return L.pcp_attn_varlen_fp8kv(q, key_cache, value_cache, self.k_descale[:R], self.v_descale[:R],
                                           block_table_dev, self.rows_dev[:n], scale, out=out, lse=lse,
                                           workspace=self.workspace, flags=flags, status=self.status,
                                           stream=stream)
        return L.pcp_attn_varlen(q, key_cache, value_cache, block_table_dev, self.rows_dev[:n], scale,
                                 out=out, lse=lse, workspace=self.workspace, flags=flags,
                                 status=self.status, stream=stream)

    def run(self, q, k_new, v_new, key_cache, value_cache, block_table_dev, scale: float, stream=None):
        """Steps 2-4 for a plan already built with :meth:`build_plan`."""
        self.upload_plan(stream)
        self.write_cache(k_new, v_new, key_cache, value_cache, stream)
        return self.attend(q, key_cache, value_cache, block_table_dev, scale, stream)

    def check_status(self) -> None:
        """Raise if a kernel reported an error (synchronises the device)."""
        s = int(self.status.item())
        if s != 0:
            self.status.zero_()
            raise L.PcpError(s, "device status")


def plan_summary(plan: dict, num_shards: int) -> str:
    """A few lines on a row plan: rows and tokens per shard, prefill / decode /
    prefix rows, the longest row and key range, and the slot mapping's PAD
    count and range."""
    rows = np.asarray(plan["rows"]).reshape(-1, len(L.ROW_FIELDS)).astype(np.int64)
    slots = np.asarray(plan["slot_mapping"])
    lines = [f"[pcp] plan: {rows.shape[0]} rows ({int((rows[:, 7] == 0).sum())} prefill, "
             f"{int((rows[:, 7] == 1).sum())} decode), {int(rows[:, 3].sum())} tokens, {num_shards} shards"]
    for s in range(num_shards):
        r = rows[rows[:, 1] == s]
        if r.shape[0] == 0:
            lines.append(f"[pcp]   shard {s}: no rows")
            continue
        lines.append(f"[pcp]   shard {s}: {r.shape[0]} rows, {int(r[:, 3].sum())} tokens, q_len "
                     f"{int(r[:, 3].min())}..{int(r[:, 3].max())}, kv_end max {int(r[:, 5].max())}, "
                     f"{int((r[:, 4] > 0).sum())} with a cached prefix")
    pad = int((slots < 0).sum())
    live = slots[slots >= 0]
    rng = f"[{int(live.min())}, {int(live.max())}]" if live.size else "[]"
    lines.append(f"[pcp] slots: {slots.shape[0]} ({pad} PAD), range {rng}")
    return "\n".join(lines)


def debug_plan(plan: dict, num_shards: int) -> None:
    """Print :func:`plan_summary` to stderr when ``PCP_DEBUG=1``."""
    if os.environ.get("PCP_DEBUG", "") == "1":
        print(plan_summary(plan, num_shards), file=sys.stderr, flush=True)


def write_positions(key_cache: torch.Tensor, value_cache: torch.Tensor, block_table_host,
                    start: Sequence[int], k_list, v_list, block_size: int,
                    status: Optional[torch.Tensor] = None, fp8_scales=None) -> None:
    """Write K/V rows of positions ``[start[r], start[r] + len)`` of every request
    into the paged cache, through the library's own plan (one shard) and cache
    writer — what earlier steps of a real engine would have left in the cache.
    ``fp8_scales=(k_scale, v_scale)`` writes an FP8 cache."""
    lens = [int(k.shape[0]) for k in k_list]
    if sum(lens) == 0:
        return
    plan = L.pcp_build_row_plan(lens, list(start), block_table_host, block_size, 1, L.PCP_SPLIT_CONTIGUOUS)
    dev = key_cache.device
    slot = torch.from_numpy(plan["slot_mapping"]).to(dev)
    k = torch.cat([x.to(dev) for x in k_list], 0)
    v = torch.cat([x.to(dev) for x in v_list], 0)
    if fp8_scales is not None:
        L.pcp_kv_cache_write_fp8(k, v, slot, key_cache, value_cache, fp8_scales[0], fp8_scales[1], status=status)
    else:
        L.pcp_kv_cache_write(k, v, slot, key_cache, value_cache, status=status)
