"""Prefill Context Parallel across GPUs: one process per GPU, one PCP rank each.

"Feat/pcp qwen36 hybrid", "Changes": each PCP rank takes a contiguous slice of
the prompt; the full-attention layers all-gather K/V and run end-aligned
(bottom-right) causal attention of the slice against it. "[MRv2][PCP] Carry
the row plan ...", commit "drop pcp_has_prefill": a rank's cache writer gets
the gathered slot mapping with every entry it must not write set to PAD, and
decode rows are written by rank 0 only.

Rank r of W ranks, every rank holding a full replica of the paged cache:

1. builds the same row plan as every other rank (``num_shards = W``) and keeps
   the rows of shard r;
2. holds the new tokens it owns (``owner_shard == r``, in packed order): their
   q, k and v;
3. writes its own tokens' K/V into its cache through its PAD-masked slot view;
4. all-gathers the new tokens' K/V of every rank and writes the other ranks'
   tokens through the complementary view, so that its cache then holds every
   new token exactly as a single rank's cache would;
5. attends its own rows in its own cache, over its compact q buffer.

The index work and the collective are plain torch (any device, any process
group backend); the cache writes and the attention are the library's calls.
The collective is a single all-gather of the raw bytes of K and V together,
padded to the largest rank's token count. (The pages' alternative of a cache sharded by
token owner, with an LSE combine across ranks, is what ``PCP_ATTN_KV_SHARDS``
emulates on one GPU.)
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

import numpy as np
import torch

from . import _lib as L


def own_tokens(plan: dict, rank: int) -> np.ndarray:
    """Packed indices of the new tokens rank ``rank`` owns, ascending."""
    return np.nonzero(np.asarray(plan["owner_shard"]) == rank)[0].astype(np.int64)


def rank_rows(plan: dict, rank: int) -> np.ndarray:
    """The rows of shard ``rank`` (plan order) with ``q_start`` moved into the
    rank's compact token buffer: the position of the row's first token among
    ``own_tokens(plan, rank)``. A row is a contiguous run of packed tokens, so
    it stays contiguous in the compact buffer."""
    rows = np.asarray(plan["rows"]).reshape(-1, len(L.ROW_FIELDS))
    mine = rows[rows[:, 1] == rank].copy()
    own = own_tokens(plan, rank)
    mine[:, 2] = np.searchsorted(own, mine[:, 2]).astype(np.int32)
    return mine


def token_counts(plan: dict, world: int) -> List[int]:
    owner = np.asarray(plan["owner_shard"])
    return [int((owner == r).sum()) for r in range(world)]


def dist_all_gather(group=None) -> Callable[[torch.Tensor], List[torch.Tensor]]:
    """The collective of a torch.distributed process group: every rank's
    equally shaped tensor, in rank order."""
    import torch.distributed as dist

    def gather(x: torch.Tensor) -> List[torch.Tensor]:
        world = dist.get_world_size(group)
        out = [torch.empty_like(x) for _ in range(world)]
        dist.all_gather(out, x.contiguous(), group=group)
        return out

    return gather


def send_buffer(k_own: torch.Tensor, v_own: torch.Tensor, n_max: int) -> torch.Tensor:
    """What a rank contributes to the all-gather: the raw bytes of its K and V
    rows, padded to n_max rows ([2, n_max, bytes per row], uint8: every backend
    gathers bytes, and gloo has no 16-bit collectives)."""
    n = int(k_own.shape[0])
    nbytes = int(np.prod(tuple(k_own.shape[1:]))) * k_own.element_size()
    send = torch.zeros((2, n_max, nbytes), dtype=torch.uint8, device=k_own.device)
    send[0, :n] = k_own.reshape(n, -1).view(torch.uint8)
    send[1, :n] = v_own.reshape(n, -1).view(torch.uint8)
    return send


def gather_new_kv(k_own: torch.Tensor, v_own: torch.Tensor, plan: dict, world: int,
                  gather: Callable[[torch.Tensor], List[torch.Tensor]]):
    """Every rank's new-token K and V, in packed token order ([T, Hkv, D]).

    ``k_own`` / ``v_own`` are this rank's tokens ([n_own, Hkv, D]). Each rank
    pads its rows to the largest count, the collective gathers the raw bytes of
    K and V together, and rank r's rows land at ``own_tokens(plan, r)``."""
    counts = token_counts(plan, world)
    T = int(np.asarray(plan["owner_shard"]).shape[0])
    shape = tuple(k_own.shape[1:])
    nbytes = int(np.prod(shape)) * k_own.element_size()
    parts = gather(send_buffer(k_own, v_own, max(counts) if counts else 0))
    k_all = torch.empty((T, nbytes), dtype=torch.uint8, device=k_own.device)
    v_all = torch.empty((T, nbytes), dtype=torch.uint8, device=k_own.device)
    for r, part in enumerate(parts):
        idx = torch.from_numpy(own_tokens(plan, r)).to(k_own.device)
        if idx.numel():
            k_all[idx] = part[0, :counts[r]]
            v_all[idx] = part[1, :counts[r]]
    return k_all.view(k_own.dtype).view((T,) + shape), v_all.view(v_own.dtype).view((T,) + shape)


def other_slots(plan: dict, rank: int) -> np.ndarray:
    """The slot mapping of every new token another rank owns (PAD = -1 for this
    rank's own tokens): the complement of ``pcp_mask_slots_for_shard``."""
    slot = np.asarray(plan["slot_mapping"], dtype=np.int64)
    owner = np.asarray(plan["owner_shard"])
    return np.where(owner == rank, -1, slot).astype(np.int64)


class PcpRank:
    """One PCP rank's step on its own GPU, with every buffer preallocated.

    ``num_shards`` of the plan is the world size. ``gather`` is the
    collective (``dist_all_gather(group)`` under torch.distributed)."""

    def __init__(self, rank: int, world: int, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, split_mode: int, max_tokens: int, max_reqs: int, max_kv_len: int,
                 gather: Callable[[torch.Tensor], List[torch.Tensor]], flags: int = 0, device: str = "cuda"):
        self.rank, self.world, self.gather = rank, world, gather
        self.hq, self.hkv, self.d, self.bs = num_q_heads, num_kv_heads, head_dim, block_size
        self.split_mode, self.flags = split_mode, flags
        self.device = torch.device(device)
        self.max_rows = max(1, 2 * world * max_reqs)
        ws = L.pcp_attn_workspace_size(self.max_rows, max(max_tokens, 1), num_q_heads, head_dim, max_kv_len, flags)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device)
        self.out = torch.empty((max(max_tokens, 1), num_q_heads, head_dim), dtype=torch.bfloat16, device=self.device)
        self.lse_buf = torch.empty(max(max_tokens, 1) * num_q_heads, dtype=torch.float32, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.plan = None

    def build_plan(self, query_len: Sequence[int], num_computed: Sequence[int], block_table_host) -> dict:
        """The shared plan, this rank's rows and its token indices (host)."""
        self.plan = L.pcp_build_row_plan(query_len, num_computed, block_table_host, self.bs, self.world,
                                         self.split_mode, rows_capacity=self.max_rows)
        self.own = own_tokens(self.plan, self.rank)
        self.rows_host = rank_rows(self.plan, self.rank)
        return self.plan

    def step(self, q_own: torch.Tensor, k_own: torch.Tensor, v_own: torch.Tensor, key_cache: torch.Tensor,
             value_cache: torch.Tensor, block_table_dev: torch.Tensor, scale: float, stream=None):
        """Steps 3-5 for a plan built with :meth:`build_plan`: own write,
        all-gather, the other ranks' write, attention of this rank's rows.
        Returns (out [n_own, Hq, D], lse [Hq, n_own])."""
        plan, dev = self.plan, self.device
        slot = np.asarray(plan["slot_mapping"], dtype=np.int64)
        own_slot = torch.from_numpy(slot[self.own]).to(dev)
        L.pcp_kv_cache_write(k_own, v_own, own_slot, key_cache, value_cache, status=self.status, stream=stream)
        k_all, v_all = gather_new_kv(k_own, v_own, plan, self.world, self.gather)
        others = torch.from_numpy(other_slots(plan, self.rank)).to(dev)
        L.pcp_kv_cache_write(k_all, v_all, others, key_cache, value_cache, status=self.status, stream=stream)
        n = int(self.own.shape[0])
        rows = torch.from_numpy(self.rows_host).to(dev)
        out = self.out[:n]
        lse = self.lse_buf[:n * self.hq].view(self.hq, n)
        if rows.shape[0] == 0 or n == 0:
            return out, lse
        return L.pcp_attn_varlen(q_own, key_cache, value_cache, block_table_dev, rows, scale, out=out, lse=lse,
                                 workspace=self.workspace, flags=self.flags, status=self.status, stream=stream)

    def check_status(self) -> None:
        s = int(self.status.item())
        if s != 0:
            self.status.zero_()
            raise L.PcpError(s, "device status")
