"""Seeded synthetic workloads for Prefill Context Parallel (PCP) attention.

This module only draws inputs: request lengths, cached-prefix lengths, paged
block tables and bf16 Q/K/V values. It holds none of the method's arithmetic
(no row plan, no slot formula, no attention), so both the CPU oracle under
``oracle/`` and the CUDA library can be fed from it without sharing any code.

Five workloads are defined, each by its shape (the numbers are sizes, not
results):

* ``1``  one 512-token prompt, 2 contiguous shards, 4 q / 2 kv heads, D=64,
         block_size 16 with an identity block table;
* ``2``  8 prompts of U[512,4096] tokens, 2 shards (one head row and one tail
         row each), 16 q / 8 kv heads, D=128, shuffled pages;
* ``3``  4 requests with a cached prefix U[8192,32768] and U[1024,4096] new
         tokens in 2 shards, 32 q / 8 kv heads, D=128;
* ``4``  8 prompts of U[1024,8192] tokens (2 shards) plus 56 single-token
         decode requests with U[1024,16384] keys, 32 q / 8 kv heads, D=128;
* ``5``  one 131072-token prompt in 4 contiguous shards, 32 q / 4 kv heads,
         D=128.

Randomness: ``torch.Generator`` seeded with ``20260000 + workload_id`` draws
the lengths and the block-table permutation; every tensor of request ``r``
comes from its own generator seeded with ``tensor_seed(seed, r, kind)`` so a
test can rebuild a single request without drawing the whole batch. Values are
``torch.randn`` in float32 rounded to bf16 (round to nearest even).

FP8 (e4m3) cache inputs: the layer scales ``FP8_K_SCALE`` / ``FP8_V_SCALE``
(the N(0, 1) values stay far inside 448 x scale) and, per workload, the
descales of shape (num_reqs, num_kv_heads): the layer scales broadcast, or a
seeded factor in [0.5, 1) times them per (request, kv head), so that the
dequantised values stay N(0, 1)-sized like the bf16 inputs (the output is
rounded to bf16, whose half-ulp reaches the 1e-2 bound at |out| = 5.12).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

SPLIT_CONTIGUOUS = 0
SPLIT_DUAL_CHUNK = 1

KIND_Q, KIND_K, KIND_V, KIND_KP, KIND_VP = range(5)


def tensor_seed(seed: int, req: int, kind: int) -> int:
    """Seed of the generator that draws tensor ``kind`` of request ``req``."""
    return (seed * 100003 + req * 8 + kind) % (2 ** 63)


@dataclasses.dataclass
class WorkloadSpec:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_shards: int
    split_mode: int
    query_len: List[int]
    num_computed: List[int]
    identity_pages: bool = False
    page_slack: float = 0.05

    @property
    def num_reqs(self) -> int:
        return len(self.query_len)

    @property
    def total_q(self) -> int:
        return int(sum(self.query_len))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


def _randint(g: torch.Generator, lo: int, hi: int, n: int) -> List[int]:
    """n integers uniform in [lo, hi] (both ends inclusive)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def workload_spec(workload: int, split_mode: int = SPLIT_CONTIGUOUS) -> WorkloadSpec:
    """Shape of one of the five synthetic workloads (lengths drawn from its seed)."""
    seed = 20260000 + workload
    g = torch.Generator().manual_seed(seed)
    if workload == 1:
        return WorkloadSpec("prefill-512-2shard-gqa4x2-d64", seed, 4, 2, 64, 16, 2,
                            SPLIT_CONTIGUOUS, [512], [0], identity_pages=True)
    if workload == 2:
        n = _randint(g, 512, 4096, 8)
        return WorkloadSpec("prefill-8req-512to4096-2shard-gqa16x8-d128", seed, 16, 8, 128, 16, 2,
                            split_mode, n, [0] * 8)
    if workload == 3:
        p = _randint(g, 8192, 32768, 4)
        n = _randint(g, 1024, 4096, 4)
        return WorkloadSpec("extend-4req-prefix8kto32k-new1kto4k-gqa32x8-d128", seed, 32, 8, 128, 16, 2,
                            split_mode, n, p)
    if workload == 4:
        n = _randint(g, 1024, 8192, 8)
        c = _randint(g, 1024, 16384, 56)
        return WorkloadSpec("mixed-8prefill1kto8k-56decode1kto16k-gqa32x8-d128", seed, 32, 8, 128, 16, 2,
                            split_mode, n + [1] * 56, [0] * 8 + [x - 1 for x in c])
    if workload == 5:
        return WorkloadSpec("prefill-131072-4shard-gqa32x4-d128", seed, 32, 4, 128, 16, 4,
                            SPLIT_CONTIGUOUS, [131072], [0])
    raise ValueError(f"unknown workload {workload}")


def custom_spec(query_len: Sequence[int], num_computed: Sequence[int], *, num_q_heads: int,
                num_kv_heads: int, head_dim: int, block_size: int = 16, num_shards: int = 2,
                split_mode: int = SPLIT_CONTIGUOUS, seed: int = 1234,
                identity_pages: bool = False, name: str = "custom") -> WorkloadSpec:
    """A small ad-hoc batch (used for ragged and edge-case tests)."""
    return WorkloadSpec(name, seed, num_q_heads, num_kv_heads, head_dim, block_size, num_shards,
                        split_mode, list(map(int, query_len)), list(map(int, num_computed)),
                        identity_pages=identity_pages)


def block_tables(spec: WorkloadSpec):
    """Paged block tables: ``(block_table[R, max_blocks] int32, num_blocks)``.

    Request ``r`` owns ``ceil((num_computed + query_len) / block_size)`` pages.
    The pool holds those pages plus ``page_slack`` spare ones; pages are a
    random permutation of the pool (identity for workload 1). Unused table
    entries are -1.
    """
    g = torch.Generator().manual_seed(spec.seed + 7)
    bs = spec.block_size
    need = [-(-(p + n) // bs) for p, n in zip(spec.num_computed, spec.query_len)]
    total = sum(need)
    num_blocks = total + max(1, int(math.ceil(total * spec.page_slack)))
    if spec.identity_pages:
        perm = torch.arange(num_blocks, dtype=torch.int64)
    else:
        perm = torch.randperm(num_blocks, generator=g)
    max_blocks = max(1, max(need) if need else 1)
    table = torch.full((spec.num_reqs, max_blocks), -1, dtype=torch.int32)
    o = 0
    for r, k in enumerate(need):
        table[r, :k] = perm[o:o + k].to(torch.int32)
        o += k
    return table, num_blocks


def _randn_bf16(seed: int, shape, device: str = "cpu") -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def request_tensor(spec: WorkloadSpec, req: int, kind: int, device: str = "cpu") -> torch.Tensor:
    """One tensor of one request: q ``[N,Hq,D]``, new k/v ``[N,Hkv,D]``,
    prefix k/v ``[P,Hkv,D]`` (bf16)."""
    n, p = spec.query_len[req], spec.num_computed[req]
    rows = p if kind in (KIND_KP, KIND_VP) else n
    heads = spec.num_q_heads if kind == KIND_Q else spec.num_kv_heads
    return _randn_bf16(tensor_seed(spec.seed, req, kind), (rows, heads, spec.head_dim), device)


def packed_new_tokens(spec: WorkloadSpec, kind: int, device: str = "cpu",
                      reqs: Optional[Sequence[int]] = None) -> torch.Tensor:
    """q, k or v of every new token, packed request-major ``[T, H, D]``."""
    reqs = range(spec.num_reqs) if reqs is None else reqs
    parts = [request_tensor(spec, r, kind, device) for r in reqs]
    heads = spec.num_q_heads if kind == KIND_Q else spec.num_kv_heads
    if not parts:
        return torch.empty((0, heads, spec.head_dim), dtype=torch.bfloat16, device=device)
    return torch.cat(parts, 0)


def full_kv(spec: WorkloadSpec, req: int, device: str = "cpu"):
    """Contiguous K and V of request ``req`` over all its positions
    ``[num_computed + query_len, Hkv, D]`` (cached prefix, then new tokens)."""
    k = torch.cat([request_tensor(spec, req, KIND_KP, device), request_tensor(spec, req, KIND_K, device)], 0)
    v = torch.cat([request_tensor(spec, req, KIND_VP, device), request_tensor(spec, req, KIND_V, device)], 0)
    return k, v


def token_offsets(spec: WorkloadSpec) -> List[int]:
    """Packed offset of each request's first new token (request-major order)."""
    out, o = [], 0
    for n in spec.query_len:
        out.append(o)
        o += n
    return out


def sample_segments(segments: Sequence, per_segment: int, seed: int) -> torch.Tensor:
    """A seeded random subset of packed token indices: up to ``per_segment``
    tokens of each ``(start, length)`` segment plus its first and last token
    (sorted, unique)."""
    g = torch.Generator().manual_seed(seed)
    picks = []
    for start, n in segments:
        start, n = int(start), int(n)
        if n <= 0:
            continue
        idx = torch.randperm(n, generator=g)[:min(per_segment, n)]
        picks.append(idx + start)
        picks.append(torch.tensor([start, start + n - 1]))
    if not picks:
        return torch.empty(0, dtype=torch.int64)
    return torch.unique(torch.cat(picks)).to(torch.int64)


# Layer scales of an FP8 (e4m3) cache: N(0, 1) K/V values of magnitude < 5 map to
# codes of magnitude < 100 (K) and < 167 (V), inside e4m3's 448.
FP8_K_SCALE = 0.05
FP8_V_SCALE = 0.03


def fp8_descales(spec: WorkloadSpec, mode: str = "layer"):
    """(k_descale, v_descale), float32 [num_reqs, num_kv_heads] on the CPU:
    ``layer`` broadcasts the layer scales; ``varied`` multiplies them by a
    seeded factor in [0.5, 1) per (request, kv head)."""
    R, H = spec.num_reqs, spec.num_kv_heads
    if mode == "layer":
        return torch.full((R, H), FP8_K_SCALE), torch.full((R, H), FP8_V_SCALE)
    if mode != "varied":
        raise ValueError(mode)
    g = torch.Generator().manual_seed(tensor_seed(spec.seed, 0, 7))
    kd = FP8_K_SCALE * (0.5 + 0.5 * torch.rand((R, H), generator=g))
    vd = FP8_V_SCALE * (0.5 + 0.5 * torch.rand((R, H), generator=g))
    return kd.to(torch.float32), vd.to(torch.float32)
