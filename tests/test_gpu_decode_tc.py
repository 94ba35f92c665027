"""Decode rows on both decode kernels, against the oracle.

Decode rows ("[MRv2] FlashAttention PCP support for GQA on MRv2", overview:
mixed-batch decode next to the prefill rows) go to the tensor-core decode
kernel for head_dim 128, up to 16 q heads per kv head (8 over an FP8 cache)
and at most 1024 rows, and to the CUDA-core kernel otherwise. The tensor-core kernel walks 128-key
tiles of 2048-key splits through shared-memory rings that run on across work
items, so these cases aim at its boundaries: context lengths around the tile
and split sizes (1, 127, 128, 129, 2047, 2048, 2049 keys, ...), every block
size, every group size up to 8 and 12, 16 (padded to 1, 2, 4, 8 or 16), the FP8
cache with both converter layouts (G <= 4: K and V widened by two warp sets;
G = 8: one set), many more work items than CTAs, and a plan with more rows
than the kernel takes (the CUDA-core kernel then runs). The caches start out
NaN-filled, so a read of an unwritten slot poisons the result.
"""
import numpy as np
import pytest

import workloads as W
from pcp_case import LSE_TOL, OUT_TOL, Case

pytestmark = pytest.mark.gpu

LENGTHS = [1, 2, 127, 128, 129, 1023, 1024, 1025, 2047, 2048, 2049, 4500]


def _check(spec, kv_fp8=False, descales="layer"):
    case = Case(spec, kv_fp8=kv_fp8, descales=descales)
    out, lse = case.run()
    eo, el = case.compare(out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128])
def test_decode_lengths_every_block_size(bs):
    """Nine decode rows whose contexts end before, on and after tile and split
    boundaries, four q heads per kv head."""
    spec = W.custom_spec([1] * len(LENGTHS), LENGTHS, num_q_heads=8, num_kv_heads=2, head_dim=128,
                         block_size=bs, seed=900 + bs)
    _check(spec)


@pytest.mark.parametrize("G", [1, 2, 3, 5, 6, 7, 8, 12, 16])
def test_decode_group_sizes(G):
    """Group sizes that the kernel pads (3 -> 4, 5..7 -> 8, 12 -> 16) and the
    exact ones, beside a prefill row (16 heads: 32 P^T rows, a partial per
    softmax warpgroup)."""
    spec = W.custom_spec([1, 1, 1, 40], [700, 1030, 3, 0], num_q_heads=2 * G, num_kv_heads=2, head_dim=128,
                         seed=910 + G)
    _check(spec)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8])
def test_decode_fp8_group_sizes(G):
    """FP8 cache with a different descale per (request, kv head): G <= 4 uses two
    converter sets, G = 8 one."""
    spec = W.custom_spec([1, 1, 1, 1, 20], [1, 129, 1025, 2100, 0], num_q_heads=2 * G, num_kv_heads=2,
                         head_dim=128, seed=920 + G)
    _check(spec, kv_fp8=True, descales="varied")


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16", "fp8"])
def test_many_decode_rows(kv_fp8):
    """700 decode rows of 1 to 5000 keys: some 3500 work items, many per CTA, so
    the rings carry over from item to item."""
    rng = np.random.default_rng(931)
    p = rng.integers(1, 5001, size=700).tolist()
    spec = W.custom_spec([1] * 700, p, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=931)
    _check(spec, kv_fp8=kv_fp8)


def test_more_rows_than_the_tensor_core_kernel_takes():
    """1100 single-token requests: more rows than the tensor-core kernel's item
    table holds, so the CUDA-core decode kernel runs; same bound."""
    rng = np.random.default_rng(941)
    p = rng.integers(1, 300, size=1100).tolist()
    spec = W.custom_spec([1] * 1100, p, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=941)
    _check(spec)
