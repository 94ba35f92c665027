"""Shared set-up of GPU parity cases: draw a workload, run the PCP step through
the C ABI, run the CPU oracle on the same inputs, and compare.

Tolerances (bf16 inputs, fp32 accumulation): max |out - oracle| <= 1e-2 and
max |lse - oracle| <= 1e-3, the bound the method is held to. The FP8-cache
cases keep the same bound: the oracle attends over the same e4m3 codes (its own
encoder) times the same descales, so the kernels' only extra rounding is the
fp32 product of scale and descale.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
import torch

import oracle
import workloads as W

OUT_TOL = 1e-2
LSE_TOL = 1e-3


def _pcp():
    import context_prefill_attention_gb300 as P
    P.load()
    return P


def make_caches(spec: W.WorkloadSpec, num_blocks: int, fill=float("nan"), device="cuda"):
    shape = (num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim)
    kc = torch.full(shape, fill, dtype=torch.bfloat16, device=device)
    vc = torch.full(shape, fill, dtype=torch.bfloat16, device=device)
    return kc, vc


def make_fp8_caches(spec: W.WorkloadSpec, num_blocks: int, device="cuda"):
    """uint8 caches filled with the e4m3 NaN code, so a slot the kernels should
    not read poisons the result."""
    shape = (num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim)
    return (torch.full(shape, 0x7F, dtype=torch.uint8, device=device),
            torch.full(shape, 0x7F, dtype=torch.uint8, device=device))


FP8_K_SCALE = W.FP8_K_SCALE
FP8_V_SCALE = W.FP8_V_SCALE


class Case:
    """One workload on the GPU with its CPU copies for the oracle.

    ``kv_fp8=True`` runs the FP8 cache path; ``descales="layer"`` uses the layer
    scales broadcast to (num_reqs, Hkv), ``descales="varied"`` a seeded
    different descale per (request, kv head); ``decode_beside=True`` lets the
    step run the decode rows beside the prefill rows where it picks a split. ``inputs_hook(case)`` may modify
    ``case.q``, ``case.kfull``, ``case.vfull`` before anything is written."""

    def __init__(self, spec: W.WorkloadSpec, flags: int = 0, device: str = "cuda", kv_fp8: bool = False,
                 descales: str = "layer", inputs_hook=None, decode_beside: bool = False):
        P = _pcp()
        self.spec, self.flags, self.device, self.kv_fp8 = spec, flags, device, kv_fp8
        self.bt, self.num_blocks = W.block_tables(spec)
        self.kfull, self.vfull = [], []
        for r in range(spec.num_reqs):
            k, v = W.full_kv(spec, r)
            self.kfull.append(k)
            self.vfull.append(v)
        self.q = W.packed_new_tokens(spec, W.KIND_Q)
        if inputs_hook is not None:  # a test may reshape the seeded inputs (same tensors for both sides)
            inputs_hook(self)
        P_ = spec.num_computed
        self.k_new = torch.cat([k[p:] for k, p in zip(self.kfull, P_)], 0)
        self.v_new = torch.cat([v[p:] for v, p in zip(self.vfull, P_)], 0)
        if kv_fp8:
            self.kc, self.vc = make_fp8_caches(spec, self.num_blocks, device=device)
        else:
            self.kc, self.vc = make_caches(spec, self.num_blocks, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        fp8_scales = (FP8_K_SCALE, FP8_V_SCALE) if kv_fp8 else None
        prefix = [i for i in range(spec.num_reqs) if P_[i] > 0]
        if prefix:
            P.write_positions(self.kc, self.vc, self.bt[prefix].numpy(), [0] * len(prefix),
                              [self.kfull[i][:P_[i]] for i in prefix],
                              [self.vfull[i][:P_[i]] for i in prefix], spec.block_size, status=self.status,
                              fp8_scales=fp8_scales)
        max_kv = self.bt.shape[1] * spec.block_size
        self.step = P.PcpStep(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                              head_dim=spec.head_dim, block_size=spec.block_size, num_shards=spec.num_shards,
                              split_mode=spec.split_mode, max_tokens=spec.total_q, max_reqs=spec.num_reqs,
                              max_kv_len=max_kv, flags=flags, device=device,
                              kv_cache_dtype="fp8" if kv_fp8 else "bf16", k_scale=FP8_K_SCALE,
                              v_scale=FP8_V_SCALE, decode_beside_prefill=decode_beside)
        self.k_descale = self.v_descale = None
        if kv_fp8:
            R = spec.num_reqs
            self.k_descale, self.v_descale = W.fp8_descales(spec, descales)
            self.step.k_descale[:R].copy_(self.k_descale)
            self.step.v_descale[:R].copy_(self.v_descale)
        self.plan = self.step.build_plan(spec.query_len, spec.num_computed, self.bt)
        self.bt_dev = self.bt.to(device)
        self.q_dev = self.q.to(device)
        self.k_dev = self.k_new.to(device)
        self.v_dev = self.v_new.to(device)

    def run(self):
        out, lse = self.step.run(self.q_dev, self.k_dev, self.v_dev, self.kc, self.vc, self.bt_dev,
                                 self.spec.scale)
        torch.cuda.synchronize()
        s = int(self.step.status.item()) | int(self.status.item())
        assert s == 0, f"device status {s}"
        return out, lse

    def oracle(self, tokens):
        spec = self.spec
        rows = oracle.row_plan(spec.query_len, spec.num_computed, self.bt.numpy(), spec.block_size,
                               spec.num_shards, spec.split_mode)["rows"]
        kv_off = np.cumsum([0] + [k.shape[0] for k in self.kfull[:-1]])
        if self.kv_fp8:
            ck, cv = self.oracle_fp8_codes()
            return oracle.attention_fp8kv(rows, self.q, ck, cv, kv_off, self.k_descale.numpy(),
                                          self.v_descale.numpy(), spec.num_q_heads, spec.num_kv_heads,
                                          spec.head_dim, spec.scale, tokens)
        return oracle.attention(rows, self.q, torch.cat(self.kfull, 0), torch.cat(self.vfull, 0), kv_off,
                                spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.scale, tokens)

    def oracle_fp8_codes(self):
        """Every request's key and value codes from the oracle's own encoder
        (the layer scales), back to back."""
        if getattr(self, "_codes", None) is None:
            ks, vs = [], []
            for k, v in zip(self.kfull, self.vfull):
                L, H, D = k.shape
                ck = np.zeros((L, H, D), dtype=np.uint8)
                cv = np.zeros((L, H, D), dtype=np.uint8)
                slot = np.arange(L, dtype=np.int64)
                assert oracle.cache_write_fp8(k, slot, ck, FP8_K_SCALE) == 0
                assert oracle.cache_write_fp8(v, slot, cv, FP8_V_SCALE) == 0
                ks.append(ck)
                vs.append(cv)
            self._codes = (np.concatenate(ks, 0), np.concatenate(vs, 0))
        return self._codes

    def compare(self, out, lse, tokens: Optional[Sequence[int]] = None):
        if tokens is None:
            tokens = np.arange(self.spec.total_q, dtype=np.int64)
        tokens = np.asarray(tokens, dtype=np.int64)
        ref_o, ref_l = self.oracle(tokens)
        idx = torch.from_numpy(tokens).to(out.device)
        got_o = out.index_select(0, idx).double().cpu().numpy()
        got_l = lse.index_select(1, idx).t().double().cpu().numpy()
        assert np.isfinite(got_o).all(), "non-finite output"
        err_o = float(np.abs(got_o - ref_o).max()) if got_o.size else 0.0
        finite = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(got_l), finite)
        err_l = float(np.abs(got_l[finite] - ref_l[finite]).max()) if finite.any() else 0.0
        return err_o, err_l


def shard_segments(plan_rows: np.ndarray):
    return [(int(r[2]), int(r[3])) for r in plan_rows]
