"""Benchmark of one PCP attention step on GB300 (prints one JSON line).

A step is the whole hot path over one batch: the host row plan, its upload,
the KV-cache write of the new tokens, and attention of every row (prefill,
cached-prefix context and decode rows) through the C ABI. The default workload is the mixed prefill + decode batch (8 prompts
of U[1024,8192] tokens in 2 shard rows each plus 56 decode rows with
U[1024,16384] keys, 32 q / 8 kv heads, D=128): the one workload on which both
halves of the metric (prefill TFLOP/s and decode-row HBM GB/s) are defined,
each timed with CUDA events around its own kernel inside the step; the other
four workloads follow in "workloads".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5] [--kv-cache bf16|fp8]
    python bench.py --impl reference     # the CPU oracle on a bounded sample

``--kv-cache fp8`` runs the same step over an FP8 (e4m3) paged cache (cache
write with the layer scales, attention with per-(request, kv head) descales).

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(no data-path collective); rank 0 prints the line, value = all ranks' work /
the slowest rank's time. ``--mode pcp`` instead splits one batch over the N
ranks, one PCP shard each, with the all-gather of the new tokens' K/V.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "prefill attn TFLOP/s (% BF16 peak); decode-row HBM GB/s (% peak)"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    """Largest value of x over all ranks (identity for one rank)."""
    if ws <= 1:
        return x
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = "cuda" if backend == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int) -> None:
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


KERNEL_SOURCES = ("attn_prefill.cu", "pcp_device.cuh", "pcp_internal.h")


def _code_only(text: str) -> str:
    """Source text without // comments and blank lines (comment edits do not
    change the compiled kernel)."""
    lines = (line.split("//", 1)[0].rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash() -> str:
    """Hash of the prefill kernel's sources (code only), to tell whether a
    stored ncu traffic figure still describes the kernel being timed."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "context_prefill_attention_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload_name: str):
    """DRAM bytes per launch of the prefill kernel from the ncu capture stored in
    profiles/traffic.json, or None if it was taken on another workload or on
    other kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        e = json.load(f).get("prefill_kernel", {})
    if e.get("workload") == workload_name and e.get("source_hash") == kernel_source_hash():
        return e.get("bytes_per_launch")
    return None


def plan_work(rows: np.ndarray, hq: int, hkv: int, d: int, kv_bytes: int = 2):
    """Algorithmic work of a plan: prefill FLOPs (4 D Hq per unmasked query-key
    pair), decode FLOPs and decode bytes (K and V of every visible key once per
    kv head at kv_bytes per element, plus q, out and lse), and the cache write's
    bytes (every new token's bf16 K and V read, written at kv_bytes per element,
    plus its 8-byte slot)."""
    r = rows.astype(np.int64)
    ql, end = r[:, 3], r[:, 5]
    dec = r[:, 7] == 1
    pairs = ql * (end - ql) + ql * (ql + 1) // 2
    pre_pairs = int(pairs[~dec].sum())
    dec_keys = int(end[dec].sum())
    n_dec = int(dec.sum())
    tokens = int(ql.sum())
    return dict(prefill_flop=4.0 * d * hq * pre_pairs, decode_flop=4.0 * d * hq * dec_keys,
                decode_bytes=float(dec_keys * hkv * d * 2 * kv_bytes + n_dec * (hq * d * 2 * 2 + hq * 4)),
                write_bytes=float(tokens * (hkv * d * 2 * (2 + kv_bytes) + 8)),
                pairs=pre_pairs + dec_keys)


class ClockSampler:
    """SM clock, power and clock-event reasons while the timed steps run: read
    from NVML (ctypes, libnvidia-ml) every millisecond, so a timed region of a
    few tens of milliseconds still holds tens of samples; without NVML,
    nvidia-smi every 20 ms. Reading clocks changes no setting."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}

    def __init__(self, index: int, period_s: float = 0.001):
        self.index, self.period = index, period_s
        self.samples, self.proc, self.nvml, self.thread = [], None, None, None
        self.stop = threading.Event()
        self.source = "none"

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return None
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        return lib, h, reasons

    def _nvml_loop(self):
        import ctypes
        lib, h, reasons = self.nvml
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, ctypes.c_int(1), ctypes.byref(clk)) == 0
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            if reasons(h, ctypes.byref(rs)) != 0:
                rs.value = 0
            if ok:
                self.samples.append((float(clk.value), self.max_mhz, pw.value / 1000.0, int(rs.value)))
            time.sleep(self.period)

    def __enter__(self):
        try:
            self.nvml = self._nvml_open()
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.source = "nvml 1 ms"
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._smi_read, daemon=True)
            self.thread.start()
            self.source = "nvidia-smi 20 ms"
        except Exception:
            self.proc = None
        return self

    def _smi_read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8 and parts[0].replace(".", "").isdigit():
                bits = sum(self.REASON_BITS[n] for i, n in enumerate(names) if parts[4 + i].lower() == "active")
                mx = float(parts[1]) if parts[1].replace(".", "").isdigit() else 0.0
                self.samples.append((float(parts[0]), mx, 0.0, bits))

    def __exit__(self, *a):
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [x[0] for x in self.samples]
        reasons = sorted({n for x in self.samples for n, b in self.REASON_BITS.items() if x[3] & b})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(x[1] for x in self.samples),
                "reasons": reasons, "samples": len(self.samples), "source": self.source,
                "power_w_max": round(max(x[2] for x in self.samples), 1)}


# ---------------------------------------------------------------- GPU arm

def merge_bytes(total_q: int, hq: int, d: int) -> float:
    """Algorithmic bytes of one LSE merge of two fp32 partials [T, Hq, D] with
    their lse [Hq, T] into bf16 out and fp32 lse."""
    return float(total_q * hq * (2 * d * 4 + 2 * 4 + d * 2 + 4))


def time_lse_merge(P, total_q: int, hq: int, d: int, device: str, stream, flush, iters: int = 5):
    """pcp_lse_merge on seeded random partials of the step's [T, Hq, D] shape,
    CUDA events on the launching stream, the L2 flushed before each launch;
    returns the mean time in ms."""
    g = torch.Generator(device=device).manual_seed(7)
    oa, ob = (torch.randn((total_q, hq, d), generator=g, device=device) for _ in range(2))
    la, lb = (torch.randn((hq, total_q), generator=g, device=device) for _ in range(2))
    out = torch.empty((total_q, hq, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((hq, total_q), dtype=torch.float32, device=device)
    for _ in range(3):
        P.pcp_lse_merge(oa, la, ob, lb, out, lse, stream=stream)
    times = []
    for i in range(iters):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        P.pcp_lse_merge(oa, la, ob, lb, out, lse, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.mean(times)


def config_of(spec, n_rows: int, flags: int, kv_fp8: bool) -> dict:
    """The workload description both arms print (same keys, same values)."""
    return {"workload": spec.name + ("-fp8kv" if kv_fp8 else ""), "rows": int(n_rows), "total_q": spec.total_q,
            "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
            "block_size": spec.block_size, "num_shards": spec.num_shards, "flags": int(flags),
            "kv_cache": "fp8-e4m3" if kv_fp8 else "bf16"}


def _mk(timing: bool = True):
    return torch.cuda.Event(enable_timing=timing)


def _live_events(n: int, stream):
    """n timing events whose CUDA events exist (torch creates one at its first
    record), so that their handles can be given to the library."""
    ev = [_mk() for _ in range(n)]
    for e in ev:
        e.record(stream)
    return ev


def time_rows(P, step, q, kc, vc, bt_dev, rows_np, scale, stream, flush, iters: int = 5):
    """pcp_attn_varlen over a subset of the plan's rows (same data, same
    workspace), the L2 flushed before each call. Returns the mean ms of the
    prefill kernel and of the decode kernels (split-KV pass and merge)."""
    rows = torch.from_numpy(np.ascontiguousarray(rows_np)).to(q.device)
    T, hq = q.shape[0], q.shape[1]
    out = step.out[:T]
    lse = step.lse_buf[:T * hq].view(hq, T)

    def call():
        if step.kv_fp8:
            R = int(bt_dev.shape[0])
            P.pcp_attn_varlen_fp8kv(q, kc, vc, step.k_descale[:R], step.v_descale[:R], bt_dev, rows, scale,
                                    out=out, lse=lse, workspace=step.workspace, flags=step.flags,
                                    status=step.status, stream=stream)
        else:
            P.pcp_attn_varlen(q, kc, vc, bt_dev, rows, scale, out=out, lse=lse, workspace=step.workspace,
                              flags=step.flags, status=step.status, stream=stream)

    for _ in range(2):
        call()
    pre, dec = [], []
    for i in range(iters):
        ev = _live_events(4, stream)
        flush.fill_(i & 0xFF)
        P.pcp_set_profile_events(*ev)
        call()
        P.pcp_set_profile_events()
        torch.cuda.synchronize()
        pre.append(ev[0].elapsed_time(ev[1]))
        dec.append(ev[2].elapsed_time(ev[3]))
    step.check_status()
    return statistics.mean(pre), statistics.mean(dec)


def time_e2e(P, spec, bt, bt_dev, kc, vc, q, k, v, steps2, stream, iters: int, kernels: bool = True):
    """The step end to end from pinned host memory: each step's q, k, v and plan
    copied in, and its out and lse copied back, inside the timed region. Two
    buffer sets alternate so that step i + 1's uploads (on a copy-in stream)
    and step i - 1's downloads (on a copy-out stream) run under step i's
    kernels; the kernels stay in order on the compute stream (the cache write of
    step i + 1 after the attention of step i). With ``kernels=False`` the same
    copies run with the same stream order and no kernel: the time the host link
    alone needs for the step's bytes. Returns (ms per step, H2D bytes, D2H bytes
    per step)."""
    dev = q.device
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    host = [x.cpu().pin_memory() for x in (q, k, v)]
    bufs = [(q, k, v), tuple(torch.empty_like(x) for x in (q, k, v))]
    out_h = [torch.empty(tuple(q.shape), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lse_h = [torch.empty((spec.num_q_heads, spec.total_q), dtype=torch.float32).pin_memory() for _ in range(2)]
    ev_in = [_mk(False), _mk(False)]
    ev_comp = [_mk(False), _mk(False)]
    ev_out = [_mk(False), _mk(False)]

    def run(n, t0=None, t1=None):
        torch.cuda.synchronize()
        if t0 is not None:
            t0.record(cin)
        for i in range(n):
            b = i % 2
            st = steps2[b]
            if i >= 2:
                ev_in[b].synchronize()  # the pinned plan staging of buffer set b is free again
            st.build_plan(spec.query_len, spec.num_computed, bt)
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(ev_comp[b])  # step i - 2 has consumed buffer set b
                for d, h in zip(bufs[b], host):
                    d.copy_(h, non_blocking=True)
                st.upload_plan(cin)
                ev_in[b].record(cin)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i - 2's result has left buffer set b
            if kernels:
                st.write_cache(bufs[b][1], bufs[b][2], kc, vc, stream)
                out, lse = st.attend(bufs[b][0], kc, vc, bt_dev, spec.scale, stream)
            else:
                T = int(q.shape[0])
                out, lse = st.out[:T], st.lse_buf[:T * spec.num_q_heads].view(spec.num_q_heads, T)
            ev_comp[b].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_comp[b])
                out_h[b].copy_(out, non_blocking=True)
                lse_h[b].copy_(lse, non_blocking=True)
                ev_out[b].record(cout)
        if t1 is not None:
            cout.wait_event(ev_out[(n - 1) % 2])
            t1.record(cout)
        torch.cuda.synchronize()

    run(4)
    t0, t1 = _mk(), _mk()
    run(iters, t0, t1)
    plan = steps2[0].plan
    h2d = sum(x.numel() * x.element_size() for x in host) + plan["rows"].nbytes + plan["slot_mapping"].nbytes
    d2h = out_h[0].numel() * 2 + lse_h[0].numel() * 4
    return t0.elapsed_time(t1) / iters, int(h2d), int(d2h)


def make_step(P, spec, bt, device, flags, kv_fp8):
    return P.PcpStep(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                     block_size=spec.block_size, num_shards=spec.num_shards, split_mode=spec.split_mode,
                     max_tokens=spec.total_q, max_reqs=spec.num_reqs, max_kv_len=bt.shape[1] * spec.block_size,
                     flags=flags, device=device, kv_cache_dtype="fp8" if kv_fp8 else "bf16",
                     k_scale=W.FP8_K_SCALE, v_scale=W.FP8_V_SCALE)


def workload_line(P, workload: int, device: str, flags: int, kv_fp8: bool, flush, stream, peaks, local: int,
                  steps: int = 10):
    """Prefill TFLOP/s (attention kernel over the prefill rows), decode GB/s
    (over the decode rows, where the workload has some) and the step time of
    one more workload, with its own clock record."""
    P, spec, bt, bt_dev, kc, vc, q, k, v, step = setup(workload, device, flags, kv_fp8)
    plan = step.build_plan(spec.query_len, spec.num_computed, bt)
    rows = plan["rows"]
    kvb = 1 if kv_fp8 else 2
    work = plan_work(rows, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, kvb)
    for _ in range(3):
        step.run(q, k, v, kc, vc, bt_dev, spec.scale, stream)
    torch.cuda.synchronize()
    st = []
    with ClockSampler(local) as clocks:
        for i in range(steps):
            flush.fill_(i & 0xFF)
            e0, e1 = _mk(), _mk()
            e0.record(stream)
            step.build_plan(spec.query_len, spec.num_computed, bt)
            step.run(q, k, v, kc, vc, bt_dev, spec.scale, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            st.append(e0.elapsed_time(e1))
        dec = rows[:, 7] == 1
        out = {"name": spec.name + ("-fp8kv" if kv_fp8 else ""), "step_ms": round(statistics.mean(st), 4)}
        pms, dms = time_rows(P, step, q, kc, vc, bt_dev, rows, spec.scale, stream, flush)
        if (~dec).any():
            tf = work["prefill_flop"] / (pms * 1e-3) / 1e12
            out["prefill"] = {"tflops": round(tf, 2), "ms": round(pms, 4), "frac_bf16_peak": round(tf / peaks["bf16"], 4)}
        if dec.any():
            gbs = work["decode_bytes"] / (dms * 1e-3) / 1e9
            out["decode"] = {"gbs": round(gbs, 1), "ms": round(dms, 4), "frac_hbm_peak": round(gbs / peaks["hbm"], 4)}
    out["clocks"] = clocks.summary()
    step.check_status()
    return out


def setup(workload: int, device: str, flags: int, kv_fp8: bool = False):
    import context_prefill_attention_gb300 as P
    P.load()
    spec = W.workload_spec(workload)
    bt, nb = W.block_tables(spec)
    shape = (nb, spec.block_size, spec.num_kv_heads, spec.head_dim)
    cache_dtype = torch.uint8 if kv_fp8 else torch.bfloat16
    kc = torch.zeros(shape, dtype=cache_dtype, device=device)
    vc = torch.zeros(shape, dtype=cache_dtype, device=device)
    fp8_scales = (W.FP8_K_SCALE, W.FP8_V_SCALE) if kv_fp8 else None
    prefix = [r for r in range(spec.num_reqs) if spec.num_computed[r] > 0]
    for r in prefix:  # contexts an earlier step would have left in the cache
        P.write_positions(kc, vc, bt[r:r + 1].numpy(), [0], [W.request_tensor(spec, r, W.KIND_KP, device)],
                          [W.request_tensor(spec, r, W.KIND_VP, device)], spec.block_size,
                          fp8_scales=fp8_scales)
    q = W.packed_new_tokens(spec, W.KIND_Q, device)
    k = W.packed_new_tokens(spec, W.KIND_K, device)
    v = W.packed_new_tokens(spec, W.KIND_V, device)
    step = make_step(P, spec, bt, device, flags, kv_fp8)
    return P, spec, bt, bt.to(device), kc, vc, q, k, v, step


def run_gpu(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    kv_fp8 = args.kv_cache == "fp8"
    kvb = 1 if kv_fp8 else 2
    P, spec, bt, bt_dev, kc, vc, q, k, v, step = setup(args.workload, device, args.flags, kv_fp8)
    workload_name = spec.name + ("-fp8kv" if kv_fp8 else "")
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    peaks = load_peaks()

    def one_step(write_events=None):
        # PcpStep.run's three steps, with optional events around the cache write
        step.build_plan(spec.query_len, spec.num_computed, bt)
        step.upload_plan(stream)
        if write_events:
            write_events[0].record(stream)
        step.write_cache(k, v, kc, vc, stream)
        if write_events:
            write_events[1].record(stream)
        return step.attend(q, kc, vc, bt_dev, spec.scale, stream)

    plan = step.build_plan(spec.query_len, spec.num_computed, bt)
    rows = plan["rows"]
    work = plan_work(rows, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, kvb)
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    step.check_status()

    # ---- the timed region: exactly K steps, the L2 flushed between them
    ev = [[_mk() for _ in range(8)] for _ in range(args.steps)]
    for e in ev:
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            P.pcp_set_profile_events(ev[i][2], ev[i][3], ev[i][4], ev[i][5])
            ev[i][0].record(stream)
            one_step(ev[i][6:8])
            ev[i][1].record(stream)
        P.pcp_set_profile_events()
        torch.cuda.synchronize()
    barrier(ws)
    step.check_status()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    pre_ms = [e[2].elapsed_time(e[3]) for e in ev]        # the prefill kernel (prefill rows)
    dec_ms = [e[4].elapsed_time(e[5]) for e in ev]        # the decode kernels (decode rows)
    write_ms = [e[6].elapsed_time(e[7]) for e in ev]
    total_ms = max_over_ranks(sum(step_ms), ws)
    ms = total_ms / args.steps
    step_flop = work["prefill_flop"] + work["decode_flop"]
    value = ws * step_flop / (ms * 1e-3) / 1e12
    pre_avg = statistics.mean(pre_ms)
    achieved = work["prefill_flop"] / (pre_avg * 1e-3) / 1e12
    write_avg = statistics.mean(write_ms)
    write_gbs = work["write_bytes"] / (write_avg * 1e-3) / 1e9 if write_avg > 0 else None
    dec = rows[:, 7] == 1
    dec_line = None
    if dec.any():
        dec_avg = statistics.mean(dec_ms)
        dec_gbs = work["decode_bytes"] / (dec_avg * 1e-3) / 1e9
        dec_line = {"gbs": round(dec_gbs, 1), "ms": round(dec_avg, 4), "frac_hbm_peak": round(dec_gbs / peaks["hbm"], 4),
                    "bytes": work["decode_bytes"]}

    # ---- the same steps with the decode rows beside the prefill rows (the SMs
    # pcp_decode_sms picks from the plan); each kernel then runs on part of the
    # GPU, so the headline above keeps the sequence and this is reported apart
    beside = None
    step.decode_beside = True
    step.build_plan(spec.query_len, spec.num_computed, bt)
    if step.decode_sms > 0:
        for _ in range(args.warmup):
            one_step()
        torch.cuda.synchronize()
        ev2 = [[_mk() for _ in range(6)] for _ in range(args.steps)]
        for e in ev2:  # recorded once here so that torch accepts those the library records
            for x in e:
                x.record(stream)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            P.pcp_set_profile_events(ev2[i][2], ev2[i][3], ev2[i][4], ev2[i][5])
            ev2[i][0].record(stream)
            one_step()
            ev2[i][1].record(stream)
        P.pcp_set_profile_events()
        torch.cuda.synchronize()
        step.check_status()
        b_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev2), ws) / args.steps
        beside = {"decode_sms": step.decode_sms, "ms_per_step": round(b_ms, 4),
                  "value": round(ws * step_flop / (b_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                  "prefill_ms": round(statistics.mean(e[2].elapsed_time(e[3]) for e in ev2), 4),
                  "decode_ms": round(statistics.mean(e[4].elapsed_time(e[5]) for e in ev2), 4),
                  "timed": f"{args.steps} more steps, L2 flushed between them, decode rows on "
                           f"{step.decode_sms} SMs of a second stream beside the prefill rows "
                           "(PCP_ATTN_DECODE_SMS)"}
    step.decode_beside = False
    step.build_plan(spec.query_len, spec.num_computed, bt)

    # ---- end to end from pinned host buffers, copies overlapped with the kernels
    step2 = make_step(P, spec, bt, device, args.flags, kv_fp8)
    if kv_fp8:
        step2.k_descale.copy_(step.k_descale)
        step2.v_descale.copy_(step.v_descale)
    e2e, h2d, d2h = time_e2e(P, spec, bt, bt_dev, kc, vc, q, k, v, [step, step2], stream, max(8, args.steps))
    e2e = max_over_ranks(e2e, ws)
    copy_ms = max_over_ranks(time_e2e(P, spec, bt, bt_dev, kc, vc, q, k, v, [step, step2], stream,
                                      max(8, args.steps), kernels=False)[0], ws)
    del step2

    merge_ms = time_lse_merge(P, spec.total_q, spec.num_q_heads, spec.head_dim, device, stream, flush)
    merge_b = merge_bytes(spec.total_q, spec.num_q_heads, spec.head_dim)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded torch.randn, bf16)",
        "config": config_of(spec, rows.shape[0], args.flags, kv_fp8),
        "l2": "flushed (512 MiB write) between timed steps", "parallelism": f"replicas x{ws}",
        "prefill": {"tflops": round(achieved, 2), "ms": round(pre_avg, 4),
                    "frac_bf16_peak": round(achieved / peaks["bf16"], 4), "flop": work["prefill_flop"]},
        "decode": dec_line,
        "cache_write": {"gbs": None if write_gbs is None else round(write_gbs, 1), "ms": round(write_avg, 4),
                        "frac_hbm_peak": None if write_gbs is None else round(write_gbs / peaks["hbm"], 4),
                        "bytes": work["write_bytes"]},
        "lse_merge": {"gbs": round(merge_b / (merge_ms * 1e-3) / 1e9, 1), "ms": round(merge_ms, 4),
                      "frac_hbm_peak": round(merge_b / (merge_ms * 1e-3) / 1e9 / peaks["hbm"], 4),
                      "bytes": merge_b, "timed": "pcp_lse_merge alone on the step's [T, Hq, D] partials"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16"], 4),
                     "traffic": measured_traffic(workload_name), "kernel": "prefill_kernel",
                     "peak_source": f"{peaks['source']} bf16 burst"},
        "e2e": {"value": round(ws * step_flop / (e2e * 1e-3) / 1e12, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e, 4),
                "host_link_gbs": round((h2d + d2h) / (e2e * 1e-3) / 1e9, 1),
                "copy_only_ms": round(copy_ms, 4),
                "timed": "pinned host buffers, two buffer sets, copies on their own streams; copy_only_ms: "
                         "the same copies and stream order without the kernels"},
        "decode_beside_prefill": beside,
        "gpu_launches": args.steps * (5 + (1 if args.flags & 1 else 0)),
        "clocks": clocks.summary(),
    }
    del q, k, v, kc, vc, step
    torch.cuda.empty_cache()
    if not args.headline_only:
        others = {}
        for w in (1, 2, 3, 4, 5):
            if w == args.workload:
                continue
            others[str(w)] = workload_line(P, w, device, args.flags, kv_fp8, flush, stream, peaks, local)
            torch.cuda.empty_cache()
        line["workloads"] = others
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, bt, target_s=args.cpu_seconds, kv_fp8=kv_fp8)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_pcp(args):
    """The multi-GPU PCP step: rank i of N owns shard i of the batch's rows
    (num_shards = N), writes its own tokens' K/V, all-gathers the new tokens'
    K/V over the process group and writes the others', then attends its own
    rows (context_prefill_attention_gb300/ranks.py). The batch is fixed, so
    the scaling is strong; value = the batch's FLOPs / the slowest rank's step.
    With N = 1 the same path runs with the gather of a single rank."""
    import dataclasses
    from context_prefill_attention_gb300 import ranks as R
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        gather = R.dist_all_gather()
    else:
        gather = lambda x: [x]  # noqa: E731
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    P, spec, bt, bt_dev, kc, vc, q, k, v, _ = setup(args.workload, device, args.flags)
    spec = dataclasses.replace(spec, num_shards=ws)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    peaks = load_peaks()
    pr = R.PcpRank(rank, ws, num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                   block_size=spec.block_size, split_mode=spec.split_mode, max_tokens=spec.total_q,
                   max_reqs=spec.num_reqs, max_kv_len=bt.shape[1] * spec.block_size, gather=gather,
                   flags=args.flags, device=device)
    plan = pr.build_plan(spec.query_len, spec.num_computed, bt)
    own = torch.from_numpy(pr.own).to(device)
    q_own, k_own, v_own = q[own].contiguous(), k[own].contiguous(), v[own].contiguous()
    del q, k, v
    work = plan_work(plan["rows"], spec.num_q_heads, spec.num_kv_heads, spec.head_dim)
    mine = plan_work(pr.rows_host, spec.num_q_heads, spec.num_kv_heads, spec.head_dim)

    def one_step():
        pr.build_plan(spec.query_len, spec.num_computed, bt)
        return pr.step(q_own, k_own, v_own, kc, vc, bt_dev, spec.scale, stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    pr.check_status()
    ev = [_live_events(4, stream) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            P.pcp_set_profile_events(ev[i][2], ev[i][3])
            ev[i][0].record(stream)
            one_step()
            ev[i][1].record(stream)
        P.pcp_set_profile_events()
        torch.cuda.synchronize()
    barrier(ws)
    pr.check_status()
    ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev), ws) / args.steps
    pre_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    step_flop = work["prefill_flop"] + work["decode_flop"]
    achieved = mine["prefill_flop"] / (pre_ms * 1e-3) / 1e12 if mine["prefill_flop"] > 0 else 0.0

    # end to end: this rank's q, k, v from pinned host memory in, its out and lse back
    hq_, hk_, hv_ = (x.cpu().pin_memory() for x in (q_own, k_own, v_own))
    n_own = int(q_own.shape[0])
    out_h = torch.empty((n_own, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((spec.num_q_heads, n_own), dtype=torch.float32).pin_memory()
    e2e_ms = []
    for i in range(max(3, args.steps // 2)):
        flush.fill_(i & 0xFF)
        s0, s1 = _mk(), _mk()
        s0.record(stream)
        q_own.copy_(hq_, non_blocking=True)
        k_own.copy_(hk_, non_blocking=True)
        v_own.copy_(hv_, non_blocking=True)
        out, lse = one_step()
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        s1.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(s0.elapsed_time(s1))
    e2e = max_over_ranks(statistics.mean(e2e_ms), ws)
    h2d = sum(x.numel() * x.element_size() for x in (hq_, hk_, hv_))
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    line = {
        "metric": METRIC, "value": round(step_flop / (ms * 1e-3) / 1e12, 3), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded torch.randn, bf16)",
        "config": config_of(spec, plan["rows"].shape[0], args.flags, False),
        "l2": "flushed (512 MiB write) between timed steps", "parallelism": f"pcp x{ws} (one shard per rank)",
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16"], 4), "traffic": None, "kernel": "prefill_kernel",
                     "peak_source": f"{peaks['source']} bf16 burst", "rank": rank},
        "e2e": {"value": round(step_flop / (e2e * 1e-3) / 1e12, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e, 4)},
        "gpu_launches": args.steps * 6,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- CPU oracle

def _oracle_sample(spec, bt, target_s: float, seed: int, kv_fp8: bool = False):
    """Run the oracle on a seeded sample of the workload's query tokens, sized to
    take about target_s seconds; returns (seconds, flop of the sample, description).
    With kv_fp8 the oracle attends over its own e4m3 codes of the keys and values
    (encoded before the timed calls) with the layer-scale descales."""
    import oracle
    rows = oracle.row_plan(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size, spec.num_shards,
                           spec.split_mode)["rows"]
    q = W.packed_new_tokens(spec, W.KIND_Q)
    kfull, vfull = zip(*[W.full_kv(spec, r) for r in range(spec.num_reqs)])
    kv_off = np.cumsum([0] + [k.shape[0] for k in kfull[:-1]])
    kk, vv = torch.cat(kfull, 0), torch.cat(vfull, 0)
    if kv_fp8:
        ck = np.zeros(tuple(kk.shape), dtype=np.uint8)
        cv = np.zeros(tuple(vv.shape), dtype=np.uint8)
        slot = np.arange(kk.shape[0], dtype=np.int64)
        oracle.cache_write_fp8(kk, slot, ck, W.FP8_K_SCALE)
        oracle.cache_write_fp8(vv, slot, cv, W.FP8_V_SCALE)
        kd, vd = (x.numpy() for x in W.fp8_descales(spec, "layer"))

        def attend(tokens):
            return oracle.attention_fp8kv(rows, q, ck, cv, kv_off, kd, vd, spec.num_q_heads, spec.num_kv_heads,
                                          spec.head_dim, spec.scale, tokens)
    else:
        def attend(tokens):
            return oracle.attention(rows, q, kk, vv, kv_off, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                    spec.scale, tokens)
    rng = np.random.default_rng(seed)
    tok_rows = [(int(r[2]), int(r[3]), int(r[5])) for r in rows]   # (q_start, q_len, kv_end)
    all_tok = np.concatenate([np.arange(s, s + n) for s, n, _ in tok_rows])
    keys_of = np.concatenate([np.arange(e - n + 1, e + 1) for s, n, e in tok_rows])
    order = rng.permutation(all_tok.shape[0])
    n = 8
    while True:
        sel = order[:n]
        t0 = time.time()
        attend(all_tok[sel])
        dt = time.time() - t0
        flop = 4.0 * spec.head_dim * spec.num_q_heads * float(keys_of[sel].sum())
        if dt >= target_s * 0.5 or n >= all_tok.shape[0]:
            return dt, flop, f"{n} seeded random query tokens of {all_tok.shape[0]} (all heads)"
        n = min(all_tok.shape[0], int(n * max(2.0, min(16.0, target_s / max(dt, 1e-3)))))


def cpu_baseline(spec, bt, target_s: float = 15.0, kv_fp8: bool = False):
    import oracle
    oracle.build()
    dt, flop, desc = _oracle_sample(spec, bt, target_s, spec.seed + 99, kv_fp8)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": round(flop / dt / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc + f", fp64, {dt:.1f} s"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec = W.workload_spec(args.workload)
    bt, _ = W.block_tables(spec)
    kv_fp8 = args.kv_cache == "fp8"
    import oracle as O
    n_rows = O.row_plan(spec.query_len, spec.num_computed, bt.numpy(), spec.block_size, spec.num_shards,
                        spec.split_mode)["rows"].shape[0]
    per_step = max(1.0, args.ref_seconds / (args.steps + args.warmup))
    for i in range(args.warmup):
        _oracle_sample(spec, bt, per_step, spec.seed + 1000 + i, kv_fp8)
    tot_t, tot_f, desc = 0.0, 0.0, ""
    for i in range(args.steps):
        dt, flop, desc = _oracle_sample(spec, bt, per_step, spec.seed + 2000 + i, kv_fp8)
        tot_t += dt
        tot_f += flop
    value = tot_f / tot_t / 1e12
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded torch.randn, bf16)",
            "config": config_of(spec, n_rows, args.flags, kv_fp8),
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"per step: {desc}"},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=4)
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--kv-cache", default="bf16", choices=["bf16", "fp8"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="skip the other four workloads")
    ap.add_argument("--mode", default="replicas", choices=["replicas", "pcp"],
                    help="N GPUs: independent replicas, or one PCP shard per rank with the K/V all-gather")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.mode == "pcp":
        run_pcp(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
