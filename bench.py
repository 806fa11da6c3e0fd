#!/usr/bin/env python3
"""Attention benchmark: prints one JSON line.

A step is one pass of the hot path over one batch of synthetic input: for the default
workload (B=4, Hq=32, Hkv=8, N=2048, d=128, bf16, causal) the forward, then the backward's
three phases (prepare, main, finish), each through the C ABI on the current stream.
`value` is attention TFLOP/s (algorithmic FLOPs: forward 4*B*Hq*N^2*d, halved when causal;
backward 2.5x the forward) with the inputs already in HBM; `e2e` is the same metric with
pinned-host inputs copied in and the results (O, dQ, dK, dV) copied out inside the timed region.

Multi-GPU (torchrun): every rank runs an independent replica of the workload on its own GPU
(weak scaling, no data-path collective); a gloo barrier brackets the timed region and the
time is the maximum over ranks.  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_bf16")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="bounded CPU-baseline sample time")
    ap.add_argument("--deterministic", action="store_true", help="backward with bitwise reproducible dQ")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other configurations timed after the default workload")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """The maximum of a host scalar over all ranks (gloo; host-side timing only)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica of the step (weak scaling)."""
    return flops_per_step * world / (ms_per_step * 1e-3) / 1e12


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                data = json.load(f)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                val = data.get(key)
                if isinstance(val, dict):
                    val = val.get("value")
                if val is not None:
                    out[key] = float(val)
            if "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                out["source"] = "measured"
                return out
        except (OSError, ValueError):
            pass
    out = dict(FALLBACK_PEAKS)
    out["source"] = "fallback"
    return out


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu_id], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file.read().splitlines() if ln.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, r[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def source_stamp() -> str:
    from exact_attention_50_gb300 import build
    return build.code_stamp()


def committed_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if the kernels have not changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    ent = data.get(kernel, {}).get(workload)
    if not ent or ent.get("source_stamp") != source_stamp():
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ CPU oracle timing

def kv_oracle_sample(wl, seconds: float, seed: int = 0):
    """The oracle's KV-cache forward over whole batches of the decode workload (all heads, the
    batch's cache) until `seconds` have passed.  Returns (TFLOP/s, description)."""
    import oracle
    from exact_attention_50_gb300 import workloads as W
    Nq = wl.extra["Nq"]
    q, k, v, cl = W.kvcache_inputs(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, wl.dtype, wl.extra["lens"], seed=seed)
    t0, flops, done = time.perf_counter(), 0.0, 0
    for b in range(wl.B):
        L = int(cl[b])
        oracle.fwd_kvcache(q[b:b + 1].double().numpy(), k[b:b + 1, :, :L].double().numpy(),
                           v[b:b + 1, :, :L].double().numpy(), [L], wl.causal, wl.scale)
        flops += W.kvcache_fwd_flops([L], wl.Hq, Nq, wl.d, wl.causal)
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, f"{done} of {wl.B} batches (all {wl.Hq} heads, their whole cache), fwd, fp64"


def oracle_sample(wl, seconds: float, seed: int = 0):
    """Times the fp64 oracle on a bounded sample of the workload: whole kv groups (all query
    heads of one kv head, one batch) forward + backward, until `seconds` have passed.  Returns
    (TFLOP/s, cores, description)."""
    import numpy as np
    import torch
    import oracle
    from exact_attention_50_gb300 import workloads as W
    oracle.build()
    oracle.set_num_threads(os.cpu_count() or 1)
    cores = oracle.num_threads()
    if wl.extra.get("cross"):  # whole kv groups of one batch: fwd (KV-cache form) + cross bwd
        Nq, G = wl.extra["Nq"], wl.G
        q, k, v, _ = W.kvcache_inputs(1, G, 1, Nq, wl.N, wl.d, wl.dtype, None, seed=seed)
        dout = torch.randn(1, G, Nq, wl.d, generator=W.generator(1)).to(q.dtype)
        qn, kn, vn, dn = (t.double().numpy() for t in (q, k, v, dout))
        per_group = W.kvcache_fwd_flops([wl.N], G, Nq, wl.d, wl.causal) * 3.5
        t0, groups = time.perf_counter(), 0
        while True:
            oracle.fwd_kvcache(qn, kn, vn, None, wl.causal, wl.scale)
            oracle.bwd_cross(qn, kn, vn, dn, wl.causal, wl.scale)
            groups += 1
            if time.perf_counter() - t0 >= seconds or groups >= wl.B * wl.Hkv:
                break
        dt = time.perf_counter() - t0
        return per_group * groups / dt / 1e12, cores, \
            f"{groups} of {wl.B * wl.Hkv} kv groups ({G} query heads, {Nq} x {wl.N}), fwd+bwd, fp64"
    if "Nq" in wl.extra:
        v_, sample = kv_oracle_sample(wl, seconds, seed)
        return v_, cores, sample
    if wl.varlen:
        qkv, cu, lengths, _ = W.varlen_inputs(wl.varlen, wl.Hq, wl.d, wl.dtype, seed=seed)
        done, flops, t0 = 0, 0.0, time.perf_counter()
        cu_l = cu.tolist()
        g = torch.Generator().manual_seed(1)
        dout = torch.randn(qkv.shape[0], wl.Hq, wl.d, generator=g).to(qkv.dtype)
        for s in np.argsort(lengths):
            a, b = cu_l[s], cu_l[s + 1]
            oracle.fwd_varlen(qkv[a:b].double().numpy(), [0, b - a], wl.causal)
            flops += W.fwd_flops(1, wl.Hq, b - a, wl.d, wl.causal)
            if wl.backward:  # the sequence as a dense [1, H, L, d] problem
                q, k, v = (qkv[a:b, i].permute(1, 0, 2).unsqueeze(0).double().numpy() for i in range(3))
                oracle.bwd(q, k, v, dout[a:b].permute(1, 0, 2).unsqueeze(0).double().numpy(), wl.causal)
                flops += W.bwd_flops(1, wl.Hq, b - a, wl.d, wl.causal)
            done += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
        what = "fwd+bwd" if wl.backward else "fwd"
        return flops / dt / 1e12, cores, f"{done} of {len(lengths)} sequences (shortest first), {what}, fp64"
    G = wl.G
    q, k, v, dout = W.dense_inputs(1, G, 1, wl.N, wl.d, wl.dtype, seed=seed)
    per_group = W.fwd_flops(1, G, wl.N, wl.d, wl.causal) * (3.5 if wl.backward else 1.0)
    if per_group > 2e11:  # a whole group would run for minutes: time sampled query rows instead
        rng = np.random.default_rng(seed)
        qn, kn, vn = (t.double().numpy() for t in (q, k, v))
        t0, flops, nrows = time.perf_counter(), 0.0, 0
        while time.perf_counter() - t0 < seconds:
            rows = np.stack([np.zeros(64, int), rng.integers(0, G, 64), rng.integers(0, wl.N, 64)], 1)
            oracle.fwd_rows(qn, kn, vn, rows, wl.causal, wl.scale)
            vis = (rows[:, 2] + 1) if wl.causal else np.full(64, wl.N)
            flops += float(np.sum(4.0 * vis * wl.d))
            nrows += 64
        dt = time.perf_counter() - t0
        return flops / dt / 1e12, cores, f"{nrows} sampled query rows (fwd only), fp64"
    qn, kn, vn, dn = (t.double().numpy() for t in (q, k, v, dout))
    t0, groups = time.perf_counter(), 0
    total_groups = wl.B * wl.Hkv
    while True:
        oracle.fwd(qn, kn, vn, wl.causal, wl.scale)
        if wl.backward:
            oracle.bwd(qn, kn, vn, dn, wl.causal, wl.scale)
        groups += 1
        if time.perf_counter() - t0 >= seconds or groups >= total_groups:
            break
    dt = time.perf_counter() - t0
    what = "fwd+bwd" if wl.backward else "fwd"
    return (per_group * groups) / dt / 1e12, cores, \
        f"{groups} of {total_groups} kv groups ({G} query heads each, N={wl.N}), {what}, fp64"


# ------------------------------------------------------------------ our arm

class Step:
    """The launches of one step of a workload through the C ABI, with its inputs resident on
    the device, and what the measurement needs to know about them."""

    def __init__(self):
        self.calls = []          # [(name, fn)] in launch order; fn returns an attn status
        self.kernels = 0         # kernels launched per step
        self.fwd_f = self.bwd_f = 0.0
        self.host_in, self.dev_in, self.dev_out = [], [], []
        self.lengths = None
        self.kv_bytes = None     # decode: algorithmic HBM bytes per step
        self.nsplit = None
        self.dom = None          # (kernel name, index of its call, its algorithmic FLOPs or bytes)


def setup_step(wl, dev, lib, sp, bwd_flags) -> Step:
    import torch
    from exact_attention_50_gb300 import workloads as W
    S = Step()
    dt_code = {"f32": 0, "f16": 1, "bf16": 2}[wl.dtype]
    scale = 0.0 if wl.scale is None else float(wl.scale)
    if wl.extra.get("cross"):
        # cross-attention: Nq queries against N keys, forward (the KV-cache call without cache
        # lengths) and backward
        Nq = wl.extra["Nq"]
        q_h, k_h, v_h, _ = W.kvcache_inputs(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, wl.dtype, None, seed=0)
        do_h = torch.randn(wl.B, wl.Hq, Nq, wl.d, generator=W.generator(1)).to(q_h.dtype)
        q, k, v, dout = q_h.to(dev), k_h.to(dev), v_h.to(dev), do_h.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(wl.B, wl.Hq, Nq, dtype=torch.float32, device=dev)
        fbytes = lib.attn_fwd_kvcache_workspace_bytes(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, 0)
        fws = torch.empty(fbytes, dtype=torch.uint8, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bbytes = lib.attn_bwd_cross_workspace_bytes(wl.B, wl.Hq, Nq, wl.N, wl.d, dt_code, bwd_flags)
        bws = torch.empty(bbytes, dtype=torch.uint8, device=dev)
        S.host_in, S.dev_in, S.dev_out = [q_h, k_h, v_h, do_h], [q, k, v, dout], [o, dq, dk, dv]
        S.calls = [("fwd_cross", lambda: lib.attn_fwd_kvcache(
                        q.data_ptr(), k.data_ptr(), v.data_ptr(), None, o.data_ptr(), lse.data_ptr(), fws.data_ptr(),
                        fbytes, wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, int(wl.causal), scale, 0, dt_code, 0, sp)),
                   ("bwd_cross", lambda: lib.attn_bwd_cross(
                       q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), bws.data_ptr(), bbytes, wl.B, wl.Hq, wl.Hkv, Nq,
                       wl.N, wl.d, int(wl.causal), scale, dt_code, bwd_flags, sp))]
        S.kernels = 2 + 3
        S.fwd_f = W.kvcache_fwd_flops([wl.N] * wl.B, wl.Hq, Nq, wl.d, wl.causal)
        S.bwd_f = 2.5 * S.fwd_f
        S.dom = ("bwd_tc_kernel", 1, S.bwd_f)
        return S
    if "Nq" in wl.extra:
        Nq = wl.extra["Nq"]
        q_h, k_h, v_h, cl_h = W.kvcache_inputs(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, wl.dtype, wl.extra["lens"],
                                               seed=0)
        S.lengths = cl_h.tolist()
        q, k, v, cl = q_h.to(dev), k_h.to(dev), v_h.to(dev), cl_h.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(wl.B, wl.Hq, Nq, dtype=torch.float32, device=dev)
        S.nsplit = lib.attn_fwd_kvcache_splits(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, 0)
        nbytes = lib.attn_fwd_kvcache_workspace_bytes(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        # a step serves one new token per sequence: its query in, its output out; the caches
        # stay resident (in the end-to-end leg too: they are the state a decoder keeps)
        S.host_in, S.dev_in, S.dev_out = [q_h], [q], [o]
        # algorithmic HBM bytes: the K and V rows of each (batch, kv head) that its queries see,
        # read once, plus Q read and O and LSE written (the split partials are not counted)
        rows = wl.B * wl.Hq * Nq
        S.kv_bytes = (sum(S.lengths) * wl.Hkv * wl.d * 2 * q_h.element_size() + 2 * rows * wl.d * q_h.element_size()
                      + rows * 4)
        S.calls = [("fwd_kvcache", lambda: lib.attn_fwd_kvcache(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), cl.data_ptr(), o.data_ptr(), lse.data_ptr(), ws.data_ptr(),
            nbytes, wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, int(wl.causal), scale, 0, dt_code, 0, sp))]
        S.kernels = 2  # the forward kernel and the split combine
        S.fwd_f = W.kvcache_fwd_flops(S.lengths, wl.Hq, Nq, wl.d, wl.causal)
        S.dom = ("fwd_tc_kernel + kv_combine_kernel", 0, S.kv_bytes)
        return S
    if wl.varlen:
        qkv_h, cu_h, lengths, _ = W.varlen_inputs(wl.varlen, wl.Hq, wl.d, wl.dtype, seed=0)
        S.lengths = lengths
        T = qkv_h.shape[0]
        qkv, cu = qkv_h.to(dev), cu_h.to(dev)
        out = torch.empty(T, wl.Hq, wl.d, dtype=qkv.dtype, device=dev)
        lse = torch.empty(wl.Hq, T, dtype=torch.float32, device=dev)
        maxlen = max(lengths)
        S.host_in, S.dev_in, S.dev_out = [qkv_h], [qkv], [out]
        S.calls = [("fwd_varlen", lambda: lib.attn_fwd_varlen(
            qkv.data_ptr(), cu.data_ptr(), len(lengths), T, maxlen, out.data_ptr(), lse.data_ptr(), wl.Hq, wl.d,
            int(wl.causal), scale, dt_code, 0, sp))]
        S.kernels = 1
        S.fwd_f = W.varlen_fwd_flops(lengths, wl.Hq, wl.d, wl.causal)
        S.dom = ("fwd_tc_kernel", 0, S.fwd_f)
        if wl.backward:
            g = torch.Generator().manual_seed(1)
            do_h = torch.randn(T, wl.Hq, wl.d, generator=g).to(qkv_h.dtype)
            dout = do_h.to(dev)
            dqkv = torch.empty_like(qkv)
            nbytes = lib.attn_bwd_varlen_workspace_bytes(T, wl.Hq, wl.d)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            S.host_in.append(do_h)
            S.dev_in.append(dout)
            S.dev_out.append(dqkv)
            S.calls.append(("bwd_varlen", lambda: lib.attn_bwd_varlen(
                qkv.data_ptr(), out.data_ptr(), dout.data_ptr(), lse.data_ptr(), cu.data_ptr(), len(lengths), T,
                maxlen, dqkv.data_ptr(), ws.data_ptr(), nbytes, wl.Hq, wl.d, int(wl.causal), scale, dt_code,
                bwd_flags, sp)))
            S.kernels += 3
            S.bwd_f = 2.5 * S.fwd_f
            # one call: its prepare and finish steps are inside the time
            S.dom = ("bwd_tc_kernel", 1, S.bwd_f)
        return S
    q_h, k_h, v_h, do_h = W.dense_inputs(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.dtype, seed=0, with_dout=wl.backward)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(wl.B, wl.Hq, wl.N, dtype=torch.float32, device=dev)
    S.host_in, S.dev_in, S.dev_out = [q_h, k_h, v_h], [q, k, v], [o]
    dims = (wl.B, wl.Hq, wl.Hkv, wl.N, wl.d)
    S.calls = [("fwd", lambda: lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                             *dims, int(wl.causal), scale, dt_code, 0, sp))]
    S.kernels = 1
    S.fwd_f = W.fwd_flops(wl.B, wl.Hq, wl.N, wl.d, wl.causal)
    S.dom = ("fwd_f32_kernel" if wl.dtype == "f32" else "fwd_tc_kernel", 0, S.fwd_f)
    if wl.backward:
        dout = do_h.to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        nbytes = lib.attn_bwd_workspace_bytes(wl.B, wl.Hq, wl.N, wl.d)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        S.host_in.append(do_h)
        S.dev_in.append(dout)
        S.dev_out += [dq, dk, dv]
        S.calls += [
            ("bwd_prepare", lambda: lib.attn_bwd_prepare(o.data_ptr(), dout.data_ptr(), ws.data_ptr(), nbytes, wl.B,
                                                         wl.Hq, wl.N, wl.d, dt_code, sp)),
            ("bwd_main", lambda: lib.attn_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                                   lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                                   ws.data_ptr(), nbytes, *dims, int(wl.causal), scale, dt_code,
                                                   bwd_flags, sp)),
            ("bwd_finish", lambda: lib.attn_bwd_finish(dq.data_ptr(), ws.data_ptr(), nbytes, wl.B, wl.Hq, wl.N, wl.d,
                                                       scale, dt_code, 0, sp)),
        ]
        S.kernels += 3
        S.bwd_f = W.bwd_flops(wl.B, wl.Hq, wl.N, wl.d, wl.causal)
        S.dom = ("bwd_tc_kernel", 2, S.bwd_f)
    return S


def run_step(S, stream, evs=None):
    from exact_attention_50_gb300 import _lib
    for i, (name, c) in enumerate(S.calls):
        if evs is not None:
            evs[i].record(stream)
        st = c()
        if st != 0:
            raise RuntimeError(f"{name} failed: {_lib.status_string(st)}")
    if evs is not None:
        evs[len(S.calls)].record(stream)


def time_steps(S, stream, K, sampler=None, barrier=lambda: None):
    """K steps bracketed by a barrier and a device synchronisation on both sides, timed with
    CUDA events on the launching stream; returns (total ms, mean ms of each call)."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(S.calls) + 1)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        run_step(S, stream, evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler is not None else None
    barrier()
    per_call = [statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
                for j in range(len(S.calls))]
    return t0.elapsed_time(t1), per_call, clocks


def choose_peak(peaks, clocks, region_s: float):
    """The dense bf16 denominator for a region: the sustained (power-capped) figure only when
    the clock record shows the power cap during a region of at least a second, else the burst
    figure of a short run at full clock."""
    capped = bool(clocks) and "sw_power_cap" in clocks.get("reasons", [])
    if capped and region_s >= 1.0:
        return peaks["bf16_tflops_sustained"], "sustained", \
            f"sw_power_cap seen during a {region_s:.2f} s timed region"
    why = "no power cap in the clock record" if not capped else f"timed region only {region_s:.3f} s"
    return peaks["bf16_tflops"], "burst", f"{why}; {region_s:.3f} s timed region"


def fp32_alu_peak(sm_count: int, sm_mhz: float) -> float:
    """fp32 CUDA-core peak in TFLOP/s: SMs x 128 fp32 lanes x 2 FLOPs per FMA x SM clock."""
    return sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12


# Configurations timed after the main workload, each on its own (a few steps, inputs resident):
# the forward-only configurations, the varlen forward, the long-context step and the fp32
# CUDA-core forward at a size that is not launch-bound.
EXTRA_WORKLOADS = ("mha_f16", "mha_f16_causal", "varlen_bf16", "long_bf16", "short_bf16", "cross_bf16", "f32_bh256")


def time_extra(name, dev, lib, stream, sp, peaks, sm_count, sm_mhz, budget_s=0.4):
    import torch
    from exact_attention_50_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    S = setup_step(wl, dev, lib, sp, 0)
    for _ in range(3):
        run_step(S, stream)
    ms1, _, _ = time_steps(S, stream, 1)
    K = int(max(3, min(50, budget_s * 1e3 / max(ms1, 1e-3))))
    ms, per_call, _ = time_steps(S, stream, K)
    st = lib.attn_get_device_status(sp)
    if st != 0:
        raise RuntimeError(f"device status after {name}: {st}")
    ent = {"workload": wl.name, "steps": K, "ms_per_step": ms / K}
    burst = peaks["bf16_tflops"]
    names = [n for n, _ in S.calls]
    if wl.dtype == "f32":
        peak = fp32_alu_peak(sm_count, sm_mhz)
        tf = S.fwd_f / (per_call[0] * 1e-3) / 1e12
        ent.update({"fwd_ms": per_call[0], "fwd_tflops": tf,
                    "roofline": {"kernel": "fwd_f32_kernel", "bound": "alu", "achieved": tf, "peak": peak,
                                 "unit": "TFLOP/s", "frac": tf / peak,
                                 "peak_source": f"derived: {sm_count} SMs x 128 fp32 lanes x 2 FLOP/FMA x "
                                                f"{sm_mhz:.0f} MHz"}})
        return ent
    tf = S.fwd_f / (per_call[0] * 1e-3) / 1e12
    ent.update({"fwd_ms": per_call[0], "fwd_tflops": tf, "fwd_frac_burst": tf / burst})
    if wl.N <= 64 and not wl.varlen and "Nq" not in wl.extra:  # the short-sequence kernel
        # the short-sequence kernel is HBM-bound: Q, K, V read and O, LSE written once
        es = 2
        nbytes = wl.B * (2 * wl.Hq + 2 * wl.Hkv) * wl.N * wl.d * es + wl.B * wl.Hq * wl.N * 4
        gbs = nbytes / (per_call[0] * 1e-3) / 1e9
        ent["roofline"] = {"kernel": "fwd_short_kernel", "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": nbytes,
                           "peak_source": f"{peaks['source']} HBM copy"}
        # the same shape on the general persistent kernel (ATTN_SHORT_KERNEL=0), for comparison
        os.environ["ATTN_SHORT_KERNEL"] = "0"
        try:
            for _ in range(3):
                run_step(S, stream)
            _, per_gen, _ = time_steps(S, stream, K)
        finally:
            del os.environ["ATTN_SHORT_KERNEL"]
        ent.update({"general_kernel_fwd_ms": per_gen[0],
                    "general_kernel_fwd_tflops": S.fwd_f / (per_gen[0] * 1e-3) / 1e12})
    if len(names) > 1:
        bwd_ms = sum(per_call[1:])
        ent.update({"bwd_ms": bwd_ms, "bwd_tflops": S.bwd_f / (bwd_ms * 1e-3) / 1e12,
                    "bwd_frac_burst": S.bwd_f / (bwd_ms * 1e-3) / 1e12 / burst,
                    "step_tflops": (S.fwd_f + S.bwd_f) / (ms / K * 1e-3) / 1e12})
    if "bwd_main" in names:
        i = names.index("bwd_main")
        main_tf = S.bwd_f / (per_call[i] * 1e-3) / 1e12
        ent.update({"bwd_main_ms": per_call[i], "bwd_main_tflops": main_tf, "bwd_main_frac_burst": main_tf / burst})
    if S.lengths is not None and wl.varlen:
        ent["total_tokens"] = sum(S.lengths)
    del S
    torch.cuda.empty_cache()
    return ent


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist
    from exact_attention_50_gb300 import _lib, build
    from exact_attention_50_gb300 import workloads as W

    build.build()
    lib = _lib.load()
    wl = W.WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    bwd_flags = _lib.ATTN_FLAG_DETERMINISTIC if args.deterministic else 0
    S = setup_step(wl, dev, lib, sp, bwd_flags)
    step_flops = S.fwd_f + S.bwd_f
    kernels_per_step, lengths, nsplit = S.kernels, S.lengths, S.nsplit

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        run_step(S, stream)
    torch.cuda.synchronize()
    st = lib.attn_get_device_status(sp)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {_lib.status_string(st)}")

    # device-resident timed region (inputs larger than L2 for the default workload)
    K = args.steps
    gpu_id = "0"
    props = torch.cuda.get_device_properties(dev)
    try:
        uuid = str(getattr(props, "uuid", ""))
        if uuid:
            gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        pass
    ms_total, per_call_ms, clocks = time_steps(S, stream, K, ClockSampler(gpu_id), barrier)
    region_s = ms_total * 1e-3
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / K
    st = lib.attn_get_device_status(sp)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {_lib.status_string(st)}")
    value = replica_throughput(step_flops, world, ms_step)

    # end to end: pinned host inputs in, results out, inside the timed region.  Two forms, both
    # through the same calls: serial (copy in, step, copy out, one stream) and pipelined (two
    # sets of device buffers; step i's inputs go up on one copy stream and step i-1's results
    # come down on another while step i-1 / i compute, ordered by per-step events).  Every step
    # still moves its own inputs and results across the link inside the timed region.
    e2e = None
    if not args.no_e2e:
        hin = [t.pin_memory() for t in S.host_in]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in S.dev_out]
        Ke = args.e2e_steps or max(3, min(K, 50))
        h2d_bytes = int(sum(t.numel() * t.element_size() for t in hin))
        d2h_bytes = int(sum(t.numel() * t.element_size() for t in hout))

        def e2e_step():
            for h, d_ in zip(hin, S.dev_in):
                d_.copy_(h, non_blocking=True)
            run_step(S, stream)
            for h, d_ in zip(hout, S.dev_out):
                h.copy_(d_, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_serial = max_over_ranks(e0.elapsed_time(e1), world) / Ke

        # pipelined: a second buffer set, an upload and a download stream
        S2 = setup_step(wl, dev, lib, sp, bwd_flags)
        sets = [S, S2]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        up_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        down_done = [torch.cuda.Event() for _ in range(2)]

        def pipelined(n, t_start=None, t_end=None):
            for i in range(n):
                k = i % 2
                St = sets[k]
                with torch.cuda.stream(up):
                    if i == 0 and t_start is not None:
                        t_start.record(up)
                    if i >= 2:
                        up.wait_event(comp_done[k])  # step i-2 has read this set's inputs
                    for h, d_ in zip(hin, St.dev_in):
                        d_.copy_(h, non_blocking=True)
                    up_done[k].record(up)
                stream.wait_event(up_done[k])
                if i >= 2:
                    stream.wait_event(down_done[k])  # step i-2's results have left this set
                run_step(St, stream)
                comp_done[k].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(comp_done[k])
                    for h, d_ in zip(hout, St.dev_out):
                        h.copy_(d_, non_blocking=True)
                    down_done[k].record(down)
            if t_end is not None:
                # the timed region ends when the last download is done (every upload and step
                # precede it)
                stream.wait_event(down_done[(n - 1) % 2])
                t_end.record(stream)

        pipelined(4)
        torch.cuda.synchronize()
        barrier()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        pipelined(Ke, p0, p1)
        torch.cuda.synchronize()
        barrier()
        ms_pipe = max_over_ranks(p0.elapsed_time(p1), world) / Ke
        st = lib.attn_get_device_status(sp)
        if st != 0:
            raise RuntimeError(f"device status after the end-to-end runs: {_lib.status_string(st)}")
        e2e = {"value": replica_throughput(step_flops, world, ms_pipe), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "ms_per_step": ms_pipe, "steps": Ke,
               "mode": "pipelined: two device buffer sets, uploads and downloads on their own streams",
               "serial": {"value": replica_throughput(step_flops, world, ms_serial), "ms_per_step": ms_serial}}
        del S2

    peaks = read_peaks()
    sm_count = props.multi_processor_count
    sm_mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
    peak, peak_kind, peak_why = choose_peak(peaks, clocks, region_s)
    burst = peaks["bf16_tflops"]
    dom_name, dom_i, dom_work = S.dom
    dom_ms = per_call_ms[dom_i]
    kv_bytes = S.kv_bytes
    if kv_bytes is not None:
        # decode streams the caches once: HBM-bound; the call's time covers the forward kernel
        # and the split combine
        gbs = kv_bytes / (dom_ms * 1e-3) / 1e9
        hbm = peaks.get("hbm_gbs")
        roofline = {"kernel": dom_name, "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4) if hbm else None,
                    "traffic": committed_traffic("fwd_tc_kernel", args.workload),
                    "algorithmic_bytes": int(kv_bytes), "peak_source": f"{peaks['source']} HBM copy"}
    elif wl.dtype == "f32":
        achieved = dom_work / (dom_ms * 1e-3) / 1e12
        alu = fp32_alu_peak(sm_count, sm_mhz)
        roofline = {"kernel": dom_name, "bound": "alu", "achieved": round(achieved, 3), "peak": round(alu, 2),
                    "unit": "TFLOP/s", "frac": round(achieved / alu, 4), "traffic": None,
                    "peak_source": f"derived: {sm_count} SMs x 128 fp32 lanes x 2 FLOP/FMA x {sm_mhz:.0f} MHz"}
    else:
        achieved = dom_work / (dom_ms * 1e-3) / 1e12
        roofline = {"kernel": dom_name, "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "frac_burst": round(achieved / burst, 4),
                    "frac_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "traffic": committed_traffic(dom_name, args.workload),
                    "peak_source": f"{peaks['source']} bf16 dense, {peak_kind} ({peak_why})"}
    fwd_ms = per_call_ms[0]
    fwd_tf = S.fwd_f / (fwd_ms * 1e-3) / 1e12
    detail = {"fwd_ms": fwd_ms, "fwd_tflops": fwd_tf}
    if wl.dtype != "f32":
        detail.update({"fwd_frac": fwd_tf / peak, "fwd_frac_burst": fwd_tf / burst, "peak_kind": peak_kind})
    names = [n for n, _ in S.calls]
    if len(names) > 1:
        bwd_ms = sum(per_call_ms[1:])
        bwd_tf = S.bwd_f / (bwd_ms * 1e-3) / 1e12
        detail.update({"bwd_ms": bwd_ms, "bwd_tflops": bwd_tf, "bwd_frac": bwd_tf / peak,
                       "bwd_frac_burst": bwd_tf / burst})
        if "bwd_main" in names:
            detail["bwd_phase_ms"] = {n.split("_", 1)[1]: per_call_ms[i] for i, n in enumerate(names) if i > 0}
            main_tf = S.bwd_f / (per_call_ms[names.index("bwd_main")] * 1e-3) / 1e12
            detail.update({"bwd_main_tflops": main_tf, "bwd_main_frac": main_tf / peak,
                           "bwd_main_frac_burst": main_tf / burst})

    line = None
    if rank == 0:
        if world == 1 and not args.no_extra and args.workload == "gqa_bf16":
            del S
            torch.cuda.empty_cache()
            detail["configs"] = {n: time_extra(n, dev, lib, stream, sp, peaks, sm_count, sm_mhz)
                                 for n in EXTRA_WORKLOADS}
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            v_, cores, sample = oracle_sample(wl, args.cpu_seconds)
            cpu = {"value": v_, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
        cfg = {"workload": wl.name, "global_batch": wl.B * world if not wl.varlen else len(lengths) * world,
               "seq_len": wl.N if not wl.varlen else max(lengths), "heads_q": wl.Hq, "heads_kv": wl.Hkv,
               "head_dim": wl.d, "causal": wl.causal, "parallelism": f"replicas x{world}",
               "l2": "inputs larger than L2 (no flush)",
               "step": "fwd + bwd (prepare, main, finish)" if len(names) > 1 else "fwd"}
        if args.deterministic:
            cfg["deterministic"] = True
        if wl.varlen:
            cfg["total_tokens"] = sum(lengths)
        if wl.extra.get("cross"):
            cfg.update({"queries": wl.extra["Nq"], "keys": wl.N, "step": "cross-attention fwd + bwd"})
        elif "Nq" in wl.extra:
            cfg.update({"queries_per_sequence": wl.extra["Nq"], "cache_capacity": wl.N,
                        "cache_tokens": sum(lengths), "num_splits": nsplit, "step": "one decode forward (forward kernel + split combine)"})
        metric = "attention TFLOP/s (fwd+bwd)" if len(names) > 1 else "attention TFLOP/s (fwd)"
        line = {"metric": metric, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
                "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded N(0,1))",
                "config": cfg, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": kernels_per_step * K, "detail": detail}
    return line


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    """The fp64 CPU oracle as the reference implementation, on rank 0 only."""
    if rank != 0:
        return None
    import numpy as np
    import oracle
    from exact_attention_50_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    oracle.build()
    oracle.set_num_threads(os.cpu_count() or 1)
    cores = oracle.num_threads()
    # one step = the oracle's fwd (+bwd) of one query head over its kv head (a slice of the
    # workload), rows sampled when a whole head would take too long
    if wl.extra.get("cross"):
        Nq, G = wl.extra["Nq"], wl.G
        q, k, v, _ = W.kvcache_inputs(1, G, 1, Nq, wl.N, wl.d, wl.dtype, None, seed=0)
        import torch
        dout = torch.randn(1, G, Nq, wl.d, generator=W.generator(1)).to(q.dtype)
        qn, kn, vn, dn = (t.double().numpy() for t in (q, k, v, dout))
        rows_per_step = 64
        rng = np.random.default_rng(0)

        def step():  # sampled query rows of one kv group, forward only
            rows = np.stack([np.zeros(rows_per_step, int), rng.integers(0, G, rows_per_step),
                             rng.integers(0, Nq, rows_per_step)], 1)
            qs = qn[:, rows[:, 1], rows[:, 2]][:, None]  # [1, 1, rows, d] as one head of queries
            oracle.fwd_kvcache(qs, kn, vn, None, False, wl.scale)
            return 4.0 * wl.d * wl.N * rows_per_step
        sample = f"{rows_per_step} sampled query rows against all {wl.N} keys per step (fwd only, unmasked), fp64"
    elif "Nq" in wl.extra:
        Nq = wl.extra["Nq"]
        q, k, v, cl = W.kvcache_inputs(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, wl.dtype, wl.extra["lens"], seed=0)
        L = int(cl.min())  # the shortest cache of the batch: one batch per step
        b = int(cl.argmin())
        qn, kn, vn = q[b:b + 1].double().numpy(), k[b:b + 1, :, :L].double().numpy(), v[b:b + 1, :, :L].double().numpy()

        def step():
            oracle.fwd_kvcache(qn, kn, vn, [L], wl.causal, wl.scale)
            return W.kvcache_fwd_flops([L], wl.Hq, Nq, wl.d, wl.causal)
        sample = f"batch {b} (all {wl.Hq} heads, cache of {L} keys) per step, fwd, fp64"
    elif wl.varlen:
        qkv, cu, lengths, _ = W.varlen_inputs(wl.varlen, wl.Hq, wl.d, wl.dtype, seed=0)
        s = int(np.argmin(lengths))
        a, b = cu.tolist()[s], cu.tolist()[s + 1]
        x = qkv[a:b].double().numpy()
        import torch
        g = torch.Generator().manual_seed(1)
        dout = torch.randn(qkv.shape[0], wl.Hq, wl.d, generator=g).to(qkv.dtype)
        qd, kd, vd = (qkv[a:b, i].permute(1, 0, 2).unsqueeze(0).double().numpy() for i in range(3))
        dd = dout[a:b].permute(1, 0, 2).unsqueeze(0).double().numpy()

        def step():
            oracle.fwd_varlen(x, [0, b - a], wl.causal)
            f = W.fwd_flops(1, wl.Hq, b - a, wl.d, wl.causal)
            if wl.backward:
                oracle.bwd(qd, kd, vd, dd, wl.causal)
                f += W.bwd_flops(1, wl.Hq, b - a, wl.d, wl.causal)
            return f
        sample = (f"sequence {s} (length {b - a}) of the varlen batch per step, "
                  f"{'fwd+bwd' if wl.backward else 'fwd'}, fp64")
    else:
        q, k, v, dout = W.dense_inputs(1, 1, 1, wl.N, wl.d, wl.dtype, seed=0)
        qn, kn, vn, dn = (t.double().numpy() for t in (q, k, v, dout))
        head_flops = W.fwd_flops(1, 1, wl.N, wl.d, wl.causal) * (3.5 if wl.backward else 1.0)
        budget = 150.0 / max(1, args.steps + max(args.warmup, 3))
        if head_flops > 3e10 * budget:  # row sample sized to the per-step budget
            rows_per_step = 64
            rng = np.random.default_rng(0)

            def step():
                rows = np.stack([np.zeros(rows_per_step, int), np.zeros(rows_per_step, int),
                                 rng.integers(0, wl.N, rows_per_step)], 1)
                oracle.fwd_rows(qn, kn, vn, rows, wl.causal, wl.scale)
                vis = (rows[:, 2] + 1) if wl.causal else np.full(rows_per_step, wl.N)
                return float(np.sum(4.0 * vis * wl.d))
            sample = f"{rows_per_step} sampled query rows of one head per step (fwd only), fp64"
        else:
            def step():
                oracle.fwd(qn, kn, vn, wl.causal, wl.scale)
                if wl.backward:
                    oracle.bwd(qn, kn, vn, dn, wl.causal, wl.scale)
                return head_flops
            sample = f"one query head (N={wl.N}, d={wl.d}) per step, {'fwd+bwd' if wl.backward else 'fwd'}, fp64"
    for _ in range(max(args.warmup, 3)):
        step()
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += step()
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    return {"impl": "reference", "metric": "attention TFLOP/s (fwd+bwd)" if wl.backward else "attention TFLOP/s (fwd)",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
            "config": {"workload": wl.name},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if args.impl == "reference":
            line = run_reference(args, rank, world)
        else:
            line = run_ours(args, rank, world, local)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
