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


def workload_flops(wl, lengths=None):
    from exact_attention_50_gb300 import workloads as W
    if "Nq" in wl.extra:  # KV cache: forward only, over the keys each query sees
        return W.kvcache_fwd_flops(lengths, wl.Hq, wl.extra["Nq"], wl.d, wl.causal), 0.0
    if wl.varlen:
        f = W.varlen_fwd_flops(lengths, wl.Hq, wl.d, wl.causal)
        return f, (2.5 * f if wl.backward else 0.0)
    f = W.fwd_flops(wl.B, wl.Hq, wl.N, wl.d, wl.causal)
    return f, (W.bwd_flops(wl.B, wl.Hq, wl.N, wl.d, wl.causal) if wl.backward else 0.0)


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
    dt_code = {"f32": _lib.ATTN_F32, "f16": _lib.ATTN_F16, "bf16": _lib.ATTN_BF16}[wl.dtype]
    scale = 0.0 if wl.scale is None else float(wl.scale)
    bwd_flags = _lib.ATTN_FLAG_DETERMINISTIC if args.deterministic else 0

    lengths = None
    kv_bytes = None
    if "Nq" in wl.extra:
        Nq = wl.extra["Nq"]
        q_h, k_h, v_h, cl_h = W.kvcache_inputs(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, wl.dtype, wl.extra["lens"],
                                               seed=0)
        lengths = cl_h.tolist()
        q, k, v, cl = q_h.to(dev), k_h.to(dev), v_h.to(dev), cl_h.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(wl.B, wl.Hq, Nq, dtype=torch.float32, device=dev)
        nsplit = lib.attn_fwd_kvcache_splits(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, 0)
        nbytes = lib.attn_fwd_kvcache_workspace_bytes(wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        # a step serves one new token per sequence: its query in, its output out; the caches
        # stay resident (in the end-to-end leg too: they are the state a decoder keeps)
        host_in = [q_h]
        dev_in = [q]
        dev_out = [o]
        # algorithmic HBM bytes: the K and V rows of each (batch, kv head) that its queries see,
        # read once, plus Q read and O and LSE written (the split partials are not counted)
        rows = wl.B * wl.Hq * Nq
        kv_bytes = (sum(lengths) * wl.Hkv * wl.d * 2 * q_h.element_size() + 2 * rows * wl.d * q_h.element_size()
                    + rows * 4)

        def fwd_call():
            return lib.attn_fwd_kvcache(q.data_ptr(), k.data_ptr(), v.data_ptr(), cl.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), ws.data_ptr(), nbytes, wl.B, wl.Hq, wl.Hkv, Nq, wl.N, wl.d,
                                        int(wl.causal), scale, 0, dt_code, 0, sp)
        bwd_calls = []
    elif wl.varlen:
        qkv_h, cu_h, lengths, _ = W.varlen_inputs(wl.varlen, wl.Hq, wl.d, wl.dtype, seed=0)
        T = qkv_h.shape[0]
        qkv = qkv_h.to(dev)
        cu = cu_h.to(dev)
        out = torch.empty(T, wl.Hq, wl.d, dtype=qkv.dtype, device=dev)
        lse = torch.empty(wl.Hq, T, dtype=torch.float32, device=dev)
        maxlen = max(lengths)
        host_in = [qkv_h]
        dev_in = [qkv]
        dev_out = [out]

        def fwd_call():
            return lib.attn_fwd_varlen(qkv.data_ptr(), cu.data_ptr(), len(lengths), T, maxlen, out.data_ptr(),
                                       lse.data_ptr(), wl.Hq, wl.d, int(wl.causal), scale, dt_code, 0, sp)
        bwd_calls = []
        if wl.backward:
            g = torch.Generator().manual_seed(1)
            do_h = torch.randn(T, wl.Hq, wl.d, generator=g).to(qkv_h.dtype)
            dout = do_h.to(dev)
            dqkv = torch.empty_like(qkv)
            nbytes = lib.attn_bwd_varlen_workspace_bytes(T, wl.Hq, wl.d)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            host_in.append(do_h)
            dev_in.append(dout)
            dev_out.append(dqkv)
            bwd_calls = [
                lambda: lib.attn_bwd_varlen(qkv.data_ptr(), out.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                                            cu.data_ptr(), len(lengths), T, maxlen, dqkv.data_ptr(), ws.data_ptr(),
                                            nbytes, wl.Hq, wl.d, int(wl.causal), scale, dt_code, bwd_flags, sp),
            ]
    else:
        q_h, k_h, v_h, do_h = W.dense_inputs(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.dtype, seed=0,
                                             with_dout=wl.backward)
        q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(wl.B, wl.Hq, wl.N, dtype=torch.float32, device=dev)
        host_in = [q_h, k_h, v_h]
        dev_in = [q, k, v]
        dev_out = [o]
        args_dims = (wl.B, wl.Hq, wl.Hkv, wl.N, wl.d)

        def fwd_call():
            return lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), *args_dims,
                                int(wl.causal), scale, dt_code, 0, sp)
        bwd_calls = []
        if wl.backward:
            dout = do_h.to(dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            nbytes = lib.attn_bwd_workspace_bytes(wl.B, wl.Hq, wl.N, wl.d)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            host_in.append(do_h)
            dev_in.append(dout)
            dev_out += [dq, dk, dv]
            bwd_calls = [
                lambda: lib.attn_bwd_prepare(o.data_ptr(), dout.data_ptr(), ws.data_ptr(), nbytes, wl.B, wl.Hq,
                                             wl.N, wl.d, dt_code, sp),
                lambda: lib.attn_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), nbytes,
                                          *args_dims, int(wl.causal), scale, dt_code, bwd_flags, sp),
                lambda: lib.attn_bwd_finish(dq.data_ptr(), ws.data_ptr(), nbytes, wl.B, wl.Hq, wl.N, wl.d, scale,
                                            dt_code, 0, sp),
            ]
    calls = [fwd_call] + bwd_calls
    launches_per_step = len(calls)
    kernels_per_step = launches_per_step + (1 if kv_bytes is not None else 0)  # + the split combine
    fwd_f, bwd_f = workload_flops(wl, lengths)
    step_flops = fwd_f + bwd_f

    def run_step(evs=None):
        for i, c in enumerate(calls):
            if evs is not None:
                evs[i].record(stream)
            st = c()
            if st != 0:
                raise RuntimeError(f"call {i} failed: {_lib.status_string(st)}")
        if evs is not None:
            evs[len(calls)].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        run_step()
    torch.cuda.synchronize()
    st = lib.attn_get_device_status(sp)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {_lib.status_string(st)}")

    # device-resident timed region (inputs larger than L2 for the default workload)
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(launches_per_step + 1)] for _ in range(K)]
    gpu_id = "0"
    try:
        props = torch.cuda.get_device_properties(dev)
        uuid = str(getattr(props, "uuid", ""))
        if uuid:
            gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        run_step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    ms_total = t_start.elapsed_time(t_end)
    per_call_ms = [statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
                   for j in range(launches_per_step)]
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / K
    st = lib.attn_get_device_status(sp)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {_lib.status_string(st)}")
    value = replica_throughput(step_flops, world, ms_step)

    # end to end: pinned host inputs in, results out, inside the timed region
    e2e = None
    if not args.no_e2e:
        hin = [t.pin_memory() for t in host_in]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out]
        Ke = args.e2e_steps or max(3, min(K, 50))
        for _ in range(2):
            for h, d_ in zip(hin, dev_in):
                d_.copy_(h, non_blocking=True)
            run_step()
            for h, d_ in zip(hout, dev_out):
                h.copy_(d_, non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            for h, d_ in zip(hin, dev_in):
                d_.copy_(h, non_blocking=True)
            run_step()
            for h, d_ in zip(hout, dev_out):
                h.copy_(d_, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_e = max_over_ranks(e0.elapsed_time(e1), world)
        e2e = {"value": replica_throughput(step_flops, world, ms_e / Ke), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hin)),
               "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hout)),
               "ms_per_step": ms_e / Ke, "steps": Ke}

    peaks = read_peaks()
    # dominant kernel: the backward main kernel when there is a backward, else the forward
    if len(bwd_calls) == 3:
        dom_name, dom_ms, dom_flops = "bwd_tc_kernel", per_call_ms[2], bwd_f
    elif bwd_calls:  # one call (varlen): its prepare and finish steps are inside the time
        dom_name, dom_ms, dom_flops = "bwd_tc_kernel", per_call_ms[1], bwd_f
    else:
        dom_name, dom_ms, dom_flops = "fwd_tc_kernel", per_call_ms[0], fwd_f
    peak = peaks["bf16_tflops_sustained"] if wl.dtype != "f32" else None
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    traffic = committed_traffic(dom_name, args.workload)
    roofline = {"kernel": dom_name, "bound": "tensor", "achieved": round(achieved, 2),
                "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4) if peak else None,
                "traffic": traffic, "peak_source": f"{peaks['source']} bf16 dense, sustained"}
    if kv_bytes is not None:
        # decode streams the caches once: HBM-bound; the call's time covers the forward kernel
        # and the split combine
        gbs = kv_bytes / (per_call_ms[0] * 1e-3) / 1e9
        hbm = peaks.get("hbm_gbs")
        roofline = {"kernel": "fwd_tc_kernel + kv_combine_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                    "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4) if hbm else None,
                    "traffic": committed_traffic("fwd_tc_kernel", args.workload),
                    "algorithmic_bytes": int(kv_bytes), "peak_source": f"{peaks['source']} HBM copy"}
    fwd_ms = per_call_ms[0]
    detail = {"fwd_ms": fwd_ms, "fwd_tflops": fwd_f / (fwd_ms * 1e-3) / 1e12,
              "fwd_frac": (fwd_f / (fwd_ms * 1e-3) / 1e12) / peak if peak else None}
    if bwd_calls:
        bwd_ms = sum(per_call_ms[1:])
        detail.update({"bwd_ms": bwd_ms, "bwd_tflops": bwd_f / (bwd_ms * 1e-3) / 1e12,
                       "bwd_frac": (bwd_f / (bwd_ms * 1e-3) / 1e12) / peak if peak else None})
        if len(bwd_calls) == 3:
            detail["bwd_phase_ms"] = {"prepare": per_call_ms[1], "main": per_call_ms[2], "finish": per_call_ms[3]}

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            v_, cores, sample = oracle_sample(wl, args.cpu_seconds)
            cpu = {"value": v_, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
        cfg = {"workload": wl.name, "global_batch": wl.B * world if not wl.varlen else len(lengths) * world,
               "seq_len": wl.N if not wl.varlen else max(lengths), "heads_q": wl.Hq, "heads_kv": wl.Hkv,
               "head_dim": wl.d, "causal": wl.causal, "parallelism": f"replicas x{world}",
               "l2": "inputs larger than L2 (no flush)" if not wl.varlen else "inputs larger than L2 (no flush)",
               "step": "fwd + bwd (prepare, main, finish)" if bwd_calls else "fwd"}
        if args.deterministic:
            cfg["deterministic"] = True
        if wl.varlen:
            cfg["total_tokens"] = sum(lengths)
        if kv_bytes is not None:
            cfg.update({"queries_per_sequence": wl.extra["Nq"], "cache_capacity": wl.N,
                        "cache_tokens": sum(lengths), "num_splits": nsplit,
                        "step": "one decode forward (forward kernel + split combine)"})
        line = {"metric": "attention TFLOP/s (fwd+bwd)" if bwd_calls else "attention TFLOP/s (fwd)",
                "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
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
    if "Nq" in wl.extra:
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
