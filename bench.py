"""Benchmark of the quantised attention path on the pages' workload.

One step = one full attention call (K mean, Q/K INT8 quantisation, V E4M3 quantisation,
fused attention) over N=37810 packed tokens, H=56 heads, D=128, read as strided NHD views
of a token-major [37810, 21504] bf16 QKV buffer (synthetic, seeded; the workload of the
Sage2 call in "gb10-sage2-p0-interleave-softmax-latency.json", key q_shape).
Metric: attention TFLOPS = 4 N^2 H D / time per call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (the only other implementation of this path) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "video"
METRIC = "attention TFLOPS (4*N^2*H*D/time) and ms/call at N=37810,H=56,D=128 on 1 GB300"
UNIT = "TFLOP/s"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")
ATTN_SRC = os.path.join(ROOT, "video_diffusion_transformer_sage_gb300", "csrc", "attn_fwd.cu")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return m["bf16_tflops"], m["bf16_tflops_sustained"], m["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 200 ms; `summary()` keeps the samples taken
    between `mark_start()` and `mark_end()` (the timed region)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        import datetime
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if self.t0 is not None and not (self.t0 - 0.1 <= ts <= self.t1 + 0.1):
                    continue
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def attn_kernel_code_sha256(path: str = ATTN_SRC) -> str:
    """sha256 of the kernel code of attn_fwd.cu: the text from `namespace sage {` to the
    host-side marker (device code; the includes and the host launch code are left out)."""
    text = open(path, encoding="utf-8").read()
    i0 = text.index("namespace sage {")
    i1 = text.index("// --------------------------------------------------------------------------- host side")
    return hashlib.sha256(text[i0:i1].encode()).hexdigest()


def _traffic_per_launch():
    """dram bytes per launch of the attention kernel from the committed ncu capture, or None
    when the kernel code changed since the capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("attn_kernel_code_sha256") != attn_kernel_code_sha256():
            return None
        return t["bytes_per_launch_full_size"]
    except Exception:
        return None


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, pg, device=None) -> float:
    """Max of a per-rank float over the process group (the slowest rank's time)."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs `steps` calls of `flops_per_step`; the job takes the
    slowest rank's time."""
    return world * flops_per_step * steps / (max_ms * 1e-3) / 1e12


def run_gpu(args):
    import torch
    import video_diffusion_transformer_sage_gb300 as sage
    from video_diffusion_transformer_sage_gb300 import build as sbuild, synth

    world, rank, local = _dist()
    sbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist

    w = synth.WORKLOADS[args.workload]
    n, h, d = w.n_tokens, w.n_heads, w.head_dim
    inp = synth.make_inputs(w)
    host = inp.storage.pin_memory()
    storage = host.to(dev)
    hd = h * d

    def views(buf):
        if w.layout == "hnd":          # [3, H, N, D] -> three [N, H, D] views
            return [buf[i].transpose(0, 1) for i in range(3)]
        if w.layout == "nhd":          # [3, N, H, D] -> three contiguous [N, H, D] tensors
            return [buf[i] for i in range(3)]
        return [buf[:, i * hd:(i + 1) * hd].view(n, h, d) for i in range(3)]

    q, k, v = views(storage)
    sm_scale = 1.0 / math.sqrt(d)
    # The timed path: the method's default (E4M3 V and P), or one of its V options.
    default_path = args.v_format == "e4m3" and not args.smooth_v
    qz = sage.Quantized(n, h, d, dev, v_format=args.v_format, smooth_v=args.smooth_v)
    scratch = sage.quant_scratch(n, h, d, dev)
    scratch2 = torch.empty(2 * scratch.numel(), dtype=torch.uint8, device=dev)   # sage_quant_qkv's
    status = sage.status_block(dev)
    out = torch.empty((n, h, d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    # sage_quant_qkv: colreduce (K sums and V maxima), colfinal (K mean and V scales), quant_qk,
    # quant_v, quant_v_fixup; then the attention.  With a V option it runs the two stage calls:
    # colreduce+colfinal (K), quant_qk, colreduce+colfinal (V), quant_v, quant_v_fixup, and V
    # smoothing adds colreduce+colfinal for the V mean.
    launches_per_step = 6 if default_path else 8 + (2 if args.smooth_v else 0)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        sage.sage_quant_qkv(q, k, v, qz, scratch2, stream)
        if ev is not None:
            ev[1].record(stream)
        sage.sage_attn_fwd_quantized(qz, sm_scale, out, status, stream)
        if ev is not None:
            ev[2].record(stream)

    with ClockSampler(local) as clk:
        time.sleep(1.0)                      # let the sampler start before the timed region
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        clk.mark_start()
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    if pg:
        pg.barrier()
    code, where = sage.sage_check_device_status(status, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} at {where}")
    total_ms = reduce_max(t0.elapsed_time(t1), pg, dev)
    quant_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    ms_per_step = total_ms / args.steps
    flops = w.flops
    value = job_throughput(flops, args.steps, world, total_ms)

    # ---- end to end through the C ABI with host buffers.  Every step copies its QKV input
    # from pinned host memory (H2D), runs the whole path (sage_attn_fwd) and copies the
    # output back to pinned host memory (D2H).  Copies run on their own streams, double
    # buffered, so step i's compute overlaps step i+1's H2D and step i-1's D2H -- a serving
    # loop.  The serial variant (copy, compute, copy, in order) is reported beside it.
    # e2e and the per-call distribution time the public whole-path call (sage_attn_fwd), which
    # runs the default path: skipped when a V option is timed.
    e2e_steps = 0 if (args.no_e2e or not default_path) else max(3, args.steps)
    e2e_ms = e2e_serial_ms = float("nan")
    e2e_runs = []
    e2e_timeline = None
    host_out = [torch.empty((n, h, d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    if e2e_steps:
        ws = sage.workspace(n, h, d, dev)
        bufs = [torch.empty_like(storage) for _ in range(2)]
        outs = [torch.empty((n, h, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        comp = torch.cuda.current_stream(dev)

        def run(steps, pipelined, timeline=None):
            # The H2D of step i+1 is enqueued before the D2H of step i: a D2H waits for its
            # step's compute, and if both copy streams share one copy engine, a prefetch
            # queued behind it would wait for that compute too (measured: 29-30 ms per step
            # instead of 23.8 on some runs).  With `timeline` (a list), every copy and every call
            # is bracketed by timing events and its [start, end] in ms from the run's start is
            # appended, per step, as (h2d, compute, d2h).
            T = timeline is not None

            def ev():
                return torch.cuda.Event(enable_timing=T)

            ev_in = [ev() for _ in range(steps)]
            ev_done = [ev() for _ in range(steps)]
            ev_out = [ev() for _ in range(steps)]
            st_in = [ev() for _ in range(steps)]
            st_comp = [ev() for _ in range(steps)]
            st_out = [ev() for _ in range(steps)]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            sin = s_in if pipelined else comp
            sout = s_out if pipelined else comp
            torch.cuda.synchronize()
            a.record(comp)
            sin.wait_event(a)
            if T:
                st_in[0].record(sin)
            with torch.cuda.stream(sin):
                bufs[0].copy_(host, non_blocking=True)
            ev_in[0].record(sin)
            for i in range(steps):
                k_ = i % 2
                comp.wait_event(ev_in[i])
                if i >= 2:
                    comp.wait_event(ev_out[i - 2])      # D2H of step i-2 released output k_
                if T:
                    st_comp[i].record(comp)
                qv, kv, vv = views(bufs[k_])
                sage.sage_attn_fwd(qv, kv, vv, sm_scale, outs[k_], ws, comp)
                ev_done[i].record(comp)
                if i + 1 < steps:
                    if i >= 1:
                        sin.wait_event(ev_done[i - 1])  # compute of step i-1 released buffer (i+1)%2
                    if T:
                        st_in[i + 1].record(sin)
                    with torch.cuda.stream(sin):
                        bufs[(i + 1) % 2].copy_(host, non_blocking=True)
                    ev_in[i + 1].record(sin)
                sout.wait_event(ev_done[i])
                if T:
                    st_out[i].record(sout)
                with torch.cuda.stream(sout):
                    host_out[k_].copy_(outs[k_], non_blocking=True)
                ev_out[i].record(sout)
            comp.wait_event(ev_out[steps - 1])
            b.record(comp)
            torch.cuda.synchronize()
            if T:
                for i in range(steps):
                    timeline.append(tuple((a.elapsed_time(x), a.elapsed_time(y)) for x, y in
                                          ((st_in[i], ev_in[i]), (st_comp[i], ev_done[i]), (st_out[i], ev_out[i]))))
            return a.elapsed_time(b) / steps

        def overlap_summary(tl):
            """Mean copy and call durations, the share of each copy's time that a call overlaps, and
            the mean idle gap of the compute stream between calls (ms)."""
            def inter(x, y):
                return max(0.0, min(x[1], y[1]) - max(x[0], y[0]))
            comps = [t[1] for t in tl]
            out = {}
            for name, idx in (("h2d", 0), ("d2h", 2)):
                ivs = [t[idx] for t in tl]
                dur = [y - x for x, y in ivs]
                ov = [sum(inter(iv, c) for c in comps) for iv in ivs]
                out[f"{name}_ms"] = round(statistics.mean(dur), 3)
                out[f"{name}_overlapped_by_compute"] = round(sum(ov) / max(sum(dur), 1e-9), 3)
            out["compute_ms"] = round(statistics.mean(c[1] - c[0] for c in comps), 3)
            gaps = [comps[i][0] - comps[i - 1][1] for i in range(1, len(comps))]
            out["compute_idle_gap_ms"] = round(statistics.mean(gaps), 3) if gaps else 0.0
            return out

        run(2, True)
        # The overlap of copies with compute varies from run to run on these boxes (23.8 or
        # 26.3-30 ms per step for the same code): three runs, the median reported, all listed,
        # each with every copy and call bracketed by events so that a slow run shows where its
        # time went.
        e2e_runs, e2e_timeline = [], []
        for _ in range(3):
            tl = []
            e2e_runs.append(run(e2e_steps, True, tl))
            e2e_timeline.append(dict(overlap_summary(tl), ms_per_step=round(e2e_runs[-1], 3)))
        e2e_ms = reduce_max(statistics.median(e2e_runs), pg, dev)
        e2e_serial_ms = run(e2e_steps, False)

    # ---- per-call distribution of the public call, in the pages' protocol: after the warm-up
    # above, 5 rounds x 10 calls of sage_attn_fwd (steps a1-a8 from the strided views), each
    # call bracketed by its own CUDA events on the launching stream.
    call_timing = None
    if not args.no_call_timing and default_path:
        ws_c = sage.workspace(n, h, d, dev)
        rounds = []
        for _ in range(5):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
            torch.cuda.synchronize()
            for a_, b_ in ev:
                a_.record(stream)
                sage.sage_attn_fwd(q, k, v, sm_scale, out, ws_c, stream)
                b_.record(stream)
            torch.cuda.synchronize()
            rounds.append([a_.elapsed_time(b_) for a_, b_ in ev])
        code, where = sage.sage_check_device_status(ws_c[:256], stream)
        if code != 0:
            raise RuntimeError(f"device status {code} at {where}")
        call_timing = call_stats(rounds)

    # ---- the qk_transform stage upstream of the path (in-place RMSNorm + rotary embedding of
    # Q and K), timed on its own on a copy of the QKV buffer: 3 warm-up calls, then 20 calls,
    # CUDA events per call.  Algorithmic bytes: Q and K read and written once (8 N H D) plus
    # the fp32 cos / sin table (4 N D).
    qk_transform = None
    if not args.no_qk_transform and w.layout == "qkv":
        gq, gk = synth.qk_norm_weights(d)
        cos, sin = synth.rope_table(synth.rope_positions(n), d)
        gq, gk, cos, sin = (t_.to(dev) for t_ in (gq, gk, cos, sin))
        buf = storage.clone()
        tq, tk, _ = views(buf)
        for _ in range(3):
            sage.sage_qk_rmsnorm_rope(tq, tk, gq, gk, cos, sin, 1e-6, stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
        torch.cuda.synchronize()
        for a_, b_ in ev:
            a_.record(stream)
            sage.sage_qk_rmsnorm_rope(tq, tk, gq, gk, cos, sin, 1e-6, stream)
            b_.record(stream)
        torch.cuda.synchronize()
        t_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in ev)
        t_bytes = 8 * n * h * d + 4 * n * d
        kname = ("rmsnorm_rope_bulk_kernel<%d>" if tq.stride(1) == d and tk.stride(1) == d
                 else "rmsnorm_rope_kernel<%d>") % d
        qk_transform = {"kernel": kname, "ms": round(t_ms, 4), "bytes": t_bytes,
                        "gbs": round(t_bytes / (t_ms * 1e-3) / 1e9, 1), "calls": 20}

        # The same transform fused into the K mean and the Q / K quantisation
        # (sage_smooth_quant_qk_rmsnorm_rope: Q and K only read), against the unfused pair
        # (the in-place transform, then sage_smooth_quant_qk) on the same data; 3 warm-up calls,
        # then 20 calls each, CUDA events per call.  Bytes of the fused call: K read once and its
        # transformed rows written and read back (6 N H D), Q read once (2 N H D), fp16 codes
        # written (4 N H D), the table (4 N D).
        fz = sage.Quantized(n, h, d, dev)

        def timed(fn, calls=20):
            for _ in range(3):
                fn()
            evp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
            torch.cuda.synchronize()
            for a_, b_ in evp:
                a_.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize()
            return statistics.mean(a_.elapsed_time(b_) for a_, b_ in evp)

        fused_ms = timed(lambda: sage.sage_smooth_quant_qk_rmsnorm_rope(q, k, gq, gk, cos, sin, 1e-6, fz, scratch,
                                                                        stream))
        pair_ms = timed(lambda: (sage.sage_qk_rmsnorm_rope(tq, tk, gq, gk, cos, sin, 1e-6, stream),
                                 sage.sage_smooth_quant_qk(tq, tk, fz, scratch, stream)))
        f_bytes = 12 * n * h * d + 4 * n * d
        qk_transform["fused_with_quantise"] = {
            "call": "sage_smooth_quant_qk_rmsnorm_rope", "ms": round(fused_ms, 4), "bytes": f_bytes,
            "gbs": round(f_bytes / (fused_ms * 1e-3) / 1e9, 1), "unfused_pair_ms": round(pair_ms, 4),
            "saved_ms": round(pair_ms - fused_ms, 4)}
        del buf, fz

    # ---- the V options of the path at the same size and inputs, outside the timed region: the
    # INT8 P.V variant (INT8 V, P = rint(127 p), fp16-code MMAs) and V smoothing (the channel
    # mean taken out of V, added back in the epilogue).  3 warm-up steps, then 10 steps with
    # CUDA events around the quantisation (Q, K and V) and around the attention launch.
    variants = None
    if not args.no_variants:
        variants = {}
        for vname, fmt, smooth in (("int8_pv", "int8", False), ("e4m3_smooth_v", "e4m3", True),
                                   ("int8_pv_smooth_v", "int8", True)):
            vz = sage.Quantized(n, h, d, dev, v_format=fmt, smooth_v=smooth)
            vev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(10)]
            for i in range(13):
                e_ = vev[i - 3] if i >= 3 else None
                if e_ is not None:
                    e_[0].record(stream)
                sage.sage_smooth_quant_qk(q, k, vz, scratch, stream)
                sage.sage_quant_v(v, vz, scratch, stream)
                if e_ is not None:
                    e_[1].record(stream)
                sage.sage_attn_fwd_quantized(vz, sm_scale, out, status, stream)
                if e_ is not None:
                    e_[2].record(stream)
            torch.cuda.synchronize()
            code, where = sage.sage_check_device_status(status, stream)
            if code != 0:
                raise RuntimeError(f"device status {code} at {where} ({vname})")
            v_attn = statistics.mean(e_[1].elapsed_time(e_[2]) for e_ in vev)
            v_quant = statistics.mean(e_[0].elapsed_time(e_[1]) for e_ in vev)
            variants[vname] = {"quantise_ms": round(v_quant, 4), "attention_ms": round(v_attn, 3),
                               "attention_tflops": round(flops / (v_attn * 1e-3) / 1e12, 1),
                               "step_ms": round(v_quant + v_attn, 3)}
            del vz

    # ---- unquantised attention on the tensor cores (sage_attn_dense_bf16_tc: bf16 operands, P
    # rounded to bf16; V's transpose and the attention, 2 launches) at the same size and inputs,
    # outside the timed region: 3 warm-up calls, then 10 calls with CUDA events around each.
    dense_tc = None
    if not args.no_variants:
        dz_out = torch.empty((n, h, d), dtype=torch.bfloat16, device=dev)
        dz_ws = sage.dense_workspace(n, h, d, dev)
        for _ in range(3):
            sage.sage_attn_dense_bf16_tc(q, k, v, sm_scale, dz_out, dz_ws, stream)
        dev_ = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
        torch.cuda.synchronize()
        for a_, b_ in dev_:
            a_.record(stream)
            sage.sage_attn_dense_bf16_tc(q, k, v, sm_scale, dz_out, dz_ws, stream)
            b_.record(stream)
        torch.cuda.synchronize()
        code, where = sage.sage_check_device_status(dz_ws[:256], stream)
        if code != 0:
            raise RuntimeError(f"device status {code} at {where} (dense_tc)")
        dt_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in dev_)
        dense_tc = {"call": "sage_attn_dense_bf16_tc", "ms": round(dt_ms, 3),
                    "tflops": round(flops / (dt_ms * 1e-3) / 1e12, 1), "launches": 2,
                    "quantised_call_speedup": round(dt_ms / ms_per_step, 3)}
        del dz_out, dz_ws

    # ---- the dense quality anchor (sage_attn_dense_bf16: unquantised, fp32 arithmetic on CUDA
    # cores), timed once after one warm-up call, beside the pages' dense figure -- context only.
    dense = None
    if args.dense_anchor:
        dense_out = torch.empty((n, h, d), dtype=torch.bfloat16, device=dev)
        sage.sage_attn_dense_bf16(q, k, v, sm_scale, dense_out, stream)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a_.record(stream)
        sage.sage_attn_dense_bf16(q, k, v, sm_scale, dense_out, stream)
        b_.record(stream)
        torch.cuda.synchronize()
        d_ms = a_.elapsed_time(b_)
        dense = {"call": "sage_attn_dense_bf16", "ms": round(d_ms, 3),
                 "tflops": round(w.flops / (d_ms * 1e-3) / 1e12, 2),
                 "note": "CUDA-core fp32 correctness path; the pages' dense attention took 947.9 ms at N=37810"}
        del dense_out

    # ---- the measured tensor-core ceiling of the attention kernel's instructions (outside the
    # timed region): one CTA per SM issuing each MMA shape back to back on resident operands
    # (sage_measure_mma_rate), 1 warm-up launch, then 3 timed launches per mode with CUDA events.
    mma_ceiling = None if args.no_mma_ceiling else mma_rates(sage, dev, stream, status)

    bf16_burst, bf16_sus, hbm, peak_src = _peaks()
    if qk_transform is not None:
        qk_transform["hbm_frac"] = round(qk_transform["gbs"] / hbm, 4)
        qk_transform["fused_with_quantise"]["hbm_frac"] = round(qk_transform["fused_with_quantise"]["gbs"] / hbm, 4)
    # The fused kernel does half its FLOPs as fp16 MMAs (QK^T on INT8 codes held in fp16)
    # and half as E4M3 MMAs (PV); the E4M3 rate is twice the 16-bit rate.  Its roofline is
    # the time of both halves at their own peaks.  The burst bf16 figure applies when the
    # timed loop ran at full SM clock without a power cap (as the burst GEMM did); the
    # sustained figure (a GEMM held under the power cap, at lower clocks) otherwise.  A loop
    # shorter than the sampler's period leaves no sample; such a short burst is held to the
    # burst figure too (the larger, so the stricter, denominator).
    clocks = clk.summary()
    full_clock = (clocks.get("sm_mhz") is None
                  or (clocks["sm_mhz"] >= 0.97 * clocks["sm_max_mhz"] and "sw_power_cap" not in clocks["reasons"]))
    p16 = bf16_burst if full_clock else bf16_sus
    p8 = 2 * p16
    composite = 1.0 / (0.5 / p16 + 0.5 / p8)
    for vname, vv_ in (variants or {}).items():
        # INT8 P.V runs both contractions on fp16 operands, so the 16-bit peak is its roofline;
        # the E4M3 variant has the default path's composite roofline.
        vv_["roofline_frac"] = round(vv_["attention_tflops"] / (p16 if vname.startswith("int8") else composite), 4)
    if dense_tc is not None:
        # Both contractions on bf16 operands: the bf16 peak bounds it.
        dense_tc["roofline_frac_of_bf16_peak"] = round(dense_tc["tflops"] / p16, 4)
    attn_avg = statistics.mean(attn_ms)
    achieved = flops / (attn_avg * 1e-3) / 1e12
    # INT8 P.V runs both contractions on 16-bit operands: the bf16 peak is its roofline.
    attn_peak = p16 if args.v_format == "int8" else composite
    kname = "attn_fwd_kernel<%d, false, %s, %s>" % (d, "true" if args.v_format == "int8" else "false",
                                                    "true" if args.smooth_v else "false")
    # The measured ceiling of the kernel's own MMA mix: one key tile of one Q tile at its D.
    mix_mode = ("qk_pv_tile_mix" if d == 128 else "qk_pv_tile_mix_d64") if args.v_format == "e4m3" \
        else "qk_f16_128x128x16"
    traffic = _traffic_per_launch()
    quant_avg = statistics.mean(quant_ms)
    quant_bytes = 13 * n * h * d
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": ("fp16(int8 codes)xfp16 + fp16(int8 codes)xfp16 -> fp32, bf16 io" if args.v_format == "int8"
                                        else "fp16(int8 codes)xfp16 + e4m3xe4m3 -> fp32, bf16 io"),
        "data": "synthetic (seeded, distributions of the pages' workload)",
        "config": {"workload": f"{w.name}: N={n}, H={h}, D={d}, batch 1, non-causal, " + (
                               "HND-contiguous bf16 Q, K, V" if w.layout == "hnd" else
                               "contiguous NHD bf16 Q, K, V" if w.layout == "nhd" else
                               f"strided NHD views of a [{n}, {3 * h * d}] bf16 QKV buffer"),
                   "path": ("INT8 P.V (INT8 V, P = rint(127 p))" if args.v_format == "int8" else
                            "E4M3 V and P") + (", V mean smoothing" if args.smooth_v else ""),
                   "l2": (f"inputs larger than L2 ({host.numel() * 2 / 1e9:.2f} GB QKV buffer)"
                          if host.numel() * 2 > 129e6 else
                          f"inputs ({host.numel() * 2 / 1e6:.0f} MB) fit in L2: a small parity case, not a bench line"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(attn_peak, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / attn_peak, 4),
                     "traffic": traffic if default_path else None,
                     "kernel": kname,
                     "peak_note": (f"the {peak_src} {'burst' if full_clock else 'sustained'} bf16 {p16} TFLOP/s "
                                   "(both contractions on fp16 operands)" if args.v_format == "int8" else
                                   f"composite of the {peak_src} {'burst' if full_clock else 'sustained'} bf16 "
                                   f"{p16} TFLOP/s (QK^T, fp16 operands) and 2x that for E4M3 (PV)"),
                     "frac_of_e4m3_peak": round(achieved / p8, 4),
                     "frac_of_bf16_peak": round(achieved / p16, 4),
                     "frac_of_mma_ceiling": (round(achieved / mma_ceiling["tflops"][mix_mode], 4)
                                             if mma_ceiling else None),
                     "mma_ceiling_mode": mix_mode,
                     # against the measured dense E4M3 (kind::f8f6f4) instruction rate, 128x256x32
                     # from shared memory: what the whole contraction would take at the FP8 rate
                     "frac_of_measured_e4m3_rate": (round(achieved / mma_ceiling["tflops"]["e4m3_ss_128x256x32"], 4)
                                                    if mma_ceiling else None)},
        "mma_ceiling": mma_ceiling,
        "dense_anchor": dense,
        "dense_tc": dense_tc,
        "kernels_ms": {"quantise_all_avg": round(quant_avg, 4), "attention_avg": round(attn_avg, 3),
                       "quantise_gbs_algorithmic": round(quant_bytes / (quant_avg * 1e-3) / 1e9, 1),
                       "quantise_hbm_frac": round(quant_bytes / (quant_avg * 1e-3) / 1e9 / hbm, 4)},
        "e2e": {"value": (round(job_throughput(flops, 1, world, e2e_ms), 2) if e2e_steps else None), "unit": UNIT,
                "h2d_bytes_per_step": int(host.numel() * 2), "d2h_bytes_per_step": int(host_out[0].numel() * 2),
                "ms_per_step": round(e2e_ms, 3) if e2e_steps else None, "steps": e2e_steps,
                "how": "pinned host QKV -> H2D, sage_attn_fwd, D2H -> pinned host each step; copies on their own "
                       "streams, double-buffered (step i overlaps H2D of i+1 and D2H of i-1; the H2D of i+1 "
                       "is enqueued before the D2H of i)",
                "serial_ms_per_step": round(e2e_serial_ms, 3) if e2e_steps else None,
                "pipelined_runs_ms": [round(x, 3) for x in e2e_runs] if e2e_steps else [],
                "timeline": e2e_timeline},
        "call_timing": call_timing,
        "qk_transform": qk_transform,
        "variants": variants,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, budget_s=args.cpu_budget, v_format=args.v_format,
                                            smooth_v=args.smooth_v)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


MMA_MODES = {0: "qk_f16_128x128x16", 1: "pv_e4m3_tmemA_128x128x32", 2: "qk_pv_tile_mix",
             3: "e4m3_ss_128x256x32", 4: "f16_ss_128x256x16", 5: "pv_e4m3_tmemA_128x64x32",
             6: "qk_pv_tile_mix_d64"}
# rounds per launch: about 10-20 ms each at the nominal per-SM rates (8192 fp16 / 16384 E4M3 FLOP per clock)
MMA_ITERS = {0: 80000, 1: 80000, 2: 54000, 3: 40000, 4: 40000, 5: 80000, 6: 80000}


def mma_rates(sage, dev, stream, status):
    """TFLOP/s of each sage_measure_mma_rate mode with one CTA per SM."""
    import torch
    from video_diffusion_transformer_sage_gb300 import _lib
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for mode, name in MMA_MODES.items():
        sage.sage_measure_mma_rate(mode, MMA_ITERS[mode] // 10, sms, status, stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
        torch.cuda.synchronize()
        for a_, b_ in ev:
            a_.record(stream)
            sage.sage_measure_mma_rate(mode, MMA_ITERS[mode], sms, status, stream)
            b_.record(stream)
        torch.cuda.synchronize()
        ms = min(a_.elapsed_time(b_) for a_, b_ in ev)
        out[name] = round(_lib.MMA_RATE_FLOPS[mode] * MMA_ITERS[mode] * sms / (ms * 1e-3) / 1e12, 1)
    code, where = sage.sage_check_device_status(status, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} at {where} (MMA rate)")
    return {"tflops": out, "ctas": sms, "how": "one CTA per SM issuing each tcgen05.mma shape back to back on "
            "resident zero operands (sage_measure_mma_rate); best of 3 launches of ~20 ms"}


def _pct(xs, q):
    """Linear-interpolated percentile q (0..100) of the sorted list xs."""
    xs = sorted(xs)
    if len(xs) == 1:
        return xs[0]
    pos = (len(xs) - 1) * q / 100.0
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(xs) - 1)
    return xs[lo] + (xs[hi] - xs[lo]) * (pos - lo)


def call_stats(rounds):
    """Distribution of per-call times (ms) over all rounds, plus each round's mean."""
    xs = [x for r in rounds for x in r]
    st = {"count": len(xs), "unit": "ms", "mean": statistics.mean(xs)}
    for q in (50, 90, 95, 99):
        st[f"p{q}"] = _pct(xs, q)
    st["min"], st["max"] = min(xs), max(xs)
    st = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in st.items()}
    st["round_means"] = [round(statistics.mean(r), 4) for r in rounds]
    st["protocol"] = "3 warm-up calls, then 5 rounds x 10 calls of sage_attn_fwd, CUDA events per call"
    return st


def cpu_baseline(inp, budget_s: float = 20.0, rows_per_step: int = 8, steps: int = 0, v_format: str = "e4m3",
                 smooth_v: bool = False):
    """The oracle as it stands on the host cores: quantisation (steps 1-4) in full, then
    same-quantisation attention for sampled query rows (all heads) until `budget_s` is spent;
    time per call extrapolated as t_quant + N * t_row.  v_format / smooth_v: the path timed."""
    import oracle
    w = inp.workload
    n, h, d = w.n_tokens, w.n_heads, w.head_dim
    t = time.perf_counter()
    qz = oracle.Quantized(inp.q, inp.k, inp.v, v_format=v_format, smooth_v=smooth_v)
    t_quant = time.perf_counter() - t
    from video_diffusion_transformer_sage_gb300 import synth
    pool = synth.sample_rows(n, 4096, 17)
    done, t_attn, i = 0, 0.0, 0
    while (steps and i < steps) or (not steps and (t_attn < budget_s or done == 0)):
        rows = [pool[(i * rows_per_step + r) % len(pool)] for r in range(rows_per_step)]
        t = time.perf_counter()
        oracle.attn_sq(qz, 1.0 / math.sqrt(d), rows, tile=128)
        t_attn += time.perf_counter() - t
        done += rows_per_step
        i += 1
    t_row = t_attn / done
    t_call = t_quant + n * t_row
    return {"value": round(w.flops / t_call / 1e12, 5), "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"quantisation in full ({t_quant:.1f} s); attention for {done} sampled query "
                                        f"rows x {h} heads ({t_attn:.1f} s); call time extrapolated "
                                        f"t_quant + N*t_row = {t_call:.0f} s",
            "host_cores": os.cpu_count()}


def run_reference(args):
    """The reference arm: the CPU oracle on the same workload, K timed steps of sampled rows."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from video_diffusion_transformer_sage_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w)
    rows_per_step = 4
    cb = cpu_baseline(inp, rows_per_step=rows_per_step, steps=args.warmup + args.steps, v_format=args.v_format,
                      smooth_v=args.smooth_v)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
            "config": {"workload": f"{w.name}: N={w.n_tokens}, H={w.n_heads}, D={w.head_dim}, batch 1, non-causal, "
                                   f"strided NHD views of a [{w.n_tokens}, {3 * w.n_heads * w.head_dim}] bf16 QKV buffer"},
            "cpu_baseline": {"kind": "oracle", "cores": cb["cores"], "sample": cb["sample"], "value": cb["value"],
                             "unit": UNIT},
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-call-timing", action="store_true",
                    help="skip the 5 x 10 per-call timing of sage_attn_fwd")
    ap.add_argument("--v-format", default="e4m3", choices=["e4m3", "int8"],
                    help="the timed path's V and P codes: e4m3 (the method's default) or int8 (INT8 P.V)")
    ap.add_argument("--smooth-v", action="store_true", help="time the path with V mean smoothing")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the timing of the INT8 P.V variant and of V smoothing")
    ap.add_argument("--no-qk-transform", action="store_true",
                    help="skip the timing of the in-place RMSNorm + rotary stage")
    ap.add_argument("--dense-anchor", action="store_true",
                    help="also time one call of the unquantised dense path (slow: CUDA cores)")
    ap.add_argument("--no-mma-ceiling", action="store_true",
                    help="skip the measurement of the tensor-core rate of the kernel's MMA shapes")
    ap.add_argument("--workload", default=WORKLOAD, help="a workload of synth.WORKLOADS with qkv layout")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
