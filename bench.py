#!/usr/bin/env python
"""Benchmark of the headwise-chunked causal GQA attention layer on GB300.

One step = one pass of the whole hot path over the layer: for every head
chunk, the fused Q/K/V projection (+RoPE, +qk-RMSNorm), causal attention over
the full sequence and the Wo-slice accumulate (``--pass fwd``; with
``--pass fwdbwd`` also the chunked backward with recomputation).

The default workload is the one the attention kernels' target is stated for:
the Llama-3-8B single-rank shard (4 of 32 query heads, 1 of 8 KV heads,
d = 128, hidden 4096) over S = 1,048,576 tokens, forward and backward, one
head per chunk (the smallest workspace).  A secondary measurement of the
Llama-3.2-3B full layer at 64K tokens (forward, chunk_heads 3, 6, 24) rides
along in the same line (``secondary``; ``--no-secondary`` skips it).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--chunk-heads C] [--pass fwd|fwdbwd]

The timed region runs exactly K steps.  The other measurements of the line
(live kernel timings, the chunk sweep, the saved-O backward, e2e) take as
many steps as fit a few seconds each, at least one, at most K.

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs an
independent replica of the workload (the path has no exchange step on one
GPU): ``value`` is the sum of all ranks' FLOPs over the max-over-ranks time.
``--impl reference`` times the float64 CPU oracle (the only reference this
method has) on a bounded sample of the same workload.

``tiled_mlp`` and ``tiled_loss`` (``--no-mlp`` skips them and ``offload``)
time the sequence-tiled SwiGLU MLP (upipe_mlp_fwd / upipe_mlp_bwd) and
cross-entropy loss (upipe_loss_fwd / upipe_loss_bwd) at Llama-3-8B widths on
one rank's 131072 tokens; ``offload`` times the layer forward with its input
offloaded to host memory and an input-sized buffer prefetched beside it.

``fused_wo_forward`` (main and secondary workload; ``--no-fused`` skips it)
times the forward whose attention kernel adds the Wo-slice partial results
into out itself (upipe_attn_fwd_fused, no attention-output buffer) against
upipe_attn_fwd, with the workspace each needs.

Besides the layer number the line carries ``roofline`` (the dominant
attention kernel: algorithmic FLOPs per launch over its live CUDA-event launch
time) and ``hbm_kernels`` (the HBM-bound kernels: algorithmic bytes per layer
call over their summed live launch time), both timed through the library's
measurement hook.
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
sys.path.insert(0, ROOT)

METRIC = "attn-layer TFLOP/s & % BF16 tensor peak; peak workspace GB vs head-chunk size"
DEFAULT_WORKLOAD = "llama3-8b-rank-s1m"
SECONDARY_WORKLOAD = "llama3.2-3b-s65536"


def layer_flops(w, mode="fwd"):
    """Model FLOPs of one layer pass (unmasked causal pairs S(S+1)/2)."""
    S, hid, d = w.S, w.hidden, w.d
    pairs = S * (S + 1) / 2
    proj = 2.0 * S * hid * d * (w.Hq + 2 * w.Hkv)
    attn = 4.0 * d * w.Hq * pairs
    wo = 2.0 * S * w.Hq * d * hid
    if mode == "fwd":
        return proj + attn + wo, attn
    # backward: dX and dW of every projection (2x each GEMM) and the
    # attention backward (10 d per pair per head)
    bwd = 2 * (proj + wo) + 10.0 * d * w.Hq * pairs
    return proj + attn + wo + bwd, attn


def recompute_flops(w, saved_o=False):
    """FLOPs the backward executes beyond the model count: it projects each
    chunk's Q/K/V again and, unless the forward's attention output is saved,
    runs the chunk's attention forward again."""
    S, hid, d = w.S, w.hidden, w.d
    proj = 2.0 * S * hid * d * (w.Hq + 2 * w.Hkv)
    return proj if saved_o else proj + 4.0 * d * w.Hq * S * (S + 1) / 2


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture, keyed by kernel, workload and chunk size, with the sha256 of the
# kernel's source file at capture time: a changed kernel reports null.
NCU_TRAFFIC = {
    # full captures of these launches exceed the profiling size rule, so the
    # bytes were taken at S = 262144 (same geometry and chunk size) and scaled
    # by the causal pairs to S = 1,048,576 (x16.0); from 65536 to 262144 the
    # traffic grew 3.7-4.0x per doubling of S, in step with the pairs
    ("attn_fwd_kernel", "llama3-8b-rank-s1m", 1): (11216113664, "ea34b7bf3592d3cf"),
    ("attn_bwd_kernel", "llama3-8b-rank-s1m", 1): (53664954368, "952ce4de4e5f29cd"),
    # the separate forward's launches at the secondary workload (a full
    # capture: mean of one step's 8 chunk launches)
    ("attn_fwd_kernel", "llama3.2-3b-s65536", 3): (88330144, "ea34b7bf3592d3cf"),
}
KERNEL_SOURCES = {"attn_fwd_kernel": "attn_fwd.cu", "attn_bwd_kernel": "attn_bwd.cu"}


def kernel_source_sha(kernel):
    import hashlib
    path = os.path.join(ROOT, "headwise_chunked_attention_gb300", "csrc", KERNEL_SOURCES[kernel])
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def traffic_of(kernel, workload, ch, S=None):
    from workloads import WORKLOADS
    if S is not None and workload in WORKLOADS and S != WORKLOADS[workload].S:
        return None
    ent = NCU_TRAFFIC.get((kernel, workload, ch))
    if ent is None or ent[1] != kernel_source_sha(kernel):
        return None
    return ent[0]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return j["bf16_tflops"], j.get("bf16_tflops_sustained", j["bf16_tflops"]), \
            j["hbm_gbs"], "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


# ------------------------------------------------------- replica helpers --

def max_over_ranks(t: float, dist=None, device="cpu") -> float:
    """The slowest rank's time: the job finishes when every replica has."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return t
    import torch
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def replica_throughput(flops_per_rank_step: float, steps: int, world: int,
                       t_max: float) -> float:
    """Whole-job TFLOP/s of ``world`` independent replicas: all ranks' work
    over the max-over-ranks time (weak scaling: per-rank work is fixed)."""
    return world * flops_per_rank_step * steps / t_max / 1e12


# ---------------------------------------------------------------- clocks --

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # nvidia-smi takes a moment to start: wait for its first sample, and
        # keep only the samples taken after this point (the timed region)
        self.skip = 0
        if self.proc is not None:
            t0 = time.time()
            while time.time() - t0 < 5 and self.proc.poll() is None:
                n = self._nlines()
                if n > 0:
                    self.skip = n
                    break
                time.sleep(0.02)
        return self

    def _nlines(self):
        self.f.flush()
        try:
            return sum(1 for l in open(self.f.name) if l.strip())
        except OSError:
            return 0

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.f.flush()
        rows = [l.split(",") for l in open(self.f.name).read().strip().splitlines() if l]
        os.unlink(self.f.name)
        if len(rows) > self.skip:
            rows = rows[self.skip:]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle --

def oracle_sample(w, inp, rows_per_head=64, groups=1, target_s=None, prefix=None):
    """Time the float64 oracle on a bounded sample of the workload: the K/V
    projection of ``groups`` kv heads plus sampled query rows of each of
    their query heads (attention over all earlier keys).  Without
    ``target_s``: ``rows_per_head`` rows.  With it: seeded-shuffled batches of
    256 rows until ``target_s`` seconds of CPU work have been spent (at most
    16384 rows).  ``prefix``: the rows are drawn from the first ``prefix``
    tokens only, and K/V are projected for those tokens (a bounded sample of
    a long sequence).  Returns (TFLOP/s, seconds, flops, rows per head)."""
    import numpy as np
    import torch

    import oracle as O
    from workloads import sample_rows
    a = {k: v.to("cpu", torch.float64).numpy() for k, v in inp.items() if k != "x"}
    xb = inp["x"]
    x_src = lambda lo, hi: xb[lo:hi].to("cpu", torch.float64).numpy()
    g = w.Hq // w.Hkv
    S = min(w.S, prefix) if prefix else w.S
    t0 = time.perf_counter()
    flops = 0.0
    kv = []
    for kvh in range(groups):
        kv.append(O.project_kv(x_src, a["Wk"], a["Wv"], w, kvh, S, a.get("k_gamma")))
        flops += 2 * 2.0 * S * w.hidden * w.d
    if target_s is None:
        rows_all, batch = np.asarray(sample_rows(S, rows_per_head)), None
    else:
        rows_all = np.random.default_rng(0).permutation(
            np.asarray(sample_rows(S, min(S, 16384))))
        batch = 256
    done = 0
    for b0 in range(0, len(rows_all), batch or len(rows_all)):
        rows = np.sort(rows_all[b0:b0 + (batch or len(rows_all))])
        xq = np.concatenate([x_src(int(r), int(r) + 1) for r in rows])
        for kvh, (K, V) in enumerate(kv):
            for h in range(kvh * g, (kvh + 1) * g):
                q = O.attention_layer._qk_post(xq @ a["Wq"][h * w.d:(h + 1) * w.d].T, rows, w,
                                               a.get("q_gamma"))
                O.causal_attention(q, K, V, rows)
                flops += 2.0 * len(rows) * w.hidden * w.d + 4.0 * w.d * float(np.sum(rows + 1))
        done += len(rows)
        if target_s is not None and time.perf_counter() - t0 >= target_s:
            break
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, flops, done


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ------------------------------------------------------------------ main --

def config_of(w, ch, pass_):
    return {"workload": w.name, "S": w.S, "hidden": w.hidden, "Hq": w.Hq, "Hkv": w.Hkv,
            "d": w.d, "chunk_heads": ch, "qk_norm": bool(w.qk_norm),
            "rope_theta": w.rope_theta, "pass": pass_, "parallelism": "replicas",
            "l2": l2_note(w)}


L2_BYTES = 129e6  # GB300 L2


def l2_note(w):
    """How the timed steps relate to L2: the hidden states x alone exceed it
    for every benchmarked geometry, so each step streams its inputs from HBM."""
    xb = w.S * w.hidden * 2
    if xb > L2_BYTES:
        return "inputs larger than L2 (x alone is %.0f MB)" % (xb / 1e6)
    return "inputs fit in L2 (x is %.1f MB): not an HBM-resident timing" % (xb / 1e6)


REFERENCE_PREFIX = 65536


def run_reference(args, w, ch):
    """The reference arm: the float64 oracle as it stands, on the host cores.
    Each step is a bounded sample of the workload: the K/V projection of one
    kv head and 64 seeded query rows of each of its query heads, drawn from
    the first 65536 tokens (the whole sequence when it is shorter), so that
    a step is about a second of CPU work at every benchmarked size."""
    import torch
    from workloads import make_inputs
    wp = w.with_(S=min(w.S, REFERENCE_PREFIX))
    inp = make_inputs(wp, seed=0, device="cpu")
    times, tf = [], []
    for i in range(args.warmup + args.steps):
        v, dt, fl, _ = oracle_sample(wp, inp)
        if i >= args.warmup:
            times.append(dt)
            tf.append(v)
    value = sum(tf) / len(tf)
    sample = (f"per step: K/V projection of 1 kv head over {wp.S} tokens + 64 seeded query "
              f"rows of each of its query heads drawn from those tokens")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, ch, args.pass_),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def gpu_uuid(dev):
    import torch
    props = torch.cuda.get_device_properties(dev)
    gid = getattr(props, "uuid", None)
    if gid is None:
        return str(dev.index)
    return str(gid) if str(gid).startswith("GPU-") else "GPU-" + str(gid)


def measure(u, w, ch, mode, steps, warmup, dist, world, rank, dev, full=True, sweep_on=True,
            cpu_on=True, fused_on=True):
    """Everything one JSON line reports for workload ``w`` at ``ch`` heads per
    chunk (mode 0 forward, 1 forward + backward).  ``full``: also e2e, the
    HBM-bound kernels, the saved-O backward and the CPU baseline.
    ``fused_on``: also the forward with the fused Wo-slice accumulate."""
    import torch
    from workloads import make_inputs

    inp = make_inputs(w, seed=rank, device=str(dev), with_grad=mode == 1)
    shape = u.Shape.of(w, ch)
    torch.cuda.synchronize()
    base_alloc = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    ws = torch.empty(u.workspace_bytes(shape, mode), dtype=torch.uint8, device=dev)
    peak_ws = torch.cuda.max_memory_allocated() - base_alloc
    out = torch.empty(w.S, w.hidden, device=dev)
    lse = torch.empty(w.Hq, w.S, device=dev)
    grads = None
    if mode:
        grads = {n: torch.empty(inp[s].shape, device=dev) for n, s in
                 [("dx", "x"), ("dWq", "Wq"), ("dWk", "Wk"), ("dWv", "Wv"), ("dWo", "Wo")]}
        grads["dqg"] = torch.empty(w.d, device=dev) if w.qk_norm else None
        grads["dkg"] = torch.empty(w.d, device=dev) if w.qk_norm else None

    def step(sh=shape, wsb=ws):
        u.attn_fwd(sh, inp["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"], out, lse, wsb,
                   inp.get("q_gamma"), inp.get("k_gamma"))
        if mode:
            u.attn_bwd(sh, inp["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"], inp["dout"],
                       lse, grads["dx"], grads["dWq"], grads["dWk"], grads["dWv"],
                       grads["dWo"], wsb, inp.get("q_gamma"), inp.get("k_gamma"),
                       grads["dqg"], grads["dkg"])

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def timed(fn, k):
        barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(k):
            fn()
        e.record()
        barrier()
        return max_over_ranks(s.elapsed_time(e) / 1e3, dist, dev)

    pass_name = "fwdbwd" if mode else "fwd"
    flops, attn_flops = layer_flops(w, pass_name)
    nchunks = w.Hq // ch
    for _ in range(warmup):
        step()
    rc = u.last_error()
    if rc != 0:
        raise RuntimeError(f"device error {rc}")

    # ---- the timed region: exactly ``steps`` steps, device-resident inputs
    gid = gpu_uuid(dev)
    with Clocks(gid) as clk:
        t = timed(step, steps)
    clocks = clk.summary()
    value = replica_throughput(flops, steps, world, t)
    step_s = t / steps

    def aux(seconds):
        """Steps for a secondary measurement: about ``seconds`` of work."""
        return max(1, min(steps, int(seconds / step_s)))

    # ---- roofline of the attention kernels: algorithmic FLOPs per launch over
    # the live CUDA-event launch time, timed in separate passes (an event
    # between two launches keeps the next kernel from starting while the
    # previous one drains).  A kernel timed inside a seconds-long loop of
    # back-to-back steps runs under the power cap: it is measured against the
    # sustained peak; ms-scale steps against the burst peak.
    burst, sustained, hbm, src = peaks()
    long_loop = t >= 10.0
    peak, peak_kind = (sustained, f"sustained bf16 ({src}): timed region {t:.0f} s") if long_loop \
        else (burst, f"burst bf16 ({src}): timed region {t:.2f} s")
    pairs = w.S * (w.S + 1) / 2

    def roofline(kernel, kid, flops_per_pair, per_step):
        k = aux(4.0)
        kt = u.KernelTimer(kid, k * per_step)
        with kt:
            t_pass = timed(step, k)
        durations = kt.durations_ms()
        avg_ms = sum(durations) / max(1, len(durations))
        fl = flops_per_pair * w.d * ch * pairs
        ach = fl / (avg_ms / 1e3) / 1e12 if durations else None
        return {"kernel": kernel, "bound": "tensor",
                "achieved": round(ach, 2) if ach else None, "peak": peak,
                "unit": "TFLOP/s", "frac": round(ach / peak, 4) if ach else None,
                "frac_of_burst": round(ach / burst, 4) if ach else None,
                "frac_of_sustained": round(ach / sustained, 4) if ach else None,
                "peak_kind": peak_kind, "launches_timed": len(durations),
                "avg_launch_ms": round(avg_ms, 4), "flops_per_launch": fl,
                "ms_per_step_timed_pass": round(1e3 * t_pass / k, 3),
                "traffic": traffic_of(kernel, w.name, ch, w.S)}

    roof_fwd = roofline("attn_fwd_kernel", 0, 4.0, nchunks * (2 if mode else 1))
    roof_bwd = roofline("attn_bwd_kernel", 1, 10.0, nchunks) if mode else None

    res = {"value": value, "t": t, "flops": flops, "clocks": clocks, "roof_fwd": roof_fwd,
           "roof_bwd": roof_bwd, "peak_ws": peak_ws, "shape": shape, "nchunks": nchunks,
           "ws_planned": u.workspace_bytes(shape, mode)}

    # ---- end to end through the public API with host buffers: every step
    # uploads its inputs (x; and dout for the backward) from pinned host
    # memory and downloads its result (out; dx for the backward).  Steps are
    # pipelined: step i+1's upload and step i-1's download run on two copy
    # streams while step i computes, on double-buffered device copies when
    # the device has room for them (else one set, and the copies serialise).
    if full:
        in_names = ["x"] + (["dout"] if mode else [])
        res0 = grads["dx"] if mode else out
        hosts = {n: inp[n].cpu().pin_memory() for n in in_names}
        res_host = torch.empty(res0.shape, dtype=res0.dtype).pin_memory()
        extra = sum(inp[n].numel() * inp[n].element_size() for n in in_names) + \
            res0.numel() * res0.element_size()
        nbuf = 2 if extra + (8 << 30) < torch.cuda.mem_get_info(dev)[0] else 1
        dbufs = [{n: inp[n] for n in in_names}] + \
            [{n: torch.empty_like(inp[n]) for n in in_names} for _ in range(nbuf - 1)]
        rbufs = [res0] + [torch.empty_like(res0) for _ in range(nbuf - 1)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {k: [torch.cuda.Event() for _ in range(nbuf)] for k in ("x", "in", "done", "out")}

        def step_io(b):
            # the forward needs only x: dout's upload runs beside it
            db, rb = dbufs[b], rbufs[b]
            o_ = rb if not mode else out
            main = torch.cuda.current_stream(dev)
            main.wait_event(ev["x"][b])
            u.attn_fwd(shape, db["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"], o_, lse, ws,
                       inp.get("q_gamma"), inp.get("k_gamma"))
            if mode:
                main.wait_event(ev["in"][b])
                u.attn_bwd(shape, db["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"],
                           db["dout"], lse, rb, grads["dWq"], grads["dWk"], grads["dWv"],
                           grads["dWo"], ws, inp.get("q_gamma"), inp.get("k_gamma"),
                           grads["dqg"], grads["dkg"])

        def e2e_run(k):
            main = torch.cuda.current_stream(dev)
            s_in.wait_stream(main)
            s_out.wait_stream(main)

            def upload(i):
                b = i % nbuf
                with torch.cuda.stream(s_in):
                    if i >= nbuf:
                        s_in.wait_event(ev["done"][b])   # step i - nbuf is done with it
                    for n in in_names:           # x first, then dout
                        dbufs[b][n].copy_(hosts[n], non_blocking=True)
                        if n == "x":
                            ev["x"][b].record(s_in)
                    ev["in"][b].record(s_in)

            upload(0)
            for i in range(k):
                b = i % nbuf
                if i + 1 < k:
                    upload(i + 1)
                if i >= nbuf:
                    main.wait_event(ev["out"][b])        # its result has been downloaded
                step_io(b)
                ev["done"][b].record(main)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev["done"][b])
                    res_host.copy_(rbufs[b], non_blocking=True)
                    ev["out"][b].record(s_out)
            main.wait_stream(s_out)

        e2e_run(1)
        # ~30 s of steps: the first upload and the last download, which no
        # compute overlaps, are then a small part of the region
        k_e2e = max(2, aux(30.0))
        with Clocks(gid) as clk_e2e:
            t_e2e = timed(lambda: e2e_run(k_e2e), 1)

        def copy_gbs(dst, src_):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            dst.copy_(src_, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            return src_.numel() * src_.element_size() / (e0.elapsed_time(e1) / 1e3) / 1e9
        # the host link as this process sees it (other jobs share it): one
        # upload and one download alone, after the e2e region
        h2d_gbs = copy_gbs(dbufs[0][in_names[0]], hosts[in_names[0]])
        d2h_gbs = copy_gbs(res_host, rbufs[0])
        res["e2e"] = {"value": round(replica_throughput(flops, k_e2e, world, t_e2e), 2),
                      "unit": "TFLOP/s",
                      "h2d_bytes_per_step": int(sum(h.numel() * h.element_size()
                                                    for h in hosts.values())),
                      "d2h_bytes_per_step": int(res_host.numel() * res_host.element_size()),
                      "steps": k_e2e, "pipelined_buffers": nbuf, "clocks": clk_e2e.summary(),
                      "h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1)}
        del dbufs, rbufs, hosts, res_host

    # ---- the HBM-bound kernels: algorithmic bytes per layer call over their
    # summed live launch time (hook kernels 2, 3, 4)
    def hbm_kernel(name, kernel, bytes_per_call):
        k = aux(2.0)
        kt_ = u.KernelTimer(kernel, k * (nchunks + w.Hkv + 1))
        with kt_:
            timed(step, k)
        d_ = kt_.durations_ms()
        if not d_:
            return None
        per_call = len(d_) // k
        b = bytes_per_call(per_call)
        ach = b / (sum(d_) / k / 1e3) / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(ach / hbm, 4), "launches_timed": len(d_),
                "launches_per_call": per_call, "avg_launch_us": round(1e3 * sum(d_) / len(d_), 2),
                "bytes_per_call": int(b)}

    def wo_bytes(per_call):
        # out (+)= O_c Wo_c^T: fp32 out read and written (written only for the
        # first chunk), O_c and the Wo slice read once
        first = 1 if per_call == nchunks else 0
        rmw = (per_call - first) * 8 + first * 4
        return per_call * 2 * (w.S + w.hidden) * ch * w.d + rmw * w.S * w.hidden

    if full:
        el = 12 if w.qk_norm else 8   # fp32 g (+ fp32 y-hat) read, bf16 hi + lo written
        hk = [hbm_kernel("gemm_kernel<F32> (Wo-slice accumulate on all SMs)", 2, wo_bytes)]
        if mode:
            hk.append(hbm_kernel(
                "qk_bwd_kernel (dQ and dK RoPE/RMSNorm backward)", 3,
                lambda n: w.S * (w.Hq + w.Hkv) * (w.d * el + (4 if w.qk_norm else 0))))
            hk.append(hbm_kernel("f32_to_bf16x2_kernel (dV hi/lo split)", 4,
                                 lambda n: w.S * w.Hkv * w.d * 8))
        res["hbm_kernels"] = [h for h in hk if h]

    # ---- paired accumulates: the forward given the third chunk buffer
    # (upipe_workspace_bytes mode 2) adds two chunks per Wo-slice accumulate
    if not mode and nchunks >= 3:
        ws2 = torch.empty(u.workspace_bytes(shape, 2), dtype=torch.uint8, device=dev)
        step(shape, ws2)
        k = max(2, aux(2.0))
        tp = timed(lambda: step(shape, ws2), k)
        res["paired"] = {"tflops": round(replica_throughput(flops, k, world, tp), 2),
                         "ms_per_step": round(1e3 * tp / k, 3), "steps": k,
                         "workspace_gb": round(ws2.numel() / 1e9, 4),
                         "note": "a third chunk buffer lets each Wo-slice accumulate add two "
                                 "chunks, halving the fp32 read-modify-write passes over out"}
        del ws2

    # ---- the fused forward (upipe_attn_fwd_fused): the attention kernel adds
    # each head's Wo-slice partial result into out itself, so the workspace
    # holds no attention output.  Timed against upipe_attn_fwd, each with its
    # smallest workspace (modes 3 and 0), in alternating passes
    if fused_on:
        fwd_flops = layer_flops(w, "fwd")[0]
        wsb = {"separate": u.workspace_bytes(shape, 0), "fused": u.workspace_bytes(shape, 3)}
        wsf = {nm: torch.empty(b, dtype=torch.uint8, device=dev) for nm, b in wsb.items()}

        def fwd_of(nm):
            call = u.attn_fwd_fused if nm == "fused" else u.attn_fwd
            return lambda: call(shape, inp["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"],
                                out, lse, wsf[nm], inp.get("q_gamma"), inp.get("k_gamma"))

        fns = {nm: fwd_of(nm) for nm in wsb}
        for fn in fns.values():
            fn()
        if u.last_error() != 0:
            raise RuntimeError("device error in the fused forward comparison")
        k = max(2, int(2.0 / timed(fns["fused"], 1)))
        rates = {nm: [] for nm in fns}
        for order in (("separate", "fused"), ("fused", "separate")):
            for nm in order:
                rates[nm].append(fwd_flops * k / timed(fns[nm], k) / 1e12)
        launch_ms = {}
        for nm, kid in (("separate", 0), ("fused", 5)):
            kt = u.KernelTimer(kid, nchunks)
            with kt:
                fns[nm]()
            launch_ms[nm] = round(sum(kt.durations_ms()), 3)
        res["fused"] = {
            "chunk_heads": ch, "steps": k,
            "forward_tflops": {nm: round(sum(r) / len(r), 2) for nm, r in rates.items()},
            "forward_tflops_passes": {nm: [round(x, 2) for x in r] for nm, r in rates.items()},
            "workspace_gb": {nm: round(b / 1e9, 4) for nm, b in wsb.items()},
            "attention_kernel_ms_per_forward": launch_ms,
            "note": "upipe_attn_fwd_fused: the attention kernel adds o_h Wo_h^T into out (fp32 "
                    "TMA reduce-adds at the end of each CTA), no O buffer; 'separate' is "
                    "upipe_attn_fwd (Wo-slice GEMM per chunk, overlapped on a side stream). "
                    "The fused kernel's time includes the Wo work"}
        del wsf

    # ---- the saved-O backward: the forward keeps every head's attention
    # output and the backward reuses it instead of recomputing the attention
    if mode and full:
        o_all = torch.empty(w.S, w.Hq * w.d, dtype=torch.bfloat16, device=dev)

        def step_saved_o():
            u.attn_fwd(shape, inp["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"], out, lse,
                       ws, inp.get("q_gamma"), inp.get("k_gamma"), o_all)
            u.attn_bwd(shape, inp["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"], inp["dout"],
                       lse, grads["dx"], grads["dWq"], grads["dWk"], grads["dWv"],
                       grads["dWo"], ws, inp.get("q_gamma"), inp.get("k_gamma"),
                       grads["dqg"], grads["dkg"], attn_o=o_all)

        step_saved_o()
        k = aux(4.0)
        ts = timed(step_saved_o, k)
        so_tf = replica_throughput(flops, k, world, ts)
        res["saved_o"] = {
            "tflops": round(so_tf, 2),
            "hardware_tflops": round(so_tf * (flops + recompute_flops(w, True)) / flops, 2),
            "ms_per_step": round(1e3 * ts / k, 3), "steps": k,
            "extra_bytes": int(o_all.numel() * 2),
            "note": "forward keeps the [S, Hq*d] bf16 attention output (and, with three or more "
                    "chunks, pairs its Wo-slice accumulates); the backward skips the per-chunk "
                    "attention recompute"}
        del o_all

    # ---- chunk sweep: throughput and workspace against chunk_heads.  The
    # chunk sizes are timed in order and then in reverse, and each reports
    # the mean of its two passes: a clock that drifts through the sweep (the
    # power cap settles over seconds) then biases no chunk size against
    # another.
    sweep = []
    if sweep_on:
        rates = {c: [] for c in w.chunk_heads}
        info = {}
        for c in list(w.chunk_heads) + list(reversed(w.chunk_heads)):
            sh = u.Shape.of(w, c)
            wb = u.workspace_bytes(sh, mode)
            del ws
            torch.cuda.synchronize()
            a0 = torch.cuda.memory_allocated()
            torch.cuda.reset_peak_memory_stats()
            ws = torch.empty(wb, dtype=torch.uint8, device=dev)
            pk = torch.cuda.max_memory_allocated() - a0
            step(sh, ws)
            k = aux(2.0)
            tc = timed(lambda: step(sh, ws), k)
            rates[c].append(flops * k / tc / 1e12)
            info[c] = (wb, pk)
        for c in w.chunk_heads:
            wb, pk = info[c]
            sweep.append({"chunk_heads": c, "tflops": round(sum(rates[c]) / len(rates[c]), 2),
                          "tflops_passes": [round(r, 2) for r in rates[c]],
                          "workspace_gb": round(wb / 1e9, 4), "peak_alloc_gb": round(pk / 1e9, 4)})
        unchunked = [e for e in sweep if e["chunk_heads"] == w.Hq]
        if unchunked:
            for e in sweep:
                e["vs_unchunked"] = round(e["tflops"] / unchunked[0]["tflops"] - 1.0, 4)
    res["sweep"] = sweep

    launches = 1 + 3 * nchunks
    if mode:
        groups = w.Hkv if ch < w.Hq // w.Hkv else nchunks
        # a memset and the bound kernel; per chunk: projection, attention,
        # dO, dWo, attention backward, Q RoPE/RMSNorm backward, one dW and one
        # dx GEMM; per KV group: K RoPE/RMSNorm backward, dV split
        launches += 2 + 8 * nchunks + 2 * groups
    res["launches_per_step"] = launches

    if full and cpu_on and world == 1:
        groups = min(w.Hkv, 4)
        v, dt, fl, nrows = oracle_sample(w, {k: v for k, v in inp.items()}, groups=groups,
                                         target_s=12.0)
        res["cpu_baseline"] = {
            "value": round(v, 6), "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": f"float64 oracle: full K/V projection of {groups} kv head(s) + {nrows} "
                      "seeded random query rows of each of their query heads (attention over "
                      "all earlier keys), batches of 256 rows until 12 s of CPU work",
            # the whole layer at the sample's rate: an extrapolation, not a
            # measurement
            "full_layer_seconds_extrapolated": round(flops / (v * 1e12), 1)}
    del inp, ws, out, lse, grads
    torch.cuda.empty_cache()
    return res


def measure_mlp(u, dev, dist, steps):
    """The sequence-tiled SwiGLU MLP at its benchmark workload (Llama-3-8B
    widths, one rank's share of 1M tokens, tiles of 8192): forward and
    backward TFLOP/s over ``steps`` device-resident calls each, and the
    workspace against the untiled intermediates."""
    import torch
    from workloads import MLP_WORKLOADS, make_mlp_inputs
    w = MLP_WORKLOADS["llama3-8b-mlp-rank-s1m"]
    t = make_mlp_inputs(w, seed=0, device=str(dev), with_grad=True)
    sh = u.MlpShape(w.S, w.hidden, w.ffn, w.tile_rows)
    wsb = {m: u.mlp_workspace_bytes(sh, m) for m in (0, 1)}
    ws = torch.empty(wsb[1], dtype=torch.uint8, device=dev)
    y = torch.empty(w.S, w.hidden, device=dev)
    g = {n: torch.empty(shp, device=dev) for n, shp in
         [("dx", (w.S, w.hidden)), ("dWg", (w.ffn, w.hidden)), ("dWu", (w.ffn, w.hidden)),
          ("dWd", (w.hidden, w.ffn))]}

    def fwd():
        u.mlp_fwd(sh, t["x"], t["Wg"], t["Wu"], t["Wd"], y, ws)

    def bwd():
        u.mlp_bwd(sh, t["x"], t["Wg"], t["Wu"], t["Wd"], t["dy"], g["dx"], g["dWg"], g["dWu"],
                  g["dWd"], ws)

    for _ in range(3):
        fwd()
        bwd()
    if u.last_error() != 0:
        raise RuntimeError("device error in the MLP measurement")

    def timed(fn, k):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(k):
            fn()
        e0.record()
        torch.cuda.synchronize()
        return max_over_ranks(s0.elapsed_time(e0) / 1e3, dist, dev) / k

    k = max(3, min(steps, 20))
    shf = float(w.S) * w.hidden * w.ffn
    tf, tb = timed(fwd, k), timed(bwd, k)
    untiled = w.S * w.ffn * (2 + 4 + 2 + 2)   # a, dA, dg, du over the whole sequence
    res = {"config": {"workload": w.name, "S": w.S, "hidden": w.hidden, "ffn": w.ffn,
                      "tile_rows": w.tile_rows},
           "steps": k,
           "fwd_ms": round(1e3 * tf, 3), "bwd_ms": round(1e3 * tb, 3),
           "fwd_tflops": round(6.0 * shf / tf / 1e12, 2),
           "bwd_tflops": round(12.0 * shf / tb / 1e12, 2),
           # the backward also recomputes the gate and up projections
           "bwd_hardware_tflops": round(16.0 * shf / tb / 1e12, 2),
           "workspace_gb": {"fwd": round(wsb[0] / 1e9, 4), "bwd": round(wsb[1] / 1e9, 4),
                            "untiled_bwd": round(untiled / 1e9, 3)},
           "note": "upipe_mlp_fwd/bwd: y = (silu(x Wg^T) * (x Wu^T)) Wd^T in tiles of "
                   "tile_rows tokens; model FLOPs 6 S hidden ffn forward, 12 backward"}
    del t, ws, y, g
    torch.cuda.empty_cache()
    return res


def measure_loss(u, dev, dist, steps):
    """The sequence-tiled cross-entropy loss at its benchmark workload
    (Llama-3-8B's vocabulary of 128256, one rank's 131072 tokens, tiles of
    4096): forward and backward TFLOP/s over device-resident calls, and the
    workspace against the untiled logits."""
    import torch
    from workloads import LOSS_WORKLOADS, make_loss_inputs
    w = LOSS_WORKLOADS["llama3-8b-loss-rank-s1m"]
    t = make_loss_inputs(w, seed=0, device=str(dev))
    sh = u.LossShape(w.S, w.hidden, w.vocab, w.tile_rows)
    wsb = {m: u.loss_workspace_bytes(sh, m) for m in (0, 1)}
    ws = torch.empty(max(wsb.values()), dtype=torch.uint8, device=dev)
    loss = torch.empty(w.S, device=dev)
    lse = torch.empty(w.S, device=dev)
    dh = torch.empty(w.S, w.hidden, device=dev)
    dW = torch.empty(w.vocab, w.hidden, device=dev)

    def fwd():
        u.loss_fwd(sh, t["h"], t["W"], t["targets"], loss, lse, ws)

    def bwd():
        u.loss_bwd(sh, t["h"], t["W"], t["targets"], lse, 1.0 / w.S, dh, dW, ws)

    for _ in range(3):
        fwd()
        bwd()
    if u.last_error() != 0:
        raise RuntimeError("device error in the loss measurement")

    def timed(fn, k):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(k):
            fn()
        e0.record()
        torch.cuda.synchronize()
        return max_over_ranks(s0.elapsed_time(e0) / 1e3, dist, dev) / k

    k = max(3, min(steps, 10))
    f = 2.0 * w.S * w.hidden * w.vocab
    tf, tb = timed(fwd, k), timed(bwd, k)
    res = {"config": {"workload": w.name, "S": w.S, "hidden": w.hidden, "vocab": w.vocab,
                      "tile_rows": w.tile_rows},
           "steps": k, "mean_loss": round(float(loss.mean()), 4),
           "fwd_ms": round(1e3 * tf, 3), "bwd_ms": round(1e3 * tb, 3),
           "fwd_tflops": round(f / tf / 1e12, 2),
           "bwd_tflops": round(2.0 * f / tb / 1e12, 2),
           # the backward also recomputes the logits
           "bwd_hardware_tflops": round(3.0 * f / tb / 1e12, 2),
           "workspace_gb": {"fwd": round(wsb[0] / 1e9, 4), "bwd": round(wsb[1] / 1e9, 4),
                            "untiled_logits_fp32": round(w.S * w.vocab * 4 / 1e9, 2)},
           "note": "upipe_loss_fwd/bwd: cross entropy over the vocabulary in tiles of tile_rows "
                   "tokens; model FLOPs 2 S hidden vocab forward, 4 backward"}
    del t, ws, loss, lse, dh, dW
    torch.cuda.empty_cache()
    return res


def measure_offload(u, w, ch, dev, dist):
    """The offload of block inputs beside compute: the layer forward of ``w``
    timed alone, and with an offload of its input x to page-locked host
    memory and a prefetch of an x-sized buffer back running on the library's
    copy stream during each forward (joined at the step's end); plus each
    copy alone."""
    import torch
    from workloads import make_inputs
    t = make_inputs(w, seed=0, device=str(dev))
    sh = u.Shape.of(w, ch)
    ws = torch.empty(u.workspace_bytes(sh, 0), dtype=torch.uint8, device=dev)
    out = torch.empty(w.S, w.hidden, device=dev)
    lse = torch.empty(w.Hq, w.S, device=dev)
    host_out = torch.empty(t["x"].shape, dtype=torch.bfloat16).pin_memory()
    host_in = torch.empty(t["x"].shape, dtype=torch.bfloat16).pin_memory()
    back = torch.empty_like(t["x"])
    nbytes = t["x"].numel() * t["x"].element_size()

    def fwd():
        u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
                   t.get("q_gamma"), t.get("k_gamma"))

    def fwd_with_copies():
        a = u.offload(t["x"], host_out)
        b = u.prefetch(host_in, back)
        fwd()
        u.copy_join(a)
        u.copy_join(b)

    def timed(fn, k):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(k):
            fn()
        e0.record()
        torch.cuda.synchronize()
        return max_over_ranks(s0.elapsed_time(e0) / 1e3, dist, dev) / k

    for _ in range(2):
        fwd_with_copies()
    if u.last_error() != 0:
        raise RuntimeError("device error in the offload measurement")
    k = 3
    t_alone = timed(fwd, k)
    t_copies = timed(fwd_with_copies, k)
    t_off = timed(lambda: u.copy_join(u.offload(t["x"], host_out)), 2)
    t_pre = timed(lambda: u.copy_join(u.prefetch(host_in, back)), 2)
    flops = layer_flops(w, "fwd")[0]
    res = {"config": {"workload": w.name, "chunk_heads": ch, "pass": "fwd"},
           "bytes_each_way": nbytes, "steps": k,
           "layer_tflops_alone": round(flops / t_alone / 1e12, 2),
           "layer_tflops_with_copies": round(flops / t_copies / 1e12, 2),
           "offload_gbs_alone": round(nbytes / t_off / 1e9, 1),
           "prefetch_gbs_alone": round(nbytes / t_pre / 1e9, 1),
           "note": "upipe_offload / upipe_prefetch of a block input (x) beside the layer forward "
                   "on the library's copy stream; the host link is shared with other jobs"}
    del t, ws, out, lse, host_out, host_in, back
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--chunk-heads", type=int, default=None)
    ap.add_argument("--pass", dest="pass_", default=None, choices=["fwd", "fwdbwd"],
                    help="default: fwdbwd for workloads with a backward, else fwd")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-fused", action="store_true",
                    help="skip the fused Wo-slice forward comparison")
    ap.add_argument("--no-mlp", action="store_true",
                    help="skip the sequence-tiled MLP, loss and offload measurements")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end and HBM-kernel measurements (profiling runs)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="run the workload's geometry at this many tokens instead")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.seq_len:
        w = w.with_(S=args.seq_len)
    if args.pass_ is None:
        args.pass_ = "fwdbwd" if "bwd" in w.passes else "fwd"
    ch = args.chunk_heads or w.chunk_heads[0]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w, ch)
        return

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import __graft_entry__
    __graft_entry__.build()
    import headwise_chunked_attention_gb300 as u

    dev = torch.device("cuda", local)
    mode = 1 if args.pass_ == "fwdbwd" else 0
    r = measure(u, w, ch, mode, args.steps, args.warmup, dist, world, rank, dev,
                full=not args.no_e2e, sweep_on=not args.no_sweep, cpu_on=not args.no_cpu,
                fused_on=not args.no_fused)
    secondary = None
    if not args.no_secondary and args.workload != SECONDARY_WORKLOAD:
        w2 = WORKLOADS[SECONDARY_WORKLOAD]
        r2 = measure(u, w2, w2.chunk_heads[0], 0, args.steps, 3, dist, world, rank, dev,
                     full=False, fused_on=not args.no_fused)
        secondary = {"config": config_of(w2, w2.chunk_heads[0], "fwd"),
                     "value": round(r2["value"], 2), "unit": "TFLOP/s",
                     "ms_per_step": round(1e3 * r2["t"] / args.steps, 3),
                     "steps": args.steps, "roofline_attn_fwd": r2["roof_fwd"],
                     "chunk_sweep": r2["sweep"], "paired_accumulate": r2.get("paired"),
                     "fused_wo_forward": r2.get("fused"), "clocks": r2["clocks"]}

    mlp = None if args.no_mlp else measure_mlp(u, dev, dist, args.steps)
    loss_line = None if args.no_mlp else measure_loss(u, dev, dist, args.steps)
    # one process only: each copy pins an input-sized host buffer (8.6 GB at
    # the default workload), which N ranks on one node would multiply
    offload_line = None if (args.no_mlp or world > 1) else measure_offload(u, w, ch, dev, dist)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    burst = peaks()[0]
    flops, t = r["flops"], r["t"]
    line = {
        "metric": METRIC, "value": round(r["value"], 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # inputs, weights and dout are bf16; the attention operands (q, k, v,
        # P, dO, dS) are fp16 and every contraction accumulates in fp32
        "dtype": "bf16", "operand_dtype": "bf16 GEMM operands, fp16 attention operands, fp32 accumulate",
        "data": "synthetic", "config": config_of(w, ch, args.pass_),
        "frac_of_bf16_peak": round(r["value"] / world / burst, 4),
        # model FLOPs count each unmasked (query, key) pair and each GEMM once;
        # hardware FLOPs add what the backward recomputes
        "flops_per_step": {"model": flops,
                           "hardware": flops + (recompute_flops(w) if mode else 0.0)},
        "hardware_tflops": round(r["value"] * (flops + (recompute_flops(w) if mode else 0.0))
                                 / flops, 2),
        "peak_workspace_gb": round(r["peak_ws"] / 1e9, 4),
        "workspace_gb_planned": round(r["ws_planned"] / 1e9, 4),
        "chunk_sweep": r["sweep"],
        "saved_o_backward": r.get("saved_o"),
        "paired_accumulate": r.get("paired"),
        "fused_wo_forward": r.get("fused"),
        "roofline": r["roof_bwd"] if r["roof_bwd"] else r["roof_fwd"],
        "roofline_attn_fwd": r["roof_fwd"],
        "roofline_attn_bwd": r["roof_bwd"],
        "hbm_kernels": r.get("hbm_kernels"),
        "e2e": r.get("e2e"),
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
        "secondary": secondary,
        "tiled_mlp": mlp,
        "tiled_loss": loss_line,
        "offload": offload_line,
    }
    if "cpu_baseline" in r:
        line["cpu_baseline"] = r["cpu_baseline"]
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
