#!/usr/bin/env python3
"""Benchmark of the KDA decode state update on GB300.

Headline workload: one decode step, N=64 requests x HV=12 value heads,
K=V=128, fp32 state pool [256, 12, 128, 128], bf16 q/k/v, fp32 gates and
output (the N=64, HV=12, K=V=128 shape the pages time their gating kernel on:
ROCm/ATOM pull request 2130, What).  A "step" is one call of kda_decode_step.

Metric: state GB/s = (state bytes read + written + q/k/v/o bytes) / step time.

Timing:
  * device ("value"): inputs resident in HBM; K steps are launched back to
    back from a CUDA graph, each on a different one of R state pools whose
    combined footprint is > 4x the L2, so every step streams its state from
    HBM and also pays the write-back of earlier steps' dirty lines (the
    steady state of a model that updates a different layer's pool each step).
    CUDA events on the launching stream bracket exactly the K steps.
  * end to end ("e2e"): the same steps through the same C ABI call, but each
    step copies its inputs (q, k, v, a, b, slot ids) from pinned host memory
    and reads the output o back; the pools stay resident.
  * clocks are sampled with nvidia-smi while the timed work runs.

--impl reference times the fp64 CPU oracle (the only reference this method
has: the pages ship no code) on the host cores, on a bounded sample of the
same workload.
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

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

N, HV, K, V, SLOTS = 64, 12, 128, 128, 256
METRIC = "KDA decode state GB/s (% of HBM peak) and us/step at N=64, HV=12, K=V=128"
PEAK_FALLBACK_GBS = 6800.0
WORKLOAD = {
    "f32": "decode step, N=64 x HV=12, K=V=128, fp32 pool [256,12,128,128], bf16 q/k/v, fp32 a/b/o",
    "f16": "decode step, N=64 x HV=12, K=V=128, fp16 pool [256,12,128,128], bf16 q/k/v, fp32 a/b/o",
}


_CODE_TOKENS = None

# The sources that define the decode kernel and its launch shape: a recorded
# traffic figure stays valid while their code (comments and layout removed)
# is unchanged.  Of kda_api.cu only the lines of the decode tile shape
# (the KDA_DEC_* settings and the decode launcher) count.
DECODE_SOURCES = ("kda_common.cuh", "kda_decode_tma.cuh", "kda_api.cu")
DECODE_API_MARKERS = ("KDA_DEC_", "launch_decode", "decode_smem_bytes", "kda_decode_kernel")


def code_text(src: str) -> str:
    """C/C++/CUDA source with its comments removed and its whitespace collapsed:
    what the compiler sees, so that an edit to a comment changes nothing."""
    global _CODE_TOKENS
    import re
    if _CODE_TOKENS is None:  # string and character literals are kept whole
        _CODE_TOKENS = re.compile(r"""//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|'(?:\\.|[^'\\\n])*'""", re.S)

    def drop(m):
        tok = m.group(0)
        if tok[0] in "\"'":
            return tok
        return "\n" * tok.count("\n") if tok.startswith("/*") else ""  # lines stay lines (directives)
    kept = _CODE_TOKENS.sub(drop, src)
    lines = (" ".join(line.split()) for line in kept.splitlines())
    return "\n".join(line for line in lines if line)


def source_hash(paths=None) -> str:
    """Short hash of CUDA sources' code (comments and layout removed; default:
    the decode kernel's files): profile summaries record it, so a number
    measured on an older kernel is recognised as stale, while an edited
    comment leaves it valid."""
    import hashlib
    h = hashlib.sha256()
    if paths is None:
        csrc = os.path.join(REPO, "kda_linear_attention_gated_gb300", "csrc")
        for name in DECODE_SOURCES:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                code = code_text(f.read())
            if name == "kda_api.cu":
                code = "\n".join(l for l in code.splitlines() if any(m in l for m in DECODE_API_MARKERS))
            h.update(code.encode())
        return h.hexdigest()[:16]
    for path in paths:
        with open(path, encoding="utf-8") as f:
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]


IN_GRAPH_PREFIX = 3  # untimed launches ahead of e0 when the events are recorded inside the graph


def in_graph_events(torch):
    """Two timing events that record as nodes of a captured graph, or None
    where this torch cannot make them (the caller then times whole replays)."""
    try:
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    except TypeError:
        return None


def timed_replays(graph, stream, reps):
    """Milliseconds of `reps` replays of `graph` on `stream`, by CUDA events.
    One untimed replay is queued first, so that the GPU is busy when the start
    event is recorded and the timed replays are already queued behind it: the
    window holds the replays themselves, not the host's graph launch latency."""
    import torch
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def graph_timed(torch, stream, launch, n, warm=3):
    """Milliseconds of n launches, launch(i) for i = IN_GRAPH_PREFIX .. +n-1,
    timed by events inside one CUDA graph behind IN_GRAPH_PREFIX untimed
    launches (as for the headline: the window runs from the completion of
    the launch before the first timed one to the completion of the last).
    Where the events cannot be made, the graph holds the n launches alone and
    is timed as a whole replay with one untimed replay queued ahead.  The
    caller has made one eager launch first (module load)."""
    events = in_graph_events(torch)
    prefix = IN_GRAPH_PREFIX if events else 0
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream() if events else None
    with torch.cuda.stream(stream):
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(prefix + n):
                if events and i == prefix:
                    side.wait_stream(stream)
                    events[0].record(side)
                launch(i)
            if events:
                events[1].record(stream)
                stream.wait_stream(side)
        for _ in range(warm):
            g.replay()
    if not events:
        return timed_replays(g, stream, 1)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    return events[0].elapsed_time(events[1])


GRAPH_TIMED = ("one CUDA graph: 3 untimed launches, then the timed ones between events recorded inside "
               "the graph")


def algorithmic_bytes(n, hv, k, v, t, state_bytes, qkv_bytes, reads=1, writes=1):
    """State read + written plus q, k, v (qkv_bytes each) and fp32 o."""
    state = (reads + writes * t) * n * hv * k * v * state_bytes
    io = n * t * hv * (2 * k + v) * qkv_bytes + n * t * hv * v * 4
    return state + io


def peaks():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback", {}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling around the timed work."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if device_id:
            cmd += ["-i", device_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        rows = []
        for line in open(self.out.name):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.out.name)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


def reduce_max(x, dist, device):
    """The largest of every rank's x (x itself on one rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank, us_per_step_max, world):
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return bytes_per_step_per_rank * world / (us_per_step_max * 1e-6) / 1e9


def chunk_size(k, limit=512):
    for c in range(min(k, limit), 0, -1):
        if k % c == 0:
            return c
    return 1


def _oracle_inputs():
    import torch
    from kda_linear_attention_gated_gb300 import workloads
    inp = workloads.make_decode(n=N, hv=HV, k=K, v=V, num_slots=SLOTS, state_dtype=torch.float32,
                                qkv_dtype=torch.bfloat16, seed=0)
    pool = inp.pool.numpy().copy()
    args = [x.double().numpy() for x in (inp.q, inp.k, inp.v, inp.a, inp.b)]
    return pool, inp.init_slot.numpy(), args


def cpu_oracle_sample(target_s=12.0, nthreads=None):
    """Time the fp64 oracle on the headline workload: whole decode steps of
    N=64 x HV=12 on a 256-slot fp32 pool, repeated until about target_s."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    pool, slots, args = _oracle_inputs()
    oracle.decode_step(pool, slots, *args, nthreads=nthreads)  # load + warm
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_step(pool, slots, *args, nthreads=nthreads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    per_step = el / steps
    gbs = algorithmic_bytes(N, HV, K, V, 1, 4, 2) / per_step / 1e9
    return dict(value=round(gbs, 4), unit="GB/s", cores=nthreads, kind="oracle",
                sample=f"{steps} full decode steps (N=64 x HV=12, K=V=128, fp32 pool, bf16 q/k/v) "
                       f"in {el:.1f} s; {per_step * 1e3:.1f} ms/step",
                ms_per_step=per_step * 1e3), steps, el


def reference_sample_size(steps, full_step_s, budget_s=60.0):
    """Requests per reference step so that `steps` steps take about budget_s."""
    m = int(N * budget_s / max(steps * full_step_s, 1e-9))
    return max(1, min(N, m))


def run_reference(args, rank, world):
    """The oracle on the host cores: exactly `steps` timed steps after up to
    `warmup` untimed ones, each step the first m of the 64 requests (all 12
    heads), m chosen so the timed steps take about a minute."""
    if rank != 0:
        return 0
    import oracle
    nthreads = os.cpu_count() or 1
    pool, slots, inputs = _oracle_inputs()
    oracle.decode_step(pool, slots, *inputs, nthreads=nthreads)
    t0 = time.perf_counter()
    oracle.decode_step(pool, slots, *inputs, nthreads=nthreads)
    full = time.perf_counter() - t0
    m = reference_sample_size(args.steps, full)
    sub = [x[:m] for x in inputs]
    warm = 0
    t_w = time.perf_counter()
    while warm < args.warmup and time.perf_counter() - t_w < 10.0:
        oracle.decode_step(pool, slots[:m], *sub, nthreads=nthreads)
        warm += 1
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_step(pool, slots[:m], *sub, nthreads=nthreads)
    el = time.perf_counter() - t0
    per_step = el / args.steps
    gbs = algorithmic_bytes(m, HV, K, V, 1, 4, 2) / per_step / 1e9
    sample = (f"{args.steps} steps of {m} of the 64 requests x 12 heads each (fp32 pool, bf16 q/k/v), "
              f"{el:.1f} s, {per_step * 1e3:.3f} ms/step; full step {full * 1e3:.1f} ms")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": warm,
        "ms_per_step": round(per_step * 1e3 * N / m, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD["f32"], "global_batch": N,
                   "parallelism": "host cores (OpenMP over request x head pairs)",
                   "l2": "n/a (host)"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the fp16 / verify lines")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--workload", choices=("decode_f32", "decode_f16"), default="decode_f32",
                    help="headline workload: the decode step on an fp32 pool (the metric's) or fp16 pool")
    ap.add_argument("--case", choices=("verify_f16", "sweep", "prefill", "aux", "conv_decode"), default=None,
                    help="time one secondary case alone and print its line (profiling runs)")
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="minimum untimed load before timing (clocks ramp; 0 under a profiler)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import kda_linear_attention_gated_gb300 as kda
    from kda_linear_attention_gated_gb300 import workloads

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    kda.build()
    lib32 = kda.KdaLibrary(torch.float32)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2**20
    dev_uuid = None
    try:
        dev_uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass

    def make_pools(inp, count):
        base = inp.pool.to("cuda")
        return [base] + [base.clone() for _ in range(count - 1)]

    def bench_decode(state_dtype, qkv_dtype, seed, steps, warmup, sample_clocks, flags):
        lib = kda.KdaLibrary(state_dtype)
        inp = workloads.make_decode(n=N, hv=HV, k=K, v=V, num_slots=SLOTS, state_dtype=state_dtype,
                                    qkv_dtype=qkv_dtype, seed=seed)
        es = 4 if state_dtype == torch.float32 else 2
        active = N * HV * K * V * es
        R = max(4, math.ceil(4 * l2 / active) + 1)
        pools = make_pools(inp, R)
        d = inp.to("cuda")
        o = torch.empty(N, HV, V, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        stream = torch.cuda.Stream()
        chunk = chunk_size(steps)
        # A run that fits in one graph is timed by events recorded inside it
        # (in_graph_events): PREFIX untimed launches run first, e0 is recorded
        # on a side stream once the last of them completes, and e1 once the
        # last timed launch completes.  The window holds exactly the `steps`
        # launches, each behind its predecessor as in a long stream, and
        # neither the host's graph launch nor a first launch on an idle GPU.
        events = in_graph_events(torch) if chunk == steps else None
        prefix = IN_GRAPH_PREFIX if events else 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            # eager warm-up launch (module load) before capture
            lib.kda_decode_step(pools[0], d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status)
            stream.synchronize()
            side = torch.cuda.Stream() if events else None
            with torch.cuda.graph(g, stream=stream):
                for i in range(prefix + chunk):
                    if events and i == prefix:
                        side.wait_stream(stream)
                        events[0].record(side)
                    lib.kda_decode_step(pools[i % R], d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status,
                                        flags=flags)
                if events:
                    events[1].record(stream)
                    stream.wait_stream(side)
        # warm-up: at least `warmup` steps and at least ~1 s of load
        t_w = time.perf_counter()
        done = 0
        with torch.cuda.stream(stream):
            while done < warmup or time.perf_counter() - t_w < args.soak_seconds:
                g.replay()
                done += chunk
                if done % (chunk * 8) == 0:
                    stream.synchronize()
        sampler = ClockSampler(dev_uuid) if sample_clocks else None
        if sample_clocks and args.soak_seconds > 0:
            with torch.cuda.stream(stream):
                # keep the GPU loaded while the sampler starts
                for _ in range(max(1, int(0.3 / max(chunk * 20e-6, 1e-6)))):
                    g.replay()
        if dist is not None:
            dist.barrier()
        if events:
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                g.replay()
            torch.cuda.synchronize()
            ms = events[0].elapsed_time(events[1])
        else:
            ms = timed_replays(g, stream, steps // chunk)
        if dist is not None:
            dist.barrier()
        clocks = sampler.stop() if sampler else None
        st = int(status.item())
        if st != 0:
            raise RuntimeError(f"device status {st}: {lib.kda_strerror(st)}")
        return dict(ms_total=ms, us_per_step=ms * 1e3 / steps, pools=R, chunk=chunk, prefix=prefix,
                    bytes=algorithmic_bytes(N, HV, K, V, 1, es, 2), clocks=clocks,
                    pool_bytes=R * pools[0].numel() * es)

    def bench_e2e(steps):
        """Through the C ABI with host buffers.  Every step: one kda_stage_host
        launch copies the step's packed inputs (slot ids, q, k, v, a, b) from
        pinned host memory into one of NB device buffer sets (a kernel, one
        thread per 16 bytes, loads over the host link: no copy-engine
        transfer and its fixed cost), then kda_decode_step writes o straight
        into pinned host memory.  Both on one stream with programmatic
        dependent launch: the staging loads start while the previous decode
        drains and store after it; the decode starts while the staging runs
        and reads its inputs after it (no early state reads: its slot ids come
        from the kernel just before it).  A group of steps is captured in one
        CUDA graph and replayed, so the host's per-call work does not pace the
        GPU."""
        inp = workloads.make_decode(n=N, hv=HV, k=K, v=V, num_slots=SLOTS, state_dtype=torch.float32,
                                    qkv_dtype=torch.bfloat16, seed=0)
        R = max(4, math.ceil(4 * l2 / (N * HV * K * V * 4)) + 1)
        pools = make_pools(inp, R)
        names = ("init_slot", "q", "k", "v", "a", "b")
        srcs = [getattr(inp, n_).contiguous() for n_ in names]
        sizes = [t.numel() * t.element_size() for t in srcs]
        offs = [0]
        for sz in sizes[:-1]:
            offs.append(offs[-1] + (sz + 255) // 256 * 256)
        h2d = offs[-1] + sizes[-1]
        host = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        for t, off, sz in zip(srcs, offs, sizes):
            host[off:off + sz].copy_(t.view(-1).view(torch.uint8))
        NB = 4
        dev_in = [torch.empty(h2d, dtype=torch.uint8, device="cuda") for _ in range(NB)]
        views = [[buf[off:off + sz].view(t.dtype).view(t.shape) for t, off, sz in zip(srcs, offs, sizes)]
                 for buf in dev_in]
        o_host = [torch.empty(N, HV, V).pin_memory() for _ in range(NB)]
        d2h = o_host[0].numel() * 4
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        stream = torch.cuda.Stream()
        pdl = kda.KDA_LAUNCH_PDL
        st_ptr = status.data_ptr()

        def one(i):
            b_ = i % NB
            rc = lib32.kda_stage_host_raw([(dev_in[b_].data_ptr(), host.data_ptr(), h2d)], stream.cuda_stream, pdl)
            if rc != 0:
                raise RuntimeError(f"kda_stage_host: {lib32.kda_strerror(rc)}")
            sl, q_, k_, v_, a_, bb = views[b_]
            rc = lib32.kda_decode_step_raw(kda.pool_desc(pools[i % R]), sl.data_ptr(), None, N, q_.data_ptr(),
                                           k_.data_ptr(), v_.data_ptr(), kda.KDA_BF16, a_.data_ptr(), bb.data_ptr(),
                                           o_host[b_].data_ptr(), st_ptr, stream.cuda_stream, pdl)
            if rc != 0:
                raise RuntimeError(f"kda_decode_step: {lib32.kda_strerror(rc)}")

        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup // 10)):
                one(i)
        torch.cuda.synchronize()
        group = 50
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            for i in range(group):
                one(i)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_.replay()
        if dist is not None:
            dist.barrier()
        n_e2e = min(steps, 2000) // group * group or group
        ms = timed_replays(g_, stream, n_e2e // group)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())}")
        return dict(us_per_step=ms * 1e3 / n_e2e, steps=n_e2e, h2d=h2d, d2h=d2h,
                    mode=f"CUDA graph of {group} steps")

    def max_over_ranks(x):
        return reduce_max(x, dist, "cuda")

    peak, peak_kind, _ = peaks()
    if args.case is not None:
        if args.case == "verify_f16":
            res = {"verify_f16": bench_verify(kda, workloads, torch, args, l2, peak),
                   "step_spec_n32_t8_fp16": bench_step(kda, workloads, torch, l2, peak)}
        elif args.case == "aux":
            res = {"ckpt_flush_fp32_n64": bench_ckpt(kda, workloads, torch, peak),
                   "ckpt_load_fp32_n64": bench_ckpt(kda, workloads, torch, peak, load=True),
                   "conv_step_n64_t5_bf16": bench_conv(kda, workloads, torch, peak),
                   "copy_floor": bench_copy_floor(kda, torch, l2, peak)}
        elif args.case == "conv_decode":
            res = {f"decode_conv_{nm}_n64": bench_decode_conv(kda, workloads, torch, l2, peak, sd)
                   for nm, sd in (("fp32", torch.float32), ("fp16", torch.float16))}
            res.update({f"step_conv_n{n_sc}_t8_fp16": bench_step_conv(kda, workloads, torch, l2, peak, n_sc)
                        for n_sc in (8, 32)})
        elif args.case == "prefill":
            res = {f"prefill_{n}x{t}_fp16{'_chunked' if c else ''}": bench_prefill(kda, workloads, torch, n, t, c)
                   for c in (False, True) for n, t in ((1, 8192), (8, 1024), (64, 128))}
        else:
            res = {f"sweep_69_layers_n{n}_{nm}": bench_sweep(kda, workloads, torch, sd, n, peak)
                   for nm, sd in (("fp32", torch.float32), ("fp16", torch.float16))
                   for n in (1, 16, 64, 128)}
        if rank == 0:
            print(json.dumps({"case": args.case, "peak": peak, "peak_kind": peak_kind, **res}), flush=True)
        return 0
    # Consecutive steps update different pools (as consecutive layers do), so
    # each launch may start streaming its state while the previous one drains.
    pdl = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE
    f16_head = args.workload == "decode_f16"
    head_dtype = torch.float16 if f16_head else torch.float32
    head = bench_decode(head_dtype, torch.bfloat16, 1 if f16_head else 0, args.steps, args.warmup, True, pdl)
    us = max_over_ranks(head["us_per_step"])
    gbs_per_gpu = head["bytes"] / (us * 1e-6) / 1e9
    value = whole_job_gbs(head["bytes"], us, world)
    e2e, e2e_us, e2e_gbs = None, None, None
    if not args.no_e2e and not f16_head:
        e2e = bench_e2e(args.steps)
        e2e_us = max_over_ranks(e2e["us_per_step"])
        e2e_gbs = head["bytes"] / (e2e_us * 1e-6) / 1e9 * world

    extra = {}
    if not args.no_extra:
        plain = bench_decode(torch.float32, torch.bfloat16, 0, min(args.steps, 20000), args.warmup, False, 0)
        extra["decode_fp32_pool_no_pdl"] = {
            "us_per_step": round(plain["us_per_step"], 3),
            "gbs": round(plain["bytes"] / (plain["us_per_step"] * 1e-6) / 1e9, 1),
            "frac_of_peak": round(plain["bytes"] / (plain["us_per_step"] * 1e-6) / 1e9 / peak, 4)}
        h16 = head if f16_head else bench_decode(torch.float16, torch.bfloat16, 1, min(args.steps, 20000),
                                                  args.warmup, False, pdl)
        extra["decode_fp16_pool"] = {
            "us_per_step": round(h16["us_per_step"], 3),
            "gbs": round(h16["bytes"] / (h16["us_per_step"] * 1e-6) / 1e9, 1),
            "frac_of_peak": round(h16["bytes"] / (h16["us_per_step"] * 1e-6) / 1e9 / peak, 4),
            "bytes_per_step": h16["bytes"], "pools": h16["pools"]}
        extra["verify"] = bench_verify(kda, workloads, torch, args, l2, peak)
        extra["verify_fp32_pool"] = bench_verify(kda, workloads, torch, args, l2, peak, torch.float32)
        extra["step_spec_n32_t8_fp16"] = bench_step(kda, workloads, torch, l2, peak)
        for sd_name, sd in (("fp32", torch.float32), ("fp16", torch.float16)):
            for n_sweep in (1, 16, 64, 128):
                extra[f"sweep_69_layers_n{n_sweep}_{sd_name}"] = bench_sweep(kda, workloads, torch, sd, n_sweep, peak)
        extra["ckpt_flush_fp32_n64"] = bench_ckpt(kda, workloads, torch, peak)
        extra["ckpt_load_fp32_n64"] = bench_ckpt(kda, workloads, torch, peak, load=True)
        extra["conv_step_n64_t5_bf16"] = bench_conv(kda, workloads, torch, peak)
        for sd_name, sd in (("fp32", torch.float32), ("fp16", torch.float16)):
            extra[f"decode_conv_{sd_name}_n64"] = bench_decode_conv(kda, workloads, torch, l2, peak, sd)
        for n_sc in (8, 32):
            extra[f"step_conv_n{n_sc}_t8_fp16"] = bench_step_conv(kda, workloads, torch, l2, peak, n_sc)
        extra["copy_floor"] = bench_copy_floor(kda, torch, l2, peak)
        extra["prefill_8x1024_fp16"] = bench_prefill(kda, workloads, torch, 8, 1024)
        extra["prefill_8x1024_fp16_chunked"] = bench_prefill(kda, workloads, torch, 8, 1024, True)

    traffic = None
    tpath = os.path.join(REPO, "profiles", "decode_f32_n64_traffic.json")
    if os.path.exists(tpath):
        try:
            t = json.load(open(tpath))
            if t.get("source_hash") == source_hash():
                traffic = t["dram_bytes_per_launch"]
        except Exception:
            traffic = None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu, _, _ = cpu_oracle_sample(target_s=12.0)
        one, _, _ = cpu_oracle_sample(target_s=4.0, nthreads=1)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us / 1e3, 6), "us_per_step": round(us, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 state, f32 math" if f16_head else "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD["f16" if f16_head else "f32"], "global_batch": N * world,
                       "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {head['pools']} rotating pools, "
                             f"{head['pool_bytes'] / 1e9:.2f} GB > 4 x {l2 / 2**20:.0f} MiB L2",
                       "launch": f"CUDA graph of {head['chunk']} launches, replayed; "
                      "flags KDA_LAUNCH_PDL|KDA_LAUNCH_PDL_EARLY_STATE",
                       "timing": (f"events inside the graph: {head['prefix']} untimed launches, then e0 "
                                  f"(recorded once the last of them completes), the {head['chunk']} timed "
                                  "launches, e1 (once the last completes)") if head["prefix"] else
                                 "events around the timed graph replays, one untimed replay queued ahead"},
            "roofline": {"bound": "hbm", "achieved": round(gbs_per_gpu, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs_per_gpu / peak, 4),
                         "traffic": traffic, "peak_kind": peak_kind,
                         "bytes_per_launch": head["bytes"]},
            "cpu_baseline": cpu,
            "e2e": None if e2e is None else {
                "value": round(e2e_gbs, 2), "unit": "GB/s", "us_per_step": round(e2e_us, 3),
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "steps": e2e["steps"],
                "how": "every step one kda_stage_host launch copies its packed inputs from pinned host "
                       "memory into one of four device buffer sets (a kernel over the host link), then the "
                       "C-ABI decode call writes o into pinned host memory; one stream, flags KDA_LAUNCH_PDL "
                       "on both; " + e2e["mode"]},
            "gpu_launches": args.steps,
            "clocks": head["clocks"],
            "extra": extra,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def bench_sweep(kda, workloads, torch, state_dtype, n, peak, layers=69, replays=30):
    """The full-depth decode: one CUDA graph of `layers` decode steps, each on
    its own 256-slot pool (N requests, HV=12, K=V=128, fp32 inputs, resets ~
    Bernoulli(0.05)); 69 distinct pools, far larger than L2."""
    lib = kda.KdaLibrary(state_dtype)
    es = 4 if state_dtype == torch.float32 else 2
    dev = [workloads.make_sweep_layer(l, n, state_dtype, sentinel=0.0).to("cuda") for l in range(layers)]
    outs = [torch.empty(n, HV, V, device="cuda") for _ in range(layers)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        d = dev[0]
        lib.kda_decode_step(d.pool, d.init_slot, d.q, d.k, d.v, d.a, d.b, outs[0], status, reset=d.reset)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for l in range(layers):
                d = dev[l]
                lib.kda_decode_step(d.pool, d.init_slot, d.q, d.k, d.v, d.a, d.b, outs[l], status,
                                    reset=d.reset, flags=flags)
        for _ in range(3):
            g.replay()
    # one replay is one forward pass over the layers, as a model launches it:
    # whole replays are timed, the boundary between forwards included
    us_fwd = timed_replays(g, stream, replays) * 1e3 / replays
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    resets = sum(int(d.reset.sum().item()) for d in dev)
    state = HV * K * V * es
    byt = (layers * n - resets) * state + layers * n * state + layers * n * HV * (2 * K + V) * 4 + layers * n * HV * V * 4
    del dev, outs
    torch.cuda.empty_cache()
    return {"workload": f"{layers} layers x N={n}, HV=12, K=V=128, {'fp32' if es == 4 else 'fp16'} pools, "
                        "fp32 inputs, resets ~ Bernoulli(0.05), one CUDA graph",
            "us_per_forward": round(us_fwd, 2), "us_per_layer": round(us_fwd / layers, 3),
            "gbs": round(byt / (us_fwd * 1e-6) / 1e9, 1),
            "frac_of_peak": round(byt / (us_fwd * 1e-6) / 1e9 / peak, 4), "bytes_per_forward": byt}


def bench_prefill(kda, workloads, torch, n, t, chunked=False, reps=5):
    """Prefill of n fresh prompts of t tokens (HV=12, K=V=128, bf16 q/k/v,
    fp16 pool), final states stored once; tokens per second.  chunked: the
    two-pass form, its workspace allocated before timing."""
    lib = kda.KdaLibrary(torch.float16)
    inp = workloads.make_prefill(lens=[t] * n, state_dtype=torch.float16, num_slots=max(16, 2 * n), seed=7,
                                 reset_p=1.0)
    d = inp.to("cuda")
    o = torch.empty(n * t, HV, V, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if chunked:
        ws = torch.empty(lib.kda_prefill_workspace_bytes(d.pool, n, n * t), dtype=torch.uint8, device="cuda")
        call = lambda: lib.kda_prefill_chunked(d.pool, d.init_slot, d.final_slot, d.q, d.k, d.v, d.a, d.b, o,  # noqa
                                               status, workspace=ws, cu_seqlens=d.cu_seqlens, max_t=t, reset=d.reset)
    else:
        call = lambda: lib.kda_prefill(d.pool, d.init_slot, d.final_slot, d.q, d.k, d.v, d.a, d.b, o, status,  # noqa
                                       cu_seqlens=d.cu_seqlens, max_t=t, reset=d.reset)
    call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        call()
    e1.record()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = e0.elapsed_time(e1) / reps
    # the recurrence's own arithmetic: decay (K V), u = S^T k (2 K V), the
    # rank-1 update (2 K V) and o = S^T q (2 K V) per token and head
    flop = 7.0 * K * V * HV * n * t
    line = {"workload": f"prefill{' (two passes)' if chunked else ''}, {n} prompts x {t} tokens, HV=12, K=V=128, "
                        "bf16 q/k/v, fp16 pool",
            "ms_per_call": round(ms, 4), "tokens_per_s": round(n * t / (ms * 1e-3), 1),
            "recurrence_tflops": round(flop / (ms * 1e-3) / 1e12, 3)}
    if chunked:
        # the scan's tensor-core products as executed, per 16-token chunk and
        # head: [X | Y] (V x 32 x K) and the state update (K x V x 16), six
        # bf16 part products each, 2 flop per multiply-add
        chunks = n * ((t + 15) // 16)
        tc = chunks * HV * 6 * 2.0 * (V * 32 * K + K * V * 16)
        sus = peaks()[2].get("bf16_tflops_sustained")
        line["tensor_tflops"] = round(tc / (ms * 1e-3) / 1e12, 3)
        if sus:
            line["tensor_frac_of_bf16_sustained"] = round(tc / (ms * 1e-3) / 1e12 / float(sus), 5)
    return line


def bench_ckpt(kda, workloads, torch, peak, replays=200, load=False):
    """Checkpoint flush of 64 fp32 states (12 x 128 x 128) from a 256-slot pool
    to a 128-entry plane (load: the reverse copy); 24 pool/plane pairs rotate
    (4.8 GB, far past L2), launched with programmatic dependent launch (the
    kernel reads nothing before the previous kernel completes)."""
    lib = kda.KdaLibrary(torch.float32)
    g = torch.Generator().manual_seed(9)
    R = 24
    pools = [workloads.make_pool(g, 256, HV, K, V, torch.float32).to("cuda") for _ in range(R)]
    planes = [torch.empty(128, HV, K, V, device="cuda") for _ in range(R)]
    slots = torch.randperm(256, generator=g)[:64].to(torch.int32).to("cuda")
    entries = torch.randperm(128, generator=g)[:64].to(torch.int32).to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    call = lib.kda_ckpt_load if load else lib.kda_ckpt_flush
    with torch.cuda.stream(stream):
        call(pools[0], planes[0], slots, entries, status)
    n_timed = R * max(1, replays // R)
    us = graph_timed(torch, stream, lambda i: call(pools[i % R], planes[i % R], slots, entries, status,
                                                   flags=kda.KDA_LAUNCH_PDL), n_timed) * 1e3 / n_timed
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    byt = 2 * 64 * HV * K * V * 4
    del pools, planes
    torch.cuda.empty_cache()
    what = ("checkpoint load, 64 fp32 states [12,128,128], 128-entry plane -> 256-slot pool" if load else
            "checkpoint flush, 64 fp32 states [12,128,128], 256-slot pool -> 128-entry plane")
    return {"workload": what, "launch": f"{GRAPH_TIMED} ({n_timed}, over {R} pool/plane pairs); "
                                        "flags KDA_LAUNCH_PDL",
            "us_per_call": round(us, 3), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(byt / (us * 1e-6) / 1e9 / peak, 4), "bytes_per_call": byt}


def bench_copy_floor(kda, torch, l2, peak, states=(8, 19, 33, 64), replays=400):
    """What a pure copy reaches at the byte counts of the paths above, launched
    the same way (a CUDA graph of launches over rotating buffers, programmatic
    dependent launch): the checkpoint flush of n fp32 states [12,128,128],
    16-byte streaming loads and stores and no arithmetic, moves 2 n 786,432 B.
    n = 8 is about the conv window step's bytes, 19 exactly the verify step's
    (29,884,416 B), 33 about the fp16-pool decode's, 64 the fp32-pool
    decode's.  A kernel launched this way pays a fixed cost per launch (the
    ramp to full bandwidth and the drain), which this line measures."""
    lib = kda.KdaLibrary(torch.float32)
    st_b = HV * K * V * 4
    out = {}
    for n in states:
        byt = 2 * n * st_b
        R = max(8, math.ceil(4 * l2 / byt) + 1)
        gen = torch.Generator(device="cuda").manual_seed(11)
        pools = [torch.randn(n, HV, K, V, device="cuda", generator=gen) for _ in range(R)]
        planes = [torch.empty(n, HV, K, V, device="cuda") for _ in range(R)]
        ids = torch.arange(n, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            lib.kda_ckpt_flush(pools[0], planes[0], ids, ids, status)
        n_timed = R * max(2, replays // R)
        us = graph_timed(torch, stream, lambda i: lib.kda_ckpt_flush(pools[i % R], planes[i % R], ids, ids, status,
                                                                     flags=kda.KDA_LAUNCH_PDL),
                         n_timed) * 1e3 / n_timed
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())}")
        out[f"bytes_{byt}"] = {"us_per_call": round(us, 3), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
                               "frac_of_peak": round(byt / (us * 1e-6) / 1e9 / peak, 4)}
        del pools, planes
        torch.cuda.empty_cache()
    out["what"] = ("checkpoint flush of n fp32 states (a pure copy), n in " + str(list(states)) +
                   f"; {GRAPH_TIMED}, over rotating buffers past L2, flags KDA_LAUNCH_PDL")
    return out


def bench_conv(kda, workloads, torch, peak, replays=480):
    """The causal short convolution in front of the recurrence at the layer
    shape: N=64 requests x T=5 tokens (4 drafts + 1), C = 4608 channels (q, k,
    v of 12 heads of 128), KW=4, a bf16 window of L = KW - 1 + 4 = 7 entries
    per slot.  48 window/input/output sets rotate (about 0.5 GB, past L2),
    launched with programmatic dependent launch and early reads (each launch
    reads its window, slot ids and weights while the previous one drains;
    the sets are distinct, so no launch reads what its predecessor writes).
    Algorithmic bytes: per request and channel the KW - 1 history entries
    read, the L window entries written, T inputs read and T outputs written,
    plus the fp32 weights and bias once."""
    lib = kda.KdaLibrary(torch.float32)
    n, t, C, kw, spec = 64, 5, 4608, 4, 4
    R = 48
    sets = [workloads.make_conv(n=n, t=t, channels=C, kw=kw, num_spec=spec, num_slots=n,
                                dtype=torch.bfloat16, seed=70 + i).to("cuda") for i in range(R)]
    ys = [torch.empty_like(d.x) for d in sets]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def call(i):
        d = sets[i]
        lib.kda_conv_step(d.window, d.conv_slot, d.x, d.weight, ys[i], status, bias=d.bias,
                          cu_seqlens=d.cu_seqlens, max_t=t, accepted=d.accepted, reset=d.reset,
                          flags=kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE)
    with torch.cuda.stream(stream):
        call(0)
    n_timed = R * max(1, replays // R)
    us = graph_timed(torch, stream, lambda i: call(i % R), n_timed) * 1e3 / n_timed
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    L = kw - 1 + spec
    byt = n * C * 2 * ((kw - 1) + L + 2 * t) + C * (kw + 1) * 4
    del sets, ys
    torch.cuda.empty_cache()
    return {"workload": "conv window step, N=64 x T=5, C=4608, KW=4, bf16 window of 7 entries",
            "us_per_call": round(us, 3), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(byt / (us * 1e-6) / 1e9 / peak, 4), "bytes_per_call": byt,
            "launch": f"{GRAPH_TIMED} ({n_timed}, over {R} sets); flags KDA_LAUNCH_PDL|KDA_LAUNCH_PDL_EARLY_STATE"}


def bench_decode_conv(kda, workloads, torch, l2, peak, state_dtype, replays=400):
    """The decode step with the short convolution fused in front
    (kda_decode_conv_step) at the headline shape: N=64 x HV=12, K=V=128, q/k/v
    from a bf16 conv of width 4 over a 3-entry window (C = 4608 channels).
    Beside it, the same work as two launches: kda_conv_step (one token a
    request) then kda_decode_step, both with PDL and early reads.  That
    decode reads q/k/v buffers of the decode's own layout; turning the conv's
    [N][C] outputs into them would cost a copy or three conv launches, which
    is not counted, so the two-launch figure is a lower bound.  Rotating
    state pools past L2.  Algorithmic bytes: the state read and written, x
    read (the q/k/v bytes), the window's history read and new entries
    written, o written (a, b, weights not counted, as for the decode)."""
    lib = kda.KdaLibrary(state_dtype)
    n, hv, K, V, kw, L = 64, 12, 128, 128, 4, 3
    es = 4 if state_dtype == torch.float32 else 2
    pool_bytes = n * hv * K * V * es
    R = max(4, math.ceil(4 * l2 / pool_bytes) + 1)
    sets = [workloads.make_decode_conv(n=n, num_slots=n, num_wslots=n, state_dtype=state_dtype, seed=90 + i)
            .to("cuda") for i in range(R)]
    C = sets[0].x.shape[1]
    os_ = [torch.empty(n, hv, V, device="cuda") for _ in range(R)]
    ys = [torch.empty_like(d.x) for d in sets]
    qkv = [(torch.empty(n, hv, K, dtype=torch.bfloat16, device="cuda").normal_(),
            torch.empty(n, hv, K, dtype=torch.bfloat16, device="cuda").normal_(),
            torch.empty(n, hv, V, dtype=torch.bfloat16, device="cuda").normal_()) for _ in range(R)]
    counters = torch.zeros(n, hv, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    flags = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE

    def fused(i):
        d = sets[i % R]
        lib.kda_decode_conv_step(d.pool, d.window, d.slot_ids, d.conv_slot, d.x, d.weight, d.a, d.b, os_[i % R],
                                 status, counters, bias=d.bias, flags=flags)

    def two(i):
        d, (q, k, v) = sets[i % R], qkv[i % R]
        lib.kda_conv_step(d.window, d.conv_slot, d.x, d.weight, ys[i % R], status, bias=d.bias, max_t=1,
                          flags=flags)
        lib.kda_decode_step(d.pool, d.slot_ids, q, k, v, d.a, d.b, os_[i % R], status, flags=flags)
    with torch.cuda.stream(stream):
        fused(0)
        two(0)
    n_timed = R * max(1, replays // R)
    us = graph_timed(torch, stream, fused, n_timed) * 1e3 / n_timed
    us2 = graph_timed(torch, stream, two, n_timed) * 1e3 / n_timed
    if int(status.item()) != 0 or int(counters.abs().sum().item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    byt = 2 * pool_bytes + n * C * 2 * (1 + (kw - 1) + L) + n * hv * V * 4
    del sets, ys, qkv, os_
    torch.cuda.empty_cache()
    sd = "fp32" if state_dtype == torch.float32 else "fp16"
    return {"workload": f"decode step with the conv fused in front, N=64 x HV=12, K=V=128, {sd} pool, "
                        f"bf16 conv window of 3 entries, width 4, C=4608",
            "us_per_step": round(us, 3), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(byt / (us * 1e-6) / 1e9 / peak, 4), "bytes_per_step": byt,
            "two_launches_us": round(us2, 3),
            "two_launches": "kda_conv_step then kda_decode_step, each PDL with early reads (y's relayout into "
                            "the decode's q/k/v not counted)",
            "launch": f"{GRAPH_TIMED} ({n_timed} steps, over {R} pool/window sets); flags "
                      "KDA_LAUNCH_PDL|KDA_LAUNCH_PDL_EARLY_STATE"}


def bench_step(kda, workloads, torch, l2, peak, n=32, t=8, replays=400):
    """The general step at serving scale: N=32 requests x T=8 tokens (one
    accepted + seven drafts) on an fp16 pool, the initial state at each
    request's accepted column of an [N][8] slot table, every token's state
    stored to its column, the learned gate scale, bf16 q/k/v.  Pools rotate
    past L2; programmatic dependent launch with early state reads."""
    lib = kda.KdaLibrary(torch.float16)
    inp = workloads.make_general(n=n, t=t, num_cols=t, h_qk=HV, state_dtype=torch.float16,
                                 qkv_dtype=torch.bfloat16, num_slots=n * t, seed=10, gate_scale=True)
    per = n * (1 + t) * HV * K * V * 2
    R = max(2, math.ceil(4 * l2 / per) + 1)
    base = inp.pool.to("cuda")
    pools = [base] + [base.clone() for _ in range(R - 1)]
    d = inp.to("cuda")
    total = n * t
    o = torch.empty(total, HV, V, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    flags = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE

    def call(pool, fl):
        lib.kda_step(pool, d.slot_table, d.q, d.k, d.v, d.a, d.b, o, status, cu_seqlens=d.cu_seqlens, max_t=t,
                     accepted=d.accepted, a_log=d.a_log, dt_bias=d.dt_bias, flags=fl)
    with torch.cuda.stream(stream):
        call(pools[0], 0)
    n_timed = R * max(1, replays // R)
    us = graph_timed(torch, stream, lambda i: call(pools[i % R], flags), n_timed) * 1e3 / n_timed
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    byt = n * HV * K * V * 2 * (1 + t) + total * (HV * (2 * K + V) * 2 + HV * K * 4 + HV * 4 + HV * V * 4)
    return {"workload": f"general step (kda_step), N={n} x T={t} (1 accepted + {t - 1} drafts), fp16 pool, "
                        "accepted columns of an [N][8] slot table, learned gate scale, bf16 q/k/v",
            "us_per_step": round(us, 3), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(byt / (us * 1e-6) / 1e9 / peak, 4), "bytes_per_step": byt, "pools": R,
            "launch": f"{GRAPH_TIMED} ({n_timed}, over {R} pools); flags KDA_LAUNCH_PDL|KDA_LAUNCH_PDL_EARLY_STATE"}


def bench_step_conv(kda, workloads, torch, l2, peak, n, t=8, replays=400):
    """The speculative step with the short convolution fused in front
    (kda_step_conv): N requests x T=8 tokens (one accepted + seven drafts) on
    an fp16 pool, each request's accepted column of an [N][8] slot table, the
    learned gate scale; q/k/v from a bf16 conv of width 4 over a window of
    kernel - 1 + 7 = 10 entries (C = 4608).  Beside it, the same work as two
    launches: kda_conv_step then kda_step, both with PDL and early reads; that
    step reads q/k/v buffers of its own layout (the conv's [total][C] y would
    need a copy to become them, not counted).  Pool/window sets rotate past
    L2.  Algorithmic bytes: the initial state read and T snapshots written, x,
    a, b read, o written, the window's history read and its L entries
    written."""
    lib = kda.KdaLibrary(torch.float16)
    kw, spec = 4, t - 1
    L = kw - 1 + spec
    per = n * (1 + t) * HV * K * V * 2
    R = max(2, math.ceil(4 * l2 / per) + 1)
    sets = [workloads.make_step_conv(n=n, num_spec=spec, kw=kw, num_slots=n * t, num_wslots=n,
                                     state_dtype=torch.float16, seed=100 + i, gate_scale=True).to("cuda")
            for i in range(R)]
    C, total = sets[0].x.shape[1], n * t
    o = torch.empty(total, HV, V, device="cuda")
    ys = [torch.empty_like(d.x) for d in sets]
    qkv = [(torch.empty(total, HV, K, dtype=torch.bfloat16, device="cuda").normal_(),
            torch.empty(total, HV, K, dtype=torch.bfloat16, device="cuda").normal_(),
            torch.empty(total, HV, V, dtype=torch.bfloat16, device="cuda").normal_()) for _ in range(R)]
    counters = torch.zeros(n, HV, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    flags = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE

    def fused(i):
        d = sets[i % R]
        lib.kda_step_conv(d.pool, d.window, d.slot_table, d.conv_slot, d.x, d.weight, d.a, d.b, o, status, counters,
                          max_t=t, accepted=d.accepted, a_log=d.a_log, dt_bias=d.dt_bias, bias=d.bias, flags=flags)

    def two(i):
        d, (q, k, v) = sets[i % R], qkv[i % R]
        lib.kda_conv_step(d.window, d.conv_slot, d.x, d.weight, ys[i % R], status, bias=d.bias, max_t=t,
                          accepted=d.accepted, flags=flags)
        lib.kda_step(d.pool, d.slot_table, q, k, v, d.a, d.b, o, status, max_t=t, accepted=d.accepted,
                     a_log=d.a_log, dt_bias=d.dt_bias, flags=flags)
    with torch.cuda.stream(stream):
        fused(0)
        two(0)
    n_timed = R * max(1, replays // R)
    us = graph_timed(torch, stream, fused, n_timed) * 1e3 / n_timed
    us2 = graph_timed(torch, stream, two, n_timed) * 1e3 / n_timed
    if int(status.item()) != 0 or int(counters.abs().sum().item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    byt = (n * HV * K * V * 2 * (1 + t) + total * (C * 2 + HV * K * 4 + HV * 4 + HV * V * 4)
           + n * C * 2 * ((kw - 1) + L))
    del sets, ys, qkv
    torch.cuda.empty_cache()
    return {"workload": f"speculative step with the conv fused in front (kda_step_conv), N={n} x T={t} "
                        f"(1 accepted + {t - 1} drafts), fp16 pool, bf16 conv window of {L} entries, width {kw}, "
                        "C=4608, learned gate scale",
            "us_per_step": round(us, 3), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(byt / (us * 1e-6) / 1e9 / peak, 4), "bytes_per_step": byt,
            "two_launches_us": round(us2, 3),
            "two_launches": "kda_conv_step then kda_step, each PDL with early reads (y's relayout into the step's "
                            "q/k/v not counted)",
            "launch": f"{GRAPH_TIMED} ({n_timed} steps, over {R} pool/window sets); flags "
                      "KDA_LAUNCH_PDL|KDA_LAUNCH_PDL_EARLY_STATE"}


def bench_verify(kda, workloads, torch, args, l2, peak, state_dtype=None, replays=400):
    """Speculative verify, N=8 x T=8, HV=12, K=V=128, fp32 inputs, on an fp16
    pool (the verify workload's) or an fp32 pool."""
    state_dtype = state_dtype or torch.float16
    es = 2 if state_dtype == torch.float16 else 4
    lib = kda.KdaLibrary(state_dtype)
    n, t = 8, 8
    inp = workloads.make_verify(n=n, t=t, hv=HV, k=K, v=V, num_slots=SLOTS,
                                state_dtype=state_dtype, qkv_dtype=torch.float32, seed=2)
    per = n * (1 + t) * HV * K * V * es
    R = max(4, math.ceil(4 * l2 / per) + 1)
    base = inp.pool.to("cuda")
    pools = [base] + [base.clone() for _ in range(R - 1)]
    d = inp.to("cuda")
    o = torch.empty(n, t, HV, V, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        lib.kda_spec_verify(pools[0], d.init_slot, d.snap_slot, d.q, d.k, d.v, d.a, d.b, o, status)
    n_timed = R * max(1, replays // R)
    us = graph_timed(torch, stream,
                     lambda i: lib.kda_spec_verify(pools[i % R], d.init_slot, d.snap_slot, d.q, d.k, d.v, d.a,
                                                   d.b, o, status,
                                                   flags=kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE),
                     n_timed) * 1e3 / n_timed
    byt = algorithmic_bytes(n, HV, K, V, t, es, 4)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    return {"workload": f"spec verify, {'fp16' if es == 2 else 'fp32'} pool, N=8 x T=8, HV=12, K=V=128, fp32 q/k/v",
            "us_per_step": round(us, 3), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(byt / (us * 1e-6) / 1e9 / peak, 4), "bytes_per_step": byt,
            "pools": R, "launch": f"{GRAPH_TIMED} ({n_timed}, over {R} pools); "
                                  "flags KDA_LAUNCH_PDL|KDA_LAUNCH_PDL_EARLY_STATE"}


if __name__ == "__main__":
    sys.exit(main())
