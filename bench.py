#!/usr/bin/env python
"""Benchmark of the NVFP4 MoE router gate on GB300.

One step = one router call (runtime NVFP4 quantization of the activations,
block-scaled NVFP4 gate GEMM, sigmoid / biased top-k / renormalise / scale
epilogue, all in one kernel launch: max|x|, then the K-split GEMM with the
quantization and the epilogue inside it) over one batch of the prefill
workload: T = 4096 tokens,
D = 7168, E = 256 experts, k = 8, bf16 activations (per-token LogNormal scale),
NVFP4 gate weight resident on the GPU.  Synthetic, seeded inputs.

Printed (rank 0, one JSON line): prefill tokens/s over exactly --steps timed
steps (inputs resident in HBM, four rotating 58.7 MB activation buffers so no
step reads its input from L2).  The timed steps are replays of a CUDA graph of
16 router calls (and one graph of the remaining --steps % 16), as a serving
loop captures its step; plus
  eager         the same steps launched directly, one call after another (the
                cooperative launch then waits for the previous call to end);
  e2e           the same call with the batch copied from pinned host memory and
                the ids/weights copied back inside every timed step;
  roofline      the dominant kernel's algorithmic bytes per launch / its mean
                duration over the timed region (one launch per step), against
                MEASURED_PEAKS.json; the event-bracketed duration of a second
                pass with events around every launch is reported beside it;
  kernels       every kernel of the step, the same way;
  decode        the decode router (T = 1, 8, 64) as CUDA-graph replays;
  other_rooflines  the wide-N raw head (k = 8 and 1), the adversarial large
                batch (tokens/s), the standalone quantizer and the decode
                kernel's own duration, each against the measured HBM copy rate;
  no_cooperative  the same steps launched with NVR_FLAG_NO_COOPERATIVE;
  cpu_baseline  the CPU oracle on a bounded sample of the same batch (all
                cores, and one BLAS thread in a child process);
  clocks        SM clocks and throttle reasons sampled during the timed region.

--impl reference times the CPU oracle itself on the host cores (the pages
publish no implementation to run).  Multi-GPU (torchrun): independent replicas,
one batch per rank, no collective on the data path; value = all ranks' tokens /
the slowest rank's time.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = ("router tokens/s (prefill) & µs/call (decode T=1); % of FP4 tensor / HBM roofline")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense ratio (fp4 13.5 PF vs bf16 2.25 PF)
GRAPH_CALLS = 16                      # router calls per captured graph in the timed region


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def wait_ready(self, timeout_s=10.0):
        """Block until nvidia-smi has written its first sample (it takes a
        moment to start), so that the samples cover the timed region."""
        if self.proc is None:
            return
        t0 = time.time()
        while time.time() - t0 < timeout_s and self.proc.poll() is None:
            with open(self.path) as f:
                if f.readline().strip():
                    return
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        busy = [r[0] for r in rows if r[0] > 0.5 * r[1]] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle

def oracle_tokens_per_s(w, x32_all, packed_w, bias, budget_s=12.0, rows_per_call=64):
    """Time the oracle (as it stands) routing slices of the batch for about
    `budget_s` seconds; the per-tensor gsa is the whole batch's."""
    from oracle import quantize as Q, gemm, router
    gsa = Q.global_scale(x32_all)
    wq, ws, wg = packed_w
    t0 = time.perf_counter()
    done = 0
    r0 = 0
    while True:
        rows = x32_all[r0:r0 + rows_per_call]
        xq, xs, _ = Q.quantize(rows, gsa=gsa)
        L, _ = gemm.logits(xq, xs, gsa, wq, ws, wg)
        router.route(L, bias, w.k, w.routed_scaling, w.raw)
        done += rows.shape[0]
        r0 = (r0 + rows_per_call) % x32_all.shape[0]
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done / el, done, el


def oracle_sample_json(budget_s):
    """The oracle sample above on the prefill batch, as one JSON line (run in
    a child process by oracle_single_thread)."""
    from oracle import pipeline
    w = WL.WORKLOADS["prefill"]
    x32 = WL.bf16_bits_to_float32(WL.make_x(w, seed=WL.SEED))
    packed = pipeline.pack_weight(WL.bf16_bits_to_float32(WL.make_w(w)))
    tps, done, el = oracle_tokens_per_s(w, x32, packed, WL.make_bias(w), budget_s=budget_s)
    return json.dumps({"value": tps, "done": done, "seconds": el})


def oracle_single_thread(budget_s=8.0):
    """The same oracle sample with one BLAS / OpenMP thread, in a child
    process (the thread count of a BLAS library is fixed when it loads)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", str(budget_s)], env=env,
                           capture_output=True, text=True, timeout=600)
        d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    except Exception as e:  # reported, not fatal: the all-cores figure stands
        return {"error": "%s: %s" % (type(e).__name__, e)}
    return {"value": d["value"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "%d tokens in 64-token slices (%.1f s), one BLAS thread" % (d["done"], d["seconds"])}


# ------------------------------------------------------------------ ranks

def max_over_ranks(v, world, device):
    """The largest value of `v` over all ranks (the slowest rank's time)."""
    if world <= 1:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, steps, max_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


# ------------------------------------------------------------------ GPU arm

def kernel_names(path):
    """Launches of one router call: bf16 activations on a head of <= 256
    experts whose token tiles all fit on the GPU at once run one kernel (max|x|,
    quantization, GEMM and router epilogue); the decode path is one kernel."""
    return ["fused"] if path == "tc" else ["decode_router"]


def algorithmic(w, T, name):
    """(bytes, flops) the method must move / compute per launch of `name`."""
    D, N, k = w.D, w.N, w.k
    x_bytes = T * D * 2
    xq = T * (D // 2 + D // 16)
    wq = N * (D // 2 + D // 16)
    out = T * k * 8
    if name == "amax":
        return x_bytes, 0
    if name == "quantize":
        return x_bytes + xq, 0
    if name in ("gemm", "fused"):          # x (bf16) once from HBM, W, bias, ids/weights
        return x_bytes + wq + N * 4 + out, 2 * T * D * N
    if name == "epilogue":
        return T * N * 4 + N * 4 + out, 0                      # the logits read once, bias, outputs
    return x_bytes + wq + N * 4 + out, 2 * T * D * N           # decode_router


def traffic_table():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by kernel;
    an entry counts only while the kernel's source is unchanged."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    out = {}
    if not os.path.exists(p):
        return out
    for line in open(p):
        parts = line.split("#")[0].split()
        if len(parts) == 4:
            name, nbytes, src, digest = parts
            f = os.path.join(ROOT, "nvfp4_router_gate_gb300", "csrc", src)
            if os.path.exists(f) and hashlib.sha256(open(f, "rb").read()).hexdigest()[:16] == digest:
                out[name] = float(nbytes)
    return out


def run_gpu(args, rank, world, local_rank):
    import torch
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WL.WORKLOADS["prefill"]
    T = w.T
    x_np = WL.make_x(w, seed=WL.SEED + rank)
    W_np = WL.make_w(w)
    bias_np = WL.make_bias(w)

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    NBUF = 4                                          # 4 x 58.7 MB > 129 MB L2
    xs = [dev_bf16(x_np) for _ in range(NBUF)]
    bias = torch.from_numpy(bias_np).to(dev)
    W_fp4, W_sf, w_gsa = R.nvfp4_pack_weight(dev_bf16(W_np))
    ws = R.new_workspace(R.router_gate_workspace_size(T, w.D, w.N, w.k), dev)
    ids = [torch.empty((T, w.k), dtype=torch.int32, device=dev) for _ in range(NBUF)]
    wts = [torch.empty((T, w.k), dtype=torch.float32, device=dev) for _ in range(NBUF)]
    stream = torch.cuda.current_stream()

    def step(i):
        R.router_gate_topk(xs[i % NBUF], W_fp4, W_sf, w_gsa, bias, w.k, w.routed_scaling,
                           out_ids=ids[i % NBUF], out_w=wts[i % NBUF], workspace=ws)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(local_rank)
    sampler.start()
    sampler.wait_ready()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # the timed steps: replays of a graph of GRAPH_CALLS calls and one graph of
    # the remaining steps % GRAPH_CALLS (captured after the warm-up, which also
    # settles the launch attributes outside capture)
    n_graph, n_rem = divmod(args.steps, GRAPH_CALLS)
    sizes = ([GRAPH_CALLS] if n_graph else []) + ([n_rem] if n_rem else [])
    graphs = {}
    for n in sizes:                                   # calls per graph
        graphs[n] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[n]):
            for i in range(n):
                step(i)
        for _ in range(2):                            # untimed replays
            graphs[n].replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_graph):
        graphs[GRAPH_CALLS].replay()
    if n_rem:
        graphs[n_rem].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    plan = R.last_router_plan()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_per_step = ms / args.steps
    value = job_throughput(world, T, args.steps, ms)
    plan["cooperative"] = int(_native.lib().nvr_router_cooperative_state())

    # the same steps launched directly
    n_eager = max(3, min(args.steps, 2000))
    e0.record(stream)
    for i in range(n_eager):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    eg_ms = e0.elapsed_time(e1) / n_eager
    eager = {"ms_per_step": eg_ms, "tokens_per_s": T / (eg_ms / 1e3), "steps": n_eager,
             "hbm_frac": algorithmic(w, T, "fused")[0] / (eg_ms / 1e3) / 1e9 / load_peaks()[0]}

    # the same steps without the cooperative launch (NVR_FLAG_NO_COOPERATIVE:
    # for a caller that owns the GPU; the next call's launch then overlaps the
    # previous call's tail)
    n_nc = max(3, min(args.steps, 2000))

    def step_nc(i):
        R.router_gate_topk(xs[i % NBUF], W_fp4, W_sf, w_gsa, bias, w.k, w.routed_scaling,
                           out_ids=ids[i % NBUF], out_w=wts[i % NBUF], workspace=ws,
                           flags=R.NVR_FLAG_NO_COOPERATIVE)
    for i in range(3):
        step_nc(i)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(n_nc):
        step_nc(i)
    e1.record(stream)
    torch.cuda.synchronize()
    nc_ms = e0.elapsed_time(e1) / n_nc
    no_coop = {"ms_per_step": nc_ms, "tokens_per_s": T / (nc_ms / 1e3), "steps": n_nc,
               "hbm_frac": algorithmic(w, T, "fused")[0] / (nc_ms / 1e3) / 1e9 / load_peaks()[0]}

    # per-kernel pass (events between the launches)
    names = kernel_names("tc")
    n_prof = max(3, min(args.steps, 500))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(names))] for _ in range(n_prof)]
    for e in evs:                                     # torch creates the CUDA event lazily
        for ev in e:
            ev.record(stream)
    torch.cuda.synchronize()
    handles = [ctypes_array(e) for e in evs]
    lib = _native.lib()
    for i in range(n_prof):
        lib.nvr_set_profile_events(handles[i][0], len(names))
        step(i)
    lib.nvr_set_profile_events(None, 0)
    torch.cuda.synchronize()
    per = {n: [] for n in names}
    for e in evs:
        for j, n in enumerate(names):
            per[n].append(e[2 * j].elapsed_time(e[2 * j + 1]))
    hbm, bf16, peak_kind = load_peaks()
    fp4_peak = bf16 * FP4_OVER_BF16
    traffic = traffic_table()
    tot = sum(statistics.mean(v) for v in per.values())
    kernels = {}
    for n in names:
        t_ms = statistics.mean(per[n])
        b, f = algorithmic(w, T, n)
        ent = {"ms": t_ms, "share": t_ms / tot}
        # every kernel of the step is bound by HBM: the gate GEMM's intensity
        # (2*T*D*N flops over the bf16 x it reads, ~N/2 flop/B) is far below
        # the fp4 tensor ridge (peak fp4 rate / HBM bandwidth, ~1700 flop/B)
        ach = b / (t_ms / 1e3) / 1e9
        ent.update({"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm})
        if f:
            tf = f / (t_ms / 1e3) / 1e12
            ent.update({"tensor_achieved_tflops": tf, "tensor_peak_tflops": fp4_peak,
                        "tensor_frac": tf / fp4_peak})
        ent["traffic"] = traffic.get(n)
        kernels[n] = ent
    dom = max(names, key=lambda n: kernels[n]["ms"])
    if len(names) == 1:
        # one launch per step: its average duration over the timed region is
        # the step time (events between launches, as in the per-kernel pass,
        # remove the overlap of one launch's tail with the next one's start)
        b, _ = algorithmic(w, T, dom)
        ach = b / (ms_per_step / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": kernels[dom]["traffic"], "bytes_per_launch": b, "ms_per_launch": ms_per_step,
                "duration_source": "timed region / steps (one launch per step)",
                "event_bracketed_ms": kernels[dom]["ms"],
                "event_bracketed_frac": kernels[dom]["frac"]}
    else:
        roof = {k: kernels[dom][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
        roof["duration_source"] = "per-kernel CUDA events"
    roof["kernel"] = dom
    roof["peak_source"] = peak_kind

    # end to end: every step copies its batch in from pinned host memory and
    # its ids/weights back out; as in a serving pipeline the copy of step i+1
    # (on a copy stream) overlaps the routing of step i (host link ~209 GB/s
    # on this machine: the copy bounds the step)
    x_host = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_host = [torch.empty((T, w.k), dtype=torch.int32).pin_memory() for _ in range(2)]
    w_host = [torch.empty((T, w.k), dtype=torch.float32).pin_memory() for _ in range(2)]
    n_e2e = max(3, min(args.steps, 200))
    copy_stream = torch.cuda.Stream()

    def e2e_run(n, start_event=None):
        copied = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        if start_event is not None:
            copy_stream.wait_event(start_event)
        for i in range(n):
            if i >= NBUF:
                copy_stream.wait_event(done[i - NBUF])        # device buffer i % NBUF is free
            with torch.cuda.stream(copy_stream):
                xs[i % NBUF].copy_(x_host, non_blocking=True)
            copied[i].record(copy_stream)
            stream.wait_event(copied[i])
            step(i)
            ids_host[i % 2].copy_(ids[i % NBUF], non_blocking=True)
            w_host[i % 2].copy_(wts[i % NBUF], non_blocking=True)
            done[i].record(stream)

    e2e_run(3)
    torch.cuda.synchronize()
    barrier()
    e0.record(stream)
    e2e_run(n_e2e, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e = {"value": job_throughput(world, T, n_e2e, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": int(x_host.numel() * 2),
           "d2h_bytes_per_step": int(ids_host[0].numel() * 4 + w_host[0].numel() * 4), "steps": n_e2e,
           "pipeline": "copy of step i+1 overlaps the routing of step i (second stream)"}

    # decode router: T = 1, 8, 64 as CUDA-graph replays
    decode = {}
    if not args.skip_decode:
        dw = WL.WORKLOADS["decode"]
        gate = R.RouterGate(dev_bf16(WL.make_w(dw)), torch.from_numpy(WL.make_bias(dw)).to(dev),
                            k=dw.k, routed_scaling=dw.routed_scaling, max_tokens=64)
        for Td in (1, 8, 64):
            xd = dev_bf16(WL.make_x(dw.with_T(Td)))
            s2 = torch.cuda.Stream()
            s2.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s2):
                for _ in range(3):
                    gate(xd)
            torch.cuda.current_stream().wait_stream(s2)
            # the router calls of consecutive layers, captured in one graph as
            # a decode step would capture them; and a graph of one call (its
            # replay overhead is paid by every call)
            for calls, key in ((16, "T%d_us_per_call"), (1, "T%d_us_per_call_one_call_graph")):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for _ in range(calls):
                        gate(xd)
                for _ in range(20):
                    g.replay()
                torch.cuda.synchronize()
                reps = 2000 // calls
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                decode[key % Td] = e0.elapsed_time(e1) * 1e3 / (reps * calls)
                if calls == 1 and Td == 1:
                    # the same graph replayed once on an idle stream: launch
                    # to completion of one call
                    lat = []
                    for _ in range(200):
                        torch.cuda.synchronize()
                        e0.record(stream)
                        g.replay()
                        e1.record(stream)
                        torch.cuda.synchronize()
                        lat.append(e0.elapsed_time(e1) * 1e3)
                    decode["T1_one_call_graph_latency_us_median"] = statistics.median(lat)
        # Back-to-back replays of a one-call graph are paced by the host's
        # replay rate: the same loop over a graph of one trivial kernel
        tiny = torch.zeros(1, device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tiny.add_(1.0)
        for _ in range(20):
            g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(2000):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        decode["one_call_graph_host_floor_us"] = e0.elapsed_time(e1) * 1e3 / 2000
        decode["launches_T1"] = 1
        decode["graph"] = "per call: 16 calls captured in one CUDA graph (the layers of a decode step)"

    extra = {} if args.skip_extra else extra_rooflines(R, dev, stream, hbm, fp4_peak, traffic)

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        from oracle import pipeline
        x32 = WL.bf16_bits_to_float32(x_np)
        packed = pipeline.pack_weight(WL.bf16_bits_to_float32(W_np))
        tps, done, el = oracle_tokens_per_s(w, x32, packed, bias_np)
        cpu = {"value": tps, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": "%d tokens of the T=4096 batch in 64-token slices (%.1f s), batch gsa; "
                         "NumPy quantize + float64 GEMM + epilogue" % (done, el),
               "single_thread": oracle_single_thread()}

    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e2m1*ue4m3->f32", "data": "synthetic",
        "config": {"workload": "prefill router T=4096 D=7168 E=256 k=8, bf16 x with per-token "
                               "LogNormal(0,1) scale, NVFP4 gate W~N(0,0.02), bias U(-0.05,0.05), "
                               "routed_scaling 2.5",
                   "T": T, "D": w.D, "E": w.N, "k": w.k,
                   "l2": "inputs larger than L2: 4 rotating 58.7 MB activation buffers",
                   "timing": "%d replays of a CUDA graph of %d router calls and %d of one of %d; 'eager' "
                             "launches every step directly" % (n_graph, GRAPH_CALLS, 1 if n_rem else 0, n_rem),
                   "plan": plan,
                   "parallelism": "replicas" if world > 1 else "single"},
        "e2e": e2e, "gpu_launches": len(names) * args.steps, "roofline": roof, "kernels": kernels,
        "eager": eager, "no_cooperative": no_coop, "decode": decode, "other_rooflines": extra,
        "cpu_baseline": cpu,
        "clocks": clocks,
    }


def _timed_calls(fn, n, stream, warm=3):
    """Mean ms per call of `n` back-to-back calls (CUDA events around them all)."""
    import torch
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def _hbm_entry(nbytes, ms, hbm, traffic=None, **kw):
    ach = nbytes / (ms / 1e3) / 1e9
    ent = {"bound": "hbm", "bytes_per_call": int(nbytes), "ms_per_call": ms, "achieved": ach, "peak": hbm,
           "unit": "GB/s", "frac": ach / hbm, "traffic": traffic}
    ent.update(kw)
    return ent


def extra_rooflines(R, dev, stream, hbm, fp4_peak, traffic):
    """Rooflines of the other configurations and kernels, each timed over
    back-to-back calls with CUDA events on the launching stream:
      wide_n       the N = 129280 raw head (T = 32, k = 8 and k = 1): weight
                   streaming, 0.52 GB per call (> L2: every call reads it from HBM);
      lm_head_linear_T32  the same weight through nvfp4_linear, bf16 logits out;
      adversarial  the T = 16384, E = 384 batch (x 235 MB > L2): tokens/s too;
      quantize     nvfp4_quantize_act on the prefill batch (x read once, codes
                   and scales written), four rotating inputs;
      moe_gemm     nvfp4_moe_gemm on the prefill batch routed by the router
                   (E = 256, k = 8) into experts of N = 512, and the combine;
      decode_kernel the decode router's own device duration at T = 1 (events
                   around every launch, so no overlap with its neighbours)."""
    import torch
    from nvfp4_router_gate_gb300 import _native
    out = {}
    g = torch.Generator(device=dev)
    g.manual_seed(WL.SEED)

    # wide-N raw head: synthetic bf16 weight of the workload's distribution,
    # drawn on the device (0.93 G elements)
    wn = WL.WORKLOADS["wide_n"]
    W = (torch.randn((wn.N, wn.D), generator=g, device=dev, dtype=torch.float32) * wn.w_std).to(torch.bfloat16)
    W_fp4, W_sf, w_gsa = R.nvfp4_pack_weight(W)
    del W
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    x = torch.randn((wn.T, wn.D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    wbytes = wn.N * (wn.D // 2 + wn.D // 16)
    for k in (8, 1):
        ws = R.new_workspace(R.router_gate_workspace_size(wn.T, wn.D, wn.N, k), dev)
        ids = torch.empty((wn.T, k), dtype=torch.int32, device=dev)
        wt = torch.empty((wn.T, k), dtype=torch.float32, device=dev)
        ms = _timed_calls(lambda i: R.router_gate_topk(x, W_fp4, W_sf, w_gsa, None, k, 1.0, True, out_ids=ids,
                                                       out_w=wt, workspace=ws), 50, stream)
        nbytes = wbytes + wn.T * wn.D * 2 + wn.T * k * 8
        out["wide_n_k%d" % k] = _hbm_entry(nbytes, ms, hbm, plan=R.last_router_plan(),
                                           traffic=traffic.get("stream_topk_k8") if k == 8 else None,
                                           traffic_kernel="gemm_stream_kernel" if k == 8 else None,
                                           tensor_tflops=2 * wn.T * wn.D * wn.N / (ms / 1e3) / 1e12)
    # the same weight as an NVFP4 linear layer (lm_head shape), bf16 logits out
    ws = R.new_workspace(R.nvfp4_linear_workspace_size(wn.T, wn.D, wn.N), dev)
    lm_out = torch.empty((wn.T, wn.N), dtype=torch.bfloat16, device=dev)
    ms = _timed_calls(lambda i: R.nvfp4_linear(x, W_fp4, W_sf, w_gsa, out=lm_out, workspace=ws), 50, stream)
    nbytes = wbytes + wn.T * wn.D * 2 + wn.T * wn.N * 2
    out_l = _hbm_entry(nbytes, ms, hbm, plan=R.last_router_plan(),
                       traffic=traffic.get("stream_linear_bf16"), traffic_kernel="gemm_stream_kernel",
                       tensor_tflops=2 * wn.T * wn.D * wn.N / (ms / 1e3) / 1e12,
                       note="nvfp4_linear T=32 D=7168 N=129280 (lm_head shape), bf16 out")
    out["lm_head_linear_T32"] = out_l
    del W_fp4, W_sf, lm_out
    torch.cuda.empty_cache()

    # adversarial large batch
    aw = WL.WORKLOADS["adversarial"]
    xa = torch.from_numpy(WL.make_x(aw).view(np.int16)).view(torch.bfloat16).to(dev)
    Wa = torch.from_numpy(WL.make_w(aw).view(np.int16)).view(torch.bfloat16).to(dev)
    Wf, Wsf, wg = R.nvfp4_pack_weight(Wa)
    bias = torch.from_numpy(WL.make_bias(aw)).to(dev)
    ws = R.new_workspace(R.router_gate_workspace_size(aw.T, aw.D, aw.N, aw.k), dev)
    ids = torch.empty((aw.T, aw.k), dtype=torch.int32, device=dev)
    wt = torch.empty((aw.T, aw.k), dtype=torch.float32, device=dev)
    ms = _timed_calls(lambda i: R.router_gate_topk(xa, Wf, Wsf, wg, bias, aw.k, aw.routed_scaling, out_ids=ids,
                                                   out_w=wt, workspace=ws), 50, stream)
    nbytes = aw.T * aw.D * 2 + aw.N * (aw.D // 2 + aw.D // 16) + aw.N * 4 + aw.T * aw.k * 8
    out["adversarial"] = _hbm_entry(nbytes, ms, hbm, plan=R.last_router_plan(), tokens_per_s=aw.T / (ms / 1e3),
                                    traffic=traffic.get("fused_384"), traffic_kernel="fused_qgemm_kernel<112, 3>")
    del xa, Wa
    torch.cuda.empty_cache()

    # standalone quantizer on the prefill batch (4 rotating 58.7 MB inputs)
    pw = WL.WORKLOADS["prefill"]
    xp = torch.from_numpy(WL.make_x(pw).view(np.int16)).view(torch.bfloat16).to(dev)
    xs = [xp.clone() for _ in range(4)]
    codes = torch.empty((pw.T, pw.D // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty(R.nvr_sf_bytes(pw.T, pw.D, "tiled"), dtype=torch.uint8, device=dev)
    gsa = torch.empty(1, dtype=torch.float32, device=dev)
    wsq = R.new_workspace(R.nvfp4_quantize_workspace_size(pw.T, pw.D), dev)
    ms = _timed_calls(lambda i: R.nvfp4_quantize_act(xs[i % 4], "tiled", codes, sf, gsa, wsq), 200, stream)
    nbytes = pw.T * pw.D * 2 + pw.T * (pw.D // 2 + pw.D // 16)
    out["quantize"] = _hbm_entry(nbytes, ms, hbm, launches_per_call=2,
                                 note="amax kernel + quantize kernel; x read twice (second pass mostly from L2)")
    del xs, xp
    torch.cuda.empty_cache()

    # the grouped expert GEMM on the prefill batch, routed by the router
    # itself (E = 256, k = 8): 256 experts of N = 512 outputs (0.53 GB packed,
    # drawn on the device), y in bf16, then the weighted combine
    pw = WL.WORKLOADS["prefill"]
    xp = torch.from_numpy(WL.make_x(pw).view(np.int16)).view(torch.bfloat16).to(dev)
    gate = R.RouterGate(torch.from_numpy(WL.make_w(pw).view(np.int16)).view(torch.bfloat16).to(dev),
                        torch.from_numpy(WL.make_bias(pw)).to(dev), k=pw.k, routed_scaling=pw.routed_scaling,
                        max_tokens=pw.T)
    ids, wts = gate(xp)
    E, Nx = pw.N, 512
    We = (torch.randn((E, Nx, pw.D), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    Ef, Esf, Eg = R.nvfp4_pack_experts(We)
    del We
    torch.cuda.empty_cache()
    wsm = R.new_workspace(R.nvfp4_moe_gemm_workspace_size(pw.T, pw.D, E, pw.k), dev)
    y = torch.empty((pw.T, pw.k, Nx), dtype=torch.bfloat16, device=dev)
    comb = torch.empty((pw.T, Nx), dtype=torch.float32, device=dev)
    ms = _timed_calls(lambda i: R.nvfp4_moe_gemm(xp, ids, Ef, Esf, Eg, y=y, workspace=wsm), 20, stream)
    nbytes = E * Nx * (pw.D // 2 + pw.D // 16) + pw.T * pw.D * 2 + pw.T * pw.k * (4 + Nx * 2)
    out["moe_gemm"] = _hbm_entry(nbytes, ms, hbm, tokens_per_s=pw.T / (ms / 1e3),
                                 traffic=traffic.get("moe_gemm_kernel"), traffic_kernel="moe_gemm_kernel",
                                 tensor_tflops=2 * pw.T * pw.k * pw.D * Nx / (ms / 1e3) / 1e12,
                                 note="nvfp4_moe_gemm T=4096 routed k=8 over E=256 experts of N=512, D=7168, "
                                      "bf16 y; 4 launches (amax, route, quantize-scatter, grouped GEMM)")
    ms = _timed_calls(lambda i: R.nvfp4_moe_combine(y, wts, out=comb), 50, stream)
    nbytes = pw.T * pw.k * (Nx * 2 + 4) + pw.T * Nx * 4
    out["moe_combine"] = _hbm_entry(nbytes, ms, hbm, traffic=traffic.get("moe_combine"))
    del Ef, Esf, y, xp, gate
    torch.cuda.empty_cache()

    # the decode kernel's own device duration at T = 1: 64 back-to-back calls
    # in one CUDA graph (programmatic launch hides each launch's latency; a
    # call's work starts when its predecessor's ends), median over replays
    dw = WL.WORKLOADS["decode"]
    gate = R.RouterGate(torch.from_numpy(WL.make_w(dw).view(np.int16)).view(torch.bfloat16).to(dev),
                        torch.from_numpy(WL.make_bias(dw)).to(dev), k=dw.k, routed_scaling=dw.routed_scaling,
                        max_tokens=1)
    xd = torch.from_numpy(WL.make_x(dw.with_T(1)).view(np.int16)).view(torch.bfloat16).to(dev)
    s2 = torch.cuda.Stream()
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s2):
        for _ in range(3):
            gate(xd)
    torch.cuda.current_stream().wait_stream(s2)
    n_calls = 64
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n_calls):
            gate(xd)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    durs = []
    for _ in range(21):
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        durs.append(e0.elapsed_time(e1) / n_calls)
    durs.sort()
    ms = durs[len(durs) // 2]
    nbytes = dw.N * (dw.D // 2 + dw.D // 16) + dw.D * 2 + dw.N * 4 + dw.k * 8
    out["decode_kernel_T1"] = _hbm_entry(nbytes, ms, hbm, traffic=traffic.get("decode_router"),
                                         p10_ms=durs[2], p90_ms=durs[-3],
                                         note="latency-bound: 64 back-to-back calls in one graph, per call")
    return out


def ctypes_array(events):
    import ctypes
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def run_reference(args, rank):
    """The CPU oracle, as it stands, on the host cores (rank 0 only).  Each of
    the K timed steps routes n consecutive tokens of the T=4096 prefill batch
    (with the whole batch's gsa), n sized from one calibration slice so that
    the W + K steps take about a minute in all; consecutive steps' tokens go
    through the oracle in slices of up to 64 rows (its per-call cost)."""
    if rank != 0:
        return None
    from oracle import pipeline, quantize as Q, gemm, router
    w = WL.WORKLOADS["prefill"]
    x32 = WL.bf16_bits_to_float32(WL.make_x(w))
    W_np = WL.make_w(w)
    bias = WL.make_bias(w)
    wq, wsc, wg = pipeline.pack_weight(WL.bf16_bits_to_float32(W_np))
    gsa = Q.global_scale(x32)

    def route_tokens(total, r0):
        """Route `total` tokens from row r0 on (wrapping), 64 rows per call."""
        done = 0
        while done < total:
            n = min(64, total - done, w.T - r0)
            rows = x32[r0:r0 + n]
            xq, xs, _ = Q.quantize(rows, gsa=gsa)
            L, _ = gemm.logits(xq, xs, gsa, wq, wsc, wg)
            router.route(L, bias, w.k, w.routed_scaling, w.raw)
            done += n
            r0 = (r0 + n) % w.T
        return r0

    t0 = time.perf_counter()
    route_tokens(64, 0)                                   # calibration slice
    rate = 64.0 / (time.perf_counter() - t0)
    n = int(min(64, max(1, round(rate * 60.0 / (args.steps + args.warmup)))))
    r0 = route_tokens(args.warmup * n, 0)
    t0 = time.perf_counter()
    route_tokens(args.steps * n, r0)
    el = time.perf_counter() - t0
    done = args.steps * n
    value = done / el
    sample = ("%d steps of %d tokens of the T=4096 prefill batch (batch gsa), routed in slices of up to "
              "64 rows: NumPy quantize + float64 GEMM + epilogue" % (args.steps, n))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "prefill router T=4096 D=7168 E=256 k=8 (CPU oracle sample)",
                       "T": w.T, "D": w.D, "E": w.N, "k": w.k},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def profile_launches():
    """One warm-up call and one measured call of every hot path, for a
    profiler's launch filter (each call reads its inputs cold under ncu):
    the prefill router (fused_qgemm_kernel), the standalone quantizer on the
    prefill batch (amax_bulk_kernel, quantize_kernel), the decode router at T = 1
    (decode_router_kernel), the N = 129280 raw head at T = 32 with k = 8 and
    as a bf16 linear (gemm_stream_kernel), the grouped expert GEMM and its
    combine on the prefill routing (moe_* kernels), the adversarial batch
    (T = 16384, E = 384: the one-launch kernel for 384 experts) and the hash
    router.  Holds about 2 GB of device memory."""
    import torch
    import nvfp4_router_gate_gb300 as R
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    pw = WL.WORKLOADS["prefill"]
    xp = bf16(WL.make_x(pw))
    gate = R.RouterGate(bf16(WL.make_w(pw)), torch.from_numpy(WL.make_bias(pw)).to(dev), k=pw.k,
                        routed_scaling=pw.routed_scaling, max_tokens=pw.T)
    for _ in range(2):
        ids, wts = gate(xp)
    # the standalone quantizer on the prefill batch (amax_bulk_kernel, quantize_kernel)
    codes = torch.empty((pw.T, pw.D // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty(R.nvr_sf_bytes(pw.T, pw.D, "tiled"), dtype=torch.uint8, device=dev)
    gsa = torch.empty(1, dtype=torch.float32, device=dev)
    wsq = R.new_workspace(R.nvfp4_quantize_workspace_size(pw.T, pw.D), dev)
    for _ in range(2):
        R.nvfp4_quantize_act(xp, "tiled", codes, sf, gsa, wsq)
    del codes, sf
    dw = WL.WORKLOADS["decode"]
    dgate = R.RouterGate(bf16(WL.make_w(dw)), torch.from_numpy(WL.make_bias(dw)).to(dev), k=dw.k,
                         routed_scaling=dw.routed_scaling, max_tokens=1)
    xd = bf16(WL.make_x(dw.with_T(1)))
    for _ in range(2):
        dgate(xd)
    wn = WL.WORKLOADS["wide_n"]
    W = (torch.randn((wn.N, wn.D), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    Wf, Wsf, wg = R.nvfp4_pack_weight(W)
    del W
    xw = torch.randn((wn.T, wn.D), generator=g, device=dev).to(torch.bfloat16)
    for _ in range(2):
        R.router_gate_topk(xw, Wf, Wsf, wg, None, 8, 1.0, True)
    for _ in range(2):
        R.nvfp4_linear(xw, Wf, Wsf, wg, out_dtype=torch.bfloat16)
    del Wf, Wsf
    torch.cuda.empty_cache()
    We = (torch.randn((pw.N, 512, pw.D), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    Ef, Esf, Eg = R.nvfp4_pack_experts(We)
    del We
    for _ in range(2):
        y = R.nvfp4_moe_gemm(xp, ids, Ef, Esf, Eg, out_dtype=torch.bfloat16)
        R.nvfp4_moe_combine(y, wts)
    aw = WL.WORKLOADS["adversarial"]
    agate = R.RouterGate(bf16(WL.make_w(aw)), torch.from_numpy(WL.make_bias(aw)).to(dev), k=aw.k,
                         routed_scaling=aw.routed_scaling, max_tokens=aw.T)
    xa = bf16(WL.make_x(aw))
    for _ in range(2):
        agate(xa)
    del xa, agate
    hw = WL.HASH_ROUTER
    table = torch.from_numpy(WL.make_hash_table(hw)).to(dev)
    tids = torch.from_numpy(WL.make_token_ids(hw)).to(dev)
    for _ in range(2):
        R.router_hash_topk(tids, table, hw.n_experts, hw.routed_scaling)
    torch.cuda.synchronize()
    print(json.dumps({"profile_launches": "ok"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-extra", action="store_true")
    ap.add_argument("--oracle-sample", type=float, default=None,
                    help="time the CPU oracle for this many seconds, print one JSON line and exit")
    ap.add_argument("--profile-launches", action="store_true",
                    help="run each hot path twice and exit (for a profiler's launch filter)")
    args = ap.parse_args()
    if args.oracle_sample is not None:
        print(oracle_sample_json(args.oracle_sample))
        return
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank)
        if out is not None:
            print(json.dumps(out))
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    from nvfp4_router_gate_gb300 import build
    build.build()
    if args.profile_launches:
        profile_launches()
        return
    out = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
