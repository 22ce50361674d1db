#!/usr/bin/env python
"""Benchmark of the routed NVFP4 MoE expert layer on GB300.

One step = per-token quantization + the W4A4 forward (routing permutation,
FC1 grouped GEMM with fused activation, FC2-input requant, FC2 grouped GEMM,
deterministic finalize) over one batch of T synthetic tokens, replayed from a
CUDA graph.  Inputs are resident in HBM; L2 is flushed (a 256 MB write)
between timed steps, outside the per-step CUDA events.

Default workload: the MoE layer of the pages' benchmark shape on one GPU
(FlashInfer fork PR #1, "Performance and reproduction": hidden 7168,
intermediate 3072, 384 experts, top-6, SwiGLU) at 4096 tokens.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead
(bounded samples on the host cores).  Multi-GPU runs (torchrun) are replicas:
every rank runs the same workload on its own GPU, no collective on the data
path; value = all tokens / max-over-ranks time.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import nvfp4_token_routed_gb300 as M  # noqa: E402
from nvfp4_token_routed_gb300 import workloads as W  # noqa: E402

METRIC = "MoE-layer tokens/s and µs/layer at 1 GB300"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = W.PAGES_E384.name
DEFAULT_T = 4096
# the oracle's samples of large workloads use at most this many distinct experts
# (its weight preparation, outside the timed region, grows with the experts)
ORACLE_MAX_EXPERTS = 24


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.ALL))
    p.add_argument("--T", type=int, default=-1,
                   help="token count (default: 4096 for the default workload, else the "
                        "workload's own)")
    p.add_argument("--E", type=int, default=0, help="override the expert count (profiling cases)")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--w4a16", action="store_true", help="time the BF16-activation variant")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--with-router", action="store_true",
                   help="start each step from router logits: top-K router kernel + the layer")
    p.add_argument("--prep", action="store_true",
                   help="time in-place weight re-preparation (a refit) instead of the forward")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# Nominal dense tensor rates relative to bf16 (2.25 PFLOP/s): FP4 13.5, so x6.
FP4_OVER_BF16 = 6.0
FALLBACK_BF16_SUSTAINED_TFLOPS = 1700.0


def fp4_peak():
    """Dense NVFP4 tensor peak in TFLOP/s: the measured sustained bf16 GEMM rate
    (the GEMMs run inside a step of several launches) times the nominal
    FP4 / bf16 ratio."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]) * FP4_OVER_BF16, "measured bf16 sustained x 6"
    return FALLBACK_BF16_SUSTAINED_TFLOPS * FP4_OVER_BF16, "fallback bf16 sustained x 6"


def algorithmic_flops(wl, R):
    """Routed work of the two grouped GEMMs: 2 R H N1 (FC1) and 2 R I H (FC2)."""
    N1 = 2 * wl.I if wl.act == "swiglu" else wl.I
    return {"fc1": 2.0 * R * wl.H * N1, "fc2": 2.0 * R * wl.I * wl.H}


def kernel_hash():
    h = hashlib.sha256()
    for f in ("gemm_w4a4.cu", "gemm_common.cuh", "ptx.cuh", "internal.h"):
        with open(os.path.join(ROOT, "nvfp4_token_routed_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(workload):
    """DRAM bytes per FC1 launch from the committed ncu summary, if it still
    describes the current kernel source."""
    path = os.path.join(ROOT, "profiles", "fc1_gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("per_launch_bytes", {}).get(workload)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def workload_of(args):
    wl = W.ALL[args.workload]
    T = args.T if args.T >= 0 else (DEFAULT_T if args.workload == DEFAULT_WORKLOAD else 0)
    if T:
        wl = wl.with_T(T)
    if getattr(args, "E", 0):
        wl = wl.with_E(args.E)
    return wl


def make_inputs(wl, device):
    big = wl.E * (wl.N1 + wl.I) * wl.H > 2e9
    gen_dev = device if big else "cpu"
    x = W.make_x(wl, device=gen_dev)
    w1, w2 = W.make_weights(wl, device=gen_dev)
    ids, wts = W.make_routing(wl, device=gen_dev)
    return x, w1, w2, ids, wts


def routes_and_experts(wl, ids):
    idsn = ids.cpu().numpy().ravel()
    valid = idsn[(idsn >= 0) & (idsn < wl.E)]
    return int(valid.size), int(np.unique(valid).size)


def algorithmic_bytes(wl, R, U, w4a16=False):
    """Algorithmic DRAM bytes of the layer and of its two GEMM launches, as the
    scope table defines them: each touched expert's codes and E4M3 scales once
    (9/16 byte per weight), the tokens (bf16 in, NVFP4 out of the quantizer and
    into FC1), the FC2 input (NVFP4 written by the FC1 stage, read by FC2), the
    bf16 route rows (written by FC2, read by the finalize), the output and the
    routing ids and scores.  Workspace-only traffic (the permuted token copy, the
    fp32 activated rows) is not algorithmic; `workspace_bytes` reports it.
    W4A16 has no token or FC2-input quantization: its GEMMs read bf16 rows."""
    T, H, I, K = wl.T, wl.H, wl.I, wl.K
    N1 = 2 * I if wl.act == "swiglu" else I
    w1 = U * N1 * H * 9 / 16
    w2 = U * H * I * 9 / 16
    if w4a16:
        fc1 = w1 + 2 * T * H + 2 * R * I
        fc2 = w2 + 2 * R * I + 2 * R * H
        layer = w1 + w2 + 2 * T * H + 2 * 2 * R * I + 4 * R * H + 2 * T * H + 8 * T * K
        # the f16 copies of the token rows (written, read) and of the handoff
        # rows (the bf16 rows read twice by the conversion, the f16 rows written)
        ws = 2 * 2 * R * H + 3 * 2 * R * I
    else:
        fc1 = w1 + T * H * 9 / 16 + R * I * 9 / 16
        fc2 = w2 + R * I * 9 / 16 + 2 * R * H
        layer = (w1 + w2 + 2 * T * H + 2 * T * H * 9 / 16 + 2 * R * I * 9 / 16 + 4 * R * H
                 + 2 * T * H + 8 * T * K)
        ws = 2 * R * H * 9 / 16 + 2 * 4 * R * I + 8 * R  # permuted copy; fp32 rows, row scales
    return {"fc1": fc1, "fc2": fc2, "layer": layer, "workspace": ws}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(wl, ids, max_tokens):
    """Token indices of the oracle's bounded sample: a prefix of the batch, cut
    where it would need more than ORACLE_MAX_EXPERTS distinct experts (small
    layers: every expert is prepared once and the prefix is only cut at
    max_tokens)."""
    idsn = ids.cpu().numpy()
    full = wl.E * (wl.N1 + wl.I) * wl.H <= 1e9
    n, used = 0, set()
    while n < min(wl.T, max_tokens):
        new = used | {int(e) for e in idsn[n] if 0 <= e < wl.E}
        if not full and n > 0 and len(new) > ORACLE_MAX_EXPERTS:
            break
        used, n = new, n + 1
    return np.arange(n)


def oracle_sample_runner(wl, x, w1, w2, ids, wts, sample):
    """Prepare the oracle's weights for the experts the sample tokens use (outside
    any timing) and return a function that runs the oracle (quantize + W4A4
    forward) on a sub-range of the sample and returns its seconds."""
    from oracle import oracle as O

    idsn = ids.cpu().numpy().astype(np.int32)[sample]
    wtn = wts.cpu().numpy().astype(np.float32)[sample]
    xs = W.bf16_bits(x[torch.as_tensor(sample, device=x.device)].cpu())
    used = np.unique(idsn[(idsn >= 0) & (idsn < wl.E)])
    idx = torch.as_tensor(used, dtype=torch.long, device=w1.device)
    Wt = O.Weights(W.bf16_bits(w1.index_select(0, idx).cpu()),
                   W.bf16_bits(w2.index_select(0, idx).cpu()))
    remap = np.full(wl.E, -1, np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    sub_ids = np.where(idsn >= 0, remap[np.clip(idsn, 0, None)], -1).astype(np.int32)

    def run(start, n):
        sl = slice(start, start + n)
        t0 = time.perf_counter()
        c, f, s = O.quantize_tokens(xs[sl])
        O.forward_w4a4(Wt, c, f, s, sub_ids[sl], wtn[sl], used.size, wl.H, wl.I, wl.act)
        return time.perf_counter() - t0

    return run, O.num_threads(), int(used.size)


def cpu_baseline(wl, x, w1, w2, ids, wts, seconds):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload: the sample is run whole, repeatedly, until about `seconds` of
    oracle work have been timed."""
    sample = oracle_sample(wl, ids, max_tokens=256)
    run, cores, n_exp = oracle_sample_runner(wl, x, w1, w2, ids, wts, sample)
    n = sample.size
    total, reps = 0.0, 0
    while total < seconds or reps == 0:
        total += run(0, n)
        reps += 1
    return {"value": n * reps / total, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {wl.T} tokens of {wl.name} (all their routes, {n_exp} "
                      f"experts prepared outside the timing), quantize + W4A4 forward, "
                      f"run {reps}x, {total:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = workload_of(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"  # input generation only
    x, w1, w2, ids, wts = make_inputs(wl, dev)
    sample = oracle_sample(wl, ids, max_tokens=64)
    run, cores, n_exp = oracle_sample_runner(wl, x, w1, w2, ids, wts, sample)
    del w1, w2
    budget = 150.0  # seconds for warmup + timed steps
    steps = args.steps
    # each step is a bounded sample: one token (all its routes), cycling over the sample
    times = []
    for i in range(args.warmup):
        run(i % sample.size, 1)
    for i in range(steps):
        times.append(run(i % sample.size, 1))
        if sum(times) > budget:
            break
    mean = sum(times) / len(times)
    value = 1 / mean
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                       "K": wl.K, "act": wl.act},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"1 token per step (all its routes), cycling over the "
                                       f"first {sample.size} of the {wl.T} tokens ({n_exp} "
                                       f"experts prepared outside the timing); {len(times)} "
                                       f"steps run of {steps} asked (150 s budget)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def max_over_ranks(value, world, device=None):
    """The largest `value` over all ranks (the slowest replica sets the time);
    the identity on one rank.  The tensor lives where the backend reduces it."""
    if world <= 1:
        return float(value)
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_step, steps, max_total_ms):
    """Whole-job tokens/s of `world` independent replicas: every rank processes
    tokens_per_step per step; the job takes the slowest rank's time."""
    return world * tokens_per_step * steps / (max_total_ms / 1e3)


def run_ours(args, rank, world, local_rank):
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = workload_of(args)
    x, w1, w2, ids, wts = make_inputs(wl, dev)
    x_d, ids_d, wts_d = x.to(dev), ids.to(dev), wts.to(dev)
    w = M.prepare_weights(w1.to(dev), w2.to(dev), wl.act)
    T, H, K = wl.T, wl.H, wl.K
    codes = torch.empty(T, H // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(T, H // 16, dtype=torch.uint8, device=dev)
    scale = torch.empty(T, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = M.workspace(w, T, K, w4a16=args.w4a16, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    logits_d = None
    if args.with_router:
        g = torch.Generator(device=dev)
        g.manual_seed(W.BASE_SEED + 5)
        logits_d = torch.randn(T, wl.E, generator=g, device=dev)

    # GEMM spans (profiling pass only): the earliest CTA start and latest CTA end
    # of each grouped GEMM launch by the GPU's global timer, reset every step
    span = torch.zeros(4, dtype=torch.int64, device=dev)
    span_init = torch.tensor([-1, 0, -1, 0], dtype=torch.int64, device=dev)
    span_on = [False]

    def step():
        if span_on[0]:
            span.copy_(span_init)
        if logits_d is not None:
            M.moe_nvfp4_route_topk(logits_d, ids_d, wts_d, stream)
        if args.w4a16:
            M.moe_nvfp4_forward_w4a16(w.dims, w, x_d, ids_d, wts_d, out, ws, stream)
            return
        M.moe_nvfp4_quantize_tokens(x_d, codes, sf, scale, stream)
        M.moe_nvfp4_forward(w.dims, w, codes, sf, scale, ids_d, wts_d, out, ws, stream)

    with torch.cuda.stream(stream):
        step()  # first call runs the device check outside capture
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws, stream) == 0

    def capture():
        if args.no_graph:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        torch.cuda.synchronize()
        return g

    graph = capture()

    def run_step(g):
        if g is not None:
            g.replay()
        else:
            step()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            run_step(graph)
    torch.cuda.synchronize()

    # ---- the timed region: K steps, each bracketed by events on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            run_step(graph)
            ends[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None

    # ---- per-kernel times: the same K steps again with stage markers recorded by
    # the library between its kernels ([1] after routing, [2] after FC1, ...).
    # Markers stop kernels from overlapping their launch with the previous
    # kernel, so they get a pass of their own.
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    with torch.cuda.stream(stream):
        for e in marks:
            e.record()
    torch.cuda.synchronize()
    M.moe_nvfp4_profile_events(marks)
    span_on[0] = True
    M.moe_nvfp4_profile_spans(span)
    graph_marked = capture()
    M.moe_nvfp4_profile_events([])
    M.moe_nvfp4_profile_events(marks)
    fc1_ms, fc2_ms, fc1_span, fc2_span = [], [], [], []
    stage_ms = []  # per step: the five intervals between the library's stage markers
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()
            run_step(graph_marked)
            marks[5].synchronize()
            fc1_ms.append(marks[1].elapsed_time(marks[2]))
            fc2_ms.append(marks[3].elapsed_time(marks[4]))
            stage_ms.append([marks[j].elapsed_time(marks[j + 1]) for j in range(5)])
            sv = span.tolist()
            if sv[1] > 0:
                fc1_span.append((sv[1] - sv[0]) * 1e-6)   # ns -> ms
            if sv[3] > 0:
                fc2_span.append((sv[3] - sv[2]) * 1e-6)
    torch.cuda.synchronize()
    M.moe_nvfp4_profile_events([])
    M.moe_nvfp4_profile_spans(None)
    span_on[0] = False

    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    value = replica_throughput(world, T, args.steps, total_ms)

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs from pinned host memory and reads its output back; as a
    # serving loop would, the copies of a step overlap the computation of its
    # neighbours: two sets of device buffers, a stream for each direction, and
    # events ordering each buffer's copy in, use and copy out.  The timed
    # region runs from before the first step's input copy to the end of the
    # last step's output copy.  (Weights and inputs exceed L2, so no flush.)
    nb = 2
    x_h = x.cpu().pin_memory()
    ids_h = ids.cpu().pin_memory()
    wts_h = wts.cpu().pin_memory()
    logits_h = logits_d.cpu().pin_memory() if logits_d is not None else None
    out_h = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    x_e = [torch.empty_like(x_d) for _ in range(nb)]
    ids_e = [torch.empty_like(ids_d) for _ in range(nb)]
    wts_e = [torch.empty_like(wts_d) for _ in range(nb)]
    logits_e = [torch.empty_like(logits_d) if logits_d is not None else None for _ in range(nb)]
    out_e = [torch.empty_like(out) for _ in range(nb)]
    h2d_s = torch.cuda.Stream(device=dev)
    d2h_s = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(nb)]
    ev_done = [torch.cuda.Event() for _ in range(nb)]
    ev_out = [torch.cuda.Event() for _ in range(nb)]
    e2e_steps = min(args.steps, 500)

    def e2e_step(i):
        b = i % nb
        with torch.cuda.stream(h2d_s):
            if i >= nb:
                h2d_s.wait_event(ev_done[b])       # step i - nb is done with buffer b
            x_e[b].copy_(x_h, non_blocking=True)
            if logits_h is not None:
                logits_e[b].copy_(logits_h, non_blocking=True)
            else:
                ids_e[b].copy_(ids_h, non_blocking=True)
                wts_e[b].copy_(wts_h, non_blocking=True)
            ev_in[b].record(h2d_s)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[b])
            if i >= nb:
                stream.wait_event(ev_out[b])       # step i - nb's output has been read back
            if logits_h is not None:
                M.moe_nvfp4_route_topk(logits_e[b], ids_e[b], wts_e[b], stream)
            if args.w4a16:
                M.moe_nvfp4_forward_w4a16(w.dims, w, x_e[b], ids_e[b], wts_e[b], out_e[b], ws,
                                          stream)
            else:
                M.moe_nvfp4_quantize_tokens(x_e[b], codes, sf, scale, stream)
                M.moe_nvfp4_forward(w.dims, w, codes, sf, scale, ids_e[b], wts_e[b], out_e[b], ws,
                                    stream)
            ev_done[b].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_done[b])
            out_h[b].copy_(out_e[b], non_blocking=True)
            ev_out[b].record(d2h_s)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e_s = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    e_s.record(h2d_s)
    for i in range(e2e_steps):
        e2e_step(i)
    e_e.record(d2h_s)
    e_e.synchronize()
    e2e_ms = e_s.elapsed_time(e_e)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = replica_throughput(world, T, e2e_steps, e2e_ms)
    h2d = x_h.numel() * 2 + (logits_h.numel() * 4 if logits_h is not None
                             else ids_h.numel() * 4 + wts_h.numel() * 4)
    d2h = out_h[0].numel() * 2

    if rank != 0:
        return
    R, U = routes_and_experts(wl, ids)
    B = algorithmic_bytes(wl, R, U, args.w4a16)
    fc1_mean = statistics.fmean(fc1_ms)
    fc2_mean = statistics.fmean(fc2_ms)
    fc1_span_mean = statistics.fmean(fc1_span) if fc1_span else None
    fc2_span_mean = statistics.fmean(fc2_span) if fc2_span else None
    # the W4A4 forward runs FC1, the FC2-input requant and FC2 as one launch when
    # T*K <= min(2048, 8*E) (moe_nvfp4.h): the roofline is then that launch's,
    # FC1 and FC2 bytes over the FC1 marker interval (the FC2 one is empty)
    fused = (not args.w4a16) and T * K <= min(2048, 8 * wl.E)
    kernel_bytes = B["fc1"] + (B["fc2"] if fused else 0)
    hbm, src = peaks()
    achieved = kernel_bytes / (fc1_mean * 1e-3) / 1e9
    layer_gbs = B["layer"] / (ms_per_step * 1e-3) / 1e9
    # Bound of the kernel (and of the layer): the larger of its FLOPs at the
    # dense tensor peak of its input type and its bytes at the HBM rate.
    F = algorithmic_flops(wl, R)
    tpeak, tsrc = fp4_peak()
    if args.w4a16:
        tpeak, tsrc = tpeak / FP4_OVER_BF16, tsrc.replace(" x 6", "")
    kernel_flops = F["fc1"] + (F["fc2"] if fused else 0)
    layer_flops = F["fc1"] + F["fc2"]
    kernel_tensor = kernel_flops / (tpeak * 1e12) > kernel_bytes / (hbm * 1e9)
    layer_tensor = layer_flops / (tpeak * 1e12) > B["layer"] / (hbm * 1e9)
    kernel_tflops = kernel_flops / (fc1_mean * 1e-3) / 1e12
    layer_tflops = layer_flops / (ms_per_step * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "us_per_layer": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 x nvfp4" if args.w4a16 else "nvfp4",
        "data": "synthetic (seeded N(0,1)-family inputs)",
        "config": {"workload": wl.name + ("+w4a16" if args.w4a16 else "") + ("+router" if args.with_router else ""),
                   "T": T, "H": H, "I": wl.I, "E": wl.E, "K": K,
                   "act": wl.act, "routes": R, "experts_touched": U,
                   "l2": "flushed (256 MB write) between timed steps",
                   "graph": graph is not None, "parallelism": f"replicas x{world}"},
        "roofline": {"kernel": ("fc1 grouped GEMM (gemm_w4a16_kernel<SwiGLU|ReLU2>)" if args.w4a16
                                else "fused FC1 + requant + FC2 (gemm_w4a4_kernel, one launch)"
                                if fused else "fc1 grouped GEMM (gemm_w4a4_kernel<SwiGLU|ReLU2>)"),
                     **({"bound": "tensor", "achieved": kernel_tflops, "peak": tpeak,
                         "unit": "TFLOP/s", "frac": kernel_tflops / tpeak, "peak_source": tsrc,
                         "hbm_gbs": achieved, "hbm_frac": achieved / hbm}
                        if kernel_tensor else
                        {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": src,
                         "tflops": kernel_tflops, "tensor_frac": kernel_tflops / tpeak}),
                     "algorithmic_flops": kernel_flops,
                     "traffic": None if fused else traffic_for(wl.name),
                     "algorithmic_bytes": kernel_bytes,
                     "workspace_bytes": B["workspace"],
                     "kernel_us": fc1_mean * 1e3, "fc2_kernel_us": fc2_mean * 1e3,
                     "fc2_frac": (None if fused else
                                  B["fc2"] / (fc2_mean * 1e-3) / 1e9 / hbm),
                     "fc2_tensor_frac": (None if fused else
                                         F["fc2"] / (fc2_mean * 1e-3) / 1e12 / tpeak),
                     "timing": "CUDA events recorded by the library around the FC1 launch, "
                               "over a second pass of the same K steps",
                     # the launch's own span (earliest CTA start to latest CTA end by the
                     # GPU's global timer, same pass): the event interval minus launch latency
                     "kernel_span_us": None if fc1_span_mean is None else fc1_span_mean * 1e3,
                     "span_frac": (None if fc1_span_mean is None else
                                   kernel_bytes / (fc1_span_mean * 1e-3) / 1e9 / hbm),
                     "fc2_span_us": None if fc2_span_mean is None else fc2_span_mean * 1e3},
        "layer_roofline": ({"bound": "tensor", "algorithmic_flops": layer_flops,
                            "achieved": layer_tflops, "peak": tpeak, "unit": "TFLOP/s",
                            "frac": layer_tflops / tpeak, "hbm_frac": layer_gbs / hbm}
                           if layer_tensor else
                           {"bound": "hbm", "algorithmic_bytes": B["layer"],
                            "achieved": layer_gbs, "peak": hbm, "unit": "GB/s",
                            "frac": layer_gbs / hbm, "tensor_frac": layer_tflops / tpeak}),
        # the layer stage by stage: CUDA events recorded by the library between its
        # kernels in the marked pass (each interval includes its kernels' launch
        # latency; with the one-launch path requant and FC2 are empty)
        "stages_us": {name: statistics.fmean(v[j] for v in stage_ms) * 1e3
                      for j, name in enumerate(("route", "fc1", "requant", "fc2", "finalize"))},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copies": "pinned host memory, each step's input and output copies overlapping "
                          "its neighbours' computation (2 buffer sets, a stream per direction)"},
        # the forward's own count (moe_nvfp4_forward_kernel_count) plus the token
        # quantization (W4A4) and the router, when the step runs them
        "gpu_launches": (M.moe_nvfp4_forward_kernel_count(w.dims, T, K, args.w4a16)
                         + (0 if args.w4a16 else 1) + (1 if args.with_router else 0)) * args.steps,
        "clocks": clocks,
        "wall_s": t_wall,
    }
    if world == 1 and not args.no_cpu_baseline and not args.w4a16:
        line["cpu_baseline"] = cpu_baseline(wl, x, w1, w2, ids, wts, args.cpu_seconds)
    print(json.dumps(line), flush=True)


# Refit shape: the pages time a full requantization of 32 local experts of a
# Nemotron-3 Super layer (hidden 2688; Megatron-LM PR #8262, "Why CuTe DSL" and
# "Performance").  They do not print the expert intermediate size; 2048 (the
# intermediate of the pages' GB300 table) stands in for it, squared ReLU.
PREP_E, PREP_H, PREP_I = 32, 2688, 2048


def run_prep(args):
    """In-place moe_nvfp4_prepare_weights of PREP_E experts, CUDA events per call,
    L2 flushed between calls; the bound is HBM (BF16 read + NVFP4 written)."""
    dev = torch.device("cuda", 0)
    wl = W.Workload("relu2_prep_E32_H2688_I2048", 1, PREP_H, PREP_I, PREP_E, 1, "relu2")
    w1, w2 = W.make_weights(wl, device=dev)
    w = M.prepare_weights(w1, w2, wl.act)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        M.prepare_weights(w1, w2, wl.act, out=w)
    torch.cuda.synchronize()
    steps = min(args.steps, 200)
    ms = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        M.prepare_weights(w1, w2, wl.act, out=w)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    mean = statistics.fmean(ms)
    read = 2 * (w1.numel() + w2.numel()) * 2  # amax pass + quantize pass over the BF16 stacks
    written = w.nbytes()
    hbm, src = peaks()
    gbs = (read + written) / (mean * 1e-3) / 1e9
    print(json.dumps({
        "metric": "in-place weight re-preparation (refit) of 32 experts", "value": mean * 1e3,
        "unit": "us", "higher_is_better": False, "steps": steps, "dtype": "bf16 -> nvfp4",
        "data": "synthetic", "config": {"workload": wl.name, "E": PREP_E, "H": PREP_H, "I": PREP_I,
                                        "act": "relu2", "l2": "flushed between calls"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "peak_source": src, "bytes": read + written},
        "context": "pages: 16.7 ms for 32 Nemotron-3 Super experts with CuTe DSL (other shape)",
    }), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.prep:
        if rank == 0:
            run_prep(args)
        return
    if world > 1:
        torch.distributed.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
