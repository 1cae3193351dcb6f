#!/usr/bin/env python3
"""Throughput of the dropless MoE layer hot path (router top-K -> permute ->
grouped SwiGLU GEMMs -> combine) on one node, one process per GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one forward pass of the whole layer over one batch of T tokens of
the workload (default: Mixtral-like, T=8192, H=4096, E=8, top-2, F=14336, bf16,
synthetic seeded inputs); for the training workload (heavy skew) it is the
forward and the whole layer's backward from the gradient of its output
(combine, expert-MLP dgrad/dx/wgrad, permute and router backward). For the
2,304-expert workload the permute, GEMMs and combine consume compact routes
with about 2 % of entries -1 (the router's output, masked once before timing;
the router still runs every step). Each rank runs the same layer on its own
batch (replicas: weak scaling, no collective on the data path); --gpus N
without a launcher starts the N ranks itself (torch's launcher, one process
per GPU). Rank 0 prints one JSON line:

  value      tokens/s over all ranks, inputs resident in HBM; the step (every
             kernel of it) captured once as a CUDA graph -- the path is
             graph-capturable, group sizes stay on the device -- and every
             timed replay bracketed by CUDA events on the launching stream, L2
             flushed (512 MiB write, then a 512 MiB read that evicts the write's dirty
             lines) before every timed step, outside the timed
             interval;
  e2e        the same metric through MoELayer.forward_host with pinned host
             tensors, every call's input copy and output copy inside the timed
             interval: K consecutive calls with the overlapped transfer (each
             call's input copy and the previous call's output copy run on the
             copy engines beside the compute) timed as one region; "serial"
             beside it times each call alone with the direct transfer (x read
             and y written in host memory by the permute and the combine). A
             training layer copies x in and y out, one call at a time;
  roofline   the dominant kernel (grouped GEMM, up projection with SwiGLU):
             algorithmic FLOPs (2 * R * H * 2F) / its mean event-timed duration,
             against the measured dense bf16 burst peak (the timed loop is short
             and runs at maximum SM clock), the sustained figure given beside it;
  stages     mean per-stage time and the bandwidth / FLOP rate of each stage,
             from CUDA events recorded inside the captured graph between stages
             (external event nodes, read after each replay); where the CUDA
             runtime cannot be loaded for that, from the same steps run eagerly;
  workloads  the other workloads (DeepSeek-V3-like MXFP8, 2,304 experts, heavy-skew
             training step, NVFP4, sigmoid router), timed the same way after the
             headline one: step time, tokens/s, per-stage rates and their
             dominant kernel's roofline;
  cpu_baseline  the CPU oracle (single-threaded C) timed on this host on a
             bounded sample of the same workload (rank 0, N=1 only), with the
             host's core count beside the one thread it uses.

--impl reference times that oracle alone as the reference arm (ms_per_step: the
wall time of each timed sample; value: the whole batch over the extrapolated
step time).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; grouped-GEMM TFLOPS and permute/combine GB/s vs peak"
KERNEL_NAMES = {"gemm_up": "grouped_gemm_kernel<UP> (GEMM up + SwiGLU)",
                "gemm_down": "grouped_gemm_kernel<DOWN> (GEMM down)",
                "dgrad_dh": "grouped_gemm_kernel<DGRAD> (dh + SwiGLU backward)"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) per launch of a workload's dominant kernel, from an ncu capture,
# keyed by (workload, stage, hash of the GEMM's sources); a changed kernel reports null.
TRAFFIC_BY_SOURCE = {
    # Mixtral-like GEMM up: 2.406 GB read + 0.462 GB written (ncu dram__bytes_read.sum / _write.sum,
    # full size, one pass)
    ("mixtral", "gemm_up", "0ce0a4a81f5de628"): 2.406117632e9 + 0.46172416e9,
}


def kernel_source_hash() -> str:
    """Hash of the grouped GEMM's own sources (the kernel file and its PTX wrappers)."""
    h = hashlib.sha1()
    for f in ("gemm.cu", "sm100_ptx.cuh"):
        with open(os.path.join(ROOT, "dropless_moe_expert_router_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1].split()[0]))
                smax.append(float(r[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


class GraphStageEvents:
    """CUDA events recorded inside a captured graph as external event nodes
    (cudaEventRecordWithFlags with cudaEventRecordExternal), read back after each replay:
    per-stage device times of a graph replay, with no host launch gaps between stages.
    Uses the CUDA runtime library through ctypes; `ok` is False where it cannot be loaded."""

    def __init__(self, n: int):
        import ctypes
        import glob
        self.C = ctypes
        self.rt = None
        cands = glob.glob("/usr/local/cuda/lib64/libcudart.so*") + glob.glob("/usr/local/cuda/lib/libcudart.so*")
        for c in sorted(cands, reverse=True):
            try:
                self.rt = ctypes.CDLL(c)
                break
            except OSError:
                continue
        self.ev = []
        self.ok = self.rt is not None
        for _ in range(n if self.ok else 0):
            e = ctypes.c_void_p()
            if self.rt.cudaEventCreate(ctypes.byref(e)) != 0:
                self.ok = False
                break
            self.ev.append(e)

    def record(self, j: int, stream) -> None:
        if self.rt.cudaEventRecordWithFlags(self.ev[j], self.C.c_void_p(stream.cuda_stream), 1) != 0:
            self.ok = False

    def elapsed_ms(self, a: int, b: int) -> float:
        ms = self.C.c_float()
        if self.rt.cudaEventElapsedTime(self.C.byref(ms), self.ev[a], self.ev[b]) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return float(ms.value)


def gpu_id_for(dev_index: int) -> str:
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        return str(dev_index)


# ---------------------------------------------------------------- oracle timing
def oracle_sample(wl, x_bits, logits_np, yperm_bits, gemm_rows: int, w_bits):
    """Time the CPU oracle on one bounded sample of the workload: router, permute and
    combine over every token, the grouped MLP on `gemm_rows` permuted rows; returns
    (seconds extrapolated to the whole batch, description)."""
    import numpy as np
    import oracle as O
    t0 = time.perf_counter()
    if wl.score == "sigmoid":
        from dropless_moe_expert_router_gb300 import workloads as W
        eb = W.expert_bias(wl)
        ids, probs = O.route_sigmoid_topk(logits_np, wl.K, bias=None if eb is None else eb.numpy(),
                                          renorm=wl.renorm)
    else:
        ids, probs = O.route_topk(logits_np, wl.K, wl.renorm)
    t1 = time.perf_counter()
    op = O.permute(x_bits, ids, wl.E)
    t2 = time.perf_counter()
    R = op["R"]
    rows = np.linspace(0, R - 1, num=min(gemm_rows, R)).astype(np.int32)
    X = O.Operand(O.MAT_BF16, op["x_perm"])
    Ws = [O.Operand(O.MAT_BF16, w) for w in w_bits]
    O.swiglu_rows(X, *Ws, op["group_offsets"], rows, h_mode=O.H_BF16, want=("y_bf16",))
    t3 = time.perf_counter()
    O.combine(yperm_bits, op["row_map"], probs)
    t4 = time.perf_counter()
    gemm_full = (t3 - t2) * R / max(1, rows.size)
    total = (t1 - t0) + (t2 - t1) + gemm_full + (t4 - t3)
    desc = (f"router, permute and combine over all {wl.T} tokens; grouped SwiGLU MLP on {rows.size} of "
            f"{R} permuted rows, extrapolated by row count"
            + ("" if wl.precision == "bf16" else f" (bf16 operands; the workload's GEMMs run {wl.precision})"))
    return total, desc


def oracle_inputs(wl):
    import numpy as np
    import torch
    from dropless_moe_expert_router_gb300 import workloads as W

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    x = W.x(wl)
    w1, w3, w2 = W.weights(wl)
    return (bits(x), W.logits(wl).numpy(), bits(W.expert_out(wl)), [bits(w1), bits(w3), bits(w2)])


# ---------------------------------------------------------------- our arm
def run_ours(args, wl, rank, world, local_rank, with_e2e=True):
    import torch
    import torch.distributed as dist
    from dropless_moe_expert_router_gb300 import api
    from dropless_moe_expert_router_gb300 import workloads as W
    from dropless_moe_expert_router_gb300.layer import MoELayer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w1, w3, w2 = W.weights(wl, seed=0)                      # replicas hold the same layer
    x = W.x(wl, seed=rank).to(dev)                          # each rank its own batch
    logits = W.logits(wl, seed=rank).to(dev)
    layer = MoELayer(w1.to(dev), w3.to(dev), w2.to(dev), T=wl.T, K=wl.K, precision=wl.precision,
                     renorm=wl.renorm, id_dtype=torch.int16 if wl.id_bits == 16 else torch.int32,
                     training=wl.backward, score=wl.score,
                     expert_bias=None if W.expert_bias(wl) is None else W.expert_bias(wl).to(dev))
    del w1, w3, w2
    dy = W.dy(wl, seed=rank).to(dev) if wl.backward else None        # gradient of the layer output
    # L2 flush before every timed step, outside the timed interval: a 512 MiB write evicts
    # everything, then a 512 MiB read of another buffer evicts the write's own dirty lines (their
    # write-back would otherwise land inside the next timed step), leaving L2 clean and holding
    # nothing the step uses
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(512 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        flush_w.zero_()
        torch.amax(flush_r)               # a reduction that reads the buffer (no widened copy)
    stream = torch.cuda.current_stream()

    route = lambda: layer.stage_route(logits)
    if wl.invalid_frac > 0:
        # compact routes with invalid entries (the 2,304-expert workload: about 2 % of the [T, K]
        # ids are -1): the router's output with the workload's mask applied once, before timing,
        # is what the permute, the GEMMs and the combine consume in every step; the router still
        # runs in every step, into buffers of its own
        layer.stage_route(logits)
        mask = W.invalid_mask(wl, seed=rank).to(dev)
        route_ids, route_probs = layer.ids.clone(), layer.probs.clone()
        layer.ids.masked_fill_(mask, -1)
        layer.probs.masked_fill_(mask, 0.0)
        torch.cuda.synchronize()
        route = lambda: api.moe_route_topk(logits, wl.K, renorm=wl.renorm, id_dtype=route_ids.dtype, ids=route_ids,
                                           probs=route_probs)
    stages = [("route", route), ("permute", lambda: layer.stage_permute(x)),
              ("gemm_up", layer.stage_gemm_up), ("gemm_down", layer.stage_gemm_down),
              ("combine", layer.stage_combine)]
    if layer.nv4:
        # NVFP4: h's quantisation between the GEMMs is a stage of its own (x's is in the permute)
        stages.insert(3, ("quant_h", layer.stage_quant_h))
    if wl.backward:
        # the whole layer's backward, from dy [T, H]: combine, expert MLP (dgrad, dx, transposes,
        # wgrad), permute and router backward
        stages += [("combine_bwd", lambda: layer.stage_combine_backward(dy)),
                   ("dgrad_dh", lambda: layer.stage_dgrad_dh(layer.dy_perm, dy_quantised=layer.fp8)), ("dgrad_dx", layer.stage_dgrad_dx),
                   ("wgrad_transpose", lambda: layer.stage_transposes(x, layer.dy_perm)),
                   ("wgrad_gemm", layer.stage_wgrad_gemm), ("permute_bwd", layer.stage_permute_backward),
                   ("route_bwd", lambda: layer.stage_route_backward(logits))]

    def step():
        for _, fn in stages:
            fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert api.moe_get_device_errors() == 0, "device error during warm-up"

    # the whole step as one CUDA graph (group sizes stay on the device, so the captured step is
    # valid for any routing); replays carry no host launch gaps. Events recorded inside the graph
    # between stages give each stage's device time within the replay.
    ns = len(stages)
    gse = GraphStageEvents(ns + 1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream()
        for j, (_, fn) in enumerate(stages):
            if gse.ok:
                gse.record(j, cap)
            fn()
        if gse.ok:
            gse.record(ns, cap)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    assert api.moe_get_device_errors() == 0, "device error during graph warm-up"

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(K)]
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(gpu_id_for(local_rank))
    sampler.start()
    time.sleep(0.2)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # timed steps: graph replays; the step time and the per-stage times from the events inside
    # the graph (read after each replay), else from events around the replay plus an eager pass
    step_ms = []
    per_stage = [[] for _ in range(ns)]
    for i in range(K):
        flush_l2()                                          # outside the timed interval
        gev[i][0].record(stream)
        graph.replay()
        gev[i][1].record(stream)
        if gse.ok:
            torch.cuda.synchronize()
            for j in range(ns):
                per_stage[j].append(gse.elapsed_ms(j, j + 1))
            step_ms.append(gse.elapsed_ms(0, ns))      # first to last stage, inside the replay
    if not gse.ok:
        for i in range(K):
            flush_l2()
            e = ev[i]
            e[0].record(stream)
            for j, (_, fn) in enumerate(stages):
                fn()
                e[j + 1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    replay_ms = [a.elapsed_time(b) for a, b in gev]
    inner_ms = statistics.mean(step_ms) if step_ms else None
    step_ms = replay_ms                                   # the step time: events around each replay
    if gse.ok:
        stage_ms = {name: statistics.mean(per_stage[j]) for j, (name, _) in enumerate(stages)}
        stage_source = "events inside the graph between stages"
    else:
        stage_ms = {name: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K))
                    for j, (name, _) in enumerate(stages)}
        stage_source = "the same steps run eagerly with an event between stages"
    total_ms = sum(step_ms)

    # end to end through the host-memory call: x and logits in, y out (for the training
    # workload dy stays on the device, where the next layer's backward produces it)
    x_host = W.x(wl, seed=rank).pin_memory()
    lg_host = W.logits(wl, seed=rank).pin_memory()
    y_host = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()

    # forward-only layers: the overlapped transfer (consecutive calls overlap: this call's input
    # copy and the previous call's output copy run on the layer's copy streams beside the compute);
    # serially, one call at a time, the direct transfer (x read and y written in host memory by the
    # permute and the combine); a training layer copies
    overlap = wl.invalid_frac == 0 and not wl.backward
    serial_transfer = "copy" if (wl.backward or layer.nv4) else "direct"

    def e2e_step(transfer):
        if wl.invalid_frac > 0:
            # the routes keep their invalid entries: the same stages between the host copies
            x.copy_(x_host, non_blocking=True)
            logits.copy_(lg_host, non_blocking=True)
            step()
            y_host.copy_(layer.y, non_blocking=True)
            return
        layer.forward_host(x_host, lg_host, y_host, transfer=transfer)
        if wl.backward:
            layer.backward_full(layer.x_dev, layer.logits_dev, dy)

    e2e_ms = e2e_serial_ms = 0.0
    if with_e2e:
        for _ in range(max(2, args.warmup // 2)):
            e2e_step(serial_transfer)
        torch.cuda.synchronize()
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(K):
            flush_l2()
            e2e_ev[i][0].record(stream)
            e2e_step(serial_transfer)
            e2e_ev[i][1].record(stream)
        torch.cuda.synchronize()
        e2e_serial_ms = sum(a.elapsed_time(b) for a, b in e2e_ev)
        e2e_ms = e2e_serial_ms
        if overlap:
            # K consecutive calls as one timed region, from the first call's input copy to the last
            # call's output copy; no L2 flush between them (each call reads every expert's weights,
            # more than L2 holds)
            for _ in range(max(3, args.warmup)):
                e2e_step("overlapped")
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            flush_l2()
            # (the first input copy runs on the layer's copy stream, which does not wait for the
            # start event: with the device idle when the event is recorded, it cannot start early)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(K):
                e2e_step("overlapped")
            stream.wait_event(layer.host_event)
            b.record(stream)
            torch.cuda.synchronize()
            e2e_ms = a.elapsed_time(b)
    clocks = sampler.stop()
    errs = api.moe_get_device_errors()
    R = int(layer.perm.group_offsets[-1].item())
    active = int((layer.perm.group_sizes > 0).sum().item())      # experts that received routes
    launches = layer.launches_per_forward + (layer.launches_per_backward_full if wl.backward else 0)

    if world > 1:
        total_ms, e2e_ms, e2e_serial_ms = reduce_max_over_ranks([total_ms, e2e_ms, e2e_serial_ms], dev)
    return dict(total_ms=total_ms, e2e_ms=e2e_ms, e2e_serial_ms=e2e_serial_ms, e2e_overlap=overlap and with_e2e,
                e2e_serial_transfer=serial_transfer, stage_ms=stage_ms, stage_source=stage_source,
                inner_ms=inner_ms, clocks=clocks, R=R, active=active, errs=errs,
                h2d=x_host.numel() * 2 + lg_host.numel() * 4, d2h=y_host.numel() * 2, launches=K * launches)


def reduce_max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings over all ranks of the process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tokens_per_s(world: int, tokens_per_rank_step: int, steps: int, max_total_ms: float) -> float:
    """Tokens of all ranks over the slowest rank's timed interval."""
    return world * tokens_per_rank_step * steps / (max_total_ms / 1e3)


def stage_report(wl, R, stage_ms, active=None):
    """Algorithmic bytes / FLOPs of each stage (minimum traffic, not counters). GEMM bytes:
    operands read once (weights of the experts with routes), outputs written once."""
    T, H, E, K, F = wl.T, wl.H, wl.E, wl.K, wl.F
    Ea = E if active is None else active
    idb = 2 if wl.id_bits == 16 else 4
    fp8 = wl.precision == "mxfp8"
    nv4 = wl.precision == "nvfp4"
    b_out = 1 if fp8 else 2
    # bytes per operand element: MXFP8 code + its share of a scale; NVFP4 half a byte + 1/16
    q = (1 + 1 / 32) if fp8 else (0.5 + 1 / 16) if nv4 else 2
    bytes_ = {
        "route": T * E * 4 + T * K * (idb + 4) + (E * 4 if wl.score == "sigmoid" else 0),
        # (NVFP4: the routed tokens' amax reads x once more; rows written as codes and scales)
        "permute": T * H * 2 * (2 if nv4 else 1) + (R * H * q if nv4 else R * H * b_out + (R * H // 32 if fp8 else 0))
                   + T * K * (idb + 4) + R * 4,
        "combine": R * H * 2 + T * K * 8 + T * H * 2,
        # read dy and y_perm, write dy_perm (MXFP8: and its codes and scales); route metadata and dprobs
        "combine_bwd": T * H * 2 + R * H * 2 + R * H * 2 + (R * H * (1 + 1 / 32) if fp8 else 0) + T * K * 12,
        "permute_bwd": R * H * 2 + T * H * 2 + T * K * 4,
        "route_bwd": T * E * 4 * 2 + T * K * (idb + 4),
        # read h (or its bf16 copy), dy, x (gathered), dab in bf16; write the transposed operands
        "wgrad_transpose": R * 2 * (F + H + H + 2 * F) + R * b_out * (F + H + H + 2 * F) * (1 + (1 / 32 if fp8 else 0)),
        "quant_h": R * F * 2 + R * F * q,
        "gemm_up": R * H * q + Ea * H * 2 * F * q + R * F * (2 if nv4 else q),
        "gemm_down": R * F * q + Ea * F * H * q + R * H * 2,
        # read dy, W2, (a | b); write dab (MXFP8: and its codes and scales)
        "dgrad_dh": R * H * q + Ea * F * H * q + R * 2 * F * 2 * 2 + (R * 2 * F * (1 + 1 / 32) if fp8 else 0),
        "dgrad_dx": R * 2 * F * q + Ea * 2 * F * H * q + R * H * 2,
        "wgrad_gemm": R * (F + H + H + 2 * F) * q + Ea * 3 * H * F * 2,
    }
    flops = {"gemm_up": 4.0 * R * H * F, "gemm_down": 2.0 * R * H * F, "dgrad_dh": 2.0 * R * H * F,
             "dgrad_dx": 4.0 * R * H * F, "wgrad_gemm": 6.0 * R * H * F}
    out = {}
    for n, ms in stage_ms.items():
        d = {"us": round(ms * 1e3, 2)}
        if n in bytes_:
            d["GB/s"] = round(bytes_[n] / (ms * 1e-3) / 1e9, 1)
        if n in flops:
            d["TFLOP/s"] = round(flops[n] / (ms * 1e-3) / 1e12, 1)
        out[n] = d
    return out, flops, bytes_


# the other workloads the default run times beside the headline one, each graph-replayed
EXTRA_WORKLOADS = ("dsv3", "large_e", "heavy", "dsv3_nvfp4", "dsv3_sigmoid")


def roofline(wl, r, peaks, peak_kind):
    """The dominant kernel of a timed workload (the GEMM stage with the largest time; one launch
    per stage) against whichever peak its algorithmic work needs longer for."""
    stages, flops, gbytes = stage_report(wl, r["R"], r["stage_ms"], r["active"])
    dom = max((n for n in flops if n in r["stage_ms"] and n != "wgrad_gemm" and n != "dgrad_dx"),
              key=lambda n: r["stage_ms"][n])
    # dense peak of the GEMMs' operand type: the measured bf16 peak times the nominal ratio
    # (MXFP8 2x, NVFP4 6x: 4.5 and 13.5 against 2.25 PFLOP/s dense)
    fp8_ratio = {"mxfp8": 2.0, "nvfp4": 6.0}.get(wl.precision, 1.0)
    # The timed loop is well under a second and the SM clock stays at its maximum
    # (see "clocks"), the conditions of the burst measurement: report against the
    # burst peak, and the sustained figure beside it.
    peak = peaks["bf16_tflops"] * fp8_ratio
    peak_sustained = peaks["bf16_tflops_sustained"] * fp8_ratio
    hbm_bound = gbytes[dom] / (peaks["hbm_gbs"] * 1e9) > flops[dom] / (peak * 1e12)
    if hbm_bound:
        achieved = gbytes[dom] / (r["stage_ms"][dom] * 1e-3) / 1e9
        peak, peak_sustained = peaks["hbm_gbs"], peaks["hbm_gbs"]
    else:
        achieved = flops[dom] / (r["stage_ms"][dom] * 1e-3) / 1e12
    traffic = TRAFFIC_BY_SOURCE.get((wl.name, dom, kernel_source_hash()))
    return stages, {
        "kernel": KERNEL_NAMES[dom], "bound": "hbm" if hbm_bound else "tensor",
        "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "GB/s" if hbm_bound else "TFLOP/s",
        "frac": round(achieved / peak, 4), "traffic": traffic,
        "peak_source": (f"{peak_kind} HBM copy bandwidth" if hbm_bound else
                        f"{peak_kind} dense bf16 burst" + ({2.0: " x2 (fp8)", 6.0: " x6 (fp4)"}.get(fp8_ratio, ""))),
        "frac_of_sustained": round(achieved / peak_sustained, 4)}


def workload_config(wl, gpus):
    return {"workload": f"{wl.name}: T={wl.T} H={wl.H} E={wl.E} top-{wl.K} F={wl.F} {wl.precision}"
                        + (f", {wl.invalid_frac:.0%} invalid routes" if wl.invalid_frac > 0 else "")
                        + (", forward + backward" if wl.backward else "")
                        + (", sigmoid router" if wl.score == "sigmoid" else ""),
            "T": wl.T, "H": wl.H, "E": wl.E, "K": wl.K, "F": wl.F, "precision": wl.precision,
            "tokens_per_step_per_gpu": wl.T, "l2": "flushed before every timed step (512 MiB write, then a 512 MiB read of another buffer)",
            "parallelism": f"replicas x{gpus}"}


def host_cores():
    """Cores of this host and those this process may run on."""
    try:
        aff = len(os.sched_getaffinity(0))
    except Exception:
        aff = os.cpu_count()
    return {"host_cores": os.cpu_count(), "affinity_cores": aff}


def _free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n: int) -> int:
    """Run this command as n ranks on this node (one process per GPU) through torch's launcher,
    rendezvous on 127.0.0.1; returns the launcher's exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def selftest_launch(rank, world):
    """--selftest-launch: the rank plumbing alone, on the CPU (gloo): every rank reports a timing
    that depends on its rank; rank 0 prints the world size and the max over ranks."""
    import torch.distributed as dist
    dist.init_process_group("gloo")
    got = reduce_max_over_ranks([10.0 + rank, 50.0 - rank], "cpu")
    dist.destroy_process_group()
    if rank == 0:
        print(json.dumps({"selftest": "launch", "world": world, "max_ms": got}))
    return 0


def reference_arm(args, wl, world):
    """The reference arm: the CPU oracle as it stands, each step a bounded sample of the workload
    (its grouped MLP on a few rows, extrapolated by row count to the whole batch)."""
    xb, lg, yb, wb = oracle_inputs(wl)
    rows_per_step = max(1, args.cpu_rows // 6)
    for _ in range(args.warmup):
        oracle_sample(wl, xb, lg, yb, 1, wb)
    est, wall = [], []
    desc = ""
    for _ in range(args.steps):
        t0 = time.perf_counter()
        t, desc = oracle_sample(wl, xb, lg, yb, rows_per_step, wb)
        wall.append(time.perf_counter() - t0)
        est.append(t)
    value = wl.T * args.steps / sum(est)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            # the wall time of each timed sample; the whole batch's step, extrapolated, beside it
            "ms_per_step": sum(wall) / args.steps * 1e3,
            "ms_per_step_extrapolated": sum(est) / args.steps * 1e3,
            "timing": "value = whole-batch tokens / extrapolated step time; ms_per_step = wall time of the timed "
                      "sample (router, permute and combine over every token, the grouped MLP on "
                      f"{rows_per_step} rows)",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, world),
            "cpu_baseline": dict({"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                  "sample": desc + " (per step)"}, **host_cores()),
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="other workloads timed beside the headline one ('' for none)")
    ap.add_argument("--cpu-rows", type=int, default=24, help="grouped-MLP rows of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer leg (for profiler launch lists of the device steps alone; "
                         "the line's e2e is then null)")
    ap.add_argument("--selftest-launch", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return launch_ranks(args.gpus)                  # one process per GPU, launched here
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if args.selftest_launch:
        return selftest_launch(rank, world)

    from dropless_moe_expert_router_gb300 import workloads as W
    wl = W.get(args.workload)
    config = workload_config(wl, world)

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args, wl, world)))
        return 0

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import __graft_entry__
    __graft_entry__.build()

    r = run_ours(args, wl, rank, world, local_rank, with_e2e=not args.no_e2e)
    peaks, peak_kind = load_peaks()
    stages, roof = roofline(wl, r, peaks, peak_kind)
    extras = {}
    for name in [n for n in args.extra.split(",") if n and n != wl.name] if args.workload == "mixtral" else []:
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        xw = W.get(name)
        rx = run_ours(args, xw, rank, world, local_rank, with_e2e=False)
        st_x, roof_x = roofline(xw, rx, peaks, peak_kind)
        extras[name] = {"config": workload_config(xw, world)["workload"],
                        "value": whole_job_tokens_per_s(world, xw.T, args.steps, rx["total_ms"]),
                        "unit": "tokens/s", "ms_per_step": rx["total_ms"] / args.steps,
                        "ms_first_to_last_stage": rx["inner_ms"],
                        "gpu_launches": rx["launches"], "routes": rx["R"], "roofline": roof_x, "stages": st_x,
                        "clocks": rx["clocks"], "device_errors": rx["errs"]}
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    value = whole_job_tokens_per_s(world, wl.T, args.steps, r["total_ms"])
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["total_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.precision, "data": "synthetic", "config": config,
        "e2e": None if args.no_e2e else {
            "value": whole_job_tokens_per_s(world, wl.T, args.steps, r["e2e_ms"]), "unit": "tokens/s",
            "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
            "transfer": "overlapped" if r["e2e_overlap"] else r["e2e_serial_transfer"],
            "serial": {"value": whole_job_tokens_per_s(world, wl.T, args.steps, r["e2e_serial_ms"]),
                       "transfer": r["e2e_serial_transfer"],
                       "timing": "each call alone, L2 flushed before it, events around it"}},
        "gpu_launches": r["launches"] + sum(v["gpu_launches"] for v in extras.values()),
        "roofline": roof,
        "timing": "step = CUDA-graph replay of the whole step, CUDA events around each replay"
                  + (f" (first to last stage inside the replay: {r['inner_ms']:.4f} ms)" if r["inner_ms"] else "")
                  + f"; stages = {r['stage_source']}; e2e = "
                  + ("not run (--no-e2e)" if args.no_e2e else
                     "K consecutive MoELayer.forward_host calls (overlapped transfer) as one timed region, "
                     "from the first input copy to the last output copy" if r["e2e_overlap"]
                     else "events around each MoELayer.forward_host call")
                  + ("; workloads = the other workloads, timed the same way after the headline one"
                     if extras else ""),
        "stages": stages,
        "routes": r["R"],
        "clocks": r["clocks"],
        "device_errors": r["errs"],
    }
    if extras:
        line["workloads"] = extras
    if world == 1 and not args.no_cpu_baseline:
        xb, lg, yb, wb = oracle_inputs(wl)
        t, desc = oracle_sample(wl, xb, lg, yb, args.cpu_rows, wb)
        line["cpu_baseline"] = dict({"value": wl.T / t, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                     "sample": desc}, **host_cores())
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
