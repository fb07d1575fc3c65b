#!/usr/bin/env python
"""Benchmark of the GB300 MoE layer forward (route -> permute -> FC1+SwiGLU ->
FC2 -> combine) on seeded synthetic inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one full layer forward over one
batch of T tokens.  `value` = tokens of all ranks / max-over-ranks time, with
inputs resident in HBM; `e2e` = the same through the public API with the
token activations copied from pinned host memory and the output copied back
inside the timed region (weights are resident model parameters).  L2 is
flushed before every timed step, outside the step's own CUDA events.  The
per-kernel breakdown and the roofline of the dominant kernel come from a
second pass that replays a CUDA graph of the same forward captured with the
library's launch-event hook armed: a CUDA event node on the launching stream
right before every kernel and one after the last.  With N > 1 (torchrun, or
started by this script), the ranks split the layer by experts (--partition ep,
the default: every rank routes the same batch, computes its contiguous slot
range and its shard of the shared experts, and one all-reduce sums the
partials; strong scaling), exchange rows all-to-all (--partition a2a: every rank
holds its own batch, sends each pair's row to the rank owning its slot and gets
the expert outputs back; weak scaling) or run independent batches (--partition
replicas; weak scaling, no collective).
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
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

import torch  # noqa: E402

import moe_inputs as mi  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300; % of BF16 tensor peak (prefill) / HBM BW (decode)"
DEFAULT_WORKLOAD = "redundant_slots_prefill"

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel,
# from one ncu capture of that workload, valid only while the kernel source hashes to
# the recorded value.
NCU_TRAFFIC = {
    # FC1 of the first forward, ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum:
    # 822.25 MB read + 87.41 MB written (algorithmic 914.36 MB)
    ("qwen2_moe_like_prefill", "f3a8bb44c1835ecc"): 909.66e6,
    # 115.62 MB read + 2.99 MB written (algorithmic 115.40 MB)
    ("dsv2_lite_like_decode_t1", "f3a8bb44c1835ecc"): 118.61e6,
    # 1105.62 MB read + 33.02 MB written (algorithmic 1090.52 MB)
    ("redundant_slots_cut16", "f3a8bb44c1835ecc"): 1138.64e6,
}


# Workloads too large for a capture under the profiling size rule: FC1's DRAM traffic per
# algorithmic byte, from one capture of a cut-down case with the same H and I (its measured
# dram bytes, its algorithmic FC1 bytes), applied to the full launch's algorithmic bytes.
# Traffic grows in proportion: every slot's weight tile is streamed once and its A rows
# stay in L2 across the slot's n-tiles, at either size.
NCU_TRAFFIC_SCALED = {
    ("redundant_slots_prefill", "f3a8bb44c1835ecc"): (
        1138.64e6, 1090.52e6,
        "one capture of FC1 on the 16-slot cut (T=1024, H=7168, I=2048, E=16, k=8: 512 rows per slot)"),
}


def _traffic(workload, src_hash, fc1_bytes):
    direct = NCU_TRAFFIC.get((workload, src_hash))
    if direct is not None:
        return direct, "ncu capture of this workload's first FC1 launch"
    scaled = NCU_TRAFFIC_SCALED.get((workload, src_hash))
    if scaled is not None:
        measured, algorithmic, what = scaled
        return measured / algorithmic * fc1_bytes, f"scaled per algorithmic byte from {what}"
    return None, "no capture of the current kernel source"


def _src_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    INTERVAL_MS = 10

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.n_before = 0

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.INTERVAL_MS), "-i", str(self.dev)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # nvidia-smi takes a moment to start: let its first sample land before the
        # timed region opens, then remember how many samples predate the region
        t_end = time.time() + 5.0
        while time.time() < t_end and self._lines() == 0:
            time.sleep(0.01)
        self.n_before = self._lines()

    def _lines(self):
        try:
            with open(self.path) as f:
                return sum(1 for ln in f if ln.endswith("\n"))
        except OSError:
            return 0

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = open(self.path).readlines()
        # the samples taken inside the region, plus the last one before it opened
        n_in = 0
        first = max(0, self.n_before - 1)
        for i, line in enumerate(lines[first:], start=first):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            n_in += i >= self.n_before
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "samples_in_region": n_in, "interval_ms": self.INTERVAL_MS, "reasons": sorted(reasons)}


class L2Flush:
    """Leaves L2 holding none of a step's data: writes one buffer of at least
    twice the L2 size, then reads a second one, so no dirty line of the flush is
    left to be written back inside the next timed step."""

    def __init__(self, dev):
        l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (128 << 20))
        self.nbytes = max(2 * l2, 256 << 20)
        n = self.nbytes // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1.0)
        torch.sum(self.r, 0, out=self.sink)

    def describe(self):
        return f"write {self.nbytes >> 20} MiB, then read another {self.nbytes >> 20} MiB"


def _external_events():
    """Two timing events that can be recorded as nodes of a captured CUDA graph (None
    where this PyTorch cannot make them)."""
    try:
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    except TypeError:
        return None


def time_steps(fns, K, flush, stream):
    """K steps; each step flushes L2, then runs fns in order with a CUDA event on
    `stream` before and after each.  Returns per-fn lists of K times in ms."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(K)]
    for i in range(K):
        flush()
        e = evs[i]
        e[0].record(stream)
        for j, fn in enumerate(fns):
            fn()
            e[j + 1].record(stream)
    torch.cuda.synchronize()
    return [[e[j].elapsed_time(e[j + 1]) for e in evs] for j in range(len(fns))]


def kernel_breakdown(layer, x, n_launch, K, W, flush, stream):
    """Each kernel of one layer forward timed on its own: the forward is captured
    into a CUDA graph with the library's launch-event hook armed, so an event
    node precedes every kernel it launches and a mark follows the last, and the
    kernels run without programmatic overlap.  The graph holds exactly the
    launches of the timed forward (same kernels, tile variants and splits).
    Returns the kernels' labels and, per kernel, K times in ms (each replay after
    an L2 flush; the host waits after every replay to read the events)."""
    import serving_router_gate_gb300 as moe
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_launch + 1)]
    for e in evs:
        e.record(stream)  # creates the CUDA events
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    moe.moe_launch_events_arm(evs)
    try:
        with torch.cuda.graph(g):
            layer.forward(x)
            moe.moe_launch_events_mark()
        labels = moe.moe_launch_events_used()
    finally:
        moe.moe_launch_events_arm(None)
    if len(labels) != n_launch + 1 or labels[-1] != "mark":
        raise RuntimeError(f"launch-event hook saw {labels}, expected {n_launch} launches and a mark")
    for _ in range(W):
        g.replay()
    times = [[] for _ in range(n_launch)]
    for _ in range(K):
        flush()
        g.replay()
        torch.cuda.synchronize()
        for i in range(n_launch):
            times[i].append(evs[i].elapsed_time(evs[i + 1]))
    return labels[:-1], times


def _stage_of(label, seen):
    """The layer stage a kernel label belongs to (E4M3 activation quantisers:
    the first one quantises the GEMM inputs, the second the intermediates)."""
    if label.startswith("router_"):
        return "route"
    if label.startswith("permute_"):
        return "permute"
    if label.startswith("grouped_gemm_fc1"):
        return "fc1"
    if label.startswith("grouped_gemm_fc2"):
        return "fc2"
    if label == "quantize_act_rows":
        return "quant_h" if "fc1" in seen else "quant_x"
    return label


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, ws: int) -> float:
    """Largest value over all ranks (timing is taken as the slowest rank)."""
    if ws <= 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(tokens_per_rank: int, ms_local: float, ws: int):
    """Whole-job throughput of N independent replicas: every rank processed
    tokens_per_rank per step; the step time is the slowest rank's.  Returns
    (tokens/s over all ranks, max ms per step)."""
    ms = max_over_ranks(ms_local, ws)
    return tokens_per_rank * ws / (ms * 1e-3), ms


def _work(cfg, rows: int, active_slots: int):
    """Algorithmic flops and bytes of the layer's kernels for one batch."""
    T, H, I, k = cfg.T, cfg.H, cfg.I, cfg.k
    Ish = cfg.n_shared * cfg.I_shared
    fc1_flops = 4.0 * H * (rows * I + T * Ish)
    fc2_flops = 2.0 * H * (rows * I + T * Ish)
    # bytes per weight, per row of weights: bf16; E4M3 + an fp32 row scale; NVFP4: half a
    # byte + one E4M3 block scale per 16 elements + an fp32 row scale
    eb = 0.5 + 1.0 / 16 if cfg.fp4 else (1 if cfg.fp8 else 2)
    er = 4 if (cfg.fp8 or cfg.fp4) else 0
    w1 = active_slots * 2 * I * (H * eb + er) + 2 * Ish * (H * eb + er)
    w2 = active_slots * H * (I * eb + er) + H * (Ish * eb + er)
    # the same per GEMM input activation
    ab = 0.5 + 1.0 / 16 if cfg.fp4 else (1 if cfg.act8 else 2)
    ar = 4 if (cfg.act8 or cfg.fp4) else 0
    a_rows = rows + T * (Ish > 0)
    fc1_bytes = w1 + a_rows * (H * ab + ar) + rows * I * 2 + T * Ish * 2
    fc2_bytes = (w2 + rows * (I * ab + ar) + T * (Ish * ab + (ar if Ish else 0))
                 + rows * H * 2 + (T * H * 2 if Ish else 0))
    # the whole layer: both GEMMs' bytes plus the router's x and fp32 gate weights, the
    # permuted expert input rows written (in FC1's input format), the expert outputs read
    # back by the combine, and out
    layer_bytes = (fc1_bytes + fc2_bytes + cfg.E * H * 4 + T * H * 2 + rows * (H * ab + ar) + rows * H * 2
                   + (T * H * 2 if Ish else 0) + T * H * 2)
    return dict(fc1_flops=fc1_flops, fc2_flops=fc2_flops, fc1_bytes=fc1_bytes, fc2_bytes=fc2_bytes,
                gate_flops=2.0 * T * H * cfg.E, layer_bytes=layer_bytes)


def _oracle_nvfp4(oracle, cfg, cpu):
    """NVFP4 workloads: the oracle's own quantisation of the weights (done once, untimed),
    the shared experts as the one concatenated MLP the layer runs, NVFP4 activations."""
    if not cfg.fp4:
        return None
    d = {}
    d["W1q"], d["W1sb"], d["s1"] = oracle.quantize_nvfp4_rows(cpu["W1"])
    d["W2q"], d["W2sb"], d["s2"] = oracle.quantize_nvfp4_rows(cpu["W2"])
    if cpu["W1s"] is not None:
        c1, c2 = mi.shared_concat(cpu["W1s"], cpu["W2s"])
        cpu["W1s"], cpu["W2s"] = c1[None], c2[None]
        d["W1sq"], d["W1ssb"], d["s1s"] = oracle.quantize_nvfp4_rows(cpu["W1s"])
        d["W2sq"], d["W2ssb"], d["s2s"] = oracle.quantize_nvfp4_rows(cpu["W2s"])
    d["act4"] = True
    return d


def _oracle_fp8(oracle, cfg, cpu):
    """E4M3 workloads: the oracle's own quantisation of the weights (done once, untimed),
    the shared experts as the one concatenated MLP the layer runs."""
    if not cfg.fp8:
        return None
    q1, s1 = oracle.quantize_fp8_rows(cpu["W1"])
    q2, s2 = oracle.quantize_fp8_rows(cpu["W2"])
    f = dict(W1q=q1, s1=s1, W2q=q2, s2=s2, act8=cfg.act8)
    if cpu["W1s"] is not None:
        c1, c2 = mi.shared_concat(cpu["W1s"], cpu["W2s"])
        cpu["W1s"], cpu["W2s"] = c1[None], c2[None]
        f["W1sq"], f["s1s"] = oracle.quantize_fp8_rows(cpu["W1s"])
        f["W2sq"], f["s2s"] = oracle.quantize_fp8_rows(cpu["W2s"])
    return f


def run_cpu_baseline(inp_dev, cfg, target_s=10.0, T_cap=None):
    """The fp64 oracle on the host cores, on the first n tokens of the batch."""
    import numpy as np  # noqa: F401
    import oracle
    from moe_inputs import shared_concat  # noqa: F401
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp_dev.items()}

    fp8 = _oracle_fp8(oracle, cfg, cpu)
    fp4 = _oracle_nvfp4(oracle, cfg, cpu)

    def run(n):
        t0 = time.perf_counter()
        oracle.moe_layer(cpu["x"][:n], cpu["Wg"], cpu["bias"], cfg.k, cfg.renorm, cpu["W1"], cpu["W2"],
                         rep_offset=cpu["rep_offset"], rep_slots=cpu["rep_slots"], W1s=cpu["W1s"],
                         W2s=cpu["W2s"], shared_gate_w=cpu["w_s"], S=cfg.slots, n_group=cfg.n_group,
                         topk_group=cfg.topk_group, on_input=cfg.on_input, fp8=fp8, nvfp4=fp4)
        return time.perf_counter() - t0

    threads = oracle.get_threads()
    n0 = min(cfg.T, max(threads, 8))
    t0 = run(n0)
    n = int(max(n0, min(T_cap or cfg.T, n0 * target_s / max(t0, 1e-3))))
    n = max(1, min(n, cfg.T))
    t = run(n)
    # the same oracle on one thread, on a sample of about a quarter of that time
    oracle.set_threads(1)
    n1 = max(1, min(cfg.T, int(n / t * target_s / 4 / max(threads, 1))))
    t1 = run(n1)
    oracle.set_threads(threads)
    return dict(value=n / t, unit="tokens/s", cores=threads, kind="oracle",
                sample=f"first {n} of the {cfg.T} tokens of {cfg.name}, whole layer in fp64 "
                       f"({t:.1f} s, {threads} OpenMP threads)",
                single_thread_value=n1 / t1,
                single_thread_sample=f"first {n1} tokens, {t1:.1f} s on one thread"), t


def _ep_layer(inp, cfg, world, rank, dev, peer=None):
    """This rank's expert-parallel layer over the workload's inputs (peer: a PeerReduction
    in place of the collective all-reduce)."""
    from serving_router_gate_gb300.expert_parallel import EPMoELayer
    W1s = W2s = None
    if inp["W1s"] is not None:
        W1s, W2s = mi.shared_concat(inp["W1s"], inp["W2s"])
    d = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    return EPMoELayer(d(inp["Wg"]), d(inp["W1"]), d(inp["W2"]), cfg.k, cfg.renorm, cfg.T, world, rank,
                      logit_bias=d(inp["bias"]), rep_offset=d(inp["rep_offset"]), rep_slots=d(inp["rep_slots"]),
                      W1s=d(W1s), W2s=d(W2s), shared_gate_w=d(inp["w_s"]), on_input=cfg.on_input,
                      n_group=cfg.n_group, topk_group=cfg.topk_group, fp8=cfg.fp8, act8=cfg.act8, fp4=cfg.fp4,
                      peer=peer)


def _a2a_layer(inp, cfg, world, rank, dev, max_T=None):
    """This rank's all-to-all expert-parallel layer over the workload's weights."""
    from serving_router_gate_gb300.expert_parallel import EPAllToAllLayer
    if cfg.fp8 or cfg.fp4:
        raise SystemExit("bench.py: --partition a2a runs bf16 weights only")
    W1s = W2s = None
    if inp["W1s"] is not None:
        W1s, W2s = mi.shared_concat(inp["W1s"], inp["W2s"])
    d = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    return EPAllToAllLayer(d(inp["Wg"]), d(inp["W1"]), d(inp["W2"]), cfg.k, cfg.renorm, max_T or cfg.T, world, rank,
                           logit_bias=d(inp["bias"]), rep_offset=d(inp["rep_offset"]),
                           rep_slots=d(inp["rep_slots"]), W1s=d(W1s), W2s=d(W2s), shared_gate_w=d(inp["w_s"]),
                           n_group=cfg.n_group, topk_group=cfg.topk_group, on_input=cfg.on_input)


def bench_ours(args):
    import serving_router_gate_gb300 as moe
    from serving_router_gate_gb300.layer import HostPipeline, layer_from_inputs

    ws_, rank, local = _dist()
    cfg = mi.CONFIGS[args.workload]
    dev = torch.device("cuda", local)
    inp = mi.make_inputs(cfg, device=dev)
    # expert parallelism (more than one rank): every rank routes the whole batch, computes
    # its slot range and shared shard, and one all-reduce sums the partials; otherwise
    # (replicas) every rank runs its own batch through the whole layer
    peer = None
    if args.partition == "ep" and ws_ > 1 and args.reduce == "peer":
        from serving_router_gate_gb300.expert_parallel import PeerReduction
        peer = PeerReduction(cfg.T, cfg.H, ws_, rank, dev)
    ep = _ep_layer(inp, cfg, ws_, rank, dev, peer) if (args.partition == "ep" and ws_ > 1) else None
    # all-to-all expert parallelism: every rank holds its own batch of T tokens and the
    # experts of its slot range; rows travel to their slots' ranks and back (NCCL).  The
    # per-kernel pass and the roofline then describe the one-GPU layer on the rank's batch.
    a2a = _a2a_layer(inp, cfg, ws_, rank, dev) if (args.partition == "a2a" and ws_ > 1) else None
    layer = ep.layer if ep is not None else layer_from_inputs(inp, dev)
    x = mi.rank_tokens(cfg, rank, cfg.T, dev) if a2a is not None else inp["x"]
    T, H = cfg.T, cfg.H
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup

    for _ in range(W):
        layer.forward(x)
    torch.cuda.synchronize()
    rows = int(layer.offsets[-1])
    active = int((layer.counts > 0).sum())
    status = moe.moe_get_device_status(layer.ws)
    if status:
        raise RuntimeError(f"device status {status} after warm-up")

    if a2a is not None:
        for _ in range(W):
            a2a.forward(x)
        torch.cuda.synchronize()
    # launches one layer forward issues (the same kernels a graph replay re-issues)
    c0 = moe.moe_get_launch_count()
    layer.forward(x)
    kernels_per_step = moe.moe_get_launch_count() - c0
    if a2a is not None:
        c0 = moe.moe_get_launch_count()
        a2a.forward(x)
        a2a_launches = moe.moe_get_launch_count() - c0
    refined_per_step = moe.moe_get_route_stats(layer.ws) / (W + 1)
    flush = L2Flush(dev)

    # ---- timed pass: the whole layer, K steps (replayed from a CUDA graph of one step) ----
    # The graph holds two external event nodes, one before the forward's first kernel
    # and one after its last: their interval is the forward's device time.  Events
    # recorded on the stream around each replay also time the graph's own launch, a
    # cost a model-level graph pays once per model step rather than once per layer;
    # both are reported.
    # the expert-parallel steps run eagerly (NCCL in the step; the all-to-all one also waits
    # for its split sizes on the host)
    graph_ok = args.graph and ep is None and a2a is None
    inner = _external_events() if graph_ok else None
    if graph_ok:
        pre = (lambda: inner[0].record()) if inner else None
        post = (lambda: inner[1].record()) if inner else None
        graph = layer.capture(x, pre=pre, post=post)
    else:
        graph = None
    if graph is not None:
        step = graph.replay
    elif ep is not None:
        step = lambda: ep.forward(x)  # noqa: E731
    elif a2a is not None:
        step = lambda: a2a.forward(x)  # noqa: E731
    else:
        step = lambda: layer.forward(x)  # noqa: E731
    for _ in range(W):
        step()

    def timed_region():
        clocks = ClockSampler(torch.cuda.current_device())
        _barrier(ws_)
        torch.cuda.synchronize()
        clocks.start()
        outer, inside = [], []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(K):
            flush()
            e0.record(stream)
            step()
            e1.record(stream)
            torch.cuda.synchronize()  # the in-graph events are re-recorded by the next replay
            outer.append(e0.elapsed_time(e1))
            if inner:
                inside.append(inner[0].elapsed_time(inner[1]))
        torch.cuda.synchronize()
        rec = clocks.stop()
        _barrier(ws_)
        t_out = statistics.mean(outer)
        t_in = statistics.mean(inside) if inside else t_out
        return (t_in, t_out), rec

    (ms_local, ms_replay_local), clk = timed_region()
    # a region that saw a hardware or thermal slowdown is measured once more (power
    # capping is kept: it is the part's normal state under a dense load); decided over
    # all ranks, so that every rank measures the same number of regions
    bad = bool(clk and set(clk["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"})
    if max_over_ranks(float(bad), ws_) > 0:
        first = clk
        (ms_local, ms_replay_local), clk = timed_region()
        if clk is not None:
            clk["remeasured_after"] = first
    if ep is not None:
        # one batch of T tokens for the whole job (strong scaling)
        ms = max_over_ranks(ms_local, ws_)
        value = T / (ms * 1e-3)
    else:
        value, ms = aggregate_throughput(T, ms_local, ws_)
    ms_replay = max_over_ranks(ms_replay_local, ws_)

    # ---- e2e pass: host activations in, host output out ----
    # Right after the device-timed region, so both run under the same thermal and power
    # state (a power-capped part clocks lower as a long run goes on): the pipelined serving
    # loop first, then the serial one, then the per-kernel pass.
    x_pin = x.cpu().pin_memory()
    out_pin = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    ms_e2e = e2e_how = None
    e2e_clk = None
    if graph_ok:
        # the serving loop: batch i+1's input copy and batch i-1's output copy overlap batch
        # i's forward (HostPipeline: three streams, two device buffer pairs).  L2 is flushed
        # on the compute stream before every forward; the flushes are timed by their own
        # events and taken out of the region's length.
        pipe = HostPipeline(layer, x)
        out_pins = [out_pin, torch.empty_like(out_pin).pin_memory()]
        pipe.run([x_pin] * W, [out_pins[i & 1] for i in range(W)])
        torch.cuda.synchronize()
        fl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]

        def flushed(i):
            fl[i][0].record()
            flush()
            fl[i][1].record()

        _barrier(ws_)
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(pipe.s_in)
        pipe.run([x_pin] * K, [out_pins[i & 1] for i in range(K)], before_forward=flushed)
        b.record(pipe.s_out)
        torch.cuda.synchronize()
        e2e_clk = sampler.stop()
        region = a.elapsed_time(b) - sum(e0.elapsed_time(e1) for e0, e1 in fl)
        ms_e2e = max_over_ranks(region / K, ws_)
        e2e_how = ("pipelined (HostPipeline): every step copies its input in from pinned host memory and its "
                   "output back, on two copy streams, overlapping the neighbouring steps' forwards; the region "
                   "runs from the first input copy to the last output copy, L2 flushes excluded; measured right "
                   "after the device-timed region")
    x_dev = torch.empty_like(x)
    h2d = lambda: x_dev.copy_(x_pin, non_blocking=True)  # noqa: E731
    d2h = lambda: out_pin.copy_(layer.out[:T], non_blocking=True)  # noqa: E731
    if graph_ok:
        g_e2e = layer.capture(x_dev, pre=h2d, post=d2h)
        e2e_step = g_e2e.replay
    else:
        def e2e_step():
            h2d()
            if ep is not None:
                layer.out[:T].copy_(ep.forward(x_dev))
            elif a2a is not None:
                layer.out[:T].copy_(a2a.forward(x_dev))
            else:
                layer.forward(x_dev)
            d2h()
    for _ in range(W):
        e2e_step()
    torch.cuda.synchronize()
    _barrier(ws_)
    ms_e2e_serial = max_over_ranks(statistics.mean(time_steps([e2e_step], K, flush, stream)[0]), ws_)
    if ms_e2e is None:
        ms_e2e, e2e_how = ms_e2e_serial, ("serial: each step copies its input in, runs the forward and copies "
                                          "the output back on one stream")

    # ---- per-kernel pass: the same forward, every kernel between its own events ----
    labels, per_kernel = kernel_breakdown(layer, x, kernels_per_step, K, W, flush, stream)
    kernel_ms = {}
    for lab, t in zip(labels, per_kernel):
        st = _stage_of(lab, kernel_ms)
        kernel_ms[st] = kernel_ms.get(st, 0.0) + statistics.mean(t)
    launches_ms = [{"kernel": lab, "ms": statistics.mean(t)} for lab, t in zip(labels, per_kernel)]
    status = moe.moe_get_device_status(layer.ws)
    if status:
        raise RuntimeError(f"device status {status} after the timed runs")

    peaks = _peaks()
    wk = _work(cfg, rows, active)
    decode = T <= 256
    fc1_s = kernel_ms["fc1"] * 1e-3
    if decode:
        achieved = wk["fc1_bytes"] / fc1_s / 1e9
        roof = dict(bound="hbm", kernel="grouped_gemm_kernel<FC1+SwiGLU>", achieved=achieved, peak=peaks["hbm"],
                    unit="GB/s", frac=achieved / peaks["hbm"], peak_kind=f"{peaks['src']} hbm_gbs")
        per_unit = f"{wk['fc1_bytes']:.0f} algorithmic bytes per launch (active slots' W1 + shared W1 + A rows + h)"
    else:
        achieved = wk["fc1_flops"] / fc1_s / 1e12
        # E4M3 operands: the measured bf16 peak times the nominal fp8 / bf16 ratio (4.5 / 2.25).
        # A timed region that ran under the power cap (sw_power_cap among the sampled reasons)
        # is held to the sustained peak, measured under the same cap; otherwise to the burst one.
        # nominal dense rates: bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s
        ratio = 6.0 if cfg.fp4 else (2.0 if cfg.act8 else 1.0)
        capped = bool(clk and "sw_power_cap" in clk.get("reasons", []))
        burst, sustained = peaks["bf16"] * ratio, peaks["bf16_sustained"] * ratio
        peak = sustained if capped else burst
        which = "bf16_tflops_sustained (the timed region ran under sw_power_cap)" if capped else \
            "bf16_tflops (burst; no power capping in the timed region)"
        roof = dict(bound="tensor", kernel="grouped_gemm_kernel<FC1+SwiGLU>", achieved=achieved,
                    peak=peak, unit="TFLOP/s", frac=achieved / peak,
                    frac_of_burst=achieved / burst, frac_of_sustained=achieved / sustained,
                    peak_kind=f"{peaks['src']} {which}" + (" x 2, the nominal e4m3 / bf16 rate ratio"
                                                            if cfg.act8 else "")
                    + (" x 6, the nominal fp4 / bf16 rate ratio" if cfg.fp4 else ""))
        per_unit = f"{wk['fc1_flops']:.4g} flops per launch = 4*H*(rows*I + T*I_shared)"
    key = (args.workload, _src_hash(os.path.join(ROOT, "serving_router_gate_gb300", "csrc", "moe_grouped_gemm.cu")))
    roof["traffic"], roof["traffic_source"] = _traffic(key[0], key[1], wk["fc1_bytes"])
    roof["algorithmic_bytes"] = wk["fc1_bytes"]
    fc1_label = next(lab for lab in labels if lab.startswith("grouped_gemm_fc1"))
    roof["kernel"] = f"grouped_gemm_kernel<FC1+SwiGLU> ({fc1_label})"
    roof["timing"] = ("CUDA events recorded on the launching stream right before and after the FC1 kernel, "
                      "as nodes of a CUDA graph of the whole forward (library launch-event hook), mean of the "
                      "timed steps, each after an L2 flush")
    roof["work"] = per_unit

    total_tokens = T if ep is not None else T * ws_
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if ep is not None else "weak", "vs_baseline": None,
        "step_timing": ("device time of one forward: CUDA events recorded by external event nodes at the "
                        "head and tail of the forward's graph, mean of the K steps" if inner else
                        "CUDA events on the stream around each step"),
        "ms_per_step_with_graph_launch": ms_replay,
        "value_with_graph_launch": T * ws_ / (ms_replay * 1e-3),
        "dtype": "nvfp4" if cfg.fp4 else ("e4m3" if cfg.act8 else "bf16"), "data": "synthetic: seeded N(0,1) activations, N(0,sigma) random-init weights of the "
                                 "workload's shapes (no checkpoint)",
        "config": {"workload": cfg.name, "shape": mi.describe(cfg), "tokens_per_gpu": T,
                   "parallelism": (f"expert parallel x{ws_} (contiguous slot ranges, shared-expert shards, one "
                                   + ("reduction by peer loads of the partials in rank order (moe_ep_reduce))"
                                      if peer is not None else "fp32 all-reduce of the partials)")
                                   if ep is not None else
                                   f"all-to-all expert parallel x{ws_} (each rank its own batch, contiguous "
                                   f"slot ranges, rows dispatched to their slots' ranks and returned; the "
                                   f"per-kernel pass and roofline: the one-GPU layer on the rank's batch)"
                                   if a2a is not None else
                                   f"replicas x{ws_} (independent token batches, no collective)"),
                   "cuda_graph": bool(graph_ok),
                   "l2": f"flushed before every timed step ({flush.describe()}); each step timed by "
                         f"its own CUDA events, flush outside them"},
        "roofline": roof,
        "e2e": {"value": total_tokens / (ms_e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2, "ms_per_step": ms_e2e, "method": e2e_how, "clocks": e2e_clk,
                "serial": {"value": total_tokens / (ms_e2e_serial * 1e-3), "ms_per_step": ms_e2e_serial}},
        "gpu_launches": (a2a_launches if a2a is not None else kernels_per_step) * K,
        "clocks": clk,
        "kernels_ms": kernel_ms,
        "launches_ms": launches_ms,
        "tflops_layer": (wk["fc1_flops"] + wk["fc2_flops"] + wk["gate_flops"]) / (ms * 1e-3) / 1e12,
        "layer_hbm": {"bytes": wk["layer_bytes"], "gbs": wk["layer_bytes"] / (ms * 1e-3) / 1e9,
                      "frac": wk["layer_bytes"] / (ms * 1e-3) / 1e9 / peaks["hbm"],
                      "what": "algorithmic bytes of the whole layer step / step time, of the measured HBM peak"},
        "grouped_gemm_tflops": (wk["fc1_flops"] + wk["fc2_flops"]) / ((kernel_ms["fc1"] + kernel_ms["fc2"]) * 1e-3) / 1e12,
        "rows": rows, "active_slots": active, "router_rechecked_tokens": refined_per_step,
    }
    if "router_logits" in [l["kernel"] for l in launches_ms]:
        # the gate GEMM on CUDA cores (T E H FMAs) against the derived fp32 peak: 152 SMs x 128
        # lanes x 2 flops x the clock (the maximum, and the median the timed region sampled)
        rl_ms = sum(l["ms"] for l in launches_ms if l["kernel"] == "router_logits")
        tf = 2.0 * T * cfg.E * H / (rl_ms * 1e-3) / 1e12
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz_max = (clk or {}).get("sm_max_mhz") or 2070.0
        mhz = (clk or {}).get("sm_mhz") or mhz_max
        res["router_logits"] = {"achieved_tflops": tf, "ms": rl_ms,
                                "peak_tflops_at_max_clock": sms * 128 * 2 * mhz_max * 1e-6,
                                "frac_at_max_clock": tf / (sms * 128 * 2 * mhz_max * 1e-6),
                                "peak_tflops_at_sampled_clock": sms * 128 * 2 * mhz * 1e-6,
                                "frac_at_sampled_clock": tf / (sms * 128 * 2 * mhz * 1e-6)}
    if rank == 0 and ws_ == 1 and not args.no_cpu_baseline:
        base, _ = run_cpu_baseline(inp, cfg, target_s=args.cpu_seconds)
        res["cpu_baseline"] = base
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws_ > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def eager_kernel_medians(step, marked_step, K, flush, stream, spare_events=8):
    """Each library kernel of an eagerly launched step timed on its own: the launch-event
    hook records a CUDA event before every launch (and marked_step may add marks, e.g.
    after phases whose work is not the library's); K steps, each after an L2 flush.
    Returns the labels and the median interval of each launch position, and the per-label
    sums of those medians (marks left out)."""
    import serving_router_gate_gb300 as moe
    c0 = moe.moe_get_launch_count()
    step()
    n_launch = moe.moe_get_launch_count() - c0
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_launch + spare_events)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    per_pos, labels = None, None
    for _ in range(K):
        flush()
        moe.moe_launch_events_arm(evs)
        try:
            marked_step()
            labels = moe.moe_launch_events_used()
        finally:
            moe.moe_launch_events_arm(None)
        torch.cuda.synchronize()
        if per_pos is None:
            per_pos = [[] for _ in range(len(labels) - 1)]
        for i in range(len(labels) - 1):
            per_pos[i].append(evs[i].elapsed_time(evs[i + 1]))
    med = [statistics.median(v) for v in per_pos]
    kernels = {}
    for lab, m in zip(labels, med):
        if lab != "mark":
            kernels[lab] = kernels.get(lab, 0.0) + m
    return labels[:-1], med, kernels


def bench_a2a_local(args):
    """All-to-all expert parallelism over R ranks held by this process on one GPU
    (a2a_forward_local: the ranks' steps one after another, the exchanges as device
    copies), the workload's batch split into R ranks' batches.  Times the whole step and,
    in a second pass, every library kernel between its own events (launch-event hook,
    eager, a mark after each phase so the exchanges' copies fall in marked intervals);
    reports the row reorder kernel against the HBM peak."""
    import serving_router_gate_gb300 as moe
    from serving_router_gate_gb300.expert_parallel import a2a_forward_local
    R = args.a2a_ranks
    cfg = mi.CONFIGS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = mi.make_inputs(cfg, device=dev)
    per = -(-cfg.T // R)
    xs = list(inp["x"].split(per))
    if len(xs) != R:
        raise SystemExit(f"bench.py: {cfg.T} tokens do not make {R} ranks' batches")
    layers = [_a2a_layer(inp, cfg, R, r, dev, max_T=per) for r in range(R)]
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    K, W = args.steps, args.warmup

    def step():
        return a2a_forward_local(layers, xs)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    t = time_steps([step], K, flush, stream)[0]
    clk = clocks.stop()
    ms = statistics.mean(t)
    for L in layers:
        if moe.moe_get_device_status(L.ws):
            raise RuntimeError("device status set after the timed steps")

    # per-kernel pass: a mark after each phase, so the exchanges' copies fall in marked intervals
    labels, med, kernels = eager_kernel_medians(
        step, lambda: a2a_forward_local(layers, xs, after_phase=lambda name: moe.moe_launch_events_mark()),
        K, flush, stream)
    # row reorders: one launch per rank, moving its received rows into slot order
    rows_in = [L.rows_in for L in layers]
    H = cfg.H
    reg = [(i, m) for i, (lab, m) in enumerate(zip(labels, med)) if lab.startswith("a2a_regroup")]
    reg_bytes = sum(2 * r * H * 2 for r in rows_in)
    reg_ms = sum(m for _, m in reg)
    peaks = _peaks()
    gbs = reg_bytes / (reg_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic: seeded N(0,1) activations, N(0,sigma) random-init weights",
        "config": {"workload": cfg.name, "shape": mi.describe(cfg),
                   "parallelism": f"all-to-all expert parallel over {R} ranks held by one process on one GPU "
                                  f"({per} tokens each; the exchanges are device copies; each rank's split "
                                  f"sizes are read on the host, one synchronisation per rank per step)",
                   "l2": f"flushed before every timed step ({flush.describe()})"},
        "rows_received": rows_in,
        "kernels_ms": kernels,
        "a2a_regroup": {"bound": "hbm", "launches": len(reg), "algorithmic_bytes": reg_bytes,
                        "ms": reg_ms, "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm"],
                        "work": "2 x rows received x H x 2 bytes per launch (each row read and written once), "
                                "one launch per rank (FC2 stores its rows back in arrival order itself)",
                        "timing": "launch-event hook: a CUDA event before every library launch and a mark "
                                  "after each phase, median per launch over the steps, each after an L2 flush"},
        "clocks": clk,
    }
    print(json.dumps(res), flush=True)


def bench_ep_local(args):
    """Expert parallelism with the peer reduction over R ranks held by this process on one
    GPU (every rank routes the whole batch, computes its slot range and shared shard into
    its partial slot, raises its flag; then every rank forms the rank-order sum of all
    partials): times the whole step and reports the reduction kernel against the HBM peak
    (all ranks' buffers are local here; on R GPUs R - 1 of the R reads go to peers)."""
    import serving_router_gate_gb300 as moe
    from serving_router_gate_gb300.expert_parallel import PeerReduction
    R = args.ep_ranks
    cfg = mi.CONFIGS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = mi.make_inputs(cfg, device=dev)
    reds = PeerReduction.local_set(cfg.T, cfg.H, R, dev)
    eps = [_ep_layer(inp, cfg, R, r, dev, reds[r]) for r in range(R)]
    x = inp["x"]
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    K, W = args.steps, args.warmup

    def step():
        for e in eps:
            e.write_partial(x)
        for r in reds:
            r.reduce()

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    t = time_steps([step], K, flush, stream)[0]
    clk = clocks.stop()
    ms = statistics.mean(t)
    def marked():
        step()
        moe.moe_launch_events_mark()

    _, _, kernels = eager_kernel_medians(step, marked, K, flush, stream)
    for r in reds:
        if moe.moe_get_device_status(r.ws):
            raise RuntimeError("device status set by the reduction")
    red_ms = kernels.get("ep_reduce_kernel", 0.0)
    red_bytes = R * (R + 1) * cfg.T * cfg.H * 2  # per rank: R partials read, its output written
    peaks = _peaks()
    gbs = red_bytes / (red_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic: seeded N(0,1) activations, N(0,sigma) random-init weights",
        "config": {"workload": cfg.name, "shape": mi.describe(cfg),
                   "parallelism": f"expert parallel over {R} ranks held by one process on one GPU (slot ranges "
                                  f"and shared shards; the reduction by loads of every rank's partial)",
                   "l2": f"flushed before every timed step ({flush.describe()})"},
        "kernels_ms": kernels,
        "ep_reduce": {"bound": "hbm", "launches": R, "algorithmic_bytes": red_bytes, "ms": red_ms,
                      "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
                      "work": "per rank: the R partials [T, H] bf16 read, its output written",
                      "timing": "launch-event hook, median per launch over the steps, each after an L2 flush"},
        "clocks": clk,
    }
    print(json.dumps(res), flush=True)


def bench_reference(args):
    """The fp64 oracle, as it stands, on the host cores: each step a bounded
    sample of the workload (its first n tokens through the whole layer)."""
    ws_ = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    cfg = mi.CONFIGS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = mi.make_inputs(cfg, device=dev)
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}

    fp8 = _oracle_fp8(oracle, cfg, cpu)
    fp4 = _oracle_nvfp4(oracle, cfg, cpu)

    def step(n):
        oracle.moe_layer(cpu["x"][:n], cpu["Wg"], cpu["bias"], cfg.k, cfg.renorm, cpu["W1"], cpu["W2"],
                         rep_offset=cpu["rep_offset"], rep_slots=cpu["rep_slots"], W1s=cpu["W1s"],
                         W2s=cpu["W2s"], shared_gate_w=cpu["w_s"], S=cfg.slots, n_group=cfg.n_group,
                         topk_group=cfg.topk_group, on_input=cfg.on_input, fp8=fp8, nvfp4=fp4)

    threads = oracle.get_threads()
    n0 = min(cfg.T, max(8, threads))
    t0 = time.perf_counter()
    step(n0)
    per = (time.perf_counter() - t0) / n0
    budget = 150.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    n = max(1, min(cfg.T, int(budget / max(per, 1e-6))))
    for _ in range(args.warmup):
        step(n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(n)
    dt = (time.perf_counter() - t0) / args.steps
    v = n / dt
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws_,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic: seeded inputs of the workload's shapes",
           "config": {"workload": cfg.name, "shape": mi.describe(cfg), "tokens_per_step": n},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                            "sample": f"first {n} of the {cfg.T} tokens per step, whole layer in fp64"},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(mi.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch every step from Python instead of replaying a CUDA graph of one step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--a2a-ranks", type=int, default=0,
                    help="one GPU: run the all-to-all expert-parallel layer over this many ranks held by one "
                         "process (exchanges as device copies) and time its kernels")
    ap.add_argument("--ep-ranks", type=int, default=0,
                    help="one GPU: run expert parallelism with the peer reduction over this many ranks held by "
                         "one process and time its kernels")
    ap.add_argument("--reduce", choices=["collective", "peer"], default="collective",
                    help="--partition ep on several GPUs: the all-reduce of torch.distributed, or the library's "
                         "reduction by loads of every rank's partial (CUDA IPC)")
    ap.add_argument("--partition", choices=["ep", "a2a", "replicas"], default="ep",
                    help="with more than one rank: expert parallelism over one batch with one reduction "
                         "(default), all-to-all expert parallelism (each rank its own batch, rows dispatched "
                         "to their experts' ranks and back) or independent replicas, each with its own batch")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws = os.environ.get("WORLD_SIZE")
    if ws is None and args.gpus > 1:
        # not started by a launcher: start one rank per GPU on this node, as torchrun would
        port = os.environ.get("MASTER_PORT", "29531")
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", port, os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))
    if ws is not None and int(ws) != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but the launcher started {ws} ranks")
    if args.impl == "reference":
        bench_reference(args)
    elif args.a2a_ranks > 0 or args.ep_ranks > 0:
        if ws is not None and int(ws) > 1:
            sys.exit("bench.py: --a2a-ranks / --ep-ranks hold every rank in one process on one GPU")
        if args.a2a_ranks > 0:
            bench_a2a_local(args)
        else:
            bench_ep_local(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
