"""Benchmark of the single-GPU forward pass of one routed MoE layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step = route -> permute -> gate/up GEMM -> down GEMM -> combine over one
batch of the workload, inputs and weights resident in HBM, replayed from CUDA
graphs.  Prints one JSON line (rank 0).  With N > 1 (torchrun, one rank per
GPU) every rank runs its own replica on its own batch (no collective on the
data path) and the whole-job throughput is the tokens of all ranks over the
slowest rank's time.

--impl reference times the CPU oracle (fp64, host cores) on a bounded sample of
the same workload; it is the deliberately slow baseline of this repository.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_inputs as mi  # noqa: E402

HEADLINE = "prefill"
FFN_PART = "gate_up+down+combine"  # the moe_ffn_combine call of the one-launch step
# Workloads measured after the headline in the same process (the `workloads` record of the line).
SUB_WORKLOADS = ["mixtral_decode", "dsv3_decode", "skew_eplb", "tiny", "dsv4_fp4_decode"]
METRIC = "MoE layer tokens/s"
# ncu DRAM bytes (read + write) per launch of a workload's dominant kernel, keyed by the
# workload, the launch form (one-launch FFN or the gate/up launch) and the hash of the
# kernel source the capture was taken from; a changed kernel source gives no entry (null).
TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (one pass) on the full-size workloads: the
    # first launch of the dominant grouped GEMM kernel in a bench process.  Taken on the kernel revision
    # before FP8 / FP4 single-CTA launches moved to 64-row chunks; the present revision has no capture.
    "prefill:split:b6a55799c140746a": 4824612864 + 78791168,          # gate/up, SM pairs
    "mixtral_decode:ffn:b6a55799c140746a": 2821686528 + 5934080,      # one-launch FFN kernel (without the reduction)
    "dsv3_decode:split:b6a55799c140746a": 7491252480 + 8620800,       # gate/up
    "skew_eplb:split:b6a55799c140746a": 2876958464 + 4845312,         # gate/up
    "dsv4_fp4_decode:split:b6a55799c140746a": 5070470400 + 8520960,   # gate/up
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def src_hash(*names):
    """Hash of the kernel sources' code: comments and blank space are dropped first, so that an
    edit of a comment keeps the ncu captures keyed by it."""
    h = hashlib.sha256()
    for n in names:
        text = open(os.path.join(ROOT, "routed_expert_layer_moe_gb300", "csrc", n)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


class ClockSampler:
    """SM clocks and clock-event (throttle) reasons sampled during the timed
    region: NVML through ctypes every 2 ms, else nvidia-smi every 200 ms."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (sm_mhz, max_mhz, reason names)
        self._stop = None
        self._thread = None
        self.proc = None
        self.source = None

    def _nvml(self):
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if nv.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return None
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))

        def read():
            c = ctypes.c_uint()
            r = ctypes.c_ulonglong()
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) != 0:
                return None
            get_reasons(h, ctypes.byref(r))
            names = [n for b, n in self.REASONS.items() if r.value & b]
            return float(c.value), float(mx.value), names

        return read

    def __enter__(self):
        import threading
        read = self._nvml()
        if read is not None and read() is not None:
            self.source = "nvml"
            self._stop = threading.Event()

            def loop():
                while not self._stop.is_set():
                    s = read()
                    if s is not None:
                        self.samples.append(s)
                    time.sleep(0.002)

            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for l in out.splitlines():
                f = [x.strip() for x in l.split(",")]
                if len(f) < 9:
                    continue
                try:
                    self.samples.append((float(f[1]), float(f[2]),
                                         [n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")]))
                except ValueError:
                    continue

    def summary(self):
        if not self.samples:
            return None
        sm = [s[0] for s in self.samples]
        reasons = sorted({n for s in self.samples for n in s[2]})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s[1] for s in self.samples), "reasons": reasons,
                "samples": len(sm), "source": self.source}


# ---- the multi-rank pieces (one replica of the layer per GPU; no data-path collective) ----

def replica_seed(rank: int) -> int:
    """Each replica draws its own batch: the generator seed is the rank."""
    return rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (the timed region is bracketed by barriers on every rank)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch each step, timed by the slowest."""
    return world * tokens_per_step * steps / (total_ms * 1e-3)


def problem_of(cfg, moe):
    return moe.Problem.make(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, P=cfg.P, M_max=cfg.M_max,
                            has_shared=cfg.S, act=cfg.act, wt=cfg.wt, out=cfg.out, layout=cfg.layout)


def to_dev(a, torch, dev):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def expert_bytes(cfg):
    """Bytes of one expert's weights (W13 + W2, plus fp32 block scales for e4m3 / e2m1)."""
    esz = {"f32": 4, "bf16": 2, "e4m3": 1, "e2m1": 0.5}[cfg.wt]
    b13 = int(2 * cfg.I * cfg.H * esz)
    b2 = int(cfg.H * cfg.I * esz)
    if cfg.wt in ("e4m3", "e2m1"):
        b13 += (2 * cfg.I // 128) * (cfg.H // 128) * 4
        b2 += (cfg.H // 128) * (cfg.I // 128) * 4
    return b13, b2


def run_gpu(args, cfg, rank, world, local_rank, split, lite=False):
    """Build the layer of one workload, capture its step as CUDA graphs and time `args.steps`
    replays.  lite: the step timing alone (no end-to-end loop, no calls outside the step), for
    the workloads measured after the headline."""
    import torch

    import routed_expert_layer_moe_gb300 as moe

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    seed = replica_seed(rank)
    x, logits = mi.activations(cfg, seed)
    w13, w13s = mi.expert_weights(cfg, "w13")
    w2, w2s = mi.expert_weights(cfg, "w2")
    p = problem_of(cfg, moe)
    # EPLB replica map: the hottest logical experts of this batch, counted from
    # the GPU's own routing of it
    p2l = None
    if cfg.redundant:
        pr = moe.Problem.make(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, M_max=max(cfg.M_max, 1),
                              act=cfg.act, wt=cfg.wt, out=cfg.out, layout=cfg.layout)
        ids = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device=dev)
        wts = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device=dev)
        moe.moe_route_topk(pr, to_dev(logits, torch, dev), ids, wts)
        counts = np.bincount(ids.cpu().numpy().ravel(), minlength=cfg.E)
        p2l = mi.replica_map(counts, cfg.E, cfg.redundant)
    order = torch.from_numpy(mi.slot_experts(cfg, p2l)).to(dev)

    def slots(a):
        if a is None:
            return None
        t = to_dev(a, torch, dev)
        return t.index_select(0, order).contiguous() if (cfg.redundant or t.shape[0] != order.numel()) else t

    L = moe.MoeLayer(p, cfg.act, cfg.wt, cfg.out, slots(w13), slots(w2), slots(w13s), slots(w2s),
                     phys_to_log=None if p2l is None else torch.from_numpy(p2l).to(dev), device=dev)
    del w13, w2, w13s, w2s
    xd, ld = to_dev(x, torch, dev), to_dev(logits, torch, dev)
    stream = torch.cuda.Stream(dev)
    # eager warm-up on the capture stream (first calls cache device attributes)
    with torch.cuda.stream(stream):
        L.forward(xd, ld, stream, fused=not split)
    stream.synchronize()
    assert int(L.err.item()) == 0, "device error flag %d" % int(L.err.item())

    # route + dispatch through moe_route_permute (one launch for small batches); then
    if split:  # gate/up, down and combine as separate calls (gate/up timed on its own)
        names = ["route+permute", "gate_up", "down", "combine"]
        parts = [lambda: L.route_permute(ld, xd, stream), lambda: L.swiglu(stream),
                 lambda: L.down(stream), lambda: L.combine(stream)]
    else:  # moe_ffn_combine: gate/up and down in one launch, the combine inside the split-K reduction
        names = ["route+permute", FFN_PART]
        parts = [lambda: L.route_permute(ld, xd, stream), lambda: L.ffn_combine(stream)]
    NP = len(parts)
    graphs = []
    for fn in parts:
        try:  # keep the graph itself (not only its executable) so its kernel nodes can be counted
            g = torch.cuda.CUDAGraph(keep_graph=True)
        except TypeError:
            g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        if hasattr(g, "instantiate"):
            g.instantiate()
        graphs.append(g)
    n_launch, launch_src = count_launches(graphs, cfg, p2l is not None)

    def step():
        for g in graphs:
            g.replay()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(NP + 1)] for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        with torch.cuda.stream(stream):
            for i in range(K):
                ev[i][0].record(stream)
                for j, g in enumerate(graphs):
                    g.replay()
                    ev[i][j + 1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = ev[0][0].elapsed_time(ev[K - 1][NP])
    part_ms = {names[j]: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) for j in range(NP)}
    total_ms = max_over_ranks(total_ms, world, dev)

    mm = L.masked_m.cpu().numpy()
    base = dict(total_ms=total_ms, part_ms=part_ms, masked_m=mm, touched=int((mm > 0).sum()), clocks=clk.summary(),
                n_launch=n_launch, launch_src=launch_src, x=x, logits=logits)
    if lite:
        return base

    # ---- end to end through the host: pinned inputs in, output back, every step.  A copy
    # stream moves step i+1's inputs in (and step i-1's output out) while step i computes:
    # two device staging buffers each way, ordered by events; the step's graphs read xd / ld
    # and write L.out, which are filled from / emptied into the staging buffers on the
    # compute stream (device copies, inside the timed region like everything else).
    xh = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if x.dtype == np.uint16 else x)
    xh = (xh.view(torch.bfloat16) if x.dtype == np.uint16 else xh).pin_memory()
    lh = torch.from_numpy(logits).pin_memory()
    oh = torch.empty(L.out.shape, dtype=L.out.dtype).pin_memory()
    cs = torch.cuda.Stream(dev)
    xs = [torch.empty_like(xd) for _ in range(2)]
    ls = [torch.empty_like(ld) for _ in range(2)]
    os_ = [torch.empty_like(L.out) for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]   # staged inputs b have landed
    in_free = [torch.cuda.Event() for _ in range(2)]    # staged inputs b were copied into xd / ld
    out_ready = [torch.cuda.Event() for _ in range(2)]  # staged output b holds a step's result
    out_free = [torch.cuda.Event() for _ in range(2)]   # staged output b was read back to the host

    def run_e2e(n):
        used_in, used_out = [False, False], [False, False]

        def h2d(b):
            with torch.cuda.stream(cs):
                if used_in[b]:
                    cs.wait_event(in_free[b])
                xs[b].copy_(xh, non_blocking=True)
                ls[b].copy_(lh, non_blocking=True)
                in_ready[b].record(cs)
            used_in[b] = True

        cs.wait_stream(stream)
        h2d(0)
        for i in range(n):
            b = i & 1
            stream.wait_event(in_ready[b])
            xd.copy_(xs[b], non_blocking=True)
            ld.copy_(ls[b], non_blocking=True)
            in_free[b].record(stream)
            if i + 1 < n:
                h2d(b ^ 1)
            step()
            if used_out[b]:
                stream.wait_event(out_free[b])
            os_[b].copy_(L.out, non_blocking=True)
            out_ready[b].record(stream)
            used_out[b] = True
            with torch.cuda.stream(cs):
                cs.wait_event(out_ready[b])
                oh.copy_(os_[b], non_blocking=True)
                out_free[b].record(cs)
        stream.wait_stream(cs)

    with torch.cuda.stream(stream):
        run_e2e(max(1, args.warmup))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_e2e(K)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    assert int(L.err.item()) == 0, "device error flag %d" % int(L.err.item())

    aux = aux_timings(moe, L, cfg, ld, stream, torch) if world == 1 else None
    return dict(base, e2e_ms=e2e_ms, h2d=xh.numel() * xh.element_size() + lh.numel() * lh.element_size(),
                d2h=oh.numel() * oh.element_size(), aux=aux)


def grouped_router_params(cfg):
    """n_group / topk_group for the grouped router on this workload (8 groups, 4 kept, when E allows)."""
    ng = 8 if cfg.E % 8 == 0 else 1
    tg = max(1, ng // 2)
    while tg < ng and cfg.K > tg * (cfg.E // ng):
        tg += 1
    return ng, tg


def aux_timings(moe, L, cfg, ld, stream, torch, reps=50, window=16):
    """Device time of the calls outside the layer step: the grouped router on this
    workload's logits, one EPLB record of masked_m, one EPLB rebalance of a
    window.  Each is captured `reps` times in one graph; time / reps."""
    ng, tg = grouped_router_params(cfg)
    dev = ld.device
    win = torch.zeros((window, cfg.P), dtype=torch.int32, device=dev)
    ll = torch.empty(cfg.E, dtype=torch.int64, device=dev)
    newmap = torch.empty(cfg.P, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.empty_like(L.ids)
    w = torch.empty_like(L.w)
    calls = {
        "route_grouped": lambda: moe.moe_route_grouped_topk(L.p, ld, None, ng, tg, ids, w, stream=stream),
        "route_softmax": lambda: moe.moe_route_topk(L.p, ld, ids, w, stream),
        "eplb_record": lambda i: moe.moe_eplb_record(L.p, L.masked_m, i, window, win, stream),
        "eplb_rebalance": lambda: moe.moe_eplb_rebalance(L.p, win, window, L.p2l, ll, newmap, err, stream),
    }
    out = {"grouped_router": {"n_group": ng, "topk_group": tg}, "eplb_window": window}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                fn(i) if name == "eplb_record" else fn()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(4):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        out[name + "_us"] = round(e0.elapsed_time(e1) * 1e3 / (4 * reps), 2)
    assert int(err.item()) == 0, "EPLB rebalance flagged %d" % int(err.item())
    return out


def count_launches(graphs, cfg, with_map):
    """Kernels of this library in one step: the kernel nodes of the captured graphs
    (memset nodes excluded).  Falls back to the static count of the calls' kernels
    (route 1; permute [map] + mark + scan + scatter; gate/up 1; down 1 or 2; combine 1)."""
    try:
        import ctypes
        rt = ctypes.CDLL("libcudart.so.13")
        total = 0
        for g in graphs:
            h = ctypes.c_void_p(g.raw_cuda_graph())
            n = ctypes.c_size_t(0)
            if rt.cudaGraphGetNodes(h, None, ctypes.byref(n)) != 0:
                raise RuntimeError("cudaGraphGetNodes")
            nodes = (ctypes.c_void_p * n.value)()
            rt.cudaGraphGetNodes(h, nodes, ctypes.byref(n))
            for nd in nodes:
                t = ctypes.c_int(-1)
                rt.cudaGraphNodeGetType(ctypes.c_void_p(nd), ctypes.byref(t))
                total += t.value == 0  # cudaGraphNodeTypeKernel
        return int(total), "graph kernel nodes"
    except Exception:
        return 1 + 3 + (1 if with_map else 0) + 1 + 1 + 1, "static count"


def ffn_roofline(cfg, res, peaks, moe_src, split):
    """Roofline of the dominant kernel.  One launch of gate/up and down (default): the W13 and
    W2 (+ scales) of every slot with rows, Xg read, Hg written and read back, Yg written; its
    event-timed duration includes the split-K reduction kernel the same call enqueues.  With
    --split-ffn: the gate/up launch alone (W13 + scales, Xg read, Hg written)."""
    hbm, _, _, src = peaks
    b13, b2 = expert_bytes(cfg)
    rows = int(res["masked_m"].sum())
    esz = {"f32": 4, "bf16": 2, "e4m3": 1}[cfg.gemm]
    x_b, h_b = rows * cfg.H * esz, rows * cfg.I * esz
    if cfg.gemm == "e4m3":
        x_b += rows * (cfg.H // 128) * 4
        h_b += rows * (cfg.I // 128) * 4
    if split:
        algo = res["touched"] * b13 + x_b + h_b
        dur_s = res["part_ms"]["gate_up"] * 1e-3
        kernel = "grouped_gemm_tc (gate/up + SwiGLU)"
    else:
        ysz = 4 if cfg.gemm == "f32" else 2
        algo = res["touched"] * (b13 + b2) + x_b + 2 * h_b + rows * cfg.H * ysz + cfg.T * cfg.H * ysz
        dur_s = res["part_ms"][FFN_PART] * 1e-3
        kernel = ("moe_ffn_combine: grouped_gemm_tc, gate/up + SwiGLU + down in one launch, then the split-K "
                  "reduction with the combine")
    achieved = algo / dur_s / 1e9
    traffic = TRAFFIC.get("%s:%s:%s" % (cfg.name, "split" if split else "ffn", moe_src))
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1),
            "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
            "algorithmic_bytes": int(algo), "avg_launch_us": round(dur_s * 1e6, 2), "peak_source": src}


def tensor_roofline(cfg, res, peaks, split):
    """The dominant kernel against the dense tensor-core peak of its MMA type (the second
    fraction the prefill workload reports): useful FLOPs (2 per multiply-add over the valid
    rows) / its event-timed duration.  bf16: the measured sustained bf16 peak (the kernel runs
    inside a long step); e4m3 and e2m1 x e4m3 (kind::f8f6f4, the FP8 rate): 2 x that, the
    recipe's nominal FP8 / bf16 ratio."""
    _, _, bf16_sus, src = peaks
    rows = int(res["masked_m"].sum())
    f13 = 2.0 * rows * 2 * cfg.I * cfg.H
    f2 = 2.0 * rows * cfg.H * cfg.I
    if split:
        flops, dur = f13, res["part_ms"]["gate_up"] * 1e-3
    else:
        flops, dur = f13 + f2, res["part_ms"][FFN_PART] * 1e-3
    if cfg.gemm == "f32":
        return None
    peak = bf16_sus * (2.0 if cfg.gemm == "e4m3" else 1.0)
    ach = flops / dur / 1e12
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(ach / peak, 4), "flops": int(flops),
            "peak_source": "%s (bf16 sustained%s)" % (src, " x 2 for FP8" if cfg.gemm == "e4m3" else "")}


def cpu_baseline(cfg, x, logits, budget_s=12.0):
    """The oracle on the host cores, whole-layer tokens/s on a bounded sample of tokens."""
    import oracle

    w13, w13s = mi.expert_weights(cfg, "w13")
    w2, w2s = mi.expert_weights(cfg, "w2")
    t0 = time.time()
    oracle.layer(cfg, x, logits, w13, w13s, w2, w2s, tokens=np.array([0], np.int32))
    one = max(time.time() - t0, 1e-3)
    n = int(max(1, min(cfg.T, budget_s / one)))
    toks = np.arange(n, dtype=np.int32)
    t0 = time.time()
    oracle.layer(cfg, x, logits, w13, w13s, w2, w2s, tokens=toks)
    dt = time.time() - t0
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d of the %d tokens of one %s batch, whole layer per token, fp64" % (n, cfg.T, cfg.name)}


def run_reference(args, cfg, rank):
    """The oracle as the reference arm: each step is a bounded sample of tokens."""
    import oracle

    x, logits = mi.activations(cfg, 0)
    w13, w13s = mi.expert_weights(cfg, "w13")
    w2, w2s = mi.expert_weights(cfg, "w2")
    t0 = time.time()
    oracle.layer(cfg, x, logits, w13, w13s, w2, w2s, tokens=np.array([0], np.int32))
    one = max(time.time() - t0, 1e-3)
    total_budget = 150.0
    per_step = max(1, min(cfg.T, int(total_budget / max(1, args.steps + args.warmup) / one)))
    toks = np.arange(per_step, dtype=np.int32)
    for _ in range(args.warmup):
        oracle.layer(cfg, x, logits, w13, w13s, w2, w2s, tokens=toks)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.layer(cfg, x, logits, w13, w13s, w2, w2s, tokens=toks)
    dt = time.time() - t0
    value = per_step * args.steps / dt
    sample = "%d of the %d tokens of one %s batch per step, whole layer per token, fp64" % (per_step, cfg.T, cfg.name)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg, args.gpus),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def config_dict(cfg, n):
    return {"workload": cfg.name, "description": cfg.description, "tokens_per_step": cfg.T, "H": cfg.H, "I": cfg.I,
            "E": cfg.E, "K": cfg.K, "shared_experts": cfg.S, "physical_slots": cfg.P, "layout": cfg.layout,
            "M_max": cfg.M_max, "expert_dtype": cfg.wt, "parallelism": "replicas%d" % n if n > 1 else "single-gpu",
            "l2": "expert weights exceed L2 (129 MB), no flush" if expert_bytes(cfg)[0] * cfg.E > 2 * 129e6
            else "small workload: L2-resident (launch-latency bound)"}


def kernel_rooflines(cfg, res, peaks, split):
    """HBM roofline of each timed GEMM part of the step: algorithmic bytes (the W13 / W2 (+ block
    scales) of every slot with rows, the grouped activations read and written) over its
    event-timed duration."""
    hbm = peaks[0]
    b13, b2 = expert_bytes(cfg)
    rows = int(res["masked_m"].sum())
    esz = {"f32": 4, "bf16": 2, "e4m3": 1}[cfg.gemm]
    x_b, h_b = rows * cfg.H * esz, rows * cfg.I * esz
    if cfg.gemm == "e4m3":
        x_b += rows * (cfg.H // 128) * 4
        h_b += rows * (cfg.I // 128) * 4
    y_b = rows * cfg.H * (4 if cfg.gemm == "f32" else 2)
    parts = {"gate_up": res["touched"] * b13 + x_b + h_b, "down": res["touched"] * b2 + h_b + y_b,
             FFN_PART: res["touched"] * (b13 + b2) + x_b + 2 * h_b + y_b + cfg.T * cfg.H * (4 if cfg.gemm == "f32" else 2)}
    out = {}
    for name, algo in parts.items():
        if name in res["part_ms"]:
            ach = algo / (res["part_ms"][name] * 1e-3) / 1e9
            out[name] = {"achieved_GBps": round(ach, 1), "frac": round(ach / hbm, 4), "algorithmic_bytes": int(algo),
                         "avg_launch_us": round(res["part_ms"][name] * 1e3, 2)}
    return out


def summarize(cfg, res, peaks, moe_src, split, K):
    """The measured figures of one workload: rooflines of the dominant kernel (HBM and tensor),
    each GEMM part's HBM fraction, the step breakdown, the layer's touched-bytes rate, clocks."""
    ms = res["total_ms"] / K
    b13, b2 = expert_bytes(cfg)
    layer_bytes = res["touched"] * (b13 + b2)
    return {
        "roofline": ffn_roofline(cfg, res, peaks, moe_src, split),
        "roofline_tensor": tensor_roofline(cfg, res, peaks, split),
        "kernels_hbm": kernel_rooflines(cfg, res, peaks, split),
        "step_breakdown_us": {k: round(v * 1e3, 2) for k, v in res["part_ms"].items()},
        "touched_slots": res["touched"],
        "layer_hbm": {"touched_expert_bytes": int(layer_bytes),
                      "achieved_GBps": round(layer_bytes / (ms * 1e-3) / 1e9, 1),
                      "frac_of_peak": round(layer_bytes / (ms * 1e-3) / 1e9 / peaks[0], 4)},
        "clocks": res["clocks"],
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=HEADLINE, choices=list(mi.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the selected workload only (no `workloads` record of the other workloads)")
    ap.add_argument("--ffn", default="auto", choices=["auto", "fused", "split"],
                    help="gate/up and down as one launch (moe_grouped_ffn) or two; auto: one launch for bf16 "
                         "experts, two for e4m3 / e2m1 (the faster of the two on GB300 for each)")
    ap.add_argument("--override", default="",
                    help="comma-separated field=value changes to the workload, e.g. T=2048,E=128 (profiling cases)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    cfg = mi.CONFIGS[args.config]
    if args.override:
        kw = {}
        for item in args.override.split(","):
            k, v = item.split("=")
            kw[k.strip()] = type(getattr(cfg, k.strip()))(v)
        cfg = cfg.replace(name=cfg.name + "[" + args.override + "]", **kw)
    args.split_ffn = args.ffn == "split" or (args.ffn == "auto" and cfg.gemm != "bf16")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, cfg, rank)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    peaks = load_peaks()
    moe_src = src_hash("gemm_tc.cu", "common.cuh")
    res = run_gpu(args, cfg, rank, world, local_rank, args.split_ffn)
    if rank == 0:
        K = args.steps
        value = job_throughput(world, cfg.T, K, res["total_ms"])
        e2e = job_throughput(world, cfg.T, K, res["e2e_ms"])
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(res["total_ms"] / K, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.gemm if cfg.wt == cfg.gemm else "%s x %s" % (cfg.wt, cfg.gemm),
            "data": "synthetic (seeded generator, random-init experts)",
            "config": dict(config_dict(cfg, world), ffn="two launches" if args.split_ffn else "one launch"),
        }
        line.update(summarize(cfg, res, peaks, moe_src, args.split_ffn, K))
        line.update({
            "aux_calls_us": res["aux"],
            "e2e": {"value": round(e2e, 1), "unit": "tokens/s", "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"]},
            "gpu_launches": res["n_launch"] * K,
            "gpu_launches_per_step": {"kernels": res["n_launch"], "counted_from": res["launch_src"]},
        })
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(cfg, res["x"], res["logits"])
    # the other workloads, each measured in this process with the same step counts (one GPU only)
    if world == 1 and not args.no_workloads and not args.override:
        import torch
        del res
        torch.cuda.empty_cache()
        subs = {}
        for name in SUB_WORKLOADS:
            if name == cfg.name:
                continue
            c = mi.CONFIGS[name]
            split = args.ffn == "split" or (args.ffn == "auto" and c.gemm != "bf16")
            r = run_gpu(args, c, rank, world, local_rank, split, lite=True)
            K = args.steps
            entry = {"tokens_per_s": round(job_throughput(world, c.T, K, r["total_ms"]), 1),
                     "ms_per_step": round(r["total_ms"] / K, 4), "T": c.T, "expert_dtype": c.wt,
                     "ffn": "two launches" if split else "one launch"}
            entry.update(summarize(c, r, peaks, moe_src, split, K))
            entry["gpu_launches_per_step"] = r["n_launch"]
            subs[name] = entry
            del r
            torch.cuda.empty_cache()
        line["workloads"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
