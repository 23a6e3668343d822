"""Benchmark of the normalize-then-quantize path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs,
each operation at its largest workload, one launch each, in this order:
  (B) fused q/kv RMSNorm + MXFP8      q [8192,1536], kv [8192,512]
  (C) static per-head FP8 of Q/K/V    T = 151,153 packed tokens, H = 12, D 192/192/128
  (A) gated RMSNorm + per-token FP8   x, gate [65536, 64, 128], sigmoid
Metric: achieved HBM GB/s (algorithmic bytes: every input read once, every
output written once) over the step, per kernel and in total; rows/s per kernel.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torchrun: each rank runs the same per-GPU workload on its
own GPU (weak scaling, no collective on the data path); rank 0 prints one JSON
line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "achieved HBM GB/s and % of GB300 peak per kernel; rows/s at 1 GPU vs CPU oracle"
UNIT = "GB/s"
WORKLOAD = ("step = rmsnorm_quant_mx q[8192,1536]+kv[8192,512] -> static_head_quant "
            "Q,K[151153,12,192]+V[151153,12,128] -> gated_rmsnorm_quant_token "
            "x,gate[65536,64,128] sigmoid; seed 0")
# oracle samples (tokens of A, rows of B, tokens of C): about 10 s of one host
# core for the CPU baseline, about 2 s per step for the reference arm
CPU_SAMPLE = (4096, 8192, 16384)
REF_SAMPLE = (512, 4096, 4096)
# GB300's nominal HBM3e bandwidth (about 8 TB/s); the roofline fractions are
# given against it and against the measured copy bandwidth
NOMINAL_HBM_GBS = 8000.0
L2_NOTE = ("inputs larger than L2: (A) 2.15 GB and (C) 2.61 GB per launch; the 55 MB of (B) "
           "is evicted by the ~5 GB the other two kernels stream between its launches")


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's
    sources are unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel_key)
    if not d:
        return None
    h = hashlib.sha256()
    for rel in d["sources"]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != d["sources_sha256"]:
        return None
    return d["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# multi-rank bookkeeping (replicas: no collective on the data path)
# ---------------------------------------------------------------------------

def reduce_max(values, world: int, device="cpu"):
    """Element-wise max of per-rank timings over all ranks (every rank gets it)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def aggregate_gbs(bytes_per_rank: int, world: int, ms: float) -> float:
    """Whole-job GB/s: the bytes all ranks processed over the slowest rank's time."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# workloads and their bytes
# ---------------------------------------------------------------------------

def make_inputs(rank: int, small: bool = False):
    """Full workloads, or (small) the profiling case: 8192 tokens of the large
    gated workload (268 MB of x + gate), the q/kv workload, and the first two
    packed sequences of the static-head workload (more than L2 each)."""
    import synth
    W = synth.workloads(seed=rank)
    wl, wm, ws = W["gated_large"], W["qkv_mx"], W["static_head"]
    if small:
        wl = synth.GatedWorkload("gated_large_8192", 8192, wl.H, wl.D, wl.act, wl.eps,
                                 wl.outlier_p, wl.outlier_scale, wl.seed, wl.stream_base)
        ws = synth.StaticHeadWorkload("static_head_2seq", seed=ws.seed, stream_base=ws.stream_base,
                                      lengths=ws.lengths[:2])
    inp = {"A": {"x": wl.x(), "gate": wl.gate(), "w": wl.weight(), "w_": wl},
           "B": {"q": wm.q(), "kv": wm.kv(), "wq": wm.q_weight(), "wkv": wm.kv_weight(), "w_": wm}}
    xs = {k: ws.tensor(k) for k in ("q", "k", "v")}
    inp["C"] = {**xs, "d": ws.descales(xs), "cu": ws.cu_seqlens(), "w_": ws}
    return inp


def alg_bytes(inp) -> dict:
    return {"A": inp["A"]["w_"].algorithmic_bytes(), "B": inp["B"]["w_"].algorithmic_bytes(),
            "C": inp["C"]["w_"].algorithmic_bytes()}


def rows(inp) -> dict:
    return {"A": inp["A"]["w_"].T, "B": inp["B"]["w_"].M, "C": inp["C"]["w_"].T}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(inp, n_a, n_b, n_c, threads: int = 1):
    """Run the oracle on the first n tokens/rows of each workload, each
    operation timed on its own, on `threads` host threads (row slices of the
    same single-threaded function; 1 = as written).  Returns a dict with the
    seconds, rows and algorithmic bytes of each operation and in total."""
    import oracle as O
    a, b, c = inp["A"], inp["B"], inp["C"]
    wl, wm, ws = a["w_"], b["w_"], c["w_"]
    O.lib()

    def timed(fn, n):
        t0 = time.perf_counter()
        O.sliced(fn, n, threads=threads, min_slice=16)
        return time.perf_counter() - t0

    sec = {
        "A": timed(lambda i, j: O.gated_rmsnorm_quant_token(a["x"][i:j], a["gate"][i:j], a["w"],
                                                            wl.eps, wl.act), n_a),
        "B": timed(lambda i, j: O.rmsnorm_quant_mx(b["q"][i:j], b["wq"], b["kv"][i:j], b["wkv"],
                                                   wm.eps), n_b),
        "C": timed(lambda i, j: [O.static_head_quant(c[k][i:j], c["d"][k]) for k in ("q", "k", "v")],
                   n_c),
    }
    nrows = {"A": n_a, "B": n_b, "C": n_c}
    by = {"A": n_a * wl.H * wl.D * 5, "B": n_b * (wm.Nq * 3 + wm.Nq // 32 + wm.Nkv * 4),
          "C": n_c * ws.H * (2 * ws.Dqk + ws.Dv) * 3}
    ops = {k: {"rows": nrows[k], "seconds": sec[k], "rows_per_s": nrows[k] / sec[k],
               "GB_s": by[k] / sec[k] / 1e9} for k in sec}
    total_s = sum(sec.values())
    return {"threads": threads, "seconds": total_s, "bytes": sum(by.values()),
            "GB_s": sum(by.values()) / total_s / 1e9, "ops": ops,
            "sample": ("first %d tokens of (A) gated_large, %d rows of (B) qkv_mx, %d tokens of (C) "
                       "static_head" % (n_a, n_b, n_c))}


def cpu_baseline(inp) -> dict:
    """The oracle as it stands on the host cores: single-threaded (as written)
    and over row slices on every host thread, per operation in rows/s and
    GB/s (rows: tokens of (A) and (C), q/kv rows of (B))."""
    import oracle as O
    one = oracle_sample(inp, *CPU_SAMPLE, threads=1)
    allt = oracle_sample(inp, *CPU_SAMPLE, threads=O.host_threads())
    names = {"A": "gated_rmsnorm_quant_token", "B": "rmsnorm_quant_mx", "C": "static_head_quant"}
    return {"value": allt["GB_s"], "unit": UNIT, "cores": allt["threads"], "kind": "oracle",
            "sample": allt["sample"] + "; C oracle over row slices on every host thread "
                      "(single-threaded figures beside it)",
            "seconds": allt["seconds"],
            "single_thread": {"value": one["GB_s"], "unit": UNIT, "cores": 1,
                              "seconds": one["seconds"]},
            "per_op": {names[k]: {"rows_per_s_1_thread": one["ops"][k]["rows_per_s"],
                                  "rows_per_s_all_threads": allt["ops"][k]["rows_per_s"],
                                  "GB_s_1_thread": one["ops"][k]["GB_s"],
                                  "GB_s_all_threads": allt["ops"][k]["GB_s"]} for k in names}}


def reference_arm(args, rank: int, world: int) -> None:
    """The oracle as it stands, on the host cores, on a bounded sample of the
    same workload; rank 0 alone under torchrun."""
    if rank != 0:
        return
    import oracle as O
    inp = make_inputs(0)
    threads = O.host_threads()
    for _ in range(args.warmup):
        oracle_sample(inp, *REF_SAMPLE, threads=threads)
    dts, by, desc = [], 0, ""
    for _ in range(args.steps):
        r = oracle_sample(inp, *REF_SAMPLE, threads=threads)
        dts.append(r["seconds"])
        by, desc = r["bytes"], r["sample"] + ", the C oracle over row slices on %d host threads" % threads
    total = sum(dts)
    value = by * args.steps / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64+f32",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the fused operations against their unfused steps, and the dynamic per-head
# quantisation (reported beside the step, not part of it)
# ---------------------------------------------------------------------------

def side_measurements(dev, d16, inp_c) -> dict:
    """Median device time over 30 launches (L2 flushed before each) of: (A) at
    the gated_silu size fused and as gated norm -> bf16 -> per-token quant;
    (B) at the qkv_mx size fused and as RMSNorm -> bf16 -> MX quant plus the
    kv RMSNorm; the decode-sized (A) fused and as its two steps, replayed from
    CUDA graphs; the dynamic per-head quantisation of the static_head
    workload (max pass + quantise pass); the inverse-RoPE + MXFP8 producer of
    the o-projection input, fused and as its two steps."""
    import torch
    import synth
    import rmsnorm_fp8_activation_gb300 as B
    W = synth.workloads()
    ws, wm = W["gated_silu"], W["qkv_mx"]
    x, gt, w = d16(ws.x()), d16(ws.gate()), d16(ws.weight())
    q, kv, wq, wkv = d16(wm.q()), d16(wm.kv()), d16(wm.q_weight()), d16(wm.kv_weight())
    Q, K, V = d16(inp_c["q"]), d16(inp_c["k"]), d16(inp_c["v"])
    flush = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    fsum = torch.zeros((), dtype=torch.int64, device=dev)

    def timed(fn, n=30):
        fn()
        ts = []
        for _ in range(n):
            fsum.copy_(flush.view(torch.int64).sum())  # evicts L2 with clean lines
            # keep the GPU busy while the host enqueues the call, so that no host
            # time falls between the two events
            torch.cuda._sleep(200000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(1e3 * e0.elapsed_time(e1))
        return statistics.median(ts)

    a_fused = timed(lambda: B.fp8n_gated_rmsnorm_quant_token(x, gt, w, ws.eps, ws.act))
    a_unfused = timed(lambda: B.fp8n_quant_token(B.fp8n_gated_rmsnorm_bf16(x, gt, w, ws.eps, ws.act)))
    b_fused = timed(lambda: B.fp8n_rmsnorm_quant_mx(q, wq, kv, wkv, wm.eps))
    b_unfused = timed(lambda: (B.fp8n_quant_mx(B.fp8n_rmsnorm_bf16(q, wq, wm.eps)),
                               B.fp8n_rmsnorm_bf16(kv, wkv, wm.eps)))
    dyn = timed(lambda: B.fp8n_dynamic_head_quant(Q, K, V))
    # the o-projection input: inverse RoPE + MXFP8, fused and as its two steps
    wr = W["inv_rope_mx"]
    ro = d16(wr.o()).view(wr.T, wr.H, wr.D)
    rp = torch.from_numpy(wr.positions()).to(dev)
    rc = torch.from_numpy(wr.cos_sin()).to(dev)
    rope_fused = timed(lambda: B.fp8n_inv_rope_quant_mx(ro, rp, rc, wr.rope_off, wr.rope_dim))
    rope_unfused = timed(lambda: B.fp8n_quant_mx(
        B.fp8n_inv_rope_bf16(ro, rp, rc, wr.rope_off, wr.rope_dim)))

    # decode-sized (A) (56 tokens x 12 heads x 128), one call replayed from a
    # CUDA graph, inputs resident (as in a decode loop): device time per call
    wd = W["gated_small"]
    xd, gd, wtd = d16(wd.x()), d16(wd.gate()), d16(wd.weight())
    od = torch.empty((wd.T, wd.H * wd.D), dtype=torch.uint8, device=dev)
    sd = torch.empty((wd.T,), dtype=torch.float32, device=dev)
    yd = torch.empty((wd.T, wd.H * wd.D), dtype=torch.bfloat16, device=dev)
    cs = torch.cuda.Stream(device=dev)

    def fused_call():
        B.fp8n_gated_rmsnorm_quant_token(xd, gd, wtd, wd.eps, wd.act, out=od, scale=sd)

    def unfused_call():  # the same result through the two steps
        B.fp8n_gated_rmsnorm_bf16(xd, gd, wtd, wd.eps, wd.act, y=yd)
        B.fp8n_quant_token(yd, out=od, scale=sd)

    def graph_us(fn, per_graph: int, replays: int) -> float:
        """Device time per fn() captured per_graph times in one CUDA graph."""
        with torch.cuda.stream(cs):
            for _ in range(3):
                fn()
        cs.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for _ in range(per_graph):
                fn()
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(replays):
            g.replay()
        g1.record()
        torch.cuda.synchronize()
        return 1e3 * g0.elapsed_time(g1) / (replays * per_graph)

    small_us = graph_us(fused_call, 1, 200)
    # the same call as one node among 20 in a graph (as in a decode step's
    # graph): the graph's own launch is spread over its nodes
    nodes = 20
    small_node_us = graph_us(fused_call, nodes, 20)
    small_unfused_us = graph_us(unfused_call, 1, 200)
    small_unfused_node_us = graph_us(unfused_call, nodes, 20)
    # a plain device copy of as many bytes as the q/kv producer moves (27.5 MB
    # read, 27.5 MB written): what one stream of this size takes here
    cp_src = torch.empty(wm.algorithmic_bytes() // 4, dtype=torch.int16, device=dev)
    cp_dst = torch.empty_like(cp_src)
    copy_us = timed(lambda: cp_dst.copy_(cp_src))
    n_c = Q.numel() + K.numel() + V.numel()
    return {
        "gated_silu_fused_us": a_fused, "gated_silu_unfused_us": a_unfused,
        "gated_silu_unfused_steps": "fp8n_gated_rmsnorm_bf16 -> fp8n_quant_token",
        "qkv_mx_fused_us": b_fused, "qkv_mx_unfused_us": b_unfused,
        "qkv_mx_unfused_steps": "fp8n_rmsnorm_bf16(q) -> fp8n_quant_mx; fp8n_rmsnorm_bf16(kv)",
        "gated_small_graph_us": small_us,
        "gated_small_graph_note": "56 x 12 x 128 sigmoid, one call per graph replay, inputs resident",
        "gated_small_graph_node_us": small_node_us,
        "gated_small_graph_node_note": "the same call as one of 20 nodes of a graph (per node)",
        "gated_small_unfused_graph_us": small_unfused_us,
        "gated_small_unfused_graph_node_us": small_unfused_node_us,
        "gated_small_unfused_note": "the same result as fp8n_gated_rmsnorm_bf16 -> "
                                    "fp8n_quant_token: per replay of the two calls, and per "
                                    "pair as 20 pairs of nodes of one graph",
        "copy_55MB_us": copy_us,
        "copy_55MB_note": "torch device copy of the q/kv producer's algorithmic bytes (half read, "
                          "half written): a plain stream of this size, for context",
        "dynamic_head_quant_us": dyn,
        "dynamic_head_quant_GB_s": 5 * n_c / (dyn * 1e-6) / 1e9,
        "dynamic_head_quant_bytes": "2 B/element read twice, 1 B/element written",
        "inv_rope_mx_fused_us": rope_fused, "inv_rope_mx_unfused_us": rope_unfused,
        "inv_rope_mx_GB_s": wr.algorithmic_bytes() / (rope_fused * 1e-6) / 1e9,
        "inv_rope_mx_frac_of_peak": wr.algorithmic_bytes() / (rope_fused * 1e-6) / 1e9
        / peaks()["hbm_gbs"],
        "inv_rope_mx_workload": "o [4096,16,576] bf16, rope on the last 64 dims (rotate-half), "
                                "positions in [0,4096), fp32 cos/sin cache [4096,64]",
        "inv_rope_mx_unfused_steps": "fp8n_inv_rope_bf16 -> fp8n_quant_mx",
        "l2": "evicted before each launch by reading 256 MB (clean lines: no write-back "
              "inside the timed launch)",
    }


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def ours(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    import torch.distributed as dist

    import rmsnorm_fp8_activation_gb300 as B
    from rmsnorm_fp8_activation_gb300 import build as _build

    _build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    inp = make_inputs(rank, small=args.small)
    nbytes = alg_bytes(inp)
    nrows = rows(inp)

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    A, Bm, C = inp["A"], inp["B"], inp["C"]
    wl, wm, ws = A["w_"], Bm["w_"], C["w_"]
    g = {"x": d16(A["x"]), "gate": d16(A["gate"]), "w": d16(A["w"]),
         "q": d16(Bm["q"]), "kv": d16(Bm["kv"]), "wq": d16(Bm["wq"]), "wkv": d16(Bm["wkv"]),
         "Q": d16(C["q"]), "K": d16(C["k"]), "V": d16(C["v"]),
         "dq": torch.from_numpy(C["d"]["q"]).to(dev), "dk": torch.from_numpy(C["d"]["k"]).to(dev),
         "dv": torch.from_numpy(C["d"]["v"]).to(dev), "cu": torch.from_numpy(C["cu"]).to(dev)}
    o = {"a": torch.empty((wl.T, wl.H * wl.D), dtype=torch.uint8, device=dev),
         "as": torch.empty((wl.T,), dtype=torch.float32, device=dev),
         "bq": torch.empty((wm.M, wm.Nq), dtype=torch.uint8, device=dev),
         "bs": torch.empty((wm.M, wm.Nq // 32), dtype=torch.uint8, device=dev),
         "bk": torch.empty((wm.M, wm.Nkv), dtype=torch.bfloat16, device=dev),
         "cq": torch.empty(C["q"].shape, dtype=torch.uint8, device=dev),
         "ck": torch.empty(C["k"].shape, dtype=torch.uint8, device=dev),
         "cv": torch.empty(C["v"].shape, dtype=torch.uint8, device=dev)}
    stream = torch.cuda.Stream(device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def run_step(gi, oi, s, ev=None):
        if ev:
            ev[0].record(s)
        B.fp8n_rmsnorm_quant_mx(gi["q"], gi["wq"], gi["kv"], gi["wkv"], wm.eps, q_out=oi["bq"],
                                q_scale=oi["bs"], kv_out=oi["bk"], status=status, stream=s)
        if ev:
            ev[1].record(s)
        B.fp8n_static_head_quant(gi["Q"], gi["K"], gi["V"], gi["dq"], gi["dk"], gi["dv"],
                                 cu_seqlens=gi["cu"], q_out=oi["cq"], k_out=oi["ck"],
                                 v_out=oi["cv"], status=status, stream=s)
        if ev:
            ev[2].record(s)
        B.fp8n_gated_rmsnorm_quant_token(gi["x"], gi["gate"], gi["w"], wl.eps, wl.act,
                                         out=oi["a"], scale=oi["as"], status=status, stream=s)
        if ev:
            ev[3].record(s)

    def step(ev=None):
        run_step(g, o, stream, ev)

    def barrier():
        if world > 1:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            step(evs[k])
    t_end.record(stream)
    stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    per = {"B": [], "C": [], "A": []}
    for e in evs:
        per["B"].append(e[0].elapsed_time(e[1]))
        per["C"].append(e[1].elapsed_time(e[2]))
        per["A"].append(e[2].elapsed_time(e[3]))
    if args.small:  # profiling case: kernel times only, no bench line
        if rank == 0:
            print(json.dumps({"small": True, "ms_per_step": total_ms / args.steps,
                              "avg_us": {k: 1e3 * statistics.mean(v) for k, v in per.items()},
                              "alg_bytes": nbytes}), flush=True)
        return

    # end to end through the public API with host buffers: every step copies
    # its inputs in from pinned host memory, runs the three calls and copies
    # the outputs back.  Two device buffer sets and three streams (copies in,
    # compute, copies out) let step k's copies in overlap step k-1's compute
    # and copies out; events order each buffer's reuse.
    h_in = {k: v.cpu().pin_memory() for k, v in g.items()}
    h_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in o.items()}
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    bufs = [(g, o), ({k: torch.empty_like(v) for k, v in g.items()},
                     {k: torch.empty_like(v) for k, v in o.items()})]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in bufs]
    ev_comp = [torch.cuda.Event() for _ in bufs]
    ev_out = [torch.cuda.Event() for _ in bufs]

    def e2e_run(n):
        for k in range(n):
            b = k % 2
            gi, oi = bufs[b]
            if k >= 2:
                s_in.wait_event(ev_comp[b])   # step k-2 has read these inputs
            with torch.cuda.stream(s_in):
                for key in gi:
                    gi[key].copy_(h_in[key], non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_out[b])  # step k-2's outputs have left
            run_step(gi, oi, stream)
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for key in oi:
                    h_out[key].copy_(oi[key], non_blocking=True)
            ev_out[b].record(s_out)

    e2e_steps = max(3, min(args.steps, 10))
    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    e2e_run(e2e_steps)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    step_ms, e2e_ms = reduce_max([total_ms / args.steps, e2e_ms], world, dev)
    if rank != 0:
        return

    total_bytes = sum(nbytes.values())
    value = aggregate_gbs(total_bytes, world, step_ms)
    pk = peaks()
    kernels = {}
    names = {"A": "gated_rmsnorm_quant_token", "B": "rmsnorm_quant_mx", "C": "static_head_quant"}
    for k in ("A", "B", "C"):
        avg_ms = statistics.mean(per[k])
        gbs = nbytes[k] / (avg_ms * 1e-3) / 1e9
        kernels[names[k]] = {"avg_us": 1e3 * avg_ms, "median_us": 1e3 * statistics.median(per[k]),
                             "alg_bytes": nbytes[k], "GB_s": gbs,
                             "frac_of_peak": gbs / pk["hbm_gbs"],
                             "frac_of_nominal": gbs / NOMINAL_HBM_GBS,
                             "rows_per_s": nrows[k] / (avg_ms * 1e-3)}
    dom = max(kernels, key=lambda n: kernels[n]["avg_us"])
    dom_key = {v: k for k, v in names.items()}[dom]
    dom_ms = statistics.mean(per[dom_key])
    ach = nbytes[dom_key] / (dom_ms * 1e-3) / 1e9

    side = side_measurements(dev, d16, inp["C"]) if world == 1 else None
    cpu = cpu_baseline(inp)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16->e4m3 (f32 arithmetic)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "per_gpu_alg_bytes_per_step": total_bytes,
                       "l2": L2_NOTE, "parallelism": "replicas" if world > 1 else "1 GPU"},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
                         "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                         "frac_of_nominal": ach / NOMINAL_HBM_GBS,
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "traffic": profiled_traffic(dom)},
            "kernels": kernels,
            "status_word": int(status.item()),
            "cpu_baseline": cpu,
            "e2e": {"value": aggregate_gbs(total_bytes, world, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms},
            # one kernel per operation and step in the timed region
            "gpu_launches": 3 * args.steps,
            "clocks": clk}
    if side is not None:
        line["unfused_and_dynamic"] = side
    print(json.dumps(line), flush=True)


def profile_case(args) -> None:
    """One call repeated (for a profiler): the inverse-RoPE producer on the
    o-projection workload; the decode-sized gated call; the dynamic per-head
    quantisation of the first two packed sequences of the static-head workload
    (its max pass and its quantise pass); or the gated workload with silu as
    its two unfused steps (gated norm to bf16, then per-token quantisation)."""
    import torch
    import synth
    import rmsnorm_fp8_activation_gb300 as B
    from rmsnorm_fp8_activation_gb300 import build as _build
    _build.build()
    W = synth.workloads()
    d16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    if args.case == "inv_rope":
        w = W["inv_rope_mx"]
        o = d16(w.o()).view(w.T, w.H, w.D)
        pos, cs = torch.from_numpy(w.positions()).cuda(), torch.from_numpy(w.cos_sin()).cuda()
        fn = lambda: B.fp8n_inv_rope_quant_mx(o, pos, cs, w.rope_off, w.rope_dim)
    elif args.case == "dynamic":
        sw = W["static_head"]
        ws = synth.StaticHeadWorkload("static_head_2seq", seed=sw.seed, stream_base=sw.stream_base,
                                      lengths=sw.lengths[:2])
        Q, K, V = (d16(ws.tensor(k)) for k in ("q", "k", "v"))
        fn = lambda: B.fp8n_dynamic_head_quant(Q, K, V)
    elif args.case == "unfused":
        w = W["gated_silu"]
        x, g, wt = d16(w.x()), d16(w.gate()), d16(w.weight())
        fn = lambda: B.fp8n_quant_token(B.fp8n_gated_rmsnorm_bf16(x, g, wt, w.eps, w.act))
    else:
        w = W["gated_small"]
        x, g, wt = d16(w.x()), d16(w.gate()), d16(w.weight())
        fn = lambda: B.fp8n_gated_rmsnorm_quant_token(x, g, wt, w.eps, w.act)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"case": args.case, "calls": args.warmup + args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--small", action="store_true",
                    help="profiling case (see make_inputs); prints kernel times only")
    ap.add_argument("--case", choices=["inv_rope", "decode", "dynamic", "unfused"], default=None,
                    help="profiling case: only the inverse-RoPE producer on its workload, the "
                         "decode-sized gated call, the dynamic per-head quantisation, or the "
                         "unfused gated steps, --steps times back to back")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.case is not None:
        profile_case(args)
    elif args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        ours(args, rank, world, local_rank)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
