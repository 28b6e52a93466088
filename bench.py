#!/usr/bin/env python
"""Benchmark of one sparse-decode step (SCORE -> TOPK -> GATHER-ATT) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (default): the long-context stress configuration -- one sequence of
n = 1,048,576 cached tokens, 32 query heads on 8 KV heads, d = 128, bf16 K/V
resident in HBM; Fathom bit-plane scan at a 56-bit water-filled budget, exact
top-512 per KV head, gather-attend over the 512 selected rows.  A step is one
layer's whole hot path for all heads: read plan -> bit-plane scan -> top-k ->
gather-attend (the KV-write-path index build is done once, untimed).

Timing: W untimed warm-up steps, then exactly K steps, each timed with CUDA
events on the launching stream; L2 (129 MB) is flushed before every timed step
by writing a 256 MB buffer and then reading another 256 MB buffer (L2 then holds
clean lines of unrelated data), outside the events.  `value` = keys scored per
second = (B * Hkv * n) / step time, summed over ranks (independent replicas,
weak scaling).  One JSON line is printed by rank 0.

--impl reference times the CPU oracle on the host cores on a bounded sample
of the same workload per step (one KV head x 262,144 tokens).
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

import numpy as np  # noqa: E402

METRIC = "keys scored/s (sparse-decode step, 1M-token context)"
UNIT = "keys/s"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)  # ~1 s timed: clocks sampled within
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-variants", action="store_true", help="skip the other scorers")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--n", type=int, default=0, help="override n (testing only)")
    return p.parse_args()


# ------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(nm)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dev_tensor(x, torch):
    x = np.ascontiguousarray(x)
    v = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}.get(x.dtype, x.dtype)
    return torch.from_numpy(x.view(v)).cuda()


# ------------------------------------------------------------------------------------
class L2Flush:
    """Before every timed step: write a 256 MB buffer (larger than the 129 MB L2),
    then read another 256 MB buffer, so that the step finds L2 holding clean lines
    of unrelated data (none of its inputs, and no dirty lines of the flush left for
    the step to write back)."""

    def __init__(self, torch):
        self.a = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.b = torch.zeros(64 << 20, dtype=torch.int32, device="cuda")
        self.sink = torch.empty((), dtype=torch.int32, device="cuda")

    def zero_(self):
        self.a.zero_()
        self.sink.copy_(self.b.max())


def timed_steps(torch, fn, steps, warmup, flush_buf, ws=1):
    """Runs fn() warmup + steps times; returns per-step device ms of the timed ones.
    The L2 flush before each step sits outside the events."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush_buf.zero_()
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(steps):
        flush_buf.zero_()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    return [a.elapsed_time(b) for a, b in ev]


def capture_graph(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def launches_per_step(step, q) -> int:
    """Kernels of libsd one eager step launches, counted by the library itself
    (a graph replay of the step launches the same kernels)."""
    import torch
    import top_sparse_decode_gb300 as sd
    torch.cuda.synchronize()
    before = sd.sd_launch_count()
    step.run(q)
    torch.cuda.synchronize()
    return sd.sd_launch_count() - before


def scan_traffic(workload: str):
    """DRAM bytes per launch of the scan kernel from the committed ncu summary,
    or None when the kernel source changed since that capture."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "score_planes_tma_scan56-1m.md")
    csrc = os.path.join(ROOT, "top_sparse_decode_gb300", "csrc")
    src, hdr = os.path.join(csrc, "sd_scan_tma.cu"), os.path.join(csrc, "sd_planes.cuh")
    if not all(os.path.exists(p) for p in (prof, src, hdr)):
        return None
    text = open(prof).read()
    code = open(src).read()
    i, j = code.find("namespace sd {"), code.find("int launch_score_planes_tma(")
    if i < 0 or j < i:
        return None
    # the scan's device code: its own source and the plan and table helpers it includes
    sha = hashlib.sha256((code[i:j] + open(hdr).read()).encode()).hexdigest()
    if sha not in text:
        return None
    for line in text.splitlines():
        if line.startswith(f"traffic_bytes_per_launch[{workload}]"):
            return int(line.split("=")[1].split()[0])
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------------------------
def oracle_sample(inp, heads, n_tok, build=True):
    """Oracle inputs for a sample of the step: the first `heads` KV heads of
    sequence 0 over the first n_tok tokens, with its planes (KV-write path)."""
    import oracle
    G = inp.cfg.G
    qh = np.ascontiguousarray(inp.q[:1, : heads * G])
    Kh = np.ascontiguousarray(inp.K[:1, :heads, :n_tok])
    Vh = np.ascontiguousarray(inp.V[:1, :heads, :n_tok])
    s2 = np.ascontiguousarray(inp.sigma2[:heads])
    smp = dict(q=qh, K=Kh, V=Vh, s2=s2, heads=heads, n=n_tok)
    if build:
        t0 = time.perf_counter()
        smp["planes"], smp["scales"] = oracle.plane_build(Kh)
        smp["build_s"] = time.perf_counter() - t0
    return smp


def oracle_step(smp, k, d=128, stages=None):
    """The oracle, as it stands: plan -> bit-plane score -> top-k -> gather-attend.
    Returns seconds; with a dict `stages`, adds each stage's seconds to it."""
    import oracle
    h = smp["heads"]
    t = [time.perf_counter()]
    plan = oracle.plan(smp["q"], smp["s2"], h, oracle.PLAN_WATERFILL, 56)
    t.append(time.perf_counter())
    sc = oracle.plane_score(smp["planes"], smp["scales"], plan, smp["q"])
    t.append(time.perf_counter())
    idx, cnt = oracle.topk(sc.reshape(h, -1), k, 0, 0)
    t.append(time.perf_counter())
    oracle.gather_attend(smp["q"], smp["K"], smp["V"], idx.reshape(1, h, -1),
                         cnt.reshape(1, h), 1 / math.sqrt(d))
    t.append(time.perf_counter())
    if stages is not None:
        for nm, a, b in zip(("plan", "score", "topk", "gather_attend"), t[:-1], t[1:]):
            stages[nm] = stages.get(nm, 0.0) + (b - a)
    return t[-1] - t[0]


def cpu_model() -> str:
    """The host CPU's model string (lscpu, else /proc/cpuinfo, else the machine)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(inp, cfg, heads=None):
    """CPU baseline leg: the oracle, as it stands, on the host cores.
    Multi-thread: the whole 1M-token step (every KV head), per stage, with the
    KV-write-path index build timed apart.  Single-thread: one KV head over the
    first 262,144 tokens, per stage (about 1/32 of the step's work)."""
    import oracle
    heads = heads or cfg.Hkv
    cores = oracle.threads()
    st_mt = {}
    smp = oracle_sample(inp, heads, cfg.n)
    dt = oracle_step(smp, cfg.k, cfg.d, st_mt)
    n1 = min(cfg.n, 1 << 18)
    prev = oracle.set_threads(1)
    try:
        st_1 = {}
        smp1 = oracle_sample(inp, 1, n1)
        dt1 = oracle_step(smp1, cfg.k, cfg.d, st_1)
    finally:
        oracle.set_threads(prev)
    return {"value": heads * cfg.n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{heads} of {cfg.Hkv} KV heads x {cfg.n} tokens of the step (plan, "
                      f"bit-plane score, top-{cfg.k}, gather-attend) in {dt:.2f} s on "
                      f"{cores} threads",
            "stages_s": {k2: round(v, 4) for k2, v in st_mt.items()},
            "index_build_s": round(smp["build_s"], 4),
            "single_thread": {"value": n1 / dt1, "unit": UNIT, "cores": 1,
                              "sample": f"1 KV head x {n1} tokens of the step in {dt1:.2f} s",
                              "stages_s": {k2: round(v, 4) for k2, v in st_1.items()},
                              "index_build_s": round(smp1["build_s"], 4)}}


def run_reference(args, ws, rank):
    """Reference arm: the CPU oracle on the same workload; each step is a bounded
    sample (1 KV head x 262,144 tokens) so that K steps take well under a minute
    or two on the host cores."""
    if rank != 0:
        return
    import oracle
    import synth
    n = args.n or (1 << 20)
    cfg = synth.config(4, n=n)
    cfg_s = synth.config(4, B=1, Hkv=1, Hq=cfg.G, n=n)
    inp = synth.make_inputs(cfg_s)
    n_tok = min(n, 1 << 18)
    smp = oracle_sample(inp, 1, n_tok)
    for _ in range(args.warmup):
        oracle_step(smp, cfg.k, cfg.d)
    times = [oracle_step(smp, cfg.k, cfg.d) for _ in range(args.steps)]
    t = statistics.mean(times)
    v = n_tok / t
    sample = (f"1 of {cfg.Hkv} KV heads x {n_tok} of {n} tokens per step (plan, bit-plane "
              f"score, top-{cfg.k}, gather-attend)")
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": f"longctx-1m: B=1, Hq=32, Hkv=8, d=128, n={n}; 56-bit "
                                   f"water-filled bit-plane scan, top-{cfg.k}, gather-attend "
                                   f"(oracle on a per-step sample)", "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------
def other_configs(torch, sd, rl, synth, flush, K_st, peak_gbs):
    """The other 128k-1M-class workloads, each as one decode step (CUDA-graph replay,
    L2 flushed before every step): the batched 128k-token bit-plane step at budgets
    47, 56 and 92 bits and reading all planes, the batch-64 Quest block step, and the
    HashAttention 32k-token step with 2-layer-MLP signatures."""
    from top_sparse_decode_gb300.pipeline import DecodeStep, StepConfig, build_index
    out = {}

    def graph_us(fn):
        g = capture_graph(torch, fn)
        return statistics.mean(timed_steps(torch, g.replay, K_st, 3, flush)) * 1e3

    # Fathom, batch 4 x 131072 tokens
    c2 = synth.config(2)
    inp = synth.make_inputs(c2)
    q, K, V = dev_tensor(inp.q, torch), dev_tensor(inp.K, torch), dev_tensor(inp.V, torch)
    s2 = dev_tensor(inp.sigma2, torch)
    keys = c2.B * c2.Hkv * c2.n
    res = {}
    index = None
    for name, mode, budget in [("47", sd.SD_PLAN_WATERFILL, 47), ("56", sd.SD_PLAN_WATERFILL, 56),
                               ("92", sd.SD_PLAN_WATERFILL, 92), ("full", sd.SD_PLAN_FULL, 0)]:
        sc = StepConfig(sd.SD_IDX_PLANES, c2.B, c2.Hq, c2.Hkv, c2.n, k=c2.k, plan_mode=mode,
                        budget=budget)
        if index is None:
            index = build_index(sc, K)
        st = DecodeStep(sc, K, V, index, sigma2=s2)
        st.run(q)
        torch.cuda.synchronize()
        t_step = graph_us(lambda: st.run(q))
        t_scan = graph_us(lambda: st.stage_plan_score(q))
        plan_np = st.plan.cpu().numpy()
        sb = rl.plane_scan_bytes(plan_np, c2.n)
        res[name] = {"us_per_step": t_step, "keys_per_s": keys / (t_step * 1e-6),
                     "plan_scan_us": t_scan, "bits_per_token": rl.plane_scan_bits_per_token(plan_np),
                     "scan_bytes": sb, "scan_GBps": sb / (t_scan * 1e-6) / 1e9,
                     "scan_frac_hbm": sb / (t_scan * 1e-6) / 1e9 / peak_gbs,
                     "token_planes_per_s": rl.plane_scan_alu_ops(plan_np, c2.n) / (t_scan * 1e-6)}
        del st
    out["fathom-128k (B=4, n=131072, k=512)"] = res
    del q, K, V, s2, index, inp

    # Quest, batch 64 x 16384 tokens, top-128 blocks + 1 local block
    c3 = synth.config(3)
    inp = synth.make_inputs(c3)
    q, K, V = dev_tensor(inp.q, torch), dev_tensor(inp.K, torch), dev_tensor(inp.V, torch)
    sc = StepConfig(sd.SD_IDX_MINMAX, c3.B, c3.Hq, c3.Hkv, c3.n, k=c3.blk_k, local=c3.blk_local)
    index = build_index(sc, K)
    st = DecodeStep(sc, K, V, index)
    st.run(q)
    torch.cuda.synchronize()
    t_step = graph_us(lambda: st.run(q))
    t_scan = graph_us(lambda: st.stage_score(q))
    t_topk = graph_us(lambda: st.stage_topk())
    t_att = graph_us(lambda: st.stage_attend(q))
    sb = rl.quest_scan_bytes(c3.B, c3.Hkv, c3.n)
    gb = rl.gather_bytes(st.count.cpu().numpy())
    keys = c3.B * c3.Hkv * c3.n
    out["quest-b64-16k (B=64, n=16384, 128+1 blocks)"] = {
        "us_per_step": t_step, "keys_per_s": keys / (t_step * 1e-6),
        "scan_us": t_scan, "scan_bytes": sb, "scan_GBps": sb / (t_scan * 1e-6) / 1e9,
        "scan_frac_hbm": sb / (t_scan * 1e-6) / 1e9 / peak_gbs,
        "topk_us": t_topk, "attend_us": t_att, "gather_bytes": gb,
        "attend_GBps": gb / (t_att * 1e-6) / 1e9,
        "attend_frac_hbm": gb / (t_att * 1e-6) / 1e9 / peak_gbs}

    # OasisKV's resident set on the same step: 129 slots of 16 tokens per KV head, at
    # most C = 7 admissions per head and step (fetch ratio 0.05 of K = 128), full K/V
    # in pinned host memory; two queries alternate so that every step has misses
    R, C, rows3 = 129, 7, c3.B * c3.Hkv
    preds = []
    for qq in (q, torch.roll(q, 1, dims=2)):
        st.stage_score(qq)
        st.stage_topk()
        preds.append((st.scores.clone(), st.idx.clone(), st.count.clone()))
    Kh, Vh = K.cpu().pin_memory(), V.cpu().pin_memory()
    res = sd.Resident(rows3, R, sc.n_units)
    Kp = torch.zeros((c3.B, c3.Hkv, R * 16, 128), dtype=torch.bfloat16, device="cuda")
    Vp = torch.zeros_like(Kp)
    plan = [torch.empty((rows3, C), dtype=torch.int32, device="cuda") for _ in range(3)]
    pcnt = torch.empty(rows3, dtype=torch.int32, device="cuda")
    pool = torch.empty((rows3, sc.max_count), dtype=torch.int32, device="cuda")
    pool_cnt = torch.empty(rows3, dtype=torch.int32, device="cuda")
    shp3 = sd.make_shape(c3.B, c3.Hq, c3.Hkv, c3.n)
    counter = [0]

    def select():
        s3, i3, n3 = preds[counter[0] % 2]
        sd.sd_delta_select(shp3, st.sel, s3, i3, sc.max_count, n3, C, counter[0], res, *plan,
                           pcnt, pool, sc.max_count, pool_cnt)
        counter[0] += 1

    def transfer():
        sd.sd_resident_gather(shp3, 16, Kh, Vh, plan[0], plan[1], pcnt, C, R, Kp, Vp)

    for _ in range(4):  # fill the set
        select()
        transfer()
    t_sel = statistics.mean(timed_steps(torch, select, K_st, 3, flush)) * 1e3

    def both():
        select()
        transfer()
    t_both = statistics.mean(timed_steps(torch, both, K_st, 3, flush)) * 1e3
    select()
    torch.cuda.synchronize()
    admitted = int(pcnt.clamp(min=0).sum().item())
    xfer = rl.resident_transfer_bytes(admitted)  # K and V rows of the admitted blocks
    out["quest-b64-16k (B=64, n=16384, 128+1 blocks)"]["resident_129x16_C7"] = {
        "delta_select_us": t_sel, "select_and_transfer_us": t_both,
        "admitted_blocks_per_step": admitted, "transfer_bytes_per_step": xfer,
        "host_link_GBps": xfer / ((t_both - t_sel) * 1e-6) / 1e9 if t_both > t_sel else None}
    del Kh, Vh, Kp, Vp, preds, res
    del st, index, q, K, V, inp

    # HashAttention, 32768 tokens, 2-layer-MLP signatures, 128 + 512 window tokens
    c1 = synth.config(1)
    inp = synth.make_inputs(c1)
    q, K, V = dev_tensor(inp.q, torch), dev_tensor(inp.K, torch), dev_tensor(inp.V, torch)
    enc = sd.make_encoder(dev_tensor(inp.W1, torch), dev_tensor(inp.b1, torch),
                          dev_tensor(inp.W2, torch), dev_tensor(inp.b2, torch))
    sc = StepConfig(sd.SD_IDX_SIG, c1.B, c1.Hq, c1.Hkv, c1.n, k=c1.k, sink=c1.sink,
                    local=c1.local)
    index = build_index(sc, K, enc)
    st = DecodeStep(sc, K, V, index, enc=enc)
    st.run(q)
    torch.cuda.synchronize()
    t_step = graph_us(lambda: st.run(q))
    keys = c1.B * c1.Hkv * c1.n
    out["hash-32k (B=1, n=32768, MLP signatures)"] = {
        "us_per_step": t_step, "keys_per_s": keys / (t_step * 1e-6),
        "gather_bytes": rl.gather_bytes(st.count.cpu().numpy())}
    del st, index, q, K, V, inp
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    import torch

    import synth
    import top_sparse_decode_gb300 as sd
    from top_sparse_decode_gb300 import build as sdbuild
    from top_sparse_decode_gb300 import roofline as rl
    from top_sparse_decode_gb300.pipeline import DecodeStep, StepConfig, build_index

    if rank == 0:
        sdbuild.build()
    barrier(ws)
    torch.cuda.set_device(local)
    sd.lib()
    cfg = synth.config(4) if not args.n else synth.config(4, n=args.n)
    t_gen = time.perf_counter()
    inp = synth.make_inputs(cfg)
    log(f"[bench] inputs generated in {time.perf_counter() - t_gen:.1f} s")
    q = dev_tensor(inp.q, torch)
    K = dev_tensor(inp.K, torch)
    V = dev_tensor(inp.V, torch)
    sigma2 = dev_tensor(inp.sigma2, torch)
    flush = L2Flush(torch)
    B, Hq, Hkv, n = cfg.B, cfg.Hq, cfg.Hkv, cfg.n
    keys = B * Hkv * n

    # headline step: 56-bit water-filled bit-plane scan
    sc = StepConfig(sd.SD_IDX_PLANES, B, Hq, Hkv, n, k=cfg.k, plan_mode=sd.SD_PLAN_WATERFILL,
                    budget=56)
    index = build_index(sc, K)
    step = DecodeStep(sc, K, V, index, sigma2=sigma2)
    step.run(q)
    torch.cuda.synchronize()
    plan_np = step.plan.cpu().numpy()
    counts_np = step.count.cpu().numpy()
    scan_bytes = rl.plane_scan_bytes(plan_np, n)
    gath_bytes = rl.gather_bytes(counts_np)
    alg_bytes = scan_bytes + gath_bytes

    # graph-captured step (falls back to eager if capture is refused)
    try:
        graph = capture_graph(torch, lambda: step.run(q))
        run = graph.replay
        mode = "cuda-graph"
    except Exception as e:  # noqa: BLE001
        log(f"[bench] graph capture failed ({e}); timing eager launches")
        run = lambda: step.run(q)  # noqa: E731
        mode = "eager"

    clocks = ClockSampler(local)
    clocks.start()
    times = timed_steps(torch, run, args.steps, args.warmup, flush, ws)
    ck = clocks.stop()
    sd.sd_device_status()  # raises if a bounded wait inside a kernel ran out
    t_step = statistics.mean(times)
    t_step_max = max_over_ranks(t_step, ws)
    value = keys * ws / (t_step_max * 1e-3)

    # per-stage and dominant-kernel timings (eager, each stage alone, cold L2)
    K_st = max(10, min(args.steps, 100))
    st_prep = statistics.mean(timed_steps(torch, lambda: step.stage_prep(q), K_st, 3, flush))
    st_score = statistics.mean(timed_steps(torch, lambda: step.stage_score(q), K_st, 3, flush))
    # the plan-in-scan call writes the word maxima the step's top-k reads
    st_plan_scan = statistics.mean(timed_steps(torch, lambda: step.stage_plan_score(q), K_st, 3,
                                               flush))
    st_topk = statistics.mean(timed_steps(torch, lambda: step.stage_topk(), K_st, 3, flush))
    st_att = statistics.mean(timed_steps(torch, lambda: step.stage_attend(q), K_st, 3, flush))
    st_sa = (statistics.mean(timed_steps(torch, lambda: step.stage_select_attend(q), K_st, 3, flush))
             if step.use_sa else None)
    st_fused = (statistics.mean(timed_steps(torch, lambda: step.stage_score_topk(q), K_st, 3,
                                            flush)) if step.fused else None)
    eager = statistics.mean(timed_steps(torch, lambda: step.run(q), K_st, 3, flush))

    # marginal stage costs inside the step: cumulative prefixes, L2 flushed before each
    stages = step.stages()

    def upto(nst):
        def f():
            for _, fn in stages[:nst]:
                fn(q)
        return f

    cum = [statistics.mean(timed_steps(torch, upto(i), K_st, 3, flush))
           for i in range(1, len(stages) + 1)]
    marginal = {name: (cum[i] - (cum[i - 1] if i else 0.0)) * 1e3
                for i, (name, _) in enumerate(stages)}
    peak_gbs, peak_kind = peaks()
    scan_gbs = scan_bytes / (st_score * 1e-3) / 1e9
    alu_ops = rl.plane_scan_alu_ops(plan_np, n)

    # e2e: pinned host q in, result out, through the public API, each step
    q_host = torch.from_numpy(inp.q.view(np.int16)).pin_memory()
    res_host = torch.empty(step.result.shape, dtype=torch.float32).pin_memory()
    out_host = res_host[:step.out.numel()].view(step.out.shape)
    lse_host = res_host[step.out.numel():].view(step.lse.shape)
    q_dev = torch.empty_like(q)

    def e2e_step():
        sd.sd_copy(q_dev, q_host)          # q from pinned host memory
        step.run(q_dev)
        sd.sd_copy(res_host, step.result)  # out and lse back, one copy

    # one CUDA graph per step: the H2D copy of q, the step's kernels and the D2H
    # copy of out and lse (copy kernels over the pinned buffers' device mapping;
    # the copies run every replay)
    g_e2e = capture_graph(torch, e2e_step)
    e2e_t = statistics.mean(timed_steps(torch, g_e2e.replay, max(args.steps // 2, 10), 3, flush))
    e2e_val = keys * ws / (max_over_ranks(e2e_t, ws) * 1e-3)
    torch.cuda.synchronize()
    assert np.array_equal(out_host.numpy(), step.out.cpu().numpy())

    variants = {}
    if not args.no_variants:
        # full-depth channel subsets on the same planes: the 32 channels of largest
        # variance (the 136-bit class) and the 16 of largest query mass (SparQ r = 16,
        # 68 bits: 4 plane bits and a quarter bit of fp16 scale per channel and token)
        for vname, vmode, vbudget in [("fixed32x4", sd.SD_PLAN_FIXED, 32),
                                      ("topq16x4", sd.SD_PLAN_TOPQ, 16),
                                      ("split56", sd.SD_PLAN_SPLIT, 56)]:
            scf = StepConfig(sd.SD_IDX_PLANES, B, Hq, Hkv, n, k=cfg.k, plan_mode=vmode,
                             budget=vbudget)
            stf = DecodeStep(scf, K, V, index, sigma2=sigma2)
            stf.run(q)
            torch.cuda.synchronize()
            pf = stf.plan.cpu().numpy()
            tf = statistics.mean(timed_steps(torch, lambda: stf.run(q), K_st, 3, flush))
            tfs = statistics.mean(timed_steps(torch, lambda: stf.stage_plan_score(q), K_st, 3,
                                              flush))
            bf = rl.plane_scan_bytes(pf, n)
            variants[vname] = {"us_per_step": tf * 1e3, "keys_per_s": keys / (tf * 1e-3),
                               "plan_scan_us": tfs * 1e3, "scan_bytes": bf,
                               "scan_GBps": bf / (tfs * 1e-3) / 1e9,
                               "scan_frac_hbm": bf / (tfs * 1e-3) / 1e9 / peak_gbs}
            del stf
        # the 8-token block landmark scan (256 B of landmark per 8 tokens per KV head),
        # top-64 blocks (512 tokens), gather-attend
        scl = StepConfig(sd.SD_IDX_LANDMARK, B, Hq, Hkv, n, k=cfg.k // 8)
        il = build_index(scl, K)
        stl = DecodeStep(scl, K, V, il)
        stl.run(q)
        torch.cuda.synchronize()
        tl = statistics.mean(timed_steps(torch, lambda: stl.run(q), K_st, 3, flush))
        tls = statistics.mean(timed_steps(torch, lambda: stl.stage_score(q), K_st, 3, flush))
        bl = rl.landmark_scan_bytes(B, Hkv, n)
        variants["landmark8"] = {"us_per_step": tl * 1e3, "keys_per_s": keys / (tl * 1e-3),
                                 "scan_us": tls * 1e3, "scan_bytes": bl,
                                 "scan_GBps": bl / (tls * 1e-3) / 1e9,
                                 "scan_frac_hbm": bl / (tls * 1e-3) / 1e9 / peak_gbs}
        del stl, il
        # 32-bit Hamming (random projection), query map included
        sch = StepConfig(sd.SD_IDX_SIG, B, Hq, Hkv, n, k=cfg.k)
        enc = sd.make_encoder(dev_tensor(inp.W1, torch), dev_tensor(inp.b1, torch))
        ih = build_index(sch, K, enc)
        sth = DecodeStep(sch, K, V, ih, enc=enc)
        sth.run(q)
        torch.cuda.synchronize()
        th = statistics.mean(timed_steps(torch, lambda: sth.run(q), K_st, 3, flush))
        ths = statistics.mean(timed_steps(torch, lambda: sth.stage_score(q), K_st, 3, flush))
        bh = rl.hamming_scan_bytes(B, Hkv, n)
        variants["hamming32"] = {"us_per_step": th * 1e3, "keys_per_s": keys / (th * 1e-3),
                                 "scan_us": ths * 1e3, "scan_bytes": bh,
                                 "scan_GBps": bh / (ths * 1e-3) / 1e9,
                                 "scan_frac_hbm": bh / (ths * 1e-3) / 1e9 / peak_gbs}

        # the KV-write path's index update for one new token (n_old = n - 1): its
        # signature, the 64-token bit-plane block it fills (re-quantised), its 16-token
        # min/max block; eager calls, one launch each (K is unchanged, so every index
        # keeps its content)
        shp_a = sd.make_shape(B, Hq, Hkv, n)
        summ = torch.empty((B, Hkv, (n + 15) // 16, 2, 128), dtype=torch.int16, device="cuda")
        sd.sd_build_index(sd.SD_IDX_MINMAX, shp_a, K, None, summ)
        appends = [
            ("sig", lambda: sd.sd_append_index(sd.SD_IDX_SIG, shp_a, n - 1, K, enc, ih["sig"])),
            ("planes", lambda: sd.sd_append_index(sd.SD_IDX_PLANES, shp_a, n - 1, K, None,
                                                  index["planes"], index["scales"])),
            ("minmax", lambda: sd.sd_append_index(sd.SD_IDX_MINMAX, shp_a, n - 1, K, None,
                                                  summ))]
        variants["append_1token"] = {
            f"{name}_us": statistics.mean(timed_steps(torch, fn, K_st, 3, flush)) * 1e3
            for name, fn in appends}
        del sth, ih, summ

        # index in pinned host memory: gather the planned prefixes over the host link
        # (NVLink-C2C on a Grace host), then scan, select and attend
        hp = index["planes"].cpu().pin_memory()
        hs = index["scales"].cpu().pin_memory()
        dpl = torch.empty_like(index["planes"])
        dsc = torch.empty_like(index["scales"])
        shp = sd.make_shape(B, Hq, Hkv, n)
        sto = DecodeStep(sc, K, V, {"planes": dpl, "scales": dsc}, sigma2=sigma2)

        def offload_only():
            sd.sd_offload_gather(shp, hp, hs, step.plan, dpl, dsc)

        def offload_step():  # the plan must exist before the gather: plan, gather, then
            sto.stage_prep(q)  # the step's calls (the scan recomputes the same plan)
            sd.sd_offload_gather(shp, hp, hs, sto.plan, dpl, dsc)
            sto.stage_plan_score(q)
            sto.stage_topk()
            sto.stage_attend(q)

        to = statistics.mean(timed_steps(torch, offload_only, K_st, 3, flush))
        tos = statistics.mean(timed_steps(torch, offload_step, K_st, 3, flush))
        torch.cuda.synchronize()
        assert np.array_equal(sto.out.cpu().numpy(), step.out.cpu().numpy())
        variants["offload56"] = {"gather_us": to * 1e3, "gather_bytes": scan_bytes,
                                 "host_link_GBps": scan_bytes / (to * 1e-3) / 1e9,
                                 "us_per_step": tos * 1e3, "keys_per_s": keys / (tos * 1e-3)}
        del hp, hs, dpl, dsc, sto

    configs = {}
    if not args.no_variants:
        configs = other_configs(torch, sd, rl, synth, flush, K_st, peak_gbs)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, cfg)

    # ALU peak: the device's SMs x 128 FP32 lanes x the median SM clock seen under load
    sm_mhz = ck.get("sm_mhz") or 1920.0
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    alu_peak = sms * 128 * sm_mhz * 1e6
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"longctx-1m: B={B}, Hq={Hq}, Hkv={Hkv}, d={cfg.d}, n={n}; "
                               f"56-bit water-filled bit-plane scan, top-{cfg.k}, "
                               f"gather-attend over bf16 K/V in HBM",
                   "l2": "flushed before every timed step: a 256 MB write, then a 256 MB "
                         "read of another buffer (no dirty lines of the flush left)",
                   "launch": mode,
                   "parallelism": f"replicas x{ws}"},
        "us_per_step": t_step_max * 1e3,
        "stages_us": {"plan": st_prep * 1e3, "scan": st_score * 1e3, "topk": st_topk * 1e3,
                      "scan_topk": None if st_fused is None else st_fused * 1e3,
                      "plan_scan": st_plan_scan * 1e3,
                      "gather_attend": st_att * 1e3,
                      "select_attend": None if st_sa is None else st_sa * 1e3,
                      "step_eager": eager * 1e3},
        "stages_in_step_us": marginal,
        # the scan is bound by one bit test and one predicated FP32 add per planned
        # token-plane: the peak is the FP32 pipe (128 lanes per SM per clock)
        "roofline": {"bound": "alu", "kernel": "score_planes_tma_kernel",
                     "achieved": alu_ops / (st_score * 1e-3) / 1e12,
                     "peak": alu_peak / 1e12, "unit": "T token-planes/s",
                     "frac": alu_ops / (st_score * 1e-3) / alu_peak,
                     # the bit test and the predicated add are two issued instructions:
                     # the issue-rate bound is half the one-operation peak
                     "frac_issue_bound": 2 * alu_ops / (st_score * 1e-3) / alu_peak,
                     "traffic": scan_traffic("longctx-1m") if n == 1048576 else None,
                     "ops_per_launch": alu_ops, "alg_bytes_per_launch": scan_bytes,
                     "peak_kind": f"derived: {sms} SMs x 128 FP32 lanes x median SM clock "
                                  f"({sm_mhz:.0f} MHz); frac counts one operation per "
                                  f"token-plane, frac_issue_bound two instructions"},
        "roofline_hbm": {"bound": "hbm", "kernel": "score_planes_tma_kernel",
                         "achieved": scan_gbs, "peak": peak_gbs, "unit": "GB/s",
                         "frac": scan_gbs / peak_gbs, "peak_kind": peak_kind,
                         "alg_bytes_per_launch": scan_bytes},
        "step_bytes": {"algorithmic": alg_bytes, "scan": scan_bytes, "gather": gath_bytes,
                       "score_buffer": rl.score_buffer_bytes(B, Hkv, n),
                       "step_GBps": alg_bytes / (t_step_max * 1e-3) / 1e9},
        "plan_bits_per_token": rl.plane_scan_bits_per_token(plan_np),
        "e2e": {"value": e2e_val, "unit": UNIT,
                "h2d_bytes_per_step": int(q_host.numel() * q_host.element_size()),
                "d2h_bytes_per_step": int(out_host.numel() * 4 + lse_host.numel() * 4),
                "launch": "one CUDA graph per step: H2D copy of q from pinned memory, the "
                          "step's kernels, one D2H copy of out and lse to pinned memory "
                          "(sd_copy kernels)"},
        "gpu_launches": launches_per_step(step, q) * args.steps,
        "clocks": ck,
        "variants": variants,
        "other_configs": configs,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
