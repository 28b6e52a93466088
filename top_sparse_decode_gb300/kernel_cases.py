"""Single-kernel workloads of libsd, for profiling one kernel at a time.

    python -m top_sparse_decode_gb300.kernel_cases <case> [--reps R]

Each bandwidth case allocates inputs larger than the GB300's 129 MB L2 but at most
a few GB of device memory; the latency cases (topk_wmax, topk_quest, merge) use the
step's own, smaller shapes.  A case runs its library call R times (default 3) and
waits for the device.  Values are random (normal keys and queries, random signatures and
summaries); what a kernel reads and writes depends on the shapes and the plan, and
the cases fix those.  Cases:

  scan56        bit-plane scan, 56-bit water-filled plan computed in the scan
                (sd_plan_score), 8 KV heads x 1M tokens
  hamming       Hamming scan (sd_score SIG), 8 KV heads x 8M tokens (256 MB)
  hamming_topk  Hamming scan + exact top-512 (sd_hamming_topk), 8 x 2M tokens
  quest         Quest bound (sd_score MINMAX), 64 x 8 heads x 16,384 tokens (268 MB)
  quest_gather  gather-attend over 128 + 1 blocks of 16 tokens (2,064 rows per KV
                head), 32 x 8 heads x 16,384 tokens (270 MB gathered)
  landmark      8-token landmark scan (sd_score LANDMARK), 8 x 1M tokens (268 MB)
  build_planes, build_minmax, build_sig, build_landmark
                index builds from 8 x 1M bf16 keys (2 GB)
  append        the three one-token appends at n = 1M (planes, min/max, signature)
  plan_split    budget split across KV heads (sd_plan SPLIT), 64 x 8 heads
  delta_select  delta selection against a 129-slot resident set, 512 rows
  resident_gather  admitted blocks from pinned host K/V into the resident pool
  offload       planned-prefix gather from pinned host planes, 8 x 1M tokens
  merge         sequence-shard top-k merge, 16 shards x 512 candidates, 64 rows
  topk_wmax     top-512 of 8 rows of 1M random scores through their 32-token word
                maxima (sd_topk_wmax), as in the long-context step
  attend_1m     gather-attend of 8 rows x 512 selected tokens (sd_gather_attend), the
                long-context step's shape; K/V of 131,072 tokens
  topk_quest    top-128 of 1,024 block scores (16-token blocks, last block forced) in
                each of 64 x 8 rows (sd_topk), the Quest step's selection
"""
from __future__ import annotations

import argparse
import math

import torch

import top_sparse_decode_gb300 as sd
from top_sparse_decode_gb300.pipeline import StepConfig, build_index

DEV = "cuda"


def _bf16(shape, gen, std=1.0):
    return (torch.randn(shape, device=DEV, generator=gen) * std).bfloat16().view(torch.int16)


def _i32(shape, gen):
    return torch.randint(-2 ** 31, 2 ** 31 - 1, shape, dtype=torch.int32, device=DEV, generator=gen)


def _planes_case(gen, n=1 << 20, Hkv=8, G=4):
    K = _bf16((1, Hkv, n, 128), gen)
    sc = StepConfig(sd.SD_IDX_PLANES, 1, Hkv * G, Hkv, n)
    idx = build_index(sc, K)
    del K
    q = _bf16((1, Hkv * G, 128), gen)
    s2 = torch.exp(torch.rand((Hkv, 128), device=DEV, generator=gen) * 7.4 - 4.6)
    return sc, idx, q, s2


def make_case(name: str):
    """Returns a function running the case's call once."""
    gen = torch.Generator(device=DEV).manual_seed(20261202)
    if name == "scan56":
        sc, idx, q, s2 = _planes_case(gen)
        shp = sd.make_shape(1, sc.Hq, sc.Hkv, sc.n)
        plan = torch.empty((1, sc.Hkv, 128), dtype=torch.uint8, device=DEV)
        scores = torch.empty((sc.Hkv, sc.n), dtype=torch.float32, device=DEV)
        wmax = torch.empty((sc.Hkv, sc.n // 32), dtype=torch.float32, device=DEV)
        return lambda: sd.sd_plan_score(shp, idx["planes"], idx["scales"], q, s2,
                                        sd.SD_PLAN_WATERFILL, 56, plan, scores, wmax)
    if name in ("hamming", "hamming_topk"):
        n = (8 << 20) if name == "hamming" else (2 << 20)
        Hkv, G = 8, 4
        sig = _i32((1, Hkv, n), gen)
        qsig = _i32((1, Hkv * G), gen)
        shp = sd.make_shape(1, Hkv * G, Hkv, n)
        if name == "hamming":
            scores = torch.empty((Hkv, n), dtype=torch.int32, device=DEV)
            return lambda: sd.sd_score(sd.SD_IDX_SIG, shp, sig, None, qsig, None, scores)
        sel = sd.make_select(512)
        ws = torch.empty(max(sd.sd_hamming_topk_workspace_size(shp, sel), 256), dtype=torch.uint8,
                         device=DEV)
        idx = torch.empty((Hkv, 512), dtype=torch.int32, device=DEV)
        cnt = torch.empty((Hkv,), dtype=torch.int32, device=DEV)
        return lambda: sd.sd_hamming_topk(shp, sig, qsig, sel, idx, 512, cnt, ws)
    if name == "quest":
        B, Hkv, G, n = 64, 8, 4, 16384
        summ = _bf16((B, Hkv, n // 16, 2, 128), gen)
        q = _bf16((B, Hkv * G, 128), gen)
        shp = sd.make_shape(B, Hkv * G, Hkv, n)
        scores = torch.empty((B * Hkv, n // 16), dtype=torch.float32, device=DEV)
        return lambda: sd.sd_score(sd.SD_IDX_MINMAX, shp, summ, None, q, None, scores)
    if name == "quest_gather":
        B, Hkv, G, n, nb = 32, 8, 4, 16384, 129
        K = _bf16((B, Hkv, n, 128), gen)
        V = _bf16((B, Hkv, n, 128), gen)
        q = _bf16((B, Hkv * G, 128), gen)
        rows = B * Hkv
        blocks = torch.sort(torch.rand((rows, n // 16 - 1), device=DEV, generator=gen).argsort(
            dim=1)[:, :nb - 1], dim=1).values
        blocks = torch.cat([blocks, torch.full((rows, 1), n // 16 - 1, device=DEV)], dim=1)
        idx = (blocks[:, :, None] * 16 + torch.arange(16, device=DEV)).reshape(rows, -1)
        idx = idx.to(torch.int32).contiguous()
        cnt = torch.full((rows,), nb * 16, dtype=torch.int32, device=DEV)
        shp = sd.make_shape(B, Hkv * G, Hkv, n)
        ws = torch.empty(max(sd.sd_gather_attend_workspace_size(shp, nb * 16), 256),
                         dtype=torch.uint8, device=DEV)
        out = torch.empty((B, Hkv * G, 128), dtype=torch.float32, device=DEV)
        lse = torch.empty((B, Hkv * G), dtype=torch.float32, device=DEV)
        return lambda: sd.sd_gather_attend(shp, q, K, V, idx, nb * 16, cnt, nb * 16,
                                           1 / math.sqrt(128), out, lse, ws)
    if name == "landmark":
        Hkv, G, n = 8, 4, 1 << 20
        L = _bf16((1, Hkv, n // 8, 128), gen)
        q = _bf16((1, Hkv * G, 128), gen)
        shp = sd.make_shape(1, Hkv * G, Hkv, n)
        scores = torch.empty((Hkv, n // 8), dtype=torch.float32, device=DEV)
        return lambda: sd.sd_score(sd.SD_IDX_LANDMARK, shp, L, None, q, None, scores)
    if name.startswith("build_") or name == "append":
        Hkv, G, n = 8, 4, 1 << 20
        K = _bf16((1, Hkv, n, 128), gen)
        shp = sd.make_shape(1, Hkv * G, Hkv, n)
        W1 = torch.randn((32, 128), device=DEV, generator=gen)
        enc = sd.make_encoder(W1, torch.zeros(32, device=DEV))
        planes = torch.empty((1, Hkv, 128, 4, n // 32), dtype=torch.int32, device=DEV)
        scales = torch.empty((1, Hkv, 128, n // 64), dtype=torch.int16, device=DEV)
        summ = torch.empty((1, Hkv, n // 16, 2, 128), dtype=torch.int16, device=DEV)
        sig = torch.empty((1, Hkv, n), dtype=torch.int32, device=DEV)
        lm = torch.empty((1, Hkv, n // 8, 128), dtype=torch.int16, device=DEV)
        calls = {
            "build_planes": lambda: sd.sd_build_index(sd.SD_IDX_PLANES, shp, K, None, planes, scales),
            "build_minmax": lambda: sd.sd_build_index(sd.SD_IDX_MINMAX, shp, K, None, summ),
            "build_sig": lambda: sd.sd_build_index(sd.SD_IDX_SIG, shp, K, enc, sig),
            "build_landmark": lambda: sd.sd_build_index(sd.SD_IDX_LANDMARK, shp, K, None, lm)}
        if name != "append":
            return calls[name]
        for c in calls.values():
            c()

        def appends():
            sd.sd_append_index(sd.SD_IDX_PLANES, shp, n - 1, K, None, planes, scales)
            sd.sd_append_index(sd.SD_IDX_MINMAX, shp, n - 1, K, None, summ)
            sd.sd_append_index(sd.SD_IDX_SIG, shp, n - 1, K, enc, sig)
        return appends
    if name == "plan_split":
        B, Hkv, G = 64, 8, 4
        q = _bf16((B, Hkv * G, 128), gen)
        s2 = torch.exp(torch.rand((Hkv, 128), device=DEV, generator=gen) * 7.4 - 4.6)
        shp = sd.make_shape(B, Hkv * G, Hkv, 64)
        plan = torch.empty((B, Hkv, 128), dtype=torch.uint8, device=DEV)
        return lambda: sd.sd_plan(shp, q, s2, sd.SD_PLAN_SPLIT, 56, plan)
    if name in ("delta_select", "resident_gather"):
        B, Hkv, G, n, R, C, kb = 64, 8, 4, 16384, 129, 7, 128
        rows, nu = B * Hkv, n // 16
        shp = sd.make_shape(B, Hkv * G, Hkv, n)
        sel = sd.make_select(kb, 0, 1, 16)
        res = sd.Resident(rows, R, nu)
        preds = []
        for _ in range(2):
            scores = torch.randn((rows, nu), device=DEV, generator=gen)
            idx = torch.empty((rows, (kb + 1) * 16), dtype=torch.int32, device=DEV)
            cnt = torch.empty((rows,), dtype=torch.int32, device=DEV)
            ws = torch.empty(max(sd.sd_topk_workspace_size(rows, nu, sel), 256),
                             dtype=torch.uint8, device=DEV)
            sd.sd_topk(sd.SD_SCORE_F32, scores, rows, nu, n, sel, idx, (kb + 1) * 16, cnt, ws)
            preds.append((scores, idx, cnt))
        plan = [torch.empty((rows, C), dtype=torch.int32, device=DEV) for _ in range(3)]
        pcnt = torch.empty(rows, dtype=torch.int32, device=DEV)
        pool = torch.empty((rows, (kb + 1) * 16), dtype=torch.int32, device=DEV)
        pool_cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
        step = [0]

        def select():
            s3, i3, n3 = preds[step[0] % 2]
            sd.sd_delta_select(shp, sel, s3, i3, (kb + 1) * 16, n3, C, step[0], res, *plan, pcnt,
                               pool, (kb + 1) * 16, pool_cnt)
            step[0] += 1
        if name == "delta_select":
            return select
        Kh = _bf16((B, Hkv, n, 128), gen).cpu().pin_memory()
        Vh = _bf16((B, Hkv, n, 128), gen).cpu().pin_memory()
        Kp = torch.zeros((B, Hkv, R * 16, 128), dtype=torch.int16, device=DEV)
        Vp = torch.zeros_like(Kp)

        def gather():
            select()
            sd.sd_resident_gather(shp, 16, Kh, Vh, plan[0], plan[1], pcnt, C, R, Kp, Vp)
        return gather
    if name == "offload":
        sc, idx, q, s2 = _planes_case(gen)
        shp = sd.make_shape(1, sc.Hq, sc.Hkv, sc.n)
        plan = torch.empty((1, sc.Hkv, 128), dtype=torch.uint8, device=DEV)
        sd.sd_plan(shp, q, s2, sd.SD_PLAN_WATERFILL, 56, plan)
        hp = idx["planes"].cpu().pin_memory()
        hs = idx["scales"].cpu().pin_memory()
        dp, ds = torch.empty_like(idx["planes"]), torch.empty_like(idx["scales"])
        return lambda: sd.sd_offload_gather(shp, hp, hs, plan, dp, ds)
    if name == "topk_wmax":  # the long-context step's top-512 from scores and word maxima
        Hkv, n, k = 8, 1 << 20, 512
        scores = torch.randn((Hkv, n), device=DEV, generator=gen)
        wmax = scores.view(Hkv, n // 32, 32).amax(dim=2).contiguous()
        sel = sd.make_select(k)
        stride = k
        idx = torch.empty((Hkv, stride), dtype=torch.int32, device=DEV)
        cnt = torch.empty((Hkv,), dtype=torch.int32, device=DEV)
        ws = torch.empty(max(sd.sd_topk_workspace_size(Hkv, n, sel), 256), dtype=torch.uint8,
                         device=DEV)
        return lambda: sd.sd_topk_wmax(scores, wmax, Hkv, n, sel, idx, stride, cnt, ws)
    if name == "topk_quest":  # the Quest step's block selection: 512 rows of 1,024 blocks
        rows, nb, blk = 64 * 8, 1024, 16
        scores = torch.randn((rows, nb), device=DEV, generator=gen)
        sel = sd.make_select(128, 0, 1, blk)
        stride = 129 * blk
        idx = torch.empty((rows, stride), dtype=torch.int32, device=DEV)
        cnt = torch.empty((rows,), dtype=torch.int32, device=DEV)
        ws = torch.empty(max(sd.sd_topk_workspace_size(rows, nb, sel), 256), dtype=torch.uint8,
                         device=DEV)
        return lambda: sd.sd_topk(sd.SD_SCORE_F32, scores, rows, nb, nb * blk, sel, idx, stride,
                                  cnt, ws)
    if name == "attend_1m":  # the long-context step's gather-attend: 8 rows of 512 tokens
        Hkv, G, n, c = 8, 4, 1 << 17, 512
        K = _bf16((1, Hkv, n, 128), gen)
        V = _bf16((1, Hkv, n, 128), gen)
        q = _bf16((1, Hkv * G, 128), gen)
        idx = torch.sort(torch.rand((Hkv, n), device=DEV, generator=gen).argsort(dim=1)[:, :c],
                         dim=1).values.to(torch.int32).contiguous()
        cnt = torch.full((Hkv,), c, dtype=torch.int32, device=DEV)
        shp = sd.make_shape(1, Hkv * G, Hkv, n)
        ws = torch.empty(max(sd.sd_gather_attend_workspace_size(shp, c), 256), dtype=torch.uint8,
                         device=DEV)
        out = torch.empty((1, Hkv * G, 128), dtype=torch.float32, device=DEV)
        lse = torch.empty((1, Hkv * G), dtype=torch.float32, device=DEV)
        return lambda: sd.sd_gather_attend(shp, q, K, V, idx, c, cnt, c, 1 / math.sqrt(128), out,
                                           lse, ws)
    if name == "merge":
        S, rows, k = 16, 64, 512
        cs = torch.randn((S, rows, k), device=DEV, generator=gen)
        ci = torch.randint(0, 1 << 24, (S, rows, k), dtype=torch.int32, device=DEV, generator=gen)
        cc = torch.full((S, rows), k, dtype=torch.int32, device=DEV)
        out = torch.empty((rows, k), dtype=torch.int32, device=DEV)
        cnt = torch.empty((rows,), dtype=torch.int32, device=DEV)
        return lambda: sd.sd_topk_merge(rows, S, k, cs, ci, cc, out, k, cnt)
    raise SystemExit(f"unknown case {name!r}; see the module docstring")


def main():
    p = argparse.ArgumentParser()
    p.add_argument("case")
    p.add_argument("--reps", type=int, default=3)
    p.add_argument("--time", action="store_true",
                   help="replay the run as a CUDA graph after an L2 flush and print the mean "
                        "CUDA-event time of a replay")
    a = p.parse_args()
    from top_sparse_decode_gb300 import build
    build.build()
    fn = make_case(a.case)
    torch.cuda.synchronize()
    if not a.time:
        for _ in range(a.reps):
            fn()
        torch.cuda.synchronize()
        sd.sd_device_status()
        print(f"{a.case}: {a.reps} runs ok")
        return
    # the run as a CUDA graph (host launch cost off the device's timeline), each replay
    # after an L2 flush (write one 256 MB buffer, then read another: no dirty lines)
    # and a ~50 us device-side spin, so the replay is queued before e0 fires
    wbuf = torch.empty(64 << 20, dtype=torch.float32, device=DEV)
    rbuf = torch.ones(64 << 20, dtype=torch.float32, device=DEV)
    sink = torch.empty((), dtype=torch.float32, device=DEV)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        fn()  # warm: attributes and caches set outside the capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            fn()
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(a.reps):
        wbuf.zero_()
        sink.copy_(rbuf.max())
        torch.cuda._sleep(100000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    sd.sd_device_status()
    print(f"{a.case}: {1e3 * total / a.reps:.1f} us per run (mean of {a.reps}, L2 flushed)")


if __name__ == "__main__":
    main()
