"""One sequence split by tokens across two ranks (HashAttention 2.5, contexts beyond
one device), driven by the library's SPMD protocol (top_sparse_decode_gb300.shard:
run_sharded_step, its torch.distributed all-gathers) over gloo on CPU.  Each rank's
phases are the oracle's (no GPU here): the merged index set equals the unsharded
oracle step's exactly and the combined attention its attention."""
import math
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASE = dict(n=64 * 40 + 17, k=48, sink=5, local=33)


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleShard:
    """The phases of one shard, computed by the oracle (test infrastructure)."""

    def __init__(self, inp, cfg, shard, shards):
        import oracle
        self.o, self.cfg, self.inp = oracle, cfg, inp
        cut = oracle.shard_bounds(cfg.n, shards)
        self.a, self.b = cut[shard], cut[shard + 1]
        self.win = oracle.shard_windows(cfg.n, self.a, self.b, cfg.sink, cfg.local)
        self.K = np.ascontiguousarray(inp.K[:, :, self.a:self.b])
        self.V = np.ascontiguousarray(inp.V[:, :, self.a:self.b])
        p, s = oracle.plane_build(self.K)
        plan = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_WATERFILL, 56)
        self.scores = oracle.plane_score(p, s, plan, inp.q, n=self.b - self.a).reshape(
            cfg.B * cfg.Hkv, -1)

    def phase1(self, q):
        sc, ix, cnt = self.o.shard_candidates(self.scores, self.cfg.k, *self.win, self.a)
        return torch.from_numpy(sc), torch.from_numpy(ix), torch.from_numpy(cnt)

    def phase2(self, q, all_score, all_idx, all_count):
        S = all_score.shape[0]
        mi, mc = self.o.topk_merge([all_score[s].numpy() for s in range(S)],
                                   [all_idx[s].numpy() for s in range(S)],
                                   [all_count[s].numpy() for s in range(S)], self.cfg.k)
        self.merged = (mi, mc)
        li, lc = self.o.shard_select(mi, mc, self.a, self.b, *self.win)
        cfg = self.cfg
        out, lse = self.o.gather_attend(self.inp.q, self.K, self.V, li.reshape(cfg.B, cfg.Hkv, -1),
                                        lc.reshape(cfg.B, cfg.Hkv), 1 / math.sqrt(cfg.d))
        return torch.from_numpy(out), torch.from_numpy(lse)

    def phase3(self, all_out, all_lse):
        S = all_out.shape[0]
        return self.o.attend_combine([all_out[s].numpy() for s in range(S)],
                                     [all_lse[s].numpy() for s in range(S)])


def _rank_main(rank, ws, port, out):
    os.environ.update({"WORLD_SIZE": str(ws), "RANK": str(rank), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    import oracle
    import synth
    from top_sparse_decode_gb300.shard import run_sharded_step
    from test_shard_gloo import OracleShard
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    cfg = synth.config(0, B=2, Hq=8, Hkv=2, **CASE)
    inp = synth.make_inputs(cfg)
    sh = OracleShard(inp, cfg, rank, ws)
    o, l = run_sharded_step(sh, None)
    # the unsharded oracle step
    p, s = oracle.plane_build(inp.K)
    plan = oracle.plan(inp.q, inp.sigma2, cfg.Hkv, oracle.PLAN_WATERFILL, 56)
    sc = oracle.plane_score(p, s, plan, inp.q, n=cfg.n).reshape(4, -1)
    ri, rc = oracle.topk(sc, cfg.k, cfg.sink, cfg.local)
    ro, rl = oracle.gather_attend(inp.q, inp.K, inp.V, ri.reshape(2, 2, -1), rc.reshape(2, 2),
                                  1 / math.sqrt(cfg.d))
    # competing part of the unsharded set = the merged set, on every rank
    lead = min(cfg.sink, cfg.n)
    tail = max(cfg.n - cfg.local, lead)
    mi, mc = sh.merged
    same = all(sorted(mi[r, :mc[r]].tolist()) ==
               [t for t in ri[r, :rc[r]].tolist() if lead <= t < tail] for r in range(4))
    out.put((rank, same, float(np.abs(o - ro).max()), float(np.abs(l - rl).max())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_sharded_step_equals_unsharded_oracle():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, same, eo, el in res:
        assert same, rank
        assert eo < 1e-12 and el < 1e-12, (rank, eo, el)
