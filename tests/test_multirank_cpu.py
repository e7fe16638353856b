"""Multi-rank host logic on CPU (gloo, world_size 2): sharding independent
sequences across ranks needs no exchange — per-rank oracle results gathered
from both ranks equal the unsharded result — and the benchmark's barrier and
max-over-ranks timing work across processes."""
import os
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_delta_rule_54_gb300 import shard, synth


def _worker(rank, world, store_file, out):
    # a file store: no port to race for
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="file://" + store_file, rank=rank,
                            world_size=world)
    try:
        from oracle.chunked import chunked
        import bench

        lengths = [70, 5, 130, 64, 1, 90, 33]
        w = synth.small(B=1, T=0, Hk=1, Hv=2, Dk=16, Dv=64, h0=True, seed=3)
        d = synth.make_inputs(w, lengths=lengths)
        s0, s1, t0, t1, local = shard.shard_packed(d["cu_seqlens"].numpy(), world, rank)
        o, ht = chunked(d["q"][:, t0:t1], d["k"][:, t0:t1], d["v"][:, t0:t1], d["beta"][:, t0:t1],
                        d["g"][:, t0:t1], d["h0"][s0:s1], cu_seqlens=torch.from_numpy(local),
                        state_mode="e4m3", w_mode="e4m3")
        # gather variable-size shards (pad to the max token count)
        sizes = [None] * world
        dist.all_gather_object(sizes, (t1 - t0, s1 - s0))
        mt = max(s[0] for s in sizes)
        ms = max(s[1] for s in sizes)
        op = torch.zeros(1, mt, 2, 64, dtype=torch.float64)
        op[:, :t1 - t0] = o
        hp = torch.zeros(ms, 2, 16, 64, dtype=torch.float64)
        hp[:s1 - s0] = ht
        go = [torch.zeros_like(op) for _ in range(world)]
        gh = [torch.zeros_like(hp) for _ in range(world)]
        dist.all_gather(go, op)
        dist.all_gather(gh, hp)
        mx = bench._max_over_ranks(float(rank + 1), world, torch.device("cpu"))
        bench._barrier(world)
        if rank == 0:
            o_all = torch.cat([g[:, :s[0]] for g, s in zip(go, sizes)], 1)
            h_all = torch.cat([g[:s[1]] for g, s in zip(gh, sizes)], 0)
            o_ref, h_ref = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   cu_seqlens=d["cu_seqlens"], state_mode="e4m3", w_mode="e4m3")
            # the same per-sequence arithmetic; only the BLAS batch grouping differs
            close = lambda a, b: float((a - b).abs().max()) <= 1e-12 * float(b.abs().max())
            out.put((close(o_all, o_ref), close(h_all, h_ref), mx, [s for s in sizes]))
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_without_exchange():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    store = os.path.join(tempfile.mkdtemp(prefix="gdn_gloo_"), "store")
    procs = [ctx.Process(target=_worker, args=(r, 2, store, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    o_eq, h_eq, mx, sizes = res
    assert o_eq and h_eq
    assert mx == 2.0
    assert sum(s[1] for s in sizes) == 7


def test_shard_range_and_packed_cover_everything_once():
    for n in (0, 1, 7, 64):
        for world in (1, 2, 3, 8):
            rs = [shard.shard_range(n, world, r) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
    lens = synth.varlen_lengths(32768)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for world in (2, 4, 8):
        parts = [shard.shard_packed(cu, world, r) for r in range(world)]
        assert parts[0][0] == 0 and parts[-1][1] == len(lens)
        assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
        assert sum(p[3] - p[2] for p in parts) == 32768
