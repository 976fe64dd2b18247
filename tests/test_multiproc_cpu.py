"""N > 1 host logic on CPU with the gloo backend (world size 2).

The path shards by rows with no exchange: rank r evaluates its own rows and
the union is the single-process answer bit for bit.  Here each rank runs the
oracle on its row slice and the gathered result is compared with one
process's answer; the benchmark's timing reduction (max over ranks) and the
reference arm's "rank 0 alone prints" rule are exercised the same way.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from invariant_token_logprob_gb300.inputs import lm_head_inputs
        d = lm_head_inputs(10, 64, 700, seed=3)
        lo, hi = rank * 5, (rank + 1) * 5
        r = oracle.logprob(d["h"][lo:hi], d["W"], d["targets"][lo:hi], 1.0)
        mine = torch.from_numpy(np.stack([r["logp"], r["lse"], r["argmax"].astype(np.float64)]))
        parts = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        t = bench.max_over_ranks(float(rank + 1), world, "cpu")
        if rank == 0:
            q.put((torch.cat(parts, dim=1).numpy(), t))
    finally:
        dist.destroy_process_group()


def test_row_sharding_matches_single_process():
    import oracle
    from invariant_token_logprob_gb300.inputs import lm_head_inputs
    oracle.load()  # build before forking workers
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    d = lm_head_inputs(10, 64, 700, seed=3)
    r = oracle.logprob(d["h"], d["W"], d["targets"], 1.0)
    assert np.array_equal(got[0], r["logp"]) and np.array_equal(got[1], r["lse"])
    assert np.array_equal(got[2].astype(np.int64), r["argmax"])
    assert tmax == 2.0  # the slowest rank's time is the job's time


def test_reference_arm_rank1_exits_silently():
    """Under torchrun the reference arm runs on rank 0 only; other ranks exit 0
    without work or output."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    # rank 1 alone cannot rendezvous, so only check the early exit path that
    # needs no process group: run with a stub that skips dist init.
    code = ("import sys; sys.path.insert(0, %r); import bench;"
            "bench.dist_init = lambda: (2, 1, 1);"
            "sys.argv = ['bench.py', '--impl', 'reference', '--steps', '1', '--warmup', '0'];"
            "sys.exit(bench.main())") % ROOT
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def _shard_worker(rank, world, port, q):
    """Rank r: block statistics of its vocabulary shard (oracle, global indices),
    all-gathered as [R][T][tiles_per_shard]; rank 0 reassembles global tile order
    and merges with the oracle's fp64 merge."""
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from invariant_token_logprob_gb300.inputs import lm_head_inputs
        T, H, V, bn = 6, 32, 1900, 256
        d = lm_head_inputs(T, H, V, seed=4)
        nvt = (V + bn - 1) // bn
        nvt_s = (nvt + world - 1) // world
        lo, hi = rank * nvt_s * bn, min((rank + 1) * nvt_s * bn, V)
        tg_local = d["targets"] - lo  # targets outside the shard match no block
        bs = oracle.block_stats(d["h"], d["W"][lo:hi], tg_local, bn)
        blk = np.full((T, nvt_s, 4), np.nan)
        n = bs["m"].shape[1]
        blk[:, :n, 0], blk[:, :n, 1] = bs["m"], bs["s"]
        blk[:, :n, 2], blk[:, :n, 3] = bs["a"] + lo, bs["zt"]
        mine = torch.from_numpy(blk)
        parts = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        if rank == 0:
            g = torch.stack(parts).numpy()  # [R][T][nvt_s][4]
            glob = np.concatenate([g[r] for r in range(world)], axis=1)[:, :nvt]
            q.put(glob)
    finally:
        dist.destroy_process_group()


def test_vocab_sharded_exchange_matches_unsharded_oracle():
    import oracle
    from invariant_token_logprob_gb300.inputs import lm_head_inputs
    oracle.load()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    glob = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    d = lm_head_inputs(6, 32, 1900, seed=4)
    bs = oracle.block_stats(d["h"], d["W"], d["targets"], 256)
    assert np.array_equal(glob[..., 0], bs["m"]) and np.array_equal(glob[..., 1], bs["s"])
    assert np.array_equal(glob[..., 2].astype(np.int64), bs["a"])
    assert np.array_equal(glob[..., 3], bs["zt"])
    a = oracle.merge_blocks(glob[..., 0], glob[..., 1], glob[..., 2], glob[..., 3], d["targets"],
                            1900, 256)
    b = oracle.merge_blocks(bs["m"], bs["s"], bs["a"], bs["zt"], d["targets"], 1900, 256)
    for k in ("lse", "logp", "argmax"):
        assert np.array_equal(a[k], b[k])
    full = oracle.logprob(d["h"], d["W"], d["targets"])
    assert np.array_equal(a["argmax"], full["argmax"])
