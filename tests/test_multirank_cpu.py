"""Multi-rank host logic on CPU ranks (gloo, world size 2): bench.py's
max-over-ranks timing, barriers and rank-0-only reference arm; the pages'
sharded block with its all-reduces as real collectives between processes
(the oracle's arithmetic per rank); and the loss of one rank, which must end
the survivors' next collective with an error rather than a hang.  The
library's own block does not shard across GPUs (its shards are logical
partitions of one GPU), so its replicas exchange nothing but timing."""
import os
import socket
import subprocess
import sys
import time

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def _sharded_worker(rank, world, port, q):
    """Rank s is shard s of undercodenews.com/?p=110319, "the Original": the
    Q/K/V rows of its heads, attention over them, its columns of Wo, its
    FFN-up rows and Wd columns; the two all-reduces are gloo all_reduce
    calls.  The arithmetic per rank is the oracle's."""
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle.tp_oracle as o
    x, w, H, causal = _sharded_case()
    d = x.shape[-1]
    dh, h_l = d // H, H // world
    f_l = w["Wd"].shape[1] // world
    rows = slice(rank * h_l * dh, (rank + 1) * h_l * dh)
    cols = slice(rank * f_l, (rank + 1) * f_l)
    xb = o.to64(x[0])
    a = o.multi_head_attention(o.linear(xb, w["Wq"][rows]), o.linear(xb, w["Wk"][rows]),
                               o.linear(xb, w["Wv"][rows]), h_l, causal)
    part = torch.from_numpy(a @ o.to64(w["Wo"])[:, rows].T)
    dist.all_reduce(part)                                   # H = X + sum_s A_s Wo_s^T
    h = xb + part.numpy()
    u = o.silu(o.linear(h, w["Wg"][cols])) * o.linear(h, w["Wu"][cols])
    part = torch.from_numpy(u @ o.to64(w["Wd"])[:, cols].T)
    dist.all_reduce(part)                                   # Y = H + sum_s U_s Wd_s^T
    q.put((rank, h + part.numpy()))
    dist.destroy_process_group()


def _sharded_case():
    g = torch.Generator().manual_seed(5)
    d, H, f, T = 64, 4, 96, 12
    w = {n: torch.randn(r, c, generator=g, dtype=torch.float64) * 0.2
         for n, (r, c) in {"Wq": (d, d), "Wk": (d, d), "Wv": (d, d), "Wo": (d, d), "Wg": (f, d), "Wu": (f, d),
                           "Wd": (d, f)}.items()}
    x = torch.randn(1, T, d, generator=g, dtype=torch.float64)
    return x, w, H, True


def test_sharded_block_with_gloo_all_reduce():
    """Two processes each holding one shard, joined by real all-reduces,
    give every rank the unsharded block's output."""
    sys.path.insert(0, ROOT)
    import oracle.tp_oracle as o
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sharded_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    x, w, H, causal = _sharded_case()
    ref, _, _ = o.block_forward(x, w, H, "swiglu", causal)
    for r in (0, 1):
        assert np.max(np.abs(res[r] - ref[0])) <= 1e-12 * np.max(np.abs(ref[0]))


def _lost_rank_worker(rank, world, port, q):
    """bench.py's process group with a short timeout: rank 1 leaves before
    the first barrier (as a replica whose process died would); rank 0's
    barrier must end with an error, not wait for ever."""
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), TP_BENCH_BACKEND="gloo", TP_BENCH_PG_TIMEOUT_S="5")
    import bench
    _, _, _, pg = bench.dist_setup(world)
    if rank == 1:
        q.put((1, "left"))
        q.close()
        q.join_thread()  # the message is out before the process goes
        os._exit(0)  # no barrier, no destroy_process_group: the rank is gone
    t0 = time.monotonic()
    try:
        pg.barrier()
        q.put((0, "barrier passed"))
    except Exception as e:  # gloo reports the lost peer or the timeout
        q.put((0, f"error after {time.monotonic() - t0:.1f} s: {type(e).__name__}"))


def test_lost_rank_ends_the_survivors_barrier_with_an_error():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_lost_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(60)
        assert p.exitcode is not None, "a rank is still running"
    assert res[1] == "left"
    assert res[0].startswith("error after"), res[0]
