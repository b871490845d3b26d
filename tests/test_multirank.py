"""Multi-process paths on CPU (gloo, world size 2).

1. The benchmark's rank bookkeeping: the job time is the slowest rank's and
   the value counts the work of every replica.
2. The exchange a sequence-sharded global-query row would need: each rank
   holds partial softmax statistics over its own key shard, the ranks
   all-gather them, and the merge by softmax denominators ("LONGNET: Scaling
   Transformers to 1,000,000,000 Tokens", section 3.4, "Mixture of Dilated
   Attentions") reproduces the unsharded row.  The arithmetic here is the CPU
   oracle's; only the protocol is under test.
3. A rank that dies before that exchange: the survivor's collective gives up
   within a short process-group timeout and reports an error; it does not
   hang.  (The failure is made on the host: the rank exits.)
"""
import datetime
import os
import socket
import time

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket(); s.bind(("127.0.0.1", 0)); port = s.getsockname()[1]; s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from oracle import lg_oracle
        # 1. bookkeeping
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        v = bench.job_throughput(1e12, 4, world, t)
        # 2. sharded partial statistics for a few global query rows
        rng = np.random.default_rng(0)
        n, nk, D = 3, 64, 8
        qq, kk, vv = rng.standard_normal((n, D)), rng.standard_normal((nk, D)), rng.standard_normal((nk, D))
        lo, hi = rank * nk // world, (rank + 1) * nk // world
        mask = np.zeros((n, nk), bool); mask[:, lo:hi] = True
        m, l, acc = lg_oracle.partial_stats(qq, kk, vv, mask, 0.5)
        pack = torch.from_numpy(np.concatenate([m[:, None], l[:, None], acc], axis=1))
        parts = [torch.zeros_like(pack) for _ in range(world)]
        dist.all_gather(parts, pack)
        ms = [p[:, 0].numpy() for p in parts]; ls = [p[:, 1].numpy() for p in parts]
        accs = [p[:, 2:].numpy() for p in parts]
        o, lse = lg_oracle.merge_partials(ms, ls, accs)
        ref_o, ref_l, _ = lg_oracle.masked_attention(qq, kk, vv, np.ones((n, nk), bool), 0.5)
        q.put((rank, t, v, float(np.abs(o - ref_o).max()), float(np.abs(lse - ref_l).max())))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t, v, err_o, err_l in res:
        assert t == 15.0                                  # slowest rank's time on every rank
        assert v == pytest.approx(1e12 * 4 * 2 / 15e-3 / 1e12)
        assert err_o < 1e-12 and err_l < 1e-12


EXCHANGE_TIMEOUT_S = 10


def _worker_killed(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=EXCHANGE_TIMEOUT_S))
    if rank == 1:
        os._exit(0)            # dies after joining, before the exchange of partial statistics
    from oracle import lg_oracle
    rng = np.random.default_rng(1)
    qq, kk, vv = rng.standard_normal((2, 8)), rng.standard_normal((16, 8)), rng.standard_normal((16, 8))
    mask = np.zeros((2, 16), bool); mask[:, :8] = True
    m, l, acc = lg_oracle.partial_stats(qq, kk, vv, mask, 0.5)
    pack = torch.from_numpy(np.concatenate([m[:, None], l[:, None], acc], axis=1))
    parts = [torch.zeros_like(pack) for _ in range(world)]
    t0 = time.monotonic()
    try:
        dist.all_gather(parts, pack)
        q.put(("no error", time.monotonic() - t0))
    except Exception as e:  # the survivor learns of the dead peer from the collective
        q.put((type(e).__name__, time.monotonic() - t0))
    q.close()
    q.join_thread()            # the result reaches the parent before the hard exit
    os._exit(0)                # the process group is broken; leave without a collective teardown


def test_killed_rank_times_out_instead_of_hanging():
    """The survivor either reports the failed exchange or exits with an error
    within the process-group timeout; what must not happen is a hang."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_killed, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    survivor = procs[0]
    survivor.join(timeout=EXCHANGE_TIMEOUT_S + 60)
    hung = survivor.is_alive()
    for p in procs:
        if p.is_alive():
            p.kill()
        p.join(timeout=10)
    assert not hung, "the surviving rank hung in the exchange with a dead rank"
    try:
        what, secs = q.get(timeout=5)
    except Exception:
        what, secs = None, None
    if what is None:
        assert survivor.exitcode != 0, "the survivor neither reported the failure nor exited with an error"
    else:
        assert what != "no error", "the exchange with a dead rank did not fail"
        assert secs <= EXCHANGE_TIMEOUT_S + 5
