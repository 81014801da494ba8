"""The N > 1 benchmark path on CPU: two gloo ranks, each timing its own replica,
agree on the slowest rank's time (the only cross-rank step of the path)."""
import os
import queue
import socket
import sys
import time

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as td
    import bench
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow replica
        q.put((rank, ws, r, local, bench.max_over_ranks(mine)))
    finally:
        td.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert all(o[4] == 15.0 for o in out)


def _worker_one_rank_lost(rank, world, port, q, ready, how):
    # rank 1 is lost before the timing reduction: it either stays away from the
    # collective (a hung replica) or exits (a crashed one); rank 0 must get an
    # error from its collective within the process-group timeout, not hang.
    # Rank 1 leaves only after rank 0's process group is up (`ready`), so the
    # error comes from the collective, not from the rendezvous.
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), FLUX_BENCH_PG_TIMEOUT_S="3")
    import time
    try:
        import bench
        bench.dist_init()
        if rank == 1:
            ready.wait(60)
            if how == "stays_away":
                time.sleep(8)  # longer than rank 0's 3 s timeout
            os._exit(0)
        ready.set()
        t0 = time.time()
        try:
            bench.max_over_ranks(1.0)
            q.put(("no error", time.time() - t0))
        except Exception as e:  # noqa: BLE001 - any error from the collective is the signal
            q.put((type(e).__name__, time.time() - t0))
    except Exception as e:  # noqa: BLE001
        q.put((f"set-up failed: {e!r}", -1.0))
    # flush the queue's feeder thread before the hard exit (os._exit skips it)
    q.close()
    q.join_thread()
    os._exit(0)


@pytest.mark.parametrize("how", ["stays_away", "exits"])
def test_a_lost_replica_ends_the_other_ranks_collective_with_an_error(how):
    # the property: rank 0 does not hang.  It either reports the collective's
    # error or is ended by its communication library when the peer's
    # connection drops (both end the job; neither holds the GPU)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ready = ctx.Event()
    port = _free_port()
    procs = [ctx.Process(target=_worker_one_rank_lost, args=(r, 2, port, q, ready, how))
             for r in range(2)]
    t0 = time.time()
    for p in procs:
        p.start()
    procs[0].join(timeout=90)
    hung = procs[0].is_alive()
    ended_after = time.time() - t0
    for p in procs:
        p.join(timeout=20)
        if p.is_alive():  # pragma: no cover - never leave a child behind
            p.kill()
            p.join()
    assert not hung, "rank 0 still waits for the lost replica"
    try:
        what, waited = q.get(timeout=5)
    except queue.Empty:
        what, waited = None, None
    if what is None:
        assert procs[0].exitcode != 0, "rank 0 ended without reporting"
        assert ended_after < 60.0
    else:
        assert not what.startswith("set-up failed"), what
        assert what != "no error"
        assert 0.0 <= waited < 30.0


def test_single_process_reduction_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
