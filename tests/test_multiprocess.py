"""The bench's multi-rank path on CPU: two ranks over gloo (127.0.0.1) run the same
process-group set-up, barrier and max / sum over ranks that ``bench.py`` uses under
torchrun, where the timed value is the maximum of the ranks' times and the work is
summed (weak scaling, replicas only)."""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank: int, world: int, port: int, out) -> None:
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    w, r, _ = bench.dist_setup()
    dev = torch.device("cpu")
    secs = 1.0 + 0.5 * r  # this rank's time
    work = 100 * (r + 1)  # this rank's units
    t = bench.max_over_ranks(w, secs, dev)
    n = bench.sum_over_ranks(w, work, dev)
    bench.barrier(w)
    out.put((r, w, t, n))
    torch.distributed.destroy_process_group()


@pytest.mark.timeout(120)
def test_rank_reductions_two_ranks_gloo():
    if torch.cuda.is_available():
        pytest.skip("the gloo fallback is for hosts without a GPU")
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    for _, w, t, n in res:
        assert w == 2
        assert t == 1.5          # the slower rank's time
        assert n == 300          # both ranks' work
