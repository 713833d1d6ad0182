"""The N > 1 logic of bench.py as two gloo ranks on CPU.

bench.py runs one process per GPU under torchrun; the path shards by tokens
with no exchange, so ranks are independent replicas and only the timing is
collective: a barrier on both sides of the timed region, the slowest rank's
time (max over ranks), whole-job tokens/s = ranks x tokens / that time, and
per-rank input batches. The reference arm runs on rank 0 only. Here two
processes rendezvous over 127.0.0.1 with the gloo backend (no GPU) and
check each of those pieces."""
import argparse
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import moe_inputs as I

    r, w, _, pg = bench.dist_setup(argparse.Namespace(impl="ours"))
    out = {"rank": r, "world": w, "backend": pg.get_backend()}
    pg.barrier()
    out["max_ms"] = bench.max_over_ranks(pg, 100.0 + 7.0 * rank)   # rank 1 is slower
    out["value"] = bench.job_tokens_per_s(w, 8192, out["max_ms"] / 100)
    seeds = [bench.rank_case(I.GPTOSS, rank, j).seed for j in range(4)]
    everyone = [None] * world
    pg.all_gather_object(everyone, seeds)
    out["seeds"] = everyone
    if rank != 0:   # the reference arm prints and works on rank 0 only
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            out["ref_rc"] = bench.run_reference(
                argparse.Namespace(workload="gptoss_prefill_n8192", steps=1, warmup=0),
                rank, world, pg)
        out["ref_printed"] = buf.getvalue()
    pg.barrier()
    pg.destroy_process_group()
    q.put(out)


@pytest.mark.timeout(300)
def test_two_gloo_ranks_time_and_shard_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=240) for _ in procs), key=lambda d: d["rank"])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for d in res:
        assert d["world"] == 2 and d["backend"] == "gloo"
        assert d["max_ms"] == 107.0   # the slowest rank's time, on every rank
        assert abs(d["value"] - 2 * 8192 / 1.07e-3) < 1e-6 * d["value"]
    s0, s1 = res[0]["seeds"]
    assert res[0]["seeds"] == res[1]["seeds"] and not set(s0) & set(s1)   # own batches
    assert res[1]["ref_rc"] == 0 and res[1]["ref_printed"] == ""
