"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The path shards by request (weak scaling): every rank verifies its own batch
of the same configuration, and the ranks meet only to time the job -- the
slowest rank's timed region and the units all ranks processed.  No GPU.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench._dist() == (ws, rank, rank)
        b = bench.make_batch(rank, N=8, V=256)
        units = 3 * b.total_rows
        elapsed = 10.0 + 5.0 * rank  # rank 1 is the slow one
        dist.barrier()
        mx, tot = bench.reduce_over_ranks(ws, torch.device("cpu"), elapsed, units)
        # the reference arm runs on rank 0 only; the others return at once
        ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), ws, rank) if rank else None
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump({"mx": mx, "tot": tot, "units": units, "N": b.N, "V": b.V,
                       "cu": b.cu.tolist(), "t0": int(np.asarray(b.target).ravel()[:64].sum()),
                       "ref": ref}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ws = 2
    mp.spawn(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, join=True)
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(ws)]
    # every rank sees the slowest rank's time and the whole job's units
    for x in r:
        assert x["mx"] == 15.0
        assert x["tot"] == r[0]["units"] + r[1]["units"]
    # same configuration, independent data
    assert r[0]["N"] == r[1]["N"] == 8 and r[0]["V"] == r[1]["V"] == 256
    assert (r[0]["cu"], r[0]["t0"]) != (r[1]["cu"], r[1]["t0"])
    assert r[1]["ref"] is None


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(1, None, 12.5, 300) == (12.5, 300.0)
