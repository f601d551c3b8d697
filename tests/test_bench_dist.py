"""Replica timing across ranks (gloo, world size 2, CPU): the bench reports the
maximum over ranks and rank 0 alone prints."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, [3.5, 7.25], out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 7.25, 1: 7.25}


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks(4.0) == 4.0


def test_dist_env_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (2, 1, 1)


def test_algorithmic_flops_counts_visible_pairs():
    # QK over 576 dims and PV over 512: 2 * 1088 flop per visible (row, key).
    assert bench.algorithmic_flops([4096], 12, 1, False) == 2 * 1088 * 12 * 4096
    # Causal MTP block of 4 over L = 10: query token qi sees 10 - 4 + qi + 1 keys.
    assert bench.algorithmic_flops([10], 2, 4, True) == 2 * 1088 * 2 * (7 + 8 + 9 + 10)
    # Selected pages 0 and 2 of a 100-token request: keys 0-31 and 64-95.
    sel = np.array([[0, 2, -1]])
    assert bench.algorithmic_flops([100], 1, 1, False, sel) == 2 * 1088 * 64
    # A causal row of a 70-token request sees keys 0-31 and 64-69 of them.
    assert bench.algorithmic_flops([70], 1, 1, True, np.array([[0, 2]])) == 2 * 1088 * 38
