"""Host-side logic of bench.py without a GPU: the replica control plane (gloo,
two ranks on the CPU) and the whole-job throughput aggregation."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    ws, r, local = bench.dist_env()
    c = bench.Control(ws)
    try:
        c.barrier()
        # rank r did (r+1) units of 1e12 flops in (r+1) * 0.5 s
        total, t, value = bench.aggregate(c, (r + 1) * 1e12, (r + 1) * 0.5)
        q.put((r, total, t, value))
    finally:
        c.close()


def test_two_replicas_aggregate_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, total, t, value in res:
        assert total == pytest.approx(3e12)      # work of all ranks
        assert t == pytest.approx(1.0)           # the slowest rank's time
        assert value == pytest.approx(3.0)       # TFLOP/s of the whole job


def test_single_process_aggregate():
    import bench

    c = bench.Control(1)
    total, t, value = bench.aggregate(c, 2e12, 0.5)
    assert (total, t, value) == (2e12, 0.5, 4.0)


def test_suite_covers_every_mode_and_the_unpadded_shapes():
    import synth

    modes = {synth.CONFIGS[k][0] for k in synth.SUITE}
    assert modes == {"ptpc", "blockscale", "mxfp8", "bf16"}
    ns = {synth.CONFIGS[k][2] for k in synth.SUITE}
    assert {6288, 3648, 6400, 7168, 896} <= ns
    assert synth.gemm_flops(32768, 6400, 7168) == pytest.approx(3006.5e9, rel=1e-4)
    assert synth.gemm_bytes("ptpc", 32768, 6400, 7168) == pytest.approx(700.3e6, rel=1e-3)
