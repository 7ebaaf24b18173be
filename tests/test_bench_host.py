"""Host-side logic of bench.py without a GPU: the replica control plane (gloo,
two ranks on the CPU), the whole-job throughput aggregation, and the rule that a
stored DRAM-traffic figure is reported only for the kernel sources it was
measured on."""
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


def _traffic_rows():
    import bench

    rows = []
    for line in open(os.path.join(bench.ROOT, "profiles", "traffic.txt")):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#"):
            rows.append((f[0], f[1], float(f[2])))
    return rows


def test_stored_traffic_applies_only_to_the_sources_it_was_measured_on(monkeypatch):
    # the roofline's DRAM traffic comes from a capture of one revision of a kernel's
    # sources; for any other revision it is not reported (null)
    import bench
    import synth

    rows = _traffic_rows()
    assert rows, "profiles/traffic.txt has no rows"
    for workload, rev, nbytes in rows:
        assert workload in synth.CONFIGS
        current = bench.kernel_revision(synth.CONFIGS[workload][0])
        assert bench.stored_traffic(workload) == (nbytes if rev == current else None)
    monkeypatch.setattr(bench, "kernel_revision", lambda mode="ptpc": "000000000000")
    assert all(bench.stored_traffic(w) is None for w, _, _ in rows)


def test_kernel_revision_hashes_each_family_s_own_sources():
    import bench

    revs = {m: bench.kernel_revision(m) for m in ("ptpc", "mxfp8", "blockscale")}
    assert len(set(revs.values())) == 3
    assert all(len(r) == 12 for r in revs.values())
    assert bench.kernel_revision("bf16") == revs["ptpc"]  # one kernel file for both
    assert revs == {m: bench.kernel_revision(m) for m in revs}
