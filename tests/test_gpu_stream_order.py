"""Stream order across back-to-back launches on one stream, with no host
synchronisation between them.

Every kernel may be scheduled while the kernel before it in the stream is still
running (programmatic dependent launch) but touches global memory only after that
kernel has completed, so the launches must behave exactly as plain stream-ordered
launches.  The pattern is ROCm/mori PR 809's, Worth a reviewer's attention: calls
back to back with no host synchronisation, where a buffer must not be refilled
before every reader of the previous call has read it.  Each case makes an early
start visible if it happened:

* read after write: a bf16 GEMM whose A is the output of the GEMM launched just
  before it (that output NaN-poisoned beforehand);
* write after read: a GEMM whose output overwrites the A operand of the GEMM
  launched just before it (ptpc, blockscale, mxfp8), or the source cache of a
  gather-GEMM;
* one mxfp8 plan launched twice in a row with different scales: the second
  launch's scale-record kernel rewrites the workspace the first launch's GEMM reads;
* every kernel of the path (ptpc, bf16, blockscale, mxfp8, gather) chained ten
  times over in one CUDA graph, replayed twice.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from checker import check

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import gpu_util

    gpu_util.lib_ready()
    from fp8_scaled_gemm_sm_gb300 import binding

    return binding


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def test_gemm_reads_the_output_of_the_gemm_before_it(b):
    # C1 = A1 B1^T (bf16, long enough to still run when the next launch starts),
    # then C2 = C1 B2^T reading C1 as its A.  The reference chains the oracle on
    # its own C1; the two C1 differ at most in a last bf16 bit, far inside the bound.
    M, K1, N1, N2 = 4096, 4096, 1024, 512
    c1 = synth.make_case("bf16", M, N1, K1, seed=11)
    c2 = synth.make_case("bf16", M, N2, N1, seed=12)  # its B only; A is C1
    dev = torch.device("cuda")
    A1, B1, B2 = c1.A.to(dev), c1.B.to(dev), c2.B.to(dev)
    C1 = torch.empty((M, N1), dtype=torch.int16, device=dev)
    C2 = torch.empty((M, N2), dtype=torch.int16, device=dev)
    _, ref1 = oracle.gemm("bf16", *c1.numpy(), want_r=False)
    _, ref2 = oracle.gemm("bf16", ref1, c2.numpy()[1], None, None, want_r=False)
    h1 = b.scaled_gemm_create("bf16", N1, K1, M)
    h2 = b.scaled_gemm_create("bf16", N2, N1, M)
    try:
        for rep in range(5):
            C1.fill_(NAN_BF16)
            C2.fill_(NAN_BF16)
            s = torch.cuda.current_stream().cuda_stream
            b.scaled_gemm_launch(h1, A1.data_ptr(), B1.data_ptr(), 0, 0, C1.data_ptr(), M, s)
            b.scaled_gemm_launch(h2, C1.data_ptr(), B2.data_ptr(), 0, 0, C2.data_ptr(), M, s)
            torch.cuda.synchronize()
            r = check(C1.cpu().numpy().view(np.uint16), ref1)
            assert r["ok"], (rep, r)
            r = check(C2.cpu().numpy().view(np.uint16), ref2)
            assert r["ok"], (rep, r)
        for h in (h1, h2):
            assert b.scaled_gemm_debug_status(h)[0] == 0
    finally:
        b.scaled_gemm_destroy(h1)
        b.scaled_gemm_destroy(h2)


@pytest.mark.parametrize("mode", ["ptpc", "blockscale", "mxfp8"])
def test_gemm_output_overwrites_the_input_of_the_gemm_before_it(b, mode):
    # C1 = op(A1, B1) runs first (mxfp8: its scale-record kernel, then the GEMM);
    # the next launch (bf16) writes its output over A1's bytes.  C1 must match the
    # oracle on the original A1.
    M, N1, K1 = 4096, 1024, 4096
    c1 = synth.make_case(mode, M, N1, K1, seed=21, b_std=0.02)
    dev = torch.device("cuda")
    A1, B1, sa1, sb1 = c1.A.to(dev), c1.B.to(dev), c1.sa.to(dev), c1.sb.to(dev)
    # bf16 GEMM whose output [M2, N2] covers A1's M x K1 bytes exactly
    M2, N2, K2 = M, K1 // 2, 256
    c2 = synth.make_case("bf16", M2, N2, K2, seed=22)
    A2, B2 = c2.A.to(dev), c2.B.to(dev)
    C1 = torch.empty((M, N1), dtype=torch.int16, device=dev)
    h1 = b.scaled_gemm_create(mode, N1, K1, M)
    h2 = b.scaled_gemm_create("bf16", N2, K2, M2)
    _, ref1 = oracle.gemm(mode, *c1.numpy(), want_r=False)
    _, ref2 = oracle.gemm("bf16", *c2.numpy(), want_r=False)
    try:
        for rep in range(3):
            A1.copy_(c1.A.to(dev))
            C1.fill_(NAN_BF16)
            s = torch.cuda.current_stream().cuda_stream
            b.scaled_gemm_launch(h1, A1.data_ptr(), B1.data_ptr(), sa1.data_ptr(), sb1.data_ptr(), C1.data_ptr(), M, s)
            b.scaled_gemm_launch(h2, A2.data_ptr(), B2.data_ptr(), 0, 0, A1.data_ptr(), M2, s)
            torch.cuda.synchronize()
            r = check(C1.cpu().numpy().view(np.uint16), ref1)
            assert r["ok"], (rep, r)
            r = check(A1.view(torch.int16).cpu().numpy().view(np.uint16).reshape(M2, N2), ref2)
            assert r["ok"], (rep, r)
        for h in (h1, h2):
            assert b.scaled_gemm_debug_status(h)[0] == 0
    finally:
        b.scaled_gemm_destroy(h1)
        b.scaled_gemm_destroy(h2)


def test_gather_gemm_source_overwritten_by_the_next_launch(b):
    # the gather-GEMM reads its A rows with cp.async from the source cache; the next
    # launch (bf16) overwrites that cache.  The gathered result must be the oracle's
    # on the original cache.
    M, R, N, K = 4096, 8192, 1024, 2048
    g = synth.make_gather_case(M, R, N, K, seed=41, page=16)
    dev = torch.device("cuda")
    A_src, idx, B, sa, sb = (t.to(dev) for t in (g.A_src, g.idx, g.B, g.sa_src, g.sb))
    M2, N2, K2 = R, K // 2, 256  # bf16 output [R, K/2] covers the R x K source bytes
    c2 = synth.make_case("bf16", M2, N2, K2, seed=42)
    A2, B2 = c2.A.to(dev), c2.B.to(dev)
    C = torch.empty((M, N), dtype=torch.int16, device=dev)
    _, ref = oracle.gemm_gather(*g.numpy(), want_r=False)
    h1 = b.scaled_gemm_create("ptpc", N, K, M)
    h2 = b.scaled_gemm_create("bf16", N2, K2, M2)
    try:
        for rep in range(3):
            A_src.copy_(g.A_src.to(dev))
            C.fill_(NAN_BF16)
            s = torch.cuda.current_stream().cuda_stream
            b.scaled_gemm_launch_gather(h1, A_src.data_ptr(), R, idx.data_ptr(), B.data_ptr(), sa.data_ptr(),
                                        sb.data_ptr(), C.data_ptr(), M, s)
            b.scaled_gemm_launch(h2, A2.data_ptr(), B2.data_ptr(), 0, 0, A_src.data_ptr(), M2, s)
            torch.cuda.synchronize()
            r = check(C.cpu().numpy().view(np.uint16), ref)
            assert r["ok"], (rep, r)
        for h in (h1, h2):
            assert b.scaled_gemm_debug_status(h)[0] == 0
    finally:
        b.scaled_gemm_destroy(h1)
        b.scaled_gemm_destroy(h2)


def test_mxfp8_plan_launched_twice_in_a_row(b):
    # two launches of one mxfp8 plan with different operands and scales, back to
    # back: the second launch's record kernel must not rewrite the workspace
    # before the first launch's GEMM has finished reading it
    M, N, K = 4096, 2048, 1792
    cases = [synth.make_case("mxfp8", M, N, K, seed=31 + i, b_std=0.02) for i in range(2)]
    dev = torch.device("cuda")
    ops = [(c.A.to(dev), c.B.to(dev), c.sa.to(dev), c.sb.to(dev)) for c in cases]
    Cs = [torch.empty((M, N), dtype=torch.int16, device=dev) for _ in cases]
    refs = [oracle.gemm("mxfp8", *c.numpy(), want_r=False)[1] for c in cases]
    h = b.scaled_gemm_create("mxfp8", N, K, M)
    try:
        for rep in range(3):
            for C in Cs:
                C.fill_(NAN_BF16)
            s = torch.cuda.current_stream().cuda_stream
            for (A, B, sa, sb), C in zip(ops, Cs):
                b.scaled_gemm_launch(h, A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), M, s)
            torch.cuda.synchronize()
            for i, (C, ref) in enumerate(zip(Cs, refs)):
                r = check(C.cpu().numpy().view(np.uint16), ref)
                assert r["ok"], (rep, i, r)
        assert b.scaled_gemm_debug_status(h)[0] == 0
    finally:
        b.scaled_gemm_destroy(h)


def test_every_kernel_chained_in_a_cuda_graph(b):
    # ptpc, bf16, blockscale, mxfp8 (scale records + GEMM) and the gather-GEMM
    # launched in turn, 10 rounds, captured in one CUDA graph: every kernel
    # boundary of the path appears as a programmatic dependency in the graph.
    # After two replays every output matches the oracle and is bit-identical to
    # the first replay's.
    dev = torch.device("cuda")
    M, N, K = 512, 1024, 1024
    jobs = []
    for i, mode in enumerate(("ptpc", "bf16", "blockscale", "mxfp8")):
        c = synth.make_case(mode, M, N, K, seed=61 + i, b_std=0.02 if mode != "bf16" else 1.0)
        ops = [c.A.to(dev), c.B.to(dev)] + ([] if mode == "bf16" else [c.sa.to(dev), c.sb.to(dev)])
        C = torch.empty((M, N), dtype=torch.int16, device=dev)
        ref = oracle.gemm(mode, *c.numpy(), want_r=False)[1]
        jobs.append((mode, b.scaled_gemm_create(mode, N, K, M), ops, C, ref))
    g = synth.make_gather_case(M, 2048, N, K, seed=65, page=16)
    gops = [t.to(dev) for t in (g.A_src, g.idx, g.B, g.sa_src, g.sb)]
    gC = torch.empty((M, N), dtype=torch.int16, device=dev)
    gref = oracle.gemm_gather(*g.numpy(), want_r=False)[1]
    gh = b.scaled_gemm_create("ptpc", N, K, M)
    stream = torch.cuda.Stream()
    try:
        def launch_all():
            s = stream.cuda_stream
            for mode, h, ops, C, _ in jobs:
                sa = ops[2].data_ptr() if len(ops) > 2 else 0
                sb = ops[3].data_ptr() if len(ops) > 2 else 0
                b.scaled_gemm_launch(h, ops[0].data_ptr(), ops[1].data_ptr(), sa, sb, C.data_ptr(), M, s)
            A_src, idx, B, sa_src, sb = gops
            b.scaled_gemm_launch_gather(gh, A_src.data_ptr(), 2048, idx.data_ptr(), B.data_ptr(), sa_src.data_ptr(),
                                        sb.data_ptr(), gC.data_ptr(), M, s)

        with torch.cuda.stream(stream):
            launch_all()  # first use sets the plans' kernels up outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(10):
                launch_all()
        first = None
        for rep in range(2):
            for _, _, _, C, _ in jobs:
                C.fill_(NAN_BF16)
            gC.fill_(NAN_BF16)
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            outs = [C.cpu().numpy().view(np.uint16) for _, _, _, C, _ in jobs] + [gC.cpu().numpy().view(np.uint16)]
            refs = [ref for *_, ref in jobs] + [gref]
            names = [mode for mode, *_ in jobs] + ["gather"]
            for name, out, ref in zip(names, outs, refs):
                r = check(out, ref)
                assert r["ok"], (rep, name, r)
            if first is None:
                first = outs
            else:
                for name, a, c in zip(names, first, outs):
                    assert np.array_equal(a, c), name
        del graph
        for _, h, _, _, _ in jobs:
            assert b.scaled_gemm_debug_status(h)[0] == 0
        assert b.scaled_gemm_debug_status(gh)[0] == 0
    finally:
        for _, h, _, _, _ in jobs:
            b.scaled_gemm_destroy(h)
        b.scaled_gemm_destroy(gh)
