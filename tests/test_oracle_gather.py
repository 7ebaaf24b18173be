"""Pins for the oracle's gather-GEMM (no GPU).

The GEMM under the gather is the ptpc oracle, pinned elsewhere; these tests pin
the gather around it against properties the definition fixes: the identity
gather is the plain GEMM, a permutation of source rows permutes the output
rows (with their per-row scales), repeated indices give repeated rows, and an
index that names no row gives a zero row.  One more test plants a plausible
mistake in the gather (the scale taken from the output row instead of the
source row) and checks that a pin catches it.  Cited: ROCm/aiter PR 6539,
Technical Details (gather_kv_b_proj: rows gathered by index, then projected).
"""
import numpy as np
import pytest

import oracle
import synth


def _plain(case):
    A, idx, B, sa, sb = case.numpy()
    return A, B, sa, sb


def test_identity_gather_is_the_plain_gemm():
    c = synth.make_gather_case(96, 96, 80, 256, seed=1, page=8)
    A, B, sa, sb = _plain(c)
    idx = np.arange(96, dtype=np.int32)
    Rg, refg = oracle.gemm_gather(A, idx, B, sa, sb)
    Rp, refp = oracle.gemm("ptpc", A, B, sa, sb)
    assert np.array_equal(refg, refp)
    assert np.array_equal(Rg, Rp)


def test_permutation_permutes_rows_with_their_scales():
    c = synth.make_gather_case(64, 64, 48, 128, seed=2)
    A, B, sa, sb = _plain(c)
    assert np.unique(sa).size > 32  # per-row scales differ, so a wrong scale shows
    perm = np.random.default_rng(3).permutation(64).astype(np.int32)
    _, refg = oracle.gemm_gather(A, perm, B, sa, sb)
    _, refp = oracle.gemm("ptpc", A, B, sa, sb)
    assert np.array_equal(refg, refp[perm])


def test_repeated_indices_give_repeated_rows():
    c = synth.make_gather_case(32, 200, 64, 128, seed=4)
    A, B, sa, sb = _plain(c)
    idx = np.array([7, 7, 199, 0, 7, 199] * 5 + [3, 3], dtype=np.int32)
    _, ref = oracle.gemm_gather(A, idx, B, sa, sb)
    assert np.array_equal(ref[0], ref[1]) and np.array_equal(ref[0], ref[4])
    assert np.array_equal(ref[2], ref[5])
    _, one = oracle.gemm("ptpc", A[[7, 199, 0, 3]], B, sa[[7, 199, 0, 3]], sb)
    assert np.array_equal(ref[0], one[0]) and np.array_equal(ref[2], one[1])
    assert np.array_equal(ref[3], one[2]) and np.array_equal(ref[-1], one[3])


def test_index_outside_the_source_gives_a_zero_row():
    c = synth.make_gather_case(16, 50, 32, 64, seed=5, page=8)
    A, B, sa, sb = _plain(c)
    idx = np.array([0, -1, 49, 50, 2**31 - 1, -(2**31), 1, 10] * 2, dtype=np.int64)
    R, ref = oracle.gemm_gather(A, idx, B, sa, sb)
    bad = (idx < 0) | (idx >= 50)
    # zero rows: scale 0 times the row's sum, so +0 or -0 by the sum's sign
    assert np.all(oracle.bits_to_f64(ref[bad]) == 0.0) and np.all(R[bad] == 0.0)
    assert np.all(np.any(oracle.bits_to_f64(ref[~bad]) != 0.0, axis=1))


def test_points_match_rows():
    c = synth.make_gather_case(128, 1024, 96, 192, seed=6)
    A, idx, B, sa, sb = c.numpy()
    _, ref = oracle.gemm_gather(A, idx, B, sa, sb)
    rng = np.random.default_rng(7)
    ms, ns = rng.integers(0, 128, 300), rng.integers(0, 96, 300)
    _, pts = oracle.gemm_gather_points(A, idx, B, sa, sb, ms, ns)
    assert np.array_equal(pts, ref[ms, ns])


def test_paged_indices_are_distinct_rows_in_page_runs():
    import torch

    g = torch.Generator("cpu")
    g.manual_seed(8)
    idx = synth.paged_indices(5000, 65536, 64, g).numpy()
    assert idx.shape == (5000,) and idx.min() >= 0 and idx.max() < 65536
    assert np.unique(idx).size == idx.size
    d = np.diff(idx.astype(np.int64))
    assert np.mean(d == 1) > 0.9  # rows run in order inside a page


def test_a_planted_scale_mistake_is_caught(monkeypatch):
    # the mistake: take the per-row scale of the OUTPUT row instead of the source row
    def wrong(A_src, idx, B, sa_src, sb, rows=None, want_r=True):
        src, valid = oracle.gather_source(idx, A_src.shape[0])
        sa = np.where(valid, np.asarray(sa_src)[: len(src)], np.float32(0)).astype(np.float32)
        return oracle.gemm("ptpc", np.asarray(A_src)[src], B, sa, sb, rows=rows, want_r=want_r)

    monkeypatch.setattr(oracle, "gemm_gather", wrong)
    with pytest.raises(AssertionError):
        test_permutation_permutes_rows_with_their_scales()
