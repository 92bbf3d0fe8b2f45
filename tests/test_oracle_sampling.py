"""The oracle computes any list of 32-row blocks, which is how the full-size
GPU parity tests check the kernel on samples; its results must not depend on
which blocks are listed, in which order, or on how many threads compute them.

For a forward problem with row and column quantization, a forward problem with
the Hadamard outputs and a backward problem: a shuffled subset of the blocks
gives, row for row, the same D (fp64), the same quantized codes and scale
factors (rows of the listed blocks; whole 32-row column blocks) and the same
dprob as the run over every block; one thread and seven threads agree bit for
bit (dprob sums its per-slice terms in thread order: to 1e-13 relative)."""
import numpy as np
import pytest

import oracle as orc
from helpers import oracle_run, small_problem

CASES = {
    "fwd_e4m3_cols": dict(counts=(100, 0, 230, 64), k=96, n=384, epi="swiglu", out_fmt="e4m3", want_col=1,
                          pad_to=32, seed=71),
    "fwd_nvfp4_cols": dict(counts=(70, 130, 0, 50), k=128, n=256, in_fmt="nvfp4", epi="srelu",
                           out_fmt="e2m1", want_col=1, tanh_clamp_s=4.0, pad_to=32, seed=72),
    "bwd_dswiglu": dict(counts=(90, 0, 160), k=64, n=192, epi="dswiglu", out_fmt="e4m3", want_col=1, pad_to=32,
                        seed=73),
}


def _rows(blocks):
    return (np.asarray(blocks)[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)


@pytest.mark.parametrize("name", sorted(CASES))
def test_subset_of_blocks_matches_the_full_run(name):
    p = small_problem(**CASES[name])
    nb = p.m_pad // 32
    full = oracle_run(p, threads=3)
    rng = np.random.default_rng(0)
    sub = rng.permutation(nb)[: max(2, nb // 2)]
    part = oracle_run(p, blocks=sub, threads=2)
    rows = _rows(sub)
    # fp64 D of the listed rows, in the listed order
    assert np.array_equal(part["d_ref"], full["d_ref"][rows])
    if "dprob_ref" in full:
        np.testing.assert_allclose(part["dprob_ref"], full["dprob_ref"][rows], rtol=1e-13, atol=0)
    # quantized rows and their scale factors
    d_full, d_part = full["d"].reshape(p.m_pad, -1), part["d"].reshape(p.m_pad, -1)
    assert np.array_equal(d_part[rows], d_full[rows])
    kb = -(-p.n_out // p.sf_vec)
    offs = np.array([orc.sf_offset(r, j, 0, p.m_pad, kb) for r in rows for j in range(kb)])
    assert np.array_equal(part["sfd_row"][offs], full["sfd_row"][offs])
    # column outputs of the listed 32-row blocks
    c_full, c_part = full["d_col"].reshape(p.m_pad, -1), part["d_col"].reshape(p.m_pad, -1)
    assert np.array_equal(c_part[rows], c_full[rows])
    kbc = -(-p.m_pad // p.sf_vec)
    col_blocks = sorted({int(r) // p.sf_vec for r in rows})
    offs_c = np.array([orc.sf_offset(j, b, 0, p.n_out, kbc) for b in col_blocks for j in range(p.n_out)])
    assert np.array_equal(part["sfd_col"][offs_c], full["sfd_col"][offs_c])


def test_hadamard_outputs_of_a_subset_match_the_full_run():
    p = small_problem(counts=(64, 128, 0, 64), k=64, n=256, in_fmt="nvfp4", epi="swiglu", out_fmt="e2m1",
                      pad_to=64, seed=74)
    for rht in ("e2m1", "col_e2m1"):
        full = oracle_run(p, rht=rht, rht_norm=1.0, threads=3)
        sub = np.array([3, 0, 5], dtype=np.int64)
        part = oracle_run(p, blocks=sub, rht=rht, rht_norm=1.0, threads=1)
        assert np.array_equal(part["rht_ref"], full["rht_ref"][_rows(sub)])
        if rht == "e2m1":
            rq_full = full["rht_q"].reshape(p.m_pad, -1)
            rq_part = part["rht_q"].reshape(p.m_pad, -1)
            assert np.array_equal(rq_part[_rows(sub)], rq_full[_rows(sub)])


@pytest.mark.parametrize("name", sorted(CASES))
def test_thread_count_does_not_change_results(name):
    p = small_problem(**CASES[name])
    one, many = oracle_run(p, threads=1), oracle_run(p, threads=7)
    for key in ("d_ref", "d", "d_col", "sfd_row", "sfd_col", "amax"):
        assert np.array_equal(one[key], many[key]), key
    if "dprob_ref" in one:
        np.testing.assert_allclose(many["dprob_ref"], one["dprob_ref"], rtol=1e-13, atol=0)
        np.testing.assert_allclose(many["dbias"], one["dbias"], rtol=1e-12, atol=1e-12)
