"""The seeded input generator on the CPU (no GPU): every input format gives the
layout the C ABI and the oracle read, padding rows are zero with unit scales
and zero prob, the same seed gives the same bytes, and the named workloads'
routing has the stated structure (checked on the routing alone, which is
cheap: the full-size tensors are drawn on the GPU by the parity tests)."""
import numpy as np
import pytest
import torch

from block_scaled_grouped_gb300 import workloads as W

# (bytes per row of K elements, scale block length, scale code of 1.0)
LAYOUT = {"mxfp8_e4m3": (1.0, 32, 127), "mxfp8_e5m2": (1.0, 32, 127), "nvfp4": (0.5, 16, 0x38),
          "fp4_ue8m0_16": (0.5, 16, 127), "mxfp4": (0.5, 32, 127), "bf16": (2.0, None, None)}


@pytest.mark.parametrize("in_fmt", W.IN_FORMATS)
def test_layout_and_padding_of_every_format(in_fmt):
    counts = (70, 0, 130)
    p = W.build_problem(name="t", counts=counts, k=192, n=64, in_fmt=in_fmt, out_fmt="bf16", epi="gate",
                        seed=5, pad_to=128)
    per_elem, v, one = LAYOUT[in_fmt]
    assert p.m_pad == 128 + 0 + 256
    assert p.a.shape == (p.m_pad, int(192 * per_elem)) and p.a.dtype == torch.uint8
    assert p.b.shape == (3, 64, int(192 * per_elem))
    if v is None:
        assert p.sfa_rows.shape == (1, p.m_pad, 0) and p.sfb_rows.shape == (3, 64, 0)
    else:
        assert p.sfa_rows.shape == (1, p.m_pad, 192 // v) and p.sfb_rows.shape == (3, 64, 192 // v)
    assert p.padded_offsets.tolist() == [128, 128, 384]
    # padding rows: data 0, scale 1.0, prob 0; real rows: some nonzero data
    pad = np.r_[70:128, 258:384]
    assert torch.all(p.a[pad] == 0)
    assert torch.all(p.prob[pad] == 0)
    if v is not None:
        assert torch.all(p.sfa_rows[0, pad] == one)
    assert torch.any(p.a[:70] != 0) and torch.any(p.a[128:258] != 0)
    assert torch.all(p.prob[:70] > 0)


@pytest.mark.parametrize("in_fmt", ["mxfp8_e4m3", "nvfp4", "bf16"])
def test_same_seed_same_bytes(in_fmt):
    kw = dict(name="t", counts=(40, 90), k=128, n=64, in_fmt=in_fmt, out_fmt="bf16", epi="dswiglu", seed=9,
              pad_to=128)
    p, q = W.build_problem(**kw), W.build_problem(**kw)
    for a, b in ((p.a, q.a), (p.b, q.b), (p.sfa_rows, q.sfa_rows), (p.prob, q.prob), (p.saved_c, q.saved_c),
                 (p.beta, q.beta), (p.alpha, q.alpha)):
        assert torch.equal(a, b)
    r = W.build_problem(**dict(kw, seed=10))
    assert not torch.equal(p.b, r.b)


def test_bf16_bytes_are_the_rounded_values():
    x = torch.randn(5, 48, generator=torch.Generator().manual_seed(1))
    q, s = W.as_bf16_bytes(x)
    assert q.shape == (5, 96) and s.shape == (5, 0)
    assert torch.equal(q.view(torch.bfloat16).float(), x.to(torch.bfloat16).float())


def test_named_routings():
    # FC layers: 4096 tokens top-2 of 8 experts, each token once per expert
    tokens, probs = W.route_softmax_topk(4096, 8, 2, seed=0)
    assert sum(t.size for t in tokens) == 8192
    for t, pr in zip(tokens, probs):
        assert np.all(np.diff(t) > 0) and np.all((pr > 0) & (pr < 1))
    # fine-grained: 8192 tokens top-8 of 64 Zipf experts, four empty, one above 4096 rows
    z = W.route_zipf_gumbel_topk(8192, 64, 8, s=1.2, n_empty=4, seed=3)
    sizes = np.array([t.size for t in z])
    assert sizes.sum() == 8192 * 8 and (sizes == 0).sum() == 4 and sizes.max() > 4096
    # skewed: 65536 rows over 128 experts from Dirichlet(0.1), many empty
    d = W.dirichlet_sizes(65536, 128, 0.1, seed=4)
    assert sum(d) == 65536 and sum(1 for c in d if c == 0) > 20
