"""The seeded input generator on the CPU (no GPU): every input format gives the
layout the C ABI and the oracle read, padding rows are zero with unit scales
and zero prob, the same seed gives the same bytes, the quantizers follow the
input recipes (MXFP8: UE8M0 scale 2^ceil(log2(amax/q_max)) per 32; NVFP4: E4M3
scale RN(amax/6) per 16; FP4 with UE8M0 scales 2^ceil(log2(amax/6)); data the
nearest value, ties to even, checked by brute force), and the named workloads'
routing has the stated structure (checked on the routing alone, which is
cheap: the full-size tensors are drawn on the GPU by the parity tests)."""
import math

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


E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _nearest_e2m1(y):
    """Brute force: the nearest listed E2M1 magnitude, ties to the even code."""
    mag = abs(y)
    d = np.abs(E2M1 - min(mag, 6.0))
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if best.size == 1 or best[0] % 2 == 0 else int(best[1])
    return code | (8 if np.signbit(y) else 0)


def _blocks(x, v):
    R, K = x.shape
    return x.reshape(R, K // v, v)


@pytest.mark.parametrize("fmt,qmax", [("mxfp8_e4m3", 448.0), ("mxfp8_e5m2", 57344.0)])
def test_mxfp8_input_recipe(fmt, qmax):
    """Scale 2^ceil(log2(amax/q_max)) per 1x32 block (UE8M0), data the nearest
    FP8 value of x/scale, never above q_max (the workloads' MXFP8 recipe)."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(6, 128, generator=g) * torch.logspace(-6, 6, 6).reshape(6, 1)
    x[2, 32:64] = 0.0
    codes, sc = W.quantize_mxfp8(x, fmt)
    dt = torch.float8_e4m3fn if fmt == "mxfp8_e4m3" else torch.float8_e5m2
    vals = codes.view(dt).double().numpy()
    xb = _blocks(x.double().numpy(), 32)
    for r in range(6):
        for b in range(4):
            am = float(np.abs(xb[r, b]).max())
            if am == 0.0:
                assert sc[r, b] == 127 and np.all(vals[r, 32 * b:32 * b + 32] == 0)
                continue
            e = math.ceil(math.log2(am / qmax))
            assert int(sc[r, b]) == e + 127
            y = xb[r, b] / 2.0 ** e
            q = vals[r, 32 * b:32 * b + 32]
            assert np.all(np.abs(q) <= qmax)
            # the nearest representable value: within half a step (3 or 2 mantissa bits)
            half = 2.0 ** -4 if fmt == "mxfp8_e4m3" else 2.0 ** -3
            tiny = 2.0 ** -10 if fmt == "mxfp8_e4m3" else 2.0 ** -17
            assert np.all(np.abs(q - y) <= half * np.abs(y) + tiny)


def test_nvfp4_input_recipe():
    """Scale RN_e4m3(amax/6) per 1x16 block (the nearest E4M3 value, found by
    brute force over all positive codes), data the nearest E2M1 value of
    x/scale with ties to the even code, element 2i in the low nibble."""
    g = torch.Generator().manual_seed(4)
    x = torch.randn(4, 64, generator=g) * torch.tensor([[1e-2], [1.0], [30.0], [500.0]])
    packed, sc = W.quantize_nvfp4(x)
    e4m3 = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    xb = _blocks(x.numpy().astype(np.float32), 16)
    nib = np.stack([packed.numpy() & 0xF, packed.numpy() >> 4], axis=-1).reshape(4, 64)
    for r in range(4):
        for b in range(4):
            t = np.float32(np.abs(xb[r, b]).max()) / np.float32(6.0)
            d = np.abs(e4m3 - min(float(t), 448.0))
            near = np.flatnonzero(d == d.min())
            want = int(near[0]) if near.size == 1 or near[0] % 2 == 0 else int(near[1])
            assert int(sc[r, b]) == (want if want != 0 else 0x38)
            s = np.float32(e4m3[int(sc[r, b])])
            for j in range(16):
                y = float(np.float32(xb[r, b, j]) / s)
                assert nib[r, 16 * b + j] == _nearest_e2m1(y)


@pytest.mark.parametrize("v", [16, 32])
def test_fp4_ue8m0_input_recipe(v):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(3, 64, generator=g) * torch.tensor([[1e-3], [1.0], [1e3]])
    packed, sc = W.quantize_fp4_ue8m0(x, v)
    xb = _blocks(x.numpy().astype(np.float32), v)
    nib = np.stack([packed.numpy() & 0xF, packed.numpy() >> 4], axis=-1).reshape(3, 64)
    for r in range(3):
        for b in range(64 // v):
            am = float(np.abs(xb[r, b]).max())
            e = math.ceil(math.log2(am / 6.0))
            assert int(sc[r, b]) == e + 127
            for j in range(v):
                y = float(np.float32(xb[r, b, j]) / np.float32(2.0 ** e))
                assert nib[r, v * b + j] == _nearest_e2m1(y)
