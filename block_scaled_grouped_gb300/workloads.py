"""Seeded synthetic MoE-shaped inputs for the grouped block-scaled GEMM.

This module is the one input generator that the tests, the smoke check and the
benchmark share.  It holds the input recipe only -- routing, value draws and
the quantization of those draws into MXFP8 / FP4 codes or bfloat16 -- and none of the
operation's own arithmetic (no GEMM, no epilogue, no output quantization, no
scale-factor layout: scale factors leave here row-major and are packed by each
consumer with its own packer).

Five named workloads follow the expert-layer shapes of the pages' MoE use:

1. ``tiny``      L=2, groups 128 and 256 rows, K=N=256, MXFP8 -> BF16 + amax
2. ``fc1_swiglu`` 4096 tokens top-2 of 8 experts, K=4096, N=28672, SwiGLU, E4M3 out
3. ``fc2_gate``  same routing, K=14336, N=4096, gating, BF16 out + amax
4. ``fine_nvfp4`` 8192 tokens top-8 of 64 Zipf(1.2) experts, K=7168, N=2048,
                 NVFP4 in, sReLU with tanh clamp s=8, NVFP4 out
5. ``skewed``    L=128, 65536 rows sized by Dirichlet(0.1), K=7168, N=4096,
                 sReLU, E4M3 row + column outputs, norm_const 0.5

and two backward ones, the dSwiGLU backward of the FC1 layer (routing of 2,
K=4096, N=14336, saved C 28672 wide): ``fc1_dswiglu`` (MXFP8 in, E4M3 row and
column outputs) and ``fc1_dswiglu_bf16`` (the BF16 backend: bfloat16 in and out).

Routing and per-group/per-row scalars are drawn with numpy's PCG64 from the
workload's seed (CPU, device independent).  Matrix values are drawn with a
torch generator on the target device, in fixed-size chunks, each chunk with its
own derived seed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

IN_FORMATS = ("mxfp8_e4m3", "mxfp8_e5m2", "nvfp4", "fp4_ue8m0_16", "mxfp4", "bf16")
FP4_FORMATS = ("nvfp4", "fp4_ue8m0_16", "mxfp4")
OUT_FORMATS = ("bf16", "f16", "f32", "e4m3", "e5m2", "e2m1")
EPILOGUES = ("gate", "swiglu", "srelu", "geglu", "dswiglu", "dgeglu", "dsituglu")
BWD_EPILOGUES = ("dswiglu", "dgeglu", "dsituglu")

_ROW_CHUNK = 4096


@dataclasses.dataclass
class Problem:
    """One grouped GEMM call: shapes, formats and the input tensors."""
    name: str
    m_pad: int
    n: int
    k: int
    num_groups: int
    in_fmt: str
    out_fmt: str
    epi: str
    tanh_clamp_s: float
    want_col: bool
    norm_const: float
    counts: np.ndarray          # unpadded rows per group
    padded_offsets: torch.Tensor  # int32 (L,)
    alpha: torch.Tensor         # float32 (L,)
    prob: torch.Tensor          # float32 (m_pad,)
    a: torch.Tensor             # uint8 (m_pad, k or k/2; bf16: 2k bytes, little-endian values)
    sfa_rows: torch.Tensor      # uint8 (1, m_pad, k/v) scale codes, row-major (bf16: 0 columns)
    b: torch.Tensor             # uint8 (L, n, k or k/2 or 2k)
    sfb_rows: torch.Tensor      # uint8 (L, n, k/v) scale codes, row-major (bf16: 0 columns)
    # the backward epilogues' extra inputs (None otherwise): the saved forward
    # pre-activation C (m_pad, 2n) bf16 and its per-group scale beta (L,)
    saved_c: Optional[torch.Tensor] = None
    beta: Optional[torch.Tensor] = None

    @property
    def sf_vec(self) -> int:
        return 16 if self.in_fmt in ("nvfp4", "fp4_ue8m0_16") else 32

    @property
    def n_out(self) -> int:
        if self.epi in ("swiglu", "geglu"):
            return self.n // 2
        return 2 * self.n if self.epi in BWD_EPILOGUES else self.n

    @property
    def m_real(self) -> int:
        return int(self.counts.sum())

    @property
    def flops(self) -> float:
        """2 * valid rows * N * K: padding rows are excluded."""
        return 2.0 * self.m_real * self.n * self.k

    def describe(self) -> dict:
        return {"workload": self.name, "L": self.num_groups, "m_pad": self.m_pad,
                "m_real": self.m_real, "n": self.n, "k": self.k, "in": self.in_fmt,
                "out": self.out_fmt, "epilogue": self.epi, "tanh_clamp_s": self.tanh_clamp_s,
                "want_col": self.want_col, "norm_const": self.norm_const}


# --------------------------------------------------------------------------
# value draws
# --------------------------------------------------------------------------

def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) % (2 ** 62))
    return g


def _draw(rows: int, k: int, dist: str, device, seed: int, stream: int) -> torch.Tensor:
    g = _gen(device, seed, stream)
    x = torch.randn(rows, k, generator=g, device=device, dtype=torch.float32)
    if dist == "normal":
        return x
    if dist == "normal_over_k":          # N(0, 1/K)
        return x * (1.0 / math.sqrt(k))
    if dist == "abs_normal_x_normal":    # |N(0,1)| * N(0,1), two independent draws
        y = torch.randn(rows, k, generator=g, device=device, dtype=torch.float32)
        return x.abs() * y
    raise ValueError(dist)


# --------------------------------------------------------------------------
# input quantization (the input recipe, not the operation)
# --------------------------------------------------------------------------

def _pad_cols(x: torch.Tensor, mult: int) -> torch.Tensor:
    k = x.shape[1]
    kp = -(-k // mult) * mult
    if kp == k:
        return x
    return torch.nn.functional.pad(x, (0, kp - k))


def quantize_mxfp8(x: torch.Tensor, fmt: str):
    """float32 (R, K) -> (codes uint8 (R, K), scale codes uint8 (R, ceil(K/32))).

    One UE8M0 scale per 1x32 block, scale = 2^ceil(log2(amax/q_max)); data is the
    RNE cast of x/scale (torch's float8 conversion), clamped to +-q_max first.
    An all-zero block gets scale 1.0 (code 127) and zero data.
    """
    R, K = x.shape
    qmax = 448.0 if fmt == "mxfp8_e4m3" else 57344.0
    dt = torch.float8_e4m3fn if fmt == "mxfp8_e4m3" else torch.float8_e5m2
    xp = _pad_cols(x, 32)
    xb = xp.view(R, -1, 32)
    amax = xb.abs().amax(-1)
    mant, ex = torch.frexp(amax / qmax)
    e = torch.where(mant == 0.5, ex - 1, ex).to(torch.int32)
    e = torch.where(amax == 0, torch.zeros_like(e), e).clamp(-127, 127)
    scale = torch.ldexp(torch.ones_like(amax), e)
    q = (xb / scale.unsqueeze(-1)).clamp(-qmax, qmax).to(dt).view(torch.uint8)
    codes = q.reshape(R, -1)[:, :K].contiguous()
    return codes, (e + 127).to(torch.uint8)


def _e2m1_rne(y: torch.Tensor) -> torch.Tensor:
    """Round to the nearest E2M1 value {0,.5,1,1.5,2,3,4,6}, ties to the even
    code, saturating; returns 4-bit codes with the sign in bit 3."""
    mag = y.abs()
    code = ((mag > 0.25).to(torch.uint8) + (mag >= 0.75).to(torch.uint8)
            + (mag > 1.25).to(torch.uint8) + (mag >= 1.75).to(torch.uint8)
            + (mag > 2.5).to(torch.uint8) + (mag >= 3.5).to(torch.uint8)
            + (mag > 5.0).to(torch.uint8))
    return code | (torch.signbit(y).to(torch.uint8) << 3)


def quantize_nvfp4(x: torch.Tensor):
    """float32 (R, K) -> (packed codes uint8 (R, K/2), scale codes uint8 (R, ceil(K/16))).

    One E4M3 scale per 1x16 block, scale = RN_e4m3(amax/6); data is the E2M1
    RNE of x/scale.  Element 2i sits in the low nibble of byte i.  A block whose
    scale rounds to zero gets scale 1.0 (code 0x38).
    """
    R, K = x.shape
    assert K % 2 == 0
    xp = _pad_cols(x, 16)
    xb = xp.view(R, -1, 16)
    amax = xb.abs().amax(-1)
    s8 = (amax / 6.0).clamp(max=448.0).to(torch.float8_e4m3fn)
    sval = s8.to(torch.float32)
    zero = sval == 0
    scode = torch.where(zero, torch.full_like(s8.view(torch.uint8), 0x38), s8.view(torch.uint8))
    sval = torch.where(zero, torch.ones_like(sval), sval)
    codes = _e2m1_rne(xb / sval.unsqueeze(-1)).reshape(R, -1)[:, :K]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
    return packed, scode


def quantize_fp4_ue8m0(x: torch.Tensor, v: int):
    """float32 (R, K) -> (packed codes uint8 (R, K/2), scale codes uint8 (R, ceil(K/v))).

    One UE8M0 scale per 1xv block, scale = 2^ceil(log2(amax/6)) (so that every
    value lands inside E2M1's range), data the E2M1 RNE of x/scale; an all-zero
    block gets scale 1.0 (code 127).  Element 2i in the low nibble of byte i.
    """
    R, K = x.shape
    assert K % 2 == 0
    xp = _pad_cols(x, v)
    xb = xp.view(R, -1, v)
    amax = xb.abs().amax(-1)
    mant, ex = torch.frexp(amax / 6.0)
    e = torch.where(mant == 0.5, ex - 1, ex).to(torch.int32)
    e = torch.where(amax == 0, torch.zeros_like(e), e).clamp(-127, 127)
    scale = torch.ldexp(torch.ones_like(amax), e)
    codes = _e2m1_rne(xb / scale.unsqueeze(-1)).reshape(R, -1)[:, :K]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
    return packed, (e + 127).to(torch.uint8)


def as_bf16_bytes(x: torch.Tensor):
    """float32 (R, K) -> (bytes uint8 (R, 2K) of its round-to-nearest-even bfloat16
    values, little-endian; no scale codes: uint8 (R, 0))."""
    R, K = x.shape
    q = x.to(torch.bfloat16).contiguous().view(torch.uint8).reshape(R, 2 * K)
    return q, torch.empty(R, 0, dtype=torch.uint8, device=x.device)


def quantize(x: torch.Tensor, in_fmt: str):
    if in_fmt == "bf16":
        return as_bf16_bytes(x)
    if in_fmt == "nvfp4":
        return quantize_nvfp4(x)
    if in_fmt == "fp4_ue8m0_16":
        return quantize_fp4_ue8m0(x, 16)
    if in_fmt == "mxfp4":
        return quantize_fp4_ue8m0(x, 32)
    return quantize_mxfp8(x, in_fmt)


# --------------------------------------------------------------------------
# routing (numpy PCG64, device independent)
# --------------------------------------------------------------------------

def route_softmax_topk(T: int, L: int, topk: int, seed: int):
    """Softmax of N(0,1) router logits, top-k per token (ties to the lower
    expert index).  Returns per-expert token lists (token order) and the
    token's softmax probability for that expert."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((T, L))
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    p = z / z.sum(axis=1, keepdims=True)
    top = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    tokens, probs = [], []
    for g in range(L):
        t = np.nonzero((top == g).any(axis=1))[0]
        tokens.append(t)
        probs.append(p[t, g].astype(np.float32))
    return tokens, probs


def route_zipf_gumbel_topk(T: int, L: int, topk: int, s: float, n_empty: int, seed: int):
    """Zipf(s) expert popularity over a seeded permutation of the experts, the
    n_empty least popular set to zero weight; each token takes the top-k of
    log(weight) + Gumbel noise (distinct experts)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(L)
    w = np.zeros(L)
    ranks = np.arange(1, L + 1, dtype=np.float64)
    pop = ranks ** (-s)
    pop[L - n_empty:] = 0.0
    w[perm] = pop
    with np.errstate(divide="ignore"):
        logw = np.log(w)
    u = rng.random((T, L))
    gumbel = -np.log(-np.log(np.clip(u, 1e-300, 1.0 - 1e-16)))
    score = logw[None, :] + gumbel
    top = np.argsort(-score, axis=1, kind="stable")[:, :topk]
    tokens = [np.nonzero((top == g).any(axis=1))[0] for g in range(L)]
    return tokens


def _gamma_mt(rng: np.random.Generator, shape: float) -> float:
    """Gamma(shape, 1) by Marsaglia-Tsang; shape < 1 via the U^(1/shape) boost."""
    if shape < 1.0:
        return _gamma_mt(rng, shape + 1.0) * rng.random() ** (1.0 / shape)
    d = shape - 1.0 / 3.0
    c = 1.0 / math.sqrt(9.0 * d)
    while True:
        x = rng.standard_normal()
        v = (1.0 + c * x) ** 3
        if v <= 0:
            continue
        u = rng.random()
        if math.log(u) < 0.5 * x * x + d - d * v + d * math.log(v):
            return d * v


def dirichlet_sizes(total: int, L: int, conc: float, seed: int) -> np.ndarray:
    """Group sizes = largest-remainder rounding of total * Dirichlet(conc)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    gam = np.array([_gamma_mt(rng, conc) for _ in range(L)])
    frac = gam / gam.sum()
    raw = frac * total
    base = np.floor(raw).astype(np.int64)
    rem = total - int(base.sum())
    order = np.argsort(-(raw - base), kind="stable")
    base[order[:rem]] += 1
    return base


# --------------------------------------------------------------------------
# problem assembly
# --------------------------------------------------------------------------

def build_problem(*, name: str, counts: Sequence[int], k: int, n: int, in_fmt: str,
                  out_fmt: str, epi: str, seed: int, device="cpu",
                  a_dist: str = "normal", b_dist: str = "normal",
                  token_rows: Optional[List[np.ndarray]] = None, num_tokens: int = 0,
                  alpha=None, row_prob: Optional[List[np.ndarray]] = None,
                  norm_const: float = 1.0, tanh_clamp_s: float = 0.0,
                  want_col: bool = False, pad_to: int = 128) -> Problem:
    """Assemble a problem: group g holds counts[g] real rows followed by padding
    rows (A = 0, scale 1.0, prob = 0) up to a multiple of pad_to."""
    assert in_fmt in IN_FORMATS and out_fmt in OUT_FORMATS and epi in EPILOGUES
    counts = np.asarray(counts, dtype=np.int64)
    L = counts.size
    padded = -(-counts // pad_to) * pad_to
    offsets = np.cumsum(padded).astype(np.int64)
    m_pad = int(offsets[-1]) if L else 0
    rng = np.random.Generator(np.random.PCG64(seed))
    if alpha is None:
        alpha = rng.uniform(0.5, 2.0, size=L)
    alpha = np.asarray(alpha, dtype=np.float32)
    if row_prob is None:
        row_prob = [rng.uniform(0.0, 1.0, size=int(c)).astype(np.float32) for c in counts]

    v = 16 if in_fmt in ("nvfp4", "fp4_ue8m0_16") else 32
    kbytes = k // 2 if in_fmt in FP4_FORMATS else 2 * k if in_fmt == "bf16" else k
    kblocks = 0 if in_fmt == "bf16" else -(-k // v)
    prob = np.zeros(m_pad, dtype=np.float32)
    a = torch.zeros(m_pad, kbytes, dtype=torch.uint8, device=device)
    one_code = 0x38 if in_fmt == "nvfp4" else 127
    sfa = torch.full((1, m_pad, kblocks), one_code, dtype=torch.uint8, device=device)

    # Real-row positions in the padded layout.
    starts = np.concatenate([[0], offsets[:-1]]) if L else np.zeros(0, np.int64)
    pos = np.concatenate([starts[g] + np.arange(counts[g]) for g in range(L)]) if L else np.zeros(0, np.int64)
    for g in range(L):
        prob[starts[g]:starts[g] + counts[g]] = row_prob[g]

    # A values: routed token activations (token_rows) or independent rows.
    if token_rows is not None:
        src = np.concatenate([np.asarray(t, dtype=np.int64) for t in token_rows])
        X_rows = num_tokens
    else:
        src = np.arange(pos.size, dtype=np.int64)
        X_rows = pos.size
    # Quantize the source rows chunk by chunk, then scatter to their positions.
    codes_src = torch.empty(X_rows, kbytes, dtype=torch.uint8, device=device)
    sf_src = torch.empty(X_rows, kblocks, dtype=torch.uint8, device=device)
    for c0 in range(0, X_rows, _ROW_CHUNK):
        r = min(_ROW_CHUNK, X_rows - c0)
        x = _draw(r, k, a_dist, device, seed, 1 + c0 // _ROW_CHUNK)
        q, s = quantize(x, in_fmt)
        codes_src[c0:c0 + r] = q
        sf_src[c0:c0 + r] = s
    if pos.size:
        pos_t = torch.as_tensor(pos, device=device)
        src_t = torch.as_tensor(src, device=device)
        a[pos_t] = codes_src[src_t]
        sfa[0, pos_t] = sf_src[src_t]
    del codes_src, sf_src

    b = torch.empty(L, n, kbytes, dtype=torch.uint8, device=device)
    sfb = torch.empty(L, n, kblocks, dtype=torch.uint8, device=device)
    for g in range(L):
        for c0 in range(0, n, _ROW_CHUNK):
            r = min(_ROW_CHUNK, n - c0)
            x = _draw(r, k, b_dist, device, seed, 100_000 + g * 1000 + c0 // _ROW_CHUNK)
            q, s = quantize(x, in_fmt)
            b[g, c0:c0 + r] = q
            sfb[g, c0:c0 + r] = s

    # backward epilogues: the saved forward C, N(0, 2) rounded to bf16 (a
    # pre-activation's typical spread), and beta ~ U(0.5, 2) per group (read
    # by dSwiGLU, and by dGeGLU on bf16 inputs)
    saved_c = beta = None
    if epi in BWD_EPILOGUES:
        beta = torch.as_tensor(rng.uniform(0.5, 2.0, size=L).astype(np.float32), device=device)
        saved_c = torch.empty(m_pad, 2 * n, dtype=torch.bfloat16, device=device)
        for c0 in range(0, m_pad, _ROW_CHUNK):
            r = min(_ROW_CHUNK, m_pad - c0)
            saved_c[c0:c0 + r] = (_draw(r, 2 * n, "normal", device, seed, 200_000 + c0 // _ROW_CHUNK)
                                  * 2.0).to(torch.bfloat16)

    return Problem(
        name=name, m_pad=m_pad, n=n, k=k, num_groups=L, in_fmt=in_fmt, out_fmt=out_fmt, epi=epi,
        tanh_clamp_s=float(tanh_clamp_s), want_col=bool(want_col), norm_const=float(norm_const),
        counts=counts,
        padded_offsets=torch.as_tensor(offsets.astype(np.int32), device=device),
        alpha=torch.as_tensor(alpha, device=device),
        prob=torch.as_tensor(prob, device=device),
        a=a, sfa_rows=sfa, b=b, sfb_rows=sfb, saved_c=saved_c, beta=beta)


WORKLOADS = ("tiny", "fc1_swiglu", "fc2_gate", "fine_nvfp4", "skewed", "fc1_dswiglu", "fc1_dswiglu_bf16",
             "skinny")


def workload(name: str, device="cpu") -> Problem:
    """The five named workloads (seed = workload number - 1)."""
    if name == "tiny":
        # L=2, group rows 128 and 256 (offsets [128, 384]), K=N=256, MXFP8,
        # alpha [1, 0.5], prob ~ U(0,1), gating, BF16 D + amax.
        return build_problem(name=name, counts=[128, 256], k=256, n=256, in_fmt="mxfp8_e4m3",
                             out_fmt="bf16", epi="gate", seed=0, device=device,
                             alpha=[1.0, 0.5])
    if name in ("fc1_swiglu", "fc2_gate", "fc1_dswiglu", "fc1_dswiglu_bf16"):
        T, L = 4096, 8
        tokens, probs = route_softmax_topk(T, L, 2, seed=1)
        counts = [t.size for t in tokens]
        if name == "fc1_dswiglu":
            # the backward of the FC1 + SwiGLU layer: the routed output gradients
            # (K = 4096) against the down-projection weights (N = 14336, the
            # SwiGLU output width) give the gradient of the 28672-wide saved C;
            # E4M3 row and column outputs for the next GEMMs
            return build_problem(name=name, counts=counts, k=4096, n=14336, in_fmt="mxfp8_e4m3",
                                 out_fmt="e4m3", epi="dswiglu", seed=5, device=device,
                                 token_rows=tokens, num_tokens=T, row_prob=probs,
                                 norm_const=1.0, want_col=True)
        if name == "fc1_dswiglu_bf16":
            # the same backward on the BF16 backend: bfloat16 gradients and
            # weights, bfloat16 D_row (no column output or scales)
            return build_problem(name=name, counts=counts, k=4096, n=14336, in_fmt="bf16",
                                 out_fmt="bf16", epi="dswiglu", seed=6, device=device,
                                 token_rows=tokens, num_tokens=T, row_prob=probs)
        if name == "fc1_swiglu":
            return build_problem(name=name, counts=counts, k=4096, n=28672, in_fmt="mxfp8_e4m3",
                                 out_fmt="e4m3", epi="swiglu", seed=1, device=device,
                                 token_rows=tokens, num_tokens=T, row_prob=probs,
                                 norm_const=1.0, want_col=True)
        return build_problem(name=name, counts=counts, k=14336, n=4096, in_fmt="mxfp8_e4m3",
                             out_fmt="bf16", epi="gate", seed=2, device=device,
                             a_dist="abs_normal_x_normal", b_dist="normal_over_k",
                             token_rows=tokens, num_tokens=T, row_prob=probs)
    if name == "fine_nvfp4":
        T, L = 8192, 64
        tokens = route_zipf_gumbel_topk(T, L, 8, s=1.2, n_empty=4, seed=3)
        counts = [t.size for t in tokens]
        assert max(counts) > 4096 and min(counts) == 0
        return build_problem(name=name, counts=counts, k=7168, n=2048, in_fmt="nvfp4",
                             out_fmt="e2m1", epi="srelu", seed=3, device=device,
                             token_rows=tokens, num_tokens=T, tanh_clamp_s=8.0,
                             norm_const=1.0)
    if name == "skewed":
        counts = dirichlet_sizes(16384 * 4, 128, 0.1, seed=4)
        return build_problem(name=name, counts=counts, k=7168, n=4096, in_fmt="mxfp8_e4m3",
                             out_fmt="e4m3", epi="srelu", seed=4, device=device,
                             norm_const=0.5, want_col=True)
    if name == "skinny":
        # a decode-like step: 128 tokens routed top-8 over 64 experts (softmax of
        # N(0,1) router logits), about 16 rows per expert, each group padded to
        # 128 rows; the fine-grained layer's K = 7168, N = 2048 in MXFP8, gating,
        # BF16 D + amax.  Every expert's weights are read for a few rows, so the
        # launch is bound by HBM, not by the tensor cores.
        T, L = 128, 64
        tokens, probs = route_softmax_topk(T, L, 8, seed=7)
        counts = [t.size for t in tokens]
        return build_problem(name=name, counts=counts, k=7168, n=2048, in_fmt="mxfp8_e4m3",
                             out_fmt="bf16", epi="gate", seed=7, device=device,
                             token_rows=tokens, num_tokens=T, row_prob=probs)
    raise KeyError(name)
