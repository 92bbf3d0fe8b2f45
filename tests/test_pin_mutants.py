"""Do the oracle's pins catch plausible mistakes?  (CPU only.)

Each case below plants ONE plausible mistake in a copy of the oracle's C++
source (a dropped term, a wrong sign, bias or index, a swapped operand or
block, a rounding rule turned the wrong way), compiles the copy into a
temporary shared object, and runs the oracle's pin suite
(``tests/test_oracle_*.py``: closed forms, brute force, invariants, the
hand-worked examples, library decodings) against it in a subprocess.  The case
passes when the pin suite FAILS on the copy: a mistake that every pin lets
through marks a part of the oracle whose pins are too weak.

Two kinds of mistake are left out on purpose.  Swapping the nibble order of
the FP4 INPUTS changes nothing observable: both operands go through the same
decoder, so every dot product only sees k permuted within a pair that shares
one scale (the packed OUTPUT's nibble order is a case below).  A wrong size of
a scale buffer writes out of bounds in the copy itself rather than giving a
wrong value; every planted index stays inside its buffer, so that a copy
fails by its values and never by corrupting its own memory.

The oracle in the repository is never modified: the mistakes live in
temporary copies only.  A control case compiles the unmodified source through
the same path and requires the pin suite to pass on it, so that a broken
harness cannot pass for a caught mistake.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

import pytest

import oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, exact text in the oracle source, text that replaces it)
MUTANTS = [
    # -- number formats ("Grouped GEMM + Quant (SM100)", Data Types) --
    ("e4m3 exponent bias 8", "else v = std::ldexp(1.0 + m / 8.0, e - 7);",
     "else v = std::ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3 subnormal exponent", "if (e == 0) v = std::ldexp(m / 8.0, -6);",
     "if (e == 0) v = std::ldexp(m / 8.0, -7);"),
    ("e5m2 exponent bias 16", "else v = std::ldexp(1.0 + m / 4.0, e - 15);",
     "else v = std::ldexp(1.0 + m / 4.0, e - 16);"),
    ("e2m1 subnormal 1.0", "double v = (e == 0) ? 0.5 * m :", "double v = (e == 0) ? 1.0 * m :"),
    ("ue8m0 bias 126", "std::ldexp(1.0, int(c) - 127)", "std::ldexp(1.0, int(c) - 126)"),
    ("rne ties go down", "else pick = (lo % 2 == 0) ? lo : hi;", "else pick = lo;"),
    ("overflow to the NaN code", "if (ax >= decode(fmt, top)) return sgn | top;",
     "if (ax >= decode(fmt, top)) return sgn | (top + 1);"),
    ("ue8m0 one step up at exact powers", "int e = (m == 0.5) ? p - 1 : p;", "int e = p;"),
    ("ue8m0 rounds down", "int e = (m == 0.5) ? p - 1 : p;", "int e = p - 1;"),
    ("e5m2 infinity decoded as NaN", "if (e == 0x1F) v = (m == 0) ? INFINITY : NAN;", "if (e == 0x1F) v = NAN;"),
    ("ue8m0 0xFF decoded as a number", "return c == 0xFF ? NAN : std::ldexp(1.0, int(c) - 127);",
     "return std::ldexp(1.0, int(c) - 127);"),
    ("ue8m0 encoder overflows to the NaN code", "return uint32_t(std::min(254, std::max(0, code)));",
     "return uint32_t(std::min(255, std::max(0, code)));"),
    ("ue8m0 zero block encoded as 1.0", "if (!(sf > 0.0f)) return 0;", "if (!(sf > 0.0f)) return 127;"),
    # -- scale-factor layout ("Grouped GEMM + Quant (SM100)", Shapes) --
    ("sf layout i0/i1 swapped", "* 32 + i0) * 4 + i1) * 4 + i3;", "* 32 + i1) * 4 + i0) * 4 + i3;"),
    ("sf layout row/k tiles swapped", "return ((((l * R + i2) * KQ + i4)", "return ((((l * KQ + i4) * R + i2)"),
    ("sf vector 32 for UE8M0/16 FP4", "return (P->in_fmt == IN_NVFP4 || P->in_fmt == IN_FP4_UE8M0_16) ? 16 : 32;",
     "return (P->in_fmt == IN_NVFP4) ? 16 : 32;"),
    ("bf16 bytes big-endian", "(uint32_t(two_bytes[0]) | (uint32_t(two_bytes[1]) << 8)) << 16",
     "(uint32_t(two_bytes[1]) | (uint32_t(two_bytes[0]) << 8)) << 16"),
    # -- grouping and the GEMM (Equations, Step 1) --
    ("group boundary inclusive", "if (m >= start && m < off[g]) return g;",
     "if (m >= start && m <= off[g]) return g;"),
    ("B of group 0 for every group", "dequant_row(P, J.B + g * b_group_bytes, J.SFB, n, P->n, g, brow.data());",
     "dequant_row(P, J.B, J.SFB, n, P->n, g, brow.data());"),
    ("SFB of group 0 for every group", "sf[sf_offset(row, k / v, l, rows, kblocks)]",
     "sf[sf_offset(row, k / v, 0, rows, kblocks)]"),
    ("alpha dropped", "(is_bwd(P) ? a * a : a) * acc", "(is_bwd(P) ? a * a : 1.0) * acc"),
    ("backward alpha not squared", "(is_bwd(P) ? a * a : a) * acc", "(is_bwd(P) ? a : a) * acc"),
    ("bias of group 0", "c += double(J.bias[g * P->n + n]);", "c += double(J.bias[n]);"),
    ("bias scaled by alpha", "c += double(J.bias[g * P->n + n]);",
     "c += double(J.alpha[g]) * double(J.bias[g * P->n + n]);"),
    ("C stored before the bias",
     "if (J.bias) c += double(J.bias[g * P->n + n]);\n      if (J.c_ref) J.c_ref[size_t((bi * 32 + i) * P->n + n)] = c;",
     "if (J.c_ref) J.c_ref[size_t((bi * 32 + i) * P->n + n)] = c;\n      if (J.bias) c += double(J.bias[g * P->n + n]);"),
    ("prob of the row within the block", "const double p = J.prob[m];", "const double p = J.prob[i];"),
    # -- forward epilogue (Step 2; SwiGLU, sReLU and GLU pages) --
    ("gating prob dropped", "d = p * Cv(j);", "d = Cv(j);"),
    ("sigmoid sign", "return 1.0 / (1.0 + std::exp(-x));", "return 1.0 / (1.0 + std::exp(x));"),
    ("swiglu blocks swapped", "return 64 * b + (second ? 32 : 0) + r;", "return 64 * b + (second ? 0 : 32) + r;"),
    ("swiglu operand roles swapped", "d = p * x * (gt * orc_sigmoid(gt));", "d = p * gt * (x * orc_sigmoid(x));"),
    ("geglu slope 1", "orc_sigmoid(1.702 * g)", "orc_sigmoid(g)"),
    ("geglu +1 dropped", "return (u + 1.0) * g *", "return u * g *"),
    ("glu limit upper only on the gate", "gt = std::min(std::max(gt, -P->glu_limit), P->glu_limit);",
     "gt = std::min(gt, P->glu_limit);"),
    ("glu alpha dropped", "d *= P->glu_alpha;", "d *= 1.0;"),
    ("glu limit upper only on the input", "x = std::min(std::max(x, -P->glu_limit), P->glu_limit);",
     "x = std::min(x, P->glu_limit);"),
    ("srelu as square of |C|", "double r = c > 0.0 ? c : 0.0;", "double r = c > 0.0 ? c : -c;"),
    ("srelu clamp without s", "r = s * std::min(std::tanh(r / s), 1.0);", "r = std::min(std::tanh(r / s), 1.0);"),
    ("srelu prob inside the square", "d = p * orc_srelu(Cv(j), P->tanh_clamp_s);",
     "d = orc_srelu(p * Cv(j), P->tanh_clamp_s);"),
    ("amax without abs", "std::max(amax_local[size_t(amax_idx)], std::fabs(float(d)));",
     "std::max(amax_local[size_t(amax_idx)], float(d));"),
    # -- output quantization (Step 3) --
    ("e4m3 q_max 240", "return P->out_fmt == OUT_E4M3 ? 448.0 :", "return P->out_fmt == OUT_E4M3 ? 240.0 :"),
    ("norm dropped from the scale factor", "const float sf = (norm * amax_blk) * rcp_max;",
     "const float sf = amax_blk * rcp_max;"),
    ("norm dropped from the data scale", "? 0.0f : norm / sfd;\n  return b;", "? 0.0f : 1.0f / sfd;\n  return b;"),
    ("row SFD of the first 128-row tile", "J.sfd_row[sf_offset(m, jb / v, 0, P->m_pad, kb_row)]",
     "J.sfd_row[sf_offset(m % 128, jb / v, 0, P->m_pad, kb_row)]"),
    ("column amax without abs", "if (grp[size_t(i)] >= 0) am = std::max(am, std::fabs(Dv(i, j)));",
     "if (grp[size_t(i)] >= 0) am = std::max(am, Dv(i, j));"),
    ("column SFD of the tile's first block", "J.sfd_col[sf_offset(j, (m0 + ib) / v, 0, nd, kb_col)]",
     "J.sfd_col[sf_offset(j, m0 / v, 0, nd, kb_col)]"),
    ("row amax without abs", "for (int64_t j = jb; j < je; ++j) am = std::max(am, std::fabs(Dv(i, j)));",
     "for (int64_t j = jb; j < je; ++j) am = std::max(am, Dv(i, j));"),
    ("e5m2 q_max 61440", "OUT_E5M2 ? 57344.0 : 6.0;", "OUT_E5M2 ? 61440.0 : 6.0;"),
    ("e2m1 q_max 4", "OUT_E5M2 ? 57344.0 : 6.0;", "OUT_E5M2 ? 57344.0 : 4.0;"),
    ("UE8M0 rule for E4M3 output scales",
     "b.code = (sf_fmt(P) == F_UE8M0) ? encode_ue8m0_ceil(sf) : encode_rne_satfinite(F_E4M3, sf);",
     "b.code = encode_ue8m0_ceil(sf);"),
    ("packed E2M1 output nibbles swapped", "if (j % 2 == 0) byte = uint8_t((byte & 0xF0) | (code & 0xF));",
     "if (j % 2 == 1) byte = uint8_t((byte & 0xF0) | (code & 0xF));"),
    # -- Hadamard output (GLU + Hadamard + Quant page) --
    ("bf16 rounding one bit short", "const int q = std::max(p - 8, -133);", "const int q = std::max(p - 9, -133);"),
    ("hadamard sign flipped", "return (bits % 2) ? -1.0 : 1.0;", "return (bits % 2) ? 1.0 : -1.0;"),
    ("rowwise rht of unrounded D", "x[t] = orc_round_bf16(D[size_t(i * w + (jb - j0) + t)]);",
     "x[t] = D[size_t(i * w + (jb - j0) + t)];"),
    ("colwise rht row-major", "const int64_t e = nd * start + j * em + t0 + t;",
     "const int64_t e = nd * start + (t0 + t) * nd + j;"),
    ("colwise rht scales without the expert's segment offset", "J.sfrht[nd * start / 16 + sf_offset(",
     "J.sfrht[sf_offset("),
    ("colwise rht q_max 4", "\n        const float sf = (norm * am) * float(1.0 / 6.0);",
     "\n        const float sf = (norm * am) * float(1.0 / 4.0);"),
    ("rowwise rht scale without rht_norm", "\n          const float sf = (norm * am) * float(1.0 / 6.0);",
     "\n          const float sf = am * float(1.0 / 6.0);"),
    ("rowwise rht E2M1 nibbles swapped", "if ((jb + t) % 2 == 0) byte = uint8_t((byte & 0xF0) | (c & 0xF));",
     "if ((jb + t) % 2 == 1) byte = uint8_t((byte & 0xF0) | (c & 0xF));"),
    ("colwise rht E2M1 nibbles swapped", "if (e % 2 == 0) byte = uint8_t((byte & 0xF0) | (c & 0xF));",
     "if (e % 2 == 1) byte = uint8_t((byte & 0xF0) | (c & 0xF));"),
    # -- backward (dGLU page) --
    ("dswiglu beta dropped", "return scale_c ? double(J.beta[g]) * c : c;", "return c;"),
    ("dswiglu d input without prob", "if (is_input) d = ref * p * (gt * sg);", "if (is_input) d = ref * (gt * sg);"),
    ("dswiglu d gate derivative", "else d = ref * p * x * sg * (1.0 + gt * (1.0 - sg));",
     "else d = ref * p * x * sg * (1.0 + gt * sg);"),
    ("dswiglu dprob without G", "+= x * (gt * orc_sigmoid(gt)) * Cv(jr);", "+= x * orc_sigmoid(gt) * Cv(jr);"),
    ("saved C blocks ignore gate_first",
     "const bool second = (gate != bool(P->gate_first));\n      const double c",
     "const bool second = gate;\n      const double c"),
    ("backward blocks swapped", "const bool is_input = (second == bool(P->gate_first));",
     "const bool is_input = (second != bool(P->gate_first));"),
    ("backward amax halves swapped", "amax_idx = 2 * g + (is_input ? 0 : 1);", "amax_idx = 2 * g + (is_input ? 1 : 0);"),
    ("dgeglu slope dropped in the derivative", "(1.0 + P->geglu_alpha * gc * (1.0 - s))", "(1.0 + gc * (1.0 - s))"),
    ("dgeglu linear offset dropped", "d_gate = ref * p * (uc + P->linear_offset)", "d_gate = ref * p * (uc)"),
    ("dgeglu up mask dropped",
     "const double up_mask = (P->glu_clamp_min <= up && up <= P->glu_clamp_max) ? 1.0 : 0.0;",
     "const double up_mask = 1.0;"),
    ("dsitu b1 dropped in the derivative", "+ b1 * th_g * sg * (1.0 - sg);", "+ th_g * sg * (1.0 - sg);"),
    ("dbias of group 0", "J.dbias[g * nd + j] += D[", "J.dbias[j] += D["),
    ("dgeglu gate not clamped", "const double gc = std::min(gate, P->glu_clamp_max);", "const double gc = gate;"),
    ("dgeglu up not clamped", "const double uc = std::min(std::max(up, P->glu_clamp_min), P->glu_clamp_max);",
     "const double uc = up;"),
    ("dgeglu gate mask dropped", "const double gate_mask = gate <= P->glu_clamp_max ? 1.0 : 0.0;",
     "const double gate_mask = 1.0;"),
    ("dgeglu dprob with prob", "dprob_term = ref * gc * s * (uc + P->linear_offset);",
     "dprob_term = ref * p * gc * s * (uc + P->linear_offset);"),
    ("dsitu up gradient without dT_u", "d_up = ref * p * t_g * dtu;", "d_up = ref * p * t_g;"),
    ("dsitu sech^2 as 1 - tanh", "const double dtu = 1.0 - th_u * th_u;", "const double dtu = 1.0 - th_u;"),
    ("dsitu dprob without T_u", "dprob_term = ref * t_g * t_u;", "dprob_term = ref * t_g;"),
    ("bf16 dgeglu without beta",
     "const bool scale_c = P->epi == EPI_DSWIGLU || (P->in_fmt == IN_BF16 && P->epi == EPI_DGEGLU);",
     "const bool scale_c = P->epi == EPI_DSWIGLU;"),
    ("dswiglu beta of group 0", "return scale_c ? double(J.beta[g]) * c : c;",
     "return scale_c ? double(J.beta[0]) * c : c;"),
    ("saved C row stride n", "J.saved_c[m * 2 * P->n + 64 * b", "J.saved_c[m * P->n + 64 * b"),
    ("dprob with prob", "+= x * (gt * orc_sigmoid(gt)) * Cv(jr);", "+= p * x * (gt * orc_sigmoid(gt)) * Cv(jr);"),
    ("dprob of the last column slice only", "J.dprob_ref[size_t(bi * 32 + i)] += dprob_local[size_t(i)];",
     "J.dprob_ref[size_t(bi * 32 + i)] = dprob_local[size_t(i)];"),
    ("dsitu b2 dropped", "t_u = b2 * th_u;", "t_u = th_u;"),
]

PIN_FILES = sorted(glob.glob(os.path.join(ROOT, "tests", "test_oracle_*.py")))


def _run_pins(lib_path: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, BSGG_ORACLE_LIB=lib_path, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider", *PIN_FILES]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=180)


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    src = open(orc.source_path()).read()
    work = tmp_path_factory.mktemp("oracle_mutants")
    cases = [("control", None, None)] + MUTANTS

    def one(idx_case):
        idx, (name, old, new) = idx_case
        text = src
        if old is not None:
            assert src.count(old) == 1, f"{name}: the planted text must occur exactly once in the source"
            text = src.replace(old, new)
        cpp = os.path.join(work, f"m{idx}.cpp")
        so = os.path.join(work, f"m{idx}.so")
        with open(cpp, "w") as f:
            f.write(text)
        orc.compile_source(cpp, so)
        try:
            r = _run_pins(so)
        except subprocess.TimeoutExpired:
            return name, "timeout", ""
        return name, r.returncode, (r.stdout + r.stderr)[-2000:]

    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with cf.ThreadPoolExecutor(workers) as ex:
        res = list(ex.map(one, enumerate(cases)))
    return {name: (rc, log) for name, rc, log in res}


def test_control_copy_passes_the_pins(outcomes):
    rc, log = outcomes["control"]
    assert rc == 0, "the unmodified oracle, built by the harness, must pass its pins:\n" + log


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(outcomes, name):
    rc, log = outcomes[name]
    assert rc != "timeout", f"the pin suite did not finish on the planted mistake '{name}'"
    assert rc != 0, f"no pin caught the planted mistake '{name}'"
