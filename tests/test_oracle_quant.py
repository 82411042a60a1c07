"""Pins of the oracle's quantizer and packer (Q1-Q5).

What fixes the expected values, other than the oracle itself:
  - hand-worked cases in tests/golden/ (closed forms, ties, signs, subnormals),
  - brute force: each code is the grid point nearest to x among all 2^b codes
    with ties to the even code, computed in exact float64 arithmetic,
  - the error bound |x - x^| <= s/2 (plus the fp32 rounding of the quotient),
  - invariants: codes in range, min -> 0, max -> 2^b - 1, constant groups exact,
  - scale within half a binary16 ulp of (max - min) / (2^b - 1),
  - numpy's unpackbits as a second reading of the bit order.
"""

import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_cases(path):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        if tok[0] in ("case", "pack"):
            cur = {"name": tok[1] if tok[0] == "case" else "pack", "bits": int(tok[-1])}
            cases.append(cur)
            continue
        key, vals = tok[0], tok[1:]
        if key == "x":
            out = []
            for v in vals:
                if v.startswith("*"):
                    out.extend([out[-1]] * int(v[1:]))
                else:
                    out.append(int(v, 16))
            cur["x"] = np.array(out, dtype=np.uint16)
        elif key in ("scale", "min"):
            cur[key] = int(vals[0], 16)
        elif key == "codes":
            cur["codes"] = np.array([int(v) for v in vals], dtype=np.uint8)
        elif key == "bytes":
            cur["bytes"] = np.array([int(v, 16) for v in vals], dtype=np.uint8)
    return cases


QUANT_CASES = _parse_cases(os.path.join(GOLDEN, "quant_cases.txt"))
PACK_CASES = _parse_cases(os.path.join(GOLDEN, "pack_cases.txt"))


@pytest.mark.parametrize("case", QUANT_CASES, ids=[c["name"] for c in QUANT_CASES])
def test_golden_quant_cases(case):
    assert case["x"].size == 32 and case["codes"].size == 32
    codes, sh, mh = oracle.quantize_group(case["x"], case["bits"])
    assert sh == case["scale"], hex(sh)
    assert mh == case["min"], hex(mh)
    assert np.array_equal(codes, case["codes"]), codes


@pytest.mark.parametrize("case", PACK_CASES, ids=["int4", "int2", "int3"])
def test_golden_pack_cases(case):
    got = oracle.pack_row(case["codes"], case["bits"])
    assert np.array_equal(got, case["bytes"]), got
    assert np.array_equal(oracle.unpack_row(got, 32, case["bits"]), case["codes"])


def _groups(rng, n):
    """Random fp16 groups of several kinds: normal, outlier-scaled, tiny ranges,
    constant, integer grids with ties, mixed zeros."""
    out = []
    for i in range(n):
        kind = i % 7
        if kind == 0:
            x = rng.standard_normal(32)
        elif kind == 1:
            x = rng.standard_normal(32) * 10.0 ** rng.uniform(-3, 3)
        elif kind == 2:  # tiny ranges around a point: subnormal or zero scale
            x = rng.uniform(0, 1) + rng.integers(-40, 40, 32) * 2.0 ** -24
            x = np.where(rng.random(32) < 0.5, x * 0 + rng.integers(0, 60, 32) * 2.0 ** -24, x)
        elif kind == 3:
            x = np.full(32, rng.standard_normal())
        elif kind == 4:  # integer + half grid: many exact ties
            x = rng.integers(0, 31, 32) / 2.0
        elif kind == 5:
            x = np.where(rng.random(32) < 0.5, -0.0, 0.0) + (rng.random(32) < 0.2) * rng.standard_normal(32)
        else:
            x = rng.laplace(size=32) * 3
        out.append(np.asarray(x, np.float64).astype(np.float16).view(np.uint16))
    return out


def _brute_force_codes(x16, mn, s, bits):
    """Nearest grid point among all 2^b codes (exact float64 arithmetic), ties to
    the even code.  Returns (codes, ambiguous, exact_tie): `ambiguous` marks
    quotients within float32 rounding of a tie that are not exact ties (either
    neighbour is accepted there); exact ties are decided strictly."""
    qmax = (1 << bits) - 1
    x = x16.view(np.float16).astype(np.float64)
    cand = np.arange(qmax + 1, dtype=np.float64)
    err = np.abs(x[:, None] - (mn + cand[None, :] * s))
    best = err.min(axis=1)
    exp = np.empty(32, dtype=np.int64)
    ambiguous = np.zeros(32, bool)
    exact_tie = np.zeros(32, bool)
    for j in range(32):
        winners = np.nonzero(err[j] == best[j])[0]
        exp[j] = winners[0] if winners.size == 1 else winners[winners % 2 == 0][0]
        diff = x[j] - mn  # exact: both are binary16 values
        t = diff / s
        k = np.floor(t)
        if diff == (k + 0.5) * s and np.float32(diff) == diff:
            exact_tie[j] = True
        elif abs(t - k - 0.5) < 4e-7 * max(1.0, t):
            ambiguous[j] = True
    return exp, ambiguous, exact_tie


@pytest.mark.parametrize("bits", [4, 2, 3])
def test_brute_force_and_bounds(bits):
    rng = np.random.default_rng(7 + bits)
    qmax = (1 << bits) - 1
    n_ties = 0
    for x16 in _groups(rng, 4000):
        codes, sh, mh = oracle.quantize_group(x16, bits)
        xv = x16.view(np.float16).astype(np.float64)
        s = float(np.array(sh, np.uint16).view(np.float16))
        mn = float(np.array(mh, np.uint16).view(np.float16))
        assert mn == xv.min()
        assert not (mn == 0 and np.signbit(mn))  # -0 is stored as +0
        assert codes.max() <= qmax
        rng_f = xv.max() - xv.min()
        # scale: nearest binary16 to the fp32 quotient (within half an ulp + fp32 error)
        target = rng_f / qmax
        if target == 0:
            assert s == 0
        else:
            ulp = max(2.0 ** -24, 2.0 ** (np.floor(np.log2(target)) - 10))
            assert abs(s - target) <= ulp / 2 + target * 2.0 ** -23, (s, target)
        if s == 0:
            assert not codes.any()
            assert np.all(np.abs(xv - mn) <= qmax * 2.0 ** -25)
            continue
        xhat = mn + codes * s
        normal = s >= 2.0 ** -14
        if normal:
            assert np.all(np.abs(xv - xhat) <= s * (0.5 + 2.0 ** -18))
            assert codes[np.argmax(xv)] == qmax
        else:
            assert np.all(np.abs(xv - xhat) <= s / 2 + qmax * 2.0 ** -25 + 1e-30)
        assert codes[np.argmin(xv)] == 0
        exp, amb, tie = _brute_force_codes(x16, mn, s, bits)
        clamp = np.minimum(exp, qmax)
        ok = (codes == clamp) | (amb & (np.abs(codes.astype(np.int64) - clamp) <= 1))
        assert ok.all(), (xv, codes, clamp)
        n_ties += tie.sum()
    # the integer/half grids must have exercised exact ties
    assert n_ties > 100


def test_exact_ties_go_to_even():
    # values k + 0.5 on a unit-scale grid: exact ties in every arithmetic
    for bits in (2, 3, 4):
        qmax = (1 << bits) - 1
        x = np.zeros(32)
        x[1] = qmax
        half = np.arange(qmax) + 0.5
        x[2:2 + half.size] = half
        codes, sh, mh = oracle.quantize_group(x.astype(np.float16).view(np.uint16), bits)
        assert sh == 0x3C00
        got = codes[2:2 + half.size]
        want = np.where(np.floor(half) % 2 == 0, np.floor(half), np.ceil(half))
        assert np.array_equal(got, want.astype(np.uint8))


@pytest.mark.parametrize("bits,d", [(4, 128), (2, 128), (4, 64), (2, 32), (3, 128), (3, 64), (3, 32)])
def test_pack_bit_order_matches_unpackbits(bits, d):
    rng = np.random.default_rng(bits * 1000 + d)
    codes = rng.integers(0, 1 << bits, d).astype(np.uint8)
    packed = oracle.pack_row(codes, bits)
    assert packed.size == d * bits // 8
    # little-endian bit string: element e at bits [e*b, e*b+b)
    bitstr = np.unpackbits(packed, bitorder="little")
    w = 1 << np.arange(bits)
    back = bitstr.reshape(d, bits) @ w
    assert np.array_equal(back, codes)
    # group g occupies bytes [g*4*b, (g+1)*4*b)
    for g in range(d // 32):
        sub = oracle.pack_row(codes[32 * g:32 * g + 32], bits)
        assert np.array_equal(packed[g * 4 * bits:(g + 1) * 4 * bits], sub)
