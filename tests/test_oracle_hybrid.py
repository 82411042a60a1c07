"""Pins of the oracle's hybrid symmetric/asymmetric mode (H1-H3; InnerQ page,
section 2.2): per group the candidate with the smaller squared reconstruction
error is kept and a 1-bit mask records which.  Checked against closed forms
(groups that one of the two grids reproduces exactly), brute force (the
symmetric codes are the nearest points of the symmetric grid), an fp64
recomputation of both errors that the fp32 decision must follow whenever they
differ clearly, ties, the fp16 overflow of the symmetric min, the mask layout
in a packed cache, and append = prefill with the mode bytes included."""

import numpy as np
import pytest

import oracle

from test_oracle_cache import _numpy_dequant, _textbook


def _f16v(h):
    return float(np.array([h], np.uint16).view(np.float16)[0])


def _dequant(codes, sh, mh):
    return _f16v(mh) + codes.astype(np.float64) * _f16v(sh)


@pytest.mark.parametrize("bits,s", [(4, 0.25), (4, 3.0), (2, 0.5), (2, 1.25)])
def test_on_symmetric_grid_takes_symmetric(bits, s):
    """x = t * s with integers |t| <= 2^(b-1) - 1, both extremes present: the
    symmetric grid holds every value (error 0), the asymmetric one does not."""
    qs = (1 << (bits - 1)) - 1
    rng = np.random.default_rng(bits * 10 + int(s * 4))
    t = rng.integers(-qs, qs + 1, 32)
    t[0], t[1] = qs, -qs
    x = (t * s).astype(np.float16)
    codes, sh, mh, mode = oracle.quantize_group_hybrid(x, bits)
    assert mode == 0
    assert _f16v(sh) == s and _f16v(mh) == -(1 << (bits - 1)) * s
    assert np.array_equal(codes, t + (1 << (bits - 1)))
    assert np.array_equal(_dequant(codes, sh, mh), x.astype(np.float64))


@pytest.mark.parametrize("bits", [4, 2])
def test_on_asymmetric_grid_takes_asymmetric(bits):
    """x = 1 + c * 0.5 with c over 0 .. 2^b - 1 (both ends present): the
    asymmetric grid is exact and the symmetric one cannot be."""
    qmax = (1 << bits) - 1
    rng = np.random.default_rng(bits)
    c = rng.integers(0, qmax + 1, 32)
    c[0], c[1] = 0, qmax
    x = (1.0 + 0.5 * c).astype(np.float16)
    codes, sh, mh, mode = oracle.quantize_group_hybrid(x, bits)
    assert mode == 1
    assert np.array_equal(codes, c) and _f16v(sh) == 0.5 and _f16v(mh) == 1.0


@pytest.mark.parametrize("bits", [4, 2])
def test_ties_keep_asymmetric(bits):
    """Zero and constant groups reconstruct exactly in the asymmetric mode; the
    all-zero group also in the symmetric one (both errors 0): a tie keeps the
    asymmetric candidate."""
    for x in (np.zeros(32, np.float16), np.full(32, -3.5, np.float16)):
        codes, sh, mh, mode = oracle.quantize_group_hybrid(x, bits)
        assert mode == 1
        assert np.array_equal(_dequant(codes, sh, mh), x.astype(np.float64))
    sc, ssh, smh, ok = oracle.quantize_group_sym(np.zeros(32, np.float16), bits)
    assert ok and ssh == 0 and smh == 0 and np.all(sc == 1 << (bits - 1))


def test_symmetric_min_overflow_rules_it_out():
    """absmax 60000 (INT4): scale 8568, min -8 * 8568 is beyond fp16, so the
    symmetric candidate cannot be stored even where it would fit better."""
    x = np.zeros(32, np.float16)
    x[0], x[1] = 60000.0, -60000.0
    sc, sh, mh, ok = oracle.quantize_group_sym(x, 4)
    assert not ok and (mh & 0x7C00) == 0x7C00
    assert oracle.quantize_group_hybrid(x, 4)[3] == 1
    # INT2 (scale = absmax): min = -2 * 60000 overflows too, -2 * 30000 does not
    assert not oracle.quantize_group_sym(x, 2)[3]
    x[0], x[1] = 30000.0, -30000.0
    sc, sh, mh, ok = oracle.quantize_group_sym(x, 2)
    assert ok and _f16v(mh) == -60000.0


def _groups(rng, n):
    """Random groups: gaussian, with outliers, one-sided, and narrow ranges."""
    out = []
    for i in range(n):
        kind = i % 4
        x = rng.standard_normal(32)
        if kind == 1:
            x = np.where(rng.random(32) < 0.05, rng.standard_normal(32) * 8, x)
        elif kind == 2:
            x = np.abs(x) + rng.random() * 3
        elif kind == 3:
            x = x * 1e-3 + rng.standard_normal()
        out.append(x.astype(np.float16))
    return out


@pytest.mark.parametrize("bits", [4, 2])
def test_symmetric_codes_are_nearest_grid_points(bits):
    """Brute force over the symmetric grid {t * s : |t| <= 2^(b-1) - 1}: each
    code is the nearest point (fp64 distances; an exact tie takes the even t)."""
    half = 1 << (bits - 1)
    qs = half - 1
    rng = np.random.default_rng(100 + bits)
    for x in _groups(rng, 200):
        codes, sh, mh, ok = oracle.quantize_group_sym(x, bits)
        s = _f16v(sh)
        assert ok and _f16v(mh) == -half * s
        if s == 0:
            continue
        grid = np.arange(-qs, qs + 1)
        xv = x.astype(np.float64)
        dist = np.abs(xv[:, None] - grid[None, :] * s)
        best = dist.min(1)
        for j in range(32):
            cand = grid[dist[j] == best[j]]
            t = int(codes[j]) - half
            assert t in cand, (j, xv[j], t, cand)
            if len(cand) == 2:
                assert t % 2 == 0


@pytest.mark.parametrize("bits", [4, 2])
def test_decision_follows_the_smaller_error(bits):
    """Both candidates' squared errors recomputed in fp64 from their stored
    (codes, scale, min): the chosen mode has the smaller one whenever they
    differ by more than fp32 rounding could blur, and both modes occur."""
    rng = np.random.default_rng(7 + bits)
    modes = []
    for x in _groups(rng, 400):
        ca, ash, amh = oracle.quantize_group(x, bits)
        cs, ssh, smh, ok = oracle.quantize_group_sym(x, bits)
        codes, sh, mh, mode = oracle.quantize_group_hybrid(x, bits)
        xv = x.astype(np.float64)
        ea = ((xv - _dequant(ca, ash, amh)) ** 2).sum()
        es = ((xv - _dequant(cs, ssh, smh)) ** 2).sum()
        if ok and abs(ea - es) > 1e-5 * max(ea, es, 1e-30):
            assert mode == (0 if es < ea else 1), (ea, es, mode)
        # the stored result is the chosen candidate, unchanged
        want = (cs, ssh, smh) if mode == 0 else (ca, ash, amh)
        assert np.array_equal(codes, want[0]) and sh == want[1] and mh == want[2]
        modes.append(mode)
    assert 0 < sum(modes) < len(modes)



def _dyadic(v: float) -> int:
    """v (an fp16 or fp32 value of modest size) as an integer multiple of 2^-40."""
    n = v * (1 << 40)
    assert n == int(n)
    return int(n)


def _is_f32(n: int) -> bool:
    """A multiple of a power of two (2^-40 or 2^-80 here) is an fp32 value when
    its odd part has at most 24 bits (the magnitudes here stay in fp32's
    normal range)."""
    n = abs(n)
    if n == 0:
        return True
    n >>= (n & -n).bit_length() - 1
    return n.bit_length() <= 24


def _exact_sq_error(x, codes, sh, mh):
    """The sum of (x - (min + code * scale))^2 in exact integer arithmetic (in
    units of 2^-80), or None unless fp32 arithmetic reproduces it without a
    single rounding: every product, reconstruction, difference and square is
    an fp32 value, and all terms are multiples of the lowest set bit among them
    with a total below 2^24 such units, so every partial sum, in any order, is
    exact."""
    mn, sc = _dyadic(_f16v(mh)), _dyadic(_f16v(sh))
    terms = []
    for v, c in zip(x.astype(np.float64), codes):
        prod = int(c) * sc
        rec = mn + prod
        d = _dyadic(float(v)) - rec
        sq = d * d
        if not all(_is_f32(t) for t in (prod, rec, d, sq)):
            return None
        terms.append(sq)
    nz = [t for t in terms if t]
    if nz:
        unit = min((t & -t).bit_length() - 1 for t in nz)
        if sum(terms) >> unit >= 1 << 24:
            return None
    return sum(terms)


@pytest.mark.parametrize("bits,p_zero", [(4, 0.0), (2, 0.3)])
def test_exact_near_ties_follow_the_exact_comparison(bits, p_zero):
    """Near ties decided without rounding.  Groups on a quarter-step grid with
    ends -1.5 and 1.5 (some values pulled to 0) whose two candidate errors fp32
    arithmetic computes exactly, so the decision cannot depend on the order of
    the sums: it must be the exact comparison, symmetric only when its error is
    strictly smaller.  Errors within 8% of each other, of both signs, and exact
    ties (INT2) occur; a swapped comparison, a non-strict one or a dropped term
    fails here even though the fp64 check above only looks at clear gaps."""
    rng = np.random.default_rng(40 + bits)
    seen = {-1: 0, 0: 0, 1: 0}
    for _ in range(1500):
        k = rng.integers(-6, 7, 32)
        k[rng.random(32) < p_zero] = 0
        k[0], k[1] = -6, 6
        x = (k * 0.25).astype(np.float16)
        ca, ash, amh = oracle.quantize_group(x, bits)
        cs, ssh, smh, ok = oracle.quantize_group_sym(x, bits)
        ea, es = _exact_sq_error(x, ca, ash, amh), _exact_sq_error(x, cs, ssh, smh)
        if not ok or ea is None or es is None or abs(ea - es) * 12 > max(ea, es):
            continue
        mode = oracle.quantize_group_hybrid(x, bits)[3]
        assert mode == (0 if es < ea else 1), (bits, ea, es, mode)
        seen[(es > ea) - (es < ea)] += 1
    assert seen[-1] >= 10 and seen[1] >= 10, seen
    if bits == 2:
        assert seen[0] >= 10, seen

def test_error_is_a_sum_of_squares():
    """H2 against its definition on hand-made cases: exact reconstruction gives
    0, one element off by 0.5 gives 0.25, and the sum is over all 32."""
    x = np.arange(32, dtype=np.float16)
    codes = np.arange(32, dtype=np.uint8)
    one = int(np.array([1.0], np.float16).view(np.uint16)[0])
    assert oracle.group_sq_error(x, codes, one, 0) == 0.0
    x2 = x.copy()
    x2[5] += np.float16(0.5)
    assert oracle.group_sq_error(x2, codes, one, 0) == 0.25
    half = int(np.array([0.5], np.float16).view(np.uint16)[0])
    # every reconstruction 0.5 low: 32 * 0.25
    assert oracle.group_sq_error(x, codes, one, int(np.array([-0.5], np.float16).view(np.uint16)[0])) == 8.0
    assert oracle.group_sq_error(np.full(32, 1.0, np.float16), np.zeros(32, np.uint8), half, half) == 8.0


@pytest.mark.parametrize("bits", [4, 2])
def test_cache_mode_bytes_and_layout(bits):
    """A hybrid pack stores, per packed row, the groups' results and the mode
    byte (bit g = group g); a plain pack of the same data leaves the mode bytes
    zero and equals the asymmetric quantizer group by group."""
    rng = np.random.default_rng(20 + bits)
    B, H, L, d, Nr = 2, 2, 30, 128, 4
    k = rng.standard_normal((B, H, L, d))
    k = np.where(rng.random(k.shape) < 0.03, rng.standard_normal(k.shape) * 8, k).astype(np.float16)
    v = rng.standard_normal((B, H, L, d)).astype(np.float16)
    lens = np.array([L, 11], np.int32)
    hy = oracle.Cache(B, H, d, bits, L, Nr, 0, 1)
    pl = oracle.Cache(B, H, d, bits, L, Nr)
    assert oracle.quantize_pack(hy, k, v, lens) == 0 and oracle.quantize_pack(pl, k, v, lens) == 0
    assert np.all(pl.k_mode == 0) and np.all(pl.v_mode == 0)
    seen = set()
    for b in range(B):
        for h in range(H):
            for t in range(int(hy.packed_len[b])):
                for g in range(d // 32):
                    c, sh, mh, mode = oracle.quantize_group_hybrid(k[b, h, t, 32 * g:32 * g + 32], bits)
                    assert (hy.k_mode[b, h, t] >> g) & 1 == mode
                    assert hy.k_params[b, h, t, g] == sh | (mh << 16)
                    seen.add(mode)
                assert hy.k_mode[b, h, t] >> (d // 32) == 0
    assert seen == {0, 1}
    # decode of a hybrid cache: textbook attention over min + code * scale
    q = rng.standard_normal((B, H, d)).astype(np.float16)
    out = oracle.decode(hy, q)
    for b in range(B):
        n = int(hy.packed_len[b])
        for h in range(H):
            K = np.concatenate([_numpy_dequant(hy.k_codes[b, h, :n], hy.k_params[b, h, :n], d, bits),
                                k[b, h, n:lens[b]].astype(np.float64)])
            V = np.concatenate([_numpy_dequant(hy.v_codes[b, h, :n], hy.v_params[b, h, :n], d, bits),
                                v[b, h, n:lens[b]].astype(np.float64)])
            assert np.allclose(out[b, h], _textbook(q[b, h], K, V), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("Nr", [0, 5])
def test_hybrid_append_equals_prefill(Nr):
    rng = np.random.default_rng(30 + Nr)
    B, H, d, L, L0 = 2, 2, 64, 25, 4
    k = rng.standard_normal((B, H, L, d))
    k = np.where(rng.random(k.shape) < 0.05, rng.standard_normal(k.shape) * 8, k).astype(np.float16)
    v = rng.standard_normal((B, H, L, d)).astype(np.float16)
    full = oracle.Cache(B, H, d, 2, L, Nr, 0, 1)
    assert oracle.quantize_pack(full, k, v, np.full(B, L, np.int32)) == 0
    inc = oracle.Cache(B, H, d, 2, L, Nr, 0, 1)
    assert oracle.quantize_pack(inc, k[:, :, :L0].copy(), v[:, :, :L0].copy(), np.full(B, L0, np.int32)) == 0
    for t in range(L0, L):
        assert oracle.append(inc, k[:, :, t].copy(), v[:, :, t].copy()) == 0
    n = int(full.packed_len[0])
    for name in ("k_codes", "v_codes", "k_params", "v_params", "k_mode", "v_mode"):
        assert np.array_equal(getattr(inc, name)[:, :, :n], getattr(full, name)[:, :, :n]), name
