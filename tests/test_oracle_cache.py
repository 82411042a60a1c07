"""Pins of the oracle's residual split, sliding-window append and fp64 decode
(Q6, Q7, D1-D4), each checked against something other than the oracle itself:
  - the split: packed and residual parts hold exactly the right tokens,
  - append: packing a prefill at once equals packing a prefix and appending the
    rest, byte for byte (grouping is per token, so the flush order cannot matter),
  - decode: closed forms (identical keys -> mean of V; one token -> that value;
    q = 0 -> the mean), textbook attention (scipy softmax on the fp16 inputs)
    where dequantization is exact (on-grid data, residual-only sequences), a
    second numpy formulation of dequantize-then-attend with its own unpacking,
    GQA head mapping, and invariance under rotation of the residual ring,
  - the attention-sink window: the first min(sink, L) tokens verbatim, the rest
    split exactly as a cache without a sink splits tokens [sink:], sink-only
    sequences are textbook attention, the second formulation with the sink rows
    in front, and appends that never touch the sink.
"""

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def _textbook(q, K, V):
    """softmax(q K^T / sqrt(d)) V in float64 on given float arrays."""
    d = q.shape[-1]
    s = (K.astype(np.float64) @ q.astype(np.float64)) / np.sqrt(d)
    return softmax(s) @ V.astype(np.float64)


def _numpy_dequant(codes, params, d, bits):
    """Second reading of D1: unpack with numpy bit ops and apply min + c * scale."""
    if codes.shape[0] == 0:
        return np.zeros((0, d))
    bitstr = np.unpackbits(codes.reshape(codes.shape[0], -1), axis=1, bitorder="little")
    c = (bitstr.reshape(codes.shape[0], d, bits) * (1 << np.arange(bits))).sum(-1)
    scale = (params & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    mn = (params >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    return mn[:, np.arange(d) // 32] + c * scale[:, np.arange(d) // 32]


def _build(rng, B=2, H=2, d=64, bits=4, L=40, Nr=8, cap=None, lens=None, kscale=1.0, sink=0):
    lens = np.array(lens if lens is not None else [L] * B, np.int32)
    Lmax = int(lens.max())
    cap = cap if cap is not None else Lmax
    k = _f16(rng, (B, H, Lmax, d), kscale)
    v = _f16(rng, (B, H, Lmax, d))
    c = oracle.Cache(B, H, d, bits, cap, Nr, sink)
    err = oracle.quantize_pack(c, k, v, lens)
    return c, k, v, lens, err


@pytest.mark.parametrize("L,Nr", [(40, 8), (5, 8), (8, 8), (0, 4), (33, 0)])
def test_split(L, Nr):
    rng = np.random.default_rng(L * 31 + Nr)
    c, k, v, lens, err = _build(rng, L=L, Nr=Nr, cap=max(L, 1))
    assert err == 0
    nres = min(L, Nr)
    assert np.all(c.packed_len == L - nres) and np.all(c.res_len == nres) and np.all(c.res_head == 0)
    for b in range(2):
        for h in range(2):
            # residual = the last nres tokens verbatim, in order
            assert np.array_equal(c.k_res[b, h, :nres], k[b, h, L - nres:L].view(np.uint16))
            assert np.array_equal(c.v_res[b, h, :nres], v[b, h, L - nres:L].view(np.uint16))
            # packed slots = each token quantized on its own
            for t in range(L - nres):
                for g in range(64 // 32):
                    codes, sh, mh = oracle.quantize_group(k[b, h, t, 32 * g:32 * g + 32], 4)
                    assert c.k_params[b, h, t, g] == sh | (mh << 16)
                    assert np.array_equal(c.k_codes[b, h, t, 16 * g:16 * g + 16],
                                          oracle.pack_row(codes, 4))


def test_capacity_and_bad_length():
    rng = np.random.default_rng(3)
    c, k, v, lens, err = _build(rng, B=2, L=20, Nr=4, cap=10)
    assert err & 1 and np.all(c.packed_len == 10)
    c2 = oracle.Cache(2, 2, 64, 4, 30, 4)
    err = oracle.quantize_pack(c2, k, v, np.array([20, 25], np.int32))
    assert err & 8 and c2.packed_len[0] == 16


@pytest.mark.parametrize("bits,Nr", [(4, 8), (2, 5), (4, 0), (3, 6)])
def test_append_equals_prefill(bits, Nr):
    rng = np.random.default_rng(11 + bits + Nr)
    B, H, d, L, L0 = 2, 3, 64, 37, 3
    k = _f16(rng, (B, H, L, d), 4.0)
    v = _f16(rng, (B, H, L, d))
    full = oracle.Cache(B, H, d, bits, L, Nr)
    assert oracle.quantize_pack(full, k, v, np.full(B, L, np.int32)) == 0
    inc = oracle.Cache(B, H, d, bits, L, Nr)
    assert oracle.quantize_pack(inc, k[:, :, :L0].copy(), v[:, :, :L0].copy(), np.full(B, L0, np.int32)) == 0
    for t in range(L0, L):
        assert oracle.append(inc, k[:, :, t].copy(), v[:, :, t].copy()) == 0
    npk = L - min(L, Nr)
    assert np.array_equal(inc.packed_len, full.packed_len)
    assert np.array_equal(inc.res_len, full.res_len)
    for a in ("k_codes", "v_codes", "k_params", "v_params"):
        assert np.array_equal(getattr(inc, a)[:, :, :npk], getattr(full, a)[:, :, :npk]), a
    # the ring holds the same tokens; in age order from res_head
    for b in range(B):
        n = inc.res_len[b]
        order = (inc.res_head[b] + np.arange(n)) % max(Nr, 1)
        assert np.array_equal(inc.k_res[b][:, order], full.k_res[b][:, :n])
        assert np.array_equal(inc.v_res[b][:, order], full.v_res[b][:, :n])
    # and decode agrees exactly in value
    q = _f16(rng, (B, 2 * H, d))
    assert np.allclose(oracle.decode(inc, q), oracle.decode(full, q), rtol=1e-12, atol=1e-14)


def test_append_capacity_error():
    rng = np.random.default_rng(5)
    c, k, v, lens, err = _build(rng, B=1, H=1, L=12, Nr=4, cap=8)
    assert err == 0 and c.packed_len[0] == 8
    before = c.copy()
    e = oracle.append(c, _f16(rng, (1, 1, 64)), _f16(rng, (1, 1, 64)))
    assert e & 1
    assert np.array_equal(c.k_res, before.k_res) and c.packed_len[0] == 8


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(21)
    B, H, d, L, Nr = 1, 1, 64, 50, 6
    # an on-grid key row (per group: min -1.75, max 2, step 0.25, so scale 0.25
    # and every value reconstructs exactly), used for every token
    codes = rng.integers(0, 16, d)
    codes[0::32], codes[1::32] = 0, 15
    kq = (codes * 0.25 - 1.75).astype(np.float16)
    k = np.broadcast_to(kq, (B, H, L, d)).copy()
    v = _f16(rng, (B, H, L, d))
    c = oracle.Cache(B, H, d, 4, L, Nr)
    oracle.quantize_pack(c, k, v, np.array([L], np.int32))
    q = _f16(rng, (B, H, d))
    out = oracle.decode(c, q)[0, 0]
    vhat = np.concatenate([_numpy_dequant(c.v_codes[0, 0, :L - Nr], c.v_params[0, 0, :L - Nr], d, 4),
                           c.v_res[0, 0].view(np.float16).astype(np.float64)])
    assert np.allclose(out, vhat.mean(0), rtol=0, atol=1e-13)


def test_single_token_and_zero_query():
    rng = np.random.default_rng(22)
    d = 64
    for Nr in (0, 1):
        c, k, v, lens, _ = _build(rng, B=1, H=1, d=d, L=1, Nr=Nr)
        out = oracle.decode(c, _f16(rng, (1, 1, d)))[0, 0]
        if Nr:
            want = v[0, 0, 0].astype(np.float64)
        else:
            want = _numpy_dequant(c.v_codes[0, 0, :1], c.v_params[0, 0, :1], d, 4)[0]
        assert np.array_equal(out, want)
    c, k, v, lens, _ = _build(rng, B=1, H=1, d=d, L=30, Nr=7)
    out = oracle.decode(c, np.zeros((1, 1, d), np.float16))[0, 0]
    vhat = np.concatenate([_numpy_dequant(c.v_codes[0, 0, :23], c.v_params[0, 0, :23], d, 4),
                           c.v_res[0, 0].view(np.float16).astype(np.float64)])
    assert np.allclose(out, vhat.mean(0), rtol=0, atol=1e-13)


@pytest.mark.parametrize("bits", [4, 2])
def test_on_grid_data_is_textbook_attention(bits):
    # K and V already on the grid: every group holds integers 0..2^b-1 with 0 and
    # 2^b-1 present, so scale = 1, min = 0 and dequantization is exact.
    rng = np.random.default_rng(40 + bits)
    qmax = (1 << bits) - 1
    B, H, d, L, Nr = 1, 2, 64, 45, 5
    x = rng.integers(0, qmax + 1, (2, B, H, L, d)).astype(np.float64)
    x[..., 0::32] = 0
    x[..., 1::32] = qmax
    k = x[0].astype(np.float16)
    v = x[1].astype(np.float16)
    c = oracle.Cache(B, H, d, bits, L, Nr)
    oracle.quantize_pack(c, k, v, np.array([L], np.int32))
    assert np.all(c.k_params[:, :, :L - Nr] == 0x3C00)
    q = _f16(rng, (B, H, d), 0.3)
    out = oracle.decode(c, q)
    for h in range(H):
        want = _textbook(q[0, h], k[0, h], v[0, h])
        assert np.allclose(out[0, h], want, rtol=1e-12, atol=1e-12)


def test_residual_only_is_textbook_attention():
    rng = np.random.default_rng(50)
    c, k, v, lens, _ = _build(rng, B=2, H=1, d=64, L=6, Nr=8)
    assert np.all(c.packed_len == 0)
    q = _f16(rng, (2, 1, 64))
    out = oracle.decode(c, q)
    for b in range(2):
        assert np.allclose(out[b, 0], _textbook(q[b, 0], k[b, 0], v[b, 0]), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("bits,d,gq", [(4, 32, 1), (2, 64, 2), (4, 128, 4), (2, 32, 3), (3, 128, 4),
                                       (3, 32, 2)])
def test_second_formulation_tiny(bits, d, gq):
    rng = np.random.default_rng(bits * 100 + d + gq)
    B, H, Nr = 2, 2, 3
    lens = [8, 5]
    c, k, v, lens, _ = _build(rng, B=B, H=H, d=d, bits=bits, Nr=Nr, lens=lens, kscale=5.0)
    q = _f16(rng, (B, H * gq, d))
    out = oracle.decode(c, q)
    for b in range(B):
        L = lens[b]
        npk = L - min(L, Nr)
        for hq in range(H * gq):
            h = hq // gq
            K = np.concatenate([_numpy_dequant(c.k_codes[b, h, :npk], c.k_params[b, h, :npk], d, bits),
                                k[b, h, npk:L].astype(np.float64)])
            V = np.concatenate([_numpy_dequant(c.v_codes[b, h, :npk], c.v_params[b, h, :npk], d, bits),
                                v[b, h, npk:L].astype(np.float64)])
            want = _textbook(q[b, hq], K, V)
            assert np.allclose(out[b, hq], want, rtol=1e-12, atol=1e-13)
    # selected pairs give the same rows
    pairs = np.array([[1, H * gq - 1], [0, 0]], np.int32)
    sel = oracle.decode(c, q, pairs)
    assert np.array_equal(sel[0], out[1, H * gq - 1]) and np.array_equal(sel[1], out[0, 0])


def test_ring_rotation_invariance():
    rng = np.random.default_rng(60)
    c, k, v, lens, _ = _build(rng, B=1, H=1, d=64, L=30, Nr=6)
    q = _f16(rng, (1, 1, 64))
    base = oracle.decode(c, q)
    r = c.copy()
    r.k_res[...] = np.roll(c.k_res, 2, axis=2)
    r.v_res[...] = np.roll(c.v_res, 2, axis=2)
    r.res_head[0] = 2
    assert np.allclose(oracle.decode(r, q), base, rtol=1e-13, atol=1e-15)


def test_empty_sequence_gives_zeros():
    c = oracle.Cache(1, 1, 64, 4, 4, 4)
    out = oracle.decode(c, np.ones((1, 1, 64), np.float16))
    assert np.all(out == 0)


# ---------------------------------------------------------- attention sink --


@pytest.mark.parametrize("L,Nr,S", [(40, 8, 4), (10, 8, 4), (3, 8, 4), (4, 0, 4), (33, 0, 32), (0, 4, 4)])
def test_sink_split(L, Nr, S):
    """The sink holds tokens [0, min(S, L)) verbatim; everything after is laid
    out byte for byte as a sink-free cache lays out the prefill without them."""
    rng = np.random.default_rng(L * 7 + Nr + S)
    B, H, d = 2, 2, 64
    lens = np.array([L, max(L - 2, 0)], np.int32)
    c, k, v, lens, err = _build(rng, B=B, H=H, d=d, Nr=Nr, cap=max(L, 1), lens=lens, sink=S)
    assert err == 0
    for b in range(B):
        ns = min(S, int(lens[b]))
        assert c.sink_len[b] == ns
        assert np.array_equal(c.k_sink[b, :, :ns], k[b, :, :ns].view(np.uint16))
        assert np.array_equal(c.v_sink[b, :, :ns], v[b, :, :ns].view(np.uint16))
        rest = int(lens[b]) - ns
        ref = oracle.Cache(1, H, d, 4, max(L, 1), Nr)
        kr = k[b:b + 1, :, ns:].copy()
        vr = v[b:b + 1, :, ns:].copy()
        assert oracle.quantize_pack(ref, kr, vr, np.array([rest], np.int32)) == 0
        assert c.packed_len[b] == ref.packed_len[0] and c.res_len[b] == ref.res_len[0]
        npk = ref.packed_len[0]
        for name in ("k_codes", "v_codes", "k_params", "v_params"):
            assert np.array_equal(getattr(c, name)[b, :, :npk], getattr(ref, name)[0, :, :npk]), name
        for name in ("k_res", "v_res"):
            assert np.array_equal(getattr(c, name)[b, :, :ref.res_len[0]],
                                  getattr(ref, name)[0, :, :ref.res_len[0]]), name


def test_sink_bounds_rejected():
    with pytest.raises(ValueError):
        oracle.quantize_pack(oracle.Cache(1, 1, 64, 4, 4, 4, 257), np.zeros((1, 1, 1, 64), np.float16),
                             np.zeros((1, 1, 1, 64), np.float16), np.array([1], np.int32))


@pytest.mark.parametrize("L,Nr", [(5, 0), (9, 4), (32, 0)])
def test_sink_only_is_textbook_attention(L, Nr):
    """With nothing packed (L <= sink + Nr) every token is fp16: the output is
    textbook attention over the inputs themselves."""
    rng = np.random.default_rng(70 + L + Nr)
    c, k, v, lens, _ = _build(rng, B=2, H=1, d=64, L=L, Nr=Nr, sink=32 if L == 32 else 5)
    assert np.all(c.packed_len == 0)
    q = _f16(rng, (2, 1, 64))
    out = oracle.decode(c, q)
    for b in range(2):
        assert np.allclose(out[b, 0], _textbook(q[b, 0], k[b, 0], v[b, 0]), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("bits,S,lens", [(4, 4, [20, 3]), (2, 32, [50, 40]), (4, 1, [9, 0])])
def test_sink_second_formulation(bits, S, lens):
    """Sink rows (fp16), then the packed tokens unpacked by numpy, then the ring:
    textbook attention over that sequence equals the oracle's decode."""
    rng = np.random.default_rng(bits + S + sum(lens))
    B, H, d, gq, Nr = 2, 2, 64, 2, 3
    c, k, v, lens, _ = _build(rng, B=B, H=H, d=d, bits=bits, Nr=Nr, lens=lens, kscale=4.0, sink=S)
    q = _f16(rng, (B, H * gq, d))
    out = oracle.decode(c, q)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            assert np.all(out[b] == 0)
            continue
        ns = min(S, L)
        nres = min(Nr, L - ns)
        npk = L - ns - nres
        for hq in range(H * gq):
            h = hq // gq
            K = np.concatenate([k[b, h, :ns].astype(np.float64),
                                _numpy_dequant(c.k_codes[b, h, :npk], c.k_params[b, h, :npk], d, bits),
                                k[b, h, L - nres:L].astype(np.float64)])
            V = np.concatenate([v[b, h, :ns].astype(np.float64),
                                _numpy_dequant(c.v_codes[b, h, :npk], c.v_params[b, h, :npk], d, bits),
                                v[b, h, L - nres:L].astype(np.float64)])
            assert np.allclose(out[b, hq], _textbook(q[b, hq], K, V), rtol=1e-12, atol=1e-13)


def test_sink_fixed_after_prefill():
    """Appends go to the recent window and the packed cache only: the sink rows
    and sink_len never change, also for a sequence whose sink is not full; past
    a full sink, append equals a prefill of the same tokens."""
    rng = np.random.default_rng(80)
    B, H, d, S, Nr, L0, L = 2, 2, 64, 6, 4, 8, 30
    k = _f16(rng, (B, H, L, d), 3.0)
    v = _f16(rng, (B, H, L, d))
    inc = oracle.Cache(B, H, d, 4, L, Nr, S)
    assert oracle.quantize_pack(inc, k[:, :, :L0].copy(), v[:, :, :L0].copy(),
                                np.array([L0, 2], np.int32)) == 0
    before = inc.copy()
    for t in range(L0, L):
        assert oracle.append(inc, k[:, :, t].copy(), v[:, :, t].copy()) == 0
    for name in ("k_sink", "v_sink", "sink_len"):
        assert np.array_equal(getattr(inc, name), getattr(before, name)), name
    assert list(inc.sink_len) == [S, 2]
    full = oracle.Cache(1, H, d, 4, L, Nr, S)
    assert oracle.quantize_pack(full, k[:1], v[:1], np.array([L], np.int32)) == 0
    npk = full.packed_len[0]
    assert inc.packed_len[0] == npk and inc.res_len[0] == full.res_len[0]
    for name in ("k_codes", "v_codes", "k_params", "v_params"):
        assert np.array_equal(getattr(inc, name)[0, :, :npk], getattr(full, name)[0, :, :npk]), name
    q = _f16(rng, (B, H, d))
    assert np.allclose(oracle.decode(inc, q)[:1], oracle.decode(full, q[:1]), rtol=1e-12, atol=1e-14)
