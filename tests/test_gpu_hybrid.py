"""GPU parity of the hybrid symmetric/asymmetric mode (InnerQ page, section
2.2): every group quantized both ways, the smaller fp32 squared error kept,
the choice in a mode byte per packed row.  Codes, scales, mins and mode bytes
bit-exact with the oracle through pack, append and the fused step; decode of a
hybrid cache within max abs 2e-3 / relative L2 1e-3 of the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq, synth

from _util import assert_attn_close, assert_cache_equal, gpu_cache, ref_cache, to_np
from test_gpu_pack import _special_values

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outliers(rng, shape, p=0.01):
    """N(0, 1) with a fraction p of the elements replaced by N(0, 8^2): the
    INT4 decode-batch workload's recipe (p = 0: the INT2 workload's plain
    gaussian values)."""
    x = rng.standard_normal(shape)
    return torch.from_numpy(np.where(rng.random(shape) < p, rng.standard_normal(shape) * 8, x)
                            .astype(np.float16))


def _both(k, v, lens, bits, cap, Nr, S=0):
    B, H, Lmax, d = k.shape
    g = gpu_cache(B, H, d, bits, cap, Nr, sink=S, hybrid=1)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), lens.to(DEV))
    st, word = kvq.kvq_read_error(g)
    r = ref_cache(B, H, d, bits, cap, Nr, sink=S, hybrid=1)
    err = oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens))
    return g, r, st, word, err


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_hybrid_pack(bits, d):
    """Special values (ties, constants, +-0, subnormals, huge ranges) in K,
    outliers in V: every byte matches, and with INT4 both modes occur."""
    rng = np.random.default_rng(bits * 31 + d)
    B, H, Lmax, Nr = 3, 2, 301, 17
    k = _special_values(rng, (B, H, Lmax, d))
    v = _outliers(rng, (B, H, Lmax, d))
    lens = torch.tensor([301, 9, 150], dtype=torch.int32)
    g, r, st, word, err = _both(k, v, lens, bits, 290, Nr)
    assert st == kvq.KVQ_OK and word == 0 and err == 0
    assert_cache_equal(g, r)
    if bits == 4:  # both modes occur (INT2's three symmetric levels rarely win)
        n = int(r.packed_len[0])
        ng = d // 32
        m = (r.k_mode[0, :, :n, None] >> np.arange(ng)) & 1
        assert 0 < m.sum() < m.size


def test_hybrid_plain_cache_unchanged():
    """hybrid = 0 packs exactly as before (no mode arrays written), and the
    hybrid cache differs from it only in groups the symmetric mode won."""
    rng = np.random.default_rng(5)
    B, H, L, d = 2, 2, 200, 128
    k, v = _outliers(rng, (B, H, L, d)), _outliers(rng, (B, H, L, d))
    lens = torch.tensor([200, 77], dtype=torch.int32)
    plain = gpu_cache(B, H, d, 4, L, 8)
    kvq.kvq_quantize_pack(plain, k.to(DEV), v.to(DEV), lens.to(DEV))
    rp = ref_cache(B, H, d, 4, L, 8)
    assert oracle.quantize_pack(rp, to_np(k), to_np(v), to_np(lens)) == 0
    assert_cache_equal(plain, rp)
    g, r, st, word, err = _both(k, v, lens, 4, L, 8)
    assert_cache_equal(g, r)
    kp_h, kp_p = to_np(g.k_params).view(np.uint32), to_np(plain.k_params).view(np.uint32)
    modes = to_np(g.k_mode)
    for b in range(B):
        n = int(r.packed_len[b])
        asym = (modes[b, :, :n, None] >> np.arange(4)) & 1
        assert np.array_equal(kp_h[b, :, :n][asym == 1], kp_p[b, :, :n][asym == 1])


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("d,gq", [(128, 4), (64, 2), (128, 1)])
def test_hybrid_decode(bits, d, gq):
    rng = np.random.default_rng(bits * 100 + d + gq)
    B, H, Nr = 3, 2, 19
    lens = torch.tensor([700, 1, 243], dtype=torch.int32)
    p = 0.01 if bits == 4 else 0.0
    k, v = _outliers(rng, (B, H, 700, d), p), _outliers(rng, (B, H, 700, d), p)
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    g, r, st, word, err = _both(k, v, lens, bits, 700, Nr)
    assert st == kvq.KVQ_OK and err == 0
    want = oracle.decode(r, q.numpy())
    assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV), flags=kvq.KVQ_OUT_F32), want)
    assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV)), want)


@pytest.mark.parametrize("fused", [False, True, "early"])
@pytest.mark.parametrize("bits,d,gq,Nr", [(4, 128, 4, 16), (2, 128, 4, 0), (4, 64, 2, 8)])
def test_hybrid_steps(fused, bits, d, gq, Nr):
    """Appends through kvq_append + decode or the fused step (tensor-core path
    for head_dim 128): each packed token quantized by the hybrid rule, its mode
    byte written; bytes and outputs against the oracle after every step."""
    rng = np.random.default_rng(bits * 7 + d + Nr + bool(fused))
    flags = kvq.KVQ_STEP_EARLY_CACHE_READ if fused == "early" else 0
    B, H = 2, 2
    lens = torch.tensor([Nr + 300, 3], dtype=torch.int32)
    p = 0.01 if bits == 4 else 0.0
    k, v = _outliers(rng, (B, H, Nr + 300, d), p), _outliers(rng, (B, H, Nr + 300, d), p)
    g, r, st, word, err = _both(k, v, lens, bits, Nr + 340, Nr)
    assert st == kvq.KVQ_OK and err == 0
    ws = kvq.workspace_for(g, H * gq)
    for _ in range(12):
        kn, vn = _outliers(rng, (B, H, d), p), _outliers(rng, (B, H, d), p)
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
        out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
        if fused:
            kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV), out, ws, flags=flags)
        else:
            kvq.kvq_append(g, kn.to(DEV), vn.to(DEV))
            kvq.kvq_decode_attention(g, q.to(DEV), out, ws)
        st, word = kvq.kvq_read_error(g)
        assert st == kvq.KVQ_OK and word == 0
        assert oracle.append(r, kn.numpy(), vn.numpy()) == 0
        assert_cache_equal(g, r)
        assert_attn_close(out, oracle.decode(r, q.numpy()))


@pytest.mark.parametrize("bits", [4, 2])
def test_hybrid_pack_full_size(bits):
    """The standalone pack case (32768 tokens x 8 heads x 128, K and V) with the
    hybrid rule: the packed bytes and mode bytes of heads 0 and 5 against the
    oracle."""
    w = synth.scaled(synth.WORKLOADS[5], bits=bits)
    k, v, lens = w.prefill(device=DEV)
    g = gpu_cache(w.batch, w.num_kv_heads, w.head_dim, bits, w.len_max, 0, hybrid=1)
    kvq.kvq_quantize_pack(g, k, v, lens.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    for h in (0, 5):
        r = ref_cache(1, 1, w.head_dim, bits, w.len_max, 0, hybrid=1)
        assert oracle.quantize_pack(r, to_np(k[:, h:h + 1]), to_np(v[:, h:h + 1]), to_np(lens)) == 0
        for name in ("k_codes", "v_codes", "k_params", "v_params", "k_mode", "v_mode"):
            got = to_np(getattr(g, name)[:, h:h + 1]).view(getattr(r, name).dtype)
            assert np.array_equal(got, getattr(r, name)), (h, name)
