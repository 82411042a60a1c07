"""GPU parity of quantize/pack and append: codes, fp16 scales, fp16 mins,
residual ring and counters bit-exact with the oracle on the same seeded inputs."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq, synth

from _util import oracle_sequences, assert_cache_equal, gpu_cache, ref_cache, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _pack_both(k, v, lens, bits, cap, Nr):
    B, H, Lmax, d = k.shape
    g = gpu_cache(B, H, d, bits, cap, Nr)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), lens.to(DEV))
    st, word = kvq.kvq_read_error(g)
    r = ref_cache(B, H, d, bits, cap, Nr)
    err = oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens))
    return g, r, st, word, err


def _special_values(rng, shape):
    """fp16 data full of quantizer edge cases: ties on unit grids, constant
    groups, +-0, subnormals, tiny and huge ranges."""
    n = int(np.prod(shape))
    kind = rng.integers(0, 6, n // 32 + 1).repeat(32)[:n]
    x = rng.standard_normal(n)
    x = np.where(kind == 1, rng.integers(0, 31, n) / 2.0, x)                # ties
    x = np.where(kind == 2, np.repeat(rng.standard_normal(n // 32 + 1), 32)[:n], x)  # constant
    x = np.where(kind == 3, rng.integers(0, 50, n) * 2.0 ** -24, x)         # subnormals
    x = np.where(kind == 4, np.where(rng.random(n) < 0.5, -0.0, 0.0), x)    # signed zeros
    x = np.where(kind == 5, rng.standard_normal(n) * 3000.0, x)             # huge range
    return torch.from_numpy(x.astype(np.float16).reshape(shape))


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_pack_random_shapes(bits, d):
    rng = np.random.default_rng(bits * 7 + d)
    B, H, Lmax, Nr = 3, 2, 301, 17
    k = _special_values(rng, (B, H, Lmax, d))
    v = torch.from_numpy((rng.standard_normal((B, H, Lmax, d)) * 2).astype(np.float16))
    lens = torch.tensor([301, 9, 150], dtype=torch.int32)
    g, r, st, word, err = _pack_both(k, v, lens, bits, 290, Nr)
    assert st == kvq.KVQ_OK and word == 0 and err == 0
    assert_cache_equal(g, r)


@pytest.mark.parametrize("lens,Nr,cap", [([0, 5], 8, 10), ([8, 8], 8, 1), ([40, 1], 0, 40),
                                         ([1, 2], 1, 1)])
def test_pack_edges(lens, Nr, cap):
    rng = np.random.default_rng(sum(lens) + Nr)
    B, H, d = 2, 3, 64
    Lmax = max(max(lens), 1)
    k = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    g, r, st, word, err = _pack_both(k, v, torch.tensor(lens, dtype=torch.int32), 4, cap, Nr)
    assert st == kvq.KVQ_OK and word == 0 and err == 0
    assert_cache_equal(g, r)


def test_pack_capacity_and_bad_length_errors():
    rng = np.random.default_rng(9)
    B, H, d, Lmax = 2, 2, 64, 50
    k = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    g, r, st, word, err = _pack_both(k, k, torch.tensor([50, 20], dtype=torch.int32), 4, 30, 4)
    assert st == kvq.KVQ_ERR_CAPACITY and word & kvq.KVQ_ERRBIT_CAPACITY and err & 1
    assert_cache_equal(g, r)
    g, r, st, word, err = _pack_both(k, k, torch.tensor([51, 20], dtype=torch.int32), 4, 60, 4)
    assert word & kvq.KVQ_ERRBIT_BADLEN and err & 8
    assert int(g.packed_len[0]) == 0 and int(g.packed_len[1]) == 16
    st, word = kvq.kvq_read_error(g)
    assert st == kvq.KVQ_OK and word == 0  # cleared by the previous read


@pytest.mark.parametrize("bits", [4, 2])
def test_pack_throughput_workload_full_size(bits):
    """32768 tokens x 8 KV heads x d128 K (4 outlier channels x10) and V, Nr 0:
    every code, scale and min bit-exact."""
    w = synth.scaled(synth.WORKLOADS[5], bits=bits)
    k, v, lens = w.prefill(device=DEV)
    g, r, st, word, err = _pack_both(k, v, lens, bits, w.len_max, 0)
    assert st == kvq.KVQ_OK and err == 0
    assert_cache_equal(g, r)


@pytest.mark.parametrize("num", [1, 2, 3])
def test_pack_decode_workloads_full_size(num):
    w = synth.WORKLOADS[num]
    k, v, lens = w.prefill(device=DEV)
    g, r, st, word, err = _pack_both(k, v, lens, w.bits, w.len_max - w.residual, w.residual)
    assert st == kvq.KVQ_OK and err == 0
    assert_cache_equal(g, r)


def test_pack_ragged_batch_workload_full():
    """Llama-2-13B batch (B64, Hkv40, ragged 1024..4096, Nr96): every code,
    scale, min and window row of all 64 sequences against the oracle (one
    oracle cache per sequence, in parallel)."""
    w = synth.WORKLOADS[4]
    k, v, lens = w.prefill(device=DEV)
    cap = w.len_max - w.residual
    g = gpu_cache(w.batch, w.num_kv_heads, w.head_dim, w.bits, cap, w.residual)
    kvq.kvq_quantize_pack(g, k, v, lens.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    rs = oracle_sequences(to_np(k), to_np(v), to_np(lens), w.bits, cap, w.residual)
    for b in range(w.batch):
        assert_cache_equal(g, rs[b], batches=[b])


def _token_major(k):
    """[B][Hkv][L][d] -> a [B][L][Hkv][d] tensor, returned as its permuted
    [B][Hkv][L][d] view (the layout a prefill's projection writes)."""
    return k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


def _qkv_views(k, v, hq, seed):
    """K and V placed in a fused QKV projection output [B][L][(Hq + 2 Hkv) d]
    (random queries first), returned as the [B][Hkv][L][d] views of its key and
    value columns."""
    B, H, L, d = k.shape
    g = torch.Generator(device=k.device).manual_seed(seed)
    qkv = torch.randn(B, L, hq + 2 * H, d, generator=g, device=k.device).to(torch.float16)
    qkv[:, :, hq:hq + H] = k.permute(0, 2, 1, 3)
    qkv[:, :, hq + H:] = v.permute(0, 2, 1, 3)
    return qkv[:, :, hq:hq + H].permute(0, 2, 1, 3), qkv[:, :, hq + H:].permute(0, 2, 1, 3)


@pytest.mark.parametrize("layout", ["token", "qkv"])
@pytest.mark.parametrize("bits,d,sink,paged", [(4, 128, 0, 0), (2, 64, 5, 0), (3, 128, 0, 1),
                                               (4, 256, 3, 1), (2, 32, 0, 0)])
def test_pack_strided_layouts(layout, bits, d, sink, paged):
    """kvq_quantize_pack_strided straight from a token-major prefill or from the
    key/value columns of a fused QKV projection output: the same bytes as the
    oracle's pack of the same values (ragged lengths, window, sink, paged)."""
    rng = np.random.default_rng(bits * 100 + d + sink)
    B, H, Lmax, Nr, hq = 3, 2, 211, 9, 8
    k = _special_values(rng, (B, H, Lmax, d))
    v = torch.from_numpy((rng.standard_normal((B, H, Lmax, d)) * 2).astype(np.float16))
    lens = torch.tensor([211, 7, 160], dtype=torch.int32)
    cap = 224
    kd, vd = k.to(DEV), v.to(DEV)
    if layout == "token":
        ks, vs = _token_major(kd), _token_major(vd)
    else:
        ks, vs = _qkv_views(kd, vd, hq, 5)
    assert not ks.is_contiguous()
    g = gpu_cache(B, H, d, bits, cap, Nr, sink=sink, pages=B * cap // 32 + 3 if paged else 0,
                  seed=bits)
    kvq.kvq_quantize_pack_strided(g, ks, vs, lens.to(DEV))
    st, word = kvq.kvq_read_error(g)
    r = ref_cache(B, H, d, bits, cap, Nr, sink=sink)
    err = oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens))
    assert st == kvq.KVQ_OK and word == 0 and err == 0
    assert_cache_equal(g, r)


@pytest.mark.parametrize("layout", ["token", "qkv"])
@pytest.mark.parametrize("bits,paged", [(4, 0), (2, 0), (4, 1)])
def test_pack_strided_workload_full_size(layout, bits, paged):
    """The pack workload (32768 tokens x 8 KV heads x d128, K with outlier
    channels) packed from a token-major prefill or from the key/value columns
    of a Llama-3.1-8B fused QKV projection output (32 query heads), into a
    contiguous or a paged cache: every code, scale and min bit-exact."""
    w = synth.scaled(synth.WORKLOADS[5], bits=bits)
    k, v, lens = w.prefill(device=DEV)
    if layout == "token":
        ks, vs = _token_major(k), _token_major(v)
    else:
        ks, vs = _qkv_views(k, v, 32, 6)
    cap = w.len_max
    g = gpu_cache(w.batch, w.num_kv_heads, w.head_dim, bits, cap, 0,
                  pages=cap // 32 + 16 if paged else 0, seed=7)
    kvq.kvq_quantize_pack_strided(g, ks, vs, lens.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    del ks, vs
    r = ref_cache(w.batch, w.num_kv_heads, w.head_dim, bits, cap, 0)
    assert oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens)) == 0
    assert_cache_equal(g, r)


def test_pack_strided_rejects_bad_strides():
    g = gpu_cache(1, 2, 64, 4, 32, 0)
    k = torch.zeros(1, 2, 16, 64, dtype=torch.float16, device=DEV)
    lib = kvq.load()
    args = lambda sb, sh, st: (ctypes.byref(g.desc), ctypes.byref(g.view), kvq._ptr(k), kvq._ptr(k),
                               kvq._ptr(g.packed_len), 16, sb, sh, st, None)
    assert lib.kvq_quantize_pack_strided(*args(2048, 1024, 64)) == kvq.KVQ_OK
    assert lib.kvq_quantize_pack_strided(*args(2048, 1024, 63)) == kvq.KVQ_ERR_MISALIGNED
    assert lib.kvq_quantize_pack_strided(*args(2048, 1028, 64)) == kvq.KVQ_ERR_MISALIGNED
    assert lib.kvq_quantize_pack_strided(*args(-8, 1024, 64)) == kvq.KVQ_ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits,Nr,d", [(4, 8, 64), (2, 5, 128), (4, 0, 32), (4, 128, 128)])
def test_append_matches_oracle_and_prefill(bits, Nr, d):
    rng = np.random.default_rng(bits + Nr + d)
    B, H, L, L0 = 3, 2, 200, 2
    k = torch.from_numpy((rng.standard_normal((B, H, L, d)) * 3).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16))
    cap = L
    inc = gpu_cache(B, H, d, bits, cap, Nr)
    kvq.kvq_quantize_pack(inc, k[:, :, :L0].contiguous().to(DEV), v[:, :, :L0].contiguous().to(DEV),
                          torch.full((B,), L0, dtype=torch.int32, device=DEV))
    r = ref_cache(B, H, d, bits, cap, Nr)
    oracle.quantize_pack(r, k[:, :, :L0].numpy().copy(), v[:, :, :L0].numpy().copy(), np.full(B, L0, np.int32))
    kd, vd = k.to(DEV), v.to(DEV)
    for t in range(L0, L):
        kvq.kvq_append(inc, kd[:, :, t].contiguous(), vd[:, :, t].contiguous())
        oracle.append(r, k[:, :, t].numpy().copy(), v[:, :, t].numpy().copy())
    assert kvq.kvq_read_error(inc)[0] == kvq.KVQ_OK
    assert_cache_equal(inc, r)
    # the same bytes as packing the whole prefill at once (ring in age order)
    full = gpu_cache(B, H, d, bits, cap, Nr)
    kvq.kvq_quantize_pack(full, kd, vd, torch.full((B,), L, dtype=torch.int32, device=DEV))
    npk = L - min(L, Nr)
    for name in ("k_codes", "v_codes", "k_params", "v_params"):
        assert torch.equal(getattr(inc, name)[:, :, :npk], getattr(full, name)[:, :, :npk]), name
    for b in range(B):
        order = (int(inc.res_head[b]) + torch.arange(min(L, Nr))) % max(Nr, 1)
        assert torch.equal(inc.k_res[b][:, order.to(DEV)], full.k_res[b][:, :min(L, Nr)])


def test_append_capacity_error_leaves_cache():
    rng = np.random.default_rng(4)
    B, H, d = 2, 2, 64
    k = torch.from_numpy(rng.standard_normal((B, H, 12, d)).astype(np.float16)).to(DEV)
    g = gpu_cache(B, H, d, 4, 8, 4)
    kvq.kvq_quantize_pack(g, k, k, torch.tensor([12, 3], dtype=torch.int32, device=DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    before = [t.clone() for t in (g.k_res, g.counters, g.k_codes)]
    kvq.kvq_append(g, k[:, :, 0].contiguous(), k[:, :, 1].contiguous())
    st, word = kvq.kvq_read_error(g)
    assert st == kvq.KVQ_ERR_CAPACITY
    # sequence 0 (full) unchanged; sequence 1 (not full) took the token into its ring
    assert torch.equal(g.k_res[0], before[0][0]) and int(g.packed_len[0]) == 8
    assert int(before[1][1][1]) == 3 and int(g.res_len[1]) == 4 and int(g.packed_len[1]) == 0
