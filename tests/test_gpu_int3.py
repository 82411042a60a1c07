"""GPU parity of 3-bit codes (eight per 24 bits, TurboQuant page, section 3.1,
on the same asymmetric rule): pack, append, decode and the decode step against
the oracle -- codes, scales and mins bit-exact, outputs within max abs 2e-3 /
relative L2 1e-3 of the fp64 oracle.  head_dim 128 with up to 4 query heads
per KV head decodes on the tensor-core kernel (rows widened to INT4 in shared
memory, the fused step one launch); other shapes on the CUDA-core kernel."""

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq, synth

from _util import assert_attn_close, assert_cache_equal, gpu_cache, ref_cache, to_np
from test_gpu_pack import _special_values

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _both(k, v, lens, cap, Nr, S=0, hybrid=0):
    B, H, Lmax, d = k.shape
    g = gpu_cache(B, H, d, 3, cap, Nr, sink=S, hybrid=hybrid)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), lens.to(DEV))
    st, word = kvq.kvq_read_error(g)
    r = ref_cache(B, H, d, 3, cap, Nr, sink=S, hybrid=hybrid)
    err = oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens))
    return g, r, st, word, err


@pytest.mark.parametrize("hybrid", [0, 1])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_int3_pack(d, hybrid):
    """Special values (ties, constants, +-0, subnormals, huge ranges): every
    code byte (codes straddle bytes and 32-bit words), scale, min and mode byte."""
    rng = np.random.default_rng(300 + d + hybrid)
    B, H, Lmax, Nr = 3, 2, 301, 17
    k = _special_values(rng, (B, H, Lmax, d))
    v = torch.from_numpy((rng.standard_normal((B, H, Lmax, d)) * 2).astype(np.float16))
    lens = torch.tensor([301, 9, 150], dtype=torch.int32)
    g, r, st, word, err = _both(k, v, lens, 290, Nr, hybrid=hybrid)
    assert st == kvq.KVQ_OK and word == 0 and err == 0
    assert_cache_equal(g, r)


@pytest.mark.parametrize("d,gq,S", [(128, 4, 0), (64, 2, 32), (256, 8, 0), (32, 1, 4), (128, 1, 0),
                                    (128, 3, 32)])
def test_int3_decode(d, gq, S):
    rng = np.random.default_rng(d * 7 + gq + S)
    B, H, Nr = 3, 2, 19
    lens = torch.tensor([700, 1, 243], dtype=torch.int32)
    k = torch.from_numpy((rng.standard_normal((B, H, 700, d)) * 2).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, 700, d)).astype(np.float16))
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    g, r, st, word, err = _both(k, v, lens, 700, Nr, S)
    assert st == kvq.KVQ_OK and err == 0
    want = oracle.decode(r, q.numpy())
    assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV)), want)
    assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV), flags=kvq.KVQ_OUT_F32), want)


@pytest.mark.parametrize("fused", [False, True, "early"])
@pytest.mark.parametrize("Nr", [16, 0])
def test_int3_steps(fused, Nr):
    """Appends: the window fills, then every step packs its oldest token (or,
    with no window, the new one) -- 3-bit codes written by the append kernel."""
    rng = np.random.default_rng(40 + Nr + bool(fused))
    flags = kvq.KVQ_STEP_EARLY_CACHE_READ if fused == "early" else 0
    B, H, d, gq = 2, 2, 128, 4
    lens = torch.tensor([Nr + 200, 3], dtype=torch.int32)
    k = torch.from_numpy(rng.standard_normal((B, H, Nr + 200, d)).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, Nr + 200, d)).astype(np.float16))
    g, r, st, word, err = _both(k, v, lens, Nr + 240, Nr)
    ws = kvq.workspace_for(g, H * gq)
    for _ in range(12):
        kn = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
        vn = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
        if fused:
            out = kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV), workspace=ws,
                                      flags=flags)
        else:
            kvq.kvq_append(g, kn.to(DEV), vn.to(DEV))
            out = kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws)
        st, word = kvq.kvq_read_error(g)
        assert st == kvq.KVQ_OK and word == 0
        assert oracle.append(r, kn.numpy(), vn.numpy()) == 0
        assert_cache_equal(g, r)
        assert_attn_close(out, oracle.decode(r, q.numpy()))


def test_int3_workload_full_size():
    """The Llama-3.1-8B 32K layer (B1, Hq32, Hkv8, d128, 128-token window) with
    3-bit codes: pack bit-exact, then two decode steps, every output row against
    the oracle."""
    w = synth.scaled(synth.WORKLOADS[2], bits=3)
    k, v, lens = w.prefill(device=DEV)
    cap = w.len_max - w.residual + 8
    g = gpu_cache(w.batch, w.num_kv_heads, w.head_dim, 3, cap, w.residual)
    kvq.kvq_quantize_pack(g, k, v, lens.to(DEV))
    r = ref_cache(w.batch, w.num_kv_heads, w.head_dim, 3, cap, w.residual)
    assert oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens)) == 0
    del k, v
    assert_cache_equal(g, r)
    for step in range(2):
        kn, vn = w.new_tokens(step)
        q = w.query(step)
        out = kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV))
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        assert oracle.append(r, kn.numpy(), vn.numpy()) == 0
        err, rel = assert_attn_close(out, oracle.decode(r, q.numpy()))
        print(f"3-bit 32K step {step}: max abs {err:.2e}, rel L2 {rel:.2e}")
    assert_cache_equal(g, r)
