"""GPU parity of the paged cache (32-token pages in a pool, found through a
per-sequence block table; the paged KV cache of the TurboQuant page, section
6.1): packed rows gathered back through the block table equal the oracle's
contiguous cache bit for bit, and decode outputs are within max abs 2e-3 /
relative L2 1e-3 of the fp64 oracle.  Block tables are seeded random
injections into a pool larger than needed, so neighbouring pages of a sequence
are far apart.  A page id outside the pool raises KVQ_ERRBIT_BADPAGE: pack and
append write nothing for it, every pool access stays in bounds, and the other
sequences decode as before (that sequence's own output is undefined)."""

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq, synth

from _util import assert_attn_close, assert_cache_equal, gpu_cache, ref_cache, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _both(rng, B, H, d, bits, cap, Nr, lens, pages, S=0, hybrid=0, seed=0):
    Lmax = max(max(lens), 1)
    k = torch.from_numpy((rng.standard_normal((B, H, Lmax, d)) * 2).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    seq = torch.tensor(lens, dtype=torch.int32)
    g = gpu_cache(B, H, d, bits, cap, Nr, sink=S, hybrid=hybrid, pages=pages, seed=seed)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), seq.to(DEV))
    st, word = kvq.kvq_read_error(g)
    r = ref_cache(B, H, d, bits, cap, Nr, sink=S, hybrid=hybrid)
    err = oracle.quantize_pack(r, to_np(k), to_np(v), to_np(seq))
    return g, r, st, word, err


@pytest.mark.parametrize("bits,hybrid,S", [(4, 0, 0), (2, 0, 0), (3, 0, 0), (4, 1, 32)])
@pytest.mark.parametrize("d", [64, 128])
def test_paged_pack(bits, hybrid, S, d):
    rng = np.random.default_rng(bits * 10 + hybrid + S + d)
    B, H, cap, Nr = 3, 2, 320, 17
    lens = [cap + Nr + S, 9, 150]
    g, r, st, word, err = _both(rng, B, H, d, bits, cap, Nr, lens, 40, S, hybrid, seed=bits + d)
    assert st == kvq.KVQ_OK and word == 0 and err == 0
    assert_cache_equal(g, r)


@pytest.mark.parametrize("bits", [4, 2, 3])
@pytest.mark.parametrize("d,gq", [(128, 4), (128, 1), (64, 2)])
def test_paged_decode(bits, d, gq):
    """Tensor-core kernel (head_dim 128, page-aligned splits, four page loads per
    stage, partial last pages) and generic kernel."""
    rng = np.random.default_rng(bits * 100 + d + gq)
    B, H, cap, Nr = 3, 2, 2048, 16
    lens = [2048 + Nr, 45, 1000 + Nr]
    g, r, st, word, err = _both(rng, B, H, d, bits, cap, Nr, lens, 200, seed=d + gq)
    assert st == kvq.KVQ_OK and err == 0
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    want = oracle.decode(r, q.numpy())
    ws = kvq.workspace_for(g, H * gq)
    for _ in range(2):
        assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws), want)
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK


@pytest.mark.parametrize("fused", [False, True, "early"])
@pytest.mark.parametrize("bits,Nr,hybrid", [(4, 16, 0), (2, 0, 0), (4, 8, 1), (3, 16, 0)])
def test_paged_steps(fused, bits, Nr, hybrid):
    """Appends across page boundaries (the packed count passes multiples of
    32), through kvq_append + decode or the fused step (also with its first
    tiles copied before the grid-dependency wait)."""
    rng = np.random.default_rng(bits * 7 + Nr + bool(fused) + hybrid)
    B, H, d, gq, cap = 2, 2, 128, 4, 256
    lens = [Nr + 30, 3]
    g, r, st, word, err = _both(rng, B, H, d, bits, cap, Nr, lens, 24, hybrid=hybrid,
                                seed=bool(fused) + 1)
    flags = kvq.KVQ_STEP_EARLY_CACHE_READ if fused == "early" else 0
    assert st == kvq.KVQ_OK and err == 0
    ws = kvq.workspace_for(g, H * gq)
    for _ in range(40):
        kn = torch.from_numpy((rng.standard_normal((B, H, d)) * 2).astype(np.float16))
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
        assert_attn_close(out, oracle.decode(r, q.numpy()))
    assert_cache_equal(g, r)


def _without_packed_rows(r, b, lo, hi):
    """Sequence b of oracle cache r with packed tokens [lo, hi) left out (a
    one-sequence cache; attention does not depend on token order)."""
    B, H, d, bits, cap, Nr, S, hyb = r.shape
    o = oracle.Cache(1, H, d, bits, cap, Nr, S, hyb)
    n = int(r.packed_len[b])
    keep = np.r_[0:lo, hi:n]
    for name in ("k_codes", "v_codes", "k_params", "v_params"):
        getattr(o, name)[0, :, :len(keep)] = getattr(r, name)[b][:, keep]
    for name in ("k_res", "v_res", "k_sink", "v_sink"):
        getattr(o, name)[0] = getattr(r, name)[b]
    o.packed_len[0] = len(keep)
    o.res_len[0], o.res_head[0], o.sink_len[0] = r.res_len[b], r.res_head[b], r.sink_len[b]
    return o


def test_paged_bad_page_is_flagged_and_skipped():
    """A block-table entry outside the pool: pack flags it and writes nothing
    there; decode (both kernels) flags it and leaves that page's tokens out, so
    sequence 0's output is the attention over its other tokens and sequence 1
    is unaffected."""
    rng = np.random.default_rng(11)
    B, H, d, cap, Nr = 2, 2, 128, 256, 8
    lens = [200 + Nr, 100 + Nr]
    k = torch.from_numpy(rng.standard_normal((B, H, 208, d)).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, 208, d)).astype(np.float16))
    g = gpu_cache(B, H, d, 4, cap, Nr, pages=20, seed=3)
    g.block_table[0, 2] = 1000  # page 2 of sequence 0 (tokens 64 .. 95)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV))
    st, word = kvq.kvq_read_error(g)
    assert word == kvq.KVQ_ERRBIT_BADPAGE
    r = ref_cache(B, H, d, 4, cap, Nr)
    oracle.quantize_pack(r, k.numpy(), v.numpy(), np.array(lens, np.int32))
    r0 = _without_packed_rows(r, 0, 64, 96)
    for gq in (4, 8):  # tensor-core and generic kernels
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
        out = kvq.kvq_decode_attention(g, q.to(DEV))
        st, word = kvq.kvq_read_error(g)
        assert word & kvq.KVQ_ERRBIT_BADPAGE
        assert torch.isfinite(out).all()
        assert_attn_close(out[1:], oracle.decode(r, q.numpy())[1:])
        assert_attn_close(out[:1], oracle.decode(r0, q.numpy()[:1]))


@pytest.mark.parametrize("flags", [0, kvq.KVQ_STEP_EARLY_CACHE_READ])
def test_paged_step_into_bad_page_matches_append_then_decode(flags):
    """A fused step whose packed token lands in a page outside the pool writes
    nothing there, flags it and leaves that token out of the attention, exactly
    as kvq_append followed by kvq_decode_attention does."""
    rng = np.random.default_rng(12)
    B, H, d, cap, Nr, gq = 1, 2, 128, 128, 16, 4
    L = 64 + Nr  # 64 packed tokens: the next packed token opens page 2
    k = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16)).to(DEV)
    v = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16)).to(DEV)
    outs = []
    for fused in (True, False):
        g = gpu_cache(B, H, d, 4, cap, Nr, pages=8, seed=5)
        g.block_table[0, 2] = -1
        kvq.kvq_quantize_pack(g, k, v, torch.tensor([L], dtype=torch.int32, device=DEV))
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        rs = np.random.default_rng(13)
        kn = torch.from_numpy(rs.standard_normal((B, H, d)).astype(np.float16)).to(DEV)
        vn = torch.from_numpy(rs.standard_normal((B, H, d)).astype(np.float16)).to(DEV)
        q = torch.from_numpy(rs.standard_normal((B, H * gq, d)).astype(np.float16)).to(DEV)
        if fused:
            out = kvq.kvq_decode_step(g, q, kn, vn, flags=kvq.KVQ_OUT_F32 | flags)
        else:
            kvq.kvq_append(g, kn, vn)
            out = kvq.kvq_decode_attention(g, q, flags=kvq.KVQ_OUT_F32)
        st, word = kvq.kvq_read_error(g)
        assert word == kvq.KVQ_ERRBIT_BADPAGE
        assert g.counters[:3, 0].tolist() == [65, Nr, 1]
        outs.append(out)
    assert torch.isfinite(outs[0]).all()
    assert (outs[0] - outs[1]).abs().max().item() <= 1e-3


def test_paged_workload_full_size():
    """The Llama-3.1-8B 32K INT4 layer with its packed cache in 1024 of 1100
    shuffled 32-token pages: pack bit-exact, then three fused steps (the first
    packed token of a new page among them) against the oracle."""
    w = synth.WORKLOADS[2]
    k, v, lens = w.prefill(device=DEV)
    cap = w.len_max - w.residual + 32
    g = gpu_cache(w.batch, w.num_kv_heads, w.head_dim, w.bits, cap, w.residual, pages=1100, seed=9)
    kvq.kvq_quantize_pack(g, k, v, lens.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    r = ref_cache(w.batch, w.num_kv_heads, w.head_dim, w.bits, cap, w.residual)
    assert oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens)) == 0
    del k, v
    assert_cache_equal(g, r)
    ws = kvq.workspace_for(g, w.num_q_heads)
    for step in range(3):
        kn, vn = w.new_tokens(step)
        q = w.query(step)
        out = kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV), workspace=ws)
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        assert oracle.append(r, kn.numpy(), vn.numpy()) == 0
        err, rel = assert_attn_close(out, oracle.decode(r, q.numpy()))
        print(f"paged 32K step {step}: max abs {err:.2e}, rel L2 {rel:.2e}")
    assert_cache_equal(g, r)
