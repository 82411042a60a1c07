"""GPU parity of the attention-sink window (the first tokens of each sequence
kept in fp16, set at prefill and fixed afterwards; InnerQ page, section 2.3):
pack, append, decode and the fused step against the oracle -- cache bytes and
counters bit-exact, outputs within max abs 2e-3 / relative L2 1e-3 of the fp64
oracle.  Sink lengths cover one row, a partial and a full 64-row sink split,
several sink splits and the 256-row maximum; sequences shorter than the sink,
with nothing packed, and empty ones."""

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq, synth

from _util import assert_attn_close, assert_cache_equal, gpu_cache, ref_cache, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(rng, B, H, d, bits, cap, Nr, S, lens, kscale=2.0):
    Lmax = max(max(lens), 1)
    k = torch.from_numpy((rng.standard_normal((B, H, Lmax, d)) * kscale).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    seq = torch.tensor(lens, dtype=torch.int32)
    g = gpu_cache(B, H, d, bits, cap, Nr, sink=S)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), seq.to(DEV))
    st, word = kvq.kvq_read_error(g)
    r = ref_cache(B, H, d, bits, cap, Nr, sink=S)
    err = oracle.quantize_pack(r, to_np(k), to_np(v), to_np(seq))
    return g, r, st, word, err


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("d,S", [(64, 1), (128, 32), (128, 100), (256, 256), (32, 64)])
def test_sink_pack(bits, d, S):
    """Sink rows, packed rows shifted past the sink, window and all four
    counters equal the oracle's, for sequences longer and shorter than the sink."""
    rng = np.random.default_rng(bits * 1000 + d + S)
    lens = [S + 300, 5, 0, S + 3]
    g, r, st, word, err = _setup(rng, 4, 2, d, bits, 400, 17, S, lens)
    assert st == kvq.KVQ_OK and word == 0 and err == 0
    assert_cache_equal(g, r)
    assert to_np(g.sink_len).tolist() == [S, min(5, S), 0, S]


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("d,gq,S,Nr", [(128, 4, 32, 96), (128, 4, 130, 0), (128, 1, 256, 64),
                                       (128, 3, 1, 19), (64, 2, 32, 96), (256, 8, 100, 5)])
def test_sink_decode(bits, d, gq, S, Nr):
    """Decode over sink + packed + window: head_dim 128 with up to 4 query heads
    per KV head runs the tensor-core kernel (64-row fp16 splits over the window
    slots and then the sink rows: one split holding both, a sink-only layout,
    up to five splits), the rest the generic one.  Lengths: a long sequence, one inside the sink, one with
    nothing packed, and one with a single packed token."""
    rng = np.random.default_rng(bits * 7919 + d * 13 + gq * 3 + S + Nr)
    B, H = 4, 2
    lens = [S + Nr + 700, max(S - 1, 1), S + Nr, S + Nr + 1]
    g, r, st, word, err = _setup(rng, B, H, d, bits, 720, Nr, S, lens)
    assert st == kvq.KVQ_OK and err == 0
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    ws = kvq.workspace_for(g, H * gq)
    want = oracle.decode(r, q.numpy())
    for _ in range(2):  # the workspace is left ready for the next call
        out = kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws)
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        assert_attn_close(out, want)


def test_sink_dominates():
    """Keys of the sink rows aligned with q and everything else orthogonal to it:
    the output is (nearly) the mean of the sink values, so a dropped or
    misplaced sink row shows at once."""
    rng = np.random.default_rng(77)
    B, H, d, gq, S, Nr, L = 1, 1, 128, 4, 8, 16, 500
    q = np.zeros((B, H * gq, d), np.float16)
    q[..., 0] = 16.0
    k = (rng.standard_normal((B, H, L, d)) * 0.05).astype(np.float16)
    k[..., 0] = 0.0
    k[:, :, :S, 0] = 16.0
    v = rng.standard_normal((B, H, L, d)).astype(np.float16)
    g = gpu_cache(B, H, d, 4, L, Nr, sink=S)
    kvq.kvq_quantize_pack(g, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV),
                          torch.tensor([L], dtype=torch.int32, device=DEV))
    r = ref_cache(B, H, d, 4, L, Nr, sink=S)
    oracle.quantize_pack(r, k, v, np.array([L], np.int32))
    out = kvq.kvq_decode_attention(g, torch.from_numpy(q).to(DEV))
    want = oracle.decode(r, q)
    assert_attn_close(out, want)
    assert np.abs(want[0, 0] - v[0, 0, :S].astype(np.float64).mean(0)).max() < 1e-3


def test_sink_empty_sequence_flags_empty():
    rng = np.random.default_rng(3)
    g, r, st, word, err = _setup(rng, 2, 2, 128, 4, 64, 8, 16, [0, 40])
    q = torch.from_numpy(rng.standard_normal((2, 8, 128)).astype(np.float16))
    out = kvq.kvq_decode_attention(g, q.to(DEV))
    st, word = kvq.kvq_read_error(g)
    assert word == kvq.KVQ_ERRBIT_EMPTY
    assert torch.all(out[0] == 0)
    assert_attn_close(out[1:], oracle.decode(r, q.numpy())[1:])


def _steps(rng, B, H, d, gq, bits, cap, Nr, S, lens, nsteps, fused, flags=0):
    g, r, st, word, err = _setup(rng, B, H, d, bits, cap, Nr, S, lens)
    assert st == kvq.KVQ_OK and err == 0
    ws = kvq.workspace_for(g, H * gq)
    sink0 = (g.k_sink.clone(), g.v_sink.clone(), g.sink_len.clone())
    for _ in range(nsteps):
        kn = torch.from_numpy((rng.standard_normal((B, H, d)) * 2).astype(np.float16))
        vn = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
        if fused:
            out = kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV), workspace=ws, flags=flags)
        else:
            kvq.kvq_append(g, kn.to(DEV), vn.to(DEV))
            out = kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws)
        st, word = kvq.kvq_read_error(g)
        e = oracle.append(r, kn.numpy(), vn.numpy())
        assert st == kvq.KVQ_OK and word == 0 and e == 0
        assert_cache_equal(g, r)
        assert_attn_close(out, oracle.decode(r, q.numpy()))
    # the sink never moves after the prefill
    assert torch.equal(g.k_sink, sink0[0]) and torch.equal(g.v_sink, sink0[1])
    assert torch.equal(g.sink_len, sink0[2])


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("bits,Nr,S", [(4, 16, 32), (2, 0, 100), (4, 96, 32)])
def test_sink_steps_tensor_core(fused, bits, Nr, S):
    """Appends after a prefill with a sink, through kvq_append + decode or the
    fused step: one sequence inside its sink (its tokens then fill the window),
    one with a window that fills, one that packs every step."""
    rng = np.random.default_rng(bits * 31 + Nr + S + fused)
    _steps(rng, 3, 2, 128, 4, bits, 900, Nr, S, [S - 5, S + 3, S + Nr + 600], 12, fused)


def test_sink_steps_early_cache_read():
    rng = np.random.default_rng(1234)
    _steps(rng, 2, 2, 128, 4, 4, 900, 16, 32, [700, 20], 8, True, kvq.KVQ_STEP_EARLY_CACHE_READ)


@pytest.mark.parametrize("fused", [False, True])
def test_sink_steps_generic(fused):
    rng = np.random.default_rng(55 + fused)
    _steps(rng, 2, 2, 64, 2, 4, 300, 8, 32, [20, 200], 8, fused)


def test_sink_workload_full_size():
    """Llama-2-13B decode batch of 64 ragged sequences (1K-4K tokens, INT4,
    96-token window) with the 32-token sink of the InnerQ page's two windows:
    pack bit-exact on sampled sequences, then three fused steps (fp32 output,
    flat bar) each followed by a decode with fp16 output, every output row of
    the sampled sequences against the oracle."""
    w = synth.WORKLOADS[4]
    S = 32
    k, v, lens = w.prefill(device=DEV)
    cap = w.len_max - w.residual - S + 8
    g = gpu_cache(w.batch, w.num_kv_heads, w.head_dim, w.bits, cap, w.residual, sink=S)
    kvq.kvq_quantize_pack(g, k, v, lens.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    sample = [0, 17, 63]
    r = ref_cache(len(sample), w.num_kv_heads, w.head_dim, w.bits, cap, w.residual, sink=S)
    sl = lens[sample]
    Lm = int(sl.max())
    assert oracle.quantize_pack(r, to_np(k[sample, :, :Lm]), to_np(v[sample, :, :Lm]), to_np(sl)) == 0
    del k, v
    assert_cache_equal(g, r, batches=sample)
    ws = kvq.workspace_for(g, w.num_q_heads)
    for step in range(3):
        kn, vn = w.new_tokens(step)
        q = w.query(step)
        out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
        kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV), out, ws)
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        assert oracle.append(r, kn[sample].numpy(), vn[sample].numpy()) == 0
        want = oracle.decode(r, q[sample].numpy())
        assert_attn_close(out[sample], want)
        assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws)[sample], want)
    assert_cache_equal(g, r, batches=sample)
