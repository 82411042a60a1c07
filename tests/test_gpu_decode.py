"""GPU parity of decode attention: the fp16 output of the CUDA path against the
fp64 oracle on the same packed cache, within max abs 2e-3 and relative L2 1e-3,
on the five workloads' decode shapes (the batched one sampled) and a sweep of
small shapes with ragged tails; plus the device-side error paths."""

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq, synth

from _util import (assert_attn_close, assert_cache_equal, attn_errors, gpu_cache, oracle_sequences,
                   per_sequence, ref_cache, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(k, v, lens, bits, cap, Nr):
    B, H, Lmax, d = k.shape
    g = gpu_cache(B, H, d, bits, cap, Nr)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), lens.to(DEV))
    r = ref_cache(B, H, d, bits, cap, Nr)
    assert oracle.quantize_pack(r, to_np(k), to_np(v), to_np(lens)) == 0
    return g, r


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("d,gq", [(32, 1), (64, 2), (128, 4), (128, 3), (256, 8), (64, 16), (128, 5)])
def test_decode_sweep(bits, d, gq):
    rng = np.random.default_rng(bits * 1000 + d * 10 + gq)
    B, H, Nr = 3, 2, 19
    lens = torch.tensor([700, 1, 243], dtype=torch.int32)
    Lmax = int(lens.max())
    k = torch.from_numpy((rng.standard_normal((B, H, Lmax, d)) * 2).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    g, r = _setup(k, v, lens, bits, Lmax, Nr)
    ws = kvq.workspace_for(g, H * gq)
    out = kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws)
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    want = oracle.decode(r, q.numpy())
    assert_attn_close(out, want)
    # the workspace is left ready: a second call through it is as good
    again = kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws)
    assert_attn_close(again, want)


@pytest.mark.parametrize("Nr", [0, 64])
def test_decode_residual_only_and_packed_only(Nr):
    rng = np.random.default_rng(Nr + 5)
    B, H, d, gq = 2, 2, 128, 4
    lens = torch.tensor([40, 64], dtype=torch.int32)
    k = torch.from_numpy(rng.standard_normal((B, H, 64, d)).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, 64, d)).astype(np.float16))
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    g, r = _setup(k, v, lens, 4, 64, Nr)
    out = kvq.kvq_decode_attention(g, q.to(DEV))
    assert_attn_close(out, oracle.decode(r, q.numpy()))


def test_decode_empty_sequence_sets_error_and_zeros():
    rng = np.random.default_rng(77)
    B, H, d = 2, 1, 64
    k = torch.from_numpy(rng.standard_normal((B, H, 10, d)).astype(np.float16))
    lens = torch.tensor([10, 0], dtype=torch.int32)
    g, r = _setup(k, k, lens, 4, 10, 4)
    q = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
    out = kvq.kvq_decode_attention(g, q.to(DEV))
    st, word = kvq.kvq_read_error(g)
    assert st == kvq.KVQ_ERR_EMPTY and word == kvq.KVQ_ERRBIT_EMPTY
    assert torch.all(out[1] == 0)
    want = oracle.decode(r, q.numpy())
    assert_attn_close(out[:1], want[:1])


@pytest.mark.parametrize("num", [1, 2, 3])
def test_decode_workload_full_size(num):
    """Workloads 1-3 at full size: prefill packed (Nr in the residual), then one
    decode step of append + attention, every output row against the oracle."""
    w = synth.WORKLOADS[num]
    k, v, lens = w.prefill(device=DEV)
    cap = w.len_max - w.residual + 8
    g, r = _setup(k, v, lens, w.bits, cap, w.residual)
    kn, vn = w.new_tokens(0)
    kvq.kvq_append(g, kn.to(DEV), vn.to(DEV))
    oracle.append(r, kn.numpy(), vn.numpy())
    q = w.query(0)
    out = kvq.kvq_decode_attention(g, q.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    err, rel = assert_attn_close(out, oracle.decode(r, q.numpy()))
    print(f"workload {num}: max abs {err:.2e}, rel L2 {rel:.2e}")


def test_decode_ragged_batch_workload_full():
    """Llama-2-13B batch at full size (B64, 40 heads, ragged 1024..4096, Nr96):
    every packed byte of all 64 sequences and all 2560 (sequence, head) output
    rows against the oracle (one oracle cache per sequence, in parallel)."""
    w = synth.WORKLOADS[4]
    k, v, lens = w.prefill(device=DEV)
    cap = w.len_max - w.residual
    g = gpu_cache(w.batch, w.num_kv_heads, w.head_dim, w.bits, cap, w.residual)
    kvq.kvq_quantize_pack(g, k, v, lens.to(DEV))
    q = w.query(0)
    out = kvq.kvq_decode_attention(g, q.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    rs = oracle_sequences(to_np(k), to_np(v), to_np(lens), w.bits, cap, w.residual)
    del k, v
    for b in range(w.batch):
        assert_cache_equal(g, rs[b], batches=[b])
    qn = q.numpy()
    want = np.concatenate(per_sequence(lambda b: oracle.decode(rs[b], qn[b:b + 1]), w.batch))
    err, rel = assert_attn_close(out, want)
    print(f"workload 4 (all 2560 rows): max abs {err:.2e}, rel L2 {rel:.2e}")


def test_decode_is_stream_ordered():
    """Two decodes on a side stream, the second reusing the first's workspace:
    both match the oracle (the tensor-core path adds split results with fp32
    atomics, so the bytes may differ by rounding between runs)."""
    rng = np.random.default_rng(8)
    B, H, d, L = 1, 8, 128, 3000
    k = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16))
    g, r = _setup(k, k, torch.tensor([L], dtype=torch.int32), 4, L, 128)
    qh = rng.standard_normal((B, 32, d)).astype(np.float16)
    q = torch.from_numpy(qh).to(DEV)
    ws = kvq.workspace_for(g, 32)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        a = kvq.kvq_decode_attention(g, q, workspace=ws)
        b = kvq.kvq_decode_attention(g, q, workspace=ws)
    s.synchronize()
    want = oracle.decode(r, qh)
    assert_attn_close(a, want)
    assert_attn_close(b, want)


@pytest.mark.parametrize("bits", [4, 2])
def test_decode_far_max_takes_exact_merge(bits):
    """One packed token whose score is hundreds of log2 units above the rest,
    outside the first tile of every split: the splits' shared reference (their
    first-tile maxima) is far below it, so the head falls back to the
    log-sum-exp merge of the split partials; the output must still be the
    oracle's (here essentially that token's value row)."""
    rng = np.random.default_rng(40 + bits)
    B, H, d, gq, L, Nr = 1, 1, 128, 4, 2000, 16
    k = rng.standard_normal((B, H, L, d))
    v = rng.standard_normal((B, H, L, d))
    q = rng.standard_normal((B, H * gq, d))
    k[0, 0, 200] = 40.0 * q[0, 0]  # query 0 scores this token ~450/sqrt(d) higher
    k, v, q = (torch.from_numpy(x.astype(np.float16)) for x in (k, v, q))
    g, r = _setup(k, v, torch.tensor([L], dtype=torch.int32), bits, L, Nr)
    want = oracle.decode(r, q.numpy())
    for _ in range(2):  # the second call checks that the fallback left the workspace ready
        out = kvq.kvq_decode_attention(g, q.to(DEV))
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        assert_attn_close(out, want)
    # and a call without the far token is back on the common path, still exact
    q2 = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    assert_attn_close(kvq.kvq_decode_attention(g, q2.to(DEV)), oracle.decode(r, q2.numpy()))


def _with_outliers(rng, shape, p=0.01):
    """N(0, 1) with a fraction p (1%: workload 4's recipe) of the elements
    replaced by N(0, 8^2)."""
    x = rng.standard_normal(shape)
    x = np.where(rng.random(shape) < p, rng.standard_normal(shape) * 8.0, x)
    return torch.from_numpy(x.astype(np.float16))


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("d,gq", [(128, 4), (64, 2), (128, 8)])
def test_decode_fp32_output(bits, d, gq):
    """KVQ_OUT_F32: the same decode written as fp32, on outlier data with sharp
    attention (|O| up to about 13, where the fp16 spacing is 2^-7).  Against the
    oracle with the flat max-abs bar, which fp16 output alone can miss there.  On
    the generic kernel (deterministic) rounding the fp32 output to fp16 gives the
    fp16 output bit for bit; the allocation-free entry point writes fp32 too."""
    rng = np.random.default_rng(d * 10 + gq + bits)
    B, H, Nr = 2, 2, 16
    lens = torch.tensor([900, 50], dtype=torch.int32)
    k, v = _with_outliers(rng, (B, H, 900, d)), _with_outliers(rng, (B, H, 900, d))
    q = torch.from_numpy((rng.standard_normal((B, H * gq, d)) * 2).astype(np.float16))
    g, r = _setup(k, v, lens, bits, 900, Nr)
    want = oracle.decode(r, q.numpy())
    assert np.abs(want).max() > 2
    out32 = kvq.kvq_decode_attention(g, q.to(DEV), flags=kvq.KVQ_OUT_F32)
    assert out32.dtype == torch.float32
    assert_attn_close(out32, want)
    out16 = kvq.kvq_decode_attention(g, q.to(DEV))
    assert out16.dtype == torch.float16
    assert_attn_close(out16, want)
    if not (d == 128 and gq <= 4):
        assert torch.equal(out32.half(), out16)
    noalloc = kvq.kvq_decode_attention_noalloc(g, q.to(DEV), torch.empty_like(out32))
    assert_attn_close(noalloc, want)


@pytest.mark.parametrize("bits", [4, 2, 3])
@pytest.mark.parametrize("pages,hybrid,sink,Nr", [(0, 0, 0, 16), (64 * 40, 0, 0, 16), (0, 1, 8, 16),
                                                  (0, 0, 32, 96)])
def test_decode_several_waves(bits, pages, hybrid, sink, Nr):
    """A batch whose grid runs in several waves (40 sequences x 8 KV heads): the
    4-CTAs-per-SM variant of the tensor-core kernel, where the last packed
    split of each head also takes the fp16 rows (in two passes of 64 when the
    window and the sink hold more); plain, paged, hybrid with a sink, and a
    96-token window with a 32-token sink; decode and three fused steps against
    the oracle, bytes bit for bit."""
    rng = np.random.default_rng(bits * 100 + bool(pages) * 10 + hybrid + Nr)
    B, H, d, gq, cap = 40, 8, 128, 4, 320
    lens = [int(x) for x in rng.integers(1, cap + Nr + sink - 3, B)]
    Lmax = max(lens)
    k = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    seq = torch.tensor(lens, dtype=torch.int32)
    g = gpu_cache(B, H, d, bits, cap, Nr, sink=sink, hybrid=hybrid, pages=pages, seed=bits)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), seq.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    rs = oracle_sequences(to_np(k), to_np(v), to_np(seq), bits, cap, Nr, sink, hybrid)
    ws = kvq.workspace_for(g, H * gq)
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    qn = q.numpy()
    want = np.concatenate(per_sequence(lambda b: oracle.decode(rs[b], qn[b:b + 1]), B))
    assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws), want)
    for step in range(3):
        kn = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
        vn = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
        out = kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV), workspace=ws)
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        knn, vnn, qn = kn.numpy(), vn.numpy(), q.numpy()
        assert all(e == 0 for e in per_sequence(
            lambda b: oracle.append(rs[b], knn[b:b + 1], vnn[b:b + 1]), B))
        want = np.concatenate(per_sequence(lambda b: oracle.decode(rs[b], qn[b:b + 1]), B))
        assert_attn_close(out, want)
    for b in range(B):
        assert_cache_equal(g, rs[b], batches=[b])


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("gq", [4, 1])
def test_decode_single_split(bits, gq):
    """Short sequences and no window, so each (sequence, KV head) is one split
    that writes its output straight from its own state; a sequence of one
    token among them."""
    rng = np.random.default_rng(7 * bits + gq)
    B, H, d, cap = 3, 2, 128, 200
    lens = torch.tensor([200, 1, 77], dtype=torch.int32)
    k = torch.from_numpy(rng.standard_normal((B, H, 200, d)).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, 200, d)).astype(np.float16))
    g, r = _setup(k, v, lens, bits, cap, 0)
    ws = kvq.workspace_for(g, H * gq)
    for _ in range(2):
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
        out = kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws, flags=kvq.KVQ_OUT_F32)
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        assert_attn_close(out, oracle.decode(r, q.numpy()))


def test_decode_tall_tiles():
    """INT2 splits long enough for the 192-token tiles (4 sequences x 8 KV heads
    of up to 20,000 packed tokens: 13 packed splits per head in one wave on a
    152-SM GB300, about 1,540 tokens each), ragged so the splits end inside a
    tile at different rows; decode and two fused steps against the oracle,
    bytes bit for bit."""
    rng = np.random.default_rng(192)
    B, H, d, gq, cap, Nr = 4, 8, 128, 4, 20000, 16
    lens = [cap + Nr - 2, 19001, 12345, 3001]  # room for the two steps' packed tokens
    Lmax = max(lens)
    k = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    v = torch.from_numpy(rng.standard_normal((B, H, Lmax, d)).astype(np.float16))
    seq = torch.tensor(lens, dtype=torch.int32)
    g = gpu_cache(B, H, d, 2, cap, Nr, seed=2)
    kvq.kvq_quantize_pack(g, k.to(DEV), v.to(DEV), seq.to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    rs = oracle_sequences(to_np(k), to_np(v), to_np(seq), 2, cap, Nr)
    del k, v
    ws = kvq.workspace_for(g, H * gq)
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
    qn = q.numpy()
    want = np.concatenate(per_sequence(lambda b: oracle.decode(rs[b], qn[b:b + 1]), B))
    assert_attn_close(kvq.kvq_decode_attention(g, q.to(DEV), workspace=ws, flags=kvq.KVQ_OUT_F32), want)
    for _ in range(2):
        kn = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
        vn = torch.from_numpy(rng.standard_normal((B, H, d)).astype(np.float16))
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16))
        out = kvq.kvq_decode_step(g, q.to(DEV), kn.to(DEV), vn.to(DEV), workspace=ws)
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        knn, vnn, qn = kn.numpy(), vn.numpy(), q.numpy()
        assert all(e == 0 for e in per_sequence(
            lambda b: oracle.append(rs[b], knn[b:b + 1], vnn[b:b + 1]), B))
        want = np.concatenate(per_sequence(lambda b: oracle.decode(rs[b], qn[b:b + 1]), B))
        assert_attn_close(out, want)
    for b in range(B):
        assert_cache_equal(g, rs[b], batches=[b])
