"""The allocation-free decode entry point (for callers that cannot allocate
device memory while decoding): called through the C ABI, its output must match
the regular entry point's within the attention tolerance of the other tests,
on two calls in a row (the static scratch keeps the first call's contents).
This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from bit_quantized_kv_pack_gb300 import _build, kvq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decode_noalloc_abi(cache, q, out):
    lib = kvq.load()
    st = lib.kvq_decode_attention_noalloc(
        ctypes.byref(cache.desc), ctypes.byref(cache.view), ctypes.c_void_p(q.data_ptr()),
        int(q.shape[1]), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_uint32(kvq.KVQ_OUT_F32 if out.dtype == torch.float32 else 0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_regular_decode_twice():
    _build.build()
    rng = np.random.default_rng(2024)
    B, H, gq, d, Nr = 2, 8, 4, 128, 128
    lens = torch.tensor([5000, 1300], dtype=torch.int32)
    L = int(lens.max())
    cache = kvq.KVCache(B, H, d, 4, L, Nr, device=DEV)
    k = torch.from_numpy((rng.standard_normal((B, H, L, d)) * 2).astype(np.float16)).to(DEV)
    v = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16)).to(DEV)
    kvq.kvq_quantize_pack(cache, k, v, lens.to(DEV))
    assert kvq.kvq_decode_workspace_bytes(cache.desc, H * gq) <= kvq.NOALLOC_SCRATCH_BYTES
    for call in range(2):
        q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16)).to(DEV)
        want = kvq.kvq_decode_attention(cache, q)
        got = torch.full_like(q, float("nan"))
        assert _decode_noalloc_abi(cache, q, got) == kvq.KVQ_OK
        torch.cuda.synchronize()
        diff = (got.float() - want.float()).abs().max().item()
        rel = ((got.float() - want.float()).norm() / want.float().norm()).item()
        assert diff <= 2e-3 and rel <= 1e-3, (call, diff, rel)
    st, word = kvq.kvq_read_error(cache)
    assert st == kvq.KVQ_OK and word == 0


def test_noalloc_rejects_oversized_request():
    # a description whose decode scratch exceeds the static array
    D = kvq.CacheDesc(2048, 16, 256, 4, 32, 1 << 20, 0)
    need = kvq.kvq_decode_workspace_bytes(D, 16 * 8)
    assert need > kvq.NOALLOC_SCRATCH_BYTES
    V = kvq.CacheView(*[ctypes.c_void_p(0x100000 * (i + 1)) for i in range(16)])
    st = kvq.load().kvq_decode_attention_noalloc(ctypes.byref(D), ctypes.byref(V),
                                                 ctypes.c_void_p(0x100000), 16 * 8,
                                                 ctypes.c_void_p(0x200000), 0, None)
    assert st == kvq.KVQ_ERR_UNSUPPORTED


def test_noalloc_alternating_shapes():
    """Calls that alternate between caches of different shapes (tensor-core and
    generic kernels, different batch and head counts) share the static array:
    each call after a shape change clears its counters and accumulators first,
    so every output still matches the regular entry point."""
    rng = np.random.default_rng(77)
    caches = []
    for B, H, gq, d, L in ((2, 8, 4, 128, 3000), (3, 2, 2, 64, 700), (1, 4, 1, 128, 2000)):
        c = kvq.KVCache(B, H, d, 4, L, 16, device=DEV)
        k = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16)).to(DEV)
        v = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16)).to(DEV)
        kvq.kvq_quantize_pack(c, k, v, torch.full((B,), L, dtype=torch.int32, device=DEV))
        caches.append((c, H * gq))
    for rnd in range(3):
        for c, hq in caches:
            B, d = c.desc.batch, c.desc.head_dim
            q = torch.from_numpy(rng.standard_normal((B, hq, d)).astype(np.float16)).to(DEV)
            want = kvq.kvq_decode_attention(c, q)
            got = torch.full_like(q, float("nan"))
            assert _decode_noalloc_abi(c, q, got) == kvq.KVQ_OK
            torch.cuda.synchronize()
            diff = (got.float() - want.float()).abs().max().item()
            assert diff <= 2e-3, (rnd, B, hq, d, diff)
    for c, _ in caches:
        assert kvq.kvq_read_error(c)[0] == kvq.KVQ_OK


def test_noalloc_after_a_timeout_on_a_side_stream():
    """After a call whose bounded wait ran out (the library's testing hook makes
    one run out without faulting the GPU), kvq_read_error reports the timeout and
    the next call clears the array's counters first.  That call and the ones
    after it run on a side stream (a non-blocking torch stream): the clear is
    enqueued on the caller's stream, so it is ordered before the decode there."""
    rng = np.random.default_rng(91)
    B, H, gq, d, L = 2, 4, 4, 128, 2600
    c = kvq.KVCache(B, H, d, 4, L, 32, device=DEV)
    k = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16)).to(DEV)
    v = torch.from_numpy(rng.standard_normal((B, H, L, d)).astype(np.float16)).to(DEV)
    kvq.kvq_quantize_pack(c, k, v, torch.full((B,), L, dtype=torch.int32, device=DEV))
    q = torch.from_numpy(rng.standard_normal((B, H * gq, d)).astype(np.float16)).to(DEV)
    got = torch.empty_like(q)
    kvq.kvq_testing_wait_fault(1000)
    try:
        assert _decode_noalloc_abi(c, q, got) == kvq.KVQ_OK
        st, word = kvq.kvq_read_error(c)
    finally:
        kvq.kvq_testing_wait_fault(0)
    assert st == kvq.KVQ_ERR_TIMEOUT
    want = kvq.kvq_decode_attention(c, q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for _ in range(2):
        with torch.cuda.stream(side):
            got = torch.full_like(q, float("nan"))
            assert _decode_noalloc_abi(c, q, got) == kvq.KVQ_OK
        side.synchronize()
        diff = (got.float() - want.float()).abs().max().item()
        assert diff <= 2e-3, diff
    assert kvq.kvq_read_error(c)[0] == kvq.KVQ_OK
