"""The bounded-wait error path of the tensor-core decode, exercised without a
GPU fault: the library's testing hook arms one tile's barrier for 16 bytes more
than its copies deliver and shortens the wait limit to a millisecond.  Every
copy still completes, so nothing is in flight when the CTA gives up.  The call
must report KVQ_ERR_TIMEOUT, leave every other head's output and the cache
itself correct, and the next call (after the workspace is zeroed again, as the
header asks) must match the oracle."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq

from _util import assert_attn_close, assert_cache_equal, ref_cache

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _fault(limit_us: int) -> None:
    lib = kvq.load()
    lib.kvq_testing_wait_fault.argtypes = [ctypes.c_uint32]
    lib.kvq_testing_wait_fault.restype = None
    lib.kvq_testing_wait_fault(limit_us)


def _setup(seed, B=2, H=2, L=3000, Nr=16, gq=4):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((B, H, L, 128)).astype(np.float16)
    v = rng.standard_normal((B, H, L, 128)).astype(np.float16)
    lens = np.array([L, L - 500], np.int32)
    g = kvq.KVCache(B, H, 128, 4, L + 8, Nr, device=DEV)
    kvq.kvq_quantize_pack(g, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV),
                          torch.from_numpy(lens).to(DEV))
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    r = ref_cache(B, H, 128, 4, L + 8, Nr)
    assert oracle.quantize_pack(r, k, v, lens) == 0
    return rng, g, r


def test_decode_wait_runs_out_and_reports_timeout():
    rng, g, r = _setup(31)
    B, Hq = 2, 8
    ws = kvq.workspace_for(g, Hq)
    q = rng.standard_normal((B, Hq, 128)).astype(np.float16)
    _fault(1000)
    try:
        out = kvq.kvq_decode_attention(g, torch.from_numpy(q).to(DEV), workspace=ws,
                                       flags=kvq.KVQ_OUT_F32)
        st, word = kvq.kvq_read_error(g)
    finally:
        _fault(0)
    assert st == kvq.KVQ_ERR_TIMEOUT and word == kvq.KVQ_ERRBIT_TIMEOUT
    want = oracle.decode(r, q)
    # query heads 0..3 use KV head 0 of sequence 0, whose split 0 gave up
    assert torch.isfinite(out).all()
    assert_attn_close(out[0, 4:], want[0, 4:])
    assert_attn_close(out[1], want[1])
    ws.zero_()
    for _ in range(2):
        out = kvq.kvq_decode_attention(g, torch.from_numpy(q).to(DEV), workspace=ws)
        assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
        assert_attn_close(out, want)


def test_step_wait_runs_out_and_the_append_still_lands():
    """A fused step whose split gives up still performs the append exactly:
    the cache after it equals the oracle's after the same append."""
    rng, g, r = _setup(32)
    B, Hq = 2, 8
    ws = kvq.workspace_for(g, Hq)
    kn = rng.standard_normal((B, 2, 128)).astype(np.float16)
    vn = rng.standard_normal((B, 2, 128)).astype(np.float16)
    q = rng.standard_normal((B, Hq, 128)).astype(np.float16)
    _fault(1000)
    try:
        out = kvq.kvq_decode_step(g, torch.from_numpy(q).to(DEV), torch.from_numpy(kn).to(DEV),
                                  torch.from_numpy(vn).to(DEV), workspace=ws)
        st, word = kvq.kvq_read_error(g)
    finally:
        _fault(0)
    assert st == kvq.KVQ_ERR_TIMEOUT
    assert oracle.append(r, kn, vn) == 0
    assert_cache_equal(g, r)
    want = oracle.decode(r, q)
    assert_attn_close(out[0, 4:], want[0, 4:])
    assert_attn_close(out[1], want[1])
    ws.zero_()
    q2 = rng.standard_normal((B, Hq, 128)).astype(np.float16)
    out = kvq.kvq_decode_attention(g, torch.from_numpy(q2).to(DEV), workspace=ws)
    assert kvq.kvq_read_error(g)[0] == kvq.KVQ_OK
    assert_attn_close(out, oracle.decode(r, q2))
