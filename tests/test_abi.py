"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/kvq.h declares, and the pure host entry points
(sizes, status strings, argument validation) behave as documented.  Calls that
would launch kernels are only made with arguments the host rejects."""

import ctypes
import os
import re

import pytest

from bit_quantized_kv_pack_gb300 import _build, kvq

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kvq.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(kvq_\w+)\s*\(", text, re.M)))


def test_header_declares_and_library_exports(lib):
    names = _declared()
    assert set(kvq.EXPORTS) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in kvq.h but not exported"
    assert kvq.kvq_version() == 160


def test_status_strings(lib):
    for code in range(8):
        assert kvq.status_string(code) and kvq.status_string(code) != "unknown status"
    assert kvq.status_string(99) == "unknown status"


def _desc(**kw):
    base = dict(batch=2, num_kv_heads=8, head_dim=128, bits=4, group=32, capacity=1000, residual=128)
    base.update(kw)
    return kvq.CacheDesc(**base)


def test_cache_bytes(lib):
    D = _desc()
    assert kvq.kvq_cache_bytes(D, kvq.KVQ_ARRAY_CODES) == 2 * 8 * 1000 * 64
    assert kvq.kvq_cache_bytes(D, kvq.KVQ_ARRAY_PARAMS) == 2 * 8 * 1000 * 4 * 4
    assert kvq.kvq_cache_bytes(D, kvq.KVQ_ARRAY_RESIDUAL) == 2 * 8 * 128 * 128 * 2
    assert kvq.kvq_cache_bytes(_desc(bits=3), kvq.KVQ_ARRAY_CODES) == 2 * 8 * 1000 * 48
    D2 = _desc(bits=2, head_dim=64)
    assert kvq.kvq_cache_bytes(D2, kvq.KVQ_ARRAY_CODES) == 2 * 8 * 1000 * 16
    assert kvq.kvq_cache_bytes(D2, kvq.KVQ_ARRAY_PARAMS) == 2 * 8 * 1000 * 2 * 4
    assert kvq.kvq_cache_bytes(D, kvq.KVQ_ARRAY_SINK) == 0
    assert kvq.kvq_cache_bytes(_desc(sink=32), kvq.KVQ_ARRAY_SINK) == 2 * 8 * 32 * 128 * 2
    assert kvq.kvq_cache_bytes(D, kvq.KVQ_ARRAY_MODE) == 0
    assert kvq.kvq_cache_bytes(_desc(hybrid=1), kvq.KVQ_ARRAY_MODE) == 2 * 8 * 1000
    # paged: the arrays are sized for the pool of pages [page][head][32]
    P = _desc(capacity=1024, page_size=32, num_pages=70, hybrid=1)
    assert kvq.kvq_cache_bytes(P, kvq.KVQ_ARRAY_CODES) == 70 * 8 * 32 * 64
    assert kvq.kvq_cache_bytes(P, kvq.KVQ_ARRAY_PARAMS) == 70 * 8 * 32 * 16
    assert kvq.kvq_cache_bytes(P, kvq.KVQ_ARRAY_MODE) == 70 * 8 * 32
    assert kvq.kvq_cache_bytes(D, 7) == 0
    for bad in (dict(bits=5), dict(bits=1), dict(head_dim=96), dict(head_dim=100), dict(group=64),
                dict(batch=0), dict(residual=-1), dict(residual=2000), dict(capacity=-5),
                dict(sink=-1), dict(sink=257), dict(hybrid=2), dict(hybrid=-1),
                dict(page_size=16, num_pages=8), dict(page_size=32, num_pages=0),
                dict(page_size=32, num_pages=4, capacity=1000)):
        assert kvq.kvq_cache_bytes(_desc(**bad), kvq.KVQ_ARRAY_CODES) == 0, bad


def test_workspace_bytes(lib):
    D = _desc()
    n = kvq.kvq_decode_workspace_bytes(D, 32)
    assert n > 0 and n % 8 == 0
    assert kvq.kvq_decode_workspace_bytes(D, 12) == 0  # 12 % 8 != 0
    assert kvq.kvq_decode_workspace_bytes(D, 0) == 0


def _view(addr=0x10000):
    # fake, well-aligned addresses: only ever passed to calls the host rejects
    return kvq.CacheView(*[ctypes.c_void_p(addr + 0x1000 * i) for i in range(16)])


@pytest.mark.parametrize("kw,expect", [
    (dict(bits=5), kvq.KVQ_ERR_UNSUPPORTED),
    (dict(head_dim=96), kvq.KVQ_ERR_UNSUPPORTED),
    (dict(head_dim=40), kvq.KVQ_ERR_INVALID_ARG),
    (dict(group=16), kvq.KVQ_ERR_INVALID_ARG),
    (dict(batch=0), kvq.KVQ_ERR_INVALID_ARG),
    (dict(sink=-2), kvq.KVQ_ERR_INVALID_ARG),
    (dict(sink=512), kvq.KVQ_ERR_UNSUPPORTED),
    (dict(hybrid=3), kvq.KVQ_ERR_INVALID_ARG),
])
def test_rejects_bad_desc(lib, kw, expect):
    D, V = _desc(**kw), _view()
    P = ctypes.c_void_p
    assert lib.kvq_quantize_pack(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000),
                                 P(0x300000), 16, None) == expect
    assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000), None) == expect
    assert lib.kvq_decode_attention(ctypes.byref(D), ctypes.byref(V), P(0x100000), 8, P(0x200000),
                                    P(0x300000), 1 << 30, 0, None) == expect


def test_rejects_bad_view_and_args(lib):
    D = _desc()
    P = ctypes.c_void_p
    assert lib.kvq_append(ctypes.byref(D), None, P(0x100000), P(0x200000), None) == kvq.KVQ_ERR_INVALID_ARG
    V = _view()
    V.k_codes = 0
    assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000), None) == kvq.KVQ_ERR_INVALID_ARG
    V = _view()
    V.k_params = 0x10008  # 8-byte aligned only
    assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000), None) == kvq.KVQ_ERR_MISALIGNED
    V = _view()
    assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), P(0x100004), P(0x200000), None) == kvq.KVQ_ERR_MISALIGNED
    assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), None, P(0x200000), None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_quantize_pack(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000),
                                 P(0x300000), -1, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_quantize_pack(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000),
                                 None, 16, None) == kvq.KVQ_ERR_INVALID_ARG
    # decode: Hq not a multiple of Hkv, too small a workspace, misaligned q
    assert lib.kvq_decode_attention(ctypes.byref(D), ctypes.byref(V), P(0x100000), 12, P(0x200000),
                                    P(0x300000), 1 << 30, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    need = kvq.kvq_decode_workspace_bytes(D, 32)
    assert lib.kvq_decode_attention(ctypes.byref(D), ctypes.byref(V), P(0x100000), 32, P(0x200000),
                                    P(0x300000), need - 1, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attention(ctypes.byref(D), ctypes.byref(V), P(0x100002), 32, P(0x200000),
                                    P(0x300000), need, 0, None) == kvq.KVQ_ERR_MISALIGNED
    # flags: only KVQ_OUT_F32 (the misaligned q then fails, so nothing launches)
    assert lib.kvq_decode_attention(ctypes.byref(D), ctypes.byref(V), P(0x100000), 32, P(0x200000),
                                    P(0x300000), need, 1, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attention(ctypes.byref(D), ctypes.byref(V), P(0x100002), 32, P(0x200000),
                                    P(0x300000), need, kvq.KVQ_OUT_F32, None) == kvq.KVQ_ERR_MISALIGNED
    assert lib.kvq_read_error(None, None, None) == kvq.KVQ_ERR_INVALID_ARG


def test_rejects_bad_sink_view(lib):
    """With a sink window the sink arrays and sink_len are required and aligned;
    without one they may be NULL."""
    P = ctypes.c_void_p
    D = _desc(sink=32)
    for field in ("k_sink", "v_sink", "sink_len"):
        V = _view()
        setattr(V, field, 0)
        assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), P(0x100004), P(0x200000), None) == \
            kvq.KVQ_ERR_INVALID_ARG, field
    V = _view()
    V.v_sink = 0x10008
    assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000), None) == kvq.KVQ_ERR_MISALIGNED
    V = _view()
    V.sink_len = 0x10002
    assert lib.kvq_append(ctypes.byref(D), ctypes.byref(V), P(0x100000), P(0x200000), None) == kvq.KVQ_ERR_MISALIGNED
    # a hybrid cache needs its mode arrays
    for field in ("k_mode", "v_mode"):
        V = _view()
        setattr(V, field, 0)
        assert lib.kvq_append(ctypes.byref(_desc(hybrid=1)), ctypes.byref(V), P(0x100004), P(0x200000),
                              None) == kvq.KVQ_ERR_INVALID_ARG, field
    # a paged cache needs its block table
    V = _view()
    V.block_table = 0
    assert lib.kvq_append(ctypes.byref(_desc(capacity=1024, page_size=32, num_pages=64)), ctypes.byref(V),
                          P(0x100004), P(0x200000), None) == kvq.KVQ_ERR_INVALID_ARG
    # sink == 0: NULL sink pointers pass the view check (the misaligned k_new then fails)
    V = _view()
    V.k_sink = V.v_sink = V.sink_len = 0
    assert lib.kvq_append(ctypes.byref(_desc()), ctypes.byref(V), P(0x100004), P(0x200000), None) == \
        kvq.KVQ_ERR_MISALIGNED


def test_step_io_bytes(lib):
    D = _desc()  # B2, Hkv8, d128
    q, kv = 2 * 32 * 128 * 2, 2 * 8 * 128 * 2
    n_in = q + 2 * kv
    assert lib.kvq_step_io_bytes(ctypes.byref(D), 32) == ((n_in + 255) // 256) * 256 + 2 * q  # fp32 room
    assert lib.kvq_step_io_bytes(ctypes.byref(D), 12) == 0
    assert lib.kvq_step_io_bytes(ctypes.byref(_desc(bits=5)), 32) == 0


def test_step_host_rejects_bad_args(lib):
    D, V = _desc(), _view()
    P = ctypes.c_void_p
    io = lib.kvq_step_io_bytes(ctypes.byref(D), 32)
    ws = kvq.kvq_decode_workspace_bytes(D, 32)
    host = P(0x7000000)  # never dereferenced: every call below fails its checks first

    def call(in_h=host, out_h=host, dev=P(0x100000), dev_bytes=io, w=P(0x200000), w_bytes=ws, flags=0, hq=32):
        return lib.kvq_decode_step_host(ctypes.byref(D), ctypes.byref(V), in_h, hq, out_h, dev, dev_bytes,
                                        w, w_bytes, flags, None)
    assert call(in_h=None) == kvq.KVQ_ERR_INVALID_ARG
    assert call(out_h=None) == kvq.KVQ_ERR_INVALID_ARG
    assert call(dev=None) == kvq.KVQ_ERR_INVALID_ARG
    assert call(dev=P(0x100010)) == kvq.KVQ_ERR_MISALIGNED  # 16- but not 256-byte aligned
    assert call(dev_bytes=io - 1) == kvq.KVQ_ERR_INVALID_ARG
    assert call(w_bytes=ws - 1) == kvq.KVQ_ERR_INVALID_ARG
    assert call(flags=4) == kvq.KVQ_ERR_INVALID_ARG
    assert call(flags=kvq.KVQ_OUT_F32 | 8) == kvq.KVQ_ERR_INVALID_ARG
    assert call(hq=12) == kvq.KVQ_ERR_INVALID_ARG
    assert call(w=P(0x200008)) == kvq.KVQ_ERR_MISALIGNED


def test_missing_library_raises(tmp_path):
    import importlib
    mod = importlib.reload(kvq)
    try:
        with pytest.raises(RuntimeError, match="not built"):
            mod._lib = None
            mod.load(str(tmp_path / "nope.so"))
    finally:
        mod._lib = None

