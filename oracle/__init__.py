"""CPU oracle for the low-bit KV-cache path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package.  The product library never does, and the oracle imports
nothing from it: the two share no code.

The arithmetic lives in ``kvq_oracle.c`` (plain C, fp64 attention, its own
binary16 conversion); this module compiles it with gcc and wraps it with ctypes
over numpy arrays.  Every wrapper names the step of the method it follows; the
C file cites the passages.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvq_oracle.so")
_CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc) and return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Desc(ctypes.Structure):
    """Cache shape; the same nine integers as the library's description."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("residual", ctypes.c_int32),
        ("sink", ctypes.c_int32),
        ("hybrid", ctypes.c_int32),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f32_to_f16_array.argtypes = [P, P, i64]
            lib.oracle_f16_to_f64_array.argtypes = [P, P, i64]
            lib.oracle_quantize_group.argtypes = [P, ctypes.c_int, P, P, P]
            lib.oracle_quantize_group_sym.argtypes = [P, ctypes.c_int, P, P, P]
            lib.oracle_quantize_group_sym.restype = ctypes.c_int
            lib.oracle_group_sq_error.argtypes = [P, P, ctypes.c_uint16, ctypes.c_uint16]
            lib.oracle_group_sq_error.restype = ctypes.c_float
            lib.oracle_quantize_group_hybrid.argtypes = [P, ctypes.c_int, P, P, P]
            lib.oracle_quantize_group_hybrid.restype = ctypes.c_int
            lib.oracle_pack_row.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
            lib.oracle_pack_row.restype = ctypes.c_int
            lib.oracle_unpack_row.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
            lib.oracle_quantize_pack.argtypes = [P, P, P, i32, P, P, P, P, P, P, P, P, P]
            lib.oracle_quantize_pack.restype = ctypes.c_int
            lib.oracle_append.argtypes = [P] * 12
            lib.oracle_append.restype = ctypes.c_int
            lib.oracle_decode_pairs.argtypes = [P] * 13 + [P, i32, P, i32, P]
            lib.oracle_decode_pairs.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [P] * 13 + [P, i32, P]
            lib.oracle_decode.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    """fp16 data as its raw uint16 bits (accepts float16 or uint16 arrays)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


# ----------------------------------------------------------------- binary16 --


def f32_to_f16_bits(x) -> np.ndarray:
    """IEEE binary16 round-to-nearest-even of float32 values, as uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_bits_to_f64(h) -> np.ndarray:
    """Exact value of binary16 bit patterns."""
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_f16_to_f64_array(_ptr(h), _ptr(out), h.size)
    return out


# ----------------------------------------------------------------- quantize --


def quantize_group(x, bits: int):
    """Q1-Q4 on 32 fp16 values -> (codes uint8[32], scale_bits, min_bits)."""
    x = _u16(x)
    assert x.size == 32
    codes = np.zeros(32, dtype=np.uint8)
    sh = ctypes.c_uint16()
    mh = ctypes.c_uint16()
    _load().oracle_quantize_group(_ptr(x), bits, _ptr(codes), ctypes.byref(sh), ctypes.byref(mh))
    return codes, sh.value, mh.value


def quantize_group_sym(x, bits: int):
    """H1 (symmetric candidate) on 32 fp16 values -> (codes, scale_bits,
    min_bits, storable)."""
    x = _u16(x)
    assert x.size == 32
    codes = np.zeros(32, dtype=np.uint8)
    sh, mh = ctypes.c_uint16(), ctypes.c_uint16()
    ok = _load().oracle_quantize_group_sym(_ptr(x), bits, _ptr(codes), ctypes.byref(sh), ctypes.byref(mh))
    return codes, sh.value, mh.value, bool(ok)


def group_sq_error(x, codes, scale_bits: int, min_bits: int) -> float:
    """H2: the fp32 squared reconstruction error of one group's candidate."""
    x = _u16(x)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    return float(_load().oracle_group_sq_error(_ptr(x), _ptr(codes), scale_bits, min_bits))


def quantize_group_hybrid(x, bits: int):
    """H3 on 32 fp16 values -> (codes, scale_bits, min_bits, mode) with mode 1
    asymmetric, 0 symmetric."""
    x = _u16(x)
    assert x.size == 32
    codes = np.zeros(32, dtype=np.uint8)
    sh, mh = ctypes.c_uint16(), ctypes.c_uint16()
    mode = _load().oracle_quantize_group_hybrid(_ptr(x), bits, _ptr(codes), ctypes.byref(sh),
                                                ctypes.byref(mh))
    return codes, sh.value, mh.value, int(mode)


def pack_row(codes, bits: int) -> np.ndarray:
    """Q5: d codes -> d*bits/8 bytes."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    d = codes.size
    out = np.zeros(d * bits // 8, dtype=np.uint8)
    _load().oracle_pack_row(_ptr(codes), d, bits, _ptr(out))
    return out


def unpack_row(packed, d: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(d, dtype=np.uint8)
    _load().oracle_unpack_row(_ptr(packed), d, bits, _ptr(out))
    return out


class Cache:
    """Host copy of one layer's cache in the library's layout (numpy arrays)."""

    def __init__(self, batch, num_kv_heads, head_dim, bits, capacity, residual, sink=0, hybrid=0):
        self.desc = Desc(batch, num_kv_heads, head_dim, bits, 32, capacity, residual, sink, hybrid)
        B, H, d = batch, num_kv_heads, head_dim
        rb, ng = d * bits // 8, d // 32
        self.k_codes = np.zeros((B, H, capacity, rb), np.uint8)
        self.v_codes = np.zeros((B, H, capacity, rb), np.uint8)
        self.k_params = np.zeros((B, H, capacity, ng), np.uint32)
        self.v_params = np.zeros((B, H, capacity, ng), np.uint32)
        self.k_res = np.zeros((B, H, max(residual, 0), d), np.uint16)
        self.v_res = np.zeros((B, H, max(residual, 0), d), np.uint16)
        self.packed_len = np.zeros(B, np.int32)
        self.res_len = np.zeros(B, np.int32)
        self.res_head = np.zeros(B, np.int32)
        self.k_sink = np.zeros((B, H, max(sink, 1), d), np.uint16)  # [B][Hkv][sink][d] fp16 bits
        self.v_sink = np.zeros((B, H, max(sink, 1), d), np.uint16)
        self.sink_len = np.zeros(B, np.int32)
        # hybrid mode: per packed row, bit g = mode of group g (1 asymmetric, 0 symmetric)
        self.k_mode = np.zeros((B, H, max(capacity, 1)), np.uint8)
        self.v_mode = np.zeros((B, H, max(capacity, 1)), np.uint8)

    @property
    def shape(self):
        D = self.desc
        return D.batch, D.num_kv_heads, D.head_dim, D.bits, D.capacity, D.residual, D.sink, D.hybrid

    def copy(self) -> "Cache":
        c = Cache(*self.shape)
        for name in ("k_codes", "v_codes", "k_params", "v_params", "k_res", "v_res",
                     "packed_len", "res_len", "res_head", "k_sink", "v_sink", "sink_len",
                     "k_mode", "v_mode"):
            getattr(c, name)[...] = getattr(self, name)
        return c


def quantize_pack(cache: Cache, k, v, seq_lens) -> int:
    """Q1-Q6 for K and V of a prefill [B][Hkv][Lmax][d]; returns the error bits."""
    k, v = _u16(k), _u16(v)
    assert k.shape == v.shape and k.ndim == 4
    Lmax = k.shape[2]
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    lib = _load()
    D = ctypes.byref(cache.desc)
    e1 = lib.oracle_quantize_pack(D, _ptr(k), _ptr(seq), Lmax, _ptr(cache.k_codes),
                                  _ptr(cache.k_params), _ptr(cache.k_res), _ptr(cache.k_sink),
                                  _ptr(cache.k_mode), _ptr(cache.packed_len), _ptr(cache.res_len), _ptr(cache.res_head),
                                  _ptr(cache.sink_len))
    e2 = lib.oracle_quantize_pack(D, _ptr(v), _ptr(seq), Lmax, _ptr(cache.v_codes),
                                  _ptr(cache.v_params), _ptr(cache.v_res), _ptr(cache.v_sink),
                                  _ptr(cache.v_mode), _ptr(cache.packed_len), _ptr(cache.res_len), _ptr(cache.res_head),
                                  _ptr(cache.sink_len))
    if e1 < 0 or e2 < 0:
        raise ValueError("invalid cache description")
    return e1 | e2


def append(cache: Cache, k_new, v_new) -> int:
    """Q7: append one token per sequence ([B][Hkv][d] each); returns the error bits."""
    k_new, v_new = _u16(k_new), _u16(v_new)
    lib = _load()
    D = ctypes.byref(cache.desc)
    pl, rl, rh = cache.packed_len.copy(), cache.res_len.copy(), cache.res_head.copy()
    e1 = lib.oracle_append(D, _ptr(k_new), _ptr(cache.k_codes), _ptr(cache.k_params),
                           _ptr(cache.k_res), _ptr(cache.k_mode), _ptr(pl), _ptr(rl), _ptr(rh),
                           _ptr(cache.packed_len), _ptr(cache.res_len), _ptr(cache.res_head))
    e2 = lib.oracle_append(D, _ptr(v_new), _ptr(cache.v_codes), _ptr(cache.v_params),
                           _ptr(cache.v_res), _ptr(cache.v_mode), _ptr(pl), _ptr(rl), _ptr(rh),
                           _ptr(cache.packed_len), _ptr(cache.res_len), _ptr(cache.res_head))
    if e1 < 0 or e2 < 0:
        raise ValueError("invalid cache description")
    return e1 | e2


def decode(cache: Cache, q, pairs=None) -> np.ndarray:
    """D1-D4: fp64 attention output.

    q is fp16 [B][Hq][d].  With ``pairs`` (an int array [n][2] of (b, hq)) only
    those rows are computed and the result is [n][d]; otherwise [B][Hq][d].
    """
    q = _u16(q)
    B, Hq, d = q.shape
    lib = _load()
    args = [ctypes.byref(cache.desc), _ptr(cache.k_codes), _ptr(cache.k_params),
            _ptr(cache.k_res), _ptr(cache.k_sink), _ptr(cache.v_codes), _ptr(cache.v_params),
            _ptr(cache.v_res), _ptr(cache.v_sink), _ptr(cache.packed_len), _ptr(cache.res_len),
            _ptr(cache.res_head), _ptr(cache.sink_len), _ptr(q), Hq]
    if pairs is None:
        out = np.zeros((B, Hq, d), np.float64)
        rc = lib.oracle_decode(*args, _ptr(out))
    else:
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((pairs.shape[0], d), np.float64)
        rc = lib.oracle_decode_pairs(*args, _ptr(pairs), pairs.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError("invalid decode arguments")
    return out
