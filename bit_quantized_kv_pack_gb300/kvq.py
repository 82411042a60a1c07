"""ctypes binding of libkvq.so (include/kvq.h): same names, argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  Torch supplies
device memory (``KVCache`` allocates the layout's arrays as torch tensors) and the
stream (the current torch stream unless one is given).  The library must be
built (``bit_quantized_kv_pack_gb300._build.build()``); if it is missing, loading
raises: there is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

# ------------------------------------------------------------------- ABI ----

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_MISALIGNED = 3
KVQ_ERR_CAPACITY = 4
KVQ_ERR_CUDA = 5
KVQ_ERR_TIMEOUT = 6
KVQ_ERR_EMPTY = 7

KVQ_ERRBIT_CAPACITY = 0x1
KVQ_ERRBIT_EMPTY = 0x2
KVQ_ERRBIT_TIMEOUT = 0x4
KVQ_ERRBIT_BADLEN = 0x8
KVQ_ERRBIT_BADPAGE = 0x10

KVQ_ARRAY_CODES = 0
KVQ_ARRAY_PARAMS = 1
KVQ_ARRAY_RESIDUAL = 2
KVQ_ARRAY_SINK = 3
KVQ_ARRAY_MODE = 4

# Every function the header declares (the tests check the library exports them).
EXPORTS = ("kvq_cache_bytes", "kvq_decode_workspace_bytes", "kvq_quantize_pack",
           "kvq_quantize_pack_strided", "kvq_append",
           "kvq_decode_attention", "kvq_decode_step", "kvq_decode_step_host", "kvq_step_io_bytes",
           "kvq_decode_attention_noalloc",
           "kvq_read_error", "kvq_status_string", "kvq_version", "kvq_testing_wait_fault",
           "kvq_testing_check_arithmetic", "kvq_testing_mma_rounding")


class CacheDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("residual", ctypes.c_int32),
                ("sink", ctypes.c_int32), ("hybrid", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


class CacheView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "k_codes", "v_codes", "k_params", "v_params", "k_res", "v_res",
        "packed_len", "res_len", "res_head", "err_word", "k_sink", "v_sink", "sink_len",
        "k_mode", "v_mode", "block_table")]


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libkvq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or library_path()
            if not os.path.exists(p):
                raise RuntimeError(f"libkvq.so not built ({p}); run __graft_entry__.build()")
            lib = ctypes.CDLL(p)
            P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            DP, VP = ctypes.POINTER(CacheDesc), ctypes.POINTER(CacheView)
            lib.kvq_cache_bytes.argtypes = [DP, ctypes.c_int]
            lib.kvq_cache_bytes.restype = sz
            lib.kvq_decode_workspace_bytes.argtypes = [DP, i32]
            lib.kvq_decode_workspace_bytes.restype = sz
            lib.kvq_quantize_pack.argtypes = [DP, VP, P, P, P, i32, P]
            lib.kvq_quantize_pack.restype = ctypes.c_int
            i64 = ctypes.c_int64
            lib.kvq_quantize_pack_strided.argtypes = [DP, VP, P, P, P, i32, i64, i64, i64, P]
            lib.kvq_quantize_pack_strided.restype = ctypes.c_int
            lib.kvq_append.argtypes = [DP, VP, P, P, P]
            lib.kvq_append.restype = ctypes.c_int
            lib.kvq_decode_attention.argtypes = [DP, VP, P, i32, P, P, sz, ctypes.c_uint32, P]
            lib.kvq_decode_attention.restype = ctypes.c_int
            lib.kvq_decode_step.argtypes = [DP, VP, P, i32, P, P, P, P, sz, ctypes.c_uint32, P]
            lib.kvq_decode_step.restype = ctypes.c_int
            lib.kvq_step_io_bytes.argtypes = [DP, i32]
            lib.kvq_step_io_bytes.restype = sz
            lib.kvq_decode_step_host.argtypes = [DP, VP, P, i32, P, P, sz, P, sz, ctypes.c_uint32, P]
            lib.kvq_decode_step_host.restype = ctypes.c_int
            lib.kvq_decode_attention_noalloc.argtypes = [DP, VP, P, i32, P, ctypes.c_uint32, P]
            lib.kvq_decode_attention_noalloc.restype = ctypes.c_int
            lib.kvq_read_error.argtypes = [VP, ctypes.POINTER(ctypes.c_uint32), P]
            lib.kvq_read_error.restype = ctypes.c_int
            lib.kvq_status_string.argtypes = [ctypes.c_int]
            lib.kvq_status_string.restype = ctypes.c_char_p
            lib.kvq_version.argtypes = []
            lib.kvq_version.restype = i32
            lib.kvq_testing_wait_fault.argtypes = [ctypes.c_uint32]
            lib.kvq_testing_wait_fault.restype = None
            lib.kvq_testing_check_arithmetic.argtypes = [ctypes.POINTER(ctypes.c_uint64),
                                                         ctypes.POINTER(ctypes.c_double)]
            lib.kvq_testing_check_arithmetic.restype = ctypes.c_int
            lib.kvq_testing_mma_rounding.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int32]
            lib.kvq_testing_mma_rounding.restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().kvq_status_string(status).decode()


kvq_status_string = status_string


def _check(status: int, where: str) -> None:
    if status != KVQ_OK:
        raise KvqError(status, where)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _f16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float16 CUDA tensor")
    return t


KVQ_OUT_F32 = 2


def _out(q: torch.Tensor, out: torch.Tensor | None, flags: int):
    """The output tensor and the flags that match its dtype: float16, or float32
    (KVQ_OUT_F32).  Without `out`, the dtype follows KVQ_OUT_F32 in flags."""
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if flags & KVQ_OUT_F32 else torch.float16,
                          device=q.device)
    if out.dtype not in (torch.float16, torch.float32) or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous float16 or float32 CUDA tensor")
    if out.dtype == torch.float32:
        flags |= KVQ_OUT_F32
    else:
        flags &= ~KVQ_OUT_F32
    return out, flags


# --------------------------------------------------------------- caches ----


class KVCache:
    """One layer's packed cache in device memory (torch tensors in the layout of
    include/kvq.h).  Holds the description and the view the calls take.
    ``sink`` > 0 keeps the first ``sink`` tokens of each sequence in fp16 (the
    attention-sink window, fixed after the prefill); ``hybrid=1`` quantizes each
    group symmetrically or asymmetrically, whichever reconstructs it better, and
    keeps a mode byte per packed row.  ``page_size=32`` keeps the packed rows in
    a pool of ``num_pages`` pages [page][head][32] found through ``block_table``
    [B][capacity / 32] (filled with pages b * capacity / 32 + j when the pool has
    room, for the caller to rewrite)."""

    def __init__(self, batch, num_kv_heads, head_dim, bits, capacity, residual, device="cuda",
                 sink=0, hybrid=0, page_size=0, num_pages=0):
        self.desc = CacheDesc(batch, num_kv_heads, head_dim, bits, 32, capacity, residual, sink,
                              hybrid, page_size, num_pages)
        self.device = torch.device(device)
        B, H, d = batch, num_kv_heads, head_dim
        rb, ng = d * bits // 8, d // 32
        kw = dict(device=self.device)
        rows = (num_pages, H, page_size) if page_size else (B, H, capacity)
        self.k_codes = torch.zeros(*rows, rb, dtype=torch.uint8, **kw)
        self.v_codes = torch.zeros(*rows, rb, dtype=torch.uint8, **kw)
        self.k_params = torch.zeros(*rows, ng, dtype=torch.int32, **kw)
        self.v_params = torch.zeros(*rows, ng, dtype=torch.int32, **kw)
        npb = capacity // page_size if page_size else 0
        self.block_table = (torch.arange(B * npb, dtype=torch.int32, **kw).view(B, npb)
                            % max(num_pages, 1))
        self.k_res = torch.zeros(B, H, residual, d, dtype=torch.float16, **kw)
        self.v_res = torch.zeros(B, H, residual, d, dtype=torch.float16, **kw)
        self.k_sink = torch.zeros(B, H, sink, d, dtype=torch.float16, **kw)
        self.v_sink = torch.zeros(B, H, sink, d, dtype=torch.float16, **kw)
        mrows = rows if hybrid else (0,)
        self.k_mode = torch.zeros(*mrows, dtype=torch.uint8, **kw)
        self.v_mode = torch.zeros(*mrows, dtype=torch.uint8, **kw)
        # packed_len, res_len, res_head, sink_len
        self.counters = torch.zeros(4, B, dtype=torch.int32, **kw)
        self.err = torch.zeros(4, dtype=torch.int32, **kw)
        self.view = self._make_view()

    def _make_view(self) -> CacheView:
        r = lambda t: _ptr(t) if t.numel() else ctypes.c_void_p(0)
        return CacheView(r(self.k_codes), r(self.v_codes), r(self.k_params), r(self.v_params),
                         r(self.k_res), r(self.v_res), _ptr(self.counters[0]),
                         _ptr(self.counters[1]), _ptr(self.counters[2]), _ptr(self.err),
                         r(self.k_sink), r(self.v_sink), _ptr(self.counters[3]),
                         r(self.k_mode), r(self.v_mode), r(self.block_table))

    @property
    def packed_len(self):
        return self.counters[0]

    @property
    def res_len(self):
        return self.counters[1]

    @property
    def res_head(self):
        return self.counters[2]

    @property
    def sink_len(self):
        return self.counters[3]

    def packed_bytes(self) -> int:
        """Code + param bytes of the tokens currently packed (K and V)."""
        D = self.desc
        per_tok = 2 * (D.head_dim * D.bits // 8 + 4 * (D.head_dim // 32))
        return int(self.packed_len.sum().item()) * D.num_kv_heads * per_tok


def kvq_cache_bytes(desc: CacheDesc, which: int) -> int:
    return int(load().kvq_cache_bytes(ctypes.byref(desc), which))


def kvq_decode_workspace_bytes(desc: CacheDesc, num_q_heads: int) -> int:
    return int(load().kvq_decode_workspace_bytes(ctypes.byref(desc), num_q_heads))


def kvq_quantize_pack(cache: KVCache, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                      stream=None) -> None:
    """Pack a prefill; k, v fp16 [B][Hkv][Lmax][d], seq_lens int32 [B] on the device."""
    _f16(k, "k"), _f16(v, "v")
    if k.shape != v.shape or k.dim() != 4:
        raise ValueError("k and v must both be [B][Hkv][Lmax][d]")
    if seq_lens.dtype != torch.int32 or not seq_lens.is_cuda:
        raise ValueError("seq_lens must be an int32 CUDA tensor")
    st = load().kvq_quantize_pack(ctypes.byref(cache.desc), ctypes.byref(cache.view), _ptr(k),
                                  _ptr(v), _ptr(seq_lens), int(k.shape[2]),
                                  _stream(stream, k.device))
    _check(st, "kvq_quantize_pack")


def kvq_quantize_pack_strided(cache: KVCache, k: torch.Tensor, v: torch.Tensor,
                              seq_lens: torch.Tensor, stream=None) -> None:
    """Pack a prefill from any strided view: k, v fp16 of logical shape
    [B][Hkv][Lmax][d] with head_dim contiguous (for example a permuted view of a
    token-major [B][L][Hkv][d] tensor, or of the key/value columns of a fused
    QKV projection output).  Nothing is copied: the library reads through the
    strides."""
    for t, name in ((k, "k"), (v, "v")):
        if t.dtype != torch.float16 or not t.is_cuda or t.dim() != 4 or t.stride(3) != 1:
            raise ValueError(f"{name} must be a float16 CUDA [B][Hkv][Lmax][d] view with d contiguous")
    if k.shape != v.shape or k.stride() != v.stride():
        raise ValueError("k and v must have the same shape and strides")
    if seq_lens.dtype != torch.int32 or not seq_lens.is_cuda:
        raise ValueError("seq_lens must be an int32 CUDA tensor")
    st = load().kvq_quantize_pack_strided(ctypes.byref(cache.desc), ctypes.byref(cache.view),
                                          _ptr(k), _ptr(v), _ptr(seq_lens), int(k.shape[2]),
                                          int(k.stride(0)), int(k.stride(1)), int(k.stride(2)),
                                          _stream(stream, k.device))
    _check(st, "kvq_quantize_pack_strided")


def kvq_append(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Append one token per sequence; k_new, v_new fp16 [B][Hkv][d]."""
    _f16(k_new, "k_new"), _f16(v_new, "v_new")
    st = load().kvq_append(ctypes.byref(cache.desc), ctypes.byref(cache.view), _ptr(k_new),
                           _ptr(v_new), _stream(stream, k_new.device))
    _check(st, "kvq_append")


def workspace_for(cache: KVCache, num_q_heads: int) -> torch.Tensor:
    """A zeroed decode workspace (zeroed once; the decode keeps it ready)."""
    n = kvq_decode_workspace_bytes(cache.desc, num_q_heads)
    if n == 0:
        raise KvqError(KVQ_ERR_INVALID_ARG, "kvq_decode_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=cache.device)


def kvq_decode_attention(cache: KVCache, q: torch.Tensor, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None, stream=None,
                         flags: int = 0) -> torch.Tensor:
    """O = softmax(q K^T / sqrt(d)) V; q fp16 [B][Hq][d] -> out [B][Hq][d], fp16
    or fp32 (an fp32 `out`, or flags=KVQ_OUT_F32)."""
    _f16(q, "q")
    out, flags = _out(q, out, flags)
    if workspace is None:
        workspace = workspace_for(cache, q.shape[1])
    st = load().kvq_decode_attention(ctypes.byref(cache.desc), ctypes.byref(cache.view), _ptr(q),
                                     int(q.shape[1]), _ptr(out), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), int(flags),
                                     _stream(stream, q.device))
    _check(st, "kvq_decode_attention")
    return out


KVQ_STEP_EARLY_CACHE_READ = 1
KVQ_STEP_HOST_MAPPED = 4


def kvq_decode_step(cache: KVCache, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream=None, flags: int = 0) -> torch.Tensor:
    """One serving-loop step: append k_new/v_new (fp16 [B][Hkv][d]), then decode
    attention of q over the updated cache; one kernel launch where the tensor-core
    kernel applies.  flags=KVQ_STEP_EARLY_CACHE_READ: the kernel enqueued just
    before does not write this cache (see kvq.h).  An fp32 `out` (or
    KVQ_OUT_F32 in flags) gives fp32 output."""
    _f16(q, "q"), _f16(k_new, "k_new"), _f16(v_new, "v_new")
    out, flags = _out(q, out, flags)
    if workspace is None:
        workspace = workspace_for(cache, q.shape[1])
    st = load().kvq_decode_step(ctypes.byref(cache.desc), ctypes.byref(cache.view), _ptr(q),
                                int(q.shape[1]), _ptr(k_new), _ptr(v_new), _ptr(out),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                int(flags), _stream(stream, q.device))
    _check(st, "kvq_decode_step")
    return out


def kvq_step_io_bytes(cache: KVCache, num_q_heads: int) -> int:
    return int(load().kvq_step_io_bytes(ctypes.byref(cache.desc), int(num_q_heads)))


def step_io_for(cache: KVCache, num_q_heads: int) -> torch.Tensor:
    """Device staging for kvq_decode_step_host (256-byte aligned)."""
    n = kvq_step_io_bytes(cache, num_q_heads)
    if n == 0:
        raise ValueError("invalid cache description or head count")
    buf = torch.empty(n + 256, dtype=torch.uint8, device=cache.device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


def kvq_decode_step_host(cache: KVCache, in_host: torch.Tensor, num_q_heads: int,
                         out_host: torch.Tensor, dev_io: torch.Tensor | None, workspace: torch.Tensor,
                         stream=None, flags: int = 0) -> None:
    """One step from host memory: in_host = [q | k_new | v_new] fp16 (pinned for
    an asynchronous call), out_host fp16 [B][Hq][d]; copies, step and copy back
    enqueued on the stream by one library call.  An fp32 out_host gives fp32
    output.  flags | KVQ_STEP_HOST_MAPPED (pinned, device-mapped buffers): the
    step reads and writes them in place, no copies, dev_io unused."""
    if in_host.is_cuda or out_host.is_cuda:
        raise ValueError("in_host and out_host must be host tensors")
    flags = (flags | KVQ_OUT_F32) if out_host.dtype == torch.float32 else (flags & ~KVQ_OUT_F32)
    io_ptr = _ptr(dev_io) if dev_io is not None else ctypes.c_void_p(0)
    io_bytes = dev_io.numel() * dev_io.element_size() if dev_io is not None else 0
    st = load().kvq_decode_step_host(ctypes.byref(cache.desc), ctypes.byref(cache.view),
                                     _ptr(in_host), int(num_q_heads), _ptr(out_host), io_ptr,
                                     io_bytes, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), int(flags),
                                     _stream(stream, workspace.device))
    _check(st, "kvq_decode_step_host")


NOALLOC_SCRATCH_BYTES = 8 << 20


def kvq_decode_attention_noalloc(cache: KVCache, q: torch.Tensor, out: torch.Tensor | None = None,
                                 stream=None) -> torch.Tensor:
    """Decode attention for callers that cannot allocate device scratch: the
    library's own static device array holds the split partials.  Calls that
    overlap on the GPU share that array and race; keep them on one stream."""
    _f16(q, "q")
    out, flags = _out(q, out, 0)
    st = load().kvq_decode_attention_noalloc(ctypes.byref(cache.desc), ctypes.byref(cache.view),
                                             _ptr(q), int(q.shape[1]), _ptr(out), int(flags),
                                             _stream(stream, q.device))
    _check(st, "kvq_decode_attention_noalloc")
    return out


def kvq_read_error(cache: KVCache, stream=None) -> tuple[int, int]:
    """(status, raw error word); synchronizes the stream and clears the word."""
    word = ctypes.c_uint32(0)
    st = load().kvq_read_error(ctypes.byref(cache.view), ctypes.byref(word),
                               _stream(stream, cache.device))
    return st, word.value


def kvq_version() -> int:
    return int(load().kvq_version())


def kvq_testing_wait_fault(limit_us: int) -> None:
    """Testing hook (see kvq.h): limit_us > 0 makes one bounded wait of the next
    tensor-core decode calls run out after limit_us microseconds; 0 turns it off."""
    load().kvq_testing_wait_fault(int(limit_us))


def kvq_testing_check_arithmetic():
    """Testing hook (see kvq.h): ([mismatches, in domain] for the divisors 15, 7,
    3, the reciprocal's worst relative error over the fp16 scales)."""
    mm = (ctypes.c_uint64 * 6)()
    worst = ctypes.c_double(0.0)
    _check(load().kvq_testing_check_arithmetic(mm, ctypes.byref(worst)),
           "kvq_testing_check_arithmetic")
    return [(int(mm[2 * i]), int(mm[2 * i + 1])) for i in range(3)], worst.value


def kvq_testing_mma_rounding(n: int = 8):
    """Testing hook (see kvq.h): the eight MMA rounding cases' results."""
    out = (ctypes.c_float * 8)()
    _check(load().kvq_testing_mma_rounding(out, int(n)), "kvq_testing_mma_rounding")
    return [float(out[i]) for i in range(n)]
