"""Shared helpers of the GPU parity tests: run the same seeded inputs through the
CUDA path (C ABI via the ctypes binding) and the CPU oracle, and compare."""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from bit_quantized_kv_pack_gb300 import kvq

ATOL = 2e-3   # max abs error of the fp16 attention output vs the fp64 oracle
RTOL_L2 = 1e-3  # relative L2 error of the same


def gpu_cache(B, H, d, bits, cap, Nr, dev="cuda", sink=0, hybrid=0, pages=0, seed=0):
    """A device cache; pages > 0 makes it paged with a pool of that many
    32-token pages and a block table drawn as a seeded random injection."""
    if not pages:
        return kvq.KVCache(B, H, d, bits, cap, Nr, device=dev, sink=sink, hybrid=hybrid)
    c = kvq.KVCache(B, H, d, bits, cap, Nr, device=dev, sink=sink, hybrid=hybrid, page_size=32,
                    num_pages=pages)
    perm = np.random.default_rng(seed).permutation(pages)[:B * (cap // 32)]
    c.block_table.copy_(torch.from_numpy(perm.astype(np.int32)).view(B, cap // 32))
    return c


class _Logical:
    """A paged cache's packed arrays gathered through its block table into the
    contiguous [B][Hkv][cap] layout (numpy-style indexing, for comparisons)."""

    def __init__(self, g):
        bt = g.block_table.long()
        B, npb = bt.shape
        for name in ("k_codes", "v_codes", "k_params", "v_params", "k_mode", "v_mode"):
            pool = getattr(g, name)
            if pool.numel() == 0:
                setattr(self, name, pool)
                continue
            x = pool[bt]  # [B][npb][H][32](...)
            x = x.transpose(1, 2).contiguous()  # [B][H][npb][32](...)
            setattr(self, name, x.view(B, x.shape[1], npb * 32, *x.shape[4:]))
        for name in ("k_res", "v_res", "k_sink", "v_sink", "packed_len", "res_len", "res_head",
                     "sink_len"):
            setattr(self, name, getattr(g, name))


def logical(g):
    return _Logical(g) if g.desc.page_size else g


def ref_cache(B, H, d, bits, cap, Nr, sink=0, hybrid=0):
    return oracle.Cache(B, H, d, bits, cap, Nr, sink, hybrid)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def assert_cache_equal(g, r, batches=None):
    """Packed bytes of every used slot, the residual ring, the sink rows and the
    counters."""
    g = logical(g)
    pl = to_np(g.packed_len)
    rl = to_np(g.res_len)
    rh = to_np(g.res_head)
    sl = to_np(g.sink_len)
    S = r.desc.sink
    rows = range(len(r.packed_len)) if batches is None else batches
    for i, b in enumerate(rows):
        assert pl[b] == r.packed_len[i], (b, pl[b], r.packed_len[i])
        assert rl[b] == r.res_len[i] and rh[b] == r.res_head[i], b
        n = int(r.packed_len[i])
        names = ("k_codes", "v_codes", "k_params", "v_params")
        if r.desc.hybrid:
            names += ("k_mode", "v_mode")
        for name in names:
            got = to_np(getattr(g, name)[b, :, :n]).view(getattr(r, name).dtype)
            want = getattr(r, name)[i, :, :n]
            if not np.array_equal(got, want):
                bad = np.argwhere(got != want)[:5]
                raise AssertionError(f"{name} differs for sequence {b} at {bad.tolist()}")
        nres = int(r.res_len[i])
        for name in ("k_res", "v_res"):
            got = to_np(getattr(g, name)[b]).view(np.uint16)
            want = getattr(r, name)[i]
            assert np.array_equal(got[:, :nres], want[:, :nres]), (name, b)
        if S > 0:
            ns = int(r.sink_len[i])
            assert sl[b] == ns, (b, sl[b], ns)
            for name in ("k_sink", "v_sink"):
                got = to_np(getattr(g, name)[b]).view(np.uint16)
                assert np.array_equal(got[:, :ns], getattr(r, name)[i][:, :ns]), (name, b)


def attn_errors(out: torch.Tensor, want: np.ndarray):
    o = to_np(out.float()).astype(np.float64)
    err = np.abs(o - want)
    rel = np.linalg.norm(o - want) / max(np.linalg.norm(want), 1e-300)
    return float(err.max()), float(rel)


def f16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the fp16 spacing at |x|: the most rounding a value to fp16 can move
    it (taking the spacing above |x|, the larger one at a power of two)."""
    return np.spacing(np.abs(x).astype(np.float16)).astype(np.float64) / 2


def assert_attn_close(out, want, atol=ATOL, rtol=RTOL_L2):
    """Max abs error <= atol and relative L2 <= rtol against the fp64 oracle.
    An fp16 output also carries its own rounding, which no fp16 result avoids:
    up to half an fp16 spacing of |O|, which reaches 2e-3 at |O| = 4 (the
    nearest fp16 to a value of 4 or more can be farther than atol from it), so
    there an element may be off by atol plus that; below |O| = 4 fp16 output is
    held to atol like fp32 output."""
    err, rel = attn_errors(out, want)
    o = to_np(out.float()).astype(np.float64)
    assert np.isfinite(o).all()
    bound = atol
    if out.dtype == torch.float16:
        bound = atol + np.where(np.abs(want) >= 4.0, f16_half_ulp(want), 0.0)
    excess = float((np.abs(o - want) - bound).max())
    assert excess <= 0 and rel <= rtol, \
        f"max abs {err:.3e} (bound {atol} + fp16 rounding exceeded by {excess:.2e}), rel L2 {rel:.3e} (<= {rtol})"
    return err, rel


def per_sequence(fn, n, threads=None):
    """fn(b) for b in range(n) on a thread pool: the oracle is a C library whose
    ctypes calls release the interpreter lock, so sequences run in parallel."""
    with ThreadPoolExecutor(max_workers=threads or min(n, os.cpu_count() or 1)) as ex:
        return list(ex.map(fn, range(n)))


def oracle_sequences(k, v, lens, bits, cap, Nr, sink=0, hybrid=0):
    """One one-sequence oracle cache per sequence of a prefill (k, v host numpy
    [B][Hkv][Lmax][d] fp16, lens int32 [B]), packed in parallel."""
    B, H, _, d = k.shape

    def one(b):
        L = max(int(lens[b]), 1)
        r = ref_cache(1, H, d, bits, cap, Nr, sink, hybrid)
        err = oracle.quantize_pack(r, np.ascontiguousarray(k[b:b + 1, :, :L]),
                                   np.ascontiguousarray(v[b:b + 1, :, :L]),
                                   np.ascontiguousarray(lens[b:b + 1], dtype=np.int32))
        assert err == 0, (b, err)
        return r

    return per_sequence(one, B)
