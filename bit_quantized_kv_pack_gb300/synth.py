"""Seeded synthetic inputs (shared by the tests, the smoke check and the benchmark).

This module holds no arithmetic of the quantization or attention method: only
random numbers and the shapes of the workloads.  Both the CUDA path and the CPU
oracle receive the tensors it returns.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", 2014) used as a counter-based stream.  Output i of stream
(seed, tensor_id) is mix64(key + (i + 1) * 0x9E3779B97F4A7C15) with
key = mix64(seed * 0x9E3779B97F4A7C15 + tensor_id); a uniform in [0, 1) takes the
top 53 bits.  Normals come from the Box-Muller transform in double precision
(element i uses outputs 2i and 2i + 1) and are rounded to float32, then to
float16, both to nearest even.  Everything is computed with torch tensor ops, on
the CPU by default (the values do not depend on chunking).

Workloads (shapes of the decode layers the pages name: Llama-3.1-8B and
Llama-2-13B; seeds are 1000 + the workload number):
  1 tiny    B1, Hq = Hkv = 1, d64, L256, Nr64, INT4; q, K, V ~ N(0, 1)
  2 8b-32k  B1, Hq32, Hkv8, d128, L32768, Nr128, INT4; V, q ~ N(0, 1);
            K ~ N(0, 1) with 4 seed-chosen channels per KV head scaled x10
  3 8b-128k same as 2 at L131072, INT2
  4 13b-b64 B64, Hq = Hkv = 40, d128, L_b ~ U{1024..4096}, Nr96, INT4;
            K, V ~ N(0, 1) with each element replaced with probability 0.01 by N(0, 8^2)
  5 pack    32768 tokens x 8 KV heads x d128 K (outlier channels as 2) and V, INT4 and INT2, Nr0
"""

from __future__ import annotations

import dataclasses
import math

import torch

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_CHUNK = 1 << 22


def _s64(x: int) -> int:
    """An unsigned 64-bit constant as the int64 with the same bits."""
    x &= (1 << 64) - 1
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def _key(seed: int, tensor_id: int) -> int:
    z = torch.tensor([_s64(seed * _GOLDEN + tensor_id)], dtype=torch.int64)
    return int(_mix64(z)[0])


def raw64(seed: int, tensor_id: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """Outputs start .. start+n-1 of stream (seed, tensor_id) as int64 bit patterns."""
    idx = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    return _mix64(idx * _s64(_GOLDEN) + _key(seed, tensor_id))


def uniform(seed: int, tensor_id: int, n: int, start: int = 0, device="cpu") -> torch.Tensor:
    """n doubles in [0, 1)."""
    return _lsr(raw64(seed, tensor_id, start, n, device), 11).to(torch.float64) * (2.0 ** -53)


def normal(seed: int, tensor_id: int, n: int, start: int = 0, device="cpu") -> torch.Tensor:
    """n standard normal doubles (Box-Muller); element i uses outputs 2i, 2i+1."""
    u = uniform(seed, tensor_id, 2 * n, 2 * start, device).view(n, 2)
    r = torch.sqrt(-2.0 * torch.log1p(-u[:, 0]))
    return r * torch.cos((2.0 * math.pi) * u[:, 1])


def to_f16(x64: torch.Tensor) -> torch.Tensor:
    return x64.to(torch.float32).to(torch.float16)


def normal_f16(seed: int, tensor_id: int, shape, sigma: float = 1.0, device="cpu") -> torch.Tensor:
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float16, device=device)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        out[s:s + m] = to_f16(normal(seed, tensor_id, m, s, device) * sigma)
    return out.view(*shape)


# Tensor ids of the streams.
T_Q, T_K, T_V, T_KNEW, T_VNEW, T_CHAN, T_LENS, T_MASK_K, T_MASK_V, T_OUT_K, T_OUT_V = range(1, 12)


def outlier_channels(seed: int, num_kv_heads: int, head_dim: int, count: int) -> torch.Tensor:
    """[Hkv][count] distinct channel indices per KV head (the `count` smallest of
    head_dim uniforms)."""
    u = uniform(seed, T_CHAN, num_kv_heads * head_dim).view(num_kv_heads, head_dim)
    return torch.argsort(u, dim=1, stable=True)[:, :count].sort(dim=1).values


@dataclasses.dataclass
class Workload:
    """Shape and value recipe of one synthetic workload."""

    number: int
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    bits: int
    residual: int
    len_min: int
    len_max: int
    k_outlier_channels: int = 0    # channels per KV head scaled x10
    sparse_outlier_p: float = 0.0  # element replacement probability
    sparse_outlier_sigma: float = 0.0

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def gq(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def seq_lens(self) -> torch.Tensor:
        if self.len_min == self.len_max:
            return torch.full((self.batch,), self.len_max, dtype=torch.int32)
        u = uniform(self.seed, T_LENS, self.batch)
        span = self.len_max - self.len_min + 1
        return (self.len_min + torch.floor(u * span).to(torch.int64)).to(torch.int32)

    def _kv(self, which: str, shape, device="cpu", start: int = 0) -> torch.Tensor:
        """K or V with the workload's outlier structure, fp16 of `shape`:
        [B][Hkv][L][d] for a prefill or [B][Hkv][d] for append tokens (which use
        streams of their own, `start` elements in for later steps).  Outlier
        channels are multiplied by 10 and sparse outliers replace the element,
        both before rounding to fp16."""
        tid = {"k": T_K, "v": T_V, "knew": T_KNEW, "vnew": T_VNEW}[which]
        is_k = which in ("k", "knew")
        n = math.prod(shape)
        d = self.head_dim
        per_head = n // (shape[0] * self.num_kv_heads)  # elements of one (b, h)
        chan_mult = None
        if is_k and self.k_outlier_channels:
            ch = outlier_channels(self.seed, self.num_kv_heads, d, self.k_outlier_channels)
            chan_mult = torch.ones(self.num_kv_heads, d, dtype=torch.float64)
            chan_mult.scatter_(1, ch, 10.0)
            chan_mult = chan_mult.to(device)
        out = torch.empty(n, dtype=torch.float16, device=device)
        for s in range(0, n, _CHUNK):
            m = min(_CHUNK, n - s)
            x = normal(self.seed, tid, m, start + s, device)
            if chan_mult is not None:
                idx = torch.arange(s, s + m, dtype=torch.int64, device=device)
                head = (idx // per_head) % self.num_kv_heads
                x = x * chan_mult[head, idx % d]
            if self.sparse_outlier_p > 0.0:
                mtid = T_MASK_K if is_k else T_MASK_V
                otid = T_OUT_K if is_k else T_OUT_V
                hit = uniform(self.seed, mtid, m, start + s, device) < self.sparse_outlier_p
                pos = torch.nonzero(hit).squeeze(1)
                if pos.numel():
                    x[pos] = _normal_at(self.seed, otid, pos + start + s) * self.sparse_outlier_sigma
            out[s:s + m] = to_f16(x)
        return out.view(*shape)

    def prefill(self, device="cpu"):
        """(K, V, seq_lens): K, V fp16 [B][Hkv][len_max][d]."""
        shape = (self.batch, self.num_kv_heads, self.len_max, self.head_dim)
        return self._kv("k", shape, device), self._kv("v", shape, device), self.seq_lens()

    def query(self, step: int = 0, device="cpu") -> torch.Tensor:
        """q fp16 [B][Hq][d]; `step` selects an independent draw."""
        n = self.batch * self.num_q_heads * self.head_dim
        x = to_f16(normal(self.seed, T_Q, n, step * n, device))
        return x.view(self.batch, self.num_q_heads, self.head_dim)

    def new_tokens(self, step: int = 0, device="cpu"):
        """(k_new, v_new) fp16 [B][Hkv][d] for decode step `step`, with the same
        outlier structure as the prefill."""
        shape = (self.batch, self.num_kv_heads, self.head_dim)
        n = math.prod(shape)
        return (self._kv("knew", shape, device, step * n), self._kv("vnew", shape, device, step * n))


def _normal_at(seed: int, tensor_id: int, positions: torch.Tensor) -> torch.Tensor:
    """Normals of stream (seed, tensor_id) at arbitrary element positions."""
    key = _key(seed, tensor_id)
    c1 = (2 * positions + 1) * _s64(_GOLDEN) + key
    c2 = (2 * positions + 2) * _s64(_GOLDEN) + key
    u1 = _lsr(_mix64(c1), 11).to(torch.float64) * (2.0 ** -53)
    u2 = _lsr(_mix64(c2), 11).to(torch.float64) * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos((2.0 * math.pi) * u2)


WORKLOADS = {
    1: Workload(1, "tiny-d64-int4-L256", 1, 1, 1, 64, 4, 64, 256, 256),
    2: Workload(2, "llama3.1-8b-int4-32k", 1, 32, 8, 128, 4, 128, 32768, 32768,
                k_outlier_channels=4),
    3: Workload(3, "llama3.1-8b-int2-128k", 1, 32, 8, 128, 2, 128, 131072, 131072,
                k_outlier_channels=4),
    4: Workload(4, "llama2-13b-int4-b64-ragged", 64, 40, 40, 128, 4, 96, 1024, 4096,
                sparse_outlier_p=0.01, sparse_outlier_sigma=8.0),
    5: Workload(5, "pack-32k-x8-d128", 1, 8, 8, 128, 4, 0, 32768, 32768,
                k_outlier_channels=4),
}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller test sizes)."""
    return dataclasses.replace(w, **changes)
