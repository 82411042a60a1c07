"""Host-side helpers the parity tests and the benchmark rely on, checked on
the CPU: the gather of a paged cache's pool through its block table into the
contiguous layout the oracle uses, the packed-token count of a prefill with a
sink and a window, the code-width override of a workload, and the rule that a
committed profile's DRAM traffic is used only while the sources it was taken on
are unchanged."""

import numpy as np
import torch

import bench
from bit_quantized_kv_pack_gb300 import kvq, synth

from _util import logical


def test_paged_gather_matches_loops():
    rng = np.random.default_rng(1)
    B, H, d, bits, cap, pages = 3, 2, 64, 4, 96, 11
    c = kvq.KVCache(B, H, d, bits, cap, 8, device="cpu", hybrid=1, page_size=32, num_pages=pages)
    perm = rng.permutation(pages)[:B * cap // 32]
    c.block_table.copy_(torch.from_numpy(perm.astype(np.int32)).view(B, cap // 32))
    for name in ("k_codes", "v_codes", "k_params", "v_params", "k_mode", "v_mode"):
        t = getattr(c, name)
        t.copy_(torch.from_numpy(rng.integers(0, 200, t.shape)).to(t.dtype))
    g = logical(c)
    bt = c.block_table.numpy()
    for name in ("k_codes", "k_params", "v_mode"):
        pool, got = getattr(c, name).numpy(), getattr(g, name).numpy()
        assert got.shape[:3] == (B, H, cap)
        for b in range(B):
            for h in range(H):
                for t in range(cap):
                    assert np.array_equal(got[b, h, t], pool[bt[b, t // 32], h, t % 32]), (name, b, h, t)
    # a contiguous cache is returned as it is
    plain = kvq.KVCache(1, 1, d, bits, 8, 0, device="cpu")
    assert logical(plain) is plain


def test_packed_per_seq():
    w = synth.WORKLOADS[4]  # Nr = 96
    lens = torch.tensor([0, 20, 96, 97, 140, 4096], dtype=torch.int32)
    assert bench.packed_per_seq(w, lens) == [0, 0, 0, 1, 44, 4000]
    # with a 32-token sink the first 32 tokens leave the packed count too
    assert bench.packed_per_seq(w, lens, 32) == [0, 0, 0, 0, 12, 3968]


def test_workload_bits_override():
    w = bench.workload_for(2, 3)
    assert w.bits == 3 and w.name == "llama3.1-8b-int3-32k"
    assert w.len_max == synth.WORKLOADS[2].len_max and w.seed == synth.WORKLOADS[2].seed
    assert bench.workload_for(3).name == "llama3.1-8b-int2-128k"


def test_profile_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    """The bench line's roofline traffic comes from a committed ncu summary only
    while its source hash matches the current kernel sources: a copy of the
    sources with one byte changed makes it null."""
    import shutil
    csrc = tmp_path / "bit_quantized_kv_pack_gb300" / "csrc"
    shutil.copytree(bench.os.path.join(bench.ROOT, "bit_quantized_kv_pack_gb300", "csrc"), csrc)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for kind, name, hash_fn, read in (
            ("decode_step", "w", bench.decode_source_hash, bench.profiled_traffic),
            ("quantize_pack", "w", bench.pack_source_hash, bench.profiled_pack_traffic)):
        prof = tmp_path / "profiles" / f"{kind}_{name}.md"
        prof.write_text(f"# summary\n\nsource_hash: {hash_fn()}\ntraffic_bytes_per_launch: 12345\n")
        assert read(name) == 12345.0
        assert read("absent") is None
    def touch(name):
        f = csrc / name
        f.write_bytes(f.read_bytes() + b"\n")
    touch("kvq_decode_tc.cu")  # a decode source only
    assert bench.profiled_traffic("w") is None
    assert bench.profiled_pack_traffic("w") == 12345.0
    touch("kvq_quant.cu")  # a pack source
    assert bench.profiled_pack_traffic("w") is None
