#!/usr/bin/env python3
"""Decode-step benchmark of the low-bit KV-cache path on GB300.

Workload (default): the Llama-3.1-8B-shaped INT4 32K decode layer -- B1, Hq32,
Hkv8, d128, 32640 packed tokens + a 128-token fp16 residual window, group 32.
A step is one pass of the whole decode hot path, one kvq_decode_step call: the
append of the step's new K/V token (the residual window is full, so its oldest
token is quantized and packed) and decode attention of the step's 32 query
heads over the updated cache -- one kernel launch on the tensor-core path.

Timing: W warm-up steps, then R >= 10 timed regions of exactly K steps each;
a region is one replay of a CUDA graph of K consecutive steps between CUDA
events (synchronize, and a barrier for N > 1, on both sides), and the median
region gives the step time.  Step i runs on cache copy i % n; the copies total
at least 3x the L2 cache, so the packed cache streams from HBM.  value = packed
code + scale bytes per step (K and V, all heads, the tokens the decode reads) /
step time.  The roofline is that of the step kernel; kvq_decode_attention alone
is timed the same way and reported beside it.  By default the line also carries
the 128K INT2 layer, the batched Llama-2-13B layer and the standalone
quantize/pack case under "workloads", each timed the same way with its own
roofline and clock record.

Output: one JSON line (see --help).  --impl reference times the CPU oracle
(the plain fp64 implementation) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

WORKLOAD = 2
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ("kvq_decode.cu", "kvq_decode_generic.cu", "kvq_decode_common.cuh",
                  "kvq_decode_tc.cu", "kvq_ptx.cuh", "kvq_internal.cuh")


# ----------------------------------------------------------------- helpers --

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_across_ranks(ms_per_step: float, e2e_value: float, step_bytes: int, device):
    """Whole-job figures of N independent replicas: the step time is the max over
    ranks, the throughput counts every rank's bytes over that time (weak
    scaling), and the end-to-end throughputs add up.  Works with any
    torch.distributed backend (nccl on GPUs, gloo on CPU)."""
    import torch.distributed as dist
    world = dist.get_world_size()
    t = torch.tensor([ms_per_step, e2e_value], dtype=torch.float64, device=device)
    tmax = t.clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    tsum = t.clone()
    dist.all_reduce(tsum, op=dist.ReduceOp.SUM)
    ms_all = float(tmax[0])
    value_all = step_bytes * world / (ms_all * 1e-3) / 1e9
    return ms_all, value_all, float(tsum[1])


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def decode_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_quantized_kv_pack_gb300", "csrc")
    for n in DECODE_SOURCES:
        p = os.path.join(csrc, n)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str, fused: bool = True):
    """DRAM bytes per launch of the roofline kernel from the committed ncu
    summary, if it was taken on the current decode sources (else None)."""
    kind = "decode_step" if fused else "decode"
    p = os.path.join(ROOT, "profiles", f"{kind}_{workload_name}.md")
    if not os.path.exists(p):
        return None
    src_hash, traffic = None, None
    for line in open(p):
        if line.startswith("source_hash:"):
            src_hash = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    if src_hash != decode_source_hash():
        return None
    return traffic


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        import threading
        self._first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self

        def reader():
            for ln in self.proc.stdout:
                if ln.strip():
                    self.lines.append(ln.strip())
                    self._first.set()
        self._thread = threading.Thread(target=reader, daemon=True)
        self._thread.start()
        # nvidia-smi's start-up can stall the GPU briefly: let it reach steady
        # sampling before the timed region begins
        self._first.wait(timeout=10.0)
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ our arm ------

def workload_for(num, bits=0):
    """Workload `num`, with its code width changed to `bits` when given."""
    from bit_quantized_kv_pack_gb300 import synth
    w = synth.WORKLOADS[num]
    if bits and bits != w.bits:
        w = synth.scaled(w, bits=bits, name=w.name.replace(f"int{w.bits}", f"int{bits}"))
    return w


def packed_per_seq(w, lens, sink=0):
    """Packed tokens of each sequence after the prefill: its length minus the
    sink rows and the fp16 window."""
    out = []
    for L in lens.tolist():
        ns = min(int(L), sink)
        out.append(int(L) - ns - min(int(L) - ns, w.residual))
    return out


def workload_config(w, packed_tokens, extra=None):
    """The config object of the JSON line (both arms)."""
    cfg = {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "bits": w.bits,
           "packed_tokens_per_head": packed_tokens, "residual": w.residual, "group": 32,
           "step": "kvq_decode_step: append + decode attention"}
    cfg.update(extra or {})
    return cfg


def build_state(dev, appends_per_copy, l2_bytes, workload, sink=0, hybrid=0, bits=0, paged=0):
    """Pack the workload once, clone it into enough copies to exceed 3x L2,
    and pre-generate the per-step queries and new tokens on the device.
    `appends_per_copy(ncopy)` is how many fused steps each copy will take."""
    from bit_quantized_kv_pack_gb300 import kvq

    w = workload_for(workload, bits)
    k, v, lens = w.prefill(device=dev)
    npk_b = packed_per_seq(w, lens, sink)
    npk0 = sum(npk_b)  # packed tokens over the batch, per KV head
    per_tok = 2 * (w.head_dim * w.bits // 8 + 4 * (w.head_dim // 32))
    step_bytes0 = npk0 * w.num_kv_heads * per_tok
    res_bytes = w.batch * w.num_kv_heads * (w.residual + sink) * w.head_dim * 2 * 2
    ncopy = max(2, math.ceil(3 * l2_bytes / (step_bytes0 + res_bytes)))
    cap = max(npk_b) + appends_per_copy(ncopy) + 8
    paging = {}
    if paged:  # 32-token pages, each copy's block table a seeded shuffle of its pool
        cap = (cap + 31) // 32 * 32
        paging = dict(page_size=32, num_pages=w.batch * cap // 32)
    base = kvq.KVCache(w.batch, w.num_kv_heads, w.head_dim, w.bits, cap, w.residual, device=dev,
                       sink=sink, hybrid=hybrid, **paging)
    if paged:
        gen = torch.Generator().manual_seed(1000 + workload)
        base.block_table.copy_(torch.randperm(paging["num_pages"], generator=gen, dtype=torch.int32)
                               .view(w.batch, cap // 32))
    kvq.kvq_quantize_pack(base, k, v, lens.to(dev))
    st, word = kvq.kvq_read_error(base)
    if st != kvq.KVQ_OK:
        raise RuntimeError(f"prefill pack failed: {kvq.status_string(st)}")
    del k, v
    copies = [base]
    for _ in range(ncopy - 1):
        c = kvq.KVCache(w.batch, w.num_kv_heads, w.head_dim, w.bits, cap, w.residual, device=dev,
                        sink=sink, hybrid=hybrid, **paging)
        for name in ("k_codes", "v_codes", "k_params", "v_params", "k_res", "v_res", "k_sink",
                     "v_sink", "k_mode", "v_mode", "block_table", "counters"):
            getattr(c, name).copy_(getattr(base, name))
        copies.append(c)
    q = torch.stack([w.query(s, device=dev) for s in range(ncopy)])
    kn, vn = zip(*[w.new_tokens(s, device=dev) for s in range(ncopy)])
    kn, vn = torch.stack(kn), torch.stack(vn)
    out = torch.empty_like(q)
    ws = kvq.workspace_for(base, w.num_q_heads)
    return dict(w=w, copies=copies, q=q, kn=kn, vn=vn, out=out, ws=ws, npk0=npk0,
                per_tok=per_tok, nslot=ncopy, step_bytes=step_bytes0)


def capture(state, nsteps, fused=True):
    """A graph of `nsteps` consecutive steps, step i on cache copy i % ncopy:
    fused steps (append + attention, one kvq_decode_step each) or decode-only
    launches (kvq_decode_attention)."""
    from bit_quantized_kv_pack_gb300 import kvq
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    n = state["nslot"]
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(nsteps):
                j = i % n
                c = state["copies"][j]
                if fused:
                    # consecutive steps use different cache copies, so the kernel
                    # before each step never writes its cache
                    kvq.kvq_decode_step(c, state["q"][j], state["kn"][j], state["vn"][j],
                                        state["out"][j], state["ws"],
                                        flags=kvq.KVQ_STEP_EARLY_CACHE_READ)
                else:
                    kvq.kvq_decode_attention(c, state["q"][j], state["out"][j], state["ws"])
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_region(g, world=1):
    """ms of one replay of g (exactly its steps), bracketed by CUDA events on the
    stream the graph replays on, with a synchronize (and, for N > 1, a barrier)
    on both sides."""
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    b.synchronize()
    if world > 1:
        torch.distributed.barrier()
    return a.elapsed_time(b)


def regions_for(args):
    """Timed regions per measurement (the median of them is reported)."""
    return max(10, args.regions)


def run_decode_workload(args, workload, dev, l2, local, world, sink=0, hybrid=0, bits=0, paged=0):
    """One decode workload: W warm-up steps, then R timed regions of exactly K
    fused steps each (median reported), the decode-only launches timed the same
    way, and the end-to-end steps through the host-buffer entry point."""
    K, W, R = args.steps, args.warmup, regions_for(args)
    e2e_steps = args.e2e_steps

    def appends(ncopy):  # fused steps each copy takes: warm-up, regions, e2e
        return (math.ceil(W / ncopy) + R * math.ceil(K / ncopy) + 4 * math.ceil(e2e_steps / ncopy)
                + 4)

    st = build_state(dev, appends, l2, workload, sink, hybrid, bits, paged)
    w, ncopy = st["w"], st["nslot"]
    g_step = capture(st, K, True)
    g_dec = capture(st, K, False)
    g_warm = capture(st, W, True)
    g_warm.replay()  # exactly W warm-up steps
    g_dec.replay()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_step = [time_region(g_step, world) for _ in range(R)]
        t_dec = [time_region(g_dec, world) for _ in range(R)]
        # keep the same kernels running long enough for several clock samples
        # (decode only: appends would grow the caches)
        t_end = time.time() + 0.6
        while time.time() < t_end:
            t_dec.append(time_region(g_dec))
    torch.cuda.synchronize()
    ms_step = statistics.median(t_step) / K
    ms_dec = statistics.median(t_dec) / K
    step_bytes = st["step_bytes"]
    peak, peak_kind = measured_peak()
    res_bytes = w.batch * w.num_kv_heads * (w.residual + sink) * w.head_dim * 2 * 2
    qo_bytes = 2 * w.batch * w.num_q_heads * w.head_dim * 2
    fused = w.head_dim == 128 and 1 <= w.num_q_heads // w.num_kv_heads <= 4
    options = bool(sink or hybrid or bits or paged)
    if fused:  # the dominant kernel is the step kernel itself (one launch per step)
        rf_kernel, rf_us = "decode_step (append + split-KV decode + combine, one launch)", ms_step * 1e3
    else:
        rf_kernel, rf_us = "decode (split-KV + combine)", ms_dec * 1e3
    achieved = step_bytes / (rf_us * 1e-6) / 1e9
    e2e = run_e2e(st, e2e_steps)
    return {
        "workload": w.name,
        "us_per_step": round(ms_step * 1e3, 3),
        "ms_per_step": round(ms_step, 6),
        "value": round(step_bytes / (ms_step * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "regions": {"count": R, "steps_each": K,
                    "us_per_step_min": round(min(t_step) / K * 1e3, 3),
                    "us_per_step_max": round(max(t_step) / K * 1e3, 3)},
        "all_bytes_gbs": round((step_bytes + res_bytes + qo_bytes) / (ms_step * 1e-3) / 1e9, 2),
        "gpu_launches": (1 if fused else 2) * K,
        "roofline": {"bound": "hbm", "kernel": rf_kernel,
                     "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if options else profiled_traffic(w.name, fused),
                     "algorithmic_bytes_per_launch": step_bytes,
                     "us_per_launch": round(rf_us, 3)},
        "decode_only": {"us_per_launch": round(ms_dec * 1e3, 3),
                        "achieved": round(step_bytes / (ms_dec * 1e-3) / 1e9, 2),
                        "frac": round(step_bytes / (ms_dec * 1e-3) / 1e9 / peak, 4),
                        "how": "kvq_decode_attention alone, same copies, median of the same regions"},
        "e2e": e2e,
        "clocks": clk.summary(),
        "config": workload_config(w, st["npk0"], {
            "l2": f"rotating {ncopy} cache copies ({ncopy * step_bytes / 2**20:.0f} MiB "
                  f"packed) > 3x L2 ({l2 / 2**20:.0f} MiB)",
            "timing": f"median of {R} regions, each one CUDA graph replay of exactly {K} steps "
                      f"between CUDA events", "parallelism": "replicas",
            **({"sink": sink} if sink else {}),
            **({"hybrid": "sym/asym per group, mode bytes"} if hybrid else {}),
            **({"paged": "32-token pages, shuffled block tables"} if paged else {})}),
        "_state": st,
    }


def run_ours(args, rank, world, local):
    from bit_quantized_kv_pack_gb300 import _build
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    head = run_decode_workload(args, args.workload, dev, l2, local, world, args.sink, args.hybrid,
                               args.bits, args.paged)
    head.pop("_state")
    extra = {}
    if args.extra_workloads and not (args.sink or args.hybrid or args.bits or args.paged):
        for wl in (3, 4):
            if wl != args.workload:
                r = run_decode_workload(args, wl, dev, l2, local, world)
                r.pop("_state")
                torch.cuda.empty_cache()
                extra[r["workload"]] = r
        pk = run_pack(args, rank, world, local, with_cpu=False)
        extra[pk["config"]["workload"]] = pk

    ms_step = head["ms_per_step"]
    step_bytes = head["roofline"]["algorithmic_bytes_per_launch"]
    e2e = head["e2e"]
    if world > 1:
        ms_all, value_all, e2e["value"] = reduce_across_ranks(ms_step, e2e["value"], step_bytes, dev)
    else:
        ms_all, value_all = ms_step, head["value"]
    res = {
        "metric": "quantized-KV decode attention: achieved HBM GB/s (% of peak), us/step",
        "value": round(value_all, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_all, 6),
        "us_per_step": round(ms_all * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": f"u{head['config']['bits']} codes, fp16 scale/min, fp32 accumulate",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, fp16)",
        "config": head["config"],
        "regions": head["regions"],
        "all_bytes_gbs": head["all_bytes_gbs"],
        "gpu_launches": head["gpu_launches"],
        "roofline": head["roofline"],
        "decode_only": head["decode_only"],
        "e2e": e2e,
        "clocks": head["clocks"],
    }
    if extra:
        res["workloads"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_seconds, workload=args.workload, sink=args.sink,
                                           bits=args.bits, hybrid=args.hybrid)
        res["cpu_baseline_all_cores"] = cpu_baseline_all_cores(res["cpu_baseline"], args.workload,
                                                               sink=args.sink, bits=args.bits,
                                                               hybrid=args.hybrid)
    return res


def run_e2e(st, nsteps):
    """The same steps end to end through the library's host-buffer entry point,
    kvq_decode_step_host, one call per step, with the step's input block
    [q | k_new | v_new] in pinned host memory and its output read back into
    pinned host memory every step, in its two modes:
      mapped: the step kernel reads the input block and writes out in place over
              the host link (KVQ_STEP_HOST_MAPPED), consecutive steps chained as
              programmatic dependents (the early-read flag);
      copies: one host-to-device copy, the step, one device-to-host copy.
    The line's e2e is the faster; both are reported."""
    from bit_quantized_kv_pack_gb300 import kvq
    n = st["nslot"]
    w = st["w"]
    hq = w.num_q_heads
    ins = torch.cat([st["q"].reshape(n, -1), st["kn"].reshape(n, -1), st["vn"].reshape(n, -1)], 1)
    in_h = ins.cpu().pin_memory()
    out_h = torch.empty_like(st["q"], device="cpu").pin_memory()
    dev_io = kvq.step_io_for(st["copies"][0], hq)
    K = max(n, nsteps)
    step_bytes = st["step_bytes"]
    modes = {"mapped": (kvq.KVQ_STEP_HOST_MAPPED | kvq.KVQ_STEP_EARLY_CACHE_READ, None),
             "copies": (kvq.KVQ_STEP_EARLY_CACHE_READ, dev_io)}
    # per-slot buffers and the stream handle are taken once, as a serving loop
    # holding its own buffers would
    ins_j = [in_h[j] for j in range(n)]
    outs_j = [out_h[j] for j in range(n)]
    stream = torch.cuda.current_stream().cuda_stream
    res = {}
    for name, (flags, io) in modes.items():
        def step(i):
            j = i % n
            kvq.kvq_decode_step_host(st["copies"][j], ins_j[j], hq, outs_j[j], io, st["ws"],
                                     stream=stream, flags=flags)

        for i in range(n):
            step(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(K):
            step(i)
        b.record()
        b.synchronize()
        ms = a.elapsed_time(b) / K
        res[name] = {"value": round(step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                     "us_per_step": round(ms * 1e3, 3)}
    best = min(res, key=lambda k: res[k]["us_per_step"])
    how = {"mapped": "one kvq_decode_step_host call per step with KVQ_STEP_HOST_MAPPED: the step "
                     "kernel reads pinned [q|k_new|v_new] and writes out to pinned host memory in "
                     "place (NVLink-C2C), no copy-engine copies",
           "copies": "one kvq_decode_step_host call per step: pinned [q|k_new|v_new] copied to the "
                     "device, fused step, out copied back to pinned host memory"}
    return {**res[best], "mode": best,
            "h2d_bytes_per_step": int(in_h[0].numel() * in_h.element_size()),
            "d2h_bytes_per_step": int(out_h[0].numel() * out_h.element_size()),
            "how": how[best], "modes": res}


# ---------------------------------------------------------- oracle arm -----

def cpu_baseline(seconds: float, steps: int | None = None, workload: int = WORKLOAD, sink: int = 0,
                 bits: int = 0, hybrid: int = 0):
    """The CPU oracle as it stands (single thread) on whole steps of the same
    workload: append + fp64 decode of every query head."""
    import oracle
    from bit_quantized_kv_pack_gb300 import synth

    w = workload_for(workload, bits)
    k, v, lens = w.prefill()
    npk_b = packed_per_seq(w, lens, sink)
    npk0 = sum(npk_b)
    n_steps_max = steps if steps is not None else 1000
    r = oracle.Cache(w.batch, w.num_kv_heads, w.head_dim, w.bits, max(npk_b) + n_steps_max + 8,
                     w.residual, sink, hybrid)
    oracle.quantize_pack(r, k.numpy(), v.numpy(), lens.numpy())
    del k, v
    per_tok = 2 * (w.head_dim * w.bits // 8 + 4 * (w.head_dim // 32))
    step_bytes = npk0 * w.num_kv_heads * per_tok
    t0 = time.time()
    n = 0
    while True:
        kn, vn = w.new_tokens(n)
        oracle.append(r, kn.numpy(), vn.numpy())
        oracle.decode(r, w.query(n).numpy())
        n += 1
        el = time.time() - t0
        if (steps is not None and n >= steps) or (steps is None and el >= seconds):
            break
    el = time.time() - t0
    return {"value": round(step_bytes * n / el / 1e9, 6), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "sample": f"{n} whole steps (append + decode of all {w.num_q_heads} "
                                        f"query heads of {w.name}), {el:.1f} s, single thread",
            "s_per_step": round(el / n, 4)}


def _oracle_units_worker(job):
    """One process of the all-cores CPU baseline: whole decode steps (append +
    fp64 decode of every query head) for its (sequence, KV head) units, each in
    a cache of its own.  Returns the seconds of its step loop."""
    workload, units, n_steps, sink, bits, hybrid = job
    import oracle
    from bit_quantized_kv_pack_gb300 import synth
    w = workload_for(workload, bits)
    k, v, lens = w.prefill()
    gq = w.num_q_heads // w.num_kv_heads
    caches = []
    for b, h in units:
        L = int(lens[b])
        r = oracle.Cache(1, 1, w.head_dim, w.bits, L + n_steps + 8, w.residual, sink, hybrid)
        oracle.quantize_pack(r, k[b:b + 1, h:h + 1].numpy().copy(), v[b:b + 1, h:h + 1].numpy().copy(),
                             lens[b:b + 1].numpy().copy())
        caches.append((b, h, r))
    t0 = time.perf_counter()
    for st in range(n_steps):
        kn, vn = w.new_tokens(st)
        q = w.query(st)
        for b, h, r in caches:
            oracle.append(r, kn[b:b + 1, h:h + 1].numpy().copy(), vn[b:b + 1, h:h + 1].numpy().copy())
            oracle.decode(r, q[b:b + 1, h * gq:(h + 1) * gq].numpy().copy())
    return time.perf_counter() - t0


def cpu_baseline_all_cores(single: dict, workload: int = WORKLOAD, seconds: float = 10.0,
                           sink: int = 0, bits: int = 0, hybrid: int = 0):
    """The same oracle on all host cores: (sequence, KV head) units spread over
    spawned processes, each running whole steps on its units; throughput = step
    bytes x steps / the slowest process's time."""
    import multiprocessing as mp
    from bit_quantized_kv_pack_gb300 import synth
    w = workload_for(workload, bits)
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    procs = max(1, min(os.cpu_count() or 1, len(units)))
    share = [units[i::procs] for i in range(procs)]
    per_step_one = single["s_per_step"] * max(len(x) for x in share) / len(units)
    n_steps = max(3, int(seconds / max(per_step_one, 1e-6)))
    from concurrent.futures import ProcessPoolExecutor
    # spawn (never fork after CUDA); a worker that fails to start raises instead
    # of being restarted, and a stuck one times out
    try:
        with ProcessPoolExecutor(max_workers=procs, mp_context=mp.get_context("spawn")) as ex:
            futs = [ex.submit(_oracle_units_worker, (workload, sh, n_steps, sink, bits, hybrid))
                    for sh in share]
            times = [f.result(timeout=600) for f in futs]
    except Exception as e:  # report, do not hang the benchmark
        return {"value": None, "unit": "GB/s", "cores": procs, "kind": "oracle",
                "sample": f"not measured: {type(e).__name__}: {e}"[:200]}
    el = max(times)
    step_bytes = single["value"] * 1e9 * single["s_per_step"]
    return {"value": round(step_bytes * n_steps / el / 1e9, 6), "unit": "GB/s", "cores": procs,
            "kind": "oracle", "sample": f"{n_steps} whole steps on {procs} processes "
                                        f"({len(units)} (sequence, KV head) units), slowest {el:.1f} s"}


REF_SLICE = 2048  # packed tokens one reference step decodes


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands (single thread), W untimed
    and then exactly K timed steps.  A step is a bounded sample of the workload:
    the append of the step's new token (every sequence and KV head), then the
    fp64 decode of the gq query heads of one KV head over a REF_SLICE-token slice
    of that head's packed cache (the head and the slice rotate) -- a piece of a
    full step, credited with the slice's packed bytes."""
    if rank != 0:
        return None
    import numpy as np
    import oracle
    from bit_quantized_kv_pack_gb300 import synth

    w = workload_for(args.workload, args.bits)
    k, v, lens = w.prefill()
    npk_b = packed_per_seq(w, lens, args.sink)
    n_total = args.warmup + args.steps
    r = oracle.Cache(w.batch, w.num_kv_heads, w.head_dim, w.bits, max(npk_b) + n_total + 8, w.residual,
                     args.sink, args.hybrid)
    oracle.quantize_pack(r, k.numpy(), v.numpy(), lens.numpy())
    del k, v
    per_tok = 2 * (w.head_dim * w.bits // 8 + 4 * (w.head_dim // 32))
    gq = w.num_q_heads // w.num_kv_heads

    def step(i):
        kn, vn = w.new_tokens(i)
        oracle.append(r, kn.numpy(), vn.numpy())
        b, h = (i // w.num_kv_heads) % w.batch, i % w.num_kv_heads
        lp = int(r.packed_len[b])
        n = min(REF_SLICE, lp)
        t0 = (i * REF_SLICE) % max(lp - n + 1, 1)
        sl = oracle.Cache(1, 1, w.head_dim, w.bits, max(n, 1), 0)  # one KV head, gq query heads
        for name in ("k_codes", "v_codes", "k_params", "v_params"):
            getattr(sl, name)[0, 0, :n] = getattr(r, name)[b, h, t0:t0 + n]
        sl.packed_len[0] = n
        q = w.query(i).numpy()[b:b + 1, h * gq:(h + 1) * gq]
        oracle.decode(sl, np.ascontiguousarray(q))
        return n * per_tok

    for i in range(args.warmup):
        step(i)
    t_start = time.perf_counter()
    nbytes = 0
    for i in range(args.warmup, n_total):
        nbytes += step(i)
    el = time.perf_counter() - t_start
    value = nbytes / el / 1e9
    sample = (f"{args.steps} steps, each the append of the step's token and the fp64 decode of the {gq} "
              f"query heads of one KV head over {REF_SLICE} of its packed tokens ({w.name}); "
              f"{el:.2f} s, single thread")
    return {
        "impl": "reference",
        "metric": "quantized-KV decode attention: achieved HBM GB/s (% of peak), us/step",
        "value": round(value, 6), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, fp16)",
        "config": workload_config(w, sum(npk_b), {
            **({"sink": args.sink} if args.sink else {}),
            **({"hybrid": "sym/asym per group, mode bytes"} if args.hybrid else {})}),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


PACK_SOURCES = ("kvq_quant.cu", "kvq_internal.cuh")


def pack_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_quantized_kv_pack_gb300", "csrc")
    for n in PACK_SOURCES:
        p = os.path.join(csrc, n)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_pack_traffic(workload_name: str):
    """DRAM bytes per launch of the INT4 pack from its committed ncu summary, if
    taken on the current pack sources (else None)."""
    p = os.path.join(ROOT, "profiles", f"quantize_pack_{workload_name}.md")
    if not os.path.exists(p):
        return None
    src_hash, traffic = None, None
    for line in open(p):
        if line.startswith("source_hash:"):
            src_hash = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if src_hash == pack_source_hash() else None


def run_pack(args, rank, world, local, with_cpu=True):
    """Standalone quantize/pack: fp16 K and V of 32768 tokens x 8 KV heads x d128
    (4 outlier channels x10 in K) packed to INT4 and to INT2, all tokens packed
    (no window).  Two input copies alternate so the 134 MB input is not served
    from L2 (129 MB) between packs.  Each timed region is exactly K launches
    (after W warm-ups) between CUDA events; the median of R regions is reported.
    value = input bytes / time (INT4); the roofline counts input + output bytes."""
    from bit_quantized_kv_pack_gb300 import _build, kvq, synth
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peak()
    K, R = args.steps, regions_for(args)
    out = {}
    with ClockSampler(local) as clk:
        for bits in (4, 2):
            w = synth.scaled(synth.WORKLOADS[5], bits=bits)
            ins = []
            for _ in range(2):
                k, v, lens = w.prefill(device=dev)
                ins.append((k, v, lens.to(dev)))
            in_bytes = 2 * ins[0][0].numel() * 2
            cache = kvq.KVCache(w.batch, w.num_kv_heads, w.head_dim, bits, w.len_max, 0, device=dev,
                                hybrid=args.hybrid)
            out_bytes = sum(cache.k_codes.numel() + cache.k_params.numel() * 4 + cache.k_mode.numel()
                            for _ in range(2))
            for i in range(args.warmup):
                k, v, lens = ins[i % 2]
                kvq.kvq_quantize_pack(cache, k, v, lens)
            ts = []
            for _ in range(R):
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for i in range(K):
                    k, v, lens = ins[i % 2]
                    kvq.kvq_quantize_pack(cache, k, v, lens)
                b.record()
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3 / K)
            st, _ = kvq.kvq_read_error(cache)
            if st != kvq.KVQ_OK:
                raise RuntimeError(f"pack failed: {kvq.status_string(st)}")
            us = statistics.median(ts)
            out[bits] = dict(us=us, gbs=in_bytes / (us * 1e-6) / 1e9,
                             traffic_gbs=(in_bytes + out_bytes) / (us * 1e-6) / 1e9,
                             algo=in_bytes + out_bytes)
            del ins, cache
            torch.cuda.empty_cache()
    name = "pack-32768x8x128-kv"
    res = {
        "metric": "quantize/pack throughput: input GB/s (fp16 K+V in, codes + scale/min out)",
        "value": round(out[4]["gbs"], 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(out[4]["us"] * 1e-3, 6),
        "us_per_step": round(out[4]["us"], 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 in, u4/u2 codes + fp16 scale/min out, fp32 arithmetic",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, fp16)",
        "config": {"workload": name, "tokens": 32768, "num_kv_heads": 8,
                   "head_dim": 128, "group": 32, "l2": "two input copies alternate",
                   "timing": f"median of {R} regions of exactly {K} launches between CUDA events",
                   **({"hybrid": "sym/asym per group, mode bytes"} if args.hybrid else {})},
        "int2": {"us_per_step": round(out[2]["us"], 3), "value": round(out[2]["gbs"], 2),
                 "frac": round(out[2]["traffic_gbs"] / peak, 4)},
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "kernel": "quantize_pack (INT4)",
                     "achieved": round(out[4]["traffic_gbs"], 2), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(out[4]["traffic_gbs"] / peak, 4),
                     "traffic": None if args.hybrid else profiled_pack_traffic(name),
                     "algorithmic_bytes_per_launch": out[4]["algo"],
                     "us_per_launch": round(out[4]["us"], 3),
                     "note": "achieved counts input + output bytes"},
        "clocks": clk.summary(),
    }
    if with_cpu and rank == 0 and not args.no_cpu_baseline:
        import oracle
        w = synth.scaled(synth.WORKLOADS[5], bits=4)
        k, v, lens = w.prefill()
        r = oracle.Cache(w.batch, w.num_kv_heads, w.head_dim, 4, w.len_max, 0, 0, args.hybrid)
        t0 = time.perf_counter()
        n = 0
        while n < 1 or time.perf_counter() - t0 < min(args.cpu_seconds, 10.0):
            oracle.quantize_pack(r, k.numpy(), v.numpy(), lens.numpy())
            n += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(n * 2 * k.numel() * 2 / el / 1e9, 4), "unit": "GB/s",
                               "cores": 1, "kind": "oracle",
                               "sample": f"{n} whole INT4 packs of the same K and V, {el:.1f} s, single thread"}
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20, help="steps per timed region (K)")
    ap.add_argument("--warmup", type=int, default=5, help="untimed warm-up steps (W >= 3)")
    ap.add_argument("--regions", type=int, default=15,
                    help="timed regions of K steps each (at least 10); the median is reported")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=WORKLOAD, choices=(1, 2, 3, 4, 5),
                    help="decode workload (default 2: Llama-3.1-8B INT4 32K); 5 = the "
                         "standalone quantize/pack throughput case (INT4 and INT2)")
    ap.add_argument("--no-extra-workloads", dest="extra_workloads", action="store_false",
                    help="time only the headline workload (by default the 128K INT2 layer, the "
                         "batched Llama-2-13B layer and the pack case are added to the line)")
    ap.add_argument("--sink", type=int, default=0,
                    help="attention-sink rows kept fp16 per sequence (0..256; default 0)")
    ap.add_argument("--hybrid", type=int, default=0, choices=(0, 1),
                    help="1: hybrid symmetric/asymmetric groups with mode bytes (default 0)")
    ap.add_argument("--bits", type=int, default=0, choices=(0, 2, 3, 4),
                    help="code width instead of the workload's own (3: the 3-bit variant)")
    ap.add_argument("--paged", type=int, default=0, choices=(0, 1),
                    help="1: packed rows in 32-token pages found through shuffled block tables")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_info()
    if world > 1:
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.workload == 5:
            res = run_pack(args, rank, world, local) if args.impl == "ours" else \
                {"impl": "reference", "unavailable": "the pack case is not the benchmark's decode "
                 "workload; the CPU oracle's pack time is the cpu_baseline of the ours line"}
        elif args.impl == "reference":
            res = run_reference(args, rank, world)
        else:
            res = run_ours(args, rank, world, local)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
