#!/usr/bin/env python3
"""Benchmark of the speculative-KV-coding hot path on GB300.

One step = the whole path over one synthetic cache: encode (rank, model CDF,
interleaved rANS, size scan, compaction into the container), decode (search,
rANS update, stream reads, output) and the ideal-bits reduction.  The default
workload is the Qwen3-32B-shaped bf16 cache (64 layers x {K,V} x 8 heads x
8192 tokens x 128 = 1.07G scalars, calibrated sigma).  ``value`` is raw-KV
bytes per second of the whole step (2 bytes per bf16 scalar), inputs resident
in HBM.  The line also carries, measured in the same run, the Qwen3-8B-shaped
FP8 cache and the 2^32-scalar long-context FP8 cache at 1K/4K/16K-scalar
chunks (``workloads``), each with its coded size against the coder's own model
bits.

``--impl reference`` times the oracle (plain C, one chunk per task on every
host core) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "raw-KV encode & decode GB/s on 1 GB300 (% of roofline); bits/scalar vs ideal"
DEFAULT_WORKLOAD = "qwen3-32b-bf16"
# bytes one status read copies back to the host: the 64-byte workspace head
# (skv_encode and skv_encode_finish read it twice, skv_decode, skv_ideal_bits
# and skv_decode_status once; skv_encode_with_bits twice, three times when its
# ideal-bits pass runs apart)
HEAD_BYTES = 64
# the other full-size workloads measured in the same run: (workload, token
# block, lanes) -- the long-context cache at 1K, 4K and 16K scalars per chunk
EXTRA_WORKLOADS = (("qwen3-8b-e4m3", 0, 0), ("long-32k-e4m3", 8, 1), ("long-32k-e4m3", 32, 1),
                   ("long-32k-e4m3", 128, 4))
# launches of our kernels per step: encode (prep, encode, 2 scans, compact),
# decode (prep, header check, decode; bf16 adds the inverse p-hat table),
# ideal bits (prep, bits, final sum); with per-block scales one more in each
# (scale estimate, scale load, scale estimate).  With the ideal bits inside the
# encoder (fused_bits) they cost one launch, the final sum, and no scale pass.
def launches_per_step(bf16: bool, block_scale: bool, adaptive_blocks: int = 0,
                      fused_bits: bool = False) -> int:
    if adaptive_blocks:   # one phase per token block (tables, chunks, update)
        nb = adaptive_blocks
        return (5 + 3 * nb - 1) + (4 + 2 * nb + nb - 1) + (2 + nb + nb - 1)
    if fused_bits:
        return 5 + 1 + (4 if bf16 else 3) + (2 if block_scale else 0)
    return 5 + (4 if bf16 else 3) + 3 + (3 if block_scale else 0)


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a host float over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def layer_range(rank: int, world: int, layers: int):
    """The contiguous layers [l0, l1) of one cache that `rank` codes: chunks are
    independent, so a layer range is a contiguous chunk range of the container."""
    return rank * layers // world, (rank + 1) * layers // world


def payload_bases(total: int, world: int, device=None):
    """Every rank's payload size, gathered (the one collective of the sharded
    path), and their exclusive scan: (base of each rank's part in the single
    container's payload, the whole payload size)."""
    if world <= 1:
        return [0], int(total)
    import torch
    import torch.distributed as dist
    t = torch.tensor([int(total)], dtype=torch.int64, device=device)
    got = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(got, t)
    sizes = [int(g.item()) for g in got]
    bases = [sum(sizes[:r]) for r in range(world)]
    return bases, sum(sizes)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Algorithmic work per scalar, in thread-instructions.  The irreducible part
# of every operation is the pair of exact cum evaluations that gives a symbol's
# frequency; its cost is measured: k_model_bits does exactly that pair per
# scalar (with the symbol's loads and rank, and a log2), and ncu counts 160
# thread-instructions per scalar for bf16 and 105 for e4m3.  On top of it:
# encode's rANS division, renormalisation and word store (at least ~10 bf16,
# ~15 e4m3: the bf16 encoder executes 185 in all, measured), decode's state
# update, stream read and store (~20), whatever its search costs.  Ideal bits:
# two Gaussian bin masses, the p-hat term and one logarithm (70 bf16, 50 e4m3:
# estimates; inside the bf16 encoder they add 86 thread-instructions per
# scalar, measured).  Each figure stays below what the kernels execute.
ALG_OPS = {2: {"encode": 170, "decode": 180, "ideal_bits": 70, "encode_with_bits": 240},
           1: {"encode": 120, "decode": 125, "ideal_bits": 50, "encode_with_bits": 170},
           # order-0 baseline: one cum evaluation is an E_q load, a multiply and
           # a shift (about 8); encode = 2 of them + the divide, renormalisation,
           # rank and loads = 70; decode = the table bracket + ~6 bisection
           # steps + 2 evaluations + the state update = 90; ideal bits = one
           # log2 = 20 (estimates)
           "o0": {"encode": 70, "decode": 90, "ideal_bits": 20, "encode_with_bits": 90}}
OPS_BASIS = {
    "encode": "per scalar: the exact cum pair (measured by ncu on k_model_bits: 160 bf16 / "
              "105 e4m3 thread-instructions) + the rANS division, renormalisation and word "
              "store (estimate, >= 10 bf16 / 15 e4m3)",
    "decode": "per scalar, the minimum any decoder of this model executes: the exact cum pair "
              "that verifies the symbol (measured by ncu on k_model_bits: 160 bf16 / 105 e4m3 "
              "thread-instructions) + the state update, stream read and store (estimate, ~20); "
              "no search",
    "ideal_bits": "per scalar: the Gaussian bin masses, the p-hat term and the logarithm "
                  "(estimate: 70 bf16, 50 e4m3)",
    "encode_with_bits": "per scalar: encode's figure + ideal bits' figure"}
KERNEL = {"encode": "k_encode", "decode": "k_decode", "ideal_bits": "k_ideal",
          "encode_with_bits": "k_encode (ideal bits inside)"}
KERNEL_O0 = {"encode": "k_encode", "decode": "k_decode_o0", "ideal_bits": "k_ideal"}


def issue_peak_gops():
    """Thread-instruction issue peak: SMs x 4 schedulers x 32 lanes x max SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = 2070.0
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return sms * 128 * mhz * 1e6 / 1e9, sms, mhz


def roofline(med_ms, n, container_bytes, bps, workload, order0=False, fused_bits=True):
    """ALU roofline of the dominant kernel (and of each kernel), plus its HBM view.
    encode_with_bits: the encoder with the ideal bits inside (fused_bits) or
    the encoder and the ideal-bits kernel back to back; its algorithmic bytes
    are one read of the inputs either way."""
    peak_ops, sms, mhz = issue_peak_gops()
    hbm_peak, peak_kind = measured_peaks()
    cb = container_bytes / n
    mub = 0 if order0 else 2          # the order-0 baseline reads no mu
    alg_bytes = {"encode": bps + mub + cb, "decode": cb + mub + bps, "ideal_bits": bps + mub,
                 "encode_with_bits": bps + mub + cb}
    ops_tab = ALG_OPS["o0"] if order0 else ALG_OPS[bps]
    kname = dict(KERNEL_O0 if order0 else KERNEL)
    kname["encode_with_bits"] = KERNEL["encode_with_bits"] if fused_bits else "k_encode + k_ideal"
    kernels = {}
    for op, ms in med_ms.items():
        ops = ops_tab[op] * n / (ms * 1e-3) / 1e9
        gbs = alg_bytes[op] * n / (ms * 1e-3) / 1e9
        kernels[op] = {"kernel": kname[op], "ms": round(ms, 4),
                       "alu_frac": round(ops / peak_ops, 4),
                       "hbm_frac": round(gbs / hbm_peak, 4)}
    top = max(med_ms, key=med_ms.get)
    ms = med_ms[top]
    achieved = ops_tab[top] * n / (ms * 1e-3) / 1e9
    gbs = alg_bytes[top] * n / (ms * 1e-3) / 1e9
    roof = {"bound": "alu", "kernel": kname[top], "achieved": round(achieved, 1),
            "peak": round(peak_ops, 1), "unit": "Gop/s", "frac": round(achieved / peak_ops, 4),
            "traffic": load_traffic(kname[top], workload),
            "ops_per_scalar": ops_tab[top], "ops_basis": OPS_BASIS[top],
            "peak_source": "%d SMs x 128 lanes x %.0f MHz (issue peak)" % (sms, mhz),
            "hbm": {"achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(gbs / hbm_peak, 4),
                    "algorithmic_bytes_per_scalar": round(alg_bytes[top], 4),
                    "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind}}
    return roof, kernels


def load_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel, {}).get(workload)
    if not ent:
        return None
    import importlib
    B = importlib.import_module("lossless_kv_cache_fixed_gb300.build")  # the module, not P.build()
    if ent.get("source_digest") != B.source_digest():
        return None
    return ent.get("bytes_per_launch")


# ----------------------------------------------------------------------------
# oracle timing (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------

def oracle_sample_step(O, m, kv, mu, chunks):
    """Encode, decode and ideal bits of the listed chunks, single-threaded."""
    s = m.s
    D, T, Tb = s.D, s.T, s.Tb
    ntb = (T + Tb - 1) // Tb
    dec = _scratch_for(kv)
    if getattr(m.s, "adaptive", 0):
        dec[:] = kv        # adaptive tables read the row's earlier blocks from here
    scalars = 0
    for c in chunks:
        words = O._encode_chunk_raw(m, kv, mu, c)
        rc = O.decode_chunk(m, words, mu, c, dec)
        if rc != 0:
            raise RuntimeError("oracle decode failed rc=%d" % rc)
        row, tb = divmod(c, ntb)
        t0 = tb * Tb
        tn = min(Tb, T - t0)
        base = row * T * D + t0 * D
        O.ideal_bits(m, kv, mu, base, base + tn * D)
        scalars += tn * D
    return scalars


_SCRATCH = {}


def _scratch_for(kv):
    key = (kv.dtype.str, kv.size)
    if key not in _SCRATCH:
        import numpy as np
        _SCRATCH[key] = np.empty_like(kv)
    return _SCRATCH[key]


def oracle_setup(workload_name, seed, device, block_scale=False, order0=False, adaptive=False,
                 token_block=0):
    import oracle as O
    import synth
    O.build()
    spec = synth.WORKLOADS[workload_name]
    if token_block:
        spec = spec.scaled(Tb=token_block)
    w = synth.make(spec, device=device, seed=seed)
    kv, mu, sigma, counts = synth.to_numpy(w)
    s = w.spec
    if order0:
        m = O.Model(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G, None, counts=counts,
                    weights=(0, 0, 100), adaptive=adaptive)
        return O, w, m, kv.reshape(-1), None
    m = O.Model(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G, sigma, counts=counts,
                block_scale=block_scale)
    return O, w, m, kv.reshape(-1), mu.reshape(-1)


def time_oracle(O, m, kv, mu, nchunks_total, budget_chunks, threads=1):
    """Time the oracle on an evenly spread, deterministic sample of chunks, on
    `threads` host threads (one slice of the sample each; every chunk is coded
    single-threaded, and the C calls release the interpreter lock)."""
    step = max(1, nchunks_total // budget_chunks)
    chunks = list(range(0, nchunks_total, step))[:budget_chunks]
    t0 = time.perf_counter()
    if threads <= 1:
        scalars = oracle_sample_step(O, m, kv, mu, chunks)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=threads) as ex:
            scalars = sum(ex.map(lambda cs: oracle_sample_step(O, m, kv, mu, cs),
                                 [chunks[i::threads] for i in range(threads)]))
    dt = time.perf_counter() - t0
    return scalars, dt, chunks


def host_cpu():
    """(CPU model name, host cores this process may use)."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                name = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not name:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu part")):
                        name = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return name or platform.machine(), max(1, cores)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def make_codec(P, w, s, dev, flags):
    """Codec for workload w coded with the chunking of spec s (its Tb and G)."""
    import numpy as np
    import torch
    import synth
    ecdf = phat = None
    if s.dtype == synth.BF16:
        E, ph = P.skv_build_ecdf(w.counts.cpu().numpy().astype(np.uint64))
        ecdf = torch.from_numpy(E.view(np.int32)).to(dev)
        phat = torch.from_numpy(ph).to(dev)
    order0 = bool(flags & P.SKV_FLAG_ORDER0)
    codec = P.Codec(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G,
                    None if order0 else w.sigma.to(dev), ecdf, phat, flags=flags)
    return codec, ecdf, phat


def device_inputs(w, order0=False):
    import torch
    import synth
    kv = (w.kv.view(torch.int16) if w.spec.dtype == synth.BF16 else w.kv).reshape(-1)
    # the order-0 baseline codes the cache alone: no prediction is read
    mu = None if order0 else w.mu.view(torch.int16).reshape(-1)
    return kv, mu


def time_steps(codec, kv, mu, out, dec, steps, warmup, world, clock_index=None, exchange=None,
               with_bits=True):
    """W untimed steps, then K steps timed with CUDA events on the launching
    stream between barriers and synchronisations.  A step is encode with the
    ideal bits (skv_encode_with_bits) and decode; with_bits=False (adaptive
    counts) runs encode, decode and ideal bits apart.  exchange(nb), when
    given, runs after each encode (the ranks' payload sizes)."""
    import torch
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        if with_bits:
            _, nb, bits = codec.encode_with_bits(kv, mu, out=out)
        else:
            _, nb = codec.encode(kv, mu, out=out)
        if exchange is not None:
            exchange(nb)
        if ev:
            ev[1].record(stream)
        codec.decode(out, nb, mu, out=dec)
        if ev:
            ev[2].record(stream)
        if not with_bits:
            bits = codec.ideal_bits(kv, mu)
        if ev:
            ev[3].record(stream)
        return nb, bits

    for _ in range(warmup):
        nb, bits = step()
    torch.cuda.synchronize()
    if not torch.equal(dec, kv):
        raise RuntimeError("decode mismatch in warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(clock_index) as clk:
        start.record(stream)
        for i in range(steps):
            nb, bits = step(evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    t = {"encode_with_bits" if with_bits else "encode": [e[0].elapsed_time(e[1]) for e in evs],
         "decode": [e[1].elapsed_time(e[2]) for e in evs]}
    if not with_bits:
        t["ideal_bits"] = [e[2].elapsed_time(e[3]) for e in evs]
    return {"ms": start.elapsed_time(stop), "nb": nb, "bits": bits, "clk": clk, "t": t}


def time_alone(codec, kv, mu, out, reps=5):
    """Median ms of encode and of ideal bits each called on its own (after
    the timed region, for the per-kernel view when the step runs them as one
    call)."""
    import torch
    stream = torch.cuda.current_stream()
    res = {}
    for op, fn in (("encode", lambda: codec.encode(kv, mu, out=out)),
                   ("ideal_bits", lambda: codec.ideal_bits(kv, mu))):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        res[op] = statistics.median(ts)
    return res


def medians(t):
    return {op: statistics.median(v) for op, v in t.items()}


def size_accounting(n, nb, nchunks, bits, model_bits):
    """Coded size against the continuous ideal and against the coder's own
    model bits (sum of M - log2 freq), whole container and payload alone."""
    payload = 8.0 * (nb - 64 - 8 * (nchunks + 1))
    return {"bits_per_scalar": round(8.0 * nb / n, 5),
            "payload_bits_per_scalar": round(payload / n, 5),
            "ideal_bits_per_scalar": round(bits / n, 5),
            "model_bits_per_scalar": round(model_bits / n, 5),
            "overhead_pct": round(100.0 * (8.0 * nb / bits - 1.0), 3),
            "overhead_vs_model_pct": round(100.0 * (8.0 * nb / model_bits - 1.0), 3),
            "payload_overhead_vs_model_pct": round(100.0 * (payload / model_bits - 1.0), 3)}


def run_gpu(args):
    import torch

    import synth
    import lossless_kv_cache_fixed_gb300 as P

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    _init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    P.build()

    spec = synth.WORKLOADS[args.workload]
    if args.adaptive and not args.token_block:
        args.token_block = 128   # the entropy-estimation page's N_update
    if args.lanes or args.token_block:
        spec = spec.scaled(G=args.lanes or spec.G, Tb=args.token_block or spec.Tb)
    if args.layers:
        spec = spec.scaled(L=args.layers)   # a smaller case of the same recipe (profiling)
    # one cache; under torchrun each rank holds and codes a contiguous layer range of it
    l0, l1 = layer_range(rank, world, spec.L)
    w = synth.make(spec, device=dev, seed=0, layers=(l0, l1))
    s = w.spec
    bps = 2 if s.dtype == synth.BF16 else 1
    flags = (P.SKV_FLAG_DECODE_BISECT if args.decode_bisect else 0) | (
        P.SKV_FLAG_BLOCK_SCALE if args.block_scale else 0) | (
        P.SKV_FLAG_ORDER0 if args.order0 else 0) | (P.SKV_FLAG_ADAPTIVE if args.adaptive else 0)
    codec, ecdf, phat = make_codec(P, w, s, dev, flags)
    kv, mu = device_inputs(w, args.order0)
    n = s.n
    raw = n * bps
    out = torch.empty(codec.max_bytes, dtype=torch.uint8, device=dev)
    dec = torch.empty_like(kv)

    nch_part = s.L * 2 * s.H * ((s.T + s.Tb - 1) // s.Tb)
    exchange = None
    if world > 1:
        # the placement of this rank's part in the single container
        def exchange(nb):
            return payload_bases(nb - 64 - 8 * (nch_part + 1), world, dev)
    with_bits = not args.adaptive     # skv_encode_with_bits takes no adaptive counts
    r = time_steps(codec, kv, mu, out, dec, args.steps, args.warmup, world, local, exchange,
                   with_bits=with_bits)
    nb, bits, clk = r["nb"], r["bits"], r["clk"]
    ms = max_over_ranks(r["ms"], world, dev)
    ms_step = ms / args.steps
    raw_all = spec.n * bps            # the whole cache, over all ranks
    value = raw_all / (ms_step * 1e-3) / 1e9
    model_bits = None if args.adaptive else codec.model_bits(kv, mu)
    med = medians(r["t"])
    alone = time_alone(codec, kv, mu, out) if with_bits else None
    fused = codec.encode_with_bits_fused() if with_bits else False

    # ---- end to end through the C ABI with host buffers ----
    e2e = off = None
    if not args.no_e2e:
        e2e = end_to_end(P, codec, s, w, ecdf, phat, flags, kv, mu, out, raw, world, dev, args,
                         raw_all)
        # range decode (the offload paths) takes whole containers only for adaptive counts
        if not args.adaptive:
            kv_h = kv.cpu().pin_memory()
            off = offload(codec, out, nb, kv, kv_h, mu, s, raw, world, dev, args)
            del kv_h
    line = finish_line(args, rank, world, s, n, nb, bits, model_bits, bps, ms_step, value,
                       med, clk, e2e, w, off, alone=alone, fused_bits=fused)
    # the other full-size workloads, one after another on the freed device
    del codec, kv, mu, out, dec, w, ecdf, phat
    torch.cuda.empty_cache()
    if world == 1 and not args.no_extra and args.workload == DEFAULT_WORKLOAD and not (
            args.order0 or args.adaptive or args.block_scale or args.decode_bisect
            or args.lanes or args.token_block or args.layers):
        extra = extra_workloads(P, dev, args, rank, world, local)
        if line is not None:
            line["workloads"] = extra
    return line


def extra_workloads(P, dev, args, rank, world, local):
    """Encode, decode and ideal bits of the FP8 8B cache and of the long-context
    FP8 cache at each chunk size: GB/s per operation, coded size against the
    model bits (the pages' FP8 model has no floor, so its continuous ideal is no
    bound there), each timed region with its own clock record."""
    import torch
    import synth
    res = {}
    steps, warmup = max(3, min(args.steps, 5)), 3
    have = None
    w = None
    for name, tb, G in EXTRA_WORKLOADS:
        spec = synth.WORKLOADS[name]
        if have != name:
            w = None
            torch.cuda.empty_cache()
            w = synth.make(spec, device=dev, seed=0)
            have = name
        s = spec.scaled(Tb=tb or spec.Tb, G=G or spec.G)
        bps = 2 if s.dtype == synth.BF16 else 1
        codec, _, _ = make_codec(P, w, s, dev, 0)
        kv, mu = device_inputs(w)
        out = torch.empty(codec.max_bytes, dtype=torch.uint8, device=dev)
        dec = torch.empty_like(kv)
        r = time_steps(codec, kv, mu, out, dec, steps, warmup, world, local)
        mbits = codec.model_bits(kv, mu)
        ms = max_over_ranks(r["ms"], world, dev) / steps
        raw = s.n * bps
        nch = s.L * 2 * s.H * ((s.T + s.Tb - 1) // s.Tb)
        med = medians(r["t"])
        fused = codec.encode_with_bits_fused()
        alone = time_alone(codec, kv, mu, out, reps=3)
        _, kernels = roofline(med, s.n, r["nb"], bps, name, fused_bits=fused)
        _, k_alone = roofline(alone, s.n, r["nb"], bps, name)
        med.update(alone)
        key = name if not tb else "%s/%dK" % (name, s.Tb * s.D // 1024)
        ent = {"workload": name, "symbols": "bf16" if bps == 2 else "e4m3",
               "scalars": s.n, "token_block": s.Tb, "lanes": s.G, "chunk_scalars": s.Tb * s.D,
               "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 4),
               "value": round(world * raw / (ms * 1e-3) / 1e9, 3),
               "fused_bits": fused}
        ent.update(op_gbs(med, raw))
        ent.update(size_accounting(s.n, r["nb"], nch, r["bits"], mbits))
        ent["kernels"] = kernels
        ent["kernels_alone"] = k_alone
        ent["clocks"] = r["clk"].summary()
        res[key] = ent
        del codec, kv, mu, out, dec
        torch.cuda.empty_cache()
    return res


def end_to_end(P, codec, s, w, ecdf, phat, flags, kv, mu, out, raw, world, dev, args,
               raw_all=None):
    """The step through the C ABI with the inputs in pinned host memory and the
    results read back every step.  Modes that produce the product's single
    container lead; the layer-group split (separate containers) rides along."""
    import torch
    n = s.n
    raw_all = raw_all or raw          # all ranks' raw bytes: the figures are whole-job
    kv_h = kv.cpu().pin_memory()
    mu_h = None if mu is None else mu.cpu().pin_memory()
    box_h = torch.empty(codec.max_bytes, dtype=torch.uint8).pin_memory()
    kv_back = torch.empty_like(kv_h).pin_memory()
    kv_d = torch.empty_like(kv)
    mu_d = None if mu is None else torch.empty_like(mu)
    box_d = out
    mub = 0 if mu is None else 2      # mu bytes per scalar moved
    # the step's calls, as in the device-timed step: encode with the ideal bits
    # and decode (adaptive counts: encode, decode and ideal bits)
    with_bits = not flags & P.SKV_FLAG_ADAPTIVE
    fused = with_bits and codec.encode_with_bits_fused()
    heads = 1 + (2 if fused else 3)   # status reads per step (decode + encode's)

    def encode_and_bits(kv_in, mu_in, box):
        if with_bits:
            _, nbx, tot = codec.encode_with_bits(kv_in, mu_in, out=box)
            return nbx, tot
        _, nbx = codec.encode(kv_in, mu_in, out=box)
        return nbx, None

    def e2e_step():
        kv_d.copy_(kv_h, non_blocking=True)
        if mu_d is not None:
            mu_d.copy_(mu_h, non_blocking=True)
        nb2, tot = encode_and_bits(kv_d, mu_d, box_d)
        box_h[:nb2].copy_(box_d[:nb2], non_blocking=True)
        box_d[:nb2].copy_(box_h[:nb2], non_blocking=True)
        codec.decode(box_d, nb2, mu_d, out=kv_d)
        kv_back.copy_(kv_d, non_blocking=True)
        if tot is None:
            tot = codec.ideal_bits(kv_d, mu_d)
        torch.cuda.synchronize()
        return nb2, tot

    def timed(fn, reps):
        for _ in range(max(1, args.warmup)):
            fn()
        barrier(world)
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            res = fn()
            ts.append(time.perf_counter() - t0)
        return ts, res

    ts, (nb2, _) = timed(e2e_step, args.steps)
    if not torch.equal(kv_back, kv_h):
        raise RuntimeError("end-to-end round trip mismatch")
    # the median step: a single slow step (the host side) does not set the figure
    e2e_s = max_over_ranks(statistics.median(ts), world, dev)
    staged_e2e = {"value": round(raw_all / e2e_s / 1e9, 3), "unit": "GB/s",
                  "h2d_bytes_per_step": int(raw + mub * n + nb2),
                  "d2h_bytes_per_step": int(nb2 + raw + heads * HEAD_BYTES),
                  "mode": "one container: staging copies to and from device buffers "
                          "(the container makes a round trip through host memory)",
                  "step_s_spread": spread(ts)}

    # the same step with the kernels reading and writing the pinned host buffers
    # directly (mapped memory over the CPU-GPU link): no staging copies
    def e2e_zero_copy():
        nb3, tot = encode_and_bits(kv_h, mu_h, box_h)
        codec.decode(box_h, nb3, mu_h, out=kv_back)
        if tot is None:
            tot = codec.ideal_bits(kv_h, mu_h)
        return nb3, tot

    kv_back.zero_()
    ts, (nb3, _) = timed(e2e_zero_copy, args.steps)
    if not torch.equal(kv_back, kv_h):
        raise RuntimeError("zero-copy round trip mismatch")
    zc_s = max_over_ranks(statistics.median(ts), world, dev)
    zc = {"value": round(raw_all / zc_s / 1e9, 3), "unit": "GB/s",
          # encode reads kv and mu, decode the container and mu, and the
          # ideal bits, unless inside the encoder, kv and mu again
          "h2d_bytes_per_step": int(raw + mub * n + nb3 + mub * n
                                    + (0 if fused else raw + mub * n)),
          "d2h_bytes_per_step": int(nb3 + raw + heads * HEAD_BYTES),
          "mode": "one container: kernels read and write pinned host memory over the link",
          "step_s_spread": spread(ts)}
    del box_h
    modes = [zc, staged_e2e]
    single = e2e_single_pipelined(P, codec, s, w, ecdf, phat, flags, kv_h, mu_h, raw_all, world,
                                  dev, args)
    if single:
        modes.append(single)
    committed = e2e_single_committed(P, codec, s, w, ecdf, phat, flags, kv_h, mu_h, raw_all,
                                     world, dev, args)
    if committed:
        modes.append(committed)
    groups = []
    for to_host in (False, True):
        g = e2e_pipelined(P, s, w, ecdf, phat, flags, kv_h, mu_h, raw_all, world, dev, args,
                          decode_to_host=to_host)
        if g:
            groups.append(g)
    # the headline is the fastest mode that writes the product's single container
    modes.sort(key=lambda m: -m["value"])
    e2e = dict(modes[0])
    e2e["other_modes"] = modes[1:] + sorted(groups, key=lambda m: -m["value"])
    return e2e


def e2e_single_pipelined(P, codec, s, w, ecdf, phat, flags, kv_h, mu_h, raw_all, world, dev,
                         args, groups=8, ranges=4, decode_to_host=False):
    """The end-to-end step writing one container, pipelined: the layer groups'
    inputs are copied in on a copy stream while the groups already in are
    encoded (skv_encode_range) and their ideal bits computed; skv_encode_finish
    writes the container; its copy out and the copies out of the decoded
    cache, range by range, overlap the range decodes (skv_decode_range).
    decode_to_host: one decode writes the cache straight into the pinned host
    buffer instead (its stores cross the link while it runs)."""
    import torch
    if s.L % groups or mu_h is None or flags & P.SKV_FLAG_ADAPTIVE:
        return None
    main = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    lp = s.L // groups
    per = kv_h.numel() // groups
    nc = codec.num_chunks()
    cpg = nc // groups
    gcodecs = [P.Codec(s.dtype, lp, s.H, s.T, s.D, s.Tb, s.G,
                       w.sigma[g * lp:(g + 1) * lp].to(dev).contiguous(), ecdf, phat, flags=flags)
               for g in range(groups)]
    kv_d = torch.empty(kv_h.numel(), dtype=kv_h.dtype, device=dev)
    mu_d = torch.empty(mu_h.numel(), dtype=mu_h.dtype, device=dev)
    box_d = torch.empty(codec.max_bytes, dtype=torch.uint8, device=dev)
    back_d = torch.empty_like(kv_d)
    back_h = torch.empty_like(kv_h).pin_memory()
    cuts = [nc * i // ranges for i in range(ranges + 1)]
    per_chunk = s.Tb * s.D       # scalars of a full chunk (token blocks divide T here)
    state = {"box_h": None}

    def step():
        evs = []
        with torch.cuda.stream(cin):
            for g in range(groups):
                kv_d[g * per:(g + 1) * per].copy_(kv_h[g * per:(g + 1) * per], non_blocking=True)
                mu_d[g * per:(g + 1) * per].copy_(mu_h[g * per:(g + 1) * per], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cin)
                evs.append(ev)
        bits = 0.0
        for g in range(groups):
            main.wait_event(evs[g])
            codec.encode_range(kv_d, mu_d, g * cpg, (g + 1) * cpg, first=(g == 0), stream=main)
            bits += gcodecs[g].ideal_bits(kv_d[g * per:(g + 1) * per], mu_d[g * per:(g + 1) * per],
                                          stream=main)
        _, nb = codec.encode_finish(out=box_d, stream=main)
        if state["box_h"] is None or state["box_h"].numel() < nb:
            state["box_h"] = torch.empty(nb, dtype=torch.uint8).pin_memory()
        box_h = state["box_h"]
        cout.wait_stream(main)
        with torch.cuda.stream(cout):
            box_h[:nb].copy_(box_d[:nb], non_blocking=True)
        if decode_to_host:
            codec.decode_range(box_d, nb, 0, nc, mu_d, back_h, first=True, stream=main)
        else:
            for r in range(ranges):
                codec.decode_range(box_d, nb, cuts[r], cuts[r + 1], mu_d, back_d, first=(r == 0),
                                   stream=main)
                ev = torch.cuda.Event()
                ev.record(main)
                cout.wait_event(ev)
                a, b = cuts[r] * per_chunk, cuts[r + 1] * per_chunk
                with torch.cuda.stream(cout):
                    back_h[a:b].copy_(back_d[a:b], non_blocking=True)
        codec.decode_status(stream=main)
        cout.synchronize()
        return nb, bits

    if s.T % s.Tb:
        return None
    for _ in range(max(1, args.warmup)):
        step()
    barrier(world)
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        nb, _ = step()
        ts.append(time.perf_counter() - t0)
    if not torch.equal(back_h, kv_h):
        raise RuntimeError("pipelined single-container round trip mismatch")
    dt = max_over_ranks(statistics.median(ts), world, dev)
    return {"value": round(raw_all / dt / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": int(kv_h.numel() * kv_h.element_size() + 2 * s.n),
            "d2h_bytes_per_step": int(nb + kv_h.numel() * kv_h.element_size()
                                      + (groups + 3) * HEAD_BYTES),
            "mode": "one container, pipelined: %d layer groups copied in while earlier groups "
                    "are encoded (skv_encode_range) and their ideal bits computed, then "
                    "skv_encode_finish; %s" % (
                        groups, "the container copied out while one decode writes the cache "
                        "straight into pinned host memory" if decode_to_host else
                        "the container and %d decoded chunk ranges (skv_decode_range) copied "
                        "out while later ranges decode" % ranges),
            "container_bytes": int(nb), "step_s_spread": spread(ts)}


def e2e_single_committed(P, codec, s, w, ecdf, phat, flags, kv_h, mu_h, raw_all, world, dev,
                         args, groups=4, layer_cuts=None):
    """The end-to-end step writing one container, committed as it is encoded:
    the layer groups' inputs are copied in on a copy stream; each group, once
    in, is encoded (skv_encode_range, with SKV_RANGE_BITS: its ideal bits inside
    the encoder, where the encoder fuses them for a group of its size; else an
    ideal-bits pass on a stream of its own) and placed in the container
    (skv_encode_commit), then decoded from the container (skv_decode_range with
    SKV_RANGE_PARTIAL) on a third stream, beside the next group's encode; a
    second copy stream takes the decoded scalars and the container bytes
    committed so far back to host memory while later groups are still being
    copied in and coded.  skv_encode_finish writes the header at the end.
    4 groups of the Qwen3-32B-shaped cache: 68.2 GB/s (65.0 with the ideal-bits
    pass beside the encodes)."""
    import torch
    if layer_cuts is None:
        if s.L % groups:
            return None
        layer_cuts = [s.L * g // groups for g in range(groups + 1)]
    groups = len(layer_cuts) - 1
    if mu_h is None or flags & P.SKV_FLAG_ADAPTIVE or s.T % s.Tb:
        return None
    main = torch.cuda.current_stream()
    cin, cout, dst = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    bst = torch.cuda.Stream()
    nc = codec.num_chunks()
    per_layer = kv_h.numel() // s.L           # scalars of one layer (K and V)
    cpl = nc // s.L                           # chunks of one layer
    sc = [l * per_layer for l in layer_cuts]  # scalar cuts
    cc = [l * cpl for l in layer_cuts]        # chunk cuts
    hb = 64 + 8 * (nc + 1)        # header and offset table
    gcodecs = [P.Codec(s.dtype, layer_cuts[g + 1] - layer_cuts[g], s.H, s.T, s.D, s.Tb, s.G,
                       w.sigma[layer_cuts[g]:layer_cuts[g + 1]].to(dev).contiguous(), ecdf, phat,
                       flags=flags)
               for g in range(groups)]
    # the groups' ideal bits inside their encodes (SKV_RANGE_BITS) where the
    # encoder fuses them for a group of this size, else a pass beside them
    fused = all(gc.encode_with_bits_fused() for gc in gcodecs)
    kv_d = torch.empty(kv_h.numel(), dtype=kv_h.dtype, device=dev)
    mu_d = torch.empty(mu_h.numel(), dtype=mu_h.dtype, device=dev)
    box_d = torch.empty(codec.max_bytes, dtype=torch.uint8, device=dev)
    box_h = torch.empty(codec.max_bytes, dtype=torch.uint8).pin_memory()
    back_d = torch.empty_like(kv_d)
    back_h = torch.empty_like(kv_h).pin_memory()
    ends = torch.zeros(groups, dtype=torch.int64).pin_memory()   # written by the device

    def step():
        evs = []
        with torch.cuda.stream(cin):
            for g in range(groups):
                a, b = sc[g], sc[g + 1]
                kv_d[a:b].copy_(kv_h[a:b], non_blocking=True)
                mu_d[a:b].copy_(mu_h[a:b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cin)
                evs.append(ev)
        bits = 0.0
        sent = hb
        for g in range(groups):
            main.wait_event(evs[g])
            c0, c1 = cc[g], cc[g + 1]
            a, b = sc[g], sc[g + 1]
            codec.encode_range(kv_d, mu_d, c0, c1, first=(g == 0), bits=fused, stream=main)
            codec.encode_commit(c0, c1, box_d, end_bytes=ends[g:g + 1], stream=main)
            committed = torch.cuda.Event()
            committed.record(main)
            if not fused:
                # the group's ideal bits beside its encode (the call synchronises bst)
                bst.wait_event(evs[g])
                bits += gcodecs[g].ideal_bits(kv_d[a:b], mu_d[a:b], stream=bst)
            committed.synchronize()          # the commit has run: ends[g] holds its size
            end = int(ends[g])
            # the group decodes on its own stream, beside the next group's encode
            dst.wait_stream(main)
            codec.decode_range(box_d, box_d.numel(), c0, c1, mu_d, back_d, first=(g == 0),
                               partial=True, stream=dst)
            with torch.cuda.stream(cout):
                cout.wait_stream(main)
                box_h[sent:end].copy_(box_d[sent:end], non_blocking=True)
                cout.wait_stream(dst)
                back_h[a:b].copy_(back_d[a:b], non_blocking=True)
            sent = end
        _, nb = codec.encode_finish(out=box_d, stream=main)
        if fused:
            bits = codec.encode_range_bits(stream=main)
        cout.wait_stream(main)
        with torch.cuda.stream(cout):
            box_h[:hb].copy_(box_d[:hb], non_blocking=True)
        codec.decode_status(stream=dst)
        cout.synchronize()
        return nb, bits

    for _ in range(max(1, args.warmup)):
        step()
    barrier(world)
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        nb, _ = step()
        ts.append(time.perf_counter() - t0)
    if not torch.equal(back_h, kv_h):
        raise RuntimeError("committed single-container round trip mismatch")
    box_d2, _ = codec.encode(kv_d, mu_d)
    if not torch.equal(box_h[:nb].to(dev), box_d2[:nb]):
        raise RuntimeError("committed container differs from skv_encode's")
    del box_d2
    dt = max_over_ranks(statistics.median(ts), world, dev)
    return {"value": round(raw_all / dt / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": int(kv_h.numel() * kv_h.element_size() + 2 * s.n),
            "d2h_bytes_per_step": int(nb + kv_h.numel() * kv_h.element_size() + 8 * groups
                                      + ((4 if fused else groups + 3) * HEAD_BYTES)),
            "mode": "one container, committed as it is encoded: %d layer groups copied in "
                    "while earlier groups are encoded (skv_encode_range%s) and committed "
                    "(skv_encode_commit), and decoded from the container being written "
                    "(skv_decode_range, SKV_RANGE_PARTIAL, beside the next group's encode); "
                    "their decoded scalars and the container's committed bytes copied out as "
                    "they are ready; skv_encode_finish writes the header"
                    % (groups, " with SKV_RANGE_BITS: the ideal bits inside the encoder" if fused
                       else "; their ideal bits computed alongside"),
            "container_bytes": int(nb), "step_s_spread": spread(ts)}


def spread(ts):
    """Median, minimum and maximum of per-step wall times (s)."""
    return {"median": round(statistics.median(ts), 5), "min": round(min(ts), 5),
            "max": round(max(ts), 5), "n": len(ts)}


def e2e_pipelined(P, s, w, ecdf, phat, flags, kv_h, mu_h, raw, world, dev, args, parts=4,
                  decode_to_host=False):
    """The end-to-end step with the cache split into layer groups, each coded as
    its own container on its own stream from its own host thread: one group's
    host-device copies run on the copy engines while other groups compute.
    decode_to_host: the decoder writes the cache straight into the pinned host
    buffer (its stores cross the link), and the container is copied out on a
    second stream as soon as it is written, so the copy engine carries only the
    inputs and the containers."""
    import threading
    import torch
    if s.L % parts or mu_h is None:
        return None
    lp = s.L // parts
    per = kv_h.numel() // parts
    groups = []
    for g in range(parts):
        sig = w.sigma[g * lp:(g + 1) * lp].to(dev).contiguous()
        codec = P.Codec(s.dtype, lp, s.H, s.T, s.D, s.Tb, s.G, sig, ecdf, phat, flags=flags)
        st = torch.cuda.Stream()
        groups.append(dict(
            codec=codec, stream=st,
            kv_h=kv_h[g * per:(g + 1) * per], mu_h=mu_h[g * per:(g + 1) * per],
            kv_d=torch.empty(per, dtype=kv_h.dtype, device=dev),
            mu_d=torch.empty(per, dtype=mu_h.dtype, device=dev),
            box_d=torch.empty(codec.max_bytes, dtype=torch.uint8, device=dev),
            box_h=torch.empty(codec.max_bytes, dtype=torch.uint8).pin_memory(),
            back_d=torch.empty(per, dtype=kv_h.dtype, device=dev),
            back_h=torch.empty(per, dtype=kv_h.dtype).pin_memory(), nb=0,
            out_stream=torch.cuda.Stream()))

    def run(gr):
        st = gr["stream"]
        with torch.cuda.stream(st):
            gr["kv_d"].copy_(gr["kv_h"], non_blocking=True)
            gr["mu_d"].copy_(gr["mu_h"], non_blocking=True)
            _, nb = gr["codec"].encode(gr["kv_d"], gr["mu_d"], out=gr["box_d"], stream=st)
            if decode_to_host:
                # the encode call has synchronised its stream: the container is
                # complete, and its copy out overlaps the decode
                with torch.cuda.stream(gr["out_stream"]):
                    gr["box_h"][:nb].copy_(gr["box_d"][:nb], non_blocking=True)
                gr["codec"].decode(gr["box_d"], nb, gr["mu_d"], out=gr["back_h"], stream=st)
            else:
                gr["box_h"][:nb].copy_(gr["box_d"][:nb], non_blocking=True)
                gr["codec"].decode(gr["box_d"], nb, gr["mu_d"], out=gr["back_d"], stream=st)
                gr["back_h"].copy_(gr["back_d"], non_blocking=True)
            gr["codec"].ideal_bits(gr["kv_d"], gr["mu_d"], stream=st)
            st.synchronize()
            gr["out_stream"].synchronize()
            gr["nb"] = nb

    def step():
        ts = [threading.Thread(target=run, args=(gr,)) for gr in groups]
        for t in ts:
            t.start()
        for t in ts:
            t.join()

    for _ in range(max(1, args.warmup)):
        step()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = max_over_ranks((time.perf_counter() - t0) / args.steps, world, dev)
    for gr in groups:
        if not torch.equal(gr["back_h"], gr["kv_h"]):
            raise RuntimeError("pipelined end-to-end round trip mismatch")
    nbs = sum(gr["nb"] for gr in groups)
    return {"value": round(raw / dt / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": int(raw + 2 * s.n),
            "d2h_bytes_per_step": int(nbs + raw + parts * 4 * HEAD_BYTES),
            "mode": "%d layer groups, each its own container on its own stream and host "
                    "thread (separate containers, not the product's single one): copies "
                    "overlap other groups' kernels%s" % (
                        parts, "; the decoder writes the cache straight into pinned host "
                        "memory" if decode_to_host else ""),
            "container_bytes": int(nbs)}


def offload(codec, out, nb, kv, kv_h, mu, s, raw, world, dev, args, pieces=4):
    """The cache held compressed in pinned host memory and brought back to the
    device where mu is (the pages' section "该方法的用途"): raw KV bytes delivered
    per second by (a) a plain copy of the raw cache over the link, (b) decoding
    the container in place from host memory, (c) copying the container's chunk
    ranges in on a second stream while the previous range decodes."""
    import torch
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    nc = (s.L * 2 * s.H) * ((s.T + s.Tb - 1) // s.Tb)
    head = 64 + 8 * (nc + 1)
    box_h = torch.empty(nb, dtype=torch.uint8).pin_memory()
    box_h.copy_(out[:nb])
    box_d = torch.empty(nb, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(kv)
    offs = box_h[64:head].view(torch.int64)
    cuts = [nc * i // pieces for i in range(pieces + 1)]
    reps = max(3, min(args.steps, 10))

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        for _ in range(reps):
            fn()
        b.record(main)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b) / reps, world, dev)

    def raw_copy():
        dst.copy_(kv_h, non_blocking=True)

    def box_copy():
        box_d.copy_(box_h, non_blocking=True)

    def direct():
        codec.decode_range(box_h, nb, 0, nc, mu, dst, first=True)

    def staged():
        side.wait_stream(main)
        box_d[:head].copy_(box_h[:head], non_blocking=True)
        codec.decode_range(box_d, nb, 0, 0, mu, dst, first=True)
        evs = []
        with torch.cuda.stream(side):
            for i in range(pieces):
                a, b = head + int(offs[cuts[i]]), head + (int(offs[cuts[i + 1]]) if cuts[i + 1] < nc
                                                         else nb - head)
                box_d[a:b].copy_(box_h[a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(side)
                evs.append(e)
        for i in range(pieces):
            main.wait_event(evs[i])
            codec.decode_range(box_d, nb, cuts[i], cuts[i + 1], mu, dst)

    # the link's own rate: best of two timings of each plain copy
    t_raw = min(timed(raw_copy), timed(raw_copy))
    t_box = min(timed(box_copy), timed(box_copy))
    t_dir, t_stg = timed(direct), timed(staged)
    codec.decode_status()
    if not torch.equal(dst, kv):
        raise RuntimeError("offload decode mismatch")
    g = lambda nbytes, ms: round(world * nbytes / (ms * 1e-3) / 1e9, 2)
    return {"unit": "GB/s of raw KV delivered to the device (mu already there)",
            "raw_h2d": g(raw, t_raw), "container_h2d_link": g(nb, t_box),
            "direct_decode_from_host": g(raw, t_dir),
            "staged_pipelined_decode": g(raw, t_stg), "pieces": pieces,
            "staged_note": "each range decode costs about one chunk's decode latency, so "
                           "the pipeline only pays with few, large ranges",
            "raw_over_container": round(raw / nb, 3),
            "best_vs_raw_copy": round(max(t_raw / t_dir, t_raw / t_stg), 3)}


def op_gbs(med, raw):
    """Raw GB/s of each timed operation: encode_gbs, decode_gbs, ..."""
    return {op + "_gbs": round(raw / (ms * 1e-3) / 1e9, 2) for op, ms in med.items()}


def finish_line(args, rank, world, s, n, nb, bits, model_bits, bps, ms_step, value, med, clk,
                e2e, w, off=None, alone=None, fused_bits=False):
    """med: median ms of each operation of the timed step; alone: encode and
    ideal bits timed on their own after it (when the step runs them as one)."""
    if rank != 0:
        return None
    import synth
    raw = n * bps

    # ---- roofline of the dominant kernel ----
    roof, kernels = roofline(med, n, nb, bps, args.workload, order0=args.order0,
                             fused_bits=fused_bits)
    k_alone = None
    if alone:
        _, k_alone = roofline(alone, n, nb, bps, args.workload, order0=args.order0)

    # ---- oracle on the host cores, bounded sample: one core, then all ----
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle as O
        kvn, mun, sig, cnt = synth.to_numpy(w)
        if args.order0:
            m = O.Model(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G, None, counts=cnt,
                        weights=(0, 0, 100), adaptive=args.adaptive)
            mun = None
        else:
            m = O.Model(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G, sig, counts=cnt,  # same chunking
                        block_scale=args.block_scale)
            mun = mun.reshape(-1)
        nch = m.num_chunks()
        kvn = kvn.reshape(-1)
        cpu_model, cores = host_cpu()
        if args.adaptive:
            cores = 1    # adaptive tables read the row's earlier blocks: one thread
        sc1, dt1, ch1 = time_oracle(O, m, kvn, mun, nch, args.cpu_sample_chunks)
        one = {"value": round(sc1 * bps / dt1 / 1e9, 6), "unit": "GB/s", "cores": 1,
               "sample": "%d of %d chunks (%d scalars, every %d-th chunk), %.1f s" % (
                   len(ch1), nch, sc1, max(1, nch // args.cpu_sample_chunks), dt1)}
        budget = min(nch, args.cpu_sample_chunks * cores)
        scn, dtn, chn = time_oracle(O, m, kvn, mun, nch, budget, threads=cores)
        cpu = {"value": round(scn * bps / dtn / 1e9, 6), "unit": "GB/s", "cores": cores,
               "kind": "oracle", "cpu_model": cpu_model,
               "sample": "%d of %d chunks (%d scalars, every %d-th chunk): encode + decode + "
                         "ideal bits, plain C, one slice of chunks per host thread, %.1f s" % (
                             len(chn), nch, scn, max(1, nch // budget), dtn),
               "single_core": one}

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "int64",
        "data": "synthetic",
        "config": {"workload": args.workload, "symbols": "bf16" if bps == 2 else "e4m3",
                   "layers": s.L if world == 1 else args.layers or synth.WORKLOADS[args.workload].L,
                   "heads": s.H, "tokens": s.T, "head_dim": s.D,
                   "scalars_per_gpu": n, "token_block": s.Tb, "lanes": s.G,
                   "block_scale": bool(args.block_scale),
                   "coder": coder_name(args),
                   "parallelism": "one GPU" if world == 1 else
                                  "the cache's layers split over %d ranks: one container, one "
                                  "all-gather of the parts' payload sizes per step" % world,
                   "l2": "inputs larger than L2: %.0f MB KV + %.0f MB mu per step" % (
                       raw / 1e6, 2 * n / 1e6),
                   "step": ("encode with the ideal bits (skv_encode_with_bits: %s) + decode" % (
                       "inside the encoder" if fused_bits else "the ideal-bits pass behind the "
                       "encoder") if "encode_with_bits" in med else
                       "encode + decode + ideal bits")},
    }
    line.update(op_gbs(med, raw))
    if alone:
        line.update({k.replace("_gbs", "_alone_gbs"): v for k, v in op_gbs(alone, raw).items()})
    nch = s.L * 2 * s.H * ((s.T + s.Tb - 1) // s.Tb)
    if model_bits is not None:
        line.update(size_accounting(n, nb, nch, bits, model_bits))
    else:
        line.update({"bits_per_scalar": round(8.0 * nb / n, 5),
                     "ideal_bits_per_scalar": round(bits / n, 5),
                     "overhead_pct": round(100.0 * (8.0 * nb / bits - 1.0), 3)})
    line.update({
        "roofline": roof,
        "kernels": kernels,
        "kernels_alone": k_alone,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "offload": off,
        "gpu_launches": launches_per_step(bps == 2, args.block_scale,
                                          s.T // s.Tb + (s.T % s.Tb > 0) if args.adaptive else 0,
                                          fused_bits) * args.steps,
        "clocks": clk.summary(),
    })
    return line


def coder_name(args) -> str:
    if args.adaptive:
        return "order-0 with adaptive per-row counts"
    return "order-0 baseline (p-hat alone)" if args.order0 else "speculative (mu, sigma mixture)"


def run_reference(args):
    """The oracle as the reference arm, on the host cores of this machine."""
    rank, world, local = _dist()
    if rank != 0:
        return None
    import torch
    device = "cuda" if torch.cuda.is_available() else "cpu"
    if args.adaptive and not args.token_block:
        args.token_block = 128
    O, w, m, kv, mu = oracle_setup(args.workload, 0, device, block_scale=args.block_scale,
                                   order0=args.order0, adaptive=args.adaptive,
                                   token_block=args.token_block)
    s = w.spec
    bps = 2 if s.dtype == 0 else 1
    nch = m.num_chunks()
    cpu_model, cores = host_cpu()
    if args.adaptive:
        cores = 1        # adaptive tables read the row's earlier blocks: one thread
    per_step = max(1, args.ref_chunks_per_step) * cores
    stride = max(1, nch // (per_step * max(1, args.steps + args.warmup)))
    order = list(range(0, nch, stride))
    k = 0
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(max_workers=cores)

    def step():
        nonlocal k
        chunks = [order[(k + i) % len(order)] for i in range(per_step)]
        k += per_step
        return sum(pool.map(lambda cs: oracle_sample_step(O, m, kv, mu, cs),
                            [chunks[i::cores] for i in range(cores)]))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    sc = 0
    for _ in range(args.steps):
        sc += step()
    dt = time.perf_counter() - t0
    v = sc * bps / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 3), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
        "config": {"workload": args.workload, "scalars_per_gpu": s.n, "token_block": s.Tb,
                   "lanes": s.G, "block_scale": bool(args.block_scale),
                   "coder": coder_name(args)},
        "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model,
                         "sample": "%d chunks per step of %d scalars each (every %d-th chunk), "
                                   "encode + decode + ideal bits, one slice of chunks per host "
                                   "thread" % (per_step, s.Tb * s.D, stride)},
        "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["skv", "reference"], default="skv")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-sample-chunks", type=int, default=384)
    ap.add_argument("--ref-chunks-per-step", type=int, default=24)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host round trip")
    ap.add_argument("--no-extra", action="store_true",
                    help="measure the named workload only (not the FP8 and long-context caches)")
    ap.add_argument("--lanes", type=int, default=0, help="override the workload's lanes per chunk")
    ap.add_argument("--token-block", type=int, default=0, help="override the token block")
    ap.add_argument("--layers", type=int, default=0,
                    help="only the first N layers' shape (a smaller case for profiling)")
    ap.add_argument("--decode-bisect", action="store_true",
                    help="decode with the reference bisection search")
    ap.add_argument("--block-scale", action="store_true",
                    help="per-(chunk, 8-channel group) sigma scales in the container")
    ap.add_argument("--order0", action="store_true",
                    help="the order-0 baseline coder (p-hat alone, no mu/sigma; bf16)")
    ap.add_argument("--adaptive", action="store_true",
                    help="adaptive counts per row on the order-0 coder (token block 128)")
    args = ap.parse_args(argv)
    if args.adaptive:
        args.order0 = True
    if args.warmup < 3 and args.impl == "skv":
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    rank, world, _ = _dist()
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
