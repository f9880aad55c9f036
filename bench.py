"""Benchmark: TurboQuant compressed-KV decode attention.

Default workload, long_256k (one replica per GPU): 64 layers, 8 KV heads, 64
query heads, head_dim 128, keys 3-bit prod, values 3-bit MSE, 262,144 tokens
prefilled by chunked encode (8192-token chunks), then decode steps that each
append 2 tokens per layer and attend with query length 2 over every layer.
Other workloads of the same family (--workload): stack_32k (64 layers,
32,768 tokens, 4-bit MSE keys and values, q_len 2, no append), paged_batch
(32 ragged sequences in 16-token blocks handed out in a shuffled order, one
token appended per sequence per step, q_len 1), layer_d256 (one head_dim-256
layer, 8192 tokens, group values) and tiny (one layer, 512 tokens).

A step = for each layer: the append of the step's tokens and the decode
attention, through tq_decode_step (the append runs inside the decode's
query-prep launch; --step-api separate: tq_encode_append then
tq_decode_attention), or tq_decode_attention alone for workloads without an
append. `value` is the compressed bytes the step's decode reads (valid tokens
x heads x layers x record bytes, summed over the sequences) divided by the
step time, summed over ranks. Inputs are resident in HBM before the timed
region; caches larger than L2 need no flush, smaller ones are flushed by a
write of 512 MB between timed steps (outside the timed events).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compressed-KV decode-attn HBM GB/s (% of peak) and steps/s @256k; encode Mtok/s"
UNIT = "GB/s"


# DRAM traffic of the dominant decode kernel as an ncu capture measured it,
# valid only for the kernel sources it was measured on (profiles/
# decode_traffic_<workload>.txt: the sources' sha256, the bytes per launch and
# the capture command); otherwise the roofline's traffic is null.
TRAFFIC_SOURCES = ["decode_mma.cuh", "decode_mma_impl.cuh", "decode_mma_a.cu", "decode_mma_b.cu",
                   "decode_mma_c.cu", "decode_step.cu", "decode.cu", "tc_ptx.cuh", "tq_internal.h"]


def decode_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "turboquant_compressed_kv_tq_gb300", "csrc")
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(workload: str):
    """(bytes per launch, source line) from the committed capture record when
    it was taken on the current kernel sources, else (None, reason)."""
    path = os.path.join(ROOT, "profiles", f"decode_traffic_{workload}.txt")
    try:
        rec = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("sources_sha256") != decode_sources_sha256():
            return None, "ncu capture taken on other kernel sources"
        return float(rec["dram_bytes_per_launch"]), rec.get("command", path)
    except (OSError, KeyError, ValueError):
        return None, "no ncu capture of these kernel sources"


def _peaks(key: str = "hbm_gbs"):
    """A measured peak of this GPU pool (HBM copy GB/s or bf16 TFLOP/s), else
    the earlier single measurement the pool's notes give as a fallback."""
    fallback = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p[key]), "measured"
    except Exception:
        return fallback[key], "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity for a single process)."""
    if world == 1:
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


def aggregate(bytes_per_step: float, step_ms_local: float, world: int, device=None):
    """Whole-job throughput of `world` replicas: every rank processed
    `bytes_per_step` per step; the job's step time is the slowest rank's.
    Returns (GB/s over all ranks, max step ms)."""
    step_ms = reduce_max(step_ms_local, world, device)
    return world * bytes_per_step / (step_ms * 1e-3) / 1e9, step_ms


# ------------------------------------------------------------------ oracle baseline

class OracleSample:
    """Oracle records of a bounded sample of a workload: layer 0, sequence 0,
    `kv_heads` KV heads at the sequence's full prefill length (encoded once, by
    the oracle, from the same device-generated inputs the GPU arm encodes)."""

    def __init__(self, w, kv_heads=1, device="cuda"):
        import oracle as O
        from turboquant_compressed_kv_tq_gb300 import workloads as wl
        O.build()
        self.O, self.w = O, w
        self.kv_heads = min(kv_heads, w.num_kv_heads)
        D, N = w.head_dim, w.seq_lens[0]
        self.kc = O.Codec(D, w.key.bits, w.key.mode, w.key.seed, w.key.group_size)
        self.vc = O.Codec(D, w.value.bits, w.value.mode, w.value.seed, w.value.group_size)
        K = wl.kv_chunk(w, 0, 0, 0, N, "k", device)[:self.kv_heads].float().cpu().numpy()
        V = wl.kv_chunk(w, 0, 0, 0, N, "v", device)[:self.kv_heads].float().cpu().numpy()
        self.q = wl.queries(w, 0, 0, device)[0].double().cpu().numpy()
        self.recs = [(self.kc.encode(K[h]), self.vc.encode(V[h])) for h in range(self.kv_heads)]
        self.nbytes = self.kv_heads * N * (self.kc.record_bytes + self.vc.record_bytes)

    def decode_seconds(self):
        """Wall time of the oracle's rotated-domain decode of the sample."""
        w, G = self.w, self.w.gqa
        t0 = time.perf_counter()
        for h in range(self.kv_heads):
            self.O.decode_rotated(self.q[h * G:(h + 1) * G], self.kc, self.recs[h][0], self.vc,
                                  self.recs[h][1], 1 / math.sqrt(w.head_dim), w.q_len)
        return time.perf_counter() - t0

    def describe(self):
        w = self.w
        return (f"oracle rotated-domain decode (fp64, OpenMP over query rows) of {w.name}: layer 0, "
                f"sequence 0, {self.kv_heads} KV head(s) x {w.gqa * w.q_len} query rows, N={w.seq_lens[0]}, "
                f"{self.nbytes / 1e6:.1f} MB of compressed records per sample")


def cpu_baseline(w, kv_heads=2, device="cuda", min_repeats=3, min_seconds=10.0, max_repeats=60):
    """Oracle decode throughput on the host cores (GB/s of compressed bytes):
    the median of timed samples, repeated until about `min_seconds` of decode
    work (at least `min_repeats`, at most `max_repeats`). Returns (value,
    cores, sample, seconds)."""
    smp = OracleSample(w, kv_heads, device)
    times = []
    while len(times) < max_repeats and (len(times) < min_repeats or sum(times) < min_seconds):
        times.append(smp.decode_seconds())
    t = statistics.median(times)
    desc = smp.describe() + f"; median of {len(times)} timed decodes"
    return smp.nbytes / t / 1e9, smp.O.num_threads(), desc, sum(times)


def cpu_baseline_one_core(w, device="cuda"):
    """The same oracle decode on one host core: one KV head of the sample,
    timed once. Returns (value, sample)."""
    smp = OracleSample(w, 1, device)
    cores = smp.O.num_threads()
    smp.O.set_num_threads(1)
    try:
        t = smp.decode_seconds()
    finally:
        smp.O.set_num_threads(cores)
    return smp.nbytes / t / 1e9, smp.describe() + "; one timed decode on 1 thread"


def _workload(args):
    from turboquant_compressed_kv_tq_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]()
    if args.layers:
        # fewer layers of the same workload: a small case for profiler captures,
        # never a headline number (the layer count is in config.workload)
        w = dataclasses.replace(w, num_layers=args.layers)
    return w


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import torch
    w = _workload(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    smp = OracleSample(w, 1, dev)
    for _ in range(args.warmup):
        smp.decode_seconds()
    times = [smp.decode_seconds() for _ in range(args.steps)]
    total = sum(times)
    val = smp.nbytes * args.steps / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": _workload_text(w)},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": smp.O.num_threads(), "kind": "oracle",
                             "sample": smp.describe()},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _codec_text(c):
    name = {0: "MSE", 1: "prod", 2: "group"}[c.mode]
    return f"{c.bits}-bit {name}" + (f" (group {c.group_size})" if c.mode == 2 else "")


def _workload_text(w):
    lens = w.seq_lens
    n = f"N={lens[0]}" if len(lens) == 1 else f"N in [{min(lens)}, {max(lens)}] (sum {sum(lens)})"
    return (f"{w.name}: {w.num_layers} layers, batch {w.batch}, {w.num_kv_heads} KV heads, {w.num_q_heads} "
            f"query heads, head_dim {w.head_dim}, {n} prefilled in {w.prefill_chunk}-token chunks"
            f"{f' then +{w.append_per_step} token(s) per sequence per step' if w.append_per_step else ''}, "
            f"q_len {w.q_len}, {w.block_tokens}-token blocks{' (shuffled)' if w.shuffle_blocks else ''}; "
            f"keys {_codec_text(w.key)}, values {_codec_text(w.value)}; {str(w.dtype).split('.')[-1]} inputs "
            f"N(0, {w.std}^2){' x per-head scale U' + str(w.head_scale_range) if w.head_scale_range else ''}")


# ------------------------------------------------------------------ GPU arm

def measure_prefill_attention(tq, wl, dev, reps: int = 3):
    """Prefill attention of one layer with the long-context codecs: an 8192-token
    chunk (64 query heads) attending to a 24,576-token compressed prefix and
    causally to itself. Useful FLOPs: 2 x (QK^T + PV) over the causal key ranges."""
    import torch
    base = wl.long_256k()
    C, P = 8192, 24576
    w = dataclasses.replace(base, num_layers=1, seq_lens=(P + C,), q_len=C)
    D, Hkv, Hq, BT = w.head_dim, w.num_kv_heads, w.num_q_heads, w.block_tokens
    N = P + C
    nblk = N // BT
    kc = tq.Codec(D, w.key.bits, w.key.mode, w.key.seed)
    vc = tq.Codec(D, w.value.bits, w.value.mode, w.value.seed)
    cache = tq.CompressedKVCache(kc, vc, 1, nblk, BT, Hkv, dev)
    starts = torch.arange(0, N, w.prefill_chunk, dtype=torch.int32, device=dev)
    for c in range(N // w.prefill_chunk):
        k = wl.kv_chunk(w, 0, 0, c * w.prefill_chunk, w.prefill_chunk, "k", dev).unsqueeze(0)
        v = wl.kv_chunk(w, 0, 0, c * w.prefill_chunk, w.prefill_chunk, "v", dev).unsqueeze(0)
        cache.append(0, k, v, starts[c:c + 1], None, nblk)
    q = wl.queries(w, 0, 0, dev)
    sl = torch.tensor([N], dtype=torch.int32, device=dev)
    ws = torch.empty(cache.prefill_workspace_bytes(1, Hq, C), dtype=torch.uint8, device=dev)
    out = torch.empty(1, Hq, C, D, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cache.prefill_attention(0, q, sl, None, nblk, out, ws)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cache.prefill_attention(0, q, sl, None, nblk, out, ws)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    assert tq.tq_device_error() == 0
    ms = statistics.median(times)
    keys = C * P + C * (C + 1) / 2            # visible keys summed over the chunk's positions
    flops = 2.0 * 2.0 * Hq * keys * D
    return {"workload": f"long_256k codecs, one layer: {C}-token chunk, {P}-token compressed prefix, "
                        f"{Hq} query heads, GQA {Hq // Hkv}, causal", "ms": ms,
            "tflops_useful": flops / (ms * 1e-3) / 1e12, "chunk_tokens_per_s": C / (ms * 1e-3),
            "kernel": "qfrag_kernel + prefill_tc_kernel (tcgen05, TMEM)"}


def run_gpu(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from turboquant_compressed_kv_tq_gb300 import build as tqbuild
    if rank == 0 or not os.path.exists(tqbuild.LIB):
        tqbuild.build()
    barrier(world)
    import turboquant_compressed_kv_tq_gb300 as tq
    from turboquant_compressed_kv_tq_gb300 import workloads as wl

    w = _workload(args)
    L, B, Hkv, Hq, D, Lq = w.num_layers, w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim, w.q_len
    A = w.append_per_step
    lens0 = list(w.seq_lens)
    total_steps = args.warmup + args.steps
    caps = [n + A * total_steps for n in lens0]
    cap = max(caps)
    BT = w.block_tokens
    paged = w.shuffle_blocks or B > 1
    if paged:
        table_h, nblk = wl.block_table(w, caps)
        max_blocks = table_h.shape[1]
        table = table_h.to(dev)
    else:
        max_blocks = nblk = (cap + BT - 1) // BT
        table = None
    kc = tq.Codec(D, w.key.bits, w.key.mode, w.key.seed, w.key.group_size)
    vc = tq.Codec(D, w.value.bits, w.value.mode, w.value.seed, w.value.group_size)
    cache = tq.CompressedKVCache(kc, vc, L, nblk, BT, Hkv, dev)
    rec_bytes = kc.record_bytes + vc.record_bytes

    stream = torch.cuda.current_stream(dev)
    # ---------------- prefill: chunked encode of every layer and sequence (timed)
    enc_ms = 0.0
    chunk = w.prefill_chunk
    for layer in range(L):
        jobs = []
        for b in range(B):
            for c0 in range(0, lens0[b], chunk):
                n = min(chunk, lens0[b] - c0)
                jobs.append((b, c0,
                             wl.kv_chunk(w, layer, b + rank * B, c0, n, "k", dev).unsqueeze(0),
                             wl.kv_chunk(w, layer, b + rank * B, c0, n, "v", dev).unsqueeze(0),
                             torch.tensor([c0], dtype=torch.int32, device=dev)))
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for b, c0, k, v, start in jobs:
            cache.append(layer, k, v, start, table[b:b + 1] if paged else None, max_blocks)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        enc_ms += e0.elapsed_time(e1)
        del jobs
    assert tq.tq_device_error() == 0

    # ---------------- decode-step inputs, resident on the device
    steps_in = []
    for s in range(total_steps):
        q = torch.stack([wl.queries(w, layer, s, dev) for layer in range(L)])      # [L, B, Hq, Lq, D]
        if A:
            k_new = torch.stack([torch.stack([wl.kv_chunk(w, layer, b + rank * B, lens0[b] + A * s, A, "k", dev)
                                              for b in range(B)]) for layer in range(L)])
            v_new = torch.stack([torch.stack([wl.kv_chunk(w, layer, b + rank * B, lens0[b] + A * s, A, "v", dev)
                                              for b in range(B)]) for layer in range(L)])
            steps_in.append((k_new.contiguous(), v_new.contiguous(), q.contiguous()))
        else:
            steps_in.append((None, None, q.contiguous()))
    lens_pre = [torch.tensor([n + A * s for n in lens0], dtype=torch.int32, device=dev) for s in range(total_steps)]
    lens_post = [t + A for t in lens_pre]
    ws = torch.empty(cache.workspace_bytes(B, Hq, Lq, cap), dtype=torch.uint8, device=dev)
    out = torch.empty(L, B, Hq, Lq, D, dtype=torch.float32, device=dev)
    # caches that fit in L2 (129 MB) with room to spare are flushed before each step
    l2_resident = sum(lens0) * Hkv * rec_bytes * L < 64e6
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if l2_resident else None

    fused = args.step_api == "fused"

    def step(s, inputs=None):
        k_new, v_new, q = inputs if inputs is not None else steps_in[s]
        for layer in range(L):
            if A and fused:
                # one call: the append runs inside the decode's query-prep launch
                cache.decode_step(layer, k_new[layer], v_new[layer], q[layer], lens_pre[s], table, max_blocks,
                                  cap, out[layer], ws)
                continue
            if A:
                cache.append(layer, k_new[layer], v_new[layer], lens_pre[s], table, max_blocks)
            cache.decode(layer, q[layer], lens_post[s], table, max_blocks, cap, out[layer], ws)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(dev)
    # small workloads are launch-bound on the host: each timed step of an
    # L2-resident cache is replayed from a CUDA graph of its launches
    graphs = None
    if l2_resident:
        try:
            graphs, graph_launches = [], 0
            for s in range(args.warmup, total_steps):
                gph = torch.cuda.CUDAGraph()
                n0 = tq.tq_launch_count()
                with torch.cuda.graph(gph):
                    step(s)
                graph_launches += tq.tq_launch_count() - n0   # kernels each replay launches
                graphs.append(gph)
            torch.cuda.synchronize(dev)
        except Exception as exc:   # capture refused: time the eager calls instead
            print(f"CUDA graph capture unavailable ({exc}); timing eager launches", file=sys.stderr)
            graphs = None
    # ---------------- timed region
    n_launch0 = tq.tq_launch_count()
    barrier(world)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if l2_resident else 1)]
    with ClockSampler(local) as clk:
        if l2_resident:
            # caches that fit in L2: each step timed alone after a flush write
            for i, s in enumerate(range(args.warmup, total_steps)):
                flush.fill_(i & 255)
                evs[i][0].record(stream)
                if graphs is not None:
                    graphs[i].replay()
                else:
                    step(s)
                evs[i][1].record(stream)
        else:
            evs[0][0].record(stream)
            for s in range(args.warmup, total_steps):
                step(s)
            evs[0][1].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    launches = tq.tq_launch_count() - n_launch0   # this library's kernels only (the flush is torch's)
    if graphs is not None:
        launches += graph_launches   # replays launch the captured kernels again
    step_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    # bytes the decode of step s reads: valid tokens x heads x layers x record bytes
    dec_bytes = [L * Hkv * sum(n + A * s + A for n in lens0) * rec_bytes for s in range(args.warmup, total_steps)]
    bytes_per_step = sum(dec_bytes) / args.steps
    value, step_ms_max = aggregate(bytes_per_step, step_ms, world, dev)

    # ---------------- roofline: the decode of one layer is the dominant launch;
    # inside a step a layer's preparation kernel overlaps the previous layer's
    # decode, so the decode's in-step duration per launch is the step time
    # over the layers (CUDA events on the launching stream, timed region above)
    per_launch_bytes = bytes_per_step / L
    launch_ms = step_ms / L
    peak, peak_kind = _peaks()
    achieved = per_launch_bytes / (launch_ms * 1e-3) / 1e9
    traffic, traffic_src = measured_traffic(w.name)
    # the decode call timed alone between events (which serialise it with its
    # neighbours), for reference
    e_iso = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
    s_last = total_steps - 1
    torch.cuda.synchronize(dev)
    for layer in range(L):
        e_iso[layer][0].record(stream)
        cache.decode(layer, steps_in[s_last][2][layer], lens_post[s_last], table, max_blocks, cap, out[layer], ws)
        e_iso[layer][1].record(stream)
    torch.cuda.synchronize(dev)
    iso_ms = sum(a.elapsed_time(b) for a, b in e_iso) / L

    # ---------------- end to end through the API with host buffers
    pin_in = [tuple(None if t is None else t.cpu().pin_memory() for t in steps_in[s])
              for s in range(args.warmup, total_steps)]
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    dev_in = tuple(None if t is None else torch.empty_like(t) for t in steps_in[0])
    h2d = sum(t.numel() * t.element_size() for t in pin_in[0] if t is not None)
    d2h = out_host.numel() * out_host.element_size()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for i, s in enumerate(range(args.warmup, total_steps)):
        for d, h in zip(dev_in, pin_in[i]):
            if d is not None:
                d.copy_(h, non_blocking=True)
        step(s, dev_in)
        out_host.copy_(out, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    e2e_s = reduce_max(e2e_s, world, dev)
    e2e_value = world * bytes_per_step / e2e_s / 1e9
    assert tq.tq_device_error() == 0

    enc_tokens = sum(lens0) * L * Hkv
    pfa = None
    if rank == 0 and not args.no_prefill_attention and w.name == "long_256k" and not args.layers:
        del steps_in, pin_in
        pfa = measure_prefill_attention(tq, wl, dev)
        peak_t, _ = _peaks("bf16_tflops")
        pfa["frac_of_bf16_peak"] = pfa["tflops_useful"] / peak_t if peak_t else None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            v, cores, sample, secs = cpu_baseline(w, kv_heads=2, device=dev)
            v1, sample1 = cpu_baseline_one_core(w, device=dev)
            cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                   "seconds": round(secs, 2), "one_core": {"value": v1, "unit": UNIT, "cores": 1, "sample": sample1}}
        clocks = clk.summary()
        plan = tq.tq_decode_plan(cache.desc, B, Hq, Lq, cap,
                                 torch.cuda.get_device_properties(dev).multi_processor_count)
        dominant = ("split_mma_kernel (tensor-core split-K decode" +
                    (")" if D == 128 else f", head_dim {D}: two 128-column value halves per unit)")
                    if plan["tensor_cores"] else "split_kernel + merge_kernel (SIMT decode)")
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16+f32", "data": "synthetic",
            "config": {"workload": _workload_text(w),
                       "bytes_per_step": bytes_per_step, "record_bytes_per_token_head": rec_bytes,
                       "l2": ("caches fit in L2: a 512 MB write flushes L2 before each timed step"
                              + ("; each step replayed from a CUDA graph" if graphs is not None else "")
                              if l2_resident else
                              f"inputs larger than L2: each step reads {bytes_per_step / 1e9:.2f} GB of records"),
                       "step_api": ("tq_decode_step" if (fused and A) else
                                    "tq_encode_append + tq_decode_attention" if A else "tq_decode_attention"),
                       "block_tokens": BT, "block_table": "shuffled" if w.shuffle_blocks else
                       ("identity" if paged else "none (contiguous)"), "replicas": world},
            "steps_per_s": 1000.0 / step_ms_max,
            "us_per_step": 1000.0 * step_ms_max,
            "hbm_frac_of_measured": value / world / peak,
            "encode": {"prefill_s": enc_ms / 1e3,
                       "mtok_s": enc_tokens / (enc_ms * 1e-3) / 1e6,
                       "unit": "M token-head-layers/s",
                       "model_tokens_per_s": sum(lens0) / (enc_ms * 1e-3),
                       "gb_s_in_out": (enc_tokens * (2 * 2 * D + rec_bytes)) / (enc_ms * 1e-3) / 1e9},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                         "traffic_source": traffic_src, "kernel": dominant + ", one layer per launch",
                         "avg_launch_ms": launch_ms, "launch_timing": "in-step: step time / layers",
                         "isolated_call_ms": iso_ms, "algorithmic_bytes_per_launch": per_launch_bytes},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if pfa:
            result["prefill_attention"] = pfa
        if cpu:
            result["cpu_baseline"] = cpu
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: the workload's own: 256 decode steps for long_256k, else 20)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="long_256k",
                    choices=["long_256k", "stack_32k", "paged_batch", "layer_d256", "tiny"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-api", default="fused", choices=["fused", "separate"],
                    help="decode step per layer: tq_decode_step (append fused into the decode's first launch) "
                         "or tq_encode_append then tq_decode_attention")
    ap.add_argument("--no-prefill-attention", action="store_true",
                    help="skip the one-layer prefill-attention measurement")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first L layers (profiling case; default: all of the workload's)")
    args = ap.parse_args(argv)
    if args.steps <= 0:
        args.steps = 256 if args.workload == "long_256k" else 20
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
