#!/usr/bin/env python
"""Benchmark of the DropKV score -> select -> compact path on one GB300 per rank.

One step = the whole path (window attention, scoring, pool + protect, bottom-k
selection, compaction) over one layer of the named workload, inputs already
resident in HBM.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--impl reference times the fp64 CPU oracle on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from kv_cache_eviction_dropkv_gb300 import synth  # noqa: E402

METRIC = "DropKV scored tokens/s and ms per layer at n=128K; achieved HBM GB/s vs peak"
UNIT = "tokens/s"
SEL_CHUNK = 16384         # slots per CTA in the selection kernels
CLUSTER_MAX_CHUNKS = 8    # heads of up to 8 chunks are selected by one cluster launch


def kernels_per_step(n_max, select="head"):
    """Kernels one step launches: window attention, split merge, score, then
    either one cluster selection that also pools, or (heads longer than 8
    chunks) pool+protect, clear and 3 radix kernels; then compaction.  The
    layer-wide selection: pool+protect, clear and 5 kernels."""
    if select == "layer":
        return 3 + 1 + 6 + 1
    chunks = -(-n_max // SEL_CHUNK)
    return 3 + (1 if chunks <= CLUSTER_MAX_CHUNKS else 5) + 1
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=synth.HEADLINE, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--score", choices=["dropkv", "snapkv"], default="dropkv",
                    help="score kind: the DropKV perturbation score (default) or the SnapKV baseline")
    ap.add_argument("--select", choices=["head", "layer"], default="head",
                    help="bottom-k per KV head (default) or one pool per sequence over its KV heads (AdaDropKV)")
    ap.add_argument("--prefill", action="store_true",
                    help="the eviction fused into the prompt's causal attention over every query row "
                         "(dropkv_evict_prefill), against that attention followed by dropkv_evict")
    ap.add_argument("--decode", type=int, default=0, metavar="M",
                    help="decode-time re-scoring: evict the workload once, append M decode tokens to the "
                         "compacted cache, and time score -> select -> compact of M rows on that grown cache")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(spec, rank):
    """Each rank scores its own layer: the workload's seed offset by the rank
    (weak scaling, no data exchanged between ranks)."""
    return spec.seed + rank


def reduce_max(x, world):
    """Maximum of a per-rank value over all ranks (the slowest rank sets the
    step time); the identity for one rank."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, step_ms):
    """Whole-job units per second: every rank processed units_per_rank in the
    (max-reduced) step time."""
    return units_per_rank * world / (step_ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def config_of(spec, lengths, score="dropkv", select="head"):
    return {"workload": spec.name, "score": score, "select": select, "B": spec.B, "Hq": spec.Hq, "Hkv": spec.Hkv, "d": spec.d, "n_max": spec.n_max,
            "n_tokens": int(sum(lengths)), "w": spec.w, "pool_kernel": spec.pool_kernel, "protect": spec.protect,
            "budget_pct_kept": spec.budget_pct, "inputs": "bf16",
            "l2": "inputs %s than L2 (K+V %.0f MB); between steps a 256 MB write flushes L2 and a 256 MB read cleans it" % (
                "larger" if kv_bytes(spec) > 129e6 else "smaller", kv_bytes(spec) / 1e6)}


def kv_bytes(spec):
    return 2 * spec.B * spec.Hkv * spec.n_max * spec.d * 2


def workload_bytes(spec, lengths, kept, score="dropkv", select="head"):
    """Algorithmic bytes of one step: each attention pass reads K and V once
    (the SnapKV score reads only K), pass 2 writes a raw score per head-token,
    pooling reads and writes one score, the selection writes the kept indices
    (plus its score re-reads where it has them), and compaction moves the kept
    K and V rows and reads their indices."""
    U_tok = spec.Hkv * int(sum(lengths))                  # head-tokens
    kv = (4 if score == "dropkv" else 2) * spec.d         # K (+ V) bytes per head-token
    p1 = U_tok * kv
    p2 = U_tok * (kv + 4)                                 # + raw score write
    pool = U_tok * 8
    # selection: the cluster kernel selects from the pooled scores it has just
    # made in shared memory (pool's 8 B cover its reads and writes); the
    # multi-kernel path for heads longer than 8 chunks reads the scores 3 times
    sel_passes = 0 if -(-spec.n_max // SEL_CHUNK) <= CLUSTER_MAX_CHUNKS else 3
    if select == "layer":
        sel_passes = 5                                    # three digit histograms, counts, write
    sel = U_tok * 4 * sel_passes + spec.Hkv * int(sum(kept)) * 4
    comp = spec.Hkv * int(sum(kept)) * (4 + 2 * 2 * spec.d * 2)
    return {"window_attention": p1, "score": p2, "pool_protect": pool, "select": sel, "compact": comp,
            "path": p1 + p2 + pool + sel + comp}


def source_hash():
    h = hashlib.sha256()
    for f in ("dropkv_attn.cu", "sm103_ptx.cuh", "dropkv_internal.cuh"):
        with open(os.path.join(ROOT, "kv_cache_eviction_dropkv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [ln.strip().split(",") for ln in self.out.read().splitlines() if ln.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for nm, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def run_reference(args, spec, wl):
    """Reference arm: the fp64 CPU oracle on the host cores, same workload,
    metric and unit.  Each step scores the whole layer with one thread per
    host core (the oracle spreads (sequence, KV head, query head) items over
    them) and counts the layer's tokens."""
    import oracle
    lengths = wl.lengths.numpy()
    nproc = os.cpu_count() or 1

    def step(i):
        oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, spec.pool_kernel, spec.protect, nthreads=nproc,
                        kind=args.score)
        return int(lengths.sum())

    for i in range(args.warmup):
        step(i)
    times, units = [], 0.0
    for i in range(args.steps):
        t0 = time.perf_counter()
        units += step(args.warmup + i)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = units / total
    sample = "per step the whole layer (%d KV heads x %d query heads, %d tokens), fp64, %d threads" % (
        spec.B * spec.Hkv, spec.Hq // spec.Hkv, int(lengths.sum()), nproc)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator; stands in for RULER/LongBench layers)",
            "config": config_of(spec, lengths, args.score),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nproc, "nproc": nproc, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def prefill_flops(spec, lengths):
    """Algorithmic FLOPs of the causal attention over every query row: per
    query head, row i multiplies its query with i + 1 keys (q.k, 2d FLOPs each)
    and sums i + 1 value rows (2d each): 2 d n_b (n_b + 1) per head."""
    return sum(spec.Hq * 2 * spec.d * int(nb) * (int(nb) + 1) for nb in lengths)


def prefill_leg(args, spec, wl, op, dev, stream, flush, clean, world, rank):
    """--prefill: one step = dropkv_evict_prefill (the causal attention over
    every query row of the layer, with the eviction fused in), beside the
    unfused pair (dropkv_prefill_attention, then dropkv_evict over the window
    rows: pass 1 reads K and V once more) and the attention alone.  Query rows
    are seeded N(0, 1) bf16, the workload's window rows at the tail."""
    from kv_cache_eviction_dropkv_gb300 import _binding as B
    rng = np.random.default_rng(spec.seed + 77)
    lengths_np = wl.lengths.numpy()
    q_full = synth.bf16_round(rng.standard_normal((spec.B, spec.Hq, spec.n_max, spec.d)).astype(np.float32))
    for b in range(spec.B):
        nb = int(lengths_np[b])
        q_full[b, :, nb - spec.w:nb] = wl.q[b]
    qwin = torch.stack([q_full[b, :, int(lengths_np[b]) - spec.w:int(lengths_np[b])] for b in range(spec.B)])
    q, qw = q_full.to(dev), qwin.contiguous().to(dev)
    k, v = wl.k.to(dev), wl.v.to(dev)
    lengths, ev = wl.lengths.to(dev), wl.evict_k.to(dev)
    out = torch.empty_like(q)

    def fused():
        op.run_prefill(q, k, v, lengths, ev, out, stream=stream, keep_raw=False)

    def unfused():
        op.prefill_attention(q, k, v, lengths, out, stream=stream)
        op.run(qw, k, v, lengths, ev, stream=stream, keep_raw=False)

    def attention():
        op.prefill_attention(q, k, v, lengths, out, stream=stream)

    def timed(fn, K):
        ts = []
        for i in range(K):
            flush.fill_(float(i))
            clean.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b_) for a, b_ in ts]

    for fn in (fused, unfused, attention):
        for i in range(max(3, args.warmup)):
            fn()
    op.check(stream)
    K = args.steps
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES") else 0)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    t_fused = timed(fused, K)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    t_unfused = timed(unfused, K)
    t_att = timed(attention, K)
    op.check(stream)
    med = lambda xs: float(sorted(xs)[len(xs) // 2])
    step_ms = reduce_max(sum(t_fused) / K, world)
    units = int(lengths_np.sum())
    flops = prefill_flops(spec, lengths_np)
    att_ms = med(t_att)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = {}
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            peaks = json.load(f)
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops / (att_ms / 1e3) / 1e12
    return {"metric": METRIC, "value": job_throughput(units, world, step_ms), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded generator; stands in for RULER/LongBench layers)",
            "config": dict(config_of(spec, lengths_np), mode="prefill-fused"),
            "roofline": {"bound": "tensor", "kernel": "prefill_attention", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": "measured (bf16 burst)" if "bf16_tflops" in peaks else "fallback",
                         "traffic": None, "algorithmic_flops_per_launch": flops},
            "prefill": {"fused_ms": med(t_fused), "unfused_ms": med(t_unfused), "attention_ms": att_ms,
                        "saved_ms": med(t_unfused) - med(t_fused),
                        "note": "fused = dropkv_evict_prefill; unfused = dropkv_prefill_attention then "
                                "dropkv_evict on the window rows (pass 1 reads K and V again); medians"},
            "gpu_launches": 5 * K, "clocks": clocks}


def oracle_decode_workload(wl, m, seed):
    """The decode-time workload of the reference arm: the oracle's prefill
    kept set, gathered on the host, grown by the same m seeded tokens."""
    import oracle
    from kv_cache_eviction_dropkv_gb300.decode import append_decode_tokens
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect,
                          nthreads=os.cpu_count() or 1)
    idx = torch.from_numpy(ref["kept_idx"]).long().clamp(min=0)[..., None].expand(-1, -1, -1, s.d)
    return append_decode_tokens(wl, torch.gather(wl.k, 2, idx), torch.gather(wl.v, 2, idx), m, seed)


def window_rows_probe(spec, wl, dev, stream, m, reps):
    """Upper bound on what an incremental re-score could save: a re-score has
    to stream K and V through both passes for any new window row, so reusing
    the w - m surviving rows' statistics would at most shrink window attention
    to m rows per query head.  Times window attention on the same cache with
    all w rows and with min(m, w) rows."""
    from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B
    out = {}
    lengths = wl.lengths.to(dev)
    k, v = wl.k.to(dev), wl.v.to(dev)
    for rows in sorted({spec.w, min(m, spec.w)}):
        op = DropKV(spec.B, spec.Hq, spec.Hkv, spec.d, spec.n_max, rows, spec.pool_kernel, spec.protect,
                    out_rows=spec.n_max, device=dev)
        q = wl.q[:, :, spec.w - rows:].contiguous().to(dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(reps)]
        for row in evs:
            for e in row:
                e.record(stream)
        for i in range(reps):
            B.dropkv_score_timed(op.shape, q, k, v, lengths, op.pool_kernel, op.protect, op.scores, None,
                                 op.workspace, op.status, evs[i][1:6], stream)
        torch.cuda.synchronize()
        op.check(stream)
        t = sorted(evs[i][1].elapsed_time(evs[i][2]) for i in range(reps))
        t2 = sorted(evs[i][1].elapsed_time(evs[i][5]) for i in range(reps))
        out["w%d" % rows] = {"window_attention_ms": t[reps // 2], "score_call_ms": t2[reps // 2]}
    full, part = out["w%d" % spec.w], out["w%d" % min(m, spec.w)]
    out["max_saving_ms"] = full["window_attention_ms"] - part["window_attention_ms"]
    out["note"] = ("an incremental re-score still reads K and V in both passes (the new rows need their own "
                   "window attention, and every surviving row's p and a change when rows are evicted); at most "
                   "it runs window attention on min(m, w) instead of w rows per query head (medians of %d)" % reps)
    return out


def cpu_baseline(spec, wl, score="dropkv"):
    """The fp64 oracle on the host: the whole layer with one thread per core,
    and a bounded sample on one thread (one query head of one KV head over all
    of its sequence's tokens, 1/Hq of the layer's scoring work, scaled to the
    tokens it represents)."""
    import oracle
    nproc = os.cpu_count() or 1
    units = int(wl.lengths.sum())
    t0 = time.perf_counter()
    oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, spec.pool_kernel, spec.protect, nthreads=nproc,
                    kind=score)
    dt_all = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.run_path(wl.q[:1, :1], wl.k[:1, :1], wl.v[:1, :1], wl.lengths[:1], wl.evict_k[:1], spec.pool_kernel,
                    spec.protect, nthreads=1, kind=score)
    dt_one = time.perf_counter() - t0
    one_units = int(wl.lengths[0]) / spec.Hq
    return {"value": units / dt_all, "unit": UNIT, "cores": nproc, "nproc": nproc, "kind": "oracle",
            "threads": nproc, "seconds": dt_all,
            "one_thread": {"value": one_units / dt_one, "threads": 1, "seconds": dt_one,
                           "sample": "one query head of one KV head (1/%d of the layer)" % spec.Hq},
            "sample": "one full layer (%d KV heads, %d tokens), fp64, %.2f s on %d threads (nproc %d)" % (
                spec.B * spec.Hkv, units, dt_all, nproc, nproc)}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    spec = synth.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        wl = synth.make_workload(args.workload)
        if args.decode:
            wl = oracle_decode_workload(wl, args.decode, spec.seed + 1000)
            spec = wl.spec
        run_reference(args, spec, wl)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, _build
    _build.build_library()

    # each rank scores its own layer (weak scaling, no data-path collective)
    wl = synth.make_workload(args.workload, seed=rank_seed(spec, rank))
    if args.decode:
        from kv_cache_eviction_dropkv_gb300.decode import grow_after_eviction
        wl = grow_after_eviction(wl, args.decode, seed=rank_seed(spec, rank) + 1000, device=dev)
        spec = wl.spec
    lengths_np = wl.lengths.numpy()
    kept_np = wl.kept_len()
    units = int(sum(lengths_np))
    layer = args.select == "layer"
    # the layer-wide selection keeps a data-dependent count per head: room for n_max rows
    op = DropKV(spec.B, spec.Hq, spec.Hkv, spec.d, spec.n_max, spec.w, spec.pool_kernel, spec.protect,
                out_rows=spec.n_max if layer else int(kept_np.max()), device=dev, kind=args.score)
    q, k, v = wl.q.to(dev), wl.k.to(dev), wl.v.to(dev)
    lengths, ev = wl.lengths.to(dev), wl.evict_k.to(dev)
    if layer:
        ev = ev * spec.Hkv            # the same total budget as per-head selection
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    if args.prefill:
        line = prefill_leg(args, spec, wl, op, dev, stream, flush, clean, world, rank)
        if rank == 0:
            print(json.dumps(line))
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    def flush_l2(i):
        # write a buffer larger than L2 (evicts the previous step's data), then
        # read another one so that the dirty lines are written back here and
        # not inside the next step's timed kernels
        flush.fill_(float(i))
        return clean.sum()

    def step(events=None):
        if events is None:
            if layer:
                op.run_layer(q, k, v, lengths, ev, stream=stream, keep_raw=False)
            else:
                op.run(q, k, v, lengths, ev, stream=stream, keep_raw=False)
        else:
            B.dropkv_score_timed(op.shape, q, k, v, lengths, op.pool_kernel, op.protect, op.scores, None,
                                 op.workspace, op.status, events[1:6], stream, kind=args.score)
            if layer:
                op.select_layer(lengths, ev, stream)
            else:
                op.select(lengths, ev, stream)
            events[6].record(stream)
            if layer:
                op.compact_heads(k, v, stream)
            else:
                op.compact(k, v, stream)

    for w in range(max(3, args.warmup)):
        flush_l2(w)
        step()
    op.check(stream)

    K = args.steps
    # timed steps: one event pair per step (events between the kernels of a
    # step would serialise their programmatic dependent launches)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in ev0 + ev1:          # torch creates the CUDA event on its first record()
        e.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local])
                           if os.environ.get("CUDA_VISIBLE_DEVICES") else local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush_l2(i)
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    op.check(stream)
    t_step = [ev0[i].elapsed_time(ev1[i]) for i in range(K)]

    # per-kernel phases, in separate steps with events at the phase boundaries
    KP = max(3, min(K, 50))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(KP)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(KP):
        flush_l2(i)
        evs[i][0].record(stream)
        step(evs[i])
        evs[i][7].record(stream)
    torch.cuda.synchronize()
    op.check(stream)

    def ms(a, b):
        return [evs[i][a].elapsed_time(evs[i][b]) for i in range(KP)]

    # warm L2: the same steps back to back without the flush (at n = 128K the
    # 537 MB of K + V is four times the L2, so the two numbers stay close)
    KW = max(3, min(K, 50))
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for i in range(KW):
        step()
    w1.record(stream)
    torch.cuda.synchronize()
    op.check(stream)
    warm_ms = reduce_max(w0.elapsed_time(w1) / KW, world)

    phases = {"window_attention": ms(1, 2), "split_merge": ms(2, 3), "score": ms(3, 4), "pool_protect": ms(4, 5),
              "select": ms(5, 6), "compact": ms(6, 7)}
    step_ms = reduce_max(sum(t_step) / K, world)
    value = job_throughput(units, world, step_ms)

    nbytes = workload_bytes(spec, lengths_np, kept_np, args.score, args.select)
    peak, peak_kind = measured_peaks()
    phase_ms = {kname: sum(v_) / KP for kname, v_ in phases.items()}
    dom = max(("window_attention", "score"), key=lambda kk: phase_ms[kk])
    achieved = nbytes[dom] / (phase_ms[dom] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": peak_kind,
                "traffic": recorded_traffic(dom, spec.name if args.score == "dropkv" else spec.name + ":" + args.score),
                "algorithmic_bytes_per_launch": nbytes[dom]}
    path_gbs = nbytes["path"] / (step_ms / 1e3) / 1e9

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": step_ms, "ms_per_step_median": reduce_max(float(sorted(t_step)[K // 2]), world),
            "head_tokens_per_s": value * spec.Hkv, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded generator; stands in for RULER/LongBench layers)",
            "config": config_of(spec, lengths_np, args.score, args.select),
            "roofline": roofline,
            "path_roofline": {"achieved": path_gbs, "peak": peak, "unit": "GB/s", "frac": path_gbs / peak,
                              "algorithmic_bytes_per_step": nbytes["path"]},
            "phases_ms": phase_ms, "phases_note": "per-kernel times from %d separate steps with events at the phase boundaries, run as the three separate calls (pooling in its own kernel; the timed step pools inside the selection)" % KP,
            "warm": {"value": job_throughput(units, world, warm_ms), "ms_per_step": warm_ms, "steps": KW,
                     "note": "no L2 flush between steps"},
            "wall_s_timed": wall, "gpu_launches": kernels_per_step(spec.n_max, args.select) * K,
            "clocks": clocks}

    if args.decode:
        line["decode"] = {"m": args.decode, "cache_rows": int(spec.n_max),
                          "reading": "prefill eviction, then m decode tokens appended to the compacted cache, "
                                     "window moved to the newest w positions, m rows evicted again",
                          "incremental": window_rows_probe(spec, wl, dev, stream, args.decode, 20)}
    if not args.no_e2e:
        line["e2e"] = e2e_leg(op, wl, dev, stream, args, world)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, wl, args.score)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def e2e_leg(op, wl, dev, stream, args, world):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads the kept set and the
    compacted K/V back.  As a serving loop would, the steps are pipelined over
    two buffer sets: step s+1's upload (copy stream) and step s-1's download
    (a third stream) overlap step s's scoring; every step's copies lie inside
    the timed region."""
    from kv_cache_eviction_dropkv_gb300 import DropKV
    Bn, Hq, Hkv, d, n_max, w = op.shape.astuple()
    ops = [op, DropKV(Bn, Hq, Hkv, d, n_max, w, op.pool_kernel, op.protect, out_rows=op.out_rows, device=dev,
                      kind=op.kind)]
    hq, hk, hv = wl.q.pin_memory(), wl.k.pin_memory(), wl.v.pin_memory()
    hl, he = wl.lengths.pin_memory(), wl.evict_k.pin_memory()
    if args.select == "layer":
        he = (wl.evict_k * Hkv).pin_memory()
    hin = (hq, hk, hv, hl, he)
    dins = [[torch.empty_like(t, device=dev) for t in hin] for _ in range(2)]
    layer = args.select == "layer"
    outs = [[o.kept_len_heads if layer else o.kept_len, o.kept_idx, o.k_out, o.v_out] for o in ops]
    houts = [[torch.empty_like(t, device="cpu").pin_memory() for t in outs[0]] for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in hin)
    bo = sum(t.numel() * t.element_size() for t in houts[0])
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    for e in ev_up + ev_run + ev_down:
        e.record(stream)

    def one(i):
        bsel = i % 2
        o, dq, dk, dv, dl, de = ops[bsel], *dins[bsel]
        s_up.wait_event(ev_run[bsel])             # scoring of step i-2 has read this input set
        with torch.cuda.stream(s_up):
            for src, dst in zip(hin, dins[bsel]):
                dst.copy_(src, non_blocking=True)
            ev_up[bsel].record(s_up)
        stream.wait_event(ev_up[bsel])
        stream.wait_event(ev_down[bsel])          # step i-2's outputs have been read back
        if layer:
            o.run_layer(dq, dk, dv, dl, de, stream=stream, keep_raw=False)
        else:
            o.run(dq, dk, dv, dl, de, stream=stream, keep_raw=False)
        ev_run[bsel].record(stream)
        s_down.wait_event(ev_run[bsel])
        with torch.cuda.stream(s_down):
            for src, dst in zip(outs[bsel], houts[bsel]):
                dst.copy_(src, non_blocking=True)
            ev_down[bsel].record(s_down)

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    K = max(2, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0.record(s_up)
    for i in range(K):
        one(i)
    e1.record(s_down)
    torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1) / K, world)
    for o in ops:
        o.check(stream)
    units = int(wl.lengths.sum())
    return {"value": job_throughput(units, world, ms), "unit": UNIT, "ms_per_step": ms, "steps": K,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "pipelined": "two buffer sets: upload of step s+1 and download of step s-1 overlap the scoring of step s"}


if __name__ == "__main__":
    main()
