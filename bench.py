#!/usr/bin/env python3
"""Benchmark of the Kamera relocate + patch + paged-scatter operator on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--no-sweep]

A step is one call of the operator over the whole workload (all chunks, all
layers, all heads): descriptor decode, RoPE phase, canonical read, rotation,
rank-m patch, bf16 rounding and paged scatter, in one kernel launch.  The
headline workload is the Qwen2.5-VL-7B shaped recall batch (28 layers, 4 KV
heads, head_dim 128, 8 chunks of 1296 tokens, rank-32 patches on K and V).
Its inputs (1.35 GB moved per step) are larger than the 129 MB L2, so no
flush is needed between timed steps; smaller sweep workloads flush L2 between
launches instead.

The metric is algorithmic bytes per second (canonical rows read + patch
factors read + rows written + int64 slot map) and tokens reinstated per
second; ``roofline.frac`` is that bandwidth over the measured HBM copy peak.

``--impl reference`` times the fp64 CPU oracle (the correctness reference of
this project) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "relocated KV GB/s (read+write) & tokens reinstated/s; % of GB300 HBM peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ utils
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s, the burst figure: a kernel timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest `value` over all ranks (the slowest rank sets the job time)."""
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: int, world: int, seconds_per_step: float) -> float:
    """Whole-job GB/s: every rank processes its own copy of the workload (weak scaling)."""
    return bytes_per_rank * world / seconds_per_step / 1e9


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

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
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
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
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def flush_l2(buf: torch.Tensor):
    buf.add_(1)


# --------------------------------------------------------------- workload
def make_call(K, wl, chunks_dev, err):
    """The operator call of one step, through the C ABI binding."""
    rope = K.Rope(wl.base, wl.rot_dim, 0 if wl.kind in ("mla", "mla_ingest") else wl.rot_offset, wl.pairing)
    n = len(wl.chunks)
    ml, mr = wl.max_len, max((c.rank for c in wl.chunks), default=0)
    if wl.kind == "gqa":
        return lambda: K.kamera_relocate_patch(wl.pool_k, wl.pool_v, wl.store_k, wl.store_v, rope, chunks_dev,
                                               n, ml, mr, err)
    if wl.kind == "mla":
        return lambda: K.kamera_mla_relocate_patch(wl.pool_k, wl.store_k, wl.kv_lora, rope, chunks_dev, n, ml,
                                                   mr, err)
    if wl.kind == "ingest":
        return lambda: K.kamera_ingest_canonical(wl.pool_k, wl.pool_v, wl.store_k, wl.store_v, rope, chunks_dev,
                                                 n, ml, err)
    if wl.kind == "mla_ingest":
        return lambda: K.kamera_mla_ingest_canonical(wl.pool_k, wl.store_k, wl.kv_lora, rope, chunks_dev, n, ml,
                                                     err)
    return lambda: K.kamera_slide_inplace(wl.pool_k, rope, chunks_dev, n, ml, err)


# workloads bench.py can time as its headline: the configured ones and the tiny
# chunk replicated 4096 times in one call (the bandwidth form of the tiny case)
BENCH_WORKLOADS = dict(W.CONFIGS, tiny_gqa_x4096=lambda: W.tiny_gqa_x(4096))


def config_block(spec, name):
    blk = {"workload": name, "layers": spec.L, "chunks": len(spec.lens), "tokens": W.tokens(spec),
           "rank": spec.m, "page_size": spec.page, "algorithmic_bytes": W.algorithmic_bytes(spec)}
    if isinstance(spec, W.MlaSpec):
        blk.update({"attention": "MLA" if spec.kind == "mla" else "MLA canonical ingest (pool -> store)",
                    "kv_lora": spec.kv_lora, "rope_dim": spec.rope})
    else:
        blk.update({"attention": {"gqa": "GQA/MHA", "slide": "slide (rotate-only, in place)",
                                  "ingest": "GQA/MHA canonical ingest (pool -> store)"}[spec.kind],
                    "kv_heads": spec.H, "head_dim": spec.d})
    return blk


def time_launches(call, steps, flush_buf=None):
    """Per-launch device times (ms) with CUDA events on the launching stream."""
    s = torch.cuda.current_stream()
    evs = []
    for _ in range(steps):
        if flush_buf is not None:
            flush_l2(flush_buf)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        call()
        b.record(s)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def kernel_of(spec) -> str:
    """The kernel a workload's call spends its time in: the relocation calls of the
    configured workloads all carry patches, so they take the tensor-core kernel,
    except calls of short chunks (<= 128 tokens) with ranks <= 8, which the
    library sends to the CUDA-core kernel."""
    if spec.kind in ("gqa", "mla") and spec.m <= 8 and max(spec.lens) <= 128:
        return "rows_simt_kernel"
    return {"slide": "slide_kernel", "ingest": "ingest_kernel", "mla_ingest": "ingest_kernel"}.get(
        spec.kind, "relocate_patch_umma_kernel")


def sweep(K, dev, peak, skip, only=None):
    """Every configured workload, timed per launch (median) with L2 flushes."""
    out = {}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    specs = [(n, f()) for n, f in W.CONFIGS.items()] + [("tiny_gqa_x4096", W.tiny_gqa_x(4096))]
    for name, spec in specs:
        if name in skip or (only is not None and name not in only):
            continue
        try:
            wl = W.make(spec, dev)
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            ch = K.pack_chunks(wl.chunks, device=dev)
            call = make_call(K, wl, ch, err)
            for _ in range(3):
                call()
            ts = time_launches(call, 10 if W.algorithmic_bytes(spec) > 1e9 else 20, flush)
            t = float(np.median(ts)) * 1e-3
            b = W.algorithmic_bytes(spec)
            out[name] = {"gbs": b / t / 1e9, "tokens_per_s": W.tokens(spec) / t, "ms": t * 1e3,
                         "frac_of_hbm_peak": b / t / 1e9 / peak, "bytes": b, "l2": "flushed between launches",
                         "kernel": kernel_of(spec), "traffic": traffic_record(kernel_of(spec), name),
                         "device_err": int(err.item())}
            del wl, ch, call
            torch.cuda.empty_cache()
        except Exception as e:  # report, keep the headline
            out[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
    for name, f in W.FORMATION.items():
        if name in skip or (only is not None and name not in only):
            continue
        try:
            out[name] = formation_entry(K, f(), dev, peak, flush)
        except Exception as e:  # report, keep the headline
            out[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
    for name, f in W.ATTENTION.items():
        if name in skip or (only is not None and name not in only):
            continue
        try:
            spec = f()
            entry = {"mla_attend": mla_attend_entry, "prefill": prefill_entry}.get(spec.kind, attend_entry)
            out[name] = entry(K, spec, dev, peak, flush)
        except Exception as e:  # report, keep the headline
            out[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return out


def attend_entry(K, spec, dev, peak, flush):
    """Decode attention over reused chunks (one query token per sequence and
    query head), timed per launch with L2 flushes."""
    a = W.make_attend(spec, dev)
    chunks = K.pack_chunks(a.chunks, device=dev)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=dev)
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing)
    ml, mr = max(c.length for c in a.chunks), max(c.rank for c in a.chunks)
    out = torch.empty_like(a.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        K.kamera_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, len(a.chunks), ml, mr,
                               layer=spec.layer, out=out, err=err)

    for _ in range(3):
        call()
    t = float(np.median(time_launches(call, 10, flush))) * 1e-3
    b = W.attend_bytes(spec)
    tok = sum(c.length for c in a.chunks)
    return {"ms": t * 1e3, "gbs": b / t / 1e9, "frac_of_hbm_peak": b / t / 1e9 / peak, "bytes": b,
            "tokens_attended_per_s": tok / t, "sequences": len(spec.seqs), "rank": spec.m,
            "l2": "flushed between launches", "kernel": "attend_kernel",
            "traffic": traffic_record("attend_kernel", spec.name), "device_err": int(err.item())}


def prefill_entry(K, spec, dev, peak, flush):
    """Prefill attention over reused chunks (T new query tokens per sequence),
    timed per launch with L2 flushes; a dense contraction on the tensor cores,
    so its roofline is the bf16 tensor peak (the folded form's flops)."""
    a = W.make_attend(spec, dev)
    chunks = K.pack_chunks(a.chunks, device=dev)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=dev)
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing)
    ml, mr = max(c.length for c in a.chunks), max(c.rank for c in a.chunks)
    out = torch.empty_like(a.q)
    lse = torch.empty(a.q.shape[:3], dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        K.kamera_prefill_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, len(a.chunks), ml, mr,
                                       layer=spec.layer, out=out, lse=lse, err=err)

    for _ in range(3):
        call()
    t = float(np.median(time_launches(call, 10, flush))) * 1e-3
    fl = W.prefill_flops(spec)
    tf_peak, tf_src = measured_bf16_peak()
    tok = sum(c.length for c in a.chunks)
    return {"ms": t * 1e3, "tflops": fl / t / 1e12, "frac_of_bf16_peak": fl / t / 1e12 / tf_peak,
            "bf16_peak_tflops": tf_peak, "bf16_peak_source": tf_src, "flops": fl,
            "query_tokens_per_s": len(spec.seqs) * spec.T / t, "tokens_attended_per_s": tok * spec.T / t,
            "sequences": len(spec.seqs), "query_tokens": spec.T, "rank": spec.m,
            "l2": "flushed between launches", "kernel": "prefill_kernel",
            "traffic": traffic_record("prefill_kernel", spec.name), "device_err": int(err.item())}


def mla_attend_entry(K, spec, dev, peak, flush):
    """MLA decode attention over reused chunks (absorbed form, one query token per
    sequence and query head), timed per launch with L2 flushes."""
    a = W.make_mla_attend(spec, dev)
    chunks = K.pack_chunks(a.chunks, device=dev)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=dev)
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing)
    ml, mr = max(c.length for c in a.chunks), max(c.rank for c in a.chunks)
    out = torch.empty(a.q.shape[0], spec.Hq, spec.kv_lora, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        K.kamera_mla_attend_reused(a.store, spec.kv_lora, a.q, rope, chunks, seq, len(a.chunks), ml, mr,
                                   layer=spec.layer, out=out, err=err)

    for _ in range(3):
        call()
    t = float(np.median(time_launches(call, 10, flush))) * 1e-3
    b = W.mla_attend_bytes(spec)
    tok = sum(c.length for c in a.chunks)
    return {"ms": t * 1e3, "gbs": b / t / 1e9, "frac_of_hbm_peak": b / t / 1e9 / peak, "bytes": b,
            "tokens_attended_per_s": tok / t, "sequences": len(spec.seqs), "rank": spec.m,
            "l2": "flushed between launches", "kernel": "mla_attend_kernel",
            "traffic": traffic_record("mla_attend_kernel", spec.name), "device_err": int(err.item())}


def formation_entry(K, spec, dev, peak, flush):
    """Patch formation of one chunk's deficits (all (kv, layer, head) blocks in
    one call), timed per launch with L2 flushes."""
    x = W.make_deficit(spec, dev)
    xb = x.reshape(spec.kv * spec.L, spec.length, spec.H, spec.d).permute(0, 2, 1, 3)
    u = torch.empty(spec.kv * spec.L, spec.H, spec.length, spec.m, dtype=torch.bfloat16, device=dev)
    v = torch.empty(spec.kv * spec.L, spec.H, spec.d, spec.m, dtype=torch.bfloat16, device=dev)
    sig = torch.empty(spec.kv * spec.L, spec.H, spec.m, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        K.kamera_form_patch(xb, spec.m, u=u, v=v, sigma=sig, err=err)

    for _ in range(3):
        call()
    t = float(np.median(time_launches(call, 10, flush))) * 1e-3
    b, fl = W.deficit_bytes(spec), W.deficit_flops(spec)
    return {"ms": t * 1e3, "blocks": W.deficit_blocks(spec), "blocks_per_s": W.deficit_blocks(spec) / t,
            "tokens_per_s": spec.length / t, "gbs": b / t / 1e9, "frac_of_hbm_peak": b / t / 1e9 / peak,
            "bytes": b, "contraction_tflops": fl / t / 1e12, "rank": spec.m,
            "l2": "flushed between launches", "kernel": "patch_form_kernel",
            "traffic": traffic_record("patch_form_kernel", spec.name), "device_err": int(err.item())}


def _replica(wl):
    """A second device copy of the workload's tensors (same shapes, fresh memory)."""
    import dataclasses
    cl = lambda t: None if t is None else t.clone()
    chunks = [dataclasses.replace(c, slots=c.slots.clone(), patches=[p.clone() for p in c.patches])
              for c in wl.chunks]
    return dataclasses.replace(wl, chunks=chunks, store_k=cl(wl.store_k), store_v=cl(wl.store_v),
                               pool_k=cl(wl.pool_k), pool_v=cl(wl.pool_v))


def e2e_measure(K, wl, steps, warmup):
    """Same metric through the C ABI with host buffers: every step copies its
    inputs host->device from pinned memory, runs the operator and reads the
    pool back device->host, all inside the timed region.  Steps alternate
    between two device buffer sets on two streams, so one step's read-back
    overlaps the next step's upload (the link carries both directions at
    once); workloads above 16 GB on the device run one set, serially."""
    ingest = wl.kind in ("ingest", "mla_ingest")

    def inputs(w):
        t = []
        for c in w.chunks:
            t += list(c.patches) + [c.slots]
        if ingest:              # the live cache is the input, the canonical store the result
            t += [x for x in (w.pool_k, w.pool_v) if x is not None]
            return t
        t += [x for x in (w.store_k, w.store_v) if x is not None]
        if w.kind == "slide":   # in place: the pool is the step's input too
            t.append(w.pool_k)
        return t

    def outputs(w):
        if ingest:
            return [x for x in (w.store_k, w.store_v) if x is not None]
        return [x for x in (w.pool_k, w.pool_v) if x is not None]

    dev_bytes = sum(t.numel() * t.element_size() for t in inputs(wl) + outputs(wl))
    sets = [wl, _replica(wl)] if dev_bytes <= (16 << 30) else [wl]
    host_in = [t.cpu().pin_memory() for t in inputs(wl)]
    chunks_dev = [K.pack_chunks(w.chunks, device=wl.pool_k.device) for w in sets]
    chunks_host = [c.cpu().pin_memory() for c in chunks_dev]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outputs(w)] for w in sets]
    errs = [torch.zeros(1, dtype=torch.int32, device=wl.pool_k.device) for _ in sets]
    calls = [make_call(K, w, c, e) for w, c, e in zip(sets, chunks_dev, errs)]
    streams = [torch.cuda.Stream() for _ in sets]
    h2d = sum(t.numel() * t.element_size() for t in host_in) + chunks_host[0].numel()
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])

    def step(i):
        k = i % len(sets)
        with torch.cuda.stream(streams[k]):
            for d, h in zip(inputs(sets[k]), host_in):
                d.copy_(h, non_blocking=True)
            chunks_dev[k].copy_(chunks_host[k], non_blocking=True)
            calls[k]()
            for h, d in zip(host_out[k], outputs(sets[k])):
                h.copy_(d, non_blocking=True)

    main = torch.cuda.current_stream()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(main)
    for st in streams:
        st.wait_stream(main)
    for i in range(steps):
        step(i)
    for st in streams:
        main.wait_stream(st)
    b.record(main)
    torch.cuda.synchronize()
    t = a.elapsed_time(b) / 1e3 / steps
    del sets
    return {"value": W.algorithmic_bytes(wl.spec) / t / 1e9, "unit": "GB/s", "ms_per_step": t * 1e3,
            "tokens_per_s": wl.tokens / t, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "buffer_sets": len(streams)}


KERNEL_UNITS = {   # the translation unit each timed kernel is compiled from
    "relocate_patch_umma_kernel": "kamera_umma.cu",
    "rows_simt_kernel": "kamera_simt.cu",
    "slide_kernel": "kamera_slide.cu",
    "ingest_kernel": "kamera_ingest.cu",
    "patch_form_kernel": "kamera_patchform.cu",
    "attend_kernel": "kamera_attend.cu",
    "mla_attend_kernel": "kamera_attend_mla.cu",
    "prefill_kernel": "kamera_prefill.cu",
}


def kernel_sources(B, kernel: str):
    """The files a kernel is built from: its translation unit, the library's
    internal headers and the C ABI header."""
    import glob
    return sorted([os.path.join(B.CSRC, KERNEL_UNITS[kernel])] + glob.glob(os.path.join(B.CSRC, "*.cuh")) +
                  glob.glob(os.path.join(B.CSRC, "*.h")) + [os.path.join(B.INCLUDE, "kamera.h")])


def source_digest(kernel: str) -> str:
    import hashlib
    from position_invariant_kv_chunk_gb300 import build as B
    h = hashlib.sha256()
    for src in kernel_sources(B, kernel):
        h.update(open(src, "rb").read())
    return h.hexdigest()[:16]


def traffic_record(kernel: str, workload: str):
    """ncu DRAM bytes (read + write) per launch of `kernel` on `workload`, if the
    committed record (profiles/dram_traffic.txt: kernel, workload, source hash,
    bytes, ...) was taken on the kernel's current sources (matching hash)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(kernel)
    for ln in open(path):
        f = ln.split()
        if len(f) >= 4 and f[0] == kernel and f[1] == workload and f[2] == digest:
            return float(f[3])
    return None


# ------------------------------------------------------------- CPU oracle
def oracle_sample(spec, target_s=8.0, max_layers=None):
    """Time the fp64 oracle on a bounded sample of `spec` (first chunks, fewer
    layers), growing the sample until it takes about target_s seconds."""
    import oracle as O
    from tests.harness import snapshot, run_oracle
    orc = O.default()
    L = 1
    nchunks = 1
    while True:
        lens = spec.lens[:nchunks]
        sub = W.scaled(spec, L=L, lens=lens, name=spec.name)
        wl = W.make(sub, "cpu")
        h = snapshot(wl)
        t0 = time.perf_counter()
        run_oracle(wl, h, orc)
        dt = time.perf_counter() - t0
        if dt >= target_s or (nchunks >= len(spec.lens) and L >= (max_layers or spec.L)):
            break
        grow = max(1.5, min(8.0, target_s / max(dt, 1e-3)))
        if nchunks < len(spec.lens):
            nchunks = min(len(spec.lens), int(np.ceil(nchunks * grow)))
        else:
            L = min(max_layers or spec.L, int(np.ceil(L * grow)))
    b = W.algorithmic_bytes(sub)
    return {"value": b / dt / 1e9, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{sub.L} of {spec.L} layers x {len(lens)} of {len(spec.lens)} chunks "
                      f"({W.tokens(sub)} tokens, {b} algorithmic bytes) in {dt:.2f} s",
            "tokens_per_s": W.tokens(sub) / dt, "seconds": dt, "bytes": b}


# ---------------------------------------------------------------- arms
def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    spec = BENCH_WORKLOADS[args.config]()
    for _ in range(args.warmup):
        oracle_sample(spec, target_s=1.0)
    vals = []
    meta = None
    for _ in range(args.steps):
        r = oracle_sample(spec, target_s=args.ref_seconds)
        vals.append(r["value"])
        meta = r
    v = float(np.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": meta["seconds"] * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_block(spec, args.config),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": meta["cores"], "kind": "oracle",
                             "sample": meta["sample"]},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def ours_arm(args):
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    import position_invariant_kv_chunk_gb300 as K
    K.load_library()
    peak, peak_src = measured_peaks()

    spec = BENCH_WORKLOADS[args.config]()
    if args.layers:
        spec = W.scaled(spec, L=args.layers, name=spec.name)
    wl = W.make(spec, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    chunks_dev = K.pack_chunks(wl.chunks, device=dev)
    call = make_call(K, wl, chunks_dev, err)
    big = W.algorithmic_bytes(spec) > 4 * L2_BYTES
    flush = None if big else torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    for _ in range(args.warmup):
        if flush is not None:
            flush_l2(flush)
        call()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    s = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        evs[0].record(s)
        for i in range(args.steps):
            if flush is not None:
                flush_l2(flush)
            call()
            evs[i + 1].record(s)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    total_ms = evs[0].elapsed_time(evs[-1])
    if flush is not None:  # kernel-only durations without the flush
        launch_ms = time_launches(call, args.steps, flush)
    else:
        launch_ms = step_ms
    t_max = max_over_ranks(total_ms, pg, dev)
    ms_per_step = t_max / args.steps
    bytes_step = W.algorithmic_bytes(spec)
    value = job_throughput(bytes_step, world, ms_per_step * 1e-3)
    launch_avg = float(np.mean(launch_ms))
    achieved = bytes_step / (launch_avg * 1e-3) / 1e9
    dev_err = int(err.item())

    if rank != 0:
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return 0

    kernel_name = kernel_of(spec)
    e2e = e2e_measure(K, wl, max(2, min(args.steps, 10)), 1)
    e2e["value"] *= world
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes of the named workload)",
        "config": {**config_block(spec, args.config),
                   "tokens_reinstated_per_s": W.tokens(spec) * world / (ms_per_step * 1e-3),
                   "pct_of_hbm_peak": 100.0 * value / world / peak,
                   "l2": "inputs larger than L2 (no flush)" if big else "L2 flushed between steps",
                   "device_err": dev_err},
        "clocks": clk.summary(),
        "e2e": e2e,
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic_record(kernel_name, args.config),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s", "launch_ms": launch_avg,
                     "bytes_per_launch": bytes_step},
    }
    if world == 1 and not args.no_cpu_baseline:
        cb = oracle_sample(spec, target_s=args.ref_seconds)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if world == 1 and not args.no_sweep:
        del wl, chunks_dev, call
        torch.cuda.empty_cache()
        line["per_config"] = sweep(K, dev, peak, skip={args.config} if args.skip_headline_in_sweep else set(),
                                   only=set(args.sweep_only.split(",")) if args.sweep_only else None)
    print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", choices=sorted(BENCH_WORKLOADS), default="qwen_recall")
    ap.add_argument("--no-sweep", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-headline-in-sweep", action="store_true")
    ap.add_argument("--sweep-only", default="", help="comma-separated workloads the sweep is limited to")
    ap.add_argument("--ref-seconds", type=float, default=8.0, help="oracle seconds per sample")
    ap.add_argument("--layers", type=int, default=0,
                    help="run the workload with this many layers (a smaller case for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return reference_arm(args)
    return ours_arm(args)


if __name__ == "__main__":
    sys.exit(main())
