"""Benchmark of the compressed-KV hot path on one GB300 (or N, one process each).

One step = one autoregressive chunk step of a LongCat-like attention layer
(16 KV heads, head_dim 128, chunks of 3 latent frames of 30x52 = 4680
tokens): compress the newest chunk's K and V into the cache (k-means with
C=256 and 8 Lloyd iterations, INT2 residual, group 64) and run attention of
that chunk's 4680 queries over the whole compressed cache of 8 chunks
(37,440 tokens), reading codes directly.  Synthetic seeded data shaped like
the workload; inputs resident in HBM at the start of the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  The reference arm times the CPU oracle on
the host cores on a bounded sample of the same step.
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
sys.path.insert(0, ROOT)

METRIC = "KV compress GB/s and fused INT2 attention tok/s, % of GB300 HBM roofline"
WORKLOAD = "longcat"
UNIT = "tok/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes (read + write) of one k_attention_ws launch of the bench
# workload, from an ncu capture of `dram__bytes_read.sum,dram__bytes_write.sum`
# on the same command, keyed by the SHA-256 of the kernel's code (comments
# stripped) so that a changed kernel reports null until re-measured.
ATTN_SOURCES = ("attention_ws.cuh", "attention_ws.cu", "umma.cuh", "common.cuh")
ATTN_TRAFFIC = {
    "7c1747e6d35b97ea03205edafaf6f72f8da0695c97a526e7fe74b55fe0a24d75": 80429056 + 3645440,
}


def _attn_source_hash():
    """SHA-256 of the attention kernel's sources with comments and blank
    lines removed, so that only a change of code invalidates the recorded
    traffic."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        with open(os.path.join(ROOT, "video_diffusion_kv_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        code = "\n".join(line.rstrip() for line in src.split("\n") if line.strip())
        h.update(code.encode())
    return h.hexdigest()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


def _workload(cache_chunks=None):
    import dataclasses

    from video_diffusion_kv_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    if cache_chunks:
        w = dataclasses.replace(w, n_chunks=cache_chunks)
    return w


def _config(w, extra=None):
    cfg = {
        "workload": ("longcat-like layer: %d KV heads, d=%d, cache of %d chunks x %d tokens (%d), "
                     "C=%d, INT%d group %d, %d Lloyd iters; step = compress K+V of the newest chunk "
                     "+ attention of its %d queries over the cache" %
                     (w.H, w.d, w.n_chunks, w.N, w.tokens, w.C, w.bits, w.group, w.iters, w.Nq)),
        "tokens_per_chunk": w.N, "cache_tokens": w.tokens, "heads": w.H, "head_dim": w.d,
        "clusters": w.C, "bits": w.bits, "group": w.group, "lloyd_iters": w.iters, "stages": w.L,
    }
    if extra:
        cfg.update(extra)
    return cfg


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines, self.first = index, None, [], 0

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi takes a while to start: wait (up to 3 s) for its first
            # sample so that the samples fall inside the timed region
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)
            self.first = len(self.lines)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # samples taken from the start of the timed region on (the last one
        # read before it started, if none fell inside)
        for ln in self.lines[self.first:] or self.lines[-1:]:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed

def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(x, ws, device=None):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ CPU oracle timing

def oracle_step_sample(w, seed=0, heads=None, q_rows=1):
    """Time the oracle on a bounded sample of one step: compress the newest
    chunk's K and V for `heads` heads (one thread per head) and attention of
    `q_rows` query rows per head over the full cache.  Returns (seconds
    scaled to the whole step, threads used, description)."""
    import numpy as np

    import oracle
    from video_diffusion_kv_gb300 import synth
    oracle.build()
    cores = os.cpu_count() or 1
    hs = heads or max(1, min(w.H, cores))
    last = w.n_chunks - 1
    k = synth.chunk_kv(w, seed, last, synth.KIND_K)[:, :hs]
    v = synth.chunk_kv(w, seed, last, synth.KIND_V)[:, :hs]
    t0 = time.perf_counter()
    ko = oracle.compress_chunk(k, w.C, w.L, w.bits, w.group, w.iters, seed=seed, chunk=last, nthreads=hs)
    vo = oracle.compress_chunk(v, w.C, w.L, w.bits, w.group, w.iters, seed=seed, chunk=last, nthreads=hs)
    t_comp = time.perf_counter() - t0
    # attention over a cache of n_chunks copies-in-shape of the reconstruction
    kh = np.concatenate([ko["xhat"]] * w.n_chunks, 0)
    vh = np.concatenate([vo["xhat"]] * w.n_chunks, 0)
    q = synth.queries(w, seed, last)[:q_rows, :hs]
    t0 = time.perf_counter()
    oracle.attention(q, kh, vh, nthreads=min(cores, hs * q_rows))
    t_attn = time.perf_counter() - t0
    rounds_full = -(-w.H // min(cores, w.H))
    rounds_sample = -(-hs // min(cores, hs))
    scale_heads = rounds_full / rounds_sample
    attn_rounds_full = -(-(w.H * w.Nq) // cores)
    attn_rounds_sample = -(-(hs * q_rows) // min(cores, hs * q_rows))
    t_full = t_comp * scale_heads + t_attn * attn_rounds_full / attn_rounds_sample
    desc = ("oracle compress of the newest chunk's K and V for %d of %d heads (%d threads) + fp64 "
            "attention of %d query row(s) x %d heads over %d cached tokens; scaled to the full step "
            "(%d heads, %d queries) by rounds of %d-thread parallel work" %
            (hs, w.H, hs, q_rows, hs, kh.shape[0], w.H, w.Nq, cores))
    return t_full, min(cores, max(hs, hs * q_rows)), desc, t_comp + t_attn


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    w = _workload()
    for _ in range(args.warmup):
        oracle_step_sample(w, seed=1)
    times, walls, desc, thr = [], [], "", 1
    for s in range(args.steps):
        t_full, thr, desc, wall = oracle_step_sample(w, seed=2 + s)
        times.append(t_full)
        walls.append(wall)
    ms = 1e3 * statistics.mean(times)
    value = w.Nq / (ms / 1e3)
    # n_gpus is the launch's N (the oracle itself runs on rank 0's host cores)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, {"parallelism": "host threads"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "sample_wall_s_per_step": statistics.mean(walls)}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ own arm

def launches_per_compress(p):
    """Kernels one qvg_compress_chunk call launches (see csrc/api.cu): per
    stage the residual quantiser, and with centroids the row norms, the
    init, iters x (assign, update) and the final assignment; then the chunk
    table."""
    per_stage = 1  # residual quantise (+ pack, stage residual, PSAC)
    if p.C > 0:
        per_stage += 1 + 1 + 2 * p.iters + 1
    return per_stage * p.L + 1


def kernel_extras(qvg, p, w, kc, vc, q, k_raw, flush, dev, last, slots_per_chunk, reps=5):
    """Separately timed kernels on the same cache (outside the step): the
    decompress of the newest chunk (fp32 and bf16 output) and of the whole
    cache (fp32), a decode-like
    attention point (16 queries over the whole cache), each with its
    algorithmic bytes and the fraction of the measured HBM peak; and the
    attention of one AR step (older chunks compressed, the newest chunk raw),
    with its FLOP rate."""
    import torch
    peaks, _ = _peaks()
    hbm = peaks["hbm_gbs"]
    nb, ng = w.d * w.bits // 8, w.d // w.group
    row_bytes = nb + 2 * ng + (1 if w.C > 0 else 0)          # codes + fp16 scales + id, per token and head
    cent_bytes = w.C * w.d * 2 * w.H                           # one chunk's bf16 centroids (all heads)

    def timed(fn):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    res = {}
    tok0 = last * slots_per_chunk
    for name, dt, osz in (("decompress_f32", qvg.QVG_OUT_F32, 4), ("decompress_bf16", qvg.QVG_OUT_BF16, 2)):
        dout = torch.empty((w.N, w.H, w.d), dtype=torch.float32 if osz == 4 else torch.bfloat16, device=dev)
        ms = timed(lambda: qvg.decompress(p, kc, tok0, w.N, out_dtype=dt, out=dout))
        nbytes = w.N * w.H * row_bytes + cent_bytes + w.N * w.H * w.d * osz
        res[name] = {"ms": ms, "bytes": nbytes, "GB/s": nbytes / (ms / 1e3) / 1e9,
                     "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm,
                     "what": "newest chunk of the K cache (%d tokens x %d heads)" % (w.N, w.H)}
    # the whole cache (every chunk), where the launch's fixed costs are small
    # against its bytes
    # (every slot: the tile padding of each chunk is written as zeros)
    nslots = kc.n_tokens
    dall = torch.empty((nslots, w.H, w.d), dtype=torch.float32, device=dev)
    ms = timed(lambda: qvg.decompress(p, kc, 0, nslots, out_dtype=qvg.QVG_OUT_F32, out=dall))
    nbytes = w.tokens * w.H * row_bytes + w.n_chunks * cent_bytes + nslots * w.H * w.d * 4
    res["decompress_f32_cache"] = {"ms": ms, "bytes": nbytes, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                   "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm,
                                   "what": "whole K cache (%d tokens in %d slots x %d heads)"
                                           % (w.tokens, nslots, w.H)}
    del dall
    q16 = q[:16].contiguous()
    out16 = torch.empty((16, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    ms = timed(lambda: qvg.attention(p, q16, kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out16))
    nbytes = 2 * (w.tokens * w.H * row_bytes + w.n_chunks * cent_bytes)
    res["attention_decode16"] = {"ms": ms, "bytes": nbytes, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                 "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm,
                                 "what": "16 queries over the whole compressed K and V cache"}
    # one AR step's attention: the newest chunk's queries over the older
    # chunks (compressed) and the newest chunk's own raw bf16 K/V
    tc_peak = peaks["bf16_tflops"]
    kc.reset(last, last * slots_per_chunk)
    vc.reset(last, last * slots_per_chunk)
    k_cur, v_cur = k_raw
    out_ar = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    ms = timed(lambda: qvg.attention_ar(p, q, kc, vc, k_cur, v_cur, out_dtype=qvg.QVG_OUT_BF16, out=out_ar))
    kc.reset(last + 1, (last + 1) * slots_per_chunk)
    vc.reset(last + 1, (last + 1) * slots_per_chunk)
    flops = 4.0 * w.Nq * w.tokens * w.d * w.Hq
    res["attention_ar_step"] = {"ms": ms, "TFLOP/s": flops / (ms / 1e3) / 1e12,
                                "frac_tensor": flops / (ms / 1e3) / 1e12 / tc_peak,
                                "what": "%d queries over %d compressed chunks + the current chunk's %d raw tokens"
                                        % (w.Nq, last, w.N)}
    assert qvg.get_status() == qvg.QVG_OK
    return res


def run_own(args):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import video_diffusion_kv_gb300 as qvg
    from video_diffusion_kv_gb300 import synth

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = _workload(args.cache_chunks)
    seed = 100 + rank
    p = qvg.Params(C=w.C, L=w.L, bits=w.bits, group=w.group, iters=w.iters, seed=seed)
    slots_per_chunk = -(-w.N // qvg.QVG_TILE) * qvg.QVG_TILE
    cap = w.n_chunks * slots_per_chunk
    kc = qvg.CompressedKV(p, w.H, w.d, cap, w.n_chunks, device=dev)
    vc = qvg.CompressedKV(p, w.H, w.d, cap, w.n_chunks, device=dev)
    ws_bytes = qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d)
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    last = w.n_chunks - 1
    for k in range(last):  # prefill the older chunks (untimed)
        qvg.compress_chunk(p, synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_K), dev), kc, workspace=workspace)
        qvg.compress_chunk(p, synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_V), dev), vc, workspace=workspace)
    k_host = synth.chunk_kv(w, seed, last, synth.KIND_K)
    v_host = synth.chunk_kv(w, seed, last, synth.KIND_V)
    q_host = synth.queries(w, seed, last)
    k_new, v_new, q = synth_dev(k_host, dev), synth_dev(v_host, dev), synth_dev(q_host, dev)
    out = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kc.reset(last, last * slots_per_chunk)
        vc.reset(last, last * slots_per_chunk)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        qvg.compress_chunk(p, k_new, kc, workspace=workspace)
        e[1].record(stream)
        qvg.compress_chunk(p, v_new, vc, workspace=workspace)
        e[2].record(stream)
        qvg.attention(p, q, kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out)
        e[3].record(stream)
        return e

    for _ in range(args.warmup):
        flush.zero_()
        step()
    assert qvg.get_status() == qvg.QVG_OK
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    evs = []
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()  # L2 flush between steps, outside the timed events
        evs.append(step())
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    _barrier(ws)
    comp = [e[0].elapsed_time(e[2]) for e in evs]
    attn = [e[2].elapsed_time(e[3]) for e in evs]
    tot = [e[0].elapsed_time(e[3]) for e in evs]
    ms_step = _max_over_ranks(statistics.mean(tot), ws, dev if ws > 1 else None)
    ms_comp = statistics.mean(comp)
    ms_attn = statistics.mean(attn)
    status = qvg.get_status()

    extras = kernel_extras(qvg, p, w, kc, vc, q, (k_new, v_new), flush, dev, last, slots_per_chunk) if rank == 0 else {}

    if args.no_e2e:
        if rank == 0:
            print(json.dumps({"attention_ms": ms_attn, "compress_ms": ms_comp, "ms_per_step": ms_step,
                              "device_status": int(status), "kernels": extras}), flush=True)
        return 0
    # end-to-end through the public API with host buffers
    pin = lambda a: torch.from_numpy(a).to(torch.bfloat16).pin_memory()
    k_pin, v_pin, q_pin = pin(k_host), pin(v_host), pin(q_host)
    out_pin = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    k_d, v_d, q_d = torch.empty_like(k_new), torch.empty_like(v_new), torch.empty_like(q)

    # the inputs arrive on a copy stream, in the order they are needed, so
    # that V's and Q's copies run under the compression of K
    copy_stream = torch.cuda.Stream(dev)
    arrived = [torch.cuda.Event() for _ in range(3)]

    def e2e_step():
        kc.reset(last, last * slots_per_chunk)
        vc.reset(last, last * slots_per_chunk)
        with torch.cuda.stream(copy_stream):
            for dst, src, ev in ((k_d, k_pin, arrived[0]), (v_d, v_pin, arrived[1]), (q_d, q_pin, arrived[2])):
                dst.copy_(src, non_blocking=True)
                ev.record(copy_stream)
        cur = torch.cuda.current_stream(dev)
        cur.wait_event(arrived[0])
        qvg.compress_chunk(p, k_d, kc, workspace=workspace)
        cur.wait_event(arrived[1])
        qvg.compress_chunk(p, v_d, vc, workspace=workspace)
        cur.wait_event(arrived[2])
        qvg.attention(p, q_d, kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out)
        out_pin.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(max(3, args.steps // 2)):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        torch.cuda.synchronize()
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
    e2e = _max_over_ranks(statistics.mean(e2e_ms), ws, dev if ws > 1 else None)
    h2d = sum(t.numel() * t.element_size() for t in (k_pin, v_pin, q_pin))
    d2h = out_pin.numel() * out_pin.element_size()

    if rank != 0:
        return 0
    peaks, peak_src = _peaks()
    flops_attn = 4.0 * w.Nq * w.tokens * w.d * w.Hq
    achieved = flops_attn / (ms_attn / 1e3) / 1e12
    # The attention kernel runs QK^T and PV on the tensor cores (fp16
    # operands, fp32 accumulation): tensor roofline, dense 16-bit peak.
    tc_peak = peaks["bf16_tflops"]
    in_bytes = 2 * w.N * w.H * w.d * 2
    # the distance GEMMs of compress (K and V, iters + 1 assignments each),
    # against the bf16 tensor peak: the compress path is bound by compute
    comp_gflop = 2.0 * 2 * w.N * w.C * w.d * (w.iters + 1) * w.H / 1e9
    line = {
        "metric": METRIC, "value": ws * w.Nq / (ms_step / 1e3), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16/fp16 MMA, fp32 accum",
        "data": "synthetic",
        "config": _config(w, {"parallelism": "replicas (one layer per GPU)" if ws > 1 else "single GPU",
                               "l2": "flushed between steps (256 MiB write, outside the timed events)",
                               "out_dtype": "bf16"}),
        "compress": {"ms": ms_comp, "GB/s": in_bytes / (ms_comp / 1e3) / 1e9,
                     "frac_hbm": (in_bytes / (ms_comp / 1e3) / 1e9) / peaks["hbm_gbs"],
                     "gflop": comp_gflop, "TFLOP/s": comp_gflop / ms_comp,
                     "frac_tensor": comp_gflop / ms_comp / peaks["bf16_tflops"]},
        "attention": {"ms": ms_attn, "tok/s": w.Nq / (ms_attn / 1e3), "TFLOP/s": achieved},
        "kernels": extras,
        "roofline": {"kernel": "k_attention_ws", "bound": "tensor", "achieved": achieved,
                     "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                     "traffic": ATTN_TRAFFIC.get(_attn_source_hash()),
                     "peak_source": "%s bf16 dense burst (MEASURED_PEAKS.json); fp16 runs at the same rate" % peak_src,
                     "mma_flops_per_algorithmic_flop": 1.0},
        "clocks": clk,
        "e2e": {"value": ws * w.Nq / (e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e},
        "gpu_launches": args.steps * (2 * launches_per_compress(p) + 1),
        "device_status": int(status),
        "wall_s_timed": t_wall,
        "peaks_source": peak_src,
    }
    if not args.no_configs:
        # the other configurations of the workload list, measured on the same GPU after the timed steps
        cfgs = {}
        for name, fn in (("tiny", measure_tiny), ("qvgpro", measure_qvgpro), ("quantwm", measure_quantwm),
                         ("rollout", measure_rollout)):
            t0 = time.perf_counter()
            cfgs[name] = fn(qvg, synth, flush, peaks, dev)
            cfgs[name]["bench_wall_s"] = time.perf_counter() - t0
            torch.cuda.empty_cache()
        line["configs"] = cfgs
        line["device_status_after_configs"] = int(qvg.get_status())
    if ws == 1 and not args.no_cpu_baseline:
        t_full, thr, desc, _ = oracle_step_sample(w, seed=seed)
        line["cpu_baseline"] = {"value": w.Nq / t_full, "unit": UNIT, "cores": thr, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ studies of the other workloads

def _rel(x, y):
    import numpy as np
    return float(np.linalg.norm((x - y).astype(np.float64)) / np.linalg.norm(x.astype(np.float64)))


def _timer(flush, reps=5, warm=2):
    """Median CUDA-event time (ms) of fn() on the current stream, L2 flushed
    before each timed call (outside the events); before() runs untimed."""
    import torch

    def timed(fn, before=None):
        ts = []
        for rep in range(warm + reps):
            if before:
                before()
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if rep >= warm:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)
    return timed


def _rates(nbytes=None, flops=None, ms=None, peaks=None):
    """Throughput of one timed call and its fractions of the measured HBM and
    dense 16-bit tensor peaks."""
    out = {"ms": ms}
    if nbytes is not None:
        gbs = nbytes / (ms / 1e3) / 1e9
        out.update({"bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]})
    if flops is not None:
        tf = flops / (ms / 1e3) / 1e12
        out.update({"flops": flops, "TFLOP/s": tf, "frac_tensor": tf / peaks["bf16_tflops"]})
    return out


def _compress_counts(w, p, N=None):
    """Algorithmic bytes (bf16 input read, compressed rows written) and the
    distance-GEMM flops of compressing one chunk of K and one of V."""
    N = N or w.N
    nb, ng = w.d * p.bits // 8, w.d // p.group
    row = nb + 2 * ng + (1 if p.C > 0 else 0)
    in_b = 2 * N * w.H * w.d * 2
    out_b = 2 * p.L * (N * w.H * row + w.H * p.C * w.d * 2)
    flops = 2 * p.L * 2.0 * N * min(p.C, N) * w.d * (p.iters + 1) * w.H
    return in_b + out_b, flops


def _cache_read_bytes(w, p, n_tokens):
    nb, ng = w.d * p.bits // 8, w.d // p.group
    row = nb + 2 * ng + (1 if p.C > 0 else 0)
    n_chunks = -(-n_tokens // w.N)
    return 2 * p.L * (n_tokens * w.H * row + n_chunks * w.H * p.C * w.d * 2)


def measure_tiny(qvg, synth, flush, peaks, dev="cuda"):
    """Config 1: 2 heads, d=64, 4 chunks x 256 tokens, C=16, INT2 G=32, 10
    Lloyd iterations; 256 queries over the 1024 cached tokens."""
    import torch
    w = synth.WORKLOADS["tiny"]
    seed = 31
    p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=seed)
    per = -(-w.N // 128) * 128
    kc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks, device=dev)
    vc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks, device=dev)
    kd = [synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_K), dev) for k in range(w.n_chunks)]
    vd = [synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_V), dev) for k in range(w.n_chunks)]
    ws = torch.empty(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d), dtype=torch.uint8, device=dev)
    for k in range(w.n_chunks):
        qvg.compress_chunk(p, kd[k], kc, workspace=ws)
        qvg.compress_chunk(p, vd[k], vc, workspace=ws)
    last = w.n_chunks - 1
    q = synth_dev(synth.queries(w, seed, w.n_chunks), dev)
    out = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    timed = _timer(flush)

    def rewind():
        kc.reset(last, last * per)
        vc.reset(last, last * per)

    def comp():
        qvg.compress_chunk(p, kd[last], kc, workspace=ws)
        qvg.compress_chunk(p, vd[last], vc, workspace=ws)

    ms_c = timed(comp, rewind)
    nbytes, flops = _compress_counts(w, p)
    ms_a = timed(lambda: qvg.attention(p, q, kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out))
    dall = torch.empty((kc.n_tokens, w.H, w.d), dtype=torch.float32, device=dev)
    ms_d = timed(lambda: qvg.decompress(p, kc, 0, kc.n_tokens, out=dall))
    return {"workload": "tiny: 2 KV heads, d=64, 4 chunks x 256 tokens, C=16, INT2 G=32, 10 Lloyd iters",
            "compress_KV_newest": dict(_rates(nbytes, flops, ms_c, peaks), what="K and V of one 256-token chunk; "
                                       "launch-bound (report absolute time)"),
            "attention": dict(_rates(_cache_read_bytes(w, p, w.tokens), 4.0 * w.Nq * w.tokens * w.d * w.Hq, ms_a, peaks),
                              **{"tok/s": w.Nq / (ms_a / 1e3), "what": "256 queries over 1024 cached tokens"}),
            "decompress_f32_cache": _rates(_cache_read_bytes(w, p, w.tokens) / 2 + kc.n_tokens * w.H * w.d * 4,
                                           None, ms_d, peaks),
            "ratio": qvg.compression_ratio(p, w.H, w.d, w.N, w.n_chunks)}


def measure_qvgpro(qvg, synth, flush, peaks, dev="cuda"):
    """Config 3, QVG-Pro on the tiny shapes: INT2 G=32 with L = 1, 2, 3 and
    INT4 G=32 with L = 1, 2; relative Frobenius error of K and V after each
    stage count, the compression ratio counting codes, fp16 scales, ids and
    bf16 centroids, and the compress / attention times."""
    import numpy as np
    import torch
    w = synth.WORKLOADS["qvgpro"]
    seed = 5
    per = -(-w.N // 128) * 128
    timed = _timer(flush)
    xs = {kind: [synth.chunk_kv(w, seed, k, kind) for k in range(w.n_chunks)] for kind in (synth.KIND_K, synth.KIND_V)}
    xd = {kind: [synth_dev(x, dev) for x in xs[kind]] for kind in xs}
    q = synth_dev(synth.queries(w, seed, w.n_chunks), dev)
    out = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    arms = []
    for bits, stages in ((2, 3), (4, 2)):
        for L in range(1, stages + 1):
            p = qvg.Params(C=w.C, L=L, bits=bits, group=w.group, iters=w.iters, seed=seed)
            cs = {}
            errs = {}
            ws = torch.empty(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d), dtype=torch.uint8, device=dev)
            for kind, name in ((synth.KIND_K, "K"), (synth.KIND_V, "V")):
                c = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks, device=dev)
                for x in xd[kind]:
                    qvg.compress_chunk(p, x, c, workspace=ws)
                xh = qvg.decompress(p, c, 0, c.n_tokens).cpu().numpy()
                errs[name] = _rel(np.concatenate(xs[kind], 0), xh)
                cs[name] = c
            last = w.n_chunks - 1

            def rewind():
                for c in cs.values():
                    c.reset(last, last * per)

            def comp():
                qvg.compress_chunk(p, xd[synth.KIND_K][last], cs["K"], workspace=ws)
                qvg.compress_chunk(p, xd[synth.KIND_V][last], cs["V"], workspace=ws)

            ms_c = timed(comp, rewind)
            ms_a = timed(lambda: qvg.attention(p, q, cs["K"], cs["V"], out_dtype=qvg.QVG_OUT_BF16, out=out))
            rtn = qvg.Params(C=0, L=1, bits=bits, group=w.group, iters=0)
            nbytes, flops = _compress_counts(w, p)
            arms.append({"bits": bits, "stages": L, "rel_err_K": errs["K"], "rel_err_V": errs["V"],
                         "ratio": qvg.compression_ratio(p, w.H, w.d, w.N, w.n_chunks),
                         "ratio_rtn_same_bits": qvg.compression_ratio(rtn, w.H, w.d, w.N, w.n_chunks),
                         "compress_KV_newest": _rates(nbytes, flops, ms_c, peaks),
                         "attention": _rates(_cache_read_bytes(w, p, w.tokens), 4.0 * w.Nq * w.tokens * w.d * w.Hq,
                                             ms_a, peaks)})
    return {"workload": "QVG-Pro on the tiny shapes: 2 heads, d=64, 4 chunks x 256 tokens, C=16, G=32, 10 iters",
            "arms": arms}


def measure_quantwm(qvg, synth, flush, peaks, dev="cuda", nthreads=None):
    """Config 4, the QuantWM world-model cache: 24 heads, d=128, 8 chunks of
    3 frames of 22x40 (21,120 tokens), C=256, INT2 G=64, 8 iterations.
    History queries (4 frames) give the QSAC weights and the PSAC basis; the
    top-1 attention-token shift rate of an 880-token query frame (the GPU's
    top-1 over the compressed cache) is measured against the oracle's argmax
    over the bf16 cache for the arms QVG, +QSAC, +PSAC and both."""
    import numpy as np
    import torch

    import oracle
    w = synth.WORKLOADS["quantwm"]
    seed = 7
    timed = _timer(flush)
    qh = synth_dev(synth.history_queries(w, seed), dev)
    M, wq, cnt = qvg.query_stats(qh, w.H)
    U, eig, frac = qvg.psac_basis(M, cnt)
    ms_stats = timed(lambda: qvg.query_stats(qh, w.H, M=M, w=wq, count=cnt))
    ms_basis = timed(lambda: qvg.psac_basis(M, cnt))
    wh = wq.cpu().numpy()
    act = synth.active_channels(w, seed)
    on = np.zeros(wh.shape, bool)
    for h in range(w.H):
        on[h, act[h]] = True
    ks = [synth.chunk_kv(w, seed, k, synth.KIND_K) for k in range(w.n_chunks)]
    vs = [synth.chunk_kv(w, seed, k, synth.KIND_V) for k in range(w.n_chunks)]
    kd = [synth_dev(x, dev) for x in ks]
    vd = [synth_dev(x, dev) for x in vs]
    qf = synth.history_queries(w, seed, n_tokens=w.Nq, stream=1)
    qfd = synth_dev(qf, dev)
    kall = np.concatenate(ks, 0)
    t0 = time.perf_counter()
    ref = oracle.top1(qf, kall, nthreads=nthreads or os.cpu_count() or 1)  # [Hq, Nq] token indices
    t_oracle = time.perf_counter() - t0
    per = -(-w.N // 128) * 128
    keep = np.concatenate([np.arange(k * per, k * per + w.N) for k in range(w.n_chunks)])
    arms = {}
    for name, flags in (("QVG", 0), ("QSAC", qvg.QVG_QSAC), ("PSAC", qvg.QVG_PSAC),
                        ("QSAC+PSAC", qvg.QVG_QSAC | qvg.QVG_PSAC)):
        p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=seed, flags=flags)
        pv = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=seed)
        kc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks, device=dev)
        vc = qvg.CompressedKV(pv, w.H, w.d, w.n_chunks * per, w.n_chunks, device=dev)
        ws = torch.empty(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d), dtype=torch.uint8, device=dev)
        for k in range(w.n_chunks):
            qvg.compress_chunk(p, kd[k], kc, qsac_w=wq, psac_basis=U, workspace=ws)
            qvg.compress_chunk(pv, vd[k], vc, workspace=ws)
        _, _, top1 = qvg.attention(p, qfd, kc, vc, want_top1=True)
        slots = top1.cpu().numpy()
        tok = (slots // per) * w.N + slots % per  # slot -> token index
        kh = qvg.decompress(p, kc, 0, kc.n_tokens).cpu().numpy()
        last = w.n_chunks - 1

        def rewind():
            kc.reset(last, last * per)
            vc.reset(last, last * per)

        def comp():
            qvg.compress_chunk(p, kd[last], kc, qsac_w=wq, psac_basis=U, workspace=ws)
            qvg.compress_chunk(pv, vd[last], vc, workspace=ws)

        ms_c = timed(comp, rewind)
        ms_a = timed(lambda: qvg.attention(p, qfd, kc, vc))
        nbytes, flops = _compress_counts(w, p)
        arms[name] = {"shift_rate": float((tok != ref).mean()),
                      "rel_err_K": _rel(kall, kh[keep]),
                      "ratio_K": qvg.compression_ratio(p, w.H, w.d, w.N, w.n_chunks,
                                                      with_psac=bool(flags & qvg.QVG_PSAC)),
                      "compress_KV_newest": _rates(nbytes, flops * (2 if flags & qvg.QVG_QSAC else 1), ms_c, peaks),
                      "attention": dict(_rates(_cache_read_bytes(w, p, w.tokens),
                                               4.0 * w.Nq * w.tokens * w.d * w.Hq, ms_a, peaks),
                                        **{"tok/s": w.Nq / (ms_a / 1e3)})}
        del kc, vc
    return {"workload": "QuantWM: 24 heads, d=128, 8 chunks x 2640 tokens (21,120), C=256, INT2 G=64, 8 iters; "
                        "880 query tokens; shift rate = GPU top-1 over the compressed cache vs the oracle's "
                        "argmax over the bf16 cache",
            "qsac_weight": {"active_channels_mean": float(wh[on].mean()), "other_channels_mean": float(wh[~on].mean()),
                            "min": float(wh.min()), "max": float(wh.max())},
            "energy_frac_top8_mean": float(frac.mean().item()),
            "query_stats_ms": ms_stats, "psac_basis_ms": ms_basis,
            "oracle_top1_s": t_oracle, "arms": arms}


def measure_rollout(qvg, synth, flush, peaks, dev="cuda"):
    """Config 5, the one-minute rollout: 288 frames of 30x52 streamed in 96
    chunks of 4680 tokens (449,280), 8 heads, d=128, INT2 C=256 G=64, 8
    iterations.  After compressing each chunk its 4680 queries attend over
    the whole compressed cache.  Chunks are drawn from the stationary
    16-prototype mixture; 12 distinct chunks are generated and cycled."""
    import torch
    w = synth.WORKLOADS["rollout"]
    seed = 9
    p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=seed)
    per = -(-w.N // 128) * 128
    kc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks, device=dev)
    vc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks, device=dev)
    uniq = 12
    K = [synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_K), dev) for k in range(uniq)]
    V = [synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_V), dev) for k in range(uniq)]
    Q = [synth_dev(synth.queries(w, seed, k), dev) for k in range(uniq)]
    out = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d), dtype=torch.uint8, device=dev)
    # one untimed chunk through a scratch cache first, so that the first
    # timed step does not include the kernels' first-launch loading
    scratch_k = qvg.CompressedKV(p, w.H, w.d, per, 1, device=dev)
    scratch_v = qvg.CompressedKV(p, w.H, w.d, per, 1, device=dev)
    qvg.compress_chunk(p, K[0], scratch_k, workspace=ws)
    qvg.compress_chunk(p, V[0], scratch_v, workspace=ws)
    qvg.attention(p, Q[0], scratch_k, scratch_v, out_dtype=qvg.QVG_OUT_BF16, out=out)
    torch.cuda.synchronize()
    del scratch_k, scratch_v
    points, comp_ms, step_ms = [], [], []
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for k in range(w.n_chunks):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        qvg.compress_chunk(p, K[k % uniq], kc, workspace=ws)
        qvg.compress_chunk(p, V[k % uniq], vc, workspace=ws)
        e[1].record()
        qvg.attention(p, Q[k % uniq], kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out)
        e[2].record()
        torch.cuda.synchronize()
        comp_ms.append(e[0].elapsed_time(e[1]))
        step_ms.append(e[0].elapsed_time(e[2]))
        if k in (0, 7, 23, 47, 71, 95):
            nk = (k + 1) * w.N
            ms = e[1].elapsed_time(e[2])
            points.append(dict(_rates(_cache_read_bytes(w, p, nk), 4.0 * w.Nq * nk * w.d * w.Hq, ms, peaks),
                               chunks=k + 1, cache_tokens=nk))
    t_wall = time.perf_counter() - t_wall
    timed = _timer(flush)
    ms_last = timed(lambda: qvg.attention(p, Q[(w.n_chunks - 1) % uniq], kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out))
    dall = torch.empty((w.N, w.H, w.d), dtype=torch.float32, device=dev)
    ms_d = timed(lambda: qvg.decompress(p, kc, kc.n_tokens - per, w.N, out=dall))
    nbytes, flops = _compress_counts(w, p)
    return {"workload": "rollout: 8 heads, d=128, 96 chunks x 4680 tokens (449,280), C=256, INT2 G=64, 8 iters",
            "points": points,
            "last_chunk_attention": dict(_rates(_cache_read_bytes(w, p, w.tokens),
                                                4.0 * w.Nq * w.tokens * w.d * w.Hq, ms_last, peaks),
                                         **{"tok/s": w.Nq / (ms_last / 1e3),
                                            "what": "4680 queries over 449,280 cached tokens, L2 flushed"}),
            "compress_KV_per_chunk": _rates(nbytes, flops, statistics.median(comp_ms), peaks),
            "decompress_newest_chunk_f32": _rates(_cache_read_bytes(w, p, w.N) / 2 + w.N * w.H * w.d * 4, None,
                                                  ms_d, peaks),
            "rollout_s": sum(step_ms) / 1e3, "rollout_wall_s": t_wall,
            "cache_bytes_compressed": kc.nbytes + vc.nbytes,
            "cache_bytes_bf16": qvg.kv_bytes_uncompressed(1, w.H, w.d, w.tokens)}


def _study(fn, name):
    def run(args):
        import torch

        import __graft_entry__
        __graft_entry__.build()
        import video_diffusion_kv_gb300 as qvg
        from video_diffusion_kv_gb300 import synth
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        peaks, _ = _peaks()
        res = fn(qvg, synth, flush, peaks)
        print(json.dumps({"study": name, "status": qvg.get_status(), **res}), flush=True)
        return 0
    return run


study_tiny = _study(measure_tiny, "tiny")
study_qvgpro = _study(measure_qvgpro, "qvgpro")
study_quantwm = _study(measure_quantwm, "quantwm")
study_rollout = _study(measure_rollout, "rollout")


def study_outlier(args):
    """Outlier split on the LongCat-like layer (16 heads, d=128, 8 chunks of
    4680 tokens, C=256, INT2 G=64): with and without the split, the
    relative Frobenius error of K and V over the whole cache, the
    compression ratio counting the side list, the time to compress the
    newest chunk (K and V) and the attention of its 4680 queries over the
    whole compressed cache (median of 5, L2 flushed before each)."""
    import statistics
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import video_diffusion_kv_gb300 as qvg
    from video_diffusion_kv_gb300 import synth
    w = synth.WORKLOADS["longcat"]
    seed = 12
    per = -(-w.N // 128) * 128
    ks = [synth.chunk_kv(w, seed, k, synth.KIND_K) for k in range(w.n_chunks)]
    vs = [synth.chunk_kv(w, seed, k, synth.KIND_V) for k in range(w.n_chunks)]
    q = synth_dev(synth.queries(w, seed, w.n_chunks - 1), "cuda")
    kd = [synth_dev(x, "cuda") for x in ks]
    vd = [synth_dev(x, "cuda") for x in vs]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    keep = np.concatenate([np.arange(k * per, k * per + w.N) for k in range(w.n_chunks)])
    arms = {}
    for name, flags in (("plain", 0), ("outlier_split", qvg.QVG_OUTLIER)):
        p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=seed, flags=flags)
        kc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks)
        vc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks)
        ws = torch.empty(max(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d), 1), dtype=torch.uint8,
                         device="cuda")
        for k in range(w.n_chunks):
            qvg.compress_chunk(p, kd[k], kc, workspace=ws)
            qvg.compress_chunk(p, vd[k], vc, workspace=ws)
        errs = {}
        for nm, c, xs in (("K", kc, ks), ("V", vc, vs)):
            xh = qvg.decompress(p, c, 0, c.n_tokens).cpu().numpy()[keep]
            errs[nm] = _rel(np.concatenate(xs, 0), xh)
        last = w.n_chunks - 1

        def timed(fn):
            ts = []
            for rep in range(7):
                kc.reset(last, last * per)
                vc.reset(last, last * per)
                if fn is attend:  # attention reads the whole cache: put the newest chunk back
                    kc.reset(last + 1, (last + 1) * per)
                    vc.reset(last + 1, (last + 1) * per)
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                if rep >= 2:
                    ts.append(e0.elapsed_time(e1))
            return statistics.median(ts)

        def compress():
            qvg.compress_chunk(p, kd[last], kc, workspace=ws)
            qvg.compress_chunk(p, vd[last], vc, workspace=ws)

        def attend():
            qvg.attention(p, q, kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out)

        tcs = timed(compress)
        ms_a = timed(attend)
        arms[name] = {"rel_err_K": errs["K"], "rel_err_V": errs["V"],
                      "ratio": qvg.compression_ratio(p, w.H, w.d, w.N, w.n_chunks),
                      "compress_ms_KV": tcs, "attention_ms": ms_a,
                      "attention_TFLOP/s": 4.0 * w.Nq * w.tokens * w.d * w.Hq / ms_a / 1e9}
    print(json.dumps({"study": "outlier", "workload": "16 heads, d=128, 8 chunks x 4680 tokens, C=256, INT2 G=64, 8 iters",
                      "status": qvg.get_status(), "arms": arms}), flush=True)
    return 0


def study_paths(args):
    """Attention read paths on the LongCat-like layer (16 heads, d=128, 8
    chunks of 4680 tokens, C=256, 8 iters): 4680 queries over the whole
    compressed cache for one-stage INT2 G=64 (plain, and with the outlier
    split), the split with G=16, two stages (QVG-Pro), PSAC on the keys
    (rank-8 orthonormal basis, seeded) and temporal anchors (chunks 0 and 4
    kept as bf16, read as raw tiles between the INT2 ones).  Median of 5 launches, L2 flushed
    before each; plus the time to compress the newest chunk (K and V)."""
    import statistics
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import video_diffusion_kv_gb300 as qvg
    from video_diffusion_kv_gb300 import synth
    w = synth.WORKLOADS["longcat"]
    seed = 13
    per = -(-w.N // 128) * 128
    kd = [synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_K), "cuda") for k in range(w.n_chunks)]
    vd = [synth_dev(synth.chunk_kv(w, seed, k, synth.KIND_V), "cuda") for k in range(w.n_chunks)]
    q = synth_dev(synth.queries(w, seed, w.n_chunks - 1), "cuda")
    rng = np.random.default_rng(seed)
    U = np.stack([np.linalg.qr(rng.standard_normal((w.d, qvg.QVG_PSAC_RANK)))[0] for _ in range(w.H)])
    U = torch.from_numpy(U.astype(np.float32)).cuda()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    arms = {}
    for name, kw in (("L1_G64", {}), ("outlier_G64", dict(flags=qvg.QVG_OUTLIER)),
                     ("outlier_G16", dict(flags=qvg.QVG_OUTLIER, group=16)), ("L2_G64", dict(L=2)),
                     ("psac_G64", dict(flags=qvg.QVG_PSAC)), ("anchors_every4", dict(anchor_every=4))):
        p = qvg.Params(**{**dict(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=seed), **kw})
        pv = qvg.Params(**{**p.__dict__, "flags": p.flags & ~qvg.QVG_PSAC})
        kc = qvg.CompressedKV(p, w.H, w.d, w.n_chunks * per, w.n_chunks)
        vc = qvg.CompressedKV(pv, w.H, w.d, w.n_chunks * per, w.n_chunks)
        ws = torch.empty(max(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d), 1), dtype=torch.uint8,
                         device="cuda")
        psac = U if p.flags & qvg.QVG_PSAC else None

        def compress(k):
            qvg.compress_chunk(p, kd[k], kc, psac_basis=psac, workspace=ws)
            qvg.compress_chunk(pv, vd[k], vc, workspace=ws)

        for k in range(w.n_chunks):
            compress(k)
        last = w.n_chunks - 1

        def timed(fn, before=None):
            ts = []
            for rep in range(7):
                if before:
                    before()
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                if rep >= 2:
                    ts.append(e0.elapsed_time(e1))
            return statistics.median(ts)

        def rewind():
            kc.reset(last, last * per)
            vc.reset(last, last * per)

        ms_c = timed(lambda: compress(last), rewind)
        ms_a = timed(lambda: qvg.attention(p, q, kc, vc, out_dtype=qvg.QVG_OUT_BF16, out=out))
        arms[name] = {"attention_ms": ms_a, "attention_TFLOP/s": 4.0 * w.Nq * w.tokens * w.d * w.Hq / ms_a / 1e9,
                      "compress_ms_KV": ms_c, "ratio": qvg.compression_ratio(p, w.H, w.d, w.N, w.n_chunks)}
        del kc, vc
    print(json.dumps({"study": "paths", "workload": "16 heads, d=128, 8 chunks x 4680 tokens, C=256, INT2, 8 iters; "
                      "4680 queries", "status": qvg.get_status(), "arms": arms}), flush=True)
    return 0


def study_layers(args):
    """Multi-layer streaming rollout: a 48-layer stack of LongCat-like layers
    (16 KV heads, d=128; INT2 C=256 G=64, 8 iterations) generates 8 chunks of
    4680 tokens (37,440 tokens, about the 38K-token, 5-second LongCat-Video
    clip of the QVG notes).  Each chunk step runs, for every layer in order,
    the AR-step attention of the chunk's 4680 queries over the layer's
    compressed history plus the chunk's own raw K/V (qvg_attention_ar), then
    compresses the chunk's K and V into that layer's cache.  Reports the
    time of each chunk step, and the memory held against the uncompressed
    size 2 x layers x KV heads x head_dim x tokens x 2 B ("The 2-bit
    quantisation trap", section 1).  Layers draw from a pool of 4 synthetic
    chunk sets (seeded per position), cycled over the layers."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import video_diffusion_kv_gb300 as qvg
    from video_diffusion_kv_gb300 import synth
    w = synth.WORKLOADS["longcat"]
    layers, pool = 48, 4
    p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=21)
    per = -(-w.N // 128) * 128
    cap = w.n_chunks * per
    base = torch.cuda.memory_allocated()
    kcs = [qvg.CompressedKV(p, w.H, w.d, cap, w.n_chunks) for _ in range(layers)]
    vcs = [qvg.CompressedKV(p, w.H, w.d, cap, w.n_chunks) for _ in range(layers)]
    held = torch.cuda.memory_allocated() - base
    K = [[synth_dev(synth.chunk_kv(w, 21 + j, k, synth.KIND_K), "cuda") for k in range(w.n_chunks)] for j in range(pool)]
    V = [[synth_dev(synth.chunk_kv(w, 21 + j, k, synth.KIND_V), "cuda") for k in range(w.n_chunks)] for j in range(pool)]
    Q = [[synth_dev(synth.queries(w, 21 + j, k), "cuda") for k in range(w.n_chunks)] for j in range(pool)]
    ws = torch.empty(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d), dtype=torch.uint8, device="cuda")
    aws = torch.empty(max(qvg.workspace_size(p, qvg.QVG_OP_ATTENTION, w.Nq, w.H, w.d, w.Hq), 1), dtype=torch.uint8,
                      device="cuda")
    out = torch.empty((w.Nq, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    steps = []
    for k in range(w.n_chunks):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        evs = []
        e[0].record()
        for li in range(layers):
            j = li % pool
            ea = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ea[0].record()
            qvg.attention_ar(p, Q[j][k], kcs[li], vcs[li], K[j][k], V[j][k], out_dtype=qvg.QVG_OUT_BF16, out=out,
                             workspace=aws)
            ea[1].record()
            qvg.compress_chunk(p, K[j][k], kcs[li], workspace=ws)
            qvg.compress_chunk(p, V[j][k], vcs[li], workspace=ws)
            ea[2].record()
            evs.append(ea)
        e[1].record()
        torch.cuda.synchronize()
        ta = sum(ea[0].elapsed_time(ea[1]) for ea in evs)
        tc = sum(ea[1].elapsed_time(ea[2]) for ea in evs)
        tokens = (k + 1) * w.N
        steps.append({"chunk": k + 1, "cache_tokens_after": tokens, "step_ms": e[0].elapsed_time(e[1]),
                      "attention_ms": ta, "compress_ms": tc})
    tokens = w.tokens
    comp = sum(c.nbytes for c in kcs + vcs)
    bf16 = qvg.kv_bytes_uncompressed(layers, w.H, w.d, tokens)
    ratio = qvg.compression_ratio(p, w.H, w.d, w.N, w.n_chunks)
    print(json.dumps({"study": "layers", "workload": "48 layers x 16 KV heads x d=128, 8 chunks x 4680 tokens "
                      "(37,440), INT2 C=256 G=64, 8 iters; per layer: AR-step attention then compress K and V",
                      "status": qvg.get_status(), "steps": steps,
                      "total_ms": sum(x["step_ms"] for x in steps),
                      "memory": {"cache_bytes_allocated": held, "cache_bytes_sized": comp,
                                 "bf16_bytes_same_tokens": bf16, "ratio_stored": ratio,
                                 "device_bytes_in_use": torch.cuda.memory_allocated()},
                      "page_scale": {"what": "32 KV heads x d=128 x 48 layers (a LongCat-Video-sized stack) at 37,440 tokens",
                                     "bf16_bytes": qvg.kv_bytes_uncompressed(layers, 32, w.d, tokens),
                                     "compressed_bytes": qvg.kv_bytes_uncompressed(layers, 32, w.d, tokens) / ratio}}),
          flush=True)
    return 0


def synth_dev(a, dev):
    import torch
    return torch.from_numpy(a).to(dev, torch.bfloat16).contiguous()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="time the device step only (profiling)")
    ap.add_argument("--cache-chunks", type=int, default=None, help="smaller cache (profiling cases)")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations' measurements")
    ap.add_argument("--workload", default="longcat",
                    choices=["longcat", "tiny", "qvgpro", "quantwm", "rollout", "outlier", "paths", "layers"],
                    help="longcat: the benchmark line; the others print their study line")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "own":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "longcat":
        return {"tiny": study_tiny, "qvgpro": study_qvgpro, "quantwm": study_quantwm, "rollout": study_rollout,
                "outlier": study_outlier, "paths": study_paths, "layers": study_layers}[args.workload](args)
    return run_own(args)


if __name__ == "__main__":
    sys.exit(main())
