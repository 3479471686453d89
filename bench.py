"""Benchmark of one batched paged-KV decode step on GB300.

A step = paged_decode_attention_append (the new K/V token of each sequence
written into its block by the split-KV main kernel just before it loads that
block, then the combine kernel) -> sample_tokens, over one batch of the
Llama-style GQA workload: batch 64, 32 query / 8 KV heads, head_dim 128,
block_size 16, lengths uniform in [512, 4096], shuffled block tables, bf16 KV,
logits over a 128256-token vocabulary (T = 0.7, top_k = 50, top_p = 0.9).

Printed (one JSON line, rank 0):
  value          algorithmic HBM bytes of the whole step / device step time (GB/s)
  sampled_tokens_per_s   batch / device step time
  roofline       paged_decode_attention_append's achieved GB/s (CUDA events around each
                 call in a second timed run of up to 500 steps) against the
                 measured copy peak
  e2e            the same metric with host buffers: every step one pinned H2D copy
                 of all its inputs, the three calls, D2H of the sampled tokens;
                 the copies double-buffered on a second stream so that a step's
                 upload overlaps the previous step's kernels (serial_*: without)
  graph          the step captured as a CUDA graph (20 steps per graph) and replayed
  cpu_baseline   the float64 oracle on this host's cores on a bounded sample
Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_decode_table_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of HBM peak); sampled tokens/sec"
WORKLOAD = 2
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _bf16_peak():
    """Measured dense bf16 TFLOP/s (burst) from MEASURED_PEAKS.json, else the fallback 1900."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        for k in ("bf16_tflops", "bf16_tflops_burst"):
            if k in d:
                return float(d[k])
    return 1900.0


def _source_hash():
    h = hashlib.sha256()
    for rel in ("paged_kv_decode_table_gb300/csrc/decode_attention.cu",
                "paged_kv_decode_table_gb300/csrc/pkv_common.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_per_launch():
    """DRAM bytes per attention call from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "decode_attention_gqa_b64_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_sha256_16") != _source_hash():
        return None
    try:
        return int(float(kv["traffic_bytes_per_call"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="pkv_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax = [], None
        for r in rows:
            try:
                sm.append(float(r[0]))
                smax = float(r[1])
            except ValueError:
                continue
            for i, n in enumerate(names):
                if r[4 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    n = int(os.environ.get("WORLD_SIZE", "1"))
    if n > 1 and not torch.distributed.is_initialized():
        backend = os.environ.get("PKV_DIST_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        torch.distributed.init_process_group(backend)
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return n, rank, local


def _max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t)
    return float(t.item())


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _config(w, inp, extra=None):
    sl = inp["seq_lens"]
    cfg = {
        "workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
        "head_dim": w.head_dim, "block_size": w.block_size, "seq_len_range": [w.len_lo, w.len_hi],
        "total_tokens": int(sl.to(torch.int64).sum()), "num_blocks": inp["num_blocks"], "vocab": w.vocab,
        "sampler": {"temperature": w.temperature, "top_k": w.top_k, "top_p": w.top_p},
        "kv_dtype": "bf16", "logits_dtype": "f32",
        "step": "paged_decode_attention_append (split-KV main with the KV append, combine) -> sample_tokens",
    }
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------- oracle baseline
def _oracle_sample_step(w, host_inp, n_seq: int, n_rows: int):
    """One bounded oracle step: append for every sequence, attention for the
    first n_seq sequences (all heads), sampler for the first n_rows rows.
    Returns (seconds, algorithmic bytes processed)."""
    import numpy as np
    import oracle
    h = host_inp
    t0 = time.perf_counter()
    K, V = h["k_cache"], h["v_cache"]
    oracle.kv_append(h["k_new"], h["v_new"], K, V, h["block_tables"], h["seq_lens"], w.block_size)
    rows = np.arange(n_seq * w.n_q_heads, dtype=np.int64)
    oracle.paged_attention(h["q"], K, V, h["block_tables"], h["seq_lens"], rows=rows)
    oracle.sample_batch(h["logits"][:n_rows], h["temperature"][:n_rows], h["top_k"][:n_rows],
                        h["top_p"][:n_rows], h["seeds"][:n_rows], h["offsets"][:n_rows])
    dt = time.perf_counter() - t0
    sl = h["seq_lens"][:n_seq].astype(np.int64)
    e = w.elem_bytes
    attn = int(sl.sum()) * w.n_kv_heads * w.head_dim * 2 * e + 2 * n_seq * w.n_q_heads * w.head_dim * e \
        + 4 * int(((sl + w.block_size - 1) // w.block_size).sum()) + 4 * n_seq
    append = 2 * (2 * w.batch * w.n_kv_heads * w.head_dim * e) + 8 * w.batch
    samp = 4 * n_rows * w.vocab + n_rows * 32 + 4 * n_rows
    return dt, attn + append + samp


def _host_copy(inp):
    import numpy as np
    out = {}
    for k, v in inp.items():
        if not isinstance(v, torch.Tensor):
            out[k] = v
            continue
        t = v.detach().contiguous().cpu()
        if t.dtype == torch.bfloat16:
            out[k] = t.view(torch.int16).numpy().view(np.uint16).copy()
        elif k in ("seeds", "offsets"):
            out[k] = t.numpy().view(np.uint64).copy()
        else:
            out[k] = t.numpy().copy()
    return out


def cpu_baseline(w, inp, budget_s: float = 12.0):
    import oracle
    oracle.build()
    h = _host_copy(inp)
    n_seq, n_rows = 2, 2
    dt, by = _oracle_sample_step(w, h, n_seq, n_rows)       # also warms the library
    # grow the sample to roughly fill the time budget
    scale = max(1.0, min(w.batch / n_seq, budget_s / max(dt, 1e-3)))
    n_seq = int(min(w.batch, max(1, n_seq * scale)))
    n_rows = int(min(w.batch, max(1, n_rows * scale)))
    # repeat the (possibly whole-batch) step until about budget_s of CPU work is timed
    tot_t, tot_b, reps = 0.0, 0, 0
    while tot_t < budget_s and reps < 1000:
        dt, by = _oracle_sample_step(w, h, n_seq, n_rows)
        tot_t += dt
        tot_b += by
        reps += 1
    return {"value": tot_b / tot_t / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} x (append of all {w.batch} sequences + attention of {n_seq} sequences x "
                      f"{w.n_q_heads} heads + sampler on {n_rows} rows), float64 C oracle, {tot_t:.1f} s"}


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = W.workload(WORKLOAD)
    inp = W.make_decode_inputs(w, "cpu")
    h = _host_copy(inp)
    # each step: a bounded sample sized so that warmup + steps stay within ~2 minutes
    dt1, _ = _oracle_sample_step(w, h, 1, 1)
    per_step_budget = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    n = max(1, min(w.batch, int(per_step_budget / max(dt1, 1e-4))))
    for _ in range(args.warmup):
        _oracle_sample_step(w, h, n, n)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, by = _oracle_sample_step(w, h, n, n)
        tot_t += dt
        tot_b += by
    val = tot_b / tot_t / 1e9
    cb = {"value": val, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
          "sample": f"per step: append of all {w.batch} sequences + attention of {n} sequences x "
                    f"{w.n_q_heads} heads + sampler on {n} rows (float64 C oracle)"}
    line = {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot_t / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, inp, {"impl_note": "float64 CPU oracle on a bounded sample per step"}),
            "impl": "reference", "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm
def run_gpu(args):
    import paged_kv_decode_table_gb300 as pkv
    from paged_kv_decode_table_gb300 import build as pkv_build
    world, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv_build.build()
    pkv.load_library()
    w = W.workload(WORKLOAD)
    inp = W.make_decode_inputs(w, dev)
    B = w.batch
    bytes_step = W.step_bytes(w, inp["seq_lens"])
    out = torch.empty_like(inp["q"])
    tokens = torch.empty(B, dtype=torch.int32, device=dev)
    ws = torch.empty(pkv.decode_workspace_bytes(B, w.n_q_heads, w.head_dim), dtype=torch.uint8, device=dev)
    status = pkv.new_status(dev)
    k_cache, v_cache = inp["k_cache"], inp["v_cache"]

    def make_step(d):
        """The public API's prepared step (buffers checked once) over the inputs d."""
        return pkv.DecodeStep(d["q"], d["k_new"], d["v_new"], k_cache, v_cache, d["block_tables"], d["seq_lens"],
                              d["logits"], d["temperature"], d["top_k"], d["top_p"], d["seeds"], d["offsets"],
                              out=out, tokens=tokens, workspace=ws, status=status)

    dstep = make_step(inp)
    step = dstep.run
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if pkv.check_status(status) != 0:
        raise SystemExit(f"device status {pkv.status_string(pkv.check_status(status))} during warm-up")

    stream = torch.cuda.current_stream(dev)
    # Timed region 1 (the headline): K whole steps back to back, events only at
    # its ends, so that the kernels of a step chain as they would in a server.
    # Timed region 2 (the roofline): K2 more steps with events around every
    # paged_decode_attention_append call, giving that call's average device duration.
    k2 = min(args.steps, 500)
    a0 = [torch.cuda.Event(enable_timing=True) for _ in range(k2)]
    a1 = [torch.cuda.Event(enable_timing=True) for _ in range(k2)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    # a spin kernel (about 15 us of GPU time per step, outside the events) while
    # the host enqueues the K steps, so that the timed region holds the steps'
    # device time and no wait for the host's first launches (a serving loop
    # keeps the host ahead of the GPU the same way)
    torch.cuda._sleep(int(min(args.steps, 4000) * 30_000))
    t0.record(stream)
    for i in range(args.steps):
        step()
    t1.record(stream)
    for i in range(k2):
        a0[i].record(stream)
        dstep.run_attention()
        a1[i].record(stream)
        dstep.run_sampler()
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    ms_local = t0.elapsed_time(t1) / args.steps
    ms = _max_over_ranks(ms_local, world, dev)
    attn_ms = sum(a0[i].elapsed_time(a1[i]) for i in range(k2)) / k2
    if pkv.check_status(status) != 0:
        raise SystemExit(f"device status {pkv.status_string(pkv.check_status(status))} in the timed region")

    # the same step captured as a CUDA graph of kGraphSteps steps and replayed:
    # the per-call host work (argument checks, launches) leaves the timed region
    graph = None
    if world == 1:
        kGraphSteps, reps = 20, max(3, args.steps // 20)
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        dstep.set_stream(gs)
        with torch.cuda.stream(gs):
            with torch.cuda.graph(g, stream=gs):
                for _ in range(kGraphSteps):
                    step()
        dstep.set_stream(stream)
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        gms = g0.elapsed_time(g1) / (reps * kGraphSteps)
        graph = {"value": bytes_step["total"] / (gms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": gms,
                 "steps_per_graph": kGraphSteps, "replays": reps}
        del g
        if pkv.check_status(status) != 0:
            raise SystemExit(f"device status {pkv.status_string(pkv.check_status(status))} in the graph replays")

    # end to end through the public API with host buffers: every step copies all
    # of its inputs host -> device (one pinned buffer holding them at 256-byte
    # aligned offsets, one copy) and reads its tokens back device -> host.
    # Pipelined (the reported value): the copies run on a second stream into two
    # device input buffers, so that the upload of step i + 1 overlaps the
    # kernels of step i.  Serial: the same copies on the compute stream.
    keys = [k for k, v in inp.items() if isinstance(v, torch.Tensor) and k not in ("k_cache", "v_cache")]
    nbytes = {k: inp[k].numel() * inp[k].element_size() for k in keys}
    offs, total = {}, 0
    for k in keys:
        offs[k] = total
        total += (nbytes[k] + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k in keys:
        host_buf[offs[k]:offs[k] + nbytes[k]].copy_(inp[k].contiguous().reshape(-1).view(torch.uint8).cpu())
    h2d = sum(nbytes.values())
    dbufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    dviews = [{k: b[offs[k]:offs[k] + nbytes[k]].view(inp[k].dtype).view(inp[k].shape) for k in keys} for b in dbufs]
    tok_host = [torch.empty(B, dtype=torch.int32).pin_memory() for _ in range(2)]
    cstream = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(10, min(args.steps, 200))

    vsteps = [make_step(d) for d in dviews]

    def run_views(j):
        vsteps[j].run()

    def e2e_step_pipelined(i):
        j = i & 1
        cstream.wait_event(free[j])             # step i - 2 is done with buffer j
        with torch.cuda.stream(cstream):
            dbufs[j].copy_(host_buf, non_blocking=True)
            ready[j].record(cstream)
        stream.wait_event(ready[j])
        run_views(j)
        free[j].record(stream)
        tok_host[j].copy_(tokens, non_blocking=True)

    def e2e_step_serial(i):
        dbufs[0].copy_(host_buf, non_blocking=True)
        run_views(0)
        tok_host[0].copy_(tokens, non_blocking=True)

    def time_e2e(fn):
        for j in range(2):
            free[j].record(stream)
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        _barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            fn(i)
        stream.wait_stream(cstream)
        e1.record(stream)
        torch.cuda.synchronize()
        return _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    e2e_ms = time_e2e(e2e_step_pipelined)
    e2e_serial_ms = time_e2e(e2e_step_serial)
    if pkv.check_status(status) != 0:
        raise SystemExit(f"device status {pkv.status_string(pkv.check_status(status))} in the end-to-end steps")
    if not all(torch.equal(t, tokens.cpu()) for t in tok_host):
        raise SystemExit("end-to-end tokens differ from the device-resident step")

    per_config = measure_per_config(pkv, dev) if world == 1 else None

    total_bytes = _sum_over_ranks(float(bytes_step["total"]), world, dev)
    value = total_bytes / (ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    attn_bytes = bytes_step["attention"] + bytes_step["append"]
    attn_gbs = attn_bytes / (attn_ms * 1e-3) / 1e9
    traffic = _traffic_per_launch()
    fast = True  # bf16, D=128, BS=16, Hkv=8: TMA/mma path -> main and combine kernels
    launches = args.steps * ((2 if fast else 2 + 1) + 1)  # attention with the append (+ combine) + sampler
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(w, inp, {
            "l2": f"no flush: every step reads {bytes_step['total'] / 1e6:.0f} MB (> 126 MB L2)",
            "parallelism": f"dp{world} (independent sequence shards, no collective)",
            "bytes_per_step": bytes_step}),
        "sampled_tokens_per_s": B * world / (ms * 1e-3),
        "pct_of_8TBps": value / 8000.0 * 100.0,
        "pct_of_measured_peak": value / peak * 100.0,
        "roofline": {"kernel": "paged_decode_attention_append (split-KV main with the KV append + combine "
                               "kernels), per call",
                     "bound": "hbm", "achieved": attn_gbs, "peak": peak, "unit": "GB/s",
                     "frac": attn_gbs / peak, "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic, "algorithmic_bytes_per_call": attn_bytes,
                     "ms_per_call": attn_ms},
        "e2e": {"value": total_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": B * 4,
                "mode": "pipelined: one pinned H2D copy per step on a copy stream, double-buffered, overlapping "
                        "the previous step's kernels; tokens D2H every step",
                "serial_ms_per_step": e2e_serial_ms,
                "serial_value": total_bytes / (e2e_serial_ms * 1e-3) / 1e9},
        "gpu_launches": launches,
        "graph": graph,
        "per_config": per_config,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ---------------------------------------------------------------- other configurations
def measure_per_config(pkv, dev, calls: int = 30):
    """The other workloads' hot calls, each timed with CUDA events on its stream
    around every call (median and mean of `calls` calls after 3 warm-up calls):
    the attention call with the append on the long-context (B 8, 64/8 heads,
    L 32K..128K) and fragmented batch-512 workloads, whose 2.7 GB and 1.2 GB of
    KV exceed L2, and the sampler alone on the batch-64, batch-512 and stress
    workloads with L2 flushed (a 256 MB write, then a 256 MB read) before every call.  Fractions are
    of the measured copy peak and of 8 TB/s."""
    peak, _ = _peaks()
    flush = _l2_flusher(dev)

    def stats(fn, flush_fn=None):
        t = _time_calls(fn, calls, flush=flush_fn)
        return t

    res = {}
    for num in (3, 4):
        w = W.workload(num)
        inp = W.make_decode_inputs(w, dev, with_logits=False)
        out = torch.empty_like(inp["q"])
        ws = torch.empty(pkv.decode_workspace_bytes(w.batch, w.n_q_heads, w.head_dim), dtype=torch.uint8,
                         device=dev)
        st = pkv.new_status(dev)
        sb = W.step_bytes(w, inp["seq_lens"])
        by = sb["attention"] + sb["append"]
        t = stats(lambda: pkv.paged_decode_attention_append(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                                            inp["v_cache"], inp["block_tables"], inp["seq_lens"],
                                                            out=out, workspace=ws, status=st))
        if pkv.check_status(st) != 0:
            raise SystemExit(f"device status {pkv.status_string(pkv.check_status(st))} on workload {w.name}")
        gbs = by / (t["median_us"] * 1e-6) / 1e9
        res[f"config{num}_attention"] = {
            "workload": w.name, "call": "paged_decode_attention_append", "algorithmic_bytes": by,
            "median_us": t["median_us"], "mean_us": t["mean_us"], "p90_us": t["p90_us"], "calls": calls,
            "GB/s": gbs, "frac_of_measured": gbs / peak, "frac_of_8TBps": gbs / 8000.0,
            "l2": "no flush: the call reads more than the 126 MB L2"}
        del inp, out, ws
        torch.cuda.empty_cache()
    for num in (2, 4, 5):
        w = W.workload(num)
        si = W.make_sampler_inputs(w, dev)
        tok = torch.empty(w.batch, dtype=torch.int32, device=dev)
        st = pkv.new_status(dev)
        t = stats(lambda: pkv.sample_tokens(si["logits"], si["temperature"], si["top_k"], si["top_p"], si["seeds"],
                                            si["offsets"], tokens=tok, status=st), flush)
        if pkv.check_status(st) != 0:
            raise SystemExit(f"device status {pkv.status_string(pkv.check_status(st))} on the sampler, {w.name}")
        by = 4 * w.batch * w.vocab + w.batch * 32
        gbs = by / (t["median_us"] * 1e-6) / 1e9
        res[f"config{num}_sampler"] = {
            "workload": f"{w.batch} x {w.vocab} logits ({w.name})", "call": "sample_tokens",
            "algorithmic_bytes": by, "median_us": t["median_us"], "mean_us": t["mean_us"], "p90_us": t["p90_us"],
            "calls": calls, "tokens_per_s": w.batch / (t["median_us"] * 1e-6), "GB/s": gbs,
            "frac_of_measured": gbs / peak, "frac_of_8TBps": gbs / 8000.0,
            "l2": "flushed before every call (256 MB write, then 256 MB read of another buffer, outside the events)"}
        del si
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- extra measurements
def _l2_flusher(dev):
    """L2 flush run before every timed call, outside the events: a 256 MB
    write (larger than the 126 MB L2), then a 256 MB read of another buffer, so
    that the dirty lines the write leaves are written back here rather than
    inside the next timed call."""
    wbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush():
        wbuf.fill_(1)
        rbuf.sum()
    return flush


def _time_calls(fn, n: int, flush=None):
    """Per-call device times (us) with CUDA events on the current stream; when
    `flush` is given it runs before every call, outside the events (L2 flush)."""
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    # a spin kernel ahead of the loop keeps the GPU busy while the host enqueues
    # every call, so no event pair spans host time
    torch.cuda._sleep(int(n * 400_000))
    for e0, e1 in ev:
        if flush is not None:
            flush()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    t = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev)
    return {"median_us": t[len(t) // 2], "mean_us": sum(t) / len(t), "p90_us": t[min(len(t) - 1, (9 * len(t)) // 10)],
            "n": n}


def run_extras(args):
    """One JSON line per extra measurement (not part of the default bench line):
    attention calls on the batch-64, long-context and fragmented workloads, the
    sampler alone on its three workloads (L2 flushed between calls), the sampler
    variants (min-p, typical sampling, logits processors), speculative
    verification, chunked prefill, block copies, and attention over forked
    sequences that share prefix blocks."""
    import numpy as np
    import paged_kv_decode_table_gb300 as pkv
    from paged_kv_decode_table_gb300 import build as pkv_build
    pkv_build.build()
    pkv.load_library()
    peak, _ = _peaks()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = _l2_flusher(dev)
    clocks = ClockSampler(0)
    clocks.start()

    def emit(d):
        print(json.dumps(d), flush=True)

    for num in (2, 3, 4):
        w = W.workload(num)
        inp = W.make_decode_inputs(w, dev, with_logits=False)
        out = torch.empty_like(inp["q"])
        ws = torch.empty(pkv.decode_workspace_bytes(w.batch, w.n_q_heads, w.head_dim), dtype=torch.uint8,
                         device=dev)
        by = W.step_bytes(w, inp["seq_lens"])["attention"]
        t = _time_calls(lambda: pkv.paged_decode_attention(inp["q"], inp["k_cache"], inp["v_cache"],
                                                           inp["block_tables"], inp["seq_lens"], out=out,
                                                           workspace=ws), 50)
        gbs = by / (t["median_us"] * 1e-6) / 1e9
        emit({"extra": "paged_decode_attention", "workload": w.name, "bytes": by, **t, "GB/s": gbs,
              "frac_of_measured": gbs / peak, "frac_of_8TBps": gbs / 8000.0})
        del inp, out, ws
        torch.cuda.empty_cache()

    for num, label, topk in ((2, "T0.7 k50 p0.9", None), (4, "T1.0 p0.95", None), (4, "T1.0 k50 p0.95", 50),
                             (5, "stress: mixed T / k / p", None)):
        w = W.workload(num)
        si = W.make_sampler_inputs(w, dev)
        if topk is not None:
            si["top_k"].fill_(topk)
        tok = torch.empty(w.batch, dtype=torch.int32, device=dev)
        t = _time_calls(lambda: pkv.sample_tokens(si["logits"], si["temperature"], si["top_k"], si["top_p"],
                                                  si["seeds"], si["offsets"], tokens=tok), 50, flush=flush)
        by = 4 * w.batch * w.vocab
        emit({"extra": "sample_tokens", "workload": f"{w.batch}x{w.vocab} {label}", **t,
              "tokens_per_s": w.batch / (t["median_us"] * 1e-6), "logits_GB/s": by / (t["median_us"] * 1e-6) / 1e9,
              "frac_of_measured": by / (t["median_us"] * 1e-6) / 1e9 / peak})
        del si
        torch.cuda.empty_cache()

    # sampler variants on the batch-64 logits: min-p after top-p, typical sampling,
    # and the logits processors (constraint masks on every row, 200 penalised
    # tokens per row)
    w = W.workload(2)
    si = W.make_sampler_inputs(w, dev)
    tok = torch.empty(w.batch, dtype=torch.int32, device=dev)
    by = 4 * w.batch * w.vocab
    mp = torch.full((w.batch,), 0.05, dtype=torch.float32, device=dev)
    t = _time_calls(lambda: pkv.sample_tokens(si["logits"], si["temperature"], si["top_k"], si["top_p"], si["seeds"],
                                              si["offsets"], tokens=tok, min_p=mp), 50, flush=flush)
    emit({"extra": "sample_tokens_min_p", "workload": f"{w.batch}x{w.vocab} T0.7 k50 p0.9 min_p0.05", **t,
          "tokens_per_s": w.batch / (t["median_us"] * 1e-6), "logits_GB/s": by / (t["median_us"] * 1e-6) / 1e9,
          "frac_of_measured": by / (t["median_us"] * 1e-6) / 1e9 / peak})
    for tpv in (0.9, 0.2):
        tpt = torch.full((w.batch,), tpv, dtype=torch.float32, device=dev)
        t = _time_calls(lambda: pkv.sample_tokens_typical(si["logits"], si["temperature"], tpt, si["seeds"],
                                                          si["offsets"], tokens=tok), 20, flush=flush)
        emit({"extra": "sample_tokens_typical", "workload": f"{w.batch}x{w.vocab} T0.7 typical_p {tpv}", **t,
              "tokens_per_s": w.batch / (t["median_us"] * 1e-6), "logits_GB/s": by / (t["median_us"] * 1e-6) / 1e9,
              "frac_of_measured": by / (t["median_us"] * 1e-6) / 1e9 / peak})
    rng = np.random.default_rng(3)
    words = (w.vocab + 31) // 32
    mask = torch.from_numpy(rng.integers(0, 2**32, (w.batch, words), dtype=np.uint64).astype(np.uint32).view(np.int32)).to(dev)
    npen = 200
    toks = torch.from_numpy(np.concatenate([rng.choice(w.vocab, npen, replace=False) for _ in range(w.batch)]).astype(np.int32)).to(dev)
    cnts = torch.from_numpy(rng.integers(1, 6, w.batch * npen).astype(np.int32)).to(dev)
    rp = torch.arange(0, w.batch * npen + 1, npen, dtype=torch.int32, device=dev)
    rep = torch.full((w.batch,), 1.2, dtype=torch.float32, device=dev)
    frq = torch.full((w.batch,), 0.3, dtype=torch.float32, device=dev)
    prs = torch.full((w.batch,), 0.2, dtype=torch.float32, device=dev)
    lg = si["logits"].clone()
    t = _time_calls(lambda: pkv.apply_logits_processors(lg, allow_mask=mask, row_ptr=rp, tokens=toks, counts=cnts,
                                                        repetition=rep, frequency=frq, presence=prs), 50, flush=flush)
    pby = w.batch * words * 4 + w.batch * w.vocab // 2 * 4 + w.batch * npen * 16   # mask, ~half the row banned, lists
    emit({"extra": "apply_logits_processors", "workload": f"{w.batch}x{w.vocab}, random masks, {npen} penalised "
          f"tokens per row", "bytes": pby, **t, "GB/s": pby / (t["median_us"] * 1e-6) / 1e9,
          "frac_of_measured": pby / (t["median_us"] * 1e-6) / 1e9 / peak})
    del si, lg, mask
    torch.cuda.empty_cache()

    # speculative verification: 64 requests, 4 drafts each, 128256-token vocabulary
    B, gamma, V = 64, 4, 128256
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    tgt = torch.randn((B, gamma + 1, V), generator=g, device=dev) * 2.0
    drf = (tgt[:, :gamma] + 0.5 * torch.randn((B, gamma, V), generator=g, device=dev)).contiguous()
    x = torch.topk(drf, 4, dim=2).indices[..., 1].to(torch.int32).contiguous()
    seq = torch.full((B,), 2048, dtype=torch.int32, device=dev)
    temp = torch.full((B,), 0.8, dtype=torch.float32, device=dev)
    sd = torch.arange(B, dtype=torch.int64, device=dev)
    off = torch.zeros(B, dtype=torch.int64, device=dev)
    wsv = torch.empty(pkv.spec_verify_workspace_bytes(B, gamma), dtype=torch.uint8, device=dev)
    t = _time_calls(lambda: pkv.spec_verify(tgt, drf, x, seq, temp, sd, off, workspace=wsv), 50, flush=flush)
    _, nacc, _ = pkv.spec_verify(tgt, drf, x, seq, temp, sd, off, workspace=wsv)
    emitted = int(nacc.sum()) + B
    by = B * (2 * gamma + 1) * V * 4
    emit({"extra": "spec_verify", "workload": f"{B} requests x {gamma} drafts, V {V}, T 0.8", "bytes": by, **t,
          "GB/s": by / (t["median_us"] * 1e-6) / 1e9, "frac_of_measured": by / (t["median_us"] * 1e-6) / 1e9 / peak,
          "accepted_drafts": int(nacc.sum()), "emitted_tokens_per_s": emitted / (t["median_us"] * 1e-6)})
    del tgt, drf
    torch.cuda.empty_cache()

    # chunked prefill: 16 sequences, a 512-token chunk each after a 1024..4096-token prefix
    Bp, chunk, Hq, Hkv_p, Dp, BSp = 16, 512, 32, 8, 128, 16
    gen = torch.Generator().manual_seed(5)
    prefix = torch.randint(1024, 4097, (Bp,), generator=gen)
    Lp = (prefix + chunk).to(torch.int32)
    nbp = (Lp + BSp - 1) // BSp
    NBp = int(nbp.sum())
    permp = torch.randperm(NBp, generator=gen).to(torch.int32)
    MBp = int(nbp.max())
    btp = torch.full((Bp, MBp), -1, dtype=torch.int32)
    o = 0
    for b in range(Bp):
        btp[b, :nbp[b]] = permp[o:o + int(nbp[b])]
        o += int(nbp[b])
    Kp = torch.randn((NBp, Hkv_p, BSp, Dp), device=dev).to(torch.bfloat16)
    Vp = torch.randn((NBp, Hkv_p, BSp, Dp), device=dev).to(torch.bfloat16)
    qp = torch.randn((Bp * chunk, Hq, Dp), device=dev).to(torch.bfloat16)
    qs = torch.arange(0, Bp * chunk + 1, chunk, dtype=torch.int32, device=dev)
    btp, Lpd = btp.to(dev), Lp.to(dev)
    outp = torch.empty_like(qp)
    t = _time_calls(lambda: pkv.paged_prefill_attention(qp, Kp, Vp, btp, Lpd, qs, out=outp), 20, flush=flush)
    # causal pairs: token i of a chunk sees prefix + i + 1 positions
    pairs = sum(int(prefix[b]) * chunk + chunk * (chunk + 1) // 2 for b in range(Bp))
    flops = 4 * Hq * Dp * pairs
    kv_bytes = int(Lp.sum()) * Hkv_p * Dp * 2 * 2
    tf = flops / (t["median_us"] * 1e-6) / 1e12
    emit({"extra": "paged_prefill_attention", "workload": f"{Bp} x {chunk}-token chunks, prefix 1024..4096, "
          f"{Hq}q/{Hkv_p}kv, D {Dp}", "flops": flops, "kv_bytes": kv_bytes, **t, "TFLOP/s": tf,
          "frac_of_bf16_dense": tf / _bf16_peak(), "kv_GB/s": kv_bytes / (t["median_us"] * 1e-6) / 1e9})
    del Kp, Vp, qp, outp
    torch.cuda.empty_cache()

    # copy-on-write block copies: 1024 pairs of 64 KB blocks (bf16, 8 KV heads, 16 slots, D 128)
    NB, Hkv, BS, D = 4096, 8, 16, 128
    K = torch.randn((NB, Hkv, BS, D), device=dev).to(torch.bfloat16)
    V = torch.randn((NB, Hkv, BS, D), device=dev).to(torch.bfloat16)
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(1)).to(torch.int32)
    src, dst = perm[:1024].to(dev), perm[1024:2048].to(dev)
    t = _time_calls(lambda: pkv.copy_blocks(K, V, src, dst), 50, flush=flush)
    by = 1024 * 2 * 2 * Hkv * BS * D * 2   # pools x (read + write) per pair
    emit({"extra": "copy_blocks", "pairs": 1024, "block_bytes_per_pool": Hkv * BS * D * 2, "bytes": by, **t,
          "GB/s": by / (t["median_us"] * 1e-6) / 1e9, "frac_of_measured": by / (t["median_us"] * 1e-6) / 1e9 / peak})
    del K, V
    torch.cuda.empty_cache()

    # forked sequences: 4 prompts of 2048..4096 tokens, 16 branches each, one decode step
    # in; attention reads each shared prompt block once from HBM and 15 more times from L2
    gen = torch.Generator().manual_seed(77)
    lens = torch.randint(2048, 4097, (4,), generator=gen).tolist()
    Hq = 32
    MB = 4200 // BS
    NB = sum(-(-L // BS) for L in lens) + 4 * 16 * 2 + 8
    pool = pkv.BlockPool(NB, BS, MB)
    K = torch.randn((NB, Hkv, BS, D), device=dev).to(torch.bfloat16)
    V = torch.randn((NB, Hkv, BS, D), device=dev).to(torch.bfloat16)
    kids = []
    for p, L in enumerate(lens):
        pool.add(1000 + p, L)
        for c in range(16):
            pool.fork(1000 + p, p * 16 + c)
            kids.append(p * 16 + c)
        pool.free(1000 + p)
    pairs = [x for x in (pool.append(s) for s in kids) if x is not None]
    if pairs:
        pkv.copy_blocks(K, V, torch.tensor([x[0] for x in pairs], dtype=torch.int32, device=dev),
                        torch.tensor([x[1] for x in pairs], dtype=torch.int32, device=dev))
    bt, sl = pool.tables(kids)
    bt, sl = bt.to(dev), sl.to(dev)
    q = torch.randn((len(kids), Hq, D), device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    t = _time_calls(lambda: pkv.paged_decode_attention(q, K, V, bt, sl, out=out), 50, flush=flush)
    logical = int(sl.sum()) * Hkv * D * 2 * 2
    unique = (NB - pool.num_free()) * Hkv * BS * D * 2 * 2
    emit({"extra": "paged_decode_attention_forked", "workload": f"4 prompts x 16 branches, lengths {lens}",
          "logical_kv_bytes": logical, "unique_kv_bytes": unique, **t,
          "logical_GB/s": logical / (t["median_us"] * 1e-6) / 1e9,
          "unique_GB/s": unique / (t["median_us"] * 1e-6) / 1e9, "cow_pairs": len(pairs)})
    emit({"extra": "clocks", "over": "every measurement above", **clocks.stop()})
    return 0


def run_spec_case(args):
    """The speculative-verification case its profile is captured on (the
    extras workload: 64 requests, 4 drafts each, 128256-token vocabulary,
    T 0.8); `--warmup` untimed calls, then `--steps` timed ones, L2 flushed
    before every call (CUDA events on the stream around each call)."""
    import paged_kv_decode_table_gb300 as pkv
    from paged_kv_decode_table_gb300 import build as pkv_build
    pkv_build.build()
    pkv.load_library()
    dev = torch.device("cuda", 0)
    B, gamma, V = 64, 4, 128256
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    tgt = torch.randn((B, gamma + 1, V), generator=g, device=dev) * 2.0
    drf = (tgt[:, :gamma] + 0.5 * torch.randn((B, gamma, V), generator=g, device=dev)).contiguous()
    x = torch.topk(drf, 4, dim=2).indices[..., 1].to(torch.int32).contiguous()
    seq = torch.full((B,), 2048, dtype=torch.int32, device=dev)
    temp = torch.full((B,), 0.8, dtype=torch.float32, device=dev)
    sd = torch.arange(B, dtype=torch.int64, device=dev)
    off = torch.zeros(B, dtype=torch.int64, device=dev)
    wsv = torch.empty(pkv.spec_verify_workspace_bytes(B, gamma), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    st = pkv.new_status()
    for _ in range(args.warmup):
        flush.zero_()
        pkv.spec_verify(tgt, drf, x, seq, temp, sd, off, workspace=wsv, status=st)
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkv.spec_verify(tgt, drf, x, seq, temp, sd, off, workspace=wsv, status=st)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1000)
    assert pkv.check_status(st) == 0
    print(json.dumps({"case": f"speculative verification {B} requests x {gamma} drafts, V {V}", "calls": args.steps,
                      "median_us": statistics.median(times) if times else None}))
    return 0


def run_typical_case(args):
    """The typical-sampling case the typical sampler profile is captured on: the
    sampler rows of the batch-64 GQA workload (64 x 128256 logits, T 0.7) with
    typical_p 0.9; `--warmup` untimed calls, then `--steps` timed ones (CUDA
    events on the stream, logits resident in L2 after the first call)."""
    import paged_kv_decode_table_gb300 as pkv
    from paged_kv_decode_table_gb300 import build as pkv_build
    pkv_build.build()
    pkv.load_library()
    dev = torch.device("cuda", 0)
    w = W.workload(2)
    si = W.make_sampler_inputs(w, dev)
    tok = torch.empty(w.batch, dtype=torch.int32, device=dev)
    tpt = torch.full((w.batch,), 0.9, dtype=torch.float32, device=dev)
    st = pkv.new_status()
    for _ in range(args.warmup):
        pkv.sample_tokens_typical(si["logits"], si["temperature"], tpt, si["seeds"], si["offsets"], tokens=tok, status=st)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        pkv.sample_tokens_typical(si["logits"], si["temperature"], tpt, si["seeds"], si["offsets"], tokens=tok, status=st)
    e1.record()
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    print(json.dumps({"case": f"typical sampling {w.batch} x {w.vocab}, T 0.7, typical_p 0.9", "calls": args.steps,
                      "us_per_call": e0.elapsed_time(e1) / max(1, args.steps) * 1000}))
    return 0


def run_sampler_case(args):
    """The sampler case its profiles are captured on: sample_tokens alone on the
    logits of workload `--sampler-case` (2: 64 x 128256, T 0.7, top-k 50,
    top-p 0.9; 4: 512 x 32000, T 1, top-p 0.95; 5: the 256 x 152064 stress
    rows; `--sampler-top-k K` sets every row's top-k to K); `--warmup` untimed
    calls, then `--steps` timed ones (CUDA events on the stream; the logits
    stay in L2 between calls when they fit)."""
    import paged_kv_decode_table_gb300 as pkv
    from paged_kv_decode_table_gb300 import build as pkv_build
    pkv_build.build()
    pkv.load_library()
    dev = torch.device("cuda", 0)
    w = W.workload(args.sampler_case)
    si = W.make_sampler_inputs(w, dev)
    if args.sampler_top_k is not None:
        si["top_k"].fill_(args.sampler_top_k)
    tok = torch.empty(w.batch, dtype=torch.int32, device=dev)
    st = pkv.new_status()
    call = lambda: pkv.sample_tokens(si["logits"], si["temperature"], si["top_k"], si["top_p"], si["seeds"],
                                     si["offsets"], tokens=tok, status=st)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    topk = "" if args.sampler_top_k is None else f", top-k {args.sampler_top_k}"
    print(json.dumps({"case": f"sample_tokens {w.batch} x {w.vocab} ({w.name}){topk}", "calls": args.steps,
                      "us_per_call": e0.elapsed_time(e1) / max(1, args.steps) * 1000}))
    return 0


def run_prefill_case(args):
    """The chunked-prefill case the prefill profile is captured on:
    `--prefill-seqs` sequences (default 4) with a 512-token chunk each after a
    1024..4096-token prefix, 32 query / 8 KV heads, D 128, block 16, bf16;
    `--warmup` untimed calls, then `--steps` timed ones (CUDA events on the
    stream)."""
    import paged_kv_decode_table_gb300 as pkv
    from paged_kv_decode_table_gb300 import build as pkv_build
    pkv_build.build()
    pkv.load_library()
    dev = torch.device("cuda", 0)
    Bp, chunk, Hq, Hkv, D, BS = args.prefill_seqs, 512, 32, 8, 128, 16
    gen = torch.Generator().manual_seed(5)
    prefix = torch.randint(1024, 4097, (Bp,), generator=gen)
    L = (prefix + chunk).to(torch.int32)
    nb = (L + BS - 1) // BS
    NB = int(nb.sum())
    perm = torch.randperm(NB, generator=gen).to(torch.int32)
    bt = torch.full((Bp, int(nb.max())), -1, dtype=torch.int32)
    o = 0
    for b in range(Bp):
        bt[b, :nb[b]] = perm[o:o + int(nb[b])]
        o += int(nb[b])
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    K = torch.randn((NB, Hkv, BS, D), generator=g, device=dev).to(torch.bfloat16)
    V = torch.randn((NB, Hkv, BS, D), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((Bp * chunk, Hq, D), generator=g, device=dev).to(torch.bfloat16)
    qs = torch.arange(0, Bp * chunk + 1, chunk, dtype=torch.int32, device=dev)
    bt, L = bt.to(dev), L.to(dev)
    out = torch.empty_like(q)
    st = pkv.new_status()
    for _ in range(args.warmup):
        pkv.paged_prefill_attention(q, K, V, bt, L, qs, out=out, status=st)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        pkv.paged_prefill_attention(q, K, V, bt, L, qs, out=out, status=st)
    e1.record()
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    print(json.dumps({"case": f"prefill {Bp} x 512-token chunks", "calls": args.steps,
                      "us_per_call": e0.elapsed_time(e1) / max(1, args.steps) * 1000}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extras", action="store_true",
                    help="print extra measurement lines (other workloads, sampler alone, block copies)")
    ap.add_argument("--prefill-case", action="store_true",
                    help="time the small chunked-prefill case of the prefill profile (--warmup, --steps calls)")
    ap.add_argument("--prefill-seqs", type=int, default=4, help="sequences of the --prefill-case workload")
    ap.add_argument("--spec-case", action="store_true",
                    help="time the speculative-verification case of its profile (--warmup, --steps calls)")
    ap.add_argument("--typical-case", action="store_true",
                    help="time the typical-sampling case of the typical sampler profile (--warmup, --steps calls)")
    ap.add_argument("--sampler-case", type=int, default=0, choices=[0, 2, 4, 5],
                    help="time sample_tokens alone on the logits of workload 2, 4 or 5 (--warmup, --steps calls)")
    ap.add_argument("--sampler-top-k", type=int, default=None, help="with --sampler-case: every row's top-k")
    args = ap.parse_args()
    if args.sampler_case:
        return run_sampler_case(args)
    if args.prefill_case:
        return run_prefill_case(args)
    if args.typical_case:
        return run_typical_case(args)
    if args.spec_case:
        return run_spec_case(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.extras:
        return run_extras(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
