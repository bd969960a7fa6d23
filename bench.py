#!/usr/bin/env python3
"""Benchmark of libkda on one GB300 (or N replicas, one per GPU).

One step = one ``kda_chunk_fwd`` over the long-context prefill workload: one
sequence of 1,048,576 tokens x 32 heads, d_k = d_v = 128, chunk 64, bf16
q/k/v, fp32 gates (log_alpha = -softplus(N(-6, 1))) and state, drawn on the
device with a seeded generator -- every prefill stage of the hot path (chunk
table, prep, state scan, outputs), the largest single-GPU workload named for
this path.  Its inputs (51.7 GB) dwarf the 129 MB L2, so no flush is needed.

Timing: CUDA events on the launch stream, W untimed warm-up calls, about
0.3 s of back-to-back calls (--preroll; the first call after an idle gap runs
slower while the clocks come back), then K timed calls, barrier and
synchronize on both sides, max over ranks.  libkda itself records events
between its kernels (kda_chunk_fwd_ws_timed, which runs them one after
another) for the per-kernel device times behind the roofline figures, which
take the method's algorithmic bytes and flops per (token, head); the engine's
own scratch traffic is reported apart.  The end-to-end figure goes through
kda_chunk_fwd_host (page-locked host buffers, copies in and out inside the
timed region).

Extra rows in the same line: the single-head-group prefill (H=16, T=4096,
L2 flushed before each step), the packed 32-sequence prefill with its
backward, K3-range gates, the fused prologue and value-head groups, the
backward of the head-group workload, the decode step (256 sequences x 32
heads, 512 MiB state, 64 steps), the multi-token recurrent pass and the
short convolution.

``--impl reference`` times the fp64 CPU oracle (the reference arm of this
repository) on a bounded sample of the same workload on the host cores;
``--impl reference --sweep`` times it on every named workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s & % bf16 tensor peak; decode state GB/s % of HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--engine", choices=["auto", "tensor", "simt"], default="auto")
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--preroll", type=float, default=0.3,
                    help="seconds of back-to-back steps before each timed loop (0: none, "
                         "for profiler runs)")
    ap.add_argument("--profile", choices=["prefill", "backward", "backward_recurrent", "decode",
                                          "recurrent", "conv"],
                    default=None,
                    help="run only one small case, --warmup + --steps plain calls and nothing "
                         "else (for counter captures): the single-head-group prefill, its "
                         "chunk-form or recurrent-form backward, the decode step (256 x 32 "
                         "heads), the 8-token multi-token pass, or the short convolution")
    ap.add_argument("--sweep", action="store_true",
                    help="with --impl reference: time the oracle on every named workload "
                         "(one JSON line each)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained",
                                                     p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no data-path collective)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int = 0):
        self.proc = None
        self.dev = device_index
        self.out_path = None

    def start(self):
        import tempfile
        try:
            fd, self.out_path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            uuid = self._uuid()
            if uuid:
                cmd += ["-i", uuid]
            self.fh = open(self.out_path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def _uuid(self):
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.dev).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.out_path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out_path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# algorithmic work per (token, head): the figures behind the roofline
# ---------------------------------------------------------------------------

def path_bytes_per_tok_head(d: int) -> int:
    """Whole-path minimum: q, k, v, out (bf16) and log_alpha (fp32) once, beta."""
    return 4 * 2 * d + 4 * d + 4


def prefill_flops_per_tok_head(d: int, C: int) -> int:
    """Dense chunk contractions: K K^T, Q K^T, A^kk (beta V), A^kk (beta Gamma K),
    A^qk E (5 x 2Cd) plus W S, K_end^T E, Q_hat S (3 x 2d^2)."""
    return 10 * C * d + 6 * d * d


# The method's algorithmic work per (token, head) at d = 128, C = 64 (the
# roofline's numerators): q, k, v, out in bf16, log_alpha in fp32 and beta read
# or written once, and the dense chunk contractions.
PATH_BYTES = path_bytes_per_tok_head(128)
PATH_FLOPS = prefill_flops_per_tok_head(128, 64)
# The tensor-core engine's own scratch traffic per (token, head) of each
# kernel, beyond the method's bytes: the prep writes one 74,496-byte image per
# (chunk, head) (-M', P', Q', Z in f16, Gamma_last and beta); the scan reads
# its 48 KB -M'/P' part once per 64-wide value tile and writes the chunk's
# state (f16, 32 KB); the output pass reads Q' and Z (24 KB) and the
# state (32 KB).  Per token: divide by the chunk's 64 tokens.
SCRATCH_BYTES = {"prep": 74496 / 64, "scan": (2 * 49152 + 32768) / 64,
                 "out": (24576 + 32768) / 64}

PROFILE_FILES = {
    "prep": ("chunk_prep_prefill_T4096_H16.md", 4096 * 16),
    "scan": ("chunk_scan_prefill_T4096_H16.md", 4096 * 16),
    "out": ("chunk_out_prefill_T4096_H16.md", 4096 * 16),
    "recurrent_step": ("recurrent_step_decode_256x32_d128.md", None),
    "recurrent_fwd": ("recurrent_fwd_decode_256x32x8_d128.md", None),
    "short_conv_fwd": ("short_conv_fwd_prefill_C12288_T4096.md", None),
    "recurrent_bwd": ("recurrent_bwd_prefill_T4096_H16.md", None),
    # the chunk-form backward's own kernels, captured on its benchmark workload
    "chunk_bwd_aux": ("chunk_bwd_aux_T4096_H16.md", None),
    "chunk_rscan": ("chunk_rscan_T4096_H16.md", None),
    "chunk_grad_g1": ("chunk_grad_g1_T4096_H16.md", None),
    "chunk_grad_g2": ("chunk_grad_g2_T4096_H16.md", None),
}


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, or None when there is none or the kernel's source has
    changed since the counters were taken (source hash recorded alongside)."""
    import hashlib
    name = PROFILE_FILES.get(kernel, (None, None))[0]
    if not name:
        return None
    path = os.path.join(ROOT, "profiles", name)
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.split(":", 1)[0] in ("source_sha256", "dram_bytes_per_launch"):
                    k, val = line.split(":", 1)
                    fields[k] = val.strip()
        digest, srcs = fields["source_sha256"].split("  ", 1)
        srcs = srcs.strip("() ").split(" + ")
        h = hashlib.sha256()
        for src in srcs:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != digest:
            return None
        return int(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def profiled_traffic_scaled(kernel: str, units: int):
    """profiled_traffic scaled to a launch of `units` (token, head) pairs: the
    prefill kernels' summaries come from the single-head-group workload (the
    full-size workloads are too large for a counter capture), and their traffic
    grows in proportion to the (chunk, head) items.  Returns (bytes, note)."""
    t = profiled_traffic(kernel)
    base = PROFILE_FILES.get(kernel, (None, None))[1]
    if t is None or not base:
        return t, None
    if units == base:
        return t, "ncu capture of this workload"
    return (int(round(t * units / base)),
            f"ncu capture at {base} (token, head) units, scaled by {units / base:g}")


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on host cores
# ---------------------------------------------------------------------------

def oracle_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


PREROLL_SECONDS = 0.3


def preroll(step, seconds: float = None):
    """Runs `step` back to back for about `seconds` (default --preroll) so that
    the timed loop that follows starts on a GPU in its loaded state: the first
    call after an idle gap runs at about half speed while the clocks come
    back up."""
    import torch
    if seconds is None:
        seconds = PREROLL_SECONDS
    seconds = min(seconds, PREROLL_SECONDS)
    if seconds <= 0:
        return
    t0 = time.time()
    while time.time() - t0 < seconds:
        for _ in range(16):
            step()
        torch.cuda.synchronize()


REF_SAMPLE_TOKENS = 2048  # reference arm: first tokens of the long-context recipe per step


def run_reference(args, dist: Dist):
    """The oracle, as it stands, on the host cores: each step is the fp64 token
    recurrence over a bounded sample of the headline workload (its first
    REF_SAMPLE_TOKENS tokens x 32 heads, drawn on the host with the same
    recipe), so the whole --steps/--warmup run stays within a few minutes."""
    if dist.rank != 0:
        return
    import oracle
    from kimi_delta_attention_chunkwise_gb300 import inputs
    Ts = REF_SAMPLE_TOKENS
    w = inputs.long_context_prefix(Ts)
    arrs = [w.q, w.k, w.v, w.log_alpha, w.beta]
    oracle.build()
    thr = oracle_threads()
    for _ in range(args.warmup):
        oracle.recurrent(*arrs, w.scale, None, [0, Ts], threads=thr)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.recurrent(*arrs, w.scale, None, [0, Ts], threads=thr)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = Ts * args.steps / total
    sample = (f"first {Ts} of 1048576 tokens x {w.H} heads of the long-context workload per "
              "step (host-drawn, same recipe), fp64 token recurrence")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "long_context_T1048576_H32_d128: B=1, one sequence of 1048576 "
                               "tokens x 32 heads, d_k=d_v=128, chunk 64, bf16 q/k/v, fp32 "
                               "log_alpha = -softplus(N(-6,1)), zero initial state, seeded",
                   "sample_tokens": Ts},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_sweep(args, dist: Dist):
    """The oracle, as it stands, on each named workload (host cores): the
    tiny fp32 one, the head-group prefill (all cores and one core), the
    packed 32-sequence batch, the 1M-token recipe's first 8,192 tokens and
    the 64 decode steps of 256 sequences x 32 heads.  One JSON line each."""
    if dist.rank != 0:
        return
    import numpy as np
    import oracle
    from kimi_delta_attention_chunkwise_gb300 import inputs
    oracle.build()
    thr = oracle_threads()

    def decode_as_prefill():
        dw = inputs.batched_decode()
        steps, N, H, d = dw.q.shape
        # sequence n's 64 steps as one 64-token sequence: [N * steps, H, d]
        seqs = lambda a: np.ascontiguousarray(np.swapaxes(a, 0, 1)).reshape((N * steps,) + a.shape[2:])
        cu = np.arange(0, N * steps + 1, steps, dtype=np.int32)
        return (dw.name, seqs(dw.q), seqs(dw.k), seqs(dw.v), seqs(dw.log_alpha), seqs(dw.beta),
                dw.scale, dw.initial_state, cu, N)

    def prefill(w, name=None):
        return (name or w.name, w.q, w.k, w.v, w.log_alpha, w.beta, w.scale, w.initial_state,
                w.cu_seqlens, len(w.cu_seqlens) - 1)

    jobs = [(lambda: prefill(inputs.tiny_f32()), thr),
            (lambda: prefill(inputs.head_group_prefill()), thr),
            (lambda: prefill(inputs.head_group_prefill()), 1),
            (lambda: prefill(inputs.varlen_prefill()), thr),
            (lambda: prefill(inputs.long_context_prefix(8192)), thr),
            (decode_as_prefill, thr)]
    for make, cores in jobs:
        name, q, k, v, la, b, scale, s0, cu, n_seqs = make()
        T, H = q.shape[0], q.shape[1]
        t0 = time.perf_counter()
        oracle.recurrent(q, k, v, la, b, scale, s0, cu, threads=cores)
        sec = time.perf_counter() - t0
        print(json.dumps({"sweep": name, "impl": "reference", "kind": "oracle",
                          "cores": cores, "sequences": n_seqs, "tokens": T, "heads": H,
                          "seconds": sec, "tok_heads_per_s": T * H / sec,
                          "tokens_per_s": T / sec, "precision": "f64"}), flush=True)
        del q, k, v, la, b, s0


def cpu_baseline():
    """The oracle as it stands on the headline workload's 8,192-token
    checkpoint prefix (all 32 heads, host-drawn with the same recipe),
    repeated to about 10 s of wall time (at most 40 runs)."""
    import oracle
    from kimi_delta_attention_chunkwise_gb300 import inputs
    oracle.build()
    thr = oracle_threads()
    w = inputs.long_context_prefix(8192)
    runs, t_total = 0, 0.0
    while runs < 40 and (t_total < 10.0 or runs == 0):
        t0 = time.perf_counter()
        oracle.recurrent(w.q, w.k, w.v, w.log_alpha, w.beta, w.scale, None, w.cu_seqlens,
                         threads=thr)
        t_total += time.perf_counter() - t0
        runs += 1
    return {"value": w.T * runs / t_total, "unit": "tokens/s", "cores": thr, "kind": "oracle",
            "sample": f"the headline workload's first {w.T} tokens x {w.H} heads (its parity "
                      f"checkpoint; host-drawn, same recipe) x {runs} run(s), fp64 token "
                      f"recurrence, {t_total:.1f} s"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def timed_loop(call, steps, stream, dist, flush=None):
    """`steps` calls, each bracketed by CUDA events on the launch stream (an L2
    flush before each when `flush` is given, outside the events); barrier and
    synchronize on both sides.  Returns (total ms, max over ranks; per-step ms)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    dist.barrier()
    torch.cuda.synchronize()
    for a, b in evs:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    per = [a.elapsed_time(b) for a, b in evs]
    return dist.max(sum(per)), per


def stage_times(timed_call, reps, flush=None):
    """Per-kernel device times (ms) of the tensor-core engine, averaged over
    `reps` calls of kda_chunk_fwd_ws_timed (library-recorded events between
    its kernels, which runs them one after another)."""
    import torch
    names = ["chunk_table", "prep", "scan", "out"]
    acc = None
    for _ in range(reps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
        for e in evs:
            e.record()
        if flush is not None:
            flush.zero_()
        n_rec = timed_call(evs)
        torch.cuda.synchronize()
        n = max(0, n_rec - 1)
        t = [evs[j].elapsed_time(evs[j + 1]) for j in range(n)]
        acc = t if acc is None else [x + y for x, y in zip(acc, t)]
    acc = [x / reps for x in (acc or [])]
    if len(acc) == 4:
        return dict(zip(names, acc))
    return {f"stage{j}": x for j, x in enumerate(acc)}


def prefill_roofline(stages, units, call_ms, peaks, traffic=None, traffic_note=None):
    """The roofline of one prefill launch: the dominant kernel's event time
    against the method's algorithmic work for the units the launch processes
    (PATH_BYTES and the dense-contraction flops per (token, head)), with the
    whole call's figures beside it; the engine's own scratch traffic of that
    kernel is reported apart (overhead_bytes)."""
    dom = max(stages, key=stages.get)
    t = stages[dom] / 1e3
    alg_bytes = PATH_BYTES * units
    alg_flops = PATH_FLOPS * units
    achieved = alg_bytes / t / 1e9
    return {
        "kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
        "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
        "traffic_note": traffic_note, "peak_source": peaks["source"],
        "algorithmic_bytes_per_launch": alg_bytes, "launch_ms": stages[dom],
        "overhead_bytes": SCRATCH_BYTES.get(dom, 0) * units,
        "overhead_note": "the engine's own scratch traffic of this kernel (images, states), "
                         "not part of the algorithmic bytes",
        "tensor_tflops": alg_flops / t / 1e12,
        "tensor_frac": alg_flops / t / 1e12 / peaks["bf16_tflops"],
        "whole_call": {"ms": call_ms, "gbs": alg_bytes / (call_ms / 1e3) / 1e9,
                       "frac": alg_bytes / (call_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                       "tflops": alg_flops / (call_ms / 1e3) / 1e12,
                       "tensor_frac": alg_flops / (call_ms / 1e3) / 1e12
                       / peaks["bf16_tflops"]},
    }


def run_ours(args, dist: Dist):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import build, inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(dist.local_rank)
    build.build()
    peaks = load_peaks()
    dev = torch.device("cuda", dist.local_rank)
    stream = torch.cuda.current_stream()

    # ---------------- the headline: one 1,048,576-token sequence x 32 heads ----------------
    x = inputs.long_context_device(device=str(dev))
    q, k, v, la, beta, cu = (x[n] for n in ("q", "k", "v", "log_alpha", "beta", "cu_seqlens"))
    scale = x["scale"]
    T, H, d = q.shape
    C = 64
    units = T * H
    out = torch.empty_like(q)
    fin = torch.empty((1, H, d, d), dtype=torch.float32, device=dev)
    call = lambda: kda.kda_chunk_fwd(q, k, v, la, beta, scale, None, cu, out, fin,
                                     engine=args.engine)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(dist.local_rank)
    sampler.start()
    preroll(call)
    kda.kda_chunk_path_counts()  # cleared: the timed calls' paths are counted below
    total_ms, per = timed_loop(call, args.steps, stream, dist)
    clocks = sampler.stop()
    paths = kda.kda_chunk_path_counts()
    ms_per_step = total_ms / args.steps
    value = units // H * args.steps * dist.world / (total_ms / 1e3)
    stages = stage_times(lambda evs: kda.kda_chunk_fwd_ws_timed(
        q, k, v, la, beta, scale, None, cu, out, fin, evs, engine=args.engine)[2], 2)
    traffic, tnote = profiled_traffic_scaled(max(stages, key=stages.get), units)
    roofline = prefill_roofline(stages, units, ms_per_step, peaks, traffic, tnote)

    # ---------------- end to end: the same call on host buffers ----------------
    # Inputs go to page-locked host memory (drawn on the device above), the
    # device copies are freed, and every step copies its inputs in and its
    # outputs out through kda_chunk_fwd_host on one stream.
    pinned = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
    hq, hk, hv, hla, hb, hcu = (pinned(t) for t in (q, k, v, la, beta, cu))
    del q, k, v, la, beta, out, x, call
    kda.binding._ws_cache.clear()
    torch.cuda.empty_cache()
    hout = torch.empty((T, H, d), dtype=torch.bfloat16, pin_memory=True)
    hfin = torch.empty((1, H, d, d), dtype=torch.float32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hla, hb, hcu))
    d2h = hout.numel() * 2 + hfin.numel() * 4
    hshape = kda.make_shape(1, T, H, d, d, kda.KDA_DTYPE_BF16)
    scratch = torch.empty(kda.kda_chunk_fwd_host_scratch_size(hshape) + 256, dtype=torch.uint8,
                          device=dev)
    e2e_call = lambda: kda.kda_chunk_fwd_host(hq, hk, hv, hla, hb, scale, None, hcu, hout, hfin,
                                              scratch=scratch, stream=stream,
                                              engine=args.engine)
    e2e_steps = max(1, min(args.steps, 5))
    for _ in range(min(args.warmup, 2)):
        e2e_call()
    torch.cuda.synchronize()
    e2e_ms, _ = timed_loop(e2e_call, e2e_steps, stream, dist)
    e2e = {"value": T * e2e_steps * dist.world / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
           "api": "kda_chunk_fwd_host (page-locked host buffers, copies in and out inside "
                  "the timed region, one stream)"}
    del hq, hk, hv, hla, hb, hcu, hout, hfin, scratch
    torch.cuda.empty_cache()

    # ---------------- the other rows ----------------
    rows = {}
    rows["prefill_T4096_H16"] = run_head_group(args, dist, peaks, dev, stream)
    rows["prefill_varlen_32seq"] = run_varlen(args, dist, peaks, dev, stream)
    rows["prefill_k3_gates"] = run_k3_gates(args, dist, dev, stream)
    w2 = inputs.head_group_prefill()
    t2 = lambda a, dt=None: torch.from_numpy(a).to(dev, dt)
    dev2 = (t2(w2.q, torch.bfloat16), t2(w2.k, torch.bfloat16), t2(w2.v, torch.bfloat16),
            t2(w2.log_alpha), t2(w2.beta), t2(w2.cu_seqlens))
    rows["prefill_variants"] = run_prefill_variants(args, dist, dev, stream, w2, dev2)
    rows["backward"] = run_backward(args, dist, peaks, dev, stream, w2, dev2)
    if not args.skip_decode:
        rows["decode"] = run_decode(args, dist, peaks, dev, stream)
        rows["recurrent_fwd"] = run_recurrent_fwd(args, dist, peaks, dev, stream)
        rows["short_conv"] = run_short_conv(args, dist, peaks, dev, stream)

    flops_call = PATH_FLOPS * units
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"long_context_T{T}_H{H}_d{d}: B=1, one sequence of {T} tokens "
                               f"x {H} heads, d_k=d_v={d}, chunk {C}, bf16 q/k/v, fp32 "
                               "log_alpha = -softplus(N(-6,1)), zero initial state, seeded",
                   "engine": args.engine,
                   "l2": "inputs (51.7 GB) far larger than the 129 MB L2; no flush",
                   "parallelism": "replicas" if dist.world > 1 else "single GPU"},
        "tflops": flops_call / (ms_per_step / 1e3) / 1e12,
        "tensor_frac_of_bf16_peak": flops_call / (ms_per_step / 1e3) / 1e12
                                    / peaks["bf16_tflops"],
        "path_gbs": PATH_BYTES * units / (ms_per_step / 1e3) / 1e9,
        "stages_ms": stages,
        "stages_note": "per-kernel device times from separate calls with library-recorded "
                       "events between the kernels (which run them one after another); the "
                       "headline times the plain public call, whose kernels overlap",
        "decay_paths": {"mid": paths[0], "half": paths[1], "direct": paths[2]},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    line.update(rows)
    if not args.skip_cpu_baseline and dist.rank == 0 and dist.world == 1:
        line["cpu_baseline"] = cpu_baseline()
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def run_head_group(args, dist, peaks, dev, stream):
    """B=1, H=16, T=4096 (the single-head-group prefill): the public call with
    an L2 flush (256 MiB write) before every timed step, since its ~100 MB of
    inputs would otherwise stay in the 129 MB L2."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import inputs
    w = inputs.head_group_prefill()
    T, H, d = w.T, w.H, w.d_k
    t = lambda a, dt=None: torch.from_numpy(a).to(dev, dt)
    q, k, v = (t(a, torch.bfloat16) for a in (w.q, w.k, w.v))
    la, beta, cu = t(w.log_alpha), t(w.beta), t(w.cu_seqlens)
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((1, H, d, d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    call = lambda: kda.kda_chunk_fwd(q, k, v, la, beta, w.scale, None, cu, out, fin,
                                     engine=args.engine)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    preroll(lambda: (flush.zero_(), call()))
    total_ms, _ = timed_loop(call, args.steps, stream, dist, flush)
    ms = total_ms / args.steps
    stages = stage_times(lambda evs: kda.kda_chunk_fwd_ws_timed(
        q, k, v, la, beta, w.scale, None, cu, out, fin, evs, engine=args.engine)[2],
        max(3, min(args.steps, 10)), flush)
    units = T * H
    traffic, tnote = profiled_traffic_scaled(max(stages, key=stages.get), units)
    return {"workload": f"{w.name}: B=1, H={H}, T={T}, d={d}, chunk 64, bf16, zero initial "
                        "state, seed 1; L2 flushed before each timed step",
            "value": T * dist.world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "stages_ms": stages,
            "roofline": prefill_roofline(stages, units, ms, peaks, traffic, tnote)}


def run_varlen(args, dist, peaks, dev, stream):
    """32 packed sequences, lengths ~ U[512, 8192] (136,134 tokens), H=32,
    initial states ~ N(0, 0.02), drawn on the device; inputs far larger than
    L2 (no flush).  Also the gradients of this workload (chunk-form backward)."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import inputs
    x = inputs.varlen_device(device=str(dev))
    q = x["q"]
    T, H, d = q.shape
    N = len(x["lengths"])
    out = torch.empty_like(q)
    fin = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    args_ = (q, x["k"], x["v"], x["log_alpha"], x["beta"], x["scale"], x["initial_state"],
             x["cu_seqlens"])
    call = lambda: kda.kda_chunk_fwd(*args_, out, fin, engine=args.engine)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    preroll(call)
    steps = max(3, min(args.steps, 10))
    total_ms, _ = timed_loop(call, steps, stream, dist)
    ms = total_ms / steps
    stages = stage_times(lambda evs: kda.kda_chunk_fwd_ws_timed(
        *args_, out, fin, evs, engine=args.engine)[2], 2)
    gen = torch.Generator(device=dev)
    gen.manual_seed(8)
    do = torch.randn(q.shape, generator=gen, device=dev).to(torch.bfloat16)
    bwd = lambda: kda.kda_chunk_bwd(*args_, do, None)
    bwd()
    torch.cuda.synchronize()
    bms, _ = timed_loop(bwd, 2, stream, dist)
    units = T * H
    res = {"workload": f"varlen_32seq_H{H}_d{d}: {N} packed sequences, lengths ~ U[512, 8192] "
                       f"({T} tokens), H={H}, initial states N(0, 0.02), drawn on the device",
           "value": T * dist.world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
           "stages_ms": stages, "roofline": prefill_roofline(stages, units, ms, peaks),
           "backward": {"ms_per_call": bms / 2, "tokens_per_s": T * dist.world / (bms / 2e3),
                        "form": "chunk (kda_chunk_bwd, forward recompute included)"}}
    del x, q, out, fin, do
    torch.cuda.empty_cache()
    return res


def run_k3_gates(args, dist, dev, stream):
    """The single-head-group shape with K3-range gates: log alpha =
    -5 sigmoid(g), g ~ N(0, 1) (range (-5, 0), midpoint -2.5), L2 flushed
    before each step, and how the prep evaluated each chunk's decayed
    products (mid-chunk reference, half-chunk references, direct)."""
    import numpy as np
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import inputs
    w = inputs.head_group_prefill()
    rng = np.random.default_rng(12)
    la_np = (-5.0 / (1.0 + np.exp(-rng.standard_normal(w.log_alpha.shape)))).astype(np.float32)
    t = lambda a, dt=None: torch.from_numpy(a).to(dev, dt)
    q, k, v = (t(a, torch.bfloat16) for a in (w.q, w.k, w.v))
    la, beta, cu = t(la_np), t(w.beta), t(w.cu_seqlens)
    out = torch.empty_like(q)
    fin = torch.empty((1, w.H, w.d_k, w.d_v), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    call = lambda: kda.kda_chunk_fwd(q, k, v, la, beta, w.scale, None, cu, out, fin,
                                     engine=args.engine)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    preroll(lambda: (flush.zero_(), call()))
    kda.kda_chunk_path_counts()
    total_ms, _ = timed_loop(call, args.steps, stream, dist, flush)
    paths = kda.kda_chunk_path_counts()
    ms = total_ms / args.steps
    return {"workload": f"{w.name} with log_alpha = -5 sigmoid(N(0, 1)) (K3 gate range); "
                        "L2 flushed before each timed step",
            "value": w.T * dist.world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "decay_paths": {"mid": paths[0], "half": paths[1], "direct": paths[2]}}


def run_profile_case(args, dist):
    """--profile prefill: the single-head-group prefill (B=1, H=16, T=4096)
    called --warmup + --steps times through the public call, no timing, no
    other row: a small case for a profiler to capture (inputs ~100 MB,
    scratch ~113 MB).  --profile backward / backward_recurrent: its gradients
    through kda_chunk_bwd / kda_recurrent_bwd instead."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import build, inputs
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(dist.local_rank)
    build.build()
    dev = torch.device("cuda", dist.local_rank)
    w = inputs.head_group_prefill()
    t = lambda a, dt=None: torch.from_numpy(a).to(dev, dt)
    q, k, v = (t(a, torch.bfloat16) for a in (w.q, w.k, w.v))
    la, beta, cu = t(w.log_alpha), t(w.beta), t(w.cu_seqlens)
    out = torch.empty_like(q)
    fin = torch.empty((1, w.H, w.d_k, w.d_v), dtype=torch.float32, device=dev)
    n = args.warmup + args.steps
    if args.profile in ("decode", "recurrent", "conv"):
        st = run_profile_other(args, dev)
        if dist.rank == 0:
            print(json.dumps({"profile_case": args.profile, "calls": n, "device_status": st}),
                  flush=True)
        return
    if args.profile in ("backward", "backward_recurrent"):
        import numpy as np
        rng = np.random.default_rng(8)
        do = t(rng.standard_normal((w.T, w.H, w.d_v)).astype(np.float32), torch.bfloat16)
        dsf = t(rng.standard_normal((1, w.H, w.d_k, w.d_v)).astype(np.float32))
        fn = kda.kda_chunk_bwd if args.profile == "backward" else kda.kda_recurrent_bwd
        for _ in range(n):
            fn(q, k, v, la, beta, w.scale, None, cu, do, dsf)
    else:
        for _ in range(n):
            kda.kda_chunk_fwd(q, k, v, la, beta, w.scale, None, cu, out, fin,
                              engine=args.engine)
    st = kda.kda_device_status()
    if dist.rank == 0:
        print(json.dumps({"profile_case": w.name, "what": args.profile, "calls": n,
                          "device_status": st}), flush=True)


def run_profile_other(args, dev):
    """--profile decode / recurrent / conv: the decode step of 256 sequences x
    32 heads (512 MiB state), the 8-token multi-token pass on the same batch,
    or the short convolution at K3 width (12,288 channels, 4,096 tokens),
    --warmup + --steps calls each."""
    import numpy as np
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import inputs
    n = args.warmup + args.steps
    t = lambda a, dt=None: torch.from_numpy(a).to(dev, dt)
    if args.profile == "decode":
        dw = inputs.batched_decode(steps=n)
        q, k, v = (t(a, torch.bfloat16) for a in (dw.q, dw.k, dw.v))
        la, b, state = t(dw.log_alpha), t(dw.beta), t(dw.initial_state)
        out = torch.empty(q.shape[1:], dtype=torch.bfloat16, device=dev)
        for i in range(n):
            kda.kda_recurrent_step(q[i], k[i], v[i], la[i], b[i], dw.scale, state, out)
    elif args.profile == "recurrent":
        N, H, d, L = 256, 32, 128, 8
        w = inputs.prefill(5, [L] * N, H=H, d=d, dtype="bf16", init_std=0.02)
        q, k, v = (t(a, torch.bfloat16) for a in (w.q, w.k, w.v))
        la, b, cu, pool = t(w.log_alpha), t(w.beta), t(w.cu_seqlens), t(w.initial_state)
        slots = torch.arange(N, dtype=torch.int32, device=dev).flip(0).contiguous()
        for _ in range(n):
            kda.kda_recurrent_fwd(q, k, v, la, b, w.scale, pool, cu, slots)
    else:
        C, W = 12288, 4
        rng = np.random.default_rng(6)
        lengths = [1000, 17, 2048, 1031]
        T = sum(lengths)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=dev)
        x = t(rng.standard_normal((T, C)).astype(np.float32), torch.bfloat16)
        wt = t((rng.standard_normal((C, W)) * 0.5).astype(np.float32))
        bias = t(rng.standard_normal(C).astype(np.float32))
        cin = torch.zeros((len(lengths), C, W), dtype=torch.bfloat16, device=dev)
        cout = torch.empty_like(cin)
        for _ in range(n):
            kda.kda_short_conv_fwd(x, wt, bias, cu, cin, cout, silu=True)
    return kda.kda_device_status()


def run_decode(args, dist, peaks, dev, stream):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import inputs
    S = args.decode_steps
    dw = inputs.batched_decode(steps=S)
    N, H, d = dw.q.shape[1], dw.q.shape[2], dw.q.shape[3]
    q = torch.from_numpy(dw.q).to(dev, torch.bfloat16)
    k = torch.from_numpy(dw.k).to(dev, torch.bfloat16)
    v = torch.from_numpy(dw.v).to(dev, torch.bfloat16)
    la = torch.from_numpy(dw.log_alpha).to(dev)
    b = torch.from_numpy(dw.beta).to(dev)
    state = torch.from_numpy(dw.initial_state).to(dev)
    out = torch.empty((N, H, d), dtype=torch.bfloat16, device=dev)
    for t in range(min(args.warmup, S)):
        kda.kda_recurrent_step(q[t], k[t], v[t], la[t], b[t], dw.scale, state, out)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(S + 1)]
    preroll(lambda: kda.kda_recurrent_step(q[0], k[0], v[0], la[0], b[0], dw.scale, state, out))
    dist.barrier()
    torch.cuda.synchronize()
    evs[0].record(stream)
    for t in range(S):
        kda.kda_recurrent_step(q[t], k[t], v[t], la[t], b[t], dw.scale, state, out)
        evs[t + 1].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    per = [evs[t].elapsed_time(evs[t + 1]) for t in range(S)]
    total_ms = dist.max(sum(per))
    bytes_step = (2 * d * d * 4 + 3 * 2 * d + 2 * d + 4 * d + 4) * N * H
    gbs = bytes_step * S * dist.world / (total_ms / 1e3) / 1e9
    return {"workload": f"{N} sequences x {H} heads, d={d}, fp32 state "
                        f"{N * H * d * d * 4 / 2**20:.0f} MiB, {S} steps (state > L2)",
            "value": gbs, "unit": "GB/s", "us_per_step": 1e3 * total_ms / S,
            "median_us_per_step": 1e3 * statistics.median(per),
            "gpu_launches": S,
            "roofline": {"kernel": "recurrent_step", "bound": "hbm", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": profiled_traffic("recurrent_step"),
                         "bytes_per_launch": bytes_step, "peak_source": peaks["source"]}}


def run_recurrent_fwd(args, dist, peaks, dev, stream):
    """Multi-token recurrent pass: every sequence of the decode batch takes 8
    new tokens in one call (a speculative-verification step), states in a
    slot pool; the state crosses HBM once in each direction per call."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kimi_delta_attention_chunkwise_gb300 import inputs
    N, H, d, L = 256, 32, 128, 8
    w = inputs.prefill(5, [L] * N, H=H, d=d, dtype="bf16", init_std=0.02,
                       name="multi_token_decode")
    to = lambda x, dt=None: torch.from_numpy(x).to(dev, dt)
    q, k, v = to(w.q, torch.bfloat16), to(w.k, torch.bfloat16), to(w.v, torch.bfloat16)
    la, b, cu = to(w.log_alpha), to(w.beta), to(w.cu_seqlens)
    pool = to(w.initial_state)
    slots = torch.arange(N, dtype=torch.int32, device=dev).flip(0).contiguous()
    out = torch.empty((w.T, H, d), dtype=torch.bfloat16, device=dev)
    call = lambda: kda.kda_recurrent_fwd(q, k, v, la, b, w.scale, pool, cu, slots, out)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    reps = 20
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    preroll(call)
    dist.barrier()
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(reps):
        call()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(reps)]
    total_ms = dist.max(sum(per))
    # state read + written once per (sequence, head); per token q, k, v, out
    # (bf16), log_alpha (fp32), beta
    bytes_call = (2 * d * d * 4 + L * (4 * 2 * d + 4 * d + 4)) * N * H
    gbs = bytes_call * reps * dist.world / (total_ms / 1e3) / 1e9
    return {"workload": f"{N} sequences x {H} heads x {L} new tokens, d={d}, bf16, fp32 state "
                        f"pool {N * H * d * d * 4 / 2**20:.0f} MiB (reversed slot order)",
            "value": N * L * reps * dist.world / (total_ms / 1e3), "unit": "tokens/s",
            "us_per_call": 1e3 * total_ms / reps, "gbs": gbs, "gpu_launches": reps,
            "roofline": {"kernel": "recurrent_fwd", "bound": "hbm", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "traffic": profiled_traffic("recurrent_fwd"),
                         "bytes_per_launch": bytes_call, "peak_source": peaks["source"]}}


def run_prefill_variants(args, dist, dev, stream, w, dev_inputs):
    """The head-group prefill workload again, (a) with the whole fused input
    prologue on (raw q/k, beta logits, K3 gate projections) and (b) with
    value-head groups (8 q/k heads shared by the 16 value heads).  Timed
    like the headline (L2 flushed before every step)."""
    import numpy as np
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    q, k, v, la, beta, cu = dev_inputs
    T, H, d = q.shape
    rng = np.random.default_rng(7)
    gate = (torch.from_numpy((rng.standard_normal((H, d)) * 0.5 - 3.0).astype(np.float32)).to(dev),
            torch.from_numpy(rng.uniform(-1, 1, H).astype(np.float32)).to(dev))
    g_raw = torch.from_numpy(rng.standard_normal((T, H, d)).astype(np.float32)).to(dev)
    beta_raw = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(dev)
    q_raw, k_raw = q * 3, k * 3
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    fin = torch.empty((1, H, d, d), device=dev)
    qg, kg = q[:, : H // 2].contiguous(), k[:, : H // 2].contiguous()
    cases = {
        "prologue": lambda: kda.kda_chunk_fwd(q_raw, k_raw, v, g_raw, beta_raw, w.scale, None, cu,
                                             out, fin, l2norm_qk=True, beta_logits=True,
                                             gate=gate),
        "value_groups": lambda: kda.kda_chunk_fwd(qg, kg, v, la, beta, w.scale, None, cu, out,
                                                 fin),
    }
    res = {}
    for name, fn in cases.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        preroll(lambda: (flush.zero_(), fn()))
        dist.barrier()
        torch.cuda.synchronize()
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ms = dist.max(sum(a.elapsed_time(b) for a, b in evs)) / args.steps
        res[name] = {"value": T * dist.world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms}
    res["prologue"]["workload"] = ("the headline workload with raw q/k (L2-normalised in-kernel), "
                                   "beta logits and K3 gate projections (bias, A_log)")
    res["value_groups"]["workload"] = (f"the headline workload with {H // 2} q/k heads shared by "
                                       f"{H} value heads")
    del flush
    return res


# Dense products of the chunk-form backward per (token, head), d = 128, C = 64,
# from the kernels' valid rows (per chunk, divided by its C tokens):
#   forward recompute without the output pass   8Cd + 4d^2
#   X_c = Q'^T dO_c and the reverse scan's -M'^T dS  2d^2 + 2d^3 / C
#   G1: [U | W], dE^T, W S_c, S_c [dO ; dE]^T, E dO^T, dS E^T   8Cd + 10d^2
#   G2: dA, A^T [dE | dW], A^T dA, dR, [X1 | X2], Y               16Cd + 4C^2
_C, _D = 64, 128
BWD_FLOPS_PER_UNIT = ((8 * _C * _D + 4 * _D * _D) + (2 * _D * _D + 2 * _D ** 3 // _C)
                      + (8 * _C * _D + 10 * _D * _D) + (16 * _C * _D + 4 * _C * _C))
# Compulsory bytes per (token, head): q, k, v, d_out (bf16) and log_alpha,
# beta in; dq, dk, dv, dlog_alpha (fp32) and dbeta out.
BWD_BYTES_PER_UNIT = 4 * 2 * 128 + 4 * 128 + 4 + 4 * 4 * 128 + 4


def run_backward(args, dist, peaks, dev, stream, w, dev_inputs):
    """Gradients of the head-group prefill workload (1 sequence x 16 heads x
    4,096 tokens) with output and final-state gradients, timed like the
    headline: the chunk form (kda_chunk_bwd: forward recompute, reverse scan
    and the per-chunk gradient products on the tensor cores) and the
    token-recurrence form (kda_recurrent_bwd)."""
    import numpy as np
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    q, k, v, la, beta, cu = dev_inputs
    T, H, d = q.shape
    rng = np.random.default_rng(8)
    do = torch.from_numpy(rng.standard_normal((T, H, d)).astype(np.float32)).to(dev, torch.bfloat16)
    dsf = torch.from_numpy(rng.standard_normal((1, H, d, d)).astype(np.float32)).to(dev)
    reps = max(3, min(args.steps, 5))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(call):
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        preroll(call, 0.1)
        dist.barrier()
        torch.cuda.synchronize()
        evs[0].record(stream)
        for _ in range(reps):
            call()
        evs[1].record(stream)
        torch.cuda.synchronize()
        return dist.max(evs[0].elapsed_time(evs[1])) / reps

    ms_chunk = timed(lambda: kda.kda_chunk_bwd(q, k, v, la, beta, w.scale, None, cu, do, dsf))
    # DRAM bytes of one call: its kernels' ncu captures on this workload (the
    # forward recompute's prep and scan from the prefill capture)
    parts = [profiled_traffic(k_) for k_ in ("prep", "scan", "chunk_bwd_aux", "chunk_rscan",
                                            "chunk_grad_g1", "chunk_grad_g2")]
    traffic = sum(parts) if all(p_ is not None for p_ in parts) else None
    ms_rec = timed(lambda: kda.kda_recurrent_bwd(q, k, v, la, beta, w.scale, None, cu, do, dsf))
    units = T * H
    bytes_call = BWD_BYTES_PER_UNIT * units + H * d * d * 4
    gbs = bytes_call / (ms_chunk / 1e3) / 1e9
    tfl = BWD_FLOPS_PER_UNIT * units / (ms_chunk / 1e3) / 1e12
    gbs_rec = bytes_call / (ms_rec / 1e3) / 1e9
    return {"workload": f"gradients of the single-head-group workload (1 x {H} heads x {T} "
                        "tokens, d=128, bf16 in, fp32 gradients) through the chunk form "
                        "(kda_chunk_bwd, its forward recompute included)",
            "value": T * dist.world / (ms_chunk / 1e3), "unit": "tokens/s",
            "ms_per_step": ms_chunk,
            "roofline": {"kernel": "chunk_bwd (whole call)", "bound": "latency",
                         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "tensor_tflops": tfl,
                         "tensor_frac": tfl / peaks["bf16_tflops"],
                         "bytes_per_launch": bytes_call,
                         "flops_per_unit": BWD_FLOPS_PER_UNIT, "peak_source": peaks["source"],
                         "traffic": traffic,
                         "traffic_note": "sum of the DRAM bytes of its kernels' ncu captures",
                         "note": "seven kernels and one flag memset per call (forward "
                                 "recompute: chunk table, prep, scan; X_c beside the reverse "
                                 "scan; two gradient kernels); per-kernel shares in profiles/"},
            "recurrent_form": {"ms_per_step": ms_rec, "value": T * dist.world / (ms_rec / 1e3),
                               "unit": "tokens/s",
                               "workload": "the same gradients through kda_recurrent_bwd "
                                           "(token recurrence with 8-token checkpoints)",
                               "roofline": {"kernel": "recurrent_bwd", "bound": "hbm",
                                            "achieved": gbs_rec, "peak": peaks["hbm_gbs"],
                                            "unit": "GB/s", "frac": gbs_rec / peaks["hbm_gbs"],
                                            "traffic": profiled_traffic("recurrent_bwd"),
                                            "bytes_per_launch": bytes_call,
                                            "peak_source": peaks["source"],
                                            "note": "the per-token walk is latency-bound "
                                                    "(barriers), not HBM-bound"}}}


def run_short_conv(args, dist, peaks, dev, stream):
    """The layer's short convolution at K3 width (96 heads x 128 = 12,288
    channels, 4 taps, SiLU, bf16) over 4 packed sequences totalling 4,096
    tokens, caches in and out; then one decode step for 256 sequences."""
    import numpy as np
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    C, W, N = 12288, 4, 4
    rng = np.random.default_rng(6)
    lengths = [1000, 17, 2048, 1031]
    T = sum(lengths)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=dev)
    x = torch.from_numpy(rng.standard_normal((T, C)).astype(np.float32)).to(dev, torch.bfloat16)
    w = torch.from_numpy((rng.standard_normal((C, W)) * 0.5).astype(np.float32)).to(dev)
    b = torch.from_numpy(rng.standard_normal(C).astype(np.float32)).to(dev)
    cin = torch.zeros((N, C, W), dtype=torch.bfloat16, device=dev)
    cout = torch.empty_like(cin)
    y = torch.empty_like(x)
    call = lambda: kda.kda_short_conv_fwd(x, w, b, cu, cin, cout, y, silu=True)
    ND = 256
    xd = torch.from_numpy(rng.standard_normal((ND, C)).astype(np.float32)).to(dev, torch.bfloat16)
    cache = torch.zeros((ND, C, W), dtype=torch.bfloat16, device=dev)
    yd = torch.empty_like(xd)
    step = lambda: kda.kda_short_conv_step(xd, w, cache, b, yd, silu=True)
    for _ in range(max(3, args.warmup)):
        call(); step()
    torch.cuda.synchronize()
    # the calls are short next to a Python launch: capture each in a CUDA graph
    # and time replays, so the device time is what is measured
    reps = 20
    res = {}
    for name, fn in (("prefill", call), ("step", step)):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        graph.replay()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        preroll(graph.replay)
        dist.barrier()
        torch.cuda.synchronize()
        evs[0].record(stream)
        for _ in range(reps):
            graph.replay()
        evs[1].record(stream)
        torch.cuda.synchronize()
        res[name] = dist.max(evs[0].elapsed_time(evs[1])) / reps
    # bytes: x read once, y written once, weights and bias, caches in and out
    b_pre = 2 * T * C * 2 + C * (W + 1) * 4 + 2 * N * C * W * 2
    b_step = 2 * ND * C * 2 + C * (W + 1) * 4 + 2 * ND * C * W * 2
    gbs = b_pre / (res["prefill"] / 1e3) / 1e9
    return {"workload": f"C={C} channels, {W} taps, SiLU, bf16; prefill {T} tokens in {N} "
                        f"sequences; decode step for {ND} sequences",
            "value": gbs, "unit": "GB/s", "us_per_call": 1e3 * res["prefill"],
            "step_us": 1e3 * res["step"],
            "step_gbs": b_step / (res["step"] / 1e3) / 1e9, "gpu_launches": 2 * reps,
            "roofline": {"kernel": "short_conv_fwd", "bound": "hbm", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "traffic": profiled_traffic("short_conv_fwd"), "bytes_per_launch": b_pre,
                         "peak_source": peaks["source"]}}


def main():
    global PREROLL_SECONDS
    args = parse_args()
    PREROLL_SECONDS = max(0.0, args.preroll)
    dist = Dist()
    try:
        if args.impl == "reference":
            if args.sweep:
                run_reference_sweep(args, dist)
            else:
                run_reference(args, dist)
        elif args.profile:
            run_profile_case(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
