#!/usr/bin/env python3
"""Benchmark of libkda on one GB300 (or N replicas, one per GPU).

One step = one ``kda_chunk_fwd`` over the single-head-group prefill workload
(B=1, H=16, T=4096, d_k=d_v=128, chunk 64, bf16 q/k/v, fp32 gates and state,
seeded synthetic inputs), i.e. every prefill stage of the hot path.  The
decode row (``kda_recurrent_step``, 256 sequences x 32 heads, 512 MiB fp32
state, 64 steps) is measured in the same run and reported under "decode".

Timing: CUDA events on the launch stream, W untimed warm-up steps, about
0.3 s of back-to-back steps (--preroll; the first call after an idle gap runs
at half speed while the clocks come back), then K timed steps with an L2
flush (256 MiB write) before each (the prefill inputs, ~100 MB, would
otherwise stay in the 129 MB L2), barrier and synchronize on both sides, max
over ranks.  libkda itself records events between its kernels
(kda_chunk_fwd_ws_timed, which runs them one after another), which gives the
per-kernel device times behind the roofline figures.  The end-to-end figure
goes through kda_chunk_fwd_host (host buffers, copies inside the timed
region).  The multi-token pass, the short convolution, the prologue and
value-group variants and the backward are measured in the same run.

``--impl reference`` times the fp64 CPU oracle (the reference arm of this
repository) on a bounded sample of the same workload on the host cores.

``--sweep`` prints, instead of the headline line, one JSON line for each of
the two larger prefill workloads (32 packed sequences x 32 heads with their
backward; one 1,048,576-token sequence x 32 heads); with ``--impl
reference`` it times the oracle on every named workload.
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
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the headline, time the packed 32-sequence workload and "
                         "the 1,048,576-token sequence (one JSON line each); with "
                         "--impl reference, time the oracle on every named workload")
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

def prefill_flops_per_tok_head(d: int, C: int) -> int:
    """Dense chunk contractions: K K^T, Q K^T, A^kk (beta V), A^kk (beta Gamma K),
    A^qk E (5 x 2Cd) plus W S, K_end^T E, Q_hat S (3 x 2d^2)."""
    return 10 * C * d + 6 * d * d


def stage_work(d: int, C: int):
    """Per (token, head) compulsory bytes and issued tensor-core flops of each
    kernel of the tensor-core engine (its own inputs read once, its outputs
    written once).  The per-(chunk, head) image holds -M' (d x d), P' (d x C),
    Q' (C x d), Z (C x C) in f16 plus Gamma_last and beta in fp32; the scan
    reads its -M'/P' part once per value tile and writes S_c (d x d, f16) per
    chunk; the output pass reads Q'/Z (with 8 KB of filler rows), S_c and v."""
    nt = 2                                            # value tiles per head
    img = (2 * d * d + 2 * d * C + 2 * C * d + 2 * C * C + 4 * d + 4 * C) / C
    prep_bytes = 2 * 2 * d + 4 * d + 4 + img          # q, k, log_alpha, beta -> image
    scan_bytes = (nt * (2 * d * d + 2 * d * C) / C    # -M', P' per value tile
                  + 2 * d + 4 * d / C * nt + 4 * nt   # v, Gamma_last, beta
                  + 2 * d * d / C)                    # S_c out (f16)
    out_bytes = ((2 * C * d + 2 * C * C + 2 * 64 * 64 + 2 * d * d) / C  # Q', Z, filler, S_c
                 + 2 * d + 4 + 2 * d)                 # v, beta in; out (bf16)
    prep_flops = 10 * C * d + 2 * d * d + 2 * C * C   # [K;Q]K^T, W, M', P', A^qk W, Z
    scan_flops = 2 * d * d + 2 * d * d * d / C        # P' (beta V), M' S_c
    out_flops = 2 * d * d + 2 * C * d                 # Q' S_c, Z (beta V)
    return {"prep": (prep_bytes, prep_flops), "scan": (scan_bytes, scan_flops),
            "out": (out_bytes, out_flops)}


PROFILE_FILES = {
    "prep": "chunk_prep_prefill_T4096_H16.md",
    "scan": "chunk_scan_prefill_T4096_H16.md",
    "out": "chunk_out_prefill_T4096_H16.md",
    "recurrent_step": "recurrent_step_decode_256x32_d128.md",
    "recurrent_fwd": "recurrent_fwd_decode_256x32x8_d128.md",
    "short_conv_fwd": "short_conv_fwd_prefill_C12288_T4096.md",
    "recurrent_bwd": "recurrent_bwd_prefill_T4096_H16.md",
}


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, or None when there is none or the kernel's source has
    changed since the counters were taken (source hash recorded alongside)."""
    import hashlib
    name = PROFILE_FILES.get(kernel)
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


def path_bytes_per_tok_head(d: int) -> int:
    """Whole-path minimum: q, k, v, out (bf16) and log_alpha (fp32) once, beta."""
    return 4 * 2 * d + 4 * d + 4


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


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    import oracle
    from kimi_delta_attention_chunkwise_gb300 import inputs
    w = inputs.head_group_prefill()
    Ts = 512  # bounded sample: the first 512 tokens of the workload, all 16 heads
    sl = slice(0, Ts)
    arrs = [w.q[sl], w.k[sl], w.v[sl], w.log_alpha[sl], w.beta[sl]]
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
    sample = (f"first {Ts} of {w.T} tokens x {w.H} heads of the prefill workload per step, "
              f"fp64 token recurrence")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + " (B=1, chunk 64, seed 1)", "sample_tokens": Ts},
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


def cpu_baseline(w):
    """The oracle as it stands on the whole prefill workload, repeated to at
    least ~10 s of wall time (bounded: at most 40 runs)."""
    import oracle
    oracle.build()
    thr = oracle_threads()
    runs, t_total = 0, 0.0
    while runs < 40 and (t_total < 10.0 or runs == 0):
        t0 = time.perf_counter()
        oracle.recurrent(w.q, w.k, w.v, w.log_alpha, w.beta, w.scale, None, w.cu_seqlens,
                         threads=thr)
        t_total += time.perf_counter() - t0
        runs += 1
    return {"value": w.T * runs / t_total, "unit": "tokens/s", "cores": thr, "kind": "oracle",
            "sample": f"the whole workload ({w.T} tokens x {w.H} heads) x {runs} run(s), "
                      f"fp64 token recurrence, {t_total:.1f} s"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, dist: Dist):
    import numpy as np
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

    # ---------------- prefill workload ----------------
    w = inputs.head_group_prefill()
    T, H, d, C = w.T, w.H, w.d_k, w.chunk_size
    q = torch.from_numpy(w.q).to(dev, torch.bfloat16)
    k = torch.from_numpy(w.k).to(dev, torch.bfloat16)
    v = torch.from_numpy(w.v).to(dev, torch.bfloat16)
    la = torch.from_numpy(w.log_alpha).to(dev)
    beta = torch.from_numpy(w.beta).to(dev)
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((1, H, d, d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # creates the underlying CUDA event
        return evs

    MAXEV = 8
    warm_evs = new_events(MAXEV)
    n_rec = 0
    for _ in range(args.warmup):
        kda.kda_chunk_fwd(q, k, v, la, beta, w.scale, None, cu, out, fin, engine=args.engine)
        _, _, n_rec = kda.kda_chunk_fwd_ws_timed(q, k, v, la, beta, w.scale, None, cu, out, fin,
                                                 warm_evs, engine=args.engine)
    torch.cuda.synchronize()
    n_stages = max(1, n_rec - 1)
    step_evs = [new_events(MAXEV) for _ in range(args.steps)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()

    # the headline: the public call, as a user makes it (no events between its kernels)
    sampler = ClockSampler(dist.local_rank)
    sampler.start()

    def headline_step():
        flush.zero_()
        kda.kda_chunk_fwd(q, k, v, la, beta, w.scale, None, cu, out, fin, engine=args.engine)

    preroll(headline_step)
    dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        kda.kda_chunk_fwd(q, k, v, la, beta, w.scale, None, cu, out, fin, engine=args.engine)
        ends[i].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()

    # per-kernel device times (the roofline inputs): the same call with
    # library-recorded events between its kernels; not part of the headline
    preroll(headline_step)
    for i in range(args.steps):
        flush.zero_()
        kda.kda_chunk_fwd_ws_timed(q, k, v, la, beta, w.scale, None, cu, out, fin, step_evs[i],
                                   engine=args.engine)
    torch.cuda.synchronize()

    step_ms = [starts[i].elapsed_time(ends[i]) for i in range(args.steps)]
    stage_ms = [[step_evs[i][s].elapsed_time(step_evs[i][s + 1]) for s in range(n_stages)]
                for i in range(args.steps)]
    total_ms = dist.max(sum(step_ms))
    ms_per_step = total_ms / args.steps
    tokens = T * args.steps * dist.world
    value = tokens / (total_ms / 1e3)
    flops_step = prefill_flops_per_tok_head(d, C) * T * H
    tflops = flops_step * args.steps * dist.world / (total_ms / 1e3) / 1e12

    stage_avg = [statistics.mean(s[j] for s in stage_ms) for j in range(n_stages)]
    if n_stages == 4:
        names = ["chunk_table", "prep", "scan", "out"]
    else:
        names = [f"stage{j}" for j in range(n_stages)]
        names[-1] = "chunk_simt" if n_stages == 1 else names[-1]
    dom = max(range(n_stages), key=lambda j: stage_avg[j])
    work = stage_work(d, C)
    if names[dom] in work:
        bpt, fpt = work[names[dom]]
    else:
        bpt, fpt = path_bytes_per_tok_head(d), prefill_flops_per_tok_head(d, C)
    dom_s = stage_avg[dom] / 1e3
    achieved_gbs = bpt * T * H / dom_s / 1e9
    roofline = {"kernel": names[dom], "bound": "hbm", "achieved": achieved_gbs,
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": profiled_traffic(names[dom]),
                "peak_source": peaks["source"],
                "bytes_per_launch": bpt * T * H, "launch_ms": stage_avg[dom],
                "tensor_tflops": fpt * T * H / dom_s / 1e12,
                "tensor_frac": fpt * T * H / dom_s / 1e12 / peaks["bf16_tflops"]}

    # ---------------- end to end through the public API, host buffers ----------------
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    hq, hk, hv = (pin(a).to(torch.bfloat16).pin_memory() for a in (w.q, w.k, w.v))
    hla, hb, hcu = pin(w.log_alpha), pin(w.beta), pin(w.cu_seqlens)
    hout = torch.empty((T, H, d), dtype=torch.bfloat16).pin_memory()
    hfin = torch.empty((1, H, d, d), dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hla, hb, hcu))
    d2h = hout.numel() * 2 + hfin.numel() * 4

    # The public host-buffer call (kda_chunk_fwd_host: copies in, prefill,
    # copies out) on two streams with two scratch buffers and two sets of host
    # outputs, steps alternating: one step's copies overlap the other
    # stream's kernels.  Every step copies its inputs in and its results out.
    hshape = kda.make_shape(1, T, H, d, d, kda.KDA_DTYPE_BF16)
    hbytes = kda.kda_chunk_fwd_host_scratch_size(hshape)
    e2e_streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    scratches = [torch.empty(hbytes + 256, dtype=torch.uint8, device=dev) for _ in range(2)]
    houts = [(hout, hfin), (torch.empty_like(hout).pin_memory(),
                            torch.empty_like(hfin).pin_memory())]

    def e2e_step(i):
        s = e2e_streams[i % 2]
        with torch.cuda.stream(s):
            flush.zero_()
        kda.kda_chunk_fwd_host(hq, hk, hv, hla, hb, w.scale, None, hcu, houts[i % 2][0],
                               houts[i % 2][1], scratch=scratches[i % 2], stream=s,
                               engine=args.engine)

    def e2e_run(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in e2e_streams:
            s.wait_event(e0)
        for i in range(n):
            e2e_step(i)
        for s in e2e_streams:
            ev = torch.cuda.Event()
            ev.record(s)
            stream.wait_event(ev)
        e1.record(stream)
        return e0, e1

    for _ in range(args.warmup):
        e2e_run(2)
    torch.cuda.synchronize()
    preroll(lambda: e2e_run(2))
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = e2e_run(args.steps)
    torch.cuda.synchronize()
    dist.barrier()
    e2e_ms = dist.max(e0.elapsed_time(e1))
    e2e = {"value": T * args.steps * dist.world / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": e2e_ms / args.steps,
           "api": "kda_chunk_fwd_host (host buffers), two streams, steps alternating"}

    # ---------------- decode rows ----------------
    variants = run_prefill_variants(args, dist, dev, stream, w, (q, k, v, la, beta, cu))
    backward = run_backward(args, dist, peaks, dev, stream, w, (q, k, v, la, beta, cu))
    decode = recurrent = conv = None
    if not args.skip_decode:
        decode = run_decode(args, dist, peaks, dev, stream)
        recurrent = run_recurrent_fwd(args, dist, peaks, dev, stream)
        conv = run_short_conv(args, dist, peaks, dev, stream)

    del flush
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: B=1, H={H}, T={T}, d_k=d_v={d}, chunk {C}, "
                               "bf16 q/k/v, fp32 gates/state, zero initial state, seed 1",
                   "engine": args.engine, "l2": "flushed (256 MiB write) before each timed step",
                   "parallelism": "replicas" if dist.world > 1 else "single GPU"},
        "tflops": tflops, "tensor_frac_of_bf16_peak": tflops / peaks["bf16_tflops"],
        "path_gbs": path_bytes_per_tok_head(d) * T * H * args.steps * dist.world
                    / (total_ms / 1e3) / 1e9,
        "stages_ms": dict(zip(names, stage_avg)),
        "stages_note": "per-kernel device times from a separate run with library-recorded events "
                       "between the kernels; the headline times the plain public call",
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": n_stages * args.steps,
        "clocks": clocks,
        "decode": decode,
        "recurrent_fwd": recurrent,
        "short_conv": conv,
        "prefill_variants": variants,
        "backward": backward,
    }
    if not args.skip_cpu_baseline and dist.rank == 0 and dist.world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


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


def run_backward(args, dist, peaks, dev, stream, w, dev_inputs):
    """Gradients of the head-group prefill workload (1 sequence x 16 heads x
    4,096 tokens): the recurrent backward with output and final-state
    gradients, timed like the headline."""
    import numpy as np
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    q, k, v, la, beta, cu = dev_inputs
    T, H, d = q.shape
    rng = np.random.default_rng(8)
    do = torch.from_numpy(rng.standard_normal((T, H, d)).astype(np.float32)).to(dev, torch.bfloat16)
    dsf = torch.from_numpy(rng.standard_normal((1, H, d, d)).astype(np.float32)).to(dev)
    call = lambda: kda.kda_recurrent_bwd(q, k, v, la, beta, w.scale, None, cu, do, dsf)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 5))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    preroll(call, 0.1)
    dist.barrier()
    torch.cuda.synchronize()
    evs[0].record(stream)
    for _ in range(reps):
        call()
    evs[1].record(stream)
    torch.cuda.synchronize()
    ms = dist.max(evs[0].elapsed_time(evs[1])) / reps
    # compulsory bytes: q, k, v, d_out (bf16), log_alpha, beta in; dq, dk, dv,
    # dlog_alpha (fp32), dbeta out; the final-state gradient in
    bytes_call = (4 * 2 * d + 4 * d + 4 + 4 * 4 * d + 4) * T * H + H * d * d * 4
    gbs = bytes_call / (ms / 1e3) / 1e9
    return {"workload": f"gradients of the headline workload (1 x {H} heads x {T} tokens, d={d}, "
                        "bf16 in, fp32 gradients), recurrent form with 8-token checkpoints",
            "value": T * dist.world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "roofline": {"kernel": "recurrent_bwd", "bound": "hbm", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": profiled_traffic("recurrent_bwd"),
                         "bytes_per_launch": bytes_call, "peak_source": peaks["source"],
                         "note": "the per-token walk is latency-bound (barriers), not HBM-bound"}}


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


def run_sweep(args, dist: Dist):
    """The two larger prefill workloads through the public call: 32 packed
    sequences (lengths ~ U[512, 8192], H=32, initial states given) and one
    1,048,576-token sequence (H=32).  Both hold far more than L2, so no flush.
    Per-kernel times come from a second run with library-recorded events."""
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

    def workloads():
        w = inputs.varlen_prefill()
        t = lambda a, dt=None: torch.from_numpy(a).to(dev, dt) if dt else torch.from_numpy(a).to(dev)
        yield (w.name, dict(q=t(w.q, torch.bfloat16), k=t(w.k, torch.bfloat16),
                            v=t(w.v, torch.bfloat16), log_alpha=t(w.log_alpha), beta=t(w.beta),
                            cu_seqlens=t(w.cu_seqlens), initial_state=t(w.initial_state),
                            scale=w.scale), len(w.meta["lengths"]))
        del w
        x = inputs.long_context_device(device=str(dev))
        x["initial_state"] = None
        yield ("long_context_T1048576_H32_d128", x, 1)

    for name, x, n_seqs in workloads():
        q = x["q"]
        T, H, d = q.shape
        out = torch.empty_like(q)
        fin = torch.empty((n_seqs, H, d, d), dtype=torch.float32, device=dev)
        call = lambda: kda.kda_chunk_fwd(q, x["k"], x["v"], x["log_alpha"], x["beta"],
                                         x["scale"], x["initial_state"], x["cu_seqlens"], out,
                                         fin, engine=args.engine)
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        steps = max(1, min(args.steps, 10))
        sampler = ClockSampler(dist.local_rank)
        sampler.start()
        preroll(call)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            call()
        end.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        clocks = sampler.stop()
        ms = dist.max(start.elapsed_time(end)) / steps
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
        for e in evs:
            e.record(stream)
        _, _, n_rec = kda.kda_chunk_fwd_ws_timed(q, x["k"], x["v"], x["log_alpha"], x["beta"],
                                                 x["scale"], x["initial_state"],
                                                 x["cu_seqlens"], out, fin, evs,
                                                 engine=args.engine)
        torch.cuda.synchronize()
        names = ["chunk_table", "prep", "scan", "out"] if n_rec == 5 else \
            [f"stage{j}" for j in range(max(0, n_rec - 1))]
        stages = {nm: evs[j].elapsed_time(evs[j + 1]) for j, nm in enumerate(names)}
        flops = prefill_flops_per_tok_head(d, 64) * T * H
        path_bytes = path_bytes_per_tok_head(d) * T * H
        line = {"sweep": name, "impl": "ours", "n_gpus": dist.world, "steps": steps,
                "tokens": T, "heads": H, "sequences": n_seqs, "ms_per_call": ms,
                "tokens_per_s": T * dist.world / (ms / 1e3),
                "tflops": flops / (ms / 1e3) / 1e12,
                "tensor_frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                "path_gbs": path_bytes / (ms / 1e3) / 1e9,
                "path_frac_of_hbm": path_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                "stages_ms": stages, "clocks": clocks, "data": "synthetic"}
        if n_seqs > 1:
            # the gradients of the packed workload (d_out ~ N(0, 1), no final-state gradient)
            gen = torch.Generator(device=dev)
            gen.manual_seed(8)
            do = torch.randn(q.shape, generator=gen, device=dev).to(torch.bfloat16)
            bwd = lambda: kda.kda_recurrent_bwd(q, x["k"], x["v"], x["log_alpha"], x["beta"],
                                                x["scale"], x["initial_state"],
                                                x["cu_seqlens"], do, None)
            for _ in range(2):
                bwd()
            torch.cuda.synchronize()
            reps = 2
            start.record(stream)
            for _ in range(reps):
                bwd()
            end.record(stream)
            torch.cuda.synchronize()
            bms = dist.max(start.elapsed_time(end)) / reps
            line["backward"] = {"ms_per_call": bms, "tokens_per_s": T * dist.world / (bms / 1e3),
                                "form": "recurrent, 8-token checkpoints"}
            del do
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
        del x, q, out, fin
        torch.cuda.empty_cache()


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
        elif args.sweep:
            run_sweep(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
