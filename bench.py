"""Benchmark: fused attention backward TFLOP/s on one GB300 (and N replicas).

One step = the whole hot path on one batch of synthetic bf16 input: forward
(O, LSE) then backward (preprocess, main kernel, dQ conversion), all through
the C ABI.  The default workload is causal, H=16, d=128, T=32768, B=1 (32K
tokens); `--workload` names any other (the GPT-2-shaped packed layer, the
sweep, the (192,128) points, the variable-length deterministic batch).
`value` = backward FLOPs 2*B*H*T^2*(3*dqk+2*dv)/2 (per sequence for a
variable-length batch) / backward time, summed over ranks.  Inputs of the
32K-token workloads (5 x 134 MB) exceed the 126 MB L2, so no flush is needed
between steps.  The same line carries the inference-mode forward
(`fwd_inference`), the time of the other dQ reduction mode (deterministic or
fast), the HBM rates of the two memory-bound kernels (`aux_kernels`) and the
end-to-end figure through host buffers (`e2e`).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--gpus N without a launcher starts N ranks itself (replicas, one per GPU);
under torchrun it must match WORLD_SIZE.  --impl reference times the fp64 CPU
oracle (the reference arm for this workload) on a bounded sample of the same
workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from attention_backward_flashattention_gb300 import binding  # noqa: E402
from attention_backward_flashattention_gb300 import synthetic as syn  # noqa: E402

METRIC = "attn bwd TFLOP/s (bf16, causal, d=128, 32K tok) and % of GB300 BF16 peak"
UNIT = "TFLOP/s"
WORKLOAD = syn.HEADLINE


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_burst": p["bf16_tflops"], "bf16_sustained": p["bf16_tflops_sustained"],
                "hbm": p["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def _config(w, extra=None):
    tensor_mb = w.total_tokens * w.H * w.dqk * 2 / 1e6
    l2 = (f"inputs larger than L2 (5 x {tensor_mb:.0f} MB bf16), no flush" if tensor_mb * 5 > 130
          else f"inputs ({5 * tensor_mb:.0f} MB) fit in L2: steps re-read them from L2")
    c = {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "dqk": w.dqk, "dv": w.dv,
         "causal": w.causal, "layout": "packed (B,T,3,H,d)" if w.layout == syn.LAYOUT_PACKED
         else ("varlen (sum T,H,d)" if w.varlen else "BTHD"),
         "deterministic": w.deterministic, "l2": l2}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


KERNEL_SOURCES = ("attn_bwd.cu", "attn_common.cuh", "attn_internal.h", "ptx.cuh")


def kernel_sources_sha256():
    """SHA-256 over the sources the backward main kernel is compiled from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "attention_backward_flashattention_gb300", "csrc", name),
                  "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _ncu_record(kernel_name, workload):
    """The committed ncu counters of `kernel_name` on `workload`
    (profiles/ncu_traffic.json, keyed by kernel, then workload) when the
    kernel's sources are unchanged since they were taken; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_name, {}).get(workload)
    if not rec or rec.get("sources_sha256") != kernel_sources_sha256():
        return None
    return rec


# ---------------------------------------------------------------------------
# workload plumbing (layouts, problems, byte counts)
# ---------------------------------------------------------------------------
def _cu(w):
    return None if not w.varlen else [0] + list(np.cumsum(w.varlen).astype(int))


def _lengths(w):
    return list(w.varlen) if w.varlen else [w.T] * w.B


def _q_tiles(w):
    return sum(-(-L // 128) for L in _lengths(w))


def aux_bytes(w):
    """Bytes the backward's two memory-bound kernels move per launch.

    preprocess: reads O and dO (bf16) and LSE, writes -D and -LSE*log2(e) per
    padded query row (fp32) and zeroes the fp32 dQ accumulator;
    'algorithmic' counts only the reads and the D / LSE writes (the operation
    D = rowsum(dO * O)), 'moved' adds the accumulator's zeroing.
    dQ conversion: reads the fp32 accumulator, writes bf16 dQ."""
    rows = w.total_tokens
    padded = _q_tiles(w) * 128
    H = w.H
    pre_alg = rows * H * (2 * w.dv * 2 + 4) + 2 * padded * H * 4
    pre_moved = pre_alg + padded * H * w.dqk * 4
    cvt = padded * H * w.dqk * 4 + rows * H * w.dqk * 2
    return {"pre_algorithmic": pre_alg, "pre_moved": pre_moved, "convert": cvt}


def _problems(t, cu):
    """(B,T,H,d) or (sum T,H,d) tensor -> list of float64 [T][d] per (sequence, head)."""
    t = t.float()
    if cu is None:
        x = t.permute(0, 2, 1, 3).contiguous()
        return list(x.reshape(-1, x.shape[2], x.shape[3]).double().numpy())
    return [t[cu[s]:cu[s + 1], h, :].double().numpy()
            for s in range(len(cu) - 1) for h in range(t.shape[1])]


# ---------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(w, rows_per_head, seed=0, x=None):
    """Time the oracle's row-by-row backward on `rows_per_head` random query
    rows of every (sequence, head) problem of `w` (one OpenMP thread per
    problem).  Returns (TFLOP/s in the metric's FLOP convention, seconds,
    threads, description)."""
    import oracle
    oracle.build()
    if x is None:
        x = syn.make_inputs(w)
    cu = _cu(w)
    q, k, v, dO = (_problems(x[n], cu) for n in ("q", "k", "v", "dO"))
    rng = np.random.default_rng(seed)
    rows = [np.sort(rng.choice(len(a), size=min(rows_per_head, len(a)), replace=False))
            .astype(np.int32) for a in q]
    per = 2.0 * (3 * w.dqk + 2 * w.dv)
    flops = sum(per * ((r + 1).sum() if w.causal else len(a) * len(r)) for r, a in zip(rows, q))
    t0 = time.perf_counter()
    oracle.backward(q, k, v, dO, w.causal, w.scale, rows=rows)
    dt = time.perf_counter() - t0
    desc = (f"oracle row-by-row backward (recomputes each row's forward), {rows_per_head} "
            f"random query rows x {len(q)} (sequence, head) problems of {w.name}; FLOPs "
            f"counted as the rows' share of 2*H*T^2*(3*dqk+2*dv)/2")
    return flops / dt / 1e12, dt, oracle.num_threads(), desc


def max_over_ranks(values, world, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the
    job's time); identity on one rank."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_tflops(flops_per_rank, world, steps, seconds):
    """Whole-job throughput: every rank processes `flops_per_rank` per step."""
    return world * flops_per_rank * steps / seconds / 1e12


def peak_for(peaks, timed_region_s):
    """The bf16 denominator for a kernel timed inside a region of this length:
    the burst figure below 2 s (the cuBLAS burst is a short loop too), the
    sustained one (measured over seconds under the power cap) above."""
    if timed_region_s < 2.0:
        return peaks["bf16_burst"], f"bf16 burst ({peaks['source']}; timed region " \
                                    f"{timed_region_s:.2f} s < 2 s)"
    return peaks["bf16_sustained"], f"bf16 sustained ({peaks['source']}; timed region " \
                                    f"{timed_region_s:.2f} s)"


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Problem:
    """Device tensors of one workload in its own layout, and the C-ABI calls
    of its forward and backward (argument marshalling only)."""

    def __init__(self, w, x, dev):
        self.w = w
        self.cu = _cu(w)
        self.varlen = self.cu is not None
        B, H, dqk, dv = w.B, w.H, w.dqk, w.dv
        self.Tq = w.total_tokens if self.varlen else w.T
        if w.layout == syn.LAYOUT_PACKED:
            self.qkv = x["qkv"].to(dev)
            self.q, self.k, self.v = (self.qkv.select(-3, i) for i in range(3))
            self.gqkv = torch.empty_like(self.qkv)
            self.dq, self.dk, self.dv = (self.gqkv.select(-3, i) for i in range(3))
        else:
            self.q, self.k, self.v = (x[n].to(dev) for n in ("q", "k", "v"))
            self.dq, self.dk, self.dv = (torch.empty_like(t) for t in (self.q, self.k, self.v))
        self.dO = x["dO"].to(dev)
        lead = (self.Tq,) if self.varlen else (B, w.T)
        self.o = torch.empty(*lead, H, dv, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(*((H, self.Tq) if self.varlen else (B, H, w.T)),
                               dtype=torch.float32, device=dev)
        self.ws_bytes = binding.attn_bwd_workspace_size(B, H, self.Tq, self.Tq, dqk, dv,
                                                        self.varlen, True)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)

    def fwd(self, stream, with_lse=True):
        w = self.w
        rc = binding.attn_fwd(self.q, self.k, self.v, self.o, self.lse if with_lse else None,
                              w.B, w.H, self.Tq, self.Tq, w.dqk, w.dv, w.causal, w.scale,
                              self.cu, w.layout, stream)
        assert rc == 0, rc

    def bwd(self, stream, deterministic):
        w = self.w
        rc = binding.attn_bwd(self.q, self.k, self.v, self.o, self.dO, self.lse, self.dq,
                              self.dk, self.dv, w.B, w.H, self.Tq, self.Tq, w.dqk, w.dv,
                              w.causal, w.scale, self.cu, w.layout, deterministic, self.ws,
                              self.ws_bytes, stream)
        assert rc == 0, rc

    def status_ok(self):
        return binding.attn_bwd_status(self.ws) == 0 and binding.attn_fwd_status() == 0


def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _time_loop(stream, steps, body):
    """Device time (ms) of `steps` calls of body(), CUDA events on `stream`."""
    a, b = _events(2)
    a.record(stream)
    for _ in range(steps):
        body()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def e2e_step_host(args, w, x, dev, stream, K):
    """Host tensors in, gradients out, through attn_step_host (fixed-length
    (B,T,H,d) only): ms per step and the bytes copied each way.

    With --e2e-slots 2 (the default) consecutive steps alternate between two
    scratch buffers, each with its own streams and host output tensors, the
    way a training loop double-buffers its batches: step k+1's input copies
    run while step k's kernels and gradient copies finish.  Every step still
    copies all its inputs in and all its gradients out inside the timed
    region."""
    B, H, T, dqk, dv = w.B, w.H, w.T, w.dqk, w.dv
    hq, hk, hv, hdo = (x[n].pin_memory() for n in ("q", "k", "v", "dO"))
    G = args.e2e_heads_per_group
    scratch_bytes = binding.attn_step_host_scratch_size(B, H, T, dqk, dv, G, w.deterministic)
    slots = []
    for i in range(max(1, args.e2e_slots)):
        slots.append({
            "out": tuple(torch.empty(x[n].shape, dtype=torch.bfloat16, pin_memory=True)
                         for n in ("q", "k", "v")),
            "scratch": torch.empty(scratch_bytes, dtype=torch.uint8, device=dev),
            "cs": stream if i == 0 else torch.cuda.Stream(dev),
            "cs2": torch.cuda.Stream(dev) if args.e2e_streams == 2 else None,
            "hs": torch.cuda.Stream(dev), "ds": torch.cuda.Stream(dev)})
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in slots[0]["out"])

    def step(k):
        sl = slots[k % len(slots)]
        hdq, hdk, hdv = sl["out"]
        rc = binding.attn_step_host(hq, hk, hv, hdo, None, hdq, hdk, hdv, B, H, T, dqk, dv,
                                    w.causal, w.scale, w.deterministic, G, sl["scratch"],
                                    scratch_bytes, sl["cs"], sl["cs2"], sl["hs"], sl["ds"])
        assert rc == 0, rc

    def status_ok():
        return all(binding.attn_step_host_status(sl["scratch"], B, H, T, dqk, dv, G,
                                                 w.deterministic, sl["cs"]) == 0 for sl in slots)

    for k in range(len(slots)):
        step(k)
    torch.cuda.synchronize()
    if not status_ok():
        raise RuntimeError("device status error in the e2e warm-up")
    a, b = _events(2)
    a.record(stream)
    for sl in slots[1:]:
        sl["cs"].wait_event(a)
    for k in range(K):
        step(k)
    for sl in slots[1:]:
        e = torch.cuda.Event()
        e.record(sl["cs"])
        stream.wait_event(e)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    if not status_ok():
        raise RuntimeError("device status error in the e2e region")
    api = ("attn_step_host (pinned host tensors; forward + backward; copies of one head group "
           "overlap the kernels of another"
           + ("; consecutive steps alternate between %d scratch buffers, so one step's copies "
              "overlap the next step's kernels" % len(slots) if len(slots) > 1 else "") + ")")
    return ms, h2d, d2h, api, {"heads_per_group": G or -(-H // 2),
                               "compute_streams": args.e2e_streams, "slots": len(slots)}


def e2e_copies(w, x, prob, stream, K):
    """Layouts attn_step_host does not take (packed QKV, variable length):
    pinned host inputs copied in, attn_fwd + attn_bwd, gradients copied out,
    all on one stream."""
    names = ("qkv", "dO") if w.layout == syn.LAYOUT_PACKED else ("q", "k", "v", "dO")
    host_in = [x[n].contiguous().pin_memory() for n in names]
    dev_in = [prob.qkv, prob.dO] if w.layout == syn.LAYOUT_PACKED else \
        [prob.q, prob.k, prob.v, prob.dO]
    dev_out = [prob.gqkv] if w.layout == syn.LAYOUT_PACKED else [prob.dq, prob.dk, prob.dv]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def step():
        with torch.cuda.stream(stream):
            for h, d in zip(host_in, dev_in):
                d.copy_(h, non_blocking=True)
            prob.fwd(stream)
            prob.bwd(stream, w.deterministic)
            for d, h in zip(dev_out, host_out):
                h.copy_(d, non_blocking=True)

    step()
    torch.cuda.synchronize()
    ms = _time_loop(stream, K, step) / K
    if not prob.status_ok():
        raise RuntimeError("device status error in the e2e region")
    return ms, h2d, d2h, "pinned host copies in, attn_fwd + attn_bwd, gradients out (one stream)", {}


def run_ours(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = WORKLOAD
    x = syn.make_inputs(w)
    prob = Problem(w, x, dev)
    stream = torch.cuda.current_stream()
    det = w.deterministic
    launches_per_step = 1 + 3
    for _ in range(args.warmup):
        prob.fwd(stream)
        prob.bwd(stream, det)
    torch.cuda.synchronize()
    if not prob.status_ok():
        raise RuntimeError("device status error during warm-up")

    K = args.steps
    ev = [_events(9) for _ in range(K)]
    for e in ev:       # create the events before the timed region
        for z in e:
            z.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler()
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start, t_stop = _events(2)
    t_start.record(stream)
    for i in range(K):
        e = ev[i]
        e[0].record(stream)
        prob.fwd(stream)
        e[1].record(stream)
        binding.attn_profile_main_kernel(e[3], e[4])
        binding.attn_profile_aux_kernels(e[5], e[6], e[7], e[8])
        prob.bwd(stream, det)
        e[2].record(stream)
    t_stop.record(stream)
    torch.cuda.synchronize()
    binding.attn_profile_main_kernel(None, None)
    binding.attn_profile_aux_kernels(None, None, None, None)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if rank == 0 else None
    total_ms = t_start.elapsed_time(t_stop)
    sums = [sum(ev[i][a].elapsed_time(ev[i][b]) for i in range(K))
            for a, b in ((0, 1), (1, 2), (3, 4), (5, 6), (7, 8))]
    if not prob.status_ok():
        raise RuntimeError("device status error in the timed region")

    # end to end through host buffers, right after the device-timed steps (as a
    # caller would run it), with its own clock record
    e2e_sampler = ClockSampler()
    if rank == 0:
        e2e_sampler.start()
    if w.layout == syn.LAYOUT_BTHD and not w.varlen:
        e2e_ms, h2d, d2h, api, e2e_extra = e2e_step_host(args, w, x, dev, stream, K)
    else:
        e2e_ms, h2d, d2h, api, e2e_extra = e2e_copies(w, x, prob, stream, K)
    e2e_clocks = e2e_sampler.stop() if rank == 0 else None

    # inference-mode forward (lse = NULL) and the other dQ reduction mode
    inf_ms = _time_loop(stream, K, lambda: prob.fwd(stream, with_lse=False))
    Kd = min(K, 10)
    other_ms = _time_loop(stream, Kd, lambda: prob.bwd(stream, not det))
    if not prob.status_ok():
        raise RuntimeError("device status error in the extra timings")

    total_ms, fwd_sum, bwd_sum, main_sum, pre_sum, cvt_sum, inf_ms, other_ms, e2e_ms = \
        max_over_ranks([total_ms, *sums, inf_ms, other_ms, e2e_ms], world, dev)
    if rank != 0:
        return None

    peaks = _peaks()
    bwd_flops, fwd_flops = w.bwd_flops(), w.fwd_flops()
    value = job_tflops(bwd_flops, world, K, bwd_sum * 1e-3)
    main_avg_s = main_sum / K * 1e-3
    achieved = bwd_flops / main_avg_s / 1e12
    timed_region_s = total_ms * 1e-3
    peak, peak_kind = peak_for(peaks, timed_region_s)
    rec = _ncu_record("attn_bwd_main_kernel", w.name)
    nb = aux_bytes(w)
    pre_s, cvt_s = pre_sum / K * 1e-3, cvt_sum / K * 1e-3
    aux = {
        "attn_bwd_pre_kernel": {
            "avg_ms": pre_s * 1e3, "bytes_moved": nb["pre_moved"],
            "bytes_algorithmic": nb["pre_algorithmic"],
            "gbs": nb["pre_moved"] / pre_s / 1e9,
            "frac_of_hbm": nb["pre_moved"] / pre_s / 1e9 / peaks["hbm"],
            "gbs_algorithmic": nb["pre_algorithmic"] / pre_s / 1e9},
        "attn_bwd_convert_kernel": {
            "avg_ms": cvt_s * 1e3, "bytes_moved": nb["convert"],
            "gbs": nb["convert"] / cvt_s / 1e9,
            "frac_of_hbm": nb["convert"] / cvt_s / 1e9 / peaks["hbm"]},
        "hbm_peak_gbs": peaks["hbm"], "unit": "GB/s",
        "bytes": "moved = every byte the kernel reads or writes as built (the preprocess also "
                 "zeroes the fp32 dQ accumulator); algorithmic = O, dO, LSE read and D written",
    }
    inf_per = fwd_flops / (inf_ms / K * 1e-3) / 1e12
    fwd_inf = {"value": world * inf_per, "unit": UNIT, "ms": inf_ms / K,
               "frac_of_burst": inf_per / peaks["bf16_burst"],
               "mode": "attn_fwd with lse = NULL (inference: no statistics written)"}
    det_key = "bwd_fast_ms" if det else "bwd_deterministic_ms"
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        tf, secs, cores, desc = oracle_sample(w, args.cpu_rows, x=x)
        cpu = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc, "seconds": round(secs, 2)}
    extra = {"parallelism": f"replicas x{world} (independent heads, no exchange)",
             "bwd_kernel": args.bwd_kernel}
    if w.varlen:
        extra["seqlens"] = list(w.varlen)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(w, extra),
        "pct_of_bf16_peak": {"burst": 100.0 * value / world / peaks["bf16_burst"],
                             "sustained": 100.0 * value / world / peaks["bf16_sustained"],
                             "peaks": peaks["source"]},
        "bwd_ms": bwd_sum / K, "fwd_ms": fwd_sum / K,
        "fwd_tflops": world * fwd_flops * K / (fwd_sum * 1e-3) / 1e12,
        "fwd_inference": fwd_inf,
        det_key: other_ms / Kd,
        "deterministic_cost_pct": 100.0 * ((bwd_sum / K) / (other_ms / Kd) - 1.0) if det else
        100.0 * ((other_ms / Kd) / (bwd_sum / K) - 1.0),
        "roofline": {"kernel": "attn_bwd_main_kernel", "bound": "tensor", "achieved": achieved,
                     "peak": peak, "unit": UNIT, "frac": achieved / peak,
                     "peak_kind": peak_kind,
                     "frac_of_burst": achieved / peaks["bf16_burst"],
                     "frac_of_sustained": achieved / peaks["bf16_sustained"],
                     "traffic": None if rec is None else rec["bytes_per_launch"],
                     "tensor_pipe_pct_ncu": None if rec is None else rec.get("tensor_pipe_pct"),
                     "algorithmic_flops_per_launch": bwd_flops,
                     "avg_launch_ms": main_avg_s * 1e3},
        "aux_kernels": aux,
        "cpu_baseline": cpu,
        "e2e": {"value": world * bwd_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "api": api, "clocks": e2e_clocks, **e2e_extra},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    return line


def run_fwd_only(args, rank, world):
    """Inference-mode forward (lse=NULL) of the workload alone: forward TFLOP/s.
    A separate measurement (`--fwd-only`); the default line carries the same
    figure as `fwd_inference`."""
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = WORKLOAD
    x = syn.make_inputs(w)
    prob = Problem(w, x, dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        prob.fwd(stream, with_lse=False)
    torch.cuda.synchronize()
    K = args.steps
    sampler = ClockSampler()
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total_ms = _time_loop(stream, K, lambda: prob.fwd(stream, with_lse=False))
    clocks = sampler.stop() if rank == 0 else None
    if binding.attn_fwd_status() != 0:
        raise RuntimeError("device status error in the timed region")
    (total_ms,) = max_over_ranks([total_ms], world, dev)
    if rank != 0:
        return None
    peaks = _peaks()
    flops = w.fwd_flops()
    value = job_tflops(flops, world, K, total_ms * 1e-3)
    per = flops / (total_ms / K * 1e-3) / 1e12
    peak, peak_kind = peak_for(peaks, total_ms * 1e-3)
    return {
        "metric": "attn fwd TFLOP/s (bf16, inference: no LSE)", "value": value, "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": _config(w, {"mode": "forward only, lse=NULL"}),
        "roofline": {"kernel": "attn_fwd_kernel", "bound": "tensor", "achieved": per,
                     "peak": peak, "unit": UNIT, "frac": per / peak, "peak_kind": peak_kind,
                     "frac_of_burst": per / peaks["bf16_burst"], "traffic": None,
                     "algorithmic_flops_per_launch": flops},
        "gpu_launches": K, "clocks": clocks,
    }


def block_sparse_mask(w, density, seed=0):
    """Seeded random block mask of workload `w`, one per head: each pair of
    128-row blocks kept with probability `density`, the diagonal always kept
    (every query then sees at least its own block).  uint8 [1][H][n][n]."""
    n = -(-w.T // 128)
    m = (np.random.default_rng(seed).random((1, w.H, n, n)) < density).astype(np.uint8)
    m[..., np.arange(n), np.arange(n)] = 1
    return m


def visible_pairs(w, mask):
    """(query, key) pairs that the kept blocks and the causal band leave, summed
    over heads and batch (the FLOP count's pair term; T a multiple of 128)."""
    n = mask.shape[-1]
    qt, kt = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    per_pair = np.full((n, n), 128.0 * 128.0)
    if w.causal:
        per_pair = np.where(kt < qt, 128.0 * 128.0, np.where(kt == qt, 128.0 * 129.0 / 2, 0.0))
    return w.B * float((mask.astype(np.float64) * per_pair).sum())


def run_block_sparse(args, rank, world):
    """Forward + backward of the workload under a random block mask of the
    given density (`--block-density`): TFLOP/s over the visible pairs only.
    A separate measurement (not the headline line)."""
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = WORKLOAD
    if w.varlen or w.layout != syn.LAYOUT_BTHD:
        raise ValueError("the block-sparse bench takes fixed-length (B,T,H,d) workloads")
    if w.T % 128:
        raise ValueError("block-sparse bench wants T a multiple of 128")
    x = syn.make_inputs(w)
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    mask = block_sparse_mask(w, args.block_density, seed=rank)
    bm = torch.from_numpy(mask).to(dev)
    B, H, T, dqk, dv = w.B, w.H, w.T, w.dqk, w.dv
    o = torch.empty(B, T, H, dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    dq, dk, dvt = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = binding.attn_bwd_workspace_size(B, H, T, T, dqk, dv, False, False)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    wl, wr = -1, -1

    def fwd():
        rc = binding.attn_fwd_ex(q, k, v, o, lse, B, H, T, T, dqk, dv, w.causal, wl, wr, bm, 1,
                                 H, w.scale, None, None, 0, stream)
        assert rc == 0, rc

    def bwd():
        rc = binding.attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dvt, B, H, T, T, dqk, dv, w.causal,
                                 wl, wr, bm, 1, H, w.scale, None, None, 0, False, ws, need,
                                 stream)
        assert rc == 0, rc

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    K = args.steps
    sampler = ClockSampler()
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * K)]
    for s_ in range(K):  # the inputs (> L2) are re-read from HBM every step
        ev[3 * s_].record(stream)
        fwd()
        ev[3 * s_ + 1].record(stream)
        bwd()
        ev[3 * s_ + 2].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if rank == 0 else None
    if binding.attn_fwd_status() != 0 or binding.attn_bwd_status(ws) != 0:
        raise RuntimeError("device status error in the timed region")
    fwd_ms = sum(ev[3 * s_].elapsed_time(ev[3 * s_ + 1]) for s_ in range(K))
    bwd_ms = sum(ev[3 * s_ + 1].elapsed_time(ev[3 * s_ + 2]) for s_ in range(K))
    fwd_ms, bwd_ms = max_over_ranks([fwd_ms, bwd_ms], world, dev)
    if rank != 0:
        return None
    pairs = visible_pairs(w, mask)
    bwd_flops = 2.0 * pairs * (3 * dqk + 2 * dv)
    fwd_flops = 2.0 * pairs * (dqk + dv)
    peaks = _peaks()
    per = bwd_flops / (bwd_ms / K * 1e-3) / 1e12
    kept = float(mask.mean())
    return {
        "metric": "attn bwd TFLOP/s (bf16, block-sparse, visible pairs only)",
        "value": job_tflops(bwd_flops, world, K, bwd_ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": bwd_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": _config(w, {"block_mask": f"random per head, density {args.block_density} "
                                            f"(diagonal kept; {kept:.3f} of block pairs kept)",
                              "dense_bwd_flops": w.bwd_flops()}),
        "fwd_tflops": job_tflops(fwd_flops, world, K, fwd_ms * 1e-3), "fwd_ms": fwd_ms / K,
        "roofline": {"kernel": "attn_bwd (pre + main + convert)", "bound": "tensor",
                     "achieved": per, "peak": peak_for(peaks, (fwd_ms + bwd_ms) * 1e-3)[0],
                     "unit": UNIT,
                     "frac": per / peak_for(peaks, (fwd_ms + bwd_ms) * 1e-3)[0],
                     "peak_kind": peak_for(peaks, (fwd_ms + bwd_ms) * 1e-3)[1], "traffic": None,
                     "algorithmic_flops_per_launch": bwd_flops},
        "gpu_launches": 4 * K, "clocks": clocks,
    }


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = WORKLOAD
    x = syn.make_inputs(w)
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(w, max(4, rows // 8), seed=1000, x=x)
    tfs, secs = [], []
    desc, cores = "", 1
    for s in range(args.steps):
        tf, dt, cores, desc = oracle_sample(w, rows, seed=s, x=x)
        tfs.append(tf)
        secs.append(dt)
    value = sum(tf * dt for tf, dt in zip(tfs, secs)) / sum(secs)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(secs) / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def launch_ranks(n):
    """`--gpus N` without a launcher: start N ranks of this command under
    torch.distributed.run (one process per GPU, rendezvous on 127.0.0.1) and
    return their exit status."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    global WORKLOAD
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--cpu-rows", type=int, default=1024, help="oracle rows per head (cpu_baseline)")
    ap.add_argument("--workload", default=syn.HEADLINE.name,
                    help="workload name: " + ", ".join(syn.ALL))
    ap.add_argument("--ref-rows", type=int, default=48, help="oracle rows per head per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-heads-per-group", type=int, default=0,
                    help="head-group size of the e2e pipeline (0: the library's choice)")
    ap.add_argument("--e2e-streams", type=int, default=1, choices=(1, 2),
                    help="compute streams of the e2e pipeline")
    ap.add_argument("--e2e-slots", type=int, default=2, choices=(1, 2),
                    help="scratch buffers that consecutive e2e steps alternate between")
    ap.add_argument("--fwd-only", action="store_true",
                    help="time the inference-mode forward (lse=NULL) instead of the step")
    ap.add_argument("--block-density", type=float, default=0.0,
                    help="time forward + backward under a random block mask of this density")
    ap.add_argument("--bwd-kernel", default="auto", choices=("auto", "one-cta", "cta-pair"),
                    help="backward main kernel where both apply (d=128, no block mask)")
    args = ap.parse_args()
    if args.workload not in syn.ALL:
        ap.error(f"unknown workload {args.workload!r}")
    WORKLOAD = syn.ALL[args.workload]
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus > 1:
        sys.exit(launch_ranks(args.gpus))
    world = int(env_world or "1")
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        sys.exit(2)
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group(backend=backend)
    if args.impl == "ours":
        from attention_backward_flashattention_gb300 import build as build_mod
        if rank == 0 or world == 1:
            build_mod.build()
        if world > 1:
            torch.distributed.barrier()
        binding.attn_debug_set_bwd_variant({"auto": 0, "one-cta": 1, "cta-pair": 2}[args.bwd_kernel])
        if args.block_density > 0:
            line = run_block_sparse(args, rank, world)
        elif args.fwd_only:
            line = run_fwd_only(args, rank, world)
        else:
            line = run_ours(args, rank, world)
    else:
        line = run_reference(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
