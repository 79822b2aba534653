#!/usr/bin/env python3
"""Benchmark of the Ulysses attention layer on GB300.

One step is the whole hot path on one batch of seeded synthetic input:

  Q, K, V seq->head, attention forward, O head->seq,
  dO seq->head, attention backward, dQ, dK, dV head->seq

(forward-only workloads stop after O head->seq). The default workload is the
Llama-8B-shaped forward+backward layer at sl=32768: P=8 virtual ranks, 32 query
heads, 8 kv heads, head size 128, bf16, causal.

Where the shape allows it (``--path auto``, the default), the step runs the
fused entry points ulysses_layer_fwd / ulysses_layer_bwd: the exchanges happen
inside the attention kernels, which read and write the sequence shards through
their TMA tensor maps. ``--path explicit`` runs the exchange kernels between
the attention calls instead. Either way the exchange kernels are also timed in
a loop of their own, for the exchange GB/s part of the metric.

Output: one JSON line on rank 0. ``value`` is tokens/s over the whole job,
timed with CUDA events with inputs already resident in HBM. ``e2e`` is the
same metric through the public API, with the host->device copy of the step's
inputs and the device->host copy of its outputs inside the timed region.
``--impl reference`` times the CPU oracle instead, on a bounded sample.

At N = 1 the line also carries ``configs``: short timed runs, in the same
process after the headline one, of every other workload (the 128K layer with
a rows/s figure for the oracle's 1024-row spot check, the packed 64K layer,
the 8K forward, and the tiny fp32 layer with the whole oracle timed on all
host cores and on one), each with its kernels' rates and fractions.
``--no-configs`` skips them.

Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own GPU. The path has no exchange between GPUs: all P ranks of one layer
are virtual shards on one GPU. Rank 0 prints the job line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import WORKLOADS, doc_offsets_for, make_global_inputs, split_shards  # noqa: E402

METRIC = "attn fwd+bwd tokens/s & TFLOPS (% bf16 peak); exchange GB/s (% HBM) at 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# Work accounting (algorithmic, not measured)
# ---------------------------------------------------------------------------
def visible_pairs(sl, causal, offs):
    """Visible (query, key) pairs of one (batch, head): the work the mask leaves."""
    offs = offs or [0, sl]
    tot = 0
    for a, b in zip(offs[:-1], offs[1:]):
        n = b - a
        tot += n * (n + 1) // 2 if causal else n * n
    return tot


def attn_flops(w, sl=None, offs=None):
    """Forward flops: 2 GEMMs (QK^T, PV) of 2*hs flops per visible pair and head."""
    sl = sl or w.sl
    offs = offs if offs is not None else doc_offsets_for(w)
    return 4.0 * w.hs * w.hc * w.bs * visible_pairs(sl, w.causal, offs)


def exchange_bytes(w, H):
    """One exchange reads and writes the whole [sl, bs, H, hs] tensor once."""
    return 2.0 * w.sl * w.bs * H * w.hs * w.elem_bytes


KERNEL_SOURCES = {
    "attn_bwd_dkdv_kernel<0>": "ulysses_sequence_attention_gb300/csrc/attn_bwd_sm103.cu",
    "attn_bwd_dkdv_kernel<1>": "ulysses_sequence_attention_gb300/csrc/attn_bwd_sm103.cu",
    "attn_bwd_dq_kernel": "ulysses_sequence_attention_gb300/csrc/attn_bwd_sm103.cu",
    "attn_bwd_dq_stored_kernel": "ulysses_sequence_attention_gb300/csrc/attn_bwd_sm103.cu",
    "attn_fwd_sm103_kernel": "ulysses_sequence_attention_gb300/csrc/attn_fwd_sm103.cu",
}


def kernel_work(w, offs, ds_bytes=0):
    """Per timed kernel id: (CUDA kernel name, bound, algorithmic work of one step, unit).

    Tensor kernels count 2*hs flops per visible (query, key) pair, head and
    GEMM. The forward needs 2 GEMMs (S = Q K^T, O = P V). The dK/dV kernel
    needs 4 (S, dP = dO V^T, dV = P^T dO, dK = dS^T Q), none of them repeated
    inside it. The recomputing dQ kernel issues 3 (S, dP, dQ = dS K), of which
    S and dP repeat the dK/dV kernel's: its algorithmic share of the 5-GEMM
    backward is the dQ GEMM alone. With stored dS (ds_bytes > 0: the area's
    blocks, zero block excluded) the dQ kernel is one GEMM at 128 flops per
    byte of dS, below the machine balance: it is counted as byte-bound, one
    read of every stored block, of K and one write of dQ. Byte-bound kernels
    count one read and one write of what they move.
    """
    fl2 = attn_flops(w, offs=offs) / 2.0   # one GEMM over the visible pairs
    tok = w.sl * w.bs
    eb = w.elem_bytes
    dq = (("attn_bwd_dq_stored_kernel", "hbm", ds_bytes + tok * (w.hc + w.hkv) * w.hs * eb, "byte") if ds_bytes
          else ("attn_bwd_dq_kernel", "tensor", 1 * fl2, "flop"))
    return {
        "attn_fwd": ("attn_fwd_sm103_kernel", "tensor", 2 * fl2, "flop"),
        # <1>: the instantiation that also writes dS
        "bwd_dkdv": ("attn_bwd_dkdv_kernel<1>" if ds_bytes else "attn_bwd_dkdv_kernel<0>", "tensor", 4 * fl2, "flop"),
        "bwd_dq": dq,
        "bwd_prep": ("attn_bwd_prep_kernel", "hbm", tok * w.hc * (2 * w.hs * eb + 4), "byte"),
        "seq_to_head": ("seq_to_head_kernel", "hbm",
                        exchange_bytes(w, w.hc) * (2 if w.backward else 1) + 2 * exchange_bytes(w, w.hkv), "byte"),
        "head_to_seq": ("head_to_seq_kernel", "hbm",
                        exchange_bytes(w, w.hc) * (2 if w.backward else 1)
                        + (2 * exchange_bytes(w, w.hkv) if w.backward else 0), "byte"),
    }


def captured_traffic(kernel, workload):
    """DRAM bytes per launch from the ncu summary in profiles/traffic.txt.

    The figure applies only while the kernel's source is the one that was
    captured (sha256 prefix); otherwise the traffic is unknown (None).
    """
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = KERNEL_SOURCES.get(kernel)
    if not os.path.exists(path) or src is None:
        return None, None
    digest = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            if parts[2] != digest or parts[3] == "null":
                return None, None
            return float(parts[3]), " ".join(parts[4:])
    return None, None


def max_over_ranks(ms: float, device, world: int) -> float:
    """The job's time: the largest of the ranks' times (all ranks get it)."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank_step: int, steps: int, world: int, job_ms: float) -> float:
    """Whole-job throughput: the tokens every rank processed over the job's (slowest rank's) time."""
    return tokens_per_rank_step * steps * world / (job_ms / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# Our implementation
# ---------------------------------------------------------------------------
def device_inputs(w, dev):
    """N(0,1) sequence shards drawn on the device from a generator seeded with the workload's seed.

    For the throughput-only configurations beside the headline workload: the
    kernels' work depends on the shapes and the mask, not on the values, and
    a device draw avoids minutes of host-side generation at 128K tokens.
    """
    g = torch.Generator(device=dev).manual_seed(w.seed)
    n = w.sl // w.P

    def shards(H):
        return [torch.randn((n, w.bs, H, w.hs), generator=g, device=dev).to(w.torch_dtype) for _ in range(w.P)]

    out = {"q": shards(w.hc), "k": shards(w.hkv), "v": shards(w.hkv)}
    if w.backward:
        out["do"] = shards(w.hc)
    return out


def run_ours(args, w, rank, world, steps=None, warmup=None, with_e2e=None, on_device=False):
    """Time the layer on workload w; returns the raw timings (run_summary turns them into rates)."""
    import ulysses_sequence_attention_gb300 as U
    from ulysses_sequence_attention_gb300 import _binding as B

    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    with_e2e = (not args.no_e2e) if with_e2e is None else with_e2e
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    offs = doc_offsets_for(w)
    P = w.P
    if on_device:
        x = None
        seq = device_inputs(w, dev)
    else:
        x = make_global_inputs(w)
        seq = {k: [t.to(dev) for t in split_shards(v, P)] for k, v in x.items()}
    fused = None if args.path == "auto" else args.path == "fused"
    L = U.UlyssesLayer(w.sl, w.bs, w.hc, w.hkv, w.hs, P, w.causal, offs, w.torch_dtype, device=str(dev),
                       fused=fused, ds_budget=args.ds_budget)
    o = L.new_seq_shards(w.hc)
    if w.backward:
        dq, dk, dv = L.new_seq_shards(w.hc), L.new_seq_shards(w.hkv), L.new_seq_shards(w.hkv)
    h = L.h
    stream = torch.cuda.current_stream(dev)
    ev = {}

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        ev.setdefault(name, []).append(e)

    def heads(H):
        return [torch.empty((w.sl, w.bs, H, w.hs), dtype=w.torch_dtype, device=dev) for _ in range(P)]

    # Head-shard buffers: the explicit path's intermediates, and the targets of
    # the exchange measurement on either path.
    hb = {"qh": heads(L.Hq), "kh": heads(L.Hk), "vh": heads(L.Hk), "oh": heads(L.Hq)}
    if w.backward:
        hb.update(doh=heads(L.Hq), dqh=heads(L.Hq), dkh=heads(L.Hk), dvh=heads(L.Hk))
    lse = [torch.empty((w.bs, L.Hq, w.sl), dtype=torch.float32, device=dev) for _ in range(P)]
    ws = torch.empty((max(B.ulysses_workspace_size(h), 16) + 3) // 4, dtype=torch.float32, device=dev)

    def step(timed):
        """One pass of the whole hot path on resident inputs."""
        if L.fused:
            if timed:
                mark("fwd0")
            B.ulysses_layer_fwd(h, seq["q"], seq["k"], seq["v"], o, lse)
            if timed:
                mark("fwd1")
            if w.backward:
                B.ulysses_layer_bwd(h, seq["q"], seq["k"], seq["v"], o, seq["do"], lse, dq, dk, dv, ws)
                if timed:
                    mark("bwd1")
            return
        if timed:
            mark("fwd0")
        B.ulysses_seq_to_head_qkv(h, seq["q"], seq["k"], seq["v"], hb["qh"], hb["kh"], hb["vh"])
        B.ulysses_attn_fwd(h, hb["qh"], hb["kh"], hb["vh"], hb["oh"], lse)
        B.ulysses_head_to_seq(h, w.hc, hb["oh"], o)
        if timed:
            mark("fwd1")
        if w.backward:
            B.ulysses_seq_to_head(h, w.hc, seq["do"], hb["doh"])
            B.ulysses_attn_bwd(h, hb["qh"], hb["kh"], hb["vh"], hb["oh"], hb["doh"], lse,
                               hb["dqh"], hb["dkh"], hb["dvh"], ws)
            B.ulysses_head_to_seq_qkv(h, hb["dqh"], hb["dkh"], hb["dvh"], dq, dk, dv)
            if timed:
                mark("bwd1")

    def exchange_step():
        """The explicit exchanges of one step: Q, K, V (and dO) seq->head, O (and dQ, dK, dV) head->seq."""
        mark("x0")
        B.ulysses_seq_to_head_qkv(h, seq["q"], seq["k"], seq["v"], hb["qh"], hb["kh"], hb["vh"])
        mark("x1")
        B.ulysses_head_to_seq(h, w.hc, hb["oh"], o)
        mark("x2")
        if w.backward:
            B.ulysses_seq_to_head(h, w.hc, seq["do"], hb["doh"])
            B.ulysses_head_to_seq_qkv(h, hb["dqh"], hb["dkh"], hb["dvh"], dq, dk, dv)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def read_timing():
        out = {}
        for i, name in enumerate(U.KERNEL_NAMES):
            ms, n = U.ulysses_timing_read(h, i)
            if n:
                out[name] = {"total_ms": ms, "launches": n, "ms_per_step": ms / steps}
        return out

    for _ in range(warmup):
        step(False)
    torch.cuda.synchronize(dev)
    st = U.ulysses_get_status(h)
    if st != U.ULYSSES_OK:
        raise RuntimeError(f"device status after warm-up: {U.ulysses_strerror(st)}")

    clocks = ClockSampler(dev.index)
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    n0 = U.ulysses_launch_count()
    U.ulysses_timing_enable(h, True)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step(True)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    launches = U.ulysses_launch_count() - n0
    kernels = read_timing()
    U.ulysses_timing_enable(h, False)
    clk = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    if U.ulysses_get_status(h) != U.ULYSSES_OK:
        raise RuntimeError("device status after the timed region is not OK")

    # The exchange kernels, timed on their own (on the fused path the step
    # runs none: the attention kernels read and write the sequence shards).
    for _ in range(3):
        exchange_step()
    torch.cuda.synchronize(dev)
    ev.pop("x0", None), ev.pop("x1", None), ev.pop("x2", None)
    U.ulysses_timing_enable(h, True)
    for _ in range(steps):
        exchange_step()
    torch.cuda.synchronize(dev)
    xk = read_timing()
    U.ulysses_timing_enable(h, False)
    for name in ("seq_to_head", "head_to_seq"):
        if name in xk:
            kernels.setdefault(name, dict(xk[name], region="exchange-only loop of the same step's exchanges"))

    def span(a, z):
        return [ea.elapsed_time(ez) for ea, ez in zip(ev[a], ev[z])]

    fwd_ms = statistics.mean(span("fwd0", "fwd1"))
    bwd_ms = statistics.mean(span("fwd1", "bwd1")) if w.backward else 0.0
    s2h_ms = statistics.mean(span("x0", "x1"))
    h2s_ms = statistics.mean(span("x1", "x2"))

    elapsed_ms = max_over_ranks(elapsed_ms, dev, world)
    ms_per_step = elapsed_ms / steps
    value = job_tokens_per_s(w.sl * w.bs, steps, world, elapsed_ms)

    e2e = None
    if with_e2e and x is not None:
        e2e = run_e2e(args, w, L, x, dev, world, barrier)

    result = {"ms_per_step": ms_per_step, "value": value, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
              "s2h_qkv_ms": s2h_ms, "h2s_o_ms": h2s_ms, "launches": launches, "clocks": clk, "e2e": e2e,
              "kernels": kernels, "path": "fused" if L.fused else "explicit",
              "ds_bytes": B.ulysses_ds_bytes(h)[0] if L.stores_ds else 0, "steps": steps,
              "timed_s": elapsed_ms / 1e3}
    del L, seq, hb, ws, lse, o
    if w.backward:
        del dq, dk, dv
    torch.cuda.empty_cache()
    return result


def run_e2e(args, w, L, x, dev, world, barrier):
    """The same metric through the public API with host<->device copies in the timed region.

    Fused shapes go through HostSteps (ulysses_host_begin/_step/_end): each
    step copies its Q/K/V/dO shards in from pinned host memory and its
    O/dQ/dK/dV shards out, on the library's copy streams, overlapped with the
    neighbouring steps' kernels. Other shapes run UlyssesLayer with the copies
    on the compute stream. CUDA events on the compute stream bracket the run;
    ulysses_host_end makes the closing event wait for every copy.
    """
    import ulysses_sequence_attention_gb300 as U
    P = w.P
    stream = torch.cuda.current_stream(dev)
    pin = {k: [t.pin_memory() for t in split_shards(v, P)] for k, v in x.items()}

    def host_out():
        mk = lambda H: [torch.empty((w.sl // P, w.bs, H, w.hs), dtype=w.torch_dtype, pin_memory=True)  # noqa: E731
                        for _ in range(P)]
        return {"o": mk(w.hc), "dq": mk(w.hc), "dk": mk(w.hkv), "dv": mk(w.hkv)}

    if L.fused and w.backward:
        hs = U.HostSteps(L)
        outs = [host_out(), host_out()]       # one set per device slot
        h2d, d2h = hs.host_bytes_per_step()

        def run(nsteps):
            hs.begin(stream)
            for i in range(nsteps):
                hs.step(pin, outs[i % 2], stream)
            hs.end(stream)
        how = "HostSteps: copies on the library's copy streams, overlapped with neighbouring steps"
    else:
        dseq = {k: [torch.empty_like(t, device=dev) for t in v] for k, v in pin.items()}
        o = L.new_seq_shards(w.hc)
        outs_dev = [o]
        if w.backward:
            dq, dk, dv = L.new_seq_shards(w.hc), L.new_seq_shards(w.hkv), L.new_seq_shards(w.hkv)
            outs_dev += [dq, dk, dv]
        host = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in grp] for grp in outs_dev]
        h2d = sum(t.numel() * t.element_size() for k, v in pin.items() if w.backward or k != "do" for t in v)
        d2h = sum(t.numel() * t.element_size() for grp in outs_dev for t in grp)

        def run(nsteps):
            for _ in range(nsteps):
                for k in pin:
                    if k == "do" and not w.backward:
                        continue
                    for src, dst in zip(pin[k], dseq[k]):
                        dst.copy_(src, non_blocking=True)
                L.forward(dseq["q"], dseq["k"], dseq["v"], o)
                if w.backward:
                    L.backward(dseq["do"], dq, dk, dv)
                for grp, hgrp in zip(outs_dev, host):
                    for src, dst in zip(grp, hgrp):
                        dst.copy_(src, non_blocking=True)
        how = "UlyssesLayer with the copies on the compute stream"

    run(args.warmup)
    torch.cuda.synchronize(dev)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    run(args.steps)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms = max_over_ranks(t0.elapsed_time(t1), dev, world)
    return {"value": job_tokens_per_s(w.sl * w.bs, args.steps, world, ms), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.steps, "how": how}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(w, sl_sample):
    """Time the oracle's whole layer (fwd, and bwd if the workload has one) at sl_sample.

    Same P, heads, head size and mask kind as the workload. Returns
    (seconds, tokens/s scaled to the full workload by visible-pair work).
    """
    import oracle
    from workloads import random_inputs
    offs = None
    if w.ndoc:
        # the same number of documents, scaled down
        full = doc_offsets_for(w)
        offs = sorted({round(o * sl_sample / w.sl) for o in full})
    x = random_inputs(sl_sample, w.bs, w.hc, w.hkv, w.hs, w.torch_dtype, w.seed, with_grad=w.backward)
    qs, ks, vs = (oracle.shard_sequence(x[n], w.P) for n in ("q", "k", "v"))
    t0 = time.perf_counter()
    oracle.ulysses_forward(qs, ks, vs, w.P, causal=w.causal, doc_offsets=offs)
    if w.backward:
        oracle.ulysses_backward(qs, ks, vs, oracle.shard_sequence(x["do"], w.P), w.P, causal=w.causal,
                                doc_offsets=offs)
    sec = time.perf_counter() - t0
    work_ratio = attn_flops(w) / attn_flops(w, sl_sample, offs)
    return sec, w.sl * w.bs / (sec * work_ratio)


def run_reference(args, w, rank, world):
    if rank != 0:
        return None
    sl_sample = args.ref_sl
    for _ in range(args.warmup):
        oracle_sample(w, sl_sample)
    secs, vals = [], []
    for _ in range(args.steps):
        s, v = oracle_sample(w, sl_sample)
        secs.append(s)
        vals.append(v)
    value = statistics.mean(vals)
    sample = (f"oracle (torch fp64 CPU) whole layer {'fwd+bwd' if w.backward else 'fwd'} at sl={sl_sample} "
              f"(same P/heads/hs/mask), tokens/s scaled to sl={w.sl} by visible-pair work")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"kind": "oracle", "cores": torch.get_num_threads(), **cpu_info(), "sample": sample,
                             "value": value, "unit": "tokens/s"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return line


def workload_config(w):
    return {"workload": w.name, "P": w.P, "global_batch": w.bs, "seq_len": w.sl, "hc": w.hc, "hkv": w.hkv,
            "hs": w.hs, "causal": w.causal, "ndoc": w.ndoc or 1, "backward": w.backward,
            "parallelism": f"ulysses sp{w.P} (virtual ranks on one GPU)",
            "l2": "inputs larger than L2 (Q alone %.0f MiB)" % (w.sl * w.bs * w.hc * w.hs * w.elem_bytes / 2**20)}


# ---------------------------------------------------------------------------
# Rates, fractions and the roofline of one timed run
# ---------------------------------------------------------------------------
FLOP_PER_CYCLE_SM = 8192   # M=256, N=128, K=16 UMMA on a CTA pair every 64 cycles (measured, sm_103a)
FP32_FLOP_PER_CYCLE_SM = 256  # 128 fp32 FMA lanes per SM, 2 flop each: the fp32 path's (CUDA-core) peak
SM_MAX_MHZ = 2070          # GB300's maximum SM clock, for runs too short for a clock sample
SUSTAINED_AFTER_S = 2.0    # a timed region at least this long is compared with the sustained peak


def sm_count():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def run_summary(w, r, peaks, src):
    """Per-kernel rates and fractions, the attention and exchange figures, and the dominant kernel's roofline.

    Tensor fractions: ``frac_burst`` against the burst cuBLAS bf16 rate,
    ``frac_sustained`` against the rate cuBLAS holds for seconds under the
    power cap, and ``frac_of_clock_peak`` against the UMMA issue rate at the
    SM clock sampled during the run (8192 flop/cycle/SM x SMs x median MHz).
    ``frac`` is the burst fraction for a timed region under two seconds, the
    sustained one otherwise.
    """
    steps = r["steps"]
    offs = doc_offsets_for(w)
    burst = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", burst)
    long_run = r["timed_s"] >= SUSTAINED_AFTER_S
    clk = (r["clocks"] or {}).get("sm_mhz")
    clock_peak = FLOP_PER_CYCLE_SM * sm_count() * clk * 1e6 / 1e12 if clk else None
    # The fp32 path runs on the CUDA cores: its peak is the fp32 FMA rate at
    # the sampled clock (the maximum clock when the run was too short to sample).
    alu_mhz = clk or SM_MAX_MHZ
    alu_peak = FP32_FLOP_PER_CYCLE_SM * sm_count() * alu_mhz * 1e6 / 1e12

    def tensor_fracs(tf):
        if w.dtype != "bf16":   # no bf16 tensor peak applies
            return {"tflops": tf, "frac_alu": tf / alu_peak}
        out = {"tflops": tf, "frac_burst": tf / burst, "frac_sustained": tf / sustained}
        if clock_peak:
            out["frac_of_clock_peak"] = tf / clock_peak
        return out

    fl_fwd = attn_flops(w, offs=offs)
    fl_bwd = 2.5 * fl_fwd if w.backward else 0.0
    ds_blocks = max(r["ds_bytes"] - 32768, 0)   # the stored blocks, zero block excluded
    work = kernel_work(w, offs, ds_blocks)
    per_kernel = {}
    for name, k in r["kernels"].items():
        cname, bound, units, unit = work[name]
        rate = units * steps / (k["total_ms"] * 1e-3)
        per_kernel[name] = dict(k, kernel=cname, bound="alu" if unit == "flop" and w.dtype != "bf16" else bound,
                                **(tensor_fracs(rate / 1e12) if unit == "flop" else
                                   {"gbs": rate / 1e9, "frac_hbm": rate / 1e9 / peaks["hbm_gbs"]}))
        if name == "bwd_dq" and not ds_blocks:   # S and dP are issued again here: 3 GEMMs run, 1 is its own
            per_kernel[name]["issued_tflops"] = 3 * rate / 1e12
    km = {n: k["ms_per_step"] for n, k in r["kernels"].items()}
    attn_fwd_ms = km["attn_fwd"]
    attn_bwd_ms = sum(km.get(n, 0.0) for n in ("bwd_prep", "bwd_dkdv", "bwd_dq"))
    fwd_tf = fl_fwd / (attn_fwd_ms * 1e-3) / 1e12
    bwd_tf = fl_bwd / (attn_bwd_ms * 1e-3) / 1e12 if w.backward else None
    x_bytes = exchange_bytes(w, w.hc) + 2 * exchange_bytes(w, w.hkv)
    s2h_gbs = x_bytes / (r["s2h_qkv_ms"] * 1e-3) / 1e9
    h2s_gbs = exchange_bytes(w, w.hc) / (r["h2s_o_ms"] * 1e-3) / 1e9
    # the dominant kernel: the largest share of the timed step's device time
    top = max((n for n in r["kernels"] if "region" not in r["kernels"][n]),
              key=lambda n: r["kernels"][n]["total_ms"])
    cname, bound, units, unit = work[top]
    k = r["kernels"][top]
    avg_ms = k["total_ms"] / k["launches"]
    per_launch = units * steps / k["launches"]
    achieved = per_launch / (avg_ms * 1e-3) / (1e12 if unit == "flop" else 1e9)
    alu = unit == "flop" and w.dtype != "bf16"
    if alu:
        bound, peak = "alu", alu_peak
        peak_source = (f"derived: {FP32_FLOP_PER_CYCLE_SM} fp32 flop/cycle/SM x {sm_count()} SMs x "
                       f"{alu_mhz:.0f} MHz ({'sampled' if clk else 'maximum'} SM clock)")
    elif unit == "flop":
        peak, peak_name = (sustained, "bf16_tflops_sustained") if long_run else (burst, "bf16_tflops")
    else:
        peak, peak_name = peaks["hbm_gbs"], "hbm_gbs"
    if not alu:
        peak_source = (f"{src} {peak_name} (timed region {r['timed_s']:.2f} s: "
                       f"{'sustained' if long_run else 'burst'} peak)")
    traffic, traffic_how = captured_traffic(cname, w.name)
    roof = {"bound": bound, "kernel": cname, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s" if unit == "flop" else "GB/s", "frac": achieved / peak, "traffic": traffic,
            "traffic_source": traffic_how,
            "peak_source": peak_source,
            "algorithmic_per_launch": per_launch, "algorithmic_unit": unit, "avg_launch_ms": avg_ms,
            "launches": k["launches"],
            "share_of_step": k["total_ms"] / (r["ms_per_step"] * steps),
            "timing": "CUDA events recorded by the library around each launch on its stream"}
    if unit == "flop" and not alu:
        roof.update({"frac_sustained": achieved / sustained, "frac_burst": achieved / burst})
        if clock_peak:
            roof["frac_of_clock_peak"] = achieved / clock_peak
            roof["clock_peak"] = {"tflops": clock_peak, "sm_mhz": clk, "sms": sm_count(),
                                  "flop_per_cycle_sm": FLOP_PER_CYCLE_SM}
    attention = {"fwd_ms": attn_fwd_ms, "fwd_tflop": fl_fwd / 1e12,
                 **{"fwd_" + a: b for a, b in tensor_fracs(fwd_tf).items()},
                 "kernel_times": "per-kernel CUDA events: forward kernel; backward prep + dK/dV + dQ",
                 "layer_fwd_ms": r["fwd_ms"],
                 "layer_times": "CUDA events around the layer's forward and backward calls (exchanges included)"}
    if w.backward:
        attention.update({"bwd_ms": attn_bwd_ms, "bwd_tflop": fl_bwd / 1e12,
                          **{"bwd_" + a: b for a, b in tensor_fracs(bwd_tf).items()},
                          # 4 GEMMs (2.0x the forward): the figure without recomputing S
                          "bwd_tflops_no_recompute": 0.8 * bwd_tf, "layer_bwd_ms": r["bwd_ms"]})
    exchange = {"s2h_qkv_ms": r["s2h_qkv_ms"], "s2h_qkv_gbs": s2h_gbs, "s2h_qkv_frac_hbm": s2h_gbs / peaks["hbm_gbs"],
                "h2s_o_ms": r["h2s_o_ms"], "h2s_o_gbs": h2s_gbs, "h2s_o_frac_hbm": h2s_gbs / peaks["hbm_gbs"],
                "bytes_rule": "read + write of the whole tensor per exchange",
                "timed": ("the explicit exchange kernels in a loop of their own; the fused step runs none "
                          "(the attention kernels read and write the sequence shards)" if r["path"] == "fused" else
                          "the explicit exchange kernels, in a loop of their own"),
                "hbm_peak_gbs": peaks["hbm_gbs"], "hbm_peak_source": src}
    backward_dq = None
    if w.backward:
        backward_dq = ({"how": "stored dS: the dK/dV kernel writes bf16 dS, dQ = s dS K reads it back",
                        "ds_bytes": r["ds_bytes"]} if ds_blocks else
                       {"how": "recomputed: the dQ kernel forms S, P, dP and dS again"})
    return {"kernels": per_kernel, "roofline": roof, "attention": attention, "exchange": exchange,
            "backward_dq": backward_dq}


# The other workloads of the layer, timed in the same process after the
# headline one: (workload, timed steps, inputs drawn on the device).
OTHER_CONFIGS = (("alst_128k", 4, True), ("packed_64k", 10, True), ("llama8b_8k", 20, True), ("tiny", 20, False))


def run_configs(args, main_w, rank, world):
    """Short timed runs of every other workload (N = 1), each summarised like the headline one."""
    peaks, src = load_peaks()
    out = {}
    for name, steps, on_device in OTHER_CONFIGS:
        if name == main_w.name:
            continue
        w = WORKLOADS[name]
        r = run_ours(args, w, rank, world, steps=steps, warmup=3, with_e2e=False, on_device=on_device)
        rs = run_summary(w, r, peaks, src)
        entry = {"config": workload_config(w), "steps": steps, "ms_per_step": r["ms_per_step"],
                 "tokens_per_s": r["value"], "path": r["path"], "clocks": r["clocks"],
                 "inputs": ("device-side N(0,1) draw of the workload's shapes, seeded with its seed"
                            if on_device else "the workload's seeded host recipe"),
                 "kernels": {n: {a: b for a, b in k.items() if a not in ("total_ms", "launches")}
                             for n, k in rs["kernels"].items()},
                 "attention": rs["attention"], "exchange": {a: b for a, b in rs["exchange"].items()
                                                            if a.endswith(("_ms", "_gbs", "_hbm"))},
                 "roofline": {a: rs["roofline"][a] for a in ("kernel", "bound", "achieved", "unit", "frac",
                                                              "frac_burst", "frac_sustained", "frac_of_clock_peak")
                              if a in rs["roofline"]},
                 "backward_dq": rs["backward_dq"]}
        if name == "tiny":
            entry["oracle"] = oracle_whole_layer_timing(w)
        if name == "alst_128k":
            entry["oracle_spot_check"] = oracle_row_sample_timing(w, 1024)
        out[name] = entry
    return out


def cpu_info():
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = None
    try:
        p = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in p.stdout.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                model = line.split(":", 1)[1].strip()
                if line.startswith("Model name"):
                    break
    except Exception:
        pass
    import platform
    return {"cores_available": cores, "cpu_model": model or platform.processor() or platform.machine()}


def with_threads(n, fn):
    old = torch.get_num_threads()
    torch.set_num_threads(n)
    try:
        return fn()
    finally:
        torch.set_num_threads(old)


def cpu_baseline(w, sl_sample):
    info = cpu_info()
    n = info["cores_available"]
    sec, val = with_threads(n, lambda: oracle_sample(w, sl_sample))
    return {"value": val, "unit": "tokens/s", "cores": n, "kind": "oracle", **info,
            "sample": (f"oracle (torch fp64 CPU, {n} threads) whole layer {'fwd+bwd' if w.backward else 'fwd'} "
                       f"at sl={sl_sample} (same P/heads/hs/mask) took {sec:.2f} s; tokens/s scaled to "
                       f"sl={w.sl} by visible-pair work")}


def oracle_whole_layer_timing(w):
    """The oracle on the whole (small) workload: all host cores, then one."""
    info = cpu_info()
    res = {**info}
    oracle_sample(w, w.sl)   # untimed first call (library set-up, page-ins)
    for label, n in (("all_cores", info["cores_available"]), ("one_core", 1)):
        sec, _ = with_threads(n, lambda: oracle_sample(w, w.sl))
        res[label] = {"threads": n, "seconds": sec, "tokens_per_s": w.sl * w.bs / sec}
    return res


def oracle_row_sample_timing(w, rows):
    """The oracle's spot check of the 128K workload: O, LSE and dQ of `rows` random query rows.

    Rows/s of the sampled check, and the extrapolation to every row of the
    layer (labelled as such: the full oracle at this size is ~490 TFLOP of fp64).
    """
    import oracle
    import numpy as np
    info = cpu_info()
    g = torch.Generator("cpu").manual_seed(w.seed)
    rng = np.random.default_rng(w.seed)
    heads = 32
    per_head = rows // heads
    s = 1.0 / math.sqrt(w.hs)
    # one head's tensors serve every head: the check's cost depends on the shapes only
    q, k, v, do = (torch.randn(w.sl, w.hs, generator=g, dtype=torch.float64) for _ in range(4))

    def run():
        t0 = time.perf_counter()
        for _ in range(heads):
            rr = torch.tensor(np.sort(rng.choice(w.sl, per_head, replace=False)))
            oracle.attention_head_dq_rows(q, k, v, do, s, w.causal, doc_offsets_for(w), rr)
        return time.perf_counter() - t0

    sec = with_threads(info["cores_available"], run)
    n = heads * per_head
    total_rows = w.sl * w.bs * w.hc
    return {**info, "threads": info["cores_available"], "rows": n, "seconds": sec, "rows_per_s": n / sec,
            "extrapolated_layer_fwd_s": total_rows / (n / sec),
            "note": "rows/s of the sampled O/LSE/dQ check; the layer figure is an extrapolation, not a run"}


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_32k", choices=sorted(WORKLOADS))
    ap.add_argument("--path", choices=["auto", "fused", "explicit"], default="auto",
                    help="fused: exchanges inside the attention kernels (where the shape allows); "
                         "explicit: exchange kernels between the attention calls")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ds-budget", type=int, default=None,
                    help="bytes the backward may keep dS in (default: the layer's; 0 recomputes dQ)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the short timed runs of the other workloads (the `configs` object)")
    ap.add_argument("--cpu-sl", type=int, default=4096, help="oracle sample length for cpu_baseline")
    ap.add_argument("--ref-sl", type=int, default=1024, help="oracle sample length per reference step")
    ap.add_argument("--sl", type=int, default=None,
                    help="run the workload's shape at another sequence length (profiling a smaller case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = WORKLOADS[args.workload]
    if args.sl is not None:
        import dataclasses
        if w.ndoc:
            ap.error("--sl applies to single-document workloads")
        if args.sl % w.P:
            ap.error("--sl must be divisible by P")
        w = dataclasses.replace(w, sl=args.sl, name=f"{w.name}@sl{args.sl}")

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")

    r = run_ours(args, w, rank, world)
    configs = None
    if not args.no_configs and world == 1:
        configs = run_configs(args, w, rank, world)
    if rank == 0:
        peaks, src = load_peaks()
        rs = run_summary(w, r, peaks, src)
        cpu = None
        if not args.no_cpu_baseline:
            cpu = cpu_baseline(w, args.cpu_sl)
        line = {"metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else "f32",
                "data": "synthetic (seeded N(0,1) Q/K/V/dO of the workload's shape)",
                "config": workload_config(w),
                "roofline": rs["roofline"],
                "cpu_baseline": cpu,
                "e2e": r["e2e"],
                "gpu_launches": r["launches"],
                "kernels": rs["kernels"],
                "clocks": r["clocks"],
                "path": r["path"],
                "backward_dq": rs["backward_dq"],
                "attention": rs["attention"],
                "exchange": rs["exchange"],
                "configs": configs,
                "context": "pages' figure (not a target): ALST trains a 500K-token sequence for Llama-8B on one H100"}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
