"""Benchmark: attention forward TFLOPS and paged-decode HBM GB/s on one GB300.

One step = one pass of the whole hot path: the fused prefill forward on the
GQA causal workload (B=4, Hq=32, Hkv=8, Sq=Sk=4096, d=128, bf16, BSHD) followed
by one paged-KV decode step (32 sequences, Hq=32, Hkv=8, lengths U[1024, 8192],
16-token pages).  `value` is the prefill TFLOPS (4*B*Hq*Sq*Sk*d / 2 flops per
launch, causal) over the K timed steps; the decode GB/s (algorithmic K+V bytes
per launch / time) is reported beside it.  Inputs are seeded synthetic data of
those shapes, resident in HBM when the timed region starts, and larger than
L2 (no flush needed).

Beside the headline the same line carries:
  sustained  the same step back to back for at least a second, with its own
             clock record, against the sustained tensor peak;
  workloads  every other prefill workload (tiny BHSD, MQA causal, ragged self
             and cross attention, the packed varlen batch, chunked prefill on
             a paged cache), each launched alone after an L2 flush, with its
             TFLOP/s, roofline fraction and the DRAM traffic of its own ncu
             capture;
  e2e        the headline prefill from pinned host memory through attn_fwd_host;
  decode_append, cpu_baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                    [--no-workloads] [--no-cpu-baseline]

Under torchrun (N > 1) every rank runs its own replica of the step (weak
scaling, no collective on the data path); timing is bracketed by a barrier and
the max over ranks is reported.  `--impl reference` times the fp64 CPU oracle
on bounded samples of the same workload instead (the slow reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from exact_attention_forward_06_gb300 import inputs  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "dram_traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PREFILL_KERNEL_SRC = os.path.join(ROOT, "exact_attention_forward_06_gb300", "csrc", "prefill_tc.cu")
DECODE_KERNEL_SRC = os.path.join(ROOT, "exact_attention_forward_06_gb300", "csrc", "decode.cu")


# ---------------------------------------------------------------------------- helpers

def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(path):
    """Hash of a kernel source's code: comments removed and whitespace collapsed,
    so that an edit to comments alone does not mark its ncu counters stale."""
    with open(path, "rb") as f:
        text = f.read().decode()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def traffic_for(workload, src_path):
    """DRAM bytes per launch of `workload` from its committed ncu summary, or
    None if absent or stale.

    Each entry of profiles/dram_traffic.json is keyed by workload and holds
    dram__bytes_read.sum + dram__bytes_write.sum of one captured launch of that
    workload, with a hash of the kernel source it was taken on; when the source
    has changed since, the figure no longer describes the kernel and None is
    reported until it is captured again.
    """
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)[workload]
    except (OSError, ValueError, KeyError):
        return None
    if t.get("source_sha256_16") != source_hash(src_path):
        return None
    return t["bytes_per_launch"]


def reduce_max_over_ranks(x: float) -> float:
    """Max of a host scalar over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- prefill cases

class DenseCase:
    """A dense batch (attn_fwd): B sequences of equal lengths in BSHD or BHSD."""

    def __init__(self, w):
        self.w = w
        self.name = w.name
        self.flops = w.flops
        self.host = inputs.make_prefill(w)
        self.lse_shape = (w.B, w.Hq, w.Sq)
        self.config = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "d": w.d, "layout": w.layout,
                       "causal": w.causal}
        self.flop_note = "4*B*Hq*Sq*Sk*d" + ("/2" if w.causal else "")
        self.bytes = byte_floor(w.B * w.Sq, w.Hq, w.B * w.Sk, w.Hkv, w.d)
        self.api = "exact_attention_forward_06_gb300.fwd (C ABI attn_fwd)"

    def workspace_bytes(self, A):
        w = self.w
        return A.fwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.causal)

    def call(self, A, dev_in, out, lse, stream):
        q, k, v = dev_in
        w = self.w
        A.fwd(q, k, v, causal=w.causal, scale=w.scale, layout=w.layout, out=out, lse=lse, stream=stream)

    def oracle_sample(self, seconds, seed):
        q_h, k_h, v_h = self.host
        return _oracle_sample(self.w, q_h, k_h, v_h, seconds, seed)


class VarlenCase:
    """A packed batch of variable-length sequences (attn_fwd_varlen)."""

    def __init__(self, w):
        self.w = w
        self.name = w.name
        self.flops = w.flops
        self.host = inputs.make_varlen(w)
        self.lq, self.lk = w.lengths()
        total_q = self.host[0].shape[0]
        self.lse_shape = (w.Hq, total_q)
        self.config = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "total_q": total_q, "total_k": self.host[1].shape[0],
                       "lengths": f"U[{w.len_lo},{w.len_hi}] seed {w.seed}", "max_seqlen": max(self.lq), "d": w.d,
                       "layout": "thd (packed)", "causal": w.causal}
        self.flop_note = "sum over sequences of 4*Hq*Lq*Lk*d" + ("/2" if w.causal else "")
        self.bytes = byte_floor(total_q, w.Hq, self.host[1].shape[0], w.Hkv, w.d)
        self.api = "exact_attention_forward_06_gb300.fwd_varlen (C ABI attn_fwd_varlen)"

    def workspace_bytes(self, A):
        return 0

    def call(self, A, dev_in, out, lse, stream):
        q, k, v, cu_q, cu_k = dev_in
        w = self.w
        A.fwd_varlen(q, k, v, cu_q, cu_k, max_seqlen_q=max(self.lq), max_seqlen_k=max(self.lk), causal=w.causal,
                     scale=w.scale, out=out, lse=lse, stream=stream)

    def oracle_sample(self, seconds, seed):
        return _oracle_sample_varlen(self, seconds, seed)


class PagedCase(VarlenCase):
    """Chunked prefill against a paged KV cache (attn_fwd_paged)."""

    def __init__(self, w):
        self.w = w
        self.name = w.name
        self.flops = w.flops
        self.host = inputs.make_paged_prefill(w)
        self.lq, self.lk = w.lengths()
        total_q = self.host[0].shape[0]
        self.lse_shape = (w.Hq, total_q)
        self.config = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "total_q": total_q,
                       "chunks": f"U[{w.chunk_lo},{w.chunk_hi}]", "contexts": f"U[{w.ctx_lo},{w.ctx_hi}]",
                       "seed": w.seed, "cache_tokens": sum(self.lk), "page_size": w.page_size, "d": w.d,
                       "layout": "thd chunks, paged cache", "causal": w.causal}
        self.flop_note = "4*Hq*d per visible pair; causal pairs Lq*(Lk-Lq) + Lq^2/2 per sequence"
        self.bytes = byte_floor(total_q, w.Hq, sum(self.lk), w.Hkv, w.d)
        self.api = "exact_attention_forward_06_gb300.fwd_paged (C ABI attn_fwd_paged)"

    def call(self, A, dev_in, out, lse, stream):
        q, kp, vp, table, lens, cu_q = dev_in
        A.fwd_paged(q, kp, vp, table, lens, cu_q, max_seqlen_q=max(self.lq), causal=self.w.causal,
                    scale=self.w.scale, out=out, lse=lse, stream=stream)

    def oracle_sample(self, seconds, seed):
        return _oracle_sample_paged(self, seconds, seed)


def byte_floor(total_q, Hq, total_k, Hkv, d):
    """The fewest bytes a launch can move: Q read and O written once, K and V
    read once, the fp32 log-sum-exp written once."""
    return 2 * total_q * Hq * d * 2 + 2 * total_k * Hkv * d * 2 + total_q * Hq * 4


def make_case(name):
    if name in inputs.PAGED_PREFILL_WORKLOADS:
        return PagedCase(inputs.PAGED_PREFILL_WORKLOADS[name])
    if name in inputs.VARLEN_WORKLOADS:
        return VarlenCase(inputs.VARLEN_WORKLOADS[name])
    return DenseCase(inputs.PREFILL_WORKLOADS[name])


# ---------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import exact_attention_forward_06_gb300 as A
    A.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    case = make_case(args.workload)
    wd = inputs.PAGED_DECODE

    # Inputs (seeded, synthetic), resident on the device.
    dev_in = [t.to(dev) for t in case.host]
    out = torch.empty_like(dev_in[0])
    lse = torch.empty(case.lse_shape, device=dev, dtype=torch.float32)
    dq_h, kp_h, vp_h, table_h, lens_h = inputs.make_decode(wd)
    dq, kp, vp, table, lens = (t.to(dev) for t in (dq_h, kp_h, vp_h, table_h, lens_h))
    dout = torch.empty_like(dq)
    dlse = torch.empty((wd.B, wd.Hq), device=dev, dtype=torch.float32)
    ws = torch.empty(A.decode_workspace_bytes(wd.B, wd.Hq, wd.d, wd.max_blocks), device=dev, dtype=torch.uint8)
    # Workspace for the prefill's tail split, when the shape gets one on this device.
    fws_bytes = case.workspace_bytes(A)
    fws = torch.empty(fws_bytes, device=dev, dtype=torch.uint8) if fws_bytes else None
    A.set_workspace(fws)
    stream = torch.cuda.current_stream(dev)

    def prefill():
        case.call(A, dev_in, out, lse, stream)

    def decode():
        A.decode_paged(dq, kp, vp, table, lens, scale=wd.scale, out=dout, lse=dlse, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        prefill()
        decode()
    torch.cuda.synchronize(dev)
    code, site = A.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} at site {site} after warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        start.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
            decode()
            ev[i][2].record(stream)
        stop.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    code, site = A.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} at site {site} after the timed steps")
    total_ms = start.elapsed_time(stop)
    prefill_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    decode_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    total_ms = reduce_max_over_ranks(total_ms)
    prefill_ms = reduce_max_over_ranks(prefill_ms)
    decode_ms = reduce_max_over_ranks(decode_ms)

    # The same step back to back for at least a second: the clocks and the
    # tensor peak that hold for a kernel timed inside a long run.
    sustained = run_sustained(prefill, decode, case.flops, total_ms / K, dev, stream, peaks, peak_src,
                              args.sustained_seconds)
    A.set_workspace(None)

    # End to end through the public API: pinned host inputs -> device -> result back to pinned host.
    e2e = run_e2e(A, case, dev, stream, args)
    # The fused append + decode step on the same decode workload (timed on its own, outside the step).
    dec_append = run_decode_append(A, wd, lens_h, dev, stream, args)
    del dev_in, out, lse
    # Every other prefill workload, each on its own.
    workloads = None if args.no_workloads else run_workloads(A, args, dev, stream, peaks, peak_src, skip=case.name)

    if rank != 0:
        return None
    flops = case.flops
    tflops = world * flops / (prefill_ms * 1e-3) / 1e12
    per_launch_tflops = flops / (prefill_ms * 1e-3) / 1e12
    kv_bytes = inputs.decode_kv_bytes(lens_h.tolist(), wd.Hkv, wd.d)
    dec_gbs_launch = kv_bytes / (decode_ms * 1e-3) / 1e9
    traffic = traffic_for(case.name, PREFILL_KERNEL_SRC)
    dec_traffic = traffic_for(wd.name, DECODE_KERNEL_SRC)
    clk = clocks.summary()
    line = {
        "metric": "attn fwd TFLOPS (bf16, d=128) and % of GB300 bf16 peak; paged decode HBM GB/s",
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded randn, bf16)",
        "config": {"workload": case.name, **case.config,
                   "decode_workload": wd.name, "decode_B": wd.B, "decode_Hq": wd.Hq, "decode_Hkv": wd.Hkv,
                   "decode_lengths": f"U[{wd.len_lo},{wd.len_hi}] seed {wd.seed}, sum {int(lens_h.sum())}",
                   "page_size": wd.page_size, "l2": "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}"},
        "prefill_ms_per_launch": round(prefill_ms, 4),
        "prefill_tail_split_workspace_bytes": fws_bytes,
        "roofline": {"bound": "tensor", "achieved": round(per_launch_tflops, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(per_launch_tflops / peaks["bf16_tflops"], 4),
                     "traffic": traffic, "peak_source": f"{peak_src} bf16_tflops (burst: {K} steps, "
                                                        f"{total_ms:.1f} ms timed)",
                     "kernel": "attn::g1::prefill_kernel",
                     "algorithmic": f"{flops:.4g} flop per launch ({case.flop_note})"},
        "decode": {"value": round(dec_gbs_launch * world, 1), "unit": "GB/s", "ms_per_launch": round(decode_ms, 4),
                   "roofline": {"bound": "hbm", "achieved": round(dec_gbs_launch, 1), "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": round(dec_gbs_launch / peaks["hbm_gbs"], 4),
                                "traffic": dec_traffic, "peak_source": f"{peak_src} hbm_gbs",
                                "kernel": "attn::dec::split_kernel + merge_kernel",
                                "algorithmic": f"{kv_bytes} B K+V per launch (4096 B per token)"}},
        "sustained": sustained,
        "workloads": workloads,
        "decode_append": dec_append,
        "e2e": e2e,
        "gpu_launches": (4 if fws_bytes else 3) * K,
        "clocks": clk,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(case, seconds=args.cpu_seconds)
    return line


def run_sustained(prefill, decode, flops, step_ms, dev, stream, peaks, peak_src, seconds):
    """The benchmark step repeated back to back for about `seconds`, timed as a
    whole and per prefill launch, with the clocks sampled meanwhile."""
    n = max(1, int(math.ceil(seconds * 1e3 / max(step_ms, 1e-3))))
    pre = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        s.record(stream)
        for a, b in pre:
            a.record(stream)
            prefill()
            b.record(stream)
            decode()
        e.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    total_ms = reduce_max_over_ranks(s.elapsed_time(e))
    prefill_ms = reduce_max_over_ranks(sum(a.elapsed_time(b) for a, b in pre) / n)
    tf = flops / (prefill_ms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    return {"steps": n, "seconds": round(total_ms / 1e3, 3), "ms_per_step": round(total_ms / n, 4),
            "value": round(_world() * tf, 2), "unit": "TFLOP/s", "prefill_ms_per_launch": round(prefill_ms, 4),
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tf / peak, 4),
                         "peak_source": f"{peak_src} bf16_tflops_sustained (seconds-long run)"},
            "clocks": clocks.summary()}


# Prefill workloads reported beside the headline, in this order.
OTHER_WORKLOADS = [inputs.TINY_BHSD.name, inputs.MQA_CAUSAL.name, inputs.RAGGED_SELF.name, inputs.RAGGED_CROSS.name,
                   inputs.VARLEN_CAUSAL.name, inputs.PAGED_PREFILL.name, inputs.GQA_SHORT_QUERY.name]
L2_BYTES = 129 << 20         # GB300's L2
L2_FLUSH_BYTES = 256 << 20   # about twice the L2


def workload_roofline(case, ms, peaks, peak_src, traffic):
    """The roofline a prefill workload sits under: the tensor peak when its
    flops per byte of the byte floor exceed the ridge point (burst tensor peak
    over copy bandwidth), else HBM, with the byte floor as the algorithmic
    bytes (a short query against long keys streams K and V)."""
    intensity = case.flops / case.bytes
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if intensity >= ridge:
        tf = case.flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(tf / peaks["bf16_tflops"], 4), "traffic": traffic,
                "peak_source": f"{peak_src} bf16_tflops (burst: one launch at a time)",
                "kernel": "attn::g1::prefill_kernel",
                "algorithmic": f"{case.flops:.4g} flop per launch ({case.flop_note})",
                "intensity_flop_per_byte": round(intensity, 1), "ridge_flop_per_byte": round(ridge, 1)}
    gbs = case.bytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
            "peak_source": f"{peak_src} hbm_gbs", "kernel": "attn::g1::prefill_kernel",
            "algorithmic": f"{case.bytes} B per launch (Q and O once, K and V once, fp32 lse)",
            "intensity_flop_per_byte": round(intensity, 1), "ridge_flop_per_byte": round(ridge, 1)}


def run_workloads(A, args, dev, stream, peaks, peak_src, skip=None):
    """Each prefill workload on its own: CUDA events around every launch, at
    least `args.steps` launches and about half a second of them.  A workload
    whose inputs and outputs together exceed L2 runs back to back like the
    headline; a smaller one gets an L2 flush (a 256 MB write, outside the
    timed events) before every launch.  Reports value, the roofline fraction
    (against the burst tensor peak, or HBM for a workload whose intensity is
    below the ridge point), and the DRAM traffic of the workload's own ncu
    capture."""
    flush = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    result = {}
    for name in OTHER_WORKLOADS:
        if name == skip:
            continue
        case = make_case(name)
        dev_in = [t.to(dev) for t in case.host]
        out = torch.empty_like(dev_in[0])
        lse = torch.empty(case.lse_shape, device=dev, dtype=torch.float32)
        fws_bytes = case.workspace_bytes(A)
        fws = torch.empty(fws_bytes, device=dev, dtype=torch.uint8) if fws_bytes else None
        A.set_workspace(fws)

        resident = sum(t.numel() * t.element_size() for t in dev_in) + out.numel() * out.element_size() + \
            lse.numel() * lse.element_size()
        needs_flush = resident <= L2_BYTES

        def one():
            if needs_flush:
                flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            case.call(A, dev_in, out, lse, stream)
            b.record(stream)
            return a, b

        for _ in range(args.warmup):
            one()
        torch.cuda.synchronize(dev)
        a, b = one()
        torch.cuda.synchronize(dev)
        est = max(a.elapsed_time(b), 1e-3)
        n = max(args.steps, min(400, int(math.ceil(500.0 / (est + (0.06 if needs_flush else 0.0))))))
        barrier()
        with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
            evs = [one() for _ in range(n)]
            torch.cuda.synchronize(dev)
        barrier()
        code, site = A.device_status()
        A.set_workspace(None)
        if code != 0:
            raise RuntimeError(f"device status {code} at site {site} in workload {name}")
        ms = reduce_max_over_ranks(sum(x.elapsed_time(y) for x, y in evs) / n)
        tf = case.flops / (ms * 1e-3) / 1e12
        result[name] = {
            "value": round(_world() * tf, 2), "unit": "TFLOP/s", "ms_per_launch": round(ms, 4), "launches": n,
            "config": case.config, "api": case.api, "tail_split_workspace_bytes": fws_bytes,
            "l2": ("flushed (256 MB write) before every timed launch" if needs_flush else
                   f"inputs and outputs ({resident / 1e6:.0f} MB) larger than L2 (no flush)"),
            "roofline": workload_roofline(case, ms, peaks, peak_src, traffic_for(name, PREFILL_KERNEL_SRC)),
            "clocks": clocks.summary(),
        }
        del dev_in, out, lse, fws
        torch.cuda.empty_cache()
    return result


def run_decode_append(A, wd, lens_h, dev, stream, args):
    """The fused append + decode call on the decode workload's lengths: a pool
    with pages for L + 1 tokens, the new token appended at position L."""
    q_h, kp_h, vp_h, table_h, _ = inputs.make_decode(wd, seqlens=(lens_h + 1).tolist())
    g = torch.Generator().manual_seed(wd.seed + 7)
    k_new = torch.randn(wd.B, wd.Hkv, wd.d, generator=g).to(torch.bfloat16).to(dev)
    v_new = torch.randn(wd.B, wd.Hkv, wd.d, generator=g).to(torch.bfloat16).to(dev)
    q, kp, vp, table, lens = (t.to(dev) for t in (q_h, kp_h, vp_h, table_h, lens_h))
    out = torch.empty_like(q)
    lse = torch.empty((wd.B, wd.Hq), device=dev, dtype=torch.float32)
    ws = torch.empty(A.decode_workspace_bytes(wd.B, wd.Hq, wd.d, wd.max_blocks), device=dev, dtype=torch.uint8)

    def call():
        A.decode_paged_append(q, k_new, v_new, kp, vp, table, lens, scale=wd.scale, out=out, lse=lse, workspace=ws,
                              stream=stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    n = max(3, args.steps)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(n):
        call()
    e.record(stream)
    torch.cuda.synchronize(dev)
    code, site = A.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} at site {site} in the fused append")
    ms = reduce_max_over_ranks(s.elapsed_time(e) / n)
    kv_bytes = inputs.decode_kv_bytes((lens_h + 1).tolist(), wd.Hkv, wd.d)
    return {"value": round(_world() * kv_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_launch": round(ms, 4),
            "kernel": "attn::dec::split_kernel (fused append) + merge_kernel",
            "algorithmic": f"{kv_bytes} B K+V per launch (L+1 keys per sequence)"}


def run_e2e_host(A, case, dev, stream, args):
    """End to end through attn_fwd_host: pinned host inputs in, pinned host
    outputs back, the library's own chunked copy/compute overlap inside."""
    w = case.w
    q, k, v = (t.pin_memory() for t in case.host)
    out_h = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(case.lse_shape, dtype=torch.float32).pin_memory()
    ws = torch.empty(A.fwd_host_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d), device=dev, dtype=torch.uint8)

    def step():
        A.fwd_host(q, k, v, causal=w.causal, scale=w.scale, layout=w.layout, out=out_h, lse=lse_h, workspace=ws,
                   stream=stream)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    n = max(1, args.steps // 2)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    s.record(stream)
    for _ in range(n):
        step()
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = reduce_max_over_ranks(s.elapsed_time(e) / n)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    return {"value": round(_world() * case.flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "api": "exact_attention_forward_06_gb300.fwd_host (C ABI attn_fwd_host: pinned host buffers in and out)"}


def run_e2e(A, case, dev, stream, args):
    if isinstance(case, DenseCase):
        return run_e2e_host(A, case, dev, stream, args)
    pinned = [t.pin_memory() for t in case.host]
    dev_in = [torch.empty_like(t, device=dev) for t in pinned]
    out_h = torch.empty_like(pinned[0]).pin_memory()
    lse_h = torch.empty(case.lse_shape, dtype=torch.float32).pin_memory()
    out = torch.empty_like(dev_in[0])
    lse = torch.empty(case.lse_shape, device=dev, dtype=torch.float32)

    def step():
        for d_t, h_t in zip(dev_in, pinned):
            d_t.copy_(h_t, non_blocking=True)
        case.call(A, dev_in, out, lse, stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    n = max(1, args.steps // 2)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    s.record(stream)
    for _ in range(n):
        step()
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = reduce_max_over_ranks(s.elapsed_time(e) / n)
    world = _world()
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    return {"value": round(world * case.flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "api": f"{case.api} with pinned host copies"}


# ---------------------------------------------------------------------------- CPU oracle arms

def _row_flops(w, rows):
    """Matmul flops of the sampled rows: 4*d per visible key."""
    tot = 0
    for _, _, i in rows:
        n = min(w.Sk, i + 1 + w.Sk - w.Sq) if w.causal else w.Sk
        tot += 4 * w.d * max(0, n)
    return tot


def _oracle_sample(w, q_h, k_h, v_h, seconds, seed):
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)

    def rows_of(n):
        return np.stack([rng.integers(0, w.B, n), rng.integers(0, w.Hq, n), rng.integers(0, w.Sq, n)], 1)

    kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk, d=w.d, layout=w.layout, causal=w.causal,
              scale=w.scale)
    # calibrate on a small batch, then size the sample to about `seconds`
    probe = rows_of(max(8, oracle.num_threads()))
    t0 = time.perf_counter()
    oracle.attention_rows(q_h, k_h, v_h, probe, **kw)
    dt = time.perf_counter() - t0
    n = max(len(probe), int(len(probe) * seconds / max(dt, 1e-3)))
    for _ in range(2):
        # the probe over-estimates the time per row (fixed costs); re-size once
        # if the sample ran well short of `seconds`
        rows = rows_of(n)
        t0 = time.perf_counter()
        oracle.attention_rows(q_h, k_h, v_h, rows, **kw)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * seconds:
            break
        n = int(n * seconds / max(dt, 1e-3))
    return _row_flops(w, rows), dt, len(rows)


def _oracle_sample_varlen(case, seconds, seed):
    """Uniformly drawn (sequence, head, row) triples of a packed batch, each row
    through the oracle over its own sequence."""
    import numpy as np
    import oracle
    w = case.w
    q_h, k_h, v_h, cu_q, cu_k = case.host
    rng = np.random.default_rng(seed)
    weights = np.array(case.lq, dtype=np.float64) / sum(case.lq)

    def run(n):
        seqs = rng.choice(w.B, size=n, p=weights)
        flops = 0
        for b in np.unique(seqs):
            m = int((seqs == b).sum())
            Lq, Lk = case.lq[b], case.lk[b]
            q0, k0 = int(cu_q[b]), int(cu_k[b])
            rows = np.stack([np.zeros(m, np.int64), rng.integers(0, w.Hq, m), rng.integers(0, Lq, m)], 1)
            oracle.attention_rows(q_h[q0:q0 + Lq][None], k_h[k0:k0 + Lk][None], v_h[k0:k0 + Lk][None], rows, B=1,
                                  Hq=w.Hq, Hkv=w.Hkv, Sq=Lq, Sk=Lk, d=w.d, causal=w.causal, scale=w.scale)
            for i in rows[:, 2]:
                nk = min(Lk, int(i) + 1 + Lk - Lq) if w.causal else Lk
                flops += 4 * w.d * max(0, nk)
        return flops

    t0 = time.perf_counter()
    probe_n = max(8, oracle.num_threads())
    run(probe_n)
    dt = time.perf_counter() - t0
    n = max(probe_n, int(probe_n * seconds / max(dt, 1e-3)))
    t0 = time.perf_counter()
    flops = run(n)
    return flops, time.perf_counter() - t0, n


def _oracle_sample_paged(case, seconds, seed):
    """Uniformly drawn (sequence, head, chunk row) triples, each through the
    oracle over its sequence's keys gathered from the pages."""
    import numpy as np
    import oracle
    w = case.w
    q_h, kp, vp, table, lens, cu_q = case.host
    rng = np.random.default_rng(seed)
    weights = np.array(case.lq, dtype=np.float64) / sum(case.lq)
    gathered = {}

    def run(n):
        seqs = rng.choice(w.B, size=n, p=weights)
        flops = 0
        for b in np.unique(seqs):
            m = int((seqs == b).sum())
            Lq, Lk = case.lq[b], case.lk[b]
            q0 = int(cu_q[b])
            if b not in gathered:
                gathered[b] = (oracle.gather_pages(kp, table[b], Lk), oracle.gather_pages(vp, table[b], Lk))
            k_b, v_b = gathered[b]
            rows = np.stack([np.zeros(m, np.int64), rng.integers(0, w.Hq, m), rng.integers(0, Lq, m)], 1)
            oracle.attention_rows(q_h[q0:q0 + Lq][None], k_b[None], v_b[None], rows, B=1, Hq=w.Hq, Hkv=w.Hkv,
                                  Sq=Lq, Sk=Lk, d=w.d, causal=w.causal, scale=w.scale)
            for i in rows[:, 2]:
                nk = min(Lk, int(i) + 1 + Lk - Lq) if w.causal else Lk
                flops += 4 * w.d * max(0, nk)
        return flops

    probe_n = max(8, oracle.num_threads())
    run(probe_n)                       # gathers every drawn sequence once
    t0 = time.perf_counter()
    run(probe_n)
    dt = time.perf_counter() - t0
    n = max(probe_n, int(probe_n * seconds / max(dt, 1e-3)))
    t0 = time.perf_counter()
    flops = run(n)
    return flops, time.perf_counter() - t0, n


def cpu_baseline(case, seconds):
    import oracle
    flops, dt, n = case.oracle_sample(seconds, seed=1)
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} uniformly drawn query rows of {case.name} (fp64 C oracle, OpenMP), {dt:.1f} s"}


def run_reference(args, rank, world):
    import oracle
    if rank != 0:
        return None
    case = make_case(args.workload)
    per_step = max(1.0, min(6.0, 60.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        case.oracle_sample(per_step / 2, seed=100 + i)
    tot_flops, tot_t, tot_rows = 0, 0.0, 0
    for i in range(args.steps):
        f, dt, n = case.oracle_sample(per_step, seed=i)
        tot_flops += f
        tot_t += dt
        tot_rows += n
    value = tot_flops / tot_t / 1e12
    return {
        "impl": "reference",
        "metric": "attn fwd TFLOPS (bf16, d=128) and % of GB300 bf16 peak; paged decode HBM GB/s",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded randn, bf16 inputs)",
        "config": {"workload": case.name, **case.config},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{tot_rows} uniformly drawn query rows of {case.name} over {args.steps} steps"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ---------------------------------------------------------------------------- main

def _world():
    return int(os.environ.get("WORLD_SIZE", "1"))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=inputs.GQA_CAUSAL.name,
                    choices=sorted(inputs.PREFILL_WORKLOADS) + sorted(inputs.VARLEN_WORKLOADS) +
                    sorted(inputs.PAGED_PREFILL_WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--sustained-seconds", type=float, default=1.5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the record of the other prefill workloads")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = _world()
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            line = run_reference(args, rank, world)
        else:
            line = run_ours(args, rank, world, local_rank)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    main()
