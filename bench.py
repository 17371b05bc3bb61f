#!/usr/bin/env python
"""Benchmark of the hybrid (ordinary + frozen heads) causal attention layer.

One step = forward + backward of the layer over one synthetic batch, through
the C ABI of libsaf.so. Default workload: GPT-2-124M-shaped layer with 25% of
heads frozen (B=8, H=12 with heads 3, 7, 11 frozen, T=4096, d=64, bf16).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs its own batch of
the same workload (weak scaling, no collective on the data path); the time
is the max over ranks and the value the work of all ranks over that time.
`--gpus N` without torchrun starts the N ranks itself (torchrun on 127.0.0.1).

Besides the headline workload, the line carries `other_workloads`: the other
bench workloads of the same layer (50% frozen, the 1B-shaped layer at 8K, the
16K prefill), each timed in the same run with its all-ordinary comparison, and
`trainable_patterns`: the time of the pattern gradient (saf_pattern_grad_tc) that
the trainable-pattern variant adds to a step.

    python bench.py --workload W --record-traffic ncu.csv

stores the DRAM bytes per launch of fwd_tc_kernel / bwd_tc_kernel from an ncu
capture (`--metrics dram__bytes_read.sum,dram__bytes_write.sum --csv`) in
profiles/traffic.json, keyed by the hash of the kernel's sources at the time
of recording; the bench line reports `roofline.traffic` only for a key that
matches the sources it runs.
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

from softmax_attention_hybrid_gb300 import flops as F  # noqa: E402
from softmax_attention_hybrid_gb300.inputs import WORKLOADS, make_inputs, Workload  # noqa: E402

METRIC = "hybrid attention fwd+bwd TFLOP/s and tokens/s at 1 GB300; % of bf16 tensor peak"
DEFAULT_WORKLOAD = "gpt2_124m_25"
# timed after the headline workload in the same run, each with its all-ordinary run
OTHER_WORKLOADS = ("gpt2_124m_50", "1b_25", "prefill_16k", "prefill_b64_4k", "prefill_b64_4k_50", "gqa_32q8kv_4k",
                   "gqa_32q8kv_d128", "1b_d96")
L2_FLUSH_BYTES = 256 << 20  # larger than the 129 MB L2


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


# the sources that decide a kernel's DRAM traffic: its own file, the shared
# device helpers, and the launch sequence with the kernels around it
KERNEL_SOURCES = {"bwd": ("bwd_tc.cu", "tc_common.cuh", "saf_internal.h", "prep.cu", "saf_api.cu"),
                  "fwd": ("fwd_tc.cu", "tc_common.cuh", "saf_internal.h", "prep.cu", "saf_api.cu")}


def _src_hash(kernel=None):
    """Hash of the library sources (all of them, or those of one kernel)."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "softmax_attention_hybrid_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) if kernel else None
    for name in sorted(names or os.listdir(csrc)):
        if name.endswith((".cu", ".h", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    if not names:
        with open(os.path.join(ROOT, "include", "saf.h"), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
                uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            except Exception:
                uuid = None
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if uuid:
                cmd += ["-i", uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for nm, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        loaded = [x for x in sm if x > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# ---------------------------------------------------------------------------

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w: Workload, x, batches=2):
    """A bounded sample of the workload for the fp64 CPU oracle: every head of
    the first `batches` batch entries, forward and backward (forward only for
    forward-only workloads), with the same head mix as the workload.
    Returns (fn, flops, description)."""
    import oracle
    nb = min(batches, w.B)
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    G = w.H // (w.Hkv or w.H)   # query heads per key/value head
    sl = {(b, h): [x[n][b, h if n in ("q", "do") else h // G].double().numpy() for n in ("q", "k", "v", "do")]
          for b in range(nb) for h in range(w.H)}
    flops = F.layer_flops(nb, w.H, sum(1 for h in range(w.H) if x["frozen"][h]), w.T, w.d,
                          backward=not w.fwd_only)

    def run():
        for (b, h), (q, k, v, do) in sl.items():
            fzh = bool(x["frozen"][h])
            oracle.head_fwd(q, k, v, a[h], r[h], fzh)
            if not w.fwd_only:
                oracle.head_bwd(q, k, v, do, a[h], r[h], fzh)

    desc = (f"batch entries 0..{nb - 1} (all {w.H} heads) of {w.name}, T={w.T}, "
            f"{'fwd' if w.fwd_only else 'fwd+bwd'}, fp64 NumPy/OpenBLAS, one slice at a time")
    return run, flops, desc


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, w):
    rank, world, local = dist_info()
    if rank != 0:
        return 0
    x = make_inputs(w, seed=0)
    run, flops, desc = oracle_sample(w, x, batches=1)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "F": w.F, "T": w.T, "d": w.d,
                   "sample": desc},
        # tokens/s of the full layer at the sample's FLOP rate
        "tokens_per_s": w.B * w.T * value * 1e12 / F.layer_flops(w.B, w.H, w.F, w.T, w.d, not w.fwd_only),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

KERNEL_FLOP_UNITS = {
    # (ordinary contractions, frozen contractions) per (batch, head) per launch
    "fwd": (2, 1),
    "bwd_kv": (4, 1),     # S recompute, dV, dP, dK | dV
    "bwd_q": (1, 0),      # dQ (its S and dP recomputes are not counted)
    "bwd": (5, 1),
    "dq_finish": (0, 0),
    "bwd_delta": (0, 0),
    "lognorm": (0, 0),
    "pattern_prep": (0, 0),
}


# what bounds each kernel: the bf16 kernels are tensor-core contractions,
# the fp32 CUDA-core kernels are FMA-bound ("alu")
def kernel_bound(name, dtype):
    # bf16 runs every main kernel on the tensor cores (bwd_kv / bwd_q: the d = 96, 128 path)
    return "tensor" if dtype == "bf16" and name in ("fwd", "bwd", "bwd_kv", "bwd_q") else "alu"


def e2e_chunk_sizes(B, spec=""):
    """Batch entries per chunk of the end-to-end step: four equal chunks when the
    batch allows (fewer, smaller chunks leave the kernels short of work), else halves."""
    if spec:
        sizes = [int(x) for x in spec.split(",")]
    elif B % 4 == 0 and B >= 8:
        sizes = [B // 4] * 4
    elif B % 2 == 0:
        sizes = [B // 2] * 2
    else:
        sizes = [B]
    if sum(sizes) != B or min(sizes) < 1:
        raise ValueError(f"e2e chunks {sizes} do not partition the batch {B}")
    return sizes


class Layer:
    """Device buffers of one workload and one step of the layer through the C ABI."""

    def __init__(self, saf, w: Workload, seed, dev):
        self.saf, self.w = saf, w
        self.x = make_inputs(w, seed=seed)
        self.frozen = self.x["frozen"]
        self.g = {n: self.x[n].to(dev) for n in ("q", "k", "v", "do", "a", "r")}
        B, H, T, d = w.B, w.H, w.T, w.d
        self.gqa = w.Hkv is not None and w.Hkv != H
        self.o = torch.empty_like(self.g["q"])
        self.lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.g["q"])
        self.dk, self.dv = torch.empty_like(self.g["v"]), torch.empty_like(self.g["v"])
        self.ws = saf.alloc_workspace(B, H, T, d, self.g["v"].dtype, not w.fwd_only, dev)
        self.kernels = {"fwd": saf.SAF_KERNEL_FWD, "lognorm": saf.SAF_KERNEL_LOGNORM,
                        "pattern_prep": saf.SAF_KERNEL_PATTERN_PREP}
        if not w.fwd_only:
            self.kernels.update({"bwd_kv": saf.SAF_KERNEL_BWD_KV, "bwd_q": saf.SAF_KERNEL_BWD_Q,
                                 "bwd": saf.SAF_KERNEL_BWD, "dq_finish": saf.SAF_KERNEL_DQ_FINISH,
                                 "bwd_delta": saf.SAF_KERNEL_BWD_DELTA})

    def prepare(self, mask):
        """Frozen-pattern state for fixed (a, r): the normalisers computed once."""
        self.state = self.saf.saf_frozen_prepare(self.g["a"], self.g["r"], mask, self.w.T, self.g["v"].dtype)

    def step_prepared(self, mask):
        saf, g = self.saf, self.g
        saf.saf_attn_fwd_prepared(g["q"], g["k"], g["v"], g["a"], g["r"], mask, self.state, o=self.o, lse=self.lse,
                                  workspace=self.ws)
        if not self.w.fwd_only:
            saf.saf_attn_bwd_prepared(g["q"], g["k"], g["v"], self.o, g["do"], self.lse, g["a"], g["r"], mask,
                                      self.state, dq=self.dq, dk=self.dk, dv=self.dv, workspace=self.ws)

    def step(self, mask):
        saf, g = self.saf, self.g
        fwd = saf.saf_attn_fwd_gqa if self.gqa else saf.saf_attn_fwd
        bwd = saf.saf_attn_bwd_gqa if self.gqa else saf.saf_attn_bwd
        fwd(g["q"], g["k"], g["v"], g["a"], g["r"], mask, o=self.o, lse=self.lse, workspace=self.ws)
        if not self.w.fwd_only:
            bwd(g["q"], g["k"], g["v"], self.o, g["do"], self.lse, g["a"], g["r"], mask, dq=self.dq, dk=self.dk,
                dv=self.dv, workspace=self.ws)


def timed(saf, lay, mask, K, trace, flush, stream, world, prepared=False):
    """K steps, each after an L2 flush, bracketed by CUDA events on the launching
    stream. trace: the kernel brackets that get their own events. Events between
    two launches cost a little time and stop the next launch from starting early,
    so the headline run brackets the dominant kernel alone and a separate run
    brackets every kernel for the per-kernel breakdown.
    Returns (per-step ms, per-kernel mean ms, launches)."""
    def new_event():
        # torch creates the CUDA event on first record; record once so that
        # the handle handed to the library is a real event
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)
        return ev

    evs = [(new_event(), new_event()) for _ in range(K)]
    kev = {nm: [(new_event(), new_event()) for _ in range(K)] for nm in trace}
    barrier(world)
    torch.cuda.synchronize()
    n0 = saf.saf_launch_count()
    for i in range(K):
        flush.fill_(float(i))
        for nm in trace:
            saf.saf_set_trace_events(lay.kernels[nm], kev[nm][i][0], kev[nm][i][1])
        evs[i][0].record(stream)
        if prepared:
            lay.step_prepared(mask)
        else:
            lay.step(mask)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    saf.saf_set_trace_events(saf.SAF_KERNEL_NONE)
    launches = saf.saf_launch_count() - n0
    ms = [s.elapsed_time(e) for s, e in evs]
    kms = {}
    for nm in trace:
        # a kernel this path never launches keeps the events' creation
        # records, which precede the step's start event
        if evs[0][0].elapsed_time(kev[nm][0][0]) < 0:
            continue
        vals = [s.elapsed_time(e) for s, e in kev[nm]]
        kms[nm] = sum(vals) / len(vals)
    return ms, kms, launches


def spread(ms):
    return {"min": min(ms), "median": statistics.median(ms), "max": max(ms),
            "stdev": statistics.pstdev(ms) if len(ms) > 1 else 0.0}


def kernel_roofline(name, kms, w, peaks, peak_src):
    """Achieved rate of kernel `name` (counted FLOP per launch / its mean launch time)."""
    units_o, units_f = KERNEL_FLOP_UNITS[name]
    c = 2 * F.pairs(w.T) * w.d
    kflops = w.B * ((w.H - w.F) * units_o + w.F * units_f) * c
    achieved = kflops / (kms[name] * 1e-3) / 1e12
    if kernel_bound(name, w.dtype) == "tensor":
        peak = peaks["bf16_tflops"]
        bound, note = "tensor", f"bf16 dense, burst, {peak_src}"
    else:
        # fp32 FMA pipes: 152 SMs x 128 FMA/clk x 2 FLOP at the max SM clock
        peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        bound, note = "alu", "fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock (derived)"
    return {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": note, "flops_per_launch": kflops, "ms_per_launch": kms[name]}


def time_prepared(saf, lay, args, dom, flush, stream, world, dev, flops, ao_ms):
    """The same step with the frozen heads' normalisers prepared once, outside the
    timed region (the paper keeps them as persistent state per frozen head)."""
    lay.prepare(lay.frozen)
    for _ in range(max(1, args.warmup // 2)):
        lay.step_prepared(lay.frozen)
    ms, _, _ = timed(saf, lay, lay.frozen, args.steps, [dom], flush, stream, world, prepared=True)
    pm = max_over_ranks(sum(ms) / len(ms), world, dev)
    out = {"ms_per_step": pm, "value": flops / (pm * 1e-3) / 1e12, "unit": "TFLOP/s",
           "note": "normalisers of the frozen heads prepared once before the timed region "
                   "(saf_frozen_prepare); the headline recomputes them in every step"}
    if ao_ms:
        out["speedup_vs_all_ordinary"] = ao_ms / pm
    return out


def backward_ms(kms):
    """Time of the backward kernels of a step: the fused kernel (d = 64), or the
    key-block and query-block passes (d = 96, 128)."""
    if "bwd" in kms:
        return kms["bwd"]
    return (kms.get("bwd_kv", 0.0) + kms.get("bwd_q", 0.0)) or None


def time_pattern_grad(saf, lay, args, flush, stream, world, dev, step_ms, bwd_ms):
    """The trainable-pattern variant's extra work (App. C.3.2): da, dr of the frozen
    heads from the step's V, dO, o and lse through saf_pattern_grad_tc, each call
    after an L2 flush and bracketed by CUDA events on the launching stream."""
    w, g = lay.w, lay.g
    H, T = w.H, w.T
    nf = sum(lay.frozen)
    ws = torch.empty(max(saf.saf_pattern_grad_tc_workspace_bytes(w.B, H, T, nf), 256), dtype=torch.uint8,
                     device=dev)
    da = torch.empty((H, T), dtype=torch.float32, device=dev)
    dr = torch.empty((H, T), dtype=torch.float32, device=dev)

    def call():
        saf.saf_pattern_grad_tc(g["v"], g["do"], lay.o, lay.lse, g["a"], g["r"], lay.frozen, da=da, dr=dr,
                                workspace=ws)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    if saf.saf_device_status(ws) != saf.SAF_OK:
        raise RuntimeError("device status after the pattern-gradient warm-up is not ok")
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    pm = max_over_ranks(sum(s.elapsed_time(e) for s, e in evs) / K, world, dev)
    out = {"ms": pm, "fraction_of_step": pm / step_ms,
           "note": "saf_pattern_grad_tc (tcgen05, fixed-order sums): gradients of a and r of the frozen heads, "
                   "timed alone after the step that produced o and lse"}
    if bwd_ms:
        out["fraction_of_bwd"] = pm / bwd_ms
    return out


def measure_workload(saf, w, args, dev, world, rank, stream, flush, peaks, peak_src):
    """Hybrid and all-ordinary step times of one more workload (no end-to-end leg)."""
    lay = Layer(saf, w, rank, dev)
    for _ in range(args.warmup):
        lay.step(lay.frozen)
    torch.cuda.synchronize()
    if saf.saf_device_status(lay.ws) != saf.SAF_OK:
        raise RuntimeError(f"device status after warm-up ({w.name}) is not ok")
    _, kms, _ = timed(saf, lay, lay.frozen, args.steps, list(lay.kernels), flush, stream, world)
    dom = max(kms, key=kms.get)
    ms, kms_dom, _ = timed(saf, lay, lay.frozen, args.steps, [dom], flush, stream, world)
    step_ms = max_over_ranks(sum(ms) / len(ms), world, dev)
    flops = F.layer_flops(w.B, w.H, w.F, w.T, w.d, backward=not w.fwd_only) * world
    out = {"ms_per_step": step_ms, "ms_spread": spread(ms), "value": flops / (step_ms * 1e-3) / 1e12,
           "unit": "TFLOP/s", "frac_of_bf16_peak": flops / world / (step_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
           "tokens_per_s": w.B * w.T * world / (step_ms * 1e-3),
           "config": {"B": w.B, "H": w.H, "Hkv": w.Hkv or w.H, "F": w.F, "T": w.T, "d": w.d, "dtype": w.dtype,
                      "fwd_only": w.fwd_only},
           "roofline": kernel_roofline(dom, kms_dom, w, peaks, peak_src), "kernel_ms": kms}
    if w.F > 0:
        zero = [0] * w.H
        for _ in range(max(1, args.warmup // 2)):
            lay.step(zero)
        ms0, _, _ = timed(saf, lay, zero, args.steps, [dom], flush, stream, world)
        ao = max_over_ranks(sum(ms0) / len(ms0), world, dev)
        out["all_ordinary"] = {"ms_per_step": ao, "speedup": ao / step_ms,
                               "ideal_speedup": F.layer_flops(w.B, w.H, 0, w.T, w.d, not w.fwd_only) /
                               F.layer_flops(w.B, w.H, w.F, w.T, w.d, not w.fwd_only)}
        out["prepared_normalisers"] = time_prepared(saf, lay, args, dom, flush, stream, world, dev, flops, ao)
        if not w.fwd_only and not lay.gqa:
            lay.step(lay.frozen)
            out["trainable_patterns"] = time_pattern_grad(saf, lay, args, flush, stream, world, dev, step_ms,
                                                          backward_ms(kms))
    del lay
    torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    from softmax_attention_hybrid_gb300 import saf

    lay = Layer(saf, w, rank, dev)
    x, frozen, g = lay.x, lay.frozen, lay.g
    B, H, T, d = w.B, w.H, w.T, w.d
    o, lse, dq, dk, dv, ws = lay.o, lay.lse, lay.dq, lay.dk, lay.dv, lay.ws
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = _peaks()

    for _ in range(args.warmup):
        lay.step(frozen)
    torch.cuda.synchronize()
    status = saf.saf_device_status(ws)
    if status != saf.SAF_OK:
        raise RuntimeError(f"device status after warm-up: {saf.saf_error_string(status)}")

    # per-kernel breakdown (every bracket traced), which also names the dominant kernel
    _, kms, _ = timed(saf, lay, frozen, args.steps, list(lay.kernels), flush, stream, world)
    dom = max(kms, key=kms.get)

    # the clock sampler runs through a soak of the same step (about 1 s, so that it
    # collects samples under load) and then through the timed region
    clocks = ClockSampler(local)
    clocks.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(20):
            lay.step(frozen)
        torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ms, kms_dom, launches = timed(saf, lay, frozen, args.steps, [dom], flush, stream, world)
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    clk["window"] = f"{args.soak_s:.1f} s soak of the same step, then the timed region"

    step_ms = max_over_ranks(sum(ms) / len(ms), world, dev)
    total_flops = F.layer_flops(B, H, w.F, T, d, backward=not w.fwd_only) * world
    value = total_flops / (step_ms * 1e-3) / 1e12
    tokens = B * T * world / (step_ms * 1e-3)

    # all-ordinary run of the same kernels on the same inputs
    allord = None
    if args.all_ordinary and w.F > 0:
        for _ in range(max(1, args.warmup // 2)):
            lay.step([0] * H)
        # traced like the hybrid run, so that both carry the same event overhead
        ms0, _, _ = timed(saf, lay, [0] * H, args.steps, [dom], flush, stream, world)
        _, kms0, _ = timed(saf, lay, [0] * H, args.steps, list(lay.kernels), flush, stream, world)
        ao_ms = max_over_ranks(sum(ms0) / len(ms0), world, dev)
        allord = {"ms_per_step": ao_ms, "speedup": ao_ms / step_ms,
                  "ideal_speedup": F.layer_flops(B, H, 0, T, d, not w.fwd_only) /
                  F.layer_flops(B, H, w.F, T, d, not w.fwd_only),
                  "kernel_ms": kms0}

    prepared = None
    trainable = None
    if w.F > 0:
        prepared = time_prepared(saf, lay, args, dom, flush, stream, world, dev, total_flops,
                                 allord["ms_per_step"] if allord else None)
    if w.F > 0:
        if not w.fwd_only and not lay.gqa:
            lay.step(frozen)   # o and lse of the frozen-mask step
            trainable = time_pattern_grad(saf, lay, args, flush, stream, world, dev, step_ms, backward_ms(kms))

    # end to end: host buffers in, host buffers out, through the same C ABI
    e2e = None
    if args.e2e:
        host_in = {n: x[n].pin_memory() for n in ("q", "k", "v", "do", "a", "r")}
        host_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
        if w.fwd_only:
            for n in ("dq", "dk", "dv"):
                host_out.pop(n)
        in_names = ("q", "k", "v", "a", "r") + (() if w.fwd_only else ("do",))
        h2d = sum(host_in[n].numel() * host_in[n].element_size() for n in in_names)
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        dev_out = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}

        # The batch goes through in chunks of batch entries (slices are independent), so
        # that the host-to-device copy of chunk c + 1 and the device-to-host copy of
        # chunk c - 1 run on their own streams while chunk c computes. Every byte of the
        # step's inputs and results still crosses in the timed region.
        sizes = e2e_chunk_sizes(B, args.e2e_chunks)
        nch = len(sizes)
        bounds = [sum(sizes[:c]) for c in range(nch + 1)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        per_batch = ("q", "k", "v", "do")

        def e2e_step():
            s_in.wait_stream(stream)   # the previous step (and the L2 flush) are done with the buffers
            ev_in = []
            with torch.cuda.stream(s_in):
                for n in ("a", "r"):
                    if n in in_names:
                        g[n].copy_(host_in[n], non_blocking=True)
                for c in range(nch):
                    sl = slice(bounds[c], bounds[c + 1])
                    for n in in_names:
                        if n in per_batch:
                            g[n][sl].copy_(host_in[n][sl], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(s_in)
                    ev_in.append(e)
            for c in range(nch):
                sl = slice(bounds[c], bounds[c + 1])
                stream.wait_event(ev_in[c])
                fwd = saf.saf_attn_fwd_gqa if lay.gqa else saf.saf_attn_fwd
                bwd = saf.saf_attn_bwd_gqa if lay.gqa else saf.saf_attn_bwd
                fwd(g["q"][sl], g["k"][sl], g["v"][sl], g["a"], g["r"], frozen, o=o[sl], lse=lse[sl], workspace=ws)
                if not w.fwd_only:
                    bwd(g["q"][sl], g["k"][sl], g["v"][sl], o[sl], g["do"][sl], lse[sl], g["a"], g["r"], frozen,
                        dq=dq[sl], dk=dk[sl], dv=dv[sl], workspace=ws)
                e = torch.cuda.Event()
                e.record(stream)
                s_out.wait_event(e)
                with torch.cuda.stream(s_out):
                    for n, t in host_out.items():
                        t[sl].copy_(dev_out[n][sl], non_blocking=True)
            stream.wait_stream(s_out)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        K = args.steps
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        barrier(world)
        for i in range(K):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            e2e_step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in evs) / K, world, dev)
        e2e = {"value": total_flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "chunks": sizes}

    # the other workloads of the same layer, timed in the same run (not the headline)
    others = None
    if args.other_workloads:
        del lay, g, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
        others = {}
        for name in OTHER_WORKLOADS:
            if name != w.name:
                others[name] = measure_workload(saf, WORKLOADS[name], args, dev, world, rank, stream, flush,
                                                peaks, peak_src)

    if rank != 0:
        return 0

    # dominant kernel: the longest kernel of the step, timed by its own events
    # inside the timed region
    roofline = None
    if dom in kms_dom:
        roofline = kernel_roofline(dom, kms_dom, w, peaks, peak_src)
        roofline["traffic"] = traffic_for(dom, w.name)
        roofline["kernel_ms"] = kms

    cpu = None
    if args.cpu_baseline and world == 1:
        run, sflops, desc = oracle_sample(w, x)
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
        cpu = {"value": sflops / dt / 1e12, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
               "sample": desc, "seconds": dt}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "F": w.F, "T": w.T, "d": w.d,
                   "frozen_heads": [h for h in range(H) if frozen[h]],
                   "l2": "flushed (256 MB write) before every timed step; inputs also exceed L2",
                   "parallelism": f"replicas x{world}, one batch per GPU"},
        "tokens_per_s": tokens,
        "frac_of_bf16_peak": value / world / peaks["bf16_tflops"],
        "ms_spread": spread(ms),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "all_ordinary": allord,
        "prepared_normalisers": prepared,
        "trainable_patterns": trainable,
        "other_workloads": others,
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
        "peaks": {"source": peak_src, "bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"]},
        "src": _src_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# DRAM traffic of the dominant kernels, from an ncu capture
# ---------------------------------------------------------------------------

TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
NCU_KERNELS = {"fwd_tc_kernel": "fwd", "bwd_tc_kernel": "bwd"}


def traffic_for(kernel, workload):
    """DRAM bytes per launch of `kernel` at `workload`, if a capture was taken on
    the current sources of that kernel (else None)."""
    if not os.path.exists(TRAFFIC_PATH):
        return None
    with open(TRAFFIC_PATH) as f:
        tt = json.load(f)
    return tt.get(f"{kernel}|{workload}|{_src_hash(kernel)}")


def record_traffic(csv_path, workload, out_path):
    """Read an ncu CSV with dram__bytes_read.sum and dram__bytes_write.sum per
    launch and store read + write bytes per launch of each tensor-core kernel,
    keyed by kernel, workload and the hash of the kernel's sources as they are
    now (run this where and when the capture ran, on the same sources)."""
    import csv
    scale = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "kibyte": 1024.0, "mibyte": 1024.0 ** 2,
             "gibyte": 1024.0 ** 3}
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    per = {}
    for row in csv.DictReader(lines):
        kname = row.get("Kernel Name", "")
        short = next((v for k, v in NCU_KERNELS.items() if k in kname), None)
        metric = row.get("Metric Name", "")
        if short is None or metric not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        val = float(row["Metric Value"].replace(",", "")) * scale[row.get("Metric Unit", "byte").lower()]
        per.setdefault(short, {}).setdefault(row["ID"], 0.0)
        per[short][row["ID"]] += val
    tt = {}
    if os.path.exists(out_path):
        with open(out_path) as f:
            tt = json.load(f)
    # drop entries of sources that no longer exist
    tt = {k: v for k, v in tt.items() if k.rsplit("|", 1)[-1] == _src_hash(k.split("|", 1)[0])}
    for short, launches in per.items():
        vals = list(launches.values())
        tt[f"{short}|{workload}|{_src_hash(short)}"] = sum(vals) / len(vals)
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    with open(out_path, "w") as f:
        json.dump(tt, f, indent=1, sort_keys=True)
    print(json.dumps({"recorded": {s: len(v) for s, v in per.items()}, "workload": workload, "out": out_path}))
    return 0 if per else 1


def spawn_ranks(args):
    """`--gpus N` without a torchrun environment: start N local ranks the way the
    driver does (torchrun, one process per GPU, rendezvous on 127.0.0.1)."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-all-ordinary", dest="all_ordinary", action="store_false")
    ap.add_argument("--e2e-chunks", default="",
                    help="batch entries per chunk of the end-to-end step, e.g. 2,2,2,2 (default: by batch size)")
    ap.add_argument("--no-other-workloads", dest="other_workloads", action="store_false",
                    help="time only the named workload (by default the other bench workloads are timed too)")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="seconds of untimed steps under the clock sampler before the timed region")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="store the DRAM bytes of an ncu capture (--csv, dram__bytes_read/write.sum) of --workload")
    ap.add_argument("--traffic-out", default=TRAFFIC_PATH)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    w = WORKLOADS[args.workload]
    if args.record_traffic:
        return record_traffic(args.record_traffic, w.name, args.traffic_out)
    rank, world, _ = dist_info()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return spawn_ranks(args)
    if "WORLD_SIZE" in os.environ and world != args.gpus:
        print(json.dumps({"error": f"--gpus {args.gpus} but WORLD_SIZE={world}"}), flush=True)
        return 2
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
