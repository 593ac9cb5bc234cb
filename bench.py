"""Benchmark: packed (block-diagonal causal) attention forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole path over one batch: segment-range tile table,
forward, tile table again, delta, dQ, dK/dV -- the same kernels, in the same
order, as pa_fwd followed by pa_bwd. The default workload is the 8k row
(B=1, N=8192, Hq=32, Hkv=8, D=128, bf16) in one segment; the same row split
into packed segments is measured too and reported under "packed".

Timing: W warm-up steps, then K timed steps; every step is bracketed by CUDA
events on the launching stream, with the L2 flushed (a 256 MiB write) between
steps outside the events; reported times are the median over the K steps. Useful FLOPs count only visible pairs (j <= i, same
segment, padding segments excluded): 4*D per pair forward, 10*D backward.
Under torchrun each rank runs its own replica of the workload (weak scaling,
no collective on the data path); the reported time is the max over ranks.

--impl reference times the fp64 CPU oracle on this machine's host cores on a
bounded sample of the same workload (one query head with its kv head per
step), in the same metric.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "packed causal attn fwd+bwd useful TFLOPS at N=8192; % of GB300 bf16 tensor peak"
UNIT = "TFLOPS"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
KERNEL_SOURCES = {"fwd": "fwd.cu", "dq": "bwd_dq.cu", "dkv": "bwd_dkv.cu", "delta": "prologue.cu"}
# algorithmic flops per visible pair, per kernel (executed by the split design)
FLOPS_PER_PAIR = {"fwd": 4, "dq": 6, "dkv": 8}


# ------------------------------------------------------------------ accounting
def segment_lengths(w: synth.Workload):
    for b in range(w.B):
        lens = list(w.lengths[b])
        pad = w.pad[b] if w.pad else 0
        yield lens, pad


def visible_pairs_per_head(w: synth.Workload, exclude_padding: bool = True) -> int:
    """Pairs (i, j) with j <= i in the same segment, summed over rows; the
    padding segment (last of a row, when the row has padding) is excluded."""
    total = 0
    for lens, pad in segment_lengths(w):
        use = lens[:-1] if (exclude_padding and pad) else lens
        total += sum(L * (L + 1) // 2 for L in use)
    return total


def useful_flops(w: synth.Workload) -> float:
    return 14.0 * w.D * visible_pairs_per_head(w) * w.Hq


def executed_tile_pairs(w: synth.Workload) -> int:
    """(query tile, key tile) pairs the kernels visit per head (range-overlap walk)."""
    T = w.N // 128
    n = 0
    for b in range(w.B):
        s = w.seg[b].reshape(T, 128)
        lo, hi = s.min(1), s.max(1)
        for tq in range(T):
            n += int(np.sum((lo[: tq + 1] <= hi[tq]) & (lo[tq] <= hi[: tq + 1])))
    return n


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", 0)),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel and on this workload (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "segment_masked_causal_gb300", "csrc", KERNEL_SOURCES[kernel])
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d.get("source_sha256_16"):
        return None
    return float(d["bytes_per_launch"])


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank processes its own independent batch of the same shape."""
    return base_seed + 7919 * rank


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ the GPU arm
class Runner:
    def __init__(self, w: synth.Workload, dev, seed: int):
        import torch
        import segment_masked_causal_gb300 as pa
        self.pa, self.torch, self.w, self.dev = pa, torch, w, dev
        w2 = synth.Workload(w.name, w.B, w.Hq, w.Hkv, w.N, w.D, seed, w.seg, w.lengths, w.pad)
        t = w2.tensors()
        self.host = t
        to = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)
        self.q, self.k, self.v, self.do = (to(t[x]) for x in ("q", "k", "v", "do"))
        self.seg = torch.from_numpy(w.seg).to(dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.ws = pa.workspace(self.q, self.k)
        self.flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush(self):
        self.flush_buf.zero_()

    def step(self, events=None, causal=False):
        """The kernels of pa_fwd + pa_bwd, one call per kernel, events between."""
        pa, seg = self.pa, (None if causal else self.seg)
        q, k, v, do = self.q, self.k, self.v, self.do
        ev = events or [None] * 7
        rec = lambda e: e is not None and e.record()
        rec(ev[0])
        pa.pa_build_tile_table(q, k, seg, self.ws)
        rec(ev[1])
        pa.pa_fwd_tiles(q, k, v, seg, self.out, self.lse, self.ws)
        rec(ev[2])
        pa.pa_build_tile_table(q, k, seg, self.ws)
        rec(ev[3])
        pa.pa_bwd_delta(q, k, self.out, do, self.lse, self.ws)
        rec(ev[4])
        pa.pa_bwd_dq(q, k, v, do, self.lse, seg, self.dq, self.ws)
        rec(ev[5])
        pa.pa_bwd_dkv(q, k, v, do, self.lse, seg, self.dk, self.dv, self.ws)
        rec(ev[6])

    def checked_step(self, causal=False):
        """One untimed step that reads the status word after the forward and
        after the backward (each tile-table step clears it)."""
        pa, seg = self.pa, (None if causal else self.seg)
        pa.pa_build_tile_table(self.q, self.k, seg, self.ws)
        pa.pa_fwd_tiles(self.q, self.k, self.v, seg, self.out, self.lse, self.ws)
        st = pa.pa_device_status(self.ws)
        if st != 0:
            raise RuntimeError(f"device status after the forward {st:#x}")
        pa.pa_build_tile_table(self.q, self.k, seg, self.ws)
        pa.pa_bwd_delta(self.q, self.k, self.out, self.do, self.lse, self.ws)
        pa.pa_bwd_dq(self.q, self.k, self.v, self.do, self.lse, seg, self.dq, self.ws)
        pa.pa_bwd_dkv(self.q, self.k, self.v, self.do, self.lse, seg, self.dk, self.dv, self.ws)
        st = pa.pa_device_status(self.ws)
        if st != 0:
            raise RuntimeError(f"device status after the backward {st:#x}")

    def timed(self, steps: int, warmup: int, causal=False, sampler=None):
        torch = self.torch
        self.checked_step(causal)
        for _ in range(warmup):
            self.step(causal=causal)
            self.flush()
        torch.cuda.synchronize()
        barrier(self.dev)
        if sampler:
            sampler.start()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
        for i in range(steps):
            self.flush()
            self.step(evs[i], causal=causal)
        torch.cuda.synchronize()
        barrier(self.dev)
        clocks = sampler.stop() if sampler else None
        status = self.pa.pa_device_status(self.ws)
        if status != 0:
            raise RuntimeError(f"device status {status:#x}")
        per = {"table_fwd": [], "fwd": [], "table_bwd": [], "delta": [], "dq": [], "dkv": [], "step": []}
        keys = ["table_fwd", "fwd", "table_bwd", "delta", "dq", "dkv"]
        for e in evs:
            for n, key in enumerate(keys):
                per[key].append(e[n].elapsed_time(e[n + 1]))
            per["step"].append(e[0].elapsed_time(e[6]))
        return {k: statistics.median(v) for k, v in per.items()}, clocks

    def e2e(self, steps: int, warmup: int):
        """Public pa_fwd + pa_bwd with pinned host inputs/outputs: every step
        copies q, k, v, dO and seg host -> device and O, lse, dQ, dK, dV
        device -> host inside the timed region. As a training loop would,
        the copies run on streams of their own with two device buffer sets,
        so a step's input copy and the previous step's output copy overlap
        the kernels of the step between them; every step still moves all of
        its bytes."""
        torch, pa = self.torch, self.pa
        pin = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
        h_in = {x: pin(self.host[x]) for x in ("q", "k", "v", "do")}
        h_seg = torch.from_numpy(self.w.seg).pin_memory()
        outs = (("o", self.out), ("lse", self.lse), ("dq", self.dq), ("dk", self.dk), ("dv", self.dv))
        h_out = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in outs}
        # two device sets of inputs and outputs: set 0 is the bench's own tensors
        sets = [{"q": self.q, "k": self.k, "v": self.v, "do": self.do, "seg": self.seg,
                 **{n: t for n, t in outs}}]
        sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        in_done = [torch.cuda.Event() for _ in sets]
        cmp_done = [torch.cuda.Event() for _ in sets]
        out_done = [torch.cuda.Event() for _ in sets]

        def one(i):
            d = sets[i % 2]
            with torch.cuda.stream(s_in):  # inputs, once step i-2's kernels have read this set
                s_in.wait_event(cmp_done[i % 2])
                for x in ("q", "k", "v", "do"):
                    d[x].copy_(h_in[x], non_blocking=True)
                d["seg"].copy_(h_seg, non_blocking=True)
                in_done[i % 2].record(s_in)
            with torch.cuda.stream(s_cmp):  # kernels, once step i-2's outputs have been read back
                s_cmp.wait_event(in_done[i % 2])
                s_cmp.wait_event(out_done[i % 2])
                pa.pa_fwd(d["q"], d["k"], d["v"], d["seg"], d["o"], d["lse"], self.ws, stream=s_cmp)
                pa.pa_bwd(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], d["seg"], d["dq"], d["dk"], d["dv"],
                          self.ws, stream=s_cmp)
                cmp_done[i % 2].record(s_cmp)
            with torch.cuda.stream(s_out):  # outputs
                s_out.wait_event(cmp_done[i % 2])
                for n, _ in outs:
                    h_out[n].copy_(d[n], non_blocking=True)
                out_done[i % 2].record(s_out)

        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        barrier(self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(steps):
            one(i)
        s_out.wait_stream(s_in)  # the end event comes after every stream's last operation
        s_out.wait_stream(s_cmp)
        e1.record(s_out)
        torch.cuda.synchronize()
        barrier(self.dev)
        ms = e0.elapsed_time(e1) / steps
        h2d = sum(t.numel() * t.element_size() for t in h_in.values()) + h_seg.numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in h_out.values())
        return ms, h2d, d2h


def host_link_gbs(dev, nbytes: int = 256 << 20, reps: int = 3):
    """Pinned-memory copy rates of this machine, host to device and back (GB/s,
    each direction alone), so that the e2e figure can be read against the
    link it rides on. None if the measurement fails."""
    import torch
    try:
        h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        d.copy_(h)
        h.copy_(d)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rates = {}
        for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
            e0.record()
            for _ in range(reps):
                dst.copy_(src, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            rates[name] = round(nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
        del h, d
        return rates
    except Exception:
        return None


def cpu_baseline(w: synth.Workload, seconds: float = 12.0, max_heads: int = 8):
    """The oracle, as it stands, on a bounded sample: complete fwd+bwd of one
    query head against its kv head (the per-head share of dK/dV), repeated over
    heads until `seconds` have passed."""
    import oracle
    t = w.tensors()
    done, elapsed = 0, 0.0
    G = w.Hq // w.Hkv
    while done < min(max_heads, w.Hq) and (elapsed < seconds or done == 0):
        h = (done * 5) % w.Hq
        hk = h // G
        q = synth.bf16_bits_to_f64(t["q"][:, h:h + 1])
        k = synth.bf16_bits_to_f64(t["k"][:, hk:hk + 1])
        v = synth.bf16_bits_to_f64(t["v"][:, hk:hk + 1])
        do = synth.bf16_bits_to_f64(t["do"][:, h:h + 1])
        t0 = time.perf_counter()
        oracle.attention(q, k, v, w.seg, w.scale, do)
        elapsed += time.perf_counter() - t0
        done += 1
    flops = 14.0 * w.D * visible_pairs_per_head(w) * done
    return {"value": flops / elapsed / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} of {w.Hq} query heads of {w.name}, each a complete fp64 forward+backward against "
                      f"its kv head ({elapsed:.1f} s)"}


def run_ours(args):
    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    if args.gpus != world:
        # one rank per GPU: N GPUs come from a launcher's N processes (torchrun);
        # a single process times one GPU whatever --gpus says
        print(f"bench.py: --gpus {args.gpus} with {world} process(es): timing {world} GPU(s), one per process",
              file=sys.stderr, flush=True)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if local == 0:
        import __graft_entry__
        __graft_entry__.build()
    barrier(dev)
    import segment_masked_causal_gb300 as pa
    pa.lib()

    w = synth.workload(args.workload)
    r = Runner(w, dev, replica_seed(w.seed, rank))
    sampler = ClockSampler(local) if rank == 0 else None
    t, clocks = r.timed(args.steps, args.warmup, sampler=sampler)
    step_ms = reduce_max(t["step"], dev)
    kern = {k: reduce_max(t[k], dev) for k in ("table_fwd", "fwd", "table_bwd", "delta", "dq", "dkv")}
    flops = useful_flops(w)
    value = flops * world / (step_ms * 1e-3) / 1e12
    pk = peaks()
    pairs = visible_pairs_per_head(w) * w.Hq
    dom = max(("fwd", "dq", "dkv"), key=lambda k: kern[k])
    achieved = FLOPS_PER_PAIR[dom] * w.D * pairs / (kern[dom] * 1e-3) / 1e12
    traffic = kernel_traffic(dom, w.name)
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": traffic,
                "peak_source": pk["source"] + " bf16 burst (MEASURED_PEAKS.json)" if pk["source"] == "measured"
                else "fallback 1.9 PFLOP/s"}
    # per query row: read O and dO (bf16) and lse; write delta and lse*log2(e)
    delta_bytes = 2 * 2 * w.B * w.Hq * w.N * w.D + 3 * 4 * w.B * w.Hq * w.N
    kernels = {k: {"ms": round(v, 4)} for k, v in kern.items()}
    for k in ("fwd", "dq", "dkv"):
        kernels[k]["tflops"] = round(FLOPS_PER_PAIR[k] * w.D * pairs / (kern[k] * 1e-3) / 1e12, 2)
    kernels["delta"]["gbs"] = round(delta_bytes / (kern["delta"] * 1e-3) / 1e9, 1)
    kernels["delta"]["hbm_frac"] = round(kernels["delta"]["gbs"] / pk["hbm_gbs"], 4)

    e2e_ms, h2d, d2h = r.e2e(args.steps, args.warmup)
    e2e_ms = reduce_max(e2e_ms, dev)
    link = host_link_gbs(dev)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "segments": sum(len(l) for l in w.lengths), "seed": w.seed,
                   "l2": "flushed between timed steps (256 MiB write, outside the events)",
                   "parallelism": "replicas" if world == 1 else f"replicas x{world} (no data-path collective)"},
        "frac_of_peak": round(value / world / pk["bf16_tflops"], 4),
        "frac_of_sustained_peak": (round(value / world / pk["bf16_tflops_sustained"], 4)
                                   if pk.get("bf16_tflops_sustained") else None),
        "useful_tflop_per_step": round(flops / 1e12, 4),
        "executed_tile_pairs_per_head": executed_tile_pairs(w),
        "kernels": kernels,
        "roofline": roofline,
        "gpu_launches": 6 * args.steps,
        "e2e": {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "overlap": "input and output copies on their own streams, two device buffer sets",
                "host_link_gbs": link},
        "clocks": clocks,
    }
    if not args.no_extras and w.name == "8k_one_segment":
        line["packed"] = packed_extras(dev, rank, args)
        line["head_dim_96"] = head_dim_96_extra(dev, rank, args)
        line["staged_layouts"] = staged_layout_extras(dev, rank, args)
        line["configs"] = config_extras(dev, rank, args)
        line["single_pass_backward"] = single_pass_extra(dev, rank, args)
    if not args.no_extras and w.name == "8k_one_segment" and rank == 0 and world == 1:
        line["linear_cross_entropy"] = lce_extra()
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def packed_extras(dev, rank, args):
    """The 8k row in packed segments, and the causal entry points on the
    one-segment row: per-kernel times for the skip speedup (packed vs causal on
    the same length) and the identical-work overhead (packed kernels with one
    segment vs the causal ones)."""
    steps = max(3, min(args.steps, 10))
    one = synth.workload("8k_one_segment")
    pk = synth.workload("8k_packed")
    r1 = Runner(one, dev, replica_seed(one.seed, rank))
    t_packed1, _ = r1.timed(steps, 2)
    t_causal, _ = r1.timed(steps, 2, causal=True)
    del r1
    r2 = Runner(pk, dev, replica_seed(pk.seed, rank))
    t_multi, _ = r2.timed(steps, 2)
    del r2
    flops = useful_flops(pk)
    out = {"workload": pk.name, "segments": len(pk.lengths[0]),
           "useful_tflops": round(flops / (t_multi["step"] * 1e-3) / 1e12, 3),
           "ms_per_step": round(t_multi["step"], 4),
           "visible_fraction_of_causal": round(visible_pairs_per_head(pk) / visible_pairs_per_head(one), 4),
           "executed_tile_fraction_of_causal": round(executed_tile_pairs(pk) / executed_tile_pairs(one), 4)}
    for k in ("fwd", "dq", "dkv", "step"):
        out[k] = {"causal_ms": round(t_causal[k], 4), "packed_one_segment_ms": round(t_packed1[k], 4),
                  "packed_multi_ms": round(t_multi[k], 4),
                  "skip_speedup_vs_causal": round(t_causal[k] / t_multi[k], 3),
                  "one_segment_overhead_vs_causal": round(t_packed1[k] / t_causal[k] - 1.0, 4)}
    return out


def oracle_estimate(w: synth.Workload, max_rows: int = 2048) -> dict:
    """The fp64 oracle's time for a whole fwd+bwd step of `w` on this host's
    cores. The oracle's time does not depend on the values, so one query
    head's worth of seeded inputs of the workload's shape is drawn. Rows with
    up to ~4e9 (pairs x D) per head: the complete forward + backward of one
    query head against its kv head (that head's share of dK/dV), times Hq.
    Longer rows: forward and dQ of `max_rows` query rows spread evenly over
    the head, scaled by visible pairs; the oracle's dK/dV visits the same pairs
    with the same work per pair as its dQ, so the step is forward + 2 x dQ."""
    import oracle
    oracle.build()
    shape = (w.B, 1, w.N, w.D)
    q, k, v, do = (synth.bf16_bits_to_f64(synth.bf16_normal(w.seed, 11 + i, shape)) for i in range(4))
    per_head = visible_pairs_per_head(w, exclude_padding=False)
    if per_head * w.D <= 4e9:
        t0 = time.perf_counter()
        oracle.attention(q, k, v, w.seg, w.scale, do)
        sec = (time.perf_counter() - t0) * w.Hq
        sample = "complete fp64 forward + backward of one query head, times Hq"
    else:
        flat = w.B * w.N
        rows = np.unique(np.linspace(0, flat - 1, min(max_rows, flat)).astype(np.int64))
        # visible pairs of the sampled rows: the row's position in its segment, plus one
        pos = np.concatenate([np.concatenate([np.arange(L) for L in lens]) for lens, _ in segment_lengths(w)])
        pairs = float(np.sum(pos[rows] + 1))
        t0 = time.perf_counter()
        o, lse, delta = oracle.forward(q, k, v, w.seg, w.scale, do, rows=rows)
        t1 = time.perf_counter()
        lse_f, delta_f = np.zeros((w.B, 1, w.N)), np.zeros((w.B, 1, w.N))
        lse_f.reshape(-1)[rows], delta_f.reshape(-1)[rows] = lse.reshape(-1), delta.reshape(-1)
        oracle.dq(q, k, v, w.seg, w.scale, do, lse_f, delta_f, rows=rows)
        t2 = time.perf_counter()
        sec = ((t1 - t0) + 2 * (t2 - t1)) / pairs * per_head * w.Hq
        sample = (f"forward and dQ of {len(rows)} query rows of one head, scaled by visible pairs "
                  f"(step = forward + 2 x dQ)")
    return {"seconds_per_step_est": round(sec, 2), "cores": oracle.num_threads(), "sample": sample}


def _kernel_ms(t):
    return {k: round(t[k], 4) for k in ("fwd", "delta", "dq", "dkv")}


def config_extras(dev, rank, args):
    """Every other configuration of the target, each timed as the main line
    is (the steps of pa_fwd + pa_bwd, L2 flushed between steps): config 2
    (2k GQA causal), config 3 (short packed rows, the pages' Alpaca
    analogue) against the causal entry points and the same rows in one
    segment, and config 5 (32k / 64k rows at head dim 64, one segment and
    packed). Each reports useful TFLOP/s, its fraction of the measured bf16
    peak and the oracle's estimated time for the same step."""
    steps = max(3, min(args.steps, 10))
    pk = peaks()
    out = {}

    def entry(w, t):
        flops = useful_flops(w)
        return {"B": w.B, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                "segments": sum(len(l) for l in w.lengths), "ms_per_step": round(t["step"], 4),
                "useful_tflops": round(flops / (t["step"] * 1e-3) / 1e12, 3),
                "frac_of_peak": round(flops / (t["step"] * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                "kernels_ms": _kernel_ms(t)}

    def run(w, causal=False):
        r = Runner(w, dev, replica_seed(w.seed, rank))
        t, _ = r.timed(steps, 2, causal=causal)
        del r
        return t

    w2 = synth.workload("causal_2k_gqa")
    out["causal_2k_gqa"] = entry(w2, run(w2))
    # config 3: packed rows vs the causal kernels on the same tokens, and the
    # packed kernels on the same shape in one segment per row
    w3 = synth.workload("packed_4x4096_short")
    t_multi = run(w3)
    t_causal = run(w3, causal=True)
    one = synth.custom(w3.B, w3.Hq, w3.Hkv, w3.N, w3.D, [[w3.N]] * w3.B, seed=w3.seed)
    t_one = run(one)
    e = entry(w3, t_multi)
    e["visible_fraction_of_causal"] = round(visible_pairs_per_head(w3) / visible_pairs_per_head(one), 4)
    e["executed_tile_fraction_of_causal"] = round(executed_tile_pairs(w3) / executed_tile_pairs(one), 4)
    for k in ("fwd", "dq", "dkv", "step"):
        e[k] = {"causal_ms": round(t_causal[k], 4), "packed_one_segment_ms": round(t_one[k], 4),
                "packed_multi_ms": round(t_multi[k], 4),
                "skip_speedup_vs_causal": round(t_causal[k] / t_multi[k], 3),
                "one_segment_overhead_vs_causal": round(t_one[k] / t_causal[k] - 1.0, 4)}
    out["packed_4x4096_short"] = e
    for n in (32, 64):
        w1 = synth.workload(f"long_{n}k_one_segment")
        wp = synth.workload(f"long_{n}k_packed")
        t1, tp = run(w1), run(wp)
        out[w1.name] = entry(w1, t1)
        e = entry(wp, tp)
        e["executed_tile_fraction_of_one_segment"] = round(executed_tile_pairs(wp) / executed_tile_pairs(w1), 4)
        e["skip_speedup_vs_one_segment"] = {k: round(t1[k] / tp[k], 3) for k in ("fwd", "dq", "dkv", "step")}
        out[wp.name] = e
    if rank == 0 and not args.no_cpu:
        for name in out:
            out[name]["oracle"] = oracle_estimate(synth.workload(name))
    return out


def single_pass_extra(dev, rank, args, names=("8k_one_segment", "8k_packed", "packed_4x4096_short", "causal_2k_gqa",
                                               "long_32k_one_segment", "long_32k_packed", "long_64k_one_segment",
                                               "long_64k_packed")):
    """The split backward (tile table + delta + dQ + dK/dV kernels) against
    the single-pass backward (pa_bwd_fused: tile table + delta with the
    accumulator zeroed + one kernel + the bf16 rounding), each timed as a
    whole with CUDA events, L2 flushed before every call, median of the
    steps, on configs 2-5."""
    import torch
    import segment_masked_causal_gb300 as pa
    steps = max(3, min(args.steps, 10))
    out = {}
    for name in names:
        w = synth.workload(name)
        r = Runner(w, dev, replica_seed(w.seed, rank))
        r.checked_step()
        fws = torch.empty(pa.pa_bwd_fused_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.D), dtype=torch.uint8,
                          device=dev)
        fdq, fdk, fdv = torch.empty_like(r.dq), torch.empty_like(r.dk), torch.empty_like(r.dv)
        q, k, v, do, seg = r.q, r.k, r.v, r.do, r.seg

        def split():
            pa.pa_build_tile_table(q, k, seg, r.ws)
            pa.pa_bwd_delta(q, k, r.out, do, r.lse, r.ws)
            pa.pa_bwd_dq(q, k, v, do, r.lse, seg, r.dq, r.ws)
            pa.pa_bwd_dkv(q, k, v, do, r.lse, seg, r.dk, r.dv, r.ws)

        def fused():
            pa.pa_bwd_fused(q, k, v, r.out, do, r.lse, seg, fdq, fdk, fdv, fws)

        res = {}
        for key, fn, ws in (("split_ms", split, r.ws), ("single_pass_ms", fused, fws)):
            for _ in range(2):
                fn()
                r.flush()
            evs = []
            for _ in range(steps):
                r.flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                evs.append((a, b))
            torch.cuda.synchronize()
            st = pa.pa_device_status(ws)
            if st != 0:
                raise RuntimeError(f"device status {st:#x} after the {key[:-3]} backward")
            res[key] = round(statistics.median(a.elapsed_time(b) for a, b in evs), 4)
        res["single_pass_speedup"] = round(res["split_ms"] / res["single_pass_ms"], 3)
        res["dk_dv_bitwise_equal"] = bool(torch.equal(fdk, r.dk) and torch.equal(fdv, r.dv))
        out[name] = res
        del r, fws, fdq, fdk, fdv
        torch.cuda.empty_cache()
    return out


def head_dim_96_extra(dev, rank, args):
    """The same 8k one-segment step at head dim 96 (the 128-wide kernels on
    tiles whose columns 96..127 are zero-filled): useful TFLOP/s counted at
    D = 96, and per-kernel times."""
    steps = max(3, min(args.steps, 10))
    w = synth.workload("8k_one_segment_d96")
    r = Runner(w, dev, replica_seed(w.seed, rank))
    t, _ = r.timed(steps, 2)
    del r
    return {"workload": w.name, "useful_tflops": round(useful_flops(w) / (t["step"] * 1e-3) / 1e12, 3),
            "ms_per_step": round(t["step"], 4), **{k + "_ms": round(t[k], 4) for k in ("fwd", "dq", "dkv")}}


def staged_layout_extras(dev, rank, args):
    """The full public calls (pa_fwd + pa_bwd) on the 8k one-segment row with
    contiguous tensors, on the same values held as (B, N, H, D) memory (the
    strided calls, which copy in and out of the workspace), and on a row of
    8,000 tokens (N not a multiple of 128, same copies)."""
    import torch
    import segment_masked_causal_gb300 as pa
    steps = max(3, min(args.steps, 10))
    bf = torch.bfloat16

    def timed(q, k, v, do, seg, strided):
        B, Hq, N, D = q.shape
        mk = (lambda t: torch.empty_strided(t.shape, t.stride(), dtype=bf, device=dev))
        out, dq, dk, dv = mk(q), mk(q), mk(k), mk(k)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
        ws = pa.workspace(q, k, strided=strided)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def one():
            if strided:
                pa.pa_fwd_strided(q, k, v, seg, out, lse, ws)
                pa.pa_bwd_strided(q, k, v, out, do, lse, seg, dq, dk, dv, ws)
            else:
                pa.pa_fwd(q, k, v, seg, out, lse, ws)
                pa.pa_bwd(q, k, v, out, do, lse, seg, dq, dk, dv, ws)
        for _ in range(2):
            one()
            flush.zero_()
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            one()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        if pa.pa_device_status(ws) != 0:
            raise RuntimeError("device status after staged-layout run")
        return statistics.median(ts)

    one_seg = synth.workload("8k_one_segment")
    r = Runner(one_seg, dev, replica_seed(one_seg.seed, rank))
    t_plain = timed(r.q, r.k, r.v, r.do, r.seg, False)
    bnhd = lambda t: t.transpose(1, 2).contiguous().transpose(1, 2)
    t_bnhd = timed(bnhd(r.q), bnhd(r.k), bnhd(r.v), bnhd(r.do), r.seg, True)
    del r
    w8000 = synth.custom(1, 32, 8, 8000, 128, [[8000]], seed=one_seg.seed)
    r = Runner(w8000, dev, replica_seed(one_seg.seed, rank))
    t_8000 = timed(r.q, r.k, r.v, r.do, r.seg, False)
    del r
    return {"workload": one_seg.name, "ms_contiguous": round(t_plain, 4),
            "bnhd_strided": {"ms": round(t_bnhd, 4), "overhead_vs_contiguous": round(t_bnhd / t_plain - 1, 4)},
            "n8000": {"ms": round(t_8000, 4),
                      "useful_tflops": round(useful_flops(w8000) / (t_8000 * 1e-3) / 1e12, 3)}}


LCE_SHAPE = (8192, 151936, 4096)  # tokens, vocabulary, hidden: the README's isolated loss-layer shape


def lce_measure(steps: int = 5, warmup: int = 2, shape=None) -> dict:
    """The fused linear cross-entropy forward (pa_lce_fwd) and backward
    (pa_lce_bwd, with and without the head's gradient) at N = 8192,
    V = 151,936, D = 4096 in bf16 (mlx-train-perf 0.5.1 README, "The fused
    cross-entropy loss", its isolated measurement). Seeded device-side
    normals (head scaled by 2/sqrt(D)); the 1.2 GB head is larger than L2.
    Tensor-bound: 2 N V D flops for the forward."""
    import torch
    import segment_masked_causal_gb300 as pa
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    N, V, D = shape or LCE_SHAPE
    gen = torch.Generator(device=dev)
    gen.manual_seed(1008)
    H = torch.randn((N, D), generator=gen, device=dev).to(torch.bfloat16)
    W = (torch.randn((V, D), generator=gen, device=dev) * (2.0 / math.sqrt(D))).to(torch.bfloat16)
    T = torch.randint(0, V, (N,), generator=gen, device=dev, dtype=torch.int32)
    nll, lse, tgt = (torch.empty(N, dtype=torch.float32, device=dev) for _ in range(3))
    ws = torch.empty(pa.pa_lce_workspace_bytes(N, V, D), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        pa.pa_lce_fwd(H, W, T, nll, lse, tgt, ws)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        a.record()
        pa.pa_lce_fwd(H, W, T, nll, lse, tgt, ws)
        b.record()
    torch.cuda.synchronize()
    status = pa.pa_device_status(ws)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    tflops = 2.0 * N * V * D / (ms * 1e-3) / 1e12
    pk = peaks()
    out = {"workload": f"N{N} V{V} D{D} bf16", "ms": round(ms, 4), "tflops": round(tflops, 2),
           "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": pk["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": round(tflops / pk["bf16_tflops"], 4)},
           "launches_per_call": 2, "device_status": status,
           "finite": bool(torch.isfinite(nll).all().item() and torch.isfinite(lse).all().item())}
    # the backward for L = mean NLL: dz recomputed per vocabulary chunk, then
    # dW = dz^T H and dH = dz W (6 N V D flops with the head training, 4 N V D
    # without)
    g = torch.full((N,), 1.0 / N, dtype=torch.float32, device=dev)
    dh, dw = torch.empty_like(H), torch.empty_like(W)
    wsb = torch.empty(pa.pa_lce_bwd_workspace_bytes(N, V, D), dtype=torch.uint8, device=dev)
    for train in (True, False):
        for _ in range(warmup):
            pa.pa_lce_bwd(H, W, T, lse, g, dh, dw if train else None, wsb)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            a.record()
            pa.pa_lce_bwd(H, W, T, lse, g, dh, dw if train else None, wsb)
            b.record()
        torch.cuda.synchronize()
        st_b = pa.pa_device_status(wsb)
        ms_b = statistics.median(a.elapsed_time(b) for a, b in evs)
        fl = (6.0 if train else 4.0) * N * V * D
        tf = fl / (ms_b * 1e-3) / 1e12
        key = "backward" if train else "backward_frozen_head"
        out[key] = {"ms": round(ms_b, 4), "tflops": round(tf, 2), "frac_of_peak": round(tf / pk["bf16_tflops"], 4),
                    "device_status": st_b, "finite": bool(torch.isfinite(dh.float()).all().item()),
                    "workspace_bytes": wsb.numel()}
    return out


def lce_extra() -> dict:
    """lce_measure in a child process, so that whatever happens there cannot
    take the main measurement down with it."""
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--lce-only"], capture_output=True,
                           text=True, timeout=300)
        lines = [x for x in r.stdout.strip().splitlines() if x.startswith("{")]
        if r.returncode == 0 and lines:
            return json.loads(lines[-1])
        return {"error": f"exit {r.returncode}: " + (r.stderr.strip().splitlines() or ["no output"])[-1][:300]}
    except Exception as e:  # a timeout or a launch failure is reported, not raised
        return {"error": repr(e)[:300]}


# ------------------------------------------------------------------ the reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = synth.workload(args.workload)
    t = w.tensors()
    G = w.Hq // w.Hkv
    pairs = visible_pairs_per_head(w)

    def one(i):
        h = (i * 5) % w.Hq
        hk = h // G
        f = lambda x, a, b: synth.bf16_bits_to_f64(t[x][:, a:b])
        oracle.attention(f("q", h, h + 1), f("k", hk, hk + 1), f("v", hk, hk + 1), w.seg, w.scale, f("do", h, h + 1))

    for i in range(args.warmup):
        one(i)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        one(args.warmup + i)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.median(times)
    value = 14.0 * w.D * pairs / (ms * 1e-3) / 1e12
    sample = f"one query head (rotating) of {w.Hq} of {w.name} per step, complete fp64 forward+backward"
    line = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "sample": "1 query head per step"},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="8k_one_segment", choices=synth.WORKLOADS)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip the packed / causal comparison runs")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--lce-only", action="store_true",
                    help="only the fused linear cross-entropy forward and backward, printed as one JSON line")
    ap.add_argument("--lce-shape", default=None,
                    help="N,V,D for --lce-only (default 8192,151936,4096, the README's isolated-loss shape)")
    ap.add_argument("--single-pass-only", action="store_true",
                    help="only the split vs single-pass backward comparison on --workload, one JSON line")
    args = ap.parse_args(argv)
    if args.lce_only:
        shape = tuple(int(x) for x in args.lce_shape.split(",")) if args.lce_shape else None
        print(json.dumps(lce_measure(shape=shape)), flush=True)
        return
    if args.single_pass_only:
        import torch
        dev = torch.device("cuda:0")
        print(json.dumps(single_pass_extra(dev, 0, args, names=(args.workload,))), flush=True)
        return
    args.warmup = max(3, args.warmup)  # at least 3 warm-up steps, whatever was asked
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
