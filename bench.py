#!/usr/bin/env python
"""Benchmark of the low-bit all-reduce hot path on GB300.

One step = a simulated W=8 low-bit all-reduce of a GPT-1.3B-shaped flat
gradient (8 rank arrays of 1.3e9 bf16 elements, N(0, 1e-3^2), per-rank seeds)
on one GPU:
  stage 1  8 encoder launches (4-bit, block 128, round to nearest, error
           feedback): read g (bf16) + e, write e', codes, fp16 scales;
  stage 2  8 chunk decoder launches (chunk c = blocks [c*ceil(nb/8), ...)):
           unpack + dequantise the 8 ranks' codes, rank-ordered fp32 sum,
           stage-2 error feedback, requantise to 4 bits, repack.
Metric: GB/s of gradient input processed, counted as fp32 (4 bytes per
element of the 8 ranks), plus the dominant kernel's fraction of the measured
HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every GPU is one rank of the real low-bit all-reduce
(W = N ranks of 1.3e9 bf16 elements each): its encoder, an all-to-all of the
packed chunks over NCCL, the decoder of its own chunk and an all-gather of the
requantised chunks; value = all ranks' elements / the slowest rank's step
time.  --replicas instead runs N independent copies of the single-GPU
simulation.  --impl reference times the CPU oracle (single
thread) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantize-pack & unpack-reduce-requant GB/s of fp32 input; % of HBM roofline"
UNIT = "GB/s"
WORKLOAD = "allreduce_w8_gpt1p3b"
W_RANKS = 8
N_PER_RANK = 1_300_000_000
BITS, BLOCK = 4, 128
ENC_BYTES_PER_ELEM = 2 + 4 + 4 + BITS / 8 + 2 / BLOCK           # g bf16, e in, e' out, codes, scales
DEC_BYTES_PER_ELEM = W_RANKS * (BITS / 8 + 2 / BLOCK) + 4 + 4 + BITS / 8 + 2 / BLOCK  # W inputs, e2 r/w, out

# DRAM traffic per element measured by ncu (dram__bytes_read.sum +
# dram__bytes_write.sum per launch / its elements), valid only while the
# sources of the two kernels' translation units (TRAFFIC_SOURCES) hash to
# `src`.  Captured on the same step with 6e7 elements per rank (3.4 GB on the
# device; each encoder launch moves 0.63 GB, five times the L2), caches left
# alone between launches (ncu --cache-control none), averaged over the step's
# 8 encoder and 8 decoder launches; the step's total equals its algorithmic
# bytes to 0.1 % (the last encoder's dirty lines are written back, and
# counted, during the first decoder), and the bytes per element do not depend
# on the size once it is well above the L2 (2e8 per rank gave 10.5057 and
# 12.6902 on earlier sources).  At 6e7 per rank the encoder launch already
# takes the same spread grid as at full size (sixteen waves of two-row CTAs).
TRAFFIC_SOURCES = ("launch.h", "codec.cuh", "encode_impl.cuh", "encode_bf16.cu", "decode_impl.cuh",
                   "decode_w8.cu")
NCU_TRAFFIC = {
    "encode": {"src": "617886ee3ae3f995", "bytes_per_elem": 10.4931},
    "decode": {"src": "617886ee3ae3f995", "bytes_per_elem": 12.7284},
}


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed, so that a
    comment edit does not invalidate measured traffic figures (the kernel
    sources hold no comment markers inside string literals)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_src_hash(files=None) -> str:
    """Hash of the kernel sources' code (comments and layout ignored): all of
    them, or the named files of the kernel directory."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_gradient_communication_gb300", "csrc")
    names = sorted(files) if files is not None else sorted(
        f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in names:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class AllReduceW8:
    """Device buffers and the launch sequence of one simulated all-reduce.
    p1 / p2 default to the headline parameters (4-bit, block 128, RTN)."""

    def __init__(self, torch, bc, synth, n, W, device, p1=None, p2=None):
        self.torch, self.bc, self.n, self.W = torch, bc, n, W
        base1 = p1 or bc.QParams(BITS, BLOCK, bc.RTN)
        self.p1 = [bc.QParams(base1.bits, base1.block, base1.rounding, seed=1000 + w,
                              hadamard=base1.hadamard) for w in range(W)]
        self.p2 = p2 or bc.QParams(BITS, BLOCK, bc.RTN, philox_stream=1)
        self.x = [synth.gradients("normal", n, 1000 + w, dtype=torch.bfloat16, device=device, sigma=1e-3)
                  for w in range(W)]
        self.err = [torch.zeros(n, dtype=torch.float32, device=device) for _ in range(W)]
        self.codes, self.scales = zip(*[bc.alloc_codes(n, self.p1[0], device) for _ in range(W)])
        self.err2 = torch.zeros(n, dtype=torch.float32, device=device)
        self.codes_out, self.scales_out = bc.alloc_codes(n, self.p2, device)
        self.side = torch.cuda.Stream(device=device)   # the second stream of decode()
        B1, B2 = self.p1[0].block, self.p2.block
        U = max(B1, B2)                          # chunks are whole blocks of both stages
        units = (n + U - 1) // U
        cu = (units + W - 1) // W
        self.chunks = []
        for c in range(W):
            u0, u1 = c * cu, min((c + 1) * cu, units)
            if u0 >= u1:
                break
            self.chunks.append((u0 * U, min(u1 * U, n)))

    def encode(self, stream=None):
        for w in range(self.W):
            self.encode_rank(w, stream)

    def encode_rank(self, w, stream=None):
        self.bc.quantize_pack(self.x[w], self.p1[w], self.err[w], self.codes[w], self.scales[w],
                              stream=stream)

    def decode(self, stream=None):
        """The W chunk decoders, alternately on the caller's stream and a second
        one (joined back before return).  They read the encoders' outputs and
        write disjoint chunks, so their order does not matter; on two streams one
        decoder's last wave overlaps the next one's first (8 x 1.625e8 outputs:
        2.55 -> 2.46 ms for the eight, the same bits)."""
        torch = self.torch
        main = stream or torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        self.side.wait_event(fork)
        for c in range(len(self.chunks)):
            self.decode_chunk(c, main if c % 2 == 0 else self.side)
        join = torch.cuda.Event()
        join.record(self.side)
        main.wait_event(join)

    def decode_chunk(self, c, stream=None):
        """Chunk c's decoder: the W ranks' codes of chunk c (what the all-to-all
        delivers to rank c), summed, requantised into chunk c of the output."""
        lo, hi = self.chunks[c]
        b1, B1 = self.p1[0].bits, self.p1[0].block
        b2, B2 = self.p2.bits, self.p2.block
        hi1 = (hi + B1 - 1) // B1 * B1
        hi2 = (hi + B2 - 1) // B2 * B2
        cin = [x[lo * b1 // 8: hi1 * b1 // 8] for x in self.codes]
        sin = [x[lo // B1: hi1 // B1] for x in self.scales]
        self.bc.unpack_dequant_reduce_requant(
            cin, sin, hi - lo, self.p1[0], sum_out=None, err2=self.err2[lo:hi],
            p_out=self.p2.shifted(lo), codes_out=self.codes_out[lo * b2 // 8: hi2 * b2 // 8],
            scales_out=self.scales_out[lo // B2: hi2 // B2], stream=stream)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import _build, synth

    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    n, W = args.n, W_RANKS

    # CPU baseline first (the oracle is single threaded, rank 0, N=1 only)
    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(torch, synth, args.cpu_sample)
        cpu_all = cpu_all_cores_sample(args.cpu_sample)

    ar = AllReduceW8(torch, bc, synth, n, W, dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        ar.encode()
        ar.decode()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for k in range(K):
        ev[k][0].record(stream)
        ar.encode()
        ev[k][1].record(stream)
        ar.decode()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    enc_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    step_ms = total_ms / K

    # end to end: pinned host gradients -> device, the step, requantised result -> host
    e2e = run_e2e(torch, bc, ar, args, dev) if not args.no_e2e else None
    n_chunks = len(ar.chunks)
    if world > 1:
        t = torch.tensor([e2e["step_ms"] if e2e else 0.0], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if e2e:
            e2e["step_ms"] = float(t.item())

    legs = None
    if rank == 0 and world == 1 and not args.no_legs:
        del ar
        torch.cuda.empty_cache()
        legs = target_legs(torch, bc, synth, args.leg_steps)
    if rank != 0:
        return
    elems = W * n * world
    value = elems * 4 / (step_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak_gbs()
    enc_launch_s = enc_ms / W * 1e-3
    dec_launch_s = dec_ms / n_chunks * 1e-3
    enc_bytes = n * ENC_BYTES_PER_ELEM
    dec_bytes = (n / n_chunks) * DEC_BYTES_PER_ELEM
    enc_gbs = enc_bytes / enc_launch_s / 1e9
    dec_gbs = dec_bytes / dec_launch_s / 1e9
    src = kernel_src_hash()
    tsrc = kernel_src_hash(TRAFFIC_SOURCES)
    tr = NCU_TRAFFIC.get("encode")
    traffic = round(tr["bytes_per_elem"] * n) if tr and tr["src"] == tsrc else None
    trd = NCU_TRAFFIC.get("decode")
    dec_traffic = round(trd["bytes_per_elem"] * n / n_chunks) if trd and trd["src"] == tsrc else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "ranks_simulated": W, "elements_per_rank": n,
                   "input_dtype": "bf16", "bits": BITS, "block": BLOCK, "rounding": "rtn",
                   "error_feedback": "stage1+stage2", "chunks": n_chunks,
                   "l2": "inputs larger than L2 (%.1f GB of gradients per step)" % (W * n * 2 / 1e9),
                   "input_gbs_bf16": round(W * n * 2 * world / (step_ms * 1e-3) / 1e9, 2),
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "roofline": {"bound": "hbm", "kernel": "encode16_kernel<bf16,4,ef,rtn>",
                     "achieved": round(enc_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(enc_gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic, "bytes_per_launch": enc_bytes,
                     "launch_ms": round(enc_launch_s * 1e3, 4)},
        "kernels": {
            "encode": {"gbs": round(enc_gbs, 1), "frac": round(enc_gbs / peak, 4),
                       "launch_ms": round(enc_launch_s * 1e3, 4), "bytes_per_elem": ENC_BYTES_PER_ELEM},
            "decode_w8": {"gbs": round(dec_gbs, 1), "frac": round(dec_gbs / peak, 4),
                          "launch_ms": round(dec_launch_s * 1e3, 4), "bytes_per_elem": DEC_BYTES_PER_ELEM,
                          "traffic": dec_traffic, "bytes_per_launch": dec_bytes},
        },
        "gpu_launches": K * (W + n_chunks),
        "clocks": clk,
        "kernel_src": src,
        "traffic_src": tsrc,
    }
    if legs:
        line["kernels"].update(legs)
    if e2e:
        line["e2e"] = {"value": round(elems * 4 / (e2e["step_ms"] * 1e-3) / 1e9, 2), "unit": UNIT,
                       "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "ms_per_step": round(e2e["step_ms"], 3)}
    if cpu:
        line["cpu_baseline"] = cpu
        line["cpu_baseline_all_cores"] = cpu_all
    print(json.dumps(line), flush=True)


def sharded_rank(torch, bc, synth, sharded, n, rank, world, device, bucket_bytes, codec=None, exchange=None,
                 grad=None):
    """One rank of the real multi-GPU all-reduce of the headline workload: this
    rank's 1.3e9-element bf16 gradient (N(0, 1e-3^2), seed 1000 + rank), 4-bit
    block-128 round-to-nearest encoder with error feedback, stage-2
    requantisation with error feedback, buckets of bucket_bytes."""
    if grad is None:
        grad = synth.gradients("normal", n, 1000 + rank, dtype=torch.bfloat16, device=device, sigma=1e-3)
    ar = sharded.LowBitAllReduce(n, torch.bfloat16, bc.QParams(BITS, BLOCK, bc.RTN, seed=1000 + rank),
                                 bc.QParams(BITS, BLOCK, bc.RTN, philox_stream=1), device=device,
                                 bucket_bytes=bucket_bytes, codec=codec, exchange=exchange)
    return ar, grad


def run_sharded(args, rank, world, local_rank):
    """N > 1: every GPU is one rank of the low-bit all-reduce (W = N): encode
    its own gradient, all-to-all of the chunks over NCCL, decode-reduce-requant
    of its own chunk, all-gather of the requantised chunks.  value = all ranks'
    gradient elements (counted as fp32 bytes) / the slowest rank's step time.
    By default the gradient is one bucket, as in the single-GPU workload (one
    encoder launch per rank, W chunks); --bucket-mb splits it into fusion
    buckets whose exchange overlaps the next bucket's encoder (each bucket
    costs a few Python-issued calls, so small buckets make the step host-bound)."""
    import torch
    import torch.distributed as dist

    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import _build, sharded, synth

    if rank == 0:
        _build.build()
    dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    n = args.n
    ar, grad = sharded_rank(torch, bc, synth, sharded, n, rank, world, dev, args.bucket_mb << 20)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        ar(grad)
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    for k in range(K):
        ev[k][0].record(stream)
        state = ar.send(grad)
        ev[k][1].record(stream)            # every bucket's encoder is queued before this
        ar.finish(ar.reduce(state))
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    t = torch.tensor([ev[0][0].elapsed_time(ev[K - 1][2]),
                      sum(e[0].elapsed_time(e[1]) for e in ev) / K], device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    step_ms, enc_ms = float(t[0]) / K, float(t[1])

    # end to end: pinned host gradient in, gathered requantised codes + scales out, every step
    e2e = None
    if not args.no_e2e:
        host_g = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
        host_g.copy_(grad)
        out_c = torch.empty(bc.packed_bytes(n, BITS, BLOCK), dtype=torch.uint8, device=dev)
        out_s = torch.empty(bc.num_blocks(n, BLOCK), dtype=torch.int16, device=dev)
        host_c = torch.empty(out_c.numel(), dtype=torch.uint8, pin_memory=True)
        host_s = torch.empty(out_s.numel(), dtype=torch.int16, pin_memory=True)
        steps = max(1, min(K, args.e2e_steps))
        dist.barrier()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            grad.copy_(host_g, non_blocking=True)
            ar(grad, out_codes=out_c, out_scales=out_s)
            host_c.copy_(out_c, non_blocking=True)
            host_s.copy_(out_s, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        te = torch.tensor([a.elapsed_time(b) / steps], device=dev)
        dist.all_reduce(te, op=dist.ReduceOp.MAX)
        e2e = {"step_ms": float(te), "h2d": n * 2, "d2h": host_c.numel() + host_s.numel() * 2}
    if rank != 0:
        return
    peak, peak_kind = measured_peak_gbs()
    enc_gbs = n * ENC_BYTES_PER_ELEM / (enc_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(world * n * 4 / (step_ms * 1e-3) / 1e9, 2), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "ranks": world, "elements_per_rank": n, "input_dtype": "bf16",
                   "bits": BITS, "block": BLOCK, "rounding": "rtn", "error_feedback": "stage1+stage2",
                   "buckets": len(ar.buckets), "bucket_bytes": args.bucket_mb << 20,
                   "l2": "inputs larger than L2 (%.1f GB of gradient per rank)" % (n * 2 / 1e9),
                   "parallelism": f"sharded low-bit all-reduce over NCCL, {world} ranks (all-to-all + all-gather)"},
        "roofline": {"bound": "hbm", "kernel": ("encode16_kernel<bf16,4,ef,rtn>" if args.bucket_mb == 0 else
                                "encode_kernel or encode16_kernel<bf16,4,ef,rtn> by bucket size (all buckets of one step)"),
                     "achieved": round(enc_gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(enc_gbs / peak, 4),
                     "peak_kind": peak_kind, "traffic": None, "bytes_per_launch": n * ENC_BYTES_PER_ELEM,
                     "launch_ms": round(enc_ms, 4)},
        "gpu_launches": K * 2 * len(ar.buckets),
        "clocks": clk, "kernel_src": kernel_src_hash(),
    }
    if e2e:
        line["e2e"] = {"value": round(world * n * 4 / (e2e["step_ms"] * 1e-3) / 1e9, 2), "unit": UNIT,
                       "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "ms_per_step": round(e2e["step_ms"], 3)}
    print(json.dumps(line), flush=True)


def target_legs(torch, bc, synth, K):
    """Short timed legs for the other target points of the method's
    measurement plan, each on its own full-size workload (inputs larger than
    L2): device time per launch (CUDA events on the launching stream, launch
    queued before the start event; see _timed), algorithmic bytes per launch,
    GB/s and the fraction of the measured HBM copy bandwidth."""
    peak, _ = measured_peak_gbs()
    legs = {}

    def leg(name, fn, nbytes, steps, note):
        for _ in range(3):
            fn()
        ms = _timed(torch, fn, steps)
        legs[name] = {"gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4),
                      "launch_ms": round(ms, 4), "bytes_per_launch": nbytes, "workload": note}

    wl = synth.WORKLOADS["sweep_laplace_256m"]
    x = synth.gradients(wl.kind, wl.n, wl.seed, **wl.params)
    deq = torch.empty(wl.n, device="cuda")
    for rounding, tag in ((bc.RTN, "rtn"), (bc.SR, "sr")):
        p = bc.QParams(4, 128, rounding, seed=wl.sr_seed)
        codes, scales = bc.alloc_codes(wl.n, p)
        note = f"268,435,456 fp32 Laplace(0, 1e-3), 4-bit, block 128, {tag}, no error feedback"
        leg(f"sweep_b4_B128_{tag}_encode", lambda: bc.quantize_pack(x, p, None, codes, scales),
            wl.n * (4 + 0.5 + 2 / 128), K, note)
        if rounding == bc.RTN:
            leg("sweep_b4_B128_decode_w1",
                lambda: bc.unpack_dequant_reduce_requant([codes], [scales], wl.n, p, sum_out=deq),
                wl.n * (0.5 + 2 / 128 + 4), K, note + "; W=1 decoder to fp32")
        del codes, scales
    del x, deq

    wl = synth.WORKLOADS["allgather_decode_gpt1p3b"]
    x = synth.gradients(wl.kind, wl.n, wl.seed, dtype=torch.bfloat16, **wl.params)
    p = bc.QParams(wl.bits, wl.block)
    codes, scales = bc.quantize_pack(x, p)
    del x
    out = torch.empty(wl.n, dtype=torch.bfloat16, device="cuda")
    leg("allgather_decode_b4_B128_bf16", lambda: bc.unpack_dequant(codes, scales, wl.n, p, 1.0 / wl.ranks, out),
        wl.n * (0.5 + 2 / 128 + 2), K, "1.3e9 4-bit block-128 codes to the bf16 mean of 8 ranks")
    del codes, scales, out

    wl = synth.WORKLOADS["gpt6p7b_2bit_buckets"]
    x = synth.gradients(wl.kind, wl.n, wl.seed, dtype=torch.bfloat16, **wl.params)
    err = torch.zeros(wl.n, device="cuda")
    p = bc.QParams(wl.bits, wl.block, wl.rounding, seed=wl.sr_seed)
    codes, scales = bc.alloc_codes(wl.n, p)
    sched = bc.Scheduler(2, wl.bucket_bytes)
    leg("gpt6p7b_2bit_buckets_encode", lambda: sched.quantize_pack(x, p, err, codes, scales),
        wl.n * (2 + 8 + wl.bits / 8 + 2 / wl.block), max(3, K // 4),
        "6.7e9 bf16 with 0.1% outliers, 2-bit block 64, stochastic rounding, error feedback, "
        "512 buckets of 25 MiB on two streams (one step = all buckets)")
    sched.close()
    del x, err, codes, scales
    torch.cuda.empty_cache()
    return legs


def run_e2e(torch, bc, ar, args, dev):
    """Host -> device copies of the 8 ranks' gradients (pinned), the step, and
    the requantised codes + scales back to the host, all inside the timed
    region.  Copies run on their own streams and wait only for what they
    overwrite: rank w's gradient copy for the previous step's encoder w, chunk
    c's decoder for the previous step's copy-out of chunk c.  So the next
    step's copies in stream behind this step's kernels, as in a training loop
    that overlaps communication with compute, while every step still moves
    its own bytes across the host link."""
    W, n = ar.W, ar.n
    host_x = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(W)]
    for w in range(W):
        host_x[w].copy_(ar.x[w])
    host_codes = torch.empty(ar.codes_out.numel(), dtype=torch.uint8, pin_memory=True)
    host_scales = torch.empty(ar.scales_out.numel(), dtype=torch.int16, pin_memory=True)
    compute = torch.cuda.current_stream()
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_x)
    d2h = host_codes.numel() + host_scales.numel() * 2
    b2, B2 = ar.p2.bits, ar.p2.block
    enc_done = [None] * W                      # previous step's encoder w has read x[w]
    out_done = [None] * len(ar.chunks)         # previous step's chunk c is back on the host

    def step():
        arrived = []
        for w in range(W):
            with torch.cuda.stream(h2d_stream):
                if enc_done[w] is not None:
                    h2d_stream.wait_event(enc_done[w])
                ar.x[w].copy_(host_x[w], non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d_stream)
            arrived.append(e)
        for w in range(W):
            compute.wait_event(arrived[w])
            ar.encode_rank(w)
            e = torch.cuda.Event()
            e.record(compute)
            enc_done[w] = e
        for c, (lo, hi) in enumerate(ar.chunks):
            if out_done[c] is not None:
                compute.wait_event(out_done[c])
            ar.decode_chunk(c)
            ev = torch.cuda.Event()
            ev.record(compute)
            d2h_stream.wait_event(ev)
            hi2 = (hi + B2 - 1) // B2 * B2
            with torch.cuda.stream(d2h_stream):
                host_codes[lo * b2 // 8: hi2 * b2 // 8].copy_(ar.codes_out[lo * b2 // 8: hi2 * b2 // 8],
                                                              non_blocking=True)
                host_scales[lo // B2: hi2 // B2].copy_(ar.scales_out[lo // B2: hi2 // B2], non_blocking=True)
                e = torch.cuda.Event()
                e.record(d2h_stream)
            out_done[c] = e

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(compute)
    h2d_stream.wait_event(t0)                  # no copy of the timed steps starts before t0
    d2h_stream.wait_event(t0)
    for _ in range(steps):
        step()
    compute.wait_stream(d2h_stream)            # the last step's results are on the host
    compute.wait_stream(h2d_stream)
    t1.record(compute)
    torch.cuda.synchronize()
    # the copies back must hold the last step's result (no copy raced its decoder)
    if not (torch.equal(host_codes, ar.codes_out.cpu()) and torch.equal(host_scales, ar.scales_out.cpu())):
        raise RuntimeError("e2e: host copy of the result differs from the device result")
    return {"step_ms": t0.elapsed_time(t1) / steps, "h2d": h2d, "d2h": d2h}


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_sample_step(O, xs_bits, S):
    """One sampled step on the host: 8 rank encoders over S elements each,
    then the W=8 decoder over the same S elements (one chunk)."""
    import numpy as np
    p1 = O.params(BITS, BLOCK)
    enc = []
    t0 = time.perf_counter()
    for w in range(W_RANKS):
        e = np.zeros(S, np.float32)
        enc.append(O.quantize_pack(xs_bits[w], p1, e))
    e2 = np.zeros(S, np.float32)
    O.unpack_dequant_reduce_requant([c for c, _ in enc], [s for _, s in enc], S, p1, False, e2,
                                    O.params(BITS, BLOCK, philox_stream=1))
    return time.perf_counter() - t0


def _sample_inputs(S):
    import numpy as np

    from bit_gradient_communication_gb300 import synth
    xs = []
    for w in range(W_RANKS):
        x = synth.np_gradients("normal", S, 1000 + w, sigma=1e-3)
        # bf16 bits by round-to-nearest-even of the fp32 draw (host-side input recipe)
        u = x.view(np.uint32).astype(np.uint64)
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        xs.append(u.astype(np.uint16))
    return xs


def _oracle_sample_threads(O, xs_bits, S, threads):
    """The same sampled step split into `threads` block-aligned slices, each an
    independent problem (zero error buffers, its own slice of every rank), run
    on host threads; the oracle's C functions release the GIL."""
    import concurrent.futures as cf
    unit = BLOCK * 64
    per = -(-S // (threads * unit)) * unit
    bounds = [(lo, min(lo + per, S)) for lo in range(0, S, per)]

    def one(b):
        lo, hi = b
        _oracle_sample_step(O, [x[lo:hi] for x in xs_bits], hi - lo)

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, bounds))
    return time.perf_counter() - t0, len(bounds)


def _host_cpu():
    """The host's CPU model and logical CPU count (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"model": model, "logical_cpus": os.cpu_count()}


def cpu_baseline_sample(torch, synth, S):
    import oracle as O
    O.build()
    xs = _sample_inputs(S)
    t = _oracle_sample_step(O, xs, S)
    return {"value": round(W_RANKS * S * 4 / t / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"8 rank encoders over {S} bf16 elements each + the W=8 decoder over "
                      f"{S} elements (one chunk), single-threaded C++ oracle, {t:.2f} s",
            "host": _host_cpu()}


def cpu_all_cores_sample(S):
    """A second CPU figure: the unchanged oracle on every host core at once."""
    import oracle as O
    xs = _sample_inputs(S)
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    t, used = _oracle_sample_threads(O, xs, S, threads)
    return {"value": round(W_RANKS * S * 4 / t / 1e9, 4), "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"the cpu_baseline sample split into {used} block-aligned slices on {used} host "
                      f"threads, {t:.2f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle as O
    O.build()
    S = args.ref_sample
    xs = _sample_inputs(S)
    for _ in range(args.warmup):
        _oracle_sample_step(O, xs, S)
    ts = [_oracle_sample_step(O, xs, S) for _ in range(args.steps)]
    t = sum(ts) / len(ts)
    value = W_RANKS * S * 4 / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "ranks_simulated": W_RANKS, "elements_per_rank": args.n,
                   "input_dtype": "bf16", "bits": BITS, "block": BLOCK, "rounding": "rtn",
                   "error_feedback": "stage1+stage2",
                   "sample_elements_per_rank": S},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"per step: 8 rank encoders over {S} bf16 elements + the W=8 "
                                   f"decoder over {S} elements, single-threaded C++ oracle"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# other workloads (python bench.py --workload NAME): one JSON line each
# ---------------------------------------------------------------------------

def _timed(torch, fn, K, flush=None):
    """Average device time of fn() over K calls (events on the current stream);
    flush() runs between calls, outside the timed intervals."""
    st = torch.cuda.current_stream()
    if flush is not None:
        # one untimed round first: the flush's own kernels load and allocate on
        # first use, and a host stall there would drain the queue into the
        # first timed interval
        flush()
        fn()
        torch.cuda.synchronize()
    total = 0.0
    for _ in range(K):
        if flush is not None:
            flush()
        elif hasattr(torch.cuda, "_sleep"):
            # keep the device busy (~50 us) while the host marshals the call's
            # arguments, so that the start event fires only when the launch is
            # already queued (the flush does the same where there is one)
            torch.cuda._sleep(100_000)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        b.synchronize()
        total += a.elapsed_time(b)
    return total / K


def run_workload(args):
    import torch

    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import _build, synth
    _build.build()
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS[args.workload]
    if args.wl_n:
        # a smaller case of the same kernels, for profilers
        wl = dataclasses.replace(wl, n=args.wl_n)
    peak, peak_kind = measured_peak_gbs()
    l2_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # > 129 MB L2
    l2_clean = torch.ones(256 << 20, dtype=torch.uint8, device="cuda")

    def flush():
        # write a buffer larger than L2, then read another one: the inputs are
        # evicted and the lines left behind are clean, so the timed kernel does
        # not also pay for writing back the flush's own dirty lines
        l2_buf.fill_(1)
        l2_clean.max()

    K, warm = args.steps, args.warmup
    lines = []
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    if args.workload == "sweep_laplace_256m":
        x = synth.gradients(wl.kind, wl.n, wl.seed, **wl.params)
        deq = torch.empty(wl.n, device="cuda")
        only = None
        if args.sweep_filter:
            fb, fB, fr = args.sweep_filter.split(",")
            only = (int(fb), int(fB), bc.SR if fr == "sr" else bc.RTN)
        for bits in (1, 2, 4, 8, 12, 16):
            for block in (32, 64, 128, 256, 1024, 4096):
                for rounding in (bc.RTN, bc.SR):
                    if only and (bits, block, rounding) != only:
                        continue
                    p = bc.QParams(bits, block, rounding, seed=wl.sr_seed)
                    codes, scales = bc.alloc_codes(wl.n, p)
                    enc = lambda: bc.quantize_pack(x, p, None, codes, scales)
                    dec = lambda: bc.unpack_dequant_reduce_requant([codes], [scales], wl.n, p, sum_out=deq)
                    for _ in range(warm):
                        enc()
                        dec()
                    te = _timed(torch, enc, K)
                    td = _timed(torch, dec, K)
                    cb = bits / 8 + 2 / block
                    eb, db = wl.n * (4 + cb), wl.n * (cb + 4)
                    lines.append({"bits": bits, "block": block, "rounding": "sr" if rounding else "rtn",
                                  "encode_gbs": round(eb / te / 1e6, 1), "encode_frac": round(eb / te / 1e6 / peak, 4),
                                  "decode_gbs": round(db / td / 1e6, 1), "decode_frac": round(db / td / 1e6 / peak, 4),
                                  "encode_input_gbs": round(wl.n * 4 / te / 1e6, 1)})
                    del codes, scales
        best = max(lines, key=lambda r: r["encode_input_gbs"])
        head = next((r for r in lines if r["bits"] == 4 and r["block"] == 128 and r["rounding"] == "rtn"),
                    lines[0])
        out = {"metric": METRIC, "value": head["encode_input_gbs"], "unit": UNIT, "n_gpus": 1, "steps": K,
               "warmup": warm, "higher_is_better": True, "dtype": "f32", "data": "synthetic",
               "config": {"workload": wl.name, "n": wl.n, "input_dtype": "f32",
                          "l2": "inputs larger than L2 (1.07 GB)", "value_is": "encoder, 4-bit, block 128, RTN"},
               "roofline": {"bound": "hbm", "kernel": "encode16_kernel<f32,4,noef,rtn>",
                            "achieved": head["encode_gbs"], "peak": peak, "unit": "GB/s",
                            "frac": head["encode_frac"], "peak_kind": peak_kind},
               "best_encode_input_gbs": best["encode_input_gbs"], "sweep": lines}
        print(json.dumps(out), flush=True)
        return
    if args.workload == "roundtrip_1m":
        x = synth.gradients(wl.kind, wl.n, wl.seed, **wl.params)
        p = bc.QParams(wl.bits, wl.block)
        codes, scales = bc.alloc_codes(wl.n, p)
        deq = torch.empty(wl.n, device="cuda")
        step = lambda: bc.roundtrip(x, p, None, codes, scales, deq)
        for _ in range(warm):
            step()
        t = _timed(torch, step, K, flush)
        # one pass: read x, write codes + scales and the dequantised fp32 result
        algo = wl.n * (4 + wl.bits / 8 + 2 / wl.block + 4)
        extra = {"l2": "flushed between timed iterations (256 MB write, then 256 MB read)",
                 "passes": "one (encoder with fused dequantisation)"}
    elif args.workload == "bucket25mb_f32":
        # one 25 MiB fusion bucket per call: the encoder entry point directly
        xs = [synth.gradients(wl.kind, wl.n, t, **wl.params) for t in range(10)]
        per_bits = {}
        for bits in (1, 2, 4, 8):
            err = torch.zeros(wl.n, device="cuda")
            codes, scales = bc.alloc_codes(wl.n, bc.QParams(bits, wl.block))
            it = [0]

            def step():
                t = it[0] % 10
                bc.quantize_pack(xs[t], bc.QParams(bits, wl.block, wl.rounding, seed=wl.sr_seed,
                                                   index_offset=t * wl.n), err, codes, scales)
                it[0] += 1
            for _ in range(warm):
                step()
            tb = _timed(torch, step, K, flush)
            tw = _timed(torch, step, K)          # back to back: part of the 82 MB stays in L2
            algo_b = wl.n * (4 + 4 + 4 + bits / 8 + 2 / wl.block)
            per_bits[bits] = {"ms": round(tb, 4), "input_gbs": round(wl.n * 4 / tb / 1e6, 1),
                              "gbs": round(algo_b / tb / 1e6, 1), "frac": round(algo_b / tb / 1e6 / peak, 4),
                              "warm_l2_ms": round(tw, 4), "warm_l2_gbs": round(algo_b / tw / 1e6, 1)}
        t = per_bits[4]["ms"]
        algo = wl.n * (12 + 0.5 + 2 / wl.block)
        extra = {"l2": "flushed between timed iterations (256 MB write, then 256 MB read); warm_l2_* without it",
                 "per_bits": per_bits, "value_is": "4-bit, L2 flushed"}
    elif args.workload in ("allgather_decode_gpt1p3b", "allgather_decode_hs_gpt1p3b"):
        # every rank's decode of the all-gathered 4-bit codes into its bf16 mean
        # gradient (with the inverse rotation for the Hadamard-smoothed codes)
        x = synth.gradients(wl.kind, wl.n, wl.seed, dtype=dt, **wl.params)
        p = bc.QParams(wl.bits, wl.block, hadamard=wl.hadamard)
        codes, scales = bc.quantize_pack(x, p)
        out = torch.empty(wl.n, dtype=torch.bfloat16, device="cuda")
        step = lambda: bc.unpack_dequant(codes, scales, wl.n, p, 1.0 / wl.ranks, out)
        for _ in range(warm):
            step()
        t = _timed(torch, step, K)
        algo = wl.n * (wl.bits / 8 + 2 / wl.block + 2)
        extra = {"l2": "inputs larger than L2 (3.3 GB per step)", "output": "bf16", "mul": "1/8",
                 "hadamard": wl.hadamard}
    elif args.workload == "tlq_hs_w8_gpt1p3b":
        # two-level quantisation with Hadamard smoothing: stage 1 8-bit groups of
        # 512, stage 2 4-bit groups of 128, both rotated by H = 128
        p1 = bc.QParams(8, 512, bc.RTN, hadamard=128)
        p2 = bc.QParams(4, 128, bc.RTN, philox_stream=1, hadamard=128)
        ar = AllReduceW8(torch, bc, synth, wl.n, wl.ranks, torch.device("cuda"), p1, p2)
        for _ in range(warm):
            ar.encode()
            ar.decode()
        te = _timed(torch, ar.encode, K)
        td = _timed(torch, ar.decode, K)
        t = te + td
        enc_b = wl.n * (2 + 8 + 1 + 2 / 512)
        dec_b = wl.n / len(ar.chunks) * (8 * (1 + 2 / 512) + 8 + 0.5 + 2 / 128)
        enc_gbs = enc_b / (te / wl.ranks) / 1e6
        dec_gbs = dec_b / (td / len(ar.chunks)) / 1e6
        algo = wl.n * wl.ranks * (2 + 8 + 1 + 2 / 512) + wl.n * (8 * (1 + 2 / 512) + 8 + 0.5 + 2 / 128)
        extra = {"l2": "inputs larger than L2", "stage1": "8-bit B512 H128 EF", "stage2": "4-bit B128 H128 EF2",
                 "encode_gbs": round(enc_gbs, 1), "encode_frac": round(enc_gbs / peak, 4),
                 "decode_gbs": round(dec_gbs, 1), "decode_frac": round(dec_gbs / peak, 4)}
        wl_elems = wl.n * wl.ranks
    elif args.workload == "qwd_gpt6p7b_w8":
        # sharded weight all-gather of a 6.7B model over 8 ranks: this rank
        # encodes its shard's weight difference (sender), then applies all 8
        # gathered shards to its reference copy and writes bf16 weights
        # shards padded to whole groups, so every shard starts on a group boundary
        shard = (wl.n // wl.ranks + wl.block - 1) // wl.block * wl.block
        n_all = shard * wl.ranks
        p = bc.QParams(wl.bits, wl.block, bc.RTN)
        w = synth.gradients(wl.kind, shard, wl.seed, dtype=dt, **wl.params)
        ref_shard = w.float() - 1e-3
        ref_all = torch.zeros(n_all, device="cuda")
        w_all = torch.empty(n_all, dtype=torch.bfloat16, device="cuda")
        codes_all, scales_all = bc.alloc_codes(n_all, p)
        nb_shard = shard // wl.block
        cs, ss = codes_all[: shard * wl.bits // 8], scales_all[:nb_shard]
        def enc():
            bc.qwd_encode(w, ref_shard, p, cs, ss)
        def app():
            bc.qwd_apply(codes_all, scales_all, n_all, p, ref_all, w_all)
        for r in range(wl.ranks):       # every shard's codes, as if gathered from its owner
            bc.qwd_encode(w, ref_shard.clone(), p, codes_all[r * shard * wl.bits // 8:(r + 1) * shard * wl.bits // 8],
                          scales_all[r * nb_shard:(r + 1) * nb_shard])
        for _ in range(warm):
            enc()
            app()
        te = _timed(torch, enc, K)
        ta = _timed(torch, app, K)
        t = te + ta
        enc_b = shard * (2 + 4 + 4 + wl.bits / 8 + 2 / wl.block)
        app_b = n_all * (wl.bits / 8 + 2 / wl.block + 4 + 4 + 2)
        algo = enc_b + app_b
        extra = {"l2": "inputs larger than L2", "shards": wl.ranks, "shard_elems": shard, "weights_out": "bf16",
                 "encode_gbs": round(enc_b / te / 1e6, 1), "encode_frac": round(enc_b / te / 1e6 / peak, 4),
                 "apply_gbs": round(app_b / ta / 1e6, 1), "apply_frac": round(app_b / ta / 1e6 / peak, 4)}
    elif args.workload == "gpt6p7b_2bit_buckets":
        sched = bc.Scheduler(2, wl.bucket_bytes)
        x = synth.gradients(wl.kind, wl.n, wl.seed, dtype=dt, **wl.params)
        err = torch.zeros(wl.n, device="cuda")
        p = bc.QParams(wl.bits, wl.block, wl.rounding, seed=wl.sr_seed)
        codes, scales = bc.alloc_codes(wl.n, p)
        step = lambda: sched.quantize_pack(x, p, err, codes, scales)
        for _ in range(warm):
            step()
        t = _timed(torch, step, K)
        algo = wl.n * (2 + 8 + wl.bits / 8 + 2 / wl.block)
        extra = {"l2": "inputs larger than L2 (67 GB per step)" if not args.wl_n else "one pass per step",
                 "buckets": len(bc.plan_buckets(wl.n, 2, wl.block, wl.bucket_bytes)) - 1, "streams": 2}
    elif args.workload == "local_sum_w8_gpt1p3b":
        # pipeline-A's full-precision local reduce on the node leader: the fp32
        # sum of the 8 local ranks' bf16 gradients in rank order
        xs = [synth.gradients(wl.kind, wl.n, wl.seed + w, dtype=dt, **wl.params) for w in range(wl.ranks)]
        out_sum = torch.empty(wl.n, device="cuda")
        step = lambda: bc.sum_ranks(xs, out=out_sum)
        for _ in range(warm):
            step()
        t = _timed(torch, step, K)
        algo = wl.n * (wl.ranks * 2 + 4)
        extra = {"l2": "inputs larger than L2 (26 GB per step)", "ranks": wl.ranks, "output": "fp32"}
        wl_elems = wl.n * wl.ranks
    elif args.workload == "local_decode_w8_gpt1p3b":
        # pipeline-A's local stage with local quantisation, on the node leader:
        # the 8 local ranks' 4-bit codes decoded into their rank-ordered fp32 sum
        p = bc.QParams(wl.bits, wl.block)
        cs, ss = [], []
        for w in range(wl.ranks):
            x = synth.gradients(wl.kind, wl.n, wl.seed + w, dtype=dt, **wl.params)
            c, s_ = bc.quantize_pack(x, p)
            cs.append(c)
            ss.append(s_)
            del x
        out_sum = torch.empty(wl.n, device="cuda")
        step = lambda: bc.unpack_dequant_reduce_requant(cs, ss, wl.n, p, sum_out=out_sum)
        for _ in range(warm):
            step()
        t = _timed(torch, step, K)
        algo = wl.n * (wl.ranks * (wl.bits / 8 + 2 / wl.block) + 4)
        extra = {"l2": "inputs larger than L2 (5.3 GB of codes per call)", "ranks": wl.ranks, "output": "fp32 sum"}
        wl_elems = wl.n * wl.ranks
    else:
        raise SystemExit(f"workload {args.workload}: use the default run")
    gbs = algo / t / 1e6
    elems = locals().get("wl_elems", wl.n)
    out = {"metric": METRIC, "value": round(elems * 4 / t / 1e6, 2), "unit": UNIT, "n_gpus": 1, "steps": K,
           "warmup": warm, "ms_per_step": round(t, 4), "higher_is_better": True, "dtype": "f32",
           "data": "synthetic", "config": {"workload": wl.name, "n": wl.n, "input_dtype": wl.dtype,
                                           "bits": wl.bits, "block": wl.block, **extra},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "peak_kind": peak_kind}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--n", type=int, default=N_PER_RANK, help="elements per simulated rank")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-sample", type=int, default=1 << 23)
    ap.add_argument("--ref-sample", type=int, default=1 << 21)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-legs", action="store_true", help="skip the target-point legs after the headline")
    ap.add_argument("--leg-steps", type=int, default=20, help="timed launches per target-point leg")
    ap.add_argument("--sweep-filter", default=None,
                    help="bits,block,rtn|sr: run one configuration of sweep_laplace_256m")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="another workload recipe from synth.WORKLOADS (one JSON line of its own)")
    ap.add_argument("--replicas", action="store_true",
                    help="N > 1: run N independent copies of the single-GPU simulation instead of the sharded all-reduce")
    ap.add_argument("--bucket-mb", type=int, default=0,
                    help="N > 1: fusion bucket size in MiB of bf16 gradient (0: one bucket per rank, the workload's "
                         "own structure: one encoder launch, W chunks)")
    ap.add_argument("--wl-n", type=int, default=0,
                    help="run --workload with this many elements instead (a small case for profilers)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload != WORKLOAD:
        run_workload(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        # NCCL's communicator lines (ranks, devices) on stdout, for checking the ranks
        os.environ.setdefault("NCCL_DEBUG", "INFO")
        os.environ.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if world > 1 and not args.replicas:
            run_sharded(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
