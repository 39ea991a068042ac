#!/usr/bin/env python3
"""Benchmark: 2-bit omni KV decode attention on one GB300 (or N replicas).

Workload (default): Qwen2.5-Omni-3B-shaped decode - 36 layers, 16 query / 2 kv
heads, head_dim 128, one session holding a 32,768-token cache built by
appending 1-s chunks of 640 video + 25 audio tokens (a 32-token text turn
every 30 chunks); 2-bit codes, key group 32. One step = one okvq_decode over
all layers (the split-K fused attention kernel + the merge / inverse-rotation
kernel). Two replicas of the cache alternate so consecutive steps never find
their 194 MB of codes in the 129 MB L2.

Prints one JSON line (rank 0). --impl reference times the CPU oracle instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_rht_gb300 import synth  # noqa: E402

METRIC = "2-bit KV decode attention: context tokens/s and HBM GB/s (% of GB300 peak)"
UNIT = "context tokens/s"


def decode_source_sha256():
    """Hash of the decode kernel's own sources (okvq_decode.cu and the two headers it
    includes; the merge kernel lives in okvq_combine.cu), compared with the one stored
    beside the ncu traffic figure: a changed kernel makes the stored figure stale."""
    import hashlib
    h = hashlib.sha256()
    for f in ("okvq_decode.cu", "okvq_internal.h", "okvq_device.h"):
        with open(os.path.join(ROOT, "bit_kv_cache_rht_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def algorithmic_bytes(w, lengths, key_codec="omni"):
    """Decode bytes per step: codes, statistics, norms, fp16 tail keys, modality ids, q and out.
    TurboQuant keys: codes and a 2-byte norm per token-head, no statistics, no tail."""
    sh = w.shape
    d, b, G = sh.head_dim, sh.bits, sh.group_size
    per_unit = 0
    for T in lengths:
        if key_codec == "turbo":
            per_unit_T = T * (2 * d * b // 8 + 2 + 2)
        else:
            per_unit_T = T * (2 * d * b // 8 + 2) + (T // G) * 4 * d + (T % G) * 2 * d
        per_unit += per_unit_T * sh.num_layers * sh.num_kv_heads
    mod = sum(lengths)
    q_bytes = 2 * len(lengths) * sh.num_layers * sh.num_q_heads * d     # fp16 queries in, and as many outputs
    rot = sh.num_layers * sh.num_kv_heads * sh.num_modalities * d * d * 4
    return per_unit + mod + q_bytes, q_bytes, rot     # split kernel bytes, merge kernel out bytes, R bytes


def rank_env():
    """(world size, rank, local rank) from the launcher's environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(vals, world, device):
    """Each rank's timings -> the maximum over the ranks (the job ends with its slowest
    replica); the identity with one rank. `device` carries the reduction (the GPU with
    NCCL, the CPU with gloo)."""
    if world <= 1:
        return [float(v) for v in vals]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tokens(world, steps, lengths):
    """Context tokens the whole job decodes: every replica decodes every session each step
    (weak scaling: the work per GPU is fixed)."""
    return world * steps * sum(lengths)


def make_workload(args):
    """The named synthetic workload at the requested code width and key group size."""
    return synth.WORKLOADS[args.workload](bits=getattr(args, "bits", 2), group_size=getattr(args, "group_size", 32))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """fp16 tensor peak (TFLOP/s): the measured bf16 cuBLAS burst figure (fp16 runs at
    the bf16 rate), else the profiling fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 cuBLAS burst; fp16 at the same rate)"
    return 1900.0, "fallback"


class ClockSampler:
    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + q, "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, gpu_index=0):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[0] == str(gpu_index):
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def device_session_kv(w, s, torch, device):
    """fp16 K, V [T][L][Hkv][d] of session s, drawn on the device with the synthetic
    recipe: the workload's per-channel scales and modality means per layer; z ~ N(0, 1);
    keys add a per-channel Gaussian random walk of step 0.02 per token (torch
    generators seeded by (workload seed, session, layer); the parity tests draw the
    same recipe with numpy)."""
    sh = w.shape
    mod = torch.from_numpy(w.sessions[s].modality()).to(device).long()
    T = len(mod)
    K = torch.empty((T, sh.num_layers, sh.num_kv_heads, sh.head_dim), dtype=torch.float16, device=device)
    V = torch.empty_like(K)
    for l in range(sh.num_layers):
        kscale, vscale, mu = w.layer_params(l)
        g = torch.Generator(device=device).manual_seed(((int(w.seed) * 1000003 + s) * 1009 + l) & 0x7FFFFFFF)
        shp = (T, sh.num_kv_heads, sh.head_dim)
        z = torch.randn(shp, device=device, generator=g)
        # the random walk along the token axis, scanned as the innermost dimension
        steps = torch.randn((sh.num_kv_heads * sh.head_dim, T), device=device, generator=g) * 0.02
        drift = torch.cumsum(steps, dim=1).t().reshape(shp)
        K[:, l] = (torch.from_numpy(kscale).to(device) * z + drift).half()
        z = torch.randn(shp, device=device, generator=g)
        V[:, l] = (torch.from_numpy(vscale).to(device) * z + torch.from_numpy(mu).to(device)[mod]).half()
    return K, V


def calibrate(w, torch, device):
    """Value rotations of the workload from its calibration slice, by the calibration
    kernel (one untimed call loads the module, the second is timed)."""
    from bit_kv_cache_rht_gb300.okvq import calibrate_rotations
    sh = w.shape
    Vc, modc = w.calibration_slice()
    Vcd, Mcd = torch.from_numpy(Vc).to(device), torch.from_numpy(modc).to(device)
    st = torch.cuda.current_stream()
    calibrate_rotations(Vcd, Mcd, sh.num_modalities)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(st)
    rot, _, sweeps = calibrate_rotations(Vcd, Mcd, sh.num_modalities, return_sweeps=True)
    c1.record(st)
    R = rot.cpu().numpy()
    sw = sweeps.cpu().numpy().astype(np.int64)
    if np.any(sw < 0):
        raise RuntimeError("calibration: Jacobi did not converge for %d units" % int((sw < 0).sum()))
    ms = c0.elapsed_time(c1)
    # shared-memory traffic of the rotating sweeps: per round, rows p, q (2 loads + 2 stores)
    # and columns p, q of A and V (4 + 4) for 64 pairs x 128 entries, 4 B each
    smem_bytes = float(np.maximum(sw - 1, 0).sum()) * 127 * 64 * 128 * 12 * 4
    smem_peak = 152 * 128 * 2.07e9 / 1e9          # GB/s: 32 banks x 4 B per clock per SM at 2.07 GHz
    calib = {"ms": ms, "units": int(sw.size), "tokens": int(Vc.shape[0]),
             "sweeps_mean": float(sw.mean()), "sweeps_max": int(sw.max()),
             "roofline": {"bound": "smem", "achieved": smem_bytes / (ms / 1e3) / 1e9, "peak": smem_peak,
                          "unit": "GB/s", "frac": smem_bytes / (ms / 1e3) / 1e9 / smem_peak,
                          "peak_kind": "nominal (152 SMs x 128 B/clk x 2.07 GHz)"}}
    del Vcd, Mcd, rot
    return R, calib


def build_cache(w, torch, device, replicas=2, key_codec="omni", keep_layer0=False):
    from bit_kv_cache_rht_gb300.okvq import Cache, OKVQ_KEYS_GROUP_RANGE, OKVQ_KEYS_TURBOQUANT
    sh = w.shape
    st = torch.cuda.current_stream()
    R, calib = calibrate(w, torch, device)
    caches = [Cache(len(w.sessions), sh.num_layers, sh.num_q_heads, sh.num_kv_heads, w.max_tokens, R,
                    head_dim=sh.head_dim, group_size=sh.group_size, bits=sh.bits, num_modalities=sh.num_modalities,
                    hadamard_seed=w.hadamard_seed,
                    key_codec=OKVQ_KEYS_TURBOQUANT if key_codec == "turbo" else OKVQ_KEYS_GROUP_RANGE)
              for _ in range(replicas)]
    for c in caches:
        c.rotations_used = R          # the value rotations the caches were created with
    append_ms = [[] for _ in range(replicas)]
    for s in range(len(w.sessions)):
        if not w.sessions[s].length:
            continue
        K, V = device_session_kv(w, s, torch, device)
        M = torch.from_numpy(w.sessions[s].modality()).to(device)
        if keep_layer0 and s == 0:     # the inputs of layer 0, for the CPU leg's state comparison
            caches[0].layer0_kv = (K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy())
        for rep, c in enumerate(caches):
            ev = []
            for a, b in w.sessions[s].chunk_bounds():
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                c.append(s, K[a:b], V[a:b], M[a:b])
                e1.record(st)
                ev.append((e0, e1, b - a))
            torch.cuda.synchronize()
            append_ms[rep] += [(e0.elapsed_time(e1), n) for e0, e1, n in ev]
        del K, V, M
    torch.cuda.synchronize()
    for c in caches:
        if c.check_errors() != 0:
            raise RuntimeError("device error word set after append")
    torch.cuda.empty_cache()
    return caches, append_ms, calib


def compaction_leg(c, w, torch, Q, out, peak, steps):
    """Retention-shaped eviction (sinks of 64 video / 8 audio tokens per 1-s chunk,
    text and the last 4 chunks kept) and the largest ordered-suffix compaction on
    one cache replica, then decode steps over the compacted cache (an L2-sized
    buffer is rewritten between steps)."""
    sh = w.shape
    T = w.sessions[0].length
    ranges = synth.retention_ranges(w.sessions[0], keep_recent=4)
    dead = np.zeros(T, bool)
    for a, b in ranges:
        dead[a:b] = True
    gran = c.compaction_granule()
    keep = [a for a in range(0, T, gran) if not dead[a:a + gran].all()]
    live_slots = sum(min(gran, T - a) for a in keep)
    max_saving = -(-T // 64) - (-(-live_slots // 64))
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    # a ~2 ms busy kernel ahead of each timed call: the host-side planning overlaps it,
    # so the events bracket the device work (copies and kernels) alone
    torch.cuda.synchronize()
    torch.cuda._sleep(4_000_000)
    ev[0].record(st)
    c.evict(0, ranges)
    ev[1].record(st)
    torch.cuda._sleep(4_000_000)
    ev[2].record(st)
    new_len, moved = c.compact(0, max(1, max_saving))
    ev[3].record(st)
    torch.cuda.synchronize()
    if c.check_errors() != 0:
        raise RuntimeError("device error word set after compaction")
    # bytes a move must read and write: codes, norms, key statistics (or key norms),
    # tile masks of every (layer, kv head), and the granule's modality ids
    B = sh.head_dim * sh.bits // 8
    per_unit = 2 * gran * B + 2 * gran + (4 * sh.head_dim if c.key_codec == 0 else 2 * gran) + gran // 16
    move_bytes = 2 * moved * (sh.num_layers * sh.num_kv_heads * per_unit + gran)
    compact_ms = ev[2].elapsed_time(ev[3])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=Q.device)
    for _ in range(3):
        c.decode(Q, out)
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        c.decode(Q, out)
        b.record(st)
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return {"deleted_tokens": int(dead.sum()), "slots_before": T, "slots_after": int(new_len),
            "moved_granules": int(moved), "granule": gran, "evict_ms": ev[0].elapsed_time(ev[1]),
            "compact_ms": compact_ms, "compact_bytes": move_bytes,
            "compact_gbs": move_bytes / (compact_ms / 1e3) / 1e9,
            "compact_frac": move_bytes / (compact_ms / 1e3) / 1e9 / peak,
            "decode_ms_after": tot / steps, "l2": "256 MB buffer rewritten before each decode"}


def pseudo_leg(torch, device, peak, steps=10, near_tokens=8192, prototypes=3072, per_proto=8):
    """ProtoKV-style far memory next to the compressed cache: a near window of the
    last 8,192 tokens of the 3B-shaped stream (2-bit) and 3,072 prototypes x 8
    fp16 pseudo tokens per (layer, kv head) (near : far = 1 : 3, the pages'
    default split), drawn on the device from a seeded generator (centres ~ N(0,
    scale^2) with per-channel scales log-uniform in [0.5, 4], residuals 0.25 of the
    scale; masses log-uniform in [1, 300], a tenth inactive). The 0.9 GB of pseudo
    tokens exceed L2, so every step reads them from HBM."""
    w = synth.qwen3b(tokens=near_tokens)
    sh = w.shape
    caches, _, _ = build_cache(w, torch, device, replicas=1)
    c = caches[0]
    g = torch.Generator(device=device).manual_seed(0x50F7)
    shp = (1, sh.num_layers, sh.num_kv_heads)
    nf = prototypes * per_proto
    scale = torch.exp(torch.empty(shp + (1, sh.head_dim), device=device).uniform_(math.log(0.5), math.log(4.0),
                                                                                    generator=g))
    kf = (scale * (torch.randn(shp + (prototypes, sh.head_dim), device=device, generator=g)
                   .repeat_interleave(per_proto, dim=3)
                   + 0.25 * torch.randn(shp + (nf, sh.head_dim), device=device, generator=g))).half()
    vf = (scale * (torch.randn(shp + (prototypes, sh.head_dim), device=device, generator=g)
                   .repeat_interleave(per_proto, dim=3)
                   + 0.25 * torch.randn(shp + (nf, sh.head_dim), device=device, generator=g))).half()
    mass = torch.exp(torch.empty(shp + (prototypes,), device=device).uniform_(0.0, math.log(300.0), generator=g))
    mass = torch.where(torch.rand(shp + (prototypes,), device=device, generator=g) < 0.1, torch.zeros_like(mass),
                       mass.round())
    Q = torch.from_numpy(w.queries(0)).to(device)
    out = torch.empty_like(Q)
    for _ in range(3):
        c.decode_pseudo(Q, kf, vf, mass, per_proto, out)
        c.decode(Q, out)
    torch.cuda.synchronize()
    c.profile_enable(True)
    for _ in range(steps):
        c.decode(Q, out)
    torch.cuda.synchronize()
    near_split, near_merge = (list(x) for x in c.profile_read())
    c.profile_enable(False)
    c.profile_enable(True)
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        c.decode_pseudo(Q, kf, vf, mass, per_proto, out)
    e1.record(st)
    torch.cuda.synchronize()
    ps_split, ps_merge = (list(x) for x in c.profile_read())
    c.profile_enable(False)
    if c.check_errors() != 0:
        raise RuntimeError("device error word set after the pseudo-token decode")
    step_ms = e0.elapsed_time(e1) / steps
    far_ms = float(np.mean(ps_split)) - float(np.mean(near_split))
    units = sh.num_layers * sh.num_kv_heads
    far_bytes = units * (nf * sh.head_dim * 2 * 2 + prototypes * 4) + 2 * Q.numel() * 2
    return {"near_tokens": near_tokens, "prototypes": prototypes, "per_prototype": per_proto, "far_tokens": nf,
            "ms_per_step": step_ms, "context_tokens_per_s": (near_tokens + nf) / (step_ms / 1e3),
            "near_decode_ms": float(np.mean(near_split)), "near_plus_far_ms": float(np.mean(ps_split)),
            "merge_ms": float(np.mean(ps_merge)),
            "far_kernel_ms": far_ms, "far_bytes": far_bytes,
            "far_roofline": {"bound": "hbm", "achieved": far_bytes / (far_ms / 1e3) / 1e9, "peak": peak,
                             "unit": "GB/s", "frac": far_bytes / (far_ms / 1e3) / 1e9 / peak,
                             "note": "far kernel time = (near + far kernels) - (near kernel alone), CUDA events"}}




def timed_steps(caches, Q, out, torch, steps, warmup):
    """Warm-up steps, a profiled pass (per-kernel CUDA events: decode kernel, merge
    kernel), then `steps` back-to-back decode steps timed with CUDA events on the
    launching stream (the replicas alternate). Returns (total ms, split ms list,
    merge ms list)."""
    st = torch.cuda.current_stream()
    for i in range(warmup):
        caches[i % len(caches)].decode(Q, out)
    torch.cuda.synchronize()
    for c in caches:
        c.profile_enable(True)
    for i in range(steps):
        caches[i % len(caches)].decode(Q, out)
    torch.cuda.synchronize()
    split_ms, merge_ms = [], []
    for c in caches:
        a, b = c.profile_read()
        split_ms += list(a)
        merge_ms += list(b)
        c.profile_enable(False)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(steps):
        caches[i % len(caches)].decode(Q, out)
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), split_ms, merge_ms


def append_rates(chunks):
    """Append rates of one replica's chunks [(ms, tokens)]: the steady state (every chunk
    after the first call, whose host side also sets the kernels' attributes and looks
    up the tensor-map encoder) and the plain total over all chunks."""
    rest = chunks[1:] or chunks
    ms = [x for x, _ in rest]
    toks = [n for _, n in rest]
    return {"tokens_per_s": sum(toks) / (sum(ms) / 1e3), "ms_per_chunk_median": float(np.median(ms)),
            "tokens_per_chunk_median": float(np.median(toks)), "chunks_counted": len(rest),
            "tokens_per_s_all_chunks": sum(n for _, n in chunks) / (sum(x for x, _ in chunks) / 1e3)}


def config_summary(w, args, torch, device, peak, steps, warmup, key_codec="omni", workload=None):
    """One extra configuration of the default run: its caches built on the device,
    decode steps timed as for the headline line (two replicas alternate unless one
    cache alone is more than four times the L2), every cache freed afterwards."""
    sh = w.shape
    lengths = [s.length for s in w.sessions]
    split_bytes, out_bytes, rot_bytes = algorithmic_bytes(w, lengths, key_codec)
    replicas = 2 if split_bytes < 4 * 129e6 else 1
    caches, append_ms, _ = build_cache(w, torch, device, replicas=replicas, key_codec=key_codec,
                                       keep_layer0=workload is not None)
    Q = torch.from_numpy(w.queries(0)).to(device)
    out = torch.empty_like(Q)
    ms, split_ms, merge_ms = timed_steps(caches, Q, out, torch, steps, warmup)
    errs = [c.check_errors() for c in caches]
    ap = append_rates(append_ms[0])
    bnd = None
    if workload is not None and not args.no_cpu_baseline:
        bnd = dict(boundary_counts(workload, sh.bits, sh.group_size, caches[0]),
                   of="layer 0 of session 0 (%d tokens), every kv head: GPU state against the oracle fed the same "
                      "inputs and rotations" % lengths[0])
    del caches, Q, out
    torch.cuda.empty_cache()
    if any(errs):
        raise RuntimeError("device error word set in %s" % w.name)
    ms_step = ms / steps
    avg_split = float(np.mean(split_ms))
    step_us = 1e3 * (np.asarray(split_ms) + np.asarray(merge_ms))
    achieved = split_bytes / (avg_split / 1e3) / 1e9
    return {"workload": config_of(w, args)["workload"], "sessions": len(lengths), "context_tokens": sum(lengths),
            "steps": steps, "warmup": warmup, "ms_per_step": ms_step,
            "context_tokens_per_s": sum(lengths) / (ms_step / 1e3),
            "hbm_gbs_step": (split_bytes + out_bytes) / (ms_step / 1e3) / 1e9,
            "latency_us": {"p50": float(np.percentile(step_us, 50)), "p99": float(np.percentile(step_us, 99))},
            "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "bytes_per_launch": split_bytes,
                         "avg_launch_ms": avg_split, "merge_kernel_avg_ms": float(np.mean(merge_ms))},
            "boundary_codes": bnd,
            "append_tokens_per_s": ap["tokens_per_s"], "append_ms_per_chunk_median": ap["ms_per_chunk_median"],
            "append_tokens_per_chunk_median": ap["tokens_per_chunk_median"],
            "l2": "two cache replicas alternate" if replicas == 2 else "one cache, %.1f GB per step" % (
                split_bytes / 1e9)}


def streaming_summary(args, torch, device, peak, tokens=131072):
    """The streaming configuration: 1-s chunks [2,304 video, 25 audio] of the 3B head
    shape appended one by one, one decode query after every chunk. Reports append
    throughput on these chunks, decode latency against context length (CUDA events
    around the device work of each call, host work included), and plain decodes at
    the final length for comparison (no append in between)."""
    from bit_kv_cache_rht_gb300.okvq import Cache
    w = synth.streaming(tokens=tokens, bits=getattr(args, "bits", 2), group_size=getattr(args, "group_size", 32))
    sh = w.shape
    R, _ = calibrate(w, torch, device)
    c = Cache(1, sh.num_layers, sh.num_q_heads, sh.num_kv_heads, w.max_tokens, R, head_dim=sh.head_dim,
              group_size=sh.group_size, bits=sh.bits, num_modalities=sh.num_modalities,
              hadamard_seed=w.hadamard_seed)
    K, V = device_session_kv(w, 0, torch, device)
    M = torch.from_numpy(w.sessions[0].modality()).to(device)
    Q = torch.from_numpy(w.queries(0)).to(device)
    out = torch.empty_like(Q)
    st = torch.cuda.current_stream()
    rows = []
    for a, b in w.sessions[0].chunk_bounds():
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(st)
        c.append(0, K[a:b], V[a:b], M[a:b])
        ev[1].record(st)
        c.decode(Q, out)
        ev[2].record(st)
        rows.append((b, b - a, ev))
    torch.cuda.synchronize()
    if c.check_errors() != 0:
        raise RuntimeError("device error word set in the streaming run")
    res = [(T, n, e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])) for T, n, e in rows]
    # plain decodes at the final length
    for _ in range(5):
        c.decode(Q, out)
    torch.cuda.synchronize()
    plain = []
    for _ in range(20):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        c.decode(Q, out)
        e1.record(st)
        torch.cuda.synchronize()
        plain.append(e0.elapsed_time(e1))
    c.close()
    del K, V, M, c
    torch.cuda.empty_cache()
    full = [r for r in res if r[1] == 2329]
    ap_tok = sum(n for _, n, _, _ in full)
    ap_ms = sum(x for _, _, x, _ in full)
    T_end, _, _, dec_last = res[-1]
    return {"workload": "streaming: 3B head shape, 1-s chunks [2,304 video, 25 audio] appended to %d tokens, a "
                        "decode after every chunk" % T_end,
            "chunks": len(res), "append_tokens_per_s_2329": ap_tok / (ap_ms / 1e3),
            "append_ms_per_2329_chunk": float(np.median([x for _, _, x, _ in full])),
            "decode_ms_after_append_at_context": [[T, round(d, 4)] for T, _, _, d in res[::8]] + [[T_end,
                                                                                                  round(dec_last, 4)]],
            "decode_ms_after_last_append": dec_last, "plain_decode_ms_at_final_length": float(np.median(plain)),
            "context_tokens_per_s_final": T_end / (float(np.median(plain)) / 1e3),
            "note": "decode after an append includes the host work split and its upload on the stream"}


def streaming_run(args, torch, device, peak):
    """--workload streaming: the streaming summary as its own JSON line."""
    s = streaming_summary(args, torch, device, peak)
    w = make_workload(args)
    line = {"metric": METRIC, "value": s["context_tokens_per_s_final"], "unit": UNIT, "n_gpus": 1,
            "steps": 20, "warmup": 5, "ms_per_step": s["plain_decode_ms_at_final_length"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16 operands, f32 accumulate",
            "data": "synthetic", "config": config_of(w, args), "streaming": s}
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands (plain numpy, fp64), timed on host cores
# ---------------------------------------------------------------------------

def cpu_model():
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20)
        for line in r.stdout.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def _oracle_for_layers(args, layers, R=None, kv=None):
    """Oracle state of session 0 of the workload for the listed layers (appended in
    the workload's chunks), the value rotations R (the GPU's, when given) and the
    inputs kv = (K, V) [T][len(layers)][Hkv][d] (the GPU cache's, when given; else the
    workload's numpy draw)."""
    from oracle import okvq_oracle as o
    w = make_workload(args)
    sh = w.shape
    if R is None:
        Vc, modc = w.calibration_slice()
        R = o.calibrate_rotations(Vc, modc, sh.num_modalities)[0].astype(np.float32)
    oc = o.OracleCache(1, sh.num_layers, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.group_size, sh.bits,
                       w.max_tokens, w.hadamard_seed, R, layers=layers, key_codec=args.key_codec)
    K, V = w.session_kv(0, layers) if kv is None else kv
    mod = w.sessions[0].modality()
    for a, b in w.sessions[0].chunk_bounds():
        oc.append(0, K[a:b], V[a:b], mod[a:b], layers_in=layers)
    return w, oc


def _worker(conn, args, layers, R):
    """One host core: the oracle state of its layers, then full-step decodes on command."""
    w, oc = _oracle_for_layers(args, layers, R)
    Q = w.queries(0)
    conn.send("ready")
    while True:
        cmd = conn.recv()
        if cmd == "stop":
            break
        t0 = time.perf_counter()
        oc.decode(Q)
        conn.send(time.perf_counter() - t0)


def _all_core_steps(args, R, steps, warmup):
    """Full decode steps of session 0 on every host core: the layers are dealt out
    to one spawned process per core, each holding its layers' oracle state; a step
    is all processes decoding their layers, timed from the command to the last
    answer (wall clock)."""
    import multiprocessing as mp
    w = make_workload(args)
    L = w.shape.num_layers
    ncores = min(os.cpu_count() or 1, L)
    ctx = mp.get_context("spawn")
    procs, conns = [], []
    for i in range(ncores):
        a, b = ctx.Pipe()
        p = ctx.Process(target=_worker, args=(b, args, list(range(i, L, ncores)), R), daemon=True)
        p.start()
        procs.append(p)
        conns.append(a)
    for c in conns:
        assert c.recv() == "ready"
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        for c in conns:
            c.send("step")
        for c in conns:
            c.recv()
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    for c in conns:
        c.send("stop")
    for p in procs:
        p.join(timeout=30)
    return times, ncores


def compare_with_oracle(state, oc):
    """Boundary-code accounting of one GPU-stored layer against the oracle (layer 0,
    session 0, every kv head): codes whose pre-quantization value lies within 1e-5
    of a decision threshold are flagged by the oracle; the GPU may pick either side
    there. Every other code, the statistics and the tail must match bit for bit."""
    from oracle import okvq_oracle as o
    r = dict(k_codes=0, k_flagged=0, k_differ_flagged=0, k_differ_strict=0, v_codes=0, v_flagged=0,
             v_differ_flagged=0, v_differ_strict=0, norms=0, norm_flagged=0, norm_differ_flagged=0,
             norm_differ_strict=0, stats_equal=True, tail_equal=True)
    bits = oc.bits
    for h in range(oc.Hkv):
        e = oc.units[(0, oc.layers[0], h)].export()
        for kind in ("k", "v"):
            g = o.unpack_codes(state[kind + "codes"][h], bits)
            ref = o.unpack_codes(e[kind + "codes"], bits)
            bnd = e[kind + "bnd"]
            d = g != ref
            r[kind + "_codes"] += int(d.size)
            r[kind + "_flagged"] += int(bnd.sum())
            r[kind + "_differ_flagged"] += int((d & bnd).sum())
            r[kind + "_differ_strict"] += int((d & ~bnd).sum())
        gn, on = state["vnorm"][h].view(np.uint16), e["vnorm"].view(np.uint16)
        d = gn != on
        r["norms"] += int(d.size)
        r["norm_flagged"] += int(e["nbnd"].sum())
        r["norm_differ_flagged"] += int((d & e["nbnd"]).sum())
        r["norm_differ_strict"] += int((d & ~e["nbnd"]).sum())
        if "kstats" in state:
            r["stats_equal"] &= bool(np.array_equal(state["kstats"][h].view(np.uint16), e["kstats"].view(np.uint16)))
            r["tail_equal"] &= bool(np.array_equal(state["ktail"][h].view(np.uint16), e["ktail"].view(np.uint16)))
    return r


def cpu_baseline_child(args):
    """Time the oracle as it stands on the host cores (no GPU in this process):
    single-threaded on layer 0 of session 0 (repeated decodes for --cpu-seconds,
    extrapolated linearly to every layer), then full steps on every core; with
    --gpu-state, also the boundary-code accounting of the GPU's layer 0."""
    R = None
    state = None
    if args.gpu_state:
        z = np.load(args.gpu_state)
        R = z["R"]
        kv0 = (z["K0"][:, None], z["V0"][:, None])
        state = {k: z[k] for k in z.files if k not in ("R", "K0", "V0")}
    w, oc = _oracle_for_layers(args, [0], R, kv0 if state is not None else None)
    sh = w.shape
    Q = w.queries(0)
    reps, t_total = 0, 0.0
    while t_total < args.cpu_seconds or reps == 0:
        t0 = time.perf_counter()
        oc.decode(Q)
        t_total += time.perf_counter() - t0
        reps += 1
        if reps >= args.cpu_max_reps:
            break
    per_sample = t_total / reps
    T0 = w.sessions[0].length
    T_all = sum(x.length for x in w.sessions)
    step_s = per_sample * sh.num_layers * T_all / T0      # linear in layers and in cached tokens
    res = {"single_core": {"value": T_all / step_s, "unit": UNIT, "cores": 1,
                           "sample": "oracle decode of layer 0 of session 0 (%d of %d (layer, kv head) units), %d "
                                     "repetitions, %.1f s of CPU time, extrapolated linearly to all %d layers%s"
                                     % (sh.num_kv_heads, sh.num_layers * sh.num_kv_heads, reps, t_total,
                                        sh.num_layers, "" if len(w.sessions) == 1 else
                                        " and all %d sessions' tokens" % len(w.sessions)),
                           "step_s_extrapolated": step_s}}
    if state is not None:
        res["boundary"] = compare_with_oracle(state, oc)
    if args.all_cores:
        times, ncores = _all_core_steps(args, R, args.all_core_steps, 1)
        st = statistics.median(times)
        T_s0 = w.sessions[0].length
        res["all_cores"] = {"value": T_s0 / st, "unit": UNIT, "cores": ncores, "step_s": st,
                            "steps": len(times),
                            "sample": "full decode steps of session 0 (%d tokens, all %d layers), layers dealt to %d "
                                      "spawned processes, one per core, wall clock per step (median of %d)"
                                      % (T_s0, sh.num_layers, ncores, len(times))
                                      + ("" if len(w.sessions) == 1 else "; session 0 only")}
    print(json.dumps(res))


def save_layer0_state(cache, path):
    """Layer 0 of session 0 as the GPU stored it, with the rotations and inputs it was
    built from (the CPU side's boundary-code accounting reads this file)."""
    st0 = cache.export_state(0)
    arrays = {k: np.ascontiguousarray(v[0]) for k, v in st0.items() if k != "mod" and v.ndim >= 2}
    arrays["R"] = np.asarray(cache.rotations_used, np.float32)
    arrays["K0"], arrays["V0"] = cache.layer0_kv
    np.savez(path, **arrays)


def boundary_child(args):
    """The oracle's layer 0 of session 0, fed the GPU cache's inputs and rotations, and
    the boundary-code accounting of the GPU's stored state against it."""
    z = np.load(args.gpu_state)
    kv0 = (z["K0"][:, None], z["V0"][:, None])
    state = {k: z[k] for k in z.files if k not in ("R", "K0", "V0")}
    _, oc = _oracle_for_layers(args, [0], z["R"], kv0)
    print(json.dumps(compare_with_oracle(state, oc)))


def boundary_counts(workload, bits, group_size, cache):
    """Boundary-code accounting of one configuration (CPU child, no GPU)."""
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    try:
        save_layer0_state(cache, path)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                   CUDA_VISIBLE_DEVICES="")
        cmd = [sys.executable, os.path.abspath(__file__), "--boundary-child", "--workload", workload, "--bits",
               str(bits), "--group-size", str(group_size), "--key-codec", "omni", "--gpu-state", path]
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, check=True).stdout
        return json.loads(out.strip().splitlines()[-1])
    finally:
        os.unlink(path)


def run_cpu_baseline(args, gpu_state=None, all_cores=True, steps=3):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", "--workload", args.workload,
           "--bits", str(getattr(args, "bits", 2)), "--group-size", str(getattr(args, "group_size", 32)),
           "--cpu-seconds", str(args.cpu_seconds), "--cpu-max-reps", str(args.cpu_max_reps),
           "--key-codec", args.key_codec, "--all-core-steps", str(steps)]
    if all_cores:
        cmd.append("--all-cores")
    if gpu_state:
        cmd += ["--gpu-state", gpu_state]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        return {"error": "cpu baseline failed: " + r.stderr[-400:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_entry(res):
    """The line's cpu_baseline object: all host cores on full steps when measured,
    the single-core figure beside it."""
    model = cpu_model()
    if "error" in res:
        return {"value": None, "unit": UNIT, "cores": None, "kind": "oracle", "sample": res["error"]}
    sc = res["single_core"]
    ac = res.get("all_cores")
    head = ac if ac else sc
    out = {"value": head["value"], "unit": UNIT, "cores": head["cores"], "kind": "oracle", "sample": head["sample"],
           "cpu_model": model, "nproc": os.cpu_count(), "single_core": sc}
    if ac:
        out["all_cores"] = ac
    return out


def reference_arm(args):
    """--impl reference: the oracle on every host core, timing full decode steps of
    the workload's session 0 (no extrapolation: every step decodes every layer)."""
    if rank_env()[1] != 0:         # under a multi-rank launch, rank 0 alone times the oracle
        return
    ns = argparse.Namespace(**vars(args))
    times, ncores = _all_core_steps(ns, None, args.steps, args.warmup)
    w = make_workload(args)
    T0 = w.sessions[0].length
    st = statistics.median(times)
    v = T0 / st
    sample = ("full decode steps of session 0 (%d tokens, all %d layers) on %d spawned processes (one per core, "
              "layers dealt out), wall clock per step, median of %d" % (T0, w.shape.num_layers, ncores, len(times)))
    if len(w.sessions) > 1:
        sample += "; session 0 of %d" % len(w.sessions)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": st * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": ncores, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model(), "nproc": os.cpu_count()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_of(w, args):
    sh = w.shape
    lengths = [x.length for x in w.sessions]
    cache = ("%d-token cache" % lengths[0]) if len(lengths) == 1 else (
        "%d sessions of %d-%d tokens (%d in all)" % (len(lengths), min(lengths), max(lengths), sum(lengths)))
    return {"workload": "%s: %d layers, %d q / %d kv heads, head_dim %d, %s, %d-bit codes, group %d"
                        % (w.name, sh.num_layers, sh.num_q_heads, sh.num_kv_heads, sh.head_dim,
                           cache, sh.bits, sh.group_size),
            "sessions": len(w.sessions), "context_tokens": sum(lengths), "bits": sh.bits,
            "group_size": sh.group_size,
            "key_codec": "turboquant (per-token norm, fixed scale)" if getattr(args, "key_codec", "omni") == "turbo"
                         else "omnikvquant (per-group min-max ranges)",
            "l2": "inputs larger than L2: two cache replicas (2 x %.0f MB) alternate between steps"
                  % (algorithmic_bytes(w, [s.length for s in w.sessions], getattr(args, "key_codec", "omni"))[0]
                     / 1e6),
            "parallelism": "replicas" if getattr(args, "gpus", 1) > 1 else "single GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="okvq", choices=["okvq", "reference"])
    ap.add_argument("--workload", default="qwen3b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-max-reps", type=int, default=1000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only (no extra configurations)")
    ap.add_argument("--key-codec", default="omni", choices=["omni", "turbo"],
                    help="omni: per-group key ranges (the method); turbo: the TurboQuant comparison codec")
    ap.add_argument("--bits", type=int, default=2, choices=[2, 4])
    ap.add_argument("--group-size", type=int, default=32, choices=[32, 64])
    ap.add_argument("--cpu-baseline-child", action="store_true")
    ap.add_argument("--boundary-child", action="store_true")
    ap.add_argument("--all-cores", action="store_true")
    ap.add_argument("--all-core-steps", type=int, default=3)
    ap.add_argument("--gpu-state", default=None)
    args = ap.parse_args()
    if args.cpu_baseline_child:
        return cpu_baseline_child(args)
    if args.boundary_child:
        return boundary_child(args)
    if args.impl == "reference":
        return reference_arm(args)
    args.warmup = max(args.warmup, 3)

    import torch
    import torch.distributed as dist
    world, rank, local = rank_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    from bit_kv_cache_rht_gb300 import okvq
    okvq.load()

    if args.workload == "streaming":
        return streaming_run(args, torch, device, peaks()[0])
    w = make_workload(args)
    sh = w.shape
    caches, append_ms, calib = build_cache(w, torch, device, replicas=2, key_codec=args.key_codec,
                                           keep_layer0=not args.no_cpu_baseline)
    lengths = [s.length for s in w.sessions]
    split_bytes, out_bytes, rot_bytes = algorithmic_bytes(w, lengths, args.key_codec)
    step_bytes = split_bytes + out_bytes

    Q = torch.from_numpy(w.queries(0)).to(device)
    out = torch.empty_like(Q)
    st = torch.cuda.current_stream()
    sampler = ClockSampler()
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms, split_ms, merge_ms = timed_steps(caches, Q, out, torch, args.steps, args.warmup)
    if world > 1:
        dist.barrier()

    # end to end through okvq_decode_host: every step copies the queries from pinned
    # host memory, decodes and delivers the outputs to pinned host memory. Timed two
    # ways: host wall clock around the calls and a final synchronisation (the line's
    # value), and CUDA events on the stream (device time only).
    q_host = Q.cpu().pin_memory()
    o_host = torch.empty(Q.shape, dtype=torch.float16).pin_memory()
    for i in range(4):
        caches[i % 2].decode_host(q_host, o_host)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        caches[i % 2].decode_host(q_host, o_host)
    torch.cuda.synchronize()
    e2e_wall_ms = (time.perf_counter() - t0) * 1e3
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(st)
    for i in range(args.steps):
        caches[i % 2].decode_host(q_host, o_host)
    f1.record(st)
    torch.cuda.synchronize()
    e2e_ev_ms = f0.elapsed_time(f1)
    clocks = sampler.stop(local) if rank == 0 else None

    t_max, e2e_max, e2e_ev_max = max_over_ranks([ms, e2e_wall_ms, e2e_ev_ms], world, device)
    total_tokens = job_tokens(world, args.steps, lengths)
    value = total_tokens / (t_max / 1e3)

    if rank == 0:
        peak, peak_kind = peaks()
        avg_split = float(np.mean(split_ms))
        step_us = 1e3 * (np.asarray(split_ms) + np.asarray(merge_ms))
        achieved = split_bytes / (avg_split / 1e3) / 1e9
        ms_step = t_max / args.steps
        ap = append_rates(append_ms[0])
        # append, steady state (every chunk after the first call): reads fp16 K and V, writes codes, norms, statistics; flops of the value
        # rotation (2 d^2 per token-head) and the key transform; the binding one of the two
        ap_bytes_tok = sh.num_layers * sh.num_kv_heads * (2 * 2 * sh.head_dim + 2 * sh.head_dim * sh.bits // 8 + 2
                                                           + 4 * sh.head_dim / sh.group_size) + 1
        ap_flops_tok = sh.num_layers * sh.num_kv_heads * (2 * sh.head_dim ** 2 + 10 * sh.head_dim)
        ap_gbs = ap["tokens_per_s"] * ap_bytes_tok / 1e9
        ap_tfs = ap["tokens_per_s"] * ap_flops_tok / 1e12
        traffic = None
        tp = os.path.join(ROOT, "profiles", "decode_traffic.json")
        if os.path.exists(tp):
            with open(tp) as f:
                tj = json.load(f)
            # DRAM bytes of one decode launch from an ncu capture, valid only while the
            # decode kernel's sources are the ones that capture measured
            if (tj.get("workload") == args.workload and tj.get("source_sha256") == decode_source_sha256()
                    and args.key_codec == "omni"):
                traffic = tj.get("bytes_per_launch")
        tc_peak, tc_kind = tensor_peak()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 operands, f32 accumulate", "data": "synthetic",
            "config": config_of(w, args),
            "hbm_gbs_step": step_bytes / (ms_step / 1e3) / 1e9,
            "latency_us": {"p50": float(np.percentile(step_us, 50)), "p99": float(np.percentile(step_us, 99)),
                           "of": "decode + merge kernels per step, profiled pass (%d steps)" % len(step_us)},
            "roofline": {"bound": "hbm", "kernel": "decode_kernel (split-K fused 2-bit attention)",
                         "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "bytes_per_launch": split_bytes, "avg_launch_ms": avg_split,
                         "merge_kernel_avg_ms": float(np.mean(merge_ms)),
                         "with_R_frac_step": (step_bytes + rot_bytes) / (ms_step / 1e3) / 1e9 / peak},
            "append": {"tokens_per_s": ap["tokens_per_s"], "ms_per_chunk_median": ap["ms_per_chunk_median"],
                       "tokens_per_chunk_median": ap["tokens_per_chunk_median"], "chunks": len(append_ms[0]),
                       "tokens_per_s_all_chunks": ap["tokens_per_s_all_chunks"],
                       "of": "every chunk after the first call (CUDA events around each okvq_append_chunk on the "
                             "stream, both grids); tokens_per_s_all_chunks: every chunk, the first call's one-time "
                             "host setup included",
                       "gbs": ap_gbs, "tflops": ap_tfs,
                       "roofline": {"bound": "hbm" if ap_gbs / peak >= ap_tfs / tc_peak else "tensor",
                                    "bytes_frac": ap_gbs / peak, "flops_frac": ap_tfs / tc_peak,
                                    "frac": max(ap_gbs / peak, ap_tfs / tc_peak),
                                    "flops": "2 d^2 + 10 d per token-head (the value rotation, on the tensor "
                                             "cores, and the key transform)",
                                    "flops_peak_tflops": tc_peak, "flops_peak_kind": tc_kind}},
            "calibration": dict(calib, kernel="calib_kernel (value-rotation covariance + Jacobi eigenbasis)"),
            "e2e": {"value": total_tokens / (e2e_max / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(Q.numel() * 2),
                    "d2h_bytes_per_step": int(out.numel() * 2), "ms_per_step_wall": e2e_max / args.steps,
                    "device_event_value": total_tokens / (e2e_ev_max / 1e3),
                    "how": "okvq_decode_host: pinned-host queries read over the host link by the query staging "
                           "kernel and outputs stored into pinned host memory by the merge kernel, every step (3 "
                           "launches a step); value = host wall clock around %d calls and a final "
                           "synchronisation; device_event_value = CUDA events on the stream" % args.steps},
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
        }
        default = (args.workload == "qwen3b" and sh.bits == 2 and sh.group_size == 32 and args.key_codec == "omni"
                   and world == 1)
        gpu_state = None
        if not args.no_cpu_baseline:
            # the GPU-stored state of layer 0 (session 0) and the rotations it used: the
            # CPU leg compares the oracle's codes with it (boundary-code accounting)
            fd, gpu_state = tempfile.mkstemp(suffix=".npz")
            os.close(fd)
            save_layer0_state(caches[0], gpu_state)
        if default:
            line["compaction"] = compaction_leg(caches[0], w, torch, Q, out, peak, 10)
        del caches
        torch.cuda.empty_cache()
        if default:
            line["pseudo_tokens"] = pseudo_leg(torch, device, peak)
            if not args.no_extra:
                cfg = {}
                ns = argparse.Namespace(**vars(args))
                cfg["qwen7b_2bit_g32"] = config_summary(synth.qwen7b(), ns, torch, device, peak, 20, 5,
                                                        workload="qwen7b")
                cfg["multisession_2bit_g32"] = config_summary(synth.multisession(), ns, torch, device, peak, 20, 5,
                                                              workload="multisession")
                cfg["multisession_4bit_g32"] = config_summary(synth.multisession(bits=4), ns, torch, device, peak, 20,
                                                              5, workload="multisession")
                cfg["streaming"] = streaming_summary(ns, torch, device, peak)
                line["configs"] = cfg
        if not args.no_cpu_baseline:
            res = run_cpu_baseline(args, gpu_state=gpu_state, all_cores=True, steps=3)
            if gpu_state:
                os.unlink(gpu_state)
            line["cpu_baseline"] = cpu_baseline_entry(res)
            if "boundary" in res:
                line["boundary_codes"] = dict(res["boundary"], of="layer 0 of session 0, every kv head: GPU state "
                                              "against the oracle fed the same inputs and rotations")
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
