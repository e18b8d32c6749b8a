"""Benchmark of the Lynx hot path on one GB300 (or N, one process per GPU).

One step = one pass of the whole hot path over a Qwen3-235B-A22B-shaped KV
cache, layer by layer (94 layers x 4 KV heads x 128 channels x 131,072 tokens,
K and V: 385,024 pages, 25.2e9 BF16 bytes, 16 query heads; synthetic, seeded):

  encode              lynx_encode_pages, one call per layer (4,096 pages)
  reconstruct_anchor  lynx_reconstruct from the Anchor alone, BF16 out, per layer
  reconstruct_full    lynx_reconstruct from Anchor + Residual, BF16 out, per layer
  decode_anchor_b1    1-token draft decode over the Anchor planes, B = 1, the
                      full 131,072-token context, per layer
  verify_full_t8      8-token causal verification over the full codes, per layer
  decode_bf16_b1      the BF16-page baseline decode, B = 1, per layer

value = sum over the step's kernels of each kernel's headline bytes (encode:
BF16 bytes in; reconstruct and decode: packed KV bytes read; BF16 baseline:
BF16 KV bytes read) / step time, in GB/s.  The two numbers the metric names
(encode GB/s of BF16 in, Anchor decode GB/s of packed KV read) and their
fractions of the measured HBM bandwidth are top-level keys; every kernel's
numbers are under "kernels".  The Qwen-32B-shaped 64-layer cache step, the
decode-attention sweep and the comparators are under "other_workloads".

--impl reference times the CPU oracle on a bounded sample of the same step.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV encode GB/s (BF16 in) and Anchor-KV decode-attn GB/s, % of GB300 HBM peak"
UNIT = "GB/s"


class Cache:
    """Shape of a multi-layer KV cache held as pages: layer l owns pages
    [l * per_layer, (l + 1) * per_layer), its K pages first (head-major, npph
    pages per head), then its V pages."""

    def __init__(self, name, n_layers, hkv, hq, n_tok, seed):
        self.name, self.n_layers, self.hkv, self.hq, self.n_tok, self.seed = name, n_layers, hkv, hq, n_tok, seed
        self.npph = n_tok // 256
        self.per = hkv * self.npph            # pages per tensor (K or V) per layer
        self.per_layer = 2 * self.per
        self.n_pages = n_layers * self.per_layer


QWEN235B = Cache("Qwen3-235B-A22B-shaped KV cache: 94 layers x 4 KV heads x 128 x 131072 tokens, K and V "
                 "(385024 pages of 128x256 BF16, 25.2e9 B), 16 query heads; layer-streamed: encode, both "
                 "reconstructs, B=1 anchor draft decode, T=8 full-code verification and the BF16 decode, "
                 "one call per layer", 94, 4, 16, 131072, 7)

# the Qwen-32B-shaped 64-layer cache (other_workloads; module globals used by its helpers)
WORKLOAD = ("Qwen-32B-shaped KV cache: 64 layers x 8 KV heads x 128 x 16384 tokens, K and V "
            "(65536 pages of 128x256 BF16, 4.29e9 B); decode B=1 and B=8 (anchor), T=8 verify (full), "
            "32 query heads")
N_LAYERS, HKV, HQ, N_TOK = 64, 8, 32, 16384
NPPH = N_TOK // 256                 # pages per head
PER = HKV * NPPH                    # pages per tensor per layer (512)
N_PAGES = 2 * N_LAYERS * PER        # 65536
E2E_CHUNKS = 8                       # layer chunks of the end-to-end step's copy pipeline


def set_layers(n):
    """A main cache with fewer layers (profiling captures of a small case)."""
    global QWEN235B
    c = QWEN235B
    QWEN235B = Cache(c.name.replace(f"{c.n_layers} layers", f"{n} layers"), n, c.hkv, c.hq, c.n_tok, c.seed)


PLANE, META, PAGE = 16384, 9216, 65536

# per-page byte counts (headline, moved) of each kernel
BYTES = {
    "encode": (PAGE, PAGE + 2 * PLANE + META),
    "reconstruct_anchor": (PLANE + META, PLANE + META + PAGE),
    "reconstruct_full": (2 * PLANE + META, 2 * PLANE + META + PAGE),
    "decode_anchor": (PLANE + META, PLANE + META),
    "decode_full": (2 * PLANE + META, 2 * PLANE + META),
    "decode_bf16": (PAGE, PAGE),
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


NOMINAL_HBM_GBS = 8000.0   # GB300's nominal HBM3e bandwidth (context for frac_of_hbm, which uses the measured copy)


def tensor_peak():
    """Dense bf16 tensor-core TFLOP/s for a kernel timed alone (the measured
    burst figure), and where it came from."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def attn_flops(B, T, G, Hkv, n_keys):
    """Algorithmic attention FLOPs of a decode call: Q K^T and P V, 2 * 128 each
    per query row per key (4 D T G per token per KV head)."""
    return 4.0 * 128 * T * G * n_keys * Hkv * B


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm

class Buffers:
    """Device buffers of one cache: the BF16 pages, the encoded pools, a
    reconstruction buffer of one layer, queries, page tables, outputs."""


def build_cache(torch, L, inputs, dev, c: Cache):
    """The cache's BF16 pages (seeded, generated per (layer, K or V) on the
    device), empty encoded pools and one layer's reconstruction buffer."""
    b = Buffers()
    outl = inputs.outlier_pairs(c.hkv, c.seed)
    b.x = torch.empty((c.n_pages, 128, 256), dtype=torch.bfloat16, device=dev)
    for layer in range(c.n_layers):
        for t in range(2):
            i = layer * c.per_layer + t * c.per
            b.x[i:i + c.per] = inputs.kv_pages_torch(c.hkv, c.n_tok, inputs.layer_seed(c.seed, layer, t), outl, dev)
    b.anc = torch.empty((c.n_pages, 128, 128), dtype=torch.uint8, device=dev)
    b.res = torch.empty_like(b.anc)
    b.meta = torch.empty((c.n_pages, L.META_FLOATS), dtype=torch.float32, device=dev)
    b.recon = torch.empty((c.per_layer, 128, 256), dtype=torch.bfloat16, device=dev)
    # one sequence per layer: B = 1, page ids relative to the layer's K (or V) pages
    b.pt = torch.arange(c.per, dtype=torch.int32, device=dev).view(1, c.hkv, c.npph)
    b.ctx = torch.full((1,), c.n_tok, dtype=torch.int32, device=dev)
    b.q1 = inputs.queries_torch((c.n_layers, 1, c.hq, 128), c.seed + 1, dev)
    b.qv = inputs.queries_torch((c.n_layers, 8, c.hq, 128), c.seed + 3, dev)

    def ws(T):
        n = L.lynx_decode_attn_workspace_size(1, T, c.hq, c.hkv, 128, c.npph)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    b.ws1, b.wsv = ws(1), ws(8)
    f32 = dict(dtype=torch.float32, device=dev)
    # separate outputs for every call, so that a readback returns each one's result
    b.oa, b.la = torch.empty((c.n_layers, 1, c.hq, 128), **f32), torch.empty((c.n_layers, 1, c.hq), **f32)
    b.ob, b.lb = torch.empty((c.n_layers, 1, c.hq, 128), **f32), torch.empty((c.n_layers, 1, c.hq), **f32)
    b.ov, b.lv = torch.empty((c.n_layers, 8, c.hq, 128), **f32), torch.empty((c.n_layers, 8, c.hq), **f32)
    return b


def layer_calls(L, c: Cache, b):
    """The step's six calls on layer l, as functions of (l, x, anc, res, meta):
    the buffers are passed so that the end-to-end pipeline can run the same calls."""
    p = L.Params()

    def sl(l):
        return slice(l * c.per_layer, (l + 1) * c.per_layer)

    def kv(t, l):       # (K view, V view) of a pool at layer l
        return t[l * c.per_layer:], t[l * c.per_layer + c.per:]

    def enc(l, x, anc, res, meta):
        L.lynx_encode_pages(x[sl(l)], p, anc[sl(l)], res[sl(l)], meta[sl(l)])

    def rec_a(l, x, anc, res, meta):
        L.lynx_reconstruct(anc[sl(l)], None, meta[sl(l)], p, out=b.recon)

    def rec_f(l, x, anc, res, meta):
        L.lynx_reconstruct(anc[sl(l)], res[sl(l)], meta[sl(l)], p, out=b.recon)

    def dec_a(l, x, anc, res, meta):
        (ka, va), (km, vm) = kv(anc, l), kv(meta, l)
        L.lynx_decode_attn(b.q1[l:l + 1], ka, None, km, va, None, vm, b.pt, b.ctx, c.hkv, p,
                           out=b.oa[l:l + 1], lse=b.la[l:l + 1], workspace=b.ws1)

    def ver_f(l, x, anc, res, meta):
        (ka, va), (kr, vr), (km, vm) = kv(anc, l), kv(res, l), kv(meta, l)
        L.lynx_decode_attn(b.qv[l:l + 1], ka, kr, km, va, vr, vm, b.pt, b.ctx, c.hkv, p, causal=True,
                           out=b.ov[l:l + 1], lse=b.lv[l:l + 1], workspace=b.wsv)

    def dec_b(l, x, anc, res, meta):
        xk, xv = kv(x, l)
        L.lynx_decode_attn_bf16(b.q1[l:l + 1], xk, xv, b.pt, b.ctx, c.hkv, out=b.ob[l:l + 1],
                                lse=b.lb[l:l + 1], workspace=b.ws1)

    n = c.n_pages
    # (name, call, launches per layer, headline bytes, moved bytes) over all layers
    return [
        ("encode", enc, 1, n * BYTES["encode"][0], n * BYTES["encode"][1]),
        ("reconstruct_anchor", rec_a, 1, n * BYTES["reconstruct_anchor"][0], n * BYTES["reconstruct_anchor"][1]),
        ("reconstruct_full", rec_f, 1, n * BYTES["reconstruct_full"][0], n * BYTES["reconstruct_full"][1]),
        ("decode_anchor_b1", dec_a, 2, n * BYTES["decode_anchor"][0], n * BYTES["decode_anchor"][1]),
        ("verify_full_t8", ver_f, 2, n * BYTES["decode_full"][0], n * BYTES["decode_full"][1]),
        ("decode_bf16_b1", dec_b, 2, n * BYTES["decode_bf16"][0], n * BYTES["decode_bf16"][1]),
    ]


def step_kernels(L, c: Cache, b):
    """(name, callable over all layers, launches, headline bytes, moved bytes)."""
    out = []
    for name, fn, lpl, head, moved in layer_calls(L, c, b):
        def run(fn=fn):
            for l in range(c.n_layers):
                fn(l, b.x, b.anc, b.res, b.meta)
        out.append((name, run, lpl * c.n_layers, head, moved))
    return out


def build_buffers(torch, L, inputs, dev, seed=0):
    """The Qwen-32B-shaped 64-layer cache of other_workloads (whole-cache calls)."""
    outl = inputs.outlier_pairs(HKV, seed)
    x = torch.empty((N_PAGES, 128, 256), dtype=torch.bfloat16, device=dev)
    for layer in range(N_LAYERS):
        for t in range(2):
            i = (2 * layer + t) * PER
            x[i:i + PER] = inputs.kv_pages_torch(HKV, N_TOK, inputs.layer_seed(seed, layer, t), outl, dev)
    anc = torch.empty((N_PAGES, 128, 128), dtype=torch.uint8, device=dev)
    res = torch.empty_like(anc)
    meta = torch.empty((N_PAGES, L.META_FLOATS), dtype=torch.float32, device=dev)
    recon = torch.empty((N_PAGES, 128, 256), dtype=torch.bfloat16, device=dev)

    def table(B, layer_of):
        t = torch.empty((B, HKV, NPPH), dtype=torch.int32)
        base = torch.arange(NPPH, dtype=torch.int32)
        for b in range(B):
            lay = layer_of(b)
            for h in range(HKV):
                t[b, h] = 2 * lay * PER + h * NPPH + base
        return t.to(dev)

    pt1 = table(N_LAYERS, lambda b: b)
    pt8 = table(8 * N_LAYERS, lambda b: (b // 8 + b % 8) % N_LAYERS)
    ctx1 = torch.full((N_LAYERS,), N_TOK, dtype=torch.int32, device=dev)
    ctx8 = torch.full((8 * N_LAYERS,), N_TOK, dtype=torch.int32, device=dev)
    q1 = inputs.queries_torch((N_LAYERS, 1, HQ, 128), seed + 1, dev)
    q8 = inputs.queries_torch((8 * N_LAYERS, 1, HQ, 128), seed + 2, dev)
    qv = inputs.queries_torch((N_LAYERS, 8, HQ, 128), seed + 3, dev)

    def ws(B, T):
        n = L.lynx_decode_attn_workspace_size(B, T, HQ, HKV, 128, NPPH)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=dev)

    f32 = dict(dtype=torch.float32, device=dev)
    b = dict(x=x, anc=anc, res=res, meta=meta, recon=recon, pt1=pt1, pt8=pt8, ctx1=ctx1, ctx8=ctx8,
             q1=q1, q8=q8, qv=qv, ws1=ws(N_LAYERS, 1), ws8=ws(8 * N_LAYERS, 1), wsv=ws(N_LAYERS, 8),
             o1=torch.empty((N_LAYERS, 1, HQ, 128), **f32), o8=torch.empty((8 * N_LAYERS, 1, HQ, 128), **f32),
             ov=torch.empty((N_LAYERS, 8, HQ, 128), **f32), ob=torch.empty((N_LAYERS, 1, HQ, 128), **f32))
    b["l1"] = torch.empty((N_LAYERS, 1, HQ), **f32)
    b["l8"] = torch.empty((8 * N_LAYERS, 1, HQ), **f32)
    b["lv"] = torch.empty((N_LAYERS, 8, HQ), **f32)
    b["lb"] = torch.empty((N_LAYERS, 1, HQ), **f32)
    return b


def kernel_list(torch, L, b):
    """(name, callable, launches, headline bytes, moved bytes) of the 64-layer cache's
    whole-cache calls (each call covers all 64 layers)."""
    anc, res, meta = b["anc"], b["res"], b["meta"]
    # K pages of layer l are pages 2l*512 + ..., V pages follow 512 pages later
    kA, vA = anc, anc[PER:]
    kR, vR = res, res[PER:]
    kM, vM = meta, meta[PER:]
    xk, xv = b["x"], b["x"][PER:]
    p = L.Params()
    dec_pages1 = N_LAYERS * HKV * NPPH
    dec_pages8 = 8 * dec_pages1

    def dec_anchor(q, pt, ctx, o, l, ws):
        return lambda: L.lynx_decode_attn(q, kA, None, kM, vA, None, vM, pt, ctx, HKV, p, out=o, lse=l,
                                          workspace=ws)
    return [
        ("encode", lambda: L.lynx_encode_pages(b["x"], p, anc, res, meta), 1,
         N_PAGES * BYTES["encode"][0], N_PAGES * BYTES["encode"][1]),
        ("reconstruct_anchor", lambda: L.lynx_reconstruct(anc, None, meta, p, out=b["recon"]), 1,
         N_PAGES * BYTES["reconstruct_anchor"][0], N_PAGES * BYTES["reconstruct_anchor"][1]),
        ("reconstruct_full", lambda: L.lynx_reconstruct(anc, res, meta, p, out=b["recon"]), 1,
         N_PAGES * BYTES["reconstruct_full"][0], N_PAGES * BYTES["reconstruct_full"][1]),
        ("decode_anchor_b1", dec_anchor(b["q1"], b["pt1"], b["ctx1"], b["o1"], b["l1"], b["ws1"]), 2,
         2 * dec_pages1 * BYTES["decode_anchor"][0], 2 * dec_pages1 * BYTES["decode_anchor"][1]),
        ("decode_anchor_b8", dec_anchor(b["q8"], b["pt8"], b["ctx8"], b["o8"], b["l8"], b["ws8"]), 2,
         2 * dec_pages8 * BYTES["decode_anchor"][0], 2 * dec_pages8 * BYTES["decode_anchor"][1]),
        ("verify_full_t8", lambda: L.lynx_decode_attn(b["qv"], kA, kR, kM, vA, vR, vM, b["pt1"], b["ctx1"], HKV, p,
                                                       causal=True, out=b["ov"], lse=b["lv"], workspace=b["wsv"]),
         2, 2 * dec_pages1 * BYTES["decode_full"][0], 2 * dec_pages1 * BYTES["decode_full"][1]),
        ("decode_bf16_b1", lambda: L.lynx_decode_attn_bf16(b["q1"], xk, xv, b["pt1"], b["ctx1"], HKV, out=b["ob"],
                                                           lse=b["lb"], workspace=b["ws1"]), 2,
         2 * dec_pages1 * BYTES["decode_bf16"][0], 2 * dec_pages1 * BYTES["decode_bf16"][1]),
    ]


def reduce_max(value, world, dist, device=None):
    """Largest value over the ranks (a job's time is its slowest rank's)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(head_bytes_per_rank, world, ms_step):
    """Whole-job GB/s: the bytes all ranks processed in one step over the
    (slowest rank's) step time; every rank runs the same workload (weak scaling)."""
    return world * head_bytes_per_rank / (ms_step * 1e6)


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def profile_traffic(name):
    """DRAM traffic per launch (bytes) of the call `name` from the committed
    capture summary (profiles/traffic.json, written by ``--write-traffic``), if
    the kernel's sources are unchanged since the capture; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get(name)
    if not e:
        return None
    return e["bytes_per_launch"] if e.get("source_sha") == source_sha(e.get("sources", [])) else None


def write_traffic(csv_path, entries):
    """profiles/traffic.json from an ncu CSV of a small one-kernel capture
    (``--metrics dram__bytes_read.sum,dram__bytes_write.sum``).  ``entries``:
    name=kernel_regex:scale pairs; the traffic of a full-size call is the mean
    captured launch's read + write bytes times ``scale`` (the units a full call
    processes over the units the captured launch processed)."""
    import csv
    import re
    rows = list(csv.reader(open(csv_path)))
    hdr = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    cols = rows[hdr]
    ki, mi, vi, ui = (cols.index(k) for k in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit"))
    unit = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    d = json.load(open(TRAFFIC_FILE)) if os.path.exists(TRAFFIC_FILE) else {}
    for spec in entries:
        name, rest = spec.split("=", 1)
        pat, scale = rest.rsplit(":", 1)
        per_launch = {}
        for r in rows[hdr + 1:]:
            if len(r) <= max(ki, mi, vi, ui) or not re.search(pat, r[ki]):
                continue
            if r[mi] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                per_launch.setdefault(r[mi], []).append(float(r[vi].replace(",", "")) * unit.get(r[ui], 1))
        if len(per_launch) != 2:
            raise SystemExit(f"no DRAM rows for {pat} in {csv_path}")
        b = sum(statistics.mean(v) for v in per_launch.values()) * float(scale)
        srcs = KERNEL_SOURCES[name]
        d[name] = {"bytes_per_launch": int(b), "sources": srcs, "source_sha": source_sha(srcs),
                   "capture": os.path.basename(csv_path), "kernel_regex": pat, "scale": float(scale),
                   "launches_captured": len(next(iter(per_launch.values())))}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)


# the CUDA sources each timed call runs (kernel file first, then shared headers)
KERNEL_SOURCES = {
    "encode": ["encode.cu", "lynx_internal.cuh"],
    "reconstruct_anchor": ["reconstruct.cu", "lynx_internal.cuh"],
    "reconstruct_full": ["reconstruct.cu", "lynx_internal.cuh"],
    "decode_anchor_b1": ["decode_draft.cu", "decode_common.cuh", "lynx_internal.cuh"],
    "decode_anchor_b8": ["decode_draft.cu", "decode_common.cuh", "lynx_internal.cuh"],
    "verify_full_t8": ["decode_tc.cu", "decode_common.cuh", "lynx_internal.cuh"],
    "decode_bf16_b1": ["decode_bf16.cu", "decode_common.cuh", "lynx_internal.cuh"],
}


def source_sha(names):
    """sha256 (first 16 hex digits) over the named csrc files, in order; None if one is missing."""
    h = hashlib.sha256()
    for n in names:
        path = os.path.join(ROOT, "progressive_kv_quantization_gb300", "csrc", n)
        if not os.path.exists(path):
            return None
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16] if names else None


def time_kernels(torch, ks, steps, warmup, barrier, stream, clocks=None):
    """Warm-up, then `steps` steps of the calls `ks`, each call bracketed by
    CUDA events on `stream`; returns (per-call mean ms, total ms, clocks)."""
    for _ in range(warmup):
        for k in ks:
            k[1]()
    torch.cuda.synchronize()
    ev = {k[0]: [] for k in ks}
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        for name, fn, _, _, _ in ks:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ev[name].append((e0, e1))
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop() if clocks is not None else None
    per = {name: statistics.mean(e0.elapsed_time(e1) for e0, e1 in v) for name, v in ev.items()}
    return per, t0.elapsed_time(t1), clk


def kernel_table(ks, per_ms, attn_shape, n_keys, G, Hkv):
    """Per-call numbers: time, headline and moved GB/s, fractions of the measured and
    nominal HBM bandwidth; decode calls also their attention FLOP rate."""
    gbps_peak, _ = peaks()
    tflops_peak, _ = tensor_peak()
    kern = {}
    for name, _, launches, head, moved in ks:
        ms = per_ms[name]
        kern[name] = {"ms": round(ms, 4), "GBps_headline": round(head / ms / 1e6, 1),
                      "GBps_moved": round(moved / ms / 1e6, 1),
                      "frac_of_hbm": round(moved / ms / 1e6 / gbps_peak, 3),
                      "frac_of_nominal_hbm": round(moved / ms / 1e6 / NOMINAL_HBM_GBS, 3), "launches": launches,
                      "headline_bytes": head, "moved_bytes": moved}
        if name in attn_shape:
            B, T = attn_shape[name]
            tf = attn_flops(B, T, G, Hkv, n_keys) / ms / 1e9
            kern[name]["attn_tflops"] = round(tf, 1)
            kern[name]["frac_of_bf16_tensor"] = round(tf / tflops_peak, 4)
    return kern


def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist
    from progressive_kv_quantization_gb300 import build as _build
    from progressive_kv_quantization_gb300 import inputs
    from progressive_kv_quantization_gb300 import lynx as L

    _build.build()
    L.load()
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    c = QWEN235B
    b = build_cache(torch, L, inputs, dev, c)
    ks = step_kernels(L, c, b)
    if args.only:
        ks = [k for k in ks if k[0] in args.only.split(",")]
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    per_ms, ms_total, clk = time_kernels(torch, ks, args.steps, args.warmup, barrier, stream, clocks)
    L.lynx_device_status()
    ms_total = reduce_max(ms_total, world, dist if world > 1 else None, dev)
    ms_step = ms_total / args.steps
    gbps_peak, peak_kind = peaks()
    attn_shape = {"decode_anchor_b1": (c.n_layers, 1), "verify_full_t8": (c.n_layers, 8),
                  "decode_bf16_b1": (c.n_layers, 1)}
    kern = kernel_table(ks, per_ms, attn_shape, c.n_tok, c.hq // c.hkv, c.hkv)
    head_total = sum(k[3] for k in ks)
    value = job_value(head_total, world, ms_step)
    dom = max(kern, key=lambda n: kern[n]["ms"])
    roof = {"kernel": dom, "bound": "hbm", "achieved": kern[dom]["GBps_moved"], "peak": gbps_peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": kern[dom]["frac_of_hbm"],
            "traffic": profile_traffic(dom), "source": KERNEL_SOURCES[dom][0]}
    if rank == 0 and not args.no_e2e and "decode_anchor_b1" in kern:
        kern["decode_anchor_b1"]["graph_ms"] = round(_graph_ms(torch, dict((k[0], k[1]) for k in ks)[
            "decode_anchor_b1"], 5), 4)
        kern["decode_anchor_b1"]["graph_frac_of_hbm"] = round(
            kern["decode_anchor_b1"]["moved_bytes"] / kern["decode_anchor_b1"]["graph_ms"] / 1e6 / gbps_peak, 3)
    pm1_file = None
    if rank == 0 and not args.no_cpu_baseline:
        pm1_file = gpu_codes_of_oracle_sample(torch, L, inputs, dev)
    e2e = run_e2e_layers(torch, L, c, b, ks, dev) if rank == 0 and not args.no_e2e else None
    del b
    torch.cuda.empty_cache()
    other = None
    if rank == 0 and not args.no_e2e and not args.only:
        other = run_other_workloads(torch, L, inputs, dev, args)
    if rank != 0:
        return None
    launches = args.steps * sum(k[2] for k in ks)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": c.name, "pages": c.n_pages, "bf16_bytes": c.n_pages * PAGE,
                   "l2": "inputs larger than L2 (25.2e9 B cache; each layer's calls read 0.1-0.3 GB, "
                         "the next layer's pages are not in L2), no flush",
                   "alpha": 100.0, "eps": 1e-6, "parallelism": f"replicas x{world} (one cache per GPU)"},
        "kernels": kern,
        "encode_GBps_bf16_in": kern.get("encode", {}).get("GBps_headline"),
        "encode_frac_of_hbm": kern.get("encode", {}).get("frac_of_hbm"),
        "decode_anchor_GBps_packed": kern.get("decode_anchor_b1", {}).get("GBps_headline"),
        "decode_anchor_frac_of_hbm": kern.get("decode_anchor_b1", {}).get("frac_of_hbm"),
        "roofline": roof,
        "e2e": e2e,
        "other_workloads": other,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        cb = cpu_baseline_subprocess(args.cpu_seconds, pm1_file)
        line["cpu_baseline"] = cb.get("single")
        line["cpu_baseline_all_cores"] = cb.get("all_cores")
        line["code_pm1"] = cb.get("pm1")
    return line


def run_other_workloads(torch, L, inputs, dev, args):
    """The Qwen-32B-shaped 64-layer cache (whole-cache calls, device-timed), the
    split-stream transfer, the token-major encoder and the comparators on it,
    then the decode-attention sweep."""
    b = build_buffers(torch, L, inputs, dev, seed=0)
    ks = kernel_list(torch, L, b)
    per_ms, ms_total, _ = time_kernels(torch, ks, max(3, args.steps // 2), 3, lambda: None,
                                       torch.cuda.current_stream())
    L.lynx_device_status()
    attn_shape = {"decode_anchor_b1": (N_LAYERS, 1), "decode_anchor_b8": (8 * N_LAYERS, 1),
                  "verify_full_t8": (N_LAYERS, 8), "decode_bf16_b1": (N_LAYERS, 1)}
    kern = kernel_table(ks, per_ms, attn_shape, N_TOK, HQ // HKV, HKV)
    steps = max(3, args.steps // 2)
    q32 = {"workload": WORKLOAD, "ms_per_step": round(ms_total / steps, 4),
           "value": round(sum(k[3] for k in ks) / (ms_total / steps) / 1e6, 1), "kernels": kern}
    out = {"qwen32b_step": q32,
           "progressive": run_progressive(torch, L, b, dev),
           "encode_tokens": run_encode_tokens(torch, L, b),
           "comparators": run_comparators(torch, L, b, dev)}
    del b
    torch.cuda.empty_cache()
    out["decode_sweep"] = run_decode_sweep(torch, L, inputs, dev)
    return out


def cpu_baseline_subprocess(seconds, pm1_file=None):
    """The oracle timed in a fresh process on the host cores (single-threaded,
    then one process per core), plus the rounding-edge code comparison of the
    GPU's codes on the oracle's sample (``pm1_file``)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--cpu-only-seconds", str(seconds)]
    if pm1_file:
        cmd += ["--pm1-codes", pm1_file]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"single": {"value": None, "error": r.stderr[-300:]}}
    return json.loads(r.stdout.strip().splitlines()[-1])["cpu_legs"]


def _host_mem_available():
    """MemAvailable of the host in bytes (None where /proc/meminfo is absent)."""
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) * 1024
    except OSError:
        pass
    return None


def run_e2e_layers(torch, L, c: Cache, b, ks, dev, n_chunks=12, steps=5):
    """The step through host buffers: every step copies the BF16 cache and the
    queries in from pinned host memory and reads every call's results back (the
    encoded planes and metadata, and the three decode calls' outputs and
    log-sum-exps), through the same per-layer calls as the device-timed step.

    Layer-streamed in chunks of layers: chunk k's BF16 pages and queries are
    copied in on an upload stream; once they have landed, the compute stream
    runs the six calls on each of its layers, and a readback stream returns the
    chunk's planes, metadata and outputs.  Later chunks' uploads overlap earlier
    chunks' compute.  Readbacks start once every upload of the step has finished
    (on this host link, transfers in both directions at once were measured to
    drop at times from 342 GB/s to ~130 GB/s).  The next step's uploads wait
    until the previous step no longer reads the BF16 cache.  Each step is timed
    on its own; the median is reported (the host link is shared)."""
    host_need = c.n_pages * (PAGE + 2 * PLANE + META) + (2 << 30)
    avail = _host_mem_available()
    if avail is not None and avail < 2 * host_need:
        return {"value": None, "skipped": f"host MemAvailable {avail / 1e9:.0f} GB < 2 x {host_need / 1e9:.0f} GB "
                                          "of pinned buffers the step needs"}
    calls = layer_calls(L, c, b)
    pin = dict(pin_memory=True)
    host_x = torch.empty(b.x.shape, dtype=torch.bfloat16, **pin)
    host_x.copy_(b.x)
    h_q = {k: torch.empty(getattr(b, k).shape, dtype=torch.bfloat16, **pin).copy_(getattr(b, k)) for k in ("q1", "qv")}
    outs = ("anc", "res", "meta", "oa", "la", "ob", "lb", "ov", "lv")
    h_out = {k: torch.empty(getattr(b, k).shape, dtype=getattr(b, k).dtype, **pin) for k in outs}
    h2d = host_x.numel() * 2 + sum(v.numel() * v.element_size() for v in h_q.values())
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    bounds = [round(k * c.n_layers / n_chunks) for k in range(n_chunks + 1)]
    chunks = [(bounds[k], bounds[k + 1]) for k in range(n_chunks) if bounds[k + 1] > bounds[k]]
    comp, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_cmp = [torch.cuda.Event() for _ in chunks]
    ev_free = torch.cuda.Event()
    ev_free.record(comp)

    def one():
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_free)           # the previous step no longer reads the cache
            for k, (l0, l1) in enumerate(chunks):
                pg = slice(l0 * c.per_layer, l1 * c.per_layer)
                b.x[pg].copy_(host_x[pg], non_blocking=True)
                b.q1[l0:l1].copy_(h_q["q1"][l0:l1], non_blocking=True)
                b.qv[l0:l1].copy_(h_q["qv"][l0:l1], non_blocking=True)
                ev_in[k].record(s_in)
        for k, (l0, l1) in enumerate(chunks):
            comp.wait_event(ev_in[k])
            with torch.cuda.stream(comp):
                for l in range(l0, l1):
                    for _, fn, _, _, _ in calls:
                        fn(l, b.x, b.anc, b.res, b.meta)
            ev_cmp[k].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_in[-1])    # after the step's last upload
                s_out.wait_event(ev_cmp[k])
                pg = slice(l0 * c.per_layer, l1 * c.per_layer)
                for name in ("anc", "res", "meta"):
                    h_out[name][pg].copy_(getattr(b, name)[pg], non_blocking=True)
                for name in ("oa", "la", "ob", "lb", "ov", "lv"):
                    h_out[name][l0:l1].copy_(getattr(b, name)[l0:l1], non_blocking=True)
        ev_free.record(comp)
        comp.wait_stream(s_out)                # results are on the host when the step ends

    one()
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    marks[0].record(comp)
    s_in.wait_event(marks[0])
    for k in range(steps):
        one()
        marks[k + 1].record(comp)
    torch.cuda.synchronize()
    L.lynx_device_status()
    per_step = sorted(marks[k].elapsed_time(marks[k + 1]) for k in range(steps))
    ms = per_step[len(per_step) // 2]
    head_total = sum(k[3] for k in ks)
    same = all(bool(torch.equal(h_out[n], getattr(b, n).cpu())) for n in ("oa", "ob", "ov"))
    del host_x, h_out
    return {"value": round(head_total / (ms * 1e6), 1), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "statistic": "median step", "step_ms": [round(x, 3) for x in per_step], "chunks": len(chunks),
            "outputs_read_back_match_device": same}


def gpu_codes_of_oracle_sample(torch, L, inputs, dev):
    """Encodes, on the GPU, the BF16 pages of the CPU oracle's sample (the same
    seeded generator) and saves the planes to a temporary file, for the oracle
    leg to compare its own codes with (the rounding-edge +-1 code fraction)."""
    import numpy as np
    kb, vb = oracle_sample_pages()
    x = torch.from_numpy(np.concatenate([kb, vb]).view(np.int16)).view(torch.bfloat16).to(dev)
    a, r, _ = L.lynx_encode_pages(x)
    torch.cuda.synchronize()
    fd, path = tempfile.mkstemp(prefix="lynx_pm1_", suffix=".npz")
    os.close(fd)
    np.savez(path, anchor=a.cpu().numpy(), residual=r.cpu().numpy())
    return path


def run_progressive(torch, L, b, dev, reps=3):
    """The paper's split-stream transfer on one box (paper §4.2, Stream SerDes):
    the 64-layer cache is encoded layer by layer on a compute stream while
    each encoded layer goes device -> pinned host -> device, its Anchor plane and
    metadata on high-priority streams and its Residual plane on low-priority
    ones (progressive.ProgressiveTransfer.encode_and_send).  Reported: the time
    from the first encode until every layer's encode has finished, until every
    Anchor has landed (draft decoding can run everywhere) and until every
    Residual has landed (verification can run everywhere), against the same
    round trip of the BF16 cache; also the transfer alone of the already
    encoded cache; medians of ``reps`` runs (the host link is shared)."""
    from progressive_kv_quantization_gb300.progressive import ProgressiveTransfer
    layers = [(2 * l * PER, 2 * (l + 1) * PER) for l in range(N_LAYERS)]
    src = (b["anc"], b["res"], b["meta"])
    dst = tuple(torch.empty_like(t) for t in src)
    tr = ProgressiveTransfer(layers, dev)
    h_x = torch.empty(b["x"].shape, dtype=torch.bfloat16, pin_memory=True)
    d_x = torch.empty_like(b["x"])
    s_o, s_i, comp = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    staged = [torch.cuda.Event() for _ in layers]
    enc, anchor, full, send_a, send_f, bf16 = [], [], [], [], [], []
    for _ in range(reps + 1):
        torch.cuda.synchronize()
        tr.encode_and_send(b["x"], src, dst, stream=comp)
        a, f = tr.times_ms()
        enc.append(tr.start.elapsed_time(tr.encoded[-1]))
        anchor.append(a)
        full.append(f)
        torch.cuda.synchronize()
        tr.send(src, dst)
        a, f = tr.times_ms()
        send_a.append(a)
        send_f.append(f)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s_o):                     # the BF16 cache along the same two-stream path
            e0.record(s_o)
            for (lo, hi), ev in zip(layers, staged):
                h_x[lo:hi].copy_(b["x"][lo:hi], non_blocking=True)
                ev.record(s_o)
        with torch.cuda.stream(s_i):
            s_i.wait_event(e0)
            for (lo, hi), ev in zip(layers, staged):
                s_i.wait_event(ev)
                d_x[lo:hi].copy_(h_x[lo:hi], non_blocking=True)
            e1.record(s_i)
        e1.synchronize()
        bf16.append(e0.elapsed_time(e1))
    med = lambda v: round(statistics.median(v[1:]), 3)    # the first run warms the path
    exact = all(bool(torch.equal(x, y)) for x, y in zip(src, dst)) and bool(torch.equal(d_x, b["x"]))
    return {"encode_done_ms": med(enc), "anchor_ready_ms": med(anchor), "full_ready_ms": med(full),
            "bf16_ms": med(bf16), "send_only": {"anchor_ready_ms": med(send_a), "full_ready_ms": med(send_f)},
            "anchor_bytes": int(src[0].numel() + src[2].numel() * 4), "residual_bytes": int(src[1].numel()),
            "bf16_bytes": int(b["x"].numel() * 2),
            "path": "encode per layer on a compute stream; each layer device -> pinned host -> device, "
                    "Anchor + metadata on high-priority streams, Residual on low-priority streams",
            "bytes_unchanged": exact, "statistic": f"median of {reps}"}


def run_encode_tokens(torch, L, b, reps=5):
    """lynx_encode_tokens on the same cache held token-major, the layout of paged
    attention: the 64 layers' K and V become one [16384 tokens][1024 x 128] BF16
    tensor (row t = token t of every layer, K/V and KV head), so one call writes
    exactly the pages lynx_encode_pages writes (checked byte for byte).  Median of
    ``reps`` CUDA-event timings; the 4.29e9-byte input is larger than L2."""
    n_heads = N_PAGES // NPPH                          # layers x {K, V} x KV heads
    x_tm = b["x"].view(n_heads, NPPH, 128, 256).permute(1, 3, 0, 2).reshape(N_TOK, n_heads * 128).contiguous()
    anc, res, meta = torch.empty_like(b["anc"]), torch.empty_like(b["res"]), torch.empty_like(b["meta"])
    p = L.Params()
    times = []
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        L.lynx_encode_tokens(x_tm, n_heads, p, anc, res, meta)
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times[1:])
    same = bool(torch.equal(anc, b["anc"])) and bool(torch.equal(res, b["res"])) and bool(torch.equal(meta, b["meta"]))
    gbps_peak, _ = peaks()
    head, moved = N_PAGES * BYTES["encode"][0], N_PAGES * BYTES["encode"][1]
    del x_tm
    return {"ms": round(ms, 4), "GBps_headline": round(head / ms / 1e6, 1), "GBps_moved": round(moved / ms / 1e6, 1),
            "frac_of_hbm": round(moved / ms / 1e6 / gbps_peak, 3), "identical_to_page_encode": same,
            "layout": f"[{N_TOK} tokens][{n_heads} x 128] BF16 (layer x K/V x KV head per row)",
            "statistic": f"median of {reps}"}


def run_comparators(torch, L, b, dev, reps=3):
    """The Table-3 analogue on the benchmark's synthetic cache: for Lynx (full
    codes; anchor only, the draft), Lynx-INT8, Lynx-INT4 and uniform INT8 / INT4,
    the KV vNMSE (mean over token vectors -- one head's 128 channels at one
    token -- of ||x_hat - x||^2 / ||x||^2, from float32 reconstructions) and the
    attention vNMSE (the B = 64, T = 1 decode's output rows against the same
    decode over the BF16 pages; uniform codes and the other split widths'
    Anchors through their BF16 reconstruction), with each variant's encode time
    (median of ``reps`` CUDA-event timings) and its bytes per KV value; then the
    Anchor alone of the split stream at widths 2, 3, 5 and 6 bits."""
    p = L.Params()
    x = b["x"]
    n = x.shape[0]
    chunk = 8192
    gbps_peak, _ = peaks()

    def timed(fn):
        ts = []
        for _ in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts[1:])

    def kv_vnmse(recon_f32):   # recon_f32(lo, hi, out) fills out with pages lo..hi in float32
        tot, cnt = 0.0, 0
        buf = torch.empty((chunk, 128, 256), dtype=torch.float32, device=dev)
        for lo in range(0, n, chunk):
            hi = min(lo + chunk, n)
            recon_f32(lo, hi, buf[:hi - lo])
            xf = x[lo:hi].float()
            d = (buf[:hi - lo] - xf).pow(2).sum(dim=1) / xf.pow(2).sum(dim=1).clamp_min(1e-30)
            tot += float(d.double().sum())
            cnt += d.numel()
        return tot / cnt

    q, pt, ctx, ws = b["q1"], b["pt1"], b["ctx1"], b["ws1"]
    kA, vA, kR, vR, kM, vM = b["anc"], b["anc"][PER:], b["res"], b["res"][PER:], b["meta"], b["meta"][PER:]
    o_ref, _ = L.lynx_decode_attn_bf16(q, x, x[PER:], pt, ctx, HKV, workspace=ws)
    o_ref = o_ref.clone()

    def attn_vnmse(o):
        a, r = o.double().reshape(-1, 128), o_ref.double().reshape(-1, 128)
        return float(((a - r).pow(2).sum(dim=1) / r.pow(2).sum(dim=1)).mean())

    rows = {}
    # Lynx split stream (the step's encode output): full codes and the Anchor alone
    t_enc = timed(lambda: L.lynx_encode_pages(x, p, kA, kR, kM))
    o_buf = torch.empty_like(o_ref)
    l_buf = torch.empty(o_ref.shape[:-1], dtype=torch.float32, device=dev)
    full_o, _ = L.lynx_decode_attn(q, kA, kR, kM, vA, vR, vM, pt, ctx, HKV, p, workspace=ws)
    t_full = timed(lambda: L.lynx_decode_attn(q, kA, kR, kM, vA, vR, vM, pt, ctx, HKV, p, out=o_buf, lse=l_buf,
                                              workspace=ws))
    rows["lynx_full"] = {"bytes_per_value": 1.0 + 9216 / 32768, "encode_ms": round(t_enc, 4),
                         "decode_ms": round(t_full, 4),
                         "kv_vnmse": kv_vnmse(lambda lo, hi, o: L.lynx_reconstruct(
                             kA[lo:hi], kR[lo:hi], kM[lo:hi], p, out=o, out_dtype=torch.float32)),
                         "attn_vnmse": attn_vnmse(full_o)}
    anc_o, _ = L.lynx_decode_attn(q, kA, None, kM, vA, None, vM, pt, ctx, HKV, p, workspace=ws)
    t_anc = timed(lambda: L.lynx_decode_attn(q, kA, None, kM, vA, None, vM, pt, ctx, HKV, p, out=o_buf, lse=l_buf,
                                             workspace=ws))
    rows["lynx_anchor"] = {"bytes_per_value": 0.5 + 9216 / 32768, "encode_ms": round(t_enc, 4),
                           "decode_ms": round(t_anc, 4),
                           "kv_vnmse": kv_vnmse(lambda lo, hi, o: L.lynx_reconstruct(
                               kA[lo:hi], None, kM[lo:hi], p, out=o, out_dtype=torch.float32)),
                           "attn_vnmse": attn_vnmse(anc_o)}
    for name in ("lynx_int8", "lynx_int4", "uniform_int8", "uniform_int4"):
        _, cb, mf = L.VARIANTS[name]
        codes = torch.empty((n, cb), dtype=torch.uint8, device=dev)
        meta = torch.empty((n, mf), dtype=torch.float32, device=dev)
        t = timed(lambda: L.lynx_encode_variant(x, name, p, codes, meta))
        ent = {"bytes_per_value": (cb + 4 * mf) / 32768, "encode_ms": round(t, 4),
               "encode_frac_of_hbm": round((n * (PAGE + cb + 4 * mf)) / t / 1e6 / gbps_peak, 3),
               "kv_vnmse": kv_vnmse(lambda lo, hi, o: L.lynx_reconstruct_variant(
                   codes[lo:hi], meta[lo:hi], name, p, out=o, out_dtype=torch.float32))}
        if name == "lynx_int4":
            o4, _ = L.lynx_decode_attn_int4(q, codes, meta, codes[PER:], meta[PER:], pt, ctx, HKV, p, workspace=ws)
            ent["attn_vnmse"] = attn_vnmse(o4)
            ent["decode_ms"] = round(timed(lambda: L.lynx_decode_attn_int4(
                q, codes, meta, codes[PER:], meta[PER:], pt, ctx, HKV, p, out=o_buf, lse=l_buf, workspace=ws)), 4)
        elif name.startswith("uniform"):
            bits = 8 if name == "uniform_int8" else 4
            if bits == 8:
                c_lo, c_hi = L.lynx_split_nibbles(codes.view(n, 128, 256))
                kh, vh = c_hi, c_hi[PER:]
            else:
                c_lo, kh, vh = codes.view(n, 128, 128), None, None
            call = lambda out=None, lse=None: L.lynx_decode_attn_uniform(
                q, bits, c_lo, kh, meta, c_lo[PER:], vh, meta[PER:], pt, ctx, HKV, out=out, lse=lse, workspace=ws)
            ou, _ = call()
            ent["attn_vnmse"] = attn_vnmse(ou)
            ent["decode_ms"] = round(timed(lambda: call(o_buf, l_buf)), 4)
            del c_lo, kh, vh
        else:
            rec = L.lynx_reconstruct_variant(codes, meta, name, p)
            o8, _ = L.lynx_decode_attn_bf16(q, rec, rec[PER:], pt, ctx, HKV, workspace=ws)
            ent["attn_vnmse"] = attn_vnmse(o8)
            del rec
        rows[name] = ent
        del codes, meta
    # the split stream at other widths: the draft (Anchor-only) accuracy against its size
    for A in (2, 3, 5, 6):
        R = 8 - A
        an = torch.empty((n, 128, 32 * A), dtype=torch.uint8, device=dev)
        rs = torch.empty((n, 128, 32 * R), dtype=torch.uint8, device=dev)
        mt = torch.empty_like(b["meta"])
        t = timed(lambda: L.lynx_encode_split(x, A, p, an, rs, mt))
        rec = L.lynx_reconstruct_split(an, None, mt, A, p)
        oa, _ = L.lynx_decode_attn_bf16(q, rec, rec[PER:], pt, ctx, HKV, workspace=ws)
        rows[f"lynx_split_{A}+{R}_anchor"] = {
            "bytes_per_value": (32 * A * 128 + 9216) / 32768, "encode_ms": round(t, 4),
            "kv_vnmse": kv_vnmse(lambda lo, hi, o: L.lynx_reconstruct_split(
                an[lo:hi], None, mt[lo:hi], A, p, out=o, out_dtype=torch.float32)),
            "attn_vnmse": attn_vnmse(oa)}
        del an, rs, mt, rec
    for r in rows.values():
        r["kv_vnmse"] = float(f"{r['kv_vnmse']:.4g}")
        r["attn_vnmse"] = float(f"{r['attn_vnmse']:.4g}")
    return {"rows": rows, "attention": "B=64, T=1 decode vs the same decode over the BF16 pages",
            "decode": "decode_ms: the same B=64, T=1 decode through the fused kernel for that format "
                      "(Lynx-INT8 values are Lynx's full codes)",
            "kv": "token vectors of the 64-layer cache, float32 reconstructions"}


def _median_ms(torch, fn, reps):
    ts = []
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts[1:])


def _graph_ms(torch, fn, reps):
    """Median over ``reps`` replays of a CUDA graph holding the launches of one
    ``fn()`` call (captured after an eager warm-up call), each replay bracketed
    by CUDA events: the GPU time of the call without the host-side cost of the
    Python binding, as a decode loop that replays a captured graph sees it."""
    fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    del g
    return statistics.median(ts)


def _graph_loop_ms(torch, fn, n_calls=100, reps=3):
    """Per-call GPU time of ``n_calls`` back-to-back calls captured in one CUDA
    graph (median of ``reps`` replays / n_calls): a decode loop without the
    per-replay launch of the graph itself."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n_calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / n_calls)
    del g
    return statistics.median(ts)


def run_decode_sweep(torch, L, inputs, dev, reps=5):
    """The decode-attention sweep workload: 8 KV heads x 128, 32 query heads,
    contexts 4K / 16K / 128K tokens x batch 1 / 16 x T = 1 / 8 / 32 (causal for
    T > 1), over Anchor-only planes, Anchor + Residual planes and BF16 pages;
    every sequence has its own pages (16 x 128K-token caches, 131,072 pages).
    GB/s = KV bytes read (packed planes + metadata, or BF16) / time; median of
    ``reps`` CUDA-event timings of a CUDA-graph replay of the call ("ms") and of
    the eager Python call ("eager_ms", which adds the binding's host-side time
    wherever the GPU finishes before the host has issued the launches); calls
    under 0.1 ms also as a graph of 100 back-to-back calls ("loop_ms" per call,
    the working set staying in L2 from call to call)."""
    Hkv, Hq, n_max, B_max = 8, 32, 131072, 16
    npph = n_max // 256
    outl = inputs.outlier_pairs(Hkv, 5)
    per_seq = 2 * Hkv * npph                        # K then V pages of one sequence
    n = B_max * per_seq
    x = torch.empty((n, 128, 256), dtype=torch.bfloat16, device=dev)
    for b in range(B_max):
        for t in range(2):
            i = b * per_seq + t * Hkv * npph
            x[i:i + Hkv * npph] = inputs.kv_pages_torch(Hkv, n_max, 900 + 2 * b + t, outl, dev)
    a, r, m = L.lynx_encode_pages(x)
    gbps_peak, _ = peaks()
    tflops_peak, _ = tensor_peak()
    rows = []
    for ctx_len in (4096, 16384, 131072):
        mp = ctx_len // 256
        for B in (1, 16):
            pt = torch.tensor([[[b * per_seq + h * npph + j for j in range(mp)] for h in range(Hkv)]
                               for b in range(B)], dtype=torch.int32, device=dev)
            ctx = torch.full((B,), ctx_len, dtype=torch.int32, device=dev)
            for T in (1, 8, 32):
                q = inputs.queries_torch((B, T, Hq, 128), 50 + T, dev)
                nb = L.lynx_decode_attn_workspace_size(B, T, Hq, Hkv, 128, mp)
                ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
                o = torch.empty((B, T, Hq, 128), dtype=torch.float32, device=dev)
                l_ = torch.empty((B, T, Hq), dtype=torch.float32, device=dev)
                causal = T > 1
                vo = Hkv * npph
                calls = {
                    "anchor": (lambda: L.lynx_decode_attn(q, a, None, m, a[vo:], None, m[vo:], pt, ctx, Hkv,
                                                          causal=causal, out=o, lse=l_, workspace=ws), 25600),
                    "full": (lambda: L.lynx_decode_attn(q, a, r, m, a[vo:], r[vo:], m[vo:], pt, ctx, Hkv,
                                                        causal=causal, out=o, lse=l_, workspace=ws), 41984),
                    "bf16": (lambda: L.lynx_decode_attn_bf16(q, x, x[vo:], pt, ctx, Hkv, causal=causal, out=o,
                                                             lse=l_, workspace=ws), 65536),
                }
                for mode, (fn, page_bytes) in calls.items():
                    eager = _median_ms(torch, fn, reps)
                    ms = _graph_ms(torch, fn, reps)
                    moved = 2 * B * Hkv * mp * page_bytes
                    tf = attn_flops(B, T, Hq // Hkv, Hkv, ctx_len) / ms / 1e9
                    row = {"ctx": ctx_len, "B": B, "T": T, "kv": mode, "ms": round(ms, 4),
                           "eager_ms": round(eager, 4), "GBps": round(moved / ms / 1e6, 1),
                           "frac_of_hbm": round(moved / ms / 1e6 / gbps_peak, 3),
                           "attn_tflops": round(tf, 1), "frac_of_bf16_tensor": round(tf / tflops_peak, 4)}
                    if ms < 0.1:   # small calls: also as a loop of 100 captured calls
                        row["loop_ms"] = round(_graph_loop_ms(torch, fn), 4)
                    rows.append(row)
    del x, a, r, m
    return {"rows": rows, "statistic": f"median of {reps}; ms = CUDA-graph replay, eager_ms = Python call",
            "tensor_roof": "attn_tflops = 4 * 128 * T * G FLOPs per key per KV head per sequence / ms, against the "
                           "measured dense bf16 peak (MEASURED_PEAKS bf16_tflops)",
            "l2": "KV read per call 0.1-21 GB: the 4K contexts at B = 1 (25-65 MB) fit in L2"}


# ------------------------------------------------------------------ oracle arm

SAMPLE_TOKENS = 32768      # tokens of the oracle's sample: one KV head of one layer, 128 pages of K and of V


def oracle_sample_pages(index=0, n_tok=SAMPLE_TOKENS):
    """BF16 pages (K, V) of the oracle's sample ``index``: one KV head of the
    Qwen3-235B-shaped cache's distribution (head 0's outlier channels, layer
    ``index``'s seeds), n_tok tokens."""
    from progressive_kv_quantization_gb300 import inputs
    c = QWEN235B
    outl = inputs.outlier_pairs(c.hkv, c.seed)[:1]
    kb = inputs.kv_pages_np(1, n_tok, inputs.layer_seed(c.seed, index, 0), outl)
    vb = inputs.kv_pages_np(1, n_tok, inputs.layer_seed(c.seed, index, 1), outl)
    return kb, vb


def oracle_sample_step(index=0, n_tok=SAMPLE_TOKENS, pages=None, stages=None):
    """One bounded sample of the step for the CPU oracle: one KV head of one
    layer (n_tok tokens of K and V) through the step's six operations: encode,
    both reconstructs, the B=1 anchor draft decode, the T=8 causal verification
    over the full codes and the BF16 decode, with G = 4 query heads.  Returns
    (headline bytes, seconds of oracle work); input generation is not timed.
    ``stages``: a dict that receives the oracle's encode stages (for the code
    comparison)."""
    import numpy as np

    from oracle import attention as at
    from oracle import lynx_oracle as lo
    from progressive_kv_quantization_gb300 import inputs

    c = QWEN235B
    eps = np.float32(1e-6)
    kb, vb = pages if pages is not None else oracle_sample_pages(index, n_tok)
    G = c.hq // c.hkv
    npph = n_tok // 256
    q1 = inputs.queries_np((1, 1, G, 128), 3 + index)
    qv = inputs.queries_np((1, 8, G, 128), 5 + index)
    table = np.arange(npph, dtype=np.int32)[None, None]
    ctx = np.array([n_tok])
    scale = 1 / math.sqrt(128)
    t0 = time.perf_counter()
    ka, kr, km, kst = lo.encode_pages(kb, 100.0, eps, return_stages=True)
    va, vr, vm, vst = lo.encode_pages(vb, 100.0, eps, return_stages=True)
    kd_a = lo.reconstruct(ka, None, km, 100.0, eps)
    vd_a = lo.reconstruct(va, None, vm, 100.0, eps)
    kd_f = lo.reconstruct(ka, kr, km, 100.0, eps)
    vd_f = lo.reconstruct(va, vr, vm, 100.0, eps)
    qf = lambda q: lo.bf16_to_f32(q).astype(np.float64)
    at.decode_attention(qf(q1), lambda ids: (kd_a[ids], vd_a[ids]), table, ctx, 1, scale, False)
    at.decode_attention(qf(qv), lambda ids: (kd_f[ids], vd_f[ids]), table, ctx, 1, scale, True)
    at.decode_attention(qf(q1), lambda ids: (lo.bf16_to_f32(kb[ids]).astype(np.float64),
                                             lo.bf16_to_f32(vb[ids]).astype(np.float64)), table, ctx, 1, scale, False)
    sec = time.perf_counter() - t0
    if stages is not None:
        stages.update(anchor=np.concatenate([ka, va]), residual=np.concatenate([kr, vr]),
                      Y=np.concatenate([kst.Y, vst.Y]))
    n = 2 * npph
    head = n * (BYTES["encode"][0] + BYTES["reconstruct_anchor"][0] + BYTES["reconstruct_full"][0]
                + BYTES["decode_anchor"][0] + BYTES["decode_full"][0] + BYTES["decode_bf16"][0])
    return head, sec


def _sample_desc(n, n_tok, cores):
    return (f"{n} x (one KV head of one layer of the Qwen3-235B-shaped cache: {n_tok // 256} pages of K and of V, "
            f"{n_tok} tokens, 4 query heads) through encode, both reconstructs, B=1 anchor draft decode, T=8 "
            f"full-code verification and BF16 decode; numpy, {cores} process(es) of 1 thread")


def run_reference_sample(seconds=15.0, steps=None, warmup=0, n_tok=SAMPLE_TOKENS, stages=None):
    """Times the oracle on repeated bounded samples in this process (one BLAS /
    OpenMP thread); ``stages`` receives the first sample's encode stages."""
    pages = oracle_sample_pages(0, n_tok)
    for _ in range(warmup):
        oracle_sample_step(0, n_tok, pages)
    tot_b, tot_s, n = 0, 0.0, 0
    while (steps is None and (tot_s < seconds or n == 0)) or (steps is not None and n < steps):
        bb, ss = oracle_sample_step(0, n_tok, pages, stages=stages if n == 0 else None)
        tot_b += bb
        tot_s += ss
        n += 1
    v = tot_b / tot_s / 1e9
    return {"value": v, "seconds": tot_s, "samples": n,
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": _sample_desc(n, n_tok, 1), "seconds": round(tot_s, 2)}}


def _all_cores_worker(index, n_tok, barrier, queue):
    pages = oracle_sample_pages(index, n_tok)
    barrier.wait()
    queue.put(oracle_sample_step(index, n_tok, pages))


def run_reference_all_cores(n_tok=SAMPLE_TOKENS, procs=None):
    """The oracle on every host core at once: one process per core, each running
    its own sample (a different layer's seeds) after a common barrier; value =
    all samples' bytes / the slowest process's oracle time."""
    import multiprocessing as mp
    procs = procs or os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier, queue = ctx.Barrier(procs), ctx.Queue()
    ps = [ctx.Process(target=_all_cores_worker, args=(i, n_tok, barrier, queue)) for i in range(procs)]
    for p in ps:
        p.start()
    res = [queue.get(timeout=900) for _ in ps]
    for p in ps:
        p.join()
    tot_b = sum(r[0] for r in res)
    sec = max(r[1] for r in res)
    return {"value": round(tot_b / sec / 1e9, 4), "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": _sample_desc(procs, n_tok, procs), "seconds": round(sec, 2)}


def pm1_fraction(gpu_file, st):
    """The rounding-edge comparison of the GPU's codes with the oracle's on the
    sample's pages (``st``: the oracle's encode stages of that sample): the
    fraction of codes that differ, and whether every difference is a +-1 step
    where the oracle's float64 Y lies within 1e-5 of a rounding edge (the bar:
    bit-exact codes except there, fraction < 1e-4)."""
    import numpy as np

    from oracle import lynx_oracle as lo
    g = np.load(gpu_file)

    def codes(a, r):
        qa = lo.unpack_nibbles(a).astype(np.int32)
        qr = lo.unpack_nibbles(r).astype(np.int32)
        S = np.where(qa < 0, -1, 1)
        I = 16 * np.where(S > 0, qa, -qa - 1) + 7 - qr
        return S, I

    sg, ig = codes(g["anchor"], g["residual"])
    so, io = codes(st["anchor"], st["residual"])
    diff = (sg != so) | (ig != io)
    Y = st["Y"]
    edge = np.abs(Y - np.floor(Y) - 0.5) < 1e-5
    ok = bool(np.all(edge[diff]) and np.all(np.abs(ig - io)[diff] <= 1))
    return {"fraction": float(diff.mean()), "codes_compared": int(diff.size), "differing": int(diff.sum()),
            "all_at_rounding_edges": ok, "bar": "fraction < 1e-4, differences only +-1 within 1e-5 of an edge",
            "sample": f"{diff.size // 32768} pages of the oracle sample (K and V of one KV head)"}


def main():
    if "--impl" in sys.argv and "reference" in sys.argv:
        # the oracle runs single-threaded: fix the thread count before numpy loads
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["lynx", "reference"], default="lynx")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-only-seconds", type=float, default=None)
    ap.add_argument("--pm1-codes", default=None, help="GPU codes of the oracle sample (internal)")
    ap.add_argument("--layers", type=int, default=94, help="layers of the main cache (94 = the workload)")
    ap.add_argument("--only", default="", help="comma-separated call names to run (profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip e2e and the other workloads (profiling)")
    ap.add_argument("--write-traffic", nargs="+", default=None,
                    help="CSV name=kernel_regex:scale ...: write profiles/traffic.json from an ncu capture")
    args = ap.parse_args()
    if args.write_traffic:
        write_traffic(args.write_traffic[0], args.write_traffic[1:])
        return
    if args.layers != QWEN235B.n_layers:
        set_layers(args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        # the CPU oracle: rank 0 only; other ranks exit without work
        if rank != 0:
            return
        if args.cpu_only_seconds is not None:
            # the GPU arm's cpu_baseline leg: single-threaded, all cores, code comparison
            st = {}
            r = run_reference_sample(seconds=args.cpu_only_seconds, stages=st)
            legs = {"single": r["cpu_baseline"], "all_cores": run_reference_all_cores()}
            if args.pm1_codes:
                try:
                    legs["pm1"] = pm1_fraction(args.pm1_codes, st)
                finally:
                    os.unlink(args.pm1_codes)
            print(json.dumps({"cpu_legs": legs}), flush=True)
            return
        # the reference arm: one sample per step (~8 s), so that --steps K --warmup W ends in minutes
        r = run_reference_sample(steps=args.steps, warmup=args.warmup)
        line = {"metric": METRIC, "value": round(r["value"], 4), "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1000 * r["seconds"] / max(r["samples"], 1), 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference",
                "config": {"workload": QWEN235B.name,
                           "sample": "one KV head of one layer, 128 pages of K and V, per step (CPU oracle)"},
                "cpu_baseline": r["cpu_baseline"],
                "e2e": {"value": round(r["value"], 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    line = run_gpu(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
