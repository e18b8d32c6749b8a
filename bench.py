"""Benchmark of the Lynx hot path on one GB300 (or N, one process per GPU).

One step = one pass of the whole hot path over a Qwen-32B-shaped KV cache
(64 layers x 8 KV heads x 128 channels x 16,384 tokens, K and V: 65,536 pages,
4.29e9 BF16 bytes, synthetic, seeded):

  encode            lynx_encode_pages over all 65,536 pages (one launch)
  reconstruct_anchor / reconstruct_full   lynx_reconstruct, BF16 out
  decode_anchor_b1  1-token draft decode, 32 query heads (GQA 4:1), one
                    sequence per layer (B = 64)
  decode_anchor_b8  the same with 8 sequences per layer (B = 512; sequence b of
                    layer l reads layer (l + b) mod 64)
  verify_full_t8    8-token causal verification over the full codes (B = 64)
  decode_bf16_b1    the BF16-page baseline kernel, B = 64, 1 token

value = sum over the step's kernels of each kernel's headline bytes (encode:
BF16 bytes in; reconstruct and decode: packed KV bytes read; BF16 baseline:
BF16 KV bytes read) / step time, in GB/s.  The per-kernel numbers, including
the two the metric names (encode GB/s of BF16 in, anchor decode GB/s of packed
KV read), are under "kernels".

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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV encode GB/s (BF16 in) and Anchor-KV decode-attn GB/s, % of GB300 HBM peak"
UNIT = "GB/s"
WORKLOAD = ("Qwen-32B-shaped KV cache: 64 layers x 8 KV heads x 128 x 16384 tokens, K and V "
            "(65536 pages of 128x256 BF16, 4.29e9 B); decode B=1 and B=8 (anchor), T=8 verify (full), "
            "32 query heads")
N_LAYERS, HKV, HQ, N_TOK = 64, 8, 32, 16384
NPPH = N_TOK // 256                 # pages per head
PER = HKV * NPPH                    # pages per tensor per layer (512)
N_PAGES = 2 * N_LAYERS * PER        # 65536
E2E_CHUNKS = 8                       # page chunks of the end-to-end step's copy pipeline


def set_layers(n):
    """Smaller caches (fewer layers) for profiling captures."""
    global N_LAYERS, N_PAGES
    N_LAYERS = n
    N_PAGES = 2 * N_LAYERS * PER
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

def build_buffers(torch, L, inputs, dev, seed=0):
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

    b = dict(x=x, anc=anc, res=res, meta=meta, recon=recon, pt1=pt1, pt8=pt8, ctx1=ctx1, ctx8=ctx8,
             q1=q1, q8=q8, qv=qv, ws1=ws(N_LAYERS, 1), ws8=ws(8 * N_LAYERS, 1), wsv=ws(N_LAYERS, 8),
             o1=torch.empty((N_LAYERS, 1, HQ, 128), dtype=torch.float32, device=dev),
             o8=torch.empty((8 * N_LAYERS, 1, HQ, 128), dtype=torch.float32, device=dev),
             ov=torch.empty((N_LAYERS, 8, HQ, 128), dtype=torch.float32, device=dev))
    b["l1"] = torch.empty((N_LAYERS, 1, HQ), dtype=torch.float32, device=dev)
    b["l8"] = torch.empty((8 * N_LAYERS, 1, HQ), dtype=torch.float32, device=dev)
    b["lv"] = torch.empty((N_LAYERS, 8, HQ), dtype=torch.float32, device=dev)
    return b


def kernel_list(torch, L, b):
    """(name, callable, launches, headline bytes, moved bytes) of the step's kernels."""
    anc, res, meta = b["anc"], b["res"], b["meta"]
    # K pages of layer l are pages 2l*512 + ..., V pages follow 512 pages later
    kA, vA = anc, anc[PER:]
    kR, vR = res, res[PER:]
    kM, vM = meta, meta[PER:]
    xk, xv = b["x"], b["x"][PER:]
    n_pool = N_PAGES - PER
    p = L.Params()
    dec_pages1 = N_LAYERS * HKV * NPPH
    dec_pages8 = 8 * dec_pages1

    def dec_anchor(q, pt, ctx, o, l, ws):
        return lambda: L.lynx_decode_attn(q, kA, None, kM, vA, None, vM, pt, ctx, HKV, p, out=o, lse=l,
                                          workspace=ws)
    ks = [
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
        ("decode_bf16_b1", lambda: L.lynx_decode_attn_bf16(b["q1"], xk, xv, b["pt1"], b["ctx1"], HKV, out=b["o1"],
                                                           lse=b["l1"], workspace=b["ws1"]), 2,
         2 * dec_pages1 * BYTES["decode_bf16"][0], 2 * dec_pages1 * BYTES["decode_bf16"][1]),
    ]
    del n_pool
    return ks


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


def profile_traffic(name):
    """DRAM traffic per launch from the committed ncu summary, if the kernel's
    source is unchanged since it was captured; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(name)
    if not e:
        return None
    return e["bytes_per_launch"] if e.get("source_sha") == source_sha(e.get("sources", [])) else None


# the CUDA sources each timed call runs (kernel file first, then shared headers)
KERNEL_SOURCES = {
    "encode": ["encode.cu", "lynx_internal.cuh"],
    "reconstruct_anchor": ["reconstruct.cu", "lynx_internal.cuh"],
    "reconstruct_full": ["reconstruct.cu", "lynx_internal.cuh"],
    "decode_anchor_b1": ["decode_narrow.cu", "decode_common.cuh", "lynx_internal.cuh"],
    "decode_anchor_b8": ["decode_narrow.cu", "decode_common.cuh", "lynx_internal.cuh"],
    "verify_full_t8": ["decode_tc.cu", "decode_common.cuh", "lynx_internal.cuh"],
    "decode_bf16_b1": ["decode_attn.cu", "lynx_internal.cuh"],
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
    b = build_buffers(torch, L, inputs, dev, seed=rank)
    ks = kernel_list(torch, L, b)
    if args.only:
        ks = [k for k in ks if k[0] in args.only.split(",")]
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        for k in ks:
            k[1]()
    torch.cuda.synchronize()
    L.lynx_device_status()

    ev = {k[0]: [] for k in ks}
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
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
    clk = clocks.stop()
    L.lynx_device_status()
    ms_total = reduce_max(t0.elapsed_time(t1), world, dist if world > 1 else None, dev)
    ms_step = ms_total / args.steps
    gbps_peak, peak_kind = peaks()
    tflops_peak, _ = tensor_peak()
    # (B, T) of the decode calls, G = 4, 8 KV heads, 16,384 keys
    attn_shape = {"decode_anchor_b1": (N_LAYERS, 1), "decode_anchor_b8": (8 * N_LAYERS, 1),
                  "verify_full_t8": (N_LAYERS, 8), "decode_bf16_b1": (N_LAYERS, 1)}
    kern = {}
    for name, _, launches, head, moved in ks:
        ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev[name])
        kern[name] = {"ms": round(ms, 4), "GBps_headline": round(head / ms / 1e6, 1),
                      "GBps_moved": round(moved / ms / 1e6, 1),
                      "frac_of_hbm": round(moved / ms / 1e6 / gbps_peak, 3),
                      "frac_of_nominal_hbm": round(moved / ms / 1e6 / NOMINAL_HBM_GBS, 3), "launches": launches,
                      "headline_bytes": head, "moved_bytes": moved}
        if name in attn_shape:
            B, T = attn_shape[name]
            tf = attn_flops(B, T, HQ // HKV, HKV, N_TOK) / ms / 1e9
            kern[name]["attn_tflops"] = round(tf, 1)
            kern[name]["frac_of_bf16_tensor"] = round(tf / tflops_peak, 4)
    head_total = sum(k[3] for k in ks)
    value = job_value(head_total, world, ms_step)
    dom = max(kern, key=lambda n: kern[n]["ms"])
    src = KERNEL_SOURCES[dom][0]
    roof = {"kernel": dom, "bound": "hbm", "achieved": kern[dom]["GBps_moved"], "peak": gbps_peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": kern[dom]["frac_of_hbm"],
            "traffic": profile_traffic(dom), "source": src}
    e2e = run_e2e(torch, L, b, ks, args, dev) if rank == 0 and not args.no_e2e else None
    prog = run_progressive(torch, L, b, dev) if rank == 0 and not args.no_e2e else None
    tok = run_encode_tokens(torch, L, b) if rank == 0 and not args.no_e2e else None
    cmp_ = run_comparators(torch, L, b, dev) if rank == 0 and not args.no_e2e else None
    other = None
    if rank == 0 and not args.no_e2e and N_LAYERS == 64:
        from progressive_kv_quantization_gb300 import inputs as inp
        other = {"decode_sweep": run_decode_sweep(torch, L, inp, dev),
                 "qwen235b": run_qwen235b(torch, L, inp, dev)}
    if rank != 0:
        return None
    launches = args.steps * sum(k[2] for k in ks)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD if N_LAYERS == 64 else WORKLOAD.replace("64 layers", f"{N_LAYERS} layers"),
                   "pages": N_PAGES, "bf16_bytes": N_PAGES * PAGE,
                   "l2": "inputs larger than L2 (4.29e9 B cache), no flush",
                   "alpha": 100.0, "eps": 1e-6, "parallelism": f"replicas x{world} (one cache per GPU)"},
        "kernels": kern,
        "encode_GBps_bf16_in": kern.get("encode", {}).get("GBps_headline"),
        "decode_anchor_GBps_packed": kern.get("decode_anchor_b1", {}).get("GBps_headline"),
        "roofline": roof,
        "e2e": e2e,
        "progressive": prog,
        "encode_tokens": tok,
        "comparators": cmp_,
        "other_workloads": other,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args.cpu_seconds)
    return line


def cpu_baseline_subprocess(seconds):
    """The oracle timed in a fresh single-threaded process on the host cores."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--impl", "reference", "--cpu-only-seconds",
                        str(seconds)], capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "error": r.stderr[-300:]}
    return json.loads(r.stdout.strip().splitlines()[-1])["cpu_baseline"]


def run_e2e(torch, L, b, ks, args, dev):
    """The same step's work through host buffers: the BF16 cache and the queries
    are copied in from pinned host memory, and the step's results (encoded
    planes, metadata, attention outputs) are read back, every step.

    The step runs per chunk of E2E_CHUNKS: chunk c is 64 / E2E_CHUNKS layers
    (their K and V pages are contiguous).  Its BF16 pages are copied in on an
    upload stream; once they have landed, the compute stream encodes them and
    runs every call of the step on those layers (both reconstructions, the
    decodes of the sequences that read them, the verification and the BF16
    decode), and a readback stream returns its planes, metadata and outputs.
    Later chunks' uploads overlap earlier chunks' compute.  The readbacks start
    once every upload of the step has finished: on this host link, transfers in
    both directions at once were measured to drop at times from 342 GB/s to
    ~130 GB/s, which made the step time vary 3x.  The next step's uploads wait
    until the previous step no longer reads the BF16 cache; a step ends when all
    its readbacks have finished."""
    n_chunks = E2E_CHUNKS
    lpc = N_LAYERS // n_chunks                # layers per chunk
    ppc = N_PAGES // n_chunks                 # pages per chunk (K and V of lpc layers)
    anc, res, meta = b["anc"], b["res"], b["meta"]
    kA, vA, kR, vR, kM, vM = anc, anc[PER:], res, res[PER:], meta, meta[PER:]
    xk, xv = b["x"], b["x"][PER:]
    p = L.Params()
    host_x = torch.empty(b["x"].shape, dtype=torch.bfloat16, pin_memory=True)
    host_x.copy_(b["x"])
    # the B = 8 sequences grouped by the layer their pages belong to
    layer8 = [(s // 8 + s % 8) % N_LAYERS for s in range(8 * N_LAYERS)]
    idx8 = [torch.tensor([s for s in range(8 * N_LAYERS) if layer8[s] // lpc == c], device=dev)
            for c in range(n_chunks)]
    c8 = [{k: b[k].index_select(0, idx8[c]).contiguous() for k in ("q8", "pt8", "ctx8")} for c in range(n_chunks)]
    h_q = {k: torch.empty(b[k].shape, dtype=b[k].dtype, pin_memory=True).copy_(b[k]) for k in ("q1", "qv")}
    h_q8 = [torch.empty(c["q8"].shape, dtype=c["q8"].dtype, pin_memory=True).copy_(c["q8"]) for c in c8]
    o8 = [{"o": torch.empty((len(idx8[c]), 1, HQ, 128), dtype=torch.float32, device=dev),
           "l": torch.empty((len(idx8[c]), 1, HQ), dtype=torch.float32, device=dev)} for c in range(n_chunks)]
    h_out = {k: torch.empty(b[k].shape, dtype=b[k].dtype, pin_memory=True) for k in ("anc", "res", "meta", "o1", "ov", "l1", "lv")}
    h_o8 = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o8[c].items()} for c in range(n_chunks)]

    def ws(B, T):
        n = L.lynx_decode_attn_workspace_size(B, T, HQ, HKV, 128, NPPH)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    ws1, ws8, wsv = ws(lpc, 1), ws(8 * lpc, 1), ws(lpc, 8)
    h2d = host_x.numel() * 2 + sum(v.numel() * v.element_size() for v in h_q.values()) + \
        sum(v.numel() * v.element_size() for v in h_q8)
    d2h = sum(v.numel() * v.element_size() for v in h_out.values()) + \
        sum(v.numel() * v.element_size() for d in h_o8 for v in d.values())
    # compute, uploads and readbacks each on a stream of their own (none of them the
    # legacy default stream, which would order itself against the others)
    comp, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n_chunks)]
    ev_cmp = [torch.cuda.Event() for _ in range(n_chunks)]
    ev_free = torch.cuda.Event()
    ev_free.record(comp)
    steps = max(5, min(args.steps, 9))

    def one():
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_free)           # the previous step no longer reads the cache
            for c in range(n_chunks):
                lo, hi = c * ppc, (c + 1) * ppc
                sl = slice(c * lpc, (c + 1) * lpc)
                b["x"][lo:hi].copy_(host_x[lo:hi], non_blocking=True)
                b["q1"][sl].copy_(h_q["q1"][sl], non_blocking=True)
                b["qv"][sl].copy_(h_q["qv"][sl], non_blocking=True)
                c8[c]["q8"].copy_(h_q8[c], non_blocking=True)
                ev_in[c].record(s_in)
        for c in range(n_chunks):
            lo, hi = c * ppc, (c + 1) * ppc
            sl = slice(c * lpc, (c + 1) * lpc)
            comp.wait_event(ev_in[c])
            cs = torch.cuda.stream(comp)
            cs.__enter__()
            L.lynx_encode_pages(b["x"][lo:hi], p, anc[lo:hi], res[lo:hi], meta[lo:hi])
            L.lynx_reconstruct(anc[lo:hi], None, meta[lo:hi], p, out=b["recon"][lo:hi])
            L.lynx_reconstruct(anc[lo:hi], res[lo:hi], meta[lo:hi], p, out=b["recon"][lo:hi])
            L.lynx_decode_attn(b["q1"][sl], kA, None, kM, vA, None, vM, b["pt1"][sl], b["ctx1"][sl], HKV, p,
                               out=b["o1"][sl], lse=b["l1"][sl], workspace=ws1)
            L.lynx_decode_attn(c8[c]["q8"], kA, None, kM, vA, None, vM, c8[c]["pt8"], c8[c]["ctx8"], HKV, p,
                               out=o8[c]["o"], lse=o8[c]["l"], workspace=ws8)
            L.lynx_decode_attn(b["qv"][sl], kA, kR, kM, vA, vR, vM, b["pt1"][sl], b["ctx1"][sl], HKV, p,
                               causal=True, out=b["ov"][sl], lse=b["lv"][sl], workspace=wsv)
            L.lynx_decode_attn_bf16(b["q1"][sl], xk, xv, b["pt1"][sl], b["ctx1"][sl], HKV, out=b["o1"][sl],
                                    lse=b["l1"][sl], workspace=ws1)
            cs.__exit__(None, None, None)
            ev_cmp[c].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_in[n_chunks - 1])   # after the step's last upload
                s_out.wait_event(ev_cmp[c])
                for k in ("anc", "res", "meta"):
                    h_out[k][lo:hi].copy_(b[k][lo:hi], non_blocking=True)
                for k in ("o1", "ov", "l1", "lv"):
                    h_out[k][sl].copy_(b[k][sl], non_blocking=True)
                for k in ("o", "l"):
                    h_o8[c][k].copy_(o8[c][k], non_blocking=True)
        ev_free.record(comp)
        comp.wait_stream(s_out)                # results are on the host when the step ends

    one()
    torch.cuda.synchronize()
    # each step timed on its own; the host link is shared, so the median step is reported
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    marks[0].record(comp)
    s_in.wait_event(marks[0])
    for k in range(steps):
        one()
        marks[k + 1].record(comp)
    torch.cuda.synchronize()
    per_step = sorted(marks[k].elapsed_time(marks[k + 1]) for k in range(steps))
    ms = per_step[len(per_step) // 2]
    head_total = sum(k[3] for k in ks)
    return {"value": round(head_total / (ms * 1e6), 1), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "statistic": "median step", "step_ms": [round(x, 3) for x in per_step], "chunks": n_chunks}


def run_progressive(torch, L, b, dev, reps=3):
    """The paper's split-stream transfer on one box (paper §4.2): the encoded
    64-layer cache goes device -> pinned host -> device layer by layer, every
    layer's Anchor plane and metadata first, the Residual planes after them
    (progressive.ProgressiveTransfer).  Reported: the time until every Anchor
    (draft decoding can run) and until every Residual (verification can run)
    has landed, against the same round trip of the BF16 cache; medians of
    ``reps`` runs (the host link is shared)."""
    from progressive_kv_quantization_gb300.progressive import ProgressiveTransfer
    layers = [(2 * l * PER, 2 * (l + 1) * PER) for l in range(N_LAYERS)]
    src = (b["anc"], b["res"], b["meta"])
    dst = tuple(torch.empty_like(t) for t in src)
    tr = ProgressiveTransfer(layers, dev)
    h_x = torch.empty(b["x"].shape, dtype=torch.bfloat16, pin_memory=True)
    d_x = torch.empty_like(b["x"])
    s_o, s_i = torch.cuda.Stream(), torch.cuda.Stream()
    staged = [torch.cuda.Event() for _ in layers]
    anchor, full, bf16 = [], [], []
    for _ in range(reps + 1):
        torch.cuda.synchronize()
        tr.send(src, dst)
        a, f = tr.times_ms()
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
        anchor.append(a)
        full.append(f)
        bf16.append(e0.elapsed_time(e1))
    med = lambda v: round(statistics.median(v[1:]), 3)    # the first run warms the path
    exact = all(bool(torch.equal(x, y)) for x, y in zip(src, dst)) and bool(torch.equal(d_x, b["x"]))
    return {"anchor_ready_ms": med(anchor), "full_ready_ms": med(full), "bf16_ms": med(bf16),
            "anchor_bytes": int(src[0].numel() + src[2].numel() * 4), "residual_bytes": int(src[1].numel()),
            "bf16_bytes": int(b["x"].numel() * 2), "path": "device -> pinned host -> device, per layer",
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


def run_qwen235b(torch, L, inputs, dev, reps=3):
    """The Qwen3-235B-shaped workload: 94 layers x K, V x 4 KV heads x 128 x
    131,072 tokens (385,024 pages, 25.2e9 BF16 bytes), 16 query heads: the
    layer-streamed encode (one lynx_encode_pages call per layer, 4,096 pages) and
    the Anchor-only decode at B = 1 over the full context (one call per layer),
    each timed over all 94 layers (CUDA events around the 94 calls; median of
    ``reps``); the decode also as one CUDA graph of the 94 calls ("graph_ms")."""
    n_layers, Hkv, Hq, n_tok = 94, 4, 16, 131072
    npph = n_tok // 256
    per_layer = 2 * Hkv * npph
    n = n_layers * per_layer
    outl = inputs.outlier_pairs(Hkv, 7)
    x = torch.empty((n, 128, 256), dtype=torch.bfloat16, device=dev)
    for layer in range(n_layers):
        for t in range(2):
            i = layer * per_layer + t * Hkv * npph
            x[i:i + Hkv * npph] = inputs.kv_pages_torch(Hkv, n_tok, inputs.layer_seed(7, layer, t), outl, dev)
    a = torch.empty((n, 128, 128), dtype=torch.uint8, device=dev)
    r = torch.empty_like(a)
    m = torch.empty((n, L.META_FLOATS), dtype=torch.float32, device=dev)
    p = L.Params()

    def encode_all():
        for layer in range(n_layers):
            sl = slice(layer * per_layer, (layer + 1) * per_layer)
            L.lynx_encode_pages(x[sl], p, a[sl], r[sl], m[sl])
    t_enc = _median_ms(torch, encode_all, reps)
    q = inputs.queries_torch((1, 1, Hq, 128), 77, dev)
    pt = torch.arange(Hkv * npph, dtype=torch.int32, device=dev).view(1, Hkv, npph)
    ctx = torch.full((1,), n_tok, dtype=torch.int32, device=dev)
    nb = L.lynx_decode_attn_workspace_size(1, 1, Hq, Hkv, 128, npph)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
    o = torch.empty((1, 1, Hq, 128), dtype=torch.float32, device=dev)
    l_ = torch.empty((1, 1, Hq), dtype=torch.float32, device=dev)
    layers = [(a[k * per_layer:], m[k * per_layer:], a[k * per_layer + Hkv * npph:], m[k * per_layer + Hkv * npph:])
              for k in range(n_layers)]

    def decode_all():
        for ka, km, va, vm in layers:
            L.lynx_decode_attn(q, ka, None, km, va, None, vm, pt, ctx, Hkv, p, out=o, lse=l_, workspace=ws)
    t_dec = _median_ms(torch, decode_all, reps)
    t_graph = _graph_ms(torch, decode_all, reps)
    gbps_peak, _ = peaks()
    enc_moved, dec_moved = n * BYTES["encode"][1], n * BYTES["decode_anchor"][1]
    del x, a, r, m
    return {"pages": n, "bf16_bytes": n * PAGE,
            "encode": {"ms": round(t_enc, 3), "GBps_bf16_in": round(n * PAGE / t_enc / 1e6, 1),
                       "frac_of_hbm": round(enc_moved / t_enc / 1e6 / gbps_peak, 3), "launches": n_layers},
            "decode_anchor_b1": {"ms": round(t_dec, 3), "GBps_packed": round(dec_moved / t_dec / 1e6, 1),
                                 "frac_of_hbm": round(dec_moved / t_dec / 1e6 / gbps_peak, 3),
                                 "graph_ms": round(t_graph, 3),
                                 "graph_GBps_packed": round(dec_moved / t_graph / 1e6, 1),
                                 "graph_frac_of_hbm": round(dec_moved / t_graph / 1e6 / gbps_peak, 3),
                                 "launches": 2 * n_layers},
            "statistic": f"median of {reps} passes over the 94 layers"}


# ------------------------------------------------------------------ oracle arm

def oracle_sample_step():
    """A bounded sample of the step for the CPU oracle: one layer's K and V of
    one KV head (64 + 64 pages) through encode, both reconstructs, the draft
    decode at B=1 and B=8, the T=8 verification and the BF16 decode.
    Returns (headline bytes, seconds)."""
    import numpy as np

    from oracle import attention as at
    from oracle import lynx_oracle as lo
    from progressive_kv_quantization_gb300 import inputs

    eps = np.float32(1e-6)
    outl = inputs.outlier_pairs(1, 0, count=1)
    kb = inputs.kv_pages_np(1, N_TOK, 1, outl)
    vb = inputs.kv_pages_np(1, N_TOK, 2, outl)
    G = HQ // HKV
    q1 = inputs.queries_np((1, 1, G, 128), 3)
    q8 = inputs.queries_np((8, 1, G, 128), 4)
    qv = inputs.queries_np((1, 8, G, 128), 5)
    table1 = np.arange(NPPH, dtype=np.int32)[None, None]
    table8 = np.repeat(table1, 8, axis=0)
    ctx1 = np.array([N_TOK])
    ctx8 = np.full(8, N_TOK)
    scale = 1 / math.sqrt(128)
    t0 = time.perf_counter()
    ka, kr, km = lo.encode_pages(kb, 100.0, eps)
    va, vr, vm = lo.encode_pages(vb, 100.0, eps)
    kd_a = lo.reconstruct(ka, None, km, 100.0, eps)
    vd_a = lo.reconstruct(va, None, vm, 100.0, eps)
    kd_f = lo.reconstruct(ka, kr, km, 100.0, eps)
    vd_f = lo.reconstruct(va, vr, vm, 100.0, eps)
    fa = lambda ids: (kd_a[ids], vd_a[ids])
    ff = lambda ids: (kd_f[ids], vd_f[ids])
    fb = lambda ids: (lo.bf16_to_f32(kb[ids]).astype(np.float64), lo.bf16_to_f32(vb[ids]).astype(np.float64))
    qf = lambda q: lo.bf16_to_f32(q).astype(np.float64)
    at.decode_attention(qf(q1), fa, table1, ctx1, 1, scale, False)
    at.decode_attention(qf(q8), fa, table8, ctx8, 1, scale, False)
    at.decode_attention(qf(qv), ff, table1, ctx1, 1, scale, True)
    at.decode_attention(qf(q1), fb, table1, ctx1, 1, scale, False)
    sec = time.perf_counter() - t0
    n = 2 * NPPH
    head = (n * BYTES["encode"][0] + n * BYTES["reconstruct_anchor"][0] + n * BYTES["reconstruct_full"][0]
            + n * BYTES["decode_anchor"][0] * (1 + 8) + n * BYTES["decode_full"][0] + n * BYTES["decode_bf16"][0])
    return head, sec


def run_reference_sample(seconds=15.0, steps=None, warmup=0):
    """Times the oracle on repeated bounded samples (the caller's process runs
    with one BLAS / OpenMP thread)."""
    for _ in range(warmup):
        oracle_sample_step()
    tot_b, tot_s, n = 0, 0.0, 0
    while (steps is None and (tot_s < seconds or n == 0)) or (steps is not None and n < steps):
        bb, ss = oracle_sample_step()
        tot_b += bb
        tot_s += ss
        n += 1
    v = tot_b / tot_s / 1e9
    return {"value": v, "seconds": tot_s, "samples": n,
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": (f"{n} x (one layer's K and V of one KV head: 2 x 64 pages, 16384 tokens, "
                                        "4 query heads) through encode, both reconstructs, B=1 and B=8 draft "
                                        "decode, T=8 verify, BF16 decode; numpy, 1 thread"),
                             "seconds": round(tot_s, 2)}}


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
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-only-seconds", type=float, default=None)
    ap.add_argument("--layers", type=int, default=64, help="cache layers (64 = the benchmark workload)")
    ap.add_argument("--only", default="", help="comma-separated kernel names to run (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.layers != 64:
        set_layers(args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        # the CPU oracle: rank 0 only; other ranks exit without work
        if rank != 0:
            return
        if args.cpu_only_seconds is not None:
            r = run_reference_sample(seconds=args.cpu_only_seconds)
        else:
            r = run_reference_sample(steps=args.steps, warmup=args.warmup)
        line = {"metric": METRIC, "value": round(r["value"], 4), "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1000 * r["seconds"] / max(r["samples"], 1), 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference",
                "config": {"workload": WORKLOAD, "sample": "one KV head of one layer per step (CPU oracle)"},
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
