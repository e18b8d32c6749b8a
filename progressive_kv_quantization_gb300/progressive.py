"""Split-stream (progressive) transfer of an encoded KV cache on one box.

The Lynx paper (§4.2, Stream SerDes and Figure 7) pushes each object's
Anchor (with its metadata) and Residual through two separate queues, the
Anchor queue first, and transmits object i while object i + 1 is being
quantised; the receiving decode instance drafts on the Anchor KV as soon as it
lands and verifies once the Residual has refined it to the full codes.  Here
the "wire" between a producing and a consuming set of device buffers is a round
trip through pinned host memory (device -> host -> device), an object is one
layer's page range, and the ordering is carried by CUDA streams and events:

  * the producer encodes layer after layer on its compute stream
    (``encode_and_send``); each layer's copies wait only for that layer's
    encode, so layer i moves while layer i + 1 is encoded;
  * outbound, a high-priority stream copies each layer's Anchor plane and
    metadata to the host and a low-priority stream its Residual plane; the
    Residual queue drains behind the Anchor queue (a Residual copy starts once
    every Anchor has gone out, as a strict priority queue does while the link
    is the bottleneck), so the link carries every Anchor first;
  * inbound, two more streams of the same priorities copy each piece to the
    destination as soon as its outbound copy has finished (per-layer events),
    Residuals again behind all Anchors; ``anchor_ready[l]`` fires when layer
    l's Anchor and metadata are in place, ``full_ready[l]`` when its Residual
    is too.

A consumer makes its draft decode of layer l wait for ``anchor_ready[l]`` and
its verification (or full reconstruction) of layer l wait for
``full_ready[l]`` (``Stream.wait_event``), so each layer's verification is
chained on its own Residual.  The transfer moves bytes only; the encode is the
library's kernel; no computation runs on the host.
"""
from __future__ import annotations

import torch


class ProgressiveTransfer:
    """Anchor-first transfer of page ranges ``layers`` (a list of (first, end)
    page indices, one per layer, in sending order) between encoded pools with
    the layouts of ``lynx_encode_pages`` (anchor / residual u8[N, 128, 128],
    meta f32[N, 2304]).  Staging buffers in pinned host memory are allocated
    once, for the largest page index used."""

    def __init__(self, layers, device=None):
        self.layers = [(int(a), int(b)) for a, b in layers]
        if not self.layers or any(a < 0 or b <= a for a, b in self.layers):
            raise ValueError("layers must be non-empty (first, end) page ranges")
        n = max(b for _, b in self.layers)
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        pin = dict(pin_memory=True)
        self.h_anchor = torch.empty((n, 128, 128), dtype=torch.uint8, **pin)
        self.h_residual = torch.empty((n, 128, 128), dtype=torch.uint8, **pin)
        self.h_meta = torch.empty((n, 2304), dtype=torch.float32, **pin)
        # a smaller number is a higher priority; torch maps values outside the
        # device's range to its nearest end, so -64 is the highest available
        high, low = -64, 0
        mk = lambda prio: torch.cuda.Stream(device=self.device, priority=prio)
        self.s_anchor_out, self.s_residual_out = mk(high), mk(low)
        self.s_anchor_in, self.s_residual_in = mk(high), mk(low)
        nl = len(self.layers)
        ev = lambda timing=False: [torch.cuda.Event(enable_timing=timing) for _ in range(nl)]
        self.anchor_ready = ev(True)
        self.full_ready = ev(True)
        self.encoded = ev(True)
        self._staged_anchor = ev()
        self._staged_residual = ev()
        self.start = torch.cuda.Event(enable_timing=True)

    def _send_anchor(self, k, src, dst, after):
        """Queue layer k's Anchor + metadata, outbound and inbound, after event ``after``."""
        a, b = self.layers[k]
        sa, _, sm = src
        da, _, dm = dst
        with torch.cuda.stream(self.s_anchor_out):
            self.s_anchor_out.wait_event(after)
            self.h_anchor[a:b].copy_(sa[a:b], non_blocking=True)
            self.h_meta[a:b].copy_(sm[a:b], non_blocking=True)
            self._staged_anchor[k].record(self.s_anchor_out)
        with torch.cuda.stream(self.s_anchor_in):
            self.s_anchor_in.wait_event(self._staged_anchor[k])
            da[a:b].copy_(self.h_anchor[a:b], non_blocking=True)
            dm[a:b].copy_(self.h_meta[a:b], non_blocking=True)
            self.anchor_ready[k].record(self.s_anchor_in)

    def _send_residual(self, k, src, dst):
        """Queue layer k's Residual, outbound once every Anchor has gone out and
        inbound once every Anchor has landed (call after every _send_anchor)."""
        a, b = self.layers[k]
        _, sr, _ = src
        _, dr, _ = dst
        with torch.cuda.stream(self.s_residual_out):
            self.s_residual_out.wait_event(self._staged_anchor[-1])
            self.h_residual[a:b].copy_(sr[a:b], non_blocking=True)
            self._staged_residual[k].record(self.s_residual_out)
        with torch.cuda.stream(self.s_residual_in):
            self.s_residual_in.wait_event(self.anchor_ready[-1])
            self.s_residual_in.wait_event(self._staged_residual[k])
            dr[a:b].copy_(self.h_residual[a:b], non_blocking=True)
            self.full_ready[k].record(self.s_residual_in)

    def send(self, src, dst, after=None):
        """Queue the transfer of an already encoded src = (anchor, residual,
        meta) into dst (same layouts, on the device).  ``after``: an event the
        transfer waits for; default: the work queued so far on the current
        stream.  Returns immediately; use the per-layer events."""
        cur = torch.cuda.current_stream(self.device)
        if after is None:
            after = torch.cuda.Event()
            after.record(cur)
        self.start.record(cur)
        for k in range(len(self.layers)):
            self._send_anchor(k, src, dst, after)
        for k in range(len(self.layers)):
            self._send_residual(k, src, dst)
        return self

    def encode_and_send(self, x, src, dst, params=None, stream=None):
        """Encode the BF16 pages ``x`` layer by layer into src = (anchor,
        residual, meta) on ``stream`` (default: the current stream) with
        ``lynx_encode_pages``, and queue each layer's Anchor transfer into dst
        as soon as that layer is encoded, so that layer i is transmitted while
        layer i + 1 is encoded; the Residuals follow the last Anchor.  Returns
        immediately; use the per-layer events (``encoded[l]`` fires when layer
        l's encode has finished)."""
        from progressive_kv_quantization_gb300 import lynx as L
        params = params if params is not None else L.Params()
        stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        sa, sr, sm = src
        self.start.record(stream)
        for k, (a, b) in enumerate(self.layers):
            with torch.cuda.stream(stream):
                L.lynx_encode_pages(x[a:b], params, sa[a:b], sr[a:b], sm[a:b])
                self.encoded[k].record(stream)
            self._send_anchor(k, src, dst, self.encoded[k])
        for k in range(len(self.layers)):
            self._send_residual(k, src, dst)
        return self

    def times_ms(self):
        """(time until every Anchor has landed, time until every Residual has
        landed), in ms from the start of the transfer; synchronises."""
        self.full_ready[-1].synchronize()
        self.anchor_ready[-1].synchronize()
        return (max(self.start.elapsed_time(e) for e in self.anchor_ready),
                max(self.start.elapsed_time(e) for e in self.full_ready))
