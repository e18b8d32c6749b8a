"""Split-stream (progressive) transfer of an encoded KV cache on one box.

The Lynx paper (§4.2, Stream SerDes) ships each layer's Anchor plane with its
metadata first and the Residual plane after it, so that the receiving decode
instance can start drafting on the Anchor KV while the Residual is still on
the wire, and verify once it lands.  Here the "wire" between a producing and a
consuming set of device buffers is a round trip through pinned host memory
(device -> host -> device), and the ordering is carried by CUDA streams and
events:

  * an outbound stream copies, layer by layer, every Anchor plane with its
    metadata to the host, then every Residual plane;
  * an inbound stream copies each piece to the destination as soon as its
    outbound copy has finished (per-layer events), in the same order, so the
    two directions of the host link overlap and every Anchor lands before any
    Residual; ``anchor_ready[l]`` fires when layer l's Anchor and metadata are
    in place, ``full_ready[l]`` when its Residual is.

A consumer makes its draft decode of layer l wait for ``anchor_ready[l]`` and
its verification wait for ``full_ready[l]`` (``Stream.wait_event``).  The
transfer moves bytes only; no computation runs on the host.
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
        self.s_out = torch.cuda.Stream(device=self.device)
        self.s_in = torch.cuda.Stream(device=self.device)
        self.anchor_ready = [torch.cuda.Event(enable_timing=True) for _ in self.layers]
        self.full_ready = [torch.cuda.Event(enable_timing=True) for _ in self.layers]
        self._staged = [torch.cuda.Event() for _ in range(2 * len(self.layers))]
        self.start = torch.cuda.Event(enable_timing=True)

    def send(self, src, dst, after=None):
        """Queue the transfer of src = (anchor, residual, meta) into dst (same
        layouts, on the device).  ``after``: an event the transfer waits for (the
        producer's encode); default: the work queued so far on the current
        stream.  Returns immediately; use the per-layer events."""
        sa, sr, sm = src
        da, dr, dm = dst
        cur = torch.cuda.current_stream(self.device)
        if after is None:
            after = torch.cuda.Event()
            after.record(cur)
        n = len(self.layers)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(after)
            self.start.record(self.s_out)
            for k, (a, b) in enumerate(self.layers):              # Anchors and metadata first
                self.h_anchor[a:b].copy_(sa[a:b], non_blocking=True)
                self.h_meta[a:b].copy_(sm[a:b], non_blocking=True)
                self._staged[k].record(self.s_out)
            for k, (a, b) in enumerate(self.layers):              # then the Residuals
                self.h_residual[a:b].copy_(sr[a:b], non_blocking=True)
                self._staged[n + k].record(self.s_out)
        with torch.cuda.stream(self.s_in):
            self.s_in.wait_event(self.start)
            for k, (a, b) in enumerate(self.layers):
                self.s_in.wait_event(self._staged[k])
                da[a:b].copy_(self.h_anchor[a:b], non_blocking=True)
                dm[a:b].copy_(self.h_meta[a:b], non_blocking=True)
                self.anchor_ready[k].record(self.s_in)
            for k, (a, b) in enumerate(self.layers):
                self.s_in.wait_event(self._staged[n + k])
                dr[a:b].copy_(self.h_residual[a:b], non_blocking=True)
                self.full_ready[k].record(self.s_in)
        return self

    def times_ms(self):
        """(time until every Anchor has landed, time until every Residual has
        landed), in ms from the start of the transfer; synchronises."""
        self.full_ready[-1].synchronize()
        return self.start.elapsed_time(self.anchor_ready[-1]), self.start.elapsed_time(self.full_ready[-1])
