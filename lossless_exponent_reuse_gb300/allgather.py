"""One exponent-reuse Allgather of a flat bf16 buffer, R simulated ranks on one GPU.

The R senders' payloads are laid out in this GPU's memory exactly as an
Allgather would deliver them (rank r's payload at row r), so the receiver
side runs on the real gathered layout; no collective is involved.

CIERA ("Cross-Iteration Exponent Reuse for Lossless Allgather in Sharded MoE
Training"), Section 3.1: every sender keeps the exponents it sent last
iteration, every receiver keeps the exponents of every shard (ExpCache);
both caches persist across iterations.  The first call is a cold start.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import ciera


class SimulatedAllgather:
    """Device state of one plan: both exponent caches, payloads, descriptors."""

    def __init__(self, numel: int, block: int, ranks: int, device="cuda",
                 keep_flags: bool = False, hashed: bool = False, rans: bool = False,
                 raw_ahead: bool = True):
        if hashed and rans:
            raise ValueError("the hashed change test and RANS payloads are separate senders")
        self.plan = ciera.Plan(numel, block, ranks)
        info = self.plan.info
        self.numel = numel
        self.device = torch.device(device)
        self.hashed = hashed
        self.rans = rans
        # raw_ahead=False: every shard takes the look-back scan (same bytes)
        self.extra_flags = 0 if raw_ahead else ciera.NO_RAW_AHEAD
        # RANS: each shard's exponent histogram, this call's and the previous one's
        self.hist = ([torch.zeros((ranks, 256), dtype=torch.int32, device=device)
                      for _ in range(2)] if rans else None)
        # the sender's state: exponents per value, or (hashed) 16 bytes per block
        self.hash_cache = (torch.zeros((ranks, max(info.blocks_per_shard, 1), 2),
                                       dtype=torch.int64, device=device) if hashed else None)
        self.sender_cache = torch.zeros(1 if hashed else max(numel, 1), dtype=torch.uint8,
                                        device=device)
        self.recv_cache = torch.zeros(max(numel, 1), dtype=torch.uint8, device=device)
        self.payloads = self.plan.new_payloads(device=device)
        self.descs = self.plan.new_descs(device=device)
        self.workspace = self.plan.new_workspace(device=device)
        self.flags = (torch.zeros((ranks, max(info.blocks_per_shard, 1)), dtype=torch.uint8,
                                  device=device) if keep_flags else None)
        self.out = torch.empty(max(numel, 1), dtype=torch.uint16, device=device)
        self.iteration = 0

    def compress(self, w: torch.Tensor, stream=None) -> None:
        if self.rans:
            prev, cur = self.hist[self.iteration % 2], self.hist[(self.iteration + 1) % 2]
            self.plan.compress_rans(w, self.sender_cache, prev, cur, self.payloads, self.descs,
                                    self.workspace, cold=self.iteration == 0,
                                    flags_out=self.flags, stream=stream)
        elif self.hashed:
            self.plan.compress_hashed(w, self.hash_cache, self.payloads, self.descs,
                                      self.workspace, cold=self.iteration == 0,
                                      flags_out=self.flags, extra_flags=self.extra_flags,
                                      stream=stream)
        else:
            self.plan.compress(w, self.sender_cache, self.payloads, self.descs, self.workspace,
                               cold=self.iteration == 0, flags_out=self.flags,
                               extra_flags=self.extra_flags, stream=stream)

    def decompress(self, stream=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        o = self.out if out is None else out
        self.plan.decompress(self.payloads, self.descs, self.recv_cache, o, self.workspace,
                             rans=self.rans, stream=stream)
        self.iteration += 1
        return o

    def step(self, w: torch.Tensor, stream=None) -> torch.Tensor:
        """Sender side for all ranks, then the fused gather-decompress."""
        self.compress(w, stream=stream)
        return self.decompress(stream=stream)

    def step_host(self, w_host: torch.Tensor, out_host: torch.Tensor, w_dev: torch.Tensor,
                  stream=None) -> None:
        """End-to-end from host memory: copy this iteration's weights in,
        run the path, copy the rebuilt weights out (pinned buffers)."""
        w_dev.view(torch.int16).copy_(w_host.view(torch.int16), non_blocking=True)
        self.step(w_dev, stream=stream)
        out_host.view(torch.int16).copy_(self.out[: self.numel].view(torch.int16),
                                         non_blocking=True)

    def status(self, stream=None) -> int:
        return ciera.status(self.workspace, stream=stream)

    def descriptors(self):
        return ciera.decode_descs(self.descs)


class HostStreamer:
    """Steps whose weights come from pinned host memory and whose rebuilt
    weights go back to it, with the copies of neighbouring steps overlapped:
    the upload of step i+1 and the download of step i run on their own
    streams (the link carries both directions at once) while the path runs on
    the caller's stream.  Device staging is double-buffered and every reuse
    of a buffer waits, by event, for its previous reader."""

    def __init__(self, ag: SimulatedAllgather):
        n = max(ag.numel, 1)
        dev = ag.device
        self.ag = ag
        self.w_buf = [torch.empty(n, dtype=torch.int16, device=dev) for _ in range(2)]
        self.out_buf = [torch.empty(n, dtype=torch.int16, device=dev) for _ in range(2)]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.ev_in, self.ev_done, self.ev_out = ev(), ev(), ev()
        self.count = 0

    def step(self, w_host: torch.Tensor, out_host: torch.Tensor) -> None:
        """Enqueue one step (asynchronous; ``finish`` joins it)."""
        n = self.ag.numel
        b = self.count % 2
        compute = torch.cuda.current_stream(self.ag.device)
        if self.count >= 2:
            self.s_in.wait_event(self.ev_done[b])        # step count-2 has read w_buf[b]
        with torch.cuda.stream(self.s_in):
            self.w_buf[b][:n].copy_(w_host.view(torch.int16), non_blocking=True)
            self.ev_in[b].record(self.s_in)
        compute.wait_event(self.ev_in[b])
        if self.count >= 2:
            compute.wait_event(self.ev_out[b])           # step count-2 has left out_buf[b]
        self.ag.compress(self.w_buf[b][:n])
        self.ag.decompress(out=self.out_buf[b])
        self.ev_done[b].record(compute)
        self.s_out.wait_event(self.ev_done[b])
        with torch.cuda.stream(self.s_out):
            out_host.view(torch.int16).copy_(self.out_buf[b][:n], non_blocking=True)
            self.ev_out[b].record(self.s_out)
        self.count += 1

    def finish(self) -> None:
        """Make the caller's stream wait for every enqueued copy."""
        compute = torch.cuda.current_stream(self.ag.device)
        compute.wait_stream(self.s_in)
        compute.wait_stream(self.s_out)
