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

    def step_host(self, session: ciera.HostSession, w_host: torch.Tensor,
                  out_host: torch.Tensor, w_dev: torch.Tensor, chunks: int = 1,
                  stream=None) -> None:
        """End-to-end from host memory (ciera_step_host): this iteration's
        weights are copied in from ``w_host`` (pinned) to ``w_dev``, the path
        runs, and the rebuilt weights land in ``out_host``, in chunks of ranks
        whose copies overlap the kernels.  Exact sender only."""
        if self.rans or self.hashed:
            raise ValueError("step_host drives the exact sender")
        session.step(self.plan, w_host, out_host, w_dev, self.sender_cache, self.payloads,
                     self.descs, self.recv_cache, self.out, self.workspace,
                     cold=self.iteration == 0, extra_flags=self.extra_flags, chunks=chunks,
                     stream=stream)
        self.iteration += 1

    def status(self, stream=None) -> int:
        return ciera.status(self.workspace, stream=stream)

    def descriptors(self):
        return ciera.decode_descs(self.descs)
