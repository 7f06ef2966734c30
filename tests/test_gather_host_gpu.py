"""Two receiver-side boundaries, checked against the CPU oracle.

* ciera_decompress_gather: the R payloads arrive in R separately allocated
  buffers (what a grouped broadcast would deliver: Algorithm 1's receiver,
  one Recv() per shard), addressed through a device table of pointers.
* ciera_step_host: one call from host memory to host memory -- upload,
  sender, gather-decompress, download -- in chunks of ranks whose copies
  overlap the kernels.

CIERA Section 3.1 and Appendix A, Algorithm 1.
"""
import numpy as np
import pytest
import torch

import oracle
from harness import OracleAny, compare_any, to_np_u16, to_np_u8
from lossless_exponent_reuse_gb300 import ciera, workloads
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = pytest.mark.gpu

# (values, ranks, block): staged fast path, 32 blocks per tile, byte-wise
# path with a partial last shard, a short last shard of partial blocks, and
# two empty last shards (50 values over 12 ranks of 5)
CASES = [(196608, 3, 4096), (131072, 4, 256), (100003, 3, 100), (40000, 7, 4096),
         (50, 12, 4)]


def _seq(n, R, B, iters, seed, p_block=0.2):
    wl = workloads.small(f"g{seed}", [(n,)], ranks=R, block=B, iterations=iters, step=1e-3,
                         seed=seed, p_block=p_block)
    return [w.cuda() for w in workloads.sequence(wl, iters)]


def _scatter(ag, capacity, shift=0):
    """Copy each rank's payload slot into its own allocation; return the
    buffers (kept alive by the caller) and the device table of their
    addresses (+ shift bytes)."""
    bufs = []
    for r in range(ag.plan.info.ranks):
        b = torch.zeros(capacity + 256, dtype=torch.uint8, device="cuda")
        b[:ag.payloads.shape[1]].copy_(ag.payloads[r])
        bufs.append(b)
    table = torch.tensor([b.data_ptr() + shift for b in bufs], dtype=torch.int64, device="cuda")
    return bufs, table


def _rans_plan(n, R, B):
    """The RANS sender takes staged plans only: B, N and S multiples of 16."""
    return B % 16 == 0 and B >= 256 and n % 16 == 0 and (-(-n // R)) % 16 == 0


@pytest.mark.parametrize("n,R,B,sender",
                         [c + ("exact",) for c in CASES] +
                         [c + ("rans",) for c in CASES if _rans_plan(*c)])
def test_gather_from_separate_buffers_matches_the_oracle(n, R, B, sender):
    seq = _seq(n, R, B, 4, seed=n % 1000 + R)
    rans = sender == "rans"
    ag = SimulatedAllgather(n, B, R, rans=rans)
    ost = OracleAny(n, R, B, sender)
    cap = ag.plan.info.payload_capacity
    for t, w in enumerate(seq):
        ag.compress(w)
        bufs, table = _scatter(ag, cap)
        ag.plan.decompress_gather(table, cap + 256, ag.descs, ag.recv_cache, ag.out,
                                  ag.workspace, rans=rans)
        ag.iteration += 1
        torch.cuda.synchronize()
        assert ag.status() == ciera.OK
        w_np = to_np_u16(w)
        compare_any(ag, ost, w_np, ost.step(w_np), tag=f"gather {sender} t={t}")
        del bufs


def test_gather_skips_missing_and_misaligned_payloads():
    """A NULL entry and (on the staged path) an entry that is not 16-byte
    aligned are never dereferenced: the rank is skipped, its output and
    ExpCache slices stay as they were, CIERA_E_CORRUPT is reported, and
    every other rank is rebuilt."""
    n, R, B = 196608, 3, 4096
    seq = _seq(n, R, B, 2, seed=5)
    ag = SimulatedAllgather(n, B, R)
    cap = ag.plan.info.payload_capacity
    S = ag.plan.info.shard_len
    ag.step(seq[0])
    assert ag.status() == ciera.OK
    ag.compress(seq[1])
    bufs, table = _scatter(ag, cap)
    for bad_rank, bad in ((1, 0), (2, bufs[2].data_ptr() + 8)):
        before_out = ag.out.clone()
        before_rc = ag.recv_cache.clone()
        t2 = table.clone()
        t2[bad_rank] = bad
        ag.plan.decompress_gather(t2, cap + 256, ag.descs, ag.recv_cache, ag.out, ag.workspace)
        torch.cuda.synchronize()
        assert ag.status() == ciera.E_CORRUPT
        lo, hi = bad_rank * S, min(n, (bad_rank + 1) * S)
        assert torch.equal(ag.out[lo:hi].view(torch.int16), before_out[lo:hi].view(torch.int16))
        assert torch.equal(ag.recv_cache[lo:hi], before_rc[lo:hi])
        for r in range(R):
            if r != bad_rank:
                a, z = r * S, min(n, (r + 1) * S)
                assert torch.equal(ag.out[a:z].view(torch.int16), seq[1][a:z].view(torch.int16))
        # the good table rebuilds everything again
        ag.plan.decompress_gather(table, cap + 256, ag.descs, ag.recv_cache, ag.out,
                                  ag.workspace)
        torch.cuda.synchronize()
        assert ag.status() == ciera.OK
        assert torch.equal(ag.out[:n].view(torch.int16), seq[1].view(torch.int16))


@pytest.mark.parametrize("n,R,B", CASES)
@pytest.mark.parametrize("chunks", [1, 2, 5, 64])
def test_step_host_matches_the_oracle(n, R, B, chunks):
    """Host buffers in, host buffers out: every step's rebuilt values in
    out_host equal the input, and the device-side results (descriptors,
    payloads, both caches) equal the oracle's, for chunkings that divide R,
    do not, and exceed it."""
    seq = _seq(n, R, B, 4, seed=3 * n % 997 + chunks)
    ag = SimulatedAllgather(n, B, R)
    ost = OracleAny(n, R, B, "exact")
    session = ciera.HostSession(64)
    w_dev = torch.empty(n, dtype=torch.int16, device="cuda")
    out_host = torch.empty(n, dtype=torch.int16).pin_memory()
    for t, w in enumerate(seq):
        w_host = w.view(torch.int16).cpu().pin_memory()
        out_host.fill_(0x7FFF)
        ag.step_host(session, w_host, out_host, w_dev, chunks=chunks)
        torch.cuda.current_stream().synchronize()
        assert ag.status() == ciera.OK
        w_np = to_np_u16(w)
        np.testing.assert_array_equal(out_host.numpy().view(np.uint16), w_np)
        compare_any(ag, ost, w_np, ost.step(w_np), tag=f"host chunks={chunks} t={t}")


def test_step_host_full_layer_round_trip():
    """The OLMoE MoE layer (402,653,184 values, 16 ranks) through
    ciera_step_host in 8 chunks for three iterations: out_host equals the
    input every time, and two sampled ranks' payloads equal the oracle's."""
    wl = workloads.workload(2)
    n = wl.layer_numel
    ag = SimulatedAllgather(n, wl.block, wl.ranks)
    session = ciera.HostSession(16)
    w_dev = torch.empty(n, dtype=torch.int16, device="cuda")
    out_host = torch.empty(n, dtype=torch.int16).pin_memory()
    w = workloads.initial_layer(wl, 0, "cuda")
    caches = {r: np.zeros(oracle.shard_len(n, wl.ranks, r), np.uint8) for r in (0, 11)}
    for t in range(3):
        if t > 0:
            w = workloads.step_layer(wl, w, 0, t)
        w_host = w.view(torch.int16).cpu().pin_memory()
        ag.step_host(session, w_host, out_host, w_dev, chunks=8)
        torch.cuda.current_stream().synchronize()
        assert ag.status() == ciera.OK
        assert torch.equal(out_host, w_host)
        descs = ag.descriptors()
        for r, sc in caches.items():
            b, ln = oracle.shard_begin(n, wl.ranks, r), oracle.shard_len(n, wl.ranks, r)
            payload, _, d = oracle.compress_shard(to_np_u16(w[b:b + ln]), wl.block, sc, t == 0)
            assert descs[r] == {k: int(v) for k, v in d.items()}, (t, r)
            np.testing.assert_array_equal(to_np_u8(ag.payloads[r, :d["payload_bytes"]]), payload)
    del ag, w_dev
    torch.cuda.empty_cache()
