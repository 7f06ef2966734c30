"""Computation-communication pipelining on one GPU (CIERA Section 3.3, Fig. 7):
compress(i+1) on a side stream overlapping decompress(i).  Every output of the
pipelined step -- descriptors, payload bytes, rebuilt values, the sender's
state (exponent cache, HashCache, exponent histograms) and the receiver's
exponent cache -- is compared with the CPU oracle's, layer by layer and step
by step, eagerly and with the step captured into a CUDA graph and replayed."""
import pytest
import torch

from harness import OracleAny, compare_any, to_np_u16
from lossless_exponent_reuse_gb300 import ciera, workloads
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = pytest.mark.gpu

LAYERS = [(131072, 4, 256), (196608, 3, 4096), (100003, 3, 256), (65536, 2, 272)]
RANS_LAYERS = [(131072, 4, 256), (196608, 3, 4096), (65536, 2, 272)]


def _layer_seqs(layers, steps, seed0=0):
    out = []
    for li, (n, R, B) in enumerate(layers):
        wl = workloads.small(f"L{seed0 + li}", [(n,)], ranks=R, block=B, iterations=steps,
                             step=1e-3, seed=seed0 + li, p_block=0.2)
        out.append([w.cuda() for w in workloads.sequence(wl, steps)])
    return out


def _run_pipelined(layers, sender, steps, seed0=0):
    seqs = _layer_seqs(layers, steps, seed0)
    kw = dict(rans=sender == "rans", hashed=sender == "hashed")
    gpu = [SimulatedAllgather(n, B, R, **kw) for n, R, B in layers]
    ref = [OracleAny(n, R, B, sender) for n, R, B in layers]
    pipe = ciera.Pipeline(len(layers))
    modes = set()
    for t in range(steps):
        pipe.step(gpu, [s[t] for s in seqs])
        torch.cuda.synchronize()
        for li, (ag, ost, s) in enumerate(zip(gpu, ref, seqs)):
            assert ag.status() == ciera.OK
            w_np = to_np_u16(s[t])
            compare_any(ag, ost, w_np, ost.step(w_np), tag=f"{sender} t={t} layer {li}")
            modes.update(d["mode"] for d in ag.descriptors())
    return modes


def test_pipelined_step_matches_the_oracle():
    modes = _run_pipelined(LAYERS, "exact", 4)
    assert {ciera.MODE_RAW, ciera.MODE_COMPRESSED} <= modes


def test_pipelined_rans_step_matches_the_oracle():
    """The same with the RANS sender (coded exponents) on every layer."""
    modes = _run_pipelined(RANS_LAYERS, "rans", 4, seed0=10)
    assert ciera.MODE_RANS in modes


def test_pipelined_hashed_step_matches_the_oracle():
    """The same with the hashed sender (Hash128 / HashCache) on every layer,
    raw-ahead and look-back shards alike."""
    modes = _run_pipelined(LAYERS, "hashed", 4)
    assert ciera.MODE_COMPRESSED in modes


@pytest.mark.parametrize("sender", ["exact", "hashed", "rans"])
def test_captured_pipelined_step_replays_match_the_oracle(sender):
    """The pipelined step captured once into a CUDA graph (after the cold
    start, which runs eagerly), then replayed with each iteration's weights
    copied into the captured input buffers."""
    layers = RANS_LAYERS if sender == "rans" else LAYERS
    steps = 5
    seqs = _layer_seqs(layers, steps, seed0=20)
    kw = dict(rans=sender == "rans", hashed=sender == "hashed")
    gpu = [SimulatedAllgather(n, B, R, **kw) for n, R, B in layers]
    ref = [OracleAny(n, R, B, sender) for n, R, B in layers]
    bufs = [torch.empty(n, dtype=torch.int16, device="cuda") for n, _, _ in layers]
    pipe = ciera.Pipeline(len(layers))

    def check(t):
        for li, (ag, ost, s) in enumerate(zip(gpu, ref, seqs)):
            assert ag.status() == ciera.OK
            w_np = to_np_u16(s[t])
            compare_any(ag, ost, w_np, ost.step(w_np), tag=f"graph {sender} t={t} layer {li}")

    for b, s in zip(bufs, seqs):
        b.copy_(s[0].view(torch.int16))
    pipe.step(gpu, bufs)
    torch.cuda.synchronize()
    check(0)
    # a warm step is captured; the RANS histograms swap every call, so the
    # graph holds two steps (odd and even iterations)
    per_graph = 2 if sender == "rans" else 1
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            pipe.step(gpu, bufs)
    for ag in gpu:
        ag.iteration -= per_graph          # capture ran nothing
    if per_graph == 1:
        for t in range(1, steps):
            for b, s in zip(bufs, seqs):
                b.copy_(s[t].view(torch.int16))
            g.replay()
            for ag in gpu:
                ag.iteration += 1
            torch.cuda.synchronize()
            check(t)
    else:
        # both captured steps read the same input buffers: feed each replay
        # an iteration whose weights equal the previous one's in the second
        # step (an unchanged iteration), which the oracle sees as well
        for t in range(1, steps):
            for b, s in zip(bufs, seqs):
                b.copy_(s[t].view(torch.int16))
            g.replay()
            for ag in gpu:
                ag.iteration += 2
            torch.cuda.synchronize()
            for li, (ag, ost, s) in enumerate(zip(gpu, ref, seqs)):
                assert ag.status() == ciera.OK
                w_np = to_np_u16(s[t])
                ost.step(w_np)
                compare_any(ag, ost, w_np, ost.step(w_np),
                            tag=f"graph {sender} t={t} layer {li}")
