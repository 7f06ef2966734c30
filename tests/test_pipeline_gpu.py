"""Computation-communication pipelining on one GPU (CIERA Section 3.3):
compress(i+1) on a side stream overlapping decompress(i).  The pipelined
step must equal layer-by-layer calls byte for byte, eagerly and when the
step is captured into a CUDA graph and replayed."""
import pytest
import torch

from lossless_exponent_reuse_gb300 import ciera, workloads
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = pytest.mark.gpu

LAYERS = [(131072, 4, 256), (196608, 3, 4096), (100003, 3, 256), (65536, 2, 272)]


def _layer_seqs(steps):
    out = []
    for li, (n, R, B) in enumerate(LAYERS):
        wl = workloads.small(f"L{li}", [(n,)], ranks=R, block=B, iterations=steps, step=1e-3,
                             seed=li, p_block=0.2)
        out.append([w.cuda() for w in workloads.sequence(wl, steps)])
    return out


def _compare(a, b, tag):
    assert a.descriptors() == b.descriptors(), tag
    for r, d in enumerate(a.descriptors()):
        pb = d["payload_bytes"]
        assert torch.equal(a.payloads[r, :pb], b.payloads[r, :pb]), (tag, r)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16)), tag
    assert torch.equal(a.sender_cache, b.sender_cache), tag
    assert torch.equal(a.recv_cache, b.recv_cache), tag


def test_pipelined_step_equals_layer_by_layer():
    seqs = _layer_seqs(4)
    seq_layers = [SimulatedAllgather(n, B, R) for n, R, B in LAYERS]
    pipe_layers = [SimulatedAllgather(n, B, R) for n, R, B in LAYERS]
    pipe = ciera.Pipeline(len(LAYERS))
    for t in range(4):
        for ag, s in zip(seq_layers, seqs):
            ag.step(s[t])
        pipe.step(pipe_layers, [s[t] for s in seqs])
        torch.cuda.synchronize()
        for li, (a, b) in enumerate(zip(seq_layers, pipe_layers)):
            assert b.status() == ciera.OK
            _compare(a, b, f"t={t} layer {li}")
            assert torch.equal(b.out[:LAYERS[li][0]].view(torch.int16),
                               seqs[li][t].view(torch.int16))


def test_captured_pipelined_step_replays():
    seqs = _layer_seqs(5)
    eager = [SimulatedAllgather(n, B, R) for n, R, B in LAYERS]
    graphed = [SimulatedAllgather(n, B, R) for n, R, B in LAYERS]
    bufs = [torch.empty(n, dtype=torch.int16, device="cuda") for n, _, _ in LAYERS]
    pipe = ciera.Pipeline(len(LAYERS))
    for ag, s in zip(eager, seqs):
        ag.step(s[0])
    for ag, b, s in zip(graphed, bufs, seqs):
        b.copy_(s[0].view(torch.int16))
        ag.step(b)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pipe.step(graphed, bufs)
    for ag in graphed:
        ag.iteration -= 1          # capture ran nothing
    for t in range(1, 5):
        for b, s in zip(bufs, seqs):
            b.copy_(s[t].view(torch.int16))
        g.replay()
        for ag, s in zip(eager, seqs):
            ag.step(s[t])
        torch.cuda.synchronize()
        for li, (a, b) in enumerate(zip(eager, graphed)):
            assert b.status() == ciera.OK
            _compare(a, b, f"replay t={t} layer {li}")


RANS_LAYERS = [(131072, 4, 256), (196608, 3, 4096), (65536, 2, 272)]


def test_pipelined_rans_step_equals_layer_by_layer():
    """The same with the RANS sender (coded exponents) on every layer."""
    seqs = []
    for li, (n, R, B) in enumerate(RANS_LAYERS):
        wl = workloads.small(f"R{li}", [(n,)], ranks=R, block=B, iterations=4, step=1e-3,
                             seed=10 + li, p_block=0.2)
        seqs.append([w.cuda() for w in workloads.sequence(wl, 4)])
    seq_layers = [SimulatedAllgather(n, B, R, rans=True) for n, R, B in RANS_LAYERS]
    pipe_layers = [SimulatedAllgather(n, B, R, rans=True) for n, R, B in RANS_LAYERS]
    pipe = ciera.Pipeline(len(RANS_LAYERS))
    modes = set()
    for t in range(4):
        for ag, s in zip(seq_layers, seqs):
            ag.step(s[t])
        pipe.step(pipe_layers, [s[t] for s in seqs])
        torch.cuda.synchronize()
        for li, (a, b) in enumerate(zip(seq_layers, pipe_layers)):
            assert b.status() == ciera.OK
            _compare(a, b, f"rans t={t} layer {li}")
            assert all(torch.equal(x, y) for x, y in zip(a.hist, b.hist))
            modes.update(d["mode"] for d in b.descriptors())
            assert torch.equal(b.out[:RANS_LAYERS[li][0]].view(torch.int16),
                               seqs[li][t].view(torch.int16))
    assert ciera.MODE_RANS in modes


def test_pipelined_hashed_step_equals_layer_by_layer():
    """The same with the hashed sender (Hash128 / HashCache) on every layer,
    raw-ahead and look-back shards alike."""
    seqs = _layer_seqs(4)
    seq_layers = [SimulatedAllgather(n, B, R, hashed=True) for n, R, B in LAYERS]
    pipe_layers = [SimulatedAllgather(n, B, R, hashed=True) for n, R, B in LAYERS]
    pipe = ciera.Pipeline(len(LAYERS))
    for t in range(4):
        for ag, s in zip(seq_layers, seqs):
            ag.step(s[t])
        pipe.step(pipe_layers, [s[t] for s in seqs])
        torch.cuda.synchronize()
        for li, (a, b) in enumerate(zip(seq_layers, pipe_layers)):
            assert b.status() == ciera.OK
            assert a.descriptors() == b.descriptors(), (t, li)
            for r, d in enumerate(a.descriptors()):
                pb = d["payload_bytes"]
                assert torch.equal(a.payloads[r, :pb], b.payloads[r, :pb]), (t, li, r)
            assert torch.equal(a.hash_cache, b.hash_cache), (t, li)
            assert torch.equal(a.recv_cache, b.recv_cache), (t, li)
            assert torch.equal(b.out[:LAYERS[li][0]].view(torch.int16),
                               seqs[li][t].view(torch.int16))
