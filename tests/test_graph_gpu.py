"""A warm step (compress of all ranks + gather-decompress) captured once into
a CUDA graph and replayed iteration after iteration, with each iteration's
weights copied into the captured input buffer, must give byte for byte what
eager calls give.  Replays reuse the captured kernel arguments, so the
look-back tags must come from the device (per workspace), not the host."""
import numpy as np
import pytest
import torch

from lossless_exponent_reuse_gb300 import ciera
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = pytest.mark.gpu


def _seq(n, steps, seed, block):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 0.02, n).astype(np.float32)
    w = (x.view(np.uint32) >> 16).astype(np.uint16)
    out = [w]
    for t in range(1, steps):
        w = w.copy()
        # exponent changes in about an eighth of the blocks
        w[rng.choice(n, size=max(1, n // (8 * block)), replace=False)] ^= np.uint16(0x0080)
        w ^= rng.integers(0, 2, n).astype(np.uint16) * np.uint16(0x0001)     # mantissa noise
        out.append(w)
    return [torch.from_numpy(v.view(np.int16)).cuda() for v in out]


@pytest.mark.parametrize("n,ranks,block,hashed", [(131072, 4, 256, False),
                                                  (3 * 65536, 3, 4096, False),
                                                  (131072, 4, 256, True)])
def test_graph_replays_match_eager(n, ranks, block, hashed):
    torch.cuda.set_device(0)
    seq = _seq(n, 6, n + block, block)
    eager = SimulatedAllgather(n, block, ranks, keep_flags=True, hashed=hashed)
    graphed = SimulatedAllgather(n, block, ranks, keep_flags=True, hashed=hashed)
    w_buf = torch.empty(n, dtype=torch.int16, device="cuda")
    # iteration 0 (the cold start) eagerly on both
    eager.step(seq[0])
    w_buf.copy_(seq[0])
    graphed.step(w_buf)
    torch.cuda.synchronize()
    # capture one warm step
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.compress(w_buf)
        graphed.decompress()
    for t in range(1, len(seq)):
        w_buf.copy_(seq[t])
        g.replay()
        eager.step(seq[t])
        torch.cuda.synchronize()
        assert eager.status() == ciera.OK and graphed.status() == ciera.OK
        de, dg = eager.descriptors(), graphed.descriptors()
        assert de == dg, t
        for r, d in enumerate(de):
            pb = d["payload_bytes"]
            assert torch.equal(eager.payloads[r, :pb], graphed.payloads[r, :pb]), (t, r)
        assert torch.equal(eager.flags, graphed.flags)
        assert torch.equal(eager.out.view(torch.int16), graphed.out.view(torch.int16))
        assert torch.equal(graphed.out[:n].view(torch.int16), seq[t])
        assert torch.equal(eager.recv_cache, graphed.recv_cache)
        if hashed:
            assert torch.equal(eager.hash_cache, graphed.hash_cache)
        else:
            assert torch.equal(eager.sender_cache, graphed.sender_cache)
    assert any(d["mode"] == ciera.MODE_COMPRESSED for d in graphed.descriptors())
