"""A warm step (compress of all ranks + gather-decompress) captured once into
a CUDA graph and replayed iteration after iteration, with each iteration's
weights copied into the captured input buffer, must give byte for byte what
the CPU oracle gives: flags, descriptors, payloads, rebuilt values and both
sides' state.  Replays reuse the captured kernel arguments, so the look-back
tags must come from the device (per workspace), not the host.
CIERA Section 3.1 and Appendix A, Algorithm 1."""
import numpy as np
import pytest
import torch

from harness import OracleAny, compare_any, to_np_u16
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
def test_graph_replays_match_the_oracle(n, ranks, block, hashed):
    torch.cuda.set_device(0)
    seq = _seq(n, 6, n + block, block)
    graphed = SimulatedAllgather(n, block, ranks, keep_flags=True, hashed=hashed)
    ost = OracleAny(n, ranks, block, "hashed" if hashed else "exact")
    w_buf = torch.empty(n, dtype=torch.int16, device="cuda")
    # iteration 0 (the cold start) eagerly
    w_buf.copy_(seq[0])
    graphed.step(w_buf)
    torch.cuda.synchronize()
    w_np = to_np_u16(seq[0])
    compare_any(graphed, ost, w_np, ost.step(w_np), tag="t=0", check_flags=True)
    # capture one warm step
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.compress(w_buf)
        graphed.decompress()
    graphed.iteration -= 1          # capture ran nothing
    for t in range(1, len(seq)):
        w_buf.copy_(seq[t])
        g.replay()
        graphed.iteration += 1
        torch.cuda.synchronize()
        assert graphed.status() == ciera.OK
        w_np = to_np_u16(seq[t])
        compare_any(graphed, ost, w_np, ost.step(w_np), tag=f"t={t}", check_flags=True)
    assert any(d["mode"] == ciera.MODE_COMPRESSED for d in graphed.descriptors())
