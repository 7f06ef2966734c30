"""GPU parity of ciera_compress_hashed (the paper's Hash128/HashCache change
test, CIERA Section 3.1 and Appendix A, Algorithm 1) with the oracle, byte
for byte: flags, descriptors, payloads, the HashCache, and the receiver's
rebuilt values and ExpCache."""

import numpy as np
import pytest
import torch

import oracle
from harness import eq16, raw_ahead_sequence, to_np_u16, to_np_u8
from lossless_exponent_reuse_gb300 import ciera, workloads
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = pytest.mark.gpu


def _bf16(rng, n, sigma=0.02):
    x = rng.normal(0.0, sigma, n).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _sequence(n, block, seed):
    rng = np.random.default_rng(seed)
    w0 = _bf16(rng, n)
    w1 = w0 ^ (rng.integers(0, 2, n).astype(np.uint16) * np.uint16(0x8041))
    w2 = w1.copy()
    if n:
        w2[rng.choice(n, size=max(1, n // 3000), replace=False)] ^= np.uint16(0x0080)
    w3 = w2 ^ np.uint16(0x0080)
    return [w0, w1, w2, w3]


def run_hashed_parity(seq, ranks, block, tag="", raw_ahead=True):
    n = seq[0].size
    ag = SimulatedAllgather(n, block, ranks, keep_flags=True, hashed=True, raw_ahead=raw_ahead)
    S = oracle.shard_size(n, ranks) if n else 0
    nb = oracle.num_blocks(S, block) if n else 0
    hc = np.zeros((ranks, max(nb, 1), 2), np.uint64)
    rcache = np.zeros(n, np.uint8)
    for t, w in enumerate(seq):
        wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.uint16)
        ag.step(wd)
        assert ag.status() == ciera.OK, tag
        pay, descs, flags = oracle.compress_plan_hashed(w, ranks, block, hc, cold=t == 0)
        st, out = oracle.decompress_plan(pay, descs, n, ranks, block, rcache)
        assert st == 0
        gd = ag.descriptors()
        gp = to_np_u8(ag.payloads)
        gf = to_np_u8(ag.flags)
        for r in range(ranks):
            od = descs[r]
            assert (gd[r]["mode"], gd[r]["n_changed_blocks"], gd[r]["body_bytes"],
                    gd[r]["payload_bytes"]) == (int(od["mode"]), int(od["n_changed_blocks"]),
                                                int(od["body_bytes"]),
                                                int(od["payload_bytes"])), (tag, t, r)
            pb = int(od["payload_bytes"])
            np.testing.assert_array_equal(gp[r, :pb], pay[r, :pb], err_msg=f"{tag} t={t} r={r}")
            ln = oracle.shard_len(n, ranks, r)
            k = oracle.num_blocks(ln, block) if ln else 0
            np.testing.assert_array_equal(gf[r, :k], flags[r, :k])
            np.testing.assert_array_equal(
                ag.hash_cache[r, :k].cpu().numpy().view(np.uint64), hc[r, :k],
                err_msg=f"{tag} t={t} r={r} hash cache")
        np.testing.assert_array_equal(to_np_u16(ag.out[:n]), out)
        np.testing.assert_array_equal(out, w)
        np.testing.assert_array_equal(to_np_u8(ag.recv_cache[:n]), rcache)
    return ag


CASES = [
    (131072, 4, 256),      # staged, 32-block tiles
    (131069, 4, 256),      # staged plan, ragged last tile (byte-wise tile)
    (100003, 3, 256),      # shard size not a multiple of 16: byte-wise path
    (61438, 3, 4096),
    (65536, 2, 272),       # 30-block tiles, partial last block
    (98304, 3, 16384),     # 48 KB of staging
    (50000, 2, 5000),      # block not a multiple of 8 or 16
    (40000, 2, 20000),     # block larger than a tile target
    (5, 8, 256),           # empty ranks
]


@pytest.mark.parametrize("n,ranks,block", CASES)
def test_hashed_edge_sequences(n, ranks, block):
    run_hashed_parity(_sequence(n, block, n + block), ranks, block,
                      tag=f"n={n} R={ranks} B={block}")


def test_hashed_raw_ahead_predictions_and_rewrites():
    n, ranks, block = 4 * 65536, 4, 4096
    run_hashed_parity(raw_ahead_sequence(n, ranks, block, seed=5), ranks, block,
                      tag="raw-ahead hashed")


def test_hashed_workload_1_and_clustered():
    wl = workloads.workload(1)
    run_hashed_parity([w.numpy().copy() for w in workloads.sequence(wl, 3)], wl.ranks,
                      wl.block, tag="cfg1")
    wl = workloads.small("clustered", [(64, 4096)], ranks=4, block=4096, iterations=4,
                         step=1e-3, p_block=0.1)
    ag = run_hashed_parity([w.numpy().copy() for w in workloads.sequence(wl, 4)], wl.ranks,
                           wl.block, tag="clustered")
    assert any(d["mode"] == ciera.MODE_COMPRESSED for d in ag.descriptors())


def test_hashed_matches_exact_sender_on_workload_2_full_size():
    wl = workloads.workload(2)
    n = wl.layer_numel
    exact = SimulatedAllgather(n, wl.block, wl.ranks, keep_flags=True)
    hashed = SimulatedAllgather(n, wl.block, wl.ranks, keep_flags=True, hashed=True)
    w = workloads.initial_layer(wl, 0, "cuda")
    for t in range(3):
        if t:
            w = workloads.step_layer(wl, w, 0, t)
        exact.compress(w)
        hashed.compress(w)
        assert exact.descriptors() == hashed.descriptors()
        assert torch.equal(exact.flags, hashed.flags)
        for r, d in enumerate(exact.descriptors()):
            assert torch.equal(exact.payloads[r, :d["payload_bytes"]],
                               hashed.payloads[r, :d["payload_bytes"]])
        hashed.decompress()
        exact.decompress()
        assert eq16(hashed.out[:n], w)
    assert exact.status() == ciera.OK and hashed.status() == ciera.OK
