"""GPU parity: libciera's kernels against the CPU oracle, byte for byte.

Cases span several tiles, ragged tails, every code path (staged and
byte-wise, multi-block tiles, blocks larger than a tile, empty ranks, raw
payloads that hold unchanged blocks) and the method's degenerate iterations:
cold start, zero exponent change, sparse change, clustered change, every
exponent changed.  CIERA Section 3.1 and Appendix A, Algorithm 1.
"""
import numpy as np
import pytest
import torch

from harness import eq16, exps_dev, raw_ahead_sequence, run_parity
from lossless_exponent_reuse_gb300 import ciera, workloads
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = pytest.mark.gpu


def _bf16(rng, n, sigma=0.02):
    x = rng.normal(0.0, sigma, n).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def edge_sequence(n, block, seed=0):
    """cold, zero-change, sparse, clustered, all-changed, sparse again."""
    rng = np.random.default_rng(seed)
    w0 = _bf16(rng, n)
    w1 = w0 ^ (rng.integers(0, 2, n).astype(np.uint16) * np.uint16(0x8041))  # sign/mantissa only
    w2 = w1.copy()
    idx = rng.choice(n, size=max(1, n // 2000), replace=False) if n else []
    w2[idx] ^= np.uint16(0x0080)
    w3 = w2.copy()
    nb = (n + block - 1) // block
    for k in rng.choice(max(nb, 1), size=max(1, nb // 5), replace=False) if n else []:
        j = k * block + rng.integers(0, max(1, min(block, n - k * block)))
        if j < n:
            w3[j] ^= np.uint16(0x0100)
    w4 = w3 ^ np.uint16(0x0080)
    w5 = w4.copy()
    if n:
        w5[rng.integers(0, n, 3)] ^= np.uint16(0x0080)
    return [w0, w1, w2, w3, w4, w5]


def test_workload_1_three_iterations():
    wl = workloads.workload(1)
    seq = [w.numpy().copy() for w in workloads.sequence(wl, wl.iterations)]
    run_parity(seq, wl.ranks, wl.block, tag="cfg1")


CASES = [
    # (numel, ranks, block)
    (131072, 4, 256),      # staged, 16-block tiles
    (131069, 4, 256),      # staged plan, ragged last tile of the last shard
    (100003, 3, 256),      # shard size not a multiple of 16: byte-wise path
    (61438, 3, 4096),      # staged, one block per tile, ragged tail
    (65536, 2, 272),       # staged, 15-block tiles, partial last block
    (98304, 3, 16384),     # staged, 64 KB of shared memory per CTA
    (40000, 2, 20000),     # block larger than the staged limit
    (50000, 2, 5000),      # block not a multiple of 16
    (70000, 7, 100),       # small odd block
    (12345, 2, 1),         # one value per block: raw payloads may hold unchanged blocks
    (10000, 5, 3),
    (5, 8, 4),             # empty ranks
    (0, 3, 4),             # empty tensor
    (8192, 1, 16),         # single rank
]


@pytest.mark.parametrize("n,ranks,block", CASES)
def test_edge_sequences(n, ranks, block):
    run_parity(edge_sequence(n, block, seed=n + block), ranks, block,
               tag=f"n={n} R={ranks} B={block}")


@pytest.mark.parametrize("n,ranks,block", [c for c in CASES if c[2] >= 256])
def test_edge_sequences_look_back_only(n, ranks, block):
    # the same sequences with raw-ahead off: every shard takes the look-back
    run_parity(edge_sequence(n, block, seed=n + block), ranks, block,
               tag=f"look-back n={n} R={ranks} B={block}", raw_ahead=False)


@pytest.mark.parametrize("n,ranks,block", [
    (4 * 65536, 4, 4096),       # 8 tiles per shard
    (3 * 40960, 3, 256),        # 32-block tiles, 5 tiles per shard
    (2 * 98304, 2, 16384),      # one block per tile
    (81904, 20, 4096),          # partial last shard of 4080 values: raw-ahead too
    (81914, 20, 4096),          # partial last shard of 4090 values: look-back, byte-wise
    (304, 20, 256),             # 16-value shards of one partial block, an empty last rank
])
def test_raw_ahead_predictions_and_rewrites(n, ranks, block):
    seq = raw_ahead_sequence(n, ranks, block, seed=n)
    ag, _ = run_parity(seq, ranks, block, tag=f"raw-ahead n={n} B={block}")
    d = ag.descriptors()
    assert d[0]["mode"] == ciera.MODE_RAW
    if ag.plan.info.blocks_per_shard > 1:              # the last iteration is even
        assert d[1]["mode"] == ciera.MODE_COMPRESSED


def test_raw_payload_with_one_unchanged_block():
    # B = 16 on 4096-value shards: the bitmap (32 bytes) is larger than one
    # block, so "all blocks but one changed" is raw yet holds an unchanged block
    n, R, B = 8192, 2, 16
    p = ciera.Plan(n, B, R)
    assert p.info.raw_fixup
    rng = np.random.default_rng(9)
    w0 = _bf16(rng, n)
    w1 = w0.copy()
    for k in range(n // B):
        if k % (4096 // B) != 7:
            w1[k * B + 3] ^= np.uint16(0x0080)
    ag, ost = run_parity([w0, w1], R, B, tag="raw-with-unchanged")
    d = ag.descriptors()
    assert all(x["mode"] == ciera.MODE_RAW for x in d)
    assert all(x["n_changed_blocks"] == 4096 // B - 1 for x in d)


def test_clustered_workload_compresses():
    wl = workloads.small("clustered", [(64, 4096)], ranks=4, block=4096, iterations=4,
                         step=1e-3, p_block=0.1)
    seq = [w.numpy().copy() for w in workloads.sequence(wl, wl.iterations)]
    ag, _ = run_parity(seq, wl.ranks, wl.block, tag="clustered")
    assert any(x["mode"] == ciera.MODE_COMPRESSED for x in ag.descriptors())


def test_rank_range_matches_full_launch():
    n, R, B = 131072, 4, 256
    seq = edge_sequence(n, B, seed=3)[:3]
    full = SimulatedAllgather(n, B, R, keep_flags=True)
    part = SimulatedAllgather(n, B, R, keep_flags=True)
    S = full.plan.info.shard_len
    for t, w in enumerate(seq):
        wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.uint16)
        full.compress(wd)
        for r in range(R):  # one rank per call, as a real sender would
            part.plan.compress(wd[r * S:(r + 1) * S], part.sender_cache[r * S:(r + 1) * S],
                               part.payloads[r:r + 1], part.descs[r:r + 1], part.workspace,
                               cold=t == 0, rank_begin=r, rank_count=1,
                               flags_out=part.flags[r:r + 1])
        assert full.descriptors() == part.descriptors()
        for r, d in enumerate(full.descriptors()):
            pb = d["payload_bytes"]
            assert torch.equal(full.payloads[r, :pb], part.payloads[r, :pb])
        assert torch.equal(full.flags, part.flags)
        assert torch.equal(full.sender_cache, part.sender_cache)
        full.decompress()
        part.iteration += 1


def test_corrupt_descriptor_is_reported_and_skipped():
    n, R, B = 131072, 4, 256
    seq = edge_sequence(n, B, seed=4)
    ag = SimulatedAllgather(n, B, R)
    for w in seq[:2]:
        ag.step(torch.from_numpy(w.view(np.int16)).cuda().view(torch.uint16))
        assert ag.status() == ciera.OK
    w = torch.from_numpy(seq[2].view(np.int16)).cuda().view(torch.uint16)
    ag.compress(w)
    d = ag.descriptors()
    assert d[1]["mode"] == ciera.MODE_COMPRESSED
    before = ag.out.clone()
    # lie about the number of changed blocks of rank 1
    ag.descs[1, 4:8] = torch.tensor(list((d[1]["n_changed_blocks"] + 1).to_bytes(4, "little")),
                                    dtype=torch.uint8, device="cuda")
    ag.decompress()
    assert ag.status() == ciera.E_CORRUPT
    S = ag.plan.info.shard_len
    assert eq16(ag.out[S:2 * S], before[S:2 * S])                  # skipped
    assert eq16(ag.out[:S], w[:S]) and eq16(ag.out[2 * S:], w[2 * S:])
    assert ag.status() == ciera.OK                                  # cleared


@pytest.mark.parametrize("raw_ahead", [True, False])
def test_bounded_wait_reports_timeout_and_context_survives(raw_ahead):
    # a cold call is raw-ahead: the shard's last tile waits for tile 0's
    # aggregate; without raw-ahead every later tile's look-back waits for it
    n, R, B = 4 * 4096 * 8, 4, 4096                                # 8 tiles per shard
    rng = np.random.default_rng(11)
    w = torch.from_numpy(_bf16(rng, n).view(np.int16)).cuda().view(torch.uint16)
    ag = SimulatedAllgather(n, B, R)
    ciera.set_wait_timeout_ns(2_000_000)
    try:
        extra = ciera.DEBUG_SKIP_FIRST_PUBLISH | (0 if raw_ahead else ciera.NO_RAW_AHEAD)
        ag.plan.compress(w, ag.sender_cache, ag.payloads, ag.descs, ag.workspace, cold=True,
                         extra_flags=extra)
        assert ag.status() == ciera.E_TIMEOUT
    finally:
        ciera.set_wait_timeout_ns(1_000_000_000)
    # the context is still usable and the next call is correct
    ag.iteration = 0
    out = ag.step(w)
    assert ag.status() == ciera.OK
    assert eq16(out[:n], w)


def test_cache_invariants_and_round_trip_on_workload_2_shape_slice():
    # one expert's three matrices of the OLMoE layer, 16 ranks, block 4096
    wl = workloads.small("expert", [(2048, 1024), (2048, 1024), (1024, 2048)], ranks=16,
                         block=4096, iterations=4, step=1e-5)
    seq = [w.numpy().copy() for w in workloads.sequence(wl, wl.iterations)]
    ag, _ = run_parity(seq, wl.ranks, wl.block, tag="expert")
    w_last = torch.from_numpy(seq[-1].view(np.int16)).cuda().view(torch.uint16)
    assert torch.equal(ag.recv_cache, exps_dev(w_last))
    assert torch.equal(ag.sender_cache, exps_dev(w_last))


def test_step_host_round_trips_every_edge_case():
    # weights from pinned host memory, rebuilt weights back (ciera_step_host),
    # over the edge-case sequence, in chunks of one rank
    n, R, B = 131072, 4, 256
    seq = edge_sequence(n, B, seed=21)
    ag = SimulatedAllgather(n, B, R)
    session = ciera.HostSession(4)
    w_dev = torch.empty(n, dtype=torch.int16, device="cuda")
    host = [torch.from_numpy(w.view(np.int16)).pin_memory() for w in seq]
    outs = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in seq]
    for w, o in zip(host, outs):
        ag.step_host(session, w, o, w_dev, chunks=4)
    torch.cuda.synchronize()
    assert ag.status() == ciera.OK
    for w, o in zip(host, outs):
        assert torch.equal(w, o)
