"""GPU parity of ciera_compress_rans and the RANS receiver with the oracle
(CIERA Section 3.1: the changed exponents entropy-coded with ANS), byte for
byte: descriptors, payloads (sign+mantissa bytes, bitmap, frequency table,
record offsets, rANS records, padding), flags, the exponent histograms,
both exponent caches and the rebuilt values."""
import numpy as np
import pytest
import torch

import oracle
from harness import to_np_u16, to_np_u8
from lossless_exponent_reuse_gb300 import ciera
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = pytest.mark.gpu


def _bf16(rng, n, sigma=0.02):
    x = rng.normal(0.0, sigma, n).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _scale_some(rng, w, frac, block):
    """Multiply a random subset of values (in a random subset of blocks) by
    factors that move their exponents; other blocks keep their exponents."""
    n = w.size
    out = w.copy()
    if n == 0:
        return out
    nb = (n + block - 1) // block
    blocks = rng.choice(nb, size=max(1, int(nb * frac)), replace=False)
    for k in blocks:
        lo, hi = k * block, min(n, (k + 1) * block)
        idx = lo + rng.choice(hi - lo, size=max(1, (hi - lo) // 50), replace=False)
        f = (out[idx].astype(np.uint32) << 16).view(np.float32)
        with np.errstate(over="ignore", invalid="ignore"):   # inf/NaN patterns are fine
            f = f * rng.choice(np.array([0.25, 0.5, 2.0, 3.0], np.float32), size=idx.size)
        out[idx] = (f.view(np.uint32) >> 16).astype(np.uint16)
    return out


def rans_sequence(n, block, seed):
    rng = np.random.default_rng(seed)
    w0 = _bf16(rng, n)
    w1 = _scale_some(rng, w0, 0.3, block)       # some blocks change
    w2 = w1.copy()                              # nothing changes
    w3 = w2 ^ np.uint16(0x0080)                 # every exponent changes (low bit)
    w4 = rng.integers(0, 1 << 16, n, dtype=np.uint16)  # table of w3 fits w4 badly: raw
    w5 = _scale_some(rng, w4, 0.2, block)       # sparse changes under a flat table
    w6 = _scale_some(rng, _bf16(rng, n), 1.0, block)
    return [w0, w1, w2, w3, w4, w5, w6]


class OracleRans:
    """R oracle senders and one oracle receiver, across iterations."""

    def __init__(self, n, ranks, block):
        self.n, self.ranks, self.block = n, ranks, block
        self.scache = np.zeros(n, np.uint8)
        self.rcache = np.zeros(n, np.uint8)
        self.hist = np.zeros((ranks, 256), np.uint32)
        self.t = 0

    def step(self, w):
        n, R, B = self.n, self.ranks, self.block
        res = []
        out = np.zeros(n, np.uint16)
        hist_cur = np.zeros((R, 256), np.uint32)
        for r in range(R):
            b = oracle.shard_begin(n, R, r)
            ln = oracle.shard_len(n, R, r)
            sc = self.scache[b:b + ln].copy()
            pay, flags, desc, h = oracle.compress_shard_rans(w[b:b + ln], B, sc, self.t == 0,
                                                             self.hist[r])
            self.scache[b:b + ln] = sc
            hist_cur[r] = h
            rc = self.rcache[b:b + ln].copy()
            st, o = oracle.decompress_shard_any(pay, desc, ln, B, rc)
            assert st == 0
            self.rcache[b:b + ln] = rc
            out[b:b + ln] = o
            res.append((pay, flags, desc))
        self.hist = hist_cur
        self.t += 1
        return res, out


def run_rans_parity(seq, ranks, block, tag=""):
    n = seq[0].size
    ag = SimulatedAllgather(n, block, ranks, keep_flags=True, rans=True)
    ref = OracleRans(n, ranks, block)
    modes = set()
    for t, w in enumerate(seq):
        wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.uint16)
        ag.step(wd)
        assert ag.status() == ciera.OK, (tag, t)
        res, out = ref.step(w)
        gd = ag.descriptors()
        gp = to_np_u8(ag.payloads)
        gf = to_np_u8(ag.flags)
        gh = ag.hist[t % 2 ^ 1].cpu().numpy().view(np.uint32)
        for r in range(ranks):
            pay, flags, od = res[r]
            modes.add(int(od["mode"]))
            assert (gd[r]["mode"], gd[r]["n_changed_blocks"], gd[r]["body_bytes"],
                    gd[r]["payload_bytes"]) == (int(od["mode"]), int(od["n_changed_blocks"]),
                                                int(od["body_bytes"]),
                                                int(od["payload_bytes"])), (tag, t, r)
            pb = int(od["payload_bytes"])
            np.testing.assert_array_equal(gp[r, :pb], pay[:pb], err_msg=f"{tag} t={t} r={r}")
            k = flags.size
            np.testing.assert_array_equal(gf[r, :k], flags, err_msg=f"{tag} t={t} r={r} flags")
            np.testing.assert_array_equal(gh[r], ref.hist[r], err_msg=f"{tag} t={t} r={r} hist")
        np.testing.assert_array_equal(to_np_u16(ag.out[:n]), out, err_msg=f"{tag} t={t}")
        np.testing.assert_array_equal(out, w)
        np.testing.assert_array_equal(to_np_u8(ag.sender_cache[:n]), ref.scache)
        np.testing.assert_array_equal(to_np_u8(ag.recv_cache[:n]), ref.rcache)
    return ag, modes


CASES = [
    (131072, 4, 256),       # 32-block tiles
    (90048, 3, 4096),       # 2-block tiles, partial last block
    (98304, 3, 16384),      # one block per tile
    (65536, 2, 272),        # 30-block tiles, partial last block
    (150400, 2, 1504),      # 5-block tiles; the receiver's 10-block tiles straddle bitmap words
    (131056, 32, 1024),     # 32 ranks, a short last shard
    (8176, 32, 256),        # tiny shards (always raw: sections alone reach 2*len)
    (76512, 300, 256),      # 300 ranks: a short shard and an empty one
]


@pytest.mark.parametrize("n,ranks,block", CASES)
def test_rans_parity(n, ranks, block):
    plan = ciera.Plan(n, block, ranks)
    assert plan.info.fast_path and plan.info.shard_len % 16 == 0 and n % 16 == 0
    seq = rans_sequence(n, block, seed=n * 31 + ranks * 7 + block)
    _, modes = run_rans_parity(seq, ranks, block, tag=f"{n}/{ranks}/{block}")
    if plan.info.shard_len >= 4096:
        assert modes == {ciera.MODE_RAW, ciera.MODE_RANS}, modes
    else:
        assert modes == {ciera.MODE_RAW}, modes


def test_rans_multi_tile_lookback():
    # 4 Mi values: 128 tiles per shard, records placed by the look-back
    seq = rans_sequence(1 << 22, 4096, seed=11)[:3]
    ag, modes = run_rans_parity(seq, 4, 4096, tag="4Mi")
    assert ciera.MODE_RANS in modes


def test_rans_record_sizes_match_descriptors():
    """Payload bytes are D plus the records, and the offset table ends there."""
    n, R, B = 131072, 4, 256
    seq = rans_sequence(n, B, seed=5)[:2]
    ag, _ = run_rans_parity(seq, R, B)
    gp = to_np_u8(ag.payloads)
    for r, d in enumerate(ag.descriptors()):
        if d["mode"] != ciera.MODE_RANS:
            continue
        ln = oracle.shard_len(n, R, r)
        nb = oracle.num_blocks(ln, B)
        A = (ln + 15) // 16 * 16
        C = (A + (nb + 7) // 8 + 15) // 16 * 16
        O = C + 512
        offs = gp[r, O:O + 4 * (nb + 1)].view(np.uint32)
        assert d["body_bytes"] + int(offs[nb]) == d["payload_bytes"]
        assert np.all(np.diff(offs.astype(np.int64)) >= 0)


def _compressed_rans_state(n=131072, R=4, B=256, seed=3):
    seq = rans_sequence(n, B, seed=seed)[:2]
    ag, _ = run_rans_parity(seq, R, B)
    return ag


def test_rans_corrupt_table_is_reported():
    ag = _compressed_rans_state()
    d = ag.descriptors()
    r = next(i for i, x in enumerate(d) if x["mode"] == ciera.MODE_RANS)
    ln = ag.plan.info.shard_len
    nb = ag.plan.info.blocks_per_shard
    C = ((ln + 15) // 16 * 16 + (nb + 7) // 8 + 15) // 16 * 16
    # the oracle rejects the same corruption
    pay = to_np_u8(ag.payloads)[r, :d[r]["payload_bytes"]].copy()
    pay[C:C + 2] = 0
    rc = np.zeros(ln, np.uint8)
    st, _ = oracle.decompress_shard_any(pay, d[r], ln, 256, rc)
    assert st != 0
    ag.payloads[r, C:C + 2] = 0
    ag.decompress()
    assert ag.status() == ciera.E_CORRUPT


def test_rans_corrupt_record_is_reported():
    ag = _compressed_rans_state()
    d = ag.descriptors()
    r = next(i for i, x in enumerate(d) if x["mode"] == ciera.MODE_RANS and x["n_changed_blocks"])
    D = d[r]["body_bytes"]
    pay = to_np_u8(ag.payloads)[r, :d[r]["payload_bytes"]].copy()
    # the first record's lane 0 word count, one larger
    cnt = int(pay[D]) | (int(pay[D + 1]) << 8)
    bad = cnt + 1
    pay[D], pay[D + 1] = bad & 0xFF, bad >> 8
    rc = to_np_u8(ag.recv_cache).copy()
    ln = ag.plan.info.shard_len
    st, _ = oracle.decompress_shard_any(pay, d[r], ln, 256, rc[r * ln:(r + 1) * ln])
    assert st != 0
    ag.payloads[r, D] = bad & 0xFF
    ag.payloads[r, D + 1] = bad >> 8
    ag.decompress()
    assert ag.status() == ciera.E_CORRUPT


def test_rans_payload_needs_the_rans_flag():
    ag = _compressed_rans_state()
    assert any(x["mode"] == ciera.MODE_RANS for x in ag.descriptors())
    ag.plan.decompress(ag.payloads, ag.descs, ag.recv_cache, ag.out, ag.workspace, rans=False)
    assert ag.status() == ciera.E_CORRUPT


def test_rans_tile_records_larger_than_staging():
    """A tile whose records exceed one byte per value (high-entropy changed
    exponents) is decoded from global memory instead of shared memory."""
    n, R, B = 4 * 65536, 4, 4096
    rng = np.random.default_rng(23)
    w0 = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    w1 = w0.copy()
    S = n // R
    for r in range(R):
        w1[r * S:r * S + 2 * B] = rng.integers(0, 1 << 16, 2 * B, dtype=np.uint16)
    w2 = w1.copy()
    w2[3 * B:4 * B] ^= np.uint16(0x0080)        # one block of tile 1, rank 0
    ag, modes = run_rans_parity([w0, w1, w2], R, B, tag="big-records")
    assert ciera.MODE_RANS in modes
    # the oracle's payload of iteration 1 had > T*B record bytes in tile 0
    ref = OracleRans(n, R, B)
    ref.step(w0)
    res, _ = ref.step(w1)
    pay, _, d = res[0]
    assert int(d["mode"]) == ciera.MODE_RANS
    nb = S // B
    A = S
    C = (A + (nb + 7) // 8 + 15) // 16 * 16
    offs = pay[C + 512:C + 512 + 4 * (nb + 1)].view(np.uint32)
    assert int(offs[2]) - int(offs[0]) > 2 * B


def test_rans_receiver_rejects_compressed_payloads():
    """CIERA_DECOMPRESS_RANS takes the RANS sender's modes (RANS, RAW); a
    COMPRESSED payload of the exact sender is reported as corrupt."""
    n, R, B = 131072, 4, 256
    seq = rans_sequence(n, B, seed=9)[:2]
    ag = SimulatedAllgather(n, B, R)
    for w in seq:
        ag.step(torch.from_numpy(w.view(np.int16)).cuda().view(torch.uint16))
    assert ag.status() == ciera.OK
    assert any(d["mode"] == ciera.MODE_COMPRESSED for d in ag.descriptors())
    ag.plan.decompress(ag.payloads, ag.descs, ag.recv_cache, ag.out, ag.workspace, rans=True)
    assert ag.status() == ciera.E_CORRUPT


def test_rans_rank_ranges_match_full_launch():
    """One RANS call per rank (each with its own histogram rows and the
    payload, descriptor and flag rows of that rank) gives the bytes of one
    call over all ranks, including the partial shard."""
    n, R, B = 131056, 32, 1024
    seq = rans_sequence(n, B, seed=21)[:4]
    full = SimulatedAllgather(n, B, R, keep_flags=True, rans=True)
    part = SimulatedAllgather(n, B, R, keep_flags=True, rans=True)
    S = full.plan.info.shard_len
    for t, w in enumerate(seq):
        wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.uint16)
        full.compress(wd)
        prev, cur = part.hist[t % 2], part.hist[(t + 1) % 2]
        for r in range(R):
            lo, hi = r * S, min(n, (r + 1) * S)
            part.plan.compress_rans(wd[lo:hi], part.sender_cache[lo:hi], prev[r:r + 1],
                                    cur[r:r + 1], part.payloads[r:r + 1], part.descs[r:r + 1],
                                    part.workspace, cold=t == 0, rank_begin=r, rank_count=1,
                                    flags_out=part.flags[r:r + 1])
        assert part.status() == ciera.OK
        assert full.descriptors() == part.descriptors(), t
        for r, d in enumerate(full.descriptors()):
            pb = d["payload_bytes"]
            assert torch.equal(full.payloads[r, :pb], part.payloads[r, :pb]), (t, r)
        assert torch.equal(full.flags, part.flags)
        assert torch.equal(full.sender_cache, part.sender_cache)
        assert torch.equal(full.hist[(t + 1) % 2], cur)
        full.decompress()
        part.iteration += 1
        assert torch.equal(full.out[:n].view(torch.int16), wd.view(torch.int16))
