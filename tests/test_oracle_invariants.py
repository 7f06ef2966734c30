"""Pins the oracle with invariants the method fixes (CIERA Section 3.1,
Section 3.2, Appendix A Algorithm 1; lossless reconstruction, Section 4.6):

* round trip: the receiver rebuilds every value bit for bit;
* sizes: zero exponent change -> len + ceil(n_b/8) bytes; every block
  changed -> raw, body identical to the input bytes; in general
  len + (values in changed blocks) + ceil(n_b/8), raw when not smaller;
* caches: after a call both hold the exponents of the new weights;
* flag truth: a block is flagged iff some exponent differs between the
  previous and the current weights (computed from the weights themselves);
* exhaustive tiny cases over every subset of changed positions.
"""

import numpy as np
import pytest

import oracle
from lossless_exponent_reuse_gb300 import workloads


def _exps(w):
    # exponent field by numeric decoding (frexp) -- independent of bit masks
    f = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a = np.abs(f)
    out = np.zeros(w.shape, dtype=np.int64)
    fin = np.isfinite(a) & (a >= 2.0 ** -126)
    _, e2 = np.frexp(a[fin])
    out[fin] = e2 - 1 + 127
    out[~np.isfinite(a)] = 255
    return out.astype(np.uint8)


def _expected_sizes(w_prev, w_cur, B, cold):
    n = w_cur.size
    nb = (n + B - 1) // B
    flags = np.zeros(nb, dtype=np.uint8)
    ep, ec = _exps(w_prev), _exps(w_cur)
    for k in range(nb):
        lo, hi = k * B, min(n, (k + 1) * B)
        flags[k] = 1 if (cold or np.any(ep[lo:hi] != ec[lo:hi])) else 0
    changed_vals = sum(min(n, (k + 1) * B) - k * B for k in range(nb) if flags[k])
    bm = (nb + 7) // 8
    comp = n + changed_vals + bm
    raw = cold or n == 0 or comp >= 2 * n
    return flags, raw, (2 * n if raw else comp), (2 * n if raw else n + changed_vals)


def _roundtrip_check(w_prev, w_cur, B, cold=False):
    n = w_cur.size
    scache = _exps(w_prev).copy()
    rcache = _exps(w_prev).copy()
    payload, flags, d = oracle.compress_shard(w_cur, B, scache, cold)
    eflags, raw, pbytes, bbytes = _expected_sizes(w_prev, w_cur, B, cold)
    np.testing.assert_array_equal(flags, eflags)
    assert d["mode"] == (oracle.RAW if raw else oracle.COMPRESSED)
    assert d["payload_bytes"] == pbytes and d["body_bytes"] == bbytes
    assert d["n_changed_blocks"] == int(eflags.sum())
    if raw:
        np.testing.assert_array_equal(payload, w_cur.view(np.uint8))
    np.testing.assert_array_equal(scache, _exps(w_cur))
    st, out = oracle.decompress_shard(payload, d, n, B, rcache)
    assert st == 0
    np.testing.assert_array_equal(out, w_cur)
    np.testing.assert_array_equal(rcache, _exps(w_cur))
    return d


def _rand_bf16(rng, n, sigma=0.02):
    x = rng.normal(0, sigma, n).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any bf16 will do


def test_zero_change_is_half_plus_flags():
    rng = np.random.default_rng(1)
    for n, B in [(4096, 256), (5000, 64), (1, 1), (33, 4)]:
        w = _rand_bf16(rng, n)
        # mantissa/sign-only edits keep every exponent
        w2 = w ^ rng.integers(0, 2, n, dtype=np.uint16) * np.uint16(0x8001)
        d = _roundtrip_check(w, w2, B)
        nb = (n + B - 1) // B
        if n + (nb + 7) // 8 < 2 * n:
            assert d["mode"] == oracle.COMPRESSED
            assert d["payload_bytes"] == n + (nb + 7) // 8
            assert d["n_changed_blocks"] == 0


def test_all_changed_falls_back_to_raw():
    rng = np.random.default_rng(2)
    for n, B in [(4096, 256), (777, 5), (8, 8)]:
        w = _rand_bf16(rng, n)
        w2 = w ^ np.uint16(0x0080)          # flips every exponent
        d = _roundtrip_check(w, w2, B)
        assert d["mode"] == oracle.RAW and d["payload_bytes"] == 2 * n
        assert d["n_changed_blocks"] == (n + B - 1) // B


def test_cold_start_is_raw_and_seeds_caches():
    rng = np.random.default_rng(3)
    w = _rand_bf16(rng, 1000)
    d = _roundtrip_check(np.zeros(1000, np.uint16), w, 64, cold=True)
    assert d["mode"] == oracle.RAW and d["n_changed_blocks"] == (1000 + 63) // 64


@pytest.mark.parametrize("cfg", [1])
def test_workload_sequence_roundtrip_and_flag_truth(cfg):
    wl = workloads.workload(cfg)
    seq = [w.numpy().copy() for w in workloads.sequence(wl, wl.iterations)]
    n, R, B = seq[0].size, wl.ranks, wl.block
    scache = np.zeros(n, np.uint8)
    rcache = np.zeros(n, np.uint8)
    prev = None
    for t, w in enumerate(seq):
        payloads, descs, flags = oracle.compress_plan(w, R, B, scache, cold=(t == 0))
        st, out = oracle.decompress_plan(payloads, descs, n, R, B, rcache)
        assert st == 0
        np.testing.assert_array_equal(out, w)
        np.testing.assert_array_equal(scache, _exps(w))
        np.testing.assert_array_equal(rcache, _exps(w))
        for r in range(R):
            b, ln = oracle.shard_begin(n, R, r), oracle.shard_len(n, R, r)
            if prev is None:
                assert flags[r].all()
                continue
            ef, raw, pb, bb = _expected_sizes(prev[b:b + ln], w[b:b + ln], B, False)
            np.testing.assert_array_equal(flags[r, :len(ef)], ef)
            assert descs[r]["payload_bytes"] == pb
        prev = w


def test_exponent_change_statistics_of_workload_1():
    # step 1e-4 on N(0, 0.02): a few percent of exponents change per step
    wl = workloads.workload(1)
    w0, w1 = [w.numpy() for w in workloads.sequence(wl, 2)]
    rate = np.mean(_exps(w0) != _exps(w1))
    assert 0.005 < rate < 0.08


# every subset of changed positions on tiny shards
@pytest.mark.parametrize("B", [1, 2, 3, 4, 16])
@pytest.mark.parametrize("R", [1, 2, 3, 5])
def test_exhaustive_tiny(B, R):
    rng = np.random.default_rng(100 * B + R)
    for n in (0, 1, 2, 3, 5, 8):
        base = _rand_bf16(rng, n) if n else np.zeros(0, np.uint16)
        for mask in range(1 << n):
            cur = base.copy()
            pos = [j for j in range(n) if mask >> j & 1]
            cur[pos] ^= np.uint16(0x0080)                   # exponent changes here
            cur ^= rng.integers(0, 2, n, dtype=np.uint16) * np.uint16(0x8041)  # sign/mantissa noise
            _check_plan(base, cur, R, B, set(pos))
    # n = 12: a sample of subsets
    base = _rand_bf16(rng, 12)
    for mask in rng.integers(0, 1 << 12, 64):
        cur = base.copy()
        pos = [j for j in range(12) if int(mask) >> j & 1]
        cur[pos] ^= np.uint16(0x0080)
        _check_plan(base, cur, R, B, set(pos))


def _check_plan(prev, cur, R, B, changed_positions):
    n = cur.size
    scache = _exps(prev).copy()
    rcache = _exps(prev).copy()
    payloads, descs, flags = oracle.compress_plan(cur, R, B, scache, cold=False)
    st, out = oracle.decompress_plan(payloads, descs, n, R, B, rcache)
    assert st == 0
    np.testing.assert_array_equal(out, cur)
    np.testing.assert_array_equal(scache, _exps(cur))
    np.testing.assert_array_equal(rcache, _exps(cur))
    S = (n + R - 1) // R if n else 0
    for r in range(R):
        b = min(r * S, n)
        ln = max(0, min(b + S, n) - b)
        nb = (ln + B - 1) // B
        truth = [int(any(b + k * B <= j < b + min(ln, (k + 1) * B) for j in changed_positions))
                 for k in range(nb)]
        assert list(flags[r, :nb]) == truth
        ch_vals = sum(min(ln, (k + 1) * B) - k * B for k in range(nb) if truth[k])
        comp = ln + ch_vals + (nb + 7) // 8
        d = descs[r]
        if ln == 0 or comp >= 2 * ln:
            assert d["mode"] == oracle.RAW and d["payload_bytes"] == 2 * ln
            np.testing.assert_array_equal(payloads[r, :2 * ln], cur[b:b + ln].view(np.uint8))
        else:
            assert d["mode"] == oracle.COMPRESSED and d["payload_bytes"] == comp
            assert d["body_bytes"] == ln + ch_vals


def test_corrupt_descriptor_is_rejected():
    rng = np.random.default_rng(5)
    w = _rand_bf16(rng, 64)
    w2 = w ^ np.uint16(0x0001)
    sc = _exps(w).copy()
    payload, flags, d = oracle.compress_shard(w2, 16, sc, False)
    assert d["mode"] == oracle.COMPRESSED
    for bad in (dict(d, n_changed_blocks=1), dict(d, body_bytes=d["body_bytes"] - 1),
                dict(d, mode=7), dict(d, mode=oracle.RAW)):
        st, _ = oracle.decompress_shard(payload, bad, 64, 16, _exps(w).copy())
        assert st == -1
