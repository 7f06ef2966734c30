"""Pins the oracle's payload layout to hand-derived worked examples
(tests/golden/*.txt; CIERA Section 3.1, Section 3.2 and Appendix A,
Algorithm 1)."""
import os

import numpy as np
import pytest

import golden_io
import oracle


@pytest.mark.parametrize("path", golden_io.all_fixtures(), ids=os.path.basename)
def test_golden_fixture(path):
    g = golden_io.load(path)
    n, R, B = g["n"], g["ranks"], g["block"]
    w = g["w"]
    scache = g["sender_cache"].copy()
    rcache = g["recv_cache"].copy()
    payloads, descs, flags = oracle.compress_plan(w, R, B, scache, bool(g["cold"]))
    assert len(g["rank_data"]) == R
    for rd in g["rank_data"]:
        r = rd["rank"]
        b, ln = oracle.shard_begin(n, R, r), oracle.shard_len(n, R, r)
        d = descs[r]
        assert (int(d["mode"]), int(d["n_changed_blocks"]), int(d["body_bytes"]),
                int(d["payload_bytes"])) == rd["desc"]
        pb = int(d["payload_bytes"])
        np.testing.assert_array_equal(payloads[r, :pb], rd["payload"])
        np.testing.assert_array_equal(flags[r, :oracle.num_blocks(ln, B)], rd["flags"])
        np.testing.assert_array_equal(scache[b:b + ln], rd["sender_cache_after"])
    st, out = oracle.decompress_plan(payloads, descs, n, R, B, rcache)
    assert st == 0
    np.testing.assert_array_equal(out, w)
    for rd in g["rank_data"]:
        r = rd["rank"]
        b, ln = oracle.shard_begin(n, R, r), oracle.shard_len(n, R, r)
        np.testing.assert_array_equal(rcache[b:b + ln], rd["recv_cache_after"])
