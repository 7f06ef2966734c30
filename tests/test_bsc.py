"""Benefit-driven shard selection (CIERA Section 3.2): pins of the oracle and
parity of libciera's ciera_bsc_select with it (host only)."""
import numpy as np
import pytest

import oracle
from lossless_exponent_reuse_gb300 import ciera

# A cost model under which the gain is plain byte counting:
# g_i = N_i (1 - q_i) - ceil(ceil(N_i/4096)/8) seconds (link 1 B/s, free kernels)
BYTES = dict(link_Bps=1.0, t_fixed_s=0.0, hbm_Bps=1e300, block=4096)

#          N       q     gain (hand)            M = N (W = 2)  ratio
# A      1000    0.5     500 - 1 = 499          1000           0.499
# B     32768    0.9     3276.8 - 1 = 3275.8    32768          0.09997
# C       100    0.0     100 - 1 = 99           100            0.99
# D       500    1.0     0 - 1 = -1             never
# E       900    0.5     450 - 1 = 449          900            0.4989
N = [1000, 32768, 100, 500, 900]
Q = [0.5, 0.9, 0.0, 1.0, 0.5]


@pytest.mark.parametrize("budget,expect", [
    (50, ""),          # nothing fits, not even C
    (100, "C"),
    (1050, "CE"),      # C; A (1100) does not fit, is skipped; E still fits
    (1100, "AC"),      # C then A by ratio; E no longer fits
    (33000, "ACE"),    # order C, A, E, B: E (total 2000) fits, B (34768) does not
    (34767, "ACE"),
    (34768, "ABCE"),   # everything with a positive gain
    (10**12, "ABCE"),
])
def test_hand_example(budget, expect):
    sel, gain, cnt = oracle.bsc_select(N, Q, 2, budget, **BYTES)
    got = "".join(c for c, s in zip("ABCDE", sel) if s)
    assert got == expect and cnt == len(expect)
    np.testing.assert_allclose(gain, [499.0, 3275.8, 99.0, -1.0, 449.0], rtol=1e-12)


def test_unlimited_budget_selects_exactly_the_profitable_shards():
    # the gain's sign is the per-tensor predicate with q_hat = q_i
    rng = np.random.default_rng(1)
    n = rng.integers(1, 10**8, 200)
    q = rng.random(200)
    sel, gain, _ = oracle.bsc_select(n, q, 16, 10**18)
    for i in range(200):
        assert bool(sel[i]) == (gain[i] > 0)
        assert (gain[i] > 0) == oracle.should_compress(int(n[i]), q_hat=float(q[i]))


def test_single_rank_caches_nothing_and_selects_nothing():
    sel, gain, cnt = oracle.bsc_select([10**7, 10**8], [0.0, 0.1], 1, 10**12)
    assert cnt == 0 and not sel.any()


def test_budget_is_respected_and_selection_grows_with_it():
    rng = np.random.default_rng(2)
    n = rng.integers(10**5, 10**7, 64)
    q = rng.random(64) * 0.5
    prev = -1
    for budget in [0, 10**6, 10**7, 10**8, 10**9, 10**10]:
        sel, _, cnt = oracle.bsc_select(n, q, 8, budget)
        assert int((7 * n * sel).sum()) <= budget
        assert cnt >= prev
        prev = cnt


def test_library_matches_oracle():
    rng = np.random.default_rng(3)
    saved = ciera.get_cost_model()
    try:
        for model in [dict(link_Bps=8e9, q_hat=0.22, t_fixed_s=20e-6, hbm_Bps=8e12, block=4096),
                      dict(link_Bps=1.0, q_hat=0.0, t_fixed_s=0.0, hbm_Bps=1e300, block=4096),
                      dict(link_Bps=50e9, q_hat=0.5, t_fixed_s=5e-6, hbm_Bps=6.8e12, block=512)]:
            ciera.set_cost_model(**model)
            kw = {k: model[k] for k in ("link_Bps", "t_fixed_s", "hbm_Bps", "block")}
            for trial in range(20):
                m = int(rng.integers(0, 40))
                n = rng.integers(1, 10**8, m)
                q = rng.random(m)
                world = int(rng.integers(1, 33))
                budget = int(rng.integers(0, 10**10))
                sel_o, gain_o, _ = oracle.bsc_select(n, q, world, budget, **kw)
                sel_l, gain_l = ciera.bsc_select(n, q, world, budget)
                assert [bool(x) for x in sel_o] == sel_l
                np.testing.assert_allclose(gain_l, gain_o, rtol=1e-12, atol=0)
        # the hand example through the library
        ciera.set_cost_model(link_Bps=1.0, q_hat=0.0, t_fixed_s=0.0, hbm_Bps=1e300, block=4096)
        sel, gain = ciera.bsc_select(N, Q, 2, 1050)
        assert sel == [False, False, True, False, True]
    finally:
        ciera.set_cost_model(**saved)


def test_library_rejects_bad_input():
    with pytest.raises(ciera.CieraError):
        ciera.bsc_select([10], [1.5], 2, 100)
    with pytest.raises(ciera.CieraError):
        ciera.bsc_select([10], [0.5], 0, 100)
    with pytest.raises(ciera.CieraError):
        ciera.bsc_select([-1], [0.5], 2, 100)
    assert ciera.bsc_select([], [], 4, 100) == ([], [])
