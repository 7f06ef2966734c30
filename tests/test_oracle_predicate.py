"""Pins the oracle's per-tensor predicate (CIERA Section 3.2, gain g_i).

Hand derivation with the defaults (link 8e9 B/s, q = 0.22, t_fixed = 20 us,
hbm 8e12 B/s, B = 4096):
  saved = (2N - N - 0.22N - ceil(ceil(N/4096)/8)) / 8e9
        ~ N * (0.78 / 8e9 - 1 / (32768 * 8e9))  = N * 9.74962e-11
  cost  = 20e-6 + 4.22 N / 8e12                  = 20e-6 + N * 5.275e-13
  saved > cost  <=>  N > 20e-6 / 9.69687e-11 ~ 206,252
so the decision flips near N = 206,250; with link 16e9 the saving halves and
the flip moves to 20e-6 / (4.875e-11 - 1.9e-15 - 5.275e-13) ~ 414,760.
"""
import oracle


def _flip(lo, hi, **kw):
    """Smallest N in [lo, hi] that compresses (the decision is monotone there)."""
    assert not oracle.should_compress(lo, **kw) and oracle.should_compress(hi, **kw)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if oracle.should_compress(mid, **kw):
            hi = mid
        else:
            lo = mid
    return hi


def test_default_threshold_near_206k():
    n_min = _flip(1000, 10_000_000)
    assert 206_150 <= n_min <= 206_350, n_min


def test_threshold_moves_with_link_bandwidth():
    n_min = _flip(1000, 100_000_000, link_Bps=16e9)
    assert 414_300 <= n_min <= 415_200, n_min


def test_olmoe_tensors_classify():
    # two norms [2048] and the router 64x2048 are declined; attention 2048^2
    # and expert matrices 2048x1024 are compressed
    assert not oracle.should_compress(2048)
    assert not oracle.should_compress(64 * 2048)
    assert oracle.should_compress(2048 * 2048)
    assert oracle.should_compress(2048 * 1024)
    # the whole accepted bucket of one layer
    assert oracle.should_compress(4 * 2048 * 2048 + 64 * 3 * 2048 * 1024)


def test_every_block_changing_never_pays():
    # q = 1: the expected payload is 2N + bitmap, so nothing is saved
    for n in (1, 4096, 10**6, 10**9):
        assert not oracle.should_compress(n, q_hat=1.0)


def test_free_kernels_reduce_to_byte_count():
    # t_fixed = 0 and an unbounded memory rate: compress iff the payload is
    # smaller, i.e. (1 - q) N > ceil(ceil(N/B)/8)
    kw = dict(t_fixed_s=0.0, hbm_Bps=1e300)
    assert not oracle.should_compress(1, q_hat=0.0, block=1, **kw)   # 1 > 1 fails
    assert oracle.should_compress(2, q_hat=0.0, block=1, **kw)       # 2 > 1
    assert not oracle.should_compress(10, q_hat=0.9, block=8, **kw)  # 1 > 1 fails
    assert oracle.should_compress(20, q_hat=0.9, block=8, **kw)      # 2 > 1
    assert not oracle.should_compress(0, q_hat=0.0, block=1, **kw)   # nothing to send
