"""Randomised GPU parity: seeded random plans (sizes, ranks, block sizes;
staged and byte-wise paths, ragged tails, empty ranks) and random iteration
sequences (no change, sparse and clustered exponent changes, every exponent
changed, arbitrary bit patterns including inf/NaN/subnormal encodings), with
raw-ahead on or off, through the exact, hashed and RANS senders; every output
byte against the oracle (CIERA Section 3.1, Appendix A Algorithm 1)."""
import numpy as np
import pytest

from harness import run_parity
from test_hashed_gpu import run_hashed_parity
from test_rans_gpu import run_rans_parity
from lossless_exponent_reuse_gb300 import ciera

pytestmark = pytest.mark.gpu

BLOCKS = [1, 3, 16, 100, 256, 272, 512, 1000, 4096, 5000, 8192, 16384, 20000]


def _bf16(rng, n):
    x = rng.normal(0.0, rng.choice([0.002, 0.02, 1.0]), n).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def random_sequence(rng, n, block, iters=5):
    """w_0 random; each next iteration one of: no change, sign/mantissa only,
    sparse exponent flips, some blocks perturbed, every exponent changed,
    arbitrary 16-bit patterns."""
    w = _bf16(rng, n) if rng.random() < 0.8 else rng.integers(0, 1 << 16, n, dtype=np.uint16)
    seq = [w]
    for _ in range(iters - 1):
        w = w.copy()
        kind = rng.integers(0, 6)
        if n == 0 or kind == 0:
            pass
        elif kind == 1:
            w ^= (rng.integers(0, 2, n).astype(np.uint16) * np.uint16(0x8041))
        elif kind == 2:
            idx = rng.integers(0, n, max(1, n // int(rng.choice([50, 2000, 100000]))))
            w[idx] ^= np.uint16(0x0080)
        elif kind == 3:
            nb = (n + block - 1) // block
            for k in rng.choice(nb, size=max(1, nb // int(rng.choice([2, 5, 20]))), replace=False):
                lo, hi = k * block, min(n, (k + 1) * block)
                j = lo + rng.integers(0, hi - lo, max(1, (hi - lo) // 10))
                w[j] ^= np.uint16(0x0100)
        elif kind == 4:
            w ^= np.uint16(0x0080)
        else:
            w = rng.integers(0, 1 << 16, n, dtype=np.uint16)
        seq.append(w)
    return seq


def staged_plan(rng, max_n=300_000):
    """A plan on the staged path: blocks a multiple of 16 in [256, 16384],
    shards of S values and N both multiples of 16, R (S - 1) < N <= R S so
    that ceil(N/R) = S; with more ranks than S/16 the last shards can be
    short or empty."""
    block = int(rng.choice([256, 272, 512, 1024, 4096, 8192, 16384]))
    ranks = int(rng.integers(1, 41))
    S = 16 * int(rng.integers(1, max(2, max_n // 16 // ranks)))
    k_lo = ranks * (S - 1) // 16 + 1          # N > R (S - 1)
    n = 16 * int(rng.integers(k_lo, ranks * S // 16 + 1))
    return n, ranks, block


def random_plan(seed):
    rng = np.random.default_rng(seed)
    if rng.random() < 0.5:
        n, ranks, block = staged_plan(rng)
    else:
        block = int(rng.choice(BLOCKS))
        ranks = int(rng.integers(1, 41))
        n = int(rng.integers(0, 300_000)) if rng.random() < 0.9 else int(rng.integers(0, 64))
    return rng, n, ranks, block


@pytest.mark.parametrize("seed", range(40))
def test_random_exact(seed):
    rng, n, ranks, block = random_plan(seed)
    raw_ahead = bool(rng.integers(0, 2))
    run_parity(random_sequence(rng, n, block), ranks, block, raw_ahead=raw_ahead,
               tag=f"seed={seed} n={n} R={ranks} B={block} raw_ahead={raw_ahead}")


@pytest.mark.parametrize("seed", range(100, 120))
def test_random_hashed(seed):
    rng, n, ranks, block = random_plan(seed)
    if ciera.Plan(n, block, ranks).info.tile_blocks > 32:
        block = 256                     # the hashed sender needs blocks of >= 256 values
    raw_ahead = bool(rng.integers(0, 2))
    run_hashed_parity(random_sequence(rng, n, block), ranks, block, raw_ahead=raw_ahead,
                      tag=f"seed={seed} n={n} R={ranks} B={block} raw_ahead={raw_ahead}")


@pytest.mark.parametrize("seed", range(200, 216))
def test_random_rans(seed):
    # the RANS sender needs the staged plan: shards and N multiples of 16,
    # blocks a multiple of 16 in [256, 16384]
    rng = np.random.default_rng(seed)
    n, ranks, block = staged_plan(rng)
    info = ciera.Plan(n, block, ranks).info
    assert info.fast_path and info.shard_len % 16 == 0 and n % 16 == 0
    run_rans_parity(random_sequence(rng, n, block, iters=6), ranks, block,
                    tag=f"seed={seed} n={n} R={ranks} B={block}")
