"""Pins of the oracle's hashed change test (CIERA Section 3.1 and Appendix A,
Algorithm 1: Hash128 from two 64-bit SplitMix64-based hashes, HashCache).

* SplitMix64 against its published outputs from seed 0 (the reference
  implementation's test vector);
* the hash of a 9-exponent block computed from the definition in Python
  integers (word packing, key index, length term), with the output function
  pinned by the same published outputs;
* the empty block hashes to 0 (fin(0) = 0, a closed form);
* a change of any single exponent always changes both hashes (each word term
  is a bijection of the word, so the sum moves by a nonzero amount, and the
  final mix is a bijection);
* the hashed sender emits the exact sender's flags, payloads and descriptors
  on real weight sequences (no collisions), and its cache holds the current
  blocks' hashes.
"""
import numpy as np
import pytest

import oracle
from lossless_exponent_reuse_gb300 import workloads

SEED1, SEED2 = 0x6A09E667F3BCC908, 0xBB67AE8584CAA73B


def test_splitmix64_published_outputs_from_seed_zero():
    assert oracle.splitmix64(0, 1) == 0xE220A8397B1DCDAF
    assert oracle.splitmix64(0, 2) == 0x6E789E6AA1B965F4
    assert oracle.splitmix64(0, 3) == 0x06C45D188009454F


M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def _fin(z):
    """SplitMix64's output function (Steele, Lea and Flood, 2014), in Python
    integers; pinned below by the generator's published seed-0 outputs."""
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_nine_exponent_block_hash_from_the_definition():
    """h_s of a 9-exponent block written out from the definition of the
    block hash: two little-endian exponent words (the second holds one
    exponent and seven zero bytes), keys = SplitMix64 outputs 1 and 2 from
    the seed (state s + i * golden, i = 1, 2), and the length 9 added before
    the final mix."""
    # the output function, through the published outputs 1..3 from seed 0
    assert [_fin(i * GOLDEN & M64) for i in (1, 2, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    e = np.array([0x7A, 0x7B, 0x7C, 0x79, 0x80, 0x00, 0xFF, 0x7D, 0x81], np.uint8)
    word0 = 0x7D_FF_00_80_79_7C_7B_7A      # e0 in the lowest byte
    word1 = 0x81
    for seed in (SEED1, SEED2):
        k1 = _fin((seed + 1 * GOLDEN) & M64)
        k2 = _fin((seed + 2 * GOLDEN) & M64)
        h = _fin((9 + _fin(word0 ^ k1) + _fin(word1 ^ k2)) & M64)
        assert oracle.exp_hash64(e, seed) == h, hex(seed)
    # and for a block given as bf16 values (exponent = bits 14..7)
    vals = (e.astype(np.uint16) << 7) | np.uint16(0x8000) | np.uint16(0x0055)
    assert oracle.block_hash128(vals) == (oracle.exp_hash64(e, SEED1),
                                          oracle.exp_hash64(e, SEED2))


def test_empty_block_hashes_to_zero():
    assert oracle.exp_hash64(np.zeros(0, np.uint8), SEED1) == 0
    assert oracle.block_hash128(np.zeros(0, np.uint16)) == (0, 0)


@pytest.mark.parametrize("L", [1, 7, 8, 9, 64, 100])
def test_every_single_exponent_change_changes_both_hashes(L):
    rng = np.random.default_rng(L)
    e = rng.integers(0, 256, L).astype(np.uint8)
    base = (oracle.exp_hash64(e, SEED1), oracle.exp_hash64(e, SEED2))
    for i in range(L):
        for delta in (1, 128, 255):
            f = e.copy()
            f[i] ^= np.uint8(delta)
            h = (oracle.exp_hash64(f, SEED1), oracle.exp_hash64(f, SEED2))
            assert h[0] != base[0] and h[1] != base[1], (i, delta)


def test_position_and_length_matter():
    e = np.arange(16, dtype=np.uint8)
    swapped = e.copy()
    swapped[:8], swapped[8:] = e[8:], e[:8]            # swap the two words
    assert oracle.exp_hash64(e, SEED1) != oracle.exp_hash64(swapped, SEED1)
    assert oracle.exp_hash64(e[:15], SEED1) != oracle.exp_hash64(
        np.concatenate([e[:15], [0]]).astype(np.uint8), SEED1)
    assert oracle.exp_hash64(e, SEED1) != oracle.exp_hash64(e, SEED2)


def test_hash128_uses_the_exponents_only():
    rng = np.random.default_rng(3)
    v = rng.integers(0, 1 << 16, 300).astype(np.uint16)
    w = v ^ (rng.integers(0, 2, 300).astype(np.uint16) * np.uint16(0x807F))  # sign+mantissa only
    assert oracle.block_hash128(v) == oracle.block_hash128(w)
    assert oracle.block_hash128(v) != oracle.block_hash128(v ^ np.uint16(0x0080))


@pytest.mark.parametrize("block,ranks,p_block", [(256, 4, None), (512, 3, 0.3), (300, 2, 0.2)])
def test_hashed_sender_equals_exact_sender(block, ranks, p_block):
    wl = workloads.small("h", [(96, 512)], ranks=ranks, block=block, iterations=4, step=1e-3,
                         p_block=p_block)
    seq = [w.numpy().copy() for w in workloads.sequence(wl, 4)]
    n = seq[0].size
    S = oracle.shard_size(n, ranks)
    nb = oracle.num_blocks(S, block)
    sc = np.zeros(n, np.uint8)
    hc = np.zeros((ranks, nb, 2), np.uint64)
    for t, w in enumerate(seq):
        pe, de, fe = oracle.compress_plan(w, ranks, block, sc, cold=t == 0)
        ph, dh, fh = oracle.compress_plan_hashed(w, ranks, block, hc, cold=t == 0)
        np.testing.assert_array_equal(fe, fh)
        np.testing.assert_array_equal(de, dh)
        for r in range(ranks):
            pb = int(de[r]["payload_bytes"])
            np.testing.assert_array_equal(pe[r, :pb], ph[r, :pb])
        # the cache holds every current block's hash
        for r in range(ranks):
            b, ln = oracle.shard_begin(n, ranks, r), oracle.shard_len(n, ranks, r)
            for k in range(oracle.num_blocks(ln, block)):
                lo, hi = b + k * block, b + min(ln, (k + 1) * block)
                assert tuple(int(x) for x in hc[r, k]) == oracle.block_hash128(w[lo:hi])
