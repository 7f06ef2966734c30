"""Pins of the oracle's rANS coding of changed exponents (CIERA Section 3.1:
changed exponents entropy-coded with ANS; our own rANS from Duda's published
method, reading R15 of the design notes).

* a one-symbol block coded by hand (uniform table);
* table normalisation by hand;
* round trips over many distributions and lengths, and rejection of
  damaged records;
* coded size against the information content of the block under the table
  (sum of log2(4096 / f) bits plus the lanes' final states);
* RANS payloads rebuild the weights exactly and carry the sign+mantissa
  bytes of every value at fixed positions.
"""
import math

import numpy as np
import pytest

import oracle
from lossless_exponent_reuse_gb300 import workloads


def test_one_symbol_block_by_hand():
    # uniform table: f = 16, cum[s] = 16 s.  Lane 0 codes symbol 127 from the
    # initial state 2^16: x = ((2^16 // 16) << 12) + 2^16 % 16 + 16 * 127
    #   = 2^24 + 2032 = 0x010007F0 -> stream words 0x0100, 0x07F0.
    # Lanes 1..31 code nothing: their stream is the initial state 0x0001, 0x0000.
    f = np.full(256, 16, np.uint16)
    rec = oracle.rans_encode_block(np.array([127], np.uint8), f)
    expect = [2, 0] * 32 + [0x00, 0x01, 0xF0, 0x07] + [0x01, 0x00, 0x00, 0x00] * 31
    assert rec.tolist() == expect                      # 64 + 128 = 192 bytes, 16-aligned
    st, out = oracle.rans_decode_block(rec, 1, f)
    assert st == 0 and out.tolist() == [127]


def test_renormalising_block_by_hand():
    """A 65-exponent block whose lane 0 renormalises twice, derived by hand
    from the coding step x' = ((x // f) << 12) + x % f + cum[s], preceded by
    emitting the low 16 bits of x (x >>= 16) whenever x >= f << 20.

    Table: h[127] = 15, h[130] = 1 -> f[127] = 1 + 15*3840/16 = 3601,
    f[130] = 1 + 3840/16 = 241, the other 254 symbols 1; the sum is 4096, so
    nothing is added.  cum[127] = 127 (127 symbols of frequency 1 below it);
    cum[200] = 198 + 3601 + 241 = 4040, cum[201] = 4041, cum[202] = 4042.

    Lane 0 codes positions 0, 32, 64 = symbols 200, 201, 202, backwards:
      x = 0x10000 (the initial state)
      s=202: x < 1 << 20;  x = (0x10000 << 12) + 4042        = 0x10000FCA
      s=201: x >= 1 << 20: emit 0x0FCA, x = 0x1000;
             x = (0x1000 << 12) + 4041                      = 0x01000FC9
      s=200: x >= 1 << 20: emit 0x0FC9, x = 0x0100;
             x = (0x0100 << 12) + 4040                      = 0x00100FC8
      final state: low 0x0FC8, high 0x0010.
    Emitted 0x0FCA, 0x0FC9, 0x0FC8, 0x0010; the decoder reads them last
    first: 0x0010, 0x0FC8, 0x0FC9, 0x0FCA (4 words).
    Lanes 1..31 code symbol 127 at positions l and l + 32 (f = 3601, bound
    3601 << 20, never reached):
      x = 0x10000: 65536 = 18*3601 + 718 -> x = 18*4096 + 718 + 127 = 74573
      x = 74573 = 20*3601 + 2553 -> x = 20*4096 + 2553 + 127 = 84600 = 0x14A78
    so each reads 0x0001, 0x4A78 (2 words).
    Record: 32 uint16 counts (4, then 2 x 31), lane 0's 4 words, 31 x 2
    words: 64 + 8 + 124 = 196 bytes, zero-padded to 208.
    """
    h = np.zeros(256, np.uint32)
    h[127], h[130] = 15, 1
    f = oracle.rans_table(h)
    assert (int(f[127]), int(f[130]), int(f.sum())) == (3601, 241, 4096)
    e = np.full(65, 127, np.uint8)
    e[[0, 32, 64]] = [200, 201, 202]
    words = [4] + [2] * 31 + [0x0010, 0x0FC8, 0x0FC9, 0x0FCA] + [0x0001, 0x4A78] * 31
    expect = np.array(words, np.uint16).view(np.uint8).tolist() + [0] * 12
    rec = oracle.rans_encode_block(e, f)
    assert len(rec) == 208
    assert rec.tolist() == expect
    st, out = oracle.rans_decode_block(rec, 65, f)
    assert st == 0 and out.tolist() == e.tolist()


def test_table_normalisation_by_hand():
    h = np.zeros(256, np.uint32)
    h[5], h[9] = 3, 1                 # 1 + 3*3840/4 = 2881, 1 + 3840/4 = 961, 254 x 1
    f = oracle.rans_table(h)
    assert (f[5], f[9]) == (2881, 961) and int(f.sum()) == 4096 and f.min() == 1
    h = np.zeros(256, np.uint32)
    h[:4] = [1, 1, 1, 4]              # 1 + 548 (x3), 1 + 2194, 252 x 1 -> 4094: +2 to s=3
    assert oracle.rans_table(h)[:5].tolist() == [549, 549, 549, 2197, 1]
    assert oracle.rans_table(np.zeros(256, np.uint32)).tolist() == [16] * 256


@pytest.mark.parametrize("L", [1, 31, 32, 33, 100, 4096, 5000])
@pytest.mark.parametrize("dist", ["gauss", "uniform", "single", "two"])
def test_round_trip_and_size_bound(L, dist):
    rng = np.random.default_rng(L * 7 + len(dist))
    if dist == "gauss":
        e = np.clip(np.round(rng.normal(118, 2.0, L)), 0, 255).astype(np.uint8)
    elif dist == "uniform":
        e = rng.integers(0, 256, L).astype(np.uint8)
    elif dist == "single":
        e = np.full(L, 121, np.uint8)
    else:
        e = rng.choice([0, 255], L).astype(np.uint8)
    f = oracle.rans_table(np.bincount(e, minlength=256).astype(np.uint32))
    rec = oracle.rans_encode_block(e, f)
    st, out = oracle.rans_decode_block(rec, L, f)
    assert st == 0
    np.testing.assert_array_equal(out, e)
    info_bits = sum(math.log2(4096 / int(f[s])) for s in e)
    # each lane: its final state (32 bits) and less than 16 bits of slack;
    # 64-byte header; up to 15 bytes of padding
    assert rec.size * 8 <= info_bits + 32 * 48 + 64 * 8 + 15 * 8, (rec.size, info_bits)
    assert rec.size % 16 == 0


def test_damaged_records_are_rejected():
    rng = np.random.default_rng(9)
    e = np.clip(np.round(rng.normal(118, 2.0, 4096)), 0, 255).astype(np.uint8)
    f = oracle.rans_table(np.bincount(e, minlength=256).astype(np.uint32))
    rec = oracle.rans_encode_block(e, f)
    bad = rec.copy()
    bad[0] += 1                                   # lane 0 claims one more word
    assert oracle.rans_decode_block(bad, 4096, f)[0] == -1
    assert oracle.rans_decode_block(rec[:100], 4096, f)[0] == -1
    bad = rec.copy()
    bad[64 + 3] ^= 0x40                           # lane 0's state
    assert oracle.rans_decode_block(bad, 4096, f)[0] == -1


def _exps(w):
    return ((w >> 7) & 0xFF).astype(np.uint8)


@pytest.mark.parametrize("block,p_block", [(4096, None), (4096, 0.2), (256, 0.3), (300, None)])
def test_rans_shard_round_trip(block, p_block):
    wl = workloads.small("r", [(64, 4096)], ranks=1, block=block, iterations=4, step=1e-4,
                         p_block=p_block)
    seq = [w.numpy().copy() for w in workloads.sequence(wl, 4)]
    n = seq[0].size
    sc = np.zeros(n, np.uint8)
    rc = np.zeros(n, np.uint8)
    hist = np.zeros(256, np.uint32)
    sc_exact = np.zeros(n, np.uint8)
    for t, w in enumerate(seq):
        payload, flags, d, hist_next = oracle.compress_shard_rans(w, block, sc, t == 0, hist)
        _, flags_exact, d_exact = oracle.compress_shard(w, block, sc_exact, t == 0)
        np.testing.assert_array_equal(flags, flags_exact)
        # the table's source: every 16th exponent of the shard
        np.testing.assert_array_equal(hist_next, np.bincount(_exps(w)[::16], minlength=256))
        np.testing.assert_array_equal(sc, _exps(w))
        st, out = oracle.decompress_shard_any(payload, d, n, block, rc)
        assert st == 0
        np.testing.assert_array_equal(out, w)
        np.testing.assert_array_equal(rc, _exps(w))
        if t == 0:
            assert d["mode"] == oracle.RAW
        else:
            assert d["mode"] == oracle.RANS
            # every value's sign+mantissa byte at its own position
            sm = (((w >> 8) & 0x80) | (w & 0x7F)).astype(np.uint8)
            np.testing.assert_array_equal(payload[:n], sm)
            assert d["payload_bytes"] < 2 * n
            if d_exact["mode"] == oracle.RAW:
                assert d["payload_bytes"] < d_exact["payload_bytes"]
            # the offset table: prefixes of the record sizes, empty for kept
            # blocks, 16-byte steps, the last entry the records' total
            nb = flags.size
            A = (n + 15) // 16 * 16
            C = (A + (nb + 7) // 8 + 15) // 16 * 16
            O = C + 512
            D = (O + 4 * (nb + 1) + 15) // 16 * 16
            assert d["body_bytes"] == D
            offs = payload[O:O + 4 * (nb + 1)].view(np.uint32).astype(np.int64)
            sizes = np.diff(offs)
            assert offs[0] == 0 and np.all(sizes % 16 == 0)
            np.testing.assert_array_equal(sizes > 0, flags.astype(bool))
            assert offs[nb] == d["payload_bytes"] - D
            # the bitmap and the frequency table
            bits = np.unpackbits(payload[A:A + (nb + 7) // 8], bitorder="little")[:nb]
            np.testing.assert_array_equal(bits, flags)
            np.testing.assert_array_equal(payload[C:C + 512].view(np.uint16),
                                          oracle.rans_table(hist))
        hist = hist_next
