"""Pins the oracle's split and merge (CIERA, Section 3.1, SplitExpMant and
Merge) against the numeric meaning of every bf16 bit pattern.

The expected exponent and sign+mantissa byte of each of the 65536 patterns
are recovered from the decoded value (math.frexp on the float), not from bit
masks, so a wrong shift, mask or field order in the oracle fails here.
"""
import math
import struct

import oracle


def _value(p):
    return struct.unpack("<f", struct.pack("<I", p << 16))[0]


def _numeric_fields(p):
    """(sign, biased exponent, 7-bit mantissa) of bf16 pattern p, from its value."""
    x = _value(p)
    sign = 1 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if math.isnan(x):
        return sign, 255, None            # mantissa: any nonzero payload
    if math.isinf(x):
        return sign, 255, 0
    if a == 0.0:
        return sign, 0, 0
    if a < 2.0 ** -126:                   # subnormal: a = m * 2^-133
        m = a / 2.0 ** -133
        assert m == int(m)
        return sign, 0, int(m)
    f, e2 = math.frexp(a)                 # a = f * 2^e2, f in [0.5, 1)
    unbiased = e2 - 1
    frac = a / 2.0 ** unbiased - 1.0      # in [0, 1)
    m = frac * 128.0
    assert m == int(m)
    return sign, unbiased + 127, int(m)


def test_split_matches_numeric_decoding_all_patterns():
    nan_seen = 0
    for p in range(1 << 16):
        sign, e, m = _numeric_fields(p)
        assert oracle.exp_of(p) == e, hex(p)
        sm = oracle.sm_of(p)
        assert sm >> 7 == sign, hex(p)
        if m is None:
            nan_seen += 1
            assert sm & 0x7F != 0, hex(p)
        else:
            assert sm & 0x7F == m, hex(p)
    assert nan_seen == 2 * 127             # 2 signs x 127 nonzero payloads


def test_join_inverts_split_all_patterns():
    for p in range(1 << 16):
        assert oracle.join(oracle.sm_of(p), oracle.exp_of(p)) == p, hex(p)


def test_split_is_a_bijection():
    pairs = {(oracle.exp_of(p), oracle.sm_of(p)) for p in range(1 << 16)}
    assert len(pairs) == 1 << 16


def test_known_values():
    # textbook bf16 encodings
    assert (oracle.exp_of(0x3F80), oracle.sm_of(0x3F80)) == (127, 0x00)   # 1.0
    assert (oracle.exp_of(0xC000), oracle.sm_of(0xC000)) == (128, 0x80)   # -2.0
    assert (oracle.exp_of(0x4049), oracle.sm_of(0x4049)) == (128, 0x49)   # 3.140625
    assert _value(0x4049) == 3.140625
