"""CPU oracle for cross-iteration exponent reuse (CIERA) on bf16 weights.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The library never imports
this package, and this package never imports the library.

The arithmetic lives in ``ciera_oracle.c`` (plain C, one element at a time);
this module compiles it with gcc into ``oracle/_build/`` and exposes numpy
wrappers.  Source for every step: "CIERA: Cross-Iteration Exponent Reuse for
Lossless Allgather in Sharded MoE Training", Section 3.1 (Exponent Reuse),
Section 3.2 (Benefit-driven Selective Compression) and Appendix A
(Algorithm 1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ciera_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libciera_oracle.so")

COMPRESSED = 0
RAW = 1

# Descriptor record: mode u32, n_changed_blocks u32, body_bytes u64,
# payload_bytes u64 (24 bytes, little-endian, no padding).
DESC_DTYPE = np.dtype([("mode", "<u4"), ("n_changed_blocks", "<u4"),
                       ("body_bytes", "<u8"), ("payload_bytes", "<u8")])


class _Desc(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_uint32), ("n_changed_blocks", ctypes.c_uint32),
                ("body_bytes", ctypes.c_uint64), ("payload_bytes", ctypes.c_uint64)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared object with gcc; returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if force or not fresh:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c99", "-Wall", "-Wextra", "-shared",
                        "-fPIC", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64, u32, vp = ctypes.c_int64, ctypes.c_uint, ctypes.c_void_p
            L.oracle_exp.argtypes = [u32]
            L.oracle_exp.restype = u32
            L.oracle_sm.argtypes = [u32]
            L.oracle_sm.restype = u32
            L.oracle_join.argtypes = [u32, u32]
            L.oracle_join.restype = u32
            for name in ("oracle_shard_size", "oracle_num_blocks", "oracle_bitmap_bytes"):
                getattr(L, name).argtypes = [i64, i64]
                getattr(L, name).restype = i64
            for name in ("oracle_shard_begin", "oracle_shard_len"):
                getattr(L, name).argtypes = [i64, i64, i64]
                getattr(L, name).restype = i64
            L.oracle_compress_shard.argtypes = [vp, i64, i64, vp, ctypes.c_int, vp, vp,
                                                ctypes.POINTER(_Desc)]
            L.oracle_compress_shard.restype = ctypes.c_int
            L.oracle_decompress_shard.argtypes = [vp, ctypes.POINTER(_Desc), i64, i64, vp, vp]
            L.oracle_decompress_shard.restype = ctypes.c_int
            L.oracle_compress_plan.argtypes = [vp, i64, i64, i64, vp, ctypes.c_int, vp, i64,
                                               vp, vp]
            L.oracle_compress_plan.restype = ctypes.c_int
            L.oracle_decompress_plan.argtypes = [vp, i64, vp, i64, i64, i64, vp, vp]
            L.oracle_decompress_plan.restype = ctypes.c_int
            L.oracle_should_compress.argtypes = [i64, ctypes.c_double, ctypes.c_double,
                                                 ctypes.c_double, ctypes.c_double, i64]
            L.oracle_should_compress.restype = ctypes.c_int
            L.oracle_bsc_select.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, i64,
                                            ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                            i64, vp, vp]
            L.oracle_bsc_select.restype = ctypes.c_int
            u64 = ctypes.c_uint64
            L.oracle_splitmix64.argtypes = [u64, u64]
            L.oracle_splitmix64.restype = u64
            L.oracle_exp_hash64.argtypes = [vp, i64, u64]
            L.oracle_exp_hash64.restype = u64
            L.oracle_block_hash128.argtypes = [vp, i64, vp]
            L.oracle_block_hash128.restype = None
            L.oracle_compress_shard_hashed.argtypes = [vp, i64, i64, vp, ctypes.c_int, vp, vp,
                                                       ctypes.POINTER(_Desc)]
            L.oracle_compress_shard_hashed.restype = ctypes.c_int
            L.oracle_compress_plan_hashed.argtypes = [vp, i64, i64, i64, vp, ctypes.c_int, vp,
                                                      i64, vp, vp]
            L.oracle_compress_plan_hashed.restype = ctypes.c_int
            L.oracle_rans_table.argtypes = [vp, vp]
            L.oracle_rans_table.restype = None
            L.oracle_rans_encode_block.argtypes = [vp, i64, vp, vp]
            L.oracle_rans_encode_block.restype = i64
            L.oracle_rans_decode_block.argtypes = [vp, i64, i64, vp, vp]
            L.oracle_rans_decode_block.restype = ctypes.c_int
            L.oracle_compress_shard_rans.argtypes = [vp, i64, i64, vp, ctypes.c_int, vp, vp, vp,
                                                     vp, ctypes.POINTER(_Desc)]
            L.oracle_compress_shard_rans.restype = ctypes.c_int
            L.oracle_decompress_shard_rans.argtypes = [vp, ctypes.POINTER(_Desc), i64, i64, vp,
                                                       vp]
            L.oracle_decompress_shard_rans.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---- element-level ---------------------------------------------------------

def exp_of(w: int) -> int:
    return int(lib().oracle_exp(int(w)))


def sm_of(w: int) -> int:
    return int(lib().oracle_sm(int(w)))


def join(sm: int, e: int) -> int:
    return int(lib().oracle_join(int(sm), int(e)))


# ---- sharding --------------------------------------------------------------

def shard_size(n: int, ranks: int) -> int:
    return int(lib().oracle_shard_size(n, ranks))


def shard_begin(n: int, ranks: int, r: int) -> int:
    return int(lib().oracle_shard_begin(n, ranks, r))


def shard_len(n: int, ranks: int, r: int) -> int:
    return int(lib().oracle_shard_len(n, ranks, r))


def num_blocks(length: int, block: int) -> int:
    return int(lib().oracle_num_blocks(length, block))


def bitmap_bytes(length: int, block: int) -> int:
    return int(lib().oracle_bitmap_bytes(length, block))


# ---- one shard -------------------------------------------------------------

def compress_shard(shard: np.ndarray, block: int, sender_cache: np.ndarray, cold: bool):
    """Sender side for one shard.  Updates ``sender_cache`` in place.

    Returns (payload bytes [payload_bytes], flags u8[n_blocks], desc dict).
    """
    shard = np.ascontiguousarray(shard, dtype=np.uint16)
    assert sender_cache.dtype == np.uint8 and sender_cache.size == shard.size
    n = shard.size
    payload = np.zeros(max(2 * n, 1), dtype=np.uint8)
    flags = np.zeros(max(num_blocks(n, block), 1), dtype=np.uint8)
    d = _Desc()
    lib().oracle_compress_shard(_ptr(shard), n, block, _ptr(sender_cache), int(bool(cold)),
                                _ptr(payload), _ptr(flags), ctypes.byref(d))
    desc = dict(mode=d.mode, n_changed_blocks=d.n_changed_blocks,
                body_bytes=d.body_bytes, payload_bytes=d.payload_bytes)
    return payload[: d.payload_bytes].copy(), flags[: num_blocks(n, block)].copy(), desc


def decompress_shard(payload: np.ndarray, desc: dict, length: int, block: int,
                     recv_cache: np.ndarray):
    """Receiver side for one shard.  Updates ``recv_cache`` in place.

    Returns (status, out u16[length]); status is 0, or -1 for a descriptor
    that does not match the payload.
    """
    buf = np.zeros(max(2 * length, 1), dtype=np.uint8)
    src = np.ascontiguousarray(payload, dtype=np.uint8)
    buf[: min(src.size, buf.size)] = src[: buf.size]
    out = np.zeros(max(length, 1), dtype=np.uint16)
    d = _Desc(desc["mode"], desc["n_changed_blocks"], desc["body_bytes"], desc["payload_bytes"])
    st = lib().oracle_decompress_shard(_ptr(buf), ctypes.byref(d), length, block,
                                       _ptr(recv_cache), _ptr(out))
    return int(st), out[:length].copy()


# ---- whole plan (all ranks) --------------------------------------------------

def compress_plan(w: np.ndarray, ranks: int, block: int, sender_cache: np.ndarray,
                  cold: bool, stride: int | None = None):
    """Sender side for every rank.  Updates ``sender_cache`` (u8[N]) in place.

    Returns (payloads u8[ranks, stride], descs DESC_DTYPE[ranks],
    flags u8[ranks, blocks_per_full_shard]).
    """
    w = np.ascontiguousarray(w, dtype=np.uint16)
    n = w.size
    s = shard_size(n, ranks) if n else 0
    if stride is None:
        stride = max(2 * s, 1)
    payloads = np.zeros((ranks, stride), dtype=np.uint8)
    descs = np.zeros(ranks, dtype=DESC_DTYPE)
    fstride = num_blocks(s, block) if n else 0
    flags = np.zeros((ranks, max(fstride, 1)), dtype=np.uint8)
    lib().oracle_compress_plan(_ptr(w), n, ranks, block, _ptr(sender_cache), int(bool(cold)),
                               _ptr(payloads), stride, _ptr(descs), _ptr(flags))
    return payloads, descs, flags[:, :fstride]


def decompress_plan(payloads: np.ndarray, descs: np.ndarray, n: int, ranks: int, block: int,
                    recv_cache: np.ndarray):
    """Receiver side for every rank.  Updates ``recv_cache`` in place.

    Returns (status, out u16[N]).
    """
    payloads = np.ascontiguousarray(payloads, dtype=np.uint8)
    descs = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
    out = np.zeros(max(n, 1), dtype=np.uint16)
    st = lib().oracle_decompress_plan(_ptr(payloads), payloads.shape[1], _ptr(descs), n, ranks,
                                      block, _ptr(recv_cache), _ptr(out))
    return int(st), out[:n]


# ---- predicate ---------------------------------------------------------------

DEFAULT_COST_MODEL = dict(link_Bps=8e9, q_hat=0.22, t_fixed_s=20e-6, hbm_Bps=8e12, block=4096)


def should_compress(numel: int, link_Bps=8e9, q_hat=0.22, t_fixed_s=20e-6, hbm_Bps=8e12,
                    block=4096) -> bool:
    return bool(lib().oracle_should_compress(numel, link_Bps, q_hat, t_fixed_s, hbm_Bps, block))


def bsc_select(numel, q, world: int, budget_bytes: int, link_Bps=8e9, t_fixed_s=20e-6,
               hbm_Bps=8e12, block=4096):
    """Section 3.2 shard selection.  Returns (selected u8[n], gain f64[n], count)."""
    numel = np.ascontiguousarray(numel, dtype=np.int64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    n = numel.size
    sel = np.zeros(max(n, 1), dtype=np.uint8)
    gain = np.zeros(max(n, 1), dtype=np.float64)
    cnt = lib().oracle_bsc_select(_ptr(numel) if n else None, _ptr(q) if n else None, n, world,
                                  budget_bytes, link_Bps, t_fixed_s, hbm_Bps, block, _ptr(sel),
                                  _ptr(gain))
    return sel[:n], gain[:n], int(cnt)


# ---- hashed sender (Hash128 + HashCache) -------------------------------------

def splitmix64(seed: int, index: int) -> int:
    """Output number `index` (1-based) of SplitMix64 started at `seed`."""
    return int(lib().oracle_splitmix64(seed & (2**64 - 1), index))


def exp_hash64(exps: np.ndarray, seed: int) -> int:
    exps = np.ascontiguousarray(exps, dtype=np.uint8)
    return int(lib().oracle_exp_hash64(_ptr(exps) if exps.size else None, exps.size,
                                       seed & (2**64 - 1)))


def block_hash128(vals: np.ndarray):
    vals = np.ascontiguousarray(vals, dtype=np.uint16)
    out = np.zeros(2, dtype=np.uint64)
    lib().oracle_block_hash128(_ptr(vals) if vals.size else None, vals.size, _ptr(out))
    return int(out[0]), int(out[1])


def compress_plan_hashed(w: np.ndarray, ranks: int, block: int, hash_cache: np.ndarray,
                         cold: bool, stride: int | None = None):
    """Sender side for every rank with the hashed change test.  ``hash_cache``
    (u64[ranks, blocks_per_full_shard, 2]) is updated in place.  Returns
    (payloads, descs, flags) like compress_plan."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    n = w.size
    s = shard_size(n, ranks) if n else 0
    if stride is None:
        stride = max(2 * s, 1)
    payloads = np.zeros((ranks, stride), dtype=np.uint8)
    descs = np.zeros(ranks, dtype=DESC_DTYPE)
    fstride = num_blocks(s, block) if n else 0
    flags = np.zeros((ranks, max(fstride, 1)), dtype=np.uint8)
    assert hash_cache.dtype == np.uint64 and hash_cache.size >= 2 * ranks * fstride
    lib().oracle_compress_plan_hashed(_ptr(w), n, ranks, block, _ptr(hash_cache),
                                      int(bool(cold)), _ptr(payloads), stride, _ptr(descs),
                                      _ptr(flags))
    return payloads, descs, flags[:, :fstride]


# ---- rANS-coded changed exponents (RANS payloads) ----------------------------

RANS = 2


def rans_table(hist) -> np.ndarray:
    hist = np.ascontiguousarray(hist, dtype=np.uint32)
    assert hist.size == 256
    freq = np.zeros(256, dtype=np.uint16)
    lib().oracle_rans_table(_ptr(hist), _ptr(freq))
    return freq


def rans_encode_block(exps: np.ndarray, freq: np.ndarray) -> np.ndarray:
    exps = np.ascontiguousarray(exps, dtype=np.uint8)
    freq = np.ascontiguousarray(freq, dtype=np.uint16)
    L = exps.size
    rec = np.zeros(64 + 32 * (4 + 2 * ((L + 31) // 32)) + 16, dtype=np.uint8)
    size = lib().oracle_rans_encode_block(_ptr(exps) if L else None, L, _ptr(freq), _ptr(rec))
    return rec[:size].copy()


def rans_decode_block(rec: np.ndarray, L: int, freq: np.ndarray):
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    freq = np.ascontiguousarray(freq, dtype=np.uint16)
    out = np.zeros(max(L, 1), dtype=np.uint8)
    st = lib().oracle_rans_decode_block(_ptr(rec), rec.size, L, _ptr(freq), _ptr(out))
    return int(st), out[:L]


def compress_shard_rans(shard, block, sender_cache, cold, hist_prev):
    """RANS sender for one shard.  Updates ``sender_cache``.  Returns
    (payload, flags, desc, hist_cur)."""
    shard = np.ascontiguousarray(shard, dtype=np.uint16)
    n = shard.size
    hist_prev = np.ascontiguousarray(hist_prev, dtype=np.uint32)
    hist_cur = np.zeros(256, dtype=np.uint32)
    payload = np.zeros(max(2 * n, 1), dtype=np.uint8)
    flags = np.zeros(max(num_blocks(n, block), 1), dtype=np.uint8)
    d = _Desc()
    lib().oracle_compress_shard_rans(_ptr(shard), n, block, _ptr(sender_cache), int(bool(cold)),
                                     _ptr(hist_prev), _ptr(hist_cur), _ptr(payload), _ptr(flags),
                                     ctypes.byref(d))
    desc = dict(mode=d.mode, n_changed_blocks=d.n_changed_blocks, body_bytes=d.body_bytes,
                payload_bytes=d.payload_bytes)
    return payload[:d.payload_bytes].copy(), flags[:num_blocks(n, block)].copy(), desc, hist_cur


def decompress_shard_any(payload, desc, length, block, recv_cache):
    """Receiver for one shard, any mode (RAW, COMPRESSED, RANS)."""
    if desc["mode"] != RANS:
        return decompress_shard(payload, desc, length, block, recv_cache)
    buf = np.ascontiguousarray(payload, dtype=np.uint8)
    if buf.size == 0:
        buf = np.zeros(1, np.uint8)
    out = np.zeros(max(length, 1), dtype=np.uint16)
    d = _Desc(desc["mode"], desc["n_changed_blocks"], desc["body_bytes"], desc["payload_bytes"])
    st = lib().oracle_decompress_shard_rans(_ptr(buf), ctypes.byref(d), length, block,
                                            _ptr(recv_cache), _ptr(out))
    return int(st), out[:length].copy()
