"""Parity harness: runs the same seeded weight sequence through libciera on
the GPU and through the CPU oracle, and compares every output byte for byte:
per-block flags, descriptors, payload bytes, the rebuilt tensor and both
exponent caches."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from lossless_exponent_reuse_gb300 import ciera
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather


def exps_dev(w_u16: torch.Tensor) -> torch.Tensor:
    """Exponent bytes of bf16 bit patterns, computed with torch ops (test side)."""
    return ((w_u16.view(torch.int16).to(torch.int32) >> 7) & 0xFF).to(torch.uint8)


def eq16(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality of two 16-bit tensors (compared as int16)."""
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


class OracleState:
    def __init__(self, n, ranks, block):
        self.n, self.ranks, self.block = n, ranks, block
        self.scache = np.zeros(n, np.uint8)
        self.rcache = np.zeros(n, np.uint8)
        self.t = 0

    def step(self, w: np.ndarray):
        payloads, descs, flags = oracle.compress_plan(w, self.ranks, self.block, self.scache,
                                                      cold=self.t == 0)
        st, out = oracle.decompress_plan(payloads, descs, self.n, self.ranks, self.block,
                                         self.rcache)
        assert st == 0
        self.t += 1
        return payloads, descs, flags, out


def compare_step(ag: SimulatedAllgather, ost: OracleState, w_np: np.ndarray, o_payloads,
                 o_descs, o_flags, o_out, tag=""):
    n, R, B = ost.n, ost.ranks, ost.block
    g_descs = ag.descriptors()
    g_payloads = to_np_u8(ag.payloads)
    g_flags = to_np_u8(ag.flags)
    for r in range(R):
        od = o_descs[r]
        gd = g_descs[r]
        assert (gd["mode"], gd["n_changed_blocks"], gd["body_bytes"], gd["payload_bytes"]) == (
            int(od["mode"]), int(od["n_changed_blocks"]), int(od["body_bytes"]),
            int(od["payload_bytes"])), f"{tag} rank {r} descriptor"
        pb = int(od["payload_bytes"])
        if not np.array_equal(g_payloads[r, :pb], o_payloads[r, :pb]):
            bad = np.nonzero(g_payloads[r, :pb] != o_payloads[r, :pb])[0]
            raise AssertionError(f"{tag} rank {r} payload differs at {bad[:10]} of {pb}")
        ln = oracle.shard_len(n, R, r)
        nb = oracle.num_blocks(ln, B) if ln else 0
        np.testing.assert_array_equal(g_flags[r, :nb], o_flags[r, :nb],
                                      err_msg=f"{tag} rank {r} flags")
    np.testing.assert_array_equal(to_np_u16(ag.out[:n]), o_out, err_msg=f"{tag} out")
    np.testing.assert_array_equal(to_np_u8(ag.sender_cache[:n]), ost.scache,
                                  err_msg=f"{tag} sender cache")
    np.testing.assert_array_equal(to_np_u8(ag.recv_cache[:n]), ost.rcache,
                                  err_msg=f"{tag} receiver cache")
    np.testing.assert_array_equal(o_out, w_np, err_msg=f"{tag} oracle round trip")


def run_parity(seq_np, ranks, block, device="cuda", tag="", raw_ahead=True):
    """seq_np: list of uint16 numpy arrays (w_0, w_1, ...).  raw_ahead=False
    sends every shard through the look-back scan."""
    n = seq_np[0].size
    ag = SimulatedAllgather(n, block, ranks, device=device, keep_flags=True,
                            raw_ahead=raw_ahead)
    ost = OracleState(n, ranks, block)
    for t, w in enumerate(seq_np):
        w_dev = torch.from_numpy(w.view(np.int16)).to(device).view(torch.uint16)
        ag.step(w_dev)
        st = ag.status()
        assert st == ciera.OK, f"{tag} t={t} status {ciera.strerror(st)}"
        o_payloads, o_descs, o_flags, o_out = ost.step(w)
        compare_step(ag, ost, w, o_payloads, o_descs, o_flags, o_out, tag=f"{tag} t={t}")
    return ag, ost


def raw_ahead_sequence(n, ranks, block, iters=7, seed=0):
    """Shard 0 changes every block every iteration (raw-ahead predicted right
    after the cold start); shard 1 alternates between every block changed
    and one changed value (predicted raw, then compacted: a rewrite every
    other iteration); the remaining shards change sparsely."""
    rng = np.random.default_rng(seed)
    S = -(-n // ranks)
    w = (rng.normal(0.0, 0.02, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    seq = [w.copy()]
    for t in range(1, iters):
        w = w.copy()
        w[:S] ^= np.uint16(0x0080)
        if t % 2:
            w[S:2 * S] ^= np.uint16(0x0080)
        else:
            w[S + int(rng.integers(0, S))] ^= np.uint16(0x0080)
        if ranks > 2:
            idx = rng.integers(2 * S, n, max(1, (n - 2 * S) // 50000))
            w[idx] ^= np.uint16(0x0100)
        seq.append(w)
    return seq


class OracleAny:
    """The oracle's side of one plan for any of the three senders: the
    sender's state (exponent cache; HashCache for the hashed change test;
    exponent cache and per-rank exponent histograms for RANS payloads) and
    the receiver's exponent cache, carried from call to call."""

    def __init__(self, n, ranks, block, sender="exact"):
        self.n, self.ranks, self.block, self.sender = n, ranks, block, sender
        S = oracle.shard_size(n, ranks) if n else 0
        self.scache = np.zeros(n, np.uint8)
        self.rcache = np.zeros(n, np.uint8)
        self.hcache = (np.zeros((ranks, max(oracle.num_blocks(S, block), 1), 2), np.uint64)
                       if sender == "hashed" else None)
        self.hist = [np.zeros(256, np.uint32) for _ in range(ranks)]
        self.t = 0

    def step(self, w: np.ndarray):
        """One call of the sender for every rank and of the receiver.
        Returns (per-rank payload bytes, per-rank descriptor dicts, flags
        u8[ranks, blocks], rebuilt values)."""
        n, R, B = self.n, self.ranks, self.block
        cold = self.t == 0
        payloads, descs, flags = [], [], []
        out = np.zeros(n, np.uint16)
        if self.sender in ("exact", "hashed"):
            if self.sender == "exact":
                P, D, F = oracle.compress_plan(w, R, B, self.scache, cold=cold)
            else:
                P, D, F = oracle.compress_plan_hashed(w, R, B, self.hcache, cold=cold)
            st, out = oracle.decompress_plan(P, D, n, R, B, self.rcache)
            assert st == 0
            for r in range(R):
                d = {k: int(D[r][k]) for k in ("mode", "n_changed_blocks", "body_bytes",
                                               "payload_bytes")}
                descs.append(d)
                payloads.append(P[r, :d["payload_bytes"]])
            flags = F
        else:
            nbmax = oracle.num_blocks(oracle.shard_size(n, R), B) if n else 0
            flags = np.zeros((R, nbmax), np.uint8)
            for r in range(R):
                b, ln = oracle.shard_begin(n, R, r), oracle.shard_len(n, R, r)
                sc = self.scache[b:b + ln].copy()
                p, f, d, h = oracle.compress_shard_rans(w[b:b + ln], B, sc, cold, self.hist[r])
                self.scache[b:b + ln] = sc
                self.hist[r] = h
                rc = self.rcache[b:b + ln].copy()
                st, o = oracle.decompress_shard_any(p, d, ln, B, rc)
                assert st == 0
                self.rcache[b:b + ln] = rc
                out[b:b + ln] = o
                flags[r, :f.size] = f
                payloads.append(p)
                descs.append({k: int(v) for k, v in d.items()})
        self.t += 1
        return payloads, descs, flags, out


def compare_any(ag: SimulatedAllgather, ost: OracleAny, w_np: np.ndarray, result, tag="",
                check_flags=False):
    """Every output of one GPU step against the oracle's: descriptors,
    payload bytes, rebuilt values, both sides' state, and (when the GPU
    state keeps them) the per-block flags."""
    payloads, descs, flags, out = result
    n = ost.n
    g_descs = ag.descriptors()
    g_payloads = to_np_u8(ag.payloads)
    for r in range(ost.ranks):
        assert g_descs[r] == descs[r], f"{tag} rank {r} descriptor {g_descs[r]} != {descs[r]}"
        pb = descs[r]["payload_bytes"]
        if not np.array_equal(g_payloads[r, :pb], payloads[r][:pb]):
            bad = np.nonzero(g_payloads[r, :pb] != payloads[r][:pb])[0]
            raise AssertionError(f"{tag} rank {r} payload differs at {bad[:10]} of {pb}")
    if check_flags:
        nb = flags.shape[1]
        np.testing.assert_array_equal(to_np_u8(ag.flags)[:, :nb], flags, err_msg=f"{tag} flags")
    np.testing.assert_array_equal(to_np_u16(ag.out[:n]), out, err_msg=f"{tag} out")
    np.testing.assert_array_equal(out, w_np, err_msg=f"{tag} oracle round trip")
    np.testing.assert_array_equal(to_np_u8(ag.recv_cache[:n]), ost.rcache,
                                  err_msg=f"{tag} receiver cache")
    if ost.sender == "hashed":
        g_h = ag.hash_cache.cpu().numpy().view(np.uint64)
        nb = ost.hcache.shape[1]
        np.testing.assert_array_equal(g_h[:, :nb], ost.hcache, err_msg=f"{tag} HashCache")
    else:
        np.testing.assert_array_equal(to_np_u8(ag.sender_cache[:n]), ost.scache,
                                      err_msg=f"{tag} sender cache")
    if ost.sender == "rans":
        cur = ag.hist[ag.iteration % 2].cpu().numpy().view(np.uint32)
        for r in range(ost.ranks):
            np.testing.assert_array_equal(cur[r], ost.hist[r], err_msg=f"{tag} rank {r} hist")
