"""Full-size workloads on the GPU, in the launch configuration the benchmark
times (all ranks in one compress launch, one fused gather-decompress).

Sampled ranks are recomputed by the CPU oracle shard by shard and compared
byte for byte (payload, flags, descriptor, rebuilt values, both caches); the
whole tensor is checked through properties that hold at any size: the
round trip is exact and both caches equal the new exponents.
CIERA Section 3.1, Section 3.2 and Appendix A, Algorithm 1.
"""
import numpy as np
import pytest
import torch

import oracle
from harness import exps_dev, to_np_u16, to_np_u8
from lossless_exponent_reuse_gb300 import ciera, workloads
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _check_iteration(ag, w, sampled, t, tag):
    """Run one iteration of `w` (device uint16) and check it."""
    n = ag.numel
    R = ag.plan.info.ranks
    B = ag.plan.info.block
    S = ag.plan.info.shard_len
    snap = {}
    for r in sampled:
        b, ln = oracle.shard_begin(n, R, r), oracle.shard_len(n, R, r)
        snap[r] = (b, ln, to_np_u8(ag.sender_cache[b:b + ln]).copy(),
                   to_np_u8(ag.recv_cache[b:b + ln]).copy(), to_np_u16(w[b:b + ln]).copy())
    ag.step(w)
    assert ag.status() == ciera.OK, tag
    # whole tensor: exact round trip and cache invariants
    assert torch.equal(ag.out[:n].view(torch.int16), w.view(torch.int16)), tag
    e = exps_dev(w)
    assert torch.equal(ag.sender_cache[:n], e), tag
    assert torch.equal(ag.recv_cache[:n], e), tag
    descs = ag.descriptors()
    for r in sampled:
        b, ln, sc, rc, ws = snap[r]
        payload, flags, d = oracle.compress_shard(ws, B, sc, cold=t == 0)
        gd = descs[r]
        assert (gd["mode"], gd["n_changed_blocks"], gd["body_bytes"], gd["payload_bytes"]) == (
            d["mode"], d["n_changed_blocks"], d["body_bytes"], d["payload_bytes"]), (tag, r)
        pb = d["payload_bytes"]
        np.testing.assert_array_equal(to_np_u8(ag.payloads[r, :pb]), payload,
                                      err_msg=f"{tag} rank {r} payload")
        np.testing.assert_array_equal(to_np_u8(ag.flags[r, :len(flags)]), flags,
                                      err_msg=f"{tag} rank {r} flags")
        np.testing.assert_array_equal(to_np_u8(ag.sender_cache[b:b + ln]), sc)
        st, out = oracle.decompress_shard(payload, d, ln, B, rc)
        assert st == 0
        np.testing.assert_array_equal(to_np_u16(ag.out[b:b + ln]), out)
        np.testing.assert_array_equal(to_np_u8(ag.recv_cache[b:b + ln]), rc)
    return descs


def _run(wl, iterations, sampled, layer=0):
    dev = "cuda"
    n = wl.layer_numel
    ag = SimulatedAllgather(n, wl.block, wl.ranks, device=dev, keep_flags=True)
    w = workloads.initial_layer(wl, layer, dev)
    all_descs = []
    for t in range(iterations):
        if t > 0:
            w = workloads.step_layer(wl, w, layer, t)
        all_descs.append(_check_iteration(ag, w, sampled, t, f"{wl.name} t={t}"))
    del ag
    torch.cuda.empty_cache()
    return all_descs


def _exp_change_rate(a, b):
    return float((exps_dev(a) != exps_dev(b)).float().mean())


def test_workload_1_matrix_all_iterations():
    wl = workloads.workload(1)
    descs = _run(wl, wl.iterations, sampled=[0, 1, 2, 3])
    assert all(d["mode"] == ciera.MODE_RAW for d in descs[0])      # cold start


def test_workload_2_olmoe_layer_all_iterations():
    wl = workloads.workload(2)
    descs = _run(wl, wl.iterations, sampled=[0, 7, 15])
    assert len(descs) == 10
    assert all(d["mode"] == ciera.MODE_RAW for d in descs[0])      # cold start


def test_workload_3_warmup_and_forced_change():
    wl = workloads.workload(3)
    descs = _run(wl, wl.iterations, sampled=[3, 12])
    forced = descs[3]
    blocks = wl.layer_numel // wl.ranks // wl.block
    assert all(d["mode"] == ciera.MODE_RAW and d["n_changed_blocks"] == blocks for d in forced)


def test_workload_5_finegrained_layer_every_rate():
    """All 16 iterations: the cold start, then five at each step size
    (about 0.1 %, 1 % and 10 % of exponents change), sampled ranks against
    the oracle at every one of them."""
    wl = workloads.workload(5)
    assert wl.iterations == 16
    dev = "cuda"
    n = wl.layer_numel
    ag = SimulatedAllgather(n, wl.block, wl.ranks, device=dev, keep_flags=True)
    w = workloads.initial_layer(wl, 0, dev)
    rates = {}
    for t in range(wl.iterations):
        if t > 0:
            w_new = workloads.step_layer(wl, w, 0, t)
            rates.setdefault(wl.step_of(t), []).append(_exp_change_rate(w, w_new))
            w = w_new
        # ranks 0 and 31 at every iteration, one more rank that moves along
        _check_iteration(ag, w, [0, 31, 1 + (5 * t) % 30], t, f"{wl.name} t={t}")
    del ag, w
    torch.cuda.empty_cache()
    mean = {k: sum(v) / len(v) for k, v in rates.items()}
    assert len(mean) == 3 and all(len(v) == 5 for v in rates.values())
    lo, mid, hi = (mean[k] for k in sorted(mean))
    assert 0.0003 < lo < 0.003 and 0.003 < mid < 0.03 and 0.03 < hi < 0.3, mean


def test_workload_2_clustered_variant():
    wl = workloads.workload(2, "clustered0.1")
    descs = _run(wl, 3, sampled=[5])
    assert all(d["mode"] == ciera.MODE_COMPRESSED for d in descs[2])


@pytest.mark.parametrize("layer", [0, 9])
def test_workload_4_layer_bucket_and_declines(layer):
    """All 5 iterations of one layer's bucket of accepted tensors (layer 0
    and layer 9 of the 16), sampled ranks against the oracle each time."""
    wl = workloads.workload(4)
    offs = workloads.layer_offsets(wl)
    accepted = [(name, o, k) for name, o, k in offs if ciera.should_compress(k)]
    declined = [name for name, o, k in offs if not ciera.should_compress(k)]
    assert sorted(declined) == ["input_norm", "post_attn_norm", "router"]
    for name, o, k in offs:
        assert ciera.should_compress(k) == oracle.should_compress(k), name
    n = sum(k for _, _, k in accepted)
    assert n == 419_430_400
    dev = "cuda"
    ag = SimulatedAllgather(n, wl.block, wl.ranks, device=dev, keep_flags=True)
    full = workloads.initial_layer(wl, layer, dev)
    for t in range(wl.iterations):
        if t > 0:
            full = workloads.step_layer(wl, full, layer, t)
        bucket = torch.cat([full[o:o + k].view(torch.int16) for _, o, k in accepted]).view(
            torch.uint16)
        _check_iteration(ag, bucket, [0, 3 + t % 4, 7], t, f"cfg4 layer{layer} t={t}")
    del ag, full, bucket
    torch.cuda.empty_cache()


def _run_rans(wl, iterations, sampled):
    """The RANS sender and receiver at full size: every iteration, sampled
    ranks against the oracle byte for byte (payload, flags, descriptor,
    histogram, caches, rebuilt values), the whole tensor by properties."""
    dev = "cuda"
    n = wl.layer_numel
    R, B = wl.ranks, wl.block
    ag = SimulatedAllgather(n, B, R, device=dev, keep_flags=True, rans=True)
    ref = {}
    for r in sampled:
        ln = oracle.shard_len(n, R, r)
        ref[r] = dict(sc=np.zeros(ln, np.uint8), rc=np.zeros(ln, np.uint8),
                      hist=np.zeros(256, np.uint32))
    w = workloads.initial_layer(wl, 0, dev)
    modes = set()
    for t in range(iterations):
        if t > 0:
            w = workloads.step_layer(wl, w, 0, t)
        tag = f"{wl.name} rans t={t}"
        shards = {r: to_np_u16(w[oracle.shard_begin(n, R, r):][:oracle.shard_len(n, R, r)])
                  for r in sampled}
        ag.step(w)
        assert ag.status() == ciera.OK, tag
        assert torch.equal(ag.out[:n].view(torch.int16), w.view(torch.int16)), tag
        e = exps_dev(w)
        assert torch.equal(ag.sender_cache[:n], e), tag
        assert torch.equal(ag.recv_cache[:n], e), tag
        descs = ag.descriptors()
        hist_gpu = ag.hist[(t + 1) % 2].cpu().numpy().view(np.uint32)
        for r in sampled:
            b, ln = oracle.shard_begin(n, R, r), oracle.shard_len(n, R, r)
            st = ref[r]
            payload, flags, d, h = oracle.compress_shard_rans(shards[r], B, st["sc"], t == 0,
                                                              st["hist"])
            st["hist"] = h
            gd = descs[r]
            modes.add(int(d["mode"]))
            assert (gd["mode"], gd["n_changed_blocks"], gd["body_bytes"], gd["payload_bytes"]) == (
                d["mode"], d["n_changed_blocks"], d["body_bytes"], d["payload_bytes"]), (tag, r)
            pb = int(d["payload_bytes"])
            np.testing.assert_array_equal(to_np_u8(ag.payloads[r, :pb]), payload[:pb],
                                          err_msg=f"{tag} rank {r} payload")
            np.testing.assert_array_equal(to_np_u8(ag.flags[r, :len(flags)]), flags)
            np.testing.assert_array_equal(hist_gpu[r], h, err_msg=f"{tag} rank {r} histogram")
            np.testing.assert_array_equal(to_np_u8(ag.sender_cache[b:b + ln]), st["sc"])
            rs, out = oracle.decompress_shard_any(payload, d, ln, B, st["rc"])
            assert rs == 0
            np.testing.assert_array_equal(to_np_u16(ag.out[b:b + ln]), out)
            np.testing.assert_array_equal(to_np_u8(ag.recv_cache[b:b + ln]), st["rc"])
    del ag
    torch.cuda.empty_cache()
    return modes


def test_workload_2_rans_sender():
    modes = _run_rans(workloads.workload(2), 3, sampled=[0, 15])
    assert ciera.MODE_RANS in modes


def test_workload_2_clustered_rans_sender():
    modes = _run_rans(workloads.workload(2, "clustered0.1"), 3, sampled=[6])
    assert ciera.MODE_RANS in modes
