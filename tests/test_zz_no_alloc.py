"""ciera_compress_noalloc: the sender side for callers that cannot allocate
device memory where they compress (for instance inside a communication hook
or an allocator callback).  Its scratch is a fixed array inside libciera;
its results must equal ciera_compress's, call after call.

Called through the C ABI with ctypes.  Collected last on purpose, so that a
run stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from lossless_exponent_reuse_gb300 import ciera, workloads

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_compress_matches_workspace_compress_two_calls():
    torch.cuda.set_device(0)
    wl = workloads.small("noalloc", [(64, 4096), (48, 4096)], ranks=4, block=4096,
                         iterations=2, step=1e-3, p_block=0.25)
    seq = [w.to("cuda") for w in workloads.sequence(wl, 2, device="cpu")]
    n = seq[0].numel()
    plan = ciera.Plan(n, wl.block, wl.ranks)
    info = plan.info
    R, nb = info.ranks, info.blocks_per_shard
    L = ciera.lib()
    stream = torch.cuda.current_stream().cuda_stream

    def bufs():
        return dict(cache=torch.zeros(n, dtype=torch.uint8, device="cuda"),
                    pay=plan.new_payloads(), desc=plan.new_descs(),
                    flags=torch.zeros((R, nb), dtype=torch.uint8, device="cuda"))

    ref, new = bufs(), bufs()
    ws = plan.new_workspace()
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    for t, w in enumerate(seq):
        flags = ciera.COLD if t == 0 else 0
        assert L.ciera_compress(plan.handle, 0, R, _ptr(w), _ptr(ref["cache"]), _ptr(ref["pay"]),
                                ref["pay"].stride(0), _ptr(ref["desc"]), _ptr(ref["flags"]),
                                _ptr(ws), flags, stream) == ciera.OK
        assert L.ciera_compress_noalloc(plan.handle, 0, R, _ptr(w), _ptr(new["cache"]),
                                        _ptr(new["pay"]), new["pay"].stride(0),
                                        _ptr(new["desc"]), _ptr(new["flags"]), _ptr(status),
                                        flags, stream) == ciera.OK
        torch.cuda.synchronize()
        assert ciera.status(ws) == ciera.OK
        assert int(status.item()) == 0
        dr, dn = ciera.decode_descs(ref["desc"]), ciera.decode_descs(new["desc"])
        assert dr == dn
        for r, d in enumerate(dr):
            pb = d["payload_bytes"]
            assert torch.equal(ref["pay"][r, :pb], new["pay"][r, :pb]), (t, r)
        assert torch.equal(ref["flags"], new["flags"])
        assert torch.equal(ref["cache"], new["cache"])
        if t == 1:
            assert any(d["mode"] == ciera.MODE_COMPRESSED for d in dn)


def test_noalloc_rejects_plans_larger_than_its_scratch():
    plan = ciera.Plan(1 << 31, 256, 64)       # workspace far beyond 8 MiB
    assert plan.info.workspace_bytes > (8 << 20)
    fake = ctypes.c_void_p(4096)              # never dereferenced: the size check fails first
    L = ciera.lib()
    assert L.ciera_compress_noalloc(plan.handle, 0, 64, fake, fake, fake,
                                    plan.info.payload_capacity, fake, None, None, 0,
                                    None) == ciera.E_INVAL
