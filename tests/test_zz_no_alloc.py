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


class _Case:
    """One plan with its seeded weight sequence, the state of a reference
    sender (ciera_compress with its own workspace) and of an allocation-free
    one (ciera_compress_noalloc)."""

    def __init__(self, name, shapes, ranks, block, iterations, p_block):
        wl = workloads.small(name, shapes, ranks=ranks, block=block, iterations=iterations,
                             step=1e-3, p_block=p_block)
        self.seq = [w.to("cuda") for w in workloads.sequence(wl, iterations, device="cpu")]
        self.n = self.seq[0].numel()
        self.plan = ciera.Plan(self.n, block, ranks)
        info = self.plan.info
        self.R, nb = info.ranks, info.blocks_per_shard

        def bufs():
            return dict(cache=torch.zeros(self.n, dtype=torch.uint8, device="cuda"),
                        pay=self.plan.new_payloads(), desc=self.plan.new_descs(),
                        flags=torch.zeros((self.R, nb), dtype=torch.uint8, device="cuda"))

        self.ref, self.new = bufs(), bufs()
        self.ws = self.plan.new_workspace()

    def step(self, t, with_flags):
        """Iteration t through both senders; compare everything they return."""
        L = ciera.lib()
        stream = torch.cuda.current_stream().cuda_stream
        w = self.seq[t]
        ref, new = self.ref, self.new
        flags = ciera.COLD if t == 0 else 0
        status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
        assert L.ciera_compress(self.plan.handle, 0, self.R, _ptr(w), _ptr(ref["cache"]),
                                _ptr(ref["pay"]), ref["pay"].stride(0), _ptr(ref["desc"]),
                                _ptr(ref["flags"]), _ptr(self.ws), flags, stream) == ciera.OK
        assert L.ciera_compress_noalloc(self.plan.handle, 0, self.R, _ptr(w),
                                        _ptr(new["cache"]), _ptr(new["pay"]),
                                        new["pay"].stride(0), _ptr(new["desc"]),
                                        _ptr(new["flags"]) if with_flags else None,
                                        _ptr(status), flags, stream) == ciera.OK
        torch.cuda.synchronize()
        assert ciera.status(self.ws) == ciera.OK
        assert int(status.item()) == 0
        dr, dn = ciera.decode_descs(ref["desc"]), ciera.decode_descs(new["desc"])
        assert dr == dn, t
        for r, d in enumerate(dr):
            pb = d["payload_bytes"]
            assert torch.equal(ref["pay"][r, :pb], new["pay"][r, :pb]), (t, r)
        if with_flags:
            assert torch.equal(ref["flags"], new["flags"])
        assert torch.equal(ref["cache"], new["cache"])
        return dn


@pytest.mark.parametrize("with_flags", [True, False])
def test_noalloc_compress_matches_workspace_compress_two_calls(with_flags):
    """Two calls in a row (the cold start, then a step with some blocks
    changed), with and without the optional flags output (without it the flag
    bytes go to the library's own array)."""
    torch.cuda.set_device(0)
    case = _Case("noalloc", [(64, 4096), (48, 4096)], 4, 4096, 2, 0.25)
    case.step(0, with_flags)
    dn = case.step(1, with_flags)
    assert any(d["mode"] == ciera.MODE_COMPRESSED for d in dn)


def test_noalloc_plans_of_three_shapes_take_turns():
    """Calls for plans whose scratch layouts differ (blocks of 4096 and of
    256, so two and 32 blocks per tile; shards of a multiple of 16 values,
    staged through shared memory, and of 21846 values, byte by byte),
    alternating on one stream without the flags output: each call must still
    equal ciera_compress."""
    torch.cuda.set_device(0)
    a = _Case("noalloc_a", [(64, 4096), (48, 4096)], 4, 4096, 4, 0.25)
    b = _Case("noalloc_b", [(131072,)], 8, 256, 4, 0.05)
    c = _Case("noalloc_c", [(131072,)], 6, 256, 4, 0.05)
    assert a.plan.info.fast_path and b.plan.info.fast_path and not c.plan.info.fast_path
    modes = set()
    for t in range(4):
        for case in (a, b, c):
            modes.update(d["mode"] for d in case.step(t, with_flags=False))
    assert ciera.MODE_COMPRESSED in modes


def test_noalloc_rejects_plans_larger_than_its_scratch():
    plan = ciera.Plan(1 << 31, 256, 64)       # workspace far beyond 8 MiB
    assert plan.info.workspace_bytes > (8 << 20)
    fake = ctypes.c_void_p(4096)              # never dereferenced: the size check fails first
    L = ciera.lib()
    assert L.ciera_compress_noalloc(plan.handle, 0, 64, fake, fake, fake,
                                    plan.info.payload_capacity, fake, None, None, 0,
                                    None) == ciera.E_INVAL
