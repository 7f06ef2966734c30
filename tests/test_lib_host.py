"""Host-side checks of libciera that need no GPU: the library loads and
exports every function include/ciera.h declares; plan geometry; argument
validation; the predicate agrees with the oracle (CIERA Section 3.2)."""
import ctypes
import os
import re

import pytest

import oracle
from lossless_exponent_reuse_gb300 import ciera

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "ciera.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ciera_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("ciera_plan", "ciera_compress", "ciera_decompress",
                     "ciera_should_compress"):
        assert required in names


def test_library_exports_every_declared_symbol():
    L = ciera.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(declared_functions()) == set(ciera.SIGNATURES)


def test_plan_geometry():
    p = ciera.Plan((256, 512), 256, 4)
    i = p.info
    assert (i.numel, i.shard_len, i.blocks_per_shard, i.tile_blocks) == (131072, 32768, 128, 32)
    assert i.total_tiles == 4 * 4 and i.fast_path and not i.raw_fixup
    assert i.payload_capacity >= 2 * i.shard_len and i.payload_capacity % 256 == 0
    p = ciera.Plan(402653184, 4096, 16)
    assert (p.info.shard_len, p.info.blocks_per_shard, p.info.tile_blocks,
            p.info.total_tiles) == (25165824, 6144, 2, 49152)
    # ragged: 10 values over 4 ranks -> 3,3,3,1
    p = ciera.Plan(10, 2, 4)
    assert p.info.shard_len == 3 and not p.info.fast_path
    assert p.info.total_tiles == 4       # one tile per non-empty shard
    # sizes that disable the staged path
    assert not ciera.Plan(100003, 256, 3).info.fast_path     # S % 16 != 0
    assert not ciera.Plan(65536, 100, 2).info.fast_path      # B % 16 != 0
    assert not ciera.Plan(65536, 128, 2).info.fast_path      # B < 256
    assert not ciera.Plan(65536, 32768, 2).info.fast_path    # B > 16384
    assert ciera.Plan(98304, 16384, 3).info.fast_path


def test_raw_fixup_flag():
    assert ciera.Plan(8192, 16, 2).info.raw_fixup       # bitmap 32 B >= block 16
    assert ciera.Plan(12345, 1, 2).info.raw_fixup
    assert not ciera.Plan(402653184, 4096, 16).info.raw_fixup
    # partial last block of one value in an otherwise large-block shard
    assert ciera.Plan(4096 * 9 + 1, 4096, 1).info.raw_fixup


def test_plan_rejects_bad_arguments():
    for args in [((-1,), 4, 2), ((16,), 0, 2), ((16,), 4, 0), ((1 << 41,), 4096, 1),
                 ((1 << 39,), 1, 1)]:
        with pytest.raises(ciera.CieraError) as e:
            ciera.Plan(*args)
        assert e.value.status == ciera.E_INVAL


def test_compress_rejects_bad_ranges_without_touching_the_gpu():
    L = ciera.lib()
    p = ciera.Plan(1024, 256, 4)
    cap = p.info.payload_capacity
    fake = ctypes.c_void_p(4096)     # never dereferenced: the checks fail first
    args = lambda rb, rc, stride: (p.handle, rb, rc, fake, fake, fake, stride, fake, None,
                                   fake, 0, None)
    assert L.ciera_compress(*args(0, 5, cap)) == ciera.E_INVAL      # past the last rank
    assert L.ciera_compress(*args(-1, 1, cap)) == ciera.E_INVAL
    assert L.ciera_compress(*args(0, 0, cap)) == ciera.E_INVAL
    assert L.ciera_compress(*args(0, 4, cap - 1)) == ciera.E_INVAL  # short stride
    assert L.ciera_compress(p.handle, 0, 4, fake, fake, fake, cap, fake, None, fake, 0x40,
                            None) == ciera.E_INVAL                  # unknown flag
    assert L.ciera_compress(p.handle, 0, 4, fake, fake, fake, cap, fake, None, fake,
                            0x40000000, None) == ciera.E_INVAL      # unknown flag
    assert L.ciera_decompress(p.handle, fake, cap - 1, fake, fake, fake, fake, 0,
                              None) == ciera.E_INVAL
    assert L.ciera_decompress(p.handle, fake, cap, fake, fake, fake, fake, 2,
                              None) == ciera.E_INVAL                # unknown flag


def test_gather_and_host_step_reject_bad_arguments_without_touching_the_gpu():
    L = ciera.lib()
    p = ciera.Plan(1024, 256, 4)
    cap = p.info.payload_capacity
    fake = ctypes.c_void_p(4096)     # never dereferenced: the checks fail first
    gather = lambda table, capacity, flags: L.ciera_decompress_gather(
        p.handle, table, capacity, fake, fake, fake, fake, flags, None)
    assert gather(None, cap, 0) == ciera.E_INVAL                      # no pointer table
    assert gather(ctypes.c_void_p(4100), cap, 0) == ciera.E_INVAL     # table not 8-byte aligned
    assert gather(fake, cap - 1, 0) == ciera.E_INVAL                  # short capacity
    assert gather(fake, cap, 2) == ciera.E_INVAL                      # unknown flag
    h = ctypes.c_void_p()
    assert L.ciera_host_session_create(0, ctypes.byref(h)) == ciera.E_INVAL
    assert L.ciera_host_session_create(4, None) == ciera.E_INVAL
    host = ctypes.c_void_p(8192)
    assert L.ciera_step_host(None, p.handle, host, host, fake, fake, fake, cap, fake, fake, fake,
                             fake, 0, 1, None) == ciera.E_INVAL       # no session
    L.ciera_host_session_destroy(None)                                # NULL is ignored


def test_predicate_matches_oracle():
    for n in [0, 1, 2047, 2048, 131072, 200000, 206000, 206300, 207000, 2097152, 4194304,
              10**9]:
        assert ciera.should_compress(n) == oracle.should_compress(n), n


def test_predicate_cost_model_round_trip_and_agreement():
    saved = ciera.get_cost_model()
    try:
        models = [dict(link_Bps=16e9, q_hat=0.22, t_fixed_s=20e-6, hbm_Bps=8e12, block=4096),
                  dict(link_Bps=8e9, q_hat=1.0, t_fixed_s=20e-6, hbm_Bps=8e12, block=4096),
                  dict(link_Bps=50e9, q_hat=0.05, t_fixed_s=5e-6, hbm_Bps=6.8e12, block=512),
                  dict(link_Bps=8e9, q_hat=0.0, t_fixed_s=0.0, hbm_Bps=1e300, block=1)]
        for m in models:
            ciera.set_cost_model(**m)
            assert ciera.get_cost_model() == m
            for n in [1, 2, 10, 2048, 131072, 206252, 414760, 2097152, 4194304]:
                assert ciera.should_compress(n) == oracle.should_compress(n, **m), (m, n)
        for bad in [dict(link_Bps=0), dict(q_hat=1.5), dict(t_fixed_s=-1), dict(block=0),
                    dict(hbm_Bps=-3)]:
            with pytest.raises(ciera.CieraError):
                ciera.set_cost_model(**dict(models[0], **bad))
    finally:
        ciera.set_cost_model(**saved)
    assert ciera.get_cost_model() == saved


def test_timeout_setting_validation():
    with pytest.raises(ciera.CieraError):
        ciera.set_wait_timeout_ns(0)
    ciera.set_wait_timeout_ns(1_000_000_000)


def test_strerror():
    assert ciera.strerror(ciera.OK) == "ok"
    assert "corrupt" in ciera.strerror(ciera.E_CORRUPT)
    assert "timed out" in ciera.strerror(ciera.E_TIMEOUT)


def test_hashed_compress_needs_tiles_of_at_most_32_blocks():
    L = ciera.lib()
    p = ciera.Plan(1 << 20, 128, 4)           # 64 blocks per tile
    cap = p.info.payload_capacity
    fake = ctypes.c_void_p(4096)              # never dereferenced: the check fails first
    assert L.ciera_compress_hashed(p.handle, 0, 4, fake, fake, fake, cap, fake, None, fake, 0,
                                   None) == ciera.E_INVAL


def test_rans_entry_points_reject_what_the_staged_kernels_cannot_take():
    L = ciera.lib()
    fake = ctypes.c_void_p(4096)              # never dereferenced: the checks fail first
    odd = ctypes.c_void_p(4097)

    def rans(plan, w=fake, hp=fake, ho=ctypes.c_void_p(1 << 20), stride=None, flags=0):
        cap = plan.info.payload_capacity if stride is None else stride
        return L.ciera_compress_rans(plan.handle, 0, plan.info.ranks, w, fake, hp, ho, fake,
                                     cap, fake, None, fake, flags, None)

    assert rans(ciera.Plan(100003, 256, 3)) == ciera.E_INVAL    # no staged path (S % 16)
    assert rans(ciera.Plan(131069, 256, 4)) == ciera.E_INVAL    # N % 16 != 0
    assert rans(ciera.Plan(65536, 128, 2)) == ciera.E_INVAL     # block below 256
    p = ciera.Plan(131072, 256, 4)
    assert rans(p, w=odd) == ciera.E_INVAL                      # unaligned values
    assert rans(p, hp=ctypes.c_void_p(4098)) == ciera.E_INVAL   # unaligned histogram
    assert rans(p, ho=ctypes.c_void_p(4096 + 1024)) == ciera.E_INVAL  # histograms overlap
    assert rans(p, stride=p.info.payload_capacity + 8) == ciera.E_INVAL  # stride % 16
    assert rans(p, flags=0x40) == ciera.E_INVAL
    assert L.ciera_compress_rans(p.handle, 0, 4, fake, fake, None, fake, fake,
                                 p.info.payload_capacity, fake, None, fake, 0,
                                 None) == ciera.E_INVAL        # no histogram
    # the receiver takes RANS payloads only on the staged path
    q = ciera.Plan(100003, 256, 3)
    assert L.ciera_decompress(q.handle, fake, q.info.payload_capacity, fake, fake, fake, fake,
                              ciera.DECOMPRESS_RANS, None) == ciera.E_INVAL
    assert L.ciera_decompress(p.handle, fake, p.info.payload_capacity, fake, odd, fake, fake,
                              ciera.DECOMPRESS_RANS, None) == ciera.E_INVAL


def test_checked_build_compiles_and_exports_the_same_symbols():
    import ctypes as ct
    from lossless_exponent_reuse_gb300 import _build
    path = _build.build(checked=True)
    L = ct.CDLL(path)
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.ciera_strerror(ciera.E_BOUNDS) is not None


def _c_layout(struct, fields):
    """sizeof and offsetof of a header struct, from a C program built with gcc
    against include/ciera.h (host compiler only; nothing runs on a GPU)."""
    import subprocess
    import tempfile
    body = "".join(f'  printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields)
    src = ("#include <stddef.h>\n#include <stdio.h>\n#include \"ciera.h\"\n"
           f"int main(void) {{\n  printf(\"%zu\\n\", sizeof({struct}));\n{body}  return 0;\n}}\n")
    with tempfile.TemporaryDirectory() as d:
        c, exe = os.path.join(d, "l.c"), os.path.join(d, "l")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), c, "-o", exe],
                       check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    return int(out[0]), [int(v) for v in out[1:]]


@pytest.mark.parametrize("struct,cls", [("ciera_plan_info_t", ciera._Info),
                                        ("ciera_layer", ciera._Layer),
                                        ("ciera_cost_model", ciera._CostModel)])
def test_binding_struct_layouts_match_the_header(struct, cls):
    fields = [f for f, _ in cls._fields_]
    size, offsets = _c_layout(struct, fields)
    assert ctypes.sizeof(cls) == size, struct
    assert [getattr(cls, f).offset for f in fields] == offsets, struct


def test_descriptor_is_24_bytes():
    size, offsets = _c_layout("ciera_desc", ["mode", "n_changed_blocks", "body_bytes",
                                             "payload_bytes"])
    assert size == ciera.DESC_BYTES and offsets == [0, 4, 8, 16]


def test_no_raw_ahead_is_a_known_compress_flag():
    # unknown flags are refused before anything is launched; this one is not
    # refused as unknown, so the call goes on to CUDA, which fails here for
    # want of a device.  With a GPU the fake pointers would reach a kernel:
    # there the test does not run.
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU (fake device pointers)")
    L = ciera.lib()
    p = ciera.Plan(1024, 256, 4)
    cap = p.info.payload_capacity
    fake = ctypes.c_void_p(4096)
    rc = L.ciera_compress(p.handle, 0, 4, fake, fake, fake, cap, fake, None, fake,
                          ciera.NO_RAW_AHEAD, None)
    assert rc == ciera.E_CUDA
