"""Thin ctypes binding of libciera (include/ciera.h), same names as the C ABI.

Only argument marshalling happens here: torch tensors supply device memory
and the current CUDA stream; every step of compression and reconstruction
runs in libciera's sm_103a kernels.  There is no CPU fallback: without the
built library or a CUDA device the calls raise.

Method: "CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in
Sharded MoE Training", Section 3.1 (Exponent Reuse), Section 3.2
(Benefit-driven Selective Compression), Appendix A (Algorithm 1).
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence, Union

import torch

from . import _build

OK = 0
E_INVAL = -1
E_CUDA = -2
E_CORRUPT = -3
E_TIMEOUT = -4
E_INTERNAL = -5
E_BOUNDS = -6

MODE_COMPRESSED = 0
MODE_RAW = 1
MODE_RANS = 2

COLD = 1
NO_RAW_AHEAD = 2  # compress: every shard takes the look-back scan
DECOMPRESS_RANS = 1
SENDER_EXACT = 0
SENDER_RANS = 1
SENDER_HASHED = 2
DEBUG_SKIP_FIRST_PUBLISH = 0x80000000

DESC_BYTES = 24


class CieraError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} ({status})")
        self.status = status


class _Info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "numel", "ranks", "block", "shard_len", "blocks_per_shard", "tile_blocks",
        "total_tiles", "payload_capacity", "workspace_bytes")] + [
        ("fast_path", ctypes.c_int32), ("raw_fixup", ctypes.c_int32)]


class _Layer(ctypes.Structure):
    _fields_ = [("plan", ctypes.c_void_p), ("w_dev", ctypes.c_void_p),
                ("sender_cache_dev", ctypes.c_void_p), ("payloads_dev", ctypes.c_void_p),
                ("payload_stride", ctypes.c_int64), ("descs_dev", ctypes.c_void_p),
                ("recv_cache_dev", ctypes.c_void_p), ("out_dev", ctypes.c_void_p),
                ("workspace_dev", ctypes.c_void_p), ("flags", ctypes.c_uint32),
                ("sender", ctypes.c_uint32), ("hist_prev_dev", ctypes.c_void_p),
                ("hist_out_dev", ctypes.c_void_p), ("hash_cache_dev", ctypes.c_void_p)]


class _CostModel(ctypes.Structure):
    _fields_ = [("link_Bps", ctypes.c_double), ("q_hat", ctypes.c_double),
                ("t_fixed_s", ctypes.c_double), ("hbm_Bps", ctypes.c_double),
                ("block", ctypes.c_int64)]


# Every symbol include/ciera.h declares, with (restype, argtypes).
_vp, _i64, _i32, _u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
SIGNATURES = {
    "ciera_plan": (_i32, [ctypes.POINTER(ctypes.c_int64), _i32, _i64, _i32,
                          ctypes.POINTER(_vp)]),
    "ciera_plan_info": (_i32, [_vp, ctypes.POINTER(_Info)]),
    "ciera_plan_destroy": (None, [_vp]),
    "ciera_workspace_init": (_i32, [_vp, _vp, _vp]),
    "ciera_compress": (_i32, [_vp, _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _u32, _vp]),
    "ciera_decompress": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _u32, _vp]),
    "ciera_compress_hashed": (_i32, [_vp, _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _u32,
                                     _vp]),
    "ciera_compress_rans": (_i32, [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp,
                                   _u32, _vp]),
    "ciera_compress_noalloc": (_i32, [_vp, _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _u32,
                                      _vp]),
    "ciera_decompress_gather": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _u32, _vp]),
    "ciera_host_session_create": (_i32, [_i32, ctypes.POINTER(_vp)]),
    "ciera_host_session_destroy": (None, [_vp]),
    "ciera_step_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp,
                               _u32, _i32, _vp]),
    "ciera_pipeline_create": (_i32, [_i32, ctypes.POINTER(_vp)]),
    "ciera_pipeline_destroy": (None, [_vp]),
    "ciera_pipeline_step": (_i32, [_vp, _vp, _i32, _vp, _vp]),
    "ciera_status": (_i32, [_vp, _vp]),
    "ciera_should_compress": (_i32, [_i64]),
    "ciera_bsc_select": (_i32, [_vp, _vp, _i32, _i32, _i64, _vp, _vp]),
    "ciera_set_cost_model": (_i32, [ctypes.POINTER(_CostModel)]),
    "ciera_get_cost_model": (_i32, [ctypes.POINTER(_CostModel)]),
    "ciera_set_wait_timeout_ns": (_i32, [ctypes.c_uint64]),
    "ciera_strerror": (ctypes.c_char_p, [_i32]),
}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def checked_build() -> bool:
    """True when this process uses the checked build of the library
    (environment variable CIERA_CHECKED=1, read at the first load)."""
    return os.environ.get("CIERA_CHECKED", "") == "1"


def lib() -> ctypes.CDLL:
    """Load libciera (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build(checked=checked_build())
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def library_path() -> str:
    return _build.library_path(checked_build())


def strerror(status: int) -> str:
    return lib().ciera_strerror(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise CieraError(status, what)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _dev_ptr(t: Optional[torch.Tensor], name: str, dtype=None, numel=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype and not (
            dtype == torch.uint16 and t.dtype == torch.int16):
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr() if t.numel() else None


@dataclass(frozen=True)
class PlanInfo:
    numel: int
    ranks: int
    block: int
    shard_len: int
    blocks_per_shard: int
    tile_blocks: int
    total_tiles: int
    payload_capacity: int
    workspace_bytes: int
    fast_path: bool
    raw_fixup: bool


class Plan:
    """ciera_plan / ciera_plan_info / ciera_plan_destroy."""

    def __init__(self, shape: Union[int, Sequence[int]], block: int, ranks: int):
        if isinstance(shape, int):
            shape = (shape,)
        arr = (ctypes.c_int64 * max(len(shape), 1))(*shape)
        h = ctypes.c_void_p()
        _check(lib().ciera_plan(arr, len(shape), int(block), int(ranks), ctypes.byref(h)),
               "ciera_plan")
        self._h = h
        info = _Info()
        _check(lib().ciera_plan_info(h, ctypes.byref(info)), "ciera_plan_info")
        self.info = PlanInfo(info.numel, info.ranks, info.block, info.shard_len,
                             info.blocks_per_shard, info.tile_blocks, info.total_tiles,
                             info.payload_capacity, info.workspace_bytes,
                             bool(info.fast_path), bool(info.raw_fixup))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.ciera_plan_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    # ---- buffers (plain torch allocations owned by the caller) ----------
    def new_workspace(self, device="cuda") -> torch.Tensor:
        return torch.zeros(max(self.info.workspace_bytes, 1), dtype=torch.uint8, device=device)

    def new_payloads(self, ranks: Optional[int] = None, device="cuda") -> torch.Tensor:
        r = self.info.ranks if ranks is None else ranks
        return torch.zeros((r, self.info.payload_capacity), dtype=torch.uint8, device=device)

    def new_descs(self, ranks: Optional[int] = None, device="cuda") -> torch.Tensor:
        r = self.info.ranks if ranks is None else ranks
        return torch.zeros((r, DESC_BYTES), dtype=torch.uint8, device=device)

    def workspace_init(self, workspace: torch.Tensor, stream=None) -> None:
        _check(lib().ciera_workspace_init(self._h, _dev_ptr(workspace, "workspace"),
                                          _stream_handle(stream)), "ciera_workspace_init")

    # ---- the hot path -------------------------------------------------
    def compress(self, w: torch.Tensor, sender_cache: torch.Tensor, payloads: torch.Tensor,
                 descs: torch.Tensor, workspace: torch.Tensor, *, cold: bool = False,
                 rank_begin: int = 0, rank_count: Optional[int] = None,
                 flags_out: Optional[torch.Tensor] = None, extra_flags: int = 0,
                 stream=None) -> None:
        """ciera_compress: ``w`` (uint16 bits) and ``sender_cache`` (uint8) cover
        ranks [rank_begin, rank_begin + rank_count) contiguously."""
        info = self.info
        rc = info.ranks - rank_begin if rank_count is None else rank_count
        if payloads.dim() != 2 or payloads.shape[0] < rc:
            raise ValueError("payloads must be [rank_count, stride] uint8")
        if descs.numel() < rc * DESC_BYTES:
            raise ValueError("descs too small")
        if flags_out is not None and flags_out.numel() < rc * info.blocks_per_shard:
            raise ValueError("flags_out too small")
        if workspace.numel() < info.workspace_bytes:
            raise ValueError("workspace too small")
        flags = (COLD if cold else 0) | int(extra_flags)
        _check(lib().ciera_compress(
            self._h, int(rank_begin), int(rc),
            _dev_ptr(w, "w", torch.uint16), _dev_ptr(sender_cache, "sender_cache", torch.uint8),
            _dev_ptr(payloads, "payloads", torch.uint8), payloads.stride(0),
            _dev_ptr(descs, "descs", torch.uint8), _dev_ptr(flags_out, "flags_out", torch.uint8),
            _dev_ptr(workspace, "workspace", torch.uint8), flags, _stream_handle(stream)),
            "ciera_compress")

    def compress_hashed(self, w: torch.Tensor, hash_cache: torch.Tensor, payloads: torch.Tensor,
                        descs: torch.Tensor, workspace: torch.Tensor, *, cold: bool = False,
                        rank_begin: int = 0, rank_count: Optional[int] = None,
                        flags_out: Optional[torch.Tensor] = None, extra_flags: int = 0,
                        stream=None) -> None:
        """ciera_compress_hashed: ``hash_cache`` holds 16 bytes per block
        (rank_count x blocks_per_shard x 2 uint64, any 8-byte dtype)."""
        info = self.info
        rc = info.ranks - rank_begin if rank_count is None else rank_count
        if payloads.dim() != 2 or payloads.shape[0] < rc:
            raise ValueError("payloads must be [rank_count, stride] uint8")
        if descs.numel() < rc * DESC_BYTES:
            raise ValueError("descs too small")
        if hash_cache.numel() * hash_cache.element_size() < 16 * rc * info.blocks_per_shard:
            raise ValueError("hash_cache too small")
        if workspace.numel() < info.workspace_bytes:
            raise ValueError("workspace too small")
        _check(lib().ciera_compress_hashed(
            self._h, int(rank_begin), int(rc), _dev_ptr(w, "w", torch.uint16),
            _dev_ptr(hash_cache, "hash_cache"),
            _dev_ptr(payloads, "payloads", torch.uint8), payloads.stride(0),
            _dev_ptr(descs, "descs", torch.uint8), _dev_ptr(flags_out, "flags_out", torch.uint8),
            _dev_ptr(workspace, "workspace", torch.uint8), (COLD if cold else 0) | int(extra_flags),
            _stream_handle(stream)), "ciera_compress_hashed")

    def compress_rans(self, w: torch.Tensor, sender_cache: torch.Tensor,
                      hist_prev: torch.Tensor, hist_out: torch.Tensor, payloads: torch.Tensor,
                      descs: torch.Tensor, workspace: torch.Tensor, *, cold: bool = False,
                      rank_begin: int = 0, rank_count: Optional[int] = None,
                      flags_out: Optional[torch.Tensor] = None, extra_flags: int = 0,
                      stream=None) -> None:
        """ciera_compress_rans: as ``compress``, with the changed exponents
        rANS-coded.  ``hist_prev`` / ``hist_out``: rank_count x 256 int32 (the
        exponent histogram of the previous call / of this call)."""
        info = self.info
        rc = info.ranks - rank_begin if rank_count is None else rank_count
        if payloads.dim() != 2 or payloads.shape[0] < rc:
            raise ValueError("payloads must be [rank_count, stride] uint8")
        if descs.numel() < rc * DESC_BYTES:
            raise ValueError("descs too small")
        if flags_out is not None and flags_out.numel() < rc * info.blocks_per_shard:
            raise ValueError("flags_out too small")
        if workspace.numel() < info.workspace_bytes:
            raise ValueError("workspace too small")
        flags = (COLD if cold else 0) | int(extra_flags)
        _check(lib().ciera_compress_rans(
            self._h, int(rank_begin), int(rc),
            _dev_ptr(w, "w", torch.uint16), _dev_ptr(sender_cache, "sender_cache", torch.uint8),
            _dev_ptr(hist_prev, "hist_prev", torch.int32, 256 * rc),
            _dev_ptr(hist_out, "hist_out", torch.int32, 256 * rc),
            _dev_ptr(payloads, "payloads", torch.uint8), payloads.stride(0),
            _dev_ptr(descs, "descs", torch.uint8), _dev_ptr(flags_out, "flags_out", torch.uint8),
            _dev_ptr(workspace, "workspace", torch.uint8), flags, _stream_handle(stream)),
            "ciera_compress_rans")

    def decompress(self, payloads: torch.Tensor, descs: torch.Tensor, recv_cache: torch.Tensor,
                   out: torch.Tensor, workspace: torch.Tensor, *, rans: bool = False,
                   stream=None) -> None:
        """ciera_decompress: all R payloads -> ``out`` (uint16 bits, N values);
        ``rans`` accepts RANS payloads too (CIERA_DECOMPRESS_RANS)."""
        info = self.info
        if payloads.dim() != 2 or payloads.shape[0] < info.ranks:
            raise ValueError("payloads must be [ranks, stride] uint8")
        if descs.numel() < info.ranks * DESC_BYTES:
            raise ValueError("descs too small")
        if workspace.numel() < info.workspace_bytes:
            raise ValueError("workspace too small")
        _check(lib().ciera_decompress(
            self._h, _dev_ptr(payloads, "payloads", torch.uint8), payloads.stride(0),
            _dev_ptr(descs, "descs", torch.uint8),
            _dev_ptr(recv_cache, "recv_cache", torch.uint8, info.numel),
            _dev_ptr(out, "out", torch.uint16, info.numel),
            _dev_ptr(workspace, "workspace", torch.uint8), DECOMPRESS_RANS if rans else 0,
            _stream_handle(stream)),
            "ciera_decompress")


    def decompress_gather(self, payload_ptrs: torch.Tensor, payload_capacity: int,
                          descs: torch.Tensor, recv_cache: torch.Tensor, out: torch.Tensor,
                          workspace: torch.Tensor, *, rans: bool = False, stream=None) -> None:
        """ciera_decompress_gather: ``payload_ptrs`` is a device int64 tensor of
        R device addresses (each buffer ``payload_capacity`` bytes or more)."""
        info = self.info
        if payload_ptrs.dtype != torch.int64 or payload_ptrs.numel() < info.ranks:
            raise ValueError("payload_ptrs must hold R int64 device addresses")
        if descs.numel() < info.ranks * DESC_BYTES:
            raise ValueError("descs too small")
        if workspace.numel() < info.workspace_bytes:
            raise ValueError("workspace too small")
        _check(lib().ciera_decompress_gather(
            self._h, _dev_ptr(payload_ptrs, "payload_ptrs"), int(payload_capacity),
            _dev_ptr(descs, "descs", torch.uint8),
            _dev_ptr(recv_cache, "recv_cache", torch.uint8, info.numel),
            _dev_ptr(out, "out", torch.uint16, info.numel),
            _dev_ptr(workspace, "workspace", torch.uint8), DECOMPRESS_RANS if rans else 0,
            _stream_handle(stream)),
            "ciera_decompress_gather")


class HostSession:
    """ciera_host_session_* and ciera_step_host: steps whose weights come
    from host memory and whose rebuilt weights go back to it, in one call."""

    def __init__(self, max_chunks: int):
        h = ctypes.c_void_p()
        _check(lib().ciera_host_session_create(int(max_chunks), ctypes.byref(h)),
               "ciera_host_session_create")
        self._h = h
        self.max_chunks = max_chunks

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.ciera_host_session_destroy(h)
            self._h = None

    def step(self, plan: Plan, w_host: torch.Tensor, out_host: torch.Tensor,
             w_dev: torch.Tensor, sender_cache: torch.Tensor, payloads: torch.Tensor,
             descs: torch.Tensor, recv_cache: torch.Tensor, out_dev: torch.Tensor,
             workspace: torch.Tensor, *, cold: bool = False, extra_flags: int = 0,
             chunks: int = 1, stream=None) -> None:
        n = plan.info.numel
        for name, t in (("w_host", w_host), ("out_host", out_host)):
            if t.is_cuda or not t.is_contiguous() or t.numel() < n or t.element_size() != 2:
                raise ValueError(f"{name} must be a contiguous 16-bit host tensor of N values")
        if payloads.dim() != 2 or payloads.shape[0] < plan.info.ranks:
            raise ValueError("payloads must be [ranks, stride] uint8")
        _check(lib().ciera_step_host(
            self._h, plan.handle, w_host.data_ptr() if n else None,
            out_host.data_ptr() if n else None, _dev_ptr(w_dev, "w_dev", torch.uint16, n),
            _dev_ptr(sender_cache, "sender_cache", torch.uint8, n),
            _dev_ptr(payloads, "payloads", torch.uint8), payloads.stride(0),
            _dev_ptr(descs, "descs", torch.uint8),
            _dev_ptr(recv_cache, "recv_cache", torch.uint8, n),
            _dev_ptr(out_dev, "out_dev", torch.uint16, n),
            _dev_ptr(workspace, "workspace", torch.uint8),
            (COLD if cold else 0) | int(extra_flags), int(chunks), _stream_handle(stream)),
            "ciera_step_host")


def status(workspace: torch.Tensor, stream=None) -> int:
    """ciera_status: waits for the stream; returns OK, E_CORRUPT, E_TIMEOUT or
    E_INTERNAL."""
    st = lib().ciera_status(_dev_ptr(workspace, "workspace", torch.uint8), _stream_handle(stream))
    if st == E_CUDA:
        raise CieraError(st, "ciera_status")
    return st


def should_compress(numel: int) -> bool:
    return bool(lib().ciera_should_compress(int(numel)))


def bsc_select(numel, q, world: int, cache_budget_bytes: int):
    """ciera_bsc_select: returns (selected: list[bool], gain: list[float])."""
    import numpy as np
    numel = np.ascontiguousarray(numel, dtype=np.int64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    n = numel.size
    sel = np.zeros(max(n, 1), dtype=np.uint8)
    gain = np.zeros(max(n, 1), dtype=np.float64)
    st = lib().ciera_bsc_select(numel.ctypes.data if n else None, q.ctypes.data if n else None,
                                n, int(world), int(cache_budget_bytes), sel.ctypes.data,
                                gain.ctypes.data)
    if st < 0:
        raise CieraError(st, "ciera_bsc_select")
    return [bool(x) for x in sel[:n]], [float(x) for x in gain[:n]]


def set_cost_model(link_Bps=8e9, q_hat=0.22, t_fixed_s=20e-6, hbm_Bps=8e12, block=4096) -> None:
    m = _CostModel(link_Bps, q_hat, t_fixed_s, hbm_Bps, block)
    _check(lib().ciera_set_cost_model(ctypes.byref(m)), "ciera_set_cost_model")


def get_cost_model() -> dict:
    m = _CostModel()
    _check(lib().ciera_get_cost_model(ctypes.byref(m)), "ciera_get_cost_model")
    return dict(link_Bps=m.link_Bps, q_hat=m.q_hat, t_fixed_s=m.t_fixed_s, hbm_Bps=m.hbm_Bps,
                block=m.block)


def set_wait_timeout_ns(ns: int) -> None:
    _check(lib().ciera_set_wait_timeout_ns(int(ns)), "ciera_set_wait_timeout_ns")


def decode_descs(descs: torch.Tensor) -> list:
    """Host-side view of descriptors (copies to the CPU)."""
    raw = descs.detach().to("cpu").contiguous().view(-1).numpy().tobytes()
    out = []
    import struct
    for i in range(len(raw) // DESC_BYTES):
        mode, nch, body, pay = struct.unpack_from("<IIQQ", raw, i * DESC_BYTES)
        out.append(dict(mode=mode, n_changed_blocks=nch, body_bytes=body, payload_bytes=pay))
    return out


class Pipeline:
    """ciera_pipeline_*: steps over several layers' simulated Allgathers with
    compress(i+1) on a side stream overlapping decompress(i)."""

    def __init__(self, max_layers: int):
        h = ctypes.c_void_p()
        _check(lib().ciera_pipeline_create(int(max_layers), ctypes.byref(h)),
               "ciera_pipeline_create")
        self._h = h
        self.max_layers = max_layers
        self.side = torch.cuda.Stream()

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.ciera_pipeline_destroy(h)
            self._h = None

    def step(self, layers, inputs, stream=None) -> None:
        """layers: SimulatedAllgather objects (any sender); inputs: their
        weights for this step.  Advances each layer's iteration count."""
        arr = (_Layer * len(layers))()
        for i, (ag, w) in enumerate(zip(layers, inputs)):
            hp = ho = hc = None
            if ag.rans:
                hp = _dev_ptr(ag.hist[ag.iteration % 2], "hist_prev", torch.int32)
                ho = _dev_ptr(ag.hist[(ag.iteration + 1) % 2], "hist_out", torch.int32)
            if ag.hashed:
                hc = _dev_ptr(ag.hash_cache, "hash_cache")
            sender = SENDER_RANS if ag.rans else SENDER_HASHED if ag.hashed else SENDER_EXACT
            arr[i] = _Layer(ag.plan.handle.value, _dev_ptr(w, "w", torch.uint16),
                            _dev_ptr(ag.sender_cache, "sender_cache", torch.uint8),
                            _dev_ptr(ag.payloads, "payloads", torch.uint8),
                            ag.payloads.stride(0), _dev_ptr(ag.descs, "descs", torch.uint8),
                            _dev_ptr(ag.recv_cache, "recv_cache", torch.uint8),
                            _dev_ptr(ag.out, "out", torch.uint16),
                            _dev_ptr(ag.workspace, "workspace", torch.uint8),
                            (COLD if ag.iteration == 0 else 0) | ag.extra_flags,
                            sender, hp, ho, hc)
        _check(lib().ciera_pipeline_step(self._h, arr, len(layers), _stream_handle(stream),
                                         self.side.cuda_stream), "ciera_pipeline_step")
        for ag in layers:
            ag.iteration += 1
