"""ctypes binding of ``liba2av.so`` (declared in ``include/a2av.h``).

Argument marshalling only: torch tensors are checked (device, dtype, shape,
contiguity) and their device pointers, together with the current CUDA stream,
are handed to the C ABI.  Every step of the data path runs in the library's
CUDA kernels; there is no CPU fallback, and loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

A2AV_OK = 0
A2AV_ERR_INVALID_ARG = 1
A2AV_ERR_CUDA = 2
A2AV_ERR_NO_MEMORY = 3

DEV_BAD_EXPERT = 1 << 0
DEV_WINDOW_OVERFLOW = 1 << 1
DEV_WAIT_TIMEOUT = 1 << 31

WINDOW_PACKED = 0
WINDOW_FIXED = 1
WINDOW_PADDED = 2
ORDER_SOURCE = 0  # windows in source order, each source segment sorted by expert
ORDER_EXPERT = 1  # windows grouped by local expert, sources in order inside each expert
FLAG_PACK_LSU = 1 << 0
FLAG_SPLITS_TILED = 1 << 1
FLAG_COMBINE_TMA = 1 << 2
FLAG_ROUTE_FUSED = 1 << 3
FLAG_ROUTE_WARP = 1 << 4

# Every function the header declares, for load checks.
EXPORTED = [
    "a2av_config_check", "a2av_recv_arena_rows", "a2av_plan_create", "a2av_plan_destroy",
    "a2av_dispatch", "a2av_splits", "a2av_pack", "a2av_combine", "a2av_expert_scale",
    "a2av_read_device_status", "a2av_device_status_ptr", "a2av_plan_launches",
    "a2av_status_string", "a2av_last_error", "a2av_dispatch_static",
    "a2av_dispatch_padded", "a2av_pack_padded", "a2av_exchange_padded", "a2av_set_active_tokens",
    "a2av_route", "a2av_route_splits", "a2av_set_wait_limit",
]


class Config(ctypes.Structure):
    _fields_ = [
        ("num_ranks", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("tokens_per_rank", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("window_mode", ctypes.c_int32),
        ("window_rows", ctypes.c_int64),
        ("device", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("pack_ctas_per_sm", ctypes.c_int32),
        ("pack_stage_bytes", ctypes.c_int32),
        ("pack_store_lag", ctypes.c_int32),
        ("combine_ctas_per_sm", ctypes.c_int32),
        ("combine_stage_bytes", ctypes.c_int32),
        ("combine_unroll", ctypes.c_int32),
        ("recv_order", ctypes.c_int32),
    ]


class SplitsPtrs(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "send_counts", "send_offsets", "recv_counts", "recv_offsets", "recv_expert_counts",
        "recv_total", "window_base", "recv_expert_offsets")]


class A2avError(RuntimeError):
    pass


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(path: Optional[str] = None):
    """Load liba2av.so (declaring the C signatures).  Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise A2avError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(p)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    cfgp = ctypes.POINTER(Config)
    spp = ctypes.POINTER(SplitsPtrs)
    L.a2av_config_check.argtypes = [cfgp]
    L.a2av_config_check.restype = i32
    L.a2av_recv_arena_rows.argtypes = [cfgp]
    L.a2av_recv_arena_rows.restype = ctypes.c_int64
    L.a2av_plan_create.argtypes = [cfgp, ctypes.POINTER(vp)]
    L.a2av_plan_create.restype = i32
    L.a2av_plan_destroy.argtypes = [vp]
    L.a2av_plan_destroy.restype = i32
    L.a2av_dispatch.argtypes = [vp, vp, vp, spp, vp, vp, vp]
    L.a2av_dispatch.restype = i32
    L.a2av_splits.argtypes = [vp, vp, spp, vp, vp]
    L.a2av_splits.restype = i32
    L.a2av_pack.argtypes = [vp, vp, vp, spp, vp, vp, vp]
    L.a2av_pack.restype = i32
    L.a2av_combine.argtypes = [vp, vp, vp, vp, vp, vp]
    L.a2av_combine.restype = i32
    L.a2av_expert_scale.argtypes = [vp, vp, vp, vp, vp, vp]
    L.a2av_expert_scale.restype = i32
    L.a2av_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, vp]
    L.a2av_read_device_status.restype = i32
    L.a2av_device_status_ptr.argtypes = [vp]
    L.a2av_device_status_ptr.restype = vp
    L.a2av_plan_launches.argtypes = [vp]
    L.a2av_plan_launches.restype = ctypes.c_int64
    L.a2av_status_string.argtypes = [i32]
    L.a2av_status_string.restype = ctypes.c_char_p
    L.a2av_last_error.argtypes = []
    L.a2av_last_error.restype = ctypes.c_char_p
    L.a2av_dispatch_static.argtypes = [cfgp, vp, vp, spp, vp, vp, vp, vp]
    L.a2av_dispatch_static.restype = i32
    L.a2av_dispatch_padded.argtypes = [vp, vp, vp, spp, vp, vp, vp, vp]
    L.a2av_dispatch_padded.restype = i32
    L.a2av_pack_padded.argtypes = [vp, vp, vp, spp, vp, vp, vp]
    L.a2av_pack_padded.restype = i32
    L.a2av_exchange_padded.argtypes = [vp, vp, vp, vp]
    L.a2av_exchange_padded.restype = i32
    L.a2av_set_active_tokens.argtypes = [vp, vp]
    L.a2av_set_active_tokens.restype = i32
    L.a2av_route.argtypes = [vp, vp, vp, vp, vp]
    L.a2av_route.restype = i32
    L.a2av_route_splits.argtypes = [vp, vp, vp, vp, spp, vp, vp]
    L.a2av_route_splits.restype = i32
    L.a2av_set_wait_limit.argtypes = [vp, ctypes.c_int64]
    L.a2av_set_wait_limit.restype = i32
    if path is None:
        _lib = L
    return L


def _check(L, rc: int, what: str):
    if rc != A2AV_OK:
        msg = L.a2av_status_string(rc).decode()
        detail = L.a2av_last_error().decode()
        raise A2avError(f"{what}: {msg}" + (f" ({detail})" if detail else ""))


def make_config(R, E, T, H, k, window_mode="packed", window_rows=0, device=0, flags=0,
                pack_ctas_per_sm=0, pack_stage_bytes=0, pack_store_lag=0, combine_ctas_per_sm=0,
                combine_stage_bytes=0, combine_unroll=0, recv_order="source") -> Config:
    mode = {"packed": WINDOW_PACKED, "fixed": WINDOW_FIXED, "padded": WINDOW_PADDED}.get(window_mode, window_mode)
    order = {"source": ORDER_SOURCE, "expert": ORDER_EXPERT}.get(recv_order, recv_order)
    return Config(int(R), int(E), int(T), int(H), int(k), int(mode), int(window_rows), int(device),
                  int(flags), int(pack_ctas_per_sm), int(pack_stage_bytes), int(pack_store_lag),
                  int(combine_ctas_per_sm), int(combine_stage_bytes), int(combine_unroll), int(order))


class Splits:
    """Device-resident split counts/offsets of one dispatch (int32 tensors).

    ``recv_expert_offsets`` is allocated and filled only when
    ``expert_offsets`` is true (the expert-grouped receive order needs it;
    in source order it is an optional extra output of the splits kernel)."""

    NAMES = ("send_counts", "send_offsets", "recv_counts", "recv_offsets", "recv_expert_counts",
             "recv_total", "window_base", "recv_expert_offsets")

    def __init__(self, R: int, E: int, device, expert_offsets: bool = True):
        import torch

        epr = E // R
        shapes = {"send_counts": (R, E), "send_offsets": (R, E), "recv_counts": (R, R),
                  "recv_offsets": (R, R), "recv_expert_counts": (R, R, epr), "recv_total": (R,),
                  "window_base": (R,), "recv_expert_offsets": (R, R, epr)}
        self.names = self.NAMES if expert_offsets else self.NAMES[:-1]
        for n in self.NAMES:
            setattr(self, n, torch.zeros(shapes[n], dtype=torch.int32, device=device) if n in self.names else None)
        self._ptrs = SplitsPtrs(*[getattr(self, n).data_ptr() if n in self.names else None for n in self.NAMES])

    @property
    def ptrs(self) -> SplitsPtrs:
        return self._ptrs

    def to_numpy(self) -> dict:
        return {n: getattr(self, n).cpu().numpy() for n in self.names}


def _stream_ptr(stream, device):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


class Plan:
    """A configured data plane: R emulated ranks, E experts, T tokens per rank,
    hidden H, top-k.  Owns only the library's small workspace."""

    def __init__(self, R, E, T, H, k, window_mode="packed", window_rows=0, device=None, flags=0,
                 pack_ctas_per_sm=0, pack_stage_bytes=0, pack_store_lag=0, combine_ctas_per_sm=0,
                 combine_stage_bytes=0, combine_unroll=0, recv_order="source"):
        import torch

        self.lib = load_library()
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        if dev.type != "cuda":
            raise A2avError("a2av plans live on a CUDA device")
        self.device = dev
        self.R, self.E, self.T, self.H, self.k = int(R), int(E), int(T), int(H), int(k)
        self.window_mode = window_mode
        self.window_rows = int(window_rows)
        self.recv_order = recv_order
        self.cfg = make_config(R, E, T, H, k, window_mode, window_rows, dev.index, flags,
                               pack_ctas_per_sm, pack_stage_bytes, pack_store_lag, combine_ctas_per_sm,
                               combine_stage_bytes, combine_unroll, recv_order)
        handle = ctypes.c_void_p()
        _check(self.lib, self.lib.a2av_plan_create(ctypes.byref(self.cfg), ctypes.byref(handle)), "a2av_plan_create")
        self.handle = handle
        self.arena_rows = int(self.lib.a2av_recv_arena_rows(ctypes.byref(self.cfg)))

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            _check(self.lib, self.lib.a2av_plan_destroy(self.handle), "a2av_plan_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- tensors ------------------------------------------------------------
    def new_splits(self, expert_offsets=None) -> Splits:
        """Split arrays for this plan; ``expert_offsets`` None = only when the
        receive order needs them (the expert-grouped order)."""
        if expert_offsets is None:
            expert_offsets = self.recv_order in ("expert", ORDER_EXPERT)
        return Splits(self.R, self.E, self.device, expert_offsets=bool(expert_offsets))

    def new_buffers(self):
        """(recv [arena_rows][H] bf16, slot_map [R][T][k] int32, out [R][T][H] bf16), uninitialised."""
        import torch

        recv = torch.empty((self.arena_rows, self.H), dtype=torch.bfloat16, device=self.device)
        slot_map = torch.empty((self.R, self.T, self.k), dtype=torch.int32, device=self.device)
        out = torch.empty((self.R, self.T, self.H), dtype=torch.bfloat16, device=self.device)
        return recv, slot_map, out

    def _t(self, t, dtype, shape, name):
        import torch

        if not isinstance(t, torch.Tensor):
            raise A2avError(f"{name} must be a torch tensor")
        if t.device != self.device:
            raise A2avError(f"{name} is on {t.device}, the plan is on {self.device}")
        if t.dtype != dtype:
            raise A2avError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise A2avError(f"{name} must be contiguous")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise A2avError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        return ctypes.c_void_p(t.data_ptr())

    def _rows(self, t, name):
        import torch

        return self._t(t, torch.bfloat16, (self.arena_rows, self.H), name)

    # ---- calls ----------------------------------------------------------------
    def dispatch(self, x, topk_idx, splits: Splits, recv, slot_map, stream=None):
        import torch

        args = (self.handle, self._t(x, torch.bfloat16, (self.R, self.T, self.H), "x"),
                self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"), ctypes.byref(splits.ptrs),
                self._rows(recv, "recv"), self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"),
                _stream_ptr(stream, self.device))
        _check(self.lib, self.lib.a2av_dispatch(*args), "a2av_dispatch")

    def splits(self, topk_idx, splits: Splits, slot_map, stream=None):
        import torch

        _check(self.lib, self.lib.a2av_splits(
            self.handle, self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"),
            ctypes.byref(splits.ptrs), self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"),
            _stream_ptr(stream, self.device)), "a2av_splits")

    def pack(self, x, topk_idx, splits: Splits, recv, slot_map, stream=None):
        import torch

        _check(self.lib, self.lib.a2av_pack(
            self.handle, self._t(x, torch.bfloat16, (self.R, self.T, self.H), "x"),
            self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"), ctypes.byref(splits.ptrs),
            self._rows(recv, "recv"), self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"),
            _stream_ptr(stream, self.device)), "a2av_pack")

    def route(self, logits, topk_idx, gate_w, stream=None):
        """Top-k experts and softmax gates of fp32 logits [R][T][E] (a2av_route)."""
        import torch

        _check(self.lib, self.lib.a2av_route(
            self.handle, self._t(logits, torch.float32, (self.R, self.T, self.E), "logits"),
            self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"),
            self._t(gate_w, torch.float32, (self.R, self.T, self.k), "gate_w"),
            _stream_ptr(stream, self.device)), "a2av_route")

    def route_splits(self, logits, topk_idx, gate_w, splits: Splits, slot_map, stream=None):
        """Router + splits in one kernel where possible (a2av_route_splits);
        follow with ``pack`` as after ``splits``."""
        import torch

        _check(self.lib, self.lib.a2av_route_splits(
            self.handle, self._t(logits, torch.float32, (self.R, self.T, self.E), "logits"),
            self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"),
            self._t(gate_w, torch.float32, (self.R, self.T, self.k), "gate_w"), ctypes.byref(splits.ptrs),
            self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"),
            _stream_ptr(stream, self.device)), "a2av_route_splits")

    def set_active_tokens(self, num_tokens=None):
        """Read per-rank token counts from the int32 device tensor `num_tokens`
        [R] in every later call (None: every token takes part)."""
        import torch

        if num_tokens is None:
            self._num_tokens = None
            ptr = None
        else:
            self._t(num_tokens, torch.int32, (self.R,), "num_tokens")
            self._num_tokens = num_tokens  # keep it alive while the plan may read it
            ptr = ctypes.c_void_p(num_tokens.data_ptr())
        _check(self.lib, self.lib.a2av_set_active_tokens(self.handle, ptr), "a2av_set_active_tokens")

    def new_send_buffer(self):
        """Padded plans: the worst-case send buffer, bf16 [R*R*T*k][H] (uninitialised)."""
        import torch

        return torch.empty((self.arena_rows, self.H), dtype=torch.bfloat16, device=self.device)

    def dispatch_padded(self, x, topk_idx, splits: Splits, sendbuf, recv, slot_map, stream=None):
        import torch

        _check(self.lib, self.lib.a2av_dispatch_padded(
            self.handle, self._t(x, torch.bfloat16, (self.R, self.T, self.H), "x"),
            self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"), ctypes.byref(splits.ptrs),
            self._rows(sendbuf, "sendbuf"), self._rows(recv, "recv"),
            self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"),
            _stream_ptr(stream, self.device)), "a2av_dispatch_padded")

    def pack_padded(self, x, topk_idx, splits: Splits, sendbuf, slot_map, stream=None):
        import torch

        _check(self.lib, self.lib.a2av_pack_padded(
            self.handle, self._t(x, torch.bfloat16, (self.R, self.T, self.H), "x"),
            self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"), ctypes.byref(splits.ptrs),
            self._rows(sendbuf, "sendbuf"), self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"),
            _stream_ptr(stream, self.device)), "a2av_pack_padded")

    def exchange_padded(self, sendbuf, recv, stream=None):
        _check(self.lib, self.lib.a2av_exchange_padded(
            self.handle, self._rows(sendbuf, "sendbuf"), self._rows(recv, "recv"),
            _stream_ptr(stream, self.device)), "a2av_exchange_padded")

    def combine(self, y, gate_w, slot_map, out, stream=None):
        import torch

        _check(self.lib, self.lib.a2av_combine(
            self.handle, self._rows(y, "y"), self._t(gate_w, torch.float32, (self.R, self.T, self.k), "gate_w"),
            self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"),
            self._t(out, torch.bfloat16, (self.R, self.T, self.H), "out"),
            _stream_ptr(stream, self.device)), "a2av_combine")

    def expert_scale(self, recv, topk_idx, slot_map, y, stream=None):
        import torch

        _check(self.lib, self.lib.a2av_expert_scale(
            self.handle, self._rows(recv, "recv"), self._t(topk_idx, torch.int32, (self.R, self.T, self.k), "topk_idx"),
            self._t(slot_map, torch.int32, (self.R, self.T, self.k), "slot_map"), self._rows(y, "y"),
            _stream_ptr(stream, self.device)), "a2av_expert_scale")

    def set_wait_limit(self, polls: int = -1):
        """Main-loop poll limit of the TMA kernels' bounded waits for later
        calls (0: give up at once; negative: the default)."""
        _check(self.lib, self.lib.a2av_set_wait_limit(self.handle, int(polls)), "a2av_set_wait_limit")

    def read_status(self, clear: bool = False, stream=None) -> int:
        bits = ctypes.c_uint32(0)
        _check(self.lib, self.lib.a2av_read_device_status(self.handle, ctypes.byref(bits), int(clear),
                                                          _stream_ptr(stream, self.device)), "a2av_read_device_status")
        return int(bits.value)

    @property
    def launches(self) -> int:
        return int(self.lib.a2av_plan_launches(self.handle))


def _static_shape_checks(L, cfg, x, topk_idx, splits, recv, slot_map, dev_status, R, E, T, H, k):
    """Shapes a2av_dispatch_static's kernels rely on (the C ABI only sees
    pointers): x (R,T,H), topk_idx and slot_map (R,T,k), recv with at least
    the arena's rows of H values, a dev_status element, and split arrays
    made for R ranks and E experts.  Raises A2avError before anything is
    enqueued."""
    rc = L.a2av_config_check(ctypes.byref(cfg))
    if rc != A2AV_OK:
        raise A2avError(f"a2av_dispatch_static: invalid configuration R={R} E={E} T={T} H={H} k={k}")
    want = {"x": (x, (R, T, H)), "topk_idx": (topk_idx, (R, T, k)), "slot_map": (slot_map, (R, T, k))}
    for name, (t, shape) in want.items():
        if tuple(t.shape) != shape:
            raise A2avError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    rows = int(L.a2av_recv_arena_rows(ctypes.byref(cfg)))
    if recv.dim() != 2 or recv.shape[1] != H or recv.shape[0] < rows:
        raise A2avError(f"recv has shape {tuple(recv.shape)}, expected at least ({rows}, {H})")
    if dev_status.numel() < 1:
        raise A2avError("dev_status needs one element")
    epr = E // R
    shapes = {"send_counts": (R, E), "send_offsets": (R, E), "recv_counts": (R, R), "recv_offsets": (R, R),
              "recv_expert_counts": (R, R, epr), "recv_total": (R,), "window_base": (R,),
              "recv_expert_offsets": (R, R, epr)}
    for name in splits.names:
        t = getattr(splits, name)
        if tuple(t.shape) != shapes[name]:
            raise A2avError(f"splits.{name} has shape {tuple(t.shape)}, expected {shapes[name]} (R={R}, E={E})")
    if cfg.recv_order == ORDER_EXPERT and "recv_expert_offsets" not in splits.names:
        raise A2avError("the expert-grouped receive order needs splits.recv_expert_offsets")


def dispatch_static(x, topk_idx, splits: Splits, recv, slot_map, dev_status, R, E, T, H, k,
                    window_mode="packed", window_rows=0, flags=0, stream=None, recv_order="source"):
    """Dispatch without a plan and without any allocation (a2av_dispatch_static).

    For callers that cannot allocate device memory where they dispatch (a
    framework whose caching allocator owns all device memory, a spent
    device-memory budget, a loop that cannot take cudaMalloc's implicit
    synchronisation): the kernels' scratch lives in a static device array of
    the library (1 MiB per GPU), so shapes are bounded; ``dev_status`` is a
    caller-owned int32 device tensor of one element that receives the
    A2AV_DEV_* bits.  The first call on a device (and the first with each
    configuration) does a one-time set-up, so make it before any stream
    capture; calls that overlap on the GPU share the array and race.  Every
    shape is checked here before anything is enqueued.
    """
    import torch

    L = load_library()
    dev = x.device
    cfg = make_config(R, E, T, H, k, window_mode, window_rows, dev.index if dev.index is not None else 0, flags,
                      recv_order=recv_order)
    _static_shape_checks(L, cfg, x, topk_idx, splits, recv, slot_map, dev_status, R, E, T, H, k)
    tensors = [(x, torch.bfloat16, "x"), (topk_idx, torch.int32, "topk_idx"), (recv, torch.bfloat16, "recv"),
               (slot_map, torch.int32, "slot_map"), (dev_status, torch.int32, "dev_status")]
    tensors += [(getattr(splits, n), torch.int32, f"splits.{n}") for n in splits.names]
    for t, dt, name in tensors:
        if t.device != dev or dev.type != "cuda" or t.dtype != dt or not t.is_contiguous():
            raise A2avError(f"{name}: expected a contiguous {dt} tensor on the CUDA device of x ({dev})")
    rc = L.a2av_dispatch_static(ctypes.byref(cfg), ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(topk_idx.data_ptr()),
                                ctypes.byref(splits.ptrs), ctypes.c_void_p(recv.data_ptr()),
                                ctypes.c_void_p(slot_map.data_ptr()), ctypes.c_void_p(dev_status.data_ptr()),
                                _stream_ptr(stream, dev))
    _check(L, rc, "a2av_dispatch_static")
