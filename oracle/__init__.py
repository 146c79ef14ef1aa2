"""CPU oracle of the MoE AllToAllvDynamic data plane (dispatch + top-k combine).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package.  The product
path (``combine_device_resident_gb300``) never imports it and shares no code
with it: the arithmetic lives in ``a2av_oracle.c`` (plain C, one thread, built
with ``-O2 -ffp-contract=off`` so every fp32 product and sum is rounded on its
own), and this module only marshals numpy arrays into it.

What each function computes, and the passages and readings it follows, is
written in ``a2av_oracle.c``.  Pinning status (what checks each function against
something other than itself, in ``tests/test_oracle_pins.py``):

* ``splits``     -- invariants (sum_e send = T*k, recv = transpose of per-rank
                    send counts summed over each rank's experts, exclusive-scan
                    offsets, window bases) and exhaustive brute force on tiny
                    routings;
* ``slot_map`` / ``dispatch`` -- brute force (window d = a stable sort of all
                    assignments sent to d by key (source, expert, token, slot),
                    or (expert, source, token, slot) in the expert-grouped
                    receive order), bijection onto [0, R*T*k), recv[slot] == x
                    bit for bit; the expert-order dispatch (regroup of the
                    source-order windows) against the direct offset formula
                    of ``slot_map``;
* ``recv_expert_offsets`` -- every window tiled by its (source, expert) blocks
                    in the order of the layout, against the brute-force rows;
* ``combine``    -- closed forms independent of the layout (unit weights and
                    identity experts give bf16(k*x), k in {1, 2, 4, 8}; gate sum
                    times x), numpy float32 with separate roundings, and the fp64
                    sum within 1 bf16 ulp;
* ``expert_scale`` -- closed form bf16(x * (1 + e/E)) computed by torch.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "a2av_oracle.c")
_LIB = os.path.join(_HERE, "liba2av_oracle.so")

BAD_EXPERT = 1
WINDOW_OVERFLOW = 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``liba2av_oracle.so`` next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def bind(L):
    """Declare the C signatures on a loaded oracle library and return it."""
    i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
    u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
    f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
    f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
    i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
    ci, ci64 = ctypes.c_int, ctypes.c_int64
    L.oracle_splits.restype = ctypes.c_uint32
    vp = ctypes.c_void_p  # optional int32 array (NULL = every token takes part)
    L.oracle_splits.argtypes = [ci, ci, ci, ci, ci, ci64, vp, i32p] + [i32p] * 7
    L.oracle_slot_map.restype = ctypes.c_uint32
    L.oracle_slot_map.argtypes = [ci, ci, ci, ci, ci, ci64, vp, i32p, i32p, i32p, i32p, i32p, i32p]
    L.oracle_recv_expert_offsets.restype = None
    L.oracle_recv_expert_offsets.argtypes = [ci, ci, ci, i32p, i32p, i32p]
    L.oracle_dispatch.restype = ctypes.c_uint32
    L.oracle_dispatch.argtypes = [ci, ci, ci, ci, ci, ci, ci64, vp, u16p, i32p, i32p, i32p, i32p, i32p,
                                  u16p, i32p]
    L.oracle_dispatch_ranks.restype = ctypes.c_uint32
    L.oracle_dispatch_ranks.argtypes = L.oracle_dispatch.argtypes + [ci, ci]
    L.oracle_expert_scale.restype = None
    L.oracle_expert_scale.argtypes = [ci, ci, ci64, u16p, i32p, i32p, u16p]
    L.oracle_combine.restype = None
    L.oracle_combine.argtypes = [ci, ci, u16p, f32p, i32p, i64p, ci64, u16p]
    L.oracle_combine_f64.restype = None
    L.oracle_combine_f64.argtypes = [ci, ci, u16p, f32p, i32p, i64p, ci64, f64p]
    f32p_ = f32p
    L.oracle_route.restype = None
    L.oracle_route.argtypes = [ci, ci, ci, ci, vp, f32p_, i32p, f64p]
    L.oracle_bf16_to_f32.restype = ctypes.c_float
    L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    return L


def compile_source(src: str, out: str) -> str:
    """Compile C source text into a shared library at ``out`` with the oracle's flags."""
    cfile = out + ".c"
    with open(cfile, "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-w", "-o", out, cfile, "-lm"])
    return out


def lib():
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build()))
    return _lib


def _counts_ptr(num_tokens):
    """(ctypes pointer or None, keep-alive array) for an optional per-rank token count."""
    if num_tokens is None:
        return None, None
    arr = np.ascontiguousarray(num_tokens, dtype=np.int32)
    return arr.ctypes.data_as(ctypes.c_void_p), arr


ORDER_EXPERT = 0x100  # receive order flag on the C side's window_mode


def _layout(window_mode) -> int:
    if window_mode in (0, "packed"):
        return 0
    if window_mode in (1, "fixed"):
        return 1
    if window_mode in (2, "padded"):
        return 2
    raise ValueError(window_mode)


def _mode(window_mode, recv_order="source") -> int:
    """Layout | receive order, as the C functions take it."""
    m = _layout(window_mode)
    if recv_order in (1, "expert"):
        if m == 2:
            raise ValueError("the expert-grouped receive order is not defined for the padded layout")
        return m | ORDER_EXPERT
    if recv_order not in (0, "source"):
        raise ValueError(recv_order)
    return m


def splits(R: int, E: int, idx: np.ndarray, window_mode="packed", window_rows: int = 0, num_tokens=None,
           recv_order="source") -> dict:
    """Counts and offsets of one dispatch.  idx int32 [R][T][k]; num_tokens
    int32 [R] (optional): only tokens t < num_tokens[s] take part; recv_order
    "source" (AllToAllv convention) or "expert" (expert-grouped windows)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    _, T, k = idx.shape
    if E % R:
        raise ValueError("E must be a multiple of R")
    epr = E // R
    out = {
        "send_counts": np.zeros((R, E), np.int32),
        "send_offsets": np.zeros((R, E), np.int32),
        "recv_counts": np.zeros((R, R), np.int32),
        "recv_offsets": np.zeros((R, R), np.int32),
        "recv_expert_counts": np.zeros((R, R, epr), np.int32),
        "recv_total": np.zeros((R,), np.int32),
        "window_base": np.zeros((R,), np.int32),
    }
    nt, _keep = _counts_ptr(num_tokens)
    st = lib().oracle_splits(R, E, T, k, _mode(window_mode), int(window_rows), nt, idx,
                             out["send_counts"], out["send_offsets"], out["recv_counts"],
                             out["recv_offsets"], out["recv_expert_counts"], out["recv_total"],
                             out["window_base"])
    out["recv_expert_offsets"] = np.zeros((R, R, epr), np.int32)
    lib().oracle_recv_expert_offsets(R, E, _mode(window_mode, recv_order), out["recv_offsets"],
                                     out["recv_expert_counts"], out["recv_expert_offsets"])
    out["status"] = int(st)
    return out


def slot_map(R: int, E: int, idx: np.ndarray, sp: dict, window_mode="packed", window_rows: int = 0,
             num_tokens=None, recv_order="source"):
    """(slot_map int32 [R][T][k], status) without moving any payload."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    _, T, k = idx.shape
    sm = np.empty((R, T, k), np.int32)
    nt, _keep = _counts_ptr(num_tokens)
    st = lib().oracle_slot_map(R, E, T, k, _mode(window_mode, recv_order), int(window_rows), nt, idx,
                               sp["send_offsets"], sp["recv_offsets"], sp["recv_expert_offsets"],
                               sp["window_base"], sm)
    return sm, int(st)


def arena_rows(R: int, T: int, k: int, window_mode="packed", window_rows: int = 0) -> int:
    m = _layout(window_mode)
    return R * T * k if m == 0 else (R * int(window_rows) if m == 1 else R * R * T * k)


def dispatch(R: int, E: int, x: np.ndarray, idx: np.ndarray, sp: dict, window_mode="packed",
             window_rows: int = 0, recv: Optional[np.ndarray] = None, num_tokens=None, recv_order="source",
             ranks=None, slot_map_out: Optional[np.ndarray] = None):
    """(recv uint16 [rows][H], slot_map, status).  x uint16 bf16 bits [R][T][H].
    Rows no assignment reaches keep their prior contents (zeros if recv is None).

    ``ranks=(s0, s1)``: only source ranks s0 <= s < s1 (source order only),
    writing their rows into ``recv`` and their slots into ``slot_map_out``
    (both shared by callers that run disjoint ranges, e.g. one per thread)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    _, T, H = x.shape
    k = idx.shape[2]
    rows = arena_rows(R, T, k, window_mode, window_rows)
    if recv is None:
        recv = np.zeros((rows, H), np.uint16)
    sm = np.empty((R, T, k), np.int32) if slot_map_out is None else slot_map_out
    nt, _keep = _counts_ptr(num_tokens)
    args = (R, E, T, H, k, _mode(window_mode, recv_order), int(window_rows), nt, x, idx,
            sp["send_counts"], sp["send_offsets"], sp["recv_offsets"], sp["window_base"], recv, sm)
    if ranks is None:
        st = lib().oracle_dispatch(*args)
    else:
        if recv_order not in (0, "source"):
            raise ValueError("a source-rank range is defined for the source order only")
        s0, s1 = (int(v) for v in ranks)
        if not 0 <= s0 <= s1 <= R:
            raise ValueError(f"rank range {ranks} outside [0, {R}]")
        st = lib().oracle_dispatch_ranks(*args, s0, s1)
    return recv, sm, int(st)


def expert_scale(E: int, recv: np.ndarray, idx: np.ndarray, sm: np.ndarray, y: Optional[np.ndarray] = None):
    """y[row] = bf16(recv[row] * (1 + e/E)) for every dispatched assignment."""
    recv = np.ascontiguousarray(recv, dtype=np.uint16)
    if y is None:
        y = recv.copy()
    H = recv.shape[1]
    lib().oracle_expert_scale(E, H, int(idx.size), recv, np.ascontiguousarray(idx, np.int32),
                              np.ascontiguousarray(sm, np.int32), y)
    return y


def combine(y: np.ndarray, gate: np.ndarray, sm: np.ndarray, tokens: Optional[np.ndarray] = None):
    """out uint16 [n_tokens][H] for flat token ids ``tokens`` (default: all)."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    sm = np.ascontiguousarray(sm, dtype=np.int32)
    k = sm.shape[-1]
    ntok_all = sm.size // k
    if tokens is None:
        tokens = np.arange(ntok_all, dtype=np.int64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    H = y.shape[1]
    out = np.empty((len(tokens), H), np.uint16)
    lib().oracle_combine(H, k, y, gate, sm, tokens, len(tokens), out)
    return out


def combine_f64(y: np.ndarray, gate: np.ndarray, sm: np.ndarray, tokens: Optional[np.ndarray] = None):
    y = np.ascontiguousarray(y, dtype=np.uint16)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    sm = np.ascontiguousarray(sm, dtype=np.int32)
    k = sm.shape[-1]
    if tokens is None:
        tokens = np.arange(sm.size // k, dtype=np.int64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    out = np.empty((len(tokens), y.shape[1]), np.float64)
    lib().oracle_combine_f64(y.shape[1], k, y, gate, sm, tokens, len(tokens), out)
    return out


def route(logits: np.ndarray, k: int, num_tokens=None):
    """Router: (topk_idx int32 [R][T][k], gate float64 [R][T][k]) from fp32
    logits [R][T][E]; entries of tokens that take no part stay -1 / 0."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    R, T, E = logits.shape
    idx = np.full((R, T, k), -1, np.int32)
    gate = np.zeros((R, T, k), np.float64)
    nt, _keep = _counts_ptr(num_tokens)
    lib().oracle_route(R, T, E, k, nt, logits, idx, gate)
    return idx, gate


def bf16_to_f32(bits: int) -> float:
    return float(lib().oracle_bf16_to_f32(int(bits)))


def f32_to_bf16(v: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(v)))


def run_all(R, E, x, idx, gate, window_mode="packed", window_rows=0, expert="identity", num_tokens=None,
            recv_order="source"):
    """The whole path on the CPU: splits, dispatch, expert stand-in, combine.
    With num_tokens, out rows of tokens that do not take part are zero here
    (the combine produces nothing for them)."""
    sp = splits(R, E, idx, window_mode, window_rows, num_tokens, recv_order)
    recv, sm, st = dispatch(R, E, x, idx, sp, window_mode, window_rows, num_tokens=num_tokens,
                            recv_order=recv_order)
    y = expert_scale(E, recv, idx, sm) if expert == "scale" else recv
    T = idx.shape[1]
    if num_tokens is None:
        out = combine(y, gate, sm).reshape(x.shape)
    else:
        act = [s * T + t for s in range(R) for t in range(min(max(int(num_tokens[s]), 0), T))]
        out = np.zeros((R * T, x.shape[2]), np.uint16)
        if act:
            out[act] = combine(y, gate, sm, np.array(act, np.int64))
        out = out.reshape(x.shape)
    return {"splits": sp, "recv": recv, "slot_map": sm, "y": y, "out": out,
            "status": sp["status"] | st}
