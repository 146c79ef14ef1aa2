"""Seeded synthetic inputs for the device-resident MoE dispatch/combine data plane.

This module only draws inputs: token rows ``x``, routing indices ``topk_idx`` and
gate weights ``gate_w``.  It holds none of the data plane's arithmetic (no
counting, scanning, placement or combining), so that the CPU oracle and the CUDA
path can both be fed from it without sharing any of the method.

The five named workloads are the MoE-inference shapes the AllToAllvDynamic
data plane is measured on (NCCLX, "Collective Communication for 100k+ GPUs",
Section 6.1: tokens routed to their top-k experts, sorted by expert and sent to
the rank holding each expert, then combined).  The pages give no dataset, so
every input is synthetic:

* ``x``       bf16 [R][T][H], values N(0, 1) drawn in float32 by torch's seeded
              generator on the device that will hold x (Philox on a GPU, the CPU
              generator on the host), then rounded to bf16 (round to nearest
              even).  The oracle is always fed a host copy of the very tensor
              the GPU path reads, so both sides see identical bits;
* ``topk_idx`` int32 [R][T][k], global expert ids;
* ``gate_w``  float32 [R][T][k].

Randomness: x comes from ``torch.Generator(device).manual_seed(seed)``; routing
and gate logits come from two independent numpy streams
``numpy.random.SeedSequence(seed).spawn(2)``, so the routing of a workload can be
drawn without drawing its (large) x.  Routing kinds:

* ``uniform``         top-1 uniform over the E experts;
* ``zipf``            top-1, P(Zipf rank i) proportional to i**-s, i = 1..E,
                      mapped to expert ids by a seeded permutation;
* ``zipf_distinct``   top-k distinct experts drawn one after another without
                      replacement (renormalising after each draw) from the same
                      Zipf law over a seeded permutation;
* ``hot0_distinct``   as ``zipf_distinct`` but expert 0 takes probability p0 on
                      the first draw, the remaining 1 - p0 is Zipf(s) over the
                      other allowed experts, and ``empty_ranks`` seeded ranks
                      other than rank 0 hold experts of probability zero.

Sampling without replacement is realised with the Gumbel-top-k construction:
the k largest of log(w_e) + Gumbel noise, in decreasing order, have the same
joint law as k successive weighted draws without replacement, so slot j is the
j-th draw.

Gate kinds: ``ones`` (every weight 1.0) or ``softmax`` (k logits per token drawn
N(0, 1) in float32, softmax over those k in float32 with the maximum
subtracted).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload of the data plane."""

    name: str
    R: int                      # emulated ranks (one window each)
    E: int                      # experts, E/R contiguous experts per rank
    T: int                      # tokens per rank
    H: int                      # hidden size (bf16 values per row)
    k: int                      # experts per token
    routing: str = "uniform"
    zipf_s: float = 0.0
    p0: float = 0.0
    empty_ranks: int = 0
    gate: str = "ones"
    expert: str = "identity"    # "identity" or "scale" (y = x * (1 + e/E))
    window_mode: str = "packed"  # "packed" arena or "fixed" per-rank windows
    window_rows: int = 0         # fixed mode: rows per destination window
    recv_order: str = "source"   # "source" (AllToAllv convention) or "expert" (grouped by local expert)

    @property
    def assignments(self) -> int:
        return self.R * self.T * self.k

    def algorithmic_bytes(self) -> int:
        """Payload bytes one dispatch+combine moves: read x, write k copies,
        read k copies, write out (4*R*T*H*(k+1)), plus the routing metadata
        (idx read twice, slot_map written and read, gate read: 16 B per
        assignment)."""
        rows = self.R * self.T
        return 4 * rows * self.H * (self.k + 1) + 16 * self.assignments

    def scaled(self, T: Optional[int] = None, H: Optional[int] = None, name: Optional[str] = None) -> "Workload":
        """Same routing law and rank/expert layout, smaller token count or row."""
        T2 = self.T if T is None else T
        rows = self.window_rows
        if self.window_mode == "fixed":
            rows = self.R * T2 * self.k
        return dataclasses.replace(self, T=T2, H=self.H if H is None else H,
                                   window_rows=rows, name=name or f"{self.name}-T{T2}-H{H or self.H}")


# The five workloads, with the sizes and distributions of the MoE decode shapes.
WORKLOADS = {
    1: Workload("r2-e4-t128-h256-top1-uniform", R=2, E=4, T=128, H=256, k=1),
    2: Workload("r8-e16-t1024-h5120-top1-uniform", R=8, E=16, T=1024, H=5120, k=1),
    # "buffers sized to max capacity T*k per rank": every source may send up to
    # T*k rows to one destination, so each fixed window holds R*T*k rows.
    3: Workload("r8-e128-t256-h5120-top1-zipf1.2-fixedwin", R=8, E=128, T=256, H=5120, k=1,
                routing="zipf", zipf_s=1.2, window_mode="fixed", window_rows=8 * 256 * 1),
    4: Workload("r16-e128-t4096-h5120-top2-zipf1.0-softmax-scale", R=16, E=128, T=4096, H=5120, k=2,
                routing="zipf_distinct", zipf_s=1.0, gate="softmax", expert="scale"),
    5: Workload("r32-e256-t2048-h7168-top8-hot0-zipf1.1-softmax", R=32, E=256, T=2048, H=7168, k=8,
                routing="hot0_distinct", p0=0.3, zipf_s=1.1, empty_ranks=4, gate="softmax"),
}


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 (round to nearest even) bit patterns as uint16, via torch."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _zipf_weights(n: int, s: float) -> np.ndarray:
    ranks = np.arange(1, n + 1, dtype=np.float64)
    w = ranks ** (-s)
    return w / w.sum()


def _gumbel_topk(rng: np.random.Generator, logw: np.ndarray, shape: tuple, k: int) -> np.ndarray:
    """k successive draws without replacement from weights exp(logw), per row."""
    E = logw.shape[0]
    out = np.empty(shape + (k,), dtype=np.int32)
    flat = out.reshape(-1, k)
    n = flat.shape[0]
    step = max(1, (1 << 22) // E)
    for lo in range(0, n, step):
        hi = min(n, lo + step)
        g = rng.gumbel(size=(hi - lo, E))
        key = logw[None, :] + g
        part = np.argpartition(-key, k - 1, axis=1)[:, :k]
        pk = np.take_along_axis(key, part, axis=1)
        order = np.argsort(-pk, axis=1, kind="stable")
        flat[lo:hi] = np.take_along_axis(part, order, axis=1)
    return out


def routing_weights(w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Per-expert draw weights (float64, sum 1) for the Zipf-type routings."""
    E = w.E
    if w.routing in ("zipf", "zipf_distinct"):
        perm = rng.permutation(E)
        p = np.zeros(E)
        p[perm] = _zipf_weights(E, w.zipf_s)
        return p
    if w.routing == "hot0_distinct":
        epr = E // w.R
        empty = rng.choice(np.arange(1, w.R), size=w.empty_ranks, replace=False)
        allowed = np.ones(E, dtype=bool)
        for r in empty:
            allowed[r * epr:(r + 1) * epr] = False
        allowed[0] = False
        others = np.flatnonzero(allowed)
        perm = rng.permutation(others)
        p = np.zeros(E)
        p[perm] = (1.0 - w.p0) * _zipf_weights(len(others), w.zipf_s)
        p[0] = w.p0
        return p
    raise ValueError(w.routing)


def make_routing(w: Workload, rng: np.random.Generator) -> np.ndarray:
    R, T, E, k = w.R, w.T, w.E, w.k
    if w.routing == "uniform":
        if k == 1:
            return rng.integers(0, E, size=(R, T, 1), dtype=np.int32)
        logw = np.zeros(E)
        return _gumbel_topk(rng, logw, (R, T), k)
    p = routing_weights(w, rng)
    if w.routing == "zipf":
        if k != 1:
            raise ValueError("zipf routing is top-1; use zipf_distinct for k > 1")
        return rng.choice(E, size=(R, T, 1), p=p).astype(np.int32)
    with np.errstate(divide="ignore"):
        logw = np.log(p)
    return _gumbel_topk(rng, logw, (R, T), k)


def make_gate(w: Workload, rng: np.random.Generator) -> np.ndarray:
    R, T, k = w.R, w.T, w.k
    if w.gate == "ones":
        return np.ones((R, T, k), dtype=np.float32)
    logits = rng.standard_normal((R, T, k), dtype=np.float32)
    ex = np.exp(logits - logits.max(axis=-1, keepdims=True)).astype(np.float32)
    return (ex / ex.sum(axis=-1, keepdims=True, dtype=np.float32)).astype(np.float32)


def _streams(seed: int):
    return [np.random.default_rng(ss) for ss in np.random.SeedSequence(seed).spawn(2)]


def make_x(w: Workload, seed: int = 0, device="cpu"):
    """torch bf16 tensor [R][T][H] on ``device``, N(0, 1) rounded to bf16."""
    import torch

    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    n = w.R * w.T * w.H
    x = torch.empty(n, dtype=torch.bfloat16, device=dev)
    step = 1 << 27
    for lo in range(0, n, step):
        hi = min(n, lo + step)
        x[lo:hi] = torch.randn(hi - lo, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    return x.view(w.R, w.T, w.H)


def make_logits(w: Workload, seed: int = 0, device="cpu"):
    """Router input: torch float32 logits [R][T][E] ~ N(0, 1) on ``device``
    (a separate generator stream from x: seed + 7919)."""
    import torch

    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed) + 7919)
    return torch.randn((w.R, w.T, w.E), generator=g, device=dev, dtype=torch.float32)


def bf16_bits(x) -> np.ndarray:
    """Host numpy uint16 view of a torch bf16 tensor's bit patterns."""
    import torch

    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def make_routing_gate(w: Workload, seed: int = 0) -> dict:
    """Seeded routing and gates: dict(topk_idx=int32 [R][T][k], gate_w=float32 [R][T][k])."""
    rng_route, rng_gate = _streams(seed)
    idx = np.ascontiguousarray(make_routing(w, rng_route), dtype=np.int32)
    gate = np.ascontiguousarray(make_gate(w, rng_gate), dtype=np.float32)
    return {"topk_idx": idx, "gate_w": gate}
