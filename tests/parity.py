"""Shared GPU-vs-oracle parity harness for the tests.

The GPU side runs only through the C ABI (``combine_device_resident_gb300``);
the expected side runs only the CPU oracle (``oracle``) on host copies of the
same seeded inputs.  Tolerances (from the method's statement):
  * splits, offsets, slot_map, recv rows: bit-exact;
  * combine output: within 1 bf16 ulp (ordered-integer distance, +0 == -0).
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W
from tests.bf16util import ulp_diff

SPLIT_KEYS = ("send_counts", "send_offsets", "recv_counts", "recv_offsets", "recv_expert_counts",
              "recv_total", "window_base", "recv_expert_offsets")
COMBINE_ULP_TOL = 1


def device():
    import torch

    return torch.device("cuda", 0)


def gpu_run(w: W.Workload, x, idx: np.ndarray, gate: np.ndarray, flags=0, pack_ctas_per_sm=0,
            pack_stage_bytes=0, pack_store_lag=0, combine_ctas_per_sm=0, combine_stage_bytes=0,
            combine_unroll=0, guard_rows=4, expert=None, plan=None, num_tokens=None, expert_offsets=True):
    """Run dispatch (+ expert stand-in) + combine on the GPU through the C ABI.
    Returns host copies and the plan.  x is a torch bf16 tensor on the GPU.
    expert_offsets: ask the splits kernel for recv_expert_offsets (always
    written in the expert-grouped order)."""
    import torch
    from combine_device_resident_gb300 import Plan

    dev = device()
    if plan is None:
        plan = Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=dev, flags=flags,
                    pack_ctas_per_sm=pack_ctas_per_sm, pack_stage_bytes=pack_stage_bytes,
                    pack_store_lag=pack_store_lag, combine_ctas_per_sm=combine_ctas_per_sm,
                    combine_stage_bytes=combine_stage_bytes, combine_unroll=combine_unroll,
                    recv_order=w.recv_order)
    nt_t = None
    if num_tokens is not None:
        nt_t = torch.from_numpy(np.ascontiguousarray(num_tokens, np.int32)).to(dev)
    plan.set_active_tokens(nt_t)
    rows = plan.arena_rows
    canary = torch.full((rows + guard_rows, w.H), -7.0, dtype=torch.bfloat16, device=dev)
    recv = canary[:rows]
    out = torch.full((w.R, w.T, w.H), 3.0, dtype=torch.bfloat16, device=dev)  # untouched rows stay 3.0
    slot_map = torch.empty((w.R, w.T, w.k), dtype=torch.int32, device=dev)
    sp = plan.new_splits(expert_offsets=expert_offsets or None)
    idx_t = torch.from_numpy(idx).to(dev)
    gate_t = torch.from_numpy(gate).to(dev)
    plan.read_status(clear=True)
    if w.window_mode == "padded":
        sendbuf = plan.new_send_buffer()
        plan.dispatch_padded(x, idx_t, sp, sendbuf, recv, slot_map)
    else:
        plan.dispatch(x, idx_t, sp, recv, slot_map)
    expert = expert or w.expert
    if expert == "scale":
        y = torch.empty_like(recv)
        plan.expert_scale(recv, idx_t, slot_map, y)
    else:
        y = recv
    plan.combine(y, gate_t, slot_map, out)
    torch.cuda.synchronize()
    status = plan.read_status()
    guard = canary[rows:].view(torch.int16).cpu().numpy()
    fill = int(torch.tensor(-7.0, dtype=torch.bfloat16).view(torch.int16))
    return {"plan": plan, "splits": sp.to_numpy(), "slot_map": slot_map.cpu().numpy(), "recv_t": recv,
            "y_t": y, "out_t": out, "status": status, "guard_ok": bool((guard == fill).all()),
            "idx_t": idx_t, "gate_t": gate_t, "nt_t": nt_t}


def bits(t) -> np.ndarray:
    return W.bf16_bits(t)


def check_splits(got: dict, want: dict):
    """Every split array the GPU produced (recv_expert_offsets only when asked for)."""
    for key in SPLIT_KEYS:
        if key in got:
            np.testing.assert_array_equal(got[key], want[key].reshape(got[key].shape), err_msg=key)


def valid_rows(sp: dict) -> np.ndarray:
    """Arena rows that hold a dispatched assignment: [base_d, base_d + total_d)."""
    return np.concatenate([np.arange(b, b + n) for b, n in zip(sp["window_base"], sp["recv_total"])]
                          ) if len(sp["window_base"]) else np.zeros(0, np.int64)


def full_parity(w: W.Workload, seed=0, idx=None, gate=None, x=None, **kw):
    """Element-by-element parity of the whole path on a size the oracle finishes quickly."""
    import torch

    if x is None:
        x = W.make_x(w, seed, device=device())
    if idx is None or gate is None:
        rg = W.make_routing_gate(w, seed)
        idx = rg["topk_idx"] if idx is None else idx
        gate = rg["gate_w"] if gate is None else gate
    g = gpu_run(w, x, idx, gate, **kw)
    xh = bits(x)
    nt = kw.get("num_tokens")
    ref = oracle.run_all(w.R, w.E, xh, idx, gate, w.window_mode, w.window_rows, kw.get("expert") or w.expert,
                         num_tokens=nt, recv_order=w.recv_order)
    check_splits(g["splits"], ref["splits"])
    np.testing.assert_array_equal(g["slot_map"], ref["slot_map"], err_msg="slot_map")
    assert g["status"] == ref["status"], (g["status"], ref["status"])
    rows = ref["slot_map"][ref["slot_map"] >= 0]
    recv = bits(g["recv_t"])
    np.testing.assert_array_equal(recv[np.sort(rows)], ref["recv"][np.sort(rows)], err_msg="recv rows")
    out = bits(g["out_t"])
    if nt is not None:
        # tokens that take part: the oracle's combine; the others: untouched
        act = np.zeros((w.R, w.T), bool)
        for s_ in range(w.R):
            act[s_, :min(max(int(nt[s_]), 0), w.T)] = True
        untouched = int(np.array([3.0], np.float32).view(np.uint32)[0] >> 16)
        assert (out[~act] == untouched).all(), "combine wrote rows of tokens that take no part"
        d = ulp_diff(out[act], ref["out"][act])
    else:
        d = ulp_diff(out, ref["out"])
    assert d.max(initial=0) <= COMBINE_ULP_TOL, f"combine off by {d.max()} ulp"
    assert g["guard_ok"], "a store landed past the end of the recv arena"
    g["ref"] = ref
    g["out"] = out
    torch.cuda.synchronize()
    return g
