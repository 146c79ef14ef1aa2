"""Parity at the workloads' full sizes, in the benchmark's launch configuration.

* splits, offsets and slot_map: bit-exact against the oracle for every
  assignment (the oracle computes them without moving payload);
* recv: every dispatched row equals its source token row (recv[slot] ==
  x[s][t], checked on the device in chunks -- a property that holds at any
  size, with slot_map already proven equal to the oracle's);
* rows beyond each window's recv_total are untouched (canary rows);
* combine: sampled tokens against the oracle's combine of the same tokens,
  built from the inputs alone (each token's k expert rows), within 1 bf16 ulp.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import parity as P
from tests.bf16util import ulp_diff

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sampled_reference(w, xh_rows, idx_rows, gate_rows, expert):
    """Oracle combine of n sampled tokens: their k expert rows laid out as a
    small arena, row i*k+j = expert_j(x_i)."""
    n = xh_rows.shape[0]
    k = w.k
    arena = np.repeat(xh_rows, k, axis=0)
    sm = np.arange(n * k, dtype=np.int32).reshape(n, 1, k)
    idx3 = idx_rows.reshape(n, 1, k)
    y = oracle.expert_scale(w.E, arena, idx3, sm) if expert == "scale" else arena
    return oracle.combine(y, gate_rows.reshape(n, 1, k), sm)


def _check_full(w, x, idx, gate, seed, num_tokens=None, expert_offsets=False):
    """Run the path at full size and check it (see the module docstring)."""
    import torch

    dev = P.device()
    g = P.gpu_run(w, x, idx, gate, guard_rows=2, expert_offsets=expert_offsets, num_tokens=num_tokens)
    sp = oracle.splits(w.R, w.E, idx, w.window_mode, w.window_rows, num_tokens, w.recv_order)
    P.check_splits(g["splits"], sp)
    sm_ref, st = oracle.slot_map(w.R, w.E, idx, sp, w.window_mode, w.window_rows, num_tokens, w.recv_order)
    np.testing.assert_array_equal(g["slot_map"], sm_ref)
    assert g["status"] == (sp["status"] | st) == 0
    assert g["guard_ok"]
    act = np.ones((w.R, w.T), bool)
    if num_tokens is not None:
        for s_ in range(w.R):
            act[s_, max(0, min(w.T, int(num_tokens[s_]))):] = False
    act_f = act.reshape(-1)

    # every dispatched row carries its token (on the device, chunked)
    slot_t = torch.from_numpy(sm_ref).to(dev).view(-1, w.k)
    recv = g["recv_t"]
    xf = x.view(-1, w.H)
    act_t = torch.from_numpy(act_f).to(dev)
    step = max(1, (1 << 28) // (w.H * 2 * w.k))
    for lo in range(0, xf.shape[0], step):
        hi = min(xf.shape[0], lo + step)
        keep = act_t[lo:hi]
        rows = slot_t[lo:hi][keep].reshape(-1).long()
        got = recv.index_select(0, rows).view(-1, w.k, w.H)
        want = xf[lo:hi][keep].unsqueeze(1).expand(-1, w.k, -1)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
            f"recv rows of tokens {lo}..{hi} differ from their source rows"
    if w.window_mode == "packed" and num_tokens is None:
        assert np.array_equal(np.sort(sm_ref.ravel()), np.arange(w.R * w.T * w.k))

    # combine on sampled tokens that take part (including each rank's first and last)
    rng = np.random.default_rng(seed)
    cand = np.flatnonzero(act_f)
    ends = np.concatenate([np.arange(w.R) * w.T, np.arange(w.R) * w.T + act.sum(axis=1) - 1])
    ends = ends[(ends >= 0) & act_f[np.clip(ends, 0, act_f.size - 1)]]
    pick = np.unique(np.concatenate([rng.choice(cand, size=min(cand.size, 1500), replace=False), ends]))
    pick_t = torch.from_numpy(pick).to(dev)
    got_out = P.bits(g["out_t"].view(-1, w.H).index_select(0, pick_t))
    xs = P.bits(xf.index_select(0, pick_t))
    want = _sampled_reference(w, xs, idx.reshape(-1, w.k)[pick], gate.reshape(-1, w.k)[pick], w.expert)
    d = ulp_diff(got_out, want)
    assert d.max() <= P.COMBINE_ULP_TOL
    res = {"slot_map": sm_ref, "splits": g["splits"]}
    del g
    torch.cuda.empty_cache()
    return res


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_full_size(wid):
    w = W.WORKLOADS[wid]
    rg = W.make_routing_gate(w, 0)
    x = W.make_x(w, 0, device=P.device())
    _check_full(w, x, rg["topk_idx"], rg["gate_w"], wid)  # as the benchmark calls it (no expert offsets)


@pytest.mark.parametrize("wid", [4, 5])
def test_full_size_expert_order(wid):
    import dataclasses

    w = dataclasses.replace(W.WORKLOADS[wid], recv_order="expert")
    rg = W.make_routing_gate(w, 0)
    x = W.make_x(w, 0, device=P.device())
    res = _check_full(w, x, rg["topk_idx"], rg["gate_w"], wid, expert_offsets=True)
    # each local expert's rows form one block starting at recv_expert_offsets[d][0][le]
    sp, idx, epr = res["splits"], rg["topk_idx"].reshape(-1), w.E // w.R
    rel = res["slot_map"].reshape(-1) - sp["window_base"][idx // epr]
    order = np.lexsort((rel, idx))
    e_sorted, rel_sorted = idx[order], rel[order]
    start = sp["recv_expert_offsets"][e_sorted // epr, 0, e_sorted % epr]
    first = np.r_[0, np.flatnonzero(np.diff(e_sorted)) + 1]
    pos = np.arange(e_sorted.size) - np.repeat(first, np.diff(np.r_[first, e_sorted.size]))
    np.testing.assert_array_equal(rel_sorted, start + pos)


@pytest.mark.parametrize("wid", [4, 5])
def test_full_size_router(wid):
    # the router at full size: ids bit-exact, gates within the derived bound,
    # then the path from those routings
    import torch
    from combine_device_resident_gb300 import Plan

    w = W.WORKLOADS[wid]
    dev = P.device()
    logits = W.make_logits(w, 0, device=dev)
    plan = Plan(w.R, w.E, w.T, w.H, w.k, device=dev)
    idx_t = torch.empty((w.R, w.T, w.k), dtype=torch.int32, device=dev)
    gate_t = torch.empty((w.R, w.T, w.k), dtype=torch.float32, device=dev)
    plan.route(logits, idx_t, gate_t)
    torch.cuda.synchronize()
    lh = logits.cpu().numpy()
    ridx, rgate = oracle.route(lh, w.k)
    idx = idx_t.cpu().numpy()
    np.testing.assert_array_equal(idx, ridx)
    sel = np.take_along_axis(lh.astype(np.float64), ridx.astype(np.int64), axis=-1)
    bound = (2 * np.abs(sel - sel[..., :1]).max(axis=-1, keepdims=True) + w.k + 8) * 2.0 ** -24
    gate = gate_t.cpu().numpy()
    assert (np.abs(gate.astype(np.float64) - rgate) <= bound * rgate).all()
    plan.close()
    x = W.make_x(w, 0, device=dev)
    _check_full(w, x, idx, gate, wid + 10)


def test_full_size_half_active():
    w = W.WORKLOADS[5]
    rg = W.make_routing_gate(w, 0)
    x = W.make_x(w, 0, device=P.device())
    nt = np.array([(w.T // 2 + 97 * s_) % (w.T + 1) for s_ in range(w.R)], np.int32)
    _check_full(w, x, rg["topk_idx"], rg["gate_w"], 55, num_tokens=nt)
