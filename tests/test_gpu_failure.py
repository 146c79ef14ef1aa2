"""Failure detection on the GPU without a fault: the bounded waits give up.

The TMA pack (default), the TMA combine and the lane-per-token router wait
on mbarriers for the bulk copies they issued themselves.  Every such wait is bounded: when it runs out
the kernel sets A2AV_DEV_WAIT_TIMEOUT in the plan's status word, lets every
copy it issued land (with the full bound) and returns, so the context stays
usable.  ``a2av_set_wait_limit(plan, 0)`` makes the main-loop wait give up at
once, which runs that path on purpose; the test then checks the status bit,
that the call returned, and that the next call on the same plan, with the
default limit, is parity-green against the oracle.
"""
import numpy as np
import pytest

import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

CASES = [(1, None, None, 0), (2, 1100, 264, 0), (5, 120, 72, 0), (4, 600, 136, 2)]


@pytest.mark.parametrize("wid,T,H,flags", CASES, ids=[f"w{c[0]}-f{c[3]}" for c in CASES])
def test_pack_wait_gives_up_then_next_call_is_exact(wid, T, H, flags):
    import torch

    import combine_device_resident_gb300 as A

    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    dev = P.device()
    plan = A.Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=dev, flags=flags)
    x = W.make_x(w, 0, device=dev)
    rg = W.make_routing_gate(w, 0)
    idx_t = torch.from_numpy(rg["topk_idx"]).to(dev)
    recv, slot_map, _ = plan.new_buffers()
    sp = plan.new_splits()
    plan.read_status(clear=True)
    plan.set_wait_limit(0)
    plan.dispatch(x, idx_t, sp, recv, slot_map)
    torch.cuda.synchronize()
    st = plan.read_status(clear=True)
    assert st & A.DEV_WAIT_TIMEOUT, f"status {st:#x}"
    plan.set_wait_limit(-1)
    g = P.full_parity(w, plan=plan)
    assert g["status"] == 0
    np.testing.assert_array_equal(g["out"], g["ref"]["out"])
    plan.close()


@pytest.mark.parametrize("wid,T,H", [(1, None, None), (4, 600, 136), (5, 90, 264)])
def test_tma_combine_wait_gives_up_then_next_call_is_exact(wid, T, H):
    import torch

    import combine_device_resident_gb300 as A

    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    dev = P.device()
    plan = A.Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=dev, flags=A.FLAG_COMBINE_TMA)
    x = W.make_x(w, 0, device=dev)
    rg = W.make_routing_gate(w, 0)
    idx_t = torch.from_numpy(rg["topk_idx"]).to(dev)
    gate_t = torch.from_numpy(rg["gate_w"]).to(dev)
    recv, slot_map, out = plan.new_buffers()
    sp = plan.new_splits()
    plan.read_status(clear=True)
    plan.dispatch(x, idx_t, sp, recv, slot_map)
    torch.cuda.synchronize()
    assert plan.read_status() == 0
    plan.set_wait_limit(0)
    plan.combine(recv, gate_t, slot_map, out)
    torch.cuda.synchronize()
    st = plan.read_status(clear=True)
    assert st & A.DEV_WAIT_TIMEOUT, f"status {st:#x}"
    plan.set_wait_limit(-1)
    g = P.full_parity(w, plan=plan)
    assert g["status"] == 0
    np.testing.assert_array_equal(g["out"], g["ref"]["out"])
    plan.close()


@pytest.mark.parametrize("wid,T", [(4, 300), (5, 100), (2, 200)])
def test_router_wait_gives_up_then_next_call_is_exact(wid, T):
    import torch

    import combine_device_resident_gb300 as A
    from oracle import route as oracle_route

    w = W.WORKLOADS[wid].scaled(T=T, H=8)
    dev = P.device()
    plan = A.Plan(w.R, w.E, w.T, w.H, w.k, device=dev)
    warp = A.Plan(w.R, w.E, w.T, w.H, w.k, device=dev, flags=A.FLAG_ROUTE_WARP)
    logits = W.make_logits(w, 3, device=dev)
    idx = torch.full((w.R, w.T, w.k), -9, dtype=torch.int32, device=dev)
    gate = torch.zeros((w.R, w.T, w.k), dtype=torch.float32, device=dev)
    plan.read_status(clear=True)
    plan.set_wait_limit(0)
    plan.route(logits, idx, gate)
    torch.cuda.synchronize()
    st = plan.read_status(clear=True)
    assert st & A.DEV_WAIT_TIMEOUT, f"status {st:#x}"
    plan.set_wait_limit(-1)
    plan.route(logits, idx, gate)
    widx = torch.empty_like(idx)
    wgate = torch.empty_like(gate)
    warp.route(logits, widx, wgate)  # the warp-per-token kernel waits on nothing
    torch.cuda.synchronize()
    assert plan.read_status() == 0 and warp.read_status() == 0
    ridx, _ = oracle_route(logits.cpu().numpy(), w.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(widx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(gate.cpu().numpy().view(np.uint32), wgate.cpu().numpy().view(np.uint32))
    plan.close()
    warp.close()


def test_wait_limit_is_per_plan():
    import torch

    import combine_device_resident_gb300 as A

    w = W.WORKLOADS[2].scaled(T=500, H=136)
    dev = P.device()
    short = A.Plan(w.R, w.E, w.T, w.H, w.k, device=dev)
    short.set_wait_limit(0)
    g = P.full_parity(w)  # a second plan keeps the default limit
    assert g["status"] == 0
    x = W.make_x(w, 0, device=dev)
    idx_t = torch.from_numpy(W.make_routing_gate(w, 0)["topk_idx"]).to(dev)
    recv, slot_map, _ = short.new_buffers()
    short.dispatch(x, idx_t, short.new_splits(), recv, slot_map)
    torch.cuda.synchronize()
    assert short.read_status() & A.DEV_WAIT_TIMEOUT
    short.close()
    g["plan"].close()
