"""a2av_dispatch_static: the dispatch for callers that cannot allocate device
memory where they dispatch (inside a framework whose caching allocator owns
all device memory, under a device-memory budget that is already spent, or in
a loop that cannot take cudaMalloc's implicit synchronisation).  It keeps its
kernels' scratch in a static device array of the library instead of a plan's
workspace.

Checked through the C ABI against the plan-based a2av_dispatch on the same
inputs, on two calls in a row with different routings (so contents the first
call leaves in the shared array cannot leak into the second): splits, offsets,
slot_map and every dispatched recv row bit-exact, as the integer/byte work of
dispatch is everywhere in these tests.  This file is collected last on
purpose; it also passes when run alone in a fresh process.
"""
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


def _plan_dispatch(w, x, idx_t):
    import combine_device_resident_gb300 as A

    plan = A.Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=x.device, recv_order=w.recv_order)
    recv, slot_map, _ = plan.new_buffers()
    recv.zero_()
    sp = plan.new_splits(expert_offsets=True)
    plan.dispatch(x, idx_t, sp, recv, slot_map)
    return plan, sp, recv, slot_map


def _static_dispatch(w, x, idx_t):
    import torch

    import combine_device_resident_gb300 as A
    from combine_device_resident_gb300.binding import dispatch_static

    dev = x.device
    sp = A.Splits(w.R, w.E, dev)
    arena = w.R * w.T * w.k if w.window_mode == "packed" else w.R * w.window_rows
    recv = torch.zeros((arena, w.H), dtype=torch.bfloat16, device=dev)
    slot_map = torch.full((w.R, w.T, w.k), -5, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dispatch_static(x, idx_t, sp, recv, slot_map, status, w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows,
                    recv_order=w.recv_order)
    return sp, recv, slot_map, status


@pytest.mark.parametrize("wid,T,H,order", [(5, 700, 264, "source"), (3, 900, 136, "source"), (4, 3000, 72, "source"),
                                           (5, 500, 72, "expert"), (2, 900, 64, "expert")])
def test_static_dispatch_matches_plan_dispatch_on_two_calls(wid, T, H, order):
    import dataclasses

    import torch

    dev = torch.device("cuda", 0)
    w = dataclasses.replace(W.WORKLOADS[wid].scaled(T=T, H=H), recv_order=order)
    x = W.make_x(w, 0, device=dev)
    for seed in (11, 12):
        idx_t = torch.from_numpy(W.make_routing_gate(w, seed)["topk_idx"]).to(dev)
        plan, sp_ref, recv_ref, sm_ref = _plan_dispatch(w, x, idx_t)
        sp, recv, sm, status = _static_dispatch(w, x, idx_t)
        torch.cuda.synchronize()
        for name in sp.NAMES:
            assert torch.equal(getattr(sp, name), getattr(sp_ref, name)), name
        assert torch.equal(sm, sm_ref)
        rows = sm_ref.flatten()
        rows = rows[rows >= 0].long()
        assert torch.equal(recv.index_select(0, rows).view(torch.int16),
                           recv_ref.index_select(0, rows).view(torch.int16))
        assert int(status.item()) == 0 and plan.read_status() == 0
        plan.close()


def test_static_dispatch_rejects_shapes_beyond_its_scratch():
    import torch

    import combine_device_resident_gb300 as A
    from combine_device_resident_gb300.binding import dispatch_static

    dev = torch.device("cuda", 0)
    # 64 ranks x 2048 experts x 2 tiles needs far more than 262144 int32
    R, E, T, H, k = 64, 2048, 600, 8, 4
    x = torch.zeros((R, T, H), dtype=torch.bfloat16, device=dev)
    idx = torch.zeros((R, T, k), dtype=torch.int32, device=dev)
    sp = A.Splits(R, E, dev)
    recv = torch.zeros((R * T * k, H), dtype=torch.bfloat16, device=dev)
    sm = torch.zeros((R, T, k), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(A.A2avError, match="scratch"):
        dispatch_static(x, idx, sp, recv, sm, status, R, E, T, H, k)
    torch.cuda.synchronize()
    assert int(sp.recv_total.sum().item()) == 0  # nothing was enqueued


def test_static_dispatch_rejects_wrong_shapes_before_enqueueing():
    import torch

    import combine_device_resident_gb300 as A
    from combine_device_resident_gb300.binding import dispatch_static

    dev = torch.device("cuda", 0)
    R, E, T, H, k = 4, 16, 50, 64, 2
    good = dict(x=torch.zeros((R, T, H), dtype=torch.bfloat16, device=dev),
                topk_idx=torch.zeros((R, T, k), dtype=torch.int32, device=dev),
                splits=A.Splits(R, E, dev),
                recv=torch.full((R * T * k, H), 5.0, dtype=torch.bfloat16, device=dev),
                slot_map=torch.full((R, T, k), -9, dtype=torch.int32, device=dev),
                dev_status=torch.zeros(1, dtype=torch.int32, device=dev))
    bad = {"x": torch.zeros((R, T, H - 8), dtype=torch.bfloat16, device=dev),
           "topk_idx": torch.zeros((R, T - 1, k), dtype=torch.int32, device=dev),
           "splits": A.Splits(R, 2 * E, dev),
           "recv": torch.zeros((R * T * k - 1, H), dtype=torch.bfloat16, device=dev),
           "slot_map": torch.zeros((R, T, 1), dtype=torch.int32, device=dev),
           "dev_status": torch.zeros(0, dtype=torch.int32, device=dev)}
    for name, t in bad.items():
        args = dict(good, **{name: t})
        with pytest.raises(A.A2avError):
            dispatch_static(args["x"], args["topk_idx"], args["splits"], args["recv"], args["slot_map"],
                            args["dev_status"], R, E, T, H, k)
    torch.cuda.synchronize()
    assert (good["slot_map"] == -9).all() and (good["recv"] == 5.0).all()  # nothing ran
