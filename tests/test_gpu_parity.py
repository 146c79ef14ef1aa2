"""GPU (C ABI) vs CPU oracle, element by element, on seeded inputs.

Bar: splits/offsets/slot_map/recv bit-exact; combine within 1 bf16 ulp.
Sizes are chosen so the oracle finishes in seconds while the histogram spans
several 2048-assignment tiles with a ragged last tile.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import parity as P
from tests.bf16util import is_inf, is_nan, ulp_diff

pytestmark = pytest.mark.gpu


# The five workloads at reduced T (several histogram tiles + ragged tail), full H.
SCALED = [
    (1, None, None),   # the small workload itself: R=2 E=4 T=128 H=256 k=1
    (2, 4100, 512),    # 4100 assignments/rank: 3 tiles
    (3, 2500, 520),    # Zipf 1.2, fixed windows of R*T*k rows, H not a multiple of 64
    (4, 2100, 264),    # top-2 Zipf 1.0, softmax gates, scaled experts
    (5, 600, 136),     # top-8, hot expert 0, 4 empty ranks, softmax gates
]


@pytest.mark.parametrize("wid,T,H", SCALED, ids=[f"w{s[0]}" for s in SCALED])
def test_workload_parity(wid, T, H):
    w = W.WORKLOADS[wid]
    if T is not None:
        w = w.scaled(T=T, H=H)
    P.full_parity(w)


@pytest.mark.parametrize("wid,T,H", [(5, 160, 2056)])
def test_rows_beyond_l2_parity(wid, T, H):
    # Top-8 calls whose rows exceed the L2 (168 MB here) run the
    # pack with evict-first row stores and the combine with evict-first
    # gathers; element-by-element parity on every row and output.
    g = P.full_parity(W.WORKLOADS[wid].scaled(T=T, H=H))
    np.testing.assert_array_equal(g["out"], g["ref"]["out"])


@pytest.mark.parametrize("wid", [2, 3])
def test_workload_parity_full_hidden(wid):
    # the real row sizes (H=5120) on a few hundred tokens per rank
    P.full_parity(W.WORKLOADS[wid].scaled(T=300))


@pytest.mark.parametrize("unroll", [1, 2, 4, 8])
def test_combine_unroll_variants(unroll):
    for wid, T, H in [(1, None, None), (4, 300, 1032), (5, 60, 7176)]:
        w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
        g = P.full_parity(w, combine_unroll=unroll)
        np.testing.assert_array_equal(g["out"], g["ref"]["out"])
    P.full_parity(_uniform(4, 64, 200, 48, 3), combine_unroll=unroll)


@pytest.mark.parametrize("flags", [0, 4], ids=["lsu", "tma"])
def test_combine_is_bit_exact_against_oracle(flags):
    # The kernels round each product and sum separately in slot order, exactly
    # as the oracle does, so the result is the oracle's bit for bit (the
    # stated bar, 1 ulp, is looser).
    for wid, T, H in [(4, 700, 200), (5, 300, 64), (5, 90, 7176)]:
        g = P.full_parity(W.WORKLOADS[wid].scaled(T=T, H=H), flags=flags)
        np.testing.assert_array_equal(g["out"], g["ref"]["out"])


@pytest.mark.parametrize("k,first,variant", [(2, 0, {}), (2, 0, dict(combine_unroll=1)), (2, 0, dict(combine_unroll=4)),
                                             (2, 0, dict(flags=4)), (3, 0, {}), (3, 0, dict(flags=4)),
                                             (3, 1, {}), (3, 1, dict(flags=4)), (4, 2, {}), (4, 2, dict(combine_unroll=2))],
                         ids=["k2", "k2-u1", "k2-u4", "k2-tma", "k3-generic", "k3-tma", "k3-slot0-empty",
                              "k3-slot0-empty-tma", "k4-slots01-empty", "k4-slots01-empty-u2"])
def test_combine_rounds_product_and_sum_hand_case(k, first, variant):
    # The oracle pin's slot pair whose separately rounded and fused readings
    # differ in the output bf16, through the C ABI, in slots first and
    # first + 1 (the other slots empty): every column of every token must come
    # out as the separately rounded reading.  With first > 0 the pair's first
    # value is not in slot 0, so it is accumulated on the scalar path from +0.
    import torch
    from combine_device_resident_gb300 import Plan
    from tests.test_oracle_pins import SLOT_PAIR_SEPARATE, SLOT_PAIR_W, SLOT_PAIR_Y

    R, E, T, H = 2, 4, 40, 264
    dev = P.device()
    plan = Plan(R, E, T, H, k, device=dev, **variant)
    recv, slot_map, out = plan.new_buffers()
    rows = recv.view(torch.int16)
    rows[0].fill_(int(SLOT_PAIR_Y[0].view(np.int16)))
    rows[1].fill_(int(SLOT_PAIR_Y[1].view(np.int16)))
    sm = np.full((R, T, k), -1, np.int32)
    sm[..., first], sm[..., first + 1] = 0, 1
    gate = np.full((R, T, k), np.float32(np.inf))  # empty slots: a weight used anyway would give inf or NaN
    gate[..., first:first + 2] = SLOT_PAIR_W
    slot_map.copy_(torch.from_numpy(sm))
    plan.combine(recv, torch.from_numpy(gate).to(dev), slot_map, out)
    torch.cuda.synchronize()
    got = P.bits(out)
    assert (got == SLOT_PAIR_SEPARATE).all(), np.unique(got)
    assert plan.read_status() == 0


@pytest.mark.parametrize("variant", [
    dict(flags=1),                              # LSU pack
    dict(pack_ctas_per_sm=1),                   # one TMA CTA per SM, deep ring
    dict(pack_ctas_per_sm=2, pack_store_lag=1),  # stores must finish reading before each refill
    dict(pack_stage_bytes=1024),                # rows split into several stage chunks
    dict(pack_stage_bytes=4096, pack_ctas_per_sm=3, pack_store_lag=6),
    dict(flags=2),                              # tiled splits kernel forced
    dict(flags=3),                              # tiled splits + LSU pack
    dict(flags=4),                              # TMA combine
    dict(flags=7),                              # LSU pack, tiled splits, TMA combine
    dict(flags=4, combine_ctas_per_sm=1, combine_stage_bytes=2048),   # TMA combine: deep ring, small chunks
    dict(flags=4, combine_ctas_per_sm=8, combine_stage_bytes=65536),  # TMA combine: whole rows, 2 stages
], ids=["lsu", "tma1", "lag1", "chunked", "chunked3-lag6", "tiled", "tiled-lsu", "tma-combine", "mixed",
        "comb-deep", "comb-wide"])
def test_pack_variants(variant):
    P.full_parity(W.WORKLOADS[5].scaled(T=500, H=1032), **variant)
    P.full_parity(W.WORKLOADS[2].scaled(T=900, H=2056), **variant)
    P.full_parity(W.WORKLOADS[2].scaled(T=200, H=520), **variant)  # one-CTA splits unless forced


@pytest.mark.parametrize("wid,T,H", [(1, None, None), (2, 1024, 264), (3, 256, 136), (3, 130, 40)])
def test_one_cta_and_tiled_splits_agree(wid, T, H):
    # workloads small enough for the one-CTA splits kernel, run both ways
    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    a = P.full_parity(w)
    b = P.full_parity(w, flags=2)
    assert a["plan"].cfg.flags == 0 and b["plan"].cfg.flags == 2
    np.testing.assert_array_equal(a["slot_map"], b["slot_map"])


def _uniform(R, E, T, H, k, **kw):
    return W.Workload("edge", R=R, E=E, T=T, H=H, k=k, routing="zipf_distinct" if k > 1 else "uniform",
                      zipf_s=0.0, gate="softmax" if k > 1 else "ones", **kw)


def test_all_tokens_to_one_expert():
    w = _uniform(8, 16, 3000, 64, 1)
    idx = np.full((w.R, w.T, 1), 5, np.int32)
    g = P.full_parity(w, idx=idx, gate=np.ones_like(idx, np.float32))
    assert g["splits"]["recv_total"].tolist() == [0, 0, w.R * w.T, 0, 0, 0, 0, 0]


def test_empty_ranks_and_empty_experts():
    w = _uniform(4, 16, 2500, 40, 2)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice([0, 1, 8, 9, 10], size=2, replace=False) for _ in range(w.R * w.T)]).astype(np.int32)
    idx = idx.reshape(w.R, w.T, 2)
    g = P.full_parity(w, idx=idx)
    assert g["splits"]["recv_total"][1] == 0 and g["splits"]["recv_total"][3] == 0


def test_one_expert_per_rank():
    P.full_parity(_uniform(8, 8, 700, 88, 1))


def test_every_expert_per_token():
    # k = E: each token goes to every expert (and so to every rank)
    P.full_parity(_uniform(2, 4, 900, 24, 4))


@pytest.mark.parametrize("H", [8, 200, 6152])
def test_row_sizes(H):
    P.full_parity(_uniform(4, 8, 300, H, 2))


def test_single_token():
    P.full_parity(_uniform(8, 16, 1, 5120, 2))
    P.full_parity(_uniform(1, 1, 1, 8, 1))


@pytest.mark.parametrize("k", [3, 5, 16, 32])
def test_generic_topk(k):
    P.full_parity(_uniform(4, 64, 200, 48, k))


def test_maximum_ranks_and_experts():
    P.full_parity(_uniform(64, 2048, 40, 8, 4))


def test_duplicate_experts_in_a_token():
    w = _uniform(2, 8, 1500, 16, 3)
    rng = np.random.default_rng(9)
    idx = rng.integers(0, 8, size=(w.R, w.T, 3), dtype=np.int32)  # duplicates allowed
    P.full_parity(w, idx=idx, gate=rng.random((w.R, w.T, 3), dtype=np.float32))


def test_bad_expert_ids_set_status_and_are_dropped():
    import combine_device_resident_gb300 as A

    w = _uniform(4, 16, 2200, 32, 2)
    rg = W.make_routing_gate(w, 3)
    idx = rg["topk_idx"].copy()
    idx[0, 7, 1] = -3
    idx[2, 2100, 0] = 16
    idx[3, 0, 0] = 1 << 30
    g = P.full_parity(w, idx=idx, gate=rg["gate_w"])
    assert g["status"] & A.DEV_BAD_EXPERT
    assert g["slot_map"][0, 7, 1] == -1 and g["slot_map"][2, 2100, 0] == -1


def test_fixed_window_overflow_is_flagged_and_bounded():
    import combine_device_resident_gb300 as A

    w = _uniform(4, 8, 2200, 24, 1, window_mode="fixed", window_rows=900)
    idx = np.zeros((w.R, w.T, 1), np.int32)
    idx[:, ::3] = 3  # rank 0 and 1 experts; window 0 gets ~5900 rows > 900
    g = P.full_parity(w, idx=idx, gate=np.ones_like(idx, np.float32))
    assert g["status"] & A.DEV_WINDOW_OVERFLOW
    assert (g["slot_map"] >= 0).sum() == 2 * 900
    assert g["guard_ok"]


@pytest.mark.parametrize("wid,T,H,flags", [(4, 300, 72, 0), (4, 300, 72, 4), (5, 60, 136, 0), (3, 256, 264, 0)],
                         ids=["top2", "top2-tma-combine", "top8", "top1-fixed"])
def test_non_finite_payloads(wid, T, H, flags):
    # Reading on non-finite values: the dispatch copies NaN and infinity bits
    # unchanged (bit-exact, as every recv row); the combine follows IEEE fp32
    # (a zero gate times an infinity is NaN, +inf plus -inf is NaN, a NaN stays
    # NaN); a NaN output matches any NaN, an infinity only the same infinity.
    import torch

    w = W.WORKLOADS[wid].scaled(T=T, H=H)
    dev = P.device()
    x = W.make_x(w, 0, device=dev)
    rg = W.make_routing_gate(w, 0)
    idx, gate = rg["topk_idx"], rg["gate_w"].copy()
    xb = x.view(torch.int16)
    PINF, NINF, QNAN, SNAN = 0x7F80, -0x80, 0x7FC1, -0x60  # bf16 +inf, -inf, quiet NaN, 0xFFA0 (signalling, negative)
    xb[0, 0, :] = PINF
    xb[0, 1, :] = NINF
    xb[0, 2, 3] = QNAN
    xb[0, 3, 0::2] = PINF
    xb[0, 3, 1::2] = NINF
    xb[1, 4, 7] = SNAN
    xb[1, 5, :] = PINF
    gate[0, 0, -1] = 0.0   # a zero gate on an infinite row: NaN (top-1: the only slot)
    gate[1, 5, 0] = -gate[1, 5, 0]  # opposite infinities in one sum when k > 1
    g = P.full_parity(w, x=x, idx=idx, gate=gate, flags=flags)
    ref = g["ref"]["out"].reshape(w.R * w.T, w.H)
    out = g["out"].reshape(w.R * w.T, w.H)
    assert is_nan(ref).any() and is_inf(ref).any()  # the case is not vacuous
    np.testing.assert_array_equal(is_nan(out), is_nan(ref))
    fin = ~is_nan(ref)
    np.testing.assert_array_equal(out[fin], ref[fin])  # everything else bit for bit


def test_null_and_misaligned_pointers_are_rejected():
    # Host-side argument checks of the C ABI: a null or misaligned buffer is
    # refused with A2AV_ERR_INVALID_ARG before anything is enqueued (the
    # plan's launch count does not move and the device status stays clear).
    import ctypes

    import torch
    from combine_device_resident_gb300 import Plan

    w = W.WORKLOADS[2].scaled(T=64, H=136)
    dev = P.device()
    plan = Plan(w.R, w.E, w.T, w.H, w.k, device=dev)
    L, h = plan.lib, plan.handle
    x = W.make_x(w, 0, device=dev)
    idx = torch.zeros((w.R, w.T, w.k), dtype=torch.int32, device=dev)
    gate = torch.ones((w.R, w.T, w.k), dtype=torch.float32, device=dev)
    recv, slot_map, out = plan.new_buffers()
    sp = plan.new_splits()
    spp = ctypes.byref(sp.ptrs)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    before = L.a2av_plan_launches(h)
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)  # noqa: E731
    null = ctypes.c_void_p(0)
    invalid = 1  # A2AV_ERR_INVALID_ARG
    bad_dispatch = [
        (null, p(idx), spp, p(recv), p(slot_map)),          # null x
        (p(x, 2), p(idx), spp, p(recv), p(slot_map)),       # x not 16-byte aligned
        (p(x), p(idx), spp, p(recv, 8), p(slot_map)),       # recv not 16-byte aligned
        (p(x), p(idx, 2), spp, p(recv), p(slot_map)),       # topk_idx not 4-byte aligned
        (p(x), p(idx), spp, p(recv), null),                 # null slot_map
    ]
    for a in bad_dispatch:
        assert L.a2av_dispatch(h, *a, stream) == invalid
    bad_combine = [
        (p(recv, 2), p(gate), p(slot_map), p(out)),         # y not 16-byte aligned
        (p(recv), null, p(slot_map), p(out)),               # null gate
        (p(recv), p(gate), p(slot_map), p(out, 4)),         # out not 16-byte aligned
    ]
    for a in bad_combine:
        assert L.a2av_combine(h, *a, stream) == invalid
    assert L.a2av_dispatch(None, p(x), p(idx), spp, p(recv), p(slot_map), stream) == invalid  # no plan
    torch.cuda.synchronize()
    assert L.a2av_plan_launches(h) == before
    assert plan.read_status() == 0
    plan.close()


def test_status_read_and_clear():
    w = _uniform(2, 4, 100, 8, 1)
    idx = np.full((2, 100, 1), 9, np.int32)
    g = P.gpu_run(w, W.make_x(w, 0, device=P.device()), idx, np.ones_like(idx, np.float32))
    plan = g["plan"]
    assert plan.read_status(clear=True) & 1
    assert plan.read_status() == 0


# (4, 1100, 136): a large call; (3, 256, 1032) and (4, 128, 520): few-token
# calls (fewer tokens than combine warps, rows split into pieces), which take
# the pack's early launch of the combine and the batched-metadata combine.
@pytest.mark.parametrize("wid,T,H", [(4, 1100, 136), (3, 256, 1032), (4, 128, 520)],
                         ids=["large", "few-tokens-top1", "few-tokens-top2"])
def test_graph_replay_with_new_routing_each_time(wid, T, H):
    # Capture dispatch + combine once; then rewrite topk_idx/gate_w in place and
    # replay.  The counts change with every replay while the graph stays the
    # same, and every replay matches the oracle.
    import torch
    from combine_device_resident_gb300 import Plan

    w = W.WORKLOADS[wid].scaled(T=T, H=H)
    dev = P.device()
    plan = Plan(w.R, w.E, w.T, w.H, w.k, device=dev)
    x = W.make_x(w, 0, device=dev)
    idx_t = torch.zeros((w.R, w.T, w.k), dtype=torch.int32, device=dev)
    gate_t = torch.zeros((w.R, w.T, w.k), dtype=torch.float32, device=dev)
    recv, slot_map, out = plan.new_buffers()
    sp = plan.new_splits()
    rg0 = W.make_routing_gate(w, 100)
    idx_t.copy_(torch.from_numpy(rg0["topk_idx"]))
    gate_t.copy_(torch.from_numpy(rg0["gate_w"]))
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):  # warm up outside capture
        plan.dispatch(x, idx_t, sp, recv, slot_map)
        plan.combine(recv, gate_t, slot_map, out)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.dispatch(x, idx_t, sp, recv, slot_map)
        plan.combine(recv, gate_t, slot_map, out)
    xh = P.bits(x)
    seen_totals = set()
    for seed in range(101, 105):
        rg = W.make_routing_gate(w.scaled(T=w.T), seed)
        if seed % 2:
            rg = {"topk_idx": np.roll(rg["topk_idx"], seed, axis=1), "gate_w": rg["gate_w"]}
        idx_t.copy_(torch.from_numpy(rg["topk_idx"]))
        gate_t.copy_(torch.from_numpy(rg["gate_w"]))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.run_all(w.R, w.E, xh, rg["topk_idx"], rg["gate_w"])
        P.check_splits(sp.to_numpy(), ref["splits"])
        np.testing.assert_array_equal(slot_map.cpu().numpy(), ref["slot_map"])
        assert ulp_diff(P.bits(out), ref["out"]).max() <= P.COMBINE_ULP_TOL
        seen_totals.add(tuple(ref["splits"]["recv_total"].tolist()))
    assert len(seen_totals) > 1
    assert plan.read_status() == 0


@pytest.mark.parametrize("wid,T,H,flags,graph", [(3, 256, 1032, 0, False), (1, None, None, 0, True),
                                                 (2, 700, 264, 2, False), (5, 90, 136, 0, True),
                                                 (4, 300, 136, 4, False)],
                         ids=["cluster", "cluster-graph", "tiled", "tiled-top8-graph", "tma-combine"])
def test_back_to_back_calls_reusing_buffers(wid, T, H, flags, graph):
    # Consecutive dispatch+combine calls on one stream, with no host sync
    # between them, reuse the splits arrays, slot_map and the arena.  Each
    # splits kernel is a programmatic dependent of the previous call's combine
    # and may be resident before it ends; nothing it writes may reach the
    # buffers the combine still reads.  Each call has its own routing and its
    # own out, and every out must match the oracle.
    import torch
    from combine_device_resident_gb300 import Plan

    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    dev = P.device()
    plan = Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=dev, flags=flags)
    x = W.make_x(w, 0, device=dev)
    recv, slot_map, _ = plan.new_buffers()
    sp = plan.new_splits()
    n = 6
    rgs = [W.make_routing_gate(w, 200 + i) for i in range(n)]
    idx = [torch.from_numpy(r["topk_idx"]).to(dev) for r in rgs]
    gate = [torch.from_numpy(r["gate_w"]).to(dev) for r in rgs]
    outs = [torch.full((w.R, w.T, w.H), 7.0, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    plan.read_status(clear=True)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))

    def calls():
        for i in range(n):
            plan.dispatch(x, idx[i], sp, recv, slot_map, stream=s)
            plan.combine(recv, gate[i], slot_map, outs[i], stream=s)

    if graph:
        with torch.cuda.stream(s):
            calls()  # warm-up outside capture
        torch.cuda.synchronize()
        for o in outs:
            o.fill_(7.0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            calls()
        g.replay()
    else:
        with torch.cuda.stream(s):
            calls()
    torch.cuda.synchronize()
    xh = P.bits(x)
    for i in range(n):
        ref = oracle.run_all(w.R, w.E, xh, rgs[i]["topk_idx"], rgs[i]["gate_w"], w.window_mode, w.window_rows)
        np.testing.assert_array_equal(P.bits(outs[i]), ref["out"], err_msg=f"call {i}")
    np.testing.assert_array_equal(slot_map.cpu().numpy(), ref["slot_map"])  # the last call's
    P.check_splits(sp.to_numpy(), ref["splits"])
    assert plan.read_status() == 0
    plan.close()


@pytest.mark.parametrize("wid,T,H,graph", [(3, 256, 5120, False), (3, 256, 5120, True), (1, None, None, False),
                                           (2, 512, 1032, True), (4, 2048, 520, False)])
def test_chained_calls_out_feeds_next_dispatch(wid, T, H, graph):
    # Each call's out is the next call's x (layer after layer with nothing in
    # between), on one stream and without a host sync: the next call's pack
    # loads x before its own dependency wait, so it must not be launched
    # before this call's combine has completed.  out is filled with a
    # sentinel on the stream before the combine that writes it; every
    # received row of the next call must be its out row bit for bit.
    import torch
    from combine_device_resident_gb300 import Plan

    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    dev = P.device()
    plan = Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=dev)
    n = 4
    xs = [W.make_x(w, 0, device=dev)] + [torch.empty((w.R, w.T, w.H), dtype=torch.bfloat16, device=dev)
                                          for _ in range(n)]
    bufs = [plan.new_buffers()[:2] for _ in range(2)]  # double-buffered arenas
    sps = [plan.new_splits() for _ in range(2)]
    rgs = [W.make_routing_gate(w, 300 + i) for i in range(n)]
    idx = [torch.from_numpy(r["topk_idx"]).to(dev) for r in rgs]
    gate = [torch.from_numpy(r["gate_w"]).to(dev) for r in rgs]
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))

    def calls():
        for i in range(n):
            recv, slot_map = bufs[i % 2]
            plan.dispatch(xs[i], idx[i], sps[i % 2], recv, slot_map, stream=s)
            xs[i + 1].fill_(-3.0)  # sentinel, on the stream, right before the combine writes it
            plan.combine(recv, gate[i], slot_map, xs[i + 1], stream=s)

    if graph:
        with torch.cuda.stream(s):
            calls()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            calls()
        for _ in range(3):
            g.replay()
    else:
        with torch.cuda.stream(s):
            for _ in range(3):
                calls()
    torch.cuda.synchronize()
    for i in range(n):
        xh = P.bits(xs[i])
        ref = oracle.run_all(w.R, w.E, xh, rgs[i]["topk_idx"], rgs[i]["gate_w"], w.window_mode, w.window_rows)
        np.testing.assert_array_equal(P.bits(xs[i + 1]), ref["out"], err_msg=f"call {i}")
    recv, slot_map = bufs[(n - 1) % 2]
    sm = slot_map.cpu().numpy()
    rb = P.bits(recv)
    xl = P.bits(xs[n - 1])
    for s_ in range(w.R):
        for t in range(0, w.T, max(1, w.T // 64)):
            for j in range(w.k):
                if sm[s_, t, j] >= 0:
                    np.testing.assert_array_equal(rb[sm[s_, t, j]], xl[s_, t])
    assert plan.read_status() == 0
    plan.close()


def test_plans_with_different_shapes_coexist():
    # Kernel attributes are per kernel, not per plan: a plan made later with a
    # small row must not break an earlier plan with a large one.
    big = W.WORKLOADS[5].scaled(T=200, H=7168)
    small = _uniform(2, 4, 64, 8, 1)
    xb = W.make_x(big, 0, device=P.device())
    rgb = W.make_routing_gate(big, 0)
    gbig = P.gpu_run(big, xb, rgb["topk_idx"], rgb["gate_w"])
    P.full_parity(small)
    P.full_parity(big, x=xb, idx=rgb["topk_idx"], gate=rgb["gate_w"])
    P.gpu_run(big, xb, rgb["topk_idx"], rgb["gate_w"], plan=gbig["plan"])


# ---------------------------------------------------------------------------
# padded baseline (worst-case segments, fixed-size exchange)
# ---------------------------------------------------------------------------
def _padded(w):
    import dataclasses

    return dataclasses.replace(w, window_mode="padded", window_rows=0, name=w.name + "-padded")


@pytest.mark.parametrize("wid,T,H", [(1, None, None), (2, 1100, 264), (3, 300, 136), (4, 700, 72), (5, 40, 64)])
def test_padded_parity_and_same_output_as_dynamic(wid, T, H):
    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    import dataclasses

    w = dataclasses.replace(w, window_mode="packed", window_rows=0)
    x = W.make_x(w, 0, device=P.device())
    rg = W.make_routing_gate(w, 0)
    dyn = P.full_parity(w, x=x, idx=rg["topk_idx"], gate=rg["gate_w"])
    pad = P.full_parity(_padded(w), x=x, idx=rg["topk_idx"], gate=rg["gate_w"])
    np.testing.assert_array_equal(pad["out"], dyn["out"])
    # same counts; padded offsets are the fixed segment starts
    for key in ("send_counts", "send_offsets", "recv_counts", "recv_expert_counts", "recv_total"):
        np.testing.assert_array_equal(pad["splits"][key], dyn["splits"][key])
    assert pad["splits"]["window_base"].tolist() == [d * w.R * w.T * w.k for d in range(w.R)]


@pytest.mark.parametrize("flags", [1, 2, 3], ids=["lsu", "tiled", "tiled-lsu"])
def test_padded_variants(flags):
    P.full_parity(_padded(W.WORKLOADS[4].scaled(T=1500, H=136)), flags=flags)
    P.full_parity(_padded(W.WORKLOADS[2].scaled(T=300, H=520)), flags=flags)


def test_padded_edge_cases():
    import combine_device_resident_gb300 as A

    w = _padded(_uniform(4, 8, 900, 24, 1))
    idx = np.full((w.R, w.T, 1), 3, np.int32)  # the worst case itself: every token to one expert
    g = P.full_parity(w, idx=idx, gate=np.ones_like(idx, np.float32))
    assert g["splits"]["recv_total"].tolist() == [0, w.R * w.T, 0, 0]
    rg = W.make_routing_gate(w, 1)
    bad = rg["topk_idx"].copy()
    bad[1, 5, 0] = -1
    g = P.full_parity(w, idx=bad, gate=rg["gate_w"])
    assert g["status"] & A.DEV_BAD_EXPERT


def test_padded_plan_rejects_dynamic_calls():
    import torch
    import combine_device_resident_gb300 as A

    w = _padded(_uniform(2, 4, 16, 8, 1))
    plan = A.Plan(w.R, w.E, w.T, w.H, w.k, "padded", device=P.device())
    x = W.make_x(w, 0, device=P.device())
    idx = torch.zeros((w.R, w.T, 1), dtype=torch.int32, device=P.device())
    recv, sm, out = plan.new_buffers()
    with pytest.raises(A.A2avError, match="padded"):
        plan.dispatch(x, idx, plan.new_splits(), recv, sm)


# ---------------------------------------------------------------------------
# variable batches: per-rank active token counts read from device memory
# ---------------------------------------------------------------------------
def _counts(w, seed):
    rng = np.random.default_rng(seed)
    nt = rng.integers(0, w.T + 1, size=w.R).astype(np.int32)
    nt[0] = w.T      # a full rank
    nt[-1] = 0       # an idle rank
    return nt


# (3, 256, 1032) and (4, 128, 520): few-token calls with rows split into
# pieces (the batched-metadata combine and the pack's early launch).
@pytest.mark.parametrize("wid,T,H", [(1, None, None), (2, 1000, 136), (3, 256, 72), (4, 2100, 40), (5, 300, 64),
                                     (3, 256, 1032), (4, 128, 520)])
def test_active_token_counts(wid, T, H):
    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    g = P.full_parity(w, num_tokens=_counts(w, wid))
    assert g["status"] == 0


@pytest.mark.parametrize("variant", [dict(flags=1), dict(flags=2), dict(flags=4), dict(flags=7)],
                         ids=["lsu", "tiled", "tma-combine", "all-variants"])
def test_active_token_counts_variants(variant):
    w = W.WORKLOADS[4].scaled(T=1500, H=136)
    P.full_parity(w, num_tokens=_counts(w, 3), **variant)
    w = W.WORKLOADS[2].scaled(T=600, H=264)
    P.full_parity(w, num_tokens=_counts(w, 4), **variant)


def test_active_token_counts_padded():
    w = _padded(W.WORKLOADS[4].scaled(T=700, H=72))
    P.full_parity(w, num_tokens=_counts(w, 5))


def test_active_token_counts_clamped():
    w = W.WORKLOADS[2].scaled(T=300, H=24)
    P.full_parity(w, num_tokens=np.array([-5, 400, 0, 300, 1, 299, 150, 10**6], np.int32))


def test_graph_replays_with_changing_counts_and_double_buffered_arenas():
    # One graph per receive arena (double buffering: consecutive steps never
    # share a receive buffer); between replays the routing, the gates and the
    # per-rank token counts change in device memory.  Every replay matches the
    # oracle.
    import torch
    from combine_device_resident_gb300 import Plan

    w = W.WORKLOADS[4].scaled(T=1200, H=72)
    dev = P.device()
    plan = Plan(w.R, w.E, w.T, w.H, w.k, device=dev)
    nt_t = torch.full((w.R,), w.T, dtype=torch.int32, device=dev)
    plan.set_active_tokens(nt_t)
    x = W.make_x(w, 0, device=dev)
    idx_t = torch.zeros((w.R, w.T, w.k), dtype=torch.int32, device=dev)
    gate_t = torch.zeros((w.R, w.T, w.k), dtype=torch.float32, device=dev)
    arenas = []
    for _ in range(2):
        recv, slot_map, out = plan.new_buffers()
        arenas.append((recv, slot_map, out, plan.new_splits()))
    rg = W.make_routing_gate(w, 7)
    idx_t.copy_(torch.from_numpy(rg["topk_idx"]))
    gate_t.copy_(torch.from_numpy(rg["gate_w"]))
    graphs = []
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for recv, slot_map, out, sp in arenas:  # warm-up outside capture
            plan.dispatch(x, idx_t, sp, recv, slot_map)
            plan.combine(recv, gate_t, slot_map, out)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize()
    for recv, slot_map, out, sp in arenas:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.dispatch(x, idx_t, sp, recv, slot_map)
            plan.combine(recv, gate_t, slot_map, out)
        graphs.append(g)
    xh = P.bits(x)
    for step in range(6):
        rg = W.make_routing_gate(w, 100 + step)
        nt = _counts(w, 200 + step)
        idx_t.copy_(torch.from_numpy(rg["topk_idx"]))
        gate_t.copy_(torch.from_numpy(rg["gate_w"]))
        nt_t.copy_(torch.from_numpy(nt))
        recv, slot_map, out, sp = arenas[step % 2]
        out.fill_(3.0)
        graphs[step % 2].replay()
        torch.cuda.synchronize()
        ref = oracle.run_all(w.R, w.E, xh, rg["topk_idx"], rg["gate_w"], num_tokens=nt)
        P.check_splits(sp.to_numpy(), ref["splits"])
        np.testing.assert_array_equal(slot_map.cpu().numpy(), ref["slot_map"])
        ob = P.bits(out)
        for s_ in range(w.R):
            assert ulp_diff(ob[s_, :nt[s_]], ref["out"][s_, :nt[s_]]).max(initial=0) <= P.COMBINE_ULP_TOL
    assert plan.read_status() == 0


# ---------------------------------------------------------------------------
# the router in front of the dispatch
# ---------------------------------------------------------------------------
def _gate_bound(logits64, idx):
    """Relative error bound of the fp32 gates against the fp64 reference:
    (2*max|l_j - l_0| + k + 8) * 2^-24 (rounded differences, expf within 2 ulp,
    k - 1 rounded sums, one rounded division)."""
    sel = np.take_along_axis(logits64, idx.astype(np.int64), axis=-1)
    dmax = np.abs(sel - sel[..., :1]).max(axis=-1, keepdims=True)
    return (2 * dmax + idx.shape[-1] + 8) * 2.0 ** -24


@pytest.mark.parametrize("R,T,E,k", [(2, 300, 4, 1), (8, 512, 16, 1), (16, 257, 128, 2), (4, 130, 256, 8),
                                     (2, 40, 2048, 32), (3, 33, 37 * 3, 5)])
def test_router_matches_oracle(R, T, E, k):
    import torch
    from combine_device_resident_gb300 import Plan

    dev = P.device()
    w = W.Workload("router", R=R, E=E, T=T, H=8, k=k)
    logits = W.make_logits(w, R + E, device=dev)
    logits[0, 0] = 0.25                       # all equal: lowest ids first
    logits[0, 1, :3] = float("nan")           # NaN counts as -inf
    logits[-1, -1] = float("-inf")            # every logit -inf: equal gates
    logits[-1, 0, E // 2] = logits[-1, 0].max()  # a tie at the top
    if T > 3:
        logits[0, 2, :] = -1.0                     # +0 and -0 compare equal: lower id first
        logits[0, 2, E - 1] = 0.0
        logits[0, 2, 0] = -0.0
    plan = Plan(R, E, T, 8, k, device=dev)
    idx = torch.full((R, T, k), -9, dtype=torch.int32, device=dev)
    gate = torch.zeros((R, T, k), dtype=torch.float32, device=dev)
    plan.route(logits, idx, gate)
    torch.cuda.synchronize()
    lh = logits.cpu().numpy()
    ridx, rgate = oracle.route(lh, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    g = gate.cpu().numpy().astype(np.float64)
    l64 = np.where(np.isnan(lh), -np.inf, lh.astype(np.float64))
    finite = np.isfinite(np.take_along_axis(l64, ridx[..., :1].astype(np.int64), axis=-1))
    bound = np.where(finite, _gate_bound(np.where(np.isfinite(l64), l64, -1e30), ridx), 2.0 ** -24)
    assert (np.abs(g - rgate) <= bound * rgate + 1e-45).all()


@pytest.mark.parametrize("wid,T,H", [(2, 700, 136), (4, 600, 72), (5, 120, 64)])
def test_router_then_dispatch_and_combine(wid, T, H):
    # The whole step from logits: GPU router -> dispatch -> combine against the
    # oracle's router (fp64 gates rounded to fp32) -> dispatch -> combine.
    import torch
    from combine_device_resident_gb300 import Plan

    w = W.WORKLOADS[wid].scaled(T=T, H=H)
    dev = P.device()
    x = W.make_x(w, 0, device=dev)
    logits = W.make_logits(w, 0, device=dev)
    plan = Plan(w.R, w.E, w.T, w.H, w.k, device=dev)
    idx = torch.empty((w.R, w.T, w.k), dtype=torch.int32, device=dev)
    gate = torch.empty((w.R, w.T, w.k), dtype=torch.float32, device=dev)
    recv, slot_map, out = plan.new_buffers()
    sp = plan.new_splits()
    plan.route(logits, idx, gate)
    plan.dispatch(x, idx, sp, recv, slot_map)
    plan.combine(recv, gate, slot_map, out)
    torch.cuda.synchronize()
    ridx, rgate = oracle.route(logits.cpu().numpy(), w.k)
    ref = oracle.run_all(w.R, w.E, P.bits(x), ridx, rgate.astype(np.float32))
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    P.check_splits(sp.to_numpy(), ref["splits"])
    np.testing.assert_array_equal(slot_map.cpu().numpy(), ref["slot_map"])
    assert ulp_diff(P.bits(out), ref["out"]).max() <= P.COMBINE_ULP_TOL
    assert plan.read_status() == 0


def _adversarial_logits(w, seed, dev):
    """Seeded Gaussian logits with rows built to reach every path of the
    lane-per-token router: ties across the k-th place, 32 and 33 logits tied
    at the top (every one a candidate), infinities, NaN, -0 and denormals,
    and rows where a group of 16-byte units holds only -inf (the whole-share
    fallback)."""
    import torch

    lg = W.make_logits(w, seed, device=dev)
    E, T = w.E, w.T
    rows = [lg[0, t] for t in range(min(T, 9))]
    if len(rows) > 0:
        rows[0][:] = 3.0                               # all equal
    if len(rows) > 1:
        rows[1][: min(E, 32)] = 7.0                    # 32 tied at the top
    if len(rows) > 2:
        rows[2][: min(E, 33)] = 7.0                    # 33 tied at the top
    if len(rows) > 3:
        rows[3][::3] = 1.5                             # ties straddling the k-th place
    if len(rows) > 4:
        rows[4][E // 2] = float("inf")
        rows[4][E - 1] = float("inf")                  # two +inf
    if len(rows) > 5:
        rows[5][::2] = float("nan")                    # NaN counts as -inf
    if len(rows) > 6:
        rows[6][:] = float("-inf")
        rows[6][E - 1] = -0.0                          # one finite logit
    if len(rows) > 7:
        rows[7][:] = 1e-40                             # denormals and signed zeros
        rows[7][1::4] = -0.0
        rows[7][2::4] = 0.0
    if len(rows) > 8 and E >= 8:
        rows[8][: E // 2] = float("-inf")              # half the groups' units start -inf
    return lg


@pytest.mark.parametrize("R,T,E,k", [(2, 300, 4, 1), (8, 512, 16, 1), (16, 257, 128, 2), (4, 130, 256, 8),
                                     (4, 70, 8, 8), (2, 65, 12, 4), (2, 40, 512, 8), (1, 33, 64, 3),
                                     (4, 31, 256, 7), (2, 50, 256, 1), (2, 50, 256, 2), (2, 45, 40, 5),
                                     (2, 20, 640, 8), (2, 30, 320, 2), (4, 40, 1024, 4)])
def test_router_lane_kernel_equals_warp_kernel(R, T, E, k):
    # The lane-per-token router (the default on these shapes) against the
    # warp-per-token one (A2AV_FLAG_ROUTE_WARP) and against the oracle: same
    # ids, same gate bits.  A logits array 4 bytes off a 16-byte boundary
    # makes the default plan take the warp kernel too.
    import torch
    from combine_device_resident_gb300 import FLAG_ROUTE_WARP, Plan

    dev = P.device()
    w = W.Workload("router", R=R, E=E, T=T, H=8, k=k)
    logits = _adversarial_logits(w, 11 + E, dev)
    outs = []
    for flags, shift in ((0, 0), (FLAG_ROUTE_WARP, 0), (0, 1)):
        plan = Plan(R, E, T, 8, k, device=dev, flags=flags)
        if shift:
            buf = torch.empty(logits.numel() + 4, dtype=torch.float32, device=dev)
            lg = buf[shift:shift + logits.numel()].view(R, T, E)
            lg.copy_(logits)
            assert lg.data_ptr() % 16 != 0
        else:
            lg = logits
        idx = torch.full((R, T, k), -9, dtype=torch.int32, device=dev)
        gate = torch.zeros((R, T, k), dtype=torch.float32, device=dev)
        plan.route(lg, idx, gate)
        torch.cuda.synchronize()
        assert plan.read_status() == 0
        outs.append((idx.cpu().numpy(), gate.cpu().numpy().view(np.uint32)))
    for i in (1, 2):
        np.testing.assert_array_equal(outs[0][0], outs[i][0])
        np.testing.assert_array_equal(outs[0][1], outs[i][1])
    ridx, _ = oracle.route(logits.cpu().numpy(), k)
    np.testing.assert_array_equal(outs[0][0], ridx)


@pytest.mark.parametrize("wid,T", [(4, 100), (5, 37), (2, 45)])
def test_router_leaves_inactive_tokens_alone(wid, T):
    # T not a multiple of a warp task's tokens: tasks straddle ranks and mix
    # active and inactive tokens (top-2: 2 lanes per token, top-8 and top-1: 4)
    import torch
    from combine_device_resident_gb300 import Plan

    from combine_device_resident_gb300 import FLAG_ROUTE_WARP

    w = W.WORKLOADS[wid].scaled(T=T, H=8)
    dev = P.device()
    nt = _counts(w, 9)
    logits = W.make_logits(w, 1, device=dev)
    ridx, _ = oracle.route(logits.cpu().numpy(), w.k, num_tokens=nt)
    runs = []
    for flags in (0, FLAG_ROUTE_WARP):  # the lane kernel, then the warp kernel
        plan = Plan(w.R, w.E, w.T, w.H, w.k, device=dev, flags=flags)
        plan.set_active_tokens(torch.from_numpy(nt).to(dev))
        idx = torch.full((w.R, w.T, w.k), -9, dtype=torch.int32, device=dev)
        gate = torch.full((w.R, w.T, w.k), -1.0, dtype=torch.float32, device=dev)
        plan.route(logits, idx, gate)
        torch.cuda.synchronize()
        got, g = idx.cpu().numpy(), gate.cpu().numpy()
        for s_ in range(w.R):
            np.testing.assert_array_equal(got[s_, :nt[s_]], ridx[s_, :nt[s_]])
            assert (got[s_, nt[s_]:] == -9).all()
            assert (g[s_, nt[s_]:] == -1.0).all()
        runs.append(g.view(np.uint32))
    np.testing.assert_array_equal(runs[0], runs[1])


# ---------------------------------------------------------------------------
# expert-grouped receive order
# ---------------------------------------------------------------------------
def _by_expert(w, **kw):
    import dataclasses

    return dataclasses.replace(w, recv_order="expert", name=w.name + "-by-expert", **kw)


@pytest.mark.parametrize("wid,T,H", SCALED, ids=[f"w{s[0]}" for s in SCALED])
def test_expert_order_parity(wid, T, H):
    w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
    P.full_parity(_by_expert(w))


@pytest.mark.parametrize("flags", [1, 2, 3], ids=["lsu", "tiled", "tiled-lsu"])
def test_expert_order_variants(flags):
    for wid, T, H in [(1, None, None), (2, 1100, 264), (4, 900, 72), (5, 200, 64)]:
        w = W.WORKLOADS[wid] if T is None else W.WORKLOADS[wid].scaled(T=T, H=H)
        P.full_parity(_by_expert(w), flags=flags)


@pytest.mark.parametrize("wid,T,H", [(2, 1100, 264), (4, 700, 72), (5, 300, 64)])
def test_expert_order_same_output_and_contiguous_experts(wid, T, H):
    w = W.WORKLOADS[wid].scaled(T=T, H=H)
    x = W.make_x(w, 0, device=P.device())
    rg = W.make_routing_gate(w, 0)
    src = P.full_parity(w, x=x, idx=rg["topk_idx"], gate=rg["gate_w"])
    ex = P.full_parity(_by_expert(w), x=x, idx=rg["topk_idx"], gate=rg["gate_w"])
    np.testing.assert_array_equal(ex["out"], src["out"])
    for key in P.SPLIT_KEYS[:-1]:  # the counts are the same; only the places differ
        np.testing.assert_array_equal(ex["splits"][key], src["splits"][key], err_msg=key)
    # each local expert's rows are one contiguous block, starting where
    # recv_expert_offsets says
    sp, idx, epr = ex["splits"], rg["topk_idx"], w.E // w.R
    rel = ex["slot_map"] - sp["window_base"][idx // epr]
    reo, rec = sp["recv_expert_offsets"], sp["recv_expert_counts"]
    for d in range(w.R):
        for le in range(epr):
            rows = np.sort(rel[idx == d * epr + le])
            assert rows.size == rec[d, :, le].sum()
            np.testing.assert_array_equal(rows, reo[d, 0, le] + np.arange(rows.size))


def test_expert_order_fixed_windows_overflow_and_active_counts():
    import dataclasses

    w3 = W.WORKLOADS[3].scaled(T=700, H=72)
    # windows too small for the hot ranks: rows past the window are dropped
    # by their expert-order position, with the overflow bit
    g = P.full_parity(_by_expert(w3, window_rows=300))
    assert g["status"] & 2
    # per-rank active counts in expert order
    w5 = W.WORKLOADS[5].scaled(T=500, H=64)
    nt = np.array([(s * 37) % 501 for s in range(w5.R)], np.int32)
    P.full_parity(_by_expert(w5), num_tokens=nt)
    P.full_parity(_by_expert(dataclasses.replace(w3, window_rows=w3.R * w3.T)), num_tokens=nt[:w3.R], flags=2)


def test_expert_order_plan_requires_the_offsets_array():
    import torch

    import combine_device_resident_gb300 as A

    w = _by_expert(W.WORKLOADS[1])
    plan = A.Plan(w.R, w.E, w.T, w.H, w.k, device=P.device(), recv_order="expert")
    sp = plan.new_splits()
    sp.ptrs.recv_expert_offsets = None
    recv, slot_map, _ = plan.new_buffers()
    idx_t = torch.zeros((w.R, w.T, w.k), dtype=torch.int32, device=P.device())
    with pytest.raises(A.A2avError):
        plan.splits(idx_t, sp, slot_map)


def test_expert_offsets_are_optional_in_source_order():
    # asked for or not, everything else is the same; when asked for they are
    # the oracle's
    import torch

    for wid, T, H in [(2, 1100, 264), (5, 300, 64)]:
        w = W.WORKLOADS[wid].scaled(T=T, H=H)
        x = W.make_x(w, 0, device=P.device())
        rg = W.make_routing_gate(w, 0)
        a = P.full_parity(w, x=x, idx=rg["topk_idx"], gate=rg["gate_w"], expert_offsets=True)
        b = P.full_parity(w, x=x, idx=rg["topk_idx"], gate=rg["gate_w"], expert_offsets=False)
        assert "recv_expert_offsets" in a["splits"] and "recv_expert_offsets" not in b["splits"]
        np.testing.assert_array_equal(a["slot_map"], b["slot_map"])
        np.testing.assert_array_equal(a["out"], b["out"])
        for g in (a, b):
            g["plan"].close()
        torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# router fused into the histogram (a2av_route_splits)
# ---------------------------------------------------------------------------
def _routed_step(w, x, logits, fused, nt=None, flags=0):
    """fused: a2av_route_splits with the router inside the histogram kernel;
    else the router kernel and the splits kernel as two calls."""
    import torch
    from combine_device_resident_gb300 import FLAG_ROUTE_FUSED, Plan

    dev = P.device()
    plan = Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=dev,
                flags=flags | (FLAG_ROUTE_FUSED if fused else 0), recv_order=w.recv_order)
    if nt is not None:
        plan.set_active_tokens(torch.from_numpy(nt).to(dev))
    idx = torch.full((w.R, w.T, w.k), -9, dtype=torch.int32, device=dev)
    gate = torch.full((w.R, w.T, w.k), -1.0, dtype=torch.float32, device=dev)
    recv = torch.full((plan.arena_rows, w.H), -7.0, dtype=torch.bfloat16, device=dev)
    slot_map = torch.empty((w.R, w.T, w.k), dtype=torch.int32, device=dev)
    out = torch.full((w.R, w.T, w.H), 3.0, dtype=torch.bfloat16, device=dev)
    sp = plan.new_splits(expert_offsets=True)
    if fused:
        plan.route_splits(logits, idx, gate, sp, slot_map)
    else:
        plan.route(logits, idx, gate)
        plan.splits(idx, sp, slot_map)
    plan.pack(x, idx, sp, recv, slot_map)
    plan.combine(recv, gate, slot_map, out)
    torch.cuda.synchronize()
    res = {"idx": idx.cpu().numpy(), "gate": gate.cpu().numpy(), "splits": sp.to_numpy(),
           "slot_map": slot_map.cpu().numpy(), "recv": P.bits(recv), "out": P.bits(out),
           "status": plan.read_status()}
    plan.close()
    return res


ROUTED = [
    (4, 900, 72, 0, "fused: r16 E128 top-2, cluster-eligible plan"),
    (5, 300, 64, 0, "fused: r32 E256 top-8, tiled plan"),
    (2, 1100, 64, 0, "fused: r8 E16 top-1"),
    (4, 700, 72, 2, "fused, plan forced tiled"),
]


@pytest.mark.parametrize("wid,T,H,flags,_", ROUTED, ids=[r[4] for r in ROUTED])
def test_route_splits_equals_route_then_splits_and_oracle(wid, T, H, flags, _):
    w = W.WORKLOADS[wid].scaled(T=T, H=H)
    x = W.make_x(w, 0, device=P.device())
    logits = W.make_logits(w, 0, device=P.device())
    a = _routed_step(w, x, logits, fused=True, flags=flags)
    b = _routed_step(w, x, logits, fused=False, flags=flags)
    for key in ("idx", "gate", "slot_map", "out"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    for key in a["splits"]:
        np.testing.assert_array_equal(a["splits"][key], b["splits"][key], err_msg=key)
    rows = a["slot_map"][a["slot_map"] >= 0]
    np.testing.assert_array_equal(a["recv"][rows], b["recv"][rows])
    # against the oracle's router and path
    ridx, rgate = oracle.route(logits.cpu().numpy(), w.k)
    ref = oracle.run_all(w.R, w.E, P.bits(x), ridx, rgate.astype(np.float32))
    np.testing.assert_array_equal(a["idx"], ridx)
    P.check_splits(a["splits"], ref["splits"])
    np.testing.assert_array_equal(a["slot_map"], ref["slot_map"])
    assert ulp_diff(a["out"], ref["out"]).max() <= P.COMBINE_ULP_TOL
    assert a["status"] == 0


def test_route_splits_fallback_active_tokens_and_layouts():
    # not fusable (k = 3, or E > 256): the two kernels; fusable with active
    # counts, fixed windows and the expert-grouped order
    import dataclasses

    cases = [
        (W.Workload("k3", R=3, E=111, T=200, H=40, k=3), None),
        (W.Workload("e512", R=4, E=512, T=64, H=24, k=8), None),
        (W.WORKLOADS[5].scaled(T=300, H=40), "counts"),
        (dataclasses.replace(W.WORKLOADS[3].scaled(T=500, H=40), window_rows=400), None),
        (dataclasses.replace(W.WORKLOADS[5].scaled(T=200, H=40), recv_order="expert"), "counts"),
    ]
    for w, mode in cases:
        nt = np.array([(s_ * 37 + 11) % (w.T + 1) for s_ in range(w.R)], np.int32) if mode else None
        x = W.make_x(w, 0, device=P.device())
        logits = W.make_logits(w, 3, device=P.device())
        a = _routed_step(w, x, logits, fused=True, nt=nt)
        b = _routed_step(w, x, logits, fused=False, nt=nt)
        for key in ("idx", "gate", "slot_map", "out"):
            np.testing.assert_array_equal(a[key], b[key], err_msg=f"{w.name} {key}")
        for key in a["splits"]:
            np.testing.assert_array_equal(a["splits"][key], b["splits"][key], err_msg=f"{w.name} {key}")
        assert a["status"] == b["status"]
        ridx, rgate = oracle.route(logits.cpu().numpy(), w.k, num_tokens=nt)
        ref = oracle.run_all(w.R, w.E, P.bits(x), ridx, rgate.astype(np.float32), w.window_mode, w.window_rows,
                             num_tokens=nt, recv_order=w.recv_order)
        P.check_splits(a["splits"], ref["splits"])
        np.testing.assert_array_equal(a["slot_map"], ref["slot_map"], err_msg=w.name)
        assert a["status"] == ref["status"], w.name
        if nt is not None:  # tokens that take no part keep their idx/gate/out
            for s_ in range(w.R):
                assert (a["idx"][s_, nt[s_]:] == -9).all() and (a["gate"][s_, nt[s_]:] == -1.0).all()


# ---------------------------------------------------------------------------
# seeded random shapes x options, element by element against the oracle
# ---------------------------------------------------------------------------
def _random_case(i):
    rng = np.random.default_rng(1000 + i)
    R = int(rng.choice([1, 2, 3, 4, 8, 16]))
    epr = int(rng.choice([1, 2, 3, 8]))
    E = R * epr
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.choice([1, 2, 7, 64, 257, 300]))
    H = int(rng.choice([8, 16, 72, 136, 520]))
    routing = "zipf_distinct" if k > 1 else str(rng.choice(["uniform", "zipf"]))
    w = W.Workload(f"fuzz{i}", R=R, E=E, T=T, H=H, k=k, routing=routing, zipf_s=float(rng.choice([0.0, 1.1])),
                   gate="softmax" if k > 1 else "ones", expert=str(rng.choice(["identity", "scale"])),
                   recv_order=str(rng.choice(["source", "expert"])))
    if rng.random() < 0.3:
        import dataclasses
        w = dataclasses.replace(w, window_mode="fixed", window_rows=int(rng.integers(1, T * k * R + 2)))
    nt = rng.integers(0, T + 1, size=R).astype(np.int32) if rng.random() < 0.4 else None
    flags = int(rng.choice([0, 1, 2, 3, 4]))
    return w, nt, flags


@pytest.mark.parametrize("i", range(24))
def test_random_shapes_and_options(i):
    w, nt, flags = _random_case(i)
    P.full_parity(w, seed=i, num_tokens=nt, flags=flags)


def _random_router_case(i):
    rng = np.random.default_rng(2000 + i)
    R = int(rng.choice([1, 2, 3, 4, 8, 16]))
    E = R * int(rng.choice([1, 2, 4, 8, 16, 32, 64]))
    k = int(rng.integers(1, min(E, 8) + 1))  # 1..8: the lane kernel's range (other shapes fall back)
    T = int(rng.choice([1, 3, 17, 64, 129]))
    return R, E, k, T, rng


@pytest.mark.parametrize("i", range(16))
def test_random_router_cases(i):
    # seeded shapes, logits with random ties and special values, and random
    # active counts: the default router against the oracle's ids and the
    # warp-per-token kernel's ids and gate bits
    import torch
    from combine_device_resident_gb300 import FLAG_ROUTE_WARP, Plan

    R, E, k, T, rng = _random_router_case(i)
    dev = P.device()
    lg = rng.standard_normal((R, T, E)).astype(np.float32)
    lg = np.round(lg * 4) / 4  # coarse values: ties are common
    specials = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 1e-40], dtype=np.float32)
    mask = rng.random(lg.shape) < 0.05
    lg[mask] = rng.choice(specials, size=int(mask.sum()))
    nt = rng.integers(0, T + 1, size=R).astype(np.int32) if rng.random() < 0.5 else None
    logits = torch.from_numpy(lg).to(dev)
    outs = []
    for flags in (0, FLAG_ROUTE_WARP):
        plan = Plan(R, E, T, 8, k, device=dev, flags=flags)
        if nt is not None:
            plan.set_active_tokens(torch.from_numpy(nt).to(dev))
        idx = torch.full((R, T, k), -9, dtype=torch.int32, device=dev)
        gate = torch.full((R, T, k), -1.0, dtype=torch.float32, device=dev)
        plan.route(logits, idx, gate)
        torch.cuda.synchronize()
        assert plan.read_status() == 0
        outs.append((idx.cpu().numpy(), gate.cpu().numpy().view(np.uint32)))
        plan.close()
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
    ridx, _ = oracle.route(lg, k, num_tokens=nt)
    got = outs[0][0]
    if nt is None:
        np.testing.assert_array_equal(got, ridx)
    else:
        for s_ in range(R):
            np.testing.assert_array_equal(got[s_, :nt[s_]], ridx[s_, :nt[s_]])
            assert (got[s_, nt[s_]:] == -9).all()
