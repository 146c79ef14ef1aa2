"""Pins for the CPU oracle: it is checked against things other than itself.

* a hand-worked tiny example (derivation in the comments);
* an exhaustive brute force written as a *different* formulation: window d is
  a sort of every assignment routed to rank d by key (source, expert, token,
  slot), and every count/offset is read off those sorted lists;
* the invariants the method fixes: split counts sum to T*k, received counts
  are the transpose of the per-rank send counts (summed over the destination's
  experts), no padding (slot_map is a bijection onto the packed arena), and
  dispatch followed by combine with identity experts and unit weights gives
  k*x [NCCLX pages: P1 "Inference", P2 section 3.3];
* closed forms of the combine computed without any dispatch (torch / numpy
  float32 / fp64), and bf16 rounding against torch's own conversion;
* mutation checks: plausible mistakes planted in a *copy* of the oracle's C
  source must each make at least one of these pins fail.
"""
import itertools
import os
import re

import numpy as np
import pytest

import oracle
from tests.bf16util import bits_to_f32, f32_to_bits_torch, is_nan, ulp_diff

SPLIT_KEYS = ["send_counts", "send_offsets", "recv_counts", "recv_offsets",
              "recv_expert_counts", "recv_total", "window_base"]


# ----------------------------------------------------------------------------
# brute force: an independent formulation from sorted per-destination lists
# ----------------------------------------------------------------------------
def brute_force(R, E, idx, window_mode="packed", window_rows=0, recv_order="source"):
    idx = np.asarray(idx)
    _, T, k = idx.shape
    epr = E // R
    items = [(s, int(idx[s, t, j]), t, j) for s in range(R) for t in range(T) for j in range(k)]
    valid = [it for it in items if 0 <= it[1] < E]
    status = 0 if len(valid) == len(items) else oracle.BAD_EXPERT
    windows = [sorted(it for it in valid if it[1] // epr == d) for d in range(R)]
    # the order rows take inside a window: (source, expert, token, slot), or
    # (expert, source, token, slot) for the expert-grouped view
    order = (lambda it: it) if recv_order == "source" else (lambda it: (it[1], it[0], it[2], it[3]))
    placed = [sorted(w, key=order) for w in windows]
    per_src = [sorted((e, t, j) for (s2, e, t, j) in valid if s2 == s) for s in range(R)]
    out = {
        "send_counts": np.array([[sum(1 for it in per_src[s] if it[0] == e) for e in range(E)] for s in range(R)]),
        "send_offsets": np.array([[next((i for i, it in enumerate(per_src[s]) if it[0] >= e), len(per_src[s]))
                                   for e in range(E)] for s in range(R)]),
        "recv_counts": np.array([[sum(1 for it in windows[d] if it[0] == s) for s in range(R)] for d in range(R)]),
        "recv_offsets": np.array([[next((i for i, it in enumerate(windows[d]) if it[0] >= s), len(windows[d]))
                                   for s in range(R)] for d in range(R)]),
        "recv_expert_counts": np.array([[[sum(1 for it in windows[d] if it[0] == s and it[1] == d * epr + le)
                                          for le in range(epr)] for s in range(R)] for d in range(R)]),
        "recv_total": np.array([len(w) for w in windows]),
    }
    if window_mode == "fixed":
        out["window_base"] = np.array([d * window_rows for d in range(R)])
        if any(len(w) > window_rows for w in windows):
            status |= oracle.WINDOW_OVERFLOW
    elif window_mode == "padded":
        # worst case: every (source, destination) pair owns T*k rows
        out["window_base"] = np.array([d * R * T * k for d in range(R)])
        out["recv_offsets"] = np.array([[src * T * k for src in range(R)] for _ in range(R)])
    else:
        out["window_base"] = np.array([sum(len(w) for w in windows[:d]) for d in range(R)])
    # first row of each (source, local expert) block: the rows placed before it
    if window_mode == "padded":
        out["recv_expert_offsets"] = np.array(
            [[[s * T * k + sum(1 for it in windows[d] if it[0] == s and it[1] < d * epr + le)
               for le in range(epr)] for s in range(R)] for d in range(R)])
    else:
        out["recv_expert_offsets"] = np.array(
            [[[sum(1 for it in placed[d] if order(it)[:2] < order((s, d * epr + le, 0, 0))[:2])
               for le in range(epr)] for s in range(R)] for d in range(R)])
    slot = -np.ones((R, T, k), dtype=np.int64)
    for d, w in enumerate(placed):
        for pos, (s, e, t, j) in enumerate(w):
            if window_mode == "fixed" and pos >= window_rows:
                continue
            if window_mode == "padded":
                # place inside source s's own segment of window d
                pos = sum(1 for it in w[:pos] if it[0] == s)
                slot[s, t, j] = d * R * T * k + s * T * k + pos
                continue
            slot[s, t, j] = out["window_base"][d] + pos
    out["slot_map"] = slot
    out["status"] = status
    return out


def check_against_brute(R, E, idx, window_mode="packed", window_rows=0, recv_order="source"):
    bf = brute_force(R, E, idx, window_mode, window_rows, recv_order)
    sp = oracle.splits(R, E, idx, window_mode, window_rows, recv_order=recv_order)
    for key in SPLIT_KEYS + ["recv_expert_offsets"]:
        np.testing.assert_array_equal(sp[key], bf[key].reshape(sp[key].shape), err_msg=key)
    sm, st = oracle.slot_map(R, E, idx, sp, window_mode, window_rows, recv_order=recv_order)
    np.testing.assert_array_equal(sm, bf["slot_map"], err_msg="slot_map")
    assert (sp["status"] | st) == bf["status"]
    return sp, sm


def check_dispatch_against_brute(R, E, idx, window_mode="packed", window_rows=0, recv_order="source", H=3):
    """The dispatch (payload moved the literal way) lands every row where the
    brute force puts it, carrying its token's bits."""
    bf = brute_force(R, E, idx, window_mode, window_rows, recv_order)
    T = idx.shape[1]
    x = (np.arange(R * T * H, dtype=np.uint32).reshape(R, T, H) * 7 + 0x3F80).astype(np.uint16)
    sp = oracle.splits(R, E, idx, window_mode, window_rows, recv_order=recv_order)
    recv, sm, st = oracle.dispatch(R, E, x, idx, sp, window_mode, window_rows, recv_order=recv_order)
    np.testing.assert_array_equal(sm, bf["slot_map"], err_msg="dispatch slot_map")
    for s_ in range(R):
        for t in range(T):
            for j in range(idx.shape[2]):
                if sm[s_, t, j] >= 0:
                    np.testing.assert_array_equal(recv[sm[s_, t, j]], x[s_, t])
    assert (sp["status"] | st) == bf["status"]


# ----------------------------------------------------------------------------
def test_hand_worked_example():
    # R=2 ranks, E=4 experts: experts {0,1} on rank 0, {2,3} on rank 1; T=3, k=1.
    # rank 0 routes tokens to experts [3, 0, 3]; rank 1 to [1, 2, 1].
    # send_counts: rank0 e0:1 e3:2 -> [1,0,0,2]; rank1 e1:2 e2:1 -> [0,2,1,0]
    # send_offsets (exclusive over e): [0,1,1,1] and [0,0,2,3]
    # recv_counts[d][s]: d0 gets e0+e1: s0 1, s1 2; d1 gets e2+e3: s0 2, s1 1
    # recv_offsets (exclusive over s): d0 [0,1], d1 [0,2]; totals [3,3];
    # packed window bases [0,3].
    # Window 0 in (source, expert, token) order: (s0,e0,t1) (s1,e1,t0) (s1,e1,t2) -> rows 0,1,2
    # Window 1: (s0,e3,t0) (s0,e3,t2) (s1,e2,t1) -> rows 3,4,5
    idx = np.array([[[3], [0], [3]], [[1], [2], [1]]], np.int32)
    sp = oracle.splits(2, 4, idx)
    assert sp["send_counts"].tolist() == [[1, 0, 0, 2], [0, 2, 1, 0]]
    assert sp["send_offsets"].tolist() == [[0, 1, 1, 1], [0, 0, 2, 3]]
    assert sp["recv_counts"].tolist() == [[1, 2], [2, 1]]
    assert sp["recv_offsets"].tolist() == [[0, 1], [0, 2]]
    assert sp["recv_expert_counts"].tolist() == [[[1, 0], [0, 2]], [[0, 2], [1, 0]]]
    assert sp["recv_total"].tolist() == [3, 3]
    assert sp["window_base"].tolist() == [0, 3]
    sm, st = oracle.slot_map(2, 4, idx, sp)
    assert st == 0
    assert sm[..., 0].tolist() == [[3, 0, 4], [1, 5, 2]]
    # payload: rows carry the token they came from
    x = np.arange(2 * 3 * 2, dtype=np.uint16).reshape(2, 3, 2) + 0x3F00
    recv, sm2, st2 = oracle.dispatch(2, 4, x, idx, sp)
    np.testing.assert_array_equal(sm2, sm)
    assert recv.tolist() == [x[0, 1].tolist(), x[1, 0].tolist(), x[1, 2].tolist(),
                             x[0, 0].tolist(), x[0, 2].tolist(), x[1, 1].tolist()]


def test_hand_worked_example_expert_order():
    # The routing of the example above.  Window 1 holds experts 2 and 3; in
    # the expert-grouped view expert 2's rows come first: (s1,e2,t1) -> row 3,
    # then expert 3's: (s0,e3,t0) -> 4, (s0,e3,t2) -> 5.  Window 0 is the same
    # in both orders: (s0,e0,t1) -> 0, (s1,e1,t0) -> 1, (s1,e1,t2) -> 2.
    # recv_expert_offsets[d][s][le], expert order: window 0: expert 0 starts
    # at 0 (s0 there, s1 after s0's 1 row), expert 1 at 1 (s0: 1, s1: 1 + 0);
    # window 1: expert 2 at 0 (s0: 0, s1: 0), expert 3 at 1 (s0: 1, s1: 1+2).
    # Source order: window 1's segments start at 0 (s0) and 2 (s1); s0 has no
    # expert-2 rows, so its expert-3 block also starts at 0; s1's expert-3
    # block starts after its one expert-2 row, at 3.
    idx = np.array([[[3], [0], [3]], [[1], [2], [1]]], np.int32)
    ex = oracle.splits(2, 4, idx, recv_order="expert")
    src = oracle.splits(2, 4, idx)
    for key in SPLIT_KEYS:
        np.testing.assert_array_equal(ex[key], src[key], err_msg=key)
    assert ex["recv_expert_offsets"].tolist() == [[[0, 1], [1, 1]], [[0, 1], [0, 3]]]
    assert src["recv_expert_offsets"].tolist() == [[[0, 1], [1, 1]], [[0, 0], [2, 3]]]
    sm, st = oracle.slot_map(2, 4, idx, ex, recv_order="expert")
    assert st == 0
    assert sm[..., 0].tolist() == [[4, 0, 5], [1, 3, 2]]
    x = np.arange(2 * 3 * 2, dtype=np.uint16).reshape(2, 3, 2) + 0x3F00
    recv, sm2, st2 = oracle.dispatch(2, 4, x, idx, ex, recv_order="expert")
    np.testing.assert_array_equal(sm2, sm)
    assert recv.tolist() == [x[0, 1].tolist(), x[1, 0].tolist(), x[1, 2].tolist(),
                             x[1, 1].tolist(), x[0, 0].tolist(), x[0, 2].tolist()]


@pytest.mark.parametrize("order", ["source", "expert"])
def test_exhaustive_expert_order_r2_e4(order):
    R, E, k, T = 2, 4, 1, 3
    for combo in itertools.product(range(E), repeat=R * T * k):
        idx = np.array(combo, np.int32).reshape(R, T, k)
        check_against_brute(R, E, idx, recv_order=order)
    pairs = [p for p in itertools.product(range(E), repeat=2) if p[0] != p[1]]
    for combo in itertools.product(pairs, repeat=R):
        check_dispatch_against_brute(R, E, np.array(combo, np.int32).reshape(R, 1, 2), recv_order=order)


def test_expert_order_random_fixed_and_active_against_brute():
    rng = np.random.default_rng(31)
    for R, E, T, k in [(1, 3, 5, 2), (3, 6, 7, 2), (4, 8, 9, 3), (4, 16, 20, 4)]:
        for _ in range(8):
            idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
            check_against_brute(R, E, idx, recv_order="expert")
            check_dispatch_against_brute(R, E, idx, recv_order="expert")
            for W_ in (R * T * k, 7, 1):
                check_against_brute(R, E, idx, "fixed", W_, recv_order="expert")
                check_dispatch_against_brute(R, E, idx, "fixed", W_, recv_order="expert")
            # tokens past num_tokens[s] take no part, in this order too
            nt = rng.integers(0, T + 1, size=R).astype(np.int32)
            masked = idx.copy()
            for s_ in range(R):
                masked[s_, nt[s_]:] = -1
            bf = brute_force(R, E, masked, recv_order="expert")
            sp = oracle.splits(R, E, idx, num_tokens=nt, recv_order="expert")
            np.testing.assert_array_equal(sp["recv_expert_offsets"], bf["recv_expert_offsets"])
            sm, st = oracle.slot_map(R, E, idx, sp, num_tokens=nt, recv_order="expert")
            np.testing.assert_array_equal(sm, bf["slot_map"])
            assert st == 0
    with pytest.raises(ValueError):
        oracle.splits(2, 4, np.zeros((2, 1, 1), np.int32), "padded", recv_order="expert")


def test_expert_order_blocks_tile_each_window():
    # each local expert's rows are one contiguous block, its sources back to
    # back, and the blocks tile [0, recv_total[d]) in expert order
    rng = np.random.default_rng(3)
    R, E, T, k = 4, 16, 40, 4
    idx = np.stack([np.stack([rng.choice(E, k, replace=False) for _ in range(T)]) for _ in range(R)]).astype(np.int32)
    sp = oracle.splits(R, E, idx, recv_order="expert")
    reo, rec = sp["recv_expert_offsets"], sp["recv_expert_counts"]
    sm, _ = oracle.slot_map(R, E, idx, sp, recv_order="expert")
    epr = E // R
    for d in range(R):
        nxt = 0
        for le in range(epr):
            for s_ in range(R):
                assert reo[d, s_, le] == nxt
                nxt += rec[d, s_, le]
        assert nxt == sp["recv_total"][d]
    rel = sm - sp["window_base"][idx // epr]
    le_of = idx % epr
    for d in range(R):
        for le in range(epr):
            rows = np.sort(rel[(idx // epr == d) & (le_of == le)])
            lo = reo[d, 0, le]
            np.testing.assert_array_equal(rows, np.arange(lo, lo + rows.size))


@pytest.mark.parametrize("T", [1, 2, 3])
def test_exhaustive_top1_r2_e4(T):
    R, E, k = 2, 4, 1
    for combo in itertools.product(range(E), repeat=R * T * k):
        idx = np.array(combo, np.int32).reshape(R, T, k)
        check_against_brute(R, E, idx)


def test_exhaustive_top2_distinct_r2_e4():
    R, E, k, T = 2, 4, 2, 1
    pairs = [p for p in itertools.product(range(E), repeat=2) if p[0] != p[1]]
    for combo in itertools.product(pairs, repeat=R * T):
        idx = np.array(combo, np.int32).reshape(R, T, k)
        check_against_brute(R, E, idx)


def test_exhaustive_top2_with_duplicates_r2_e4():
    # duplicates inside one token are allowed and ordered by slot j
    R, E, k, T = 2, 4, 2, 1
    for combo in itertools.product(range(E), repeat=R * T * k):
        idx = np.array(combo, np.int32).reshape(R, T, k)
        check_against_brute(R, E, idx)


@pytest.mark.parametrize("R,E,T,k", [(1, 3, 5, 2), (2, 2, 4, 1), (3, 6, 7, 2), (4, 8, 9, 3), (4, 16, 33, 4)])
def test_random_against_brute(R, E, T, k):
    rng = np.random.default_rng(R * 1000 + E * 10 + k)
    for _ in range(20):
        idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
        check_against_brute(R, E, idx)


def test_fixed_windows_and_overflow_against_brute():
    rng = np.random.default_rng(7)
    R, E, T, k = 3, 6, 6, 2
    for W in (R * T * k, 8, 5, 1, 0):
        for _ in range(10):
            idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
            check_against_brute(R, E, idx, "fixed", W)
    # all tokens to one expert with a window of T*k rows must overflow
    idx = np.zeros((R, T, k), np.int32)
    sp = oracle.splits(R, E, idx, "fixed", T * k)
    assert sp["status"] & oracle.WINDOW_OVERFLOW
    sm, st = oracle.slot_map(R, E, idx, sp, "fixed", T * k)
    assert st & oracle.WINDOW_OVERFLOW
    assert (sm[0] >= 0).all() and (sm[1:] == -1).all()


def test_padded_layout_against_brute():
    rng = np.random.default_rng(13)
    for R, E, T, k in [(2, 4, 3, 1), (3, 6, 5, 2), (4, 8, 7, 3)]:
        for _ in range(15):
            idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
            check_against_brute(R, E, idx, "padded")
    # exhaustive on the tiny case
    for combo in itertools.product(range(4), repeat=4):
        check_against_brute(2, 4, np.array(combo, np.int32).reshape(2, 2, 1), "padded")


def test_padded_and_packed_place_the_same_rows_in_the_same_order():
    # the two layouts differ only by where each (source, destination) segment
    # starts; inside a segment the order is the same
    rng = np.random.default_rng(5)
    R, E, T, k = 4, 8, 9, 2
    idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
    a = oracle.splits(R, E, idx)
    b = oracle.splits(R, E, idx, "padded")
    sa, _ = oracle.slot_map(R, E, idx, a)
    sb, _ = oracle.slot_map(R, E, idx, b, "padded")
    d = idx // (E // R)
    src = np.arange(R)[:, None, None]
    rel_a = sa - a["window_base"][d] - a["recv_offsets"][d, src]
    rel_b = sb - b["window_base"][d] - b["recv_offsets"][d, src]
    np.testing.assert_array_equal(rel_a, rel_b)
    assert (rel_b >= 0).all() and (rel_b < T * k).all()
    for key in ("send_counts", "send_offsets", "recv_counts", "recv_expert_counts", "recv_total"):
        np.testing.assert_array_equal(a[key], b[key])


def test_active_token_counts_equal_truncated_routing():
    # Tokens past num_tokens[s] take no part: the counts and rows equal those
    # of the same routing with those tokens' expert ids removed, and their
    # slots are -1 without a bad-expert status.
    rng = np.random.default_rng(21)
    for R, E, T, k in [(2, 4, 6, 1), (3, 6, 7, 2), (4, 16, 12, 3)]:
        for _ in range(10):
            idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
            nt = rng.integers(0, T + 1, size=R).astype(np.int32)
            masked = idx.copy()
            for s_ in range(R):
                masked[s_, nt[s_]:] = -1
            for mode in ("packed", "padded"):
                bf = brute_force(R, E, masked, mode)
                sp = oracle.splits(R, E, idx, mode, num_tokens=nt)
                for key in SPLIT_KEYS:
                    np.testing.assert_array_equal(sp[key], bf[key].reshape(sp[key].shape), err_msg=key)
                sm, st = oracle.slot_map(R, E, idx, sp, mode, num_tokens=nt)
                np.testing.assert_array_equal(sm, bf["slot_map"])
                assert sp["status"] == 0 and st == 0
    # clamping: negative counts take nothing, counts past T take everything
    idx = rng.integers(0, 4, size=(2, 5, 1), dtype=np.int32)
    a = oracle.splits(2, 4, idx, num_tokens=np.array([-3, 99], np.int32))
    assert a["send_counts"][0].sum() == 0 and a["send_counts"][1].sum() == 5


def test_active_token_counts_combine_only_active_tokens():
    import workloads as W

    w = W.Workload("t", R=3, E=6, T=9, H=16, k=2, routing="zipf_distinct", zipf_s=1.0, gate="softmax")
    x = W.bf16_bits(W.make_x(w, 2))
    rg = W.make_routing_gate(w, 2)
    nt = np.array([9, 4, 0], np.int32)
    full = oracle.run_all(w.R, w.E, x, rg["topk_idx"], rg["gate_w"])
    part = oracle.run_all(w.R, w.E, x, rg["topk_idx"], rg["gate_w"], num_tokens=nt)
    for s_ in range(w.R):
        np.testing.assert_array_equal(part["out"][s_, :nt[s_]], full["out"][s_, :nt[s_]])
        assert (part["out"][s_, nt[s_]:] == 0).all()
        assert (part["slot_map"][s_, nt[s_]:] == -1).all()
    assert part["splits"]["recv_total"].sum() == nt.sum() * w.k


def test_router_against_numpy_sort_and_softmax():
    # selection = a lexicographic sort by (logit descending, id ascending),
    # gates = the float64 softmax of the selected logits
    from scipy.special import softmax

    rng = np.random.default_rng(31)
    for R, T, E, k in [(2, 5, 4, 1), (3, 7, 16, 2), (2, 9, 256, 8), (1, 3, 64, 32)]:
        logits = rng.standard_normal((R, T, E)).astype(np.float32)
        logits[0, 0, :] = 0.5                      # all equal: ids in order
        logits[-1, -1, 3 % E] = np.nan             # NaN counts as -inf
        logits[-1, 1 % T, :2] = np.float32(-np.inf)
        idx, gate = oracle.route(logits, k)
        for s_ in range(R):
            for t in range(T):
                v = np.where(np.isnan(logits[s_, t]), -np.inf, logits[s_, t].astype(np.float64))
                order = np.lexsort((np.arange(E), -v))[:k]
                np.testing.assert_array_equal(idx[s_, t], order)
                np.testing.assert_allclose(gate[s_, t], softmax(v[order]), rtol=1e-12, atol=0)
    # every selected logit -inf: equal weights
    logits = np.full((1, 1, 8), -np.inf, np.float32)
    idx, gate = oracle.route(logits, 3)
    assert idx[0, 0].tolist() == [0, 1, 2] and np.allclose(gate, 1 / 3)
    # inactive tokens untouched
    logits = rng.standard_normal((2, 4, 8)).astype(np.float32)
    idx, gate = oracle.route(logits, 2, num_tokens=np.array([1, 0], np.int32))
    assert (idx[0, 1:] == -1).all() and (idx[1] == -1).all() and (idx[0, 0] >= 0).all()


def test_bad_expert_ids_are_dropped():
    R, E, T, k = 2, 4, 4, 2
    rng = np.random.default_rng(3)
    idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
    idx[0, 1, 0] = -1
    idx[1, 3, 1] = E
    sp, sm = check_against_brute(R, E, idx)
    assert sp["status"] & oracle.BAD_EXPERT
    assert sm[0, 1, 0] == -1 and sm[1, 3, 1] == -1
    assert sp["send_counts"].sum() == R * T * k - 2


# ----------------------------------------------------------------------------
# invariants on the synthetic workloads (full routing, no payload)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_invariants_on_workloads(wid):
    import workloads as W

    w = W.WORKLOADS[wid]
    idx = W.make_routing_gate(w)["topk_idx"]
    sp = oracle.splits(w.R, w.E, idx, w.window_mode, w.window_rows)
    assert sp["status"] == 0
    T, k, R, E = w.T, w.k, w.R, w.E
    epr = E // R
    # split counts sum to T*k on every rank
    assert (sp["send_counts"].sum(axis=1) == T * k).all()
    # per-rank counts equal a direct bincount of that rank's routing
    for s in range(R):
        np.testing.assert_array_equal(sp["send_counts"][s], np.bincount(idx[s].ravel(), minlength=E))
    # received counts: transpose of send counts summed over each rank's experts
    np.testing.assert_array_equal(sp["recv_counts"], sp["send_counts"].reshape(R, R, epr).sum(-1).T)
    assert sp["recv_total"].sum() == R * T * k
    sm, st = oracle.slot_map(R, E, idx, sp, w.window_mode, w.window_rows)
    assert st == 0
    if w.window_mode == "packed":
        # no padding: a bijection onto [0, R*T*k)
        assert np.array_equal(np.sort(sm.ravel()), np.arange(R * T * k))
    else:
        rel = sm - sp["window_base"][idx // epr]
        assert (rel >= 0).all() and (rel < w.window_rows).all()
        for d in range(R):
            rows = np.sort(rel[(idx // epr) == d])
            assert np.array_equal(rows, np.arange(sp["recv_total"][d]))


def test_workload_routing_laws():
    import workloads as W

    # top-k experts are distinct where the workload asks for it
    for wid in (4, 5):
        w = W.WORKLOADS[wid]
        idx = W.make_routing_gate(w)["topk_idx"].reshape(-1, w.k)
        srt = np.sort(idx, axis=1)
        assert (np.diff(srt, axis=1) > 0).all()
    # the hot expert of workload 5 holds close to the 1/k cap of assignments,
    # and four ranks receive nothing
    w = W.WORKLOADS[5]
    idx = W.make_routing_gate(w)["topk_idx"]
    share0 = (idx == 0).mean()
    assert 0.11 < share0 <= 1.0 / w.k
    per_rank = np.bincount(idx.ravel() // (w.E // w.R), minlength=w.R)
    assert (per_rank == 0).sum() == 4 and per_rank[0] > 0
    # workload 3 leaves some experts empty
    w = W.WORKLOADS[3]
    idx = W.make_routing_gate(w)["topk_idx"]
    assert (np.bincount(idx.ravel(), minlength=w.E) == 0).any()


# ----------------------------------------------------------------------------
# dispatch payload and the combine closed forms
# ----------------------------------------------------------------------------
def _small(wid, T, H, seed=0):
    import workloads as W

    w = W.WORKLOADS[wid].scaled(T=T, H=H)
    x = W.bf16_bits(W.make_x(w, seed))
    rg = W.make_routing_gate(w, seed)
    return w, x, rg["topk_idx"], rg["gate_w"]


@pytest.mark.parametrize("wid,T,H", [(1, 128, 256), (2, 40, 72), (3, 64, 40), (4, 50, 24), (5, 12, 16)])
def test_dispatch_places_every_row(wid, T, H):
    w, x, idx, gate = _small(wid, T, H)
    res = oracle.run_all(w.R, w.E, x, idx, gate, w.window_mode, w.window_rows, w.expert)
    sm, recv = res["slot_map"], res["recv"]
    assert res["status"] == 0
    R, k = w.R, w.k
    for s in range(R):
        for t in range(T):
            for j in range(k):
                assert np.array_equal(recv[sm[s, t, j]], x[s, t])
    if w.window_mode == "packed":
        assert np.array_equal(np.sort(sm.ravel()), np.arange(R * T * k))


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_identity_unit_weights_give_k_times_x(k):
    # dispatch then combine with identity experts and unit weights returns k*x,
    # which is exact in bf16 for a power of two k.
    import torch
    import workloads as W

    w = W.Workload("t", R=4, E=16, T=37, H=48, k=k, routing="zipf_distinct", zipf_s=1.0)
    x = W.bf16_bits(W.make_x(w, 1))
    idx = W.make_routing_gate(w, 1)["topk_idx"]
    gate = np.ones_like(idx, dtype=np.float32)
    res = oracle.run_all(w.R, w.E, x, idx, gate)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    want = (xt * k).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(res["out"], want)


def test_identity_softmax_weights_close_to_gate_sum_times_x():
    import workloads as W

    w, x, idx, gate = _small(5, 20, 64)
    res = oracle.run_all(w.R, w.E, x, idx, gate)
    exact = bits_to_f32(x).astype(np.float64) * gate.astype(np.float64).sum(-1, keepdims=True)
    d = ulp_diff(res["out"], f32_to_bits_torch(exact.astype(np.float32)))
    assert d.max() <= 1


def _f32_nearest_even(q):
    """fp32 nearest (ties to even) to an exact rational q in fp32's normal range."""
    from fractions import Fraction

    if q == 0:
        return np.float32(0.0)
    sign, q = (-1 if q < 0 else 1), abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    scaled = q / Fraction(2) ** (e - 23)  # in [2^23, 2^24)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2):
        n += 1
    return np.float32(sign * n * 2.0 ** (e - 23))


# A hand-made slot pair on which a separately rounded product and sum and a
# fused multiply-add give different output bf16.  Slot 0: w0 = 2 - 3*2^-8 +
# 2^-21, y0 = -1, so acc = -w0 exactly.  Slot 1: w1 = 1 + 2^-23, y1 = 3, exact
# product 3 + 3*2^-23, which rounds (a tie, to even) to 3 + 2^-21.
# Separately rounded: 3 + 2^-21 - w0 = 1 + 3*2^-8 exactly, the bf16 midpoint
# between 1 + 2^-7 and 1 + 2^-6, which rounds to the even 1 + 2^-6 = 0x3F82.
# Fused: 3 + 3*2^-23 - w0 = 1 + 3*2^-8 - 2^-23, below the midpoint, so
# 1 + 2^-7 = 0x3F81.
SLOT_PAIR_W = np.array([2.0 - 3 * 2.0 ** -8 + 2.0 ** -21, 1.0 + 2.0 ** -23], np.float32)
SLOT_PAIR_Y = np.array([0xBF80, 0x4040], np.uint16)  # bf16 -1, 3
SLOT_PAIR_SEPARATE, SLOT_PAIR_FUSED = 0x3F82, 0x3F81


def test_combine_rounds_product_and_sum_hand_case():
    from fractions import Fraction

    # the two readings, in exact rationals, do differ on this case ...
    w0, w1 = (Fraction(float(v)) for v in SLOT_PAIR_W)
    acc = _f32_nearest_even(w0 * -1)
    sep = _f32_nearest_even(Fraction(float(_f32_nearest_even(w1 * 3))) + Fraction(float(acc)))
    fused = _f32_nearest_even(w1 * 3 + Fraction(float(acc)))
    assert int(f32_to_bits_torch(np.float32([sep]))[0]) == SLOT_PAIR_SEPARATE
    assert int(f32_to_bits_torch(np.float32([fused]))[0]) == SLOT_PAIR_FUSED
    # ... and the oracle rounds the product and then the sum, in every column
    H = 16
    y = np.repeat(SLOT_PAIR_Y[:, None], H, axis=1)
    out = oracle.combine(y, SLOT_PAIR_W.reshape(1, 1, 2), np.array([[[0, 1]]], np.int32))
    assert (out == SLOT_PAIR_SEPARATE).all(), out


@pytest.mark.parametrize("wid,T,H,nthr", [(2, 40, 16, 3), (3, 64, 8, 8), (4, 50, 8, 5), (5, 12, 8, 7)])
def test_dispatch_by_rank_ranges_equals_whole_dispatch(wid, T, H, nthr):
    # The per-rank CPU setting runs disjoint source-rank ranges of the same
    # dispatch; together they must place every row and slot as one call does
    # (fixed windows with overflow included).
    import workloads as W

    w = W.WORKLOADS[wid].scaled(T=T, H=H)
    x = W.bf16_bits(W.make_x(w, 3))
    idx = W.make_routing_gate(w, 3)["topk_idx"]
    window_rows = w.window_rows if w.window_mode != "fixed" else max(1, w.window_rows // 9)
    sp = oracle.splits(w.R, w.E, idx, w.window_mode, window_rows)
    recv, sm, st = oracle.dispatch(w.R, w.E, x, idx, sp, w.window_mode, window_rows)
    recv2 = np.zeros_like(recv)
    sm2 = np.full_like(sm, -7)
    st2 = 0
    for i in range(nthr):
        s0, s1 = w.R * i // nthr, w.R * (i + 1) // nthr
        _, _, sti = oracle.dispatch(w.R, w.E, x, idx, sp, w.window_mode, window_rows, recv=recv2, ranks=(s0, s1),
                                    slot_map_out=sm2)
        st2 |= sti
    np.testing.assert_array_equal(sm2, sm)
    np.testing.assert_array_equal(recv2, recv)
    assert st2 == st
    with pytest.raises(ValueError):
        oracle.dispatch(w.R, w.E, x, idx, sp, ranks=(0, 1), recv_order="expert")


def test_combine_non_finite_values_follow_ieee():
    # Reading: infinities and NaNs in the expert outputs go through the
    # combine's fp32 products and sums as IEEE 754 defines them (a zero gate
    # times an infinity is NaN, +inf plus -inf is NaN, a NaN stays NaN).  Pinned
    # against numpy's float32 arithmetic, which shares nothing with the oracle,
    # on every pair of special and ordinary values under every pair of gates.
    vals = np.array([0x7F80, 0xFF80, 0x7FC1, 0xFFA0, 0x3FC0, 0xC000, 0x0000, 0x8000, 0x4040], np.uint16)
    gates = np.array([0.0, 1.0, 0.5, -1.0, -0.0, np.inf], np.float32)
    ys, ws = [], []
    for a in vals:
        for b in vals:
            for g0 in gates:
                for g1 in gates:
                    ys.append((a, b))
                    ws.append((g0, g1))
    n = len(ys)
    H = 2  # column 1 holds a finite control value
    y = np.zeros((2 * n, H), np.uint16)
    y[:, 0] = np.array(ys, np.uint16).reshape(-1)
    y[:, 1] = 0x3F80
    gate = np.array(ws, np.float32).reshape(1, n, 2)
    sm = np.arange(2 * n, dtype=np.int32).reshape(1, n, 2)
    out = oracle.combine(y, gate, sm)
    yf = bits_to_f32(np.array(ys, np.uint16))
    wf = np.array(ws, np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        acc = np.float32(0.0) + (wf[:, 0] * yf[:, 0]).astype(np.float32)
        acc = (acc + (wf[:, 1] * yf[:, 1]).astype(np.float32)).astype(np.float32)
        ctrl = ((np.float32(0.0) + wf[:, 0]).astype(np.float32) + wf[:, 1]).astype(np.float32)
    for col, want_f in ((0, acc), (1, ctrl)):
        got = out[:, col]
        nan = np.isnan(want_f)
        assert is_nan(got[nan]).all(), "a NaN result must come out as a NaN"
        assert not is_nan(got[~nan]).any()
        np.testing.assert_array_equal(got[~nan], f32_to_bits_torch(want_f[~nan]))
    # the cases the reading names, spelled out
    index = {(int(a), int(b), float(g0), float(g1)): i for i, ((a, b), (g0, g1)) in enumerate(zip(ys, ws))}

    def one(a, b, g0, g1):
        return int(out[index[(a, b, g0, g1)], 0])

    assert is_nan(one(0x7F80, 0x3FC0, 0.0, 1.0))       # 0 * inf
    assert one(0x7F80, 0x3FC0, 1.0, 1.0) == 0x7F80      # inf + 1.5
    assert is_nan(one(0x7F80, 0xFF80, 1.0, 0.5))       # inf + -inf
    assert is_nan(one(0x7FC1, 0x3FC0, 1.0, 1.0))       # NaN in, NaN out
    assert one(0x7F80, 0x3FC0, -1.0, 1.0) == 0xFF80     # the sign of the gate
    assert one(0x3FC0, 0x4040, np.inf, 0.0) == 0x7F80   # an infinite gate on a finite row


def test_scaled_experts_closed_form_numpy_f32():
    # out = bf16( sum_j w_j * bf16(x * (1 + e_j/E)) ), accumulated in fp32 in j order
    # from 0, products and sums rounded separately -- computed straight from
    # (x, idx, w) with numpy float32 and no dispatch at all.
    w, x, idx, gate = _small(4, 64, 40)
    res = oracle.run_all(w.R, w.E, x, idx, gate, expert="scale")
    xf = bits_to_f32(x)
    acc = np.zeros(xf.shape, np.float32)
    for j in range(w.k):
        scale = (np.float32(1.0) + idx[..., j].astype(np.float32) / np.float32(w.E)).astype(np.float32)
        yj = bits_to_f32(f32_to_bits_torch(xf * scale[..., None]))
        acc = (acc + (gate[..., j][..., None] * yj).astype(np.float32)).astype(np.float32)
    np.testing.assert_array_equal(res["out"], f32_to_bits_torch(acc))


def test_expert_scale_closed_form_torch():
    import torch

    w, x, idx, gate = _small(4, 33, 24)
    sp = oracle.splits(w.R, w.E, idx)
    recv, sm, _ = oracle.dispatch(w.R, w.E, x, idx, sp)
    y = oracle.expert_scale(w.E, recv, idx, sm)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    for s in range(w.R):
        for t in range(0, w.T, 5):
            for j in range(w.k):
                e = int(idx[s, t, j])
                want = (xt[s, t] * (1.0 + e / w.E)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                np.testing.assert_array_equal(y[sm[s, t, j]], want)


def test_combine_fp32_within_one_ulp_of_fp64():
    import workloads as W

    for wid, T, H in [(4, 64, 64), (5, 16, 64)]:
        w, x, idx, gate = _small(wid, T, H)
        res = oracle.run_all(w.R, w.E, x, idx, gate, expert=w.expert)
        f64 = oracle.combine_f64(res["y"], gate, res["slot_map"])
        want = f32_to_bits_torch(f64.astype(np.float32))  # fp64 -> fp32 is within fp32's half ulp
        assert ulp_diff(res["out"].reshape(-1, H), want).max() <= 1


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),
        # exact ties: bf16 value + half an ulp, both parities
        ((np.arange(1, 500, dtype=np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, np.inf, -np.inf], np.float32),
    ])
    want = f32_to_bits_torch(vals)
    got = np.array([oracle.f32_to_bf16(v) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, want)
    bits = rng.integers(0, 1 << 16, 5000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]
    back = np.array([oracle.bf16_to_f32(b) for b in bits], np.float32)
    np.testing.assert_array_equal(back, bits_to_f32(bits))


# ----------------------------------------------------------------------------
# mutation checks: plant a mistake in a copy of the oracle, the pins must fail
# ----------------------------------------------------------------------------
MUTANTS = {
    "transposed recv_offsets": ("(int64_t)recv_offsets[(size_t)d * R + s] + (pos[a] - so[d * epr]);\n            if (expert_order)",
                                "(int64_t)recv_offsets[(size_t)s * R + d] + (pos[a] - so[d * epr]);\n            if (expert_order)"),
    "expert blocks regrouped source-major": ("        for (int le = 0; le < epr; ++le)\n            for (int s = 0; s < R; ++s) {\n                const int32_t *sc",
                                             "        for (int s = 0; s < R; ++s)\n            for (int le = 0; le < epr; ++le) {\n                const int32_t *sc"),
    "expert offsets count own source": ("                    for (int s2 = 0; s2 < s; ++s2)\n                        v += recv_expert_counts[((size_t)d * R + s2) * epr + le];",
                                        "                    for (int s2 = 0; s2 <= s; ++s2)\n                        v += recv_expert_counts[((size_t)d * R + s2) * epr + le];"),
    "expert-order rank from segment start": ("+ (e - d * epr)] + (pos[a] - so[e]);", "+ (e - d * epr)] + (pos[a] - so[d * epr]);"),
    "inclusive send_offsets": ("            send_offsets[(size_t)s * E + e] = run;\n            run += cnt[e];",
                               "            run += cnt[e];\n            send_offsets[(size_t)s * E + e] = run;"),
    "unstable sort": ("    for (int t = 0; t < T; ++t)\n        for (int j = 0; j < k; ++j) {\n            int32_t e = idx_s[(size_t)t * k + j];\n            if (t >= Ts) {",
                      "    for (int t = T - 1; t >= 0; --t)\n        for (int j = 0; j < k; ++j) {\n            int32_t e = idx_s[(size_t)t * k + j];\n            if (t >= Ts) {"),
    "dropped gate weight": ("float prod = w[j] * oracle_bf16_to_f32(", "float prod = 1.0f * oracle_bf16_to_f32("),
    "fused multiply-add": ("float prod = w[j] * oracle_bf16_to_f32(y[(size_t)slots[j] * H + h]);\n                acc = acc + prod;",
                           "acc = fmaf(w[j], oracle_bf16_to_f32(y[(size_t)slots[j] * H + h]), acc);"),
    "truncating bf16 rounding": ("u += 0x7fffu + keep_lsb;", "u += 0u * keep_lsb;"),
    "window base off by one window": ("            window_base[d] = (int32_t)base;\n        base += recv_total[d];",
                                      "        base += recv_total[d];\n            window_base[d] = (int32_t)base;"),
    "wrong expert-to-rank map": ("            int d = e / epr;\n            int64_t rel", "            int d = e % R;\n            int64_t rel"),
    "expert scale sign": ("float scale = 1.0f + q;", "float scale = 1.0f - q;"),
    "router tie order": ("return a > b || (a == b && ia < ib);", "return a > b || (a == b && ia > ib);"),
    "router softmax shift": ("ex[j] = exp(sel[j] - sel[0]);", "ex[j] = exp(sel[j] - sel[k - 1]) * (j + 1);"),
    "padded segments by destination": ("recv_offsets[(size_t)d * R + s] = (int32_t)((int64_t)s * T * k);",
                                       "recv_offsets[(size_t)d * R + s] = (int32_t)((int64_t)d * T * k);"),
}


def _pin_suite():
    """The pins above, run against whatever library ``oracle._lib`` holds."""
    test_hand_worked_example()
    test_exhaustive_top1_r2_e4(2)
    test_exhaustive_top2_distinct_r2_e4()
    test_random_against_brute(4, 8, 9, 3)
    test_identity_unit_weights_give_k_times_x(2)
    test_identity_softmax_weights_close_to_gate_sum_times_x()
    test_scaled_experts_closed_form_numpy_f32()
    test_combine_rounds_product_and_sum_hand_case()
    test_expert_scale_closed_form_torch()
    test_bf16_rounding_matches_torch()
    test_padded_layout_against_brute()
    test_router_against_numpy_sort_and_softmax()
    test_hand_worked_example_expert_order()
    test_exhaustive_expert_order_r2_e4("expert")
    test_expert_order_random_fixed_and_active_against_brute()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    import ctypes

    src = open(os.path.join(os.path.dirname(oracle.__file__), "a2av_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    path = oracle.compile_source(src.replace(old, new), str(tmp_path / "mutant.so"))
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(path)))
    with pytest.raises(AssertionError):
        _pin_suite()
