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


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_full_size(wid):
    import torch

    w = W.WORKLOADS[wid]
    dev = P.device()
    rg = W.make_routing_gate(w, 0)
    idx, gate = rg["topk_idx"], rg["gate_w"]
    x = W.make_x(w, 0, device=dev)
    g = P.gpu_run(w, x, idx, gate, guard_rows=2, expert_offsets=False)  # as the benchmark calls it

    sp = oracle.splits(w.R, w.E, idx, w.window_mode, w.window_rows)
    P.check_splits(g["splits"], sp)
    sm_ref, st = oracle.slot_map(w.R, w.E, idx, sp, w.window_mode, w.window_rows)
    np.testing.assert_array_equal(g["slot_map"], sm_ref)
    assert g["status"] == (sp["status"] | st) == 0
    assert g["guard_ok"]

    # every dispatched row carries its token (on the device, chunked)
    slot_t = torch.from_numpy(sm_ref).to(dev).view(-1, w.k)
    recv = g["recv_t"]
    xf = x.view(-1, w.H)
    step = max(1, (1 << 28) // (w.H * 2 * w.k))
    for lo in range(0, xf.shape[0], step):
        hi = min(xf.shape[0], lo + step)
        rows = slot_t[lo:hi].reshape(-1).long()
        got = recv.index_select(0, rows).view(hi - lo, w.k, w.H)
        assert torch.equal(got.view(torch.int16), xf[lo:hi].unsqueeze(1).expand(-1, w.k, -1).view(torch.int16)), \
            f"recv rows of tokens {lo}..{hi} differ from their source rows"
    if w.window_mode == "packed":
        assert np.array_equal(np.sort(sm_ref.ravel()), np.arange(w.R * w.T * w.k))

    # combine on sampled tokens (including the first and last of every rank)
    rng = np.random.default_rng(wid)
    ntok = w.R * w.T
    pick = np.unique(np.concatenate([rng.choice(ntok, size=min(ntok, 1500), replace=False),
                                     np.arange(w.R) * w.T, np.arange(1, w.R + 1) * w.T - 1]))
    pick_t = torch.from_numpy(pick).to(dev)
    got_out = P.bits(g["out_t"].view(-1, w.H).index_select(0, pick_t))
    xs = P.bits(xf.index_select(0, pick_t))
    want = _sampled_reference(w, xs, idx.reshape(-1, w.k)[pick], gate.reshape(-1, w.k)[pick], w.expert)
    d = ulp_diff(got_out, want)
    assert d.max() <= P.COMBINE_ULP_TOL
    del g
    torch.cuda.empty_cache()
