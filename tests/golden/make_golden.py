"""Writes the regression fixtures in this folder.  It calls only ``oracle/``
(and the seeded input generator), never the CUDA library, so every stored value
is an oracle value; rerun it only when the oracle's arithmetic changes for a
reason that names the passage or reading behind the change."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def case(name, R, E, T, k, H, window_mode="packed", window_rows=0, expert="identity", seed=0):
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, E, size=(R, T, k), dtype=np.int32)
    x = (rng.integers(0x3c00, 0x4100, size=(R, T, H)) | (rng.integers(0, 2, size=(R, T, H)) << 15)).astype(np.uint16)
    gate = rng.random((R, T, k), dtype=np.float32)
    res = oracle.run_all(R, E, x, idx, gate, window_mode, window_rows, expert)
    sp = res["splits"]
    doc = {
        "about": "regression fixture written by tests/golden/make_golden.py from the CPU oracle",
        "R": R, "E": E, "T": T, "k": k, "H": H, "window_mode": window_mode, "window_rows": window_rows,
        "expert": expert,
        "topk_idx": idx.tolist(), "x_bits": x.tolist(), "gate_w_hex": [[[float(v).hex() for v in r] for r in g] for g in gate],
        "splits": {k2: sp[k2].tolist() for k2 in ("send_counts", "send_offsets", "recv_counts", "recv_offsets",
                                                    "recv_expert_counts", "recv_total", "window_base")},
        "slot_map": res["slot_map"].tolist(), "out_bits": res["out"].tolist(), "status": res["status"],
    }
    with open(os.path.join(HERE, name + ".json"), "w") as f:
        json.dump(doc, f, separators=(",", ":"))


if __name__ == "__main__":
    case("r2_e4_t5_k2_h8_packed_scale", 2, 4, 5, 2, 8, expert="scale", seed=1)
    case("r3_e6_t4_k2_h16_fixed_w5_overflow", 3, 6, 4, 2, 16, "fixed", 5, seed=2)
