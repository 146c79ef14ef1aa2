"""The oracle still reproduces the fixtures stored under tests/golden/ (regression
pins written by tests/golden/make_golden.py, which calls only the oracle)."""
import glob
import json
import os

import numpy as np
import pytest

import oracle

FILES = sorted(glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))


@pytest.mark.parametrize("path", FILES, ids=[os.path.basename(p) for p in FILES])
def test_oracle_reproduces_golden(path):
    doc = json.load(open(path))
    idx = np.array(doc["topk_idx"], np.int32)
    x = np.array(doc["x_bits"], np.uint16)
    gate = np.array([[[float.fromhex(v) for v in r] for r in g] for g in doc["gate_w_hex"]], np.float32)
    res = oracle.run_all(doc["R"], doc["E"], x, idx, gate, doc["window_mode"], doc["window_rows"], doc["expert"])
    for key, val in doc["splits"].items():
        assert res["splits"][key].tolist() == val, key
    assert res["slot_map"].tolist() == doc["slot_map"]
    assert res["out"].tolist() == doc["out_bits"]
    assert res["status"] == doc["status"]
