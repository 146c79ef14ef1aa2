"""Host-side helpers of bench.py (no GPU)."""
import bench


def test_code_only_drops_comments_and_whitespace():
    a = "int a = 1; // count\n/* block\n comment */ const char *s = \"//kept\";\n\n  char c = '/';"
    b = "int a = 1;\nconst char *s = \"//kept\"; char c = '/';"
    assert bench._code_only(a) == bench._code_only(b)
    assert '"//kept"' in bench._code_only(a)


def test_code_only_sees_code_changes():
    assert bench._code_only("x = a + b; // sum") != bench._code_only("x = a - b; // sum")
    assert bench._code_only('s = "a /* b */ c";') == 's = "a /* b */ c";'


def test_kernel_hashes_are_distinct_and_stable():
    hs = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert len(set(hs.values())) == len(hs)
    assert hs == {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}


def test_traffic_record_is_keyed_on_workload_and_kernel():
    w5 = "r32-e256-t2048-h7168-top8-hot0-zipf1.1-softmax"
    assert bench.ncu_traffic("pack", "no-such-workload") is None
    assert bench.ncu_traffic("route", w5) is None  # no capture recorded for the router
    assert bench.ncu_traffic("no-such-kernel", w5) is None


def test_traffic_records_add_up_and_match_the_workload():
    import json
    import os

    import workloads as W

    d = json.load(open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")))
    by_name = {w.name: w for w in W.WORKLOADS.values()}
    for ent in d["records"]:
        assert ent["dram_bytes_per_launch"] == ent["dram_read_bytes"] + ent["dram_write_bytes"], ent["kernel"]
        reads = [r for r, _ in ent["per_launch"]]
        writes = [w_ for _, w_ in ent["per_launch"]]
        assert ent["dram_read_bytes"] == sum(reads) // len(reads), ent["kernel"]
        assert ent["dram_write_bytes"] == sum(writes) // len(writes), ent["kernel"]
        w = by_name[ent["workload"]]
        A = w.R * w.T * w.k
        assert ent["algorithmic_bytes_per_launch"] == w.R * w.T * w.H * 2 * (1 + w.k) + 8 * A
        # measured DRAM bytes of a full-size launch: within a few % of the algorithmic bytes
        assert 0.95 < ent["dram_bytes_per_launch"] / ent["algorithmic_bytes_per_launch"] < 1.02, ent["kernel"]


def test_threaded_oracle_step_equals_one_thread_run():
    # CPU baseline setting (ii): the same oracle functions on disjoint
    # source-rank ranges, one thread each, give the one-thread results.
    import concurrent.futures

    import numpy as np

    import oracle
    import workloads as W

    for wid, T, H, nthr in [(4, 40, 16, 5), (5, 10, 8, 16), (2, 30, 8, 3)]:
        w = W.WORKLOADS[wid].scaled(T=T, H=H)
        x = W.bf16_bits(W.make_x(w, 0))
        rg = W.make_routing_gate(w, 0)
        ref = oracle.run_all(w.R, w.E, x, rg["topk_idx"], rg["gate_w"], w.window_mode, w.window_rows, w.expert)
        with concurrent.futures.ThreadPoolExecutor(max_workers=nthr) as pool:
            recv, sm, out = bench.oracle_step_threaded(w, x, rg["topk_idx"], rg["gate_w"], pool, nthr)
        np.testing.assert_array_equal(sm, ref["slot_map"])
        np.testing.assert_array_equal(recv, ref["recv"])
        np.testing.assert_array_equal(out, ref["out"])


def test_cpu_baseline_reports_both_settings():
    import workloads as W

    w = W.WORKLOADS[5].scaled(T=16, H=64)
    x = W.bf16_bits(W.make_x(w, 0))
    rg = W.make_routing_gate(w, 0)
    cb = bench.cpu_baseline(w, x, rg["topk_idx"], rg["gate_w"], budget_s=0.5, threads=4)
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] > 0
    assert cb["threads"] == 4 and cb["value_threaded"] > 0 and "4 threads" in cb["sample_threaded"]


def test_tokens_and_hidden_options_scale_the_workload():
    # --tokens and --hidden give the small cases the profiles use; the
    # router's capture keeps every token and shrinks only the rows
    import bench
    import workloads as W

    a = bench.parse_args(["--workload", "5", "--hidden", "64"])
    assert (a.tokens, a.hidden) == (0, 64)
    w = bench.resolve_workload(a)
    base = W.WORKLOADS[5]
    assert (w.R, w.E, w.T, w.k, w.H) == (base.R, base.E, base.T, base.k, 64)
    a = bench.parse_args(["--workload", "3", "--tokens", "16"])
    w = bench.resolve_workload(a)
    assert (w.T, w.H, w.window_rows) == (16, W.WORKLOADS[3].H, W.WORKLOADS[3].R * 16 * W.WORKLOADS[3].k)
    assert bench.resolve_workload(bench.parse_args([])) == W.WORKLOADS[bench.DEFAULT_WORKLOAD]
