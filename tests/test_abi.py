"""The C-ABI library builds, loads without a GPU, and exports every function
that include/*.h declares; host-only calls validate configurations."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(a2av_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from combine_device_resident_gb300 import build

    build.build()
    from combine_device_resident_gb300 import load_library

    return load_library()


def test_header_declares_the_calls():
    names = _declared_functions()
    for must in ("a2av_dispatch", "a2av_combine", "a2av_splits", "a2av_pack", "a2av_plan_create"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from combine_device_resident_gb300 import EXPORTED

    declared = _declared_functions()
    assert declared, "no declarations found"
    for name in declared:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert sorted(EXPORTED) == sorted(declared), "binding's symbol list out of step with the header"


def _cfg(**kw):
    from combine_device_resident_gb300 import make_config

    base = dict(R=8, E=16, T=1024, H=5120, k=1)
    base.update(kw)
    return make_config(**base)


def test_config_check_host_only(lib):
    ok = [_cfg(), _cfg(R=1, E=1, T=1, H=8, k=1), _cfg(R=64, E=2048, T=3, H=8, k=32),
          _cfg(window_mode="fixed", window_rows=100), _cfg(window_mode="padded"), _cfg(recv_order="expert"),
          _cfg(window_mode="fixed", window_rows=100, recv_order="expert"), _cfg(flags=1 << 3), _cfg(flags=1 << 4),
          _cfg(flags=(1 << 3) | (1 << 4))]
    bad = [_cfg(R=0), _cfg(R=65, E=130), _cfg(E=12, R=8), _cfg(E=4096, R=8), _cfg(H=12), _cfg(H=0), _cfg(k=0),
           _cfg(k=33), _cfg(T=0), _cfg(window_mode=3), _cfg(window_mode="fixed", window_rows=-1),
           _cfg(R=64, E=64, T=65536, k=8, window_mode="padded"),
           _cfg(R=64, E=64, T=1 << 20, k=32), _cfg(flags=1 << 7), _cfg(flags=1 << 5), _cfg(pack_stage_bytes=24),
           _cfg(pack_ctas_per_sm=9), _cfg(recv_order=2), _cfg(recv_order=-1),
           _cfg(window_mode="padded", recv_order="expert")]
    for c in ok:
        assert lib.a2av_config_check(ctypes.byref(c)) == 0
    for c in bad:
        assert lib.a2av_config_check(ctypes.byref(c)) == 1
    assert lib.a2av_config_check(None) == 1


def test_struct_layouts_match_the_header():
    # the binding's ctypes mirrors of a2av_config_t / a2av_splits_t
    from combine_device_resident_gb300.binding import Config, SplitsPtrs

    assert Config.recv_order.offset == Config.combine_unroll.offset + 4
    assert ctypes.sizeof(Config) == (Config.recv_order.offset + 4 + 7) // 8 * 8  # int64 member: 8-byte alignment
    assert SplitsPtrs.recv_expert_offsets.offset == 7 * ctypes.sizeof(ctypes.c_void_p)
    hdr = open(os.path.join(ROOT, "include", "a2av.h")).read()
    cfg_body = hdr[hdr.index("typedef struct {\n    int32_t num_ranks;"):hdr.index("} a2av_config_t;")]
    fields = re.findall(r"^\s*(?:u?int\d+_t)\s+(\w+);", cfg_body, re.M)
    assert fields == [f[0] for f in Config._fields_]
    sp_body = hdr[hdr.index("typedef struct {\n    int32_t *send_counts;"):hdr.index("} a2av_splits_t;")]
    assert re.findall(r"int32_t \*(\w+);", sp_body) == [f[0] for f in SplitsPtrs._fields_]


def test_arena_rows(lib):
    assert lib.a2av_recv_arena_rows(ctypes.byref(_cfg(R=32, E=256, T=2048, k=8))) == 32 * 2048 * 8
    assert lib.a2av_recv_arena_rows(ctypes.byref(_cfg(window_mode="fixed", window_rows=2048))) == 8 * 2048
    assert lib.a2av_recv_arena_rows(ctypes.byref(_cfg(H=7))) == -1
    assert lib.a2av_recv_arena_rows(ctypes.byref(_cfg(window_mode="padded"))) == 8 * 8 * 1024


def test_plan_create_rejects_bad_config_without_touching_a_gpu(lib):
    h = ctypes.c_void_p()
    assert lib.a2av_plan_create(ctypes.byref(_cfg(H=12)), ctypes.byref(h)) == 1
    assert not h.value
    assert lib.a2av_plan_create(ctypes.byref(_cfg()), None) == 1


def test_null_arguments_are_rejected(lib):
    from combine_device_resident_gb300.binding import SplitsPtrs

    sp = SplitsPtrs()
    assert lib.a2av_dispatch(None, None, None, ctypes.byref(sp), None, None, None) == 1
    assert lib.a2av_combine(None, None, None, None, None, None) == 1
    assert lib.a2av_plan_destroy(None) == 0
    assert lib.a2av_status_string(0) == b"ok"
    assert lib.a2av_status_string(1) == b"invalid argument"


def test_product_path_fails_loudly_without_library(tmp_path):
    from combine_device_resident_gb300 import binding

    with pytest.raises(binding.A2avError):
        binding.load_library(str(tmp_path / "missing.so"))


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "combine_device_resident_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.sub(r"#.*|//.*", "", src).replace("the oracle", ""), f


def test_static_dispatch_checks_every_shape_on_the_host():
    # a2av_dispatch_static's binding checks shapes before any device work, so
    # a wrong shape fails here without a GPU (host tensors, never enqueued).
    import torch

    import combine_device_resident_gb300 as A
    from combine_device_resident_gb300.binding import dispatch_static

    R, E, T, H, k = 4, 16, 50, 64, 2
    good = dict(x=torch.zeros((R, T, H), dtype=torch.bfloat16), topk_idx=torch.zeros((R, T, k), dtype=torch.int32),
                splits=A.Splits(R, E, "cpu"), recv=torch.zeros((R * T * k, H), dtype=torch.bfloat16),
                slot_map=torch.zeros((R, T, k), dtype=torch.int32), dev_status=torch.zeros(1, dtype=torch.int32))
    bad = {"x": torch.zeros((R, T, H - 8), dtype=torch.bfloat16),
           "topk_idx": torch.zeros((R, T - 1, k), dtype=torch.int32),
           "splits": A.Splits(R, 2 * E, "cpu"),
           "recv": torch.zeros((R * T * k - 1, H), dtype=torch.bfloat16),
           "slot_map": torch.zeros((R, T, 1), dtype=torch.int32),
           "dev_status": torch.zeros(0, dtype=torch.int32)}
    for name, t in bad.items():
        args = dict(good, **{name: t})
        with pytest.raises(A.A2avError, match="shape|element"):
            dispatch_static(args["x"], args["topk_idx"], args["splits"], args["recv"], args["slot_map"],
                            args["dev_status"], R, E, T, H, k)
    # right shapes, host tensors: refused for the device, still before any call
    with pytest.raises(A.A2avError, match="CUDA device"):
        dispatch_static(*good.values(), R, E, T, H, k)
    expert = A.Splits(R, E, "cpu", expert_offsets=False)
    with pytest.raises(A.A2avError, match="expert"):
        dispatch_static(good["x"], good["topk_idx"], expert, good["recv"], good["slot_map"], good["dev_status"],
                        R, E, T, H, k, recv_order="expert")
