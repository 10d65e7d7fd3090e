"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every entry point
that include/*.h declares (moe_tail.h, attnres_mix.h), and answers argument errors before
touching a device."""
import ctypes
import os
import re

import pytest

import moe_layer_tail_gb300 as mt
from moe_layer_tail_gb300 import build as mt_build
from moe_layer_tail_gb300 import inputs as gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mt_build.build()
    return mt.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_(?:tail|attnres)_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12, names
    assert {"moe_attnres_mix", "moe_attnres_mix_ctas_per_row",
            "moe_attnres_mix_get_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), "missing export " + n


def header_enum_values():
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "moe_tail.h")).read(),
                 flags=re.S)
    return {k: int(v) for k, v in re.findall(r"\b(MOE_TAIL_[A-Z0-9_]+)\s*=\s*(-?\d+)", src)}


def test_binding_constants_match_header():
    vals = header_enum_values()
    for name, v in vals.items():
        short = name[len("MOE_TAIL_"):]
        if short.startswith(("ERR_", "STATUS_", "MODE_", "DEBUG_")) or short == "OK":
            assert getattr(mt, short) == v, name
    assert {k for k in vals if k.startswith("MOE_TAIL_STATUS_")} == {
        "MOE_TAIL_STATUS_BAD_ROUTING", "MOE_TAIL_STATUS_BAD_DISTINCT", "MOE_TAIL_STATUS_TIMEOUT",
        "MOE_TAIL_STATUS_BAD_TILE"}


def test_timeline_slots_match_header():
    vals = header_enum_values()
    slots = sorted((v, k) for k, v in vals.items()
                   if k.startswith("MOE_TAIL_TL_") and k != "MOE_TAIL_TL_SLOTS")
    assert [v for v, _ in slots] == list(range(vals["MOE_TAIL_TL_SLOTS"]))
    assert [k[len("MOE_TAIL_TL_"):].lower() for _, k in slots] == list(mt.TL_NAMES)


def test_timeline_refused_without_its_flag(lib):
    import numpy as np
    buf = np.zeros(14, np.uint64)
    assert lib.moe_tail_debug_timeline(None, buf.ctypes.data, 14) == mt.ERR_INVALID_ARG


def test_weight_struct_fields_match_header():
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "moe_tail.h")).read(),
                 flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\} moe_tail_weights_t;", src).group(1)
    fields = re.findall(r"const void\*\s+(\w+);", body)
    assert [f for f, _ in mt.WeightPtrs._fields_] == fields
    assert fields[-2:] == ["shared_gate", "out_proj"]


def test_config_struct_fields_match_header():
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "moe_tail.h")).read(),
                 flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\} moe_tail_config_t;", src).group(1)
    fields = re.findall(r"(?:int32_t|uint32_t|float)\s+(\w+);", body)
    assert [f for f, _ in mt.Config._fields_] == fields
    assert fields[-1] == "attn_dim"


def test_strerror_covers_codes(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = lib.moe_tail_strerror(code).decode()
        assert s and s != "unknown error"
    assert lib.moe_tail_strerror(-99).decode() == "unknown error"


def test_null_arguments_rejected_without_device(lib):
    h = ctypes.c_void_p()
    assert lib.moe_tail_create(None, None, ctypes.byref(h)) == mt.ERR_INVALID_ARG
    assert h.value is None
    assert lib.moe_tail_run(None, None, None, None, 1, None) == mt.ERR_INVALID_ARG
    assert lib.moe_tail_run_host(None, None, None, None, 1, None) == mt.ERR_INVALID_ARG
    assert lib.moe_tail_run_attn(None, None, None, None, 1, None) == mt.ERR_INVALID_ARG
    assert lib.moe_tail_get_status(None, None) == mt.ERR_INVALID_ARG
    assert lib.moe_tail_refresh_scales(None, None) == mt.ERR_INVALID_ARG
    lib.moe_tail_destroy(None)
    assert lib.moe_tail_launches_per_run(None, 1) == 0


@pytest.mark.parametrize("field,value", [("max_rows", 0), ("max_rows", 33), ("hidden", 200),
                                         ("hidden", 384), ("hidden", 2304),
                                         ("top_k", 9), ("expert_inter", 96),
                                         ("expert_inter", 2176),
                                         ("shared_inter", 100), ("norm_topk_prob", 0),
                                         ("n_experts", 2000), ("rms_eps", 0.0),
                                         ("attn_dim", -64), ("attn_dim", 100),
                                         ("attn_dim", 65600)])
def test_unsupported_configs_refused_before_device(lib, field, value):
    cfg = mt.make_config(gen.TailShape(2, 256, 8, 2, 128, 128))
    setattr(cfg, field, value)
    w = mt.WeightPtrs(*([16] * 8))  # never dereferenced: refusal comes first
    h = ctypes.c_void_p()
    assert lib.moe_tail_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == \
        mt.ERR_UNSUPPORTED
    assert h.value is None


@pytest.mark.parametrize("flags,mode,attn", [(16, 0, 0), (1, 0, 0), (8, 0, 0), (0, 0, 64)])
def test_more_than_16_rows_only_in_the_tensor_core_forms(lib, flags, mode, attn):
    # mma.sync, cross-checking kernels, fused front, out_proj: 16 rows at most (the default
    # form and the persistent launch, both on the tensor-core kernels, take up to 32)
    cfg = mt.make_config(gen.TailShape(24, 256, 8, 2, 128, 128, Ha=attn), debug_flags=flags,
                         mode=mode)
    w = mt.WeightPtrs(*([16] * 8 + ([0, 16] if attn else [])))  # never dereferenced
    h = ctypes.c_void_p()
    assert lib.moe_tail_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == \
        mt.ERR_UNSUPPORTED
    assert h.value is None


def test_misaligned_weight_pointer_refused(lib):
    cfg = mt.make_config(gen.TailShape(2, 256, 8, 2, 128, 128))
    w = mt.WeightPtrs(*([16] * 7 + [24]))
    h = ctypes.c_void_p()
    assert lib.moe_tail_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == \
        mt.ERR_INVALID_ARG


def test_out_proj_pointer_must_match_attn_dim(lib):
    h = ctypes.c_void_p()
    cfg = mt.make_config(gen.TailShape(2, 256, 8, 2, 128, 128, Ha=128))
    w = mt.WeightPtrs(*([16] * 8))  # attn_dim > 0 but no out_proj
    assert lib.moe_tail_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == \
        mt.ERR_INVALID_ARG
    cfg = mt.make_config(gen.TailShape(2, 256, 8, 2, 128, 128))
    w = mt.WeightPtrs(*([16] * 8 + [0, 16]))  # out_proj given with attn_dim 0
    assert lib.moe_tail_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == \
        mt.ERR_INVALID_ARG
    assert h.value is None


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(mt, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        mt.load_library(str(tmp_path / "nope.so"))


# ------------------------------------------------------ the AttnRes mix (attnres_mix.h) ----

def test_attnres_mix_flags_match_header():
    src = open(os.path.join(ROOT, "include", "attnres_mix.h")).read()
    for name in ("PDL", "DEBUG_STALL"):
        v = int(re.search(r"#define MOE_ATTNRES_MIX_%s (\d+)u" % name, src).group(1))
        assert getattr(mt, "ATTNRES_MIX_" + name) == v


def test_attnres_mix_status_refuses_null(lib):
    assert lib.moe_attnres_mix_get_status(None, 0) == mt.ERR_INVALID_ARG


@pytest.mark.parametrize("hidden,n_blocks,ctas", [
    (7168, 8, 8), (8192, 31, 8), (256, 0, 2), (64, 0, 1), (1000, 3, 1), (1024, 5, 8),
    (65536, 8, 8), (65536, 31, None), (7, 0, None), (65544, 0, None), (7168, 32, None),
    (7168, -1, None)])
def test_attnres_mix_plan(lib, hidden, n_blocks, ctas):
    rc = lib.moe_attnres_mix_ctas_per_row(hidden, n_blocks)
    assert rc == (ctas if ctas is not None else mt.ERR_UNSUPPORTED)


def _mix_call(lib, **kw):
    P = ctypes.c_void_p
    args = dict(rows=8, hidden=7168, n_blocks=3, commit=0, eps=1e-6, sub=P(0x1000),
                prefix=P(0x2000), blocks=P(0x3000), q=P(0x4000), gamma=P(0x5000),
                mix=P(0x6000), y=P(0x7000), flags=0, stream=P(0))
    args.update(kw)
    return lib.moe_attnres_mix(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(rows=0), mt.ERR_INVALID_ARG),
    (dict(rows=4097), mt.ERR_INVALID_ARG),
    (dict(n_blocks=-1), mt.ERR_INVALID_ARG),
    (dict(eps=0.0), mt.ERR_INVALID_ARG),
    (dict(eps=float("nan")), mt.ERR_INVALID_ARG),
    (dict(eps=float("inf")), mt.ERR_INVALID_ARG),
    (dict(flags=4), mt.ERR_INVALID_ARG),
    (dict(flags=0x80000000), mt.ERR_INVALID_ARG),
    (dict(sub=ctypes.c_void_p(0)), mt.ERR_INVALID_ARG),
    (dict(y=ctypes.c_void_p(0x7008)), mt.ERR_INVALID_ARG),
    (dict(blocks=ctypes.c_void_p(0)), mt.ERR_INVALID_ARG),
    (dict(n_blocks=0, commit=1, blocks=ctypes.c_void_p(0)), mt.ERR_INVALID_ARG),
    (dict(hidden=7164), mt.ERR_UNSUPPORTED),
    (dict(hidden=1 << 17), mt.ERR_UNSUPPORTED),
    (dict(n_blocks=32), mt.ERR_UNSUPPORTED),
    (dict(hidden=65536, n_blocks=31), mt.ERR_UNSUPPORTED),
])
def test_attnres_mix_refuses_bad_arguments_before_any_launch(lib, kw, code):
    assert _mix_call(lib, **kw) == code


def test_check_scratch_refuses_null_handle(lib):
    assert lib.moe_tail_check_scratch(None) == mt.ERR_INVALID_ARG
