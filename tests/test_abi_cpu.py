"""The C-ABI library builds, loads and exports what include/moe_decode.h
declares; host-side argument checks (no CUDA work, no GPU needed)."""
import ctypes
import os
import re

import pytest

import quantized_moe_decode_softmax_gb300 as q
from quantized_moe_decode_softmax_gb300 import _abi
from quantized_moe_decode_softmax_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_decode.h")


@pytest.fixture(scope="module")
def libpath():
    return qbuild.build()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, re.M))


def test_header_declares_the_bound_functions():
    assert header_functions() == set(q.EXPORTED)


def test_library_exports_every_declared_symbol(libpath):
    L = ctypes.CDLL(libpath)
    for name in header_functions():
        assert hasattr(L, name), name


def test_abi_version_and_status_strings(libpath):
    assert q.moe_abi_version() == 2
    assert q.moe_status_str(q.MOE_OK) == "MOE_OK"
    assert q.moe_status_str(q.MOE_ERR_UNSUPPORTED) == "MOE_ERR_UNSUPPORTED"
    assert q.moe_status_str(99) == "MOE_ERR_UNKNOWN"


GOOD = dict(E=128, top_k=8, D=2048, Dff=768, max_tokens=64)


@pytest.mark.parametrize("change,status", [
    (dict(), q.MOE_OK),
    (dict(bits=8), q.MOE_ERR_UNSUPPORTED),
    (dict(group_size=32), q.MOE_ERR_UNSUPPORTED),
    (dict(D=2047), q.MOE_ERR_UNSUPPORTED),
    (dict(Dff=770), q.MOE_ERR_UNSUPPORTED),
    (dict(Dff=8256), q.MOE_ERR_UNSUPPORTED),
    (dict(E=2048), q.MOE_ERR_UNSUPPORTED),
    (dict(E=64, top_k=17), q.MOE_ERR_UNSUPPORTED),
    (dict(top_k=0), q.MOE_ERR_INVALID_ARG),
    (dict(E=4, top_k=5), q.MOE_ERR_INVALID_ARG),
    (dict(max_tokens=0), q.MOE_ERR_INVALID_ARG),
    (dict(max_tokens=8193), q.MOE_ERR_INVALID_ARG),
    (dict(x_dtype=7), q.MOE_ERR_INVALID_ARG),
    (dict(mma_min_tokens=-1), q.MOE_ERR_INVALID_ARG),
])
def test_config_validation(libpath, change, status):
    args = dict(GOOD)
    bits = change.pop("bits", 4) if "bits" in change else 4
    gs = change.pop("group_size", 64) if "group_size" in change else 64
    xd = change.pop("x_dtype", q.MOE_DTYPE_BF16) if "x_dtype" in change else q.MOE_DTYPE_BF16
    mm = change.pop("mma_min_tokens", 0) if "mma_min_tokens" in change else 0
    args.update(change)
    cfg = q.make_config(args["E"], args["top_k"], args["D"], args["Dff"], args["max_tokens"],
                        x_dtype=xd, router_dtype=q.MOE_DTYPE_BF16, out_dtype=q.MOE_DTYPE_BF16,
                        mma_min_tokens=mm, bits=bits, group_size=gs)
    n = ctypes.c_size_t(0)
    st = q.lib().moe_plan_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n))
    assert st == status
    if status == q.MOE_OK:
        assert n.value > 64 * 8 * (768 + 2048) * 4  # at least h and y scratch


def test_null_arguments_rejected_before_any_cuda_call(libpath):
    L = q.lib()
    planes = q.moe_expert_planes()
    assert L.moe_decode_forward(None, None, None, None, ctypes.byref(planes), 1, 8, None, None) \
        == q.MOE_ERR_INVALID_ARG
    assert L.moe_plan_create(None, None) == q.MOE_ERR_INVALID_ARG
    assert L.moe_plan_check(None) == q.MOE_ERR_INVALID_ARG
    assert L.moe_get_routing(None, *([None] * 8)) == q.MOE_ERR_INVALID_ARG
    assert L.moe_plan_free(None) == q.MOE_OK
    assert L.moe_decode_forward_layers(None, None, 1, 1, 8, None) == q.MOE_ERR_INVALID_ARG
    cfg = q.make_config(**GOOD)
    assert L.moe_plan_workspace_bytes(ctypes.byref(cfg), None) == q.MOE_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(_abi, "LIB_PATH", os.path.join(ROOT, "does-not-exist.so"))
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        _abi.lib()


def test_flag_values_match_the_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    found = {name: 1 << int(bit) for name, bit in re.findall(r"(MOE_FLAG_\w+)\s*=\s*1u\s*<<\s*(\d+)", text)}
    assert found == {name: getattr(q, name) for name in found}
    assert set(found) == {n for n in dir(q) if n.startswith("MOE_FLAG_")}


@pytest.mark.parametrize("flags,status", [
    (q.MOE_FLAG_GROUPED_COHORTS, q.MOE_OK),
    (q.MOE_FLAG_GROUPED_COHORTS | q.MOE_FLAG_F32_DEBUG | q.MOE_FLAG_TRACE, q.MOE_OK),
    (1 << 4, q.MOE_ERR_INVALID_ARG),
])
def test_plan_flags_validated(libpath, flags, status):
    cfg = q.make_config(**GOOD, flags=flags)
    n = ctypes.c_size_t(0)
    assert q.lib().moe_plan_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)) == status


# one documented rule broken at a time, from a valid configuration
_SINGLE_VIOLATIONS = [
    ("bits", 8, q.MOE_ERR_UNSUPPORTED), ("group_size", 128, q.MOE_ERR_UNSUPPORTED),
    ("D", 2048 + 32, q.MOE_ERR_UNSUPPORTED), ("Dff", 768 + 8, q.MOE_ERR_UNSUPPORTED),
    ("D", 16384 + 64, q.MOE_ERR_UNSUPPORTED), ("Dff", 8192 + 64, q.MOE_ERR_UNSUPPORTED),
    ("E", 1025, q.MOE_ERR_UNSUPPORTED), ("top_k", 17, q.MOE_ERR_UNSUPPORTED),
    ("E", 0, q.MOE_ERR_INVALID_ARG), ("top_k", 0, q.MOE_ERR_INVALID_ARG),
    ("D", 0, q.MOE_ERR_INVALID_ARG), ("Dff", -64, q.MOE_ERR_INVALID_ARG),
    ("max_tokens", 0, q.MOE_ERR_INVALID_ARG), ("max_tokens", 8193, q.MOE_ERR_INVALID_ARG),
    ("x_dtype", 2, q.MOE_ERR_INVALID_ARG), ("router_dtype", -1, q.MOE_ERR_INVALID_ARG),
    ("out_dtype", 9, q.MOE_ERR_INVALID_ARG), ("mma_min_tokens", -3, q.MOE_ERR_INVALID_ARG),
    ("flags", 1 << 5, q.MOE_ERR_INVALID_ARG),
    ("activation", 4, q.MOE_ERR_UNSUPPORTED), ("activation", -1, q.MOE_ERR_UNSUPPORTED),
    ("down_bits", 5, q.MOE_ERR_UNSUPPORTED), ("down_bits", 8, q.MOE_ERR_UNSUPPORTED),
]

# the clamp bound and the expert range (each broken alone)
_PAIR_VIOLATIONS = [
    (dict(activation=3, act_limit=0.0), q.MOE_ERR_INVALID_ARG),
    (dict(activation=3, act_limit=-1.0), q.MOE_ERR_INVALID_ARG),
    (dict(activation=3, act_limit=float("nan")), q.MOE_ERR_INVALID_ARG),
    (dict(activation=3, act_limit=float("inf")), q.MOE_ERR_INVALID_ARG),
    (dict(activation=3, act_limit=7.0), q.MOE_OK),
    (dict(activation=1, act_limit=0.0), q.MOE_OK),   # the bound is ignored elsewhere
    (dict(expert_begin=5, expert_end=3), q.MOE_ERR_INVALID_ARG),
    (dict(expert_begin=4, expert_end=4), q.MOE_ERR_INVALID_ARG),
    (dict(expert_begin=-1, expert_end=5), q.MOE_ERR_INVALID_ARG),
    (dict(expert_begin=0, expert_end=129), q.MOE_ERR_INVALID_ARG),
    (dict(expert_begin=0, expert_end=128), q.MOE_OK),
    (dict(expert_begin=64, expert_end=128), q.MOE_OK),
    (dict(down_bits=6), q.MOE_OK),
    (dict(down_bits=4), q.MOE_OK),
]


def _status(**over):
    base = dict(E=128, top_k=8, D=2048, Dff=768, bits=4, group_size=64, max_tokens=64,
                x_dtype=q.MOE_DTYPE_BF16, router_dtype=q.MOE_DTYPE_BF16,
                out_dtype=q.MOE_DTYPE_BF16, flags=0, mma_min_tokens=0, activation=0,
                act_limit=0.0, down_bits=0, expert_begin=0, expert_end=0)
    base.update(over)
    cfg = q.moe_config(base["E"], base["top_k"], base["D"], base["Dff"], base["bits"],
                       base["group_size"], base["max_tokens"], base["x_dtype"],
                       base["router_dtype"], base["out_dtype"], base["flags"],
                       base["mma_min_tokens"], base["activation"], base["act_limit"],
                       base["down_bits"], base["expert_begin"], base["expert_end"])
    n = ctypes.c_size_t(0)
    return q.lib().moe_plan_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), n.value


@pytest.mark.parametrize("field,value,status", _SINGLE_VIOLATIONS,
                         ids=[f"{f}={v}" for f, v, _ in _SINGLE_VIOLATIONS])
def test_each_documented_rule_alone(libpath, field, value, status):
    assert _status(**{field: value})[0] == status


@pytest.mark.parametrize("over,status", _PAIR_VIOLATIONS, ids=[str(o) for o, _ in _PAIR_VIOLATIONS])
def test_layer_variant_and_expert_range_rules(libpath, over, status):
    assert _status(**over)[0] == status


def test_config_struct_matches_the_header():
    """The ctypes struct lists the header's moe_config fields in order."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\}\s*moe_config;", text).group(1)
    fields = re.findall(r"(\w+)\s*;", body)
    assert fields == [f for f, _ in q.moe_config._fields_]


def test_random_valid_configs_are_accepted_and_sized(libpath):
    import random
    r = random.Random(7)
    for _ in range(300):
        E = r.randint(1, 1024)
        cfg = dict(E=E, top_k=r.randint(1, min(E, 16)), D=64 * r.randint(1, 256),
                   Dff=64 * r.randint(1, 128), max_tokens=r.randint(1, 64),
                   x_dtype=r.choice([q.MOE_DTYPE_F32, q.MOE_DTYPE_BF16]),
                   out_dtype=r.choice([q.MOE_DTYPE_F32, q.MOE_DTYPE_BF16]),
                   mma_min_tokens=r.randint(0, 64), activation=r.randint(0, 3),
                   act_limit=r.uniform(0.5, 50.0), down_bits=r.choice([0, 4, 6]))
        if r.random() < 0.5:
            b = r.randint(0, E - 1)
            cfg.update(expert_begin=b, expert_end=r.randint(b + 1, E))
        st, nbytes = _status(**cfg)
        assert st == q.MOE_OK, cfg
        # the workspace holds at least h and y in f32 for every slot
        S = cfg["max_tokens"] * cfg["top_k"]
        assert nbytes >= 4 * S * (cfg["Dff"] + cfg["D"]), cfg
        # and grows with the largest cohort
        if cfg["max_tokens"] < 64:
            assert _status(**dict(cfg, max_tokens=cfg["max_tokens"] + 1))[1] > nbytes, cfg
