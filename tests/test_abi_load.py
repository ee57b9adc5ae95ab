"""The C-ABI library loads, exports every symbol the header declares, reports
the split constants the oracle restates, and rejects bad arguments with the
documented status codes.  No compute calls: runs without a GPU."""

import ctypes
import os
import re

import pytest

from oracle import plan as OP

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("decode_attn.h", "nvfp4_mm.h")]


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    if not os.path.exists(_api.LIB_PATH):
        from invariant_decode_attention_gb300 import build
        build.build()
    _api.lib()
    return _api


def header_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b((?:decode_attn|nvfp4_mm)\w*)\s*\(",
                                text, re.M))
    return sorted(names)


def test_every_header_is_covered():
    assert sorted(os.listdir(os.path.join(ROOT, "include"))) == sorted(
        os.path.basename(h) for h in HEADERS)


def test_exports_every_declared_symbol(api):
    declared = header_functions()
    assert declared, "no declarations parsed"
    assert sorted(api.EXPORTS) == declared
    L = api.lib()
    for name in declared:
        assert hasattr(L, name), name


def test_version_names_the_constants(api):
    v = api.version()
    t, mn, mx = OP.VARIANT_CONSTANTS["fma"]
    assert f"fma: tile={t} min_tiles={mn} max_splits={mx}" in v
    t, mn, mx = OP.VARIANT_CONSTANTS["mla"]
    assert f"mla: tile={t} min_tiles={mn} max_splits={mx}" in v
    assert f"fixed_overhead={OP.BALANCED_FIXED_OVERHEAD}" in v


@pytest.mark.parametrize("g,d", [(g, d) for d in (64, 128) for g in (1, 2, 3, 4, 5, 8, 12, 15)])
def test_fma_split_constants_match_oracle(api, g, d):
    prob = api.problem(batch=3, num_q_heads=2 * g, num_kv_heads=2, head_dim_qk=d,
                       layout="paged", scale=0.1, page_size=16, width=8, num_blocks=100)
    variant, *consts = api.split_constants(prob)
    assert variant == api.VARIANT_FMA
    assert tuple(consts) == OP.VARIANT_CONSTANTS["fma"]


def test_unsupported_head_configs(api):
    for g, d in [(4, 96), (4, 256), (8, 32), (129, 128)]:
        prob = api.problem(batch=1, num_q_heads=g, num_kv_heads=1, head_dim_qk=d,
                           layout="contiguous", scale=1.0, width=4)
        with pytest.raises(api.DecodeAttnError) as e:
            api.split_constants(prob)
        assert e.value.status == api.ERR_UNSUPPORTED


def test_invalid_problems(api):
    L = api.lib()
    n = ctypes.c_size_t()
    assert L.decode_attn_workspace_bytes(None, ctypes.byref(n)) == api.ERR_INVALID_ARG
    bad = [
        dict(num_q_heads=6, num_kv_heads=4),        # H_q not a multiple of H_kv
        dict(batch=-1),
        dict(layout=7),
        dict(layout="paged", page_size=0),
        dict(scale=float("inf")),
        dict(width=-3),
    ]
    for kw in bad:
        args = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim_qk=128,
                    layout="contiguous", scale=0.1, width=16, page_size=16, num_blocks=4)
        args.update(kw)
        prob = api.problem(**args)
        assert L.decode_attn_workspace_bytes(ctypes.byref(prob), ctypes.byref(n)) == \
            api.ERR_INVALID_ARG, kw


def test_workspace_size_and_plan_argument_checks(api):
    prob = api.problem(batch=32, num_q_heads=32, num_kv_heads=8, head_dim_qk=128,
                       layout="paged", scale=0.1, page_size=16, width=512, num_blocks=9000)
    nbytes = api.workspace_bytes(prob)
    ms = OP.VARIANT_CONSTANTS["fma"][2]
    # partial outputs dominate: B * max_splits * H_q * D_v fp32
    assert nbytes >= 32 * ms * 32 * 128 * 4
    L = api.lib()
    plan = api.DaPlan()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    rc = L.decode_attn_plan(ctypes.byref(prob), api.INVARIANT, fake, fake, nbytes - 1,
                            ctypes.byref(plan), None)
    assert rc == api.ERR_WORKSPACE
    rc = L.decode_attn_plan(ctypes.byref(prob), api.INVARIANT, fake, ctypes.c_void_p((1 << 20) + 8),
                            nbytes, ctypes.byref(plan), None)
    assert rc == api.ERR_WORKSPACE  # misaligned
    rc = L.decode_attn_plan(ctypes.byref(prob), 5, fake, fake, nbytes, ctypes.byref(plan), None)
    assert rc == api.ERR_INVALID_ARG  # unknown policy
    rc = L.decode_attn_plan(ctypes.byref(prob), api.INVARIANT, None, fake, nbytes,
                            ctypes.byref(plan), None)
    assert rc == api.ERR_INVALID_ARG  # no lengths


def test_status_strings(api):
    L = api.lib()
    for code in range(5):
        assert L.decode_attn_status_string(code)
    assert L.decode_attn_status_string(99) == b"unknown status"
