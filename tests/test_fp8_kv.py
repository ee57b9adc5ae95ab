"""E4M3 (FP8) key/value caches: the CUDA-core split kernel on byte caches
against the fp64 oracle decoding the same bytes, bitwise batch invariance,
repeat runs, and the argument rules (CPU checks need no GPU)."""

import pytest
import torch

from _util import assert_parity, oracle_for
from invariant_decode_attention_gb300 import workloads as W

gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


LENGTHS = [0, 1, 15, 16, 17, 63, 64, 65, 1000, 5000, 20000]


@gpu
@pytest.mark.parametrize("layout", [W.PAGED, W.CONTIGUOUS, W.INDEXED])
@pytest.mark.parametrize("g,d", [(1, 64), (2, 128), (4, 128), (8, 64)])
def test_fp8_parity(api, layout, g, d):
    base = W.make(layout, LENGTHS, H_q=2 * g, H_kv=2, D_qk=d, page_size=16,
                  num_slots=30000 if layout == W.INDEXED else None, seed=50 + g + d)
    wl = W.quantize_fp8(base, k_scale=0.37, v_scale=3.0)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_fp8_gqa_paged_config(api):
    wl = W.gqa_paged_fp8()
    out, lse = api.run_workload(wl.to("cuda"))
    rows = list(range(0, 32, 3))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_fp8_row_solo_vs_batch_and_repeat(api):
    wl = W.quantize_fp8(W.make(W.PAGED, [4096, 300, 70000, 1, 9000], H_q=32, H_kv=8, D_qk=128,
                               page_size=16, seed=61))
    g = wl.to("cuda")
    ws = api.workspace(api.problem_for(g), "cuda")
    o, l = [t.clone() for t in api.run_workload(g, ws=ws)]
    for _ in range(4):
        o2, l2 = api.run_workload(g, ws=ws)
        assert torch.equal(o2, o) and torch.equal(l2, l)
    for r in (0, 2, 4):
        solo = W.Workload("solo", W.PAGED, g.q[r:r + 1].contiguous(), g.k, g.v,
                          g.lengths[r:r + 1].contiguous(), g.table[r:r + 1].contiguous(),
                          g.page_size, g.H_q, g.H_kv, g.D_qk, g.D_v, g.scale,
                          kv_fp8=True, k_scale=g.k_scale, v_scale=g.v_scale)
        so, sl = api.run_workload(solo)
        assert torch.equal(so[0], o[r]) and torch.equal(sl[0], l[r])


def _prob(api, **kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim_qk=128, layout="paged",
                scale=0.1, page_size=16, width=4, num_blocks=8, kv_dtype=api.KV_FP8_E4M3,
                k_scale=0.5, v_scale=0.5)
    base.update(kw)
    return api.problem(**base)


def test_fp8_argument_rules(api):
    ok = _prob(api)
    assert api.lib().decode_attn_split_constants(__import__("ctypes").byref(ok), None, None, None,
                                                 None) == 0
    bad_cases = [
        (_prob(api, k_scale=0.0), 1), (_prob(api, v_scale=float("nan")), 1),
        (_prob(api, kv_dtype=7), 1),
        (_prob(api, num_q_heads=128, num_kv_heads=1, head_dim_qk=576, head_dim_v=512,
               shared_latent=True, layout="indexed", extra_width=16, extra_num_blocks=4),
         2),                                                  # second latent source: unsupported
        (_prob(api, extra_width=16, extra_num_blocks=4), 2),  # second source: unsupported
    ]
    import ctypes
    for prob, want in bad_cases:
        assert api.lib().decode_attn_split_constants(ctypes.byref(prob), None, None, None,
                                                     None) == want
