"""NVFP4 key/value caches (E2M1 codes, one E4M3 scale per 16 elements of a
head row, one fp32 scale per cache): the CUDA-core split kernel against the
fp64 oracle decoding the same bytes, bitwise batch invariance (a ragged
sweep, solo against batched rows, repeats), and the argument rules (CPU
checks need no GPU).  The pages run NVFP4 checkpoints ("Sparse MLA decode is
not batch-invariant", Environment; "Greedy outputs depend on batch
composition", Observation) without naming a cache format; the layout is the
library's reading, stated in include/decode_attn.h."""

import ctypes

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
@pytest.mark.parametrize("g,d", [(1, 64), (2, 128), (4, 128), (8, 64), (8, 128), (3, 64)])
def test_nvfp4_parity(api, layout, g, d):
    base = W.make(layout, LENGTHS, H_q=2 * g, H_kv=2, D_qk=d, page_size=16,
                  num_slots=30000 if layout == W.INDEXED else None, seed=60 + g + d,
                  draw_kv=False)
    wl = W.nvfp4_kv(base, k_scale=0.37, v_scale=3.0, seed=61 + g + d)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_nvfp4_gqa_paged_config(api):
    wl = W.gqa_paged_nvfp4()
    out, lse = api.run_workload(wl.to("cuda"))
    rows = list(range(0, 32, 3))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_nvfp4_row_solo_vs_batch_and_repeat(api):
    wl = W.nvfp4_kv(W.make(W.PAGED, [4096, 300, 70000, 1, 9000], H_q=32, H_kv=8, D_qk=128,
                           page_size=16, seed=62, draw_kv=False), seed=63)
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
                          kv_nvfp4=True, k_blocks=g.k_blocks, v_blocks=g.v_blocks,
                          k_scale=g.k_scale, v_scale=g.v_scale)
        so, sl = api.run_workload(solo)
        assert torch.equal(so[0], o[r]) and torch.equal(sl[0], l[r])


@gpu
def test_nvfp4_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweep(range(1, 257), kv_nvfp4=True)
    o_solo, l_solo = api.run_workload(sweep.solo())
    ro, rl = oracle_for(sweep.solo_cpu())
    assert_parity(o_solo, l_solo, ro, rl)
    for i in range(len(sweep.sizes)):
        wl, pos = sweep.batch(i)
        o, l = api.run_workload(wl)
        assert torch.equal(o[pos], o_solo[0]), f"B={wl.B} pos={pos}"
        assert torch.equal(l[pos], l_solo[0]), f"B={wl.B} pos={pos}"


def _prob(api, **kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim_qk=128, layout="paged",
                scale=0.1, page_size=16, width=4, num_blocks=8, kv_dtype=api.KV_NVFP4,
                k_scale=0.5, v_scale=0.5)
    base.update(kw)
    return api.problem(**base)


def test_nvfp4_argument_rules(api):
    L = api.lib()
    ok = _prob(api)
    assert L.decode_attn_split_constants(ctypes.byref(ok), None, None, None, None) == 0
    bad_cases = [
        (_prob(api, k_scale=0.0), api.ERR_INVALID_ARG),
        (_prob(api, v_scale=float("inf")), api.ERR_INVALID_ARG),
        (_prob(api, num_q_heads=128, num_kv_heads=1, head_dim_qk=576, head_dim_v=512,
               shared_latent=True, layout="indexed"), api.ERR_UNSUPPORTED),
        (_prob(api, extra_width=16, extra_num_blocks=4), api.ERR_UNSUPPORTED),
        (_prob(api, head_dim_qk=96), api.ERR_UNSUPPORTED),
    ]
    for prob, want in bad_cases:
        assert L.decode_attn_split_constants(ctypes.byref(prob), None, None, None, None) == want
