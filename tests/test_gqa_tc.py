"""Tensor-core variant for grouped-query attention over separate K and V:
16..128 query heads per KV head at head dim 128 (the multi-head QK^T and PV
contractions go to tcgen05; "Sparse MLA decode is not batch-invariant",
FlashMLA issue #212, Summary: the op is per row over its own KV list, the
head layout is the caller's).  Parity against the fp64 oracle on every
layout and page size (box copies for contiguous caches and pages of a
multiple of 16 entries, gathers otherwise), runs of one-tile units (the copy
pipeline crossing a unit boundary every tile), bitwise batch invariance (a
ragged sweep, solo against batched rows, repeats), and the variant choice
(CPU checks need no GPU)."""

import ctypes
import dataclasses

import pytest
import torch

from _util import assert_parity, oracle_for
from invariant_decode_attention_gb300 import workloads as W
from oracle import plan as OP

gpu = pytest.mark.gpu

EDGE = [0, 1, 2, 15, 16, 17, 63, 64, 65, 511, 512, 513, 1000, 4097]


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


def _prob(api, g, d=128, **kw):
    base = dict(batch=3, num_q_heads=2 * g, num_kv_heads=2, head_dim_qk=d, layout="paged",
                scale=0.1, page_size=16, width=8, num_blocks=100)
    base.update(kw)
    return api.problem(**base)


# ---------------------------------------------------------------- CPU: choice

@pytest.mark.parametrize("g", [16, 17, 32, 64, 128])
def test_tensor_core_variant_for_large_groups(api, g):
    variant, *consts = api.split_constants(_prob(api, g))
    assert variant == api.VARIANT_GQA_TC
    assert tuple(consts) == OP.VARIANT_CONSTANTS["gqa_tc"]


def test_e4m3_cache_takes_the_tensor_core_variant(api):
    prob = _prob(api, 32, kv_dtype=api.KV_FP8_E4M3, k_scale=0.5, v_scale=0.25)
    assert api.split_constants(prob)[0] == api.VARIANT_GQA_TC


def test_nvfp4_cache_takes_the_tensor_core_variant_with_even_kv_heads(api):
    even = _prob(api, 32, kv_dtype=api.KV_NVFP4, k_scale=0.5, v_scale=0.25)
    assert api.split_constants(even)[0] == api.VARIANT_GQA_TC
    odd = _prob(api, 16, num_q_heads=48, num_kv_heads=3, kv_dtype=api.KV_NVFP4, k_scale=1.0,
                v_scale=1.0)
    assert api.split_constants(odd)[0] == api.VARIANT_FMA


def test_other_large_group_configs_stay_on_cuda_cores(api):
    for prob in (_prob(api, 16, d=64), _prob(api, 15),
                 _prob(api, 16, num_q_heads=16, num_kv_heads=1, kv_dtype=api.KV_NVFP4,
                       k_scale=1.0, v_scale=1.0),
                 _prob(api, 16, extra_width=8, extra_num_blocks=10)):
        variant, *consts = api.split_constants(prob)
        assert variant == api.VARIANT_FMA


# ---------------------------------------------------------------- GPU: parity

@gpu
@pytest.mark.parametrize("layout,page", [(W.PAGED, 16), (W.PAGED, 64), (W.PAGED, 100),
                                         (W.CONTIGUOUS, 0), (W.INDEXED, 0)])
@pytest.mark.parametrize("g", [16, 32])
def test_tc_parity_layouts(api, layout, page, g):
    wl = W.make(layout, EDGE, H_q=2 * g, H_kv=2, D_qk=128, page_size=page or 16,
                num_slots=6000, seed=500 + g + page)
    prob = api.problem_for(wl)
    assert api.split_constants(prob)[0] == api.VARIANT_GQA_TC
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
@pytest.mark.parametrize("g", [20, 48, 64, 128])
def test_tc_parity_group_sizes(api, g):
    wl = W.make(W.PAGED, [1, 77, 1024, 3000], H_q=g, H_kv=1, D_qk=128, page_size=32,
                seed=600 + g)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_tc_gqa16_config(api):
    wl = W.gqa16_paged()
    out, lse = api.run_workload(wl.to("cuda"))
    rows = list(range(0, wl.B, 5))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_tc_balanced_is_correct(api):
    wl = W.gqa16_paged()
    out, lse = api.run_workload(wl.to("cuda"), policy=api.BALANCED)
    rows = [0, 9, 31]
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_tc_out_of_range_page_sets_error(api):
    wl = W.make(W.PAGED, [40, 300], H_q=32, H_kv=2, D_qk=128, page_size=16, seed=77)
    wl.table[1, 3] = 10 ** 6
    g = wl.to("cuda")
    prob = api.problem_for(g)
    ws = api.workspace(prob)
    out = torch.empty((2, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 32), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    err = api.read_error(pl)
    assert err & api.DEVERR_INDEX and not err & api.DEVERR_TIMEOUT
    ro, rl = oracle_for(wl, rows=[0])
    assert_parity(out, lse, ro, rl, rows=[0])


# ---------------------------------------------------------------- GPU: invariance

@gpu
def test_tc_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweep(range(1, 257), H_q=128)
    o_solo, l_solo = api.run_workload(sweep.solo())
    ro, rl = oracle_for(sweep.solo_cpu())
    assert_parity(o_solo, l_solo, ro, rl)
    for i in range(len(sweep.sizes)):
        wl, pos = sweep.batch(i)
        o, l = api.run_workload(wl)
        assert torch.equal(o[pos], o_solo[0]), f"B={wl.B} pos={pos}"
        assert torch.equal(l[pos], l_solo[0]), f"B={wl.B} pos={pos}"
        if i in (0, 63, 255):
            for _ in range(3):
                o2, l2 = api.run_workload(wl)
                assert torch.equal(o2, o) and torch.equal(l2, l)


@gpu
def test_tc_repeated_runs_and_solo_rows(api):
    wl = W.gqa16_paged().to("cuda")
    ws = api.workspace(api.problem_for(wl), "cuda")
    o0, l0 = [t.clone() for t in api.run_workload(wl, ws=ws)]
    for _ in range(16):
        o, l = api.run_workload(wl, ws=ws)
        assert torch.equal(o, o0) and torch.equal(l, l0)
    for r in (0, 13, 31):
        solo = W.Workload("solo", W.PAGED, wl.q[r:r + 1].contiguous(), wl.k, wl.v,
                          wl.lengths[r:r + 1].contiguous(), wl.table[r:r + 1].contiguous(),
                          wl.page_size, wl.H_q, wl.H_kv, 128, 128, wl.scale)
        o1, l1 = api.run_workload(solo)
        assert torch.equal(o1[0], o0[r]) and torch.equal(l1[0], l0[r])


@gpu
def test_tc_runs_of_one_tile_units(api):
    # hundreds of rows of at most one tile each: a CTA takes many one-tile
    # units in a row, so its copy pipeline crosses unit boundaries every tile
    lens = [1 + (37 * i) % 64 for i in range(300)] + [5000, 0, 130]
    wl = W.make(W.PAGED, lens, H_q=64, H_kv=4, D_qk=128, page_size=16, seed=99)
    g = wl.to("cuda")
    prob = api.problem_for(g)
    ws = api.workspace(prob)
    out = torch.empty((wl.B, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.B, 64), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    assert api.read_error(pl) == 0
    rows = [0, 1, 63, 150, 299, 300, 301, 302]
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


# ---------------------------------------------------------------- E4M3 caches
# The same variant on one-byte caches: the bytes are converted to f16 in
# shared memory (exact), Q is prescaled per row by a power of two into f16's
# range, the MMAs run on f16 operands; the oracle decodes the same bytes.

@gpu
@pytest.mark.parametrize("layout,page", [(W.PAGED, 16), (W.PAGED, 100), (W.CONTIGUOUS, 0),
                                         (W.INDEXED, 0)])
@pytest.mark.parametrize("g", [16, 32])
def test_tc_fp8_parity_layouts(api, layout, page, g):
    base = W.make(layout, EDGE, H_q=2 * g, H_kv=2, D_qk=128, page_size=page or 16,
                  num_slots=6000, seed=700 + g + page)
    wl = W.quantize_fp8(base, k_scale=0.37, v_scale=3.0)
    assert api.split_constants(api.problem_for(wl))[0] == api.VARIANT_GQA_TC
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
@pytest.mark.parametrize("g", [20, 64, 128])
def test_tc_fp8_parity_group_sizes(api, g):
    wl = W.quantize_fp8(W.make(W.PAGED, [1, 77, 1024, 3000], H_q=g, H_kv=1, D_qk=128,
                               page_size=32, seed=800 + g))
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_tc_fp8_query_scales(api):
    # query rows of very different magnitudes (the per-row power-of-two
    # prescale into f16), and a row of zeros
    wl = W.quantize_fp8(W.make(W.PAGED, [500, 2000], H_q=32, H_kv=2, D_qk=128, page_size=16,
                               seed=901))
    q = wl.q.float()
    q[0, :8] *= 2.0 ** 6
    q[0, 8:16] *= 2.0 ** -20
    q[1, 3] = 0.0
    wl = dataclasses.replace(wl, q=q.to(torch.bfloat16))
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_tc_fp8_gqa16_config(api):
    wl = W.quantize_fp8(W.gqa16_paged())
    out, lse = api.run_workload(wl.to("cuda"))
    rows = list(range(0, wl.B, 5))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_tc_fp8_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweep(range(1, 257), H_q=128, kv_fp8=True)
    o_solo, l_solo = api.run_workload(sweep.solo())
    ro, rl = oracle_for(sweep.solo_cpu())
    assert_parity(o_solo, l_solo, ro, rl)
    for i in range(len(sweep.sizes)):
        wl, pos = sweep.batch(i)
        o, l = api.run_workload(wl)
        assert torch.equal(o[pos], o_solo[0]), f"B={wl.B} pos={pos}"
        assert torch.equal(l[pos], l_solo[0]), f"B={wl.B} pos={pos}"
        if i in (0, 63, 255):
            for _ in range(3):
                o2, l2 = api.run_workload(wl)
                assert torch.equal(o2, o) and torch.equal(l2, l)


@gpu
def test_tc_fp8_runs_of_one_tile_units(api):
    lens = [1 + (37 * i) % 64 for i in range(300)] + [5000, 0, 130]
    wl = W.quantize_fp8(W.make(W.PAGED, lens, H_q=64, H_kv=4, D_qk=128, page_size=16, seed=98))
    out, lse = api.run_workload(wl.to("cuda"))
    rows = [0, 1, 63, 150, 299, 300, 301, 302]
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


# ---------------------------------------------------------------- NVFP4 caches
# E2M1 codes with one E4M3 scale per 16 elements: code and block scale are
# each exact in f16 and so is their product, written as f16 operands by the
# converter; the scale rows of two neighbouring KV heads are copied together,
# so the variant takes an even number of KV heads.

@gpu
@pytest.mark.parametrize("layout,page", [(W.PAGED, 16), (W.PAGED, 100), (W.CONTIGUOUS, 0),
                                         (W.INDEXED, 0)])
@pytest.mark.parametrize("g,h_kv", [(16, 2), (32, 4)])
def test_tc_nvfp4_parity_layouts(api, layout, page, g, h_kv):
    base = W.make(layout, EDGE, H_q=h_kv * g, H_kv=h_kv, D_qk=128, page_size=page or 16,
                  num_slots=6000, seed=1100 + g + page, draw_kv=False)
    wl = W.nvfp4_kv(base, k_scale=0.37, v_scale=3.0, seed=1101 + g + page)
    assert api.split_constants(api.problem_for(wl))[0] == api.VARIANT_GQA_TC
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
@pytest.mark.parametrize("g", [20, 64, 128])
def test_tc_nvfp4_parity_group_sizes(api, g):
    wl = W.nvfp4_kv(W.make(W.PAGED, [1, 77, 1024, 3000], H_q=2 * g, H_kv=2, D_qk=128,
                           page_size=32, seed=1200 + g, draw_kv=False), seed=1201 + g)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_tc_nvfp4_block_scales_over_the_whole_e4m3_range(api):
    # block scales from the smallest subnormal (2^-9) to the largest finite
    # value (448), of both signs: every code x scale product (2^-10 .. 2688)
    # must still be exact in f16; global scales keep the scores moderate
    wl = W.nvfp4_kv(W.make(W.PAGED, [700, 2500, 64], H_q=32, H_kv=2, D_qk=128, page_size=16,
                           seed=1300, draw_kv=False), k_scale=2.0 ** -9, v_scale=2.0 ** -8,
                    seed=1301)
    g = torch.Generator().manual_seed(1302)
    for name in ("k_blocks", "v_blocks"):
        b = getattr(wl, name)
        mag = torch.randint(1, 0x7F, b.shape, generator=g, dtype=torch.int32)  # 0x01 .. 0x7E
        sign = torch.randint(0, 2, b.shape, generator=g, dtype=torch.int32) << 7
        b = (mag | sign).to(torch.uint8)
        b.view(-1)[:4] = torch.tensor([0x01, 0x7E, 0x81, 0xFE], dtype=torch.uint8)
        wl = dataclasses.replace(wl, **{name: b})
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_tc_nvfp4_gqa16_config(api):
    wl = W.gqa16_paged_nvfp4()
    assert api.split_constants(api.problem_for(wl))[0] == api.VARIANT_GQA_TC
    out, lse = api.run_workload(wl.to("cuda"))
    rows = list(range(0, wl.B, 5))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_tc_nvfp4_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweep(range(1, 257), H_q=128, kv_nvfp4=True)
    o_solo, l_solo = api.run_workload(sweep.solo())
    ro, rl = oracle_for(sweep.solo_cpu())
    assert_parity(o_solo, l_solo, ro, rl)
    for i in range(len(sweep.sizes)):
        wl, pos = sweep.batch(i)
        o, l = api.run_workload(wl)
        assert torch.equal(o[pos], o_solo[0]), f"B={wl.B} pos={pos}"
        assert torch.equal(l[pos], l_solo[0]), f"B={wl.B} pos={pos}"
        if i in (0, 63, 255):
            for _ in range(3):
                o2, l2 = api.run_workload(wl)
                assert torch.equal(o2, o) and torch.equal(l2, l)


@gpu
def test_tc_nvfp4_runs_of_one_tile_units(api):
    lens = [1 + (37 * i) % 64 for i in range(300)] + [5000, 0, 130]
    wl = W.nvfp4_kv(W.make(W.PAGED, lens, H_q=64, H_kv=4, D_qk=128, page_size=16, seed=97,
                           draw_kv=False), seed=96)
    out, lse = api.run_workload(wl.to("cuda"))
    rows = [0, 1, 63, 150, 299, 300, 301, 302]
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


# ---------------------------------------------------------------- empty cache

@gpu
@pytest.mark.parametrize("kv", ["bf16", "fp8", "nvfp4"])
def test_tc_empty_cache(api, kv):
    # a cache of zero rows (every length 0): the tensor maps stand on a zero
    # tile, no unit has tiles, every output row is 0 with lse = -inf
    wl = W.make(W.INDEXED, [0, 0, 0], H_q=32, H_kv=2, D_qk=128, num_slots=1, seed=1400)
    if kv == "fp8":
        wl = W.quantize_fp8(wl)
    elif kv == "nvfp4":
        wl = W.nvfp4_kv(wl, seed=1401)
    g = wl.to("cuda")
    prob = api.problem_for(g)
    prob.num_blocks = 0
    assert api.split_constants(prob)[0] == api.VARIANT_GQA_TC
    ws = api.workspace(prob)
    out = torch.full((3, 32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((3, 32), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    assert api.read_error(pl) == 0
    assert torch.all(out == 0) and torch.all(lse == float("-inf"))
