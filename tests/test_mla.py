"""Tensor-core (MLA-style) variant: 16..128 query heads sharing one latent KV
row of 576 dims whose first 512 are the value -- the sparse decode case of
"Sparse MLA decode is not batch-invariant" (FlashMLA issue #212).  Parity
against the fp64 oracle, bitwise batch invariance, and the variant's split
constants."""

import dataclasses

import pytest
import torch

from _util import assert_parity, oracle_for
from invariant_decode_attention_gb300 import workloads as W
from oracle import plan as OP

gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import os
    from invariant_decode_attention_gb300 import api as _api
    if not os.path.exists(_api.LIB_PATH):
        from invariant_decode_attention_gb300 import build
        build.build()
    _api.lib()
    return _api


# ---------------------------------------------------------------- CPU: constants

@pytest.mark.parametrize("h_q", [16, 64, 128])
def test_mla_split_constants_match_oracle(api, h_q):
    prob = api.problem(batch=2, num_q_heads=h_q, num_kv_heads=1, head_dim_qk=576,
                       head_dim_v=512, layout="indexed", scale=576 ** -0.5, width=2048,
                       num_blocks=65536, shared_latent=True)
    variant, *consts = api.split_constants(prob)
    assert variant == api.VARIANT_MLA
    assert tuple(consts) == OP.VARIANT_CONSTANTS["mla"]


def test_mla_unsupported_shapes(api):
    for h_q, h_kv, d_qk, d_v in [(8, 1, 576, 512), (256, 1, 576, 512), (128, 2, 576, 512),
                                 (128, 1, 512, 512), (128, 1, 576, 448)]:
        prob = api.problem(batch=1, num_q_heads=h_q, num_kv_heads=h_kv, head_dim_qk=d_qk,
                           head_dim_v=d_v, layout="indexed", scale=0.1, width=8,
                           num_blocks=64, shared_latent=True)
        with pytest.raises(api.DecodeAttnError) as e:
            api.split_constants(prob)
        assert e.value.status == api.ERR_UNSUPPORTED


def test_mla_e4m3_latent_takes_the_mla_variant(api):
    prob = api.problem(batch=2, num_q_heads=128, num_kv_heads=1, head_dim_qk=576,
                       head_dim_v=512, layout="indexed", scale=576 ** -0.5, width=2048,
                       num_blocks=65536, shared_latent=True, kv_dtype=api.KV_FP8_E4M3,
                       k_scale=1 / 64, v_scale=1 / 32)
    variant, *consts = api.split_constants(prob)
    assert variant == api.VARIANT_MLA
    assert tuple(consts) == OP.VARIANT_CONSTANTS["mla"]
    nvfp4 = api.problem(batch=2, num_q_heads=128, num_kv_heads=1, head_dim_qk=576,
                        head_dim_v=512, layout="indexed", scale=576 ** -0.5, width=2048,
                        num_blocks=65536, shared_latent=True, kv_dtype=api.KV_NVFP4,
                        k_scale=1.0, v_scale=1.0)
    with pytest.raises(api.DecodeAttnError) as e:
        api.split_constants(nvfp4)
    assert e.value.status == api.ERR_UNSUPPORTED


# ---------------------------------------------------------------- GPU: parity

@gpu
@pytest.mark.parametrize("layout", [W.INDEXED, W.PAGED, W.CONTIGUOUS])
def test_mla_small_all_layouts(api, layout):
    lens = [1, 31, 32, 33, 64, 700, 0, 2048]
    wl = W.make(layout, lens, H_q=128, H_kv=1, D_qk=576, D_v=512, latent=True,
                page_size=64, num_slots=5000, width=2048 if layout != W.PAGED else None,
                seed=40)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
@pytest.mark.parametrize("h_q", [16, 64, 100])
def test_mla_fewer_heads(api, h_q):
    wl = W.make(W.INDEXED, [300, 1500], H_q=h_q, H_kv=1, D_qk=576, D_v=512, latent=True,
                num_slots=4000, width=2048, seed=h_q)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_mla_config_full(api):
    wl = W.mla_sparse()
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_mla_balanced_is_correct(api):
    wl = W.mla_sparse()
    out, lse = api.run_workload(wl.to("cuda"), policy=api.BALANCED)
    rows = list(range(0, 64, 7))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_mla_out_of_range_index_sets_error(api):
    wl = W.make(W.INDEXED, [40, 300], H_q=128, H_kv=1, D_qk=576, D_v=512, latent=True,
                num_slots=1000, width=512, seed=77)
    wl.table[1, 5] = 5000
    g = wl.to("cuda")
    prob = api.problem_for(g)
    ws = api.workspace(prob)
    out = torch.empty((2, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 128), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, None, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    assert api.read_error(pl) & api.DEVERR_INDEX
    assert not api.read_error(pl) & api.DEVERR_TIMEOUT
    ro, rl = oracle_for(wl, rows=[0])
    assert_parity(out, lse, ro, rl, rows=[0])


# ---------------------------------------------------------------- GPU: invariance

@gpu
def test_mla_row_solo_vs_batch(api):
    wl = W.mla_sparse()
    g = wl.to("cuda")
    o, l = api.run_workload(g)
    for r in (0, 21, 63):
        solo = W.Workload("solo", W.INDEXED, g.q[r:r + 1].contiguous(), g.k, None,
                          g.lengths[r:r + 1].contiguous(), g.table[r:r + 1].contiguous(),
                          0, 128, 1, 576, 512, wl.scale)
        o1, l1 = api.run_workload(solo)
        assert torch.equal(o1[0], o[r]) and torch.equal(l1[0], l[r])
    o2, l2 = api.run_workload(g)
    assert torch.equal(o2, o) and torch.equal(l2, l)


@gpu
@pytest.mark.parametrize("fp8", [False, True])
def test_mla_q_alignment_does_not_change_bits(api, fp8):
    """q 32-byte aligned (32-byte row loads) or only 16-byte aligned (16-byte
    loads): the same bits."""
    wl = W.make(W.INDEXED, [300, 1500, 2048], H_q=128, H_kv=1, D_qk=576, D_v=512, latent=True,
                num_slots=4000, width=2048, seed=45)
    if fp8:
        wl = W.quantize_fp8(wl)
    g = wl.to("cuda")
    o32, l32 = [t.clone() for t in api.run_workload(g)]
    assert g.q.data_ptr() % 32 == 0
    store = torch.empty(g.q.numel() + 16, dtype=torch.bfloat16, device="cuda")
    q16 = store[8:8 + g.q.numel()].view_as(g.q)
    q16.copy_(g.q)
    assert q16.data_ptr() % 32 == 16
    o16, l16 = api.run_workload(dataclasses.replace(g, q=q16))
    assert torch.equal(o16, o32) and torch.equal(l16, l32)


@gpu
@pytest.mark.parametrize("name", ["mla_sparse", "mla_sparse_extra"])
def test_mla_repeated_runs_bitwise(api, name):
    """The same inputs give the same bits on every run, one workspace reused
    back to back: a result read before the tensor core finished with it (or a
    stage refilled early) shows up as a run that differs from the first."""
    wl = getattr(W, name)().to("cuda")
    ws = api.workspace(api.problem_for(wl), "cuda")
    out0, lse0 = [t.clone() for t in api.run_workload(wl, ws=ws)]
    for _ in range(16):
        out, lse = api.run_workload(wl, ws=ws)
        assert torch.equal(out, out0) and torch.equal(lse, lse0)


# ---------------------------------------------------------------- E4M3 latent cache
# One byte per latent element: the scores take k_scale times the row's 576
# bytes, the values v_scale times its first 512.  The producer gathers the
# bytes, the converter widens them to f16 in the operand stage (exact), Q is
# prescaled per row by a power of two into f16's range, the MMAs run on f16.

def _fp8(wl, k_scale=1 / 64, v_scale=1 / 32):
    return W.quantize_fp8(wl, k_scale=k_scale, v_scale=v_scale)


@gpu
@pytest.mark.parametrize("layout", [W.INDEXED, W.PAGED, W.CONTIGUOUS])
def test_mla_fp8_small_all_layouts(api, layout):
    lens = [1, 31, 32, 33, 64, 700, 0, 2048]
    wl = _fp8(W.make(layout, lens, H_q=128, H_kv=1, D_qk=576, D_v=512, latent=True,
                     page_size=64, num_slots=5000, width=2048 if layout != W.PAGED else None,
                     seed=41))
    assert api.split_constants(api.problem_for(wl))[0] == api.VARIANT_MLA
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
@pytest.mark.parametrize("h_q", [16, 64, 100])
def test_mla_fp8_fewer_heads(api, h_q):
    wl = _fp8(W.make(W.INDEXED, [300, 1500], H_q=h_q, H_kv=1, D_qk=576, D_v=512, latent=True,
                     num_slots=4000, width=2048, seed=h_q + 1))
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_mla_fp8_config_full(api):
    wl = W.mla_sparse_fp8()
    out, lse = api.run_workload(wl.to("cuda"))
    rows = list(range(0, 64, 3))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)


@gpu
def test_mla_fp8_query_scales(api):
    # query rows of very different magnitudes (the per-row power-of-two
    # prescale into f16), one head's row all zeros, and equal scales
    wl = W.make(W.INDEXED, [500, 2000], H_q=128, H_kv=1, D_qk=576, D_v=512, latent=True,
                num_slots=4000, width=2048, seed=902)
    q = wl.q.float()
    q[0, :8] *= 2.0 ** 6
    q[0, 8:16] *= 2.0 ** -20
    q[1, 3] = 0.0
    wl = _fp8(dataclasses.replace(wl, q=q.to(torch.bfloat16)), k_scale=1 / 64, v_scale=1 / 64)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@gpu
def test_mla_fp8_out_of_range_index_sets_error(api):
    wl = _fp8(W.make(W.INDEXED, [40, 300], H_q=128, H_kv=1, D_qk=576, D_v=512, latent=True,
                     num_slots=1000, width=512, seed=78))
    wl.table[1, 5] = 5000
    g = wl.to("cuda")
    prob = api.problem_for(g)
    ws = api.workspace(prob)
    out = torch.empty((2, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 128), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, None, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    err = api.read_error(pl)
    assert err & api.DEVERR_INDEX and not err & api.DEVERR_TIMEOUT
    ro, rl = oracle_for(wl, rows=[0])
    assert_parity(out, lse, ro, rl, rows=[0])


@gpu
def test_mla_fp8_row_solo_vs_batch_and_repeat(api):
    wl = W.mla_sparse_fp8()
    g = wl.to("cuda")
    ws = api.workspace(api.problem_for(g), "cuda")
    o, l = [t.clone() for t in api.run_workload(g, ws=ws)]
    for _ in range(8):
        o2, l2 = api.run_workload(g, ws=ws)
        assert torch.equal(o2, o) and torch.equal(l2, l)
    for r in (0, 21, 63):
        solo = dataclasses.replace(g, name="solo", q=g.q[r:r + 1].contiguous(),
                                   lengths=g.lengths[r:r + 1].contiguous(),
                                   table=g.table[r:r + 1].contiguous())
        o1, l1 = api.run_workload(solo)
        assert torch.equal(o1[0], o[r]) and torch.equal(l1[0], l[r])
