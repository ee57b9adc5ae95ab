"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, within the bar stated in tests/_util.py."""

import numpy as np
import pytest
import torch

from _util import assert_parity, oracle_for
from invariant_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


EDGE_LENGTHS = [0, 1, 2, 15, 16, 17, 63, 64, 65, 511, 512, 513, 1000, 4097]


def test_tiny_config(api):
    wl = W.tiny()
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@pytest.mark.parametrize("layout", [W.CONTIGUOUS, W.PAGED, W.INDEXED])
@pytest.mark.parametrize("g,d", [(1, 64), (2, 128), (4, 128), (8, 64), (4, 64), (1, 128)])
def test_edge_lengths_all_layouts(api, layout, g, d):
    wl = W.make(layout, EDGE_LENGTHS, H_q=2 * g, H_kv=2, D_qk=d, page_size=16,
                num_slots=6000, seed=100 + g + d)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@pytest.mark.parametrize("g,d", [(g, 128) for g in (3, 5, 6, 7, 8, 9, 12, 15, 16)] +
                         [(g, 64) for g in (3, 5, 6, 7, 9, 12, 15, 16)])
def test_any_group_size(api, g, d):
    # groups the kernel takes in head chunks of 4 (d = 128) or 8 (d = 64),
    # the last chunk padded past the group's end
    wl = W.make(W.PAGED, EDGE_LENGTHS, H_q=2 * g, H_kv=2, D_qk=d, page_size=16,
                seed=300 + g + d)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


@pytest.mark.parametrize("g", [3, 8, 12])
def test_any_group_size_fp8_and_extra(api, g):
    base = W.make(W.PAGED, [0, 17, 700, 5000], H_q=2 * g, H_kv=2, D_qk=128, page_size=16,
                  seed=400 + g)
    for wl in (W.quantize_fp8(base, k_scale=0.5, v_scale=2.0),
               W.with_extra(base, [3, 0, 64, 900], num_slots=1000, seed=401 + g)):
        out, lse = api.run_workload(wl.to("cuda"))
        ro, rl = oracle_for(wl)
        assert_parity(out, lse, ro, rl)


@pytest.mark.parametrize("page_size", [1, 8, 16, 32, 64, 100])
def test_page_sizes(api, page_size):
    wl = W.make(W.PAGED, [1, 99, 700, 2100], H_q=8, H_kv=2, D_qk=128, page_size=page_size,
                seed=page_size)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


def test_gqa_paged_config_full(api):
    wl = W.gqa_paged()
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


def test_long_context_config_sampled(api):
    # full size (8 rows x 131072 entries, page 64), as the bench runs it;
    # the oracle evaluates two rows' heads one by one
    wl = W.long_context()
    out, lse = api.run_workload(wl.to("cuda"))
    rows, heads = [0, 5], [0, 3, 4, 17, 31]
    ro, rl = oracle_for(wl, rows=rows, heads=heads)
    assert_parity(out, lse, ro, rl, rows=rows, heads=heads)


def test_layouts_give_identical_bits(api):
    # one logical KV list per row laid out contiguous, paged (shuffled) and
    # indexed: the kernel visits the same entries in the same order, so the
    # three results are bitwise equal
    lens = [0, 5, 64, 333, 1500, 4096]
    paged = W.make(W.PAGED, lens, H_q=16, H_kv=4, D_qk=128, page_size=16, seed=7)
    B, Lmax = len(lens), max(lens)
    kc = torch.zeros((B, Lmax, 4, 128), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    idx = torch.full((B, Lmax), -1, dtype=torch.int32)
    flat_k = paged.k.reshape(-1, 4, 128)
    flat_v = paged.v.reshape(-1, 4, 128)
    for b, L in enumerate(lens):
        t = torch.arange(L)
        rows = paged.table[b, t // 16].long() * 16 + t % 16
        kc[b, :L], vc[b, :L] = flat_k[rows], flat_v[rows]
        idx[b, :L] = rows.to(torch.int32)
    contig = W.Workload("c", W.CONTIGUOUS, paged.q, kc, vc, paged.lengths, None, 0, 16, 4,
                        128, 128, paged.scale)
    indexed = W.Workload("i", W.INDEXED, paged.q, flat_k.contiguous(), flat_v.contiguous(),
                         paged.lengths, idx, 0, 16, 4, 128, 128, paged.scale)
    # the same lists again in pages of 32 and 64 entries (shuffled tables):
    # small pages take the kernel form whose page lookups run a slice ahead
    repaged = []
    for P in (32, 64):
        n_pages = [-(-L // P) for L in lens]
        perm = torch.randperm(sum(n_pages), generator=torch.Generator().manual_seed(P))
        kp = torch.zeros((sum(n_pages), P, 4, 128), dtype=torch.bfloat16)
        vp = torch.zeros_like(kp)
        table = torch.zeros((B, max(n_pages)), dtype=torch.int32)
        first = 0
        for b, L in enumerate(lens):
            for i in range(n_pages[b]):
                pg = int(perm[first + i])
                table[b, i] = pg
                n = min(P, L - i * P)
                kp[pg, :n], vp[pg, :n] = kc[b, i * P:i * P + n], vc[b, i * P:i * P + n]
            first += n_pages[b]
        repaged.append(W.Workload(f"p{P}", W.PAGED, paged.q, kp, vp, paged.lengths, table, P, 16,
                                  4, 128, 128, paged.scale))
    res = [api.run_workload(w.to("cuda")) for w in (paged, contig, indexed, *repaged)]
    for o, l in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(l, res[0][1])
    ro, rl = oracle_for(paged)
    assert_parity(*res[0], ro, rl)


def test_balanced_policy_is_correct(api):
    wl = W.gqa_paged()
    out, lse = api.run_workload(wl.to("cuda"), policy=api.BALANCED)
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


def test_separate_plan_run_combine_match_forward(api):
    wl = W.make(W.PAGED, [3000, 70, 9000], H_q=8, H_kv=2, D_qk=128, seed=3)
    g = wl.to("cuda")
    prob = api.problem_for(g)
    ws = api.workspace(prob)
    out = torch.empty((3, 8, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((3, 8), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    o2, l2 = api.run_workload(g)
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    assert api.read_error(pl) == 0


def test_out_of_range_index_sets_error_without_fault(api):
    wl = W.make(W.INDEXED, [10, 300], H_q=4, H_kv=1, D_qk=64, num_slots=500, seed=9)
    wl.table[1, 7] = 100000          # beyond the cache
    wl.table[1, 8] = -5
    g = wl.to("cuda")
    prob = api.problem_for(g)
    ws = api.workspace(prob)
    out = torch.empty((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    assert api.read_error(pl) & api.DEVERR_INDEX
    # the well-formed row is unaffected
    ro, rl = oracle_for(wl, rows=[0])
    assert_parity(out, lse, ro, rl, rows=[0])


def test_length_beyond_capacity_is_clamped_and_flagged(api):
    wl = W.make(W.CONTIGUOUS, [40, 50], H_q=2, H_kv=1, D_qk=64, seed=11)
    wl.lengths[1] = 10 ** 6          # capacity is Lmax = 50
    g = wl.to("cuda")
    prob = api.problem_for(g)
    ws = api.workspace(prob)
    out = torch.empty((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 2), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
    api.run(pl, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    api.combine(pl, out, lse)
    assert api.read_error(pl) & api.DEVERR_LENGTH
    wl.lengths[1] = 50
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)


def test_empty_batch_is_a_no_op(api):
    prob = api.problem(batch=0, num_q_heads=4, num_kv_heads=1, head_dim_qk=64,
                       layout="contiguous", scale=0.125, width=1)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    lengths = torch.empty(0, dtype=torch.int32, device="cuda")
    api.plan(prob, api.INVARIANT, lengths, ws)


def test_cpu_tensors_are_refused(api):
    wl = W.tiny()
    with pytest.raises(ValueError):
        api.run_workload(wl)
