"""Second KV source: each row's list continues with entries gathered from a
second cache (the sparse decode call of FlashMLA issue #212 with
extra_indices_in_kvcache / extra_topk_length).  Parity against the fp64
oracle, bitwise equality with one concatenated cache, bitwise batch
invariance, and argument checks."""

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


def _concatenated(wl):
    """The same two lists per row as one index-gathered cache (main rows
    first, extra rows after them)."""
    B = wl.B
    if wl.layout == W.INDEXED:
        main_k = wl.k
        main_v = wl.v
        main_idx = wl.table
    else:  # paged main source: flatten pages into rows
        P = wl.page_size
        main_k = wl.k.reshape(-1, wl.H_kv, wl.D_qk)
        main_v = None if wl.v is None else wl.v.reshape(-1, wl.H_kv, wl.D_v)
        main_idx = torch.full((B, wl.table.shape[1] * P), -1, dtype=torch.int32)
        for b in range(B):
            L = int(wl.lengths[b])
            t = torch.arange(L)
            main_idx[b, :L] = (wl.table[b, t // P].long() * P + t % P).to(torch.int32)
    n_main = main_k.shape[0]
    k = torch.cat([main_k, wl.extra_k])
    v = None if wl.v is None else torch.cat([main_v, wl.extra_v])
    tot = wl.lengths + wl.extra_lengths
    idx = torch.full((B, max(int(tot.max()), 1)), -1, dtype=torch.int32)
    for b in range(B):
        L, Le = int(wl.lengths[b]), int(wl.extra_lengths[b])
        idx[b, :L] = main_idx[b, :L]
        idx[b, L:L + Le] = wl.extra_table[b, :Le] + n_main
    return W.Workload("cat", W.INDEXED, wl.q, k, v, tot.to(torch.int32), idx, 0, wl.H_q, wl.H_kv,
                      wl.D_qk, wl.D_v, wl.scale)


def test_mla_with_extra_source_matches_oracle_and_concatenation(api):
    wl = W.mla_sparse_extra()
    out, lse = api.run_workload(wl.to("cuda"))
    rows = list(range(0, 64, 3))
    ro, rl = oracle_for(wl, rows=rows)
    assert_parity(out, lse, ro, rl, rows=rows)
    o2, l2 = api.run_workload(_concatenated(wl).to("cuda"))
    assert torch.equal(out, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("g,d", [(4, 128), (8, 64)])
def test_gqa_paged_with_extra_source(api, g, d):
    base = W.make(W.PAGED, [0, 5, 100, 1000, 3000], H_q=2 * g, H_kv=2, D_qk=d, page_size=16,
                  seed=31)
    wl = W.with_extra(base, [7, 0, 64, 17, 700], num_slots=900, seed=32)
    out, lse = api.run_workload(wl.to("cuda"))
    ro, rl = oracle_for(wl)
    assert_parity(out, lse, ro, rl)
    o2, l2 = api.run_workload(_concatenated(wl).to("cuda"))
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_extra_source_row_solo_vs_batch(api):
    wl = W.mla_sparse_extra()
    g = wl.to("cuda")
    o, l = api.run_workload(g)
    for r in (0, 40):
        solo = W.Workload("solo", W.INDEXED, g.q[r:r + 1].contiguous(), g.k, None,
                          g.lengths[r:r + 1].contiguous(), g.table[r:r + 1].contiguous(), 0,
                          128, 1, 576, 512, wl.scale, extra_k=g.extra_k, extra_v=None,
                          extra_table=g.extra_table[r:r + 1].contiguous(),
                          extra_lengths=g.extra_lengths[r:r + 1].contiguous())
        o1, l1 = api.run_workload(solo)
        assert torch.equal(o1[0], o[r]) and torch.equal(l1[0], l[r])


def test_plan_kind_must_match_run_kind(api):
    wl = W.mla_sparse_extra().to("cuda")
    prob = api.problem_for(wl)
    ws = api.workspace(prob)
    out = torch.empty((64, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((64, 128), dtype=torch.float32, device="cuda")
    pl = api.plan(prob, api.INVARIANT, wl.lengths, ws)  # plan without the second source
    with pytest.raises(api.DecodeAttnError) as e:
        api.run_extra(pl, wl.q, wl.k, None, wl.table, wl.lengths, wl.extra_k, None,
                      wl.extra_table, wl.extra_lengths, out, lse)
    assert e.value.status == api.ERR_INVALID_ARG
    pl = api.plan_extra(prob, api.INVARIANT, wl.lengths, wl.extra_lengths, ws)
    with pytest.raises(api.DecodeAttnError):
        api.run(pl, wl.q, wl.k, None, wl.table, wl.lengths, out, lse)
