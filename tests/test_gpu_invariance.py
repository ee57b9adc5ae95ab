"""Bitwise batch invariance of the INVARIANT policy, and the BALANCED
counter-example.

A row's output and LSE must not change by a single bit with its batchmates,
its position in the batch, its page ids, the table width or a repeat of the
call (FlashMLA issue #212, Measurement: the solo re-run of row 0 with sliced
inputs and a fresh schedule is the test; "same prompt, different batch size
gives identical results", per op, is the rule of the batch-invariance gotchas
page).
"""

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


@pytest.fixture(scope="module")
def sweep():
    return W.RaggedSweep(range(1, 257))


def test_ragged_sweep_target_row_bitwise_invariant(api, sweep):
    o_solo, l_solo = api.run_workload(sweep.solo())
    # the solo result itself is correct
    q, k, v = sweep.q_t, sweep.k_t, sweep.v_t
    solo_cpu = W.Workload("solo", W.CONTIGUOUS, q[None], k[None], v[None],
                          torch.tensor([W.RAGGED_TARGET_LEN], dtype=torch.int32), None, 0,
                          32, 8, 128, 128, 128 ** -0.5)
    ro, rl = oracle_for(solo_cpu)
    assert_parity(o_solo, l_solo, ro, rl)
    for i in range(len(sweep.sizes)):
        wl, pos = sweep.batch(i)
        o, l = api.run_workload(wl)
        assert torch.equal(o[pos], o_solo[0]), f"B={wl.B} pos={pos}"
        assert torch.equal(l[pos], l_solo[0]), f"B={wl.B} pos={pos}"
        if i in (0, 63, 255):  # repeated runs: identical bits
            for _ in range(3):
                o2, l2 = api.run_workload(wl)
                assert torch.equal(o2, o) and torch.equal(l2, l)


def test_balanced_policy_is_not_invariant(api, sweep):
    # the counter-example: the batch-wide quota cuts the target row
    # differently as its batchmates change, and its bits move
    o_solo, _ = api.run_workload(sweep.solo(), policy=api.BALANCED)
    differ, max_abs = 0, 0.0
    for i in range(0, len(sweep.sizes), 5):
        wl, pos = sweep.batch(i)
        o, _ = api.run_workload(wl, policy=api.BALANCED)
        d = (o[pos].float() - o_solo[0].float()).abs().max().item()
        differ += d > 0
        max_abs = max(max_abs, d)
    print(f"BALANCED: {differ} of {len(range(0, len(sweep.sizes), 5))} batches move the "
          f"target row; max_absdiff {max_abs:.5f}")
    assert differ > 0


def test_gqa_paged_row_solo_vs_batch(api):
    wl = W.gqa_paged()
    g = wl.to("cuda")
    o, l = api.run_workload(g)
    for r in (0, 13, 31):
        solo = W.Workload("solo", W.PAGED, g.q[r:r + 1].contiguous(), g.k, g.v,
                          g.lengths[r:r + 1].contiguous(), g.table[r:r + 1].contiguous(),
                          16, 32, 8, 128, 128, wl.scale)
        o1, l1 = api.run_workload(solo)
        assert torch.equal(o1[0], o[r]) and torch.equal(l1[0], l[r])


def test_table_width_and_page_ids_do_not_matter(api):
    wl = W.make(W.PAGED, [3000, 64, 7777], H_q=32, H_kv=8, D_qk=128, page_size=16, seed=21)
    o, l = api.run_workload(wl.to("cuda"))
    # same rows, wider table, pages moved to new ids
    perm = torch.randperm(wl.k.shape[0], generator=torch.Generator().manual_seed(3))
    k2 = torch.empty_like(wl.k)
    v2 = torch.empty_like(wl.v)
    k2[perm] = wl.k
    v2[perm] = wl.v
    t2 = torch.full((3, wl.table.shape[1] + 77), -1, dtype=torch.int32)
    valid = wl.table >= 0
    t2[:, :wl.table.shape[1]] = torch.where(valid, perm[wl.table.clamp(min=0).long()].to(torch.int32),
                                            wl.table)
    wl2 = W.Workload("moved", W.PAGED, wl.q, k2, v2, wl.lengths, t2, 16, 32, 8, 128, 128, wl.scale)
    o2, l2 = api.run_workload(wl2.to("cuda"))
    assert torch.equal(o, o2) and torch.equal(l, l2)


def test_gqa_repeated_runs_bitwise(api):
    """Back-to-back runs on one workspace give identical bits."""
    wl = W.gqa_paged().to("cuda")
    ws = api.workspace(api.problem_for(wl), "cuda")
    out0, lse0 = [t.clone() for t in api.run_workload(wl, ws=ws)]
    for _ in range(8):
        out, lse = api.run_workload(wl, ws=ws)
        assert torch.equal(out, out0) and torch.equal(lse, lse0)


def test_one_plan_many_runs(api):
    """One plan, several run + combine calls: the split kernel's work queue is
    back at its start after every call, so every call computes every unit."""
    wl = W.make(W.PAGED, [0, 5000, 1, 0, 70000, 640, 3000], H_q=32, H_kv=8, D_qk=128,
                page_size=16, seed=71).to("cuda")
    prob = api.problem_for(wl)
    ws = api.workspace(prob, "cuda")
    pl = api.plan(prob, api.INVARIANT, wl.lengths, ws)
    outs = []
    for _ in range(3):
        out = torch.full((wl.B, wl.H_q, wl.D_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((wl.B, wl.H_q), float("nan"), dtype=torch.float32, device="cuda")
        api.run(pl, wl.q, wl.k, wl.v, wl.table, wl.lengths, out, lse)
        api.combine(pl, out, lse)
        outs.append((out, lse))
    for out, lse in outs:
        assert not torch.isnan(out).any() and not torch.isnan(lse).any()
        assert torch.equal(out, outs[0][0]) and torch.equal(lse, outs[0][1])
    o_ref, l_ref = api.run_workload(wl)
    assert torch.equal(outs[0][0], o_ref) and torch.equal(outs[0][1], l_ref)
