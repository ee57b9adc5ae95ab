"""The time-out path of the tensor-core kernels, made to run on purpose.

Every mbarrier wait in the tcgen05 kernels is bounded; when one runs out the
kernel records DA_DEVERR_TIMEOUT, every role leaves its loop, the copies in
flight and the tensor-core work are drained and tensor memory is freed, so
the context stays usable.  The DA_FLAG_TEST_STALL hook makes the MMA-issuing
thread of every CTA wait first on a barrier that nothing signals (2 ms
limit), which drives each role into that path from a known point: copies
issued, nothing consumed.  The tests check the error word, and that a normal
call on the same buffers right after it returns the clean result bit for bit
(a CTA that left tensor memory allocated, or an arrival still in flight into
freed shared memory, would show up there or hang the next launch's
allocation).  The CPU test checks the flag's validation.
"""

import pytest
import torch

from invariant_decode_attention_gb300 import workloads as W

gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


def _workloads():
    return {
        "mla": W.make(W.INDEXED, [40, 300, 1500, 2048], H_q=128, H_kv=1, D_qk=576, D_v=512,
                      latent=True, num_slots=4096, seed=71),
        "mla_fp8": W.quantize_fp8(W.make(W.INDEXED, [40, 300, 1500, 2048], H_q=128, H_kv=1,
                                         D_qk=576, D_v=512, latent=True, num_slots=4096,
                                         seed=76)),
        "gqa_tc": W.make(W.PAGED, [40, 300, 1500, 5000], H_q=64, H_kv=2, D_qk=128,
                         page_size=16, seed=72),
        "gqa_tc_fp8": W.quantize_fp8(W.make(W.PAGED, [40, 300, 1500, 5000], H_q=64, H_kv=2,
                                            D_qk=128, page_size=16, seed=73)),
        "gqa_tc_nvfp4": W.nvfp4_kv(W.make(W.PAGED, [40, 300, 1500, 5000], H_q=64, H_kv=2,
                                          D_qk=128, page_size=16, seed=74, draw_kv=False),
                                   seed=75),
    }


def test_flag_validation(api):
    wl = _workloads()["gqa_tc"]
    prob = api.problem_for(wl)
    prob.flags = api.FLAG_TEST_STALL
    assert api.workspace_bytes(prob) > 0
    prob.flags = 2
    with pytest.raises(RuntimeError):
        api.workspace_bytes(prob)


@gpu
@pytest.mark.parametrize("kind", ["mla", "mla_fp8", "gqa_tc", "gqa_tc_fp8", "gqa_tc_nvfp4"])
def test_stall_times_out_and_context_stays_usable(api, kind):
    wl = _workloads()[kind]
    g = wl.to("cuda")
    prob = api.problem_for(g)
    variant = api.split_constants(prob)[0]
    assert variant == (api.VARIANT_MLA if kind.startswith("mla") else api.VARIANT_GQA_TC)
    o_ref, l_ref = [t.clone() for t in api.run_workload(g)]

    prob.flags = api.FLAG_TEST_STALL
    ws = api.workspace(prob)
    out = torch.empty((g.B, g.H_q, g.D_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((g.B, g.H_q), dtype=torch.float32, device="cuda")
    for _ in range(2):  # twice: the first stalled call left nothing behind
        pl = api.plan(prob, api.INVARIANT, g.lengths, ws)
        api.run(pl, g.q, g.k, g.v, g.table, g.lengths, out, lse)
        api.combine(pl, out, lse)
        err = api.read_error(pl)
        assert err & api.DEVERR_TIMEOUT, err
        assert not err & (api.DEVERR_INDEX | api.DEVERR_LENGTH), err

    for _ in range(2):
        o, l = api.run_workload(g, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
