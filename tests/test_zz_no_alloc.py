"""decode_attn_forward_static: the forward pass for callers that cannot
allocate device memory (a plugin whose host process owns every device
allocation, a latency-critical path that must not trigger cudaMalloc's
synchronisation).  Its scratch is one fixed device array inside the library.

The test calls the entry point through the C ABI twice in a row -- two
different problems, so the second call runs on scratch the first one left
behind -- and checks each result bit for bit against the regular entry point
(decode_attn_forward with a caller-owned workspace): both run the same plan
and the same kernels, so their bits must agree.  A third call repeats the
first problem while the device's free memory and torch's allocator counters
are watched: nothing may be allocated.  It also reads a call's device error
word through the returned plan, and checks that an oversized problem is
refused.  This file is named to be collected last.
"""

import ctypes

import pytest
import torch

from invariant_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


def _cases():
    return [W.gqa_paged(), W.make(W.PAGED, [0, 9000, 77, 131072], H_q=16, H_kv=4, D_qk=128,
                                  page_size=64, seed=5)]


def _static(api, g, prob):
    out = torch.full((g.B, g.H_q, g.D_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((g.B, g.H_q), float("nan"), dtype=torch.float32, device="cuda")
    return out, lse


def test_static_entry_matches_regular_entry_on_two_calls(api):
    for wl in _cases():
        g = wl.to("cuda")
        prob = api.problem_for(g)
        assert api.workspace_bytes(prob) <= api.STATIC_WORKSPACE_BYTES
        ref_out, ref_lse = api.run_workload(g)  # decode_attn_forward, caller's workspace
        out, lse = _static(api, g, prob)
        pl = api.forward_static(prob, api.INVARIANT, g.q, g.k, g.v, g.table, g.lengths, out, lse)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        assert api.read_error(pl) == 0


def test_static_entry_allocates_nothing(api):
    g = _cases()[0].to("cuda")
    prob = api.problem_for(g)
    ref_out, ref_lse = api.run_workload(g)
    out, lse = _static(api, g, prob)
    # first call: the library's code and its array are loaded on the device
    api.forward_static(prob, api.INVARIANT, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    out2, lse2 = _static(api, g, prob)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, res0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    api.forward_static(prob, api.INVARIANT, g.q, g.k, g.v, g.table, g.lengths, out2, lse2)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == res0
    assert torch.equal(out2, ref_out) and torch.equal(lse2, ref_lse)


def test_static_entry_reports_device_errors(api):
    wl = W.make(W.PAGED, [100, 3000], H_q=32, H_kv=8, D_qk=128, page_size=16, seed=9)
    g = wl.to("cuda")
    prob = api.problem_for(g)
    bad = torch.tensor([100, 10 ** 7], dtype=torch.int32, device="cuda")  # above capacity
    out, lse = _static(api, g, prob)
    pl = api.forward_static(prob, api.INVARIANT, g.q, g.k, g.v, g.table, bad, out, lse)
    assert api.read_error(pl) & api.DEVERR_LENGTH
    # a clean call afterwards clears the word again
    pl = api.forward_static(prob, api.INVARIANT, g.q, g.k, g.v, g.table, g.lengths, out, lse)
    assert api.read_error(pl) == 0


def test_static_entry_refuses_a_problem_beyond_its_array(api):
    # 4096 rows x 64 splits x 32 heads x 128 dims of fp32 partials > 64 MiB
    prob = api.problem(batch=4096, num_q_heads=32, num_kv_heads=8, head_dim_qk=128,
                       layout="paged", scale=0.1, page_size=16, width=8, num_blocks=64)
    assert api.workspace_bytes(prob) > api.STATIC_WORKSPACE_BYTES
    L = api.lib()
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = L.decode_attn_forward_static(ctypes.byref(prob), api.INVARIANT, p, p, p, p, p, p, p,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                      None)
    assert rc == api.ERR_WORKSPACE
