"""decode_attn_forward_static: the forward pass for callers that cannot
allocate device memory (a plugin whose host process owns every device
allocation, a latency-critical path that must not trigger cudaMalloc's
synchronisation).  Its scratch is one fixed device array inside the library.

The test calls the entry point through the C ABI twice in a row -- two
different problems, so the second call runs on scratch the first one left
behind -- and checks each result against the regular entry point
(decode_attn_forward with a caller-owned workspace) within the tolerance the
parity tests use.  It also checks that an oversized problem is refused.
This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

from invariant_decode_attention_gb300 import workloads as W
from oracle import bf16 as OB

pytestmark = pytest.mark.gpu

OUT_ATOL, LSE_ATOL = 1e-2, 1e-4


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


def _close(out, lse, ref_out, ref_lse):
    o, ro = out.double().cpu().numpy(), ref_out.double().cpu().numpy()
    assert np.all(np.abs(o - ro) <= np.maximum(OUT_ATOL, OB.ulp(ro)))
    l, rl = lse.double().cpu().numpy(), ref_lse.double().cpu().numpy()
    same_inf = np.isneginf(l) & np.isneginf(rl)
    assert np.all(same_inf | (np.abs(l - rl) <= LSE_ATOL))


def test_static_entry_matches_regular_entry_on_two_calls(api):
    cases = [W.gqa_paged(), W.make(W.PAGED, [0, 9000, 77, 131072], H_q=16, H_kv=4,
                                   D_qk=128, page_size=64, seed=5)]
    for wl in cases:
        g = wl.to("cuda")
        prob = api.problem_for(g)
        assert api.workspace_bytes(prob) <= api.STATIC_WORKSPACE_BYTES
        ref_out, ref_lse = api.run_workload(g)  # decode_attn_forward, caller's workspace
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        api.forward_static(prob, api.INVARIANT, g.q, g.k, g.v, g.table, g.lengths, out, lse)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


def test_static_entry_refuses_a_problem_beyond_its_array(api):
    # 4096 rows x 64 splits x 32 heads x 128 dims of fp32 partials > 64 MiB
    prob = api.problem(batch=4096, num_q_heads=32, num_kv_heads=8, head_dim_qk=128,
                       layout="paged", scale=0.1, page_size=16, width=8, num_blocks=64)
    assert api.workspace_bytes(prob) > api.STATIC_WORKSPACE_BYTES
    L = api.lib()
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = L.decode_attn_forward_static(ctypes.byref(prob), api.INVARIANT, p, p, p, p, p, p, p,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == api.ERR_WORKSPACE
