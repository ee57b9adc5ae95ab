"""Bitwise batch invariance of every kernel family, swept like the bf16 one.

Invariance has to be shown per kernel path and cache format, not assumed
from one of them ("Batch invariance is not universal across kernel paths",
Workaround: measure it per architecture, quantization and kernel family).
Each sweep embeds one fixed target row at a random position of batches of
every size 1..256, with fresh batchmates and fresh page ids / slot ids for
the target every time; the target's bits must equal its solo run, which
itself matches the fp64 oracle, and repeated runs must be identical.

Families: the E4M3 (one-byte cache) instantiation of the CUDA-core kernel,
the CUDA-core kernel with a second KV source, the CUDA-core kernel on groups
it cuts into head chunks (8 and 3 query heads per KV head at d = 128), the
tensor-core shared-latent kernel on bf16 and on E4M3 latent caches, and the
tensor-core kernel with a second latent source.
"""

import pytest
import torch

from _util import assert_parity, oracle_for
from invariant_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SIZES = range(1, 257)
REPEAT_AT = (0, 63, 255)


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


def _sweep(api, sweep, solo_cpu):
    o_solo, l_solo = api.run_workload(sweep.solo())
    ro, rl = oracle_for(solo_cpu)
    assert_parity(o_solo, l_solo, ro, rl)
    for i in range(len(sweep.sizes)):
        wl, pos = sweep.batch(i)
        o, l = api.run_workload(wl)
        assert torch.equal(o[pos], o_solo[0]), f"B={wl.B} pos={pos}"
        assert torch.equal(l[pos], l_solo[0]), f"B={wl.B} pos={pos}"
        if i in REPEAT_AT:
            for _ in range(3):
                o2, l2 = api.run_workload(wl)
                assert torch.equal(o2, o) and torch.equal(l2, l)


def test_fp8_cache_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweep(SIZES, kv_fp8=True)
    _sweep(api, sweep, sweep.solo_cpu())


def test_extra_source_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweep(SIZES, extra=True)
    _sweep(api, sweep, sweep.solo_cpu())


@pytest.mark.parametrize("h_q", [64, 24])
def test_head_chunk_ragged_sweep_bitwise(api, h_q):
    sweep = W.RaggedSweep(SIZES, H_q=h_q)
    _sweep(api, sweep, sweep.solo_cpu())


def test_latent_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweepLatent(SIZES)
    _sweep(api, sweep, sweep.solo_cpu())


def test_latent_extra_source_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweepLatent(SIZES, extra=True)
    _sweep(api, sweep, sweep.solo_cpu())


def test_latent_fp8_ragged_sweep_bitwise(api):
    sweep = W.RaggedSweepLatent(SIZES, kv_fp8=True)
    _sweep(api, sweep, sweep.solo_cpu())
