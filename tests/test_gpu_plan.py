"""The device split plans are bit-exact against the oracle's plans."""

import random

import pytest
import torch

from oracle import plan as OP

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


def _device_plan(api, lengths, policy, capacity, variant="fma"):
    if variant == "fma":
        prob = api.problem(batch=len(lengths), num_q_heads=1, num_kv_heads=1, head_dim_qk=64,
                           layout="indexed", scale=1.0, width=capacity, num_blocks=1)
    else:  # the tensor-core variant: heads over one shared latent row (16, the fewest it
        # takes, keeps the partial buffers of a 4096-row plan at 4 GB)
        prob = api.problem(batch=len(lengths), num_q_heads=16, num_kv_heads=1, head_dim_qk=576,
                           head_dim_v=512, layout="indexed", scale=1.0, width=capacity,
                           num_blocks=1, shared_latent=True)
    variant_id, *_ = api.split_constants(prob)
    assert variant_id == (api.VARIANT_FMA if variant == "fma" else api.VARIANT_MLA)
    ws = api.workspace(prob)
    d_len = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    pl = api.plan(prob, policy, d_len, ws)
    n_splits, split_begin, work = api.copy_plan(pl)
    bounds = [split_begin[b, :int(n_splits[b]) + 1].tolist() for b in range(len(lengths))]
    return pl, bounds, work.tolist()


def _same_work(work, bounds, mx):
    """The device work list holds exactly the oracle's items, largest key
    first (items of equal key may come in any order)."""
    want = OP.work_list(bounds, mx)
    assert sorted(work) == sorted(want)
    keys = [OP.work_key(bounds, mx, w) for w in work]
    assert keys == [OP.work_key(bounds, mx, w) for w in want]


@pytest.mark.parametrize("start", range(0, 131073, 16384))
def test_invariant_plan_all_lengths_up_to_131072(api, start):
    _all_lengths(api, "fma", start, 16384)


@pytest.mark.parametrize("start", range(0, 131073, 4096))
def test_invariant_plan_all_lengths_up_to_131072_tensor_core(api, start):
    _all_lengths(api, "mla", start, 4096)


def _all_lengths(api, variant, start, n):
    lengths = list(range(start, min(start + n, 131073)))
    T, mn, mx = OP.VARIANT_CONSTANTS[variant]
    pl, bounds, work = _device_plan(api, lengths, api.INVARIANT, 131072, variant)
    assert (pl.tile_tokens, pl.min_tiles_per_split, pl.max_splits) == (T, mn, mx)
    want = OP.plan_invariant(lengths, T, mn, mx)
    assert bounds == want
    _same_work(work, want, mx)


@pytest.mark.parametrize("variant", ["fma", "mla"])
def test_invariant_and_balanced_random_batches(api, variant):
    rng = random.Random(5)
    T, mn, mx = OP.VARIANT_CONSTANTS[variant]
    for trial in range(20):
        B = rng.randint(1, 300)
        lengths = [rng.choice([0, 1, rng.randint(1, 131072), int(2 ** (17 * rng.random()))])
                   for _ in range(B)]
        pl, bounds, work = _device_plan(api, lengths, api.INVARIANT, 131072, variant)
        want = OP.plan_invariant(lengths, T, mn, mx)
        assert bounds == want
        _same_work(work, want, mx)
        pl, bounds, work = _device_plan(api, lengths, api.BALANCED, 131072, variant)
        want = OP.plan_balanced(lengths, T, mx, pl.num_parts, pl.fixed_overhead)
        assert pl.fixed_overhead == OP.BALANCED_FIXED_OVERHEAD
        assert bounds == want
        _same_work(work, want, mx)


def test_lengths_are_clamped_like_the_oracle_reads_them(api):
    T, mn, mx = OP.VARIANT_CONSTANTS["fma"]
    pl, bounds, _ = _device_plan(api, [-5, 100, 10 ** 7], api.INVARIANT, 5000)
    assert bounds == OP.plan_invariant([0, 100, 5000], T, mn, mx)
    assert api.read_error(pl) & api.DEVERR_LENGTH
