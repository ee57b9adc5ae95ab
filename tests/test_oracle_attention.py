"""Pins of the fp64 attention oracle against closed forms, brute force and
invariants -- never against itself.  CPU only.

Each test names the mistake it is there to catch.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import bf16 as OB
from invariant_decode_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf(x):
    """Values exactly representable in bf16, returned as fp64."""
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _f64(t):
    return t.double().numpy()


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_its_value_and_lse_is_the_score():
    # catches: a dropped normalisation, a wrong scale, a transposed q.k
    rng = np.random.default_rng(0)
    q = _bf(rng.standard_normal((1, 1, 16)))
    k = _bf(rng.standard_normal((1, 1, 1, 16)))
    v = _bf(rng.standard_normal((1, 1, 1, 8)))
    scale = 0.37
    out, lse = A.attend(q, k, v, [1], scale=scale, layout=A.CONTIGUOUS)
    assert np.array_equal(out[0, 0], v[0, 0, 0])
    s = scale * math.fsum(q[0, 0, d] * k[0, 0, 0, d] for d in range(16))
    assert lse[0, 0] == pytest.approx(s, abs=1e-14)


def test_equal_scores_give_mean_of_values_and_log_length():
    # q = 0 makes every score 0: out = mean(V), lse = ln(L) (natural log).
    # catches: a log2-based LSE, an off-by-one in the length, a missing max shift
    rng = np.random.default_rng(1)
    L = 37
    q = np.zeros((1, 1, 8))
    k = _bf(rng.standard_normal((1, L, 1, 8)))
    v = _bf(rng.standard_normal((1, L, 1, 5)))
    out, lse = A.attend(q, k, v, [L], scale=1.0, layout=A.CONTIGUOUS)
    mean = [math.fsum(v[0, :, 0, d]) / L for d in range(5)]
    assert np.allclose(out[0, 0], mean, rtol=0, atol=1e-15)
    assert lse[0, 0] == pytest.approx(math.log(L), abs=1e-15)


def test_two_keys_sigmoid_weights():
    # out = sigma(s1 - s2) v1 + sigma(s2 - s1) v2; catches a sign flip in the
    # shift or exponent, or swapped weights
    q = np.array([[[1.0, 2.0]]])
    k = np.array([[[[0.5, -1.0]], [[1.5, 0.25]]]])        # s = scale*(-1.5), scale*2.0
    v = np.array([[[[1.0, -2.0, 3.0]], [[4.0, 5.0, -6.0]]]])
    scale = 0.5
    s1, s2 = scale * -1.5, scale * 2.0
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    w2 = 1.0 / (1.0 + math.exp(s1 - s2))
    out, lse = A.attend(q, k, v, [2], scale=scale, layout=A.CONTIGUOUS)
    assert np.allclose(out[0, 0], w1 * v[0, 0, 0] + w2 * v[0, 1, 0], rtol=0, atol=1e-15)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(s1) + math.exp(s2)), abs=1e-15)


def test_large_scores_do_not_overflow():
    # scores of +-1000 overflow exp() without the max shift; closed form:
    # lse = s_max + log(1 + exp(s_min - s_max))
    q = np.array([[[1.0]]])
    k = np.array([[[[1000.0]], [[998.0]]]])
    v = np.array([[[[1.0]], [[0.0]]]])
    out, lse = A.attend(q, k, v, [2], scale=1.0, layout=A.CONTIGUOUS)
    assert lse[0, 0] == pytest.approx(1000.0 + math.log1p(math.exp(-2.0)), abs=1e-12)
    assert out[0, 0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-2.0)), abs=1e-15)


def test_lse_equals_direct_log_sum_exp_without_shift():
    # direct, unshifted log(sum(exp(scale q.k))) where nothing can overflow
    rng = np.random.default_rng(2)
    L, D = 50, 32
    q = _bf(rng.standard_normal((1, 1, D)))
    k = _bf(rng.standard_normal((1, L, 1, D)))
    v = _bf(rng.standard_normal((1, L, 1, D)))
    scale = D ** -0.5
    _, lse = A.attend(q, k, v, [L], scale=scale, layout=A.CONTIGUOUS)
    direct = math.log(math.fsum(
        math.exp(scale * math.fsum(q[0, 0, d] * k[0, i, 0, d] for d in range(D)))
        for i in range(L)))
    assert lse[0, 0] == pytest.approx(direct, abs=1e-13)


@pytest.mark.parametrize("L", [1, 2, 3, 7, 17])
def test_brute_force_fsum_tiny_rows(L):
    # every sum done with math.fsum on python floats: catches any slip in the
    # vectorised expression (transposed operand, wrong axis)
    rng = np.random.default_rng(10 + L)
    D, Dv = 6, 4
    q = _bf(rng.standard_normal((1, 1, D)))
    k = _bf(rng.standard_normal((1, L, 1, D)))
    v = _bf(rng.standard_normal((1, L, 1, Dv)))
    scale = 0.8
    out, lse = A.attend(q, k, v, [L], scale=scale, layout=A.CONTIGUOUS)
    s = [scale * math.fsum(q[0, 0, d] * k[0, i, 0, d] for d in range(D)) for i in range(L)]
    z = math.fsum(math.exp(x) for x in s)
    for d in range(Dv):
        ref = math.fsum(math.exp(s[i]) * v[0, i, 0, d] for i in range(L)) / z
        assert out[0, 0, d] == pytest.approx(ref, abs=1e-13)
    assert lse[0, 0] == pytest.approx(math.log(z), abs=1e-13)


def test_empty_row_gives_zero_and_minus_inf():
    q = np.ones((1, 2, 4))
    k = np.ones((1, 3, 1, 4))
    out, lse = A.attend(q, k, k, [0], scale=1.0, layout=A.CONTIGUOUS)
    assert np.all(out == 0.0) and np.all(lse == -np.inf)


# ---------------------------------------------------------- head map and MLA

def test_gqa_head_map_is_block_contiguous():
    # H_q = 4, H_kv = 2: q heads 0,1 -> kv head 0; q heads 2,3 -> kv head 1.
    # kv head 0 has all-zero values, kv head 1 all-one values.  catches an
    # interleaved map (j % H_kv) or a transposed head axis.
    rng = np.random.default_rng(3)
    L, D = 9, 8
    q = _bf(rng.standard_normal((1, 4, D)))
    k = _bf(rng.standard_normal((1, L, 2, D)))
    v = np.zeros((1, L, 2, 3))
    v[:, :, 1, :] = 1.0
    out, _ = A.attend(q, k, v, [L], scale=0.3, layout=A.CONTIGUOUS)
    assert np.allclose(out[0, :2], 0.0, atol=0) and np.allclose(out[0, 2:], 1.0, atol=1e-15)


def test_mla_latent_value_is_leading_dims():
    # shared latent row of 576 dims; V is its first 512.  single key => out
    # equals K[:512] exactly, and the trailing 64 dims still enter the score.
    rng = np.random.default_rng(4)
    cache = _bf(rng.standard_normal((10, 1, 576)))
    q = _bf(rng.standard_normal((1, 2, 576)))
    table = np.array([[7, -1, -1]], dtype=np.int32)
    out, lse = A.attend(q, cache, None, [1], scale=576 ** -0.5, layout=A.INDEXED,
                        table=table, d_v=512)
    assert np.array_equal(out[0, 0], cache[7, 0, :512])
    s = 576 ** -0.5 * math.fsum(q[0, 1, d] * cache[7, 0, d] for d in range(576))
    assert lse[0, 1] == pytest.approx(s, abs=1e-13)
    # the trailing dims matter for the score
    s_lead = 576 ** -0.5 * math.fsum(q[0, 1, d] * cache[7, 0, d] for d in range(512))
    assert abs(lse[0, 1] - s_lead) > 1e-6


# ---------------------------------------------------------------- layouts

def test_paged_shuffled_equals_contiguous_exactly():
    # same logical KV laid out through a shuffled page table; catches t // P
    # vs t % P slips and a page-table transpose
    wl = W.make(W.PAGED, [1, 15, 16, 17, 40], H_q=4, H_kv=2, D_qk=16, page_size=16, seed=5)
    B, Lmax = wl.B, int(wl.lengths.max())
    kc = torch.zeros((B, Lmax, 2, 16), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for b in range(B):
        for t in range(int(wl.lengths[b])):
            p = int(wl.table[b, t // 16])
            kc[b, t] = wl.k[p, t % 16]
            vc[b, t] = wl.v[p, t % 16]
    o1, l1 = A.attend(_f64(wl.q), _f64(wl.k), _f64(wl.v), wl.lengths.numpy(), scale=wl.scale,
                      layout=A.PAGED, table=wl.table.numpy(), page_size=16)
    o2, l2 = A.attend(_f64(wl.q), _f64(kc), _f64(vc), wl.lengths.numpy(), scale=wl.scale,
                      layout=A.CONTIGUOUS)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_indexed_equals_contiguous_and_ignores_entries_past_length():
    wl = W.make(W.INDEXED, [3, 20, 1], H_q=2, H_kv=1, D_qk=8, width=24, num_slots=50, seed=6)
    B = wl.B
    kc = torch.zeros((B, 20, 1, 8), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for b in range(B):
        for t in range(int(wl.lengths[b])):
            kc[b, t] = wl.k[int(wl.table[b, t])]
            vc[b, t] = wl.v[int(wl.table[b, t])]
    args = dict(scale=wl.scale)
    o1, l1 = A.attend(_f64(wl.q), _f64(wl.k), _f64(wl.v), wl.lengths.numpy(),
                      layout=A.INDEXED, table=wl.table.numpy(), **args)
    o2, l2 = A.attend(_f64(wl.q), _f64(kc), _f64(vc), wl.lengths.numpy(),
                      layout=A.CONTIGUOUS, **args)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # fill the padding past each row's length with valid slots: nothing changes
    table = wl.table.numpy().copy()
    for b in range(B):
        table[b, int(wl.lengths[b]):] = (np.arange(24 - int(wl.lengths[b])) * 7) % 50
    o3, l3 = A.attend(_f64(wl.q), _f64(wl.k), _f64(wl.v), wl.lengths.numpy(),
                      layout=A.INDEXED, table=table, **args)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


def test_permuting_a_rows_index_list_leaves_result_unchanged():
    wl = W.make(W.INDEXED, [300], H_q=4, H_kv=1, D_qk=32, width=300, num_slots=1000, seed=7)
    perm = np.random.default_rng(8).permutation(300)
    t2 = wl.table.numpy().copy()
    t2[0, :300] = t2[0, perm]
    o1, l1 = A.attend(_f64(wl.q), _f64(wl.k), _f64(wl.v), [300], scale=wl.scale,
                      layout=A.INDEXED, table=wl.table.numpy())
    o2, l2 = A.attend(_f64(wl.q), _f64(wl.k), _f64(wl.v), [300], scale=wl.scale,
                      layout=A.INDEXED, table=t2)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- LSE merge

@pytest.mark.parametrize("cuts", [[0, 100], [0, 1, 100], [0, 33, 34, 90, 100], [0, 0, 50, 50, 100]])
def test_lse_merge_of_split_partials_equals_unsplit(cuts):
    # the combine identity: attention over pieces, merged by LSE weights,
    # equals attention over the whole list.  Empty pieces (lse -inf) drop out.
    rng = np.random.default_rng(9)
    L, D = 100, 16
    q = _bf(rng.standard_normal(D))
    K = _bf(rng.standard_normal((L, D)))
    V = _bf(rng.standard_normal((L, D)))
    whole = A.attend_row(q, K, V, 0.25)
    parts = [A.attend_row(q, K[a:b], V[a:b], 0.25) for a, b in zip(cuts[:-1], cuts[1:])]
    out, lse = A.lse_merge(parts)
    assert np.allclose(out, whole[0], rtol=0, atol=1e-12)
    assert lse == pytest.approx(whole[1], abs=1e-12)


def test_lse_merge_all_empty():
    out, lse = A.lse_merge([(np.zeros(3), -math.inf), (np.zeros(3), -math.inf)])
    assert lse == -math.inf and np.all(out == 0)


def test_lse_merge_two_piece_closed_form():
    # two single-key pieces: merge weights are sigmoid(lse1 - lse2)
    o1, o2 = np.array([1.0, 0.0]), np.array([0.0, 1.0])
    out, lse = A.lse_merge([(o1, 0.0), (o2, math.log(3.0))])
    assert np.allclose(out, [0.25, 0.75], atol=1e-15)
    assert lse == pytest.approx(math.log(4.0), abs=1e-15)


# ---------------------------------------------------------------- bf16

def test_bf16_rounding_matches_torch_on_fp32_values():
    # fp32 inputs round once, so torch's fp32->bf16 cast is the same function
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * s
                        for s in (1e-3, 1.0, 30.0, 1e30)])
    x = np.concatenate([x, np.float32([0.0, -0.0, 1e-40, -3e-39, 3.0e38, np.inf, -np.inf])])
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = OB.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rounding_ties_to_even_and_no_double_rounding():
    one = 1.0
    u = 2.0 ** -7            # bf16 spacing on [1, 2)
    assert OB.round_to_bf16(one + u / 2) == one            # tie -> even (1.0)
    assert OB.round_to_bf16(one + 3 * u / 2) == one + 2 * u  # tie -> even
    # just above a tie, by less than fp32 can hold: rounding through fp32
    # first would land on the tie and go to even; the exact answer rounds up
    x = one + u / 2 + 2.0 ** -40
    assert OB.round_to_bf16(x) == one + u


def test_bf16_ulp_matches_page_figures():
    with open(os.path.join(GOLDEN, "bf16_ulp_page_figures.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        assert OB.ulp(case["x"]) == case["ulp"], case
    lo, hi = g["printed_range"]
    # the printed range is one ULP on [0.25, 0.5) and one ULP on [0.5, 1)
    assert abs(OB.ulp(0.3) - lo) < 1e-5 and abs(OB.ulp(0.7) - hi) < 1e-4


# ---------------------------------------------------------------- second KV source

def _two_source_case(seed=12):
    rng = np.random.default_rng(seed)
    B, H, D, Dv = 3, 4, 24, 16
    q = _bf(rng.standard_normal((B, H, D)))
    main = _bf(rng.standard_normal((40, 1, D)))
    extra = _bf(rng.standard_normal((30, 1, D)))
    lengths = np.array([5, 0, 12])
    extra_lengths = np.array([3, 7, 0])
    table = np.stack([rng.permutation(40)[:12] for _ in range(B)]).astype(np.int32)
    extra_table = np.stack([rng.permutation(30)[:8] for _ in range(B)]).astype(np.int32)
    return q, main, extra, lengths, extra_lengths, table, extra_table, Dv


def test_extra_source_equals_one_concatenated_cache():
    # the two lists read from two caches == one cache holding both, with the
    # extra indices offset past the main cache's slots
    q, main, extra, L, Le, t, te, Dv = _two_source_case()
    o1, l1 = A.attend(q, main, None, L, scale=0.2, layout=A.INDEXED, table=t, d_v=Dv,
                      extra_k=extra, extra_table=te, extra_lengths=Le)
    cat = np.concatenate([main, extra], axis=0)
    B = q.shape[0]
    tt = np.full((B, 20), -1, dtype=np.int32)
    for b in range(B):
        tt[b, :L[b]] = t[b, :L[b]]
        tt[b, L[b]:L[b] + Le[b]] = te[b, :Le[b]] + main.shape[0]
    o2, l2 = A.attend(q, cat, None, L + Le, scale=0.2, layout=A.INDEXED, table=tt, d_v=Dv)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_extra_source_is_the_lse_merge_of_the_two_lists():
    # attention over main ++ extra == LSE merge of attention over each part
    q, main, extra, L, Le, t, te, Dv = _two_source_case(13)
    o, l = A.attend(q, main, None, L, scale=0.3, layout=A.INDEXED, table=t, d_v=Dv,
                    extra_k=extra, extra_table=te, extra_lengths=Le)
    om, lm = A.attend(q, main, None, L, scale=0.3, layout=A.INDEXED, table=t, d_v=Dv)
    oe, le = A.attend(q, extra, None, Le, scale=0.3, layout=A.INDEXED, table=te, d_v=Dv)
    for b in range(q.shape[0]):
        for j in range(q.shape[1]):
            mo, ml = A.lse_merge([(om[b, j], lm[b, j]), (oe[b, j], le[b, j])])
            assert np.allclose(o[b, j], mo, rtol=0, atol=1e-12)
            assert (l[b, j] == ml == -np.inf) or abs(l[b, j] - ml) < 1e-12
