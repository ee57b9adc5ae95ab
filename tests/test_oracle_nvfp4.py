"""Pins for oracle/nvfp4.py: the E2M1 decoder against the format's value
list, the nibble and block-scale layout against hand-built matrices, and the
activation-rounded product against brute force, exact integer arithmetic and
the bf16 ties-to-even rule."""

import math

import numpy as np
import pytest

from oracle import fp8, nvfp4
from invariant_decode_attention_gb300 import workloads as W

# The sixteen E2M1 values, code by code: magnitudes 0, 0.5 (subnormal), then
# 1, 1.5, 2, 3, 4, 6 (exponent 1..3, one fraction bit); bit 3 is the sign.
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
               -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_value_list():
    got = nvfp4.decode_e2m1(np.arange(16))
    assert np.array_equal(got, np.array(E2M1_VALUES))
    assert np.signbit(got[8]) and not np.signbit(got[0])


def test_e2m1_monotone_and_symmetric():
    v = nvfp4.decode_e2m1(np.arange(16))
    assert (np.diff(v[:8]) > 0).all()
    assert np.array_equal(v[8:], -v[:8])
    assert np.abs(v).max() == 6.0


def test_nibble_order():
    # byte j holds element 2j in its low nibble and element 2j + 1 in its high one
    codes = np.array([[0x21, 0xF0, 0x7A]], dtype=np.uint8)
    assert nvfp4.unpack(codes).tolist() == [[1, 2, 0, 15, 10, 7]]


def test_block_scales_cover_sixteen_weights():
    K = 64
    codes = np.full((2, K // 2), 0x22, dtype=np.uint8)        # every weight code 2 = 1.0
    scales = np.array([[0x38, 0x40, 0x30, 0x39],                # 1, 2, 0.5, 1.125
                       [0x48, 0x28, 0x3C, 0x01]], dtype=np.uint8)  # 4, 0.25, 1.5, 2^-9
    w = nvfp4.dequantize(codes, scales, 0.5)
    want = 0.5 * np.repeat(np.array([[1.0, 2.0, 0.5, 1.125], [4.0, 0.25, 1.5, 2.0 ** -9]]),
                           16, axis=1)
    assert np.array_equal(w, want)
    with pytest.raises(ValueError):
        nvfp4.dequantize(codes, scales[:, :3], 1.0)


def test_operand_orientation():
    # W[o, k] nonzero only at (1, 5), x[i, k] nonzero only at (0, 5):
    # y = x W^T is nonzero only at (0, 1)
    K, N = 32, 3
    codes = np.zeros((N, K // 2), dtype=np.uint8)
    codes[1, 2] = 0x70                                           # element 5 = high nibble of byte 2: 6.0
    scales = np.full((N, K // 16), 0x38, dtype=np.uint8)
    x = np.zeros((2, K))
    x[0, 5] = 3.0
    y = nvfp4.matmul(x, codes, scales, 1.0)
    want = np.zeros((2, N))
    want[0, 1] = 18.0
    assert np.array_equal(y, want)


def _brute(x, codes, scales, gs):
    """Independent restatement for tiny inputs: per element, a table lookup of
    the nibble, the block's scale, and math.fsum over exact products."""
    n, K = x.shape
    N = codes.shape[0]
    s = fp8.decode_e4m3(scales)
    xr = nvfp4.round_activations(x)
    y = np.zeros((n, N))
    for i in range(n):
        for o in range(N):
            terms = []
            for k in range(K):
                byte = int(codes[o, k // 2])
                nib = byte & 0xF if k % 2 == 0 else byte >> 4
                terms.append(xr[i, k] * gs * s[o, k // 16] * E2M1_VALUES[nib])
            y[i, o] = math.fsum(terms)
    return y


def test_matmul_brute_force_tiny():
    m = W.nvfp4_matmul(3, 5, 48, seed=11)
    x, c, s = m.x.double().numpy(), m.codes.numpy(), m.scales.numpy()
    y = nvfp4.matmul(x, c, s, m.global_scale)
    ref = _brute(x, c, s, m.global_scale)
    mag = nvfp4.abs_products(x, c, s, m.global_scale)
    assert np.all(np.abs(y - ref) <= 1e-14 * mag)


def test_integer_weights_and_activations_are_exact():
    # scales 1, global scale 1: 2 W is an integer matrix; integer x is exact in
    # bf16, so 2 y is an exact integer product (numpy int64, no float at all)
    rng = np.random.default_rng(3)
    N, K, n = 7, 96, 4
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = np.full((N, K // 16), 0x38, dtype=np.uint8)
    x = rng.integers(-8, 9, (n, K)).astype(np.float64)
    twice = {0: 0, 1: 1, 2: 2, 3: 3, 4: 4, 5: 6, 6: 8, 7: 12}
    nib = nvfp4.unpack(codes)
    w2 = np.vectorize(lambda c: (-1 if c & 8 else 1) * twice[c & 7])(nib).astype(np.int64)
    want2 = x.astype(np.int64) @ w2.T
    y = nvfp4.matmul(x, codes, scales, 1.0)
    assert np.array_equal(2 * y, want2.astype(np.float64))


def test_activations_round_to_bf16_ties_to_even():
    K = 16
    codes = np.full((1, K // 2), 0x02, dtype=np.uint8)  # weight 0 = 1.0, the rest 0
    scales = np.full((1, 1), 0x38, dtype=np.uint8)
    for xv, want in [(1.0 + 2.0 ** -8, 1.0),                   # halfway: to the even 1.0
                     (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),    # halfway: to the even 1 + 2^-6
                     (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7),
                     (-(3.0 + 2.0 ** -7), -3.0)]:
        x = np.zeros((1, K))
        x[0, 0] = xv
        assert nvfp4.matmul(x, codes, scales, 1.0)[0, 0] == want


def test_global_scale_is_linear():
    m = W.nvfp4_matmul(2, 9, 64, seed=5)
    x, c, s = m.x.double().numpy(), m.codes.numpy(), m.scales.numpy()
    assert np.array_equal(nvfp4.matmul(x, c, s, 2.0), 2.0 * nvfp4.matmul(x, c, s, 1.0))


def test_rows_are_independent():
    # the definition has no batch dependence: a row's result is the same alone
    m = W.nvfp4_matmul(6, 11, 80, seed=9)
    x, c, s = m.x.double().numpy(), m.codes.numpy(), m.scales.numpy()
    y = nvfp4.matmul(x, c, s, m.global_scale)
    for i in range(6):
        assert np.array_equal(nvfp4.matmul(x[i:i + 1], c, s, m.global_scale)[0], y[i])


def test_abs_products_bound_the_result():
    m = W.nvfp4_matmul(4, 16, 128, seed=13)
    x, c, s = m.x.double().numpy(), m.codes.numpy(), m.scales.numpy()
    y = nvfp4.matmul(x, c, s, m.global_scale)
    mag = nvfp4.abs_products(x, c, s, m.global_scale)
    assert np.all(np.abs(y) <= mag) and np.all(mag > 0)


def test_generator_layout():
    m = W.nvfp4_matmul(3, 10, 64, seed=1)
    assert m.codes.shape == (10, 32) and m.scales.shape == (10, 4) and m.x.shape == (3, 64)
    e = (m.scales.numpy() >> 3) & 0xF
    assert e.min() >= 4 and e.max() <= 10 and (m.scales.numpy() < 0x80).all()
    assert m.weight_bytes() == 10 * 32 + 10 * 4


# ---------------------------------------------------------------- NVFP4 KV cache

def test_cache_blocks_run_along_each_head_row():
    # two heads of one entry, D = 32: a head row has two 16-element blocks;
    # head 0 row codes 0x21 (elements 0.5, 1.0, ...), head 1 row all code 7 (6.0)
    codes = np.zeros((1, 2, 16), dtype=np.uint8)
    codes[0, 0] = 0x21
    codes[0, 1] = 0x77
    scales = np.array([[[0x38, 0x40], [0x30, 0x48]]], dtype=np.uint8)  # 1, 2 | 0.5, 4
    got = nvfp4.dequantize_cache(codes, scales, 0.25)
    h0 = np.array([0.5, 1.0] * 8 + [1.0, 2.0] * 8) * 0.25
    h1 = np.array([3.0] * 16 + [24.0] * 16) * 0.25
    assert got.shape == (1, 2, 32)
    assert np.array_equal(got[0, 0], h0) and np.array_equal(got[0, 1], h1)


def test_attention_over_an_nvfp4_cache_by_brute_force():
    # a 5-entry cache of one KV head (D = 32) decoded by an independent table
    # of E2M1 values and the E4M3 decoder (pinned in test_oracle_fp8.py);
    # attention then by math.fsum: the oracle's view must agree to 1e-12
    from oracle import attention as A
    rng = np.random.default_rng(3)
    L, D = 5, 32
    kc = rng.integers(0, 256, (L, 1, D // 2), dtype=np.uint8)
    vc = rng.integers(0, 256, (L, 1, D // 2), dtype=np.uint8)
    ks = rng.integers(0x20, 0x40, (L, 1, D // 16), dtype=np.uint8)
    vs = rng.integers(0x20, 0x40, (L, 1, D // 16), dtype=np.uint8)
    q = rng.standard_normal((1, 2, D))

    def hand(codes, scales, g):
        out = np.zeros((L, 1, D))
        for t in range(L):
            for d in range(D):
                byte = int(codes[t, 0, d // 2])
                nib = (byte >> 4) if d % 2 else (byte & 0xF)
                out[t, 0, d] = g * float(fp8.decode_e4m3(scales[t, 0, d // 16])) * E2M1_VALUES[nib]
        return out

    K, V = hand(kc, ks, 0.5), hand(vc, vs, 2.0)
    scale = D ** -0.5
    want_o = np.zeros((2, D))
    want_l = np.zeros(2)
    for j in range(2):
        s = [scale * math.fsum(q[0, j, d] * K[t, 0, d] for d in range(D)) for t in range(L)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        Z = math.fsum(w)
        want_l[j] = m + math.log(Z)
        for d in range(D):
            want_o[j, d] = math.fsum(w[t] * V[t, 0, d] for t in range(L)) / Z
    Kd = nvfp4.dequantize_cache(kc, ks, 0.5)[None]
    Vd = nvfp4.dequantize_cache(vc, vs, 2.0)[None]
    o, l = A.attend(q, Kd, Vd, np.array([L]), scale=scale, layout="contiguous")
    assert np.allclose(o[0], want_o, rtol=0, atol=1e-12)
    assert np.allclose(l[0], want_l, rtol=0, atol=1e-12)


def test_nvfp4_workload_device_layout_is_codes_then_scales():
    wl = W.nvfp4_kv(W.make(W.PAGED, [5, 40], H_q=4, H_kv=2, D_qk=64, page_size=16, seed=3),
                    seed=4)
    assert wl.k.shape == (wl.k.shape[0], 16, 2, 32) and wl.k_blocks.shape[-1] == 4
    moved = wl.to("cpu")
    base = moved.k.data_ptr()
    assert moved.k_blocks.data_ptr() == base + moved.k.numel()
    assert np.array_equal(moved.k.numpy(), wl.k.numpy())
    assert np.array_equal(moved.v_blocks.numpy(), wl.v_blocks.numpy())
    # positive scales, no NaN code; every code value appears
    assert ((wl.k_blocks >> 3) >= 4).all() and ((wl.k_blocks & 0x80) == 0).all()
    nib = np.concatenate([wl.k.numpy().ravel() & 0xF, wl.k.numpy().ravel() >> 4])
    assert set(nib.tolist()) == set(range(16))
