"""Pins for oracle/fp8.py: the E4M3 decoder against closed forms, the
format's special codes and an independent library decode; the dequantized
cache against attention on the same values given in fp64."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import fp8


def test_closed_form_codes():
    cases = {
        0x00: 0.0, 0x80: -0.0,
        0x38: 1.0,            # e = 7, f = 0
        0x39: 1.125,          # 1 + 1/8
        0x40: 2.0, 0xC0: -2.0,
        0x30: 0.5,
        0x7E: 448.0,          # e = 15, f = 6: largest finite
        0xFE: -448.0,
        0x08: 2.0 ** -6,      # smallest normal
        0x01: 2.0 ** -9,      # smallest subnormal: (1/8) * 2^-6
        0x07: 7.0 / 8.0 * 2.0 ** -6,  # largest subnormal
        0x77: 1.875 * 2.0 ** 7,       # e = 14, f = 7
    }
    got = fp8.decode_e4m3(list(cases))
    want = np.array(list(cases.values()))
    assert np.array_equal(got, want)
    assert np.signbit(fp8.decode_e4m3([0x80]))[0]


def test_nan_codes_and_no_infinities():
    v = fp8.decode_e4m3(np.arange(256))
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(np.delete(v, [0x7F, 0xFF])).all()
    assert np.nanmax(np.abs(v)) == fp8.E4M3_MAX


def test_monotone_and_symmetric():
    pos = fp8.decode_e4m3(np.arange(0x00, 0x7F))
    assert (np.diff(pos) > 0).all()  # codes 0..126 increase strictly
    assert np.array_equal(fp8.decode_e4m3(np.arange(0x80, 0xFF)), -pos)


def test_all_codes_match_library_decode():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.decode_e4m3(np.arange(256))
    both_nan = np.isnan(lib) & np.isnan(ours)
    assert np.array_equal(np.where(both_nan, 0.0, lib), np.where(both_nan, 0.0, ours))


def test_scale_multiplies_exactly():
    codes = np.arange(0, 0x7F)
    assert np.array_equal(fp8.dequantize(codes, 0.25), fp8.decode_e4m3(codes) * 0.25)


def test_attention_over_dequantized_cache():
    # The quantized cache means attention over its decoded values: a tiny case
    # where two keys are equal and the third is far below, by brute force.
    k = np.array([0x38, 0x38, 0x80 | 0x50], dtype=np.uint8).reshape(3, 1, 1)  # 1, 1, -8
    v = np.array([0x40, 0x48, 0x38], dtype=np.uint8).reshape(3, 1, 1)         # 2, 4, 1
    K = fp8.dequantize(k, 0.5)
    V = fp8.dequantize(v, 2.0)
    q = np.array([[[4.0]]])
    out, lse = A.attend(q, K[None], V[None], np.array([3]), scale=1.0, layout=A.CONTIGUOUS)
    s = np.array([2.0, 2.0, -16.0])
    w = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
    assert np.allclose(out[0, 0, 0], (w * np.array([4.0, 8.0, 2.0])).sum(), rtol=0, atol=1e-15)
    assert np.isclose(lse[0, 0], np.log(np.exp(s).sum()), rtol=0, atol=1e-15)


def test_quantized_workload_decodes_near_its_source():
    from invariant_decode_attention_gb300 import workloads as W
    base = W.make(W.PAGED, [5, 40, 100], H_q=8, H_kv=2, D_qk=64, page_size=16, seed=7)
    wl = W.quantize_fp8(base)
    assert wl.k.dtype == torch.uint8 and wl.kv_fp8
    deq = fp8.dequantize(wl.k.numpy(), wl.k_scale)
    src = base.k.double().numpy()
    # 3 fraction bits: relative error at most 2^-4 for normal codes, absolute
    # error at most half the subnormal spacing (2^-10 * scale) below them --
    # the generator's rounding, not the oracle's arithmetic, is what this checks
    tol = np.maximum(np.abs(src) * 2.0 ** -4, 2.0 ** -10 * wl.k_scale)
    assert np.all(np.abs(deq - src) <= tol)


def test_oracle_for_quantized_workload_is_attention_on_decoded_values():
    from _util import oracle_for
    from invariant_decode_attention_gb300 import workloads as W
    wl = W.quantize_fp8(W.make(W.CONTIGUOUS, [3, 17, 0], H_q=4, H_kv=2, D_qk=64, seed=8))
    out, lse = oracle_for(wl)
    K = fp8.dequantize(wl.k.numpy(), wl.k_scale)
    V = fp8.dequantize(wl.v.numpy(), wl.v_scale)
    ref_out, ref_lse = A.attend(wl.q.double().numpy(), K, V, wl.lengths.numpy(), scale=wl.scale,
                                layout=A.CONTIGUOUS)
    assert np.array_equal(out, ref_out, equal_nan=True)
    assert np.array_equal(lse, ref_lse)
