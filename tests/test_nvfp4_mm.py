"""NVFP4 weight matmul: the tensor-core path against the fp64 oracle, bitwise
independence of a row's result from the row count n and from its position
(the property the gllm issue's GEMV/GEMM switch breaks), and the argument
rules (CPU checks need no GPU).

Tolerance.  y is an fp32 sum: per 1024-wide K chunk the tensor core adds 64
groups of 16 exact bf16 x bf16 products into an fp32 accumulator, then the
chunk sums are added and multiplied by the global scale.  Each of those
roundings is at most a few units of 2^-24 of the magnitudes summed, so for
K <= 4096 the error is below ~2^-16 * sum_k |x_k w_k|; the gate allows 2^-14
times that sum (``oracle.nvfp4.abs_products``).  A wrong nibble order, block
scale or operand orientation moves y by a large fraction of that sum and
fails it."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import nvfp4 as ON
from invariant_decode_attention_gb300 import workloads as W

gpu = pytest.mark.gpu
REL = 2.0 ** -14


@pytest.fixture(scope="module")
def api():
    from invariant_decode_attention_gb300 import api as _api
    _api.lib()
    return _api


def oracle(m, rows=None):
    x = m.x.double().numpy() if rows is None else m.x[rows].double().numpy()
    c, s = m.codes.numpy(), m.scales.numpy()
    return ON.matmul(x, c, s, m.global_scale), ON.abs_products(x, c, s, m.global_scale)


def check(y, m, rows=None):
    ref, mag = oracle(m, rows)
    got = y.double().cpu().numpy()
    err = np.abs(got - ref)
    bad = err > REL * mag
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; worst rel "
                           f"{float((err / mag).max()):.3g}")


@gpu
@pytest.mark.parametrize("n,N,K", [(1, 128, 64), (3, 128, 1024), (5, 256, 1088),
                                   (32, 128, 2048), (33, 256, 3136), (70, 384, 1216),
                                   (100, 128, 4096)])
def test_parity(api, n, N, K):
    m = W.nvfp4_matmul(n, N, K, seed=n * 7 + K)
    g = m.to("cuda")
    ybf = torch.empty((n, N), dtype=torch.bfloat16, device="cuda")
    y = api.run_nvfp4(g, y_bf16=ybf)
    torch.cuda.synchronize()
    check(y, m)
    # bf16 output is the round-to-nearest-even of the fp32 result
    assert torch.equal(ybf, y.to(torch.bfloat16))


@gpu
def test_row_bits_do_not_depend_on_n_or_position(api):
    N, K = 256, 2112  # three K chunks, the last one partial
    codes, scales, gs = W.nvfp4_weight(N, K, seed=21)
    pool = W.nvfp4_activations(300, K, seed=22)
    dc, ds = codes.cuda(), scales.cuda()
    target = pool[7:8]
    solo = api.nvfp4_mm(target.cuda(), dc, ds, gs)
    gen = torch.Generator().manual_seed(5)
    for n in (1, 2, 31, 32, 33, 64, 65, 100, 255, 300):
        others = pool[torch.randperm(300, generator=gen)[:n]]
        pos = int(torch.randint(0, n, (1,), generator=gen))
        x = others.clone()
        x[pos] = target[0]
        y = api.nvfp4_mm(x.cuda(), dc, ds, gs)
        assert torch.equal(y[pos], solo[0]), f"n={n} pos={pos}"
    # every row of a full batch equals that row alone
    y_all = api.nvfp4_mm(pool.cuda(), dc, ds, gs)
    for i in (0, 31, 32, 33, 150, 299):
        assert torch.equal(y_all[i], api.nvfp4_mm(pool[i:i + 1].cuda(), dc, ds, gs)[0])
    check(y_all[:40], W.Nvfp4Matmul("pool", pool[:40], codes, scales, gs))


@gpu
def test_bf16_activations_match_rounded_fp32(api):
    m = W.nvfp4_matmul(9, 256, 1536, seed=31)
    g = m.to("cuda")
    y32 = api.run_nvfp4(g)
    y16 = api.nvfp4_mm(g.x.to(torch.bfloat16), g.codes, g.scales, g.global_scale)
    assert torch.equal(y32, y16)


@gpu
def test_repeat_runs_and_error_word(api):
    m = W.nvfp4_matmul(40, 384, 3072, seed=41).to("cuda")
    ws = api.nvfp4_workspace(m.n, m.N, m.K)
    y0 = api.run_nvfp4(m, ws=ws).clone()
    for _ in range(8):
        assert torch.equal(api.run_nvfp4(m, ws=ws), y0)
    assert api.nvfp4_read_error(ws) == 0


@gpu
def test_projection_size_sampled(api):
    # the 8192 x 4096 projection at 32 rows (the largest the pages' GEMV path
    # takes) and 33 rows (the first their GEMM path takes): sampled rows
    # against the oracle, and the same row's bits across row counts
    m32 = W.nvfp4_proj(n=32)
    g = m32.to("cuda")
    y32 = api.run_nvfp4(g)
    rows = [0, 13, 31]
    check(y32[rows], m32, rows=rows)
    x = g.x
    y1 = api.nvfp4_mm(x[13:14].contiguous(), g.codes, g.scales, g.global_scale)
    extra = W.nvfp4_activations(224, m32.K, seed=77).cuda()
    y33 = api.nvfp4_mm(torch.cat([extra[:1], x]), g.codes, g.scales, g.global_scale)
    y256 = api.nvfp4_mm(torch.cat([extra, x]), g.codes, g.scales, g.global_scale)
    assert torch.equal(y1[0], y32[13])
    assert torch.equal(y33[14], y32[13])
    assert torch.equal(y256[224 + 13], y32[13])


@gpu
def test_zero_rows_and_special_weights(api):
    # n = 0 enqueues nothing; all-zero codes give exact zeros; a NaN block
    # scale poisons exactly the outputs of its weight row
    N, K = 128, 256
    codes, scales, gs = W.nvfp4_weight(N, K, seed=3)
    x = W.nvfp4_activations(4, K, seed=4).cuda()
    y0 = api.nvfp4_mm(x[:0], codes.cuda(), scales.cuda(), gs)
    assert y0.shape == (0, N)
    z = api.nvfp4_mm(x, torch.zeros_like(codes).cuda(), scales.cuda(), gs)
    assert torch.equal(z, torch.zeros_like(z))
    s2 = scales.clone()
    s2[5, 3] = 0x7F
    y = api.nvfp4_mm(x, codes.cuda(), s2.cuda(), gs).cpu()
    assert torch.isnan(y[:, 5]).all()
    assert torch.isfinite(torch.cat([y[:, :5], y[:, 6:]], 1)).all()


def test_argument_rules(api):
    L = api.lib()
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: every case fails before any device work
    assert L.nvfp4_mm_workspace_bytes(1, 100, 64) == 0
    assert L.nvfp4_mm_workspace_bytes(1, 128, 48) == 0
    # header, tile counters (256-byte rounded), rounded activations, partials
    assert L.nvfp4_mm_workspace_bytes(32, 128, 1024) == 256 + 256 + 32 * 1024 * 2
    assert L.nvfp4_mm_workspace_bytes(33, 128, 2048) == (256 + 256 + 64 * 2048 * 2 +
                                                         2 * 33 * 128 * 4)
    def call(x=fake, xd=0, codes=fake, scales=fake, gs=1.0, n=4, N=128, K=64, y=fake, yb=None,
             ws=fake, wsb=1 << 30):
        return L.nvfp4_mm(x, xd, codes, scales, ctypes.c_float(gs), n, N, K, y, yb, ws, wsb, None)
    assert call(xd=2) == api.ERR_INVALID_ARG
    assert call(gs=float("nan")) == api.ERR_INVALID_ARG
    assert call(gs=float("inf")) == api.ERR_INVALID_ARG
    assert call(N=100) == api.ERR_UNSUPPORTED
    assert call(K=96) == api.ERR_UNSUPPORTED
    assert call(n=-1) == api.ERR_UNSUPPORTED
    assert call(n=0, x=None, codes=None, scales=None, y=None, ws=None) == api.OK
    assert call(x=None) == api.ERR_INVALID_ARG
    assert call(y=None) == api.ERR_INVALID_ARG
    assert call(x=vp((1 << 20) + 8)) == api.ERR_INVALID_ARG
    assert call(ws=None) == api.ERR_WORKSPACE
    assert call(ws=vp((1 << 20) + 16)) == api.ERR_WORKSPACE
    assert call(wsb=100) == api.ERR_WORKSPACE
