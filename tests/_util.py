"""Helpers shared by the tests: oracle evaluation on workload tensors and the
parity tolerance.  No attention arithmetic lives here -- only marshalling."""

import numpy as np
import torch

from oracle import attention as A
from oracle import bf16 as OB
from oracle import fp8 as OF
from oracle import nvfp4 as ON

# Parity bar (out): |gpu - oracle| <= max(1e-2, one bf16 ULP of the oracle
# value).  A correctly rounded bf16 result is within half a ULP of the exact
# value; for |o| < 4 that is <= 0.0078 < 1e-2, leaving >= 0.002 for fp32
# accumulation error; for |o| >= 4 half a ULP alone exceeds 1e-2, so the bar
# there is one ULP.  LSE (fp32, natural log): |gpu - oracle| <= 1e-4.
OUT_ATOL = 1e-2
LSE_ATOL = 1e-4


class Bf16Cache:
    """Read-only view of a bf16 torch cache that the oracle can index like a
    numpy array; every read comes back as exact fp64."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        if not isinstance(idx, tuple):
            idx = (idx,)
        idx = tuple(torch.as_tensor(np.asarray(i)) if not isinstance(i, (int, slice)) else i
                    for i in idx)
        return self.t[idx].double().numpy()


class Fp8Cache:
    """Read-only view of an E4M3 byte cache (uint8 torch tensor) with its
    scale; every read is decoded by the oracle (exact fp64)."""

    def __init__(self, t, scale):
        self.t = t
        self.scale = scale
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        if not isinstance(idx, tuple):
            idx = (idx,)
        idx = tuple(torch.as_tensor(np.asarray(i)) if not isinstance(i, (int, slice)) else i
                    for i in idx)
        return OF.dequantize(self.t[idx].numpy(), self.scale)


class Nvfp4Cache:
    """Read-only view of an NVFP4 cache (codes and block-scale uint8 torch
    tensors) with its global scale; every read is decoded by the oracle."""

    def __init__(self, codes, blocks, scale):
        self.codes, self.blocks, self.scale = codes, blocks, scale
        self.shape = tuple(codes.shape[:-1]) + (codes.shape[-1] * 2,)

    def __getitem__(self, idx):
        if not isinstance(idx, tuple):
            idx = (idx,)
        idx = tuple(torch.as_tensor(np.asarray(i)) if not isinstance(i, (int, slice)) else i
                    for i in idx)
        return ON.dequantize_cache(self.codes[idx].numpy(), self.blocks[idx].numpy(), self.scale)


def oracle_for(wl, rows=None, heads=None):
    """fp64 oracle (out, lse) of a CPU workload, optionally on a subset."""
    table = None if wl.table is None else wl.table.numpy()
    if getattr(wl, "kv_nvfp4", False):
        return A.attend(wl.q.double().numpy(), Nvfp4Cache(wl.k, wl.k_blocks, wl.k_scale),
                        Nvfp4Cache(wl.v, wl.v_blocks, wl.v_scale), wl.lengths.numpy(),
                        scale=wl.scale, layout=wl.layout, table=table,
                        page_size=wl.page_size, d_v=wl.D_v, rows=rows, heads=heads)
    if getattr(wl, "kv_fp8", False):
        # a shared latent cache: values are the leading D_v bytes of each row,
        # decoded at the value scale
        v = (Fp8Cache(wl.k[..., :wl.D_v], wl.v_scale) if wl.v is None
             else Fp8Cache(wl.v, wl.v_scale))
        return A.attend(wl.q.double().numpy(), Fp8Cache(wl.k, wl.k_scale),
                        v, wl.lengths.numpy(), scale=wl.scale,
                        layout=wl.layout, table=table, page_size=wl.page_size, d_v=wl.D_v,
                        rows=rows, heads=heads)
    extra = {}
    if getattr(wl, "extra_k", None) is not None:
        extra = dict(extra_k=Bf16Cache(wl.extra_k),
                     extra_v=None if wl.extra_v is None else Bf16Cache(wl.extra_v),
                     extra_table=wl.extra_table.numpy(), extra_lengths=wl.extra_lengths.numpy())
    return A.attend(wl.q.double().numpy(), Bf16Cache(wl.k),
                    None if wl.v is None else Bf16Cache(wl.v), wl.lengths.numpy(),
                    scale=wl.scale, layout=wl.layout, table=table, page_size=wl.page_size,
                    d_v=wl.D_v, rows=rows, heads=heads, **extra)


def assert_parity(out_gpu, lse_gpu, ref_out, ref_lse, rows=None, heads=None):
    """Element-wise parity of GPU (bf16 out, fp32 lse) against the oracle."""
    o = out_gpu.double().cpu().numpy()
    l = lse_gpu.double().cpu().numpy()
    rows = range(o.shape[0]) if rows is None else rows
    heads = range(o.shape[1]) if heads is None else heads
    ri = np.ix_(list(rows), list(heads))
    o, l, ro, rl = o[ri], l[ri], ref_out[ri], ref_lse[ri]
    tol = np.maximum(OUT_ATOL, OB.ulp(ro))
    err = np.abs(o - ro)
    bad = ~(err <= tol)
    assert not bad.any(), (f"out mismatch at {np.argwhere(bad)[:5].tolist()}: "
                           f"max err {np.nanmax(err):.4g}")
    both_inf = np.isneginf(l) & np.isneginf(rl)
    lerr = np.where(both_inf, 0.0, np.abs(l - rl))
    assert np.all(lerr <= LSE_ATOL), f"lse max err {np.nanmax(lerr):.4g}"
    return float(np.max(err)) if err.size else 0.0, float(np.max(lerr)) if lerr.size else 0.0
