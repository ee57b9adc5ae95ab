"""Seeded synthetic decode-attention inputs.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.  Everything is generated on the CPU with
``torch.Generator().manual_seed(seed)`` so that both sides see identical bits.

Cache layouts (``H`` = KV heads, ``D`` = head dim, bf16):

* contiguous: ``[B, Lmax, H, D]``; row b's entry t is ``cache[b, t]``
* paged:      ``[num_pages, P, H, D]`` + ``table int32[B, width]``; entry t of
              row b is ``cache[table[b, t // P], t % P]``; unused table slots
              hold -1
* indexed:    ``[num_slots, H, D]`` + ``table int32[B, width]`` of slot indices
              (a row's top-k list); entries past the row's length hold -1

A quantized workload (``kv_fp8``) holds K and V as E4M3 bytes (uint8) with
one fp32 scale per cache; ``quantize_fp8`` makes one from a bf16 workload by
torch's own float8_e4m3fn conversion of value / scale.  An NVFP4 workload
(``kv_nvfp4``) holds, per cache, E2M1 codes ``[..., H, D/2]`` and E4M3 block
scales ``[..., H, D/16]`` drawn at random (``nvfp4_kv``); on a device the two
are views into one buffer, codes first, as the library reads them.

The named workloads follow the five configurations the pages' problem
statement is measured on (tiny dense, GQA paged, MLA-style sparse, ragged
invariance sweep, long context); sizes are spelled out in each function.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

CONTIGUOUS = "contiguous"
PAGED = "paged"
INDEXED = "indexed"


@dataclasses.dataclass
class Workload:
    name: str
    layout: str
    q: torch.Tensor                 # [B, H_q, D_qk] bf16
    k: torch.Tensor                 # key cache (or shared latent cache), bf16
    v: Optional[torch.Tensor]       # value cache, or None when V = k[..., :D_v]
    lengths: torch.Tensor           # int32 [B]
    table: Optional[torch.Tensor]   # int32 [B, width] page table / indices
    page_size: int
    H_q: int
    H_kv: int
    D_qk: int
    D_v: int
    scale: float
    # optional second, index-gathered KV source continuing each row's list
    extra_k: Optional[torch.Tensor] = None        # [slots, H_kv, D_qk]
    extra_v: Optional[torch.Tensor] = None        # [slots, H_kv, D_v] or None (latent)
    extra_table: Optional[torch.Tensor] = None    # int32 [B, extra_width]
    extra_lengths: Optional[torch.Tensor] = None  # int32 [B]
    # quantized cache: k and v are E4M3 bytes (uint8), value = scale * e4m3
    kv_fp8: bool = False
    k_scale: float = 1.0
    v_scale: float = 1.0
    # NVFP4 cache: k / v hold the E2M1 codes [..., H, D/2] (uint8), these the
    # E4M3 block scales [..., H, D/16] (uint8)
    kv_nvfp4: bool = False
    k_blocks: Optional[torch.Tensor] = None
    v_blocks: Optional[torch.Tensor] = None

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def width(self):
        """Contiguous: Lmax; paged: page-table width; indexed: index width."""
        if self.layout == CONTIGUOUS:
            return self.k.shape[1]
        return self.table.shape[1]

    @property
    def num_blocks(self):
        """Pages (paged) or slots (indexed) in the cache; rows*Lmax otherwise."""
        if self.layout == CONTIGUOUS:
            return self.k.shape[0] * self.k.shape[1]
        return self.k.shape[0]

    def kv_bytes(self):
        """Bytes of K and V the rows actually attend over (the algorithmic payload)."""
        n = int(self.lengths.to(torch.int64).sum())
        if self.extra_lengths is not None:
            n += int(self.extra_lengths.to(torch.int64).sum())
        if self.kv_nvfp4:
            per = self.H_kv * (self.D_qk // 2 + self.D_qk // 16)
            return n * 2 * per
        eb = 1 if self.kv_fp8 else 2
        per_entry_k = self.H_kv * self.D_qk * eb
        per_entry_v = 0 if self.v is None else self.H_kv * self.D_v * eb
        return n * (per_entry_k + per_entry_v)

    def to(self, device):
        def mv(t):
            return None if t is None else t.to(device)
        kv = dict(k=mv(self.k), v=mv(self.v))
        if self.kv_nvfp4:
            kv = {}
            for name in ("k", "v"):
                codes, blocks = getattr(self, name), getattr(self, name + "_blocks")
                kv[name], kv[name + "_blocks"] = nvfp4_buffer(codes, blocks, device)
        return dataclasses.replace(self, q=mv(self.q), **kv,
                                   lengths=mv(self.lengths), table=mv(self.table),
                                   extra_k=mv(self.extra_k), extra_v=mv(self.extra_v),
                                   extra_table=mv(self.extra_table),
                                   extra_lengths=mv(self.extra_lengths))


def nvfp4_buffer(codes, blocks, device):
    """One buffer on `device` holding the codes, then the block scales (the
    layout the library reads); returns (codes view, block-scales view)."""
    n = codes.numel()
    buf = torch.empty(n + blocks.numel(), dtype=torch.uint8, device=device)
    buf[:n].copy_(codes.reshape(-1))
    buf[n:].copy_(blocks.reshape(-1))
    return buf[:n].view(codes.shape), buf[n:].view(blocks.shape)


def _randn(shape, g):
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def page_table(lengths, page_size, g, width=None, spare_pages=0):
    """Random page ids for each row: every row gets ceil(L/P) distinct pages
    drawn from a shuffled pool.  Returns (table[B, width], num_pages)."""
    need = [-(-int(L) // page_size) for L in lengths]
    width = max(max(need), 1) if width is None else width
    num_pages = sum(need) + spare_pages
    perm = torch.randperm(max(num_pages, 1), generator=g)[:num_pages].to(torch.int32)
    table = torch.full((len(need), width), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, max(num_pages, 1)


def make(layout, lengths, *, H_q, H_kv, D_qk, D_v=None, page_size=16, width=None,
         num_slots=None, latent=False, seed=0, scale=None, name="custom",
         identity_table=False, draw_kv=True):
    """General seeded workload.  q, K, V ~ N(0, 1) rounded to bf16.

    latent=True makes one shared latent cache with V = K[..., :D_v] (MLA-style).
    identity_table=True lays paged rows out in consecutive pages (no shuffle).
    draw_kv=False leaves K and V undrawn (uninitialised placeholders of the
    right shapes, for a caller that replaces them); q and the table are the
    same as with draw_kv=True.
    """
    g = torch.Generator().manual_seed(seed)
    lengths = torch.as_tensor(lengths, dtype=torch.int32)
    B = lengths.numel()
    D_v = D_qk if D_v is None else D_v
    scale = 1.0 / math.sqrt(D_qk) if scale is None else scale
    q = _randn((B, H_q, D_qk), g)
    table = None
    if layout == CONTIGUOUS:
        Lmax = max(int(lengths.max()) if B else 0, 1) if width is None else width
        kshape = (B, Lmax, H_kv, D_qk)
        vshape = (B, Lmax, H_kv, D_v)
    elif layout == PAGED:
        if identity_table:
            need = [-(-int(L) // page_size) for L in lengths]
            w = max(max(need), 1) if width is None else width
            table = torch.full((B, w), -1, dtype=torch.int32)
            off = 0
            for b, n in enumerate(need):
                table[b, :n] = torch.arange(off, off + n, dtype=torch.int32)
                off += n
            num_pages = max(off, 1)
        else:
            table, num_pages = page_table(lengths.tolist(), page_size, g, width)
        kshape = (num_pages, page_size, H_kv, D_qk)
        vshape = (num_pages, page_size, H_kv, D_v)
    elif layout == INDEXED:
        w = max(int(lengths.max()) if B else 0, 1) if width is None else width
        n_slots = max(w, 1) if num_slots is None else num_slots
        table = torch.full((B, w), -1, dtype=torch.int32)
        for b in range(B):
            L = int(lengths[b])
            table[b, :L] = torch.randperm(n_slots, generator=g)[:L].to(torch.int32)
        kshape = (n_slots, H_kv, D_qk)
        vshape = (n_slots, H_kv, D_v)
    else:
        raise ValueError(layout)
    if draw_kv:
        k = _randn(kshape, g)
        v = None if latent else _randn(vshape, g)
    else:
        k = torch.empty(kshape, dtype=torch.bfloat16)
        v = None if latent else torch.empty(vshape, dtype=torch.bfloat16)
    return Workload(name, layout, q, k, v, lengths, table, page_size,
                    H_q, H_kv, D_qk, D_v, scale)


# --------------------------------------------------------------------------
# The five named configurations.
# --------------------------------------------------------------------------

def tiny(seed=1000):
    """Tiny dense decode: 4 rows, 8 q heads sharing 1 KV head, head_dim 64,
    KV lengths {17, 100, 256, 1000}, contiguous cache, scale 1/sqrt(64)."""
    return make(CONTIGUOUS, [17, 100, 256, 1000], H_q=8, H_kv=1, D_qk=64,
                seed=seed, name="tiny_dense_b4_h8x1_d64")


def gqa_paged(seed=1001, B=32):
    """GQA paged decode: 32 rows, 32 q / 8 KV heads, head_dim 128, page 16,
    shuffled page table, lengths uniform in [512, 8192]."""
    g = torch.Generator().manual_seed(seed)
    lengths = torch.randint(512, 8193, (B,), generator=g, dtype=torch.int64)
    return make(PAGED, lengths.tolist(), H_q=32, H_kv=8, D_qk=128, page_size=16,
                width=8192 // 16, seed=seed + 7919, name="gqa_paged_b32_h32x8_d128_p16")


def gqa16_paged(seed=1007, B=32):
    """GQA paged decode with 16 query heads per KV head (the tensor-core
    GQA variant's case): 32 rows, 128 q / 8 KV heads, head_dim 128, page 16,
    shuffled page table, lengths uniform in [512, 8192] -- the GQA paged
    recipe with four times the query heads."""
    g = torch.Generator().manual_seed(seed)
    lengths = torch.randint(512, 8193, (B,), generator=g, dtype=torch.int64)
    return make(PAGED, lengths.tolist(), H_q=128, H_kv=8, D_qk=128, page_size=16,
                width=8192 // 16, seed=seed + 7919, name="gqa16_paged_b32_h128x8_d128_p16")


def mla_sparse(seed=1002, B=64, num_slots=65536, max_topk=2048):
    """MLA-style sparse decode: 64 rows, 128 q heads sharing one latent KV row
    of 576 dims (the first 512 are V), 65536 cache slots, per-row distinct
    uniform top-k indices, topk_length uniform in [256, 2048], scale 576^-0.5."""
    g = torch.Generator().manual_seed(seed)
    lengths = torch.randint(256, max_topk + 1, (B,), generator=g, dtype=torch.int64)
    return make(INDEXED, lengths.tolist(), H_q=128, H_kv=1, D_qk=576, D_v=512,
                width=max_topk, num_slots=num_slots, latent=True, seed=seed + 7919,
                name="mla_sparse_b64_h128_d576v512_topk2048")


def long_context(seed=1004, B=8, L=131072, page_size=64, identity_table=False, draw_kv=True):
    """Long-context decode: 8 rows of 131072 entries each, 32 q / 8 KV heads,
    head_dim 128, paged with page 64 (shuffled table unless identity_table)."""
    return make(PAGED, [L] * B, H_q=32, H_kv=8, D_qk=128, page_size=page_size,
                seed=seed, identity_table=identity_table, draw_kv=draw_kv,
                name=f"long_context_b{B}_l{L}_h32x8_d128_p{page_size}")


# Ragged invariance sweep: one fixed target row (length 4096, GQA 32/8,
# d=128, page 16) embedded at random positions in batches of 1..256 rows whose
# other rows have log-uniform lengths in [1, 131072].
RAGGED_TARGET_LEN = 4096
RAGGED_MAX_LEN = 131072


def ragged_target(seed=1003, H_q=32):
    """The target row's own data: q [H_q, 128], K and V [4096, 8, 128] (bf16)."""
    g = torch.Generator().manual_seed(seed)
    q = _randn((H_q, 128), g)
    k = _randn((RAGGED_TARGET_LEN, 8, 128), g)
    v = _randn((RAGGED_TARGET_LEN, 8, 128), g)
    return q, k, v


def ragged_batch_lengths(B, seed):
    """Lengths of a ragged batch and the target's position in it.

    Batchmates: L = clamp(floor(2 ** (17 * U)), 1, 131072), U ~ U[0, 1).
    Returns (lengths list with the target's 4096 at `pos`, pos)."""
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(B, generator=g, dtype=torch.float64)
    lens = torch.clamp(torch.floor(torch.exp2(17.0 * u)), 1, RAGGED_MAX_LEN).to(torch.int64)
    pos = int(torch.randint(0, B, (1,), generator=g))
    lens[pos] = RAGGED_TARGET_LEN
    return lens.tolist(), pos


def ragged_page_table(lengths, seed, page_size=16, width=None):
    """Shuffled page table for a ragged batch: (table[B, width], num_pages)."""
    g = torch.Generator().manual_seed(seed + 1)
    return page_table(lengths, page_size, g, width)


def _e4m3_bytes(t, scale):
    """E4M3 bytes of value / scale (torch's float8_e4m3fn conversion)."""
    return (t.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8)


class RaggedSweep:
    """Batches of the ragged invariance sweep, assembled on a device.

    All batches share one page pool whose content is random filler (drawn on
    the device: batchmates are never compared with anything).  For each batch
    the target row's q, K and V are written into its own freshly shuffled
    pages, so the target attends over identical data at a different position,
    with different page ids and different batchmates every time.

    H_q: query heads over the 8 KV heads (32 in the sweep's configuration).
    kv_fp8: the caches hold E4M3 bytes (scales 1/64), the target's bytes
    converted once from its bf16 values.  kv_nvfp4: the caches are NVFP4
    (codes, then block scales, in one buffer per cache; global scales 1/2),
    the target's parts drawn at random like the pool's.  extra: every row's list continues
    in a second, index-gathered cache [extra_slots, 8, 128]; the target's
    RAGGED_TARGET_EXTRA extra entries are written to fresh distinct slots per
    batch, batchmates take uniform extra lengths in [0, extra_width] of
    random (possibly repeated) slots.
    """

    def __init__(self, sizes, device="cuda", seed=1003, page_size=16, kv_fp8=False,
                 extra=False, extra_slots=32768, extra_width=1024, H_q=32, kv_nvfp4=False):
        self.sizes = list(sizes)
        self.page_size = page_size
        self.device = device
        self.seed = seed
        self.kv_fp8 = kv_fp8
        self.kv_nvfp4 = kv_nvfp4
        self.extra = extra
        self.extra_slots = extra_slots
        self.extra_width = extra_width
        self.H_q = H_q
        self.q_t, self.k_t, self.v_t = ragged_target(seed, H_q)
        self.batches = []
        max_pages = 1
        for B in self.sizes:
            lens, pos = ragged_batch_lengths(B, seed=seed * 1000 + B)
            table, num_pages = ragged_page_table(lens, seed=seed * 1000 + B,
                                                 page_size=page_size,
                                                 width=RAGGED_MAX_LEN // page_size)
            self.batches.append((B, lens, pos, table))
            max_pages = max(max_pages, num_pages)
        self.num_pages = max_pages
        g = torch.Generator(device=device).manual_seed(seed)
        shape = (max_pages, page_size, 8, 128)
        self.k_pool = torch.randn(shape, generator=g, device=device, dtype=torch.bfloat16)
        self.v_pool = torch.randn(shape, generator=g, device=device, dtype=torch.bfloat16)
        n_tp = RAGGED_TARGET_LEN // page_size
        kt = self.k_t.view(n_tp, page_size, 8, 128)
        vt = self.v_t.view(n_tp, page_size, 8, 128)
        if kv_fp8:
            self.k_scale = self.v_scale = 1.0 / 64
            self.k_pool = _e4m3_bytes(self.k_pool, self.k_scale)
            self.v_pool = _e4m3_bytes(self.v_pool, self.v_scale)
            kt, vt = _e4m3_bytes(kt, self.k_scale), _e4m3_bytes(vt, self.v_scale)
        self.ktb_cpu = self.vtb_cpu = None
        if kv_nvfp4:
            self.k_scale = self.v_scale = 0.5
            gn = torch.Generator().manual_seed(seed + 29)
            shape_t = (RAGGED_TARGET_LEN, 8, 128)
            kc, kb = nvfp4_codes(shape_t, gn)
            vc, vb = nvfp4_codes(shape_t, gn)
            kt, vt = kc.view(n_tp, page_size, 8, 64), vc.view(n_tp, page_size, 8, 64)
            self.ktb_cpu = kb.view(n_tp, page_size, 8, 8)
            self.vtb_cpu = vb.view(n_tp, page_size, 8, 8)
            self._ktb, self._vtb = self.ktb_cpu.to(device), self.vtb_cpu.to(device)
            pools = []
            for _ in range(2):  # filler parts drawn on the device, codes then scales
                nc, nb = max_pages * page_size * 8 * 64, max_pages * page_size * 8 * 8
                buf = torch.empty(nc + nb, dtype=torch.uint8, device=device)
                buf[:nc] = torch.randint(0, 256, (nc,), generator=g, device=device,
                                         dtype=torch.int32).to(torch.uint8)
                e = torch.randint(4, 8, (nb,), generator=g, device=device, dtype=torch.int32)
                buf[nc:] = ((e << 3) | 5).to(torch.uint8)
                pools.append((buf[:nc].view(max_pages, page_size, 8, 64),
                              buf[nc:].view(max_pages, page_size, 8, 8)))
            (self.k_pool, self.kb_pool), (self.v_pool, self.vb_pool) = pools
        self.kt_cpu, self.vt_cpu = kt, vt  # the target's cache rows as stored
        self._kt = kt.to(device)
        self._vt = vt.to(device)
        self._qt = self.q_t.to(device)
        if extra:
            gx = torch.Generator().manual_seed(seed + 17)
            self.xk_t = _randn((RAGGED_TARGET_EXTRA, 8, 128), gx)
            self.xv_t = _randn((RAGGED_TARGET_EXTRA, 8, 128), gx)
            xshape = (extra_slots, 8, 128)
            self.xk_pool = torch.randn(xshape, generator=g, device=device, dtype=torch.bfloat16)
            self.xv_pool = torch.randn(xshape, generator=g, device=device, dtype=torch.bfloat16)
            self._xkt, self._xvt = self.xk_t.to(device), self.xv_t.to(device)

    def _wl(self, name, q, k, v, lengths, table, kb=None, vb=None, **extra):
        kw = {}
        if self.kv_fp8:
            kw = dict(kv_fp8=True, k_scale=self.k_scale, v_scale=self.v_scale)
        if self.kv_nvfp4:
            kw = dict(kv_nvfp4=True, k_blocks=kb, v_blocks=vb, k_scale=self.k_scale,
                      v_scale=self.v_scale)
        return Workload(name, PAGED, q, k, v, lengths, table, self.page_size, self.H_q, 8, 128,
                        128, 128 ** -0.5, **extra, **kw)

    def solo(self):
        """The target row alone, in its own 256 pages (and, with a second
        source, its extra entries in slots 0 .. RAGGED_TARGET_EXTRA-1 of a
        cache of their own)."""
        n_tp = RAGGED_TARGET_LEN // self.page_size
        table = torch.full((1, RAGGED_MAX_LEN // self.page_size), -1, dtype=torch.int32)
        table[0, :n_tp] = torch.arange(n_tp, dtype=torch.int32)
        extra = {}
        if self.extra:
            xt = torch.full((1, self.extra_width), -1, dtype=torch.int32)
            xt[0, :RAGGED_TARGET_EXTRA] = torch.arange(RAGGED_TARGET_EXTRA, dtype=torch.int32)
            extra = dict(extra_k=self._xkt.contiguous(), extra_v=self._xvt.contiguous(),
                         extra_table=xt.to(self.device),
                         extra_lengths=torch.tensor([RAGGED_TARGET_EXTRA], dtype=torch.int32,
                                                    device=self.device))
        k, v, kb, vb = self._kt.contiguous(), self._vt.contiguous(), None, None
        if self.kv_nvfp4:
            k, kb = nvfp4_buffer(self._kt, self._ktb, self.device)
            v, vb = nvfp4_buffer(self._vt, self._vtb, self.device)
        return self._wl("ragged_solo", self._qt[None].contiguous(), k, v,
                        torch.tensor([RAGGED_TARGET_LEN], dtype=torch.int32, device=self.device),
                        table.to(self.device), kb=kb, vb=vb, **extra)

    def solo_cpu(self):
        """The solo row as a CPU workload with a contiguous cache (for the
        oracle)."""
        extra = {}
        if self.extra:
            xt = torch.arange(RAGGED_TARGET_EXTRA, dtype=torch.int32)[None]
            extra = dict(extra_k=self.xk_t, extra_v=self.xv_t, extra_table=xt,
                         extra_lengths=torch.tensor([RAGGED_TARGET_EXTRA], dtype=torch.int32))
        kw = dict(kv_fp8=True, k_scale=self.k_scale, v_scale=self.v_scale) if self.kv_fp8 else {}
        dk = 64 if self.kv_nvfp4 else 128
        k = self.kt_cpu.reshape(RAGGED_TARGET_LEN, 8, dk)[None]
        v = self.vt_cpu.reshape(RAGGED_TARGET_LEN, 8, dk)[None]
        if self.kv_nvfp4:
            kw = dict(kv_nvfp4=True, k_scale=self.k_scale, v_scale=self.v_scale,
                      k_blocks=self.ktb_cpu.reshape(RAGGED_TARGET_LEN, 8, 8)[None],
                      v_blocks=self.vtb_cpu.reshape(RAGGED_TARGET_LEN, 8, 8)[None])
        return Workload("ragged_solo_cpu", CONTIGUOUS, self.q_t[None], k, v,
                        torch.tensor([RAGGED_TARGET_LEN], dtype=torch.int32), None, 0, self.H_q,
                        8, 128, 128, 128 ** -0.5, **extra, **kw)

    def batch(self, i):
        """(Workload on the device, target position) of the i-th batch."""
        B, lens, pos, table = self.batches[i]
        n_tp = RAGGED_TARGET_LEN // self.page_size
        pages = table[pos, :n_tp].to(device=self.device, dtype=torch.int64)
        self.k_pool[pages] = self._kt
        self.v_pool[pages] = self._vt
        nv = {}
        if self.kv_nvfp4:
            self.kb_pool[pages] = self._ktb
            self.vb_pool[pages] = self._vtb
            nv = dict(kb=self.kb_pool, vb=self.vb_pool)
        g = torch.Generator(device=self.device).manual_seed(7 * B + 1)
        q = torch.randn((B, self.H_q, 128), generator=g, device=self.device, dtype=torch.bfloat16)
        q[pos] = self._qt
        extra = {}
        if self.extra:
            gx = torch.Generator().manual_seed(self.seed * 1000 + B + 5)
            el = torch.randint(0, self.extra_width + 1, (B,), generator=gx, dtype=torch.int32)
            el[pos] = RAGGED_TARGET_EXTRA
            xt = torch.randint(0, self.extra_slots, (B, self.extra_width), generator=gx,
                               dtype=torch.int32)
            xt[torch.arange(self.extra_width)[None, :] >= el[:, None]] = -1
            slots = torch.randperm(self.extra_slots, generator=gx)[:RAGGED_TARGET_EXTRA]
            xt[pos] = -1
            xt[pos, :RAGGED_TARGET_EXTRA] = slots.to(torch.int32)
            sd = slots.to(self.device)
            self.xk_pool[sd] = self._xkt
            self.xv_pool[sd] = self._xvt
            extra = dict(extra_k=self.xk_pool, extra_v=self.xv_pool,
                         extra_table=xt.to(self.device), extra_lengths=el.to(self.device))
        wl = self._wl(f"ragged_b{B}", q, self.k_pool, self.v_pool,
                      torch.tensor(lens, dtype=torch.int32, device=self.device),
                      table.to(self.device), **nv, **extra)
        return wl, pos


# Ragged sweep of the shared-latent (MLA-style) variant: one target row
# (128 heads, top-k 1536 entries of a 65536-slot latent cache, 576 dims of
# which the first 512 are V) in batches whose other rows take top-k lengths
# log-uniform in [1, 2048]; optionally a second latent source (target: 300
# entries of a 16384-slot cache, batchmates uniform in [0, 512]).
RAGGED_TARGET_EXTRA = 700
LATENT_TARGET_LEN = 1536
LATENT_TARGET_EXTRA = 300


class RaggedSweepLatent:
    """Batches of the shared-latent ragged sweep, assembled on a device.

    The caches are pools of random filler drawn on the device; for every
    batch the target row's latent entries are written into fresh distinct
    slots (in the same order), so the target attends over identical data at
    a new position, through new slot ids, among new batchmates whose index
    lists are random (possibly repeated) slots."""

    def __init__(self, sizes, device="cuda", seed=1008, extra=False, num_slots=65536,
                 width=2048, extra_slots=16384, extra_width=512, kv_fp8=False):
        # kv_fp8: an E4M3 latent cache (one source), scores at scale 1/64 and
        # values at 1/32 of the stored bytes
        assert not (kv_fp8 and extra), "E4M3 latent cache: one source"
        self.kv_fp8 = kv_fp8
        self.k_scale, self.v_scale = (1.0 / 64, 1.0 / 32) if kv_fp8 else (1.0, 1.0)
        self.sizes = list(sizes)
        self.device = device
        self.seed = seed
        self.extra = extra
        self.num_slots, self.width = num_slots, width
        self.extra_slots, self.extra_width = extra_slots, extra_width
        g = torch.Generator().manual_seed(seed)
        self.q_t = _randn((128, 576), g)
        self.k_t = _randn((LATENT_TARGET_LEN, 1, 576), g)
        self.xk_t = _randn((LATENT_TARGET_EXTRA, 1, 576), g) if extra else None
        gd = torch.Generator(device=device).manual_seed(seed)
        self.pool = torch.randn((num_slots, 1, 576), generator=gd, device=device,
                                dtype=torch.bfloat16)
        self.xpool = (torch.randn((extra_slots, 1, 576), generator=gd, device=device,
                                  dtype=torch.bfloat16) if extra else None)
        if kv_fp8:
            self.k_t = _e4m3_bytes(self.k_t, self.k_scale)
            self.pool = _e4m3_bytes(self.pool, self.k_scale)
        self._qt, self._kt = self.q_t.to(device), self.k_t.to(device)
        self._xkt = self.xk_t.to(device) if extra else None

    def solo_cpu(self):
        """The target row alone with caches of its own (CPU tensors)."""
        table = torch.arange(LATENT_TARGET_LEN, dtype=torch.int32)[None]
        extra = {}
        if self.extra:
            extra = dict(extra_k=self.xk_t, extra_v=None,
                         extra_table=torch.arange(LATENT_TARGET_EXTRA, dtype=torch.int32)[None],
                         extra_lengths=torch.tensor([LATENT_TARGET_EXTRA], dtype=torch.int32))
        return Workload("latent_solo", INDEXED, self.q_t[None], self.k_t, None,
                        torch.tensor([LATENT_TARGET_LEN], dtype=torch.int32), table, 0, 128, 1,
                        576, 512, 576 ** -0.5, **extra, **self._fp8_kw())

    def _fp8_kw(self):
        if not self.kv_fp8:
            return {}
        return dict(kv_fp8=True, k_scale=self.k_scale, v_scale=self.v_scale)

    def solo(self):
        return self.solo_cpu().to(self.device)

    def batch(self, i):
        """(Workload on the device, target position) of the i-th batch."""
        B = self.sizes[i]
        g = torch.Generator().manual_seed(self.seed * 1000 + B)
        u = torch.rand(B, generator=g, dtype=torch.float64)
        lens = torch.clamp(torch.floor(torch.exp2(11.0 * u)), 1, self.width).to(torch.int32)
        pos = int(torch.randint(0, B, (1,), generator=g))
        lens[pos] = LATENT_TARGET_LEN
        table = torch.randint(0, self.num_slots, (B, self.width), generator=g, dtype=torch.int32)
        table[torch.arange(self.width)[None, :] >= lens[:, None]] = -1
        slots = torch.randperm(self.num_slots, generator=g)[:LATENT_TARGET_LEN]
        table[pos] = -1
        table[pos, :LATENT_TARGET_LEN] = slots.to(torch.int32)
        self.pool[slots.to(self.device)] = self._kt
        gq = torch.Generator(device=self.device).manual_seed(11 * B + 3)
        q = torch.randn((B, 128, 576), generator=gq, device=self.device, dtype=torch.bfloat16)
        q[pos] = self._qt
        extra = {}
        if self.extra:
            el = torch.randint(0, self.extra_width + 1, (B,), generator=g, dtype=torch.int32)
            el[pos] = LATENT_TARGET_EXTRA
            xt = torch.randint(0, self.extra_slots, (B, self.extra_width), generator=g,
                               dtype=torch.int32)
            xt[torch.arange(self.extra_width)[None, :] >= el[:, None]] = -1
            xs = torch.randperm(self.extra_slots, generator=g)[:LATENT_TARGET_EXTRA]
            xt[pos] = -1
            xt[pos, :LATENT_TARGET_EXTRA] = xs.to(torch.int32)
            self.xpool[xs.to(self.device)] = self._xkt
            extra = dict(extra_k=self.xpool, extra_v=None, extra_table=xt.to(self.device),
                         extra_lengths=el.to(self.device))
        wl = Workload(f"latent_ragged_b{B}", INDEXED, q, self.pool, None, lens.to(self.device),
                      table.to(self.device), 0, 128, 1, 576, 512, 576 ** -0.5, **extra,
                      **self._fp8_kw())
        return wl, pos


def with_extra(wl, extra_lengths, num_slots, width=None, seed=0):
    """The workload plus a second, index-gathered KV source: row b's list
    continues with extra_lengths[b] distinct slots of a fresh cache of
    `num_slots` rows (values N(0, 1) in bf16; latent when wl.v is None)."""
    g = torch.Generator().manual_seed(seed)
    el = torch.as_tensor(extra_lengths, dtype=torch.int32)
    w = max(int(el.max()) if el.numel() else 0, 1) if width is None else width
    table = torch.full((wl.B, w), -1, dtype=torch.int32)
    for b in range(wl.B):
        n = int(el[b])
        table[b, :n] = torch.randperm(num_slots, generator=g)[:n].to(torch.int32)
    ek = _randn((num_slots, wl.H_kv, wl.D_qk), g)
    ev = None if wl.v is None else _randn((num_slots, wl.H_kv, wl.D_v), g)
    return dataclasses.replace(wl, extra_k=ek, extra_v=ev, extra_table=table, extra_lengths=el,
                               name=wl.name + "_extra")


def mla_sparse_extra(seed=1005):
    """The MLA-style sparse workload with a second latent KV source: per row
    extra_topk uniform in [0, 512] distinct slots of a 16384-slot extra cache
    (the sparse decode path with an extra k cache)."""
    g = torch.Generator().manual_seed(seed)
    el = torch.randint(0, 513, (64,), generator=g, dtype=torch.int64)
    return with_extra(mla_sparse(), el.tolist(), 16384, width=512, seed=seed + 1)


def quantize_fp8(wl, k_scale=1.0 / 64, v_scale=1.0 / 64, name=None):
    """The same workload with its K and V caches stored as E4M3 bytes:
    ``bytes = float8_e4m3fn(value / k_scale)`` (torch's conversion, round to
    nearest even).  With N(0, 1) data and scale 1/64 every value stays far
    inside the format's range (|value / scale| < 448).  A shared latent
    cache (v None) is one byte array: its scores use k_scale, its values (the
    leading D_v bytes of each row) v_scale."""
    assert wl.extra_k is None, "one source"
    v = None if wl.v is None else _e4m3_bytes(wl.v, v_scale)
    return dataclasses.replace(wl, k=_e4m3_bytes(wl.k, k_scale), v=v, kv_fp8=True,
                               k_scale=float(k_scale), v_scale=float(v_scale),
                               name=name or wl.name + "_fp8")


def nvfp4_codes(shape, g):
    """Random NVFP4 parts for a cache of bf16 shape [..., H, D]: codes uint8
    [..., H, D/2] uniform over 0..255 (all sixteen E2M1 codes in both nibbles)
    and block scales uint8 [..., H, D/16], positive E4M3 codes with exponent
    field 4..7 and a uniform fraction (values 2^-3 .. 1.875)."""
    *lead, D = shape
    codes = torch.randint(0, 256, (*lead, D // 2), generator=g, dtype=torch.int32)
    e = torch.randint(4, 8, (*lead, D // 16), generator=g, dtype=torch.int32)
    f = torch.randint(0, 8, (*lead, D // 16), generator=g, dtype=torch.int32)
    return codes.to(torch.uint8), ((e << 3) | f).to(torch.uint8)


def nvfp4_kv(wl, k_scale=0.5, v_scale=0.5, seed=0, name=None):
    """The workload with NVFP4 K and V caches of the same shapes, drawn at
    random (nvfp4_codes) -- the format's values, not a rounding of wl's: with
    global scales 1/2 the elements are 0 .. 5.6 in magnitude."""
    assert wl.v is not None and wl.extra_k is None, "separate K and V, one source"
    g = torch.Generator().manual_seed(seed)
    kc, kb = nvfp4_codes(tuple(wl.k.shape), g)
    vc, vb = nvfp4_codes(tuple(wl.v.shape), g)
    return dataclasses.replace(wl, k=kc, v=vc, k_blocks=kb, v_blocks=vb, kv_nvfp4=True,
                               k_scale=float(k_scale), v_scale=float(v_scale),
                               name=name or wl.name + "_nvfp4")


def gqa_paged_nvfp4(seed=1001):
    """The GQA paged workload (32 rows, 32/8 heads, d = 128, page 16, lengths
    512..8192) with NVFP4 KV caches (global scales 1/2)."""
    return nvfp4_kv(gqa_paged(seed), seed=seed + 31,
                    name="gqa_paged_nvfp4_b32_h32x8_d128_p16")


def long_context_nvfp4(seed=1004):
    """The long-context workload (8 x 131072, 32/8 heads, d = 128, page 64)
    with NVFP4 KV caches (global scales 1/2)."""
    return nvfp4_kv(long_context(seed, draw_kv=False), seed=seed + 31,
                    name="long_context_nvfp4_b8_l131072_h32x8_d128_p64")


def gqa16_paged_fp8(seed=1007):
    """The 16-heads-per-KV-head GQA paged workload (32 rows, 128/8 heads,
    d = 128, page 16) with an E4M3 KV cache, scales 1/64."""
    return quantize_fp8(gqa16_paged(seed), name="gqa16_paged_fp8_b32_h128x8_d128_p16")


def mla_sparse_fp8(seed=1002):
    """The MLA-style sparse workload (64 rows, 128 heads, 576/512 latent,
    top-k <= 2048 of 65536 slots) with an E4M3 latent cache, scales 1/64."""
    return quantize_fp8(mla_sparse(seed), name="mla_sparse_fp8_b64_h128_d576_topk2048")


def gqa16_paged_nvfp4(seed=1007):
    """The 16-heads-per-KV-head GQA paged workload (32 rows, 128/8 heads,
    d = 128, page 16) with NVFP4 KV caches (global scales 1/2)."""
    return nvfp4_kv(gqa16_paged(seed), seed=seed + 31,
                    name="gqa16_paged_nvfp4_b32_h128x8_d128_p16")


def gqa_paged_fp8(seed=1001):
    """The GQA paged workload (32 rows, 32/8 heads, d = 128, page 16, lengths
    512..8192) with an E4M3 KV cache, scales 1/64."""
    return quantize_fp8(gqa_paged(seed), name="gqa_paged_fp8_b32_h32x8_d128_p16")


def long_context_fp8(seed=1004):
    """The long-context workload (8 x 131072, 32/8 heads, d = 128, page 64)
    with an E4M3 KV cache, scales 1/64."""
    return quantize_fp8(long_context(seed), name="long_context_fp8_b8_l131072_h32x8_d128_p64")


# ----------------------------------------------------------------- NVFP4 weight matmul

@dataclasses.dataclass
class Nvfp4Matmul:
    """Inputs of one weight matmul y = bf16(x) @ W^T with an NVFP4 weight.

    ``codes`` uint8 [N, K / 2]: two E2M1 codes per byte, element 2j of a row
    in the low nibble of byte j; ``scales`` uint8 [N, K / 16]: one E4M3 code
    per 16 consecutive weights of a row; ``global_scale``: one fp32 factor
    for the whole matrix; ``x`` fp32 [n, K]: the activations before rounding.
    """
    name: str
    x: torch.Tensor
    codes: torch.Tensor
    scales: torch.Tensor
    global_scale: float

    @property
    def n(self):
        return int(self.x.shape[0])

    @property
    def N(self):
        return int(self.codes.shape[0])

    @property
    def K(self):
        return int(self.x.shape[1])

    def weight_bytes(self):
        return self.codes.numel() + self.scales.numel()

    def to(self, device):
        return dataclasses.replace(self, x=self.x.to(device), codes=self.codes.to(device),
                                   scales=self.scales.to(device))

    def with_rows(self, x):
        """The same weight with other activation rows."""
        return dataclasses.replace(self, x=x)


def nvfp4_weight(N, K, seed, global_scale=1.0 / 128):
    """A random NVFP4 weight: every byte of ``codes`` uniform over 0..255 (all
    sixteen E2M1 codes in both nibbles, both zeros included) and positive
    E4M3 block scales with exponent field 4..10 and a uniform fraction, i.e.
    values 2^-3 .. 15 (no NaN code)."""
    if N <= 0 or K <= 0 or K % 16:
        raise ValueError("N > 0 and K a positive multiple of 16")
    g = torch.Generator().manual_seed(seed)
    codes = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    e = torch.randint(4, 11, (N, K // 16), generator=g, dtype=torch.int32)
    f = torch.randint(0, 8, (N, K // 16), generator=g, dtype=torch.int32)
    scales = ((e << 3) | f).to(torch.uint8)
    return codes, scales, float(global_scale)


def nvfp4_activations(n, K, seed):
    """n activation rows of N(0, 1) fp32 values (full fp32 fraction bits, so
    rounding to bf16 changes almost every one)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn((n, K), generator=g, dtype=torch.float32)


def nvfp4_matmul(n, N, K, seed, name=None):
    codes, scales, gs = nvfp4_weight(N, K, seed)
    x = nvfp4_activations(n, K, seed + 7919)
    return Nvfp4Matmul(name or f"nvfp4_n{n}_N{N}_K{K}", x, codes, scales, gs)


def nvfp4_proj(n=32, seed=1006):
    """A dense projection-sized NVFP4 weight (N = 8192 outputs, K = 4096
    inputs: 16.8 MB of codes + 2.1 MB of scales) with n activation rows;
    n = 32 is the largest row count the pages' GEMV path takes."""
    return nvfp4_matmul(n, 8192, 4096, seed, name=f"nvfp4_proj_n{n}_N8192_K4096")
