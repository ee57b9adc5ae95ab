"""Plain fp64 softmax attention for decode rows -- the oracle's definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The method (FlashMLA issue #212, "Sparse MLA decode is not batch-invariant",
Summary + Measurement) reaches exactly -- up to rounding order -- the plain
softmax-attention result of each query row over its own KV list.  This module
writes that definition out, with no tiling, splitting or reordering:

    s_i   = scale * sum_d q[d] * K[i, d]            (fp64)
    m     = max_i s_i
    lse   = m + log sum_i exp(s_i - m)              (natural log)
    out   = sum_i exp(s_i - m) * V[i, :] / sum_i exp(s_i - m)

Readings of points the pages leave open:

* GQA head map: query head ``j`` reads KV head ``j // (H_q / H_kv)``.
* Latent (MLA-style) KV: when no separate V cache is given, ``V = K[..., :D_v]``
  (the value is the leading ``D_v`` dims of the shared latent row).
* Index entries at positions ``>= length`` are never read (the page's
  ``topk_length`` equals the count of valid entries).
* An empty row (length 0) gives ``out = 0`` and ``lse = -inf``.
* ``scale`` multiplies the exact dot product; q is never pre-scaled.
"""

from __future__ import annotations

import math

import numpy as np

CONTIGUOUS = "contiguous"
PAGED = "paged"
INDEXED = "indexed"
LAYOUTS = (CONTIGUOUS, PAGED, INDEXED)


def row_entries(cache, b, length, layout, table=None, page_size=None):
    """Return row ``b``'s first ``length`` KV entries in list order.

    cache layouts (last two dims are ``[H_kv, D]``):
      contiguous: ``cache[B, Lmax, H_kv, D]``; entry t is ``cache[b, t]``
      paged:      ``cache[num_pages, P, H_kv, D]``; entry t is
                  ``cache[table[b, t // P], t % P]``
      indexed:    ``cache[num_slots, H_kv, D]``; entry t is
                  ``cache[table[b, t]]`` (``table`` holds top-k indices)
    Returns an fp64 array ``[length, H_kv, D]``.
    """
    t = np.arange(length)
    if layout == CONTIGUOUS:
        rows = cache[b, :length]
    elif layout == PAGED:
        pages = np.asarray(table[b])[t // page_size]
        rows = cache[pages, t % page_size]
    elif layout == INDEXED:
        slots = np.asarray(table[b])[:length]
        rows = cache[slots]
    else:
        raise ValueError(f"unknown layout {layout!r}")
    return np.asarray(rows, dtype=np.float64)


def attend_row(q_row, K, V, scale):
    """Softmax attention of one query vector over keys ``K[L, D]``, values ``V[L, Dv]``.

    Returns ``(out[Dv], lse)`` in fp64.  L == 0 gives zeros and ``-inf``.
    """
    L = K.shape[0]
    if L == 0:
        return np.zeros(V.shape[1], dtype=np.float64), -math.inf
    s = scale * (K @ np.asarray(q_row, dtype=np.float64))
    m = s.max()
    e = np.exp(s - m)          # shifted by the max so nothing overflows
    z = e.sum()
    return (e @ V) / z, m + math.log(z)


def attend(q, k_cache, v_cache, lengths, *, scale, layout, table=None,
           page_size=None, d_v=None, rows=None, heads=None,
           extra_k=None, extra_v=None, extra_table=None, extra_lengths=None):
    """Attention of every (row, query head) over the row's own KV list.

    q:        ``[B, H_q, D_qk]`` (any float dtype; converted to fp64 exactly)
    k_cache:  the key cache in ``layout`` (see ``row_entries``)
    v_cache:  the value cache in the same layout, or ``None`` for a shared
              latent cache where ``V = K[..., :d_v]``
    lengths:  ``[B]`` integer KV lengths (``topk_length`` for ``indexed``)
    rows, heads: optional subsets to evaluate (others are left as NaN)
    extra_*:  an optional second KV source, always index-gathered: row b's
              list continues with ``extra_k[extra_table[b, t]]`` for
              t < extra_lengths[b] (values from ``extra_v``, or the leading
              ``d_v`` dims of ``extra_k`` for a shared latent cache).  The
              FlashMLA issue #212 page re-runs rows with their
              ``extra_indices_in_kvcache`` / ``extra_topk_length`` sliced
              alongside the main indices (Measurement, item 2): the row
              attends over both lists.

    Returns ``(out[B, H_q, D_v], lse[B, H_q])`` in fp64.
    """
    q = np.asarray(q)
    B, H_q, _ = q.shape
    H_kv = k_cache.shape[-2]
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    G = H_q // H_kv
    if v_cache is None:
        if d_v is None:
            raise ValueError("d_v is required for a shared latent cache")
        Dv = d_v
    else:
        Dv = v_cache.shape[-1]
    out = np.full((B, H_q, Dv), np.nan)
    lse = np.full((B, H_q), np.nan)
    rows = range(B) if rows is None else rows
    heads = range(H_q) if heads is None else heads
    for b in rows:
        L = int(lengths[b])
        K = row_entries(k_cache, b, L, layout, table, page_size)
        if v_cache is None:
            V = K[..., :Dv]
        else:
            V = row_entries(v_cache, b, L, layout, table, page_size)
        if extra_k is not None:
            Le = int(extra_lengths[b])
            Ke = row_entries(extra_k, b, Le, INDEXED, extra_table)
            Ve = Ke[..., :Dv] if extra_v is None else row_entries(extra_v, b, Le, INDEXED,
                                                                   extra_table)
            K = np.concatenate([K, Ke], axis=0)
            V = np.concatenate([V, Ve], axis=0)
        for j in heads:
            h = j // G
            out[b, j], lse[b, j] = attend_row(q[b, j], K[:, h, :], V[:, h, :], scale)
    return out, lse


def lse_merge(partials):
    """Merge per-split partial results ``[(out_s, lse_s), ...]`` into one.

    Each partial is the softmax attention over a disjoint piece of the row's
    KV list.  The merged result is the attention over their union:

        M   = max_s lse_s
        W   = sum_s exp(lse_s - M)
        out = sum_s (exp(lse_s - M) / W) * out_s
        lse = M + log W

    Pieces with ``lse_s = -inf`` (empty) carry zero weight; if every piece is
    empty the result is ``(0, -inf)``.  Source: FlashMLA issue #212, "Where it
    comes from" (the combine step's per-split LSE rescale and fp32 sum).
    """
    outs = [np.asarray(o, dtype=np.float64) for o, _ in partials]
    lses = [float(l) for _, l in partials]
    M = max(lses)
    if M == -math.inf:
        return np.zeros_like(outs[0]), -math.inf
    w = [math.exp(l - M) for l in lses]
    W = math.fsum(w)
    out = sum((wi / W) * oi for wi, oi in zip(w, outs))
    return out, M + math.log(W)
