"""Thin Python binding of the C ABI in ``include/decode_attn.h`` and
``include/nvfp4_mm.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library.  torch tensors supply device memory and the current CUDA stream.  If
the library has not been built, or a tensor is not on a CUDA device, the
calls raise -- there is no CPU path.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libdecode_attn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = 0, 1, 2, 3, 4
INVARIANT, BALANCED = 0, 1
KV_BF16, KV_FP8_E4M3, KV_NVFP4 = 0, 1, 2
CONTIGUOUS, PAGED, INDEXED = 0, 1, 2
VARIANT_FMA, VARIANT_MLA, VARIANT_GQA_TC = 0, 1, 2
DEVERR_LENGTH, DEVERR_INDEX, DEVERR_TIMEOUT = 1, 2, 4
FLAG_TEST_STALL = 1  # da_problem.flags test hook (see include/decode_attn.h)

LAYOUT_CODES = {"contiguous": CONTIGUOUS, "paged": PAGED, "indexed": INDEXED}

# Every symbol the header declares (tests check the library exports them).
EXPORTS = (
    "decode_attn_version", "decode_attn_status_string", "decode_attn_split_constants",
    "decode_attn_workspace_bytes", "decode_attn_plan", "decode_attn_run",
    "decode_attn_combine", "decode_attn_forward", "decode_attn_read_error",
    "decode_attn_copy_plan", "decode_attn_forward_static", "decode_attn_plan_extra",
    "decode_attn_run_extra", "decode_attn_forward_extra",
    "nvfp4_mm_workspace_bytes", "nvfp4_mm", "nvfp4_mm_read_error",
)

# NVFP4 weight matmul (include/nvfp4_mm.h)
NVFP4_TILE_N, NVFP4_ROW_TILE, NVFP4_K_CHUNK = 128, 32, 1024
NVFP4_X_F32, NVFP4_X_BF16 = 0, 1

# Size of the fixed device array decode_attn_forward_static uses as scratch.
STATIC_WORKSPACE_BYTES = 64 << 20


class DaProblem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim_qk", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("width", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("shared_latent", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("extra_width", ctypes.c_int32),
        ("extra_num_blocks", ctypes.c_int64),
        ("kv_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
    ]


class DaPlan(ctypes.Structure):
    _fields_ = [
        ("prob", DaProblem),
        ("policy", ctypes.c_int32),
        ("variant", ctypes.c_int32),
        ("tile_tokens", ctypes.c_int32),
        ("min_tiles_per_split", ctypes.c_int32),
        ("max_splits", ctypes.c_int32),
        ("num_parts", ctypes.c_int32),
        ("fixed_overhead", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("device", ctypes.c_int32),
        ("has_extra", ctypes.c_int32),
        ("ws", ctypes.c_void_p),
        ("ws_bytes", ctypes.c_size_t),
        ("off_n_splits", ctypes.c_uint64),
        ("off_split_begin", ctypes.c_uint64),
        ("off_work", ctypes.c_uint64),
        ("off_item_desc", ctypes.c_uint64),
        ("off_lse_part", ctypes.c_uint64),
        ("off_o_part", ctypes.c_uint64),
    ]


class DecodeAttnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().decode_attn_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


_LIB = None


def lib():
    """Open the CUDA library (built by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    P = ctypes.POINTER
    L.decode_attn_version.restype = ctypes.c_char_p
    L.decode_attn_version.argtypes = []
    L.decode_attn_status_string.restype = ctypes.c_char_p
    L.decode_attn_status_string.argtypes = [ctypes.c_int]
    L.decode_attn_split_constants.restype = ctypes.c_int
    L.decode_attn_split_constants.argtypes = [P(DaProblem), P(i32), P(i32), P(i32), P(i32)]
    L.decode_attn_workspace_bytes.restype = ctypes.c_int
    L.decode_attn_workspace_bytes.argtypes = [P(DaProblem), P(sz)]
    L.decode_attn_plan.restype = ctypes.c_int
    L.decode_attn_plan.argtypes = [P(DaProblem), i32, vp, vp, sz, P(DaPlan), vp]
    L.decode_attn_run.restype = ctypes.c_int
    L.decode_attn_run.argtypes = [P(DaPlan), vp, vp, vp, vp, vp, vp, vp, vp]
    L.decode_attn_combine.restype = ctypes.c_int
    L.decode_attn_combine.argtypes = [P(DaPlan), vp, vp, vp]
    L.decode_attn_forward.restype = ctypes.c_int
    L.decode_attn_forward.argtypes = [P(DaProblem), i32, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    L.decode_attn_read_error.restype = ctypes.c_int
    L.decode_attn_read_error.argtypes = [P(DaPlan), P(i32), vp]
    L.decode_attn_plan_extra.restype = ctypes.c_int
    L.decode_attn_plan_extra.argtypes = [P(DaProblem), i32, vp, vp, vp, sz, P(DaPlan), vp]
    L.decode_attn_run_extra.restype = ctypes.c_int
    L.decode_attn_run_extra.argtypes = [P(DaPlan), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.decode_attn_forward_extra.restype = ctypes.c_int
    L.decode_attn_forward_extra.argtypes = [P(DaProblem), i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            vp, sz, vp, vp, vp]
    L.decode_attn_forward_static.restype = ctypes.c_int
    L.decode_attn_forward_static.argtypes = [P(DaProblem), i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                             P(DaPlan)]
    L.decode_attn_copy_plan.restype = ctypes.c_int
    L.decode_attn_copy_plan.argtypes = [P(DaPlan), vp, vp, P(i32), vp, vp]
    L.nvfp4_mm_workspace_bytes.restype = sz
    L.nvfp4_mm_workspace_bytes.argtypes = [i32, i32, i32]
    L.nvfp4_mm.restype = ctypes.c_int
    L.nvfp4_mm.argtypes = [vp, i32, vp, vp, ctypes.c_float, i32, i32, i32, vp, vp, vp, sz, vp]
    L.nvfp4_mm_read_error.restype = ctypes.c_int
    L.nvfp4_mm_read_error.argtypes = [vp, P(i32), vp]
    _LIB = L
    return L


def _check(status, where):
    if status != OK:
        raise DecodeAttnError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


# cache tensors: bf16, or E4M3 bytes (uint8 / float8_e4m3fn) for DA_KV_FP8_E4M3
_KV = (torch.bfloat16, torch.uint8) + ((torch.float8_e4m3fn,)
                                        if hasattr(torch, "float8_e4m3fn") else ())


def _dev_ptr(t: Optional[torch.Tensor], name: str, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def problem(*, batch, num_q_heads, num_kv_heads, head_dim_qk, head_dim_v=None, layout,
            scale, page_size=0, width=0, num_blocks=0, shared_latent=False, extra_width=0,
            extra_num_blocks=0, kv_dtype=KV_BF16, k_scale=1.0, v_scale=1.0) -> DaProblem:
    """Fill a ``da_problem``.  ``layout`` is a name or a DA_KV_* code."""
    if isinstance(layout, str):
        layout = LAYOUT_CODES[layout]
    return DaProblem(batch, num_q_heads, num_kv_heads, head_dim_qk,
                     head_dim_qk if head_dim_v is None else head_dim_v, layout, page_size,
                     width, num_blocks, scale, int(bool(shared_latent)), 0, extra_width,
                     extra_num_blocks, kv_dtype, k_scale, v_scale)


def problem_for(wl) -> DaProblem:
    """The ``da_problem`` of a ``workloads.Workload``."""
    extra = getattr(wl, "extra_k", None) is not None
    return problem(batch=wl.B, num_q_heads=wl.H_q, num_kv_heads=wl.H_kv, head_dim_qk=wl.D_qk,
                   head_dim_v=wl.D_v, layout=wl.layout, scale=wl.scale,
                   page_size=wl.page_size if wl.layout == "paged" else 0, width=wl.width,
                   num_blocks=wl.num_blocks, shared_latent=wl.v is None,
                   extra_width=wl.extra_table.shape[1] if extra else 0,
                   extra_num_blocks=wl.extra_k.shape[0] if extra else 0,
                   kv_dtype=(KV_NVFP4 if getattr(wl, "kv_nvfp4", False) else
                             KV_FP8_E4M3 if getattr(wl, "kv_fp8", False) else KV_BF16),
                   k_scale=getattr(wl, "k_scale", 1.0), v_scale=getattr(wl, "v_scale", 1.0))


def version() -> str:
    return lib().decode_attn_version().decode()


def split_constants(prob: DaProblem):
    """(variant, tile_tokens, min_tiles_per_split, max_splits) for ``prob``."""
    v, t, m, s = (ctypes.c_int32() for _ in range(4))
    _check(lib().decode_attn_split_constants(ctypes.byref(prob), ctypes.byref(v), ctypes.byref(t),
                                             ctypes.byref(m), ctypes.byref(s)), "split_constants")
    return v.value, t.value, m.value, s.value


def workspace_bytes(prob: DaProblem) -> int:
    n = ctypes.c_size_t()
    _check(lib().decode_attn_workspace_bytes(ctypes.byref(prob), ctypes.byref(n)),
           "workspace_bytes")
    return n.value


def workspace(prob: DaProblem, device="cuda") -> torch.Tensor:
    """A device buffer of the required size (torch allocates it; 256-byte aligned)."""
    return torch.empty(max(workspace_bytes(prob), 256), dtype=torch.uint8, device=device)


def plan(prob: DaProblem, policy: int, lengths: torch.Tensor, ws: torch.Tensor,
         stream=None) -> DaPlan:
    pl = DaPlan()
    _check(lib().decode_attn_plan(ctypes.byref(prob), policy,
                                  _dev_ptr(lengths, "lengths", torch.int32),
                                  _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                  ctypes.byref(pl), _stream(stream)), "plan")
    return pl


def run(pl: DaPlan, q, k, v, table, lengths, out, lse, stream=None):
    _check(lib().decode_attn_run(ctypes.byref(pl), _dev_ptr(q, "q", torch.bfloat16),
                                 _dev_ptr(k, "k", _KV), _dev_ptr(v, "v", _KV),
                                 _dev_ptr(table, "table", torch.int32),
                                 _dev_ptr(lengths, "lengths", torch.int32),
                                 _dev_ptr(out, "out", torch.bfloat16),
                                 _dev_ptr(lse, "lse", torch.float32), _stream(stream)), "run")


def combine(pl: DaPlan, out, lse, stream=None):
    _check(lib().decode_attn_combine(ctypes.byref(pl), _dev_ptr(out, "out", torch.bfloat16),
                                     _dev_ptr(lse, "lse", torch.float32), _stream(stream)),
           "combine")


def forward(prob: DaProblem, policy, q, k, v, table, lengths, ws, out, lse, stream=None):
    """plan + run + combine through the single C entry point."""
    _check(lib().decode_attn_forward(ctypes.byref(prob), policy, _dev_ptr(q, "q", torch.bfloat16),
                                     _dev_ptr(k, "k", _KV),
                                     _dev_ptr(v, "v", _KV),
                                     _dev_ptr(table, "table", torch.int32),
                                     _dev_ptr(lengths, "lengths", torch.int32),
                                     _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                     _dev_ptr(out, "out", torch.bfloat16),
                                     _dev_ptr(lse, "lse", torch.float32), _stream(stream)),
           "forward")


def forward_static(prob: DaProblem, policy, q, k, v, table, lengths, out, lse,
                   stream=None) -> DaPlan:
    """The forward pass with the library's own fixed device scratch array, for
    callers that cannot allocate device memory (see the header): no workspace
    argument, nothing allocated.  Raises DecodeAttnError(ERR_WORKSPACE) for a
    problem whose workspace exceeds STATIC_WORKSPACE_BYTES.  Calls sharing a
    device must not overlap on the GPU.  Returns the call's plan, which
    read_error accepts until the next call overwrites the array."""
    pl = DaPlan()
    _check(lib().decode_attn_forward_static(ctypes.byref(prob), policy,
                                            _dev_ptr(q, "q", torch.bfloat16),
                                            _dev_ptr(k, "k", _KV),
                                            _dev_ptr(v, "v", _KV),
                                            _dev_ptr(table, "table", torch.int32),
                                            _dev_ptr(lengths, "lengths", torch.int32),
                                            _dev_ptr(out, "out", torch.bfloat16),
                                            _dev_ptr(lse, "lse", torch.float32), _stream(stream),
                                            ctypes.byref(pl)),
           "forward_static")
    return pl


def plan_extra(prob: DaProblem, policy: int, lengths, extra_lengths, ws, stream=None) -> DaPlan:
    pl = DaPlan()
    _check(lib().decode_attn_plan_extra(ctypes.byref(prob), policy,
                                        _dev_ptr(lengths, "lengths", torch.int32),
                                        _dev_ptr(extra_lengths, "extra_lengths", torch.int32),
                                        _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                        ctypes.byref(pl), _stream(stream)), "plan_extra")
    return pl


def run_extra(pl: DaPlan, q, k, v, table, lengths, extra_k, extra_v, extra_indices,
              extra_lengths, out, lse, stream=None):
    _check(lib().decode_attn_run_extra(
        ctypes.byref(pl), _dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k, "k", _KV),
        _dev_ptr(v, "v", _KV), _dev_ptr(table, "table", torch.int32),
        _dev_ptr(lengths, "lengths", torch.int32), _dev_ptr(extra_k, "extra_k", torch.bfloat16),
        _dev_ptr(extra_v, "extra_v", torch.bfloat16),
        _dev_ptr(extra_indices, "extra_indices", torch.int32),
        _dev_ptr(extra_lengths, "extra_lengths", torch.int32),
        _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(lse, "lse", torch.float32),
        _stream(stream)), "run_extra")


def forward_extra(prob: DaProblem, policy, q, k, v, table, lengths, extra_k, extra_v,
                  extra_indices, extra_lengths, ws, out, lse, stream=None):
    """plan + run + combine over a main and a second (index-gathered) KV source."""
    _check(lib().decode_attn_forward_extra(
        ctypes.byref(prob), policy, _dev_ptr(q, "q", torch.bfloat16),
        _dev_ptr(k, "k", _KV), _dev_ptr(v, "v", _KV),
        _dev_ptr(table, "table", torch.int32), _dev_ptr(lengths, "lengths", torch.int32),
        _dev_ptr(extra_k, "extra_k", torch.bfloat16), _dev_ptr(extra_v, "extra_v", torch.bfloat16),
        _dev_ptr(extra_indices, "extra_indices", torch.int32),
        _dev_ptr(extra_lengths, "extra_lengths", torch.int32),
        _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
        _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(lse, "lse", torch.float32),
        _stream(stream)), "forward_extra")


def read_error(pl: DaPlan, stream=None) -> int:
    code = ctypes.c_int32()
    _check(lib().decode_attn_read_error(ctypes.byref(pl), ctypes.byref(code), _stream(stream)),
           "read_error")
    return code.value


def copy_plan(pl: DaPlan, stream=None):
    """(n_splits[B], split_begin[B, max_splits+1], work[n_work]) as CPU int32 tensors."""
    B, ms = pl.prob.batch, pl.max_splits
    n_splits = torch.zeros(B, dtype=torch.int32)
    split_begin = torch.zeros((B, ms + 1), dtype=torch.int32)
    work = torch.zeros(B * ms, dtype=torch.int32)
    n_work = ctypes.c_int32()
    _check(lib().decode_attn_copy_plan(ctypes.byref(pl), _ptr(n_splits), _ptr(split_begin),
                                       ctypes.byref(n_work), _ptr(work), _stream(stream)),
           "copy_plan")
    return n_splits, split_begin, work[:n_work.value]


def decode_attention(q, k, v, lengths, table=None, *, layout, scale, page_size=0,
                     num_blocks=None, d_v=None, policy=INVARIANT, ws=None, out=None, lse=None,
                     stream=None):
    """Batch-invariant split-KV decode attention (plan + run + combine).

    q: bf16 [B, H_q, D_qk]; k, v: bf16 caches in ``layout`` (v=None for a
    shared latent cache, then ``d_v`` gives the value width); lengths: int32
    [B]; table: int32 [B, width] page ids / indices (None when contiguous).
    Returns (out bf16 [B, H_q, D_v], lse fp32 [B, H_q]).
    """
    if isinstance(layout, str):
        layout = LAYOUT_CODES[layout]
    B, H_q, D_qk = q.shape
    H_kv = k.shape[-2]
    D_v = (v.shape[-1] if v is not None else d_v)
    if layout == CONTIGUOUS:
        width = k.shape[1]
        nb = k.shape[0] * k.shape[1]
    else:
        width = table.shape[1]
        nb = k.shape[0] if num_blocks is None else num_blocks
    prob = problem(batch=B, num_q_heads=H_q, num_kv_heads=H_kv, head_dim_qk=D_qk,
                   head_dim_v=D_v, layout=layout, scale=scale, page_size=page_size,
                   width=width, num_blocks=nb, shared_latent=v is None)
    if ws is None:
        ws = workspace(prob, q.device)
    if out is None:
        out = torch.empty((B, H_q, D_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    forward(prob, policy, q, k, v, table, lengths, ws, out, lse, stream)
    return out, lse


def run_workload(wl, policy=INVARIANT, ws=None, out=None, lse=None, stream=None):
    """decode_attention on a ``workloads.Workload`` whose tensors are on the GPU."""
    prob = problem_for(wl)
    if ws is None:
        ws = workspace(prob, wl.q.device)
    if out is None:
        out = torch.empty((wl.B, wl.H_q, wl.D_v), dtype=torch.bfloat16, device=wl.q.device)
    if lse is None:
        lse = torch.empty((wl.B, wl.H_q), dtype=torch.float32, device=wl.q.device)
    if getattr(wl, "extra_k", None) is not None:
        forward_extra(prob, policy, wl.q, wl.k, wl.v, wl.table, wl.lengths, wl.extra_k, wl.extra_v,
                      wl.extra_table, wl.extra_lengths, ws, out, lse, stream)
    else:
        forward(prob, policy, wl.q, wl.k, wl.v, wl.table, wl.lengths, ws, out, lse, stream)
    return out, lse


# ----------------------------------------------------------------- NVFP4 weight matmul

def nvfp4_workspace_bytes(n: int, N: int, K: int) -> int:
    """Workspace bytes of one ``nvfp4_mm`` call (0: shape not supported)."""
    return int(lib().nvfp4_mm_workspace_bytes(n, N, K))


def nvfp4_workspace(n: int, N: int, K: int, device="cuda") -> torch.Tensor:
    nb = nvfp4_workspace_bytes(n, N, K)
    if nb == 0:
        raise DecodeAttnError(ERR_UNSUPPORTED, f"nvfp4 shape n={n} N={N} K={K}")
    return torch.empty(nb, dtype=torch.uint8, device=device)


def nvfp4_mm(x, codes, scales, global_scale, *, y=None, y_bf16=None, ws=None, stream=None):
    """y = global_scale * bf16(x) @ W^T for an NVFP4 weight (nvfp4_mm.h).

    x: fp32 or bf16 [n, K]; codes: uint8 [N, K / 2]; scales: uint8 (or
    float8_e4m3fn) [N, K / 16]; returns y fp32 [n, N] (and fills ``y_bf16``
    when given).  Every row's result is independent of n and of the other rows.
    """
    n, K = x.shape
    N = codes.shape[0]
    if codes.shape != (N, K // 2) or scales.shape != (N, K // 16):
        raise ValueError(f"codes {tuple(codes.shape)} / scales {tuple(scales.shape)} "
                         f"do not match x {tuple(x.shape)}")
    x_dtype = {torch.float32: NVFP4_X_F32, torch.bfloat16: NVFP4_X_BF16}.get(x.dtype)
    if x_dtype is None:
        raise ValueError(f"x must be float32 or bfloat16, got {x.dtype}")
    if y is None:
        y = torch.empty((n, N), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = nvfp4_workspace(n, N, K, x.device)
    _check(lib().nvfp4_mm(_dev_ptr(x, "x"), x_dtype, _dev_ptr(codes, "codes", torch.uint8),
                          _dev_ptr(scales, "scales", _KV[1:]), ctypes.c_float(global_scale),
                          n, N, K, _dev_ptr(y, "y", torch.float32),
                          _dev_ptr(y_bf16, "y_bf16", torch.bfloat16), _dev_ptr(ws, "ws"),
                          ws.numel(), _stream(stream)), "nvfp4_mm")
    return y


def nvfp4_read_error(ws: torch.Tensor, stream=None) -> int:
    """Device error bits (DEVERR_*) of the last ``nvfp4_mm`` call on ``ws``."""
    code = ctypes.c_int32()
    _check(lib().nvfp4_mm_read_error(_dev_ptr(ws, "ws"), ctypes.byref(code), _stream(stream)),
           "nvfp4_read_error")
    return code.value


def run_nvfp4(m, ws=None, y=None, y_bf16=None, stream=None):
    """nvfp4_mm on a ``workloads.Nvfp4Matmul`` whose tensors are on the GPU."""
    return nvfp4_mm(m.x, m.codes, m.scales, m.global_scale, y=y, y_bf16=y_bf16, ws=ws,
                    stream=stream)
