"""PyTorch-facing binding of the C ABI (argument marshalling only).

Every function takes CUDA tensors, checks dtype/layout/device, allocates the
outputs and the workspace the caller did not pass, and calls the entry point
of the same name on the current CUDA stream.  All computation happens in the
library's kernels; there is no CPU or PyTorch fallback.

``AttnQAT`` mirrors the pages' ``AttentionImpl(num_heads, head_size,
softmax_scale, causal).forward(q, k, v)`` ("attn_qat_train" API page,
``AttnQatTrainImpl``): q, k, v in [B, L, H, D] layout, dropout rejected,
softmax_scale None meaning 1/sqrt(D).
"""
from __future__ import annotations

import math

import torch

from . import _lib

BF16 = torch.bfloat16


def _stream_ptr(t: torch.Tensor):
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtype=BF16):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _check_bnhd(t, name, shape=None):
    _check(t, name)
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, N, H, D] tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _rows_ld(x: torch.Tensor):
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    return x.shape[0], x.shape[1], x.stride(0)


# ------------------------------------------------------------------ quantizer

def nvfp4_global_sf(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 scalar tensor 448*6/max(amax(|x|), 1e-12) computed on the device."""
    _check(x, "x")
    rows, cols, ld = _rows_ld(x)
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=x.device)
    _lib.call("nvfp4_global_sf", _ptr(x), rows, cols, ld, _ptr(out), _stream_ptr(x))
    return out


def nvfp4_fake_quant(x: torch.Tensor, global_sf: torch.Tensor | None = None,
                     out: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                     want_scales: bool = True):
    """NVFP4 fake quantization of a bf16 [rows, cols] matrix, cols % 16 == 0.

    Returns (out bf16 [rows, cols], scales uint8 [rows, cols/16] E4M3FN bytes or
    None).  ``global_sf`` is a device fp32 scalar or None (unit scale).
    """
    _check(x, "x")
    rows, cols, ld = _rows_ld(x)
    if out is None:
        out = torch.empty((rows, cols), dtype=BF16, device=x.device)
    _check(out, "out")
    if scales is None and want_scales:
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=x.device)
    if global_sf is not None:
        _check(global_sf, "global_sf", torch.float32)
    _lib.call("nvfp4_fake_quant", _ptr(x), rows, cols, ld, _ptr(global_sf), _ptr(out),
              out.stride(0), _ptr(scales), 0 if scales is None else scales.stride(0),
              _stream_ptr(x))
    return out, scales


def nvfp4_quantize_codes(x: torch.Tensor, global_sf: torch.Tensor | None = None,
                         codes: torch.Tensor | None = None, scales: torch.Tensor | None = None):
    """Packed NVFP4 codes (uint8 [rows, cols/2], element 2i in the low nibble) and
    E4M3FN scale bytes (uint8 [rows, cols/16])."""
    _check(x, "x")
    rows, cols, ld = _rows_ld(x)
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=x.device)
    if global_sf is not None:
        _check(global_sf, "global_sf", torch.float32)
    _lib.call("nvfp4_quantize_codes", _ptr(x), rows, cols, ld, _ptr(global_sf), _ptr(codes),
              codes.stride(0), _ptr(scales), scales.stride(0), _stream_ptr(x))
    return codes, scales


# ------------------------------------------------------------------ attention

def default_scale(d: int) -> float:
    """sm_scale default of attn_qat_train(): 1/sqrt(D)."""
    return 1.0 / math.sqrt(d)


def _scale(scale, d: int) -> float:
    """The softmax scale to pass: None or NaN mean the default 1/sqrt(D)."""
    if scale is None or math.isnan(float(scale)):
        return default_scale(d)
    return float(scale)


def attn_qat_fwd_workspace(b, nq, nkv, h, d) -> int:
    return int(_lib.load().attn_qat_fwd_workspace(b, nq, nkv, h, d))


def attn_qat_bwd_workspace(b, nq, nkv, h, d) -> int:
    return int(_lib.load().attn_qat_bwd_workspace(b, nq, nkv, h, d))


NO_REGION = 2 ** 64 - 1  # SIZE_MAX: the workspace has no such region


def attn_qat_layout(b, nq, nkv, h, d, which: str = "fwd") -> dict:
    """Byte offsets of the regions of the forward ("fwd") or backward ("bwd")
    workspace (nvq_attn_layout); absent regions are left out."""
    import ctypes
    lay = _lib.AttnLayout()
    _lib.call(f"attn_qat_{which}_layout", b, nq, nkv, h, d, ctypes.addressof(lay))
    return {name: getattr(lay, name) for name, _ in lay._fields_
            if getattr(lay, name) != NO_REGION}


def _workspace(nbytes: int, device, ws: torch.Tensor | None) -> torch.Tensor:
    if ws is None or ws.numel() * ws.element_size() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    return ws


def _fwd_args(q, k, v, scale, o, stats, workspace):
    _check_bnhd(q, "q")
    b, nq, h, d = q.shape
    nkv = k.shape[1]
    _check_bnhd(k, "k", (b, nkv, h, d))
    _check_bnhd(v, "v", (b, nkv, h, d))
    scale = _scale(scale, d)
    if o is None:
        o = torch.empty_like(q)
    if stats is None:
        stats = torch.empty((b, h, 2, nq), dtype=torch.float32, device=q.device)
    ws = _workspace(attn_qat_fwd_workspace(b, nq, nkv, h, d), q.device, workspace)
    return (b, nq, nkv, h, d), scale, o, stats, ws


def attn_qat_fwd(q, k, v, scale=None, causal=False, o=None, stats=None, workspace=None):
    """Forward: returns (o bf16 [B, Nq, H, D], stats fp32 [B, H, 2, Nq] = (LSE, m))."""
    dims, scale, o, stats, ws = _fwd_args(q, k, v, scale, o, stats, workspace)
    _lib.call("attn_qat_fwd", _ptr(q), _ptr(k), _ptr(v), *dims, scale,
              int(bool(causal)), _ptr(o), _ptr(stats), _ptr(ws), ws.numel() * ws.element_size(),
              _stream_ptr(q))
    return o, stats


def attn_qat_fwd_hp(q, k, v, scale=None, causal=False, o=None, o_hp=None, stats=None,
                    workspace=None):
    """Forward with the auxiliary high-precision output: returns (o, o_hp, stats),
    o_hp = P V~ / l with P unquantized (bf16 [B, Nq, H, D]); o and stats as in
    attn_qat_fwd.  Passing o_hp as ``o`` to attn_qat_bwd takes delta from it."""
    dims, scale, o, stats, ws = _fwd_args(q, k, v, scale, o, stats, workspace)
    if o_hp is None:
        o_hp = torch.empty_like(q)
    _check_bnhd(o_hp, "o_hp", q.shape)
    _lib.call("attn_qat_fwd_hp", _ptr(q), _ptr(k), _ptr(v), *dims, scale,
              int(bool(causal)), _ptr(o), _ptr(o_hp), _ptr(stats), _ptr(ws),
              ws.numel() * ws.element_size(), _stream_ptr(q))
    return o, o_hp, stats


def attn_qat_bwd(q, k, v, o, stats, do, scale=None, causal=False, dq=None, dk=None, dv=None,
                 workspace=None):
    """Straight-through backward: returns (dq, dk, dv), bf16, shaped like q, k, v."""
    _check_bnhd(q, "q")
    b, nq, h, d = q.shape
    nkv = k.shape[1]
    _check_bnhd(k, "k", (b, nkv, h, d))
    _check_bnhd(v, "v", (b, nkv, h, d))
    _check_bnhd(o, "o", q.shape)
    _check_bnhd(do, "do", q.shape)
    _check(stats, "stats", torch.float32)
    scale = _scale(scale, d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = _workspace(attn_qat_bwd_workspace(b, nq, nkv, h, d), q.device, workspace)
    _lib.call("attn_qat_bwd", _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(stats), _ptr(do),
              _ptr(dq), _ptr(dk), _ptr(dv), b, nq, nkv, h, d, scale, int(bool(causal)),
              _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(q))
    return dq, dk, dv


def attn_qat_bwd_saved(saved, o, stats, do, scale=None, causal=False, nkv=None, dq=None,
                       dk=None, dv=None, workspace=None):
    """Straight-through backward from the quantized operands a forward left in its
    workspace ``saved`` (the ``workspace`` tensor passed to attn_qat_fwd or
    attn_qat_fwd_hp on the same q, k, v): returns (dq, dk, dv), equal to
    attn_qat_bwd's bit for bit.  ``nkv`` is the key count (default Nq)."""
    _check_bnhd(o, "o")
    b, nq, h, d = o.shape
    nkv = nq if nkv is None else int(nkv)
    _check_bnhd(do, "do", o.shape)
    _check(stats, "stats", torch.float32)
    _check(saved, "saved", torch.uint8)
    scale = _scale(scale, d)
    dq = torch.empty_like(o) if dq is None else dq
    dk = torch.empty((b, nkv, h, d), dtype=BF16, device=o.device) if dk is None else dk
    dv = torch.empty((b, nkv, h, d), dtype=BF16, device=o.device) if dv is None else dv
    need = int(_lib.load().attn_qat_bwd_saved_workspace(b, nq, nkv, h, d))
    ws = _workspace(need, o.device, workspace)
    _lib.call("attn_qat_bwd_saved", _ptr(saved), saved.numel(), _ptr(o), _ptr(stats), _ptr(do),
              _ptr(dq), _ptr(dk), _ptr(dv), b, nq, nkv, h, d, scale, int(bool(causal)), _ptr(ws),
              ws.numel() * ws.element_size(), _stream_ptr(o))
    return dq, dk, dv


# ------------------------------------------------------------------ NVFP4 linear
def nvfp4_tiled_scale_bytes(rows: int, cols: int) -> int:
    return int(_lib.load().nvfp4_tiled_scale_bytes(rows, cols))


def nvfp4_quantize_tiled(x: torch.Tensor, global_sf: torch.Tensor | None = None,
                         codes: torch.Tensor | None = None, scales: torch.Tensor | None = None):
    """Packed E2M1 codes (uint8 [rows, cols/2]) and E4M3 scales in the 128x4 tiled
    layout of block-scaled FP4 GEMMs (uint8, nvfp4_tiled_scale_bytes) of a bf16
    matrix x [rows, cols]."""
    _check(x, "x")
    rows, cols, ld = _rows_ld(x)
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(nvfp4_tiled_scale_bytes(rows, cols), dtype=torch.uint8,
                             device=x.device)
    _lib.call("nvfp4_quantize_tiled", _ptr(x), rows, cols, ld, _opt_ptr(global_sf),
              _ptr(codes), _ptr(scales), _stream_ptr(x))
    return codes, scales


def _opt_ptr(t):
    if t is None:
        return None
    _check(t, "global_sf", torch.float32)
    return _ptr(t)


def _linear_dims(x, w):
    _check(x, "x")
    _check(w, "w")
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"x [M, K] and w [N, K] expected, got {tuple(x.shape)}, {tuple(w.shape)}")
    if not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("x and w must be contiguous")
    return x.shape[0], w.shape[0], x.shape[1]


def nvfp4_linear_fwd(x, w, bias=None, x_global_sf=None, w_global_sf=None, out=None,
                     workspace=None):
    """out [M, N] bf16 = x~ w~^T (+ bias): both operands NVFP4-quantized under
    their global scales (None: 448*6/amax of the operand), FP4 block-scaled GEMM."""
    m, n, k = _linear_dims(x, w)
    if bias is not None:
        _check(bias, "bias")
    if out is None:
        out = torch.empty((m, n), dtype=BF16, device=x.device)
    ws = _workspace(int(_lib.load().nvfp4_linear_workspace(m, n, k)), x.device, workspace)
    _lib.call("nvfp4_linear_fwd", _ptr(x), _ptr(w), None if bias is None else _ptr(bias), m, n, k,
              _opt_ptr(x_global_sf), _opt_ptr(w_global_sf), _ptr(out), _ptr(ws),
              ws.numel() * ws.element_size(), _stream_ptr(x))
    return out


def nvfp4_linear_bwd(grad, x, w, need_bias=True, workspace=None):
    """Straight-through gradients (grad_x [M, K], grad_w [N, K], grad_b [N] or None), bf16."""
    m, n, k = _linear_dims(x, w)
    _check(grad, "grad")
    if tuple(grad.shape) != (m, n) or not grad.is_contiguous():
        raise ValueError("grad must be a contiguous [M, N] tensor")
    gx = torch.empty_like(x)
    gw = torch.empty_like(w)
    gb = torch.empty((n,), dtype=BF16, device=x.device) if need_bias else None
    ws = _workspace(int(_lib.load().nvfp4_linear_bwd_workspace(m, n, k)), x.device, workspace)
    _lib.call("nvfp4_linear_bwd", _ptr(grad), _ptr(x), _ptr(w), m, n, k, _ptr(gx), _ptr(gw),
              None if gb is None else _ptr(gb), _ptr(ws), ws.numel() * ws.element_size(),
              _stream_ptr(x))
    return gx, gw, gb


class NVFP4LinearFunction(torch.autograd.Function):
    """Forward: the NVFP4 linear (both operands quantized, FP4 GEMM); backward: the
    full-precision linear gradients (straight-through)."""

    @staticmethod
    def forward(ctx, x, w, bias, x_global_sf):
        shape = x.shape
        x2 = x.reshape(-1, shape[-1]).contiguous()
        out = nvfp4_linear_fwd(x2, w.contiguous(), bias, x_global_sf)
        ctx.save_for_backward(x2, w)
        ctx.has_bias, ctx.shape = bias is not None, shape
        return out.view(*shape[:-1], w.shape[0])

    @staticmethod
    def backward(ctx, grad):
        x2, w = ctx.saved_tensors
        g2 = grad.reshape(-1, grad.shape[-1]).contiguous()
        gx, gw, gb = nvfp4_linear_bwd(g2, x2, w.contiguous(), ctx.has_bias)
        return gx.view(ctx.shape), gw, gb, None


class NVFP4Linear(torch.nn.Module):
    """A bf16 linear layer whose forward runs as the NVFP4 GEMM (weight quantized
    under 448*6/amax(w) at every call, input under ``input_global_sf`` or its own
    amax) and whose backward is straight-through."""

    def __init__(self, in_features: int, out_features: int, bias: bool = True,
                 input_global_sf: torch.Tensor | None = None, device=None):
        super().__init__()
        self.weight = torch.nn.Parameter(torch.empty(out_features, in_features, dtype=BF16,
                                                     device=device))
        self.bias = torch.nn.Parameter(torch.zeros(out_features, dtype=BF16, device=device)) \
            if bias else None
        self.input_global_sf = input_global_sf
        torch.nn.init.normal_(self.weight, std=in_features ** -0.5)

    def forward(self, x):
        return NVFP4LinearFunction.apply(x, self.weight, self.bias, self.input_global_sf)


# Kernel kinds of nvq_timing_read (include/nvfp4attn.h, NVQ_KERNEL_*)
KERNEL_KINDS = {"quantize": 0, "attn_fwd": 1, "bwd_delta": 2, "bwd_dkdv": 3, "bwd_dq": 4,
                "global_sf": 5, "vsa": 6, "linear": 7}


def timing_enable(on: bool = True) -> None:
    """Start (discarding earlier records) or stop per-kernel event timing."""
    _lib.call("nvq_timing_enable", int(bool(on)))


def timing_read() -> dict:
    """{kind: (launches, total_ms)} for the launches recorded since timing_enable(True)."""
    import ctypes
    out = {}
    for name, kind in KERNEL_KINDS.items():
        n, ms = ctypes.c_int64(0), ctypes.c_double(0.0)
        _lib.call("nvq_timing_read", kind, ctypes.addressof(n), ctypes.addressof(ms))
        out[name] = (int(n.value), float(ms.value))
    return out


# ------------------------------------------------------- block-sparse (VSA)

VSA_TILE = 128  # tokens per tile: one 4x4x8 cube


def _check_tiles(kv_tiles, b, h, n):
    _check(kv_tiles, "kv_tiles", torch.int32)
    if kv_tiles.dim() != 4 or tuple(kv_tiles.shape[:3]) != (b, h, n // VSA_TILE) or \
            not kv_tiles.is_contiguous():
        raise ValueError(f"kv_tiles must be contiguous int32 [B, H, N/128, topk] = "
                         f"[{b}, {h}, {n // VSA_TILE}, topk], got {tuple(kv_tiles.shape)}")


def vsa_effective_topk(sparsity: float, num_blocks: int) -> int:
    """max(1, min(ceil((1 - sparsity) * num_blocks), num_blocks)) (the VSA metadata's formula)."""
    return max(1, min(math.ceil((1.0 - sparsity) * num_blocks), num_blocks))


def vsa_reorder(x, grid, cube=(4, 4, 8), to_cubes=True, out=None):
    """Token rows of bf16 [B, T*Hh*W, H, D] between raster and cube order."""
    _check(x, "x", torch.bfloat16)
    b, n, h, d = x.shape
    t, hh, w = grid
    if n != t * hh * w:
        raise ValueError(f"x has {n} tokens, the grid {t}x{hh}x{w}")
    out = torch.empty_like(x) if out is None else out
    _lib.call("vsa_reorder", _ptr(x), b, t, hh, w, h, d, cube[0], cube[1], cube[2],
              int(bool(to_cubes)), _ptr(out), _stream_ptr(x))
    return out


def vsa_select_tiles(q, k, topk, workspace=None):
    """int32 [B, H, N/128, topk]: per query tile the topk key tiles by cube-mean score."""
    _check_bnhd(q, "q")
    _check_bnhd(k, "k", q.shape)
    b, n, h, d = q.shape
    out = torch.empty((b, h, n // VSA_TILE, topk), dtype=torch.int32, device=q.device)
    need = vsa_select_workspace(b, n, h, d)
    ws = _workspace(need, q.device, workspace)
    _lib.call("vsa_select_tiles", _ptr(q), _ptr(k), b, n, h, d, int(topk), _ptr(out), _ptr(ws),
              ws.numel() * ws.element_size(), _stream_ptr(q))
    return out


def attn_qat_fwd_sparse(q, k, v, kv_tiles, scale=None, o=None, stats=None, workspace=None):
    """Block-sparse forward (tokens in cube order): (o, stats)."""
    _check_bnhd(q, "q")
    b, n, h, d = q.shape
    _check_bnhd(k, "k", q.shape)
    _check_bnhd(v, "v", q.shape)
    _check_tiles(kv_tiles, b, h, n)
    topk = kv_tiles.shape[-1]
    scale = _scale(scale, d)
    o = torch.empty_like(q) if o is None else o
    if stats is None:
        stats = torch.empty((b, h, 2, n), dtype=torch.float32, device=q.device)
    ws = _workspace(attn_qat_fwd_workspace(b, n, n, h, d), q.device, workspace)
    _lib.call("attn_qat_fwd_sparse", _ptr(q), _ptr(k), _ptr(v), b, n, h, d, scale, _ptr(kv_tiles),
              topk, _ptr(o), _ptr(stats), _ptr(ws), ws.numel() * ws.element_size(),
              _stream_ptr(q))
    return o, stats


def attn_qat_bwd_sparse_workspace(b, n, h, d, topk) -> int:
    return int(_lib.load().attn_qat_bwd_sparse_workspace(b, n, h, d, topk))


def vsa_select_workspace(b, n, h, d) -> int:
    return int(_lib.load().vsa_select_workspace(b, n, h, d))


def attn_qat_bwd_sparse(q, k, v, o, stats, do, kv_tiles, scale=None, dq=None, dk=None, dv=None,
                        workspace=None):
    """Block-sparse straight-through backward: (dq, dk, dv)."""
    _check_bnhd(q, "q")
    b, n, h, d = q.shape
    for t_, name in ((k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check_bnhd(t_, name, q.shape)
    _check(stats, "stats", torch.float32)
    _check_tiles(kv_tiles, b, h, n)
    topk = kv_tiles.shape[-1]
    scale = _scale(scale, d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = attn_qat_bwd_sparse_workspace(b, n, h, d, topk)
    ws = _workspace(need, q.device, workspace)
    _lib.call("attn_qat_bwd_sparse", _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(stats), _ptr(do),
              _ptr(kv_tiles), topk, _ptr(dq), _ptr(dk), _ptr(dv), b, n, h, d, scale, _ptr(ws),
              ws.numel() * ws.element_size(), _stream_ptr(q))
    return dq, dk, dv


def attn_qat_bwd_sparse_saved_workspace(b, n, h, d, topk) -> int:
    return int(_lib.load().attn_qat_bwd_sparse_saved_workspace(b, n, h, d, topk))


def attn_qat_bwd_sparse_saved(saved, o, stats, do, kv_tiles, scale=None, dq=None, dk=None,
                              dv=None, workspace=None):
    """Block-sparse backward from the quantized operands attn_qat_fwd_sparse left in
    its workspace ``saved`` (same q, k, v and kv_tiles): (dq, dk, dv), equal to
    attn_qat_bwd_sparse's bit for bit, without its quantizer pass."""
    _check_bnhd(o, "o")
    b, n, h, d = o.shape
    _check_bnhd(do, "do", o.shape)
    _check(stats, "stats", torch.float32)
    _check(saved, "saved", torch.uint8)
    _check_tiles(kv_tiles, b, h, n)
    topk = kv_tiles.shape[-1]
    scale = _scale(scale, d)
    dq = torch.empty_like(o) if dq is None else dq
    dk = torch.empty_like(o) if dk is None else dk
    dv = torch.empty_like(o) if dv is None else dv
    ws = _workspace(attn_qat_bwd_sparse_saved_workspace(b, n, h, d, topk), o.device, workspace)
    _lib.call("attn_qat_bwd_sparse_saved", _ptr(saved), saved.numel(), _ptr(o), _ptr(stats),
              _ptr(do), _ptr(kv_tiles), topk, _ptr(dq), _ptr(dk), _ptr(dv), b, n, h, d, scale,
              _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(o))
    return dq, dk, dv


def device_status(device=None) -> int:
    """Synchronize the current stream and return (and clear) the device error word."""
    s = torch.cuda.current_stream(device).cuda_stream
    return int(_lib.load().nvq_device_status(s))


DELTA_MODES = ("o", "hp")


class AttnQATFunction(torch.autograd.Function):
    """O = attention with NVFP4 fake-quantized Q, K, V, P; straight-through backward.
    ``delta_mode`` "o": the backward's delta = rowsum(dO * O); "hp": from the
    auxiliary high-precision output P V~ / l, which the forward then also computes."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal, delta_mode="o"):
        b, nq, h, d = q.shape
        # the forward's workspace keeps Q~, K~, V~ in every form the backward
        # reads: it is saved instead of q, k, v, and the backward quantizes nothing
        saved = torch.empty(attn_qat_fwd_workspace(b, nq, k.shape[1], h, d), dtype=torch.uint8,
                            device=q.device)
        if delta_mode == "hp":
            o, o_d, stats = attn_qat_fwd_hp(q, k, v, scale, causal, workspace=saved)
        elif delta_mode == "o":
            o, stats = attn_qat_fwd(q, k, v, scale, causal, workspace=saved)
            o_d = o
        else:
            raise ValueError(f"delta_mode must be one of {DELTA_MODES}, got {delta_mode!r}")
        ctx.save_for_backward(saved, o_d, stats)
        ctx.scale, ctx.causal, ctx.nkv = scale, causal, k.shape[1]
        return o

    @staticmethod
    def backward(ctx, do):
        saved, o_d, stats = ctx.saved_tensors
        dq, dk, dv = attn_qat_bwd_saved(saved, o_d, stats, do.contiguous(), ctx.scale,
                                        ctx.causal, nkv=ctx.nkv)
        return dq, dk, dv, None, None, None


class AttnQAT(torch.nn.Module):
    """``AttentionImpl(num_heads, head_size, softmax_scale, causal)`` with ``forward(q, k, v)``.

    ``delta_mode`` chooses where the backward's delta comes from.  The default
    "o" takes it from the returned output O (the exact straight-through
    derivative of the forward, the reading the parity tests use).  This differs
    from the pages: ``attn_qat_train()`` ("attn_qat_train" API page) hard-codes
    ``use_high_prec_o = True``, i.e. delta from the auxiliary high-precision
    output P V~ / l, which ``delta_mode="hp"`` selects.
    """

    def __init__(self, num_heads: int, head_size: int, softmax_scale: float | None = None,
                 causal: bool = False, dropout_p: float = 0.0, delta_mode: str = "o"):
        super().__init__()
        if delta_mode not in DELTA_MODES:
            raise ValueError(f"delta_mode must be one of {DELTA_MODES}, got {delta_mode!r}")
        if dropout_p > 0:
            raise NotImplementedError(
                f"NVFP4 Attn-QAT attention applies no dropout (got dropout_p={dropout_p})")
        if head_size not in (64, 128):
            raise ValueError(f"head_size must be 64 or 128, got {head_size}")
        self.num_heads, self.head_size = num_heads, head_size
        self.softmax_scale = default_scale(head_size) if softmax_scale is None else softmax_scale
        self.causal = causal
        self.delta_mode = delta_mode

    def forward(self, q, k, v):
        return AttnQATFunction.apply(q, k, v, self.softmax_scale, self.causal, self.delta_mode)
