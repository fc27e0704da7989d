"""NVFP4 linear oracle (TEST INFRASTRUCTURE ONLY; see ``oracle/__init__``).

Source: "nvfp4_qad.py", ``nvfp4_gemm`` and ``_NVFP4STE``.

What it computes:
  forward   both operands NVFP4-quantized in blocks of 16 along K under their
            own global scales (the weight's is ``weight_global_sf`` =
            448*6/amax(w); the input's is given, or taken the same way from x
            here when none is given), then an FP4 GEMM with
            alpha = (1/gsf_w)/gsf_x, plus bias:
                out = alpha * sum_k (code_x s_x)(code_w s_w) + bias
                    = fq(x; gsf_x) fq(w; gsf_w)^T + bias
            (the products of codes and E4M3 scales are exact, and dividing
            every dequantized value by its global scale is the same as one
            alpha).  Evaluated in float64 from the pinned quantizer ``fq``.
  backward  straight-through: the full-precision linear gradients
                grad_x = grad w,  grad_w = grad^T x,  grad_b = sum over rows of grad
  scales    the E4M3 scale bytes [rows, cols/16] placed in the 128 x 4 tiled
            layout that block-scaled FP4 GEMMs read (the pages' "layout_128x4"):
            rows padded to 128 and blocks to 4; 512-byte tiles of 128 rows x 4
            blocks, ordered by row tile then block tile; inside a tile row r is
            at (r % 32) * 16 + (r // 32) * 4 and block c at c % 4.  Padding is 0.
"""
from __future__ import annotations

import torch

from .nvfp4 import fake_quant, fq, global_sf

F64 = torch.float64


def tiled_scale_offsets(rows: int, nblocks: int) -> torch.Tensor:
    """[rows, nblocks] int64 byte offsets of each scale in the tiled layout."""
    r = torch.arange(rows, dtype=torch.long)[:, None]
    c = torch.arange(nblocks, dtype=torch.long)[None, :]
    n_bt = -(-nblocks // 4)
    tile = (r // 128) * n_bt + c // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4


def tiled_scale_bytes(rows: int, cols: int) -> int:
    nb = cols // 16
    return (-(-rows // 128) * 128) * (-(-nb // 4) * 4)


def tile_scales(sbytes: torch.Tensor) -> torch.Tensor:
    """uint8 [rows, nblocks] -> the flat tiled layout (padding zero)."""
    rows, nb = sbytes.shape
    out = torch.zeros(tiled_scale_bytes(rows, nb * 16), dtype=torch.uint8)
    out[tiled_scale_offsets(rows, nb).reshape(-1)] = sbytes.reshape(-1).to(torch.uint8)
    return out


def untile_scales(buf: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """The flat tiled layout -> uint8 [rows, cols/16]."""
    nb = cols // 16
    return buf.reshape(-1)[tiled_scale_offsets(rows, nb).reshape(-1)].reshape(rows, nb)


def quantize_tiled(x, gsf=None):
    """(packed codes uint8 [rows, cols/2] with the even element in the low nibble,
    tiled scale bytes) of a bf16 matrix; gsf None = unit global scale."""
    _, sb, codes = fake_quant(x, 1.0 if gsf is None else gsf, torch.float32, axis=-1)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed, tile_scales(sb)


def linear_fwd(x, w, bias=None, gsf_x=None, gsf_w=None):
    """out [M, N] float64 = fq(x; gsf_x) fq(w; gsf_w)^T + bias.  A None global
    scale is taken from the operand (448*6/amax, fp32)."""
    gx = global_sf(x) if gsf_x is None else float(gsf_x)
    gw = global_sf(w) if gsf_w is None else float(gsf_w)
    out = fq(x, gx, torch.float32) @ fq(w, gw, torch.float32).T
    if bias is not None:
        out = out + bias.to(F64)[None, :]
    return out


def linear_bwd(grad, x, w):
    """(grad_x [M, K], grad_w [N, K], grad_b [N]) in float64."""
    g, xx, ww = grad.to(F64), x.to(F64), w.to(F64)
    return g @ ww, g.T @ xx, g.sum(dim=0)
