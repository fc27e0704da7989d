"""Video sparse attention (VSA) block selection and token order (TEST INFRASTRUCTURE ONLY).

Source: "vsqa-preview-1.3b metadata.json", ``attention``: ``kind`` vsa,
``cube_shape`` [4, 4, 8] (frames x height x width of the latent grid),
``precision.coarse`` BF16 and ``precision.fine`` NVFP4 fake-quant,
``selection.sparsity`` 0.9 with ``selection.effective_topk`` =
max(1, min(ceil((1 - sparsity) * num_blocks), num_blocks)).

What this module computes (the block-sparse fine-attention workload):
  * cube order: the T x Hh x W latent tokens (raster order t, h, w) regrouped
    into cubes of ct x ch x cw tokens; cubes in raster order over the cube
    grid, tokens inside a cube in raster order.  One cube of 4x4x8 = 128 tokens
    is one attention tile (``attention.TILE``).
  * selection: per (batch, head), the mean of Q and of K over each cube (of the
    bf16 values), the cube-level scores mean_q . mean_k for every pair of cubes,
    and for each query cube the ``topk`` key cubes of highest score, ties to the
    lower cube index.  The lists are returned in ascending cube order.
The fine attention itself is ``attention.attn_fwd`` / ``attn_bwd`` with
``kv_tiles`` set to these lists.  The metadata names the selection mode "top-p"
next to a top-k formula; the formula is what is implemented (top-k).
"""
from __future__ import annotations

import math

import torch

F64 = torch.float64


def effective_topk(sparsity: float, num_blocks: int) -> int:
    """max(1, min(ceil((1 - sparsity) * num_blocks), num_blocks))."""
    return max(1, min(math.ceil((1.0 - sparsity) * num_blocks), num_blocks))


def cube_order(t: int, hh: int, w: int, cube=(4, 4, 8)) -> torch.Tensor:
    """perm[i] = raster token index (t, h, w) of the token at cube-order position i."""
    ct, ch, cw = cube
    if t % ct or hh % ch or w % cw:
        raise ValueError("the latent grid must be a whole number of cubes")
    tt, hi, wi = torch.meshgrid(torch.arange(t), torch.arange(hh), torch.arange(w), indexing="ij")
    token = (tt * hh + hi) * w + wi                       # raster index of each grid point
    # cube-order key of each grid point: cube raster index, then position inside the cube
    cube_id = ((tt // ct) * (hh // ch) + hi // ch) * (w // cw) + wi // cw
    inner = ((tt % ct) * ch + hi % ch) * cw + wi % cw
    key = cube_id * (ct * ch * cw) + inner
    perm = torch.empty(t * hh * w, dtype=torch.long)
    perm[key.reshape(-1)] = token.reshape(-1)
    return perm


def to_cubes(x: torch.Tensor, t: int, hh: int, w: int, cube=(4, 4, 8)) -> torch.Tensor:
    """[B, N, H, D] raster token order -> cube order."""
    return x[:, cube_order(t, hh, w, cube)]


def from_cubes(x: torch.Tensor, t: int, hh: int, w: int, cube=(4, 4, 8)) -> torch.Tensor:
    """[B, N, H, D] cube order -> raster token order."""
    out = torch.empty_like(x)
    out[:, cube_order(t, hh, w, cube)] = x
    return out


def cube_scores(q: torch.Tensor, k: torch.Tensor, tile: int = 128) -> torch.Tensor:
    """[B, H, n, n] float64 scores mean_q(i) . mean_k(j) over tiles of ``tile`` tokens
    (q, k in cube order, [B, N, H, D])."""
    b, n_tok, h, d = q.shape
    n = n_tok // tile
    qm = q.to(F64).reshape(b, n, tile, h, d).mean(dim=2)  # [B, n, H, D]
    km = k.to(F64).reshape(b, n, tile, h, d).mean(dim=2)
    return torch.einsum("bihd,bjhd->bhij", qm, km)


def select_tiles(q: torch.Tensor, k: torch.Tensor, topk: int, tile: int = 128) -> torch.Tensor:
    """[B, H, n, topk] int64: for each query tile the ``topk`` key tiles of highest
    cube score (ties to the lower index), in ascending tile order."""
    s = cube_scores(q, k, tile)
    b, h, n, _ = s.shape
    out = torch.empty(b, h, n, topk, dtype=torch.long)
    for bi in range(b):
        for hi in range(h):
            for i in range(n):
                # sort by score descending, then index ascending: lexicographic key
                order = sorted(range(n), key=lambda j: (-float(s[bi, hi, i, j]), j))
                out[bi, hi, i] = torch.tensor(sorted(order[:topk]))
    return out
