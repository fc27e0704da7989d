"""Attention forward / straight-through backward oracle in float64 (TEST INFRASTRUCTURE ONLY).

Layout: q [B, Nq, H, D], k and v [B, Nkv, H, D] (the "BLHD" tensors that
``attn_qat_train()`` receives on the "attn_qat_train" API page), values given as
bf16 numbers (any float dtype; converted to float64 here).

Forward (the ``attn_qat_train()`` flag set on that page: ``is_qat`` on Q, K, V
and P, unit global scales for both, no Q/K smoothing, no two-level P; sm_scale
defaults to 1/sqrt(D)), per (b, h):
    Q~, K~, V~ = fq16 along D (unit gsf)
    S          = scale * Q~ K~^T                 (-inf where causal and j > i)
    m          = rowmax S
    P          = exp(S - m)
    l          = sum_j P                          (unquantized row sum)
    P~         = fq16 of P along keys, blocks [16t, 16t+16) counted from key 0
    O          = P~ V~ / l
    LSE        = m + ln l
P~ is referenced to the final row max m (the exact statistics that the
"Attn-QAT Training" guide, section "Architecture-specific Triton routing",
describes as the reference order).

Backward: the exact derivative of the forward with every fq replaced by the
identity (straight-through; the backward flags ``use_qat_qkv_backward`` and
``fake_quant_p_bwd`` of ``attn_qat_train()`` say it runs on the quantized
operands), m held constant:
    A   = P / l                 (= exp(S - LSE))
    dV  = (P~ / l)^T dO
    dP  = dO V~^T
    d   = rowsum(dO * O)        O = the forward output handed to the backward
    dS  = A * (dP - d)
    dQ  = scale * dS K~
    dK  = scale * dS^T Q~
``delta_mode="hp"`` takes d from the unquantized-P output P V~ / l instead (the
"auxiliary output" reading of the metadata's backward description).

Block-sparse variant (``kv_tiles``): the fine attention of the video sparse
attention recipe in "vsqa-preview-1.3b metadata.json" (``attention.kind`` vsa,
``cube_shape`` [4, 4, 8], ``precision.fine`` NVFP4 fake-quant): tokens are in
cube order, a tile is one cube of TILE = 128 tokens, and query tile i attends
only to the key tiles listed in ``kv_tiles[b, h, i]``.  Every other score is
-inf, so P = 0 there; tile boundaries are multiples of 16, so each P~ block lies
wholly inside or wholly outside the selection and the definition above applies
unchanged.

Query rows are processed in blocks only to bound memory; nothing else is
reordered.
"""
from __future__ import annotations

import math

import torch

from .nvfp4 import fake_quant, fq

F64 = torch.float64
TILE = 128  # tokens per tile of the block-sparse variant (one 4x4x8 cube)


def _t(x) -> torch.Tensor:
    return x.to(F64) if isinstance(x, torch.Tensor) else torch.as_tensor(x, dtype=F64)


def quantize_rows(x: torch.Tensor, quant: bool) -> torch.Tensor:
    """Q~/K~/V~: fq16 along D with unit gsf (decisions in fp32 on bf16 inputs)."""
    return fq(x, 1.0, torch.float32, axis=-1) if quant else x


def _head(x, b, h):
    return _t(x)[b, :, h, :]


def _allowed(tiles, rows, keys):
    """[R, C] bool: key ``keys[c]`` lies in a tile listed for the tile of ``rows[r]``."""
    rows, keys = torch.as_tensor(rows), torch.as_tensor(keys)
    ok = torch.zeros(int(tiles.shape[0]), int(keys.max()) // TILE + 1, dtype=torch.bool)
    for i in range(tiles.shape[0]):
        for t in tiles[i].tolist():
            if t < ok.shape[1]:
                ok[i, t] = True
    return ok[rows // TILE][:, keys // TILE]


def _scores(qt_rows, kt, scale, rows, causal, tiles=None, keys=None):
    s = scale * (qt_rows @ kt.T)
    keys = torch.arange(kt.shape[0]) if keys is None else torch.as_tensor(keys)
    if causal:
        s = s.masked_fill(keys[None, :] > torch.as_tensor(rows)[:, None], float("-inf"))
    if tiles is not None:
        s = s.masked_fill(~_allowed(tiles, rows, keys), float("-inf"))
    return s


def _probs(s, quant):
    m = s.amax(dim=1)
    p = torch.exp(s - m[:, None])
    l = p.sum(dim=1)
    pt = fq(p, 1.0, torch.float64, axis=1) if quant else p
    return m, p, l, pt


class HeadProblem:
    """One (b, h) head with its quantized operands, for sampled evaluation."""

    def __init__(self, q, k, v, b, h, scale, causal=False, quant=True, kv_tiles=None):
        self.qt = quantize_rows(_head(q, b, h), quant)
        self.kt = quantize_rows(_head(k, b, h), quant)
        self.vt = quantize_rows(_head(v, b, h), quant)
        self.scale, self.causal, self.quant = float(scale), bool(causal), bool(quant)
        # this head's [n_query_tiles, topk] selected key tiles, or None (dense)
        self.tiles = None if kv_tiles is None else torch.as_tensor(kv_tiles)[b, h].long()

    def fwd_rows(self, rows):
        """(o [R, D], lse [R], m [R]) for query rows ``rows``."""
        rows = torch.as_tensor(rows, dtype=torch.long)
        s = _scores(self.qt[rows], self.kt, self.scale, rows, self.causal, self.tiles)
        m, _, l, pt = _probs(s, self.quant)
        o = (pt @ self.vt) / l[:, None]
        return o, m + torch.log(l), m

    def probs_rows(self, rows):
        """(m, l, P, P~, scale bytes) of query rows ``rows``: the forward's row
        maxima, unquantized row sums, probabilities P = exp(S - m), their
        fake-quantized P~, and the E4M3 bytes of P~'s block scales, uint8
        [R, ceil(Nkv / 16)] (None without quantization)."""
        rows = torch.as_tensor(rows, dtype=torch.long)
        s = _scores(self.qt[rows], self.kt, self.scale, rows, self.causal, self.tiles)
        m, p, l, pt = _probs(s, self.quant)
        sb = fake_quant(p, 1.0, torch.float64, axis=1)[1] if self.quant else None
        return m, l, p, pt, sb

    def o_hp_rows(self, rows):
        """The auxiliary high-precision output P V~ / l (P unquantized) for ``rows``."""
        rows = torch.as_tensor(rows, dtype=torch.long)
        s = _scores(self.qt[rows], self.kt, self.scale, rows, self.causal, self.tiles)
        _, p, l, _ = _probs(s, self.quant)
        return (p @ self.vt) / l[:, None]

    def row_stats(self, block=512):
        """(m, l) for every query row."""
        n = self.qt.shape[0]
        ms, ls = [], []
        for r0 in range(0, n, block):
            rows = torch.arange(r0, min(n, r0 + block))
            s = _scores(self.qt[rows], self.kt, self.scale, rows, self.causal, self.tiles)
            m = s.amax(dim=1)
            ms.append(m)
            ls.append(torch.exp(s - m[:, None]).sum(dim=1))
        return torch.cat(ms), torch.cat(ls)

    def dq_rows(self, rows, o_rows, do_rows, delta_mode="o"):
        """dQ for query rows ``rows``; o_rows/do_rows are those rows of O and dO."""
        rows = torch.as_tensor(rows, dtype=torch.long)
        s = _scores(self.qt[rows], self.kt, self.scale, rows, self.causal, self.tiles)
        m, p, l, pt = _probs(s, self.quant)
        a = p / l[:, None]
        do_rows = _t(do_rows)
        o_d = _t(o_rows) if delta_mode == "o" else (p @ self.vt) / l[:, None]
        delta = (do_rows * o_d).sum(dim=1)
        dp = do_rows @ self.vt.T
        ds = a * (dp - delta[:, None])
        return self.scale * (ds @ self.kt)

    def dkdv_cols(self, cols, o, do, delta_mode="o", block=512):
        """(dK [C, D], dV [C, D]) for key columns ``cols``.

        ``o`` and ``do`` are this head's full [Nq, D] O and dO.  Each column's
        P~ needs its whole 16-key block, so the blocks containing ``cols`` are
        evaluated and the requested columns picked out.
        """
        cols = torch.as_tensor(cols, dtype=torch.long)
        nkv = self.kt.shape[0]
        blocks = torch.unique(cols // 16)
        keys = torch.cat([torch.arange(int(b) * 16, min(nkv, int(b) * 16 + 16)) for b in blocks])
        pos = {int(kk): i for i, kk in enumerate(keys)}
        sel = torch.tensor([pos[int(c)] for c in cols])
        o, do = _t(o), _t(do)
        d = self.kt.shape[1]
        dk = torch.zeros(len(keys), d, dtype=F64)
        dv = torch.zeros(len(keys), d, dtype=F64)
        m_all, l_all = self.row_stats(block)
        n = self.qt.shape[0]
        for r0 in range(0, n, block):
            rows = torch.arange(r0, min(n, r0 + block))
            s = _scores(self.qt[rows], self.kt[keys], self.scale, rows, self.causal, self.tiles,
                        keys)
            m, l = m_all[rows], l_all[rows]
            p = torch.exp(s - m[:, None])
            # keys holds whole 16-key blocks in order, so fq along it is blockwise
            pt = fq(p, 1.0, torch.float64, axis=1) if self.quant else p
            a = p / l[:, None]
            if delta_mode == "o":
                delta = (do[rows] * o[rows]).sum(dim=1)
            else:
                sf = _scores(self.qt[rows], self.kt, self.scale, rows, self.causal, self.tiles)
                pf = torch.exp(sf - m[:, None])
                delta = (do[rows] * ((pf @ self.vt) / l[:, None])).sum(dim=1)
            dv += (pt / l[:, None]).T @ do[rows]
            dp = do[rows] @ self.vt[keys].T
            ds = a * (dp - delta[:, None])
            dk += self.scale * (ds.T @ self.qt[rows])
        return dk[sel], dv[sel]


def attn_fwd(q, k, v, scale=None, causal=False, quant=True, block=512, kv_tiles=None):
    """Whole-tensor forward: (o [B,Nq,H,D], lse [B,H,Nq], m [B,H,Nq]) in float64.
    ``kv_tiles``: [B, H, Nq/TILE, topk] selected key tiles (block-sparse), or None."""
    q, k, v = _t(q), _t(k), _t(v)
    bsz, nq, nh, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.zeros(bsz, nq, nh, d, dtype=F64)
    lse = torch.zeros(bsz, nh, nq, dtype=F64)
    mm = torch.zeros(bsz, nh, nq, dtype=F64)
    for b in range(bsz):
        for h in range(nh):
            hp = HeadProblem(q, k, v, b, h, scale, causal, quant, kv_tiles)
            for r0 in range(0, nq, block):
                rows = torch.arange(r0, min(nq, r0 + block))
                ob, lb, mb = hp.fwd_rows(rows)
                o[b, rows, h] = ob
                lse[b, h, rows] = lb
                mm[b, h, rows] = mb
    return o, lse, mm


def attn_fwd_hp(q, k, v, scale=None, causal=False, quant=True, block=512):
    """Whole-tensor auxiliary high-precision output P V~ / l [B, Nq, H, D] (float64):
    the forward's output with P left unquantized (Q~, K~, V~ and l as in attn_fwd)."""
    q, k, v = _t(q), _t(k), _t(v)
    bsz, nq, nh, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o_hp = torch.zeros(bsz, nq, nh, d, dtype=F64)
    for b in range(bsz):
        for h in range(nh):
            hp = HeadProblem(q, k, v, b, h, scale, causal, quant)
            for r0 in range(0, nq, block):
                rows = torch.arange(r0, min(nq, r0 + block))
                o_hp[b, rows, h] = hp.o_hp_rows(rows)
    return o_hp


def attn_bwd(q, k, v, o, do, scale=None, causal=False, quant=True, delta_mode="o", block=512,
             kv_tiles=None):
    """Whole-tensor straight-through backward: (dq, dk, dv) in float64.
    ``kv_tiles`` as in attn_fwd."""
    q, k, v, o, do = _t(q), _t(k), _t(v), _t(o), _t(do)
    bsz, nq, nh, d = q.shape
    nkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for b in range(bsz):
        for h in range(nh):
            hp = HeadProblem(q, k, v, b, h, scale, causal, quant, kv_tiles)
            for r0 in range(0, nq, block):
                rows = torch.arange(r0, min(nq, r0 + block))
                s = _scores(hp.qt[rows], hp.kt, hp.scale, rows, hp.causal, hp.tiles)
                m, p, l, pt = _probs(s, hp.quant)
                a = p / l[:, None]
                do_r = do[b, rows, h]
                o_d = o[b, rows, h] if delta_mode == "o" else (p @ hp.vt) / l[:, None]
                delta = (do_r * o_d).sum(dim=1)
                dv[b, :, h] += (pt / l[:, None]).T @ do_r
                dp = do_r @ hp.vt.T
                ds = a * (dp - delta[:, None])
                dq[b, rows, h] = hp.scale * (ds @ hp.kt)
                dk[b, :, h] += hp.scale * (ds.T @ hp.qt[rows])
    assert dk.shape[1] == nkv
    return dq, dk, dv
