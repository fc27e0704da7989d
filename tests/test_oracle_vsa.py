"""Pins of the block-sparse (VSA) parts of the oracle: cube order, the top-k
formula, the cube-score selection and block-sparse attention, each checked
against brute force or reduced to the dense attention oracle."""
import math

import torch

from oracle import attention as oa
from oracle import vsa


def test_cube_order_brute_force_small_grid():
    t, hh, w = 8, 8, 16
    expected = []
    for c0 in range(t // 4):
        for c1 in range(hh // 4):
            for c2 in range(w // 8):
                for a in range(4):
                    for bb in range(4):
                        for c in range(8):
                            expected.append(((c0 * 4 + a) * hh + (c1 * 4 + bb)) * w + c2 * 8 + c)
    assert vsa.cube_order(t, hh, w).tolist() == expected


def test_cube_order_wan_grid_and_round_trip():
    perm = vsa.cube_order(16, 28, 56)  # the 16x28x56 latent of 448x896x61 frames
    assert perm.numel() == 25088 == 196 * 128
    assert torch.equal(torch.sort(perm).values, torch.arange(25088))
    x = torch.randn(1, 8 * 8 * 16, 2, 3, generator=torch.Generator().manual_seed(5))
    assert torch.equal(vsa.from_cubes(vsa.to_cubes(x, 8, 8, 16), 8, 8, 16), x)


def test_effective_topk_formula():
    assert vsa.effective_topk(0.9, 196) == 20   # ceil(19.6)
    assert vsa.effective_topk(0.95, 196) == 10  # ceil(9.8)
    assert vsa.effective_topk(0.0, 7) == 7
    assert vsa.effective_topk(1.0, 7) == 1


def _brute_scores(q, k, tile):
    b, n_tok, h, d = q.shape
    n = n_tok // tile
    out = torch.zeros(b, h, n, n, dtype=torch.float64)
    for bi in range(b):
        for hi in range(h):
            qm = [[sum(float(q[bi, i * tile + r, hi, dd]) for r in range(tile)) / tile
                   for dd in range(d)] for i in range(n)]
            km = [[sum(float(k[bi, j * tile + r, hi, dd]) for r in range(tile)) / tile
                   for dd in range(d)] for j in range(n)]
            for i in range(n):
                for j in range(n):
                    out[bi, hi, i, j] = sum(a * c for a, c in zip(qm[i], km[j]))
    return out


def test_select_tiles_matches_brute_force_sort():
    g = torch.Generator().manual_seed(6)
    q = torch.randn(1, 6 * 8, 2, 4, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 6 * 8, 2, 4, generator=g).to(torch.bfloat16)
    got = vsa.select_tiles(q, k, topk=3, tile=8)
    s = _brute_scores(q, k, 8)
    assert torch.allclose(vsa.cube_scores(q, k, 8), s, rtol=1e-12, atol=1e-12)
    for hi in range(2):
        for i in range(6):
            rank = sorted(range(6), key=lambda j: (-float(s[0, hi, i, j]), j))
            assert got[0, hi, i].tolist() == sorted(rank[:3])


def test_select_tiles_ties_go_to_the_lower_index():
    q = torch.ones(1, 4 * 8, 1, 2)
    k = torch.ones(1, 4 * 8, 1, 2)  # every pair of tiles scores the same
    got = vsa.select_tiles(q, k, topk=2, tile=8)
    assert got[0, 0].tolist() == [[0, 1]] * 4
    k[0, 24:32] = 2.0  # tile 3 now scores highest for every query tile
    got = vsa.select_tiles(q, k, topk=2, tile=8)
    assert got[0, 0].tolist() == [[0, 3]] * 4


def _inputs(n_tiles, h, d, seed):
    g = torch.Generator().manual_seed(seed)
    n = n_tiles * oa.TILE
    return [torch.randn(1, n, h, d, generator=g).to(torch.bfloat16) for _ in range(4)]


def test_all_tiles_selected_is_dense_attention():
    q, k, v, do = _inputs(3, 1, 16, 7)
    tiles = torch.arange(3).repeat(1, 1, 3, 1)  # [1, 1, 3, 3]
    o_s, lse_s, m_s = oa.attn_fwd(q, k, v, 0.25, kv_tiles=tiles)
    o_d, lse_d, m_d = oa.attn_fwd(q, k, v, 0.25)
    assert torch.equal(o_s, o_d) and torch.equal(lse_s, lse_d) and torch.equal(m_s, m_d)
    g_s = oa.attn_bwd(q, k, v, o_d, do, 0.25, kv_tiles=tiles)
    g_d = oa.attn_bwd(q, k, v, o_d, do, 0.25)
    assert all(torch.equal(a, b) for a, b in zip(g_s, g_d))


def test_unquantized_block_sparse_softmax_by_explicit_loops():
    q, k, v, _ = _inputs(3, 1, 8, 8)
    tiles = torch.tensor([[[[0, 2], [1, 2], [0, 1]]]])
    o, lse, _ = oa.attn_fwd(q, k, v, 0.3, quant=False, kv_tiles=tiles)
    qd, kd, vd = (x.double()[0, :, 0] for x in (q, k, v))
    for r in range(0, 3 * oa.TILE, 37):
        keys = [c for t in tiles[0, 0, r // oa.TILE].tolist()
                for c in range(t * oa.TILE, (t + 1) * oa.TILE)]
        s = [0.3 * float(qd[r] @ kd[c]) for c in keys]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        den = sum(e)
        ref = sum(ei * vd[c] for ei, c in zip(e, keys)) / den
        assert torch.allclose(o[0, r, 0], ref, rtol=1e-12, atol=1e-12)
        assert abs(float(lse[0, 0, r]) - (mx + math.log(den))) < 1e-12


def test_quantized_block_sparse_equals_dense_attention_on_the_selected_keys():
    """Per query tile, the block-sparse result is dense Attn-QAT over the keys of
    its selected tiles (P~ blocks are tile-aligned), and the backward's dK, dV
    are the sums of those dense problems' dK, dV scattered back."""
    q, k, v, do = _inputs(4, 1, 16, 9)
    tiles = torch.tensor([[[[0, 3], [1, 2], [2, 3], [0, 1]]]])
    o, lse, m = oa.attn_fwd(q, k, v, 0.25, kv_tiles=tiles)
    dq, dk, dv = oa.attn_bwd(q, k, v, o, do, 0.25, kv_tiles=tiles)
    t = oa.TILE
    dk_ref = torch.zeros_like(dk)
    dv_ref = torch.zeros_like(dv)
    for i in range(4):
        rows = slice(i * t, (i + 1) * t)
        keys = torch.cat([torch.arange(j * t, (j + 1) * t) for j in tiles[0, 0, i].tolist()])
        o_i, lse_i, m_i = oa.attn_fwd(q[:, rows], k[:, keys], v[:, keys], 0.25)
        assert torch.allclose(o[:, rows], o_i, rtol=1e-12, atol=1e-13)
        assert torch.allclose(lse[:, :, rows], lse_i, rtol=0, atol=1e-12)
        assert torch.equal(m[:, :, rows], m_i)
        dq_i, dk_i, dv_i = oa.attn_bwd(q[:, rows], k[:, keys], v[:, keys], o[:, rows],
                                       do[:, rows], 0.25)
        assert torch.allclose(dq[:, rows], dq_i, rtol=1e-10, atol=1e-12)
        dk_ref[:, keys] += dk_i
        dv_ref[:, keys] += dv_i
    assert torch.allclose(dk, dk_ref, rtol=1e-10, atol=1e-12)
    assert torch.allclose(dv, dv_ref, rtol=1e-10, atol=1e-12)
