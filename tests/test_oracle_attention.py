"""Pins of the attention oracle against things other than itself.

- quantizers off: PyTorch's scaled_dot_product_attention and autograd (library)
- quantizers on: autograd of a straight-through forward built from the pinned
  quantizer (the backward formula is derived by autograd, not retyped)
- central finite differences (quantizers off)
- a pure-Python brute force with the exact rational block quantizer (P~
  referenced to the final row max, blocks of 16 keys counted from key 0)
- closed form for constant V rows; sampled evaluation == whole-tensor evaluation
"""
import math
from fractions import Fraction

import pytest
import torch

from oracle import attention as at
from oracle import nvfp4 as nv

F64 = torch.float64


def _inputs(b, nq, nkv, h, d, seed, spread=1.0):
    g = torch.Generator().manual_seed(seed)
    mk = lambda n: nv.to_bf16(torch.randn(b, n, h, d, generator=g, dtype=F64) * spread)
    return mk(nq), mk(nkv), mk(nkv), mk(nq)


def _sdpa(q, k, v, scale, causal):
    # [B, N, H, D] -> [B, H, N, D]
    o = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), is_causal=causal, scale=scale)
    return o.transpose(1, 2)


@pytest.mark.parametrize("nq,nkv,causal", [(37, 53, False), (29, 29, True), (1, 17, False)])
def test_fq_off_forward_matches_sdpa(nq, nkv, causal):
    q, k, v, _ = _inputs(2, nq, nkv, 3, 16, seed=1)
    scale = 0.3
    o, lse, m = at.attn_fwd(q, k, v, scale, causal, quant=False)
    ref = _sdpa(q, k, v, scale, causal)
    assert torch.allclose(o, ref, rtol=0, atol=1e-12)
    s = scale * torch.einsum("bqhd,bkhd->bhqk", q, k)
    if causal:
        s = s.masked_fill(torch.ones(nq, nkv, dtype=torch.bool).triu(1), float("-inf"))
    assert torch.allclose(lse, torch.logsumexp(s, dim=-1), rtol=0, atol=1e-12)
    assert torch.equal(m, s.amax(dim=-1))


@pytest.mark.parametrize("causal", [False, True])
def test_fq_off_backward_matches_autograd(causal):
    q, k, v, do = _inputs(1, 24, 24, 2, 16, seed=2)
    scale = 0.25
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    ref = _sdpa(qq, kk, vv, scale, causal)
    ref.backward(do)
    o, _, _ = at.attn_fwd(q, k, v, scale, causal, quant=False)
    dq, dk, dv = at.attn_bwd(q, k, v, o, do, scale, causal, quant=False)
    for a, b in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
        assert torch.allclose(a, b, rtol=0, atol=1e-11)


def _ste(x, xq):
    return x + (xq - x).detach()


@pytest.mark.parametrize("nq,nkv,causal", [(20, 40, False), (33, 33, True)])
def test_ste_backward_matches_autograd(nq, nkv, causal):
    """Quantizers on: the oracle backward equals autograd of the forward with every
    fq replaced by a straight-through estimator and the row max held constant."""
    q, k, v, do = _inputs(1, nq, nkv, 2, 32, seed=3)
    scale = 1 / math.sqrt(32)
    o, _, _ = at.attn_fwd(q, k, v, scale, causal, quant=True)
    dq, dk, dv = at.attn_bwd(q, k, v, o, do, scale, causal, quant=True)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    qt = _ste(qq, nv.fq(q, 1.0, torch.float32))
    kt = _ste(kk, nv.fq(k, 1.0, torch.float32))
    vt = _ste(vv, nv.fq(v, 1.0, torch.float32))
    s = scale * torch.einsum("bqhd,bkhd->bhqk", qt, kt)
    if causal:
        s = s.masked_fill(torch.ones(nq, nkv, dtype=torch.bool).triu(1), float("-inf"))
    m = s.amax(dim=-1, keepdim=True).detach()
    p = torch.exp(s - m)
    l = p.sum(dim=-1, keepdim=True)
    pt = _ste(p, nv.fq(p.detach(), 1.0, torch.float64, axis=-1))
    out = torch.einsum("bhqk,bkhd->bqhd", pt / l, vt)
    assert torch.allclose(out.detach(), o, rtol=0, atol=1e-12)
    out.backward(do)
    for a, b in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
        assert torch.allclose(a, b, rtol=0, atol=1e-11)


def test_finite_differences_fq_off():
    q, k, v, do = _inputs(1, 6, 9, 1, 8, seed=4)
    scale = 0.5
    o, _, _ = at.attn_fwd(q, k, v, scale, quant=False)
    dq, dk, dv = at.attn_bwd(q, k, v, o, do, scale, quant=False)

    def loss(q_, k_, v_):
        return float((at.attn_fwd(q_, k_, v_, scale, quant=False)[0] * do).sum())

    eps = 1e-6
    g = torch.Generator().manual_seed(0)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(6):
            idx = tuple(int(torch.randint(0, n, (1,), generator=g)) for n in grad.shape)
            args = [q.clone(), k.clone(), v.clone()]
            args[which][idx] += eps
            up = loss(*args)
            args[which][idx] -= 2 * eps
            dn = loss(*args)
            fd = (up - dn) / (2 * eps)
            assert abs(fd - float(grad[idx])) <= 1e-6 * max(1.0, abs(fd))


def test_constant_v_rows_closed_form():
    """With identical V rows u: O_i = (sum_j P~_ij / l_i) * fq(u)."""
    q, k, _, _ = _inputs(1, 19, 35, 2, 16, seed=5)
    u = nv.to_bf16(torch.randn(16, dtype=F64))
    v = u.expand(1, 35, 2, 16).clone()
    scale = 0.4
    o, lse, m = at.attn_fwd(q, k, v, scale)
    for h in range(2):
        qt = nv.fq(q[0, :, h], 1.0, torch.float32)
        kt = nv.fq(k[0, :, h], 1.0, torch.float32)
        s = scale * qt @ kt.T
        p = torch.exp(s - s.amax(1, keepdim=True))
        ratio = nv.fq(p, 1.0, torch.float64, axis=1).sum(1) / p.sum(1)
        ref = ratio[:, None] * nv.fq(u, 1.0, torch.float32)[None, :]
        assert torch.allclose(o[0, :, h], ref, rtol=0, atol=1e-13)


def test_forward_brute_force_exact_quantizer():
    """Pure-Python loops, exact rational block quantizer, explicit 16-key blocks
    from key 0 with a short last block, P~ referenced to the final row max."""
    nq, nkv, d = 3, 21, 16
    q, k, v, _ = _inputs(1, nq, nkv, 1, d, seed=6, spread=2.0)
    scale = 0.37
    o, lse, _ = at.attn_fwd(q, k, v, scale)

    def fq_vec(xs):
        out = []
        for b0 in range(0, len(xs), 16):
            out += [float(t) for t in nv.fake_quant_block_exact(xs[b0:b0 + 16])[2]]
        return out

    qt = [fq_vec(q[0, i, 0].tolist()) for i in range(nq)]
    kt = [fq_vec(k[0, j, 0].tolist()) for j in range(nkv)]
    vt = [fq_vec(v[0, j, 0].tolist()) for j in range(nkv)]
    for i in range(nq):
        s = [scale * sum(a * b for a, b in zip(qt[i], kt[j])) for j in range(nkv)]
        mx = max(s)
        p = [math.exp(x - mx) for x in s]
        l = sum(p)
        pt = fq_vec(p)
        for c in range(d):
            ref = sum(pt[j] * vt[j][c] for j in range(nkv)) / l
            assert abs(ref - float(o[0, i, 0, c])) <= 1e-12
        assert abs(mx + math.log(l) - float(lse[0, 0, i])) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_equals_whole(causal):
    q, k, v, do = _inputs(2, 40, 40, 2, 16, seed=7)
    scale = 0.3
    o, lse, m = at.attn_fwd(q, k, v, scale, causal, block=7)
    dq, dk, dv = at.attn_bwd(q, k, v, o, do, scale, causal, block=9)
    o2, _, _ = at.attn_fwd(q, k, v, scale, causal, block=512)
    assert torch.allclose(o, o2, rtol=0, atol=1e-14)
    rows = [0, 5, 17, 39]
    cols = [0, 15, 16, 33, 39]
    for b in range(2):
        for h in range(2):
            hp = at.HeadProblem(q, k, v, b, h, scale, causal)
            ob, lb, mb = hp.fwd_rows(rows)
            assert torch.allclose(ob, o[b, rows, h], rtol=0, atol=1e-14)
            assert torch.allclose(lb, lse[b, h, rows], rtol=0, atol=1e-14)
            dqr = hp.dq_rows(rows, o[b, rows, h], do[b, rows, h])
            assert torch.allclose(dqr, dq[b, rows, h], rtol=0, atol=1e-12)
            dkc, dvc = hp.dkdv_cols(cols, o[b, :, h], do[b, :, h], block=11)
            assert torch.allclose(dkc, dk[b, cols, h], rtol=0, atol=1e-12)
            assert torch.allclose(dvc, dv[b, cols, h], rtol=0, atol=1e-12)


def test_delta_modes_differ_only_through_delta():
    """delta_mode 'hp' takes d from P V~ / l; it leaves dV unchanged."""
    q, k, v, do = _inputs(1, 24, 24, 1, 16, seed=8)
    o, _, _ = at.attn_fwd(q, k, v, 0.3)
    a = at.attn_bwd(q, k, v, o, do, 0.3, delta_mode="o")
    b = at.attn_bwd(q, k, v, o, do, 0.3, delta_mode="hp")
    assert torch.equal(a[2], b[2])
    assert not torch.allclose(a[0], b[0], rtol=0, atol=1e-9)
    hp = at.HeadProblem(q, k, v, 0, 0, 0.3)
    assert torch.allclose(hp.dq_rows([3, 9], o[0, [3, 9], 0], do[0, [3, 9], 0], "hp"),
                          b[0][0, [3, 9], 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_aux_output_is_plain_attention_on_the_quantized_operands(causal):
    """P V~ / l with P unquantized is softmax attention over (Q~, K~, V~): PyTorch's
    scaled_dot_product_attention on the pinned quantizer's outputs."""
    q, k, v, _ = _inputs(2, 40, 40, 2, 32, seed=9)
    scale = 0.2
    o_hp = at.attn_fwd_hp(q, k, v, scale, causal)
    qt, kt, vt = (nv.fq(x, 1.0, torch.float32, axis=-1) for x in (q, k, v))
    ref = _sdpa(qt, kt, vt, scale, causal)
    assert torch.allclose(o_hp, ref, rtol=0, atol=1e-12)
    # it differs from the output, whose P is quantized
    o, _, _ = at.attn_fwd(q, k, v, scale, causal)
    assert not torch.allclose(o, o_hp, rtol=0, atol=1e-6)


def test_aux_output_equals_the_output_with_quantizers_off():
    q, k, v, _ = _inputs(1, 33, 21, 2, 16, seed=10)
    o, _, _ = at.attn_fwd(q, k, v, 0.4, quant=False)
    assert torch.allclose(at.attn_fwd_hp(q, k, v, 0.4, quant=False), o, rtol=0, atol=1e-13)


def test_hp_delta_is_delta_from_the_aux_output():
    """delta_mode 'hp' equals delta_mode 'o' handed the auxiliary output as O: the
    backward reads O for delta only."""
    q, k, v, do = _inputs(1, 24, 24, 2, 16, seed=11)
    o_hp = at.attn_fwd_hp(q, k, v, 0.3)
    o, _, _ = at.attn_fwd(q, k, v, 0.3)
    a = at.attn_bwd(q, k, v, o, do, 0.3, delta_mode="hp")
    b = at.attn_bwd(q, k, v, o_hp, do, 0.3, delta_mode="o")
    for x, y in zip(a, b):
        assert torch.allclose(x, y, rtol=0, atol=1e-12)
