"""The forward with the auxiliary high-precision output O_hp = P V~ / l ("Attn-QAT
Training" guide, attn_qat_train(): use_high_prec_o) and the backward whose delta
is taken from it, on the GPU through the C ABI, against the float64 oracle.

The kernel runs one query tile per CTA with the even and odd key tiles on the
two softmax pairs, so the shapes include odd key-tile counts (the second pair's
last tile is then missing), causal masking, D = 64 and ragged tails.  Its o and
stats are the plain forward's: m bit-identical, o within the last bf16 place
(the row sums are added in another order).
"""
import pytest
import torch

from nvfp4_fake_quant_gb300 import api, workloads
from oracle import attention as oa
from oracle import nvfp4 as onv

pytestmark = pytest.mark.gpu

O_RTOL, O_ATOL, G_RTOL, LSE_ATOL = 1e-2, 5e-2, 2e-2, 2e-3


def rel_l2(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b).clamp_min(1e-30))


CASES = [
    # name, B, Nq, Nkv, H, D, causal, seed
    ("tiny_config", 1, 256, 256, 2, 64, False, 0),
    ("odd_tiles_d128", 2, 300, 300, 3, 128, False, 30),
    ("cross_d128", 1, 200, 333, 2, 128, False, 31),
    ("causal_d64", 1, 300, 300, 2, 64, True, 32),
    ("causal_d128", 1, 640, 640, 1, 128, True, 33),
    ("five_tiles", 1, 640, 640, 2, 128, False, 34),
    ("short", 1, 17, 15, 1, 128, False, 35),
    ("single", 1, 1, 1, 1, 64, False, 36),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_aux_output_parity(case):
    name, b, nq, nkv, h, d, causal, seed = case
    inp = workloads.attn_inputs(b, nq, nkv, h, d, seed, causal=causal)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, o_hp, stats = api.attn_qat_fwd_hp(q, k, v, inp.scale, causal)
    o_plain, stats_plain = api.attn_qat_fwd(q, k, v, inp.scale, causal)
    dq, dk, dv = api.attn_qat_bwd(q, k, v, o_hp, stats, do, inp.scale, causal)
    assert api.device_status() == 0
    o_ref, lse_ref, _ = oa.attn_fwd(inp.q, inp.k, inp.v, inp.scale, causal)
    hp_ref = oa.attn_fwd_hp(inp.q, inp.k, inp.v, inp.scale, causal)
    g_ref = oa.attn_bwd(inp.q, inp.k, inp.v, onv.to_bf16(hp_ref), inp.do, inp.scale, causal)
    st = stats.cpu().double()
    errs = {"o": rel_l2(o, o_ref), "o_hp": rel_l2(o_hp, hp_ref),
            "o_hp_maxabs": float((o_hp.cpu().double() - hp_ref).abs().max()),
            "o_vs_plain": rel_l2(o, o_plain),
            "lse": float((st[:, :, 0] - lse_ref).abs().max()),
            "dq": rel_l2(dq, g_ref[0]), "dk": rel_l2(dk, g_ref[1]), "dv": rel_l2(dv, g_ref[2])}
    print(name, errs)
    assert errs["o"] <= O_RTOL and errs["lse"] <= LSE_ATOL, errs
    assert errs["o_hp"] <= O_RTOL and errs["o_hp_maxabs"] <= O_ATOL, errs
    assert errs["o_vs_plain"] <= 2e-3, errs
    assert torch.equal(stats[:, :, 1].cpu(), stats_plain[:, :, 1].cpu())
    assert all(errs[n] <= G_RTOL for n in ("dq", "dk", "dv")), errs


def test_hp_delta_reaches_the_gradients():
    """dQ from the hp delta is nearer the oracle's hp gradient than its O-delta one,
    and the autograd module with delta_mode='hp' gives the same bits as the calls."""
    inp = workloads.attn_inputs(1, 384, 384, 2, 128, seed=37)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, o_hp, stats = api.attn_qat_fwd_hp(q, k, v, inp.scale)
    dq, _, _ = api.attn_qat_bwd(q, k, v, o_hp, stats, do, inp.scale)
    o_ref, _, _ = oa.attn_fwd(inp.q, inp.k, inp.v, inp.scale)
    hp_ref = oa.attn_fwd_hp(inp.q, inp.k, inp.v, inp.scale)
    dq_hp = oa.attn_bwd(inp.q, inp.k, inp.v, onv.to_bf16(hp_ref), inp.do, inp.scale)[0]
    dq_o = oa.attn_bwd(inp.q, inp.k, inp.v, onv.to_bf16(o_ref), inp.do, inp.scale)[0]
    assert rel_l2(dq_hp, dq_o) > 2 * rel_l2(dq, dq_hp)
    mod = api.AttnQAT(2, 128, inp.scale, delta_mode="hp")
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = mod(qq, kk, vv)
    out.backward(do)
    assert torch.equal(out, o)
    assert torch.equal(qq.grad, dq)
    with pytest.raises(ValueError):
        api.AttnQAT(2, 128, delta_mode="x")
