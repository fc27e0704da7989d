"""Parity of the CUDA Attn-QAT forward and straight-through backward (through the
C ABI) with the float64 oracle, element by element, on shapes spanning several
128-row tiles, ragged tails (N % 128 and N % 16 != 0), cross attention, causal
masking, D = 64 and 128, and the degenerate N = 1.

Acceptance: O rel-L2 <= 1e-2 and max-abs <= 5e-2; dQ, dK, dV rel-L2 <= 2e-2;
LSE within 2e-3 absolute.  The oracle's backward takes the oracle's own O
(rounded to bf16) as its `o`; the CUDA backward takes the CUDA forward's o.
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
    # name, B, Nq, Nkv, H, D, causal, seed, dist, scale
    ("tiny_config", 1, 256, 256, 2, 64, False, 0, "normal", 1 / 8),
    ("ragged_d128", 2, 300, 300, 3, 128, False, 10, "normal", None),
    ("cross_d128", 1, 200, 333, 2, 128, False, 11, "normal", None),
    ("causal_d64", 1, 300, 300, 2, 64, True, 12, "normal", None),
    ("causal_d128", 2, 257, 257, 1, 128, True, 13, "normal", None),
    ("short", 1, 17, 15, 1, 128, False, 14, "normal", None),
    ("single", 1, 1, 1, 1, 64, False, 15, "normal", None),
    ("unit_rms", 1, 640, 640, 2, 128, False, 16, "unit_rms", None),
    ("lognormal_channels", 1, 520, 520, 2, 128, False, 17, "lognormal_channels", None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_attention_parity(case):
    name, b, nq, nkv, h, d, causal, seed, dist, scale = case
    inp = workloads.attn_inputs(b, nq, nkv, h, d, seed, scale=scale, causal=causal, dist=dist)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, stats = api.attn_qat_fwd(q, k, v, inp.scale, causal)
    dq, dk, dv = api.attn_qat_bwd(q, k, v, o, stats, do, inp.scale, causal)
    assert api.device_status() == 0
    o_ref, lse_ref, m_ref = oa.attn_fwd(inp.q, inp.k, inp.v, inp.scale, causal)
    o_ref_bf16 = onv.to_bf16(o_ref)
    dq_ref, dk_ref, dv_ref = oa.attn_bwd(inp.q, inp.k, inp.v, o_ref_bf16, inp.do, inp.scale,
                                         causal)
    st = stats.cpu().double()
    errs = {"o": rel_l2(o, o_ref), "o_maxabs": float((o.cpu().double() - o_ref).abs().max()),
            "lse": float((st[:, :, 0] - lse_ref).abs().max()),
            "m": float((st[:, :, 1] - m_ref).abs().max()),
            "dq": rel_l2(dq, dq_ref), "dk": rel_l2(dk, dk_ref), "dv": rel_l2(dv, dv_ref)}
    print(name, errs)
    assert errs["o"] <= O_RTOL, errs
    assert errs["o_maxabs"] <= O_ATOL, errs
    assert errs["lse"] <= LSE_ATOL, errs
    assert errs["m"] <= 1e-4 * max(1.0, float(m_ref.abs().max())), errs
    assert all(errs[n] <= G_RTOL for n in ("dq", "dk", "dv")), errs


def test_quantizers_matter():
    """The result must differ from unquantized attention by much more than the
    tolerance, so the parity above is not met by plain attention."""
    inp = workloads.tiny()
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    o, _ = api.attn_qat_fwd(q, k, v, inp.scale)
    o_plain, _, _ = oa.attn_fwd(inp.q, inp.k, inp.v, inp.scale, quant=False)
    o_ref, _, _ = oa.attn_fwd(inp.q, inp.k, inp.v, inp.scale)
    assert rel_l2(o_ref, o_plain) > 5e-2
    assert rel_l2(o, o_ref) < 0.2 * rel_l2(o, o_plain)


def test_repeatable_and_autograd_module():
    """Same inputs give bit-identical outputs; the autograd module matches the calls."""
    inp = workloads.attn_inputs(1, 384, 384, 2, 128, seed=21)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o1, s1 = api.attn_qat_fwd(q, k, v, inp.scale)
    o2, s2 = api.attn_qat_fwd(q, k, v, inp.scale)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    dq1, dk1, dv1 = api.attn_qat_bwd(q, k, v, o1, s1, do, inp.scale)
    mod = api.AttnQAT(2, 128, inp.scale)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = mod(qq, kk, vv)
    out.backward(do)
    assert torch.equal(out.detach(), o1)
    assert torch.equal(dk1, kk.grad) and torch.equal(dv1, vv.grad)
    assert rel_l2(qq.grad, dq1) < 1e-6  # dQ accumulates with atomics: order may vary
