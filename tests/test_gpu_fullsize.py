"""Parity at the full Wan sizes, in the launch configuration bench.py times,
on outputs the oracle computes one by one:

- forward: O, LSE and m of sampled query rows (first, last, tile edges, random)
- backward: dQ of sampled query rows and dK, dV of sampled key columns
  (including the ragged last 16-key block at N = 32760)

For the sampled dK/dV columns the oracle needs delta = rowsum(dO * o) of every
query row.  Both sides therefore take the same seeded synthetic `o` (bf16,
0.05 * N(0,1)); the backward is defined for any `o`.  The forward's own output
is checked separately on its rows, and the chain fwd -> bwd on small shapes in
test_gpu_attn.py.
"""
import pytest
import torch

from nvfp4_fake_quant_gb300 import api, workloads
from oracle import attention as oa

pytestmark = pytest.mark.gpu

O_RTOL, O_ATOL, G_RTOL, LSE_ATOL = 1e-2, 5e-2, 2e-2, 2e-3


def rel_l2(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b).clamp_min(1e-30))


def _sample(n, count, seed):
    g = torch.Generator().manual_seed(seed)
    fixed = [0, 1, 127, 128, 129, 255, 256, n // 2, n - 129, n - 128, n - 17, n - 16, n - 9, n - 8,
             n - 2, n - 1]
    rnd = torch.randint(0, n, (count,), generator=g).tolist()
    return sorted({i for i in fixed + rnd if 0 <= i < n})


@pytest.mark.parametrize("name,heads", [("wan25088", (0, 7)), ("wan32760", (0, 11))])
def test_fullsize_sampled_parity(name, heads):
    inp = getattr(workloads, name)()
    b, n, _, h, d = inp.shape
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, stats = api.attn_qat_fwd(q, k, v, inp.scale)
    g = torch.Generator().manual_seed(99)
    o_syn = (0.05 * torch.randn(b, n, h, d, generator=g)).to(torch.bfloat16)
    dq, dk, dv = api.attn_qat_bwd(q, k, v, o_syn.cuda(), stats, do, inp.scale)
    assert api.device_status() == 0
    rows = _sample(n, 40, 1)
    cols = _sample(n, 24, 2)
    o_c, st_c = o.cpu(), stats.cpu().double()
    dq_c, dk_c, dv_c = dq.cpu(), dk.cpu(), dv.cpu()
    for hh in heads:
        sl = slice(hh, hh + 1)
        hp = oa.HeadProblem(inp.q[:, :, sl], inp.k[:, :, sl], inp.v[:, :, sl], 0, 0, inp.scale)
        o_ref, lse_ref, m_ref = hp.fwd_rows(rows)
        o_got = o_c[0, rows, hh].double()
        assert rel_l2(o_got, o_ref) <= O_RTOL, (name, hh, rel_l2(o_got, o_ref))
        assert float((o_got - o_ref).abs().max()) <= O_ATOL
        assert float((st_c[0, hh, 0, rows] - lse_ref).abs().max()) <= LSE_ATOL
        assert float((st_c[0, hh, 1, rows] - m_ref).abs().max()) <= 1e-4 * max(1.0, float(m_ref.abs().max()))
        do_h = inp.do[0, :, hh].double()
        o_h = o_syn[0, :, hh].double()
        dq_ref = hp.dq_rows(rows, o_h[rows], do_h[rows])
        assert rel_l2(dq_c[0, rows, hh], dq_ref) <= G_RTOL, (name, hh, "dq")
        dk_ref, dv_ref = hp.dkdv_cols(cols, o_h, do_h, block=1024)
        assert rel_l2(dk_c[0, cols, hh], dk_ref) <= G_RTOL, (name, hh, "dk", rel_l2(dk_c[0, cols, hh], dk_ref))
        assert rel_l2(dv_c[0, cols, hh], dv_ref) <= G_RTOL, (name, hh, "dv", rel_l2(dv_c[0, cols, hh], dv_ref))
