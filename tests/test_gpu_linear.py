"""The NVFP4 linear on the GPU through the C ABI against the float64 oracle:

- tiled quantizer: packed codes and scale bytes bit-exact (unit and static global
  scale, ragged row tiles, a block count that is not a multiple of 4), padding zero;
- forward: out = fq(x) fq(w)^T + bias; the FP4 GEMM's products are exact, so the
  error is the fp32 accumulation and the bf16 rounding of out: rel-L2 <= 5e-3;
- backward: BF16 GEMMs with fp32 accumulation against float64: rel-L2 <= 1e-2 for
  grad_x, grad_w; grad_b within bf16 rounding;
- the autograd module against the calls, and the Wan FFN up-projection at full
  size on sampled rows.
"""
import pytest
import torch

from nvfp4_fake_quant_gb300 import api, workloads
from oracle import linear as ol
from oracle import nvfp4 as onv

pytestmark = pytest.mark.gpu

FWD_RTOL, BWD_RTOL = 5e-3, 1e-2


def rel_l2(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b).clamp_min(1e-30))


@pytest.mark.parametrize("rows,cols,static", [(200, 320, True), (130, 80, False), (256, 1536, True),
                                              (1, 64, False)])
def test_tiled_quantizer_is_bit_exact(rows, cols, static):
    x = workloads.quant_matrix(rows, cols, seed=50 + rows)
    gsf = onv.global_sf(x) if static else None
    gsf_t = torch.tensor([gsf], dtype=torch.float32, device="cuda") if static else None
    codes, scales = api.nvfp4_quantize_tiled(x.cuda(), gsf_t)
    assert api.device_status() == 0
    ref_codes, ref_scales = ol.quantize_tiled(x, gsf)
    assert torch.equal(codes.cpu(), ref_codes)
    assert torch.equal(scales.cpu(), ref_scales)  # includes the zero padding


# (2048, 1536, 512): 192 output tiles of 128 x 128, more than one per CTA, so both
# TMEM accumulators and the persistent loop are used; K = 320 and 192 end on a
# partial stage of the 256-element pipeline; N = 96 is a partial tile.
@pytest.mark.parametrize("m,n,k,bias", [(256, 256, 320, True), (200, 512, 128, False),
                                        (64, 96, 1536, True), (1000, 128, 64, True),
                                        (2048, 1536, 512, True), (300, 640, 192, False)])
def test_forward_parity(m, n, k, bias):
    inp = workloads.linear_inputs(m, n, k, seed=60 + m)
    b = inp.bias if bias else None
    out = api.nvfp4_linear_fwd(inp.x.cuda(), inp.w.cuda(), None if b is None else b.cuda())
    assert api.device_status() == 0
    ref = ol.linear_fwd(inp.x, inp.w, b)
    assert rel_l2(out, ref) <= FWD_RTOL, rel_l2(out, ref)
    # quantization matters: the plain bf16 product is far off
    plain = inp.x.double() @ inp.w.double().T + (0 if b is None else b.double())
    assert rel_l2(plain, ref) > 10 * rel_l2(out, ref)


def test_forward_with_given_global_scales():
    inp = workloads.linear_inputs(128, 256, 256, seed=70)
    gx, gw = 2688.0 / 7.0, 2688.0 / 0.5   # deliberately not the operands' own
    t = lambda v: torch.tensor([v], dtype=torch.float32, device="cuda")
    out = api.nvfp4_linear_fwd(inp.x.cuda(), inp.w.cuda(), None, t(gx), t(gw))
    assert api.device_status() == 0
    gx32, gw32 = float(torch.tensor(gx, dtype=torch.float32)), float(torch.tensor(gw, dtype=torch.float32))
    ref = ol.linear_fwd(inp.x, inp.w, None, gx32, gw32)
    assert rel_l2(out, ref) <= FWD_RTOL


# (2048, 1024, 2560): 240 output tiles of 128 x 256 over both gradients in one
# launch, more than one per CTA; (256, 256, 320): K = 320 is a partial 256-wide tile
@pytest.mark.parametrize("m,n,k", [(256, 256, 320), (200, 512, 128), (2048, 1024, 2560)])
def test_backward_parity(m, n, k):
    inp = workloads.linear_inputs(m, n, k, seed=80 + m)
    gx, gw, gb = api.nvfp4_linear_bwd(inp.grad.cuda(), inp.x.cuda(), inp.w.cuda())
    assert api.device_status() == 0
    rx, rw, rb = ol.linear_bwd(inp.grad, inp.x, inp.w)
    assert rel_l2(gx, rx) <= BWD_RTOL and rel_l2(gw, rw) <= BWD_RTOL
    assert torch.allclose(gb.cpu().double(), rb, rtol=1e-2, atol=1e-2)


def test_module_matches_the_calls():
    inp = workloads.linear_inputs(3 * 64, 128, 256, seed=90)
    lin = api.NVFP4Linear(256, 128, device="cuda")
    with torch.no_grad():
        lin.weight.copy_(inp.w)
        lin.bias.copy_(inp.bias)
    x = inp.x.cuda().view(3, 64, 256).requires_grad_(True)
    y = lin(x)
    y.backward(inp.grad.cuda().view(3, 64, 128))
    out = api.nvfp4_linear_fwd(inp.x.cuda(), inp.w.cuda(), inp.bias.cuda())
    gx, gw, gb = api.nvfp4_linear_bwd(inp.grad.cuda(), inp.x.cuda(), inp.w.cuda())
    assert torch.equal(y.reshape(-1, 128), out)
    assert torch.equal(x.grad.reshape(-1, 256), gx)
    assert torch.equal(lin.weight.grad, gw) and torch.equal(lin.bias.grad, gb)


def test_wan_ffn_up_fullsize_sampled():
    inp = workloads.wan_ffn_up()
    x, w, b = inp.x.cuda(), inp.w.cuda(), inp.bias.cuda()
    out = api.nvfp4_linear_fwd(x, w, b)
    gx, gw, gb = api.nvfp4_linear_bwd(inp.grad.cuda(), x, w)
    assert api.device_status() == 0
    g = torch.Generator().manual_seed(7)
    rows = sorted(set([0, 1, 127, 128, 25087] + torch.randint(0, 25088, (27,), generator=g).tolist()))
    # the global scales are those of the whole operands
    gsx, gsw = onv.global_sf(inp.x), onv.global_sf(inp.w)
    ref = ol.linear_fwd(inp.x[rows], inp.w, inp.bias, gsx, gsw)
    assert rel_l2(out.cpu()[rows], ref) <= FWD_RTOL
    rx = inp.grad[rows].double() @ inp.w.double()
    assert rel_l2(gx.cpu()[rows], rx) <= BWD_RTOL
    cols = sorted(set([0, 8959] + torch.randint(0, 8960, (14,), generator=g).tolist()))
    rw = inp.grad[:, cols].double().T @ inp.x.double()
    assert rel_l2(gw.cpu()[cols], rw) <= BWD_RTOL
    rb = inp.grad.double().sum(dim=0)
    assert torch.allclose(gb.cpu().double(), rb, rtol=1e-2, atol=0.5)
