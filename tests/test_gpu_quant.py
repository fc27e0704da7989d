"""Bit-exact parity of the standalone NVFP4 quantizer (CUDA, through the C ABI)
with the oracle: dequantized bf16 values, E4M3FN scale bytes, packed codes and
the static global scale, for unit and static global scales."""
import numpy as np
import pytest
import torch

from nvfp4_fake_quant_gb300 import api, workloads
from oracle import nvfp4 as onv

pytestmark = pytest.mark.gpu


def _check_matrix(x_cpu: torch.Tensor, gsf_dev=None, gsf_host=1.0, ld=None):
    rows, cols = x_cpu.shape
    if ld is None:
        xd = x_cpu.cuda()
    else:
        buf = torch.zeros(rows, ld, dtype=torch.bfloat16)
        buf[:, :cols] = x_cpu
        xd = buf.cuda()[:, :cols]
    out, sc = api.nvfp4_fake_quant(xd, gsf_dev)
    codes, sc2 = api.nvfp4_quantize_codes(xd, gsf_dev)
    assert api.device_status() == 0
    ref_bits, ref_sc, ref_codes = onv.quantizer_outputs(x_cpu.double(), gsf_host)
    got_bits = out.cpu().view(torch.int16)
    assert torch.equal(sc.cpu(), ref_sc), "scale bytes differ"
    assert torch.equal(sc2.cpu(), ref_sc), "scale bytes (codes call) differ"
    assert torch.equal(codes.cpu(), ref_codes), "codes differ"
    assert torch.equal(got_bits, ref_bits), "dequantized values differ"


def test_quantizer_workload_unit_and_static():
    """bf16 4096x4096 with outliers and zero blocks: unit and static gsf."""
    x = workloads.quant_matrix()
    _check_matrix(x)
    xd = x.cuda()
    gsf = api.nvfp4_global_sf(xd)
    g_ref = onv.global_sf(x.double())
    assert np.float32(gsf.item()) == np.float32(g_ref)
    _check_matrix(x, gsf, g_ref)


@pytest.mark.parametrize("rows,cols,ld,seed,spread", [(37, 80, 96, 1, 1.0), (1, 16, 16, 2, 1e-3),
                                                      (513, 208, 208, 3, 300.0),
                                                      (64, 4096, 4104, 4, 1.0),
                                                      # static scale near the fp32 range ends:
                                                      # outputs 6*448/gsf above 2^124 take the
                                                      # IEEE path; a clamped amax (1e-12) gives
                                                      # gsf = 2.688e15
                                                      (256, 64, 64, 5, 3e37), (128, 128, 128, 6, 1e-14)])
def test_quantizer_shapes_and_strides(rows, cols, ld, seed, spread):
    x = workloads.random_matrix(rows, cols, seed, spread)
    _check_matrix(x, ld=ld)
    gsf = api.nvfp4_global_sf(x.cuda())
    _check_matrix(x, gsf, onv.global_sf(x.double()), ld=ld)


def test_quantizer_every_bf16_value_and_all_ties():
    """Every finite bf16 value next to fixed companions, every E2M1 tie at every
    scale and every E4M3 midpoint."""
    b = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = b[torch.isfinite(b.float())].double()
    blocks = []
    for amax in [1.0, 6.0, 0.01171875, 2688.0, 1e30]:
        blk = torch.zeros(vals.numel(), 16, dtype=torch.float64)
        blk[:, 0] = vals
        blk[:, 1] = amax
        blocks.append(blk)
    ties = []
    for sb in range(1, 0x7F):
        s = float(onv.E4M3_VALUES[sb])
        ties.append([6 * s, 0.25 * s, 0.75 * s, 1.25 * s, -1.75 * s, 2.5 * s, 3.5 * s, 5 * s,
                     -0.5 * s, s, 1.5 * s, 2 * s, 3 * s, -4 * s, 0.0, -0.0])
    v = onv.E4M3_VALUES.tolist()
    for lo, hi in zip(v[:-1], v[1:]):
        ties.append([3 * (lo + hi)] + [0.0] * 15)
    blocks.append(torch.tensor(ties, dtype=torch.float64))
    x = torch.cat(blocks).to(torch.bfloat16)
    _check_matrix(x)


def test_quantizer_in_place():
    x = workloads.random_matrix(128, 256, 7)
    xd = x.cuda()
    out, _ = api.nvfp4_fake_quant(xd, None, out=xd)
    ref_bits, _, _ = onv.quantizer_outputs(x.double(), 1.0)
    assert torch.equal(out.cpu().view(torch.int16), ref_bits)
