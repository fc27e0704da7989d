"""Pins of the NVFP4 linear oracle against things other than itself.

- the tiled scale layout at hand-worked byte offsets, and as a bijection;
- operands already on the NVFP4 grid (fq is the identity there): the forward is a
  plain matmul;
- exact power-of-two scaling of the input (the global scale follows it exactly);
- the backward against PyTorch's autograd of torch.nn.functional.linear.
"""
import torch

from oracle import linear as ol
from oracle import nvfp4 as nv

F64 = torch.float64


def test_tiled_layout_hand_worked_offsets():
    off = ol.tiled_scale_offsets(200, 20)   # 2 row tiles x 5 block tiles
    assert int(off[0, 0]) == 0
    assert int(off[1, 0]) == 16             # next row: 16 bytes on
    assert int(off[0, 3]) == 3              # blocks 0..3 of a row are adjacent
    assert int(off[32, 0]) == 4             # row 32 shares row 0's 16 bytes, at +4
    assert int(off[33, 5]) == 533           # block tile 1 (512) + row 1 (16) + row 33 // 32 (4) + 1
    assert int(off[130, 9]) == 3617         # tile (1, 2) = 7 * 512, row 2 -> 32, block 9 % 4 -> 1
    assert int(off[127, 19]) == 4 * 512 + 31 * 16 + 3 * 4 + 3
    assert ol.tiled_scale_bytes(200, 320) == 256 * 20


def test_tiled_layout_is_a_bijection_with_zero_padding():
    g = torch.Generator().manual_seed(5)
    sb = torch.randint(1, 255, (130, 7), generator=g, dtype=torch.uint8)
    buf = ol.tile_scales(sb)
    assert buf.numel() == 256 * 8
    assert torch.equal(ol.untile_scales(buf, 130, 7 * 16), sb)
    assert int((buf != 0).sum()) == sb.numel()       # every other byte is padding, zero
    off = ol.tiled_scale_offsets(256, 8).reshape(-1)
    assert torch.equal(torch.sort(off).values, torch.arange(256 * 8))


def _grid_matrix(rows, cols, seed):
    """Values code * 2^e with every 16-block holding a 6 * 2^e (amax), so that
    with unit global scale s = 2^e exactly and fq(x) == x."""
    g = torch.Generator().manual_seed(seed)
    grid = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=F64)
    idx = torch.randint(0, 8, (rows, cols), generator=g)
    sign = torch.where(torch.rand(rows, cols, generator=g) < 0.5, -1.0, 1.0).to(F64)
    x = grid[idx] * sign
    x.view(rows, cols // 16, 16)[..., 0] = 6.0
    e = torch.randint(-3, 3, (rows, cols // 16, 1), generator=g).to(F64)
    return (x.view(rows, cols // 16, 16) * torch.pow(2.0, e)).reshape(rows, cols)


def test_operands_on_the_grid_give_a_plain_matmul():
    x, w = _grid_matrix(24, 64, 1), _grid_matrix(16, 64, 2)
    assert torch.equal(nv.fq(x, 1.0), x) and torch.equal(nv.fq(w, 1.0), w)
    b = torch.linspace(-1, 1, 16, dtype=F64)
    out = ol.linear_fwd(x, w, b, gsf_x=1.0, gsf_w=1.0)
    assert torch.equal(out, x @ w.T + b)


def test_power_of_two_scaling_of_the_input():
    g = torch.Generator().manual_seed(3)
    x = nv.to_bf16(torch.randn(32, 128, generator=g, dtype=F64))
    w = nv.to_bf16(torch.randn(48, 128, generator=g, dtype=F64))
    a = ol.linear_fwd(x, w)
    b = ol.linear_fwd(x * 8.0, w)
    assert torch.equal(b, 8.0 * a)
    # the global scale matters: unit scales quantize differently
    assert not torch.allclose(ol.linear_fwd(x, w, gsf_x=1.0, gsf_w=1.0), a, rtol=0, atol=1e-9)


def test_backward_matches_autograd_of_linear():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(20, 32, generator=g, dtype=F64, requires_grad=True)
    w = torch.randn(12, 32, generator=g, dtype=F64, requires_grad=True)
    b = torch.randn(12, generator=g, dtype=F64, requires_grad=True)
    grad = torch.randn(20, 12, generator=g, dtype=F64)
    torch.nn.functional.linear(x, w, b).backward(grad)
    gx, gw, gb = ol.linear_bwd(grad, x.detach(), w.detach())
    for got, ref in ((gx, x.grad), (gw, w.grad), (gb, b.grad)):
        assert torch.allclose(got, ref, rtol=0, atol=1e-12)
