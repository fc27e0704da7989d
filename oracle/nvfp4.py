"""NVFP4 fake-quantization oracle (TEST INFRASTRUCTURE ONLY; see ``oracle/__init__``).

What it computes ("nvfp4_qad.py", module docstring; "vsqa-preview-1.3b
metadata.json", ``attention.precision``: group_size 16, NVFP4 E2M1 values,
FP8 E4M3FN scales):

  for every block of 16 contiguous elements x_0..x_15 (the last block of a row
  may be shorter):
    1. amax   = max_i |x_i|
    2. s      = E4M3( amax * gsf / 6 )         round-to-nearest-even, saturating at 448
    3. code_i = E2M1( |x_i| * gsf / s )        grid {0,.5,1,1.5,2,3,4,6}, RNE, saturating at 6
                                               (every code is 0 when s == 0)
    4. x~_i   = sign(x_i) * code_i * s / gsf   (dequantized value; "nvfp4_qad.py",
                                               ``nvfp4_gemm``: alpha = (1/w_sf)/input_sf)

gsf is the global scale: 1.0 ("unit": attention and attention projections) or
448*6/amax(X) ("static"; ``weight_global_sf``), see ``global_sf``.

Precision of the rounding decisions.  The pages do not say in which arithmetic
amax*gsf/6 and |x|*gsf/s are formed.  Reading taken here: in the arithmetic of
the kernel, IEEE fp32 with every product and quotient rounded to nearest even,
and the decisions of steps 2 and 3 are then taken exactly on those fp32
values; step 4 is an fp32 quotient too.  ``prec=torch.float64`` runs the same
steps in fp64; the attention oracle uses it for its float64 probabilities P.
For bf16 inputs and unit gsf both precisions, and the exact rational
``fake_quant_block_exact``, take identical decisions (proved in the tests on
every bf16 value and every tie).

Representation: the E4M3FN byte of a non-negative finite value is its index in
the ascending list of the 127 such values; the E2M1 magnitude code is its
index in the 8-entry grid.  Both lists are written out from the format
definitions and checked in the tests against PyTorch's float8_e4m3fn.

Plain PyTorch CPU ops (float32/float64) are used so that large inputs run on all
host cores; nothing here is blocked, fused or reordered beyond the steps above.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

BLOCK = 16
FP4_MAX = 6.0
E4M3_MAX = 448.0
FP4_RANGE = E4M3_MAX * FP4_MAX  # 2688: "nvfp4_qad.py", FP4_RANGE


def _e4m3fn_values() -> list:
    """The 127 non-negative finite E4M3FN values; list index == bit pattern.

    E4M3FN: 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
    subnormal (m * 2^-9); pattern 0x7F is NaN and there are no infinities.
    """
    vals = []
    for byte in range(0x7F):
        e, m = byte >> 3, byte & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return vals


E4M3_VALUES = torch.tensor(_e4m3fn_values(), dtype=torch.float64)
E2M1_GRID = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)


def _t(x, dtype=torch.float64) -> torch.Tensor:
    if isinstance(x, torch.Tensor):
        return x.to(dtype)
    return torch.as_tensor(np.asarray(x), dtype=dtype)


def round_to_grid(v: torch.Tensor, grid: torch.Tensor) -> torch.Tensor:
    """Index of the grid point nearest to v >= 0; ties to the even index; saturating.

    2v and lo+hi are exact in float64 for float32/float64 v and for grid points
    with few significant bits, so the comparison is the exact decision.
    """
    v = v.to(torch.float64)
    n = grid.numel()
    hi = torch.searchsorted(grid, v.contiguous(), right=False).clamp_(0, n - 1)
    lo = (hi - 1).clamp_(min=0)
    twice = 2.0 * v
    mid = grid[lo] + grid[hi]
    pick_hi = (twice > mid) | ((twice == mid) & (hi % 2 == 0))
    idx = torch.where(pick_hi, hi, lo)
    return torch.where(v >= grid[-1], torch.full_like(idx, n - 1), idx)


def e4m3_round(v) -> torch.Tensor:
    """E4M3FN byte of RNE(v), v >= 0 finite, saturating at 448 (satfinite)."""
    return round_to_grid(_t(v), E4M3_VALUES).to(torch.uint8)


def e2m1_round(v) -> torch.Tensor:
    """E2M1 magnitude code (0..7) of RNE(v), v >= 0 finite, saturating at 6."""
    return round_to_grid(_t(v), E2M1_GRID).to(torch.uint8)


def to_bf16(x) -> torch.Tensor:
    """Round (via fp32) to bfloat16, RNE; values returned as float64."""
    return _t(x, torch.float32).to(torch.bfloat16).to(torch.float64)


def bf16_bits(x) -> torch.Tensor:
    """int16 bit patterns of x rounded (via fp32) to bfloat16, RNE."""
    return _t(x, torch.float32).to(torch.bfloat16).view(torch.int16)


def global_sf(x) -> float:
    """Static global scale 448*6/amax(|x|) as an fp32 value, amax clamped at 1e-12.

    "nvfp4_qad.py", ``weight_global_sf`` (and ``input_global_sf`` for static
    activations): fp32 quotient of 2688 by the fp32 amax of the finite tensor.
    The fp64 quotient rounded once to fp32 equals the correctly rounded fp32
    quotient (both operands carry at most 24 bits).
    """
    x = _t(x)
    amax = float(x.abs().max()) if x.numel() else 0.0
    amax = max(float(np.float32(amax)), float(np.float32(1e-12)))
    return float(np.float32(FP4_RANGE / amax))


def fake_quant(x, gsf=1.0, prec=torch.float32, axis: int = -1):
    """NVFP4 fake-quantization of ``x`` in blocks of 16 along ``axis``.

    Returns (xq, scale_bytes, codes):
      xq          dequantized values (float64 tensor shaped like x), step 4, no
                  final bf16 rounding
      scale_bytes uint8 E4M3FN bytes, x.shape with ``axis`` -> ceil(n/16)
      codes       uint8 4-bit codes (sign << 3 | magnitude index), shaped like x
    A short last block (n % 16 != 0) is quantized on its own elements.
    """
    x = _t(x).movedim(axis, -1)
    n = x.shape[-1]
    nb = -(-n // BLOCK)
    pad = nb * BLOCK - n
    xp = torch.nn.functional.pad(x, (0, pad)) if pad else x
    xb = xp.reshape(x.shape[:-1] + (nb, BLOCK))
    ax = xb.abs()
    g = torch.tensor(gsf, dtype=prec)
    six = torch.tensor(FP4_MAX, dtype=prec)
    amax = ax.amax(dim=-1)
    t = amax.to(prec) * g                                # step 2: amax*gsf (rounded in prec)
    t = t / six                                          #         then /6  (rounded in prec)
    sbyte = e4m3_round(t)
    s = E4M3_VALUES[sbyte.long()]
    y = ax.to(prec) * g                                  # step 3: |x|*gsf  (rounded in prec)
    sp = s.to(prec).unsqueeze(-1)
    nz = sp > 0
    q = torch.where(nz, y / torch.where(nz, sp, torch.ones_like(sp)), torch.zeros_like(y))
    cidx = e2m1_round(q)
    mag = E2M1_GRID[cidx.long()] * s.unsqueeze(-1)      # exact: <= 7 significant bits
    deq = (mag.to(prec) / g).to(torch.float64)           # step 4: /gsf (rounded in prec)
    neg = torch.signbit(xb)
    xq = torch.where(neg, -deq, deq)
    codes = cidx | (neg.to(torch.uint8) << 3)
    xq = xq.reshape(xp.shape)[..., :n]
    codes = codes.reshape(xp.shape)[..., :n]
    return xq.movedim(-1, axis), sbyte.movedim(-1, axis), codes.movedim(-1, axis)


def fq(x, gsf=1.0, prec=torch.float32, axis: int = -1) -> torch.Tensor:
    """Dequantized NVFP4 fake-quant values only (see ``fake_quant``)."""
    return fake_quant(x, gsf, prec, axis)[0]


def quantizer_outputs(x, gsf=1.0):
    """The standalone quantizer's outputs for a bf16 matrix x [rows, cols], cols % 16 == 0.

    Returns (out_bits int16 [rows, cols], scale_bytes uint8 [rows, cols/16],
    packed_codes uint8 [rows, cols/2], low nibble = even element).  The fp32
    dequantized value is rounded to bf16 (RNE); with unit gsf it is exact.
    """
    xq, sb, codes = fake_quant(x, gsf, torch.float32, axis=-1)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return bf16_bits(xq), sb, packed


# ----------------------------------------------------------------------------
# Exact rational version, for pinning the tensor quantizer (slow: small inputs)
# ----------------------------------------------------------------------------

def _e4m3fn_fractions() -> list:
    out = []
    for byte in range(0x7F):
        e, m = byte >> 3, byte & 7
        out.append(Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return out


E4M3_FRACTIONS = _e4m3fn_fractions()
E2M1_FRACTIONS = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2),
                  Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def rne_exact(v: Fraction, grid: list) -> int:
    """Exact nearest-grid index of v >= 0, ties to the even index, saturating."""
    if v >= grid[-1]:
        return len(grid) - 1
    for i in range(1, len(grid)):
        if v < grid[i]:
            lo, hi = grid[i - 1], grid[i]
            if v - lo != hi - v:
                return i - 1 if v - lo < hi - v else i
            return i if i % 2 == 0 else i - 1
    raise AssertionError("unreachable")


def fake_quant_block_exact(block, gsf=Fraction(1)):
    """One block in exact rational arithmetic (no intermediate rounding at all).

    Returns (scale_byte, [magnitude code indices], [dequantized Fractions]).
    """
    xs = [Fraction(v) for v in block]
    gsf = Fraction(gsf)
    amax = max(abs(v) for v in xs)
    sb = rne_exact(amax * gsf / 6, E4M3_FRACTIONS)
    s = E4M3_FRACTIONS[sb]
    idx, deq = [], []
    for v in xs:
        c = 0 if s == 0 else rne_exact(abs(v) * gsf / s, E2M1_FRACTIONS)
        idx.append(c)
        d = E2M1_FRACTIONS[c] * s / gsf
        deq.append(-d if v < 0 else d)
    return sb, idx, deq
