"""Pins of the NVFP4 quantizer oracle against things other than itself.

- PyTorch's float8_e4m3fn decoding and rounding (library routine)
- hand-worked examples (tests/golden/nvfp4_hand_examples.txt, derived from the format)
- the exact rational quantizer on every bf16 value, every tie and random blocks
- brute-force idempotence over every reachable (scale, max code) pair
- scale equivariance of the static global scale
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nvfp4 as nv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_hand_examples.txt")


def _parse_float(s):
    s = s.strip()
    return -0.0 if s == "-0" else float(s)


def load_hand_examples():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, gsf, xs, sb, ys = [p.strip() for p in line.split("|")]
            cases.append((name, float(gsf), [_parse_float(v) for v in xs.split(",")],
                          int(sb, 16), [_parse_float(v) for v in ys.split(",")]))
    return cases


def test_e4m3_table_matches_torch():
    raw = torch.arange(0, 0x7F, dtype=torch.int16).to(torch.uint8)
    ref = raw.view(torch.float8_e4m3fn).to(torch.float64)
    assert torch.equal(ref, nv.E4M3_VALUES)
    assert float(nv.E4M3_VALUES[0x7E]) == 448.0
    assert float(nv.E4M3_VALUES[0x01]) == 2.0 ** -9
    assert float(nv.E4M3_VALUES[0x38]) == 1.0
    assert [float(f) for f in nv.E4M3_FRACTIONS] == nv.E4M3_VALUES.tolist()


def test_e4m3_rounding_matches_torch():
    g = torch.Generator().manual_seed(11)
    vals = nv.E4M3_VALUES
    mids = (vals[1:] + vals[:-1]) / 2
    rnd = torch.exp2(torch.rand(200000, generator=g, dtype=torch.float64) * 20 - 12)
    v = torch.cat([vals, mids, rnd]).to(torch.float32)
    v = v[v <= 448.0]
    ours = nv.e4m3_round(v)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(ours, ref)
    # saturation (satfinite) above 448, where torch's cast would give NaN
    assert torch.all(nv.e4m3_round(torch.tensor([448.5, 464.0, 480.0, 1e6])) == 0x7E)


def test_e2m1_rounding_exact():
    grid = nv.E2M1_FRACTIONS
    pts = set()
    for i in range(len(grid)):
        pts.add(grid[i])
        if i:
            mid = (grid[i] + grid[i - 1]) / 2
            pts.update({mid, mid - Fraction(1, 1 << 20), mid + Fraction(1, 1 << 20)})
    pts.update({Fraction(7), Fraction(100)})
    pts = sorted(pts)
    ours = nv.e2m1_round(torch.tensor([float(p) for p in pts], dtype=torch.float64)).tolist()
    assert ours == [nv.rne_exact(p, grid) for p in pts]
    # ties go to the even code: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    t = nv.e2m1_round(torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))
    assert nv.E2M1_GRID[t.long()].tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


@pytest.mark.parametrize("case", load_hand_examples(), ids=lambda c: c[0])
def test_hand_examples(case):
    name, gsf, xs, sb, ys = case
    x = torch.tensor(xs, dtype=torch.float64)
    assert torch.equal(nv.to_bf16(x), x), "inputs must be bf16 values"
    bits, sbytes, _ = nv.quantizer_outputs(x[None, :], gsf)
    assert int(sbytes[0, 0]) == sb
    exp_bits = nv.bf16_bits(torch.tensor(ys, dtype=torch.float64))
    assert torch.equal(bits[0], exp_bits), (bits[0], exp_bits)
    if gsf == 1.0:
        e_sb, _, e_deq = nv.fake_quant_block_exact([Fraction(v) for v in xs])
        assert e_sb == sb
        assert [float(d) for d in e_deq] == [abs(y) if y == 0 else y for y in ys] or \
            [float(d) for d in e_deq] == ys


def _all_finite_bf16():
    b = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    v = b.view(torch.bfloat16).to(torch.float64)
    return v[torch.isfinite(v)]


def test_every_bf16_value_fp32_equals_fp64_unit_gsf():
    """With unit gsf the fp32 decisions equal fp64 ones for every bf16 value,
    in blocks whose amax is each of a spread of companions."""
    v = _all_finite_bf16()
    for amax in [2.0 ** -100, 0.01171875, 0.017578125, 1.0, 1.5, 3.0, 6.0, 100.0, 2688.0, 3e38]:
        x = torch.zeros(v.numel(), 16, dtype=torch.float64)
        x[:, 0] = v
        x[:, 1] = amax
        a32 = nv.fake_quant(x, 1.0, torch.float32)
        a64 = nv.fake_quant(x, 1.0, torch.float64)
        for p, q in zip(a32, a64):
            assert torch.equal(p, q)


def test_fp32_decisions_equal_exact_rationals_unit_gsf():
    """Every tie of both roundings, plus random bf16 blocks, against Fractions."""
    blocks = []
    for sb in range(1, 0x7F):
        s = float(nv.E4M3_VALUES[sb])
        # amax = 6*s gives scale s exactly; every E2M1 tie point times s
        blocks.append([6 * s, 0.25 * s, 0.75 * s, 1.25 * s, -1.75 * s, 2.5 * s, 3.5 * s, 5 * s,
                       -0.5 * s, s, 1.5 * s, 2 * s, 3 * s, -4 * s, 0.0, -0.0])
    vals = nv.E4M3_VALUES.tolist()
    for lo, hi in zip(vals[:-1], vals[1:]):
        blocks.append([3 * (lo + hi)] + [0.0] * 15)  # amax/6 exactly on a scale midpoint
    g = torch.Generator().manual_seed(5)
    rnd = nv.to_bf16(torch.randn(600, 16, generator=g) *
                     torch.exp2(torch.randint(-12, 12, (600, 1), generator=g).double()))
    blocks += rnd.tolist()
    x = nv.to_bf16(torch.tensor(blocks, dtype=torch.float64))
    assert torch.equal(x, torch.tensor(blocks, dtype=torch.float64))
    xq, sb, codes = nv.fake_quant(x, 1.0, torch.float32)
    for i, blk in enumerate(blocks):
        e_sb, e_idx, e_deq = nv.fake_quant_block_exact(blk)
        assert int(sb[i, 0]) == e_sb
        assert (codes[i] & 7).tolist() == e_idx
        assert xq[i].tolist() == [float(d) for d in e_deq]


def test_idempotence_reachable_pairs():
    """fq(fq(x)) == fq(x) for every reachable (scale, max code) pair but two.

    Reachable pairs are enumerated by quantizing a block whose max is each
    positive finite bf16 value.  The two exceptions: scale 2^-9 with max code 3
    (re-quantizing ties amax/6 = 2^-10 down to scale 0 and flushes the block),
    and scale 2^-8 with max code 4 (the new scale rounds down to 2^-9 and the
    max saturates at code 6).
    """
    b = torch.arange(1, 0x7F80, dtype=torch.int32).to(torch.int16)
    a = b.view(torch.bfloat16).to(torch.float64)
    x = torch.zeros(a.numel(), 16, dtype=torch.float64)
    x[:, 0] = a
    _, sb, codes = nv.fake_quant(x, 1.0, torch.float32)
    first = {}
    for amax, s, c in zip(a.tolist(), sb[:, 0].tolist(), (codes[:, 0] & 7).tolist()):
        if s:
            first.setdefault((s, c), amax)
    assert len(first) == 129
    exceptions = []
    for (s_b, ci), amax in sorted(first.items()):
        s = float(nv.E4M3_VALUES[s_b])
        # an input block whose max gives (s, ci); the others sit on every smaller code of s
        others = [gv * s for gv in nv.E2M1_GRID[:ci].tolist()]
        blk = torch.tensor(([amax] + others + [-m for m in others] + [0.0] * 16)[:16],
                           dtype=torch.float64)
        once, sb1, c1 = nv.fake_quant(blk, 1.0, torch.float32)
        assert int(sb1[0]) == s_b and int(c1[0]) & 7 == ci
        if not torch.equal(nv.fq(once, 1.0, torch.float32), once):
            exceptions.append((s, float(nv.E2M1_GRID[ci])))
    assert exceptions == [(2.0 ** -9, 3.0), (2.0 ** -8, 4.0)]


def test_static_gsf_power_of_two_equivariance():
    """fq(x; gsf) == fq(x * gsf; 1) / gsf, exact when gsf is a power of two."""
    g = torch.Generator().manual_seed(3)
    x = nv.to_bf16(torch.randn(2000, 16, generator=g, dtype=torch.float64) * 3)
    for k in [-6, -1, 3, 5]:
        gs = 2.0 ** k
        a, sa, ca = nv.fake_quant(x, gs, torch.float32)
        b, sb, cb = nv.fake_quant(x * gs, 1.0, torch.float32)
        assert torch.equal(sa, sb) and torch.equal(ca, cb)
        assert torch.equal(a, b / gs)


def test_static_gsf_matches_exact_except_near_ties():
    """fp32 decisions with a static gsf agree with exact-real ones except where the
    exact quotient lies within fp32 rounding of a tie (the documented reading).

    With gsf = fp32(2688/A) such near-ties are systematic, not rare: x*gsf/s is
    close to a ratio of short integers whenever x/A is, and only gsf's rounding
    error separates it from the tie.
    """
    g = torch.Generator().manual_seed(4)
    xm = nv.to_bf16(torch.randn(400, 16, generator=g, dtype=torch.float64) * 5)
    gsf = nv.global_sf(xm)
    xq, sb, codes = nv.fake_quant(xm, gsf, torch.float32)
    gf = Fraction(gsf)
    e2m1_ties = [(a + b) / 2 for a, b in zip(nv.E2M1_FRACTIONS[:-1], nv.E2M1_FRACTIONS[1:])]
    near = Fraction(1, 1 << 21)
    for i in range(xm.shape[0]):
        blk = xm[i].tolist()
        e_sb, e_idx, _ = nv.fake_quant_block_exact(blk, gf)
        assert int(sb[i, 0]) == e_sb  # no scale near-tie occurs in this sample
        s = nv.E4M3_FRACTIONS[e_sb]
        for j, (c, ce) in enumerate(zip((codes[i] & 7).tolist(), e_idx)):
            if c != ce:
                qx = abs(Fraction(blk[j])) * gf / s
                assert min(abs(qx - t) / t for t in e2m1_ties) < near, (i, j)
                assert abs(c - ce) == 1


def test_global_sf():
    x = torch.tensor([[1.0, -50.0, 3.0]])
    assert nv.global_sf(x) == float(np.float32(2688.0) / np.float32(50.0))
    assert nv.global_sf(torch.zeros(4)) == float(np.float32(2688.0 / np.float32(1e-12)))
    assert nv.global_sf(torch.tensor([6.0])) == 448.0


def test_code_packing_and_signs():
    x = torch.tensor([[6.0, -3.0, 0.25, -0.25, 2.5, -6.0] + [0.0] * 10])
    bits, sb, packed = nv.quantizer_outputs(x, 1.0)
    # codes: 6 -> 0x7, -3 -> 0xD, 0.25 -> 0x0, -0.25 -> 0x8 (negative zero), 2.5 -> 0x4, -6 -> 0xF
    assert packed[0, :3].tolist() == [0x7 | (0xD << 4), 0x0 | (0x8 << 4), 0x4 | (0xF << 4)]
    assert int(bits[0, 3]) == -32768  # bf16 -0.0 bit pattern 0x8000
    assert int(sb[0, 0]) == 0x38


def test_short_tail_block():
    """A row whose length is not a multiple of 16 ends in a short block that is
    quantized on its own elements (zero padding changes neither amax nor codes)."""
    g = torch.Generator().manual_seed(8)
    x = nv.to_bf16(torch.randn(3, 40, generator=g, dtype=torch.float64))
    a = nv.fq(x, 1.0, torch.float64)
    pad = torch.nn.functional.pad(x, (0, 8))
    b = nv.fq(pad, 1.0, torch.float64)[:, :40]
    assert torch.equal(a, b)
    e_sb, _, e_deq = nv.fake_quant_block_exact(x[1, 32:40].tolist())
    assert a[1, 32:40].tolist() == [float(d) for d in e_deq]
