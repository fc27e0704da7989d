"""The quantized operands inside the attention calls, compared with the oracle
byte for byte, and the agreement of the forward's and the backward's P~.

1. After attn_qat_fwd / attn_qat_fwd_hp / attn_qat_fwd_sparse / attn_qat_bwd the caller-owned
   workspaces hold the quantized Q, K, V at the offsets attn_qat_*_layout
   reports (include/nvfp4attn.h): the E2M1 codes and the 512-byte scale blocks
   of Q~ and K~ that feed the block-scaled FP4 MMA, V~ in f16, Q~/K~/V~ in
   bf16 (the forward's copies are what attn_qat_bwd_saved reads).  North-star
   acceptance asks for bit-exact codes and E4M3 scales on identical inputs,
   so every byte is compared with the oracle's quantizer
   ("nvfp4_qad.py", module docstring: blocks of 16, E4M3 scale, E2M1 codes),
   re-laid into the documented block layout; the padding tokens of the last
   128-token tile must carry scale 0.  The workspaces are filled with a
   non-zero pattern first, so nothing passes by being left untouched.

2. P~ = fq16(exp(S - m)) is computed twice: by the forward for O = P~ V~ / l
   and by the dK/dV kernel for dV = (P~ / l)^T dO, both from S on the same
   block-scaled FP4 MMAs (earlier forms of the dK/dV kernel formed S on BF16
   MMAs, equal up to the fp32 accumulation order), so a difference would show
   where P / s lies within rounding of an E2M1 decision ("Attn-QAT Training"
   guide, "Architecture-specific Triton routing": the exact-m statistics exist
   to keep dV consistent with the forward's P~).
   Both P~ are read out through the public calls, with no instrumentation:
   V = one-hot rows over one tile of keys makes O[i, c] = 1.03125 P~[i, j] / l_i
   (the fake-quantized one-hot block is 6 * E4M3(1/6) = 1.03125), and dO =
   one-hot rows over one tile of queries makes dV[j, c] = P~[i, j] / l_i.
   The test bounds how often they differ and checks that each difference is
   one E2M1 step at the block's scale.
"""
import pytest
import torch

from nvfp4_fake_quant_gb300 import api, workloads
from oracle import attention as oa
from oracle import nvfp4 as onv

pytestmark = pytest.mark.gpu

FILL = 0xA5  # workspace bytes before the call


def _bytes(ws, off, n):
    return ws[off:off + n].cpu()


def scale_blocks(sb, n, d):
    """Oracle scale bytes uint8 [B, N, H, D/16] re-laid into the documented
    512-byte blocks [B, H, ceil(N/128), D/64, 512] (flattened): token r of a
    tile, 16-element block j of a 64-element group at (r % 32) * 16 + (r / 32) * 4 + j;
    tokens past N keep scale 0."""
    b, _, h, _ = sb.shape
    nt = -(-n // 128)
    out = torch.zeros(b, h, nt, d // 64, 512, dtype=torch.uint8)
    tok = torch.arange(n)
    t, r = tok // 128, tok % 128
    for g in range(d // 64):
        for j in range(4):
            pos = (r % 32) * 16 + (r // 32) * 4 + j
            out[:, :, t, g, pos] = sb[:, tok, :, g * 4 + j].permute(0, 2, 1)
    return out.reshape(-1)


def oracle_fp4(x):
    """(packed codes, scale blocks) of a bf16 [B, N, H, D] tensor, per the oracle."""
    b, n, h, d = x.shape
    _, sb, codes = onv.quantizer_outputs(x.reshape(-1, d))
    return codes.reshape(-1), scale_blocks(sb.reshape(b, n, h, d // 16), n, d)


def oracle_fq_bits(x, dtype):
    """Bit patterns (int16) of the oracle's fq16 of x along D, in bf16 or f16 (exact)."""
    xq = onv.fq(x, 1.0, torch.float32, axis=-1)
    return xq.to(torch.float32).to(dtype).view(torch.int16).reshape(-1)


def check_fp4(ws, lay, name, x):
    codes, blocks = oracle_fp4(x)
    got_c = _bytes(ws, lay[f"{name}_codes"], codes.numel())
    got_s = _bytes(ws, lay[f"{name}_scales"], blocks.numel())
    bad_c = int((got_c != codes).sum())
    bad_s = int((got_s != blocks).sum())
    assert bad_c == 0, f"{name} codes: {bad_c} of {codes.numel()} bytes differ"
    assert bad_s == 0, f"{name} scale blocks: {bad_s} of {blocks.numel()} bytes differ"


def check_16bit(ws, off, x, dtype, what):
    want = oracle_fq_bits(x, dtype)
    got = _bytes(ws, off, 2 * want.numel()).view(torch.int16)
    bad = int((got != want).sum())
    assert bad == 0, f"{what}: {bad} of {want.numel()} values differ"


CASES = [
    # B, Nq, Nkv, H, D, causal, seed
    (1, 256, 256, 2, 64, False, 0),     # the tiny configuration
    (2, 300, 300, 3, 128, False, 10),   # ragged: 44 padding tokens in the last tile
    (1, 200, 333, 2, 128, False, 11),   # cross attention, Nq != Nkv
    (1, 17, 15, 1, 64, False, 14),      # one partial tile
    (1, 520, 520, 2, 128, True, 17),    # causal, lognormal channel scales
]


def _inputs(case):
    b, nq, nkv, h, d, causal, seed = case
    dist = "lognormal_channels" if seed == 17 else "normal"
    inp = workloads.attn_inputs(b, nq, nkv, h, d, seed, causal=causal, dist=dist)
    return inp, (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])))
def test_forward_workspace_operands_are_bit_exact(case):
    b, nq, nkv, h, d, causal, _ = case
    inp, (q, k, v, _do) = _inputs(case)
    lay = api.attn_qat_layout(b, nq, nkv, h, d, "fwd")
    ws = torch.empty((lay["total"],), dtype=torch.uint8, device="cuda")
    # both dense forwards leave every form of Q~, K~, V~ the backward reads
    for fwd in (api.attn_qat_fwd, api.attn_qat_fwd_hp):
        ws.fill_(FILL)
        fwd(q, k, v, inp.scale, causal, workspace=ws)
        assert api.device_status() == 0
        check_fp4(ws, lay, "q", inp.q)
        check_fp4(ws, lay, "k", inp.k)
        check_16bit(ws, lay["v_f16"], inp.v, torch.float16, "V~ (f16)")
        check_16bit(ws, lay["q_bf16"], inp.q, torch.bfloat16, "Q~ (bf16)")
        check_16bit(ws, lay["k_bf16"], inp.k, torch.bfloat16, "K~ (bf16)")
        check_16bit(ws, lay["v_bf16"], inp.v, torch.bfloat16, "V~ (bf16)")


@pytest.mark.parametrize("b,n_tiles,h,d,topk,seed", [(1, 3, 2, 128, 2, 30), (2, 2, 3, 64, 1, 31)])
def test_sparse_forward_workspace_operands_are_bit_exact(b, n_tiles, h, d, topk, seed):
    """The block-sparse forward leaves the same forms as the dense ones (what
    attn_qat_bwd_sparse_saved reads), whatever tiles the lists select."""
    n = n_tiles * 128
    inp = workloads.attn_inputs(b, n, n, h, d, seed)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    tiles = api.vsa_select_tiles(q, k, topk)
    lay = api.attn_qat_layout(b, n, n, h, d, "fwd")
    ws = torch.full((lay["total"],), FILL, dtype=torch.uint8, device="cuda")
    api.attn_qat_fwd_sparse(q, k, v, tiles, inp.scale, workspace=ws)
    assert api.device_status() == 0
    check_fp4(ws, lay, "q", inp.q)
    check_fp4(ws, lay, "k", inp.k)
    check_16bit(ws, lay["v_f16"], inp.v, torch.float16, "V~ (f16)")
    check_16bit(ws, lay["q_bf16"], inp.q, torch.bfloat16, "Q~ (bf16)")
    check_16bit(ws, lay["k_bf16"], inp.k, torch.bfloat16, "K~ (bf16)")
    check_16bit(ws, lay["v_bf16"], inp.v, torch.bfloat16, "V~ (bf16)")


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])))
def test_backward_workspace_operands_are_bit_exact(case):
    b, nq, nkv, h, d, causal, _ = case
    inp, (q, k, v, do) = _inputs(case)
    o, stats = api.attn_qat_fwd(q, k, v, inp.scale, causal)
    lay = api.attn_qat_layout(b, nq, nkv, h, d, "bwd")
    ws = torch.full((lay["total"],), FILL, dtype=torch.uint8, device="cuda")
    api.attn_qat_bwd(q, k, v, o, stats, do, inp.scale, causal, workspace=ws)
    assert api.device_status() == 0
    check_fp4(ws, lay, "q", inp.q)
    check_fp4(ws, lay, "k", inp.k)
    check_16bit(ws, lay["q_bf16"], inp.q, torch.bfloat16, "Q~ (bf16)")
    check_16bit(ws, lay["k_bf16"], inp.k, torch.bfloat16, "K~ (bf16)")
    check_16bit(ws, lay["v_bf16"], inp.v, torch.bfloat16, "V~ (bf16)")
    # delta = rowsum(dO * o), f32 [B, H, Nq]
    delta = _bytes(ws, lay["delta"], 4 * b * h * nq).view(torch.float32).double()
    want = (inp.do.double() * o.cpu().double()).sum(-1).permute(0, 2, 1).reshape(-1)
    mag = (inp.do.double().abs() * o.cpu().double().abs()).sum(-1).permute(0, 2, 1).reshape(-1)
    assert bool(((delta - want).abs() <= 1e-5 * mag + 1e-30).all())


# ------------------------------------------------------------------ P~ agreement

C_ONEHOT = 1.03125  # fq16 of a block holding one 1.0 and zeros: 6 * E4M3(1/6)


def _onehot(b, n, h, d, t, device="cuda"):
    """bf16 [B, n, H, d]: row t*d + c is e_c for c < d (rows of tile t), others 0."""
    x = torch.zeros(b, n, h, d, dtype=torch.bfloat16, device=device)
    rows = torch.arange(t * d, min(n, (t + 1) * d), device=device)
    x[:, rows, :, rows - t * d] = 1.0
    return x, rows.cpu()


def forward_ptilde(q, k, scale, causal):
    """P~ / l as the forward applies it, [B, H, Nq, Nkv] float64 (bf16-rounded),
    and the forward's stats (identical for every V)."""
    b, nq, h, d = q.shape
    nkv = k.shape[1]
    out = torch.zeros(b, h, nq, nkv, dtype=torch.float64)
    stats0 = None
    for t in range(-(-nkv // d)):
        v, rows = _onehot(b, nkv, h, d, t)
        o, stats = api.attn_qat_fwd(q, k, v, scale, causal)
        if stats0 is None:
            stats0 = stats
        assert torch.equal(stats, stats0)  # the statistics do not depend on V
        out[:, :, :, rows] = o[:, :, :, :len(rows)].permute(0, 2, 1, 3).cpu().double() / C_ONEHOT
    return out, stats0


def backward_ptilde(q, k, v, o, stats, scale, causal):
    """P~ / l as the dK/dV kernel applies it (dV = (P~/l)^T dO), [B, H, Nq, Nkv]."""
    b, nq, h, d = q.shape
    nkv = k.shape[1]
    out = torch.zeros(b, h, nq, nkv, dtype=torch.float64)
    for u in range(-(-nq // d)):
        do, rows = _onehot(b, nq, h, d, u)
        _, _, dv = api.attn_qat_bwd(q, k, v, o, stats, do, scale, causal)
        out[:, :, rows, :] = dv[:, :, :, :len(rows)].permute(0, 2, 3, 1).cpu().double()
    return out


def differ(a, b):
    """True where two bf16 roundings of P~/l cannot come from the same P~ (the
    nearest distinct P~ values are >= 2.3% apart; two roundings differ <= 0.8%)."""
    return (a - b).abs() > 2.0 ** -6 * torch.maximum(a.abs(), b.abs())


GRID = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)


def grid_index(c):
    """Index of the E2M1 grid value nearest to c >= 0 and whether c lies within 1% of it."""
    idx = (c[..., None] - GRID).abs().argmin(-1)
    g = GRID[idx]
    return idx, (c - g).abs() <= 0.01 * torch.maximum(g, torch.full_like(g, 0.5))


PT_CASES = [
    # B, N, H, D, causal, seed, scale
    (1, 256, 2, 64, False, 0, 1 / 8),      # the tiny configuration
    (1, 300, 1, 128, False, 10, None),     # ragged, D = 128
    (1, 200, 1, 64, True, 12, None),       # causal
]
MAX_DIFF_FRAC = 1e-3


@pytest.mark.parametrize("case", PT_CASES, ids=lambda c: "x".join(map(str, c[:4])))
def test_forward_and_backward_ptilde_agree(case):
    b, n, h, d, causal, seed, scale = case
    inp = workloads.attn_inputs(b, n, n, h, d, seed, scale=scale, causal=causal)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    pf, stats = forward_ptilde(q, k, inp.scale, causal)
    o, stats2 = api.attn_qat_fwd(q, k, v, inp.scale, causal)
    assert torch.equal(stats, stats2)
    pb = backward_ptilde(q, k, v, o, stats, inp.scale, causal)
    assert api.device_status() == 0
    st = stats.cpu().double()
    l = torch.exp(st[:, :, 0] - st[:, :, 1])[..., None]  # l = exp(LSE - m), [B, H, N, 1]
    pt_f, pt_b = pf * l, pb * l                            # P~ (to ~2^-8 relative)

    # oracle P~ and its block scales, for the step check and as a second witness
    pt_o = torch.zeros_like(pf)
    s_o = torch.zeros(b, h, n, -(-n // 16), dtype=torch.float64)
    for bb in range(b):
        for hh in range(h):
            hp = oa.HeadProblem(inp.q, inp.k, inp.v, bb, hh, inp.scale, causal)
            _, _, _, pt, sb = hp.probs_rows(torch.arange(n))
            pt_o[bb, hh] = pt
            s_o[bb, hh] = onv.E4M3_VALUES[sb.long()]

    d_fb = differ(pf, pb)
    d_fo = differ(pt_f, pt_o)
    d_bo = differ(pt_b, pt_o)
    total = pf.numel()
    print(f"P~ elements {total}: fwd!=bwd {int(d_fb.sum())}, fwd!=oracle {int(d_fo.sum())}, "
          f"bwd!=oracle {int(d_bo.sum())}")
    assert float(d_fb.sum()) <= MAX_DIFF_FRAC * total
    assert float(d_fo.sum()) <= MAX_DIFF_FRAC * total
    assert float(d_bo.sum()) <= MAX_DIFF_FRAC * total
    # every difference between the forward and the backward is one E2M1 step
    # at the block's scale
    idx = d_fb.nonzero(as_tuple=True)
    if idx[0].numel():
        s = s_o[idx[0], idx[1], idx[2], idx[3] // 16]
        cf, okf = grid_index(pt_f[idx] / s)
        cb, okb = grid_index(pt_b[idx] / s)
        assert bool(okf.all()) and bool(okb.all()), (pt_f[idx], pt_b[idx], s)
        assert bool(((cf - cb).abs() == 1).all()), (cf, cb)


@pytest.mark.parametrize("case", PT_CASES, ids=lambda c: "x".join(map(str, c[:4])))
def test_auxiliary_output_forward_ptilde_agrees(case):
    """The auxiliary-output forward ("use_high_prec_o") forms pass 2's S from 64-key FP4
    UMMAs (its half tiles) and the dense forward from 128-key ones: the row maxima must
    be the same bits, and the P~ that its o applies must be the dense forward's and the
    oracle's up to the same bounded, one-E2M1-step differences (l may differ in the
    last bits: its fp32 sums run in another order)."""
    b, n, h, d, causal, seed, scale = case
    inp = workloads.attn_inputs(b, n, n, h, d, seed, scale=scale, causal=causal)
    q, k = inp.q.cuda(), inp.k.cuda()
    pf, stats = forward_ptilde(q, k, inp.scale, causal)
    ph = torch.zeros_like(pf)
    stats_h = None
    for t in range(-(-n // d)):
        v, rows = _onehot(b, n, h, d, t)
        o, _, st = api.attn_qat_fwd_hp(q, k, v, inp.scale, causal)
        if stats_h is None:
            stats_h = st
        assert torch.equal(st, stats_h)  # the statistics do not depend on V
        ph[:, :, :, rows] = o[:, :, :, :len(rows)].permute(0, 2, 1, 3).cpu().double() / C_ONEHOT
    assert api.device_status() == 0
    assert torch.equal(stats_h[:, :, 1], stats[:, :, 1])  # m
    st_f, st_h = stats.cpu().double(), stats_h.cpu().double()
    pt_f = pf * torch.exp(st_f[:, :, 0] - st_f[:, :, 1])[..., None]
    pt_h = ph * torch.exp(st_h[:, :, 0] - st_h[:, :, 1])[..., None]

    pt_o = torch.zeros_like(pf)
    s_o = torch.zeros(b, h, n, -(-n // 16), dtype=torch.float64)
    for bb in range(b):
        for hh in range(h):
            hp = oa.HeadProblem(inp.q, inp.k, inp.v, bb, hh, inp.scale, causal)
            _, _, _, pt, sb = hp.probs_rows(torch.arange(n))
            pt_o[bb, hh] = pt
            s_o[bb, hh] = onv.E4M3_VALUES[sb.long()]
    d_fh = differ(pt_f, pt_h)
    d_ho = differ(pt_h, pt_o)
    total = pf.numel()
    print(f"P~ elements {total}: dense!=aux {int(d_fh.sum())}, aux!=oracle {int(d_ho.sum())}")
    assert float(d_fh.sum()) <= MAX_DIFF_FRAC * total
    assert float(d_ho.sum()) <= MAX_DIFF_FRAC * total
    idx = d_fh.nonzero(as_tuple=True)
    if idx[0].numel():
        s = s_o[idx[0], idx[1], idx[2], idx[3] // 16]
        cf, okf = grid_index(pt_f[idx] / s)
        ch, okh = grid_index(pt_h[idx] / s)
        assert bool(okf.all()) and bool(okh.all()), (pt_f[idx], pt_h[idx], s)
        assert bool(((cf - ch).abs() == 1).all()), (cf, ch)
