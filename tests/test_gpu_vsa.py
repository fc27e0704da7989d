"""Block-sparse (VSA) path on the GPU against the oracle, through the C ABI:

- token reordering between raster and cube order: bit-exact, both directions;
- block selection: the kernel takes fp32 cube means and scores, the oracle
  float64, so a selection may differ from the oracle's only between tiles whose
  float64 scores are within float32 rounding of each other; it is checked for
  that validity, and for exact agreement on exact ties;
- block-sparse attention forward and backward, element by element at the dense
  tolerances, with the GPU's own selection (or a hand-built list) given to both
  sides; key tiles that no query tile selects get exactly zero dK and dV;
- the config-5 workload (Wan latent 16x28x56, 196 cubes, top-20) at full size,
  on sampled rows and key columns of two heads.
"""
import pytest
import torch

from nvfp4_fake_quant_gb300 import api, workloads
from oracle import attention as oa
from oracle import nvfp4 as onv
from oracle import vsa as ov

pytestmark = pytest.mark.gpu

O_RTOL, O_ATOL, G_RTOL, LSE_ATOL = 1e-2, 5e-2, 2e-2, 2e-3


def rel_l2(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b).clamp_min(1e-30))


def test_reorder_matches_the_oracle_and_round_trips():
    g = torch.Generator().manual_seed(40)
    x = torch.randn(2, 8 * 8 * 16, 3, 64, generator=g).to(torch.bfloat16)
    c = api.vsa_reorder(x.cuda(), (8, 8, 16))
    assert torch.equal(c.cpu(), ov.to_cubes(x, 8, 8, 16))
    back = api.vsa_reorder(c, (8, 8, 16), to_cubes=False)
    assert torch.equal(back.cpu(), x)
    assert api.device_status() == 0


def check_selection(got, q, k, topk, tol_rel=1e-5):
    """Every list is ascending, distinct and in range, and is a top-k of the
    float64 scores up to float32 rounding.  Returns the rows that differ from
    the oracle's selection."""
    s = ov.cube_scores(q, k)
    ref = ov.select_tiles(q, k, topk)
    got = got.cpu().long()
    b, h, n, _ = s.shape
    tol = tol_rel * (float(s.abs().max()) + 1.0)
    differ = 0
    for bi in range(b):
        for hi in range(h):
            for i in range(n):
                g = got[bi, hi, i]
                assert bool((g[1:] > g[:-1]).all()) and int(g.min()) >= 0 and int(g.max()) < n
                if torch.equal(g, ref[bi, hi, i]):
                    continue
                differ += 1
                sel = torch.zeros(n, dtype=torch.bool)
                sel[g] = True
                row = s[bi, hi, i]
                assert float(row[sel].min()) >= float(row[~sel].max()) - tol, (bi, hi, i)
    return differ


def test_selection_is_a_valid_top_k():
    inp = workloads.attn_inputs(1, 128 * 12, 128 * 12, 2, 128, seed=41)
    q, k = inp.q.cuda(), inp.k.cuda()
    tiles = api.vsa_select_tiles(q, k, 3)
    assert api.device_status() == 0
    assert check_selection(tiles, inp.q, inp.k, 3) <= 2


def test_selection_ties_go_to_the_lower_index():
    q = torch.ones(1, 128 * 5, 1, 64, dtype=torch.bfloat16)
    k = torch.ones(1, 128 * 5, 1, 64, dtype=torch.bfloat16)
    tiles = api.vsa_select_tiles(q.cuda(), k.cuda(), 2)
    assert tiles.cpu().tolist() == [[[[0, 1]] * 5]]
    k[0, 384:512] = 2.0  # tile 3 scores highest everywhere
    tiles = api.vsa_select_tiles(q.cuda(), k.cuda(), 2)
    assert tiles.cpu().tolist() == [[[[0, 3]] * 5]]


def _parity(inp, tiles):
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, stats = api.attn_qat_fwd_sparse(q, k, v, tiles, inp.scale)
    dq, dk, dv = api.attn_qat_bwd_sparse(q, k, v, o, stats, do, tiles, inp.scale)
    assert api.device_status() == 0
    kvt = tiles.cpu().long()
    o_ref, lse_ref, m_ref = oa.attn_fwd(inp.q, inp.k, inp.v, inp.scale, kv_tiles=kvt)
    g_ref = oa.attn_bwd(inp.q, inp.k, inp.v, onv.to_bf16(o_ref), inp.do, inp.scale, kv_tiles=kvt)
    st = stats.cpu().double()
    errs = {"o": rel_l2(o, o_ref), "o_maxabs": float((o.cpu().double() - o_ref).abs().max()),
            "lse": float((st[:, :, 0] - lse_ref).abs().max()),
            "dq": rel_l2(dq, g_ref[0]), "dk": rel_l2(dk, g_ref[1]), "dv": rel_l2(dv, g_ref[2])}
    assert errs["o"] <= O_RTOL and errs["o_maxabs"] <= O_ATOL and errs["lse"] <= LSE_ATOL, errs
    assert all(errs[n] <= G_RTOL for n in ("dq", "dk", "dv")), errs
    return dk.cpu(), dv.cpu()


@pytest.mark.parametrize("b,n_tiles,h,d,topk,seed", [(1, 6, 2, 128, 2, 42), (2, 5, 3, 64, 3, 43),
                                                     (1, 4, 1, 128, 1, 44), (1, 3, 2, 128, 3, 45)])
def test_block_sparse_parity_with_the_gpu_selection(b, n_tiles, h, d, topk, seed):
    n = n_tiles * 128
    inp = workloads.attn_inputs(b, n, n, h, d, seed)
    tiles = api.vsa_select_tiles(inp.q.cuda(), inp.k.cuda(), topk)
    _parity(inp, tiles)


def test_hand_built_lists_and_unselected_key_tiles():
    """Lists in descending order; key tiles 2 and 3 are selected by no query tile."""
    inp = workloads.attn_inputs(1, 512, 512, 2, 128, seed=46)
    tiles = torch.tensor([[[1, 0]] * 4, [[0, 1]] * 4], dtype=torch.int32).reshape(1, 2, 4, 2)
    dk, dv = _parity(inp, tiles.cuda())
    assert bool((dk[:, 256:] == 0).all()) and bool((dv[:, 256:] == 0).all())


@pytest.mark.parametrize("b,n_tiles,h,d,topk,seed", [(1, 6, 2, 128, 2, 47), (2, 5, 3, 64, 3, 48)])
def test_sparse_saved_operand_backward_matches(b, n_tiles, h, d, topk, seed):
    """attn_qat_bwd_sparse_saved reads the operands attn_qat_fwd_sparse left in its
    workspace; its gradients equal attn_qat_bwd_sparse's bit for bit."""
    n = n_tiles * 128
    inp = workloads.attn_inputs(b, n, n, h, d, seed)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    tiles = api.vsa_select_tiles(q, k, topk)
    saved = torch.full((api.attn_qat_fwd_workspace(b, n, n, h, d),), 0x5A, dtype=torch.uint8,
                       device="cuda")
    o, stats = api.attn_qat_fwd_sparse(q, k, v, tiles, inp.scale, workspace=saved)
    ref = api.attn_qat_bwd_sparse(q, k, v, o, stats, do, tiles, inp.scale)
    got = api.attn_qat_bwd_sparse_saved(saved, o, stats, do, tiles, inp.scale)
    assert api.device_status() == 0
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(g, r), name


def _sample(n, count, seed):
    g = torch.Generator().manual_seed(seed)
    fixed = [0, 1, 127, 128, 129, 255, 256, n // 2, n - 129, n - 128, n - 2, n - 1]
    rnd = torch.randint(0, n, (count,), generator=g).tolist()
    return sorted({i for i in fixed + rnd if 0 <= i < n})


def test_config5_fullsize_sampled_parity():
    """The config-5 workload: raster tokens -> cube order, top-20 of 196 key cubes,
    block-sparse forward and backward, sampled against the oracle for heads 0, 11."""
    inp = workloads.vsa25088()
    grid = workloads.VSA_GRID
    b, n, _, h, d = inp.shape
    topk = api.vsa_effective_topk(0.9, n // 128)
    assert topk == 20
    qc, kc, vc, doc = (api.vsa_reorder(t.cuda(), grid) for t in (inp.q, inp.k, inp.v, inp.do))
    tiles = api.vsa_select_tiles(qc, kc, topk)
    o, stats = api.attn_qat_fwd_sparse(qc, kc, vc, tiles, inp.scale)
    g = torch.Generator().manual_seed(98)
    o_syn = (0.05 * torch.randn(b, n, h, d, generator=g)).to(torch.bfloat16)
    dq, dk, dv = api.attn_qat_bwd_sparse(qc, kc, vc, o_syn.cuda(), stats, doc, tiles, inp.scale)
    assert api.device_status() == 0
    q_c, k_c, v_c, do_c = (x.cpu() for x in (qc, kc, vc, doc))
    assert torch.equal(q_c, ov.to_cubes(inp.q, *grid))
    kvt = tiles.cpu().long()
    rows, cols = _sample(n, 30, 3), _sample(n, 16, 4)
    o_h, st_c = o.cpu(), stats.cpu().double()
    for hh in (0, 11):
        sl = slice(hh, hh + 1)
        assert check_selection(tiles[:, sl], q_c[:, :, sl], k_c[:, :, sl], topk) <= 4
        hp = oa.HeadProblem(q_c[:, :, sl], k_c[:, :, sl], v_c[:, :, sl], 0, 0, inp.scale,
                            kv_tiles=kvt[:, sl])
        o_ref, lse_ref, _ = hp.fwd_rows(rows)
        assert rel_l2(o_h[0, rows, hh], o_ref) <= O_RTOL
        assert float((st_c[0, hh, 0, rows] - lse_ref).abs().max()) <= LSE_ATOL
        do_hd, o_hd = do_c[0, :, hh].double(), o_syn[0, :, hh].double()
        dq_ref = hp.dq_rows(rows, o_hd[rows], do_hd[rows])
        assert rel_l2(dq.cpu()[0, rows, hh], dq_ref) <= G_RTOL
        dk_ref, dv_ref = hp.dkdv_cols(cols, o_hd, do_hd, block=1024)
        assert rel_l2(dk.cpu()[0, cols, hh], dk_ref) <= G_RTOL
        assert rel_l2(dv.cpu()[0, cols, hh], dv_ref) <= G_RTOL


@pytest.mark.parametrize("b,n_tiles,h,d,seed", [(1, 5, 2, 128, 60), (2, 3, 3, 64, 61)])
def test_full_lists_equal_the_dense_calls(b, n_tiles, h, d, seed):
    """With every query tile listing all key tiles in order, the block-sparse calls
    visit the same key tiles in the same order as the dense ones, through the same
    kernels' block-sparse instances: o, stats, dq, dk and dv must be the same bits."""
    n = 128 * n_tiles
    inp = workloads.attn_inputs(b, n, n, h, d, seed)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    tiles = torch.arange(n_tiles, dtype=torch.int32, device="cuda")
    kv = tiles.expand(b, h, n_tiles, n_tiles).contiguous()
    o_s, st_s = api.attn_qat_fwd_sparse(q, k, v, kv, inp.scale)
    o_d, st_d = api.attn_qat_fwd(q, k, v, inp.scale, False)
    assert api.device_status() == 0
    assert torch.equal(o_s, o_d)
    assert torch.equal(st_s, st_d)
    g_s = api.attn_qat_bwd_sparse(q, k, v, o_s, st_s, do, kv, inp.scale)
    g_d = api.attn_qat_bwd(q, k, v, o_d, st_d, do, inp.scale, False)
    assert api.device_status() == 0
    for name, x, y in zip(("dq", "dk", "dv"), g_s, g_d):
        assert torch.equal(x, y), name
