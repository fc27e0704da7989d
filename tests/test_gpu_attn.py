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
    # 13 key tiles (ragged last): pass-1 tiles unevenly over the four warpgroups,
    # barrier and scale-copy indices past their first wrap
    ("thirteen_tiles", 1, 1650, 1650, 1, 128, False, 18, "unit_rms", None),
    ("thirteen_tiles_causal", 1, 1650, 1650, 1, 64, True, 19, "normal", None),
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
    assert torch.equal(dq1, qq.grad)  # no atomics anywhere: the backward is deterministic


def test_calls_from_a_thread_without_a_current_context():
    """The C ABI works from a host thread that has made no CUDA call yet (such a
    thread has no current context; tensor-map encoding needs one).  Framework
    worker threads, such as the autograd engine's, are like that.  All buffers
    are allocated here; the new thread only calls the library."""
    import threading

    from nvfp4_fake_quant_gb300 import _lib

    inp = workloads.attn_inputs(1, 256, 256, 2, 128, seed=22)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    b, n, h, d = q.shape
    o_ref, s_ref = api.attn_qat_fwd(q, k, v, inp.scale)
    g_ref = api.attn_qat_bwd(q, k, v, o_ref, s_ref, do, inp.scale)
    o, stats = torch.empty_like(q), torch.empty_like(s_ref)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(api.attn_qat_fwd_workspace(b, n, n, h, d),
                         api.attn_qat_bwd_workspace(b, n, n, h, d)), dtype=torch.uint8,
                     device="cuda")
    torch.cuda.synchronize()
    lib = _lib.load()
    result = {}

    def worker():
        nb = ws.numel()
        result["fwd"] = lib.attn_qat_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), b, n, n, h, d,
                                         inp.scale, 0, o.data_ptr(), stats.data_ptr(),
                                         ws.data_ptr(), nb, None)
        result["bwd"] = lib.attn_qat_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         stats.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                         dk.data_ptr(), dv.data_ptr(), b, n, n, h, d, inp.scale, 0,
                                         ws.data_ptr(), nb, None)
        result["detail"] = lib.nvq_last_error_detail().decode()
        result["sync"] = lib.nvq_device_status(None)

    th = threading.Thread(target=worker)
    th.start()
    th.join()
    assert (result["fwd"], result["bwd"], result["sync"]) == (0, 0, 0), result
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(stats, s_ref)
    for g, r in zip((dq, dk, dv), g_ref):
        assert torch.equal(g, r)


def test_kernel_timing_hook_counts_every_launch():
    """nvq_timing_* files each launch of a forward + backward under its kernel
    kind, with a positive device time that fits inside the calls' wall time."""
    import time
    inp = workloads.attn_inputs(1, 384, 384, 2, 128, seed=23)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, stats = api.attn_qat_fwd(q, k, v, inp.scale)
    torch.cuda.synchronize()
    api.timing_enable(True)
    try:
        t0 = time.perf_counter()
        o, stats = api.attn_qat_fwd(q, k, v, inp.scale)
        api.attn_qat_bwd(q, k, v, o, stats, do, inp.scale)
        torch.cuda.synchronize()
        wall_ms = (time.perf_counter() - t0) * 1e3
        got = api.timing_read()
    finally:
        api.timing_enable(False)
    # one fused quantizer launch per call (q, k, v in every form the call reads)
    assert {k: n for k, (n, _) in got.items()} == {
        "quantize": 2, "attn_fwd": 1, "bwd_delta": 1, "bwd_dkdv": 1, "bwd_dq": 1, "global_sf": 0,
        "vsa": 0, "linear": 0}
    assert all(ms > 0 for n, ms in got.values() if n)
    assert sum(ms for _, ms in got.values()) <= wall_ms
    assert api.timing_read()["attn_fwd"] == (0, 0.0)  # disabled: records discarded


SAVED_CASES = [c for c in CASES if c[0] in ("tiny_config", "ragged_d128", "cross_d128",
                                            "causal_d64", "short", "thirteen_tiles")]


@pytest.mark.parametrize("case", SAVED_CASES, ids=lambda c: c[0])
def test_saved_operand_backward_matches(case):
    """attn_qat_bwd_saved reads the quantized operands the forward left in its
    workspace; its gradients equal attn_qat_bwd's (which quantizes q, k, v
    itself) bit for bit, after attn_qat_fwd and after attn_qat_fwd_hp."""
    name, b, nq, nkv, h, d, causal, seed, dist, scale = case
    inp = workloads.attn_inputs(b, nq, nkv, h, d, seed, scale=scale, causal=causal, dist=dist)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    saved = torch.full((api.attn_qat_fwd_workspace(b, nq, nkv, h, d),), 0x5A, dtype=torch.uint8,
                       device="cuda")
    o, stats = api.attn_qat_fwd(q, k, v, inp.scale, causal, workspace=saved)
    ref = api.attn_qat_bwd(q, k, v, o, stats, do, inp.scale, causal)
    got = api.attn_qat_bwd_saved(saved, o, stats, do, inp.scale, causal, nkv=nkv)
    assert api.device_status() == 0
    for n_, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(g, r), n_
    saved.fill_(0xA5)
    o2, o_hp, stats2 = api.attn_qat_fwd_hp(q, k, v, inp.scale, causal, workspace=saved)
    ref = api.attn_qat_bwd(q, k, v, o_hp, stats2, do, inp.scale, causal)
    got = api.attn_qat_bwd_saved(saved, o_hp, stats2, do, inp.scale, causal, nkv=nkv)
    assert api.device_status() == 0
    for n_, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(g, r), n_
