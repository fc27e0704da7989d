"""The allocation-free backward, attn_qat_bwd_builtin_scratch, called through
the C ABI and compared with attn_qat_bwd.

That entry point is for callers that cannot allocate device memory (code inside
a framework that owns all device memory and gives plug-ins no allocator, or on a
path where cudaMalloc would synchronize the device); its scratch is a fixed
32 MiB array in the library, shared by every call.  The backward is
deterministic, so the two entry points must agree bit for bit.  The larger
problem runs first: the second, smaller call then finds the array full of the
first call's bytes (not load-time zeros) at the offsets it uses, and must not
depend on them.  Both problems have ragged token counts (N % 128 != 0), so the
zero scales of the padding tokens are covered.  This file is collected last on
purpose, so a run that stops at the first failure has run every other test.
"""
import pytest
import torch

from nvfp4_fake_quant_gb300 import _lib, api, workloads

pytestmark = pytest.mark.gpu

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
LIMIT = 32 << 20  # bytes of the built-in scratch array


def _builtin_bwd(q, k, v, o, stats, do, scale, causal, d=None, grads=None):
    b, nq, h, dd = q.shape
    nkv = k.shape[1]
    dq, dk, dv = grads if grads is not None else \
        (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    st = _lib.load().attn_qat_bwd_builtin_scratch(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), stats.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), b, nq, nkv, h, dd if d is None else d, scale,
        int(causal), torch.cuda.current_stream().cuda_stream)
    return st, (dq, dk, dv)


# (B, Nq, Nkv, H, D, causal, seed): the larger problem first
PROBLEMS = [(1, 1000, 1000, 8, 128, False, 30), (2, 300, 300, 3, 64, True, 31)]


def test_builtin_scratch_backward_matches_workspace_backward():
    assert api.attn_qat_bwd_workspace(*PROBLEMS[0][:5]) > \
        2 * api.attn_qat_bwd_workspace(*PROBLEMS[1][:5])
    for (b, nq, nkv, h, d, causal, seed) in PROBLEMS:  # two calls in a row
        assert api.attn_qat_bwd_workspace(b, nq, nkv, h, d) <= LIMIT
        inp = workloads.attn_inputs(b, nq, nkv, h, d, seed, causal=causal)
        q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
        o, stats = api.attn_qat_fwd(q, k, v, inp.scale, causal)
        ref = api.attn_qat_bwd(q, k, v, o, stats, do, inp.scale, causal)
        st, got = _builtin_bwd(q, k, v, o, stats, do, inp.scale, causal)
        assert st == OK, _lib.STATUS.get(st, st)
        assert api.device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g, r), name


def test_builtin_scratch_rejects_before_launching():
    b, n, h, d = 1, 16384, 4, 128  # needs about 50 MB of scratch (> 32 MiB)
    assert api.attn_qat_bwd_workspace(b, n, n, h, d) > LIMIT
    x = torch.zeros(b, n, h, d, dtype=torch.bfloat16, device="cuda")
    stats = torch.zeros(b, h, 2, n, dtype=torch.float32, device="cuda")
    grads = tuple(torch.full_like(x, 7.0) for _ in range(3))
    torch.cuda.synchronize()
    assert _builtin_bwd(x, x, x, x, stats, x, 0.1, False, grads=grads)[0] == WORKSPACE
    # argument errors take precedence over the size limit, as in attn_qat_bwd
    assert _builtin_bwd(x, x, x, x, stats, x, 0.1, False, d=256, grads=grads)[0] == UNSUPPORTED
    assert _builtin_bwd(x, x, x, x, stats, x, -1.0, False, grads=grads)[0] == INVALID
    assert _builtin_bwd(x, x, x, x, stats, x, 0.1, 2, grads=grads)[0] == INVALID
    # nothing was launched or written
    assert api.device_status() == 0
    for g in grads:
        assert bool((g == 7.0).all())
