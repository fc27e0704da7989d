"""The allocation-free backward, attn_qat_bwd_builtin_scratch, called through
the C ABI and compared with attn_qat_bwd.

That entry point is for callers that cannot allocate device memory (code inside
a framework that owns all device memory, or on a path where cudaMalloc would
synchronize the device); its scratch is a fixed 32 MiB array in the library,
shared by every call.  The test runs it twice in a row on different problems,
so a second call that depended on stale scratch contents would fail, and checks
that a problem too large for the array is rejected.  This file is collected last on purpose.
"""
import pytest
import torch

from nvfp4_fake_quant_gb300 import _lib, api, workloads

pytestmark = pytest.mark.gpu

G_RTOL = 2e-2  # the gradient tolerance of the attention parity tests
WORKSPACE = 3  # NVQ_ERR_WORKSPACE


def rel_l2(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b).clamp_min(1e-30))


def _builtin_bwd(q, k, v, o, stats, do, scale, causal):
    b, nq, h, d = q.shape
    nkv = k.shape[1]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = _lib.load().attn_qat_bwd_builtin_scratch(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), stats.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), b, nq, nkv, h, d, scale, int(causal),
        torch.cuda.current_stream().cuda_stream)
    return st, (dq, dk, dv)


@pytest.mark.parametrize("shapes", [[(1, 256, 256, 2, 64, False, 0), (2, 300, 300, 3, 128, True, 1)]])
def test_builtin_scratch_backward_matches_workspace_backward(shapes):
    for (b, nq, nkv, h, d, causal, seed) in shapes:  # two calls in a row
        inp = workloads.attn_inputs(b, nq, nkv, h, d, seed)
        q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
        o, stats = api.attn_qat_fwd(q, k, v, inp.scale, causal)
        ref = api.attn_qat_bwd(q, k, v, o, stats, do, inp.scale, causal)
        st, got = _builtin_bwd(q, k, v, o, stats, do, inp.scale, causal)
        assert st == 0, _lib.STATUS.get(st, st)
        assert api.device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert rel_l2(g, r) <= G_RTOL, (name, rel_l2(g, r))


def test_builtin_scratch_rejects_problems_over_the_limit():
    b, n, h, d = 1, 16384, 4, 128  # needs about 50 MB of scratch (> 32 MiB)
    assert api.attn_qat_bwd_workspace(b, n, n, h, d) > (32 << 20)
    x = torch.zeros(b, n, h, d, dtype=torch.bfloat16, device="cuda")
    stats = torch.zeros(b, h, 2, n, dtype=torch.float32, device="cuda")
    st, _ = _builtin_bwd(x, x, x, x, stats, x, 0.1, False)
    assert st == WORKSPACE
