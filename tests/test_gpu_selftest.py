"""GPU checks of the hardware encodings the attention kernels rely on (tcgen05
UMMA descriptors for K-major and MN-major 128-byte-swizzled operands, and an A
operand held in tensor memory) and of the bounded device waits (a wait that
must run out, recorded as a status)."""
import pytest
import torch

from nvfp4_fake_quant_gb300 import _lib, api

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k,a_mn,b_mn", [(128, 128, 0, 0), (128, 128, 0, 1), (128, 128, 1, 1),
                                           (128, 128, 1, 0), (64, 128, 0, 1), (128, 64, 0, 0),
                                           (64, 64, 1, 1), (64, 128, 1, 1), (128, 128, 2, 1),
                                           (64, 128, 2, 1), (128, 64, 2, 0), (64, 64, 2, 0)])
def test_umma_descriptor_encodings(n, k, a_mn, b_mn):
    g = torch.Generator().manual_seed(100 + n + k + 2 * a_mn + b_mn)
    a = torch.randn(128, k, generator=g).to(torch.bfloat16)
    b = torch.randn(n, k, generator=g).to(torch.bfloat16)
    a_store = (a.T if a_mn == 1 else a).contiguous().cuda()  # a_mn == 2: row-major, into TMEM
    b_store = (b.T if b_mn else b).contiguous().cuda()
    c = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    _lib.call("nvq_selftest_umma", a_store.data_ptr(), b_store.data_ptr(), c.data_ptr(), n, k,
              a_mn, b_mn, torch.cuda.current_stream().cuda_stream)
    assert api.device_status() == 0
    ref = a.double() @ b.double().T
    assert torch.allclose(c.cpu().double(), ref, rtol=1e-5, atol=1e-4)


def test_bounded_wait_times_out_and_reports():
    assert api.device_status() == 0
    _lib.call("nvq_selftest_timeout", 2_000_000, torch.cuda.current_stream().cuda_stream)
    assert api.device_status() == 5  # NVQ_ERR_TIMEOUT, then cleared
    assert api.device_status() == 0
    x = torch.ones(4, 4, device="cuda")
    assert float((x + 1).sum()) == 32.0  # the context is still usable
