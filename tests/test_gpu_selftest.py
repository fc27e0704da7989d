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


# ---------------------------------------------------------------- FP4 UMMA
# Block-scaled kind::mxf4nvf4 MMA: E2M1 codes two to a byte (even element in the
# low nibble), one E4M3 scale per 16 elements of a row.  The scales sit in
# tensor memory in the layout of the 128 x 4 scale tile of block-scaled FP4
# GEMMs: per MMA (64 K-elements) four 32-bit columns; lane l of every lane
# quadrant holds, in column c, the four scale bytes (in K order) of row
# (l % 32) + 32 c.

_E2M1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)


def _e2m1_values(codes):  # uint8 [rows, K/2] -> float64 [rows, K]
    nib = torch.stack([codes & 15, codes >> 4], dim=-1).reshape(codes.shape[0], -1).long()
    mag = _E2M1[nib & 7]
    return torch.where(nib >= 8, -mag, mag)


def _e4m3_values(s):  # uint8 -> float64
    return s.contiguous().view(torch.float8_e4m3fn).to(torch.float64)


def _fp4_operands(seed, rows_a, n, k):
    g = torch.Generator().manual_seed(seed)
    a = torch.randint(0, 256, (rows_a, k // 2), generator=g, dtype=torch.uint8)
    b = torch.randint(0, 256, (n, k // 2), generator=g, dtype=torch.uint8)
    sa = torch.randint(0x28, 0x49, (rows_a, k // 16), generator=g, dtype=torch.uint8)
    sb = torch.randint(0x28, 0x49, (n, k // 16), generator=g, dtype=torch.uint8)
    return a, b, sa, sb


def _scale_words(s, rows, kk):
    """u32 [32, 4]: word (l, c) = the 4 scale bytes of row l + 32 c for MMA kk."""
    pad = torch.zeros(128, s.shape[1], dtype=torch.uint8)
    pad[:rows] = s
    blk = pad[:, 4 * kk:4 * kk + 4].reshape(4, 32, 4).permute(1, 0, 2).contiguous()
    return blk.view(torch.int32).reshape(32, 4)


def _tmem_image(sa, sb, n, nmma):
    img = torch.zeros(2, 128, 32, dtype=torch.int32)
    for m, (s, rows) in enumerate(((sa, 128), (sb, n))):
        for kk in range(nmma):
            img[m, :, 4 * kk:4 * kk + 4] = _scale_words(s, rows, kk).repeat(4, 1)
    return img


def _cp_source(sa, sb, n, nmma):
    blocks = [_scale_words(s, rows, kk).view(torch.uint8).reshape(512)
              for s, rows in ((sa, 128), (sb, n)) for kk in range(nmma)]
    return torch.cat(blocks)


def _run_fp4(a, b, img, src, n, nmma, stride, mode):
    dev = "cuda"
    a_d, b_d = a.to(dev), b.to(dev)
    img_d = img.to(dev) if img is not None else None
    src_d = src.to(dev) if src is not None else None
    c = torch.full((128, n), float("nan"), dtype=torch.float32, device=dev)
    dump = torch.zeros(128, 64, dtype=torch.int32, device=dev)
    st = _lib.call("nvq_selftest_fp4", a_d.data_ptr(), b_d.data_ptr(),
                   img_d.data_ptr() if img_d is not None else None,
                   src_d.data_ptr() if src_d is not None else None, c.data_ptr(),
                   dump.data_ptr(), n, nmma, stride, mode, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    assert api.device_status() == 0
    return c.cpu().double(), dump.cpu()


@pytest.mark.parametrize("n,nmma,mode", [(128, 2, 0), (128, 2, 1), (64, 1, 0), (64, 2, 1),
                                         (128, 1, 1), (128, 4, 0), (128, 4, 1), (64, 4, 1)])
def test_fp4_block_scaled_umma(n, nmma, mode):
    k = 64 * nmma
    a, b, sa, sb = _fp4_operands(7 + n + nmma + mode, 128, n, k)
    img = _tmem_image(sa, sb, n, nmma) if mode == 0 else None
    src = _cp_source(sa, sb, n, nmma) if mode == 1 else None
    c, dump = _run_fp4(a, b, img, src, n, nmma, 4, mode)
    av = _e2m1_values(a) * _e4m3_values(sa).repeat_interleave(16, dim=1)
    bv = _e2m1_values(b) * _e4m3_values(sb).repeat_interleave(16, dim=1)
    ref = av @ bv.T
    mag = av.abs() @ bv.abs().T
    if mode == 1:  # the copy replicated the 32 x 16-byte blocks into every lane quadrant
        want = _tmem_image(sa, sb, n, nmma)
        for m in range(2):
            assert torch.equal(dump[:, 32 * m:32 * m + 4 * nmma], want[m, :, :4 * nmma])
    assert torch.all((c - ref).abs() <= 1e-6 * mag + 1e-30), float((c - ref).abs().max())


def test_hardware_exp2_is_non_decreasing():
    """The P~ quantization forms a block's maximum of P = 2^x as 2^(max x); that is the
    same value only if the hardware 2^x (ex2.approx.ftz.f32) never decreases.  Checked
    for every pair of consecutive floats in [-200, 2] (about 2.2e9 pairs)."""
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    assert _lib.load().nvq_selftest_ex2_monotone(out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    bad, first = out.cpu().tolist()
    assert bad == 0, (bad, first)
