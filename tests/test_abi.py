"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/nvfp4attn.h declares, sizes its workspaces, and rejects bad
arguments on the host before launching anything (these calls never reach a
CUDA API, so they are safe without a device)."""
import ctypes
import os
import re

import pytest

from nvfp4_fake_quant_gb300 import _lib
from nvfp4_fake_quant_gb300 import build as nvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4attn.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
A = 0x100000  # a 256-byte-aligned non-null address that validation never dereferences


@pytest.fixture(scope="module")
def lib():
    path = nvbuild.build()
    return _lib.load(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return sorted(set(re.findall(r"\b([A-Za-z_]\w*)\s*\([^;{()]*\)\s*;", src)))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ["nvfp4_fake_quant", "nvfp4_quantize_codes", "nvfp4_global_sf", "attn_qat_fwd",
                     "attn_qat_bwd", "attn_qat_fwd_workspace", "attn_qat_bwd_workspace",
                     "nvq_device_status", "nvq_status_string", "nvq_version"]:
        assert required in names
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    cdll = ctypes.CDLL(nvbuild.LIB)
    for name in declared_functions():
        getattr(cdll, name)


def test_status_strings_and_version(lib):
    for code, name in _lib.STATUS.items():
        assert lib.nvq_status_string(code).decode() == name
    assert lib.nvq_status_string(99).decode() == "NVQ_ERR_UNKNOWN"
    assert lib.nvq_version() >> 16 == 1
    assert lib.nvq_last_error_detail() == b""  # no call on this thread has failed in CUDA


def test_workspace_sizes(lib):
    b, n, h, d = 1, 25088, 12, 128
    t = b * n * h * d * 2
    # Q~, K~, V~ (bf16), delta, then the E2M1 codes (D/2 bytes a row) and the
    # 512-byte scale blocks (one per 128 rows and 64 elements of D) of Q~ and K~
    codes = b * n * h * d // 2
    scales = b * h * ((n + 127) // 128) * (d // 64) * 512
    # forward: codes and scale blocks of Q~, K~, V~ in f16, Q~, K~ and V~ in bf16
    assert lib.attn_qat_fwd_workspace(b, n, n, h, d) == 2 * codes + 2 * scales + 4 * t
    assert lib.attn_qat_bwd_saved_workspace(b, n, n, h, d) == b * h * n * 4
    assert lib.attn_qat_bwd_workspace(b, n, n, h, d) == 3 * t + b * h * n * 4 + 2 * codes + 2 * scales
    assert lib.attn_qat_fwd_workspace(0, n, n, h, d) == 0
    assert lib.attn_qat_fwd_workspace(1, 3, 5, 1, 64) % 256 == 0


def test_workspace_layouts(lib):
    """The regions attn_qat_*_layout reports are 256-byte aligned, disjoint, of
    the documented sizes, and inside the workspace the size query returns."""
    from nvfp4_fake_quant_gb300 import api
    for (b, nq, nkv, h, d) in [(1, 25088, 25088, 12, 128), (2, 300, 333, 3, 64), (1, 1, 1, 1, 128)]:
        nt = lambda n: (n + 127) // 128
        size = {"q_codes": b * nq * h * d // 2, "k_codes": b * nkv * h * d // 2,
                "q_scales": b * h * nt(nq) * (d // 64) * 512,
                "k_scales": b * h * nt(nkv) * (d // 64) * 512,
                "v_f16": b * nkv * h * d * 2, "q_bf16": b * nq * h * d * 2,
                "k_bf16": b * nkv * h * d * 2, "v_bf16": b * nkv * h * d * 2,
                "delta": b * h * nq * 4}
        for which, query in (("fwd", lib.attn_qat_fwd_workspace),
                             ("bwd", lib.attn_qat_bwd_workspace)):
            lay = api.attn_qat_layout(b, nq, nkv, h, d, which)
            assert lay["total"] == query(b, nq, nkv, h, d)
            spans = sorted((off, off + size[name]) for name, off in lay.items() if name != "total")
            assert all(off % 256 == 0 for off, _ in spans)
            assert all(e0 <= s1 for (_, e0), (s1, _) in zip(spans, spans[1:]))
            assert spans[-1][1] <= lay["total"]
        assert set(api.attn_qat_layout(b, nq, nkv, h, d, "fwd")) == \
            {"q_codes", "k_codes", "q_scales", "k_scales", "v_f16", "q_bf16", "k_bf16", "v_bf16",
             "total"}
        assert set(api.attn_qat_layout(b, nq, nkv, h, d, "bwd")) == \
            {"q_codes", "k_codes", "q_scales", "k_scales", "q_bf16", "k_bf16", "v_bf16", "delta",
             "total"}
    lay = _lib.AttnLayout()
    assert lib.attn_qat_fwd_layout(1, 128, 128, 1, 96, ctypes.addressof(lay)) == INVALID
    assert lib.attn_qat_bwd_layout(0, 128, 128, 1, 64, ctypes.addressof(lay)) == INVALID
    assert lib.attn_qat_fwd_layout(1, 128, 128, 1, 64, None) == INVALID


def _fwd(lib, q=A, k=A, v=A, B=1, Nq=128, Nkv=128, H=1, D=128, scale=0.125, causal=0, o=A,
         stats=A, ws=A, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.attn_qat_fwd_workspace(B, Nq, Nkv, H, D) if min(B, Nq, Nkv, H) > 0 else 0
    return lib.attn_qat_fwd(q, k, v, B, Nq, Nkv, H, D, scale, causal, o, stats, ws, ws_bytes, None)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, D=96) == UNSUPPORTED
    assert _fwd(lib, D=256) == UNSUPPORTED
    assert _fwd(lib, causal=1, Nq=128, Nkv=256) == UNSUPPORTED
    assert _fwd(lib, B=0) == INVALID
    assert _fwd(lib, Nkv=0) == INVALID
    assert _fwd(lib, scale=0.0) == INVALID
    assert _fwd(lib, scale=-1.0) == INVALID
    assert _fwd(lib, scale=float("nan")) == INVALID
    assert _fwd(lib, scale=float("inf")) == INVALID
    assert _fwd(lib, causal=2) == INVALID
    assert _fwd(lib, q=None) == INVALID
    assert _fwd(lib, stats=None) == INVALID
    assert _fwd(lib, o=A + 8) == INVALID
    assert _fwd(lib, ws=None) == WORKSPACE
    assert _fwd(lib, ws_bytes=1024) == WORKSPACE
    assert _fwd(lib, ws=A + 16) == WORKSPACE


def test_fwd_hp_rejects_bad_arguments(lib):
    def fwd_hp(o_hp=A + 4096, D=128, causal=0, Nkv=128, ws_bytes=None):
        if ws_bytes is None:
            ws_bytes = lib.attn_qat_fwd_workspace(1, 128, Nkv, 1, D)
        return lib.attn_qat_fwd_hp(A, A, A, 1, 128, Nkv, 1, D, 0.1, causal, A, o_hp, A, A,
                                   ws_bytes, None)
    assert fwd_hp(o_hp=None) == INVALID
    assert fwd_hp(o_hp=A + 8) == INVALID
    assert fwd_hp(D=96) == UNSUPPORTED
    assert fwd_hp(causal=1, Nkv=256) == UNSUPPORTED
    assert fwd_hp(ws_bytes=16) == WORKSPACE


def test_bwd_rejects_bad_arguments(lib):
    def bwd(dq=A, D=128, Nq=128, Nkv=128, causal=0, ws=A, ws_bytes=None, scale=0.1):
        if ws_bytes is None:
            ws_bytes = lib.attn_qat_bwd_workspace(1, Nq, Nkv, 1, D)
        return lib.attn_qat_bwd(A, A, A, A, A, A, dq, A, A, 1, Nq, Nkv, 1, D, scale, causal, ws,
                                ws_bytes, None)
    assert bwd(D=80) == UNSUPPORTED
    assert bwd(causal=1, Nkv=64) == UNSUPPORTED
    assert bwd(dq=None) == INVALID
    assert bwd(dq=A + 2) == INVALID
    assert bwd(scale=float("nan")) == INVALID
    assert bwd(ws_bytes=0) == WORKSPACE


def test_bwd_saved_rejects_bad_arguments(lib):
    b, n, h, d = 1, 256, 2, 128
    fws = lib.attn_qat_fwd_workspace(b, n, n, h, d)
    bws = lib.attn_qat_bwd_saved_workspace(b, n, n, h, d)

    def bwd(saved=A, saved_bytes=fws, o=A, D=d, causal=0, scale=0.1, ws=A + (1 << 30),
            ws_bytes=bws, nkv=n):
        return lib.attn_qat_bwd_saved(saved, saved_bytes, o, A, A, A, A, A, b, n, nkv, h, D, scale,
                                      causal, ws, ws_bytes, None)
    assert bwd(D=96) == UNSUPPORTED
    assert bwd(causal=1, nkv=n + 1) == UNSUPPORTED
    assert bwd(scale=float("nan")) == INVALID
    assert bwd(o=None) == INVALID
    assert bwd(o=A + 8) == INVALID
    assert bwd(saved=None) == WORKSPACE
    assert bwd(saved_bytes=fws - 1) == WORKSPACE
    assert bwd(saved=A + 16) == WORKSPACE
    assert bwd(ws_bytes=bws - 1) == WORKSPACE
    assert bwd(ws=None) == WORKSPACE


def test_sparse_saved_backward_workspace_and_rejections(lib):
    """attn_qat_bwd_sparse_saved: its workspace is delta [B, H, N] f32 followed by the
    transposed lists (offsets [B, H, n_tiles + 1], entries [B, H, n_tiles, topk] int32),
    each region 256-byte aligned; bad sizes, lists and buffers are rejected before any
    device work."""
    def up(x):
        return (x + 255) // 256 * 256
    n, h, d = 25088, 12, 128
    want = up(12 * n * 4) + up(12 * 197 * 4) + up(12 * 196 * 20 * 4)
    assert lib.attn_qat_bwd_sparse_saved_workspace(1, n, h, d, 20) == want
    assert lib.attn_qat_bwd_sparse_saved_workspace(1, n, h, d, 0) == 0
    b, n, h, d, topk = 1, 512, 2, 128, 2
    fws = lib.attn_qat_fwd_workspace(b, n, n, h, d)
    bws = lib.attn_qat_bwd_sparse_saved_workspace(b, n, h, d, topk)

    def bwd(saved=A, saved_bytes=fws, o=A, tiles=A, topk=topk, n=n, D=d, scale=0.1,
            ws=A + (1 << 30), ws_bytes=bws):
        return lib.attn_qat_bwd_sparse_saved(saved, saved_bytes, o, A, A, tiles, topk, A, A, A,
                                             b, n, h, D, scale, ws, ws_bytes, None)
    assert bwd(topk=0) == INVALID
    assert bwd(topk=5) == INVALID           # more than n / 128 key tiles
    assert bwd(n=500) == INVALID            # not whole tiles
    assert bwd(tiles=None) == INVALID
    assert bwd(tiles=A + 2) == INVALID
    assert bwd(D=96) == UNSUPPORTED
    assert bwd(scale=float("nan")) == INVALID
    assert bwd(o=A + 8) == INVALID
    assert bwd(saved=None) == WORKSPACE
    assert bwd(saved_bytes=fws - 1) == WORKSPACE
    assert bwd(ws_bytes=bws - 1) == WORKSPACE
    assert bwd(ws=A + 16) == WORKSPACE


def test_quantizer_rejects_bad_arguments(lib):
    def fq(x=A, rows=4, cols=32, ld=32, gsf=None, out=A + 4096, ld_out=32, sc=A, ld_s=2):
        return lib.nvfp4_fake_quant(x, rows, cols, ld, gsf, out, ld_out, sc, ld_s, None)
    assert fq(cols=24, ld=24, ld_out=24) == INVALID     # cols % 16
    assert fq(cols=0) == INVALID
    assert fq(rows=0) == INVALID
    assert fq(ld=16) == INVALID                          # ld_x < cols
    assert fq(ld=36) == INVALID                          # ld_x % 8
    assert fq(x=None) == INVALID
    assert fq(x=A + 2) == INVALID
    assert fq(out=None) == INVALID
    assert fq(ld_out=40, out=A) == INVALID               # in place needs ld_out == ld_x
    assert fq(ld_s=1) == INVALID
    assert fq(gsf=A + 1) == INVALID
    assert lib.nvfp4_quantize_codes(A, 4, 32, 32, None, A, 12, A, 2, None) == INVALID  # ld%8
    assert lib.nvfp4_quantize_codes(A, 4, 32, 32, None, A, 16, None, 2, None) == INVALID
    assert lib.nvfp4_global_sf(A, 4, 32, 32, None, None) == INVALID
    assert lib.nvfp4_global_sf(A, 0, 32, 32, A, None) == INVALID
    assert lib.nvq_selftest_timeout(0, None) == INVALID
    assert lib.nvq_selftest_ex2_monotone(None, None) == INVALID
    assert lib.nvq_selftest_ex2_monotone(A + 4, None) == INVALID
    assert lib.nvq_selftest_umma(A, A, A, 96, 64, 0, 0, None) == INVALID
    assert lib.nvq_selftest_umma(A, A, A, 64, 64, 3, 0, None) == INVALID
    assert lib.nvq_selftest_fp4(A, A, A, None, A, A, 96, 1, 4, 0, None) == INVALID
    assert lib.nvq_selftest_fp4(A, A, A, None, A, A, 128, 3, 4, 0, None) == INVALID
    assert lib.nvq_selftest_fp4(A, A, None, None, A, A, 128, 2, 4, 0, None) == INVALID
    assert lib.nvq_selftest_fp4(A, A, None, None, A, A, 128, 2, 4, 1, None) == INVALID
    assert lib.nvq_selftest_fp4(A, A, A, None, A, A, 128, 2, 5, 0, None) == INVALID


def test_block_sparse_and_vsa_calls_reject_bad_arguments(lib):
    n, h, d = 25088, 12, 128
    assert lib.vsa_select_workspace(1, n, h, d) == 2 * 12 * 196 * 128 * 4
    assert lib.vsa_select_workspace(1, n - 8, h, d) == 0
    # the dense backward's workspace (Q~, K~, V~ bf16, delta, the FP4 operands of the
    # dQ kernel) followed by the transposed tile lists
    common = lib.attn_qat_bwd_workspace(1, n, n, h, d)
    offsets = (12 * 197 * 4 + 255) // 256 * 256  # [B, H, n_tiles + 1] int32, 256-byte aligned
    assert lib.attn_qat_bwd_sparse_workspace(1, n, h, d, 20) == common + offsets + 12 * 196 * 20 * 4
    big = 1 << 40

    def reorder(x=A, out=A + 4096, t=8, hh=8, w=16, ct=4, ch=4, cw=8, to_cubes=1):
        return lib.vsa_reorder(x, 1, t, hh, w, 2, 64, ct, ch, cw, to_cubes, out, None)
    assert reorder(out=A) == INVALID         # in place
    assert reorder(x=None) == INVALID
    assert reorder(t=6) == INVALID           # not a whole number of cubes
    assert reorder(to_cubes=2) == INVALID

    def select(nn=384, topk=2, ws=A, ws_bytes=big, dd=64):
        return lib.vsa_select_tiles(A, A, 1, nn, 2, dd, topk, A, ws, ws_bytes, None)
    assert select(topk=0) == INVALID
    assert select(topk=4) == INVALID         # more than N / 128
    assert select(nn=390) == INVALID         # N % 128
    assert select(dd=2048) == INVALID
    assert select(ws_bytes=16) == WORKSPACE

    def fwd(nn=384, topk=2, kv=A, dd=128):
        return lib.attn_qat_fwd_sparse(A, A, A, 1, nn, 2, dd, 0.1, kv, topk, A, A, A, big, None)
    assert fwd(nn=300) == INVALID
    assert fwd(topk=4) == INVALID
    assert fwd(kv=None) == INVALID
    assert fwd(kv=A + 2) == INVALID
    assert fwd(dd=96) == UNSUPPORTED
    assert lib.attn_qat_bwd_sparse(A, A, A, A, A, A, A, 0, A, A, A, 1, 384, 2, 128, 0.1, A, big,
                                   None) == INVALID  # topk 0


def test_timing_hook_arguments(lib):
    n, ms = ctypes.c_int64(-1), ctypes.c_double(-1.0)
    pn, pms = ctypes.addressof(n), ctypes.addressof(ms)
    assert lib.nvq_timing_enable(2) == INVALID
    assert lib.nvq_timing_read(8, pn, pms) == INVALID
    assert lib.nvq_timing_read(-1, pn, pms) == INVALID
    assert lib.nvq_timing_read(0, None, pms) == INVALID
    assert lib.nvq_timing_enable(1) == OK
    assert lib.nvq_timing_read(3, pn, pms) == OK  # nothing launched: no CUDA call needed
    assert (n.value, ms.value) == (0, 0.0)
    assert lib.nvq_timing_enable(0) == OK


def test_python_layer_conventions():
    from nvfp4_fake_quant_gb300 import api
    with pytest.raises(NotImplementedError):
        api.AttnQAT(12, 128, None, False, dropout_p=0.1)
    with pytest.raises(ValueError):
        api.AttnQAT(12, 96)
    assert api.AttnQAT(12, 128).softmax_scale == 1.0 / 128 ** 0.5
    assert api.default_scale(64) == 0.125
