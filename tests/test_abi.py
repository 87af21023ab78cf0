"""The C-ABI library builds, loads and exports every entry point that
include/nvfp4.h declares; host-side argument checks reject bad calls before
any launch (no GPU needed)."""

import ctypes
import os
import re

import pytest

from nvfp4_bit_numerics_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(binding.EXPORTED) == sorted(n for n in names)


def test_status_strings(lib):
    for code in range(8):
        assert lib.nvfp4_status_string(code)
    assert lib.nvfp4_status_string(99) == b"unknown status"


def test_size_queries(lib):
    assert binding.nvfp4_scale_bytes(128, 256, binding.NVFP4_SCALES_MMA) == 128 * 16
    assert binding.nvfp4_scale_bytes(256, 64, binding.NVFP4_SCALES_MMA) == 1024
    assert binding.nvfp4_scale_bytes(100, 64, binding.NVFP4_SCALES_LINEAR) == 400
    ws = binding.nvfp4_linear_workspace_bytes(128, 256, 256)
    # six tensors, 0.5 B codes + 1/16 B scales per element, plus a header
    elems = 2 * 128 * 256 + 2 * 256 * 256 + 2 * 256 * 128
    assert ws >= elems * 0.5625 + 256
    assert binding.nvfp4_linear_workspace_bytes(0, 1, 1) == 0
    # MXFP4: one byte per 32 elements, or the padded words of the tile layout
    assert binding.nvfp4_mx_scale_bytes(100, 64, binding.NVFP4_SCALES_LINEAR) == 200
    assert binding.nvfp4_mx_scale_bytes(128, 256, binding.NVFP4_SCALES_MMA) == 128 * 16


def _t(rows, cols, layout=1, codes=16, scales=16, amax=16, ts=16, fmt=0):
    return binding.nvfp4_tensor(codes, scales, amax, ts, rows, cols, layout, fmt)


def _mx(rows, cols, layout=1, codes=16, scales=16):
    return _t(rows, cols, layout, codes, scales, None, None, binding.NVFP4_FORMAT_MXFP4)


def test_gemm_argument_checks(lib):
    a, b = _t(128, 256), _t(256, 256)
    d = ctypes.c_void_p(16)
    call = lambda a_, b_, d_=d, dt=0, ldd=256: lib.nvfp4_gemm(ctypes.byref(a_), ctypes.byref(b_), d_, dt, ldd, None)
    assert lib.nvfp4_gemm(None, ctypes.byref(b), d, 0, 256, None) == binding.NVFP4_ERR_ARG
    assert call(a, b, d_=None) == binding.NVFP4_ERR_ARG
    assert call(a, b, dt=7) == binding.NVFP4_ERR_ARG
    assert call(_t(128, 256, layout=0), b) == binding.NVFP4_ERR_ARG
    assert call(_t(100, 256), b) == binding.NVFP4_ERR_SHAPE
    assert call(a, _t(256, 128)) == binding.NVFP4_ERR_SHAPE
    assert call(_t(128, 96), _t(256, 96)) == binding.NVFP4_ERR_SHAPE
    assert call(a, b, ldd=200) == binding.NVFP4_ERR_SHAPE
    assert call(a, _t(256, 256, codes=24)) == binding.NVFP4_ERR_ARG
    assert call(a, b, d_=ctypes.c_void_p(24)) == binding.NVFP4_ERR_ALIGN
    assert call(a, b, ldd=260) == binding.NVFP4_ERR_ALIGN
    # the amax variant: its slot is required and 4-byte aligned, then the same checks
    am = lambda a_, b_, amax_: lib.nvfp4_gemm_amax(ctypes.byref(a_), ctypes.byref(b_), d, 0, 256, amax_, None)
    assert am(a, b, None) == binding.NVFP4_ERR_ARG
    assert am(a, b, ctypes.c_void_p(18)) == binding.NVFP4_ERR_ALIGN
    assert am(_t(100, 256), b, ctypes.c_void_p(16)) == binding.NVFP4_ERR_SHAPE
    # formats: an NVFP4 tensor needs its tensor scale, an MXFP4 one does not;
    # mixed formats and unknown formats are rejected
    assert call(_t(128, 256, ts=None), b) == binding.NVFP4_ERR_ARG
    assert call(_mx(128, 256), _t(256, 256)) == binding.NVFP4_ERR_ARG
    assert call(_t(128, 256, fmt=2), _t(256, 256, fmt=2)) == binding.NVFP4_ERR_ARG
    assert call(_mx(100, 256), _mx(256, 256)) == binding.NVFP4_ERR_SHAPE
    assert call(_mx(128, 256, layout=0), _mx(256, 256)) == binding.NVFP4_ERR_ARG


def test_gemm2_argument_checks(lib):
    """nvfp4_gemm2 checks each of its two products as nvfp4_gemm does (BF16
    output), before any launch."""
    a, b = _t(256, 256), _t(256, 256)
    d = ctypes.c_void_p(16)

    def call(a0=a, b0=b, d0=d, l0=256, a1=a, b1=b, d1=d, l1=256):
        return lib.nvfp4_gemm2(ctypes.byref(a0), ctypes.byref(b0), d0, l0, ctypes.byref(a1), ctypes.byref(b1), d1,
                               l1, None)

    assert lib.nvfp4_gemm2(None, ctypes.byref(b), d, 256, ctypes.byref(a), ctypes.byref(b), d, 256,
                           None) == binding.NVFP4_ERR_ARG
    assert call(d0=None) == binding.NVFP4_ERR_ARG
    assert call(d1=None) == binding.NVFP4_ERR_ARG
    assert call(a0=_t(100, 256)) == binding.NVFP4_ERR_SHAPE
    assert call(b1=_t(256, 128)) == binding.NVFP4_ERR_SHAPE
    assert call(l1=200) == binding.NVFP4_ERR_SHAPE
    assert call(d1=ctypes.c_void_p(24)) == binding.NVFP4_ERR_ALIGN
    assert call(a1=_t(256, 256, ts=None)) == binding.NVFP4_ERR_ARG
    # outputs that share bytes: the same buffer, or d1 starting on d0's last row
    assert call() == binding.NVFP4_ERR_ARG
    assert call(d1=ctypes.c_void_p(16 + 255 * 256 * 2)) == binding.NVFP4_ERR_ARG


def test_gemm_quant_argument_checks(lib):
    a, b = _t(256, 256), _t(512, 256)
    yq = _t(256, 512, amax=32)
    d = ctypes.c_void_p(16)
    g = lambda a_=a, b_=b, y_=yq, d_=d, amax_=None: lib.nvfp4_gemm_quant(  # noqa: E731
        ctypes.byref(a_), ctypes.byref(b_), ctypes.byref(y_) if y_ is not None else None, d_, 512, amax_, None)
    assert g(y_=None) == binding.NVFP4_ERR_ARG
    assert g(y_=_t(256, 512, amax=None)) == binding.NVFP4_ERR_ARG         # the amax is an input
    assert g(y_=_t(256, 512, layout=0)) == binding.NVFP4_ERR_ARG          # MMA scale layout only
    assert g(y_=_t(256, 512, fmt=binding.NVFP4_FORMAT_MXFP4)) == binding.NVFP4_ERR_ARG
    assert g(amax_=ctypes.c_void_p(32)) == binding.NVFP4_ERR_ARG          # same slot as y_q->amax
    assert g(a_=_t(128, 256), y_=_t(128, 512)) == binding.NVFP4_ERR_SHAPE  # pair kernel: M % 256
    assert g(y_=_t(256, 256)) == binding.NVFP4_ERR_SHAPE
    assert g(a_=_mx(256, 256), b_=_mx(512, 256)) == binding.NVFP4_ERR_ARG
    assert g(amax_=ctypes.c_void_p(18)) == binding.NVFP4_ERR_ALIGN
    assert g(d_=ctypes.c_void_p(24)) == binding.NVFP4_ERR_ALIGN


def test_quantize_mx_argument_checks(lib):
    x = ctypes.c_void_p(16)
    out, out_t = _mx(128, 256), _mx(256, 128)
    q = lambda x_=x, r=128, c=256, k=0, o=out, ot=None: lib.nvfp4_quantize_mx(
        x_, r, c, k, ctypes.byref(o) if o is not None else None, ctypes.byref(ot) if ot is not None else None, None)
    assert q(x_=None) == binding.NVFP4_ERR_ARG
    assert q(k=3) == binding.NVFP4_ERR_ARG          # no 2D kind for MXFP4
    assert q(k=-1) == binding.NVFP4_ERR_ARG
    assert q(o=None) == binding.NVFP4_ERR_ARG
    assert q(k=2) == binding.NVFP4_ERR_ARG          # fused kind needs out_t
    assert q(o=_t(128, 256)) == binding.NVFP4_ERR_ARG  # an NVFP4 output
    assert q(r=100) == binding.NVFP4_ERR_SHAPE
    assert q(c=96) == binding.NVFP4_ERR_SHAPE
    assert q(r=0) == binding.NVFP4_ERR_SHAPE
    assert q(x_=ctypes.c_void_p(8)) == binding.NVFP4_ERR_ALIGN
    assert q(o=_mx(128, 128)) == binding.NVFP4_ERR_SHAPE
    assert q(k=1) == binding.NVFP4_ERR_SHAPE        # transposed output must be [256, 128]
    assert q(r=64, c=256, o=_mx(64, 256)) == binding.NVFP4_ERR_SHAPE  # MMA layout needs rows % 128
    assert q(o=_mx(128, 256, codes=24)) == binding.NVFP4_ERR_ARG
    # and nvfp4_quantize refuses MXFP4 outputs
    cfg = binding.nvfp4_quant_cfg(0, 0, 0, 0, 0, 0, 0)
    mxo = _t(128, 256, fmt=binding.NVFP4_FORMAT_MXFP4)
    assert lib.nvfp4_quantize(x, 128, 256, ctypes.byref(cfg), ctypes.byref(mxo), None, None) == binding.NVFP4_ERR_ARG


def test_quantize_argument_checks(lib):
    cfg = binding.nvfp4_quant_cfg(0, 0, 0, 0, 0, 0, 0)
    out = _t(128, 256)
    x = ctypes.c_void_p(16)
    q = lambda x_=x, r=128, c=256, cfg_=cfg, o=out: lib.nvfp4_quantize(x_, r, c, ctypes.byref(cfg_),
                                                                    ctypes.byref(o), None, None)
    assert q(x_=None) == binding.NVFP4_ERR_ARG
    assert q(r=100) == binding.NVFP4_ERR_SHAPE
    assert q(c=0) == binding.NVFP4_ERR_SHAPE
    assert q(r=0) == binding.NVFP4_ERR_SHAPE  # empty tensors are not quantized
    assert q(x_=ctypes.c_void_p(8)) == binding.NVFP4_ERR_ALIGN
    assert q(o=_t(128, 128)) == binding.NVFP4_ERR_SHAPE
    assert q(o=_t(64, 256)) == binding.NVFP4_ERR_SHAPE
    assert q(cfg_=binding.nvfp4_quant_cfg(9, 0, 0, 0, 0, 0, 0)) == binding.NVFP4_ERR_ARG
    assert q(cfg_=binding.nvfp4_quant_cfg(0, 5, 0, 0, 0, 0, 0)) == binding.NVFP4_ERR_ARG
    # fused kind needs the transposed output
    assert q(cfg_=binding.nvfp4_quant_cfg(2, 0, 0, 0, 0, 0, 0)) == binding.NVFP4_ERR_ARG
    assert lib.nvfp4_amax(x, 10, 17, 1, 0, ctypes.c_void_p(16), None) == binding.NVFP4_ERR_SHAPE
    assert lib.nvfp4_amax(x, 10, 16, 4, 0, ctypes.c_void_p(16), None) == binding.NVFP4_ERR_SHAPE
    assert lib.nvfp4_amax(x, 16, 16, 0, 0, ctypes.c_void_p(16), None) == binding.NVFP4_ERR_ARG


def test_linear_argument_checks(lib):
    ws = binding.nvfp4_linear_workspace_bytes(128, 256, 256)
    p = ctypes.c_void_p(16)
    f = lambda M=128, K=256, N=256, wsb=ws, w=p: lib.nvfp4_linear_fwd(p, p, M, K, N, 1, p, w, wsb, None)
    assert f(M=64) == binding.NVFP4_ERR_SHAPE
    assert f(M=0) == binding.NVFP4_ERR_SHAPE
    assert f(N=0) == binding.NVFP4_ERR_SHAPE
    assert f(wsb=ws - 1) == binding.NVFP4_ERR_WORKSPACE
    assert f(w=None) == binding.NVFP4_ERR_ARG
    assert f(w=ctypes.c_void_p(8)) == binding.NVFP4_ERR_ALIGN
    assert lib.nvfp4_linear_bwd(p, 128, 256, 256, 1, p, None, p, ws, None) == binding.NVFP4_ERR_ARG
    # BF16 layers (checked before cuBLAS is touched)
    bf = lambda M=100, K=64, N=72, x=p, y=p: lib.nvfp4_linear_bf16_fwd(x, p, M, K, N, y, None)  # noqa: E731
    assert bf(M=0) == binding.NVFP4_ERR_SHAPE
    assert bf(K=60) == binding.NVFP4_ERR_SHAPE
    assert bf(N=70) == binding.NVFP4_ERR_SHAPE
    assert bf(x=None) == binding.NVFP4_ERR_ARG
    assert bf(y=ctypes.c_void_p(24)) == binding.NVFP4_ERR_ALIGN
    bb = lambda dx=p, K=64: lib.nvfp4_linear_bf16_bwd(p, p, p, 100, K, 72, dx, p, None)  # noqa: E731
    assert bb(dx=None) == binding.NVFP4_ERR_ARG
    assert bb(K=-8) == binding.NVFP4_ERR_SHAPE
    assert bb(dx=ctypes.c_void_p(40)) == binding.NVFP4_ERR_ALIGN
