"""The plain C++ CPU oracle (oracle/cxx/nvfp4_oracle.cpp), built and called
through ctypes.  TEST INFRASTRUCTURE ONLY: only the test suite, the smoke
check and the CPU-baseline leg of the benchmark use it; the product path never
imports it.

It computes the same definitions as the numpy oracle of this package -- the
two-level NVFP4 scaling, 1x16 and 16x16 blocks, the 16x16 random Hadamard
transform, stochastic rounding with Philox4x32-10 uniforms, and an
FP64-accumulated GEMM on the dequantized operands ("Pretraining Large Language
Models with NVFP4", gist.science summary, Resumo técnico §2 and §3) -- written
a second time, element by element, in C++17 compiled with -ffp-contract=off,
with std::thread over the host's cores.  The functions below take and return
the numpy oracle's representations (float32 arrays holding BF16 values,
packed codes, linear [rows, cols/16] scale codes) so that the tests can pin
both oracles with the same checks and compare them bit for bit.
"""

import ctypes
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cxx", "nvfp4_oracle.cpp")
LIB = os.path.join(HERE, "cxx", "libnvfp4_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]

F32 = np.float32
_lib = None


def build(force=False):
    """Compile the oracle library with the host C++ compiler (if stale)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) > os.path.getmtime(SRC):
        return LIB
    cxx = os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("no C++ compiler for the oracle")
    tmp = LIB + ".tmp"
    r = subprocess.run([cxx] + FLAGS + ["-o", tmp, SRC], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        P, I64, I32, U64, U32, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                                    ctypes.c_uint32, ctypes.c_float)
        sig = {
            "ox_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "ox_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "ox_e2m1_encode_rne_n": (None, [P, I64, P]),
            "ox_e2m1_encode_sr_n": (None, [P, P, I64, P]),
            "ox_e4m3_encode_rne_sat_n": (None, [P, I64, P]),
            "ox_sr_uniform16_n": (None, [U64, U32, P, I64, P]),
            "ox_philox4x32_10": (None, [P, U32, U32, P]),
            "ox_rht_signs": (None, [U64, P]),
            "ox_rht16": (None, [P, P, P]),
            "ox_amax": (F, [P, I64, I64, I32]),
            "ox_amax_rht": (F, [P, I64, I64, I32, U64, I32]),
            "ox_quantize_rows": (I32, [P, I64, I64, I32, P, I64, F, I32, U64, U32, I32, U64, P, P, P, I32]),
            "ox_quantize_2d": (I32, [P, I64, I64, F, P, P, P, P, P, I32]),
            "ox_gemm": (None, [P, P, F, P, P, F, I64, I64, P, I64, P, I32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


# ---------------------------------------------------------------------------
# formats and generator
# ---------------------------------------------------------------------------
def e2m1_decode(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib().ox_e2m1_decode(int(v) & 0xF) for v in c.reshape(-1)]).reshape(c.shape)


def e4m3_decode(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib().ox_e4m3_decode(int(v)) for v in c.reshape(-1)]).reshape(c.shape)


def e2m1_encode_rne(v):
    shape = np.shape(v)
    v = _f32(v)
    out = np.empty(v.shape, np.uint8)
    lib().ox_e2m1_encode_rne_n(_p(v), v.size, _p(out))
    return out.reshape(shape)


def e2m1_encode_sr(v, u16):
    shape = np.broadcast_shapes(np.shape(v), np.shape(u16))
    v = _f32(np.broadcast_to(np.asarray(v, dtype=np.float32), shape))
    u = np.ascontiguousarray(np.broadcast_to(np.asarray(u16, dtype=np.uint32), shape)).reshape(v.shape)
    out = np.empty(v.shape, np.uint8)
    lib().ox_e2m1_encode_sr_n(_p(v), _p(u), v.size, _p(out))
    return out.reshape(shape)


def e4m3_encode_rne_sat(x):
    shape = np.shape(x)
    x = _f32(x)
    out = np.empty(x.shape, np.uint8)
    lib().ox_e4m3_encode_rne_sat_n(_p(x), x.size, _p(out))
    return out.reshape(shape)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    ctr = np.array([c0, c1, c2, c3], dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().ox_philox4x32_10(_p(ctr), int(k0) & 0xFFFFFFFF, int(k1) & 0xFFFFFFFF, _p(out))
    return [np.uint32(v) for v in out]


def sr_uniform16(seed, stream_id, elem_index):
    e = np.ascontiguousarray(np.asarray(elem_index, dtype=np.uint64))
    out = np.empty(e.shape, np.uint32)
    lib().ox_sr_uniform16_n(int(seed) & (2 ** 64 - 1), int(stream_id), _p(e), e.size, _p(out))
    return out


def rht_signs(seed):
    s = np.empty(16, np.float32)
    lib().ox_rht_signs(int(seed) & (2 ** 64 - 1), _p(s))
    return s.astype(np.int64)


def rht16(x, signs):
    """Q x for one 16-vector (float32)."""
    x = _f32(x).reshape(16)
    s = _f32(signs).reshape(16)
    y = np.empty(16, np.float32)
    lib().ox_rht16(_p(x), _p(s), _p(y))
    return y


# ---------------------------------------------------------------------------
# amax, quantization, GEMM
# ---------------------------------------------------------------------------
def tensor_amax(x, threads=0):
    x = _f32(x)
    if x.size == 0:
        return F32(0.0)
    x2 = x.reshape(x.shape[0], -1) if x.ndim > 1 else x.reshape(1, -1)
    return F32(lib().ox_amax(_p(x2), x2.shape[0], x2.shape[1], threads))


def amax_rht(x, rht_seed, axis, threads=0):
    x = _f32(x)
    return F32(lib().ox_amax_rht(_p(x), x.shape[0], x.shape[1], int(axis), int(rht_seed) & (2 ** 64 - 1), threads))


def _quantize(x, transpose, rounding, seed, stream_id, rht_seed, amax, ids, threads):
    x = _f32(x)
    R, C = x.shape
    rows_q, cols_q = (C, R) if transpose else (R, C)
    assert cols_q % 16 == 0
    rht = rht_seed is not None
    if amax is None:
        if rht:
            amax = amax_rht(x, rht_seed, 0 if transpose else 1, threads)
        else:
            amax = tensor_amax(x, threads)
    ids = np.arange(rows_q, dtype=np.int64) if ids is None else np.ascontiguousarray(ids, dtype=np.int64)
    codes = np.zeros((len(ids), cols_q // 2), np.uint8)
    scales = np.zeros((len(ids), cols_q // 16), np.uint8)
    ts = np.zeros(1, np.float32)
    rc = lib().ox_quantize_rows(_p(x), R, C, int(transpose), _p(ids), len(ids), F32(amax),
                                1 if rounding == "sr" else 0, int(seed) & (2 ** 64 - 1), int(stream_id), int(rht),
                                int(rht_seed or 0) & (2 ** 64 - 1), _p(codes), _p(scales), _p(ts), threads)
    if rc != 0:
        raise FloatingPointError("non-finite amax")
    return dict(codes=codes, scales=scales, amax=F32(amax), ts=F32(ts[0]))


def quantize_1d(x, rounding="rne", seed=0, stream_id=0, rht_seed=None, amax=None, row_ids=None, threads=0):
    """1x16 blocks along the last axis of x [R, C] (see the numpy oracle's
    quant.quantize_1d); ``row_ids`` selects rows with the whole tensor's amax."""
    return _quantize(x, False, rounding, seed, stream_id, rht_seed, amax, row_ids, threads)


def quantize_transpose(x, rounding="rne", seed=0, stream_id=0, rht_seed=None, amax=None, col_ids=None, threads=0):
    """x [M, C] -> x^T [C, M], optionally transformed along M, 1x16 blocks
    along M (see quant.quantize_transpose); ``col_ids`` selects output rows."""
    return _quantize(x, True, rounding, seed, stream_id, rht_seed, amax, col_ids, threads)


def quantize_2d(w, amax=None, threads=0):
    w = _f32(w)
    N, K = w.shape
    if amax is None:
        amax = tensor_amax(w, threads)
    codes = np.zeros((N, K // 2), np.uint8)
    codes_t = np.zeros((K, N // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    scales_t = np.zeros((K, N // 16), np.uint8)
    ts = np.zeros(1, np.float32)
    rc = lib().ox_quantize_2d(_p(w), N, K, F32(amax), _p(codes), _p(scales), _p(codes_t), _p(scales_t), _p(ts),
                              threads)
    if rc != 0:
        raise FloatingPointError("non-finite amax")
    return dict(codes=codes, scales=scales, codes_t=codes_t, scales_t=scales_t, scales_2d=scales[::16],
                amax=F32(amax), ts=F32(ts[0]))


def gemm_ref(a_codes, a_scales, ts_a, b_codes, b_scales, ts_b, rows=None, threads=0):
    """D = A B^T in float64 for K-major NVFP4 A [M, K], B [N, K]; ``rows``
    selects rows of D."""
    a_codes, a_scales = np.ascontiguousarray(a_codes, np.uint8), np.ascontiguousarray(a_scales, np.uint8)
    b_codes, b_scales = np.ascontiguousarray(b_codes, np.uint8), np.ascontiguousarray(b_scales, np.uint8)
    N, K = b_codes.shape[0], b_codes.shape[1] * 2
    ids = np.arange(a_codes.shape[0], dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    d = np.empty((len(ids), N), np.float64)
    lib().ox_gemm(_p(a_codes), _p(a_scales), F32(ts_a), _p(b_codes), _p(b_scales), F32(ts_b), N, K, _p(ids),
                  len(ids), _p(d), threads)
    return d


# ---------------------------------------------------------------------------
# One linear layer (the composition of the numpy oracle's linear module:
# stream 0 rounds dY, stream 1 the transformed dY^T, the seed keys the signs)
# ---------------------------------------------------------------------------
SR_STREAM_DY = 0
SR_STREAM_DYT = 1


def linear_fwd(x, w, seed, rows=None, threads=0):
    x = _f32(x)
    xq = quantize_1d(x, "rne", amax=tensor_amax(x, threads), row_ids=rows, threads=threads)
    wq = quantize_2d(w, threads=threads)
    xtq = quantize_transpose(x, "rne", rht_seed=seed, threads=threads)
    y = gemm_ref(xq["codes"], xq["scales"], xq["ts"], wq["codes"], wq["scales"], wq["ts"], threads=threads)
    return dict(y=y, xq=xq, wq=wq, xtq=xtq)


def linear_bwd(dy, fwd, seed, rows_dx=None, rows_dw=None, threads=0):
    dy = _f32(dy)
    dyq = quantize_1d(dy, "sr", seed=seed, stream_id=SR_STREAM_DY, amax=tensor_amax(dy, threads), row_ids=rows_dx,
                      threads=threads)
    dytq = quantize_transpose(dy, "sr", seed=seed, stream_id=SR_STREAM_DYT, rht_seed=seed,
                              amax=amax_rht(dy, seed, 0, threads), col_ids=rows_dw, threads=threads)
    wq, xtq = fwd["wq"], fwd["xtq"]
    dx = gemm_ref(dyq["codes"], dyq["scales"], dyq["ts"], wq["codes_t"], wq["scales_t"], wq["ts"], threads=threads)
    dw = gemm_ref(dytq["codes"], dytq["scales"], dytq["ts"], xtq["codes"], xtq["scales"], xtq["ts"], threads=threads)
    return dict(dx=dx, dw=dw, dyq=dyq, dytq=dytq)
