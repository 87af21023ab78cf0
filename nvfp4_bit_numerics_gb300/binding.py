"""ctypes binding of libnvfp4.so (include/nvfp4.h), argument marshalling only.

Every function below forwards torch tensors' device pointers, sizes and the
current CUDA stream to the C entry point of the same name; all computation
happens in the library's CUDA kernels.  PyTorch only allocates device memory
and provides streams.  There is no fallback: if the library is missing or no
GPU is present, the calls raise.
"""

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnvfp4.so")

# status codes
NVFP4_OK = 0
NVFP4_ERR_ARG = 1
NVFP4_ERR_SHAPE = 2
NVFP4_ERR_ALIGN = 3
NVFP4_ERR_NONFINITE = 4
NVFP4_ERR_TIMEOUT = 5
NVFP4_ERR_CUDA = 6
NVFP4_ERR_WORKSPACE = 7

NVFP4_SCALES_LINEAR = 0
NVFP4_SCALES_MMA = 1
NVFP4_Q_ROWWISE = 0
NVFP4_Q_TRANSPOSE = 1
NVFP4_Q_ROWWISE_AND_TRANSPOSE = 2
NVFP4_Q_2D = 3
NVFP4_ROUND_RNE = 0
NVFP4_ROUND_SR = 1
NVFP4_AMAX_PLAIN = 1
NVFP4_AMAX_RHT_ROWS = 2
NVFP4_AMAX_RHT_COLS = 4
NVFP4_OUT_BF16 = 0
NVFP4_OUT_F32 = 1
NVFP4_FORMAT_NVFP4 = 0
NVFP4_FORMAT_MXFP4 = 1

EXPORTED = [
    "nvfp4_amax", "nvfp4_quantize", "nvfp4_scale_bytes", "nvfp4_gemm", "nvfp4_linear_workspace_bytes",
    "nvfp4_linear_fwd", "nvfp4_linear_bwd", "nvfp4_linear_get_views", "nvfp4_get_status",
    "nvfp4_status_string", "nvfp4_kernel_launch_count", "nvfp4_linear_fwd_noalloc",
    "nvfp4_debug_stall_next_gemm", "nvfp4_gemm_amax", "nvfp4_quantize_mx", "nvfp4_mx_scale_bytes",
    "nvfp4_linear_bf16_fwd", "nvfp4_linear_bf16_bwd", "nvfp4_gemm_quant", "nvfp4_debug_stall_next_quantize",
    "nvfp4_gemm2",
]


class Nvfp4Error(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__("%s failed: %s (%d)" % (fn, msg, code))
        self.code = code


class nvfp4_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("scale_layout", ctypes.c_int32), ("format", ctypes.c_int32)]


class nvfp4_quant_cfg(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("rounding", ctypes.c_int32), ("rht", ctypes.c_int32),
                ("compute_amax", ctypes.c_int32), ("seed", ctypes.c_uint64), ("sr_stream", ctypes.c_uint32),
                ("sr_stream_t", ctypes.c_uint32)]


class nvfp4_linear_views(ctypes.Structure):
    _fields_ = [(n, nvfp4_tensor) for n in ("xq", "wq", "wtq", "xtq", "dyq", "dytq")]


_lib = None


def load_library(path=LIB_PATH):
    """Load libnvfp4.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libnvfp4.so not built: run nvfp4_bit_numerics_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I64, I32, U64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t
    T = ctypes.POINTER(nvfp4_tensor)
    sig = {
        "nvfp4_amax": (I32, [P, I64, I64, I32, U64, P, P]),
        "nvfp4_quantize": (I32, [P, I64, I64, ctypes.POINTER(nvfp4_quant_cfg), T, T, P]),
        "nvfp4_scale_bytes": (SZ, [I64, I64, I32]),
        "nvfp4_gemm": (I32, [T, T, P, I32, I64, P]),
        "nvfp4_gemm2": (I32, [T, T, P, I64, T, T, P, I64, P]),
        "nvfp4_gemm_amax": (I32, [T, T, P, I32, I64, P, P]),
        "nvfp4_gemm_quant": (I32, [T, T, T, P, I64, P, P]),
        "nvfp4_linear_workspace_bytes": (SZ, [I64, I64, I64]),
        "nvfp4_linear_fwd": (I32, [P, P, I64, I64, I64, U64, P, P, SZ, P]),
        "nvfp4_linear_bwd": (I32, [P, I64, I64, I64, U64, P, P, P, SZ, P]),
        "nvfp4_linear_get_views": (I32, [P, I64, I64, I64, ctypes.POINTER(nvfp4_linear_views)]),
        "nvfp4_get_status": (I32, [P]),
        "nvfp4_status_string": (ctypes.c_char_p, [I32]),
        "nvfp4_kernel_launch_count": (U64, []),
        "nvfp4_linear_fwd_noalloc": (I32, [P, P, I64, I64, I64, U64, P, P]),
        "nvfp4_debug_stall_next_gemm": (None, [I32]),
        "nvfp4_debug_stall_next_quantize": (None, [I32]),
        "nvfp4_quantize_mx": (I32, [P, I64, I64, I32, T, T, P]),
        "nvfp4_mx_scale_bytes": (SZ, [I64, I64, I32]),
        "nvfp4_linear_bf16_fwd": (I32, [P, P, I64, I64, I64, P, P]),
        "nvfp4_linear_bf16_bwd": (I32, [P, P, P, I64, I64, I64, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(fn, code):
    if code != NVFP4_OK:
        msg = load_library().nvfp4_status_string(code).decode()
        raise Nvfp4Error(fn, code, msg)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _bf16_2d(x, name):
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()):
        raise ValueError("%s must be a contiguous 2D bfloat16 CUDA tensor" % name)


class QTensor:
    """Torch-owned buffers of one quantized tensor [rows, cols] (see
    nvfp4_tensor); an MXFP4 tensor (fmt NVFP4_FORMAT_MXFP4) has no amax or
    tensor scale (None)."""

    def __init__(self, codes, scales, amax, tensor_scale, rows, cols, layout, fmt=NVFP4_FORMAT_NVFP4):
        self.codes, self.scales, self.amax, self.tensor_scale = codes, scales, amax, tensor_scale
        self.rows, self.cols, self.layout, self.fmt = rows, cols, layout, fmt

    def struct(self):
        opt = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
        return nvfp4_tensor(self.codes.data_ptr(), self.scales.data_ptr(), opt(self.amax), opt(self.tensor_scale),
                            self.rows, self.cols, self.layout, self.fmt)


def nvfp4_scale_bytes(rows, cols, layout):
    return int(load_library().nvfp4_scale_bytes(rows, cols, layout))


def empty_qtensor(rows, cols, layout=NVFP4_SCALES_MMA, device="cuda"):
    """Allocate (with torch) the buffers of a [rows, cols] NVFP4 tensor."""
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    scales = torch.zeros(nvfp4_scale_bytes(rows, cols, layout), dtype=torch.uint8, device=device)
    amax = torch.zeros(1, dtype=torch.float32, device=device)
    ts = torch.zeros(1, dtype=torch.float32, device=device)
    return QTensor(codes, scales, amax, ts, rows, cols, layout)


def nvfp4_mx_scale_bytes(rows, cols, layout):
    return int(load_library().nvfp4_mx_scale_bytes(rows, cols, layout))


def empty_mx_qtensor(rows, cols, layout=NVFP4_SCALES_MMA, device="cuda"):
    """Allocate (with torch) the buffers of a [rows, cols] MXFP4 tensor."""
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    scales = torch.zeros(nvfp4_mx_scale_bytes(rows, cols, layout), dtype=torch.uint8, device=device)
    return QTensor(codes, scales, None, None, rows, cols, layout, NVFP4_FORMAT_MXFP4)


def nvfp4_quantize_mx(x, kind=NVFP4_Q_ROWWISE, out=None, out_t=None, layout=NVFP4_SCALES_MMA, stream=None):
    """Quantize a BF16 [rows, cols] tensor to MXFP4; returns (out, out_t)
    QTensors (out_t is None unless kind is NVFP4_Q_ROWWISE_AND_TRANSPOSE)."""
    _bf16_2d(x, "x")
    rows, cols = x.shape
    if out is None:
        out = empty_mx_qtensor(cols, rows, layout, x.device) if kind == NVFP4_Q_TRANSPOSE else \
            empty_mx_qtensor(rows, cols, layout, x.device)
    if out_t is None and kind == NVFP4_Q_ROWWISE_AND_TRANSPOSE:
        out_t = empty_mx_qtensor(cols, rows, layout, x.device)
    so = out.struct()
    st = out_t.struct() if out_t is not None else None
    _check("nvfp4_quantize_mx", load_library().nvfp4_quantize_mx(
        _ptr(x), rows, cols, kind, ctypes.byref(so), ctypes.byref(st) if st is not None else None,
        _stream(stream)))
    return out, out_t


def nvfp4_amax(x, flags=NVFP4_AMAX_PLAIN, rht_seed=0, out=None, stream=None):
    """Returns a float32 tensor of 3 slots [plain, rht_rows, rht_cols]."""
    _bf16_2d(x, "x")
    if out is None:
        out = torch.zeros(3, dtype=torch.float32, device=x.device)
    _check("nvfp4_amax", load_library().nvfp4_amax(_ptr(x), x.shape[0], x.shape[1], flags, rht_seed,
                                                   _ptr(out), _stream(stream)))
    return out


def nvfp4_quantize(x, kind=NVFP4_Q_ROWWISE, rounding=NVFP4_ROUND_RNE, rht=False, seed=0, sr_stream=0,
                   sr_stream_t=0, compute_amax=True, out=None, out_t=None, layout=NVFP4_SCALES_MMA,
                   stream=None):
    """Quantize a BF16 [rows, cols] tensor; returns (out, out_t) QTensors
    (out_t is None for kinds without a transposed output)."""
    _bf16_2d(x, "x")
    rows, cols = x.shape
    if out is None:
        out = empty_qtensor(cols, rows, layout, x.device) if kind == NVFP4_Q_TRANSPOSE else \
            empty_qtensor(rows, cols, layout, x.device)
    if out_t is None and kind in (NVFP4_Q_ROWWISE_AND_TRANSPOSE, NVFP4_Q_2D):
        out_t = empty_qtensor(cols, rows, layout, x.device)
    cfg = nvfp4_quant_cfg(kind, rounding, int(bool(rht)), int(bool(compute_amax)), seed, sr_stream, sr_stream_t)
    so = out.struct()
    st = out_t.struct() if out_t is not None else None
    _check("nvfp4_quantize", load_library().nvfp4_quantize(
        _ptr(x), rows, cols, ctypes.byref(cfg), ctypes.byref(so), ctypes.byref(st) if st is not None else None,
        _stream(stream)))
    return out, out_t


def nvfp4_gemm(a, b, out=None, out_dtype=torch.bfloat16, stream=None):
    """D[M, N] = ts_a ts_b A B^T for QTensors A [M, K], B [N, K]."""
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    dt = NVFP4_OUT_F32 if out.dtype == torch.float32 else NVFP4_OUT_BF16
    sa, sb = a.struct(), b.struct()
    _check("nvfp4_gemm", load_library().nvfp4_gemm(ctypes.byref(sa), ctypes.byref(sb), _ptr(out), dt,
                                                   out.stride(0), _stream(stream)))
    return out


def nvfp4_gemm2(a0, b0, a1, b1, out0=None, out1=None, stream=None):
    """(D0, D1) = (ts A0 B0^T, ts A1 B1^T) as BF16, the two GEMMs in one launch
    when both take the CTA-pair kernel (nvfp4_gemm2 of nvfp4.h)."""
    dev = a0.codes.device
    if out0 is None:
        out0 = torch.empty((a0.rows, b0.rows), dtype=torch.bfloat16, device=dev)
    if out1 is None:
        out1 = torch.empty((a1.rows, b1.rows), dtype=torch.bfloat16, device=dev)
    s0, t0, s1, t1 = a0.struct(), b0.struct(), a1.struct(), b1.struct()
    _check("nvfp4_gemm2", load_library().nvfp4_gemm2(ctypes.byref(s0), ctypes.byref(t0), _ptr(out0), out0.stride(0),
                                                     ctypes.byref(s1), ctypes.byref(t1), _ptr(out1), out1.stride(0),
                                                     _stream(stream)))
    return out0, out1


def nvfp4_gemm_amax(a, b, out=None, out_dtype=torch.bfloat16, amax=None, stream=None):
    """nvfp4_gemm that also returns max |D| over the stored output (a float32
    device tensor of one element): (out, amax)."""
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=a.codes.device)
    dt = NVFP4_OUT_F32 if out.dtype == torch.float32 else NVFP4_OUT_BF16
    sa, sb = a.struct(), b.struct()
    _check("nvfp4_gemm_amax", load_library().nvfp4_gemm_amax(ctypes.byref(sa), ctypes.byref(sb), _ptr(out), dt,
                                                             out.stride(0), _ptr(amax), _stream(stream)))
    return out, amax


def nvfp4_gemm_quant(a, b, yq, out=None, amax_out=None, stream=None):
    """D = A B^T with D also written NVFP4-quantized into the QTensor yq
    (whose amax the caller has set); out: optional BF16 [M, N] output;
    amax_out: optional one-float tensor receiving max |D|.  Returns
    (yq, out, amax_out)."""
    sa, sb, sq = a.struct(), b.struct(), yq.struct()
    ldd = out.stride(0) if out is not None else b.rows
    _check("nvfp4_gemm_quant", load_library().nvfp4_gemm_quant(
        ctypes.byref(sa), ctypes.byref(sb), ctypes.byref(sq), _ptr(out), ldd, _ptr(amax_out), _stream(stream)))
    return yq, out, amax_out


def nvfp4_linear_workspace_bytes(M, K, N):
    return int(load_library().nvfp4_linear_workspace_bytes(M, K, N))


def linear_workspace(M, K, N, device="cuda"):
    return torch.empty(nvfp4_linear_workspace_bytes(M, K, N), dtype=torch.uint8, device=device)


def nvfp4_linear_fwd(x, w, seed, ws, y=None, stream=None):
    _bf16_2d(x, "x")
    _bf16_2d(w, "w")
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("nvfp4_linear_fwd", load_library().nvfp4_linear_fwd(
        _ptr(x), _ptr(w), M, K, N, seed, _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))
    return y


def nvfp4_linear_bwd(dy, K, seed, ws, dx=None, dw=None, stream=None):
    _bf16_2d(dy, "dy")
    M, N = dy.shape
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    if dw is None:
        dw = torch.empty((N, K), dtype=torch.bfloat16, device=dy.device)
    _check("nvfp4_linear_bwd", load_library().nvfp4_linear_bwd(
        _ptr(dy), M, K, N, seed, _ptr(dx), _ptr(dw), _ptr(ws), ws.numel(), _stream(stream)))
    return dx, dw


def nvfp4_linear_fwd_noalloc(x, w, seed, y=None, stream=None):
    """nvfp4_linear_fwd with the library's own 32 MiB device workspace, for
    callers that must not allocate a workspace (see include/nvfp4.h)."""
    _bf16_2d(x, "x")
    _bf16_2d(w, "w")
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("nvfp4_linear_fwd_noalloc", load_library().nvfp4_linear_fwd_noalloc(
        _ptr(x), _ptr(w), M, K, N, seed, _ptr(y), _stream(stream)))
    return y


def nvfp4_linear_bf16_fwd(x, w, y=None, stream=None):
    """Y = X W^T for a layer kept in BF16 (cuBLAS inside the library)."""
    _bf16_2d(x, "x")
    _bf16_2d(w, "w")
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("w must be [N, %d]" % K)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("nvfp4_linear_bf16_fwd", load_library().nvfp4_linear_bf16_fwd(_ptr(x), _ptr(w), M, K, N, _ptr(y),
                                                                         _stream(stream)))
    return y


def nvfp4_linear_bf16_bwd(dy, x, w, dx=None, dw=None, stream=None):
    """dX = dY W and dW = dY^T X for a layer kept in BF16; returns (dx, dw)."""
    for t, n in ((dy, "dy"), (x, "x"), (w, "w")):
        _bf16_2d(t, n)
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or tuple(dy.shape) != (M, N):
        raise ValueError("shapes must be dy [M, N], x [M, K], w [N, K]")
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    if dw is None:
        dw = torch.empty((N, K), dtype=torch.bfloat16, device=x.device)
    _check("nvfp4_linear_bf16_bwd", load_library().nvfp4_linear_bf16_bwd(
        _ptr(dy), _ptr(x), _ptr(w), M, K, N, _ptr(dx), _ptr(dw), _stream(stream)))
    return dx, dw


def nvfp4_linear_get_views(ws, M, K, N):
    """QTensor views (torch slices of ws) of the six quantized operands."""
    v = nvfp4_linear_views()
    _check("nvfp4_linear_get_views", load_library().nvfp4_linear_get_views(_ptr(ws), M, K, N, ctypes.byref(v)))
    base = ws.data_ptr()
    hdr = ws[:256].view(torch.float32)
    out = {}
    for name in ("xq", "wq", "wtq", "xtq", "dyq", "dytq"):
        t = getattr(v, name)
        oc, osf = t.codes - base, t.scales - base
        nsf = nvfp4_scale_bytes(t.rows, t.cols, t.scale_layout)
        codes = ws[oc:oc + t.rows * t.cols // 2].view(t.rows, t.cols // 2)
        scales = ws[osf:osf + nsf]
        ia, it = (t.amax - base) // 4, (t.tensor_scale - base) // 4
        out[name] = QTensor(codes, scales, hdr[ia:ia + 1], hdr[it:it + 1], t.rows, t.cols, t.scale_layout)
    return out


def nvfp4_get_status(stream=None):
    """Synchronises the stream; returns and clears the device status code."""
    return int(load_library().nvfp4_get_status(_stream(stream)))


def nvfp4_debug_stall_next_gemm(on=True):
    load_library().nvfp4_debug_stall_next_gemm(1 if on else 0)


def nvfp4_debug_stall_next_quantize(on=True):
    load_library().nvfp4_debug_stall_next_quantize(1 if on else 0)


def nvfp4_kernel_launch_count():
    return int(load_library().nvfp4_kernel_launch_count())
