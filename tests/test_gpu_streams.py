"""The layer step under CUDA graph capture and from concurrent host threads.

Outside capture, nvfp4_linear_fwd quantizes W on the library's per-device
side stream (forked from and joined back into the caller's stream); under
capture it enqueues everything on the caller's stream.  Both paths, and two
host threads driving their own layers at once, must give exactly the results
of a plain single-threaded run."""

import threading

import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from nvfp4_bit_numerics_gb300 import workloads
from tests.gpu_util import ensure_lib

pytestmark = pytest.mark.gpu

SHAPE = (512, 768, 1024)  # M, K, N: multiples of 256, the CTA-pair GEMM


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_lib()


def inputs(seed):
    M, K, N = SHAPE
    x, w, dy = workloads.layer_inputs(M, K, N, seed, 4, 30.0, 0.02, 1e-3)
    return x.cuda(), w.cuda(), dy.cuda()


def eager(x, w, dy, seed):
    M, K = x.shape
    N = w.shape[0]
    ws = B.linear_workspace(M, K, N)
    y = B.nvfp4_linear_fwd(x, w, seed, ws)
    dx, dw = B.nvfp4_linear_bwd(dy, K, seed, ws)
    torch.cuda.synchronize()
    assert B.nvfp4_get_status() == B.NVFP4_OK
    return y, dx, dw


def test_graph_capture_replays_bit_identical():
    M, K, N = SHAPE
    x, w, dy = inputs(11)
    seed = 77
    ref = eager(x, w, dy, seed)
    ws = B.linear_workspace(M, K, N)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.nvfp4_linear_fwd(x, w, seed, ws, y=y, stream=s)
        B.nvfp4_linear_bwd(dy, K, seed, ws, dx=dx, dw=dw, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.nvfp4_linear_fwd(x, w, seed, ws, y=y, stream=s)
        B.nvfp4_linear_bwd(dy, K, seed, ws, dx=dx, dw=dw, stream=s)
    for _ in range(3):
        for t in (y, dx, dw):
            t.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for got, want in zip((y, dx, dw), ref):
            assert torch.equal(got, want)
    assert B.nvfp4_get_status() == B.NVFP4_OK


def test_concurrent_host_threads():
    """Two threads, each with its own stream, workspace and layer, enqueue
    twenty steps at the same time; the shared side stream must keep them
    apart."""
    M, K, N = SHAPE
    seeds = [5, 6]
    data = [inputs(100 + i) for i in range(2)]
    refs = [eager(*data[i], seeds[i]) for i in range(2)]
    results = [None, None]
    errors = []
    start = threading.Barrier(2)

    def worker(i):
        try:
            x, w, dy = data[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                ws = B.linear_workspace(M, K, N)
                start.wait()
                for _ in range(20):
                    y = B.nvfp4_linear_fwd(x, w, seeds[i], ws, stream=s)
                    dx, dw = B.nvfp4_linear_bwd(dy, K, seeds[i], ws, stream=s)
                s.synchronize()
            results[i] = (y, dx, dw)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert B.nvfp4_get_status() == B.NVFP4_OK
    for i in range(2):
        for got, want in zip(results[i], refs[i]):
            assert torch.equal(got, want), i


def test_graph_capture_of_the_further_paths():
    """The MXFP4 quantize + GEMM, the GEMM with its output quantized in the
    epilogue and the BF16 layer step, captured into one graph after a first
    eager run (which creates the library's cuBLAS handle and sets kernel
    attributes): every replay gives the eager results exactly."""
    M, K, N = SHAPE
    x, w, dy = inputs(21)
    s = torch.cuda.Stream()
    qx, qw = B.empty_mx_qtensor(M, K), B.empty_mx_qtensor(N, K)
    nqx, nqw = B.empty_qtensor(M, K), B.empty_qtensor(N, K)
    y_mx = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y_bf = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    y_nv = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    yq = B.empty_qtensor(M, N)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")

    def work():
        B.nvfp4_quantize_mx(x, out=qx, stream=s)
        B.nvfp4_quantize_mx(w, out=qw, stream=s)
        B.nvfp4_gemm(qx, qw, out=y_mx, stream=s)
        B.nvfp4_quantize(x, B.NVFP4_Q_ROWWISE, out=nqx, stream=s)
        B.nvfp4_quantize(w, B.NVFP4_Q_2D, out=nqw, stream=s)
        B.nvfp4_gemm_quant(nqx, nqw, yq, out=y_nv, amax_out=amax, stream=s)
        B.nvfp4_linear_bf16_fwd(x, w, y=y_bf, stream=s)
        B.nvfp4_linear_bf16_bwd(dy, x, w, dx=dx, dw=dw, stream=s)

    outs = (y_mx, qx.codes, qx.scales, y_nv, yq.codes, yq.scales, amax, y_bf, dx, dw)
    with torch.cuda.stream(s):
        yq.amax.fill_(4.0)  # a given (delayed) amax for the quantized output
        work()
    torch.cuda.synchronize()
    ref = [t.clone() for t in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        work()
    for _ in range(2):
        for t in outs:
            t.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for got, want in zip(outs, ref):
            assert torch.equal(got, want)
    assert B.nvfp4_get_status() == B.NVFP4_OK
