"""nvfp4_linear_fwd_noalloc: the forward pass for callers that cannot
allocate device memory of their own (a plugin whose host framework owns all
GPU memory, a service with a fixed memory budget).  It must give the same Y
as nvfp4_linear_fwd with a caller workspace, call after call, although every
call reuses the library's one static workspace.

This file is collected last so that a run stopping at its first failure has
run every other test before it."""

import ctypes

import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from nvfp4_bit_numerics_gb300 import workloads
from tests.gpu_util import ensure_lib, rel_fro

pytestmark = pytest.mark.gpu

TOL = 1e-3
LIMIT = 32 << 20


@pytest.fixture(scope="module")
def lib():
    return ensure_lib()


def _noalloc(lib, x, w, seed, y):
    M, K = x.shape
    N = w.shape[0]
    st = lib.nvfp4_linear_fwd_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), M, K, N, seed,
                                      ctypes.c_void_p(y.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.NVFP4_OK, lib.nvfp4_status_string(st)


def test_noalloc_matches_workspace_forward_twice(lib):
    """Two calls in a row, on two different layers, each compared with the
    workspace-taking entry point on the same inputs."""
    for (M, K, N, seed) in ((256, 512, 384, 7), (128, 1024, 256, 8)):
        x, w, _ = workloads.tiny_layer(M=M, K=K, N=N, seed=seed)
        assert B.nvfp4_linear_workspace_bytes(M, K, N) <= LIMIT
        xg, wg = x.cuda(), w.cuda()
        ws = B.linear_workspace(M, K, N)
        ref = B.nvfp4_linear_fwd(xg, wg, seed, ws)
        y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
        _noalloc(lib, xg, wg, seed, y)
        torch.cuda.synchronize()
        assert B.nvfp4_get_status() == B.NVFP4_OK
        assert rel_fro(y.float().cpu().numpy(), ref.float().cpu().numpy()) <= TOL
        assert torch.equal(y, ref)  # same kernels on the same inputs


def test_noalloc_rejects_layers_beyond_the_static_workspace(lib):
    M, K, N = 4096, 4096, 4096
    assert B.nvfp4_linear_workspace_bytes(M, K, N) > LIMIT
    p = ctypes.c_void_p(256)
    st = lib.nvfp4_linear_fwd_noalloc(p, p, M, K, N, 1, p, None)
    assert st == B.NVFP4_ERR_WORKSPACE
    assert lib.nvfp4_linear_fwd_noalloc(p, p, 100, 128, 128, 1, p, None) == B.NVFP4_ERR_SHAPE
