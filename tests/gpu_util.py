"""Helpers shared by the GPU parity tests: build/load the library, move
tensors between torch and the oracle's numpy representation."""

import numpy as np
import torch

from nvfp4_bit_numerics_gb300 import binding, build, workloads
from oracle import formats, quant


def ensure_lib():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need CUDA")
    build.build()
    return binding.load_library()


def to_gpu_bf16(t):
    return t.contiguous().cuda()


def f32(t):
    """bf16 torch tensor (any device) -> float32 numpy (exact)."""
    return t.detach().to("cpu", torch.float32).numpy()


def gpu_qtensor_to_numpy(q):
    """QTensor on the GPU -> (codes [rows, cols/2] u8, linear scales
    [rows, cols/16] u8, amax float32, ts float32)."""
    torch.cuda.synchronize()
    codes = q.codes.cpu().numpy()
    sc = q.scales.cpu().numpy()
    if q.layout == binding.NVFP4_SCALES_MMA:
        sc = quant.unswizzle_scales(sc, q.rows, q.cols // 16)
    else:
        sc = sc.reshape(q.rows, q.cols // 16)
    return codes, sc, np.float32(q.amax.cpu().item()), np.float32(q.tensor_scale.cpu().item())


def assert_q_equal(gpu_q, ref, rows=None, what=""):
    """Bit-exact comparison of a GPU QTensor with an oracle dict."""
    codes, sc, amax, ts = gpu_qtensor_to_numpy(gpu_q)
    if rows is not None:
        codes, sc = codes[rows], sc[rows]
    rc, rs = ref["codes"], ref["scales"]
    assert amax.view(np.uint32) == np.float32(ref["amax"]).view(np.uint32), (what, amax, ref["amax"])
    assert ts.view(np.uint32) == np.float32(ref["ts"]).view(np.uint32), (what, ts, ref["ts"])
    bad_s = np.argwhere(sc != rs)
    assert bad_s.size == 0, "%s: %d scale mismatches, first %s gpu=%d ref=%d" % (
        what, len(bad_s), bad_s[0], sc[tuple(bad_s[0])], rs[tuple(bad_s[0])])
    bad = np.argwhere(codes != rc)
    assert bad.size == 0, "%s: %d code-byte mismatches of %d, first %s gpu=%#x ref=%#x" % (
        what, len(bad), codes.size, bad[0], codes[tuple(bad[0])], rc[tuple(bad[0])])


def rel_fro(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    n = np.linalg.norm(ref)
    return np.linalg.norm(a - ref) / (n if n > 0 else 1.0)


def outlier_tensor(rows, cols, seed, sigma=1.0):
    """bf16 CPU tensor ~N(0, sigma) with a few large entries and some exact
    zeros / negative zeros, for parity edge coverage."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(sigma)
    n = max(1, x.size // 300)
    idx = rng.choice(x.size, n, replace=False)
    x.reshape(-1)[idx] *= 60
    z = rng.choice(x.size, max(1, x.size // 500), replace=False)
    x.reshape(-1)[z[: len(z) // 2]] = 0.0
    x.reshape(-1)[z[len(z) // 2:]] = -0.0
    return workloads.to_bf16(x)
