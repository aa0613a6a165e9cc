"""The no-allocation dense GEMV entry point (qmv_int4_gs_noalloc).

It serves callers that cannot call cudaMalloc - code that must never make the
device synchronise, hosts that forbid device allocation after start-up, C
callers with nowhere to keep a workspace - by using a scratch array built into
the library. This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest

import datagen
import oracle
from tests.gpu_util import TOL_FP32, norm_err

torch = pytest.importorskip("torch")
q = pytest.importorskip("int4_group_quantized_gs64_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    q.build()
    lib = q.lib()
    f = lib.qmv_int4_gs_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, i32, i32, i32, vp, vp, i32, vp]
    f.restype = i32
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(L, wq, sc, x, y):
    N, K = wq.shape[0], wq.shape[1] * 2
    S = x.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.qmv_int4_gs_noalloc(_p(wq), _p(sc), N, K, 64, _p(x), _p(y), S, stream)


def test_matches_workspace_entry_point_on_two_calls(L):
    """Two calls in a row with different activations (and shapes) agree with
    qmv_int4_gs, the entry point that takes a caller workspace."""
    for (N, K, S, seed) in [(14336, 4096, 1, 0), (1000, 2048, 3, 1)]:
        wq, sc, x = datagen.dense_int4(N, K, S, seed=seed)
        dwq, dsc, dx = (torch.from_numpy(a).cuda() for a in (wq, sc, x))
        y = torch.full((S, N), float("nan"), device="cuda")
        assert _call_noalloc(L, dwq, dsc, dx, y) == 0
        ref = q.qmv_int4_gs(dwq, dsc, dx)
        torch.cuda.synchronize()
        yn, yr = y.cpu().numpy(), ref.cpu().numpy()
        _, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
        assert norm_err(yn, yr, den) <= TOL_FP32
        exact, _ = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
        assert norm_err(yn, exact, den) <= TOL_FP32


def test_exact_scratch_limit_multi_pass(L):
    """S * K == 65536 exactly (the factor block ends at the array's last byte)
    with S > 4, so the kernel walks the tokens in several passes."""
    N, K, S = 1000, 4096, 16
    wq, sc, x = datagen.dense_int4(N, K, S, seed=5)
    dwq, dsc, dx = (torch.from_numpy(a).cuda() for a in (wq, sc, x))
    ys = []
    for _ in range(2):
        y = torch.full((S, N), float("nan"), device="cuda")
        assert _call_noalloc(L, dwq, dsc, dx, y) == 0
        ys.append(y)
    ref = q.qmv_int4_gs(dwq, dsc, dx)
    torch.cuda.synchronize()
    exact, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
    for y in ys:
        yn = y.cpu().numpy()
        assert norm_err(yn, ref.cpu().numpy(), den) <= TOL_FP32
        assert norm_err(yn, exact, den) <= TOL_FP32
    assert torch.equal(ys[0], ys[1])


def test_rejects_sizes_beyond_the_static_scratch(L):
    N, K, S = 64, 4096, 17  # S * K = 69632 > 65536
    dwq = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    dsc = torch.ones((N, K // 64), device="cuda")
    dx = torch.ones((S, K), device="cuda")
    y = torch.full((S, N), 7.0, device="cuda")
    assert _call_noalloc(L, dwq, dsc, dx, y) == -3  # QMV_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
