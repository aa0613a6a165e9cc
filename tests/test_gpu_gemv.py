"""Dense int4-gs64 and int8-row GEMV on the GPU against the fp64 oracle."""
import numpy as np
import pytest

import datagen
import oracle
from tests.gpu_util import TOL_FP32, norm_err

torch = pytest.importorskip("torch")
q = pytest.importorskip("int4_group_quantized_gs64_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    q.build()
    q.lib()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_int4(wq, sc, x):
    y = q.qmv_int4_gs(dev(wq), dev(sc), dev(x))
    torch.cuda.synchronize()
    return y.cpu().numpy()


def run_int8(w, r, x):
    y = q.qmv_int8_row(dev(w), dev(r), dev(x))
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K", [(1024, 1024), (14336, 4096)], ids=["1024x1024", "14336x4096"])
def test_int4_workloads(N, K):
    wq, sc, x = datagen.dense_int4(N, K, 1)
    y = run_int4(wq, sc, x)
    ref, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
    assert norm_err(y, ref, den) <= TOL_FP32


def test_int8_workload():
    w, r, x = datagen.dense_int8(14336, 4096, 1)
    y = run_int8(w, r, x)
    ref, den = oracle.qmv_int8_row(w, r, x)
    assert norm_err(y, ref, den) <= TOL_FP32


# (the single-launch kernel takes S <= 4 with S * K <= 16384: both its 32 KB
# and 64 KB activation tables appear below, and larger S * K take the others)
SHAPES = [(1, 64, 1), (17, 64, 3), (100, 192, 5), (63, 1088, 4), (65, 4096, 8), (33, 640, 16),
          (40, 256, 17), (16, 16384, 2), (128, 2048, 33), (1000, 4096, 4), (2048, 4096, 3),
          (48, 16384, 1)]


@pytest.mark.parametrize("N,K,S", SHAPES)
def test_int4_shapes(N, K, S):
    rng = np.random.default_rng(N * 7919 + K + S)
    wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
    x = rng.normal(size=(S, K)).astype(np.float32)
    y = run_int4(wq, sc, x)
    ref, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
    assert norm_err(y, ref, den) <= TOL_FP32


# Shapes of the tensor-map kernel (N a multiple of 256, K/64 a multiple of 4):
# one tile and one stage, several passes of 8 tokens with a ragged last pass,
# and long rows whose stages are split between CTAs.
TMA_SHAPES = [(256, 256, 1), (512, 1024, 8), (768, 4096, 9), (2048, 2048, 17), (256, 16384, 2),
              (14336, 4096, 8)]


@pytest.mark.parametrize("N,K,S", TMA_SHAPES)
def test_int4_tma_shapes(N, K, S):
    rng = np.random.default_rng(N * 131 + K + S)
    wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
    x = rng.normal(size=(S, K)).astype(np.float32)
    ws = torch.full((q.qmv_gemv_workspace_bytes(K, S),), 0xFF, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the workspace left by the first
        y = q.qmv_int4_gs(dev(wq), dev(sc), dev(x), ws=ws)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).cpu()[0]) == 0  # status word: no wait timed out
        ref, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
        assert norm_err(y.cpu().numpy(), ref, den) <= TOL_FP32


@pytest.mark.parametrize("N,K,S", [(14336, 4096, 8), (256, 16384, 2)])
def test_int4_tma_split_items_any_arrival_order(N, K, S):
    """Dense mode of the tensor-map kernel with the compute warps of odd CTAs
    started 100 us late (qmv_test_split_skew): the items two CTAs share are
    finished by whichever arrives last, and y is bit-identical to the
    undelayed call's."""
    rng = np.random.default_rng(N + K + S + 5)
    wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
    x = rng.normal(size=(S, K)).astype(np.float32)
    ws = torch.zeros((q.qmv_gemv_workspace_bytes(K, S),), dtype=torch.uint8, device="cuda")
    dw, ds, dx = dev(wq), dev(sc), dev(x)
    ref = q.qmv_int4_gs(dw, ds, dx, ws=ws).cpu().numpy()
    old = q.qmv_test_split_skew(100_000)
    try:
        a = q.qmv_int4_gs(dw, ds, dx, ws=ws).cpu().numpy()
    finally:
        q.qmv_test_split_skew(old)
    b = q.qmv_int4_gs(dw, ds, dx, ws=ws).cpu().numpy()
    assert int(ws[:4].view(torch.int32).cpu()[0]) == 0
    assert np.array_equal(a, ref)
    assert np.array_equal(b, ref)
    ref64, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
    assert norm_err(a, ref64, den) <= TOL_FP32


# Pairs of matrices against one x: the pages' q_a + kv_a shape 6144 -> (2048, 576),
# ragged last row tiles (N not a multiple of 256), several token passes, and
# a pair that does not qualify for the tensor-map kernel (two GEMVs).
PAIR_SHAPES = [(2048, 576, 6144, 1), (256, 256, 256, 1), (512, 48, 1024, 3), (1024, 1040, 2048, 9),
               (100, 36, 192, 2)]


@pytest.mark.parametrize("N0,N1,K,S", PAIR_SHAPES)
def test_int4_pair(N0, N1, K, S):
    rng = np.random.default_rng(N0 + 3 * N1 + K + S)
    mats = []
    for N in (N0, N1):
        wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
        sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
        mats.append((wq, sc))
    x = rng.normal(size=(S, K)).astype(np.float32)
    ws = torch.full((q.qmv_gemv_workspace_bytes(K, S),), 0xFF, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the workspace left by the first
        y0, y1 = q.qmv_int4_gs_pair(dev(mats[0][0]), dev(mats[0][1]), dev(mats[1][0]),
                                    dev(mats[1][1]), dev(x), ws=ws)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).cpu()[0]) == 0
        for y, (wq, sc) in zip((y0, y1), mats):
            ref, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
            assert norm_err(y.cpu().numpy(), ref, den) <= TOL_FP32


# int3-g64 two-plane rows: one and many groups, ragged row counts, several
# token passes (4 a pass), the 14336 x 4096 shape, K = 16384 and 24576 (x staged
# in shared memory, fewer tokens a pass) and K = 32768 and 65536 (x read from
# global memory). Up to 4 tokens with K a multiple of 256 and x's units within
# 64 KB take the warp-MMA single launch: 14336 x 4096, a ragged last row tile
# (1000, 33 rows), one 4-group stage for one warp only (K 256), warps with no
# groups (K 4352: 68 groups as 12 a warp; K 7168), and the 64 KB unit table
# (K x tokens = 16384: 4096 x 4 and 8192 x 2; K 16384 x 2 is past it).
INT3_SHAPES = [(1, 64, 1), (17, 192, 3), (100, 1024, 5), (256, 4096, 8), (14336, 4096, 1),
               (9, 32768, 3), (5, 65536, 1), (40, 24576, 2),
               (64, 16384, 2), (1000, 1024, 4), (33, 256, 2), (300, 4352, 3), (2048, 7168, 1),
               (80, 4096, 4), (64, 8192, 2)]


@pytest.mark.parametrize("N,K,S", INT3_SHAPES)
def test_int3_shapes(N, K, S):
    rng = np.random.default_rng(N * 17 + K + S)
    wq3 = rng.integers(0, 256, size=(N, K // 64 * 24), dtype=np.uint8)
    sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
    x = rng.normal(size=(S, K)).astype(np.float32)
    y = q.qmv_int3_gs(dev(wq3), dev(sc), dev(x))
    torch.cuda.synchronize()
    ref, den = oracle.qmv_int3_gs(wq3, sc, x)
    assert norm_err(y.cpu().numpy(), ref, den) <= TOL_FP32


@pytest.mark.parametrize("K", [512, 2048])
def test_int3_all_codes_bit_exact(K):
    """Every code at every position, dyadic scales, small-integer x: exact in
    fp32 too (one x block a row at K = 512, several at 2048)."""
    rng = np.random.default_rng(13 + K)
    N = 40
    vals = rng.integers(-4, 4, size=(N, K)).astype(np.int8)
    wq3 = np.stack([oracle.pack_int3(vals[i]) for i in range(N)])
    s = (2.0 ** rng.integers(-6, 2, size=(N, K // 64))).astype(np.float32)
    x = rng.integers(-20, 21, size=(3, K)).astype(np.float32)
    y = q.qmv_int3_gs(dev(wq3), dev(s), dev(x))
    torch.cuda.synchronize()
    ref, _ = oracle.qmv_int3_gs(wq3, s, x)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


def test_int3_weights_not_16_byte_aligned():
    """Weights 4 bytes past a 16-byte boundary (the entry point asks for 4)."""
    rng = np.random.default_rng(23)
    N, K, S = 96, 4096, 2
    rb = K // 64 * 24
    flat = torch.from_numpy(rng.integers(0, 256, size=N * rb + 16, dtype=np.uint8)).cuda()
    wq3 = flat[4:4 + N * rb].view(N, rb)
    assert wq3.data_ptr() % 16 == 4
    sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
    x = rng.normal(size=(S, K)).astype(np.float32)
    y = q.qmv_int3_gs(wq3, dev(sc), dev(x))
    torch.cuda.synchronize()
    ref, den = oracle.qmv_int3_gs(wq3.cpu().numpy(), sc, x)
    assert norm_err(y.cpu().numpy(), ref, den) <= TOL_FP32


def test_int3_extreme_activations():
    """Activations from 1e-30 to 1e30 (one magnitude a group) and an all-zero
    group: each group gets its own power-of-two factor before the fp16 split."""
    rng = np.random.default_rng(17)
    N, K, S = 48, 1024, 3
    wq3 = rng.integers(0, 256, size=(N, K // 64 * 24), dtype=np.uint8)
    sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
    mag = 10.0 ** rng.integers(-30, 31, size=(S, K // 64))
    x = (rng.normal(size=(S, K // 64, 64)) * mag[:, :, None]).reshape(S, K).astype(np.float32)
    x[:, 64:128] = 0.0
    y = q.qmv_int3_gs(dev(wq3), dev(sc), dev(x))
    torch.cuda.synchronize()
    ref, den = oracle.qmv_int3_gs(wq3, sc, x)
    assert np.all(np.isfinite(y.cpu().numpy()))
    assert norm_err(y.cpu().numpy(), ref, den) <= TOL_FP32


@pytest.mark.parametrize("N,K,S", SHAPES)
def test_int8_shapes(N, K, S):
    rng = np.random.default_rng(N * 31 + K + S)
    w = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    r = np.abs(rng.normal(0, 0.01, size=N)).astype(np.float32)
    x = rng.normal(size=(S, K)).astype(np.float32)
    y = run_int8(w, r, x)
    ref, den = oracle.qmv_int8_row(w, r, x)
    assert norm_err(y, ref, den) <= TOL_FP32


def test_int4_all_equal_nibbles_bit_exact():
    """nibble == c, dyadic scales, small-integer x: every step is exact in fp32 too."""
    rng = np.random.default_rng(5)
    N, K = 96, 512
    x = rng.integers(-20, 21, size=(2, K)).astype(np.float32)
    s = (2.0 ** rng.integers(-8, 2, size=(N, K // 64))).astype(np.float32)
    for c in (0, 3, 8, 15):
        wq = np.full((N, K // 2), c | (c << 4), np.uint8)
        y = run_int4(wq, s, x)
        ref = oracle.qmv_int4_gs(wq, s, x, 64)
        assert np.array_equal(y.astype(np.float64), ref), c
        if c == 8:
            assert not np.any(y)


def test_zero_and_extreme_activations():
    rng = np.random.default_rng(9)
    N, K = 80, 1024
    wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
    x = np.zeros((1, K), np.float32)
    assert not np.any(run_int4(wq, sc, x))
    for mag in (1e-30, 1e-6, 1e6, 1e30):
        x = (rng.normal(size=(2, K)) * mag).astype(np.float32)
        ref, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
        assert norm_err(run_int4(wq, sc, x), ref, den) <= TOL_FP32, mag
    # one huge outlier among unit values
    x = rng.normal(size=(1, K)).astype(np.float32)
    x[0, 17] = 3e4
    ref, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
    assert norm_err(run_int4(wq, sc, x), ref, den) <= TOL_FP32


def test_deterministic():
    wq, sc, x = datagen.dense_int4(4096, 4096, 3)
    a = run_int4(wq, sc, x)
    b = run_int4(wq, sc, x)
    assert np.array_equal(a, b)


def test_bad_arguments_leave_output_untouched():
    y = torch.full((1, 64), 7.0, device="cuda")
    wq = torch.zeros((64, 48), dtype=torch.uint8, device="cuda")   # K = 96: not a multiple of 64
    sc = torch.ones((64, 1), device="cuda")
    x = torch.ones((1, 96), device="cuda")
    with pytest.raises(q.QmvError):
        q.qmv_int4_gs(wq, sc, x, y=y)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


# ------------------------------------------------------------------ bf16 outputs

def bf16_rne(y32):
    """fp32 -> bf16 bit patterns, round to nearest, ties to even (finite inputs)."""
    b = np.ascontiguousarray(y32, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def half_ulp_bf16(v):
    """Half the spacing of bf16 values at |v| (8 significand bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), np.finfo(np.float32).tiny)))
    return np.ldexp(1.0, (e - 8).astype(int))


def check_bf16(ybf, y32, ref, den):
    bits = ybf.view(torch.int16).cpu().numpy().view(np.uint16)
    # the fp32 result of the same kernel, rounded here: equal bit for bit
    assert np.array_equal(bits, bf16_rne(y32))
    # and within the fp32 tolerance plus half a bf16 ulp of the exact result
    g = bf16_to_f64(bits)
    bound = TOL_FP32 * den + half_ulp_bf16(np.maximum(np.abs(g), np.abs(ref)))
    assert np.all(np.abs(g - ref) <= bound)


@pytest.mark.parametrize("N,K,S", [(14336, 4096, 1), (1024, 1024, 1), (512, 1024, 9),
                                   (1000, 2048, 3), (63, 1088, 4), (40, 256, 17)])
def test_int4_bf16_output(N, K, S):
    """qmv_int4_gs_bf16 on the tensor-map path (N % 16 == 0) and the cp.async
    path (other N), one and several token passes."""
    wq, sc, x = datagen.dense_int4(N, K, S, seed=N + K + S)
    ws = torch.empty(q.qmv_gemv_workspace_bytes(K, S), dtype=torch.uint8, device="cuda")
    dwq, dsc, dx = dev(wq), dev(sc), dev(x)
    y32 = q.qmv_int4_gs(dwq, dsc, dx, ws=ws)
    ybf = q.qmv_int4_gs_bf16(dwq, dsc, dx, ws=ws)
    torch.cuda.synchronize()
    ref, den = oracle.qmv_int4_gs(wq, sc, x, 64, with_den=True)
    check_bf16(ybf, y32.cpu().numpy(), ref, den)


@pytest.mark.parametrize("N,K,S", [(14336, 4096, 1), (100, 192, 5), (33, 640, 16), (300, 4096, 4)])
def test_int8_bf16_output(N, K, S):
    w, r, x = datagen.dense_int8(N, K, S, seed=N + K + S)
    ws = torch.empty(q.qmv_gemv_workspace_bytes(K, S), dtype=torch.uint8, device="cuda")
    dw, dr, dx = dev(w), dev(r), dev(x)
    y32 = q.qmv_int8_row(dw, dr, dx, ws=ws)
    ybf = q.qmv_int8_row_bf16(dw, dr, dx, ws=ws)
    torch.cuda.synchronize()
    ref, den = oracle.qmv_int8_row(w, r, x)
    check_bf16(ybf, y32.cpu().numpy(), ref, den)
