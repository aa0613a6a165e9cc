"""Seeded synthetic inputs shared by the oracle driver, the GPU tests and the bench.

Nothing here computes any part of the quantized GEMV / MoE path: it only draws
random numbers (see ``datagen.c`` for the generator) and lays them out in the
shapes of the five workloads:

* ``dense_int4``: int4-gs64 GEMV inputs. Bytes uniform 0..255 (two offset-binary
  nibbles each), fp32 group scales ``|N(0, 0.02)| + 1e-4``, activations ``N(0, 1)``.
* ``dense_int8``: int8 weights uniform in [-127, 127], fp32 row scales ``|N(0, 0.01)|``.
* ``moe_weights``: per-expert stacked gate+up ``[2I][H/2]`` and down ``[H][I/2]``
  int4 tensors plus their ``[rows][K/64]`` scales, regenerable per expert.
* ``moe_inputs``: activations (fp32, or bf16 bits for the prefill batch) and
  router logits ``N(0, 1)``, optionally raised by +2 on a seeded set of "hot"
  experts.

Every tensor has a fixed stream id, so a sub-range (one expert, a few tokens)
can be regenerated alone with identical values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "datagen.c")
_LIB = os.path.join(_HERE, "libdatagen.so")

SEED = 0

# Fixed stream id per tensor.
STREAM = {
    "wq": 1, "scales": 2, "x": 3, "w8": 4, "rscale": 5,
    "gu_q": 10, "gu_s": 11, "dn_q": 12, "dn_s": 13,
    "moe_x": 14, "logits": 15, "hot": 16,
}

# The five workloads (sizes only; the names say what they are).
WORKLOADS = {
    0: dict(name="int4-gs64 GEMV 1024x1024, 1 token", kind="dense", N=1024, K=1024, S=1),
    1: dict(name="int4-gs64 / int8-row GEMV 14336x4096, 1 token", kind="dense", N=14336, K=4096, S=1),
    2: dict(name="MoE decode H2048 E256 I512 top8, 1 token", kind="moe", H=2048, E=256, I=512,
            k=8, T=1, hot=0, xdtype="f32"),
    3: dict(name="MoE decode H6144 E160 I2048 top8, 8 tokens, 16 hot experts", kind="moe", H=6144,
            E=160, I=2048, k=8, T=8, hot=16, xdtype="f32"),
    4: dict(name="MoE prefill H6144 E160 I2048 top8, 512 tokens bf16", kind="moe", H=6144, E=160,
            I=2048, k=8, T=512, hot=0, xdtype="bf16"),
}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``libdatagen.so`` with the host C compiler (atomic replace)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64 = ctypes.c_uint64
        vp = ctypes.c_void_p
        lib.dg_bits.argtypes = [u64, u64, u64, u64, vp]
        lib.dg_u8.argtypes = [u64, u64, u64, u64, vp]
        lib.dg_int8_sym.argtypes = [u64, u64, u64, u64, ctypes.c_int, vp]
        lib.dg_normal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double, vp]
        lib.dg_absnormal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double, vp]
        lib.dg_normal_bf16.argtypes = [u64, u64, u64, u64, ctypes.c_double, vp]
        lib.dg_choose.argtypes = [u64, u64, ctypes.c_int, ctypes.c_int, vp, vp]
        lib.dg_choose.restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- primitives

def bits(stream: int, n: int, start: int = 0, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _L().dg_bits(seed, stream, start, n, _p(out))
    return out


def u8(stream: int, shape, start: int = 0, seed: int = SEED) -> np.ndarray:
    out = np.empty(shape, np.uint8)
    _L().dg_u8(seed, stream, start, out.size, _p(out))
    return out


def int8_sym(stream: int, shape, lim: int = 127, start: int = 0, seed: int = SEED) -> np.ndarray:
    out = np.empty(shape, np.int8)
    _L().dg_int8_sym(seed, stream, start, out.size, lim, _p(out))
    return out


def normal_f32(stream: int, shape, std: float = 1.0, mean: float = 0.0, start: int = 0,
               seed: int = SEED) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _L().dg_normal_f32(seed, stream, start, out.size, mean, std, _p(out))
    return out


def absnormal_f32(stream: int, shape, std: float, add: float = 0.0, start: int = 0,
                  seed: int = SEED) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _L().dg_absnormal_f32(seed, stream, start, out.size, std, add, _p(out))
    return out


def normal_bf16_bits(stream: int, shape, std: float = 1.0, start: int = 0,
                     seed: int = SEED) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    _L().dg_normal_bf16(seed, stream, start, out.size, std, _p(out))
    return out


def choose(stream: int, n_total: int, n_pick: int, seed: int = SEED) -> np.ndarray:
    out = np.empty(n_pick, np.int32)
    scratch = np.empty(max(n_total, 1), np.int32)
    if _L().dg_choose(seed, stream, n_total, n_pick, _p(out), _p(scratch)) != 0:
        raise ValueError("bad sizes for choose")
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to fp32 (exact)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- workloads

def dense_int4(N: int, K: int, S: int = 1, seed: int = SEED):
    """int4-gs64 GEMV inputs: (wq [N][K/2] u8, scales [N][K/64] f32, x [S][K] f32)."""
    wq = u8(STREAM["wq"], (N, K // 2), seed=seed)
    sc = absnormal_f32(STREAM["scales"], (N, K // 64), std=0.02, add=1e-4, seed=seed)
    x = normal_f32(STREAM["x"], (S, K), seed=seed)
    return wq, sc, x


def dense_int8(N: int, K: int, S: int = 1, seed: int = SEED):
    """int8 per-row GEMV inputs: (w [N][K] i8, row_scale [N] f32, x [S][K] f32)."""
    w = int8_sym(STREAM["w8"], (N, K), 127, seed=seed)
    r = absnormal_f32(STREAM["rscale"], (N,), std=0.01, add=0.0, seed=seed)
    x = normal_f32(STREAM["x"], (S, K), seed=seed)
    return w, r, x


def moe_weights(E: int, H: int, I: int, experts=None, seed: int = SEED):
    """Expert weights, all experts or only those listed (in list order).

    gu_q [n][2I][H/2] u8 (gate rows 0..I-1 then up rows I..2I-1), gu_s [n][2I][H/64],
    dn_q [n][H][I/2] u8, dn_s [n][H][I/64]; scales are |N(0, 0.02)| + 1e-4.
    """
    ex = list(range(E)) if experts is None else [int(e) for e in experts]
    n = len(ex)
    gq_sz, gs_sz = 2 * I * (H // 2), 2 * I * (H // 64)
    dq_sz, ds_sz = H * (I // 2), H * (I // 64)
    out = dict(
        gu_q=np.empty((n, 2 * I, H // 2), np.uint8),
        gu_s=np.empty((n, 2 * I, H // 64), np.float32),
        dn_q=np.empty((n, H, I // 2), np.uint8),
        dn_s=np.empty((n, H, I // 64), np.float32),
    )
    if experts is None:
        out["gu_q"][...] = u8(STREAM["gu_q"], out["gu_q"].shape, seed=seed)
        out["gu_s"][...] = absnormal_f32(STREAM["gu_s"], out["gu_s"].shape, 0.02, 1e-4, seed=seed)
        out["dn_q"][...] = u8(STREAM["dn_q"], out["dn_q"].shape, seed=seed)
        out["dn_s"][...] = absnormal_f32(STREAM["dn_s"], out["dn_s"].shape, 0.02, 1e-4, seed=seed)
        return out
    for i, e in enumerate(ex):
        if not 0 <= e < E:
            raise ValueError("expert index out of range")
        out["gu_q"][i] = u8(STREAM["gu_q"], out["gu_q"].shape[1:], start=e * gq_sz, seed=seed)
        out["gu_s"][i] = absnormal_f32(STREAM["gu_s"], out["gu_s"].shape[1:], 0.02, 1e-4,
                                       start=e * gs_sz, seed=seed)
        out["dn_q"][i] = u8(STREAM["dn_q"], out["dn_q"].shape[1:], start=e * dq_sz, seed=seed)
        out["dn_s"][i] = absnormal_f32(STREAM["dn_s"], out["dn_s"].shape[1:], 0.02, 1e-4,
                                       start=e * ds_sz, seed=seed)
    return out


def hot_experts(E: int, n_hot: int, seed: int = SEED) -> np.ndarray:
    return np.sort(choose(STREAM["hot"], E, n_hot, seed=seed))


def moe_inputs(T: int, E: int, H: int, hot: int = 0, xdtype: str = "f32", seed: int = SEED,
               token_start: int = 0):
    """Router logits [T][E] fp32 (N(0,1), +2 on ``hot`` seeded experts) and activations
    x [T][H] (fp32, or bf16 bit patterns when ``xdtype == 'bf16'``)."""
    logits = normal_f32(STREAM["logits"], (T, E), start=token_start * E, seed=seed)
    if hot:
        logits[:, hot_experts(E, hot, seed)] += np.float32(2.0)
    if xdtype == "bf16":
        x = normal_bf16_bits(STREAM["moe_x"], (T, H), start=token_start * H, seed=seed)
    else:
        x = normal_f32(STREAM["moe_x"], (T, H), start=token_start * H, seed=seed)
    return x, logits
