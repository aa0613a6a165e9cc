"""fp64 CPU oracle for the int4-gs64 / int8 GEMV and the MoE expert FFN.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers. The CUDA library never
imports, links or runs anything in this folder, and this folder never touches
the CUDA library.

The arithmetic lives in ``qmv_oracle.c`` (plain C, every accumulation in
double); this module only builds it with the host C compiler and marshals
numpy arrays. Pages followed (colibri pull requests):

* PR #418 "Vulkan backend: expert tier + dense + MLA attention on any Vulkan
  1.2 GPU": int4 decodes as nibble - 8 (commit "opt-in Vulkan int4/int8
  quantized GEMV"); one scale per 64-wide group applied to the group partial
  (commit "grouped scales in the Vulkan kernels", fmt 4); hidden =
  silu(gate x) * up x (commit "qmatmul_gate_up.comp"); K experts, gate+up then
  down (commit "coli_vk_expert_group").
* PR #1338 "qwen36: Vulkan expert tier, and staged device-local uploads":
  int4-gs64 is fmt 4 / group 64 at half a byte per element; expert outputs are
  combined by weighted accumulation (fake-Vulkan gate comment).

Readings where the pages are silent are listed in ``qmv_oracle.c`` (R1-R5).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB, defines=()) -> str:
    """Compile the oracle with the host C compiler (strict IEEE double, no contraction)."""
    if (not force and out == _LIB and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-ffp-contract=off",
           *[f"-D{d}" for d in defines], src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.orc_set_threads.argtypes = [i32]
    lib.orc_get_threads.restype = i32
    lib.orc_unpack_int4.argtypes = [vp, i64, vp]
    lib.orc_pack_int4.argtypes = [vp, i64, vp]
    lib.orc_pack_int4.restype = i32
    lib.orc_dequant_int4.argtypes = [vp, vp, i32, i32, i32, vp]
    lib.orc_qmv_int4_gs.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp]
    lib.orc_qmv_int4_gs_absden.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp]
    lib.orc_matvec_f64.argtypes = [vp, i32, i32, vp, i32, vp]
    lib.orc_qmv_int8_row.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp]
    lib.orc_unpack_int3.argtypes = [vp, i64, vp]
    lib.orc_pack_int3.argtypes = [vp, i64, vp]
    lib.orc_pack_int3.restype = i32
    lib.orc_qmv_int3_gs.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp]
    lib.orc_route_topk.argtypes = [vp, i32, i32, i32, vp, vp]
    lib.orc_route_topk.restype = i32
    lib.orc_group.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
    lib.orc_group.restype = i32
    lib.orc_moe_ffn.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, i32, vp, vp, i32,
                                vp, vp, vp, vp]
    return lib


def load(path: str | None = None):
    """The oracle library (built on first use). ``path`` loads a variant build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def set_threads(n: int) -> None:
    load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(load().orc_get_threads())


# ------------------------------------------------------------------ a1

def unpack_int4(packed, lib=None) -> np.ndarray:
    """Offset-binary decode: values = nibble - 8, low nibble first (int8 array)."""
    lib = lib or load()
    b = _c(packed, np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.int8)
    lib.orc_unpack_int4(_p(b), out.size, _p(out))
    return out


def pack_int4(values, lib=None) -> np.ndarray:
    lib = lib or load()
    v = _c(values, np.int8)
    out = np.empty(v.shape[:-1] + (v.shape[-1] // 2,), np.uint8)
    if lib.orc_pack_int4(_p(v), v.size, _p(out)) != 0:
        raise ValueError("values outside [-8, 7] or odd length")
    return out


def dequant_int4(wq, scales, gs: int = 64, lib=None) -> np.ndarray:
    lib = lib or load()
    wq, scales = _c(wq, np.uint8), _c(scales, np.float32)
    N, K = wq.shape[0], wq.shape[1] * 2
    W = np.empty((N, K), np.float64)
    lib.orc_dequant_int4(_p(wq), _p(scales), N, K, gs, _p(W))
    return W


# ------------------------------------------------------------------ a2 / a3

def qmv_int4_gs(wq, scales, x, gs: int = 64, with_den: bool = False, lib=None):
    """Form (i): y[S][N] (float64); optionally also the |deq*x| denominators."""
    lib = lib or load()
    wq, scales, x = _c(wq, np.uint8), _c(scales, np.float32), _c(np.atleast_2d(x), np.float32)
    N, K, S = wq.shape[0], wq.shape[1] * 2, x.shape[0]
    y = np.empty((S, N), np.float64)
    lib.orc_qmv_int4_gs(_p(wq), _p(scales), N, K, gs, _p(x), S, _p(y))
    if not with_den:
        return y
    den = np.empty((S, N), np.float64)
    lib.orc_qmv_int4_gs_absden(_p(wq), _p(scales), N, K, gs, _p(x), S, _p(den))
    return y, den


def matvec_f64(W, x, lib=None) -> np.ndarray:
    """Form (ii): plain matvec over an explicitly dequantized matrix."""
    lib = lib or load()
    W, x = _c(W, np.float64), _c(np.atleast_2d(x), np.float32)
    N, K, S = W.shape[0], W.shape[1], x.shape[0]
    y = np.empty((S, N), np.float64)
    lib.orc_matvec_f64(_p(W), N, K, _p(x), S, _p(y))
    return y


def qmv_int8_row(w, r, x, lib=None):
    """y[S][N] = r * (w @ x) and its |.| denominators, both float64."""
    lib = lib or load()
    w, r, x = _c(w, np.int8), _c(r, np.float32), _c(np.atleast_2d(x), np.float32)
    N, K, S = w.shape[0], w.shape[1], x.shape[0]
    y = np.empty((S, N), np.float64)
    den = np.empty((S, N), np.float64)
    lib.orc_qmv_int8_row(_p(w), _p(r), N, K, _p(x), S, _p(y), _p(den))
    return y, den


# ------------------------------------------------------------------ f2: int3-g64

def unpack_int3(packed_row, n_vals: int, lib=None) -> np.ndarray:
    """Values code - 4 of one two-plane row (reading R6 in qmv_oracle.c)."""
    lib = lib or load()
    packed_row = _c(packed_row, np.uint8)
    vals = np.empty(n_vals, np.int8)
    lib.orc_unpack_int3(_p(packed_row), n_vals, _p(vals))
    return vals


def pack_int3(values, lib=None) -> np.ndarray:
    """int8 values in [-4, 3], length a multiple of 64 -> two-plane bytes."""
    lib = lib or load()
    values = _c(values, np.int8)
    out = np.empty(values.size // 64 * 24, np.uint8)
    if lib.orc_pack_int3(_p(values), values.size, _p(out)) != 0:
        raise ValueError("int3 values must lie in [-4, 3], in whole 64-groups")
    return out


def qmv_int3_gs(wq, scales, x, lib=None):
    """(y [S][N], den [S][N]) float64 for two-plane int3-g64 rows wq [N][K/64*24]."""
    lib = lib or load()
    wq, scales, x = _c(wq, np.uint8), _c(scales, np.float32), _c(np.atleast_2d(x), np.float32)
    N, K, S = wq.shape[0], wq.shape[1] // 24 * 64, x.shape[0]
    y = np.empty((S, N), np.float64)
    den = np.empty((S, N), np.float64)
    lib.orc_qmv_int3_gs(_p(wq), _p(scales), N, K, _p(x), S, _p(y), _p(den))
    return y, den


# ------------------------------------------------------------------ a4 / a5

def route_topk(logits, k: int, lib=None):
    """(ids int32 [T][k], w float64 [T][k])."""
    lib = lib or load()
    logits = _c(np.atleast_2d(logits), np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if lib.orc_route_topk(_p(logits), T, E, k, _p(ids), _p(w)) != 0:
        raise ValueError("bad routing sizes")
    return ids, w


def group(ids, E: int, lib=None):
    """(offsets [E+1], list [T*k], used experts [n_used]) as int32 arrays."""
    lib = lib or load()
    ids = _c(np.atleast_2d(ids), np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    lst = np.empty(T * k, np.int32)
    uexp = np.empty(E, np.int32)
    nu = np.zeros(1, np.int32)
    if lib.orc_group(_p(ids), T, k, E, _p(offsets), _p(lst), _p(uexp), _p(nu)) != 0:
        raise ValueError("expert id out of range")
    return offsets, lst, uexp[: int(nu[0])].copy()


# ------------------------------------------------------------------ a6 / a7

def moe_ffn(weights: dict, x, ids, w, gs: int = 64, want_h: bool = False, lib=None):
    """Expert FFN over the tokens of ``x`` (float64-widened [T][H]).

    ``weights`` holds gu_q/gu_s/dn_q/dn_s for n experts; ``ids`` [T][k] index into
    those n (the caller maps global expert ids to positions); ``w`` [T][k] fp32.
    Returns dict(out [T][H], den [T][H]) plus h / hden [T*k][I] when ``want_h``.
    """
    lib = lib or load()
    gu_q, gu_s = _c(weights["gu_q"], np.uint8), _c(weights["gu_s"], np.float32)
    dn_q, dn_s = _c(weights["dn_q"], np.uint8), _c(weights["dn_s"], np.float32)
    I = gu_q.shape[1] // 2
    H = gu_q.shape[2] * 2
    x = _c(np.atleast_2d(x), np.float64)
    ids, w = _c(np.atleast_2d(ids), np.int32), _c(np.atleast_2d(w), np.float32)
    T, k = ids.shape
    if x.shape != (T, H) or w.shape != (T, k):
        raise ValueError("shape mismatch")
    if ids.size and (ids.min() < 0 or ids.max() >= gu_q.shape[0]):
        raise ValueError("ids must index the given weight arrays")
    out = np.empty((T, H), np.float64)
    den = np.empty((T, H), np.float64)
    h = np.empty((T * k, I), np.float64) if want_h else None
    hden = np.empty((T * k, I), np.float64) if want_h else None
    lib.orc_moe_ffn(_p(gu_q), _p(gu_s), _p(dn_q), _p(dn_s), H, I, gs, _p(x), T, _p(ids), _p(w),
                    k, _p(h), _p(hden), _p(out), _p(den))
    res = dict(out=out, den=den)
    if want_h:
        res.update(h=h, hden=hden)
    return res
