"""Python binding of libqmv.so, the GB300 (sm_103a) int4-gs64 / int8 quantized GEMV library.

Argument marshalling only: every computation runs in the CUDA kernels behind
the C ABI declared in ``include/qmv.h``. Tensors are torch CUDA tensors (torch
provides device memory and streams); outputs are allocated with torch when the
caller passes none. There is no CPU fallback: if the library cannot be loaded,
every call raises.

Functions carry the C names: ``qmv_int4_gs``, ``qmv_int8_row``, their bf16-output
forms ``qmv_int4_gs_bf16`` and ``qmv_int8_row_bf16``,
``moe_route_topk``, ``moe_group``, ``moe_gate_up_silu``, ``moe_down``,
``moe_combine``, ``moe_workspace_bytes``, ``moe_expert_ffn_int4`` and
``moe_expert_ffn_int4_prefill``.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

_lib = None

QMV_STATUS = {0: "QMV_OK", -1: "QMV_EINVAL", -2: "QMV_ESHAPE", -3: "QMV_EWORKSPACE",
              -4: "QMV_ECUDA", -5: "QMV_ETIMEOUT", -6: "QMV_EALIGN"}


class QmvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = lib().qmv_status_str(status).decode() if _lib is not None else "?"
        super().__init__(f"{fn} failed: {QMV_STATUS.get(status, status)} ({msg})")
        self.status = status


class MoeDesc(ctypes.Structure):
    """Mirror of ``qmv_moe_int4``."""
    _fields_ = [("gu_q", ctypes.c_void_p), ("gu_s", ctypes.c_void_p), ("dn_q", ctypes.c_void_p),
                ("dn_s", ctypes.c_void_p), ("E", ctypes.c_int32), ("H", ctypes.c_int32),
                ("I", ctypes.c_int32), ("gs", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libqmv.so for sm_103a (in-tree)."""
    return _build.build(force=force, verbose=verbose)


def lib():
    """Load libqmv.so (it must have been built; raises otherwise)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libqmv.so is not built: call int4_group_quantized_gs64_gb300.build()")
        L = ctypes.CDLL(_build.LIB)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        P = ctypes.POINTER(MoeDesc)
        sig = {
            "qmv_version": ([], i32),
            "qmv_test_split_skew": ([i32], i32),
            "qmv_status_str": ([i32], ctypes.c_char_p),
            "qmv_gemv_workspace_bytes": ([i32, i32], sz),
            "qmv_int4_gs": ([vp, vp, i32, i32, i32, vp, vp, i32, vp, sz, vp], i32),
            "qmv_int4_gs_pair": ([vp, vp, i32, vp, vp, i32, i32, i32, vp, vp, vp, i32, vp, sz, vp],
                                 i32),
            "qmv_int3_gs": ([vp, vp, i32, i32, i32, vp, vp, i32, vp], i32),
            "qmv_int8_row": ([vp, vp, i32, i32, vp, vp, i32, vp, sz, vp], i32),
            "qmv_int4_gs_bf16": ([vp, vp, i32, i32, i32, vp, vp, i32, vp, sz, vp], i32),
            "qmv_int8_row_bf16": ([vp, vp, i32, i32, vp, vp, i32, vp, sz, vp], i32),
            "moe_route_topk": ([vp, i32, i32, i32, vp, vp, vp], i32),
            "moe_group": ([vp, i32, i32, i32, vp, vp, vp, vp, vp, vp], i32),
            "moe_gate_up_silu": ([P, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_down": ([P, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_combine": ([vp, vp, vp, i32, i32, i32, i32, vp, vp], i32),
            "moe_workspace_bytes": ([P, i32, i32], sz),
            "moe_expert_ffn_int4": ([P, vp, i32, vp, vp, i32, vp, vp, sz, vp], i32),
            "moe_ffn_prepare": ([P, vp, i32, vp, i32, vp, sz, vp], i32),
            "moe_ffn_gate_up": ([P, i32, i32, vp, sz, vp], i32),
            "moe_ffn_down": ([P, i32, i32, vp, sz, vp], i32),
            "moe_ffn_combine": ([P, vp, vp, i32, i32, vp, vp, sz, vp], i32),
            "moe_weight_path": ([P], i32),
            "moe_one_token_path": ([P, i32], i32),
            "moe_route_expert_ffn_int4": ([P, vp, vp, i32, i32, vp, vp, vp, vp, sz, vp], i32),
            "moe_expert_ffn_int4_resident": ([P, vp, vp, i32, vp, vp, i32, vp, vp, vp, sz, vp], i32),
            "moe_prefill_workspace_bytes": ([P, i32, i32], sz),
            "moe_expert_ffn_int4_prefill": ([P, vp, i32, vp, vp, i32, vp, vp, sz, vp], i32),
        }
        for name, (args, res) in sig.items():
            if hasattr(L, name):
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
        _lib = L
    return _lib


# ------------------------------------------------------------------ helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise QmvError(fn, status)


def _need(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def qmv_test_split_skew(ns: int) -> int:
    """Test hook (qmv.h): the compute warps of odd CTAs of the tensor-map kernels
    start `ns` nanoseconds late from the next launch on (0: off). Returns the
    previous value."""
    return int(lib().qmv_test_split_skew(int(ns)))


# ------------------------------------------------------------------ GEMV

def qmv_gemv_workspace_bytes(K: int, S: int) -> int:
    return int(lib().qmv_gemv_workspace_bytes(K, S))


def qmv_int4_gs(wq, scales, x, y=None, gs: int = 64, ws=None, stream=None):
    """y[S][N] = int4-gs64 W[N][K] . x[S][K]  (wq uint8 [N][K/2], scales fp32 [N][K/64])."""
    import torch
    _need(wq, torch.uint8, "wq"); _need(scales, torch.float32, "scales"); _need(x, torch.float32, "x")
    N, K = wq.shape[0], wq.shape[1] * 2
    x2 = x.view(-1, K)
    S = x2.shape[0]
    if y is None:
        y = torch.empty((S, N), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, "y")
    if ws is None:
        ws = _workspace(qmv_gemv_workspace_bytes(K, S), x.device)
    _check("qmv_int4_gs", lib().qmv_int4_gs(_ptr(wq), _ptr(scales), N, K, gs, _ptr(x2), _ptr(y), S,
                                            _ptr(ws), ws.numel(), _stream(stream)))
    return y


def qmv_int4_gs_bf16(wq, scales, x, y=None, gs: int = 64, ws=None, stream=None):
    """qmv_int4_gs with the fp32 result rounded to bf16 (ties to even): y bf16 [S][N]."""
    import torch
    _need(wq, torch.uint8, "wq"); _need(scales, torch.float32, "scales"); _need(x, torch.float32, "x")
    N, K = wq.shape[0], wq.shape[1] * 2
    x2 = x.view(-1, K)
    S = x2.shape[0]
    if y is None:
        y = torch.empty((S, N), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, "y")
    if ws is None:
        ws = _workspace(qmv_gemv_workspace_bytes(K, S), x.device)
    _check("qmv_int4_gs_bf16", lib().qmv_int4_gs_bf16(_ptr(wq), _ptr(scales), N, K, gs, _ptr(x2),
                                                      _ptr(y), S, _ptr(ws), ws.numel(),
                                                      _stream(stream)))
    return y


def qmv_int4_gs_pair(wq0, s0, wq1, s1, x, y0=None, y1=None, gs: int = 64, ws=None, stream=None):
    """(y0, y1) = (W0 . x, W1 . x) for two int4-gs64 matrices sharing x [S][K]."""
    import torch
    for t, n in ((wq0, "wq0"), (wq1, "wq1")):
        _need(t, torch.uint8, n)
    for t, n in ((s0, "s0"), (s1, "s1"), (x, "x")):
        _need(t, torch.float32, n)
    N0, K = wq0.shape[0], wq0.shape[1] * 2
    N1 = wq1.shape[0]
    if wq1.shape[1] * 2 != K:
        raise QmvError("qmv_int4_gs_pair: the two matrices need the same K")
    x2 = x.view(-1, K)
    S = x2.shape[0]
    if y0 is None:
        y0 = torch.empty((S, N0), dtype=torch.float32, device=x.device)
    if y1 is None:
        y1 = torch.empty((S, N1), dtype=torch.float32, device=x.device)
    _need(y0, torch.float32, "y0"); _need(y1, torch.float32, "y1")
    if ws is None:
        ws = _workspace(qmv_gemv_workspace_bytes(K, S), x.device)
    _check("qmv_int4_gs_pair",
           lib().qmv_int4_gs_pair(_ptr(wq0), _ptr(s0), N0, _ptr(wq1), _ptr(s1), N1, K, gs, _ptr(x2),
                                  _ptr(y0), _ptr(y1), S, _ptr(ws), ws.numel(), _stream(stream)))
    return y0, y1


def qmv_int3_gs(wq3, scales, x, y=None, gs: int = 64, stream=None):
    """y[S][N] = int3-g64 two-plane W . x  (wq3 uint8 [N][K/64*24], scales fp32 [N][K/64])."""
    import torch
    _need(wq3, torch.uint8, "wq3"); _need(scales, torch.float32, "scales")
    _need(x, torch.float32, "x")
    N, K = wq3.shape[0], wq3.shape[1] // 24 * 64
    if wq3.shape[1] % 24:
        raise QmvError("qmv_int3_gs: rows must be whole 24-byte groups")
    x2 = x.view(-1, K)
    S = x2.shape[0]
    if y is None:
        y = torch.empty((S, N), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, "y")
    _check("qmv_int3_gs", lib().qmv_int3_gs(_ptr(wq3), _ptr(scales), N, K, gs, _ptr(x2), _ptr(y),
                                            S, _stream(stream)))
    return y


def qmv_int8_row(w, row_scale, x, y=None, ws=None, stream=None):
    """y[S][N] = row_scale[N] * (w[N][K] . x[S][K])  (w int8)."""
    import torch
    _need(w, torch.int8, "w"); _need(row_scale, torch.float32, "row_scale"); _need(x, torch.float32, "x")
    N, K = w.shape
    x2 = x.view(-1, K)
    S = x2.shape[0]
    if y is None:
        y = torch.empty((S, N), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, "y")
    if ws is None:
        ws = _workspace(qmv_gemv_workspace_bytes(K, S), x.device)
    _check("qmv_int8_row", lib().qmv_int8_row(_ptr(w), _ptr(row_scale), N, K, _ptr(x2), _ptr(y), S,
                                              _ptr(ws), ws.numel(), _stream(stream)))
    return y


def qmv_int8_row_bf16(w, row_scale, x, y=None, ws=None, stream=None):
    """qmv_int8_row with the fp32 result rounded to bf16 (ties to even): y bf16 [S][N]."""
    import torch
    _need(w, torch.int8, "w"); _need(row_scale, torch.float32, "row_scale"); _need(x, torch.float32, "x")
    N, K = w.shape
    x2 = x.view(-1, K)
    S = x2.shape[0]
    if y is None:
        y = torch.empty((S, N), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, "y")
    if ws is None:
        ws = _workspace(qmv_gemv_workspace_bytes(K, S), x.device)
    _check("qmv_int8_row_bf16", lib().qmv_int8_row_bf16(_ptr(w), _ptr(row_scale), N, K, _ptr(x2),
                                                        _ptr(y), S, _ptr(ws), ws.numel(),
                                                        _stream(stream)))
    return y


# ------------------------------------------------------------------ MoE

class MoeInt4Weights:
    """Device-resident int4-gs64 expert pools (gate rows then up rows in gu_q)."""

    def __init__(self, gu_q, gu_s, dn_q, dn_s, gs: int = 64):
        import torch
        _need(gu_q, torch.uint8, "gu_q"); _need(gu_s, torch.float32, "gu_s")
        _need(dn_q, torch.uint8, "dn_q"); _need(dn_s, torch.float32, "dn_s")
        self.gu_q, self.gu_s, self.dn_q, self.dn_s = gu_q, gu_s, dn_q, dn_s
        self.E = gu_q.shape[0]
        self.I = gu_q.shape[1] // 2
        self.H = gu_q.shape[2] * 2
        self.gs = gs
        self._desc = MoeDesc(gu_q.data_ptr(), gu_s.data_ptr(), dn_q.data_ptr(), dn_s.data_ptr(),
                             self.E, self.H, self.I, gs)

    @property
    def desc(self):
        return ctypes.byref(self._desc)

    @classmethod
    def from_numpy(cls, d: dict, device="cuda"):
        import torch
        t = {k: torch.from_numpy(v).to(device) for k, v in d.items()}
        return cls(t["gu_q"], t["gu_s"], t["dn_q"], t["dn_s"])


def moe_workspace_bytes(m: MoeInt4Weights, T: int, k: int) -> int:
    return int(lib().moe_workspace_bytes(m.desc, T, k))


def _workspace(nbytes, device):
    import torch
    # 256-byte alignment: torch's caching allocator returns 512-byte aligned blocks.
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def moe_route_topk(logits, k: int, ids=None, w=None, stream=None):
    import torch
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check("moe_route_topk", lib().moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w),
                                                  _stream(stream)))
    return ids, w


def moe_group(ids, E: int, status=None, stream=None):
    """Returns (offsets [E+1], list [T*k], uexp [E], n_used [1], status [1]) int32 tensors."""
    import torch
    _need(ids, torch.int32, "ids")
    T, k = ids.shape
    dev = ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    lst = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    uexp = torch.empty(E, dtype=torch.int32, device=dev)
    n_used = torch.empty(1, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("moe_group", lib().moe_group(_ptr(ids), T, k, E, _ptr(offsets), _ptr(lst), _ptr(uexp),
                                        _ptr(n_used), _ptr(status), _stream(stream)))
    return offsets, lst[: T * k], uexp, n_used, status


def moe_gate_up_silu(m: MoeInt4Weights, x, k: int, offsets, lst, uexp, n_used, h=None, ws=None,
                     stream=None):
    import torch
    _need(x, torch.float32, "x")
    T = x.shape[0]
    if h is None:
        h = torch.zeros((T * k, m.I), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _workspace(moe_workspace_bytes(m, T, k), x.device)
    _check("moe_gate_up_silu", lib().moe_gate_up_silu(
        m.desc, _ptr(x), T, k, _ptr(offsets), _ptr(lst), _ptr(uexp), _ptr(n_used), _ptr(h),
        _ptr(ws), ws.numel(), _stream(stream)))
    return h


def moe_down(m: MoeInt4Weights, h, T: int, k: int, offsets, lst, uexp, n_used, y=None, ws=None,
             stream=None):
    import torch
    _need(h, torch.float32, "h")
    if y is None:
        y = torch.zeros((T * k, m.H), dtype=torch.float32, device=h.device)
    if ws is None:
        ws = _workspace(moe_workspace_bytes(m, T, k), h.device)
    _check("moe_down", lib().moe_down(m.desc, _ptr(h), T, k, _ptr(offsets), _ptr(lst), _ptr(uexp),
                                      _ptr(n_used), _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))
    return y


def moe_combine(y, ids, w, E: int, out=None, stream=None):
    import torch
    T, k = ids.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=y.device)
    _check("moe_combine", lib().moe_combine(_ptr(y), _ptr(ids), _ptr(w), T, k, E, H, _ptr(out),
                                            _stream(stream)))
    return out


def moe_expert_ffn_int4(m: MoeInt4Weights, x, ids, w, out=None, ws=None, stream=None):
    """out[T][H] = sum_j w[t][j] * FFN_{ids[t][j]}(x[t]) for a decode micro-batch."""
    import torch
    _need(x, torch.float32, "x"); _need(ids, torch.int32, "ids"); _need(w, torch.float32, "w")
    T, k = ids.shape
    if out is None:
        out = torch.empty((T, m.H), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _workspace(moe_workspace_bytes(m, T, k), x.device)
    _check("moe_expert_ffn_int4", lib().moe_expert_ffn_int4(
        m.desc, _ptr(x), T, _ptr(ids), _ptr(w), k, _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def moe_route_expert_ffn_int4(m: MoeInt4Weights, logits, x, k: int, ids=None, w=None, out=None,
                              ws=None, stream=None):
    """Routing plus expert FFN in one call; returns (out [T][H], ids [T][k], w [T][k])."""
    import torch
    _need(logits, torch.float32, "logits"); _need(x, torch.float32, "x")
    T = logits.shape[0]
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    if out is None:
        out = torch.empty((T, m.H), dtype=torch.float32, device=x.device)
    _need(ids, torch.int32, "ids"); _need(w, torch.float32, "w")
    if ws is None:
        ws = _workspace(moe_workspace_bytes(m, T, k), x.device)
    _check("moe_route_expert_ffn_int4", lib().moe_route_expert_ffn_int4(
        m.desc, _ptr(logits), _ptr(x), T, k, _ptr(ids), _ptr(w), _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out, ids, w


def moe_expert_ffn_int4_resident(m: MoeInt4Weights, resident, x, ids, w, out=None, served=None,
                                 ws=None, stream=None):
    """As moe_expert_ffn_int4 over the experts set in the bitmap ``resident``
    (int32 [ceil(E/32)], bit e%32 of word e/32); returns (out, served uint8 [T][k])."""
    import torch
    _need(x, torch.float32, "x"); _need(ids, torch.int32, "ids"); _need(w, torch.float32, "w")
    _need(resident, torch.int32, "resident")
    if resident.numel() * 32 < m.E:
        raise QmvError("moe_expert_ffn_int4_resident: the bitmap needs ceil(E/32) words")
    T, k = ids.shape
    if out is None:
        out = torch.empty((T, m.H), dtype=torch.float32, device=x.device)
    if served is None:
        served = torch.empty((T, k), dtype=torch.uint8, device=x.device)
    _need(served, torch.uint8, "served")
    if ws is None:
        ws = _workspace(moe_workspace_bytes(m, T, k), x.device)
    _check("moe_expert_ffn_int4_resident", lib().moe_expert_ffn_int4_resident(
        m.desc, _ptr(resident), _ptr(x), T, _ptr(ids), _ptr(w), k, _ptr(out), _ptr(served),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out, served


def moe_ffn_prepare(m: MoeInt4Weights, x, ids, ws, stream=None):
    T, k = ids.shape
    _check("moe_ffn_prepare", lib().moe_ffn_prepare(m.desc, _ptr(x), T, _ptr(ids), k, _ptr(ws),
                                                    ws.numel(), _stream(stream)))


def moe_ffn_gate_up(m: MoeInt4Weights, T: int, k: int, ws, stream=None):
    _check("moe_ffn_gate_up", lib().moe_ffn_gate_up(m.desc, T, k, _ptr(ws), ws.numel(),
                                                    _stream(stream)))


def moe_ffn_down(m: MoeInt4Weights, T: int, k: int, ws, stream=None):
    _check("moe_ffn_down", lib().moe_ffn_down(m.desc, T, k, _ptr(ws), ws.numel(), _stream(stream)))


def moe_ffn_combine(m: MoeInt4Weights, ids, w, out, ws, stream=None):
    T, k = ids.shape
    _check("moe_ffn_combine", lib().moe_ffn_combine(m.desc, _ptr(ids), _ptr(w), T, k, _ptr(out),
                                                    _ptr(ws), ws.numel(), _stream(stream)))
    return out


def moe_weight_path(m: MoeInt4Weights) -> int:
    """1: decode kernels stream weights by tensor-map (TMA) copies; 0: cp.async rings."""
    r = int(lib().moe_weight_path(m.desc))
    if r < 0:
        _check("moe_weight_path", r)
    return r


def moe_one_token_path(m: MoeInt4Weights, k: int) -> int:
    """1: moe_expert_ffn_int4 with one token runs as a single cooperative kernel."""
    r = int(lib().moe_one_token_path(m.desc, k))
    if r < 0:
        _check("moe_one_token_path", r)
    return r


def moe_prefill_workspace_bytes(m: MoeInt4Weights, T: int, k: int) -> int:
    return int(lib().moe_prefill_workspace_bytes(m.desc, T, k))


def moe_expert_ffn_int4_prefill(m: MoeInt4Weights, x_bf16, ids, w, out=None, ws=None, stream=None):
    """Batched prefill: x bf16 [T][H] -> out fp32 [T][H] on the tcgen05 tensor-core path."""
    import torch
    _need(x_bf16, torch.bfloat16, "x"); _need(ids, torch.int32, "ids"); _need(w, torch.float32, "w")
    T, k = ids.shape
    if out is None:
        out = torch.empty((T, m.H), dtype=torch.float32, device=x_bf16.device)
    if ws is None:
        ws = _workspace(moe_prefill_workspace_bytes(m, T, k), x_bf16.device)
    _check("moe_expert_ffn_int4_prefill", lib().moe_expert_ffn_int4_prefill(
        m.desc, _ptr(x_bf16), T, _ptr(ids), _ptr(w), k, _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out
