"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments on the host (no GPU needed: validation runs before any
CUDA call)."""
import ctypes
import os
import re

import pytest

import int4_group_quantized_gs64_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmv.h")

EINVAL, ESHAPE, EWORKSPACE, EALIGN = -1, -2, -3, -6


@pytest.fixture(scope="module")
def L():
    q.build()
    return q.lib()


def declared_functions():
    """Names of the functions declared in qmv.h (comments and typedefs stripped)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"^\s*#.*$", "", text, flags=re.M)
    text = re.sub(r"typedef[^;]*;", "", text, flags=re.S)
    names = []
    for stmt in text.split(";"):
        m = re.search(r"([A-Za-z_][A-Za-z0-9_]*)\s*\(", stmt)
        if m and not stmt.strip().startswith(("}", "extern")):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("qmv_gemv_workspace_bytes", "qmv_int4_gs", "qmv_int4_gs_pair", "qmv_int3_gs",
              "qmv_int8_row", "qmv_int4_gs_bf16", "qmv_int8_row_bf16",
              "moe_route_topk", "moe_group", "moe_gate_up_silu",
              "moe_down", "moe_combine", "moe_workspace_bytes", "moe_expert_ffn_int4"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in qmv.h but not exported"


def test_status_strings(L):
    assert L.qmv_version() >= 100
    for s in (0, -1, -2, -3, -4, -5, -6, 99):
        assert isinstance(L.qmv_status_str(s), bytes)


FAKE = 0x10000  # a 64 KiB-aligned non-null address: never dereferenced, validation fails first


def test_dense_validation(L):
    p = ctypes.c_void_p(FAKE)
    need = L.qmv_gemv_workspace_bytes(64, 1)
    assert need >= 64 * 4 and need % 256 == 0
    assert L.qmv_gemv_workspace_bytes(96, 1) == 0 and L.qmv_gemv_workspace_bytes(64, 0) == 0
    ok = (p, need, None)
    assert L.qmv_int4_gs(None, p, 8, 64, 64, p, p, 1, *ok) == EINVAL
    assert L.qmv_int4_gs(p, p, 8, 64, 32, p, p, 1, *ok) == EINVAL      # gs != 64
    assert L.qmv_int4_gs(p, p, 0, 64, 64, p, p, 1, *ok) == EINVAL      # N < 1
    assert L.qmv_int4_gs(p, p, 8, 64, 64, p, p, 0, *ok) == EINVAL      # S < 1
    assert L.qmv_int4_gs(p, p, 8, 96, 64, p, p, 1, *ok) == ESHAPE      # ragged K
    assert L.qmv_int4_gs(p, p, 8, 0, 64, p, p, 1, *ok) == ESHAPE
    assert L.qmv_int4_gs(ctypes.c_void_p(FAKE + 8), p, 8, 64, 64, p, p, 1, *ok) == EALIGN
    assert L.qmv_int4_gs(p, ctypes.c_void_p(FAKE + 2), 8, 64, 64, p, p, 1, *ok) == EALIGN
    assert L.qmv_int4_gs(p, p, 8, 64, 64, p, p, 1, None, need, None) == EWORKSPACE
    assert L.qmv_int4_gs(p, p, 8, 64, 64, p, p, 1, p, need - 1, None) == EWORKSPACE
    assert L.qmv_int4_gs(p, p, 8, 64, 64, p, p, 1, ctypes.c_void_p(FAKE + 128), need, None) == EWORKSPACE
    # pair: (wq0, s0, N0, wq1, s1, N1, K, gs, x, y0, y1, S, ws, bytes, stream)
    assert L.qmv_int4_gs_pair(p, p, 8, None, p, 8, 64, 64, p, p, p, 1, *ok) == EINVAL
    assert L.qmv_int4_gs_pair(p, p, 8, p, p, 0, 64, 64, p, p, p, 1, *ok) == EINVAL   # N1 < 1
    assert L.qmv_int4_gs_pair(p, p, 8, p, p, 8, 64, 64, p, p, None, 1, *ok) == EINVAL
    assert L.qmv_int4_gs_pair(p, p, 8, p, p, 8, 96, 64, p, p, p, 1, *ok) == ESHAPE
    assert L.qmv_int4_gs_pair(p, p, 8, ctypes.c_void_p(FAKE + 8), p, 8, 64, 64, p, p, p, 1,
                              *ok) == EALIGN
    assert L.qmv_int4_gs_pair(p, p, 8, p, p, 8, 64, 64, p, p, p, 1, p, need - 1, None) == EWORKSPACE
    # int3: (wq3, scales, N, K, gs, x, y, S, stream), no workspace
    assert L.qmv_int3_gs(None, p, 8, 64, 64, p, p, 1, None) == EINVAL
    assert L.qmv_int3_gs(p, p, 8, 64, 32, p, p, 1, None) == EINVAL
    assert L.qmv_int3_gs(p, p, 8, 96, 64, p, p, 1, None) == ESHAPE
    assert L.qmv_int3_gs(ctypes.c_void_p(FAKE + 2), p, 8, 64, 64, p, p, 1, None) == EALIGN
    assert L.qmv_int3_gs(p, p, 8, 64, 64, ctypes.c_void_p(FAKE + 8), p, 1, None) == EALIGN
    assert L.qmv_int8_row(p, None, 8, 64, p, p, 1, *ok) == EINVAL
    assert L.qmv_int8_row(p, p, 8, 100, p, p, 1, *ok) == ESHAPE
    assert L.qmv_int8_row(ctypes.c_void_p(FAKE + 4), p, 8, 64, p, p, 1, *ok) == EALIGN
    assert L.qmv_int8_row(p, p, 8, 64, p, p, 1, p, 0, None) == EWORKSPACE
    # bf16 outputs: same arguments, y is bf16 (2-byte aligned)
    odd = ctypes.c_void_p(FAKE + 1)
    assert L.qmv_int4_gs_bf16(p, p, 8, 64, 64, p, None, 1, *ok) == EINVAL
    assert L.qmv_int4_gs_bf16(p, p, 8, 64, 32, p, p, 1, *ok) == EINVAL
    assert L.qmv_int4_gs_bf16(p, p, 8, 96, 64, p, p, 1, *ok) == ESHAPE
    assert L.qmv_int4_gs_bf16(p, p, 8, 64, 64, p, odd, 1, *ok) == EALIGN
    assert L.qmv_int4_gs_bf16(p, p, 8, 64, 64, p, ctypes.c_void_p(FAKE + 2), 1, p, 0, None) == EWORKSPACE
    assert L.qmv_int8_row_bf16(p, None, 8, 64, p, p, 1, *ok) == EINVAL
    assert L.qmv_int8_row_bf16(p, p, 8, 100, p, p, 1, *ok) == ESHAPE
    assert L.qmv_int8_row_bf16(p, p, 8, 64, p, odd, 1, *ok) == EALIGN
    assert L.qmv_int8_row_bf16(p, p, 8, 64, p, p, 1, p, 0, None) == EWORKSPACE


def test_route_and_group_validation(L):
    p = ctypes.c_void_p(FAKE)
    assert L.moe_route_topk(p, 1, 8, 0, p, p, None) == EINVAL       # k < 1
    assert L.moe_route_topk(p, 1, 8, 9, p, p, None) == EINVAL       # k > E
    assert L.moe_route_topk(p, 1, 2048, 8, p, p, None) == EINVAL    # E > 1024
    assert L.moe_route_topk(p, 1, 64, 33, p, p, None) == EINVAL     # k > 32
    assert L.moe_route_topk(None, 0, 8, 2, None, None, None) == 0   # T == 0: nothing to do
    assert L.moe_group(p, 1, 2, 8, None, p, p, p, p, None) == EINVAL
    assert L.moe_group(p, 1 << 20, 2, 8, p, p, p, p, p, None) == EINVAL  # too many pairs


def _desc(E=8, H=128, I=64, gs=64, base=FAKE):
    return q.MoeDesc(base, base, base, base, E, H, I, gs)


def test_moe_validation(L):
    p = ctypes.c_void_p(FAKE)
    d = _desc()
    need = L.moe_workspace_bytes(ctypes.byref(d), 3, 2)
    assert need > 0 and need % 256 == 0
    assert L.moe_workspace_bytes(ctypes.byref(_desc(H=100)), 3, 2) == 0
    ws = ctypes.c_void_p(FAKE)
    args = (p, 3, p, p, 2, p)
    assert L.moe_expert_ffn_int4(ctypes.byref(d), *args, ws, need - 1, None) == EWORKSPACE
    assert L.moe_expert_ffn_int4(ctypes.byref(d), *args, ctypes.c_void_p(FAKE + 16), need, None) == EWORKSPACE
    assert L.moe_expert_ffn_int4(ctypes.byref(d), *args, None, need, None) == EWORKSPACE
    assert L.moe_expert_ffn_int4(ctypes.byref(_desc(gs=32)), *args, ws, need, None) == EINVAL
    assert L.moe_expert_ffn_int4(ctypes.byref(_desc(I=96)), *args, ws, need, None) == ESHAPE
    assert L.moe_expert_ffn_int4(ctypes.byref(_desc(E=2048)), *args, ws, need, None) == EINVAL
    assert L.moe_expert_ffn_int4(None, *args, ws, need, None) == EINVAL
    bad = q.MoeDesc(FAKE + 8, FAKE, FAKE, FAKE, 8, 128, 64, 64)
    assert L.moe_expert_ffn_int4(ctypes.byref(bad), *args, ws, need, None) == EALIGN
    # k larger than E
    assert L.moe_expert_ffn_int4(ctypes.byref(d), p, 3, p, p, 9, p, ws, need, None) == EINVAL
    # staged entry points share the workspace rule
    assert L.moe_gate_up_silu(ctypes.byref(d), p, 3, 2, p, p, p, p, p, ws, need - 1, None) == EWORKSPACE
    assert L.moe_down(ctypes.byref(d), p, 3, 2, p, p, p, p, p, ws, need - 1, None) == EWORKSPACE
    assert L.moe_combine(p, p, None, 3, 2, 8, 128, p, None) == EINVAL
    # weight-path query: same descriptor rule; a valid descriptor answers 0 or 1
    assert L.moe_weight_path(None) == EINVAL
    assert L.moe_weight_path(ctypes.byref(_desc(gs=32))) == EINVAL
    assert L.moe_weight_path(ctypes.byref(_desc(I=96))) == ESHAPE
    assert L.moe_weight_path(ctypes.byref(bad)) == EALIGN
    assert L.moe_weight_path(ctypes.byref(d)) in (0, 1)
    # fused routing + FFN: (m, logits, x, T, k, ids, w, out, ws, bytes, stream)
    assert L.moe_route_expert_ffn_int4(ctypes.byref(d), None, p, 3, 2, p, p, p, ws, need,
                                       None) == EINVAL
    assert L.moe_route_expert_ffn_int4(ctypes.byref(d), p, p, 3, 33, p, p, p, ws, need,
                                       None) == EINVAL                     # k > 32
    assert L.moe_route_expert_ffn_int4(ctypes.byref(d), p, p, 3, 2, ctypes.c_void_p(FAKE + 2), p,
                                       p, ws, need, None) == EALIGN
    assert L.moe_route_expert_ffn_int4(ctypes.byref(d), p, p, 0, 2, p, p, p, ws, need,
                                       None) == 0
    # resident variant: bitmap and served mask required, bitmap 4-byte aligned
    # (m, resident, x, T, ids, w, k, out, served, ws, bytes, stream)
    assert L.moe_expert_ffn_int4_resident(ctypes.byref(d), None, p, 3, p, p, 2, p, p, ws,
                                          need, None) == EINVAL
    assert L.moe_expert_ffn_int4_resident(ctypes.byref(d), p, p, 3, p, p, 2, p, None, ws,
                                          need, None) == EINVAL
    assert L.moe_expert_ffn_int4_resident(ctypes.byref(d), ctypes.c_void_p(FAKE + 2), p, 3, p, p,
                                          2, p, p, ws, need, None) == EALIGN
    assert L.moe_expert_ffn_int4_resident(ctypes.byref(d), p, p, 3, p, p, 2, p, p, ws,
                                          need - 1, None) == EWORKSPACE
    # one-token path query: same descriptor rule
    assert L.moe_one_token_path(None, 8) == EINVAL
    assert L.moe_one_token_path(ctypes.byref(_desc(gs=32)), 8) == EINVAL
    assert L.moe_one_token_path(ctypes.byref(_desc(I=96)), 8) == ESHAPE
    assert L.moe_one_token_path(ctypes.byref(bad), 8) == EALIGN
    assert L.moe_one_token_path(ctypes.byref(d), 8) in (0, 1)
    assert L.moe_one_token_path(ctypes.byref(d), 0) == 0


def test_workspace_grows_with_tokens(L):
    d = _desc(E=160, H=6144, I=2048)
    a = L.moe_workspace_bytes(ctypes.byref(d), 8, 8)
    b = L.moe_workspace_bytes(ctypes.byref(d), 16, 8)
    assert b > a > 8 * 8 * (2048 + 6144) * 4
