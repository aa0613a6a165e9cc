"""MoE decode on the GPU against the fp64 oracle: routing and grouping
bit-exact, gate+up+SiLU, down and the weighted combine within 2e-5."""
import numpy as np
import pytest

import datagen
import oracle
from tests.gpu_util import TOL_FP32, TOL_W, moe_oracle, norm_err

torch = pytest.importorskip("torch")
q = pytest.importorskip("int4_group_quantized_gs64_gb300")

pytestmark = pytest.mark.gpu

W2 = datagen.WORKLOADS[2]
W3 = datagen.WORKLOADS[3]
W4 = datagen.WORKLOADS[4]


@pytest.fixture(scope="module", autouse=True)
def _built():
    q.build()
    q.lib()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture(scope="module")
def pool_160():
    """All 160 experts of the H 6144 / I 2048 workloads on the device (3.4 GB)."""
    wts = datagen.moe_weights(160, 6144, 2048)
    m = q.MoeInt4Weights.from_numpy(wts)
    del wts
    return m


# ------------------------------------------------------------------ routing / grouping

@pytest.mark.parametrize("wl", [W2, W3, W4], ids=["w2", "w3", "w4"])
def test_route_matches_oracle(wl):
    _, logits = datagen.moe_inputs(wl["T"], wl["E"], 64, hot=wl["hot"])
    ids, w = q.moe_route_topk(dev(logits), wl["k"])
    torch.cuda.synchronize()
    rid, rw = oracle.route_topk(logits, wl["k"])
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=TOL_W, atol=0)


def test_route_ties_and_nan():
    logits = np.array([[1.0, 3.0, 3.0, 0.5, 2.0, 3.0, -np.inf, 0.0],
                       [np.nan, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0]], np.float32)
    ids, w = q.moe_route_topk(dev(logits), 4)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    assert ids[0].tolist() == [1, 2, 5, 4]
    assert ids[1].tolist() == [1, 2, 3, 4]
    rid, rw = oracle.route_topk(logits, 4)  # the oracle reads NaN as -inf
    assert np.array_equal(ids, rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=TOL_W, atol=0)


def test_route_nan_golden():
    """The hand-derived NaN / all -inf / signed-zero fixture, on the GPU."""
    import json
    import os
    d = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "route_nan_as_minus_inf.json")))
    logits = np.array([[float(v) for v in row] for row in d["logits"]], np.float32)
    ids, w = q.moe_route_topk(dev(logits), d["k"])
    torch.cuda.synchronize()
    assert ids.cpu().numpy().tolist() == d["expected_ids"]
    assert np.allclose(w.cpu().numpy(), d["expected_w"], rtol=TOL_W, atol=0)


def test_route_many_experts_and_k32():
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(37, 1024)).astype(np.float32)
    ids, w = q.moe_route_topk(dev(logits), 32)
    torch.cuda.synchronize()
    rid, rw = oracle.route_topk(logits, 32)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=TOL_W, atol=0)


def _lane_heavy(rng, T, E):
    """Logits whose largest values all sit on experts 3, 35, 67, ...: one lane
    of the routing warp holds the top, so it wins round after round (and has
    to rescan its experts every other round)."""
    logits = rng.normal(size=(T, E)).astype(np.float32)
    logits[:, 3::32] += 10.0
    return logits


@pytest.mark.parametrize("T,k,E", [(2, 32, 1024), (5, 8, 256), (3, 16, 40), (4, 8, 160)])
def test_route_one_lane_holds_the_top(T, k, E):
    rng = np.random.default_rng(7 * T + k + E)
    logits = _lane_heavy(rng, T, E)
    ids, w = q.moe_route_topk(dev(logits), k)
    torch.cuda.synchronize()
    rid, rw = oracle.route_topk(logits, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=TOL_W, atol=0)


def test_route_signed_zero_inf_and_nan_ties():
    """+0 and -0 tie (the lower index first), -inf ties with -inf and NaN
    counts as -inf: ids bit-exact against the oracle, which reads NaN the
    same way."""
    rng = np.random.default_rng(29)
    vals = np.array([0.0, -0.0, -np.inf, np.nan, 1.0, -1.0], np.float32)
    for E, k in ((64, 16), (200, 32), (33, 32)):
        logits = rng.choice(vals, size=(6, E)).astype(np.float32)
        ids, _ = q.moe_route_topk(dev(logits), k)
        torch.cuda.synchronize()
        rid, _ = oracle.route_topk(logits, k)
        assert np.array_equal(ids.cpu().numpy(), rid), (E, k)


@pytest.mark.parametrize("T", [1, 3])
def test_route_ffn_fused_lane_heavy_logits(T):
    """The in-kernel routing of the one-token kernel (T = 1) and of the
    grouping kernel (T = 3) on logits that make one lane win repeatedly."""
    E, H, I, k = 256, 256, 256, 8
    rng = np.random.default_rng(40 + T)
    wts = _rand_pool(rng, E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    x = rng.normal(size=(T, H)).astype(np.float32)
    logits = _lane_heavy(rng, T, E)
    out, ids, w = q.moe_route_expert_ffn_int4(m, dev(logits), dev(x), k)
    torch.cuda.synchronize()
    rid, rw = oracle.route_topk(logits, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    ref = oracle.moe_ffn(wts, x.astype(np.float64), rid, rw.astype(np.float32))
    assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32


@pytest.mark.parametrize("T,k,E", [(1, 8, 256), (8, 8, 160), (512, 8, 160), (33, 2, 7),
                                   (3000, 4, 1024), (5, 3, 6)])
def test_group_matches_oracle(T, k, E):
    rng = np.random.default_rng(T + k + E)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    off, lst, uexp, nu, st = q.moe_group(dev(ids), E)
    torch.cuda.synchronize()
    roff, rlst, ruexp = oracle.group(ids, E)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(lst.cpu().numpy(), rlst)
    n = int(nu.cpu()[0])
    assert n == len(ruexp) and np.array_equal(uexp.cpu().numpy()[:n], ruexp)
    assert int(st.cpu()[0]) == 0


def test_group_flags_bad_ids():
    ids = np.array([[0, 5], [9, 1], [-1, 2]], np.int32)  # 9 and -1 are outside [0, 6)
    off, lst, uexp, nu, st = q.moe_group(dev(ids), 6)
    torch.cuda.synchronize()
    assert int(st.cpu()[0]) == 1
    good = ids.copy()
    assert off.cpu().numpy()[-1] == 4
    assert lst.cpu().numpy()[:4].tolist() == [0, 3, 5, 1]


# ------------------------------------------------------------------ FFN stages

def _route_oracle(wl, T=None):
    T = wl["T"] if T is None else T
    x, logits = datagen.moe_inputs(T, wl["E"], wl["H"], hot=wl["hot"])
    ids, w = oracle.route_topk(logits, wl["k"])
    return x, ids, w.astype(np.float32)


def test_w2_full_layer():
    wl = W2
    wts = datagen.moe_weights(wl["E"], wl["H"], wl["I"])
    m = q.MoeInt4Weights.from_numpy(wts)
    x, ids, w = _route_oracle(wl)
    assert q.moe_one_token_path(m, wl["k"]) == 1  # one token: the single-launch kernel
    out = q.moe_expert_ffn_int4(m, dev(x), dev(ids), dev(w))
    torch.cuda.synchronize()
    ref = moe_oracle(wl["E"], wl["H"], wl["I"], x.astype(np.float64), ids, w, weights=wts)
    assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32


def _rand_pool(rng, E, H, I):
    return dict(
        gu_q=rng.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8),
        gu_s=(np.abs(rng.normal(0, 0.02, size=(E, 2 * I, H // 64))) + 1e-4).astype(np.float32),
        dn_q=rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8),
        dn_s=(np.abs(rng.normal(0, 0.02, size=(E, H, I // 64))) + 1e-4).astype(np.float32),
    )


@pytest.mark.parametrize("E,H,I,k", [(8, 256, 256, 1), (8, 256, 256, 8), (40, 512, 768, 4),
                                     (64, 1024, 256, 32), (300, 2048, 512, 8)])
def test_one_token_shapes(E, H, I, k):
    """One token on the single-launch kernel: one and many experts, k = E,
    k = 32 (every warp takes several down tiles), several gate+up tiles per CTA."""
    rng = np.random.default_rng(E * 7 + H + I + k)
    wts = _rand_pool(rng, E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    assert q.moe_one_token_path(m, k) == 1
    x = rng.normal(size=(1, H)).astype(np.float32)
    ids, w = oracle.route_topk(rng.normal(size=(1, E)).astype(np.float32), k)
    w = w.astype(np.float32)
    ws = torch.full((q.moe_workspace_bytes(m, 1, k),), 0xFF, dtype=torch.uint8, device="cuda")
    ref = oracle.moe_ffn(wts, x.astype(np.float64), ids, w)
    first = None
    for _ in range(3):  # the grid barrier's counter is cleared by every call
        out = q.moe_expert_ffn_int4(m, dev(x), dev(ids), dev(w), ws=ws)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).cpu()[0]) == 0
        o = out.cpu().numpy()
        assert norm_err(o, ref["out"], ref["den"]) <= TOL_FP32
        if first is None:
            first = o
        assert np.array_equal(o, first)


def test_one_token_bad_ids_and_fallback():
    rng = np.random.default_rng(78)
    E, H, I, k = 4, 256, 256, 3
    wts = _rand_pool(rng, E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    assert q.moe_one_token_path(m, k) == 1
    x = rng.normal(size=(1, H)).astype(np.float32)
    ids = np.array([[2, 9, 0]], np.int32)
    w = np.array([[0.5, 0.25, 0.25]], np.float32)
    ws = torch.empty(q.moe_workspace_bytes(m, 1, k), dtype=torch.uint8, device="cuda")
    out = q.moe_expert_ffn_int4(m, dev(x), dev(ids), dev(w), ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).cpu()[0]) == 1  # the bad id is flagged and skipped
    ref = moe_oracle(E, H, I, x.astype(np.float64), ids, w, weights=wts)
    assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32
    # too large for one CTA's shared memory: the grouped phases instead
    big = q.MoeInt4Weights.from_numpy(_rand_pool(rng, 2, 6144, 2048))
    assert q.moe_one_token_path(big, 2) == 0


@pytest.mark.parametrize("T,k,E,H,I", [(1, 8, 256, 2048, 512), (1, 3, 40, 256, 256),
                                       (8, 8, 160, 512, 256), (2, 32, 64, 256, 256)])
def test_route_ffn_fused(T, k, E, H, I):
    """Routing inside the one-token kernel, and routing then the phases for
    more tokens: ids bit-exact and w as moe_route_topk, out within 2e-5."""
    rng = np.random.default_rng(T + 10 * k + E)
    wts = _rand_pool(rng, E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    x = rng.normal(size=(T, H)).astype(np.float32)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    if T == 1:
        assert q.moe_one_token_path(m, k) == 1
    ws = torch.empty(q.moe_workspace_bytes(m, T, k), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        out, ids, w = q.moe_route_expert_ffn_int4(m, dev(logits), dev(x), k, ws=ws)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).cpu()[0]) == 0
        rid, rw = oracle.route_topk(logits, k)
        assert np.array_equal(ids.cpu().numpy(), rid)
        gi, gw = q.moe_route_topk(dev(logits), k)
        assert np.array_equal(w.cpu().numpy(), gw.cpu().numpy())  # the same routing code
        ref = oracle.moe_ffn(wts, x.astype(np.float64), rid, rw.astype(np.float32))
        assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32


def _bitmap(mask):
    """bool [E] -> int32 words [ceil(E/32)], bit e % 32 of word e / 32."""
    E = len(mask)
    words = np.zeros((E + 31) // 32, np.uint32)
    for e in np.flatnonzero(mask):
        words[e // 32] |= np.uint32(1) << np.uint32(e % 32)
    return words.view(np.int32)


@pytest.mark.parametrize("T,k,E,H,I,frac", [(1, 8, 64, 256, 256, 0.5), (8, 8, 40, 512, 256, 0.3),
                                            (5, 3, 6, 128, 192, 0.5), (8, 4, 16, 256, 256, 0.0),
                                            (3, 2, 7, 256, 256, 1.0), (1, 8, 300, 2048, 512, 0.7)])
def test_resident_subset(T, k, E, H, I, frac):
    """Only resident experts are computed: out is the oracle over the served
    slots (the others weighted zero), served marks exactly those slots, and a
    non-resident id is no error. Covers the single-launch one-token kernel,
    the tensor-map phases (packed), the cp.async phases and no resident expert."""
    rng = np.random.default_rng(T * 1000 + k * 10 + E)
    wts = _rand_pool(rng, E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    x = rng.normal(size=(T, H)).astype(np.float32)
    ids, w = oracle.route_topk(rng.normal(size=(T, E)).astype(np.float32), k)
    w = w.astype(np.float32)
    res = rng.random(E) < frac
    ws = torch.empty(q.moe_workspace_bytes(m, T, k), dtype=torch.uint8, device="cuda")
    out, served = q.moe_expert_ffn_int4_resident(m, dev(_bitmap(res)), dev(x), dev(ids), dev(w),
                                                 ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).cpu()[0]) == 0
    want = res[ids]
    assert np.array_equal(served.cpu().numpy(), want.astype(np.uint8))
    ref = oracle.moe_ffn(wts, x.astype(np.float64), ids, np.where(want, w, 0).astype(np.float32))
    o = out.cpu().numpy()
    assert np.all(o[~want.any(axis=1)] == 0)
    den = np.maximum(ref["den"], 1e-30)
    assert norm_err(o, ref["out"], den) <= TOL_FP32


def test_resident_all_matches_plain_call():
    """Every expert resident: the same result as moe_expert_ffn_int4, bit for bit."""
    rng = np.random.default_rng(91)
    E, H, I, T, k = 12, 256, 256, 8, 4
    wts = _rand_pool(rng, E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    x = rng.normal(size=(T, H)).astype(np.float32)
    ids, w = oracle.route_topk(rng.normal(size=(T, E)).astype(np.float32), k)
    w = w.astype(np.float32)
    a = q.moe_expert_ffn_int4(m, dev(x), dev(ids), dev(w)).cpu().numpy()
    b, served = q.moe_expert_ffn_int4_resident(m, dev(_bitmap(np.ones(E, bool))), dev(x),
                                               dev(ids), dev(w))
    assert np.array_equal(a, b.cpu().numpy())
    assert np.all(served.cpu().numpy() == 1)


def test_w2_stages_hidden():
    wl = W2
    wts = datagen.moe_weights(wl["E"], wl["H"], wl["I"])
    m = q.MoeInt4Weights.from_numpy(wts)
    x, ids, w = _route_oracle(wl)
    dids = dev(ids)
    off, lst, uexp, nu, _ = q.moe_group(dids, wl["E"])
    h = q.moe_gate_up_silu(m, dev(x), wl["k"], off, lst, uexp, nu)
    y = q.moe_down(m, h, wl["T"], wl["k"], off, lst, uexp, nu)
    out = q.moe_combine(y, dids, dev(w), wl["E"])
    torch.cuda.synchronize()
    ref = moe_oracle(wl["E"], wl["H"], wl["I"], x.astype(np.float64), ids, w, want_h=True,
                     weights=wts)
    assert norm_err(h.cpu().numpy(), ref["h"], ref["hden"]) <= TOL_FP32
    assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32


def test_w3_full_layer(pool_160):
    wl = W3
    x, ids, w = _route_oracle(wl)
    out = q.moe_expert_ffn_int4(pool_160, dev(x), dev(ids), dev(w))
    torch.cuda.synchronize()
    ref = moe_oracle(wl["E"], wl["H"], wl["I"], x.astype(np.float64), ids, w, want_h=False)
    assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32


def test_w3_hidden(pool_160):
    wl = W3
    x, ids, w = _route_oracle(wl)
    dids = dev(ids)
    off, lst, uexp, nu, _ = q.moe_group(dids, wl["E"])
    h = q.moe_gate_up_silu(pool_160, dev(x), wl["k"], off, lst, uexp, nu)
    torch.cuda.synchronize()
    ref = moe_oracle(wl["E"], wl["H"], wl["I"], x.astype(np.float64), ids, w, want_h=True)
    assert norm_err(h.cpu().numpy(), ref["h"], ref["hden"]) <= TOL_FP32


@pytest.mark.parametrize("T,k,E,H,I", [(5, 3, 6, 128, 192), (33, 2, 7, 64, 64), (1, 1, 1, 256, 128),
                                       (40, 3, 3, 192, 320), (2, 8, 8, 1024, 512),
                                       (40, 3, 3, 256, 256), (17, 4, 5, 512, 768)])
def test_ffn_shapes(T, k, E, H, I):
    """Odd shapes: ragged token counts per expert, > 16 tokens on one expert
    (several passes), a single expert, k = E. Shapes with H/64 and I/64
    multiples of 4 run the tensor-map (TMA) kernels, the rest the cp.async ones."""
    rng = np.random.default_rng(T * 100 + k + E)
    wts = dict(
        gu_q=rng.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8),
        gu_s=(np.abs(rng.normal(0, 0.02, size=(E, 2 * I, H // 64))) + 1e-4).astype(np.float32),
        dn_q=rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8),
        dn_s=(np.abs(rng.normal(0, 0.02, size=(E, H, I // 64))) + 1e-4).astype(np.float32),
    )
    m = q.MoeInt4Weights.from_numpy(wts)
    assert q.moe_weight_path(m) == int((H // 64) % 4 == 0 and (I // 64) % 4 == 0)
    x = rng.normal(size=(T, H)).astype(np.float32)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    ids, w = oracle.route_topk(logits, k)
    w = w.astype(np.float32)
    out = q.moe_expert_ffn_int4(m, dev(x), dev(ids), dev(w))
    torch.cuda.synchronize()
    ref = oracle.moe_ffn(wts, x.astype(np.float64), ids, w)
    assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32


def test_ffn_bad_ids_flag_and_skip():
    rng = np.random.default_rng(77)
    E, H, I, T, k = 4, 128, 64, 3, 2
    wts = datagen.moe_weights(E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    x = rng.normal(size=(T, H)).astype(np.float32)
    ids = np.array([[0, 1], [7, 2], [3, -2]], np.int32)
    w = np.full((T, k), 0.5, np.float32)
    ws = torch.empty(q.moe_workspace_bytes(m, T, k), dtype=torch.uint8, device="cuda")
    out = q.moe_expert_ffn_int4(m, dev(x), dev(ids), dev(w), ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).cpu()[0]) == 1
    ref = moe_oracle(E, H, I, x.astype(np.float64), ids, w, weights=wts)
    assert norm_err(out.cpu().numpy(), ref["out"], ref["den"]) <= TOL_FP32


def test_ffn_deterministic(pool_160):
    x, ids, w = _route_oracle(W3)
    a = q.moe_expert_ffn_int4(pool_160, dev(x), dev(ids), dev(w)).cpu().numpy()
    b = q.moe_expert_ffn_int4(pool_160, dev(x), dev(ids), dev(w)).cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("skew_us", [30, 150])
def test_ffn_split_items_any_arrival_order(pool_160, skew_us):
    """An item whose stages two CTAs share comes out the same whatever order
    they reach it in. With the compute warps of odd CTAs started late (the
    qmv_test_split_skew hook; 150 us is longer than a CTA's whole range), an
    even CTA ends before its odd successor has published the rest of their
    shared item, so it publishes instead of adding the fetched partial sums,
    and the successor, publishing last, writes the item after its own range;
    an odd CTA ends after its even successor published, and adds the fetched
    partial sums. The outputs must equal the undelayed call's bit for bit,
    twice on one workspace (the counters return to zero) and once more after
    the hook is off."""
    x, ids, w = _route_oracle(W3)
    dx, dids, dw = dev(x), dev(ids), dev(w)
    ref = q.moe_expert_ffn_int4(pool_160, dx, dids, dw).cpu().numpy()
    T, k = ids.shape
    ws = torch.empty(q.moe_workspace_bytes(pool_160, T, k), dtype=torch.uint8, device="cuda")
    old = q.qmv_test_split_skew(skew_us * 1000)
    try:
        a = q.moe_expert_ffn_int4(pool_160, dx, dids, dw, ws=ws).cpu().numpy()
        b = q.moe_expert_ffn_int4(pool_160, dx, dids, dw, ws=ws).cpu().numpy()
    finally:
        q.qmv_test_split_skew(old)
    c = q.moe_expert_ffn_int4(pool_160, dx, dids, dw, ws=ws).cpu().numpy()
    assert int(ws[:4].view(torch.int32).cpu()[0]) == 0
    assert np.array_equal(a, ref)
    assert np.array_equal(b, ref)
    assert np.array_equal(c, ref)


def test_ffn_phases_repeat_match_fused():
    """The four phases reproduce the fused call bit for bit, also when gate+up
    and down run again on one prepared workspace (items split between CTAs
    leave their counters at zero for the next launch)."""
    wl = W2
    wts = datagen.moe_weights(wl["E"], wl["H"], wl["I"])
    m = q.MoeInt4Weights.from_numpy(wts)
    x, ids, w = _route_oracle(wl, T=2)  # two tokens: the call runs the same phases
    dx, dids, dw = dev(x), dev(ids), dev(w)
    fused = q.moe_expert_ffn_int4(m, dx, dids, dw).cpu().numpy()
    T, k = ids.shape
    ws = torch.empty(q.moe_workspace_bytes(m, T, k), dtype=torch.uint8, device="cuda")
    q.moe_ffn_prepare(m, dx, dids, ws)
    outs = []
    for _ in range(3):
        q.moe_ffn_gate_up(m, T, k, ws)
        q.moe_ffn_down(m, T, k, ws)
        out = torch.empty((T, wl["H"]), dtype=torch.float32, device="cuda")
        outs.append(q.moe_ffn_combine(m, dids, dw, out, ws).cpu().numpy())
    assert int(ws[:4].view(torch.int32).cpu()[0]) == 0
    for o in outs:
        assert np.array_equal(o, fused)
