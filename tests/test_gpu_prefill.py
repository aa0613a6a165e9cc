"""Batched MoE prefill on the tcgen05 tensor cores against the fp64 oracle
(bf16 operands: normalised error <= 1e-2, expert selection bit-exact)."""
import numpy as np
import pytest

import datagen
import oracle
from tests.gpu_util import TOL_BF16, moe_oracle, norm_err

torch = pytest.importorskip("torch")
q = pytest.importorskip("int4_group_quantized_gs64_gb300")

pytestmark = pytest.mark.gpu

PASS_PAIRS = 64  # the prefill kernels run an expert's pairs in passes of up to 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    q.build()
    q.lib()


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run_prefill(m, xbits, ids, w):
    T, k = ids.shape
    ws = torch.empty(q.moe_prefill_workspace_bytes(m, T, k), dtype=torch.uint8, device="cuda")
    out = q.moe_expert_ffn_int4_prefill(m, bf16_dev(xbits), torch.from_numpy(ids).cuda(),
                                        torch.from_numpy(w).cuda(), ws=ws)
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).cpu()[0])
    return out.cpu().numpy(), status


def rand_experts(rng, E, H, I):
    return dict(
        gu_q=rng.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8),
        gu_s=(np.abs(rng.normal(0, 0.02, size=(E, 2 * I, H // 64))) + 1e-4).astype(np.float32),
        dn_q=rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8),
        dn_s=(np.abs(rng.normal(0, 0.02, size=(E, H, I // 64))) + 1e-4).astype(np.float32),
    )


@pytest.mark.parametrize("T,k,E,H,I", [(5, 2, 4, 256, 256), (40, 2, 4, 256, 256),
                                       (200, 2, 3, 128, 384), (70, 1, 1, 192, 128),
                                       (64, 8, 16, 512, 256), (300, 2, 4, 256, 512),
                                       (33, 4, 8, 1024, 256)])
def test_prefill_shapes(T, k, E, H, I):
    """Under 16 tokens per expert (padding), several passes of 64, one expert."""
    rng = np.random.default_rng(T * 7 + k * 3 + E)
    wts = rand_experts(rng, E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    xbits = datagen.normal_bf16_bits(99, (T, H), start=T)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    ids, w = oracle.route_topk(logits, k)
    w = w.astype(np.float32)
    out, status = run_prefill(m, xbits, ids, w)
    assert status == 0
    ref = oracle.moe_ffn(wts, datagen.bf16_bits_to_f32(xbits).astype(np.float64), ids, w)
    assert norm_err(out, ref["out"], ref["den"]) <= TOL_BF16


@pytest.mark.parametrize("lo,hi", [(-4.0, -0.55), (-3.0, -0.7), (-1.0, 0.5), (-0.58, -0.5)])
def test_prefill_scale_ranges(lo, hi):
    """Group scales 10^U(lo, hi): the tensor-map kernel's dequant takes its
    one-multiply-add form for a warp only while all 32 rows' scales lie in
    [2^-120, 1/4), else the two-step form; both must give the oracle's result:
    mixed warps, all warps in the first form, all in the second (large
    scales, scales just above 1/4)."""
    rng = np.random.default_rng(int(100 * (hi - lo)))
    E, H, I, T, k = 4, 256, 256, 48, 2
    wts = rand_experts(rng, E, H, I)
    for key in ("gu_s", "dn_s"):
        wts[key] = (10.0 ** rng.uniform(lo, hi, size=wts[key].shape)).astype(np.float32)
    m = q.MoeInt4Weights.from_numpy(wts)
    assert q.moe_weight_path(m) == 1
    xbits = datagen.normal_bf16_bits(7, (T, H), start=3)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    ids, w = oracle.route_topk(logits, k)
    w = w.astype(np.float32)
    out, status = run_prefill(m, xbits, ids, w)
    assert status == 0
    ref = oracle.moe_ffn(wts, datagen.bf16_bits_to_f32(xbits).astype(np.float64), ids, w)
    assert norm_err(out, ref["out"], ref["den"]) <= TOL_BF16


def pass_cells(ids, E, pass_tok):
    """Per token, the cells its pairs fall in: (expert, pass) for every pair,
    plus (expert, pass, "last") for the pair in a pass's last column. An
    expert's pairs run in ascending pair id, as the grouping lists them, in
    passes of pass_tok."""
    T, k = ids.shape
    flat = ids.reshape(-1)
    cells = [set() for _ in range(T)]
    for e in range(E):
        pairs = np.nonzero(flat == e)[0]
        for j, p in enumerate(pairs):
            ps = j // pass_tok
            cells[p // k].add((e, ps))
            if j == min(len(pairs), (ps + 1) * pass_tok) - 1:
                cells[p // k].add((e, ps, "last"))
    return cells


def covering_sample(ids, E, pass_tok):
    """Greedy token sample whose pairs touch every used expert, every pass of
    each expert and the last column of every pass, so that every weight tile
    the kernel streams, every pass it runs and the widest MMA column of each
    pass meet a checked output. Returns the sorted tokens and all cells."""
    cells = pass_cells(ids, E, pass_tok)
    todo = set().union(*cells)
    every = set(todo)
    chosen = []
    while todo:
        t = max(range(len(cells)), key=lambda t: (len(cells[t] & todo), -t))
        chosen.append(t)
        todo -= cells[t]
    return np.array(sorted(chosen)), every


def test_prefill_workload_512_tokens_sampled():
    """512 tokens, H 6144, E 160, I 2048, top-8: every output computed on the
    GPU; a greedy sample of tokens that touches every expert and every pass
    of 64 pairs and the last column of every pass (hence every weight row
    tile of both projections) is checked against the oracle, element by
    element."""
    wl = datagen.WORKLOADS[4]
    E, H, I, k, T = wl["E"], wl["H"], wl["I"], wl["k"], wl["T"]
    wts = datagen.moe_weights(E, H, I)
    m = q.MoeInt4Weights.from_numpy(wts)
    xbits, logits = datagen.moe_inputs(T, E, H, xdtype="bf16")
    ids_d, w_d = q.moe_route_topk(torch.from_numpy(logits).cuda(), k)
    ids, w = oracle.route_topk(logits, k)
    assert np.array_equal(ids_d.cpu().numpy(), ids)
    w = w.astype(np.float32)
    out, status = run_prefill(m, xbits, ids, w)
    assert status == 0
    assert np.all(np.isfinite(out))
    sample, cells = covering_sample(ids, E, PASS_PAIRS)
    per_tok = pass_cells(ids, E, PASS_PAIRS)
    assert set().union(*(per_tok[t] for t in sample)) == cells, "sample misses a cell"
    assert set(np.unique(ids[sample]).tolist()) == set(np.unique(ids).tolist())
    x64 = datagen.bf16_bits_to_f32(xbits[sample]).astype(np.float64)
    ref = moe_oracle(E, H, I, x64, ids[sample], w[sample], weights=wts)
    err = norm_err(out[sample], ref["out"], ref["den"])
    print(f"prefill 512 tokens: {len(sample)} tokens checked, {len(cells)} cells, "
          f"normalised error {err:.3e} (bound {TOL_BF16:.0e})")
    assert err <= TOL_BF16, err
