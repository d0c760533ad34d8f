"""Draft trees on the GPU (dflash_ddtree_build / dflash_ddtree_walk) and the draft step's
softmax normaliser (dflash_draft_step_lse) against the oracle.

Tree parity uses log-probabilities on a 1/64 grid: every prefix sum is exact in fp32 and
fp64 alike, so the GPU must pop the same nodes in the same order, ties included."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import get_config
from synth import inputs as S

from harness import LOGIT_TOL, Pair, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_inject_gb300 import build
    build.build()


def _grid_candidates(rng, n, L, kc):
    lp = -np.sort(rng.integers(0, 6 * 64, (n, L, kc)), axis=2) / 64.0      # best first, ties likely
    tok = np.stack([np.stack([rng.permutation(5000)[:kc] for _ in range(L)]) for _ in range(n)])
    return lp.astype(np.float32), tok.astype(np.int32)


@pytest.mark.parametrize("L,kc,budget,with_lse", [(1, 4, 10, 0), (7, 1, 5, 0), (7, 4, 1, 1), (7, 16, 64, 0),
                                                  (15, 32, 300, 1), (15, 8, 1024, 0), (31, 3, 200, 1)])
def test_ddtree_build_matches_oracle(L, kc, budget, with_lse):
    """with_lse: the kernel gets logits (log-probabilities plus a per-row offset on the same
    grid) and the offsets as the rows' normalisers, so it must recover the same values."""
    from block_diffusion_speculative_inject_gb300 import ddtree_build
    rng = np.random.default_rng(L * 1000 + kc * 10 + budget)
    n = 5
    lp, tok = _grid_candidates(rng, n, L, kc)
    if with_lse:
        off = (rng.integers(-64 * 8, 64 * 8, (n, L)) / 64.0).astype(np.float32)
        out = ddtree_build(torch.from_numpy(tok).cuda(), torch.from_numpy(lp + off[..., None]).cuda(), budget,
                           lse=torch.from_numpy(off).cuda())
    else:
        out = ddtree_build(torch.from_numpy(tok).cuda(), torch.from_numpy(lp).cuda(), budget)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items()}
    words = (budget + 1 + 31) // 32
    for b in range(n):
        nodes = O.ddtree_build(lp[b].astype(np.float64), tok[b], budget)
        nn = len(nodes)
        assert g["n_nodes"][b] == nn
        np.testing.assert_array_equal(g["tok"][b, :nn], [x[0] for x in nodes])
        np.testing.assert_array_equal(g["parent"][b, :nn], [x[1] for x in nodes])
        np.testing.assert_array_equal(g["depth"][b, :nn], [x[2] for x in nodes])
        np.testing.assert_array_equal(g["logp"][b, :nn], np.array([x[3] for x in nodes], dtype=np.float32))
        assert np.all(g["tok"][b, nn:] == -1)
        m = O.ddtree_mask(nodes)
        bits = g["mask"][b].view(np.uint32)
        for i in range(nn + 1):
            row = np.array([(int(bits[i, j // 32]) >> (j % 32)) & 1 for j in range(words * 32)], dtype=bool)
            np.testing.assert_array_equal(row[:nn + 1], m[i])
            assert not row[nn + 1:].any()


def test_ddtree_walk_matches_oracle():
    from block_diffusion_speculative_inject_gb300 import ddtree_build, ddtree_walk
    rng = np.random.default_rng(81)
    n, L, kc, budget = 64, 7, 4, 40
    lp = -np.sort(-np.log(rng.dirichlet(np.ones(kc), size=(n, L))), axis=2).astype(np.float32)
    tok = np.tile(np.arange(kc, dtype=np.int32), (n, L, 1))          # tokens 0..3 at every position
    tree = ddtree_build(torch.from_numpy(tok).cuda(), torch.from_numpy(lp).cuda(), budget, with_mask=False)
    g_tok, g_par = tree["tok"].cpu().numpy(), tree["parent"].cpu().numpy()
    nn = tree["n_nodes"].cpu().numpy()
    tn = rng.integers(0, kc, (n, budget + 1)).astype(np.int32)
    tn[:, 0] = g_tok[:, 0]                 # the walk enters the tree in most rows
    acc, toks, nxt = ddtree_walk(tree, L, torch.from_numpy(tn).cuda())
    acc, toks, nxt = acc.cpu().numpy(), toks.cpu().numpy(), nxt.cpu().numpy()
    for b in range(n):
        nodes = [(int(g_tok[b, i]), int(g_par[b, i]), 0, 0.0) for i in range(nn[b])]
        a, out = O.ddtree_walk(nodes, tn[b])
        assert acc[b] == a
        np.testing.assert_array_equal(toks[b, :a + 1], out)
        assert np.all(toks[b, a + 1:] == -1) and nxt[b] == out[-1]
    assert acc.max() >= 2


@pytest.mark.parametrize("name,lens", [("mini_bf16", [120, 37]), ("mini_bf16", [50, 173, 300]),
                                       ("tiny_f32", [64])])
def test_draft_lse_and_tree_from_draft(name, lens):
    """lse of the fused (2 requests) and unfused (3 requests, fp32) LM heads against the
    oracle's normaliser; a tree built from topk_val - lse on the GPU against the oracle's tree
    over the same fp32 values (nodes may differ only across a near-tie at the budget edge)."""
    from block_diffusion_speculative_inject_gb300 import Limits, ddtree_build
    cfg = get_config(name)
    pair = Pair(cfg, Limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100))
    B = len(lens)
    reqs = list(range(B))
    pair.inject(reqs, lens, "prefill", reset=True)
    anchors = S.make_anchors(cfg, B, 0, 0)
    out = pair.ctx.draft(reqs, anchors.cuda(), want_lse=True)
    lse = to_np(out["lse"])
    for i, r in enumerate(reqs):
        _, _, _, w_lg = pair.orc.draft(r, int(anchors[i]))
        np.testing.assert_allclose(lse[i], O.log_softmax_norm(w_lg), atol=LOGIT_TOL[cfg.dtype], rtol=0)
    lp = (out["topk_val"] - out["lse"][..., None]).contiguous()
    budget = 48
    tree = ddtree_build(out["topk_idx"], lp, budget, with_mask=False)
    g_tok, g_lp = tree["tok"].cpu().numpy(), tree["logp"].cpu().numpy()
    # the normaliser subtracted in the kernel: the same fp32 subtraction, the same tree
    tree2 = ddtree_build(out["topk_idx"], out["topk_val"], budget, with_mask=False, lse=out["lse"])
    for key in ("tok", "parent", "depth", "logp", "n_nodes"):
        assert torch.equal(tree[key], tree2[key]), key
    lp_np = lp.cpu().numpy().astype(np.float64)
    ti = out["topk_idx"].cpu().numpy()
    for i in range(B):
        nodes = O.ddtree_build(lp_np[i], ti[i], budget)
        want = np.array([x[3] for x in nodes])
        # the same multiset of path probabilities up to fp32 summation order
        np.testing.assert_allclose(np.sort(g_lp[i]), np.sort(want), atol=1e-4, rtol=0)
