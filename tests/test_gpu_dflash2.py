"""DFlash 2 modules on the GPU against the oracle: the two-tap dynamic convolutions in every
layer (whole draft + verify steps, tensor-core and FFMA paths, eager and graph-replayed) and
the path selector (the walk kernel on identical inputs, and inside the draft step).

Selector decisions are float decisions: the GPU scores in fp32 (and, inside the draft step,
from its own fp32 hidden rows), the oracle in fp64. So each position of the GPU's walk is
checked given the GPU's own predecessor: its pick must be the oracle's best candidate, or
within a margin of it when the oracle's best two lie closer than the margin (then both
picks are correct)."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import get_config
from synth import inputs as S

from harness import Pair, to_np
from test_gpu_parity import _limits, _run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_inject_gb300 import build
    build.build()


# ----------------------------------------------------------------------------- convolution
@pytest.mark.parametrize("lens", [[120, 37], [50, 173, 300]])
@pytest.mark.parametrize("hidden", [512, 1024])
def test_dyn_conv_steps_bf16(lens, hidden):
    """Two widths: 32 and 64 channel groups per correction row."""
    cfg = get_config("mini_bf16", dyn_conv=1, hidden=hidden)
    _run_steps(cfg, _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100), lens, steps=2)


def test_dyn_conv_steps_f32():
    cfg = get_config("tiny_f32", dyn_conv=1)
    _run_steps(cfg, _limits(max_batch=1, max_pages=8, max_positions=256, max_inject_rows=64), [64], steps=2)


def test_dyn_conv_with_variants():
    cfg = get_config("mini_bf16", n_layers=1, dyn_conv=1, block_causal=1, mask_embedding=1)
    _run_steps(cfg, _limits(max_batch=4, max_pages=16, max_positions=512, max_inject_rows=64), [90, 64], steps=1)


@pytest.mark.parametrize("hidden", [512, 1024])
def test_dyn_conv_graph_replay_matches_eager(hidden):
    """Without full logits the layer stack is captured into a CUDA graph on the second call
    and replayed after; every call must give the eager result."""
    cfg = get_config("mini_bf16", dyn_conv=1, hidden=hidden)
    pair = Pair(cfg, _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100))
    reqs = [3, 4]
    pair.inject(reqs, [77, 140], "prefill", reset=True)
    anchors = S.make_anchors(cfg, 2, 0, 0).cuda()
    ref = pair.ctx.draft(reqs, anchors, want_logits=True)
    for _ in range(3):
        out = pair.ctx.draft(reqs, anchors)
        assert torch.equal(out["argmax"], ref["argmax"])
        assert torch.equal(out["topk_idx"], ref["topk_idx"])
        assert torch.equal(out["topk_val"], ref["topk_val"])


# ----------------------------------------------------------------------------- selector
def _check_walk(got, anchor, cand, unary, gate, A, B, margin):
    """Every step of the GPU's walk against the oracle's scores given the GPU's predecessor;
    returns the number of steps whose oracle decision was clear (exact match required)."""
    prev, clear = int(anchor), 0
    for t in range(len(got)):
        _, sc = O.select_path(prev, cand[t:t + 1], unary[t:t + 1], gate[t:t + 1], A, B)
        sc = sc[0]
        j = list(cand[t]).index(int(got[t]))
        assert sc[j] >= sc.max() - margin, (t, sc[j], sc.max())
        srt = np.sort(sc)[::-1]
        if len(srt) == 1 or srt[0] - srt[1] > margin:
            assert j == int(np.argmax(sc))
            clear += 1
        prev = int(got[t])
    return clear


@pytest.mark.parametrize("dtype,r,kc", [("bf16", 256, 16), ("bf16", 64, 32), ("f32", 32, 5), ("bf16", 512, 1)])
def test_select_path_kernel_matches_oracle(dtype, r, kc):
    from block_diffusion_speculative_inject_gb300 import select_path
    rng = np.random.default_rng(r + kc)
    n, K, V = 6, 9, 3000
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    A = torch.from_numpy(rng.normal(0, 0.25, (V, r)).astype(np.float32)).to(tdt)
    B = torch.from_numpy(rng.normal(0, 0.25, (V, r)).astype(np.float32)).to(tdt)
    cand = np.stack([np.stack([rng.permutation(V)[:kc] for _ in range(K)]) for _ in range(n)]).astype(np.int32)
    unary = -np.sort(-rng.normal(0, 1, (n, K, kc)), axis=2).astype(np.float32)
    gate = rng.normal(0, 0.5, (n, K, r)).astype(np.float32)
    anchors = rng.integers(0, V, n).astype(np.int32)
    anchors[-1] = -1                     # out of range: a zero predecessor row
    sel, sc = select_path(torch.from_numpy(anchors).cuda(), torch.from_numpy(cand).cuda(),
                          torch.from_numpy(unary).cuda(), torch.from_numpy(gate).cuda(), A.cuda(), B.cuda(),
                          want_scores=True)
    torch.cuda.synchronize()
    sel, sc = sel.cpu().numpy(), sc.cpu().numpy()
    A64, B64 = A.double().numpy(), B.double().numpy()
    clear = 0
    for b in range(n):
        if anchors[b] < 0:
            # the first position's scores are the unary scores alone
            np.testing.assert_array_equal(sc[b, 0], unary[b, 0])
            continue
        clear += _check_walk(sel[b], anchors[b], cand[b], unary[b], gate[b], A64, B64, 1e-4)
        # the scores along the GPU's own walk
        prev = int(anchors[b])
        for t in range(K):
            _, want = O.select_path(prev, cand[b, t:t + 1], unary[b, t:t + 1], gate[b, t:t + 1], A64, B64)
            np.testing.assert_allclose(sc[b, t], want[0], rtol=0, atol=2e-5)
            prev = int(sel[b, t])
    assert clear >= 0.95 * (n - 1) * K


def test_select_path_argument_errors():
    from block_diffusion_speculative_inject_gb300 import DFlashError, select_path
    z = torch.zeros((2, 3, 4), dtype=torch.int32, device="cuda")
    u = torch.zeros((2, 3, 4), device="cuda")
    a = torch.zeros((2,), dtype=torch.int32, device="cuda")
    for r in (16, 48, 544):
        cb = torch.zeros((10, r), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(DFlashError):
            select_path(a, z, u, torch.zeros((2, 3, r), device="cuda"), cb, cb)


@pytest.mark.parametrize("name,lens,r", [("mini_bf16", [120, 37], 64), ("mini_bf16", [50, 173, 300], 256),
                                         ("tiny_f32", [64], 32)])
def test_draft_step_selector_matches_oracle(name, lens, r):
    """The selected path of the draft step against the oracle's walk over the same
    candidates and unary scores (the GPU's top-k), with the oracle's own gate rows."""
    cfg = get_config(name, selector_rank=r)
    pair = Pair(cfg, _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100))
    reqs = list(range(len(lens)))
    pair.inject(reqs, lens, "prefill", reset=True)
    anchors = S.make_anchors(cfg, len(lens), 0, 0)
    out = pair.ctx.draft(reqs, anchors.cuda(), want_selected=True)
    sel = out["selected"].cpu().numpy()
    ti, tv = out["topk_idx"].cpu().numpy(), to_np(out["topk_val"])
    clear = 0
    for i, q in enumerate(reqs):
        gate = pair.orc.hidden(q, int(anchors[i])) @ pair.orc.w["sel_hidden_proj"].astype(np.float64).T
        clear += _check_walk(sel[i], anchors[i], ti[i], tv[i].astype(np.float64), gate,
                             pair.orc.w["sel_pred_codebook"], pair.orc.w["sel_succ_codebook"], 2e-2)
    assert clear >= 0.6 * len(lens) * cfg.block_k
    # the argmax path is left alone and the selector really chooses
    assert np.all(out["argmax"].cpu().numpy() == ti[:, :, 0])
    assert np.any(sel != ti[:, :, 0])


def test_draft_step_selector_with_convolutions():
    cfg = get_config("mini_bf16", n_layers=1, dyn_conv=1, selector_rank=128)
    pair = Pair(cfg, _limits(max_batch=4, max_pages=16, max_positions=512, max_inject_rows=64))
    reqs = [0, 1]
    pair.inject(reqs, [90, 64], "prefill", reset=True)
    anchors = S.make_anchors(cfg, 2, 0, 0)
    out = pair.ctx.draft(reqs, anchors.cuda(), want_selected=True)
    sel, ti, tv = out["selected"].cpu().numpy(), out["topk_idx"].cpu().numpy(), to_np(out["topk_val"])
    for i, q in enumerate(reqs):
        gate = pair.orc.hidden(q, int(anchors[i])) @ pair.orc.w["sel_hidden_proj"].astype(np.float64).T
        _check_walk(sel[i], anchors[i], ti[i], tv[i].astype(np.float64), gate,
                    pair.orc.w["sel_pred_codebook"], pair.orc.w["sel_succ_codebook"], 2e-2)


def test_selected_needs_the_selector_and_topk():
    from block_diffusion_speculative_inject_gb300 import DFlashError
    cfg = get_config("mini_bf16", n_layers=1)
    pair = Pair(cfg, _limits(max_batch=2, max_pages=8, max_positions=256, max_inject_rows=64))
    pair.inject([0], [40], "prefill", reset=True)
    with pytest.raises(DFlashError, match="INVALID_ARG"):
        pair.ctx.draft([0], torch.zeros(1, dtype=torch.int32, device="cuda"), want_selected=True)


# ----------------------------------------------------------------------------- selector, sampling mode
def _check_sample_walk(sel, q_tok, q_p, anchor, cand, unary, gate, A, B, T, u, q_atol, margin):
    """Each step of the GPU's sampling walk, given the GPU's own predecessor: its candidate
    distribution against the oracle's, and its draw against the oracle's inverse CDF (exact
    unless the uniform lies within `margin` of a step boundary). Returns the exact steps."""
    prev, exact = int(anchor), 0
    V = A.shape[0]
    for t in range(len(sel)):
        _, sc = O.select_path(prev, cand[t:t + 1], unary[t:t + 1], gate[t:t + 1], A, B)
        q = O.softmax(sc[0] / T)
        k = len(cand[t])
        np.testing.assert_array_equal(q_tok[t, :k], cand[t])
        np.testing.assert_allclose(q_p[t, :k], q, rtol=0, atol=q_atol)
        full = O.subset_to_vocab(cand[t], q, V)
        cum = np.cumsum(full[np.sort(cand[t])])
        # the pick's step of the oracle's CDF (vocabulary order) holds u, up to the margin
        assert int(sel[t]) in cand[t]
        lo = full[:int(sel[t])].sum()
        assert lo - margin <= u[t] <= lo + full[int(sel[t])] + margin, (t, lo, full[int(sel[t])], u[t])
        if np.min(np.abs(cum - u[t])) > margin:
            assert int(sel[t]) == O.sample_index(full, float(u[t])), t
            exact += 1
        prev = int(sel[t])
    return exact


@pytest.mark.parametrize("dtype,r,kc,T", [("bf16", 64, 16, 0.8), ("f32", 32, 5, 1.3), ("bf16", 256, 32, 0.5)])
def test_select_sample_kernel_matches_oracle(dtype, r, kc, T):
    from block_diffusion_speculative_inject_gb300 import select_sample
    rng = np.random.default_rng(r * 3 + kc)
    n, K, V = 6, 9, 3000
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    A = torch.from_numpy(rng.normal(0, 0.25, (V, r)).astype(np.float32)).to(tdt)
    B = torch.from_numpy(rng.normal(0, 0.25, (V, r)).astype(np.float32)).to(tdt)
    cand = np.stack([np.stack([rng.permutation(V)[:kc] for _ in range(K)]) for _ in range(n)]).astype(np.int32)
    unary = -np.sort(-rng.normal(0, 1, (n, K, kc)), axis=2).astype(np.float32)
    gate = rng.normal(0, 0.5, (n, K, r)).astype(np.float32)
    anchors = rng.integers(0, V, n).astype(np.int32)
    u = rng.uniform(0, 1, (n, K)).astype(np.float32)
    sel, q_tok, q_p, q_n = select_sample(torch.from_numpy(anchors).cuda(), torch.from_numpy(cand).cuda(),
                                         torch.from_numpy(unary).cuda(), torch.from_numpy(gate).cuda(), A.cuda(),
                                         B.cuda(), T, torch.from_numpy(u).cuda())
    torch.cuda.synchronize()
    sel, q_tok, q_p, q_n = (x.cpu().numpy() for x in (sel, q_tok, q_p, q_n))
    assert np.all(q_n == kc)
    A64, B64 = A.double().numpy(), B.double().numpy()
    exact = sum(_check_sample_walk(sel[b], q_tok[b], q_p[b], anchors[b], cand[b], unary[b], gate[b], A64, B64, T,
                                   u[b].astype(np.float64), 1e-5, 5e-5) for b in range(n))
    assert exact >= 0.95 * n * K


def test_verify_sample_q_matches_oracle():
    """Rejection sampling against candidate-list draft distributions: accept lengths and
    tokens exact, with every float decision kept away from its threshold."""
    from test_gpu_sampling import _ctx, _mid_step, _safe_top_p
    B = 5
    cfg, ctx = _ctx(4999, B)
    K, V = cfg.block_k, cfg.vocab
    rng = np.random.default_rng(123)
    T, k, top_p = 0.9, 20, 0.95
    tl = rng.normal(0, 1.0, (B, K + 1, V)).astype(np.float32)
    tl64 = tl.astype(np.float64)
    tp = _safe_top_p(list(tl64.reshape(-1, V)), T, k, top_p)
    kc = 16
    q_tok = np.full((B, K, 32), -1, dtype=np.int32)
    q_p = np.zeros((B, K, 32), dtype=np.float32)
    drafts, u_acc, u_res, want = [], [], [], []
    plans = [0, 2, K, K - 1, 1]           # the position each request rejects at (K: none)
    for b in range(B):
        p_rows = [O.sampling_probs(r, T, k, tp) for r in tl64[b]]
        d, ua, q_rows = [], [], []
        for j in range(K):
            # candidates: the target's kept tokens mixed with others, so p/q varies
            kept = np.flatnonzero(p_rows[j] > 0)
            others = rng.choice(np.setdiff1d(np.arange(V), kept), kc, replace=False)
            cands = rng.permutation(np.concatenate([kept[:kc // 2], others]))[:kc]
            w = rng.uniform(0.2, 1.0, kc).astype(np.float32)
            qv = (w / w.sum()).astype(np.float32)
            q_tok[b, j, :kc] = cands
            q_p[b, j, :kc] = qv
            full = O.subset_to_vocab(cands, qv.astype(np.float64), V)
            q_rows.append(full)
            if j < plans[b]:
                # a draft the target also keeps, accepted (uniform at half the ratio)
                both = np.where(p_rows[j] > 0, full, 0.0)
                _, tok = _mid_step(both, rng)
                ratio = min(1.0, p_rows[j][tok] / full[tok])
                ua.append(ratio / 2)
            else:
                _, tok = _mid_step(full, rng)
                ratio = min(1.0, p_rows[j][tok] / full[tok])
                ua.append((ratio + 1.0) / 2 if ratio <= 0.96 else ratio / 2)
            d.append(tok)
        a = 0
        while a < K and ua[a] < O.accept_prob(p_rows[a], q_rows[a], d[a]):
            a += 1
        dist = O.residual_dist(p_rows[a], q_rows[a]) if a < K else p_rows[K]
        ur, _ = _mid_step(dist, rng)
        wa, toks = O.verify_sample(p_rows, q_rows, d, ua, ur)
        assert wa == a
        drafts.append(d)
        u_acc.append(ua)
        u_res.append(ur)
        want.append((wa, toks))
    q_n = np.full((B, K), kc, dtype=np.int32)
    acc, out, nxt = ctx.verify_sample_q(torch.from_numpy(tl).cuda(), torch.from_numpy(q_tok).cuda(),
                                        torch.from_numpy(q_p).cuda(), torch.from_numpy(q_n).cuda(),
                                        torch.tensor(drafts, dtype=torch.int32).cuda(),
                                        torch.tensor(u_acc, dtype=torch.float32).cuda(),
                                        torch.tensor(u_res, dtype=torch.float32).cuda(), T, k, tp)
    torch.cuda.synchronize()
    acc, out, nxt = acc.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy()
    for b, (wa, toks) in enumerate(want):
        assert acc[b] == wa, (b, acc[b], wa)
        np.testing.assert_array_equal(out[b, :wa + 1], toks)
        assert nxt[b] == toks[-1]
    assert len(set(acc.tolist())) > 1
    ctx.close()


def test_draft_step_sampling_selector():
    """The draft step's sampling walk against the oracle's, over the GPU's candidates with the
    oracle's own gate rows (q within the bf16 logit tolerance, draws exact away from steps)."""
    cfg = get_config("mini_bf16", selector_rank=64)
    pair = Pair(cfg, _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100))
    reqs = [0, 1, 2]
    pair.inject(reqs, [120, 37, 200], "prefill", reset=True)
    anchors = S.make_anchors(cfg, 3, 0, 0)
    T = 0.8
    u = np.random.default_rng(5).uniform(0, 1, (3, cfg.block_k)).astype(np.float32)
    out = pair.ctx.draft(reqs, anchors.cuda(), sel_uniform=torch.from_numpy(u).cuda(), sel_temperature=T)
    sel, ti, tv = out["selected"].cpu().numpy(), out["topk_idx"].cpu().numpy(), to_np(out["topk_val"])
    qt, qp = out["sel_q_tok"].cpu().numpy(), out["sel_q_p"].cpu().numpy()
    assert np.all(out["sel_q_n"].cpu().numpy() == cfg.topk)
    exact = 0
    for i, q in enumerate(reqs):
        gate = pair.orc.hidden(q, int(anchors[i])) @ pair.orc.w["sel_hidden_proj"].astype(np.float64).T
        exact += _check_sample_walk(sel[i], qt[i], qp[i], anchors[i], ti[i], tv[i].astype(np.float64), gate,
                                    pair.orc.w["sel_pred_codebook"], pair.orc.w["sel_succ_codebook"], T,
                                    u[i].astype(np.float64), 2e-2, 1e-2)
    assert exact >= 0.3 * len(reqs) * cfg.block_k
