"""Sampling mode on the GPU (dflash_sample_tokens, dflash_verify_sample) against the oracle.

The GPU computes the truncated distributions in fp32 and the oracle in fp64, so every
decision that a float takes (a top-p cut, an accept test, a draw) is set up with a margin:
top_p is moved away from every prefix mass it could cut at, accept uniforms sit far from
min(1, p/q), and draw uniforms sit in the middle of a CDF step. The integers are then
compared exactly.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import get_config
from synth import inputs as S

from harness import weights_cuda

pytestmark = pytest.mark.gpu

PARAMS = [(1.0, 20, 0.95), (0.7, 32, 1.0), (1.3, 1, 1.0), (0.9, 8, 0.6)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_inject_gb300 import build
    build.build()


def _ctx(vocab, batch):
    from block_diffusion_speculative_inject_gb300 import Context, Limits
    cfg = get_config("mini_bf16", vocab=vocab, batch=batch)
    w = S.make_weights(cfg, 3)
    return cfg, Context(cfg, weights_cuda(w), Limits(max_batch=batch, max_pages=8, max_positions=256,
                                                     max_inject_rows=64))


def _safe_top_p(rows, T, k, top_p):
    """top_p moved (downwards) until no row has a top-k prefix mass within 2e-4 of it."""
    if top_p >= 1.0:
        return top_p
    cums = [np.cumsum(np.sort(O.sampling_probs(lg, T, k, 1.0))[::-1]) for lg in rows]
    for _ in range(400):
        if all(np.min(np.abs(c - top_p)) >= 2e-4 for c in cums):
            return top_p
        top_p -= 7e-4
    raise AssertionError("no safe top_p")


def _mid_step(dist, rng):
    """A uniform in the middle of the CDF step (vocabulary order) of a likely token."""
    dist = np.asarray(dist, dtype=np.float64)
    total = dist.sum()
    cands = np.flatnonzero(dist >= 0.02 * total)
    t = int(rng.choice(cands))
    before = dist[:t].sum()
    return (before + 0.5 * dist[t]) / total, t


@pytest.mark.parametrize("vocab", [4999, 5000])
@pytest.mark.parametrize("T,k,top_p", PARAMS)
def test_sample_tokens_matches_oracle(vocab, T, k, top_p):
    cfg, ctx = _ctx(vocab, 4)
    rng = np.random.default_rng(vocab + k)
    rows = 12
    lg = rng.normal(0, 2.0, (rows, vocab)).astype(np.float32)
    lg64 = lg.astype(np.float64)
    tp = _safe_top_p(lg64, T, k, top_p)
    us, want = [], []
    for r in range(rows):
        u, t = _mid_step(O.sampling_probs(lg64[r], T, k, tp), rng)
        us.append(u)
        want.append(O.sample_token(lg64[r], u, T, k, tp))
        assert want[-1] == t
    got = ctx.sample_tokens(torch.from_numpy(lg).cuda(), torch.tensor(us, dtype=torch.float32).cuda(), T, k, tp)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), want)
    ctx.close()


def _plan(p_rows, q_rows, reject_at, rng):
    """Drafts drawn from q (mid-step uniforms), accept uniforms with margin that accept
    before `reject_at` and reject there when the ratio allows it."""
    K = len(q_rows)
    draft, u_acc, u_draft = [], [], []
    for j in range(K):
        u, d = _mid_step(q_rows[j], rng)
        draft.append(d)
        u_draft.append(u)
        ratio = min(1.0, p_rows[j][d] / q_rows[j][d])
        if j == reject_at and ratio <= 0.96:
            u_acc.append((ratio + 1.0) / 2)
        elif ratio >= 0.04:
            u_acc.append(ratio / 2)
        else:
            u_acc.append((ratio + 1.0) / 2)
    return draft, u_acc, u_draft


@pytest.mark.parametrize("vocab", [4999, 151936])
@pytest.mark.parametrize("T,k,top_p", PARAMS)
def test_verify_sample_matches_oracle(vocab, T, k, top_p):
    B = 5
    cfg, ctx = _ctx(vocab, B)
    K = cfg.block_k
    rng = np.random.default_rng(vocab * 7 + k)
    tl = rng.normal(0, 1.0, (B, K + 1, vocab)).astype(np.float32)
    dl = (tl[:, :K] + rng.normal(0, 0.7, (B, K, vocab))).astype(np.float32)   # a draft close to the target
    # request 4: the draft equals the target at positions 0-2; it accepts 0 and 1 (ratio 1,
    # uniform 0) and rejects 2 with a uniform of 1.0, leaving a zero residual: the draw then
    # comes from p (the fallback)
    dl[4, :3] = tl[4, :3]
    # request 2: the draft equals the target everywhere, so every position accepts and the
    # bonus is drawn from p_K
    dl[2] = tl[2, :K]
    tl64, dl64 = tl.astype(np.float64), dl.astype(np.float64)
    tp = _safe_top_p(list(tl64.reshape(-1, vocab)) + list(dl64.reshape(-1, vocab)), T, k, top_p)
    plans = {0: 0, 1: 3, 2: None, 3: K - 1, 4: None}
    drafts, u_acc, u_res, want = [], [], [], []
    for b in range(B):
        p_rows = [O.sampling_probs(r, T, k, tp) for r in tl64[b]]
        q_rows = [O.sampling_probs(r, T, k, tp) for r in dl64[b]]
        d, ua, _ = _plan(p_rows, q_rows, plans[b], rng)
        if b == 4:
            ua[0] = ua[1] = 0.0
            ua[2] = 1.0
        # the distribution the resample draw uses, from the oracle's own path
        a = 0
        while a < K and ua[a] < O.accept_prob(p_rows[a], q_rows[a], d[a]):
            a += 1
        dist = O.residual_dist(p_rows[a], q_rows[a]) if a < K else p_rows[K]
        ur, _ = _mid_step(dist, rng)
        wa, toks = O.verify_sample_logits(tl64[b], dl64[b], d, ua, ur, T, k, tp)
        assert wa == a
        drafts.append(d)
        u_acc.append(ua)
        u_res.append(ur)
        want.append((wa, toks))
    acc, out, nxt = ctx.verify_sample(torch.from_numpy(tl).cuda(), torch.from_numpy(dl).cuda(),
                                      torch.tensor(drafts, dtype=torch.int32).cuda(),
                                      torch.tensor(u_acc, dtype=torch.float32).cuda(),
                                      torch.tensor(u_res, dtype=torch.float32).cuda(), T, k, tp)
    torch.cuda.synchronize()
    acc, out, nxt = acc.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy()
    for b, (wa, toks) in enumerate(want):
        assert acc[b] == wa, (b, acc[b], wa)
        np.testing.assert_array_equal(out[b, :wa + 1], toks)
        assert np.all(out[b, wa + 1:] == -1)
        assert nxt[b] == toks[-1]
    assert acc[2] == K          # all accepted: the bonus came from p_K
    assert acc[4] == 2          # the fallback row
    ctx.close()


def test_sampling_parameter_errors():
    from block_diffusion_speculative_inject_gb300 import DFlashError
    cfg, ctx = _ctx(5000, 2)
    lg = torch.zeros((2, 5000), device="cuda")
    u = torch.zeros((2,), device="cuda")
    for T, k, tp in [(0.0, 5, 0.9), (1.0, 33, 0.9), (1.0, 5, 0.0), (1.0, 5, 1.5)]:
        with pytest.raises(DFlashError, match="INVALID_ARG"):
            ctx.sample_tokens(lg, u, T, k, tp)
    with pytest.raises(DFlashError, match="UNSUPPORTED"):
        ctx.sample_tokens(lg, u, 1.0, 0, 0.9)
    ctx.close()
