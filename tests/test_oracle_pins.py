"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test fixes one part of the oracle by brute force, a closed form, an independent
library routine, an invariant the pages state, or exact rational arithmetic, chosen
so that a plausible slip (dropped term, wrong sign, wrong index, transposed operand)
fails at least one of them.
"""
import itertools
import json
import os
import types
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cfg(**kw):
    base = dict(hidden=64, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=16,
                intermediate=96, vocab=300, n_feat=3, target_hidden=32, block_k=5,
                topk=8, mask_id=299, qk_norm=1, rms_eps=1e-6, rope_theta=1e4,
                input_embedding_scale=1.0, dtype="f64")
    base.update(kw)
    return types.SimpleNamespace(**base)


def _weights(c, seed=0, norm_std=0.1):
    rng = np.random.default_rng(seed)
    n = lambda *s: rng.normal(0, 0.02, s)
    nw = lambda *s: 1.0 + rng.normal(0, norm_std, s)
    w = dict(embed=n(c.vocab, c.hidden) * 20, lm_head=n(c.vocab, c.hidden),
             fc=n(c.hidden, c.n_feat * c.target_hidden) * 5, fc_norm=nw(c.hidden),
             final_norm=nw(c.hidden), layers=[])
    q, kv = c.n_q_heads * c.head_dim, c.n_kv_heads * c.head_dim
    for _ in range(c.n_layers):
        w["layers"].append(dict(
            in_norm=nw(c.hidden), wq=n(q, c.hidden) * 10, wk=n(kv, c.hidden) * 10,
            wv=n(kv, c.hidden) * 10, q_norm=nw(c.head_dim), k_norm=nw(c.head_dim),
            wo=n(c.hidden, q) * 5, post_norm=nw(c.hidden), w_gate=n(c.intermediate, c.hidden) * 5,
            w_up=n(c.intermediate, c.hidden) * 5, w_down=n(c.hidden, c.intermediate) * 5))
    return w


def _feats(c, n, seed):
    rng = np.random.default_rng(seed)
    return [rng.normal(0, 1, (n, c.target_hidden)) for _ in range(c.n_feat)]


# ----------------------------------------------------------------------------- rounding
def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 2000), rng.normal(0, 1e30, 2000),
        rng.uniform(-1, 1, 2000) * 2.0 ** -130,          # bf16 subnormal range
    ]).astype(np.float32)
    # exact ties: 1 + 2^-8 style values with odd and even neighbours
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(2 + 2 ** -7), 3 * 2 ** -9 + 2 ** -1], np.float32)
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_round_ties_to_even_by_hand():
    assert O.bf16_round(np.array([1 + 2 ** -8]))[0] == 1.0                # even neighbour is 1.0
    assert O.bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6    # even neighbour above
    assert O.bf16_round(np.array([1 + 2 ** -8 + 2 ** -30]))[0] == 1 + 2 ** -7  # past the tie
    assert np.isinf(O.bf16_round(np.array([3.5e38]))[0])


def test_f32_round_is_ieee_single():
    x = np.array([1 + 2 ** -24, 1 + 3 * 2 ** -24, 0.1])
    np.testing.assert_array_equal(O.f32_round(x), x.astype(np.float32).astype(np.float64))


# ----------------------------------------------------------------------------- elementwise
def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(2)
    x, w = rng.normal(0, 3, (7, 48)), rng.normal(1, 0.2, 48)
    want = F.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rmsnorm(x, w, 1e-6), want, rtol=1e-13, atol=1e-13)


def test_silu_softmax_match_torch():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 4, (5, 33))
    np.testing.assert_allclose(O.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-13)
    np.testing.assert_allclose(O.softmax(x), torch.softmax(torch.from_numpy(x), -1).numpy(),
                               rtol=1e-13, atol=1e-15)


def test_rope_closed_forms():
    hd, theta = 16, 1e6
    half = hd // 2
    # position 0 is the identity
    x = np.random.default_rng(4).normal(size=(3, 2, hd))
    np.testing.assert_allclose(O.rope(x, np.zeros(3), theta), x, atol=0)
    # pairs are (i, i + hd/2): e_0 at position p -> cos p at 0, sin p at hd/2 (frequency 1)
    e0 = np.zeros((1, hd)); e0[0, 0] = 1.0
    r = O.rope(e0, np.array([3]), theta)
    want = np.zeros(hd); want[0] = np.cos(3); want[half] = np.sin(3)
    np.testing.assert_allclose(r[0], want, atol=1e-15)
    # second pair rotates with frequency theta^(-2/hd); x2 maps with the opposite sign
    e1 = np.zeros((1, hd)); e1[0, half + 1] = 1.0
    ang = 5 * theta ** (-2.0 / hd)
    r = O.rope(e1, np.array([5]), theta)
    want = np.zeros(hd); want[1] = -np.sin(ang); want[half + 1] = np.cos(ang)
    np.testing.assert_allclose(r[0], want, atol=1e-15)


def test_rope_composition_and_relative_position():
    rng = np.random.default_rng(5)
    hd, theta = 32, 1e6
    q, k = rng.normal(size=(1, hd)), rng.normal(size=(1, hd))
    a, b = 1234, 40000
    np.testing.assert_allclose(O.rope(O.rope(q, [a], theta), [b], theta),
                               O.rope(q, [a + b], theta), atol=1e-9)
    d1 = np.dot(O.rope(q, [700], theta)[0], O.rope(k, [650], theta)[0])
    d2 = np.dot(O.rope(q, [30050], theta)[0], O.rope(k, [30000], theta)[0])
    assert abs(d1 - d2) < 1e-9
    # rotation keeps the norm
    assert abs(np.linalg.norm(O.rope(q, [99], theta)) - np.linalg.norm(q)) < 1e-12


# ----------------------------------------------------------------------------- context fusion
def test_fc_concat_order_block_decomposition():
    c = _cfg()
    w = _weights(c)
    od = O.OracleDraft(c, w)
    fe = _feats(c, 6, 7)
    acc = sum(fe[f] @ w["fc"][:, f * c.target_hidden:(f + 1) * c.target_hidden].T
              for f in range(c.n_feat))
    want = O.rmsnorm(acc, w["fc_norm"], c.rms_eps)
    np.testing.assert_allclose(od.fuse(fe), want, rtol=1e-12, atol=1e-12)
    # the norm really is applied: with unit weights every fused row has RMS 1
    w2 = dict(w, fc_norm=np.ones(c.hidden))
    g = O.OracleDraft(c, w2).fuse(fe)
    np.testing.assert_allclose(np.sqrt(np.mean(g * g, -1)), 1.0, rtol=1e-6)


def test_fc_shape_chain_golden():
    gold = json.load(open(os.path.join(GOLDEN, "fc_shape_chain.json")))
    c = _cfg(hidden=gold["fused_width"], n_feat=gold["n_feat"], target_hidden=gold["target_hidden"])
    rng = np.random.default_rng(0)
    w = dict(fc=rng.normal(0, 0.02, (c.hidden, c.n_feat * c.target_hidden)).astype(np.float32),
             fc_norm=np.ones(c.hidden))
    fe = [rng.normal(size=(gold["tokens"], c.target_hidden)) for _ in range(c.n_feat)]
    assert np.concatenate(fe, 1).shape == (gold["tokens"], gold["concat_width"])
    g = O.OracleDraft(c, w).fuse(fe)
    assert g.shape == (gold["tokens"], gold["fused_width"])


# ----------------------------------------------------------------------------- layer vs library
def _torch_layer(c, lw, x, ctx_k, ctx_v, pos):
    """Independent composition of the decoder layer from torch fp64 library routines."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    n = x.shape[0]
    X = t(x)
    xn = F.rms_norm(X, (c.hidden,), t(lw["in_norm"]), eps=c.rms_eps)
    q = F.linear(xn, t(lw["wq"])).view(n, c.n_q_heads, c.head_dim)
    k = F.linear(xn, t(lw["wk"])).view(n, c.n_kv_heads, c.head_dim)
    v = F.linear(xn, t(lw["wv"])).view(n, c.n_kv_heads, c.head_dim)
    q = F.rms_norm(q, (c.head_dim,), t(lw["q_norm"]), eps=c.rms_eps)
    k = F.rms_norm(k, (c.head_dim,), t(lw["k_norm"]), eps=c.rms_eps)
    q = t(O.rope(q.numpy(), pos, c.rope_theta))          # rope is pinned on its own
    k = t(O.rope(k.numpy(), pos, c.rope_theta))
    keys = torch.cat([t(ctx_k), k], 0).transpose(0, 1)    # [nkv, S, hd]
    vals = torch.cat([t(ctx_v), v], 0).transpose(0, 1)
    mask = None
    if getattr(c, "block_causal", 0):
        # context keys visible to all rows; block key i visible to block rows j >= i
        n_ctx = ctx_k.shape[0]
        mask = torch.ones((n, n_ctx + n), dtype=torch.bool)
        mask[:, n_ctx:] = torch.tril(torch.ones((n, n), dtype=torch.bool))
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], keys[None], vals[None],
                                       attn_mask=mask, enable_gqa=True)[0]   # None: bidirectional
    o = o.transpose(0, 1).reshape(n, -1)
    X = X + F.linear(o, t(lw["wo"]))
    xn2 = F.rms_norm(X, (c.hidden,), t(lw["post_norm"]), eps=c.rms_eps)
    h = F.silu(F.linear(xn2, t(lw["w_gate"]))) * F.linear(xn2, t(lw["w_up"]))
    return (X + F.linear(h, t(lw["w_down"]))).numpy()


@pytest.mark.parametrize("nq,nkv", [(4, 2), (4, 4), (6, 2), (4, 1)])
def test_layer_matches_torch_library_composition(nq, nkv):
    c = _cfg(n_q_heads=nq, n_kv_heads=nkv)
    w = _weights(c, seed=nq * 10 + nkv)
    od = O.OracleDraft(c, w)
    rng = np.random.default_rng(8)
    n_ctx = 37
    x = rng.normal(0, 1, (c.block_k + 1, c.hidden))
    ck = rng.normal(0, 1, (n_ctx, nkv, c.head_dim))
    cv = rng.normal(0, 1, (n_ctx, nkv, c.head_dim))
    pos = np.arange(n_ctx, n_ctx + c.block_k + 1)
    np.testing.assert_allclose(od.layer(x, 0, ck, cv, pos),
                               _torch_layer(c, w["layers"][0], x, ck, cv, pos),
                               rtol=1e-10, atol=1e-11)


def test_gqa_head_mapping_equals_duplicated_kv_heads():
    """nq=4, nkv=2 must equal nq=4, nkv=4 whose kv heads are [h0, h0, h1, h1]."""
    c2 = _cfg(n_q_heads=4, n_kv_heads=2, n_layers=1)
    w2 = _weights(c2, seed=11)
    c4 = _cfg(n_q_heads=4, n_kv_heads=4, n_layers=1)
    hd = c2.head_dim
    lw = dict(w2["layers"][0])
    dup = lambda m: np.concatenate([m[0:hd], m[0:hd], m[hd:2 * hd], m[hd:2 * hd]], 0)
    lw4 = dict(lw, wk=dup(lw["wk"]), wv=dup(lw["wv"]))
    w4 = dict(w2, layers=[lw4])
    rng = np.random.default_rng(12)
    x = rng.normal(0, 1, (c2.block_k + 1, c2.hidden))
    ck = rng.normal(0, 1, (9, 2, hd)); cv = rng.normal(0, 1, (9, 2, hd))
    ck4 = ck[:, [0, 0, 1, 1]]; cv4 = cv[:, [0, 0, 1, 1]]
    pos = np.arange(9, 9 + c2.block_k + 1)
    a = O.OracleDraft(c2, w2).layer(x, 0, ck, cv, pos)
    b = O.OracleDraft(c4, w4).layer(x, 0, ck4, cv4, pos)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_in_block_attention_is_bidirectional_and_context_is_a_set():
    c = _cfg(n_layers=1)
    w = _weights(c, seed=13)
    od = O.OracleDraft(c, w)
    rng = np.random.default_rng(14)
    x = rng.normal(0, 1, (c.block_k + 1, c.hidden))
    ck = rng.normal(0, 1, (20, c.n_kv_heads, c.head_dim))
    cv = rng.normal(0, 1, (20, c.n_kv_heads, c.head_dim))
    pos = np.arange(20, 20 + c.block_k + 1)
    base = od.layer(x, 0, ck, cv, pos)
    x2 = x.copy(); x2[-1] += 1.0                    # change the last mask row only
    assert np.max(np.abs(od.layer(x2, 0, ck, cv, pos)[0] - base[0])) > 1e-6   # anchor sees it
    perm = rng.permutation(20)                      # context K/V order does not matter
    np.testing.assert_allclose(od.layer(x, 0, ck[perm], cv[perm], pos), base, rtol=1e-12, atol=1e-13)


def test_injected_kv_equal_inline_prepended_rows():
    """Context K/V injected from g equal the K/V the layer computes for g rows placed in
    front of the block ([P1] Step 3: g goes through the same K/V projection and is prepended).

    With unit input-norm weights, eps = 0 and fc_norm = 1, rmsnorm(g) == g, so feeding the g
    rows through the layer's own input path reproduces exactly the injected projection.
    """
    for qk in (0, 1):
        c = _cfg(n_layers=1, rms_eps=0.0, qk_norm=qk)
        w = _weights(c, seed=15)
        w["fc_norm"] = np.ones(c.hidden)
        w["layers"][0]["in_norm"] = np.ones(c.hidden)
        od = O.OracleDraft(c, w)
        n = 11
        g = od.fuse(_feats(c, n, 16))
        kc, vc = od.project_kv(g, np.arange(n), 0)
        rng = np.random.default_rng(17)
        xb = rng.normal(0, 1, (c.block_k + 1, c.hidden))
        pos_b = np.arange(n, n + c.block_k + 1)
        injected = od.layer(xb, 0, kc, vc, pos_b)
        empty = np.zeros((0, c.n_kv_heads, c.head_dim))
        inline = od.layer(np.concatenate([g, xb]), 0, empty, empty, np.arange(n + c.block_k + 1))[n:]
        np.testing.assert_allclose(injected, inline, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------- request-level invariants
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_incremental_injection_equals_one_shot(dtype):
    c = _cfg(dtype=dtype)
    w = _weights(c, seed=18)
    rng = np.random.default_rng(19)
    n = 70
    fe = _feats(c, n, 20)
    one = O.OracleDraft(c, w); one.inject(0, fe)
    inc = O.OracleDraft(c, w)
    s = 0
    while s < n:
        m = min(int(rng.integers(1, 17)), n - s)
        inc.inject(0, [f[s:s + m] for f in fe])
        s += m
    for l in range(c.n_layers):
        np.testing.assert_array_equal(one.cache[0]["K"][l], inc.cache[0]["K"][l])
        np.testing.assert_array_equal(one.cache[0]["V"][l], inc.cache[0]["V"][l])
    np.testing.assert_array_equal(one.logits(0, 5), inc.logits(0, 5))


def test_anchor_gives_no_candidate_and_k_candidates_per_request():
    gold = json.load(open(os.path.join(GOLDEN, "block_layout.json")))
    for case in gold["cases"]:
        c = _cfg(block_k=case["K"], n_layers=1)
        w = _weights(c, seed=21)
        od = O.OracleDraft(c, w)
        od.inject(0, _feats(c, 8, 22))
        assert len(od.block_tokens(3)) == case["queries"]
        am, idx, val, lg = od.draft(0, 3)
        assert lg.shape == (case["candidates"], c.vocab)
        assert am.shape == (case["candidates"],)
        assert idx.shape == (case["candidates"], c.topk)


def test_mask_rows_depend_on_the_anchor_and_context():
    c = _cfg()
    w = _weights(c, seed=23)
    od = O.OracleDraft(c, w)
    od.inject(0, _feats(c, 12, 24))
    a = od.logits(0, 3)
    assert np.max(np.abs(a - od.logits(0, 4))) > 1e-6       # anchor token matters
    od.inject(0, _feats(c, 1, 25))
    assert np.max(np.abs(a - od.logits(0, 3))) > 1e-6       # one more context position matters


def test_requests_are_independent():
    c = _cfg(dtype="bf16")
    w = _weights(c, seed=26)
    solo = O.OracleDraft(c, w); solo.inject(7, _feats(c, 30, 27))
    mixed = O.OracleDraft(c, w)
    mixed.inject(3, _feats(c, 50, 28)); mixed.inject(7, _feats(c, 30, 27)); mixed.inject(9, _feats(c, 5, 29))
    np.testing.assert_array_equal(solo.logits(7, 11), mixed.logits(7, 11))


# ----------------------------------------------------------------------------- selection
def test_topk_and_argmax_brute_force_with_ties():
    rng = np.random.default_rng(30)
    for trial in range(200):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, n + 1))
        x = rng.integers(-3, 4, n).astype(np.float64)      # many exact ties
        want = sorted(range(n), key=lambda i: (-x[i], i))[:k]
        idx, val = O.topk_desc(x[None], k)
        assert list(idx[0]) == want
        assert list(val[0]) == [x[i] for i in want]
        assert O.argmax_lowest(x[None])[0] == want[0]


# ----------------------------------------------------------------------------- greedy verify
def test_greedy_verify_brute_force_against_prefix_formula():
    """All (draft, target) pairs with V=3, K<=3 against the cumprod formula of [P2] §2.3."""
    V = 3
    for K in range(1, 4):
        drafts = np.array(list(itertools.product(range(V), repeat=K)))
        targets = np.array(list(itertools.product(range(V), repeat=K + 1)))
        D = np.repeat(drafts, len(targets), 0)
        T = np.tile(targets, (len(drafts), 1))
        acc, out, nxt = O.verify_greedy(D, T)
        a_formula = np.cumprod(D == T[:, :-1], axis=1).sum(axis=1)
        np.testing.assert_array_equal(acc, a_formula)
        assert np.all(acc <= K)
        for i in range(len(D)):
            a = acc[i]
            emitted = out[i][out[i] >= 0]
            assert len(emitted) == a + 1 <= K + 1
            np.testing.assert_array_equal(emitted[:a], D[i, :a])
            assert emitted[a] == T[i, a] == nxt[i]


def test_greedy_verify_worked_example_golden():
    gold = json.load(open(os.path.join(GOLDEN, "verify_worked_example.json")))
    vocab = gold["vocab"]
    d = np.array([[vocab[t] for t in gold["draft"]]])
    t = np.array([[vocab[t] for t in gold["target"]]])
    acc, out, nxt = O.verify_greedy(d, t)
    assert acc[0] == gold["expected_accept_len"]
    assert list(out[0][out[0] >= 0]) == [vocab[t] for t in gold["expected_emitted"]]
    assert nxt[0] == vocab[gold["expected_next_anchor"]]


# ----------------------------------------------------------------------------- rejection sampling
def _rand_dist(rng, V, zeros=False):
    v = [int(x) for x in rng.integers(1, 9, V)]
    if zeros:
        v[int(rng.integers(0, V))] = 0
    return O.as_fraction_dist(v)


def _exact_output_distribution(p_of, q_rows, V, K):
    """Exact law of the emitted tokens, completed by the target to K+1 tokens."""
    out = {}

    def complete(seq, prob):
        if len(seq) == K + 1:
            out[tuple(seq)] = out.get(tuple(seq), 0) + prob
            return
        p = p_of(tuple(seq))
        for t in range(V):
            if p[t]:
                complete(seq + [t], prob * p[t])

    for d in itertools.product(range(V), repeat=K):
        pd = Fraction(1)
        for j in range(K):
            pd *= q_rows[j][d[j]]
        if pd == 0:
            continue
        prefix, prob = [], pd
        for j in range(K):
            p = p_of(tuple(prefix))
            a = O.accept_prob(p, q_rows[j], d[j])
            if a < 1:                                   # rejection branch
                res = O.residual_dist(p, q_rows[j])
                for t in range(V):
                    if res[t]:
                        complete(prefix + [t], prob * (1 - a) * res[t])
            prob *= a
            if prob == 0:
                break
            prefix = prefix + [d[j]]
        else:
            p = p_of(tuple(prefix))                     # all accepted: bonus from p_K
            for t in range(V):
                if p[t]:
                    complete(prefix + [t], prob * p[t])
    return out


@pytest.mark.parametrize("V,K,seed", [(3, 1, 0), (3, 2, 1), (4, 2, 2), (4, 2, 3), (2, 3, 4)])
def test_rejection_sampling_reproduces_target_exactly(V, K, seed):
    rng = np.random.default_rng(100 + seed)
    table = {}

    def p_of(prefix):
        if prefix not in table:
            table[prefix] = _rand_dist(rng, V, zeros=(len(prefix) % 2 == 1))
        return table[prefix]

    q_rows = [_rand_dist(rng, V, zeros=(j == 0)) for j in range(K)]
    got = _exact_output_distribution(p_of, q_rows, V, K)
    for seq in itertools.product(range(V), repeat=K + 1):
        want = Fraction(1)
        for i in range(K + 1):
            want *= p_of(tuple(seq[:i]))[seq[i]]
        assert got.get(seq, 0) == want, (seq, got.get(seq, 0), want)


def test_residual_falls_back_to_target_when_nothing_is_left():
    p = O.as_fraction_dist([1, 2, 3])
    assert O.residual_dist(p, p) == p
    q = O.as_fraction_dist([3, 2, 1])
    r = O.residual_dist(p, q)
    assert r == [0, 0, 1]


def test_verify_sample_monte_carlo_matches_exact_law():
    V, K = 3, 2
    rng = np.random.default_rng(7)
    table = {}

    def p_of(prefix):
        if prefix not in table:
            table[prefix] = _rand_dist(rng, V)
        return table[prefix]

    q_rows = [_rand_dist(rng, V) for _ in range(K)]
    first_exact = p_of(())
    n = 20000
    counts = np.zeros(V)
    mc = np.random.default_rng(8)
    for _ in range(n):
        d = [int(mc.choice(V, p=[float(x) for x in q_rows[j]])) for j in range(K)]
        p_rows = [p_of(tuple(d[:j])) for j in range(K + 1)]
        p_rows = [[float(x) for x in r] for r in p_rows]
        a, toks = O.verify_sample(p_rows, [[float(x) for x in r] for r in q_rows], d,
                                  mc.random(K), mc.random())
        assert 1 <= len(toks) == a + 1 <= K + 1
        counts[toks[0]] += 1
    # the first emitted token follows p(. | prefix) exactly; 5 sigma tolerance
    f = np.array([float(x) for x in first_exact])
    assert np.all(np.abs(counts / n - f) < 5 * np.sqrt(f * (1 - f) / n) + 1e-3)


@pytest.mark.parametrize("dtype,rnd", [("bf16", O.bf16_round), ("f32", O.f32_round)])
def test_cache_is_stored_in_the_storage_type_and_activations_are_not(dtype, rnd):
    """The KV cache lands on the storage grid; g and the logits are carried unrounded."""
    c = _cfg(dtype=dtype)
    w = _weights(c, seed=31)
    od = O.OracleDraft(c, w)
    fe = _feats(c, 20, 32)
    od.inject(0, fe)
    for l in range(c.n_layers):
        np.testing.assert_array_equal(rnd(od.cache[0]["K"][l]), od.cache[0]["K"][l])
        np.testing.assert_array_equal(rnd(od.cache[0]["V"][l]), od.cache[0]["V"][l])
    g = od.fuse(fe)
    assert np.any(O.bf16_round(g) != g) and np.any(O.f32_round(g) != g)


# ----------------------------------------------------------------------------- sampling mode
def test_sampling_probs_without_truncation_is_the_tempered_softmax():
    """top_k = V and top_p = 1 leave softmax(logits / T) (torch's routine) untouched."""
    rng = np.random.default_rng(41)
    for T in (0.5, 1.0, 1.7):
        lg = rng.normal(0, 2, 97)
        ref = torch.softmax(torch.tensor(lg, dtype=torch.float64) / T, 0).numpy()
        np.testing.assert_allclose(O.sampling_probs(lg, T, 97, 1.0), ref, rtol=1e-13, atol=1e-15)


def test_sampling_probs_top_k_is_the_softmax_of_the_k_largest():
    """top-k keeps torch.topk's set (distinct logits) and renormalises over it."""
    rng = np.random.default_rng(42)
    lg = rng.permutation(np.linspace(-3, 3, 64))
    for k in (1, 5, 20):
        vals, idx = torch.topk(torch.tensor(lg, dtype=torch.float64), k)
        ref = np.zeros(64)
        ref[idx.numpy()] = torch.softmax(vals / 0.8, 0).numpy()
        np.testing.assert_allclose(O.sampling_probs(lg, 0.8, k, 1.0), ref, rtol=1e-13, atol=1e-15)


def test_sampling_probs_top_p_closed_form():
    """logits (2, 1, 0, -1), T = 1, top_p = 0.8: softmax mass 0.644 < 0.8 <= 0.881 after two
    tokens, so two survive with probabilities sigmoid(1) and 1 - sigmoid(1)."""
    p = O.sampling_probs(np.array([2.0, 1.0, 0.0, -1.0]), 1.0, 4, 0.8)
    s = 1.0 / (1.0 + np.exp(-1.0))
    np.testing.assert_allclose(p, [s, 1.0 - s, 0.0, 0.0], rtol=1e-14)


def test_sampling_probs_top_p_keeps_the_shortest_sufficient_prefix():
    """The kept set is a prefix of the descending order whose softmax mass reaches top_p,
    and dropping its last token falls short (minimality), after top-k truncation."""
    rng = np.random.default_rng(43)
    for trial in range(50):
        V = int(rng.integers(5, 60))
        lg = rng.normal(0, 1.5, V)
        k = int(rng.integers(1, V + 1))
        top_p = float(rng.uniform(0.05, 0.99))
        T = float(rng.uniform(0.3, 2.0))
        p = O.sampling_probs(lg, T, k, top_p)
        kept = np.flatnonzero(p)
        order = np.argsort(-lg, kind="stable")[:k]
        full = np.exp(lg[order] / T - np.max(lg[order] / T))
        full /= full.sum()
        n = len(kept)
        assert set(kept) == set(order[:n])
        assert full[:n].sum() >= top_p - 1e-12
        if n > 1:
            assert full[:n - 1].sum() < top_p
        np.testing.assert_allclose(p.sum(), 1.0, rtol=1e-12)


def test_sampling_probs_temperature_scaling_and_ties():
    """Temperature T equals dividing the logits by T first; a tie at the top-k boundary
    keeps the lower vocabulary index."""
    lg = np.array([0.5, 2.0, -1.0, 2.0, 1.0])
    np.testing.assert_allclose(O.sampling_probs(lg, 0.25, 3, 0.9), O.sampling_probs(lg * 4, 1.0, 3, 0.9))
    p = O.sampling_probs(np.array([1.0, 3.0, 2.0, 2.0]), 1.0, 2, 1.0)
    assert p[2] > 0 and p[3] == 0


def test_sample_token_inverse_cdf_steps():
    """Draws follow the cumulative distribution in index order."""
    lg = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    assert O.sample_token(lg, 0.05, 1.0, 4, 1.0) == 0
    assert O.sample_token(lg, 0.15, 1.0, 4, 1.0) == 1
    assert O.sample_token(lg, 0.59, 1.0, 4, 1.0) == 2
    assert O.sample_token(lg, 0.61, 1.0, 4, 1.0) == 3


def test_verify_sample_logits_first_token_follows_truncated_target():
    """With drafts drawn from the truncated draft distribution, the first emitted token
    of the sampling verify follows the truncated target distribution (Monte Carlo)."""
    rng = np.random.default_rng(44)
    V, K, T, k, tp = 12, 2, 0.9, 6, 0.9
    tl = rng.normal(0, 1.2, (K + 1, V))
    dl = rng.normal(0, 1.2, (K, V))
    p0 = O.sampling_probs(tl[0], T, k, tp)
    n = 20000
    counts = np.zeros(V)
    for _ in range(n):
        d = [O.sample_token(dl[j], rng.random(), T, k, tp) for j in range(K)]
        a, toks = O.verify_sample_logits(tl, dl, d, rng.random(K), rng.random(), T, k, tp)
        assert 1 <= len(toks) == a + 1 <= K + 1
        counts[toks[0]] += 1
    assert np.all(np.abs(counts / n - p0) < 5 * np.sqrt(p0 * (1 - p0) / n) + 1e-3)


# ----------------------------------------------------------------------------- variants
def test_causal_block_layer_matches_torch_masked_attention():
    """The causal variant equals torch's scaled_dot_product_attention with a mask that
    shows every context key and block keys 0..j to block row j; a row does not depend on
    later block rows."""
    c = _cfg(n_q_heads=4, n_kv_heads=2, block_causal=1)
    w = _weights(c, seed=61)
    od = O.OracleDraft(c, w)
    rng = np.random.default_rng(62)
    n_ctx = 21
    x = rng.normal(0, 1, (c.block_k + 1, c.hidden))
    ck = rng.normal(0, 1, (n_ctx, 2, c.head_dim))
    cv = rng.normal(0, 1, (n_ctx, 2, c.head_dim))
    pos = np.arange(n_ctx, n_ctx + c.block_k + 1)
    full = od.layer(x, 0, ck, cv, pos)
    np.testing.assert_allclose(full, _torch_layer(c, w["layers"][0], x, ck, cv, pos), rtol=1e-10, atol=1e-11)
    for j in (0, 2):
        part = od.layer(x[:j + 1], 0, ck, cv, pos[:j + 1])
        np.testing.assert_allclose(part[j], full[j], rtol=1e-12, atol=1e-13)
    bi = O.OracleDraft(_cfg(n_q_heads=4, n_kv_heads=2), w).layer(x, 0, ck, cv, pos)
    assert np.abs(bi[0] - full[0]).max() > 1e-6      # the flag changes the anchor row


def test_mask_embedding_replaces_the_mask_rows_only():
    """With the trained mask embedding equal to E[mask_id] the draft is unchanged; another
    vector changes the mask rows' logits."""
    c0 = _cfg()
    c1 = _cfg(mask_embedding=1)
    w = _weights(c0, seed=63)
    fe = _feats(c0, 12, 64)
    base = O.OracleDraft(c0, w)
    base.inject(0, fe)
    same = O.OracleDraft(c1, dict(w, mask_embedding=np.array(w["embed"][c0.mask_id])))
    same.inject(0, fe)
    np.testing.assert_allclose(same.logits(0, 5), base.logits(0, 5), rtol=1e-13, atol=1e-13)
    other = O.OracleDraft(c1, dict(w, mask_embedding=np.random.default_rng(65).normal(0, 0.02, c0.hidden)))
    other.inject(0, fe)
    assert np.abs(other.logits(0, 5) - base.logits(0, 5)).max() > 1e-6


def test_output_multiplier_and_softcap_properties():
    """The scale alone is linear; the soft cap keeps the order, stays inside (-c, c) and
    inverts through atanh back to the scaled logits."""
    c0 = _cfg()
    w = _weights(c0, seed=66)
    fe = _feats(c0, 10, 67)
    raw = O.OracleDraft(c0, w)
    raw.inject(0, fe)
    r = raw.logits(0, 9)
    sc = O.OracleDraft(_cfg(output_multiplier=3.5), w)
    sc.inject(0, fe)
    np.testing.assert_allclose(sc.logits(0, 9), 3.5 * r, rtol=1e-13)
    cap = 1.0
    cp = O.OracleDraft(_cfg(output_multiplier=3.5, logit_softcap=cap), w)
    cp.inject(0, fe)
    y = cp.logits(0, 9)
    assert np.all(np.abs(y) < cap)
    for row_r, row_y in zip(r, y):
        np.testing.assert_array_equal(np.argsort(row_r, kind="stable"), np.argsort(row_y, kind="stable"))
    np.testing.assert_allclose(cap * np.arctanh(y / cap), 3.5 * r, rtol=1e-9, atol=1e-12)


# ----------------------------------------------------------------------------- DDTree
def _tuples(nodes):
    """Rank-free identity of each node: the token path from the root."""
    out = []
    for tok, parent, depth, lp in nodes:
        out.append((out[parent] if parent >= 0 else ()) + (tok,))
    return out


def test_log_softmax_norm_matches_scipy():
    from scipy.special import logsumexp
    x = np.random.default_rng(70).normal(0, 3, (4, 1000))
    np.testing.assert_allclose(O.log_softmax_norm(x), logsumexp(x, axis=-1), rtol=1e-14)


@pytest.mark.parametrize("L,kc,budget", [(3, 3, 5), (3, 4, 11), (4, 2, 9), (2, 5, 10)])
def test_ddtree_is_the_top_budget_prefixes(L, kc, budget):
    """Proposition 2 by brute force: the popped nodes are exactly the `budget` most likely
    prefixes over every depth, and each node's parent is popped before it."""
    rng = np.random.default_rng(L * 100 + kc * 10 + budget)
    for _ in range(20):
        p = rng.dirichlet(np.ones(kc + 3), size=L)[:, :kc]
        p = -np.sort(-p, axis=1)
        lp = np.log(p)
        tok = rng.permutation(1000)[:L * kc].reshape(L, kc)
        nodes = O.ddtree_build(lp, tok, budget)
        allp = []
        for d in range(1, L + 1):
            for ranks in itertools.product(range(kc), repeat=d):
                allp.append((sum(lp[i][r] for i, r in enumerate(ranks)),
                             tuple(int(tok[i][r]) for i, r in enumerate(ranks))))
        allp.sort(key=lambda e: -e[0])
        want = {t for _, t in allp[:budget]}
        assert set(_tuples(nodes)) == want
        for i, (t, parent, depth, v) in enumerate(nodes):
            assert parent < i and (parent < 0) == (depth == 1)
            if parent >= 0:
                assert nodes[parent][2] == depth - 1


def test_ddtree_mask_is_the_prefix_relation():
    rng = np.random.default_rng(71)
    lp = np.log(-np.sort(-rng.dirichlet(np.ones(6), size=4)[:, :4], axis=1))
    tok = np.arange(16).reshape(4, 4) + 100
    nodes = O.ddtree_build(lp, tok, 12)
    paths = [()] + _tuples(nodes)
    m = O.ddtree_mask(nodes)
    for i, pi in enumerate(paths):
        for j, pj in enumerate(paths):
            assert m[i, j] == (pi[:len(pj)] == pj)


def test_ddtree_walk_follows_the_target_down_the_tree():
    """The walk against a direct search: from the root, extend the accepted path while the
    target's next token labels a child of the current path."""
    rng = np.random.default_rng(72)
    lp = np.log(-np.sort(-rng.dirichlet(np.ones(5), size=3)[:, :3], axis=1))
    tok = np.array([[1, 2, 3], [1, 2, 3], [1, 2, 3]])
    nodes = O.ddtree_build(lp, tok, 9)
    paths = _tuples(nodes)
    index = {p: i for i, p in enumerate(paths)}
    for _ in range(200):
        tn = rng.integers(1, 5, len(nodes) + 1)
        a, out = O.ddtree_walk(nodes, tn)
        path, cur = (), -1
        while True:
            t = int(tn[cur + 1])
            if path + (t,) in index:
                path = path + (t,)
                cur = index[path]
            else:
                break
        assert a == len(path) and out == list(path) + [t]


# ----------------------------------------------------------------------------- DFlash 2 modules
def _conv_weights(rng, H, n=4, tap0=1.0, tap1=0.4, std=0.05):
    base = np.stack([np.stack([tap0 + rng.normal(0, 0.1, H), tap1 + rng.normal(0, 0.1, H)]) for _ in range(n)])
    proj = rng.normal(0, std, (n, 2 * (H // 16), H))
    return base, proj


def test_dyn_conv_static_taps_match_torch_depthwise_conv1d():
    """With no correction the convolution is a depthwise two-tap conv1d over the block rows
    with zero padding in front (torch's conv1d is a cross-correlation: weight[c] = (tap 1,
    tap 0))."""
    rng = np.random.default_rng(70)
    H, T = 64, 9
    x = rng.normal(0, 1, (T, H))
    base = rng.normal(0, 1, (2, H))
    y = O.dyn_conv(x, base, np.zeros((2 * H // 16, H)))
    inp = F.pad(torch.from_numpy(x.T[None]), (1, 0))                       # [1, H, T + 1]
    wt = torch.from_numpy(np.stack([base[1], base[0]], axis=1)[:, None, :])  # [H, 1, 2]
    want = F.conv1d(inp, wt, groups=H)[0].numpy().T
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("tap", [0, 1])
def test_dyn_conv_correction_is_one_value_per_16_channels(tap):
    """A single nonzero row g of the correction map (tap 0 or tap 1) changes exactly the 16
    channels of group g, by (v . x_t) times x_t (tap 0) or x_{t-1} (tap 1)."""
    rng = np.random.default_rng(71 + tap)
    H, T, G, g = 64, 6, 4, 2
    x = rng.normal(0, 1, (T, H))
    v = rng.normal(0, 1, H)
    proj = np.zeros((2 * G, H))
    proj[tap * G + g] = v
    y = O.dyn_conv(x, np.zeros((2, H)), proj)
    src = x if tap == 0 else np.vstack([np.zeros((1, H)), x[:-1]])
    want = np.zeros((T, H))
    want[:, 16 * g:16 * g + 16] = (x @ v)[:, None] * src[:, 16 * g:16 * g + 16]
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def test_dyn_conv_row_depends_on_itself_and_the_row_before_only():
    rng = np.random.default_rng(73)
    H, T = 32, 7
    x = rng.normal(0, 1, (T, H))
    base, proj = rng.normal(0, 1, (2, H)), rng.normal(0, 0.1, (2 * H // 16, H))
    y = O.dyn_conv(x, base, proj)
    for j in range(T):
        xp = x.copy()
        xp[j] += rng.normal(0, 1, H)
        d = np.abs(O.dyn_conv(xp, base, proj) - y).max(axis=1)
        changed = {t for t in range(T) if d[t] > 0}
        assert changed == ({j, j + 1} & set(range(T)))


def _torch_conv(x, base, proj):
    """The convolution from torch pieces: the static part through conv1d, the correction
    expanded to channels through a 0/1 group matrix."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    X, H = t(x), x.shape[1]
    G = H // 16
    E = torch.kron(torch.eye(G, dtype=torch.float64), torch.ones((1, 16), dtype=torch.float64))  # [G, H]
    corr = F.linear(X, t(proj))
    k0 = t(base[0]) + corr[:, :G] @ E
    k1 = t(base[1]) + corr[:, G:] @ E
    prev = F.pad(X, (0, 0, 1, 0))[:-1]
    return k0 * X + k1 * prev


def test_conv_layer_places_four_convolutions():
    """The conv layer equals a torch composition with a convolution on the attention input
    (after the input norm), on the output projection's result, on the MLP input (after the
    post-attention norm) and on the down projection's result; identity convolutions give
    back the plain layer."""
    c = _cfg(dyn_conv=1)
    w = _weights(c, seed=74)
    rng = np.random.default_rng(75)
    for lw in w["layers"]:
        lw["conv_base"], lw["conv_proj"] = _conv_weights(rng, c.hidden)
    od = O.OracleDraft(c, w)
    n_ctx = 19
    x = rng.normal(0, 1, (c.block_k + 1, c.hidden))
    ck = rng.normal(0, 1, (n_ctx, c.n_kv_heads, c.head_dim))
    cv = rng.normal(0, 1, (n_ctx, c.n_kv_heads, c.head_dim))
    pos = np.arange(n_ctx, n_ctx + c.block_k + 1)
    lw = w["layers"][0]
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    n = x.shape[0]
    X = t(x)
    xn = _torch_conv(F.rms_norm(X, (c.hidden,), t(lw["in_norm"]), eps=c.rms_eps).numpy(),
                     lw["conv_base"][0], lw["conv_proj"][0])
    q = F.rms_norm(F.linear(xn, t(lw["wq"])).view(n, c.n_q_heads, c.head_dim), (c.head_dim,), t(lw["q_norm"]),
                   eps=c.rms_eps)
    k = F.rms_norm(F.linear(xn, t(lw["wk"])).view(n, c.n_kv_heads, c.head_dim), (c.head_dim,), t(lw["k_norm"]),
                   eps=c.rms_eps)
    v = F.linear(xn, t(lw["wv"])).view(n, c.n_kv_heads, c.head_dim)
    q, k = t(O.rope(q.numpy(), pos, c.rope_theta)), t(O.rope(k.numpy(), pos, c.rope_theta))
    keys = torch.cat([t(ck), k], 0).transpose(0, 1)
    vals = torch.cat([t(cv), v], 0).transpose(0, 1)
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], keys[None], vals[None], enable_gqa=True)[0]
    o = F.linear(o.transpose(0, 1).reshape(n, -1), t(lw["wo"]))
    X = X + _torch_conv(o.numpy(), lw["conv_base"][1], lw["conv_proj"][1])
    xn2 = _torch_conv(F.rms_norm(X, (c.hidden,), t(lw["post_norm"]), eps=c.rms_eps).numpy(),
                      lw["conv_base"][2], lw["conv_proj"][2])
    h = F.silu(F.linear(xn2, t(lw["w_gate"]))) * F.linear(xn2, t(lw["w_up"]))
    want = X + _torch_conv(F.linear(h, t(lw["w_down"])).numpy(), lw["conv_base"][3], lw["conv_proj"][3])
    np.testing.assert_allclose(od.layer(x, 0, ck, cv, pos), want.numpy(), rtol=1e-10, atol=1e-11)
    # identity convolutions: the plain layer
    for lw in w["layers"]:
        lw["conv_base"] = np.stack([np.stack([np.ones(c.hidden), np.zeros(c.hidden)])] * 4)
        lw["conv_proj"] = np.zeros_like(lw["conv_proj"])
    np.testing.assert_allclose(O.OracleDraft(c, w).layer(x, 0, ck, cv, pos),
                               _torch_layer(c, w["layers"][0], x, ck, cv, pos), rtol=1e-10, atol=1e-11)


def _sel_case(rng, K=5, k=4, V=40, r=8):
    cand = np.stack([rng.permutation(V)[:k] for _ in range(K)])
    unary = -np.sort(-rng.normal(0, 1, (K, k)), axis=1)
    return cand, unary, rng.normal(0, 1, (K, r)), rng.normal(0, 1, (V, r)), rng.normal(0, 1, (V, r))


def test_select_path_without_pair_scores_is_the_argmax_path():
    rng = np.random.default_rng(80)
    cand, unary, gate, A, B = _sel_case(rng)
    for args in ((gate, np.zeros_like(A), B), (gate, A, np.zeros_like(B)), (np.zeros_like(gate), A, B)):
        toks, _ = O.select_path(7, cand, unary, *args)
        np.testing.assert_array_equal(toks, cand[:, 0])


def test_select_path_follows_a_planted_chain():
    """Codebooks that give the pair (d_{t-1}, d_t) a score of 100 and every other pair 0
    make the walk take the planted tokens, whatever their unary rank."""
    rng = np.random.default_rng(81)
    K, k, V = 5, 4, 40
    cand, unary, _, _, _ = _sel_case(rng, K, k, V)
    unary = unary / 10.0
    pick = rng.integers(0, k, K)
    d = cand[np.arange(K), pick]
    anchor = int(np.setdiff1d(np.arange(V), cand.ravel())[0])
    r = K + 1
    A, B = np.zeros((V, r)), np.zeros((V, r))
    A[anchor, 0] = 10.0
    for t in range(K):
        B[d[t], t] = 10.0
        A[d[t], t + 1] = 10.0
    toks, scores = O.select_path(anchor, cand, unary, np.ones((K, r)), A, B)
    np.testing.assert_array_equal(toks, d)
    np.testing.assert_allclose(scores[np.arange(K), pick], unary[np.arange(K), pick] + 100.0)


def test_select_path_ignores_candidate_order_and_breaks_ties_by_it():
    rng = np.random.default_rng(82)
    cand, unary, gate, A, B = _sel_case(rng)
    toks, _ = O.select_path(3, cand, unary, gate, A, B)
    perm = np.stack([rng.permutation(cand.shape[1]) for _ in range(cand.shape[0])])
    toks_p, _ = O.select_path(3, np.take_along_axis(cand, perm, 1), np.take_along_axis(unary, perm, 1), gate, A, B)
    np.testing.assert_array_equal(toks, toks_p)
    # two candidates with equal scores: the first in candidate order is taken
    cand2 = np.array([[5, 6]])
    B2 = np.zeros((10, 2))
    toks2, sc = O.select_path(1, cand2, np.array([[0.5, 0.5]]), np.ones((1, 2)), np.ones((10, 2)), B2)
    assert sc[0, 0] == sc[0, 1] and toks2[0] == 5
    toks3, _ = O.select_path(1, cand2[:, ::-1], np.array([[0.5, 0.5]]), np.ones((1, 2)), np.ones((10, 2)), B2)
    assert toks3[0] == 6


def test_draft_selector_uses_the_final_hidden_rows():
    """OracleDraft.select: zero codebooks give the draft's argmax; otherwise every pick is one
    of its position's candidates and the gate is W_h applied to the final-normed rows."""
    c = _cfg()
    w = _weights(c, seed=83)
    rng = np.random.default_rng(84)
    w["sel_hidden_proj"] = rng.normal(0, 0.3, (8, c.hidden))
    w["sel_pred_codebook"] = np.zeros((c.vocab, 8))
    w["sel_succ_codebook"] = rng.normal(0, 1, (c.vocab, 8))
    od = O.OracleDraft(c, w)
    od.inject(0, _feats(c, 14, 85))
    am, idx, val, _ = od.draft(0, 11)
    toks, _ = od.select(0, 11)
    np.testing.assert_array_equal(toks, am)
    w["sel_pred_codebook"] = rng.normal(0, 1, (c.vocab, 8))
    toks, scores = od.select(0, 11)
    gate = od.hidden(0, 11) @ w["sel_hidden_proj"].T
    want, _ = O.select_path(11, idx, val, gate, w["sel_pred_codebook"], w["sel_succ_codebook"])
    np.testing.assert_array_equal(toks, want)
    assert all(toks[t] in idx[t] for t in range(c.block_k))
    assert np.any(toks != am)


def test_select_sample_distribution_and_draws():
    """Sampling-mode selector: each position's q is the softmax of the greedy walk's scores
    over the candidates (zero elsewhere, summing to one); with zero codebooks it is the
    softmax of the unary scores; a uniform in the middle of a candidate's CDF step (in
    vocabulary order) draws that candidate; the walk continues from the drawn token."""
    rng = np.random.default_rng(90)
    K, k, V, r = 4, 5, 30, 6
    cand, unary, gate, A, B = _sel_case(rng, K, k, V, r)
    T = 0.7
    u = rng.uniform(0, 1, K)
    toks, q = O.select_sample(3, cand, unary, gate, A, B, T, u, V)
    prev = 3
    for t in range(K):
        _, sc = O.select_path(prev, cand[t:t + 1], unary[t:t + 1], gate[t:t + 1], A, B)
        want = np.exp((sc[0] - sc[0].max()) / T)
        want /= want.sum()
        np.testing.assert_allclose(q[t][cand[t]], want, rtol=1e-12)
        assert abs(q[t].sum() - 1) < 1e-12 and np.all(q[t][np.setdiff1d(np.arange(V), cand[t])] == 0)
        # the draw: the first candidate in vocabulary order whose running mass exceeds u
        order = np.argsort(cand[t])
        cum = np.cumsum(want[order])
        assert toks[t] == cand[t][order][np.searchsorted(cum, u[t], side="right")]
        prev = toks[t]
    _, q0 = O.select_sample(3, cand, unary, gate, np.zeros_like(A), B, T, u, V)
    for t in range(K):
        w = np.exp((unary[t] - unary[t].max()) / T)
        np.testing.assert_allclose(q0[t][cand[t]], w / w.sum(), rtol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rejection_sampling_with_selector_q_is_exact(seed):
    """Rejection sampling against the selector's subset distribution reproduces the target's
    distribution exactly (enumerated over all draws, exact rationals), K = 1: the subset q
    over the vocabulary is a valid draft distribution."""
    rng = np.random.default_rng(200 + seed)
    V, k = 4, 3
    cand = np.array([rng.permutation(V)[:k]])
    unary = rng.normal(0, 1, (1, k))
    gate = rng.normal(0, 1, (1, 2))
    A, B = rng.normal(0, 1, (V, 2)), rng.normal(0, 1, (V, 2))
    _, sc = O.select_path(1, cand, unary, gate, A, B)
    q = O.subset_to_vocab(cand[0], O.softmax(sc[0] / 0.9), V)
    qf = [Fraction(float(x)) for x in q]
    qf = [x / sum(qf) for x in qf]
    assert sum(1 for x in qf if x == 0) == V - k        # zero outside the candidates
    p0, p1 = _rand_dist(rng, V), _rand_dist(rng, V, zeros=True)
    law = _exact_output_distribution(lambda prefix: p0 if len(prefix) == 0 else p1, [qf], V, 1)
    for seq in itertools.product(range(V), repeat=2):
        assert law.get(seq, 0) == p0[seq[0]] * p1[seq[1]], seq


def test_ddtree_takes_every_prefix_when_the_budget_allows():
    """With a budget above the number of prefixes (sum of kc^d for d = 1..L) the tree is the
    whole prefix tree, in an order that pops every parent first, and stops there."""
    rng = np.random.default_rng(91)
    L, kc = 3, 2
    lp = np.log(-np.sort(-rng.dirichlet(np.ones(kc), size=L), axis=1))
    tok = np.arange(L * kc).reshape(L, kc)
    nodes = O.ddtree_build(lp, tok, 100)
    assert len(nodes) == sum(kc ** d for d in range(1, L + 1))
    assert len(set(_tuples(nodes))) == len(nodes)
    assert all(parent < i for i, (_, parent, _, _) in enumerate(nodes))


def test_bench_prefill_flops_match_the_scope_table():
    """The bench's prefill FLOP count (fc and every layer's K/V projection, once per
    position) for the 27B-shaped draft's whole contexts: 96.2 TF for 262,144 positions."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(os.path.dirname(GOLDEN), "..", "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from synth import get_config
    rep = bench._prefill_report(get_config("q27b_b8"), 1000.0, 8 * 32768)
    assert abs(rep["tflops"] * 1.0 - 96.2) < 0.1       # over 1 s
    assert rep["positions"] == 262144


def test_select_path_worked_example_golden():
    """The pages' walk: with the printed scores (as unary scores, no pair term) the path is
    cat, sat."""
    g = json.load(open(os.path.join(GOLDEN, "selector_walk_example.json")))
    v = g["vocab"]
    cand = np.array([[v[t] for t in pos["candidates"]] for pos in g["positions"]])
    unary = np.array([pos["scores"] for pos in g["positions"]])
    A = np.zeros((len(v), 4))
    toks, _ = O.select_path(v[g["anchor"]], cand, unary, np.ones((len(cand), 4)), A, A)
    inv = {i: t for t, i in v.items()}
    assert [inv[int(t)] for t in toks] == g["expected_path"]


@pytest.mark.parametrize("L,V,budget", [(3, 3, 5), (2, 4, 6), (3, 2, 7)])
def test_ddtree_value_is_the_expected_acceptance_under_q(L, V, budget):
    """Proposition 1: under the drafter's factorized distribution Q, the expected number of
    tokens a tree accepts (the longest prefix of Y that is a path of the tree) equals the sum
    of its nodes' prefix probabilities. Brute force over every Y in V^L."""
    rng = np.random.default_rng(L * 10 + V + budget)
    q = rng.dirichlet(np.ones(V), size=L)                       # [L][V], full distributions
    order = np.argsort(-q, axis=1, kind="stable")
    lp = np.log(np.take_along_axis(q, order, 1))
    nodes = O.ddtree_build(lp, order, budget)
    paths = set(_tuples(nodes))
    expect = 0.0
    for y in itertools.product(range(V), repeat=L):
        prob = np.prod([q[i][y[i]] for i in range(L)])
        a = 0
        while a < L and tuple(y[:a + 1]) in paths:
            a += 1
        expect += prob * a
    np.testing.assert_allclose(expect, sum(np.exp(n[3]) for n in nodes), rtol=1e-12)


# ----------------------------------------------------------------------------- block forward tail
class _Recorder(O.OracleDraft):
    """The oracle with each layer's input rows and positions recorded."""

    def layer(self, x, l, ctx_k, ctx_v, pos):
        self.seen.append((l, np.array(x), np.array(pos)))
        return super().layer(x, l, ctx_k, ctx_v, pos)


def _torch_block_logits(c, w, feats, anchor):
    """The K mask rows' logits from torch fp64 library routines alone: the context K/V from
    g = rms_norm(linear(concat(h_f), W_fc)) through each layer's k/v projection (k-norm,
    RoPE at positions 0..n-1), the block as F.embedding([anchor, mask x K]) scaled by
    input_embedding_scale on every row, the decoder layers at positions n..n+K, the final
    rms_norm of rows 1..K and F.linear with the LM-head matrix."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    n = feats[0].shape[0]
    cat = torch.cat([t(f) for f in feats], 1)
    g = F.rms_norm(F.linear(cat, t(w["fc"])), (c.hidden,), t(w["fc_norm"]), eps=c.rms_eps)
    toks = torch.tensor([anchor] + [c.mask_id] * c.block_k)
    x = F.embedding(toks, t(w["embed"])) * c.input_embedding_scale
    pos = np.arange(n, n + c.block_k + 1)
    X = x.numpy()
    for l, lw in enumerate(w["layers"]):
        k = F.linear(g, t(lw["wk"])).view(n, c.n_kv_heads, c.head_dim)
        v = F.linear(g, t(lw["wv"])).view(n, c.n_kv_heads, c.head_dim)
        k = F.rms_norm(k, (c.head_dim,), t(lw["k_norm"]), eps=c.rms_eps)
        k = O.rope(k.numpy(), np.arange(n), c.rope_theta)
        X = _torch_layer(c, lw, X, k, v.numpy(), pos)
    h = F.rms_norm(t(X)[1:], (c.hidden,), t(w["final_norm"]), eps=c.rms_eps)
    return F.linear(h, t(w["lm_head"])).numpy()


@pytest.mark.parametrize("scale", [0.5, 1.0, 3.0])
def test_block_logits_match_torch_composition(scale):
    """hidden() and logits(): the embedding gather x input_embedding_scale on all K+1 block
    rows ("DFlash 2 块扩散投机解码技术详解" §2.2), block positions ctx_len + j, the anchor
    row dropped ("DFlash：把串行 Draft 变成并行“填空”" §4.3), the final norm and the LM-head
    product, against an independent torch composition. The LM head differs from the
    embedding, so using one for the other fails."""
    c = _cfg(input_embedding_scale=scale)
    w = _weights(c, seed=40)
    assert np.max(np.abs(w["lm_head"] - w["embed"])) > 0.1
    od = O.OracleDraft(c, w)
    fe = _feats(c, 23, 41)
    od.inject(0, fe)
    for anchor in (3, 250):
        want = _torch_block_logits(c, w, fe, anchor)
        np.testing.assert_allclose(od.logits(0, anchor), want, rtol=1e-9, atol=1e-10)
        # hidden() is the final-normed K mask rows that the LM head multiplies
        np.testing.assert_allclose(od.hidden(0, anchor) @ w["lm_head"].T, want, rtol=1e-9, atol=1e-10)


def test_input_embedding_scale_multiplies_every_block_row_of_the_first_layer_input():
    c = _cfg(input_embedding_scale=2.5)
    w = _weights(c, seed=42)
    od = _Recorder(c, w)
    od.seen = []
    od.inject(0, _feats(c, 9, 43))
    od.hidden(0, 17)
    l0, x0, pos0 = od.seen[0]
    assert l0 == 0 and x0.shape == (c.block_k + 1, c.hidden)
    want = w["embed"][[17] + [c.mask_id] * c.block_k] * 2.5
    np.testing.assert_array_equal(x0, want)
    np.testing.assert_array_equal(pos0, np.arange(9, 9 + c.block_k + 1))
    # every layer sees the same block positions
    assert all(np.array_equal(p, pos0) for _, _, p in od.seen)
    # the scale acts through the residual stream: the logits move with it
    c1 = _cfg(input_embedding_scale=1.0)
    od1 = O.OracleDraft(c1, w)
    od1.inject(0, _feats(c1, 9, 43))
    assert np.max(np.abs(od1.logits(0, 17) - O.OracleDraft.logits(od, 0, 17))) > 1e-3


def test_hidden_equals_inline_prepended_context_rows():
    """One layer, unit input norm, eps 0, unit fc norm: the context enters as leading rows of
    one sequence [g rows ; scaled block embeddings] at positions 0..n+K with no cache, and
    the final-normed rows n+1..n+K of that sequence equal hidden() ("LLM的推理加速-DFlash"
    关键创新 Step 3: g goes through the same K/V projection, prepended to the block)."""
    for scale in (0.5, 4.0):
        c = _cfg(n_layers=1, rms_eps=0.0, input_embedding_scale=scale)
        w = _weights(c, seed=44)
        w["fc_norm"] = np.ones(c.hidden)
        w["layers"][0]["in_norm"] = np.ones(c.hidden)
        od = O.OracleDraft(c, w)
        n = 13
        fe = _feats(c, n, 45)
        od.inject(0, fe)
        g = od.fuse(fe)
        xb = w["embed"][[7] + [c.mask_id] * c.block_k] * scale
        empty = np.zeros((0, c.n_kv_heads, c.head_dim))
        seq = od.layer(np.concatenate([g, xb]), 0, empty, empty, np.arange(n + c.block_k + 1))
        want = O.rmsnorm(seq[n + 1:], w["final_norm"], c.rms_eps)
        np.testing.assert_allclose(od.hidden(0, 7), want, rtol=1e-10, atol=1e-11)
