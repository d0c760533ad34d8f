"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle, on the same
seeded inputs, element by element at small sizes and on whole steps of the workloads."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import get_config
from synth import inputs as S

from harness import Pair, check_argmax, check_logits, check_topk, to_np, LOGIT_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_inject_gb300 import build
    build.build()


def _limits(**kw):
    from block_diffusion_speculative_inject_gb300 import Limits
    return Limits(**kw)


# ----------------------------------------------------------------------------- verify
def test_verify_greedy_bit_exact_random_and_edges():
    from block_diffusion_speculative_inject_gb300 import Context
    cfg = get_config("mini_bf16", n_layers=1)
    pair = Pair(cfg, _limits(max_batch=4, max_pages=4, max_positions=128, max_inject_rows=16))
    K, V = cfg.block_k, 7    # tiny alphabet -> many matches
    g = torch.Generator().manual_seed(5)
    B = 1000                 # verification is not bounded by max_batch
    draft = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    target = torch.randint(0, V, (B, K + 1), generator=g, dtype=torch.int32)
    copy = torch.rand((B, K), generator=g) < 0.8
    target[:, :K] = torch.where(copy, draft, target[:, :K])
    target[0, :K] = draft[0]                  # all accepted -> bonus
    target[1, 0] = (draft[1, 0] + 1) % V      # first rejected
    acc, out, nxt = pair.ctx.verify(draft.cuda(), target.cuda())
    wa, wo, wn = O.verify_greedy(draft.numpy(), target.numpy())
    np.testing.assert_array_equal(acc.cpu().numpy(), wa)
    np.testing.assert_array_equal(out.cpu().numpy(), wo)
    np.testing.assert_array_equal(nxt.cpu().numpy(), wn)
    assert acc[0].item() == K and acc[1].item() == 0
    assert int(acc.max()) <= K


# ----------------------------------------------------------------------------- whole steps
def _run_steps(cfg, limits, ctx_lens, steps, seed=0, check_kv=True):
    pair = Pair(cfg, limits, seed=seed)
    B = len(ctx_lens)
    reqs = list(range(10, 10 + B))
    pair.inject(reqs, ctx_lens, "prefill", reset=True)
    tol = LOGIT_TOL[cfg.dtype]
    if check_kv:
        for i, r in enumerate(reqs):
            for l in range(cfg.n_layers):
                k, v = pair.ctx.export_kv(r, l, 0, ctx_lens[i])
                wk, wv = pair.orc.cache[r]["K"][l], pair.orc.cache[r]["V"][l]
                kv_tol = 1e-4 if cfg.dtype == "f32" else 3e-2
                np.testing.assert_allclose(to_np(k), wk, atol=kv_tol, rtol=0)
                np.testing.assert_allclose(to_np(v), wv, atol=kv_tol, rtol=0)
                if cfg.dtype == "bf16":
                    # the injection GEMMs accumulate exactly enough that fewer than one stored
                    # value in a thousand lands on the other bf16 neighbour of the oracle's
                    assert np.mean(to_np(k) == wk) > 0.999 and np.mean(to_np(v) == wv) > 0.999
    anchors = S.make_anchors(cfg, B, seed, 0)
    for step in range(steps):
        out = pair.ctx.draft(reqs, anchors.cuda(), want_logits=True)
        lg = to_np(out["logits"])
        am = out["argmax"].cpu().numpy()
        ti, tv = out["topk_idx"].cpu().numpy(), to_np(out["topk_val"])
        oam = np.zeros((B, cfg.block_k), dtype=np.int64)
        for i, r in enumerate(reqs):
            w_am, w_idx, w_val, w_lg = pair.orc.draft(r, int(anchors[i]))
            oam[i] = w_am
            check_logits(cfg, lg[i], w_lg, f"step {step} req {r}")
            check_argmax(am[i], w_lg, f"step {step} req {r}")
            check_topk(ti[i], tv[i], w_lg, cfg.topk, tol, f"step {step} req {r}")
            assert np.all(am[i] == ti[i][:, 0])
        # the synthetic target follows the oracle's argmax; both verifies see the same ids
        target = S.make_targets(cfg, torch.from_numpy(oam), seed, step)
        acc, toks, nxt = pair.ctx.verify(out["argmax"], target.cuda())
        wa, wo, wn = O.verify_greedy(am, target.numpy())
        np.testing.assert_array_equal(acc.cpu().numpy(), wa)
        np.testing.assert_array_equal(toks.cpu().numpy(), wo)
        np.testing.assert_array_equal(nxt.cpu().numpy(), wn)
        # next round: inject the anchor + accepted drafts (a + 1 positions)
        n_new = (acc.cpu() + 1).tolist()
        pair.inject(reqs, n_new, ("step", step))
        for i, r in enumerate(reqs):
            assert pair.ctx.context_len(r) == pair.orc.context_len(r)
        anchors = nxt.cpu()
    return pair


def test_tiny_f32_steps():
    cfg = get_config("tiny_f32")
    _run_steps(cfg, _limits(max_batch=1, max_pages=8, max_positions=256, max_inject_rows=64),
               [64], steps=3)


def test_mini_bf16_ragged_batch_steps():
    cfg = get_config("mini_bf16")
    _run_steps(cfg, _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100),
               [50, 173, 300], steps=3)


@pytest.mark.parametrize("name,scale", [("tiny_f32", 0.5), ("mini_bf16", 2.5)])
def test_input_embedding_scale_steps(name, scale):
    """input_embedding_scale multiplies every block row's embedding ("DFlash 2 块扩散投机解码技术
    详解" §2.2). The first layer's input norm cannot see it; the residual stream and so the
    logits do."""
    cfg = get_config(name, input_embedding_scale=scale)
    if name == "tiny_f32":
        lim = _limits(max_batch=1, max_pages=8, max_positions=256, max_inject_rows=64)
        lens = [64]
    else:
        lim = _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100)
        lens = [50, 173, 300]
    _run_steps(cfg, lim, lens, steps=2)


def test_mini_bf16_empty_context_and_page_edges():
    cfg = get_config("mini_bf16", n_layers=1)
    _run_steps(cfg, _limits(max_batch=4, max_pages=16, max_positions=512, max_inject_rows=64),
               [1, 63, 64, 65], steps=2)


# ----------------------------------------------------------------------------- invariants on the GPU
def test_incremental_injection_equals_one_shot():
    cfg = get_config("mini_bf16")
    w = S.make_weights(cfg, 3)
    lim = _limits(max_batch=2, max_pages=16, max_positions=512, max_inject_rows=40)
    a = Pair(cfg, lim, seed=3, weights=w)
    b = Pair(cfg, lim, seed=3, weights=w)
    n = 150
    feats = S.make_features(cfg, n, 3, "ctx")
    fg = [f.cuda() for f in feats]
    a.ctx.inject([1], [n], fg, reset=True)
    g = torch.Generator().manual_seed(4)
    s = 0
    while s < n:
        m = min(int(torch.randint(1, 17, (1,), generator=g)), n - s)
        b.ctx.inject([1], [m], [f[s:s + m].contiguous() for f in fg])
        s += m
    # The GEMM's split-K factor follows the row count of each call, so the fp32 sums differ in
    # order between chunkings, and chunks of at most 32 rows apply the fc RMSNorm as a row
    # scale after the K/V GEMM instead of before it. Both orders carry the pre-rounding K/V to
    # about 1e-7 relative (fp32 sums of exactly accumulated k-blocks), so a bf16 rounding of
    # the stored K/V lands on the other neighbour for a small fraction of values.
    for l in range(cfg.n_layers):
        for x, y in zip(a.ctx.export_kv(1, l, 0, n), b.ctx.export_kv(1, l, 0, n)):
            x, y = x.float(), y.float()
            assert torch.mean((x == y).float()).item() > 0.99
            # one unit in the last place of the value, plus an absolute floor for values that
            # RoPE's rotation made small relative to their operands (2^-15 of the largest |K|)
            ulp = torch.abs(x) * 2.0 ** -7 + 1e-30
            assert torch.all(torch.abs(x - y) <= ulp + 2.0 ** -15 * torch.abs(x).max())


def test_results_independent_of_batch_composition():
    """A request's logits do not depend on which other requests share the step. The split-K
    factor of a GEMM depends on the batch's row count, so agreement is to fp32 summation
    order (well inside the oracle tolerance), and the argmax must not move."""
    cfg = get_config("mini_bf16")
    w = S.make_weights(cfg, 6)
    lim = _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=128)
    p = Pair(cfg, lim, seed=6, weights=w)
    lens = [120, 37, 260]
    p.inject([1, 2, 3], lens, "prefill", reset=True)
    anchors = torch.tensor([5, 17, 99], dtype=torch.int32).cuda()
    full = p.ctx.draft([1, 2, 3], anchors, want_logits=True)
    solo = p.ctx.draft([2], anchors[1:2].contiguous(), want_logits=True)
    perm = p.ctx.draft([3, 1], anchors[[2, 0]].contiguous(), want_logits=True)
    for a, b in [(full["logits"][1], solo["logits"][0]), (full["logits"][2], perm["logits"][0]),
                 (full["logits"][0], perm["logits"][1])]:
        assert torch.max(torch.abs(a - b)).item() < 1e-4
    assert torch.equal(full["argmax"][1], solo["argmax"][0])
    assert torch.equal(full["argmax"][2], perm["argmax"][0])
    assert torch.equal(full["argmax"][0], perm["argmax"][1])


def test_tensor_core_gemm_matches_ffma_gemm(monkeypatch):
    """The tcgen05 path and the FFMA path of the same bf16 context agree closely, over a
    batch whose 144 block rows span two token tiles, a ragged vocabulary and split-K."""
    cfg = get_config("mini_bf16")
    w = S.make_weights(cfg, 8)
    lim = _limits(max_batch=9, max_pages=64, max_positions=512, max_inject_rows=700)
    lens = [50 + 29 * i for i in range(9)]
    outs = []
    for force in ("0", "1"):
        monkeypatch.setenv("DFLASH_FORCE_FFMA", force)
        p = Pair(cfg, lim, seed=8, weights=w)
        p.inject(list(range(9)), lens, "prefill", reset=True)
        anchors = torch.arange(9, dtype=torch.int32).cuda() * 7
        o = p.ctx.draft(list(range(9)), anchors, want_logits=True)
        k, v = p.ctx.export_kv(4, 1, 0, lens[4])
        outs.append((o["logits"].cpu(), o["argmax"].cpu(), k.float().cpu(), v.float().cpu()))
        p.ctx.close()
    (lt, at, kt, vt), (lf, af, kf, vf) = outs
    assert torch.max(torch.abs(lt - lf)).item() < 1e-3
    assert torch.mean((at == af).float()).item() > 0.99
    assert torch.max(torch.abs(kt - kf)).item() < 3e-2 and torch.mean((kt == kf).float()).item() > 0.99
    assert torch.max(torch.abs(vt - vf)).item() < 3e-2 and torch.mean((vt == vf).float()).item() > 0.99


def test_host_errors_change_no_state():
    from block_diffusion_speculative_inject_gb300 import DFlashError
    cfg = get_config("mini_bf16", n_layers=1)
    p = Pair(cfg, _limits(max_batch=2, max_pages=3, max_positions=256, max_inject_rows=64))
    p.inject([1], [100], "a", reset=True)             # 2 pages
    free = p.ctx.free_pages()
    feats = [f.cuda() for f in S.make_features(cfg, 130, 0, "b")]
    with pytest.raises(DFlashError) as e:              # needs 3 more pages, 1 free
        p.ctx.inject([2], [130], feats)
    assert e.value.status == -2
    assert p.ctx.free_pages() == free and p.ctx.context_len(1) == 100
    with pytest.raises(DFlashError) as e:
        p.ctx.draft([7], torch.zeros(1, dtype=torch.int32).cuda())
    assert e.value.status == -3
    with pytest.raises(DFlashError) as e:              # duplicate request in one call
        p.ctx.draft([1, 1], torch.zeros(2, dtype=torch.int32).cuda())
    assert e.value.status == -1
    with pytest.raises(DFlashError) as e:              # beyond max_positions
        p.ctx.inject([1], [200], [f[:1] for f in feats])
    assert e.value.status == -1 and p.ctx.context_len(1) == 100
    # a bad anchor id is caught on the device and reported by the next call
    p.ctx.draft([1], torch.tensor([10 ** 6], dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    with pytest.raises(DFlashError) as e:
        p.ctx.draft([1], torch.zeros(1, dtype=torch.int32).cuda())
    assert e.value.status == -5
    p.ctx.draft([1], torch.zeros(1, dtype=torch.int32).cuda())   # flag cleared
    # truncate / release return pages
    p.ctx.truncate(1, 10)
    assert p.ctx.free_pages() == free + 1
    p.ctx.release(1)
    assert p.ctx.free_pages() == 3


# ----------------------------------------------------------------------------- full-size workload
@pytest.mark.slow
@pytest.mark.parametrize("scale", [1.0, 2.0])
def test_q8b_b1_full_size_step(scale):
    """Qwen3-8B-shaped draft, batch 1, context 2048, K=15: two whole steps vs the oracle, at
    the workload's input_embedding_scale of 1 and at 2."""
    cfg = get_config("q8b_b1", input_embedding_scale=scale)
    _run_steps(cfg, _limits(max_batch=1, max_pages=40, max_positions=2304, max_inject_rows=2048),
               [2048], steps=2, check_kv=False)


def test_graph_replay_matches_eager(monkeypatch):
    """The draft step replayed from a captured CUDA graph gives the same argmax / top-k bits as
    the eagerly launched step, across repeated steps with changing context lengths."""
    cfg = get_config("mini_bf16")
    w = S.make_weights(cfg, 9)
    lim = _limits(max_batch=3, max_pages=48, max_positions=1024, max_inject_rows=400)
    results = []
    for no_graphs in ("1", "0"):
        monkeypatch.setenv("DFLASH_NO_GRAPHS", no_graphs)
        p = Pair(cfg, lim, seed=9, weights=w)
        p.inject([1, 2, 3], [120, 250, 64], "prefill", reset=True)
        outs = []
        for step in range(5):
            anchors = S.make_anchors(cfg, 3, 9, step).cuda()
            o = p.ctx.draft([1, 2, 3], anchors)
            outs.append((o["argmax"].cpu(), o["topk_idx"].cpu(), o["topk_val"].cpu()))
            n_new = [1 + (step + i) % 5 for i in range(3)]
            p.inject([1, 2, 3], n_new, ("g", step))
        results.append(outs)
        p.ctx.close()
    for (a1, i1, v1), (a2, i2, v2) in zip(*results):
        assert torch.equal(a1, a2) and torch.equal(i1, i2) and torch.equal(v1, v2)


@pytest.mark.parametrize("name,B,rows", [("mini_bf16", 1, 64), ("mini_bf16", 3, 100), ("mini_bf16", 3, 20),
                                         ("tiny_f32", 2, 64)])
def test_inject_blocks_appends_each_blocks_counted_prefix(name, B, rows):
    """dflash_inject_blocks on whole verify blocks (K + 1 feature rows per request, counts
    0..K+1 including both ends) against the oracle injecting the counted prefix of each block:
    the cache rows, the context lengths and the next draft. The counted rows are packed
    first: up to 32 of them take the fused cache-write epilogue, 39 the separate cache-write
    kernel, and max_inject_rows 20 cuts the packed rows into chunks."""
    cfg = get_config(name)
    Q = cfg.block_k + 1
    pair = Pair(cfg, _limits(max_batch=B, max_pages=48, max_positions=1024, max_inject_rows=rows))
    reqs = list(range(20, 20 + B))
    lens = [70, 129, 64][:B]
    pair.inject(reqs, lens, "prefill", reset=True)
    rng = np.random.default_rng(7)
    counts = [[0, Q, 5][:B], [Q, Q, 7][:B], [Q, 1, 0][:B], rng.integers(1, Q + 1, size=B).tolist()]
    if B == 1:
        counts = [[0], [Q], [1], [9]]
    for step, n_new in enumerate(counts):
        blocks = [S.make_features(cfg, Q, 0, ("block", step), r) for r in reqs]
        feats = [torch.cat([b[f] for b in blocks], 0).cuda().contiguous() for f in range(cfg.n_feat)]
        pair.ctx.inject_blocks(reqs, n_new, Q, feats)
        for r, b, n in zip(reqs, blocks, n_new):
            pair.orc.inject(r, [to_np(x[:n]).astype(np.float64) for x in b])
    kv_tol = 1e-4 if cfg.dtype == "f32" else 3e-2
    equal = total = 0
    for i, r in enumerate(reqs):
        n_all = pair.ctx.context_len(r)
        assert n_all == pair.orc.context_len(r) == lens[i] + sum(c[i] for c in counts)
        for l in range(cfg.n_layers):
            k, v = pair.ctx.export_kv(r, l, lens[i], n_all - lens[i])
            for got, want in ((k, pair.orc.cache[r]["K"][l][lens[i]:]), (v, pair.orc.cache[r]["V"][l][lens[i]:])):
                got = to_np(got)
                np.testing.assert_allclose(got, want, atol=kv_tol, rtol=0)
                equal += int(np.sum(got == want))
                total += got.size
    if cfg.dtype == "bf16":
        assert equal > 0.999 * total, f"{equal} of {total} cached values equal"
    anchors = S.make_anchors(cfg, B, 0, 3)
    out = pair.ctx.draft(reqs, anchors.cuda(), want_logits=True)
    lg, am = to_np(out["logits"]), out["argmax"].cpu().numpy()
    ti, tv = out["topk_idx"].cpu().numpy(), to_np(out["topk_val"])
    for i, r in enumerate(reqs):
        w_am, w_idx, w_val, w_lg = pair.orc.draft(r, int(anchors[i]))
        check_logits(cfg, lg[i], w_lg, f"req {r}")
        check_argmax(am[i], w_lg, f"req {r}")
        check_topk(ti[i], tv[i], w_lg, cfg.topk, LOGIT_TOL[cfg.dtype], f"req {r}")


def test_inject_blocks_rejects_counts_outside_the_block():
    cfg = get_config("mini_bf16")
    from block_diffusion_speculative_inject_gb300 import DFlashError
    pair = Pair(cfg, _limits(max_batch=2, max_pages=16, max_positions=512, max_inject_rows=64))
    pair.inject([1, 2], [10, 10], "prefill", reset=True)
    feats = [torch.zeros((2 * 16, cfg.target_hidden), dtype=torch.bfloat16, device="cuda")
             for _ in range(cfg.n_feat)]
    for n_new, rows in (([17, 1], 16), ([-1, 1], 16), ([1, 1], 0)):
        with pytest.raises(DFlashError):
            pair.ctx.inject_blocks([1, 2], n_new, rows, feats)
        assert pair.ctx.context_len(1) == 10 and pair.ctx.context_len(2) == 10
