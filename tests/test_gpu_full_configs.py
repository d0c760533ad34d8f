"""Full-size parity on the batched workloads: the CUDA library runs the whole batch, the oracle
recomputes a seeded sample of requests (per-request results do not depend on the rest of
the batch). Sampled requests get the same synthetic features on both sides; the others get
device-drawn features that only the GPU sees."""
import zlib

import numpy as np
import pytest
import torch

import oracle as O
from synth import get_config
from synth import inputs as S

from harness import LOGIT_TOL, check_argmax, check_logits, check_topk, to_np, weights_cuda, weights_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_inject_gb300 import build
    build.build()


def _device_feats(cfg, n, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    return [torch.randn((n, cfg.target_hidden), generator=g, device="cuda").to(dt) for _ in range(cfg.n_feat)]


def _run(cfg_name, sample, steps, ctx_override=None, checked=None):
    """steps verify-driven draft steps; the oracle drafts the sampled requests at the steps in
    `checked` (all by default) and follows every step's injection, so its cache of the sampled
    requests is compared with the library's over all positions injected after the prefill."""
    from block_diffusion_speculative_inject_gb300 import Context, Limits
    cfg = get_config(cfg_name)
    B = cfg.batch
    ctx_lens = ctx_override or S.make_context_lengths(cfg, 0)
    w = S.make_weights(cfg, 0)
    pages = sum((c + 64 * (steps + 2)) // 64 + 2 for c in ctx_lens)
    ctx = Context(cfg, weights_cuda(w), Limits(max_batch=B, max_requests=B, max_pages=pages,
                                               max_positions=max(ctx_lens) + 64 * (steps + 2),
                                               max_inject_rows=8192))
    orc = O.OracleDraft(cfg, weights_np(w))
    del w
    reqs = list(range(B))

    def inject(n_new, tag, reset=False):
        # the prefill as packed rows; a step's a + 1 positions per request as the target
        # hands them over: a block of K + 1 feature rows per request (dflash_inject_blocks)
        Q = cfg.block_k + 1
        parts = []
        for r, n in zip(reqs, n_new):
            rows = n if reset else Q
            if r in sample:
                f = S.make_features(cfg, rows, 0, tag, r)
                orc.inject(r, [to_np(x[:n]).astype(np.float64) for x in f], reset=reset)
                parts.append([x.cuda() for x in f])
            else:
                parts.append(_device_feats(cfg, rows, zlib.crc32(repr((tag, r)).encode())))
        feats = [torch.cat([p[f] for p in parts], 0).contiguous() for f in range(cfg.n_feat)]
        if reset:
            ctx.inject(reqs, n_new, feats, reset=True)
        else:
            ctx.inject_blocks(reqs, n_new, Q, feats)

    inject(ctx_lens, "prefill", reset=True)
    anchors = S.make_anchors(cfg, B, 0, 0)
    tol = LOGIT_TOL[cfg.dtype]
    checked = set(range(steps)) if checked is None else set(checked)
    for step in range(steps):
        # unchecked steps take the production path (CUDA graph, no logits written)
        out = ctx.draft(reqs, anchors.cuda(), want_logits=step in checked)
        am = out["argmax"].cpu().numpy()
        ti, tv = out["topk_idx"].cpu().numpy(), to_np(out["topk_val"])
        oam = am.copy()
        for r in sample if step in checked else ():
            w_am, w_idx, w_val, w_lg = orc.draft(r, int(anchors[r]))
            lg = to_np(out["logits"][r])
            check_logits(cfg, lg, w_lg, f"{cfg_name} step {step} req {r}")
            check_argmax(am[r], w_lg, f"{cfg_name} step {step} req {r}")
            check_topk(ti[r], tv[r], w_lg, cfg.topk, tol, f"{cfg_name} step {step} req {r}")
            oam[r] = w_am
        target = S.make_targets(cfg, torch.from_numpy(oam), 0, step)
        acc, toks, nxt = ctx.verify(out["argmax"], target.cuda())
        wa, wo, wn = O.verify_greedy(am, target.numpy())
        np.testing.assert_array_equal(acc.cpu().numpy(), wa)
        np.testing.assert_array_equal(toks.cpu().numpy(), wo)
        np.testing.assert_array_equal(nxt.cpu().numpy(), wn)
        inject((acc.cpu() + 1).tolist(), ("step", step))
        anchors = nxt.cpu()
        for r in sample:
            assert ctx.context_len(r) == orc.context_len(r)
    for r in sample:
        # the cache rows written by the steps' incremental injections: all within the bound,
        # and at least 99.9% of them (over every layer, K and V) equal to the oracle's
        c0, n = ctx_lens[r], ctx.context_len(r) - ctx_lens[r]
        equal = total = 0
        for l in range(cfg.n_layers):
            k, v = ctx.export_kv(r, l, c0, n)
            for got, want in ((k, orc.cache[r]["K"][l][c0:c0 + n]), (v, orc.cache[r]["V"][l][c0:c0 + n])):
                got = to_np(got)
                np.testing.assert_allclose(got, want, atol=3e-2 if cfg.dtype == "bf16" else 1e-4, rtol=0)
                equal += int(np.sum(got == want))
                total += got.size
        assert equal > 0.999 * total, f"{equal} of {total} cached values equal"
    ctx.close()


def test_q8b_b32_ragged_batch():
    """Qwen3-8B-shaped draft, 32 requests with contexts U[512, 8192], K=15; requests 3 and 17."""
    _run("q8b_b32", sample=(3, 17), steps=2)


def test_q4b_b128_large_batch():
    """Qwen3-4B-shaped draft, 128 requests of context 1024, K=7; requests 0 and 101."""
    _run("q4b_b128", sample=(0, 101), steps=2)


def test_q27b_b8_long_context():
    """27B-target-shaped draft, 8 requests of context 32768, K=15; request 5, over 64
    consecutive verify-driven steps (each injects the a + 1 positions its verify accepted, from
    the K + 1-row verify block of target features), drafts compared with the oracle at 8 of
    them, the cache rows of all 64 injections after."""
    _run("q27b_b8", sample=(5,), steps=64, checked=(0, 1, 2, 9, 21, 36, 50, 63))
