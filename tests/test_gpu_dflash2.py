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
