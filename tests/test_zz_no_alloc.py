"""dflash_topk_noalloc — the top-k entry point that allocates no device memory.

It serves callers that cannot call the CUDA allocator (work being recorded into a CUDA
graph, runtimes with a fixed device-memory budget): its candidate scratch is a fixed array
compiled into the library. Checked here against the top-k of dflash_draft_step on the same
logits, on two calls in a row. This file is collected last so a stop-at-first-failure run
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import get_config
from synth import inputs as S

pytestmark = pytest.mark.gpu


def _noalloc(lib, logits, k, stream=None):
    rows, vocab = logits.shape
    dev = logits.device
    am = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    ti = torch.full((rows, k), -1, dtype=torch.int32, device=dev)
    tv = torch.zeros((rows, k), dtype=torch.float32, device=dev)
    msg = ctypes.create_string_buffer(256)
    s = torch.cuda.current_stream() if stream is None else stream
    st = lib.dflash_topk_noalloc(ctypes.c_void_p(s.cuda_stream), rows, vocab, k,
                                 ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(am.data_ptr()),
                                 ctypes.c_void_p(ti.data_ptr()), ctypes.c_void_p(tv.data_ptr()), msg, 256)
    return st, msg.value.decode(), am, ti, tv


def test_noalloc_topk_matches_draft_step_on_two_calls():
    from block_diffusion_speculative_inject_gb300 import Context, Limits, build, library
    build.build()
    lib = library()
    cfg = get_config("mini_bf16")
    w = S.make_weights(cfg, 11)
    wg = {k: v.cuda() for k, v in w.items() if k != "layers"}
    wg["layers"] = [{k: v.cuda() for k, v in lw.items()} for lw in w["layers"]]
    ctx = Context(cfg, wg, Limits(max_batch=3, max_pages=32, max_positions=512, max_inject_rows=256))
    lens = [90, 200, 33]
    feats = [torch.cat([S.make_features(cfg, n, 11, "na", r)[f] for r, n in enumerate(lens)]).cuda()
             for f in range(cfg.n_feat)]
    ctx.inject([0, 1, 2], lens, feats, reset=True)
    for call in range(2):
        anchors = S.make_anchors(cfg, 3, 11, call).cuda()
        ref = ctx.draft([0, 1, 2], anchors, want_logits=True)
        logits = ref["logits"].reshape(-1, cfg.vocab).contiguous()
        st, msg, am, ti, tv = _noalloc(lib, logits, cfg.topk)
        torch.cuda.synchronize()
        assert st == 0, msg
        # same fp32 logits and the same tie rule: indices agree exactly, values to fp32 rounding
        np.testing.assert_array_equal(am.cpu().numpy(), ref["argmax"].reshape(-1).cpu().numpy())
        np.testing.assert_array_equal(ti.cpu().numpy(), ref["topk_idx"].reshape(-1, cfg.topk).cpu().numpy())
        np.testing.assert_allclose(tv.cpu().numpy(), ref["topk_val"].reshape(-1, cfg.topk).cpu().numpy(),
                                   rtol=0, atol=1e-6)
    ctx.close()


def test_noalloc_topk_rejects_sizes_beyond_its_scratch():
    from block_diffusion_speculative_inject_gb300 import library
    lib = library()
    logits = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    msg = ctypes.create_string_buffer(256)
    null = ctypes.c_void_p(0)
    # 5000 rows x 38 chunks x 16 > 524288 candidates: refused before any launch
    st = lib.dflash_topk_noalloc(null, 5000, 151936, 16, ctypes.c_void_p(logits.data_ptr()),
                                 ctypes.c_void_p(logits.data_ptr()), None, None, msg, 256)
    assert st == -1 and b"scratch" in msg.value
    st = lib.dflash_topk_noalloc(null, 1, 8, 33, ctypes.c_void_p(logits.data_ptr()),
                                 ctypes.c_void_p(logits.data_ptr()), None, None, msg, 256)
    assert st == -1


def test_noalloc_topk_full_vocabulary_with_ties_across_chunks():
    """vocab 151936 (38 chunks of 4096, more chunks than k = 16, so the merge takes its
    candidate-pool path) against the definition: values descending, ties to the lower index.
    Row 1 plants equal values on both sides of chunk boundaries; row 2 is constant."""
    import oracle as O
    from block_diffusion_speculative_inject_gb300 import build, library
    build.build()
    lib = library()
    g = torch.Generator().manual_seed(3)
    V, k = 151936, 16
    x = torch.randn((4, V), generator=g)
    for c in (1, 5, 17, 36):                 # 8 equal maxima straddling chunk edges
        x[1, c * 4096 - 1] = 9.0
        x[1, c * 4096] = 9.0
    x[1, 100] = 9.0
    x[2] = 0.25
    x[3, -1] = 50.0                          # the last entry of the ragged last chunk
    for call in range(2):
        st, msg, am, ti, tv = _noalloc(lib, x.cuda(), k)
        torch.cuda.synchronize()
        assert st == 0, msg
        want_idx, want_val = O.topk_desc(x.double().numpy(), k)
        np.testing.assert_array_equal(ti.cpu().numpy(), want_idx)
        np.testing.assert_array_equal(tv.cpu().numpy(), want_val.astype(np.float32))
        np.testing.assert_array_equal(am.cpu().numpy(), want_idx[:, 0])
    assert ti[1, :9].tolist() == [100, 4095, 4096, 20479, 20480, 69631, 69632, 147455, 147456]
    assert ti[2].tolist() == list(range(k))


def test_noalloc_topk_more_rows_than_a_grid_dimension_of_65535():
    from block_diffusion_speculative_inject_gb300 import library
    lib = library()
    g = torch.Generator().manual_seed(4)
    x = torch.randn((70000, 8), generator=g)
    st, msg, am, ti, tv = _noalloc(lib, x.cuda(), 1)
    torch.cuda.synchronize()
    assert st == 0, msg
    np.testing.assert_array_equal(am.cpu().numpy(), x.argmax(1).numpy())
