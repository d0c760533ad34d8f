"""Shared set-up for the GPU parity tests: the same seeded inputs fed to the CUDA library
(through the C ABI) and to the CPU oracle, plus the comparison rules."""
import numpy as np
import torch

import oracle as O
from synth import inputs as S

# Tolerances (spec contract): logits max abs 2e-2 for bf16 storage, 1e-4 for fp32;
# verification and indices bit-exact except where the oracle's gap between the two
# candidates in question is below 1e-3.
LOGIT_TOL = {"bf16": 2e-2, "f32": 1e-4}
# The same near-tie rule holds for every top-k rank, not only the first.
TIE_GAP = 1e-3


def to_np(t):
    return t.detach().cpu().float().numpy()


def weights_np(w):
    out = {k: to_np(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: to_np(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


def weights_cuda(w, device="cuda:0"):
    out = {k: v.to(device) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: v.to(device) for k, v in lw.items()} for lw in w["layers"]]
    return out


class Pair:
    """The CUDA context and the oracle for one draft shape, fed identical inputs."""

    def __init__(self, cfg, limits, seed=0, weights=None):
        from block_diffusion_speculative_inject_gb300 import Context
        self.cfg = cfg
        self.seed = seed
        w = weights if weights is not None else S.make_weights(cfg, seed)
        self.w_cpu = w
        self.wg = weights_cuda(w)
        self.ctx = Context(cfg, self.wg, limits)
        self.orc = O.OracleDraft(cfg, weights_np(w))

    def inject(self, req_ids, n_new, tag, reset=False):
        """Draws features for each request (stream tag, request) and injects on both sides."""
        per_req = [S.make_features(self.cfg, n, self.seed, tag, r) for r, n in zip(req_ids, n_new)]
        feats = [torch.cat([p[f] for p in per_req], 0).cuda().contiguous()
                 for f in range(self.cfg.n_feat)]
        self.ctx.inject(req_ids, n_new, feats, reset=reset)
        for r, p in zip(req_ids, per_req):
            self.orc.inject(r, [to_np(x).astype(np.float64) for x in p], reset=reset)
        return feats


def check_logits(cfg, got, want, what=""):
    tol = LOGIT_TOL[cfg.dtype]
    err = np.max(np.abs(got - want))
    assert err <= tol, f"{what} logits max abs err {err:.3g} > {tol}"
    return err


def check_argmax(got, logits_oracle, what=""):
    """got [K] int; logits_oracle [K, V] fp64: equal to the oracle's argmax (fp32 decision)
    except where the oracle's top-2 gap is below TIE_GAP, in which case got must be one of
    the near-tied candidates."""
    l32 = O.f32_round(logits_oracle)
    want = O.argmax_lowest(l32)
    for j in range(len(got)):
        if got[j] == want[j]:
            continue
        top = l32[j, want[j]]
        assert top - l32[j, got[j]] < TIE_GAP, \
            f"{what} row {j}: argmax {got[j]} vs oracle {want[j]} (gap {top - l32[j, got[j]]:.3g})"


def check_topk(got_idx, got_val, logits_oracle, k, tol, what="", gap=TIE_GAP):
    """Values match the oracle's sorted top-k within tol; indices equal the oracle's except
    inside runs of near-ties (oracle gap < `gap`), where they must be valid near-tied members."""
    l32 = O.f32_round(logits_oracle)
    want_idx, want_val = O.topk_desc(l32, k)
    np.testing.assert_allclose(got_val, want_val, atol=tol, rtol=0, err_msg=what)
    for j in range(got_idx.shape[0]):
        assert len(set(got_idx[j].tolist())) == k, f"{what} row {j}: duplicate indices"
        for r in range(k):
            if got_idx[j, r] == want_idx[j, r]:
                continue
            # a swap is allowed only among candidates the oracle ranks within `gap`
            assert abs(l32[j, got_idx[j, r]] - want_val[j, r]) < gap, \
                (f"{what} row {j} rank {r}: {got_idx[j, r]} vs {want_idx[j, r]}: oracle gap "
                 f"{want_val[j, r] - l32[j, got_idx[j, r]]:.3g}, gpu values {got_val[j, r]:.7g} "
                 f"(oracle {l32[j, got_idx[j, r]]:.7g} / {want_val[j, r]:.7g})")
