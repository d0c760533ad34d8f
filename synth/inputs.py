"""Seeded generators for every input of the draft step.

Nothing here computes any part of the method: the functions only draw random
tensors of the right shape and distribution (torch CPU generators, one per named
stream so that any subset can be regenerated on its own). Weights are returned
as CPU tensors in the storage dtype ("f32" -> float32, "bf16" -> bfloat16) in the
[out_features, in_features] row-major layout of a linear layer.

Recipe (the workloads fix the projection-weight and hidden-state distributions;
norm weights are not fixed, and are drawn around 1 so that a dropped or
mis-indexed norm weight changes the result):
  projection weights, embedding, LM head, fc:  N(0, 0.02)
  RMSNorm weights (fc_norm, in/post/final norm, q/k head norms): 1 + N(0, 0.1)
  target hidden states (features):              N(0, 1)
  anchor tokens:                                uniform over [0, V)
  context lengths:                              uniform integers in [ctx_min, ctx_max]
  newly accepted positions per step:            uniform integers in [1, n_new_max]
  synthetic target ids:                         the given draft argmax with probability
                                                accept_p, else uniform over [0, V);
                                                the bonus position is uniform
  dynamic convolutions (when configured):       base taps 0.5 + N(0, 0.1), correction
                                                maps N(0, 0.005)
  path selector (when configured):              codebooks N(0, 0.25), hidden map N(0, 0.02)
"""
import hashlib
from concurrent.futures import ThreadPoolExecutor

import torch

from .configs import DraftConfig

_WEIGHT_STD = 0.02
_NORM_STD = 0.1


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(*parts) -> torch.Generator:
    return torch.Generator().manual_seed(_seed(*parts))


def storage_dtype(cfg: DraftConfig) -> torch.dtype:
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def _normal(shape, std, mean, dtype, *tag):
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(0.0, std, generator=_gen(*tag))
    if mean:
        t += mean
    return t.to(dtype)


def weight_specs(cfg: DraftConfig):
    """(name, shape, std, mean) for every weight tensor; layer tensors are 'L{i}.name'."""
    H, F, V, I, hd = cfg.hidden, cfg.feat_dim, cfg.vocab, cfg.intermediate, cfg.head_dim
    specs = [
        ("embed", (V, H), _WEIGHT_STD, 0.0),
        ("lm_head", (V, H), _WEIGHT_STD, 0.0),
        ("fc", (H, F), _WEIGHT_STD, 0.0),
        ("fc_norm", (H,), _NORM_STD, 1.0),
        ("final_norm", (H,), _NORM_STD, 1.0),
    ]
    for i in range(cfg.n_layers):
        specs += [
            (f"L{i}.in_norm", (H,), _NORM_STD, 1.0),
            (f"L{i}.wq", (cfg.q_dim, H), _WEIGHT_STD, 0.0),
            (f"L{i}.wk", (cfg.kv_dim, H), _WEIGHT_STD, 0.0),
            (f"L{i}.wv", (cfg.kv_dim, H), _WEIGHT_STD, 0.0),
            (f"L{i}.q_norm", (hd,), _NORM_STD, 1.0),
            (f"L{i}.k_norm", (hd,), _NORM_STD, 1.0),
            (f"L{i}.wo", (H, cfg.q_dim), _WEIGHT_STD, 0.0),
            (f"L{i}.post_norm", (H,), _NORM_STD, 1.0),
            (f"L{i}.w_gate", (I, H), _WEIGHT_STD, 0.0),
            (f"L{i}.w_up", (I, H), _WEIGHT_STD, 0.0),
            (f"L{i}.w_down", (H, I), _WEIGHT_STD, 0.0),
        ]
        if cfg.dyn_conv:
            # four convolutions per layer: attention input / output, MLP input / output
            specs += [
                (f"L{i}.conv_base", (4, 2, H), _NORM_STD, 0.5),
                (f"L{i}.conv_proj", (4, 2 * (H // 16), H), 0.005, 0.0),
            ]
    if cfg.selector_rank:
        r = cfg.selector_rank
        specs += [
            ("sel_pred_codebook", (V, r), 0.25, 0.0),
            ("sel_succ_codebook", (V, r), 0.25, 0.0),
            ("sel_hidden_proj", (r, H), _WEIGHT_STD, 0.0),
        ]
    return specs


LAYER_KEYS = ("in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "post_norm",
              "w_gate", "w_up", "w_down")
CONV_KEYS = ("conv_base", "conv_proj")
SELECTOR_KEYS = ("sel_pred_codebook", "sel_succ_codebook", "sel_hidden_proj")


def make_weights(cfg: DraftConfig, seed: int = 0, threads: int = 8):
    """Dict with embed, lm_head, fc, fc_norm, final_norm and layers=[dict per layer]."""
    dt = storage_dtype(cfg)
    specs = weight_specs(cfg)

    def one(spec):
        name, shape, std, mean = spec
        return name, _normal(shape, std, mean, dt, "weights", cfg.name, seed, name)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        flat = dict(ex.map(one, specs))
    w = {k: flat[k] for k in ("embed", "lm_head", "fc", "fc_norm", "final_norm")}
    keys = LAYER_KEYS + (CONV_KEYS if cfg.dyn_conv else ())
    w["layers"] = [{k: flat[f"L{i}.{k}"] for k in keys} for i in range(cfg.n_layers)]
    for k in SELECTOR_KEYS:
        if k in flat:
            w[k] = flat[k]
    if cfg.mask_embedding:
        w["mask_embedding"] = _normal((cfg.hidden,), 0.02, 0.0, dt, "weights", cfg.name, seed, "mask_embedding")
    return w


def make_features(cfg: DraftConfig, n_rows: int, seed: int, *stream):
    """n_feat target hidden-state tensors, each [n_rows, target_hidden], N(0, 1).

    `stream` names the draw (e.g. ("prefill", request)) so that one request's rows can be
    regenerated without drawing the others.
    """
    dt = storage_dtype(cfg)
    return [_normal((n_rows, cfg.target_hidden), 1.0, 0.0, dt, "feat", cfg.name, seed, f, *stream)
            for f in range(cfg.n_feat)]


def make_context_lengths(cfg: DraftConfig, seed: int = 0):
    g = _gen("ctxlen", cfg.name, seed)
    return torch.randint(cfg.ctx_min, cfg.ctx_max + 1, (cfg.batch,), generator=g).tolist()


def make_n_new(cfg: DraftConfig, batch: int, seed: int, step: int):
    g = _gen("nnew", cfg.name, seed, step)
    return torch.randint(1, cfg.n_new_max + 1, (batch,), generator=g).tolist()


def make_anchors(cfg: DraftConfig, batch: int, seed: int, step: int = 0):
    g = _gen("anchor", cfg.name, seed, step)
    return torch.randint(0, cfg.vocab, (batch,), generator=g, dtype=torch.int64).to(torch.int32)


def make_targets(cfg: DraftConfig, draft_argmax, seed: int, step: int = 0, p: float = None):
    """Synthetic target ids [B, K+1] (int32) standing in for the target model.

    Position j < K copies draft_argmax[b, j] with probability p, else draws uniformly;
    the bonus position K is uniform. `draft_argmax` is an int tensor [B, K].
    """
    p = cfg.accept_p if p is None else p
    d = torch.as_tensor(draft_argmax).to(torch.int64)
    B, K = d.shape
    g = _gen("target", cfg.name, seed, step)
    coin = torch.rand((B, K), generator=g) < p
    rnd = torch.randint(0, cfg.vocab, (B, K + 1), generator=g, dtype=torch.int64)
    t = rnd.clone()
    t[:, :K] = torch.where(coin, d, rnd[:, :K])
    return t.to(torch.int32)


def make_uniforms(n: int, seed: int, *stream):
    """n float64 uniforms in [0, 1) (for sampling-based verification)."""
    g = _gen("uniform", seed, *stream)
    return torch.rand(n, generator=g, dtype=torch.float64)
