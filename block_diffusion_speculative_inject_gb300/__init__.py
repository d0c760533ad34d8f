"""DFlash batched draft step on one GB300: Python binding of libdflash (include/dflash.h).

The binding only marshals arguments: torch provides device memory and streams, every
step of the path runs in the library's CUDA kernels. If libdflash.so is missing the
import of the library raises; there is no fallback implementation.

Functions with the C names take torch tensors (device buffers) and Python ints:

    ctx = dflash_create(cfg, weights, limits)                 # -> Context
    dflash_inject_context(ctx, req_ids, n_new, feats, reset=False)
    dflash_inject_blocks(ctx, req_ids, n_new, block_rows, feats)
    dflash_draft_step(ctx, req_ids, anchors, argmax, topk_idx=None, topk_val=None, logits=None)
    dflash_verify_greedy(ctx, draft, target, accept_len, out_tokens, next_anchor)
    dflash_release / dflash_truncate / dflash_context_len / dflash_export_kv / dflash_destroy

`Context` wraps the same calls as methods and allocates outputs when asked to.
"""
import ctypes

import torch

from . import _ffi

__all__ = ["DFlashError", "Context", "Limits", "dflash_create", "dflash_destroy",
           "dflash_inject_context", "dflash_inject_blocks", "dflash_draft_step", "dflash_verify_greedy",
           "dflash_release", "dflash_truncate", "dflash_context_len", "dflash_export_kv",
           "dflash_validate_config", "make_config", "library"]


class DFlashError(RuntimeError):
    def __init__(self, status, message=""):
        self.status = status
        super().__init__(f"{_ffi.STATUS.get(status, status)}: {message}")


def library():
    return _ffi.load()


def _stream_ptr(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _i32_array(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


class Limits:
    """Context capacity: batch, live requests, pages, positions, injection chunk rows."""

    def __init__(self, max_batch=1, max_requests=None, max_pages=1024, max_positions=4096,
                 max_inject_rows=4096):
        self.max_batch = max_batch
        self.max_requests = max_requests if max_requests is not None else max_batch
        self.max_pages = max_pages
        self.max_positions = max_positions
        self.max_inject_rows = max_inject_rows


def make_config(cfg, limits: Limits):
    """A dflash_config from a draft shape (any object with the DraftConfig attributes)."""
    return _ffi.Config(
        hidden=cfg.hidden, n_layers=cfg.n_layers, n_q_heads=cfg.n_q_heads,
        n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, intermediate=cfg.intermediate,
        vocab=cfg.vocab, n_feat=cfg.n_feat, target_hidden=cfg.target_hidden,
        block_k=cfg.block_k, topk=cfg.topk, mask_token_id=cfg.mask_id, qk_norm=cfg.qk_norm,
        max_batch=limits.max_batch, max_requests=limits.max_requests,
        max_pages=limits.max_pages, page_size=64, max_positions=limits.max_positions,
        max_inject_rows=limits.max_inject_rows, rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta,
        input_embedding_scale=cfg.input_embedding_scale,
        dtype=_ffi.BF16 if cfg.dtype == "bf16" else _ffi.F32,
        block_causal=getattr(cfg, "block_causal", 0),
        output_multiplier=getattr(cfg, "output_multiplier", 1.0),
        logit_softcap=getattr(cfg, "logit_softcap", 0.0),
        dyn_conv=getattr(cfg, "dyn_conv", 0),
        selector_rank=getattr(cfg, "selector_rank", 0))


def dflash_validate_config(cfg, limits: Limits):
    lib = library()
    c = make_config(cfg, limits)
    buf = ctypes.create_string_buffer(256)
    st = lib.dflash_validate_config(ctypes.byref(c), buf, 256)
    return st, buf.value.decode()


class Context:
    """Owns one dflash_ctx. Weights are torch CUDA tensors kept alive by this object."""

    def __init__(self, cfg, weights, limits: Limits, device=0):
        self.lib = library()
        self.cfg = cfg
        self.limits = limits
        self._weights = weights
        self._c = make_config(cfg, limits)
        layers = (_ffi.LayerWeights * cfg.n_layers)()
        for i, lw in enumerate(weights["layers"]):
            for k in _ffi.LayerWeights._fields_:
                name = k[0]
                setattr(layers[i], name, lw[name].data_ptr() if lw.get(name) is not None else None)
        self._layers = layers
        self._w = _ffi.Weights(embed=weights["embed"].data_ptr(), lm_head=weights["lm_head"].data_ptr(),
                               fc=weights["fc"].data_ptr(), fc_norm=weights["fc_norm"].data_ptr(),
                               final_norm=weights["final_norm"].data_ptr(),
                               layers=ctypes.cast(layers, ctypes.POINTER(_ffi.LayerWeights)),
                               mask_embedding=(weights["mask_embedding"].data_ptr()
                                               if weights.get("mask_embedding") is not None else None),
                               **{k: (weights[k].data_ptr() if weights.get(k) is not None else None)
                                  for k in ("sel_pred_codebook", "sel_succ_codebook", "sel_hidden_proj")})
        h = ctypes.c_void_p()
        st = self.lib.dflash_create(ctypes.byref(self._c), ctypes.byref(self._w), device, ctypes.byref(h))
        if st != _ffi.OK:
            raise DFlashError(st, "dflash_create failed")
        self.h = h
        self.device = device

    # -- helpers
    def _check(self, st):
        if st != _ffi.OK:
            raise DFlashError(st, self.lib.dflash_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.lib.dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- calls
    def inject(self, req_ids, n_new, feats, reset=False, stream=None):
        n = len(req_ids)
        arr = (ctypes.c_void_p * len(feats))(*[f.data_ptr() for f in feats]) if feats else None
        st = self.lib.dflash_inject_context(self.h, _stream_ptr(stream), n, _i32_array(req_ids),
                                            _i32_array(n_new), 1 if reset else 0, arr)
        self._check(st)

    def inject_blocks(self, req_ids, n_new, block_rows, feats, stream=None):
        """Appends the first n_new[b] rows of request b's block of block_rows feature rows
        (feats[f] is [len(req_ids) * block_rows, H_t]) without gathering them first."""
        arr = (ctypes.c_void_p * len(feats))(*[f.data_ptr() for f in feats])
        st = self.lib.dflash_inject_blocks(self.h, _stream_ptr(stream), len(req_ids), _i32_array(req_ids),
                                           _i32_array(n_new), int(block_rows), arr)
        self._check(st)

    def draft(self, req_ids, anchors, argmax=None, topk_idx=None, topk_val=None, logits=None,
              want_topk=True, want_logits=False, stream=None, lse=None, want_lse=False, selected=None,
              want_selected=False, sel_uniform=None, sel_temperature=1.0):
        """One draft step. With sel_uniform [B, K] the path selector samples (its draft
        distributions come back as sel_q_tok / sel_q_p [B, K, 32] and sel_q_n [B, K])."""
        B, K, k, V = len(req_ids), self.cfg.block_k, self.cfg.topk, self.cfg.vocab
        dev = anchors.device
        if argmax is None:
            argmax = torch.empty((B, K), dtype=torch.int32, device=dev)
        if want_topk and topk_idx is None:
            topk_idx = torch.empty((B, K, k), dtype=torch.int32, device=dev)
            topk_val = torch.empty((B, K, k), dtype=torch.float32, device=dev)
        if want_logits and logits is None:
            logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
        if want_lse and lse is None:
            lse = torch.empty((B, K), dtype=torch.float32, device=dev)
        if (want_selected or sel_uniform is not None) and selected is None:
            selected = torch.empty((B, K), dtype=torch.int32, device=dev)
        q = {}
        if sel_uniform is not None:
            q = dict(sel_q_tok=torch.empty((B, K, 32), dtype=torch.int32, device=dev),
                     sel_q_p=torch.empty((B, K, 32), dtype=torch.float32, device=dev),
                     sel_q_n=torch.empty((B, K), dtype=torch.int32, device=dev))
        if selected is not None:
            out = _ffi.DraftOut(argmax=argmax.data_ptr(), topk_idx=_ptr(topk_idx), topk_val=_ptr(topk_val),
                                logits=_ptr(logits), lse=_ptr(lse), selected=selected.data_ptr(),
                                sel_temperature=float(sel_temperature), sel_uniform=_ptr(sel_uniform),
                                **{k: v.data_ptr() for k, v in q.items()})
            st = self.lib.dflash_draft_step_ex(self.h, _stream_ptr(stream), B, _i32_array(req_ids), _ptr(anchors),
                                               ctypes.byref(out))
        elif lse is not None:
            st = self.lib.dflash_draft_step_lse(self.h, _stream_ptr(stream), B, _i32_array(req_ids),
                                                _ptr(anchors), _ptr(argmax), _ptr(topk_idx),
                                                _ptr(topk_val), _ptr(logits), _ptr(lse))
        else:
            st = self.lib.dflash_draft_step(self.h, _stream_ptr(stream), B, _i32_array(req_ids),
                                            _ptr(anchors), _ptr(argmax), _ptr(topk_idx),
                                            _ptr(topk_val), _ptr(logits))
        self._check(st)
        return dict(argmax=argmax, topk_idx=topk_idx, topk_val=topk_val, logits=logits, lse=lse, selected=selected,
                    **q)

    def verify(self, draft, target, accept_len=None, out_tokens=None, next_anchor=None, stream=None):
        B, K = draft.shape
        dev = draft.device
        if accept_len is None:
            accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
            out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
            next_anchor = torch.empty((B,), dtype=torch.int32, device=dev)
        st = self.lib.dflash_verify_greedy(self.h, _stream_ptr(stream), B, _ptr(draft), _ptr(target),
                                           _ptr(accept_len), _ptr(out_tokens), _ptr(next_anchor))
        self._check(st)
        return accept_len, out_tokens, next_anchor

    def sample_tokens(self, logits, u, temperature, top_k, top_p, tokens=None, stream=None):
        """One draw per row of fp32 logits [rows, V] from the truncated distribution."""
        rows = logits.shape[0]
        if tokens is None:
            tokens = torch.empty((rows,), dtype=torch.int32, device=logits.device)
        sp = _ffi.Sampling(float(temperature), int(top_k), float(top_p))
        st = self.lib.dflash_sample_tokens(self.h, _stream_ptr(stream), rows, ctypes.byref(sp),
                                           _ptr(logits), _ptr(u), _ptr(tokens))
        self._check(st)
        return tokens

    def verify_sample(self, target_logits, draft_logits, draft, u_accept, u_resample, temperature,
                      top_k, top_p, accept_len=None, out_tokens=None, next_anchor=None, stream=None):
        """Rejection-sampling verification; returns (accept_len, out_tokens, next_anchor)."""
        B, K = draft.shape
        dev = draft.device
        if accept_len is None:
            accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
            out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
            next_anchor = torch.empty((B,), dtype=torch.int32, device=dev)
        sp = _ffi.Sampling(float(temperature), int(top_k), float(top_p))
        st = self.lib.dflash_verify_sample(self.h, _stream_ptr(stream), B, ctypes.byref(sp),
                                           _ptr(target_logits), _ptr(draft_logits), _ptr(draft),
                                           _ptr(u_accept), _ptr(u_resample), _ptr(accept_len),
                                           _ptr(out_tokens), _ptr(next_anchor))
        self._check(st)
        return accept_len, out_tokens, next_anchor

    def verify_sample_q(self, target_logits, q_tok, q_p, q_n, draft, u_accept, u_resample, temperature, top_k,
                        top_p, stream=None):
        """Rejection sampling against draft distributions given as candidate lists
        (dflash_verify_sample_q); returns (accept_len, out_tokens, next_anchor)."""
        B, K = draft.shape
        dev = draft.device
        accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        next_anchor = torch.empty((B,), dtype=torch.int32, device=dev)
        sp = _ffi.Sampling(float(temperature), int(top_k), float(top_p))
        st = self.lib.dflash_verify_sample_q(self.h, _stream_ptr(stream), B, ctypes.byref(sp), _ptr(target_logits),
                                             _ptr(q_tok), _ptr(q_p), _ptr(q_n), _ptr(draft), _ptr(u_accept),
                                             _ptr(u_resample), _ptr(accept_len), _ptr(out_tokens),
                                             _ptr(next_anchor))
        self._check(st)
        return accept_len, out_tokens, next_anchor

    def release(self, req_id):
        self._check(self.lib.dflash_release(self.h, int(req_id)))

    def truncate(self, req_id, new_len):
        self._check(self.lib.dflash_truncate(self.h, int(req_id), int(new_len)))

    def context_len(self, req_id):
        v = ctypes.c_int32()
        self._check(self.lib.dflash_context_len(self.h, int(req_id), ctypes.byref(v)))
        return v.value

    def export_kv(self, req_id, layer, pos0, n, stream=None):
        dt = torch.bfloat16 if self.cfg.dtype == "bf16" else torch.float32
        shape = (n, self.cfg.n_kv_heads, self.cfg.head_dim)
        k = torch.empty(shape, dtype=dt, device=f"cuda:{self.device}")
        v = torch.empty(shape, dtype=dt, device=f"cuda:{self.device}")
        self._check(self.lib.dflash_export_kv(self.h, _stream_ptr(stream), int(req_id), int(layer),
                                              int(pos0), int(n), _ptr(k), _ptr(v)))
        return k, v

    def free_pages(self):
        return self.lib.dflash_free_pages(self.h)

    def launch_count(self):
        return self.lib.dflash_launch_count(self.h)

    def timing_enable(self, on=True):
        self._check(self.lib.dflash_timing_enable(self.h, 1 if on else 0))

    def timing_read(self):
        """{class: dict(ms, launches, bytes, flops)} accumulated since the last read."""
        n = self.lib.dflash_timing_classes()
        ms = (ctypes.c_double * n)()
        la = (ctypes.c_int64 * n)()
        by = (ctypes.c_double * n)()
        fl = (ctypes.c_double * n)()
        self._check(self.lib.dflash_timing_read(self.h, ms, la, by, fl, n))
        out = {}
        for i in range(n):
            if la[i]:
                out[self.lib.dflash_timing_class_name(i).decode()] = dict(
                    ms=ms[i], launches=la[i], bytes=by[i], flops=fl[i])
        return out


# ----------------------------------------------------------------- C-named functions
def dflash_create(cfg, weights, limits: Limits, device=0):
    return Context(cfg, weights, limits, device)


def dflash_destroy(ctx: Context):
    ctx.close()


def dflash_inject_context(ctx: Context, req_ids, n_new, feats, reset=False, stream=None):
    ctx.inject(req_ids, n_new, feats, reset=reset, stream=stream)


def dflash_inject_blocks(ctx: Context, req_ids, n_new, block_rows, feats, stream=None):
    ctx.inject_blocks(req_ids, n_new, block_rows, feats, stream=stream)


def dflash_draft_step(ctx: Context, req_ids, anchors, argmax, topk_idx=None, topk_val=None,
                      logits=None, stream=None):
    return ctx.draft(req_ids, anchors, argmax=argmax, topk_idx=topk_idx, topk_val=topk_val,
                     logits=logits, want_topk=topk_idx is not None, stream=stream)


def dflash_verify_greedy(ctx: Context, draft, target, accept_len, out_tokens, next_anchor, stream=None):
    return ctx.verify(draft, target, accept_len, out_tokens, next_anchor, stream=stream)


def dflash_sample_tokens(ctx: Context, logits, u, temperature, top_k, top_p, tokens=None, stream=None):
    return ctx.sample_tokens(logits, u, temperature, top_k, top_p, tokens, stream=stream)


def dflash_verify_sample(ctx: Context, target_logits, draft_logits, draft, u_accept, u_resample,
                         temperature, top_k, top_p, accept_len=None, out_tokens=None,
                         next_anchor=None, stream=None):
    return ctx.verify_sample(target_logits, draft_logits, draft, u_accept, u_resample, temperature,
                             top_k, top_p, accept_len, out_tokens, next_anchor, stream=stream)


def ddtree_build(cand_tok, cand_logp, budget, with_mask=True, stream=None, lse=None):
    """Best-first draft trees (dflash_ddtree_build) from candidates [n, L, kc] (int32 tokens,
    fp32 values, best first): log-probabilities, or logits when lse [n, L] (the rows'
    normalisers, subtracted in the kernel) is given. Returns a dict of device tensors."""
    lib = library()
    n, L, kc = cand_tok.shape
    dev = cand_tok.device
    out = dict(tok=torch.empty((n, budget), dtype=torch.int32, device=dev),
               parent=torch.empty((n, budget), dtype=torch.int32, device=dev),
               depth=torch.empty((n, budget), dtype=torch.int32, device=dev),
               logp=torch.empty((n, budget), dtype=torch.float32, device=dev),
               n_nodes=torch.empty((n,), dtype=torch.int32, device=dev))
    words = (budget + 1 + 31) // 32
    out["mask"] = (torch.empty((n, budget + 1, words), dtype=torch.int32, device=dev) if with_mask else None)
    st = lib.dflash_ddtree_build(_stream_ptr(stream), n, L, kc, budget, _ptr(cand_tok), _ptr(cand_logp),
                                 _ptr(lse), _ptr(out["tok"]), _ptr(out["parent"]), _ptr(out["depth"]), _ptr(out["logp"]),
                                 _ptr(out["n_nodes"]), _ptr(out["mask"]))
    if st != _ffi.OK:
        raise DFlashError(st, "dflash_ddtree_build failed")
    return out


def select_path(anchors, cand_tok, unary, gate, pred_codebook, succ_codebook, want_scores=False, stream=None):
    """The DFlash 2 path selector's walk on its own (dflash_select_path): anchors [n],
    cand_tok / unary [n, K, kc], gate [n, K, r] fp32, codebooks [V, r] (bf16 or fp32).
    Returns (selected [n, K], scores [n, K, kc] or None)."""
    lib = library()
    n, K, kc = cand_tok.shape
    V, r = pred_codebook.shape
    dev = cand_tok.device
    dt = _ffi.BF16 if pred_codebook.dtype == torch.bfloat16 else _ffi.F32
    sel = torch.empty((n, K), dtype=torch.int32, device=dev)
    sc = torch.empty((n, K, kc), dtype=torch.float32, device=dev) if want_scores else None
    st = lib.dflash_select_path(_stream_ptr(stream), n, K, kc, r, V, dt, _ptr(anchors), _ptr(cand_tok), _ptr(unary),
                                _ptr(gate), _ptr(pred_codebook), _ptr(succ_codebook), _ptr(sel), _ptr(sc))
    if st != _ffi.OK:
        raise DFlashError(st, "dflash_select_path failed")
    return sel, sc


def select_sample(anchors, cand_tok, unary, gate, pred_codebook, succ_codebook, temperature, u, stream=None):
    """The path selector's sampling walk on its own (dflash_select_sample). Returns
    (selected [n, K], q_tok [n, K, 32], q_p [n, K, 32], q_n [n, K])."""
    lib = library()
    n, K, kc = cand_tok.shape
    V, r = pred_codebook.shape
    dev = cand_tok.device
    dt = _ffi.BF16 if pred_codebook.dtype == torch.bfloat16 else _ffi.F32
    sel = torch.empty((n, K), dtype=torch.int32, device=dev)
    q_tok = torch.empty((n, K, 32), dtype=torch.int32, device=dev)
    q_p = torch.empty((n, K, 32), dtype=torch.float32, device=dev)
    q_n = torch.empty((n, K), dtype=torch.int32, device=dev)
    st = lib.dflash_select_sample(_stream_ptr(stream), n, K, kc, r, V, dt, float(temperature), _ptr(anchors),
                                  _ptr(cand_tok), _ptr(unary), _ptr(gate), _ptr(pred_codebook), _ptr(succ_codebook),
                                  _ptr(u), _ptr(sel), _ptr(q_tok), _ptr(q_p), _ptr(q_n))
    if st != _ffi.OK:
        raise DFlashError(st, "dflash_select_sample failed")
    return sel, q_tok, q_p, q_n


def ddtree_walk(tree, L, target_next, stream=None):
    """Greedy verifier walk (dflash_ddtree_walk); returns (accept_len, out_tokens, next_anchor)."""
    lib = library()
    n, budget = tree["tok"].shape
    dev = tree["tok"].device
    acc = torch.empty((n,), dtype=torch.int32, device=dev)
    toks = torch.empty((n, L + 1), dtype=torch.int32, device=dev)
    nxt = torch.empty((n,), dtype=torch.int32, device=dev)
    st = lib.dflash_ddtree_walk(_stream_ptr(stream), n, L, budget, _ptr(tree["tok"]), _ptr(tree["parent"]),
                                _ptr(tree["n_nodes"]), _ptr(target_next), _ptr(acc), _ptr(toks), _ptr(nxt))
    if st != _ffi.OK:
        raise DFlashError(st, "dflash_ddtree_walk failed")
    return acc, toks, nxt


def dflash_release(ctx: Context, req_id):
    ctx.release(req_id)


def dflash_truncate(ctx: Context, req_id, new_len):
    ctx.truncate(req_id, new_len)


def dflash_context_len(ctx: Context, req_id):
    return ctx.context_len(req_id)


def dflash_export_kv(ctx: Context, req_id, layer, pos0, n, stream=None):
    return ctx.export_kv(req_id, layer, pos0, n, stream=stream)
