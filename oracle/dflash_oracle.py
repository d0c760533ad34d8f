"""Plain fp64 CPU oracle of the DFlash draft step (test infrastructure only).

This module is the checker the CUDA library is compared against. Only the tests,
`__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import it. It
shares no code, table or helper with the CUDA path: numpy in float64, matrix
products through numpy's BLAS, everything else written out row by row.

Sources (cited by page title and section):
  [P1] "LLM的推理加速-DFlash" — 架构设计; 关键创新 Step 1-3 (multi-layer features,
       concat + projection, K/V injection prepended to every layer's attention);
       核心推理伪代码 (the draft/verify loop); 验证 (left-to-right acceptance).
  [P2] "DFlash 2 块扩散投机解码技术详解" — §2.1 (anchor + mask block, mask_token_id),
       §2.2 (shared embedding x input_embedding_scale; fc + RMSNorm fusion; shared LM
       head), §2.3 (rejection sampling; greedy prefix formula), §4.2 (fallback to p).
  [P3] "DFlash：块扩散 + KV 注入，让投机解码的草稿不再串行" — §四 (immediate
       materialisation: K/V projection then norm + RoPE post-processing).
  [P4] "DFlash：把串行 Draft 变成并行“填空”" — §2 (at most K+1 tokens per round),
       §4-4.4 (context / anchor / mask roles; K+1 queries, K outputs), §5.1
       (normalise, K/V-project, RoPE, write the draft KV cache), §5.3 (non-causal
       in-block attention), §5.6 (the draft KV cache holds the injected context).

Readings where the pages leave a step open (each is also listed in the design notes):
  * g = RMSNorm(fc(concat_f h_f)) once; the per-layer input norm is not applied to g.
  * Per-head RMSNorm on q and k (learned weight over head_dim) before RoPE, switchable
    with `qk_norm`.
  * Rotate-half RoPE with inv_freq_i = theta^(-2i/head_dim); context position p is its
    index in the sequence, block row j (0 = anchor) sits at position ctx_len + j.
  * In-block attention is bidirectional (no mask); every block query sees the whole
    injected context.
  * Block K/V are never written to the cache; after a verify the caller injects the
    anchor plus the accepted drafts (a + 1 positions).
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * w.
  * Variants (off by default): a causal mask inside the block (block row j sees block keys
    0..j), a trained mask embedding replacing E[mask_id] for the mask rows, and the logits
    scaled by output_multiplier then soft-capped as c * tanh(logits / c).
  * Precision: the stored operands of the method — weights, the target hidden states
    and the context K/V cache — have the storage type (bf16 or fp32); the cache is
    rounded to it (round-to-nearest-even) when written. Every other value (the fused
    feature g, the residual stream, normed activations, q/k/v, attention, SwiGLU, the
    final hidden rows, logits) is an activation carried at full precision: fp64 here,
    fp32 (or an exact bf16 hi+lo pair as a tensor-core operand) on the GPU. Argmax and
    top-k are decided on the logits rounded to fp32, ties to the lowest index.
  * top-k: k values sorted descending, indices tie-broken by lowest index.
  * DFlash 2 local convolution ([P2] §3.2.3), off by default: four two-tap dynamic depthwise
    convolutions per layer — on the attention input (after the input norm), on the attention
    output (after the output projection, before the residual add), on the MLP input (after
    the post-attention norm) and on the MLP output (before the residual add). Over the K+1
    block rows of one request, y_t = k_t0 * x_t + k_t1 * x_{t-1} with x_{-1} = 0; the taps
    are k_ti[c] = base[i][c] + (P x_t)[i*G + c // 16], P [2G, H], G = H / 16 (the correction
    is computed from the convolution's own input row and shared by 16 channels).
  * DFlash 2 path selector ([P2] §3.1), off by default: over each mask position's top-k
    candidates, S_t(a, b) = U_t(b) + <A(a) * g_t, B(b)>, U_t = the draft's logits, A / B the
    predecessor / successor codebooks [V, r], g_t = W_h h_t with h_t the final-normed hidden
    row of mask position t; a greedy walk from the anchor takes the best-scoring candidate
    at each position (the first in candidate order among equal scores). In sampling mode the
    walk draws position t's token from softmax(S_t(a, .) / temperature) over the k
    candidates (inverse CDF in vocabulary order, a caller-supplied uniform); that subset
    distribution, as a distribution over the vocabulary (zero outside the candidates), is
    the draft's q in rejection sampling.
  * Sampling mode ([P2] §2.3, §3.3, §4.2): both the draft and the target distribution go
    through the same truncation — logits / temperature, keep the top_k largest (ties to
    the lower index), softmax over those, then keep the shortest prefix of them in
    descending order whose mass reaches top_p, renormalised. Draws are inverse-CDF over
    the vocabulary in index order with caller-supplied uniforms; the drafted tokens are
    inputs (drawn from q by the caller).

Parity status: every function here is pinned by the CPU tests (brute force, closed
forms, library routines or exact rational arithmetic) — see tests/test_oracle_pins.py.
"""
from fractions import Fraction

import numpy as np

__all__ = [
    "round_to", "bf16_round", "f32_round", "rmsnorm", "rope", "silu", "softmax",
    "OracleDraft", "topk_desc", "argmax_lowest", "verify_greedy",
    "accept_prob", "residual_dist", "sample_index", "verify_sample", "as_fraction_dist",
    "sampling_probs", "sample_token", "verify_sample_logits",
    "log_softmax_norm", "ddtree_build", "ddtree_mask", "ddtree_walk",
    "dyn_conv", "select_path", "select_sample", "subset_to_vocab",
]


# ----------------------------------------------------------------------------- rounding
def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value (ties to even), as float64.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the float32 exponent
    range; below 2^-126 the spacing stays 2^-133 (gradual underflow). Written from that
    definition: scale the significand to 8 bits, round half to even, scale back.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e = np.frexp(xf)                 # xf = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)             # bf16 min normal is 2^-126 = 0.5 * 2^-125
    scale = np.ldexp(1.0, 8 - e)        # 8 significant bits
    r = np.rint(xf * scale) / scale     # np.rint rounds half to even
    bf16_max = 3.3895313892515355e38    # (2 - 2^-7) * 2^127
    out[finite] = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    return out


def f32_round(x):
    """Round float64 values to the nearest float32 value (IEEE, ties to even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(dtype):
    """Rounding to the storage type (applied where the KV cache is written)."""
    if dtype == "bf16":
        return bf16_round
    if dtype == "f32":
        return f32_round
    if dtype == "f64":          # no rounding at all (used by the oracle's own pins)
        return lambda x: np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------- elementwise
def rmsnorm(x, w, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope(x, pos, theta):
    """Rotate-half rotary embedding of x [..., n, head_dim] at integer positions pos [n].

    For i < head_dim/2 the pair (x_i, x_{i+head_dim/2}) is rotated by the angle
    pos * theta^(-2i/head_dim).
    """
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [n, half]
    c, s = np.cos(ang), np.sin(ang)
    # broadcast [n, half] against x [n, heads, half] when x has a head axis
    while c.ndim < x.ndim:
        c, s = c[:, None, :], s[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def softmax(s, axis=-1):
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


# ----------------------------------------------------------------------------- the draft
def _f64(a):
    return np.asarray(a, dtype=np.float64)


class OracleDraft:
    """The DFlash draft model and its per-request context cache, in float64.

    `cfg` needs the attributes hidden, n_layers, n_q_heads, n_kv_heads, head_dim,
    intermediate, vocab, n_feat, target_hidden, block_k, topk, mask_id, qk_norm,
    rms_eps, rope_theta, input_embedding_scale, dtype. `weights` holds float arrays
    (float32 or float64) in [out, in] layout: embed, lm_head, fc, fc_norm, final_norm
    and layers = [dict(in_norm, wq, wk, wv, q_norm, k_norm, wo, post_norm, w_gate, w_up,
    w_down)]. The cache maps a request id to per-layer lists of context K and V rows.
    """

    def __init__(self, cfg, weights):
        self.cfg = cfg
        self.w = weights
        self.r = round_to(cfg.dtype)   # storage rounding of the KV cache
        self.cache = {}   # req -> {"K": [L arrays [n, nkv, hd]], "V": [...]}

    # -- context fusion and injection ([P1] Step 2-3, [P2] §2.2, [P3] §四, [P4] §5.1)
    def fuse(self, feats):
        """g = RMSNorm(concat_f(h_f) @ W_fc^T) for rows of n_feat hidden-state arrays."""
        c = self.cfg
        cat = np.concatenate([_f64(f) for f in feats], axis=1)           # [n, n_feat*H_t]
        fc_out = cat @ _f64(self.w["fc"]).T                             # [n, H]
        return rmsnorm(fc_out, self.w["fc_norm"], c.rms_eps)

    def project_kv(self, g, pos, layer):
        """Context K/V of one draft layer for fused rows g at positions pos."""
        c, r, lw = self.cfg, self.r, self.w["layers"][layer]
        n = g.shape[0]
        k = (g @ _f64(lw["wk"]).T).reshape(n, c.n_kv_heads, c.head_dim)
        v = (g @ _f64(lw["wv"]).T).reshape(n, c.n_kv_heads, c.head_dim)
        if c.qk_norm:
            k = rmsnorm(k, lw["k_norm"], c.rms_eps)
        # the cache stores K and V in the storage type
        return r(rope(k, pos, c.rope_theta)), r(v)

    def inject(self, req, feats, reset=False):
        """Append the K/V of newly accepted positions (rows of feats) to req's cache."""
        c = self.cfg
        if reset or req not in self.cache:
            self.cache[req] = {"K": [np.zeros((0, c.n_kv_heads, c.head_dim))] * c.n_layers,
                               "V": [np.zeros((0, c.n_kv_heads, c.head_dim))] * c.n_layers}
        ent = self.cache[req]
        n = feats[0].shape[0]
        if n == 0:
            return
        start = ent["K"][0].shape[0]
        pos = np.arange(start, start + n)
        g = self.fuse(feats)
        for l in range(c.n_layers):
            k, v = self.project_kv(g, pos, l)
            ent["K"][l] = np.concatenate([ent["K"][l], k], axis=0)
            ent["V"][l] = np.concatenate([ent["V"][l], v], axis=0)

    def context_len(self, req):
        return self.cache[req]["K"][0].shape[0]

    def truncate(self, req, n):
        ent = self.cache[req]
        ent["K"] = [k[:n] for k in ent["K"]]
        ent["V"] = [v[:n] for v in ent["V"]]

    # -- the query block forward ([P2] §2.1-2.2, [P4] §4-4.4 and §5.3, [P1] Step 3)
    def block_tokens(self, anchor):
        """[anchor, mask x K] — the anchor is the last verified token."""
        return [int(anchor)] + [self.cfg.mask_id] * self.cfg.block_k

    def layer(self, x, l, ctx_k, ctx_v, pos):
        """One pre-norm decoder layer over the block rows x [K+1, H]."""
        c, lw = self.cfg, self.w["layers"][l]
        nq, nkv, hd = c.n_q_heads, c.n_kv_heads, c.head_dim
        q_rows = x.shape[0]
        conv = getattr(c, "dyn_conv", 0)
        xn = rmsnorm(x, lw["in_norm"], c.rms_eps)
        if conv:
            xn = dyn_conv(xn, lw["conv_base"][0], lw["conv_proj"][0])
        q = (xn @ _f64(lw["wq"]).T).reshape(q_rows, nq, hd)
        k = (xn @ _f64(lw["wk"]).T).reshape(q_rows, nkv, hd)
        v = (xn @ _f64(lw["wv"]).T).reshape(q_rows, nkv, hd)
        if c.qk_norm:
            q = rmsnorm(q, lw["q_norm"], c.rms_eps)
            k = rmsnorm(k, lw["k_norm"], c.rms_eps)
        q = rope(q, pos, c.rope_theta)
        k = rope(k, pos, c.rope_theta)
        # context K/V first, then the block's own K/V; no mask inside the block by default
        # ([P4] §5.3); the causal variant ([P2] 1.x, "块内保持因果掩码") lets block row j see
        # block keys 0..j only
        keys = np.concatenate([ctx_k, k], axis=0)         # [n_ctx + K + 1, nkv, hd]
        vals = np.concatenate([ctx_v, v], axis=0)
        n_ctx = ctx_k.shape[0]
        group = nq // nkv
        o = np.empty((q_rows, nq, hd))
        for h in range(nq):
            kvh = h // group
            s = (q[:, h, :] @ keys[:, kvh, :].T) / np.sqrt(hd)   # [K+1, n_keys]
            if getattr(c, "block_causal", 0):
                for j in range(q_rows):
                    s[j, n_ctx + j + 1:] = -np.inf
            o[:, h, :] = softmax(s, axis=-1) @ vals[:, kvh, :]
        o = o.reshape(q_rows, nq * hd)
        attn_out = o @ _f64(lw["wo"]).T
        if conv:
            attn_out = dyn_conv(attn_out, lw["conv_base"][1], lw["conv_proj"][1])
        x = x + attn_out
        xn2 = rmsnorm(x, lw["post_norm"], c.rms_eps)
        if conv:
            xn2 = dyn_conv(xn2, lw["conv_base"][2], lw["conv_proj"][2])
        hmid = silu(xn2 @ _f64(lw["w_gate"]).T) * (xn2 @ _f64(lw["w_up"]).T)
        mlp_out = hmid @ _f64(lw["w_down"]).T
        if conv:
            mlp_out = dyn_conv(mlp_out, lw["conv_base"][3], lw["conv_proj"][3])
        return x + mlp_out

    def hidden(self, req, anchor):
        """Final-normed hidden rows of the K mask positions, [K, H]."""
        c = self.cfg
        ent = self.cache[req]
        n_ctx = ent["K"][0].shape[0]
        toks = self.block_tokens(anchor)
        emb = _f64(self.w["embed"][toks])
        if getattr(c, "mask_embedding", 0):
            # a trained mask embedding replaces the word embedding of the mask rows ([P4] §5.2)
            emb[1:] = _f64(self.w["mask_embedding"])
        x = emb * c.input_embedding_scale
        pos = np.arange(n_ctx, n_ctx + c.block_k + 1)
        for l in range(c.n_layers):
            x = self.layer(x, l, ent["K"][l], ent["V"][l], pos)
        # the anchor row yields no candidate ([P4] §4.3): only the K mask rows go on
        return rmsnorm(x[1:], self.w["final_norm"], c.rms_eps)

    def logits(self, req, anchor, chunk=16384):
        """fp64 logits [K, V] of the K mask positions (LM head in vocabulary chunks)."""
        h = self.hidden(req, anchor)
        lm = self.w["lm_head"]
        V = lm.shape[0]
        out = np.empty((h.shape[0], V))
        for v0 in range(0, V, chunk):
            out[:, v0:v0 + chunk] = h @ _f64(lm[v0:v0 + chunk]).T
        # optional output scale and soft cap ([P2] 1.x compute_logits): c * tanh(x / c)
        out = out * getattr(self.cfg, "output_multiplier", 1.0)
        cap = getattr(self.cfg, "logit_softcap", 0.0)
        if cap > 0:
            out = cap * np.tanh(out / cap)
        return out

    def draft(self, req, anchor):
        """(argmax [K], topk_idx [K, k], topk_val [K, k], logits [K, V]) for one request."""
        lg = self.logits(req, anchor)
        lg32 = f32_round(lg)
        idx, val = topk_desc(lg32, self.cfg.topk)
        return argmax_lowest(lg32), idx, val, lg

    def select(self, req, anchor, cand_tok=None, unary=None):
        """The path selector's walk ([P2] §3.1) for one request: (tokens [K], scores [K, k]).
        Candidates and their unary scores default to this oracle's own top-k of the logits;
        g_t comes from this oracle's final-normed hidden rows."""
        if cand_tok is None:
            _, cand_tok, unary, _ = self.draft(req, anchor)
        gate = self.hidden(req, anchor) @ _f64(self.w["sel_hidden_proj"]).T      # [K, r]
        return select_path(anchor, cand_tok, unary, gate, self.w["sel_pred_codebook"],
                           self.w["sel_succ_codebook"])


# ----------------------------------------------------------------------------- selection
def argmax_lowest(x):
    """Row-wise argmax; among equal maxima the lowest index wins."""
    x = np.asarray(x)
    return np.argmax(x, axis=-1)   # numpy returns the first occurrence


def topk_desc(x, k):
    """Row-wise top-k: values descending, equal values ordered by lowest index."""
    x = np.asarray(x, dtype=np.float64)
    # stable sort on (-value) keeps lower indices first among equal values
    order = np.argsort(-x, axis=-1, kind="stable")[..., :k]
    return order, np.take_along_axis(x, order, axis=-1)


# ----------------------------------------------------------------------------- verification
def verify_greedy(draft, target):
    """Greedy verification of one block per request ([P2] §2.3, [P1] 核心推理伪代码).

    draft [B, K]: the draft's tokens for the K mask positions. target [B, K+1]: the
    target's greedy token after the anchor and after each draft token. The accepted
    count a is the number of leading positions with draft == target; the round emits
    draft[:a] followed by target[a] (a correction, or the bonus when a == K), so at most
    K+1 tokens ([P4] §2). Returns (accept_len [B], out_tokens [B, K+1] padded with -1,
    next_anchor [B]).
    """
    draft = np.asarray(draft)
    target = np.asarray(target)
    B, K = draft.shape
    acc = np.zeros(B, dtype=np.int32)
    out = np.full((B, K + 1), -1, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int32)
    for b in range(B):
        a = 0
        while a < K and draft[b, a] == target[b, a]:
            a += 1
        acc[b] = a
        out[b, :a] = draft[b, :a]
        out[b, a] = target[b, a]
        nxt[b] = target[b, a]
    return acc, out, nxt


def accept_prob(p, q, d):
    """Probability of accepting draft token d: min(1, p[d] / q[d]) ([P2] §2.3)."""
    return min(1, p[d] / q[d])


def residual_dist(p, q):
    """norm(max(p - q, 0)); falls back to p when nothing is left ([P2] §2.3, §4.2).

    Works on any number type (floats or fractions.Fraction) given as sequences.
    """
    res = [max(pi - qi, 0) for pi, qi in zip(p, q)]
    total = sum(res)
    if total <= 0:
        return list(p)
    return [x / total for x in res]


def sample_index(dist, u):
    """Inverse-CDF draw: smallest i with cumsum(dist)[:i+1] > u * sum(dist)."""
    total = sum(dist)
    acc = 0
    for i, pi in enumerate(dist):
        acc += pi
        if acc > u * total:
            return i
    return len(dist) - 1


def verify_sample(p_rows, q_rows, draft, u_accept, u_resample):
    """Rejection-sampling verification of one block ([P2] §2.3, §4.2).

    p_rows [K+1][V]: the target's distribution at each block position given the anchor
    and the drafts before it; q_rows [K][V]: the draft's distribution per mask position;
    draft [K]: the drafted tokens; u_accept [K], u_resample: uniforms in [0, 1).
    Position j accepts draft[j] when u_accept[j] < min(1, p/q). On the first rejection
    the token is drawn from the residual norm(max(p_j - q_j, 0)) (p_j when that vanishes)
    and the round ends; when all K are accepted a bonus is drawn from p_K.
    Returns (accepted count a, emitted tokens, a + 1 of them).
    """
    K = len(draft)
    out = []
    for j in range(K):
        d = int(draft[j])
        if u_accept[j] < accept_prob(p_rows[j], q_rows[j], d):
            out.append(d)
            continue
        out.append(sample_index(residual_dist(p_rows[j], q_rows[j]), u_resample))
        return j, out
    out.append(sample_index(list(p_rows[K]), u_resample))
    return K, out


def as_fraction_dist(values):
    """Helper for exact tests: normalise a sequence of positive ints to Fractions."""
    total = sum(values)
    return [Fraction(v, total) for v in values]


# ----------------------------------------------------------------------------- sampling mode
def sampling_probs(logits, temperature, top_k, top_p):
    """Truncated sampling distribution of one row of logits ([P2] §3.3: the same top-k /
    top-p truncation applied to the draft and the target).

    temperature > 0; top_k in [1, V] (V keeps every token); 0 < top_p <= 1. Returns a
    length-V float64 vector: zero outside the kept set, summing to one.
    """
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    V = z.shape[0]
    k = min(int(top_k), V)
    # descending by value, ties to the lower index (a stable sort of -z)
    order = np.argsort(-z, kind="stable")
    kept = order[:k]
    e = np.exp(z[kept] - z[kept[0]])
    p = e / e.sum()
    if top_p < 1.0:
        mass = 0.0
        n = 0
        for n in range(1, k + 1):
            mass += p[n - 1]
            if mass >= top_p:
                break
        kept = kept[:n]
        p = p[:n] / p[:n].sum()
    out = np.zeros(V, dtype=np.float64)
    out[kept] = p
    return out


def sample_token(logits, u, temperature, top_k, top_p):
    """One draw from sampling_probs(...) with the uniform u (inverse CDF, index order)."""
    return sample_index(list(sampling_probs(logits, temperature, top_k, top_p)), u)


def verify_sample_logits(target_logits, draft_logits, draft, u_accept, u_resample,
                         temperature, top_k, top_p):
    """verify_sample on the truncated distributions of the target's K+1 rows and the
    draft's K rows (sampling mode of [P2] §2.3)."""
    p_rows = [sampling_probs(r, temperature, top_k, top_p) for r in target_logits]
    q_rows = [sampling_probs(r, temperature, top_k, top_p) for r in draft_logits]
    return verify_sample(p_rows, q_rows, draft, u_accept, u_resample)


# ----------------------------------------------------------------------------- DDTree
def log_softmax_norm(logits):
    """log sum_v exp(logits[v]) per row (the normaliser of the draft's softmax)."""
    x = np.asarray(logits, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True)))[..., 0]


def ddtree_build(cand_logp, cand_tok, budget):
    """Best-first draft tree ("DDTree" §2.3, Algorithm 1, and Proposition 2).

    cand_logp [L][kc]: log-probabilities of each block position's candidates, best first;
    cand_tok [L][kc]: their tokens. A prefix is a rank tuple (r_1 .. r_d) (r_i = which
    candidate position i takes); its log-probability is the sum of its entries. The heap
    starts with (best of position 1); each pop adds the prefix as a node and pushes its next
    sibling (last rank + 1) and its first child (a best candidate at the next position).
    Ties pop by (log-probability desc, depth asc, parent node asc, last rank asc).
    Returns the popped nodes in order as (token, parent node or -1 for the root, depth,
    log-probability): at most `budget` of them, prefix-closed.
    """
    import heapq
    L, kc = len(cand_logp), len(cand_logp[0])
    nodes = []
    heap = [(-float(cand_logp[0][0]), 1, -1, 0)]     # (-logp, depth, parent, rank)
    while heap and len(nodes) < budget:
        nlp, depth, parent, rank = heapq.heappop(heap)
        lp = -nlp
        me = len(nodes)
        nodes.append((int(cand_tok[depth - 1][rank]), parent, depth, lp))
        base = 0.0 if parent < 0 else nodes[parent][3]
        if rank + 1 < kc:
            heapq.heappush(heap, (-(base + float(cand_logp[depth - 1][rank + 1])), depth, parent, rank + 1))
        if depth < L:
            heapq.heappush(heap, (-(lp + float(cand_logp[depth][0])), depth + 1, me, 0))
    return nodes


def ddtree_mask(nodes):
    """Ancestor-only visibility ("DDTree" §3.3): index 0 is the root (the anchor / bonus
    token), node i is index i + 1; each index sees the root, its ancestors and itself."""
    n = len(nodes) + 1
    m = np.zeros((n, n), dtype=bool)
    m[:, 0] = True
    for i in range(1, n):
        j = i
        while j > 0:
            m[i, j] = True
            j = nodes[j - 1][1] + 1
    return m


def ddtree_walk(nodes, target_next):
    """Greedy verifier walk over the tree ("DDTree" §3.5): target_next[0] is the target's
    token after the root, target_next[i + 1] after node i. From the root, move to the child
    whose token equals the target's next token while one exists; emit the matched tokens and
    then the target's token where the walk stopped. Returns (accepted, emitted tokens)."""
    cur = -1
    out = []
    while True:
        t = int(target_next[cur + 1])
        child = [i for i, nd in enumerate(nodes) if nd[1] == cur and nd[0] == t]
        if not child:
            out.append(t)
            return len(out) - 1, out
        out.append(t)
        cur = child[0]


# ----------------------------------------------------------------------------- DFlash 2 modules
def dyn_conv(x, base, proj, group=16):
    """Two-tap dynamic depthwise convolution over the rows of one block ([P2] §3.2.3):
    y_t = k_t0 * x_t + k_t1 * x_{t-1}, the row before the first being zero. The taps are a
    learned base per channel plus a correction computed from the input row by the linear
    map `proj` [2G, H] (rows 0..G-1 tap 0, rows G..2G-1 tap 1), one value per group of
    `group` channels: k_ti[c] = base[i][c] + (proj @ x_t)[i*G + c // group]."""
    x = _f64(x)
    base, proj = _f64(base), _f64(proj)
    T, H = x.shape
    G = H // group
    corr = x @ proj.T                                      # [T, 2G]
    y = np.empty_like(x)
    for t in range(T):
        k0 = base[0] + np.repeat(corr[t, :G], group)
        k1 = base[1] + np.repeat(corr[t, G:], group)
        prev = x[t - 1] if t > 0 else np.zeros(H)
        y[t] = k0 * x[t] + k1 * prev
    return y


def select_path(anchor, cand_tok, unary, gate, pred_cb, succ_cb):
    """Greedy walk of the path selector ([P2] §3.1) over K positions with k candidates each:
    starting from the anchor as predecessor a, position t scores its candidates b by
    S_t(a, b) = unary[t, b] + sum_r pred_cb[a, r] * gate[t, r] * succ_cb[b, r] and takes the
    best (the first in candidate order among equal scores), which becomes the next
    predecessor. Returns (tokens [K], scores [K, k])."""
    cand_tok = np.asarray(cand_tok)
    unary, gate = _f64(unary), _f64(gate)
    K, k = cand_tok.shape
    prev = int(anchor)
    toks, scores = [], np.empty((K, k))
    for t in range(K):
        a = _f64(pred_cb[prev]) * gate[t]                             # [r]
        for j in range(k):
            scores[t, j] = unary[t, j] + float(a @ _f64(succ_cb[int(cand_tok[t, j])]))
        best = int(np.argmax(scores[t]))                                # first maximum
        prev = int(cand_tok[t, best])
        toks.append(prev)
    return np.array(toks, dtype=np.int64), scores


def subset_to_vocab(tokens, probs, V):
    """A distribution over k distinct candidate tokens as a length-V vector (zero elsewhere)."""
    full = np.zeros(V)
    for t, q in zip(tokens, probs):
        full[int(t)] += float(q)
    return full


def select_sample(anchor, cand_tok, unary, gate, pred_cb, succ_cb, temperature, u, V):
    """The path selector's walk in sampling mode ([P2] §3.1.3): at position t the scores
    S_t(a, b) of select_path (a = the token drawn at t-1, the anchor at t = 0) become the
    distribution softmax(S_t / temperature) over the k candidates, and the token is drawn
    from it by inverse CDF in vocabulary order with u[t]. Returns (tokens [K], q [K][V]): the
    drawn tokens and each position's subset distribution over the vocabulary."""
    cand_tok = np.asarray(cand_tok)
    K, k = cand_tok.shape
    prev = int(anchor)
    toks, q_rows = [], []
    for t in range(K):
        _, sc = select_path(prev, cand_tok[t:t + 1], np.asarray(unary)[t:t + 1], np.asarray(gate)[t:t + 1],
                            pred_cb, succ_cb)
        q = softmax(sc[0] / temperature)
        full = subset_to_vocab(cand_tok[t], q, V)
        prev = sample_index(full, float(u[t]))
        toks.append(prev)
        q_rows.append(full)
    return np.array(toks, dtype=np.int64), q_rows
