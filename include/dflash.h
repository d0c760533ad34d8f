/*
 * dflash.h — C ABI of the DFlash batched draft step on one GB300 (sm_103a).
 *
 * The library runs the hot path of DFlash block-diffusion speculative decoding:
 *   1. KV injection: target hidden states of n_feat target layers are concatenated,
 *      projected by fc and RMSNorm into the fused feature g, then put through every
 *      draft layer's K/V projection (+ per-head k-norm) and RoPE and written to the
 *      paged draft KV cache.
 *        ("LLM的推理加速-DFlash", 关键创新 Step 1-3; "DFlash 2 块扩散投机解码技术详解" §2.2;
 *         "DFlash：块扩散 + KV 注入" §四; "DFlash：把串行 Draft 变成并行“填空”" §5.1, §5.6)
 *   2. One parallel forward of the query block [anchor, MASK x K] (embedding rows times
 *      input_embedding_scale) through the draft decoder layers, attending without a mask
 *      over the injected context K/V followed by the block's own K/V.
 *        ("DFlash 2 块扩散投机解码技术详解" §2.1-2.2; "DFlash：把串行 Draft 变成并行“填空”"
 *         §4-4.4, §5.3; "LLM的推理加速-DFlash", 关键创新 Step 3)
 *   3. The LM head with per-position argmax and top-k for the K mask rows only (the
 *      anchor row yields no candidate).
 *        ("DFlash：把串行 Draft 变成并行“填空”" §4.3; "DFlash 2 块扩散投机解码技术详解" §2.2)
 *   4. Greedy verification: the longest prefix of drafts equal to the target tokens,
 *      then one target token (correction or bonus); at most K+1 tokens per round.
 *        ("DFlash 2 块扩散投机解码技术详解" §2.3; "DFlash：把串行 Draft 变成并行“填空”" §2;
 *         "LLM的推理加速-DFlash", 核心推理伪代码)
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses on the device the context was created
 *     on; host pointers are ordinary host memory read before the call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Calls only enqueue work on it and never synchronise the device. All calls on
 *     one context must be issued in one stream order (one stream, or streams the
 *     caller orders with events); the context is not thread-safe.
 *   - Weight matrices are row-major [out_features, in_features] (the nn.Linear layout),
 *     norm weights are vectors; all have the storage type of `dtype` (fp32 or bf16).
 *     The caller owns weights and every input/output buffer and keeps the weights
 *     alive and unchanged while the context exists. The library owns the paged KV
 *     pool, its page tables, scratch and pinned staging, all allocated in
 *     dflash_create and freed in dflash_destroy.
 *   - Every call returns a dflash_status. On an error no request state changes (pages
 *     are planned on the host before anything is launched); dflash_last_error()
 *     gives the reason. Device-side checks (out-of-range token ids, exhausted waits)
 *     latch a flag that the next call reports as DFLASH_ERR_DEVICE.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1,     /* a NULL/misaligned pointer, a size out of range */
  DFLASH_ERR_OUT_OF_PAGES = -2,    /* the paged KV pool cannot hold the injection   */
  DFLASH_ERR_UNKNOWN_REQUEST = -3, /* req_id was never injected or was released     */
  DFLASH_ERR_CUDA = -4,            /* a CUDA runtime/driver call failed             */
  DFLASH_ERR_DEVICE = -5,          /* a device-side check latched an error flag     */
  DFLASH_ERR_UNSUPPORTED = -6      /* a shape the kernels do not handle             */
} dflash_status;

typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 } dflash_dtype;

/* Draft-model shape and context limits. Requirements (checked by dflash_validate_config):
 * hidden (<= 8192), intermediate, n_q_heads*head_dim and n_kv_heads*head_dim multiples of 128;
 * target_hidden a multiple of 64; head_dim 64 or 128; n_q_heads a multiple of
 * n_kv_heads with n_q_heads/n_kv_heads <= 8; 1 <= block_k <= 31; 1 <= topk <= 32;
 * page_size == 64; vocab >= topk; mask_token_id in [0, vocab). */
typedef struct {
  int32_t hidden;            /* H: draft hidden size                                   */
  int32_t n_layers;          /* L: draft decoder layers                                */
  int32_t n_q_heads;         /* nq                                                     */
  int32_t n_kv_heads;        /* nkv (GQA: q head h reads kv head h / (nq/nkv))         */
  int32_t head_dim;          /* hd                                                     */
  int32_t intermediate;      /* I: SwiGLU width                                        */
  int32_t vocab;             /* V                                                      */
  int32_t n_feat;            /* number of target layers whose hidden states are fused  */
  int32_t target_hidden;     /* H_t: width of each target hidden state                 */
  int32_t block_k;           /* K mask positions; the query block has K+1 rows         */
  int32_t topk;              /* k of the per-position top-k                            */
  int32_t mask_token_id;     /* embedding row used for every mask position             */
  int32_t qk_norm;           /* 1: per-head RMSNorm (q_norm/k_norm) before RoPE        */
  int32_t max_batch;         /* most requests in one call                              */
  int32_t max_requests;      /* most live requests                                     */
  int32_t max_pages;         /* pages in the KV pool                                   */
  int32_t page_size;         /* tokens per page; must be 64                            */
  int32_t max_positions;     /* longest context + K + 1 (RoPE table length)            */
  int32_t max_inject_rows;   /* rows per internal injection chunk (scratch sizing)     */
  float rms_eps;             /* RMSNorm epsilon                                        */
  float rope_theta;          /* RoPE base                                              */
  float input_embedding_scale; /* multiplies the block's embedding rows                */
  dflash_dtype dtype;        /* storage / GEMM operand type                            */
  /* Variants ("DFlash 2 块扩散投机解码技术详解" §1.x: the causal in-block mask and the
   * optional output_multiplier / logit soft cap of compute_logits). Zero-initialised
   * fields give the default path: bidirectional block, logits unscaled, no cap. */
  int32_t block_causal;      /* 1: block row j attends to block keys 0..j only          */
  float output_multiplier;   /* logits *= m (0 is read as 1; must be > 0 otherwise)     */
  float logit_softcap;       /* c > 0: logits = c * tanh(logits / c) after the scale    */
  /* DFlash 2 modules ("DFlash 2 块扩散投机解码技术详解" §3.1, §3.2.3); zero: off. */
  int32_t dyn_conv;          /* 1: four two-tap dynamic convolutions in every layer      */
  int32_t selector_rank;     /* r > 0: the path selector with rank-r codebooks; r a
                              * multiple of 32, <= 512; needs topk outputs              */
} dflash_config;

/* One draft decoder layer (pre-norm, Qwen3-style). All [out, in] row-major. */
typedef struct {
  const void *in_norm;   /* [H]                 */
  const void *wq;        /* [nq*hd, H]          */
  const void *wk;        /* [nkv*hd, H]         */
  const void *wv;        /* [nkv*hd, H]         */
  const void *q_norm;    /* [hd] (unused when qk_norm == 0, may be NULL) */
  const void *k_norm;    /* [hd] (unused when qk_norm == 0, may be NULL) */
  const void *wo;        /* [H, nq*hd]          */
  const void *post_norm; /* [H]                 */
  const void *w_gate;    /* [I, H]              */
  const void *w_up;      /* [I, H]              */
  const void *w_down;    /* [H, I]              */
  /* dyn_conv only (else may be NULL): four two-tap dynamic depthwise convolutions, index
   * 0 on the attention input (after in_norm), 1 on the attention output (after wo, before
   * the residual add), 2 on the MLP input (after post_norm), 3 on the MLP output (after
   * w_down, before the residual add). Over the K+1 block rows of a request,
   * y_t = k_t0 * x_t + k_t1 * x_{t-1} (x_{-1} = 0), with taps
   * k_ti[c] = conv_base[j][i][c] + (conv_proj[j] x_t)[i*G + c/16], G = H/16. */
  const void *conv_base; /* [4, 2, H]           */
  const void *conv_proj; /* [4, 2*G, H]         */
} dflash_layer_weights;

typedef struct {
  const void *embed;       /* [V, H] shared token embedding                          */
  const void *lm_head;     /* [V, H] shared LM head (may equal embed)                */
  const void *fc;          /* [H, n_feat*H_t]; input column block f holds feature f  */
  const void *fc_norm;     /* [H] RMSNorm after fc                                   */
  const void *final_norm;  /* [H] RMSNorm before the LM head                         */
  const dflash_layer_weights *layers; /* host array of n_layers entries (copied)     */
  const void *mask_embedding; /* [H] or NULL: a trained mask embedding used instead of
                               * embed[mask_token_id] for the K mask rows
                               * ("DFlash：把串行 Draft 变成并行“填空”" §5.2)          */
  /* selector_rank > 0 only (else may be NULL): the path selector's codebooks and gate. */
  const void *sel_pred_codebook; /* [V, r] predecessor embedding A                   */
  const void *sel_succ_codebook; /* [V, r] successor embedding B                     */
  const void *sel_hidden_proj;   /* [r, H] gate g_t = W_h h_t of the final hidden row  */
} dflash_weights;

typedef struct dflash_ctx dflash_ctx;

/* Checks a configuration on the host only (no CUDA call). Writes a reason into msg
 * (if msg != NULL and msg_len > 0) when the status is not DFLASH_OK. */
dflash_status dflash_validate_config(const dflash_config *cfg, char *msg, int32_t msg_len);

/* Creates a context on `device`: validates cfg, checks weight pointers (non-NULL,
 * 16-byte aligned), allocates the KV pool (max_pages x n_layers x 2 x nkv x 64 x hd
 * elements), scratch and staging. *out is set only on DFLASH_OK. */
dflash_status dflash_create(const dflash_config *cfg, const dflash_weights *w,
                            int32_t device, dflash_ctx **out);

/* Frees everything the context owns (after synchronising its device). NULL is a no-op. */
void dflash_destroy(dflash_ctx *ctx);

/* KV injection ("LLM的推理加速-DFlash" 关键创新 Step 2-3; "DFlash：把串行 Draft 变成并行“填空”"
 * §4.1, §5.1): appends n_new[b] positions to request req_ids[b] for b < n_req.
 *   req_ids [n_req] host: request ids (any int32); an unknown id registers a request.
 *   n_new   [n_req] host: rows per request, >= 0.
 *   reset   1: drop each request's existing context first (prefill); 0: append.
 *   feats   host array of n_feat DEVICE pointers; feats[f] is [sum(n_new), H_t]
 *           row-major (16-byte aligned), rows grouped by request in req_ids order.
 * Position p of a request gets K = RoPE(k_norm(g Wk^T), p) and V = g Wv^T in every
 * layer, g = RMSNorm(concat_f(h_f) W_fc^T). Errors: OUT_OF_PAGES / INVALID_ARG with
 * no state change. Rows are processed in chunks of max_inject_rows. */
dflash_status dflash_inject_context(dflash_ctx *ctx, void *stream, int32_t n_req,
                                    const int32_t *req_ids, const int32_t *n_new,
                                    int32_t reset, const void *const *feats);

/* Incremental injection straight from the target's verify block ("LLM的推理加速-DFlash"
 * 关键创新 Step 3: after verification the accepted positions' target hidden states enter
 * the draft cache): the same result as dflash_inject_context (reset 0) on the gathered rows.
 *   block_rows >= 1: feats[f] is [n_req * block_rows, H_t] row-major (16-byte aligned);
 *           rows [b * block_rows, (b + 1) * block_rows) belong to request req_ids[b].
 *   n_new   [n_req] host, 0 <= n_new[b] <= block_rows: the first n_new[b] rows of request
 *           b's block are appended (typically the accept length + 1 of its verify).
 * The counted rows are packed by the library (into memory it grows on demand), so the
 * caller passes the blocks as the target produced them.
 * Errors: as dflash_inject_context; INVALID_ARG if block_rows < 1, n_req * block_rows
 * exceeds 2^31 - 1, or a count is out of range. */
dflash_status dflash_inject_blocks(dflash_ctx *ctx, void *stream, int32_t n_req,
                                   const int32_t *req_ids, const int32_t *n_new,
                                   int32_t block_rows, const void *const *feats);

/* One draft step for n_req live requests ("DFlash：把串行 Draft 变成并行“填空”" §4-4.4):
 *   req_ids  [n_req] host.
 *   anchors  [n_req] int32 DEVICE: the last verified token of each request.
 *   argmax   [n_req, K] int32 DEVICE (required): per mask position, lowest index on ties.
 *   topk_idx [n_req, K, topk] int32 DEVICE or NULL; topk_val the fp32 logits, sorted
 *            descending (ties: lower index first); both or neither.
 *   logits   [n_req, K, V] fp32 DEVICE or NULL: full logits (for inspection).
 * Block row j of request b sits at position ctx_len_b + j (row 0 is the anchor). The
 * block's own K/V are not added to the cache. */
dflash_status dflash_draft_step(dflash_ctx *ctx, void *stream, int32_t n_req,
                                const int32_t *req_ids, const int32_t *anchors,
                                int32_t *argmax, int32_t *topk_idx, float *topk_val,
                                float *logits);

/* dflash_draft_step that also writes lse [n_req, K] fp32 DEVICE (NULL: not written): the
 * log of the softmax normaliser of each mask row's logits, log sum_v exp(logits[v]), so that
 * topk_val - lse are the draft's full-vocabulary log-probabilities of its candidates (the
 * input of a draft tree, "DDTree" §2.3). Computed in fp32. */
dflash_status dflash_draft_step_lse(dflash_ctx *ctx, void *stream, int32_t n_req,
                                    const int32_t *req_ids, const int32_t *anchors,
                                    int32_t *argmax, int32_t *topk_idx, float *topk_val,
                                    float *logits, float *lse);

/* Outputs of dflash_draft_step_ex (all DEVICE; NULL: not written). argmax is required;
 * topk_idx / topk_val both or neither; lse as in dflash_draft_step_lse. selected [n_req, K]
 * int32 (needs selector_rank > 0 and the top-k outputs): the path selector's walk
 * ("DFlash 2 块扩散投机解码技术详解" §3.1) — from the anchor, position t takes the candidate b
 * of its top-k with the largest S_t(a, b) = topk_val[t, b] + <A(a) * g_t, B(b)>, a being the
 * token taken at t-1 (the anchor at t = 0), g_t = sel_hidden_proj h_t with h_t the
 * final-normed hidden row of mask position t; equal scores go to the earlier candidate.
 * Scores are computed in fp32. With sel_uniform [n_req, K] fp32 given, the walk samples
 * instead (the selector's sampling mode, §3.1.3): position t draws from
 * q = softmax(S_t(a, .) / sel_temperature) over its candidates, by inverse CDF in vocabulary
 * order against sel_uniform[b][t]; the drawn token is the next predecessor, and q goes to
 * sel_q_tok / sel_q_p [n_req, K, 32] (entries 0..topk-1) and sel_q_n [n_req, K] (= topk),
 * the draft distribution that dflash_verify_sample_q takes. */
typedef struct {
  int32_t *argmax;
  int32_t *topk_idx;
  float *topk_val;
  float *logits;
  float *lse;
  int32_t *selected;
  float sel_temperature;
  const float *sel_uniform;
  int32_t *sel_q_tok;
  float *sel_q_p;
  int32_t *sel_q_n;
} dflash_draft_out;

dflash_status dflash_draft_step_ex(dflash_ctx *ctx, void *stream, int32_t n_req,
                                   const int32_t *req_ids, const int32_t *anchors,
                                   const dflash_draft_out *out);

/* The selector's walk on its own (no context): n_req requests, K positions with kc <= 32
 * candidates each. anchors [n_req] int32, cand_tok [n_req, K, kc] int32, unary
 * [n_req, K, kc] fp32, gate [n_req, K, r] fp32, pred / succ codebooks [V, r] of `dtype`,
 * outputs selected [n_req, K] int32 and scores [n_req, K, kc] fp32 or NULL (each position's
 * scores given the predecessor taken). All DEVICE. Tokens outside [0, vocab) read as zero
 * codebook rows. Limits: 1 <= K <= 31, 1 <= kc <= 32, r a multiple of 32 in [32, 512];
 * else DFLASH_ERR_INVALID_ARG. Scratch comes from the stream-ordered allocator. */
dflash_status dflash_select_path(void *stream, int32_t n_req, int32_t K, int32_t kc, int32_t r,
                                 int32_t vocab, dflash_dtype dtype, const int32_t *anchors, const int32_t *cand_tok,
                                 const float *unary, const float *gate, const void *pred_codebook,
                                 const void *succ_codebook, int32_t *selected, float *scores);

/* The selector's sampling walk on its own (no context): as dflash_select_path, with
 * temperature > 0 and uniforms u [n_req, K]; outputs selected [n_req, K] and the draft
 * distributions q_tok / q_p [n_req, K, 32] (entries 0..kc-1), q_n [n_req, K] (= kc). */
dflash_status dflash_select_sample(void *stream, int32_t n_req, int32_t K, int32_t kc, int32_t r,
                                   int32_t vocab, dflash_dtype dtype, float temperature,
                                   const int32_t *anchors, const int32_t *cand_tok, const float *unary,
                                   const float *gate, const void *pred_codebook, const void *succ_codebook,
                                   const float *u, int32_t *selected, int32_t *q_tok, float *q_p,
                                   int32_t *q_n);

/* Greedy verification ("DFlash 2 块扩散投机解码技术详解" §2.3): for each of n_req rows,
 *   draft  [n_req, K] int32 DEVICE, target [n_req, K+1] int32 DEVICE (the target's token
 *   after the anchor and after each draft), outputs (DEVICE):
 *   accept_len [n_req] = number of leading j < K with draft[j] == target[j] (= a),
 *   out_tokens [n_req, K+1] = draft[0..a-1], target[a], then -1 padding,
 *   next_anchor [n_req] = target[a].
 * The next injection for the request is a + 1 positions (the anchor and the accepted
 * drafts). n_req may exceed max_batch. */
dflash_status dflash_verify_greedy(dflash_ctx *ctx, void *stream, int32_t n_req,
                                   const int32_t *draft, const int32_t *target,
                                   int32_t *accept_len, int32_t *out_tokens,
                                   int32_t *next_anchor);

/* Sampling mode ("DFlash 2 块扩散投机解码技术详解" §2.3 rejection sampling, §3.3 the same
 * top-k / top-p truncation on the draft and the target side, §4.2 the fallback to p).
 * A row of logits becomes a distribution by: logits / temperature; keep the top_k largest
 * (ties to the lower vocabulary index); softmax over those; keep the shortest prefix in
 * descending order whose probability mass reaches top_p; renormalise. Draws are inverse-CDF
 * over the kept tokens in vocabulary order: the first token whose running mass exceeds
 * u times the total. Uniforms are inputs (the caller owns the random stream).
 * Limits: temperature > 0, 1 <= top_k <= 32, 0 < top_p <= 1 (top_k = 0, i.e. top-p over
 * the whole vocabulary, is not supported: DFLASH_ERR_UNSUPPORTED). Computed in fp32. */
typedef struct {
  float temperature;
  int32_t top_k;
  float top_p;
} dflash_sampling;

/* One draw per row from the sampling distribution of fp32 logits [rows, V] (DEVICE,
 * row-major, V = the config's vocab) with uniforms u [rows] in [0, 1) (DEVICE fp32) into
 * tokens [rows] int32 (DEVICE). Used to draw the drafts from the draft's logits. */
dflash_status dflash_sample_tokens(dflash_ctx *ctx, void *stream, int32_t rows,
                                   const dflash_sampling *sampling, const float *logits,
                                   const float *u, int32_t *tokens);

/* Sampling verification of n_req rows (n_req <= max_batch), all DEVICE:
 *   target_logits [n_req, K+1, V] fp32: the target's logits after the anchor and after
 *                 each draft; draft_logits [n_req, K, V] fp32: the draft's logits;
 *   draft [n_req, K] int32: tokens drawn from the draft's distributions;
 *   u_accept [n_req, K] fp32, u_resample [n_req] fp32: uniforms in [0, 1).
 * Position j accepts draft[j] when u_accept[j] < min(1, p_j(d)/q_j(d)) (q_j(d) = 0 accepts
 * iff p_j(d) > 0); the first rejection emits a draw from norm(max(p_j - q_j, 0)), or from
 * p_j when that is zero, and ends the row; with all K accepted a bonus is drawn from p_K.
 * Outputs as dflash_verify_greedy: accept_len [n_req] (= a), out_tokens [n_req, K+1] (the
 * a accepted drafts, the emitted token, -1 padding), next_anchor [n_req]. */
dflash_status dflash_verify_sample(dflash_ctx *ctx, void *stream, int32_t n_req,
                                   const dflash_sampling *sampling, const float *target_logits,
                                   const float *draft_logits, const int32_t *draft,
                                   const float *u_accept, const float *u_resample,
                                   int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor);

/* dflash_verify_sample with the draft distributions given as candidate lists instead of
 * draft logits (the path selector's sampling mode, "DFlash 2 块扩散投机解码技术详解" §3.1.3:
 * its draft distribution lives on the k candidates): q_tok / q_p [n_req, K, 32] DEVICE
 * (entries 0..q_n-1, distinct tokens, probabilities summing to 1), q_n [n_req, K] DEVICE in
 * 1..32. The target side is truncated from target_logits as in dflash_verify_sample; the
 * acceptance test, residual and bonus are the same. */
dflash_status dflash_verify_sample_q(dflash_ctx *ctx, void *stream, int32_t n_req, const dflash_sampling *sp,
                                     const float *target_logits, const int32_t *q_tok, const float *q_p,
                                     const int32_t *q_n, const int32_t *draft, const float *u_accept,
                                     const float *u_resample, int32_t *accept_len, int32_t *out_tokens,
                                     int32_t *next_anchor);

/* Draft trees ("DDTree" §2.3 Algorithm 1 / Proposition 2, §3.3 ancestor-only mask, §3.5
 * the verifier walk). No context needed; all pointers DEVICE, row-major.
 * dflash_ddtree_build: per request, L block positions with kc candidates each, best first:
 *   cand_tok [n_req, L, kc] int32 and cand_logp [n_req, L, kc] fp32; cand_lse is NULL
 *   (cand_logp are log-probabilities) or [n_req, L] fp32 row normalisers subtracted from
 *   cand_logp (cand_logp = topk_val and cand_lse = lse of dflash_draft_step_lse). The
 *   `budget` most likely prefixes (a prefix takes one candidate at each of positions 1..d;
 *   its log-probability is the sum)
 *   are popped best-first from a max-heap seeded with the best candidate of position 1,
 *   each pop pushing the next sibling and the first child; ties pop by (log-probability
 *   desc, depth asc, parent asc, rank asc). With kc >= min(budget, V) the tree is the
 *   optimal one; with fewer candidates it is the best tree over those candidates.
 *   Outputs [n_req, budget] in pop order: tree_tok, tree_parent (-1: child of the root, the
 *   anchor), tree_depth (1..L), tree_logp; n_nodes [n_req] (fewer than budget only when the
 *   candidates run out; unused slots hold token -1); mask [n_req, budget+1, W] uint32 or
 *   NULL, W = ceil((budget+1)/32): row i (0 = the root, node j = row j+1) has bit j set when
 *   index j is the root, an ancestor of i, or i itself.
 *   Limits: 1 <= L <= 31, 1 <= kc <= 32, 1 <= budget <= 1024; else DFLASH_ERR_INVALID_ARG.
 * dflash_ddtree_walk: greedy verification of built trees; target_next [n_req, budget+1]
 *   int32 is the target's token after the root (index 0) and after node j (index j+1).
 *   From the root, the walk moves to the child whose token equals the target's next token
 *   while one exists. Outputs accept_len [n_req], out_tokens [n_req, L+1] (the accepted
 *   tokens, then the target's token where the walk stopped, then -1), next_anchor [n_req]. */
dflash_status dflash_ddtree_build(void *stream, int32_t n_req, int32_t L, int32_t kc, int32_t budget,
                                  const int32_t *cand_tok, const float *cand_logp, const float *cand_lse,
                                  int32_t *tree_tok,
                                  int32_t *tree_parent, int32_t *tree_depth, float *tree_logp,
                                  int32_t *n_nodes, uint32_t *mask);
dflash_status dflash_ddtree_walk(void *stream, int32_t n_req, int32_t L, int32_t budget,
                                 const int32_t *tree_tok, const int32_t *tree_parent,
                                 const int32_t *n_nodes, const int32_t *target_next,
                                 int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor);

/* Forgets a request and returns its pages to the pool (host only). Work already
 * enqueued that reads those pages must precede any later call in stream order. */
dflash_status dflash_release(dflash_ctx *ctx, int32_t req_id);

/* Shortens a request's context to new_len <= its length (host only; frees whole pages
 * past the new end). Used by schedulers that roll a request back. */
dflash_status dflash_truncate(dflash_ctx *ctx, int32_t req_id, int32_t new_len);

/* Context length of a live request (host only). */
dflash_status dflash_context_len(const dflash_ctx *ctx, int32_t req_id, int32_t *len);

/* Copies positions [pos0, pos0+n) of one layer's cached K and V of a request into
 * k_out / v_out, each [n, nkv, hd] DEVICE buffers of the storage type (inspection). */
dflash_status dflash_export_kv(dflash_ctx *ctx, void *stream, int32_t req_id, int32_t layer,
                               int32_t pos0, int32_t n, void *k_out, void *v_out);

/* Free pages in the pool (host only). */
int32_t dflash_free_pages(const dflash_ctx *ctx);

/* Text of the last error on this context ("" if none). Valid until the next call. */
const char *dflash_last_error(const dflash_ctx *ctx);

/* Static name of a status code. */
const char *dflash_status_string(dflash_status s);

/* Number of kernel launches this context has issued so far (all calls). */
int64_t dflash_launch_count(const dflash_ctx *ctx);

/* Kernel timing (tracing). With timing enabled every kernel launch is bracketed by CUDA
 * events on its stream and tagged with a kernel class and its algorithmic bytes and
 * flops. dflash_timing_read synchronises on the recorded events, adds the elapsed time
 * per class into ms[i] (milliseconds), launches[i], bytes[i], flops[i] for
 * i < min(n, dflash_timing_classes()) (any of the arrays may be NULL), then clears the
 * records. Enabling adds two event records per launch. */
dflash_status dflash_timing_enable(dflash_ctx *ctx, int32_t enable);
int32_t dflash_timing_classes(void);
const char *dflash_timing_class_name(int32_t cls);
dflash_status dflash_timing_read(dflash_ctx *ctx, double *ms, int64_t *launches, double *bytes,
                                 double *flops, int32_t n);

/* Top-k of fp32 logits that allocates nothing (no counterpart on the pages: a service of
 * this library). Same result as the top-k of dflash_draft_step (values descending, ties to
 * the lower index, argmax = first), computed as per-chunk candidates plus a merge, with the
 * candidates in a fixed 4 MiB device array compiled into the library instead of memory from
 * cudaMalloc. It is meant for callers that cannot call the CUDA allocator: code being
 * recorded into a CUDA graph, or runtimes that own a fixed device-memory budget.
 *   logits [rows, vocab] fp32 DEVICE; argmax [rows] int32 DEVICE; topk_idx [rows, k] int32
 *   and topk_val [rows, k] fp32 DEVICE or both NULL; 1 <= k <= min(32, vocab);
 *   rows * ceil(vocab / 4096) * k must not exceed 524288, and vocab not 65535 * 4096
 *   (else DFLASH_ERR_INVALID_ARG, before any launch).
 *   msg (optional, msg_len bytes) receives the reason of an error.
 * The first call on a device looks up that device's copy of the array
 * (cudaGetSymbolAddress); make it before any stream capture. Every call, from any thread
 * or stream, uses the same array: calls that overlap on the GPU race and must be ordered
 * by the caller. No slot is read before the call writes it, so nothing needs clearing. */
dflash_status dflash_topk_noalloc(void *stream, int32_t rows, int32_t vocab, int32_t k,
                                  const float *logits, int32_t *argmax, int32_t *topk_idx,
                                  float *topk_val, char *msg, int32_t msg_len);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
