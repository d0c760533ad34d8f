// Internal launchers of libdflash (not part of the C ABI).
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace dflash {

struct ModelDims {
  int H, L, nq, nkv, hd, I, V, K, n_feat, Ht, topk;
  int qk_norm;
  float eps, emb_scale;
  int causal;                 // causal mask inside the query block
  float out_mult, softcap;    // logits *= out_mult, then softcap * tanh(logits / softcap) if > 0
  int conv;                   // DFlash 2 dynamic convolutions in every layer
  int sel_r;                  // DFlash 2 path selector rank (0: off)
  int q_dim() const { return nq * hd; }
  int kv_dim() const { return nkv * hd; }
  int qkv_dim() const { return (nq + 2 * nkv) * hd; }
  int Q() const { return K + 1; }
};

// Device batch descriptor of one draft step, packed as int32:
//   ctx_len[B] | n_split[B] | split_len[B] | page_off[B+1] | pages[page_off[B]]
struct DraftBatch {
  const int32_t *ctx_len, *n_split, *split_len, *page_off, *pages;
  int B;
  int max_split;
  int min_split;        // the smallest split count of the batch (0: a request has no context)
};

// dtype (storage type of weights / features / cache): 0 = fp32, 1 = bf16.
cudaError_t gemm_simt(int dtype, const GemmDesc &d, cudaStream_t s);

// Tensor maps over the KV pool for the tensor-core attention: K blocks viewed as rows of hd
// values (box 64 x 64), V blocks ([hd][64]) as rows of 64 positions (box 64 x 128).
struct AttnMaps {
  CUtensorMap k, v;
  bool valid;
  int *err;      // device error flag raised by expired waits
  int num_sms;
};

// Split-KV attention of the query block of each request over its paged context plus the
// block's own K/V, then the split combine into the operand o [B*(K+1), q_dim].
cudaError_t launch_attention(int dtype, const ModelDims &m, const DraftBatch &b, int layer,
                             const float *qkv, const void *pool, float *part_o, float *part_ml,
                             OpOut o, const AttnMaps *maps, cudaStream_t s);

// The tensor-core split kernel (bf16 cache, head_dim 128).
cudaError_t launch_attn_split_tc(const ModelDims &m, const DraftBatch &b, int layer,
                                 const float *qkv, const AttnMaps *maps, float scale_log2,
                                 float *part_o, float *part_ml, cudaStream_t s);

// Sampling mode: truncated distributions (at most SMP_K kept tokens per row) of fp32 logits
// [rows, V], optionally with one draw per row against uniforms u; the verification of a batch
// from its target rows [B][K+1] and draft rows [B][K] of such distributions.
constexpr int SMP_K = 32;
cudaError_t launch_trunc_dist(int rows, int V, float temperature, int top_k, float top_p,
                              const float *logits, const float *u, int32_t *draw, int32_t *dist_tok,
                              float *dist_p, int32_t *dist_n, int max_ctas, cudaStream_t s);
cudaError_t launch_verify_sample(int B, int K, const int32_t *ptok, const float *pp, const int32_t *pn,
                                 const int32_t *qtok, const float *qp, const int32_t *qn,
                                 const int32_t *draft, const float *u_accept, const float *u_resample,
                                 int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor,
                                 cudaStream_t s);

// logits[i] = logit_xform(logits[i]) over n fp32 values, in place.
cudaError_t launch_logit_xform(long n, float mult, float cap, float *logits, cudaStream_t s);

// Row-wise top-k (values descending, ties to the lower index) of fp32 logits [rows, V], on at
// most max_ctas CTAs (<= 0: one per row) that loop over the rows; lse [rows] (or null) gets
// each row's log(sum exp).
cudaError_t launch_topk(int rows, int V, int k, const float *logits, int32_t *argmax,
                        int32_t *topk_idx, float *topk_val, float *lse, int max_ctas, cudaStream_t s);

// Merge of the per-tile candidates [tiles][rows][k] of the tensor-core LM-head epilogue; with
// lse non-null also each row's log(sum exp) from the tiles' (max, sum exp) partials.
cudaError_t launch_topk_merge(int tiles, int rows, int k, const int2 *cand, int32_t *argmax,
                              int32_t *topk_idx, float *topk_val, const float2 *lse_part, float *lse,
                              cudaStream_t s);

// GEMM post-ops over split-K partials ws[S][M][N] (see k_post.cu).
cudaError_t launch_post_qkv(int dtype, const ModelDims &m, int B, const float *ws, int S, float *qkv,
                            const int32_t *ctx_len, const float2 *rope, const void *q_norm,
                            const void *k_norm, cudaStream_t s);
cudaError_t launch_post_norm(int dtype, int M, int H, const float *ws, int S, float *x, OpOut out,
                             const void *w, float eps, int out_skip_k, cudaStream_t s);
cudaError_t launch_post_swiglu(int M, int I, const float *ws, int S, OpOut h, cudaStream_t s);
// out + f * out_stride + r * row_bytes  <-  in[f] + src[r] * row_bytes, r < rows, f < n_feat <= 8
cudaError_t launch_gather_rows(int n_feat, int rows, long row_bytes, const int32_t *src,
                               const void *const *in, void *out, long out_stride, cudaStream_t s);
cudaError_t launch_post_kv(int dtype, const ModelDims &m, int T, const float *ws, int S,
                           const int32_t *slot, const int32_t *pos, const float2 *rope,
                           const void *const *k_norms, void *pool, cudaStream_t s);
cudaError_t launch_embed_norm(int dtype, const ModelDims &m, int B, const int32_t *anchors, int mask_id,
                              const void *embed, const void *mask_emb, float *x, OpOut out, const void *w,
                              int *err, cudaStream_t s);

cudaError_t launch_verify(int n, int K, const int32_t *draft, const int32_t *target,
                          int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor,
                          cudaStream_t s);

// DFlash 2 modules (k_dflash2.cu). corr [M][2G] holds each row's tap corrections (G = H/16).
cudaError_t launch_conv_in(int dtype, int M, int Q, int H, OpOut in, const float *corr, const void *base,
                           OpOut out, cudaStream_t s);
cudaError_t launch_conv_out_norm(int dtype, int M, int Q, int H, const float *y, const float *corr,
                                 const void *base, float *x, OpOut out, const void *w, float eps,
                                 int out_skip_k, cudaStream_t s);
cudaError_t launch_to_op(long n, const float *src, OpOut out, cudaStream_t s);
// Sampling mode of the selector's walk (null: the greedy walk): temperature, uniforms
// [n][K], and the drawn positions' candidate distributions as lists of stride SMP_K.
struct SelSample {
  float temperature;
  const float *u;
  int32_t *q_tok;
  float *q_p;
  int32_t *q_n;
};
cudaError_t launch_select_path(int dtype, int n, int K, int kc, int r, int V, const int32_t *anchors,
                               const int32_t *cand_tok, const float *unary, const float *gate, const void *pred,
                               const void *succ, float *tab, int32_t *selected, float *scores, cudaStream_t s,
                               const SelSample *smp = nullptr);

cudaError_t launch_export_kv(int dtype, const ModelDims &m, int layer, int pos0, int n,
                             const int32_t *pages, const void *pool, void *k_out, void *v_out,
                             cudaStream_t s);

}  // namespace dflash
