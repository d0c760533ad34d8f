// Internal launchers of libdflash (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace dflash {

struct ModelDims {
  int H, L, nq, nkv, hd, I, V, K, n_feat, Ht, topk;
  int qk_norm;
  float eps, emb_scale;
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
};

// dtype: 0 = fp32, 1 = bf16 (matches dflash_dtype)
cudaError_t gemm_simt(int dtype, const GemmDesc &d, cudaStream_t s);

cudaError_t launch_embed(int dtype, const ModelDims &m, int B, const int32_t *anchors,
                         int mask_id, const void *embed, void *x, int *err, cudaStream_t s);

// out row r <- rmsnorm(in row map(r)); map(r) = r, or with skip_anchor_k = K > 0 the
// K mask rows of each (K+1)-row block: (r / K) * (K + 1) + r % K + 1.
cudaError_t launch_rmsnorm(int dtype, int rows, int H, const void *in, int ld_in, void *out,
                           int ld_out, const void *w, float eps, int skip_anchor_k,
                           cudaStream_t s);

// In place on qkv rows [B*(K+1), qkv_dim]: per-head q/k RMSNorm (if enabled) + RoPE at
// position ctx_len[b] + j, rounded to the storage type.
cudaError_t launch_qk_norm_rope(int dtype, const ModelDims &m, int B, void *qkv,
                                const int32_t *ctx_len, const float2 *rope,
                                const void *q_norm, const void *k_norm, cudaStream_t s);

// Injection epilogue: kv rows [T, L*2*kv_dim] (per layer [k | v]) -> k-norm + RoPE at
// pos[t] -> KV pool slot[t] (page * 64 + offset) in every layer.
cudaError_t launch_inject_kv(int dtype, const ModelDims &m, int T, const void *kv,
                             const int32_t *slot, const int32_t *pos, const float2 *rope,
                             const void *const *k_norms, void *pool, cudaStream_t s);

cudaError_t launch_swiglu(int dtype, int rows, int I, const void *gu, void *h, cudaStream_t s);

// Split-KV attention of the query block of each request over its paged context plus the
// block's own K/V, then the split combine into o [B*(K+1), q_dim].
cudaError_t launch_attention(int dtype, const ModelDims &m, const DraftBatch &b, int layer,
                             const void *qkv, const void *pool, float *part_o, float *part_ml,
                             void *o, cudaStream_t s);

// Row-wise top-k (values descending, ties to the lower index) of fp32 logits [rows, V].
cudaError_t launch_topk(int rows, int V, int k, const float *logits, int32_t *argmax,
                        int32_t *topk_idx, float *topk_val, cudaStream_t s);

cudaError_t launch_verify(int n, int K, const int32_t *draft, const int32_t *target,
                          int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor,
                          cudaStream_t s);

cudaError_t launch_export_kv(int dtype, const ModelDims &m, int layer, int pos0, int n,
                             const int32_t *pages, const void *pool, void *k_out, void *v_out,
                             cudaStream_t s);

}  // namespace dflash
