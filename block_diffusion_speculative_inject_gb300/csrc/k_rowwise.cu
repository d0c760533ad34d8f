// Greedy verification and the KV export (inspection) — the row-wise kernels that are not
// GEMM post-ops.
#include "kernels.h"

namespace dflash {

constexpr int PAGE = KV_PAGE;

// ------------------------------------------------------------------------- logit scale / soft cap
// The optional output scale and logit soft cap of the LM head ("DFlash 2 块扩散投机解码技术
// 详解" §1.x compute_logits), in place on fp32 logits [n] (the unfused LM-head path).
__global__ void k_logit_xform(long n, float mult, float cap, float *logits) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) logits[i] = logit_xform(logits[i], mult, cap);
}

cudaError_t launch_logit_xform(long n, float mult, float cap, float *logits, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(k_logit_xform, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, n, mult, cap, logits);
}

// ------------------------------------------------------------------------- greedy verify
// a = number of leading j < K with draft[j] == target[j]; emit draft[0..a-1] then target[a]
// ("DFlash 2 块扩散投机解码技术详解" §2.3; at most K+1 tokens: "DFlash：把串行 Draft 变成并行“填空”" §2).
__global__ void k_verify(int n, int K, const int32_t *draft, const int32_t *target,
                         int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= n) return;
  const int32_t *d = draft + (size_t)b * K;
  const int32_t *t = target + (size_t)b * (K + 1);
  int a = 0;
  while (a < K && d[a] == t[a]) ++a;
  int32_t *o = out_tokens + (size_t)b * (K + 1);
  for (int j = 0; j <= K; ++j) o[j] = j < a ? d[j] : (j == a ? t[a] : -1);
  accept_len[b] = a;
  next_anchor[b] = t[a];
}

cudaError_t launch_verify(int n, int K, const int32_t *draft, const int32_t *target,
                          int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor,
                          cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(k_verify, dim3((n + 127) / 128), dim3(128), 0, s, n, K, draft, target,
                    accept_len, out_tokens, next_anchor);
}

// ------------------------------------------------------------------------- KV export
template <typename T>
__global__ void k_export_kv(int L, int nkv, int hd, int layer, int pos0, int n,
                            const int32_t *pages, const T *pool, T *k_out, T *v_out) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  long total = (long)n * nkv * hd;
  if (i >= total) return;
  int d = i % hd;
  int h = (i / hd) % nkv;
  int t = i / ((long)hd * nkv);
  int p = pos0 + t;
  int page = pages[p / PAGE], off = p % PAGE;
  k_out[i] = pool[kv_block(page, layer, 0, h, L, nkv, hd) + (size_t)off * hd + d];
  v_out[i] = pool[kv_block(page, layer, 1, h, L, nkv, hd) + (size_t)d * PAGE + off];
}

cudaError_t launch_export_kv(int dtype, const ModelDims &m, int layer, int pos0, int n,
                             const int32_t *pages, const void *pool, void *k_out, void *v_out,
                             cudaStream_t s) {
  long total = (long)n * m.nkv * m.hd;
  if (total == 0) return cudaSuccess;
  dim3 g((unsigned)((total + 255) / 256));
  if (dtype) return launch_pdl(k_export_kv<bf16>, g, dim3(256), 0, s, m.L, m.nkv, m.hd, layer, pos0, n, pages,
                                                 (const bf16 *)pool, (bf16 *)k_out, (bf16 *)v_out);
  return launch_pdl(k_export_kv<float>, g, dim3(256), 0, s, m.L, m.nkv, m.hd, layer, pos0, n, pages,
                                            (const float *)pool, (float *)k_out, (float *)v_out);
}

}  // namespace dflash
