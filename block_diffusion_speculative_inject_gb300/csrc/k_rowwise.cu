// Row-wise kernels of the draft step: block embedding, RMSNorm, q/k head norm + RoPE,
// the injection epilogue (k-norm + RoPE + paged-cache write), SwiGLU, greedy verify and
// the KV export. All are HBM/latency-bound elementwise passes; one warp per row or per
// (row, head), 16-byte aligned rows, fp32 arithmetic and one rounding per stored value.
#include "kernels.h"

namespace dflash {

constexpr int PAGE = KV_PAGE;

// ------------------------------------------------------------------------- embedding
// Block rows of request b: row 0 is the anchor token, rows 1..K the mask token; each is
// the shared embedding row times input_embedding_scale ("DFlash 2 块扩散投机解码技术详解"
// §2.2; "DFlash：把串行 Draft 变成并行“填空”" §4).
template <typename T>
__global__ void k_embed(int H, int Q, int V, const int32_t *anchors, int mask_id, float scale,
                        const T *embed, float *x, int *err) {
  int r = blockIdx.x;
  int b = r / Q, j = r % Q;
  int tok = j == 0 ? anchors[b] : mask_id;
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) raise_err(err, DEV_ERR_TOKEN);
    tok = 0;
  }
  const T *src = embed + (size_t)tok * H;
  float *dst = x + (size_t)r * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) dst[i] = to_f(src[i]) * scale;
}

cudaError_t launch_embed(int dtype, const ModelDims &m, int B, const int32_t *anchors,
                         int mask_id, const void *embed, float *x, int *err, cudaStream_t s) {
  dim3 g(B * m.Q());
  if (dtype) k_embed<bf16><<<g, 256, 0, s>>>(m.H, m.Q(), m.V, anchors, mask_id, m.emb_scale,
                                             (const bf16 *)embed, x, err);
  else k_embed<float><<<g, 256, 0, s>>>(m.H, m.Q(), m.V, anchors, mask_id, m.emb_scale,
                                        (const float *)embed, x, err);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- RMSNorm
// y = x * rsqrt(mean(x^2) + eps) * w, written as a GEMM operand. One 128-thread CTA per row:
// the row is read once with float4 loads into registers (H <= 8192), reduced across the
// block, scaled and written.
constexpr int RN_THREADS = 128;
constexpr int RN_VEC = 16;   // float4 per thread: H <= 128 * 4 * 16 = 8192

template <typename TW>
__global__ void __launch_bounds__(RN_THREADS) k_rmsnorm(int rows, int H, const float *in, int ld_in,
                                                        OpOut out, int ld_out, const TW *w,
                                                        float eps, int skip_k) {
  __shared__ float red[RN_THREADS / 32];
  const int r = blockIdx.x;
  if (r >= rows) return;
  const int src = skip_k > 0 ? (r / skip_k) * (skip_k + 1) + r % skip_k + 1 : r;
  const float4 *xi = (const float4 *)(in + (size_t)src * ld_in);
  const int n4 = H / 4;
  float4 v[RN_VEC];
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < RN_VEC; ++t) {
    const int i = threadIdx.x + t * RN_THREADS;
    if (i < n4) {
      v[t] = xi[i];
      ss += v[t].x * v[t].x + v[t].y * v[t].y + v[t].z * v[t].z + v[t].w * v[t].w;
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < RN_THREADS / 32; ++i) tot += red[i];
  const float rs = rsqrtf(tot / (float)H + eps);
  const size_t o = (size_t)r * ld_out;
#pragma unroll
  for (int t = 0; t < RN_VEC; ++t) {
    const int i = threadIdx.x + t * RN_THREADS;
    if (i < n4) {
      const int e = 4 * i;
      write_op(out, o + e + 0, v[t].x * rs * to_f(w[e + 0]));
      write_op(out, o + e + 1, v[t].y * rs * to_f(w[e + 1]));
      write_op(out, o + e + 2, v[t].z * rs * to_f(w[e + 2]));
      write_op(out, o + e + 3, v[t].w * rs * to_f(w[e + 3]));
    }
  }
}

cudaError_t launch_rmsnorm(int dtype, int rows, int H, const float *in, int ld_in, OpOut out,
                           int ld_out, const void *w, float eps, int skip_anchor_k,
                           cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (H % 4 || H > RN_THREADS * 4 * RN_VEC || ld_in % 4) return cudaErrorInvalidValue;
  if (dtype) k_rmsnorm<bf16><<<rows, RN_THREADS, 0, s>>>(rows, H, in, ld_in, out, ld_out,
                                                        (const bf16 *)w, eps, skip_anchor_k);
  else k_rmsnorm<float><<<rows, RN_THREADS, 0, s>>>(rows, H, in, ld_in, out, ld_out,
                                                   (const float *)w, eps, skip_anchor_k);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- head norm + RoPE
// One warp rotates one head vector of hd (64 or 128) values held as hd/32 per lane:
// lane holds i = lane + 32*t; pairs are (i, i + hd/2) so for hd = 128 lane's t=0,1
// pair with t=2,3 and for hd = 64 t=0 pairs with t=1.
template <typename TW, typename TD>
__device__ __forceinline__ void head_norm_rope(const float *src, TD *dst, const TW *nw, int hd,
                                               float eps, const float2 *rope_row, int lane) {
  float v[4];
  const int per = hd / 32;
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (t < per) {
      v[t] = src[lane + 32 * t];
      ss += v[t] * v[t];
    }
  if (nw) {
    ss = warp_sum(ss);
    float rs = rsqrtf(ss / (float)hd + eps);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (t < per) v[t] = v[t] * rs * to_f(nw[lane + 32 * t]);
  }
  const int hp = per / 2;  // number of first-half slots per lane
  float o[4];
#pragma unroll
  for (int t = 0; t < 2; ++t)
    if (t < hp) {
      int i = lane + 32 * t;
      float2 cs = rope_row[i];
      float x1 = v[t], x2 = v[t + hp];
      o[t] = x1 * cs.x - x2 * cs.y;
      o[t + hp] = x2 * cs.x + x1 * cs.y;
    }
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (t < per) dst[lane + 32 * t] = from_f<TD>(o[t]);
}

template <typename TW>
__global__ void k_qk_norm_rope(int rows, int Q, int nq, int nkv, int hd, int qkv_dim,
                               float *qkv, const int32_t *ctx_len, const float2 *rope,
                               const TW *q_norm, const TW *k_norm, float eps) {
  int w = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  int heads = nq + nkv;
  if (w >= rows * heads) return;
  int r = w / heads, h = w % heads;
  int b = r / Q, j = r % Q;
  int pos = ctx_len[b] + j;
  float *p = qkv + (size_t)r * qkv_dim + (size_t)h * hd;   // q heads then k heads are contiguous
  const TW *nw = h < nq ? q_norm : k_norm;
  head_norm_rope<TW, float>(p, p, nw, hd, eps, rope + (size_t)pos * (hd / 2), lane);
}

cudaError_t launch_qk_norm_rope(int dtype, const ModelDims &m, int B, float *qkv,
                                const int32_t *ctx_len, const float2 *rope,
                                const void *q_norm, const void *k_norm, cudaStream_t s) {
  int rows = B * m.Q();
  int warps = rows * (m.nq + m.nkv);
  dim3 g((warps + 7) / 8);
  const void *qn = m.qk_norm ? q_norm : nullptr, *kn = m.qk_norm ? k_norm : nullptr;
  if (dtype) k_qk_norm_rope<bf16><<<g, 256, 0, s>>>(rows, m.Q(), m.nq, m.nkv, m.hd, m.qkv_dim(),
                                                    qkv, ctx_len, rope, (const bf16 *)qn,
                                                    (const bf16 *)kn, m.eps);
  else k_qk_norm_rope<float><<<g, 256, 0, s>>>(rows, m.Q(), m.nq, m.nkv, m.hd, m.qkv_dim(),
                                               qkv, ctx_len, rope, (const float *)qn,
                                               (const float *)kn, m.eps);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- injection epilogue
// Row t of the layer-batched K/V projection of g goes, in every layer, through the per-head
// k-norm and RoPE at its position and into its page slot; V is stored as projected
// ("DFlash：块扩散 + KV 注入" §四: projection then norm + RoPE post-processing;
// "DFlash：把串行 Draft 变成并行“填空”" §5.1).
struct KNormPtrs { const void *p[16]; };

template <typename T>
__global__ void k_inject_kv(int T_rows, int L, int nkv, int hd, const float *kv, const int32_t *slot,
                            const int32_t *pos, const float2 *rope, KNormPtrs kn, int qk_norm,
                            float eps, T *pool) {
  int w = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (w >= T_rows * L * nkv) return;
  int t = w / (L * nkv), rem = w % (L * nkv);
  int l = rem / nkv, h = rem % nkv;
  int kv_dim = nkv * hd;
  int sl = slot[t];
  int page = sl / PAGE, off = sl % PAGE;
  const float *src_k = kv + (size_t)t * (L * 2 * kv_dim) + (size_t)l * 2 * kv_dim + (size_t)h * hd;
  const float *src_v = src_k + kv_dim;
  T *dk = pool + kv_block(page, l, 0, h, L, nkv, hd) + (size_t)off * hd;
  T *dv = pool + kv_block(page, l, 1, h, L, nkv, hd) + off;     // transposed: [hd][64]
  const T *nw = qk_norm ? (const T *)kn.p[l] : nullptr;
  head_norm_rope<T, T>(src_k, dk, nw, hd, eps, rope + (size_t)pos[t] * (hd / 2), lane);
  for (int i = lane; i < hd; i += 32) dv[(size_t)i * PAGE] = from_f<T>(src_v[i]);
}

cudaError_t launch_inject_kv(int dtype, const ModelDims &m, int T, const float *kv,
                             const int32_t *slot, const int32_t *pos, const float2 *rope,
                             const void *const *k_norms, void *pool, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  KNormPtrs kn{};
  for (int l = 0; l < m.L && l < 16; ++l) kn.p[l] = k_norms[l];
  long warps = (long)T * m.L * m.nkv;
  dim3 g((unsigned)((warps + 7) / 8));
  if (dtype) k_inject_kv<bf16><<<g, 256, 0, s>>>(T, m.L, m.nkv, m.hd, kv, slot, pos, rope, kn,
                                                 m.qk_norm, m.eps, (bf16 *)pool);
  else k_inject_kv<float><<<g, 256, 0, s>>>(T, m.L, m.nkv, m.hd, kv, slot, pos, rope, kn,
                                            m.qk_norm, m.eps, (float *)pool);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- SwiGLU
// gu rows hold [gate (I) | up (I)] in fp32; h = silu(gate) * up as a GEMM operand.
__global__ void k_swiglu(long n, int I, const float *gu, OpOut h) {
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  long r = i / I, c = i % I;
  float g = gu[r * 2 * I + c], u = gu[r * 2 * I + I + c];
  write_op(h, i, g / (1.f + expf(-g)) * u);
}

cudaError_t launch_swiglu(int rows, int I, const float *gu, OpOut h, cudaStream_t s) {
  long n = (long)rows * I;
  if (n == 0) return cudaSuccess;
  k_swiglu<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(n, I, gu, h);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- greedy verify
// a = number of leading j < K with draft[j] == target[j]; emit draft[0..a-1] then target[a]
// ("DFlash 2 块扩散投机解码技术详解" §2.3; at most K+1 tokens: "DFlash：把串行 Draft 变成并行“填空”" §2).
__global__ void k_verify(int n, int K, const int32_t *draft, const int32_t *target,
                         int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor) {
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
  k_verify<<<(n + 127) / 128, 128, 0, s>>>(n, K, draft, target, accept_len, out_tokens,
                                           next_anchor);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- KV export
template <typename T>
__global__ void k_export_kv(int L, int nkv, int hd, int layer, int pos0, int n,
                            const int32_t *pages, const T *pool, T *k_out, T *v_out) {
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
  if (dtype) k_export_kv<bf16><<<g, 256, 0, s>>>(m.L, m.nkv, m.hd, layer, pos0, n, pages,
                                                 (const bf16 *)pool, (bf16 *)k_out, (bf16 *)v_out);
  else k_export_kv<float><<<g, 256, 0, s>>>(m.L, m.nkv, m.hd, layer, pos0, n, pages,
                                            (const float *)pool, (float *)k_out, (float *)v_out);
  return cudaGetLastError();
}

}  // namespace dflash
