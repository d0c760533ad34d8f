// GEMM post-ops: each sums a GEMM's S split-K partials ws[S][M][N] (fp32, in split order;
// S = 1 when the GEMM was not split) and applies the operation that follows that GEMM on
// the path, so the sum never makes an extra round trip through HBM:
//   post_qkv         q/k heads: per-head RMSNorm (if enabled) + RoPE at ctx_len[b] + j; v copied
//   post_resid_norm  x += sum (residual), then RMSNorm(x) as the next GEMM's operand
//   post_norm        RMSNorm(sum) as an operand (the fused context feature g)
//   post_swiglu      silu(gate) * up as an operand (gate = columns [0, I), up = [I, 2I))
//   post_kv          injection: every layer's k (norm + RoPE) and v into the paged cache
#include "kernels.h"

namespace dflash {

__device__ __forceinline__ float psum(const float *__restrict__ ws, int S, int M, int N, int m,
                                      int n) {
  // four independent loads in flight per round trip; the sum keeps split order
  float a = 0.f;
  int s = 0;
  for (; s + 4 <= S; s += 4) {
    const float v0 = __ldg(ws + ((size_t)(s + 0) * M + m) * N + n);
    const float v1 = __ldg(ws + ((size_t)(s + 1) * M + m) * N + n);
    const float v2 = __ldg(ws + ((size_t)(s + 2) * M + m) * N + n);
    const float v3 = __ldg(ws + ((size_t)(s + 3) * M + m) * N + n);
    a += v0;
    a += v1;
    a += v2;
    a += v3;
  }
  for (; s < S; ++s) a += __ldg(ws + ((size_t)s * M + m) * N + n);
  return a;
}

// One warp rotates one head of hd (64 or 128) values held hd/32 per lane; pairs (i, i+hd/2).
template <typename TW>
__device__ __forceinline__ void norm_rope_regs(float (&v)[4], int per, const TW *nw, int hd, float eps,
                                               const float2 *rope_row, int lane) {
  if (nw) {
    float ss = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (t < per) ss += v[t] * v[t];
    ss = warp_sum(ss);
    const float rs = rsqrtf(ss / (float)hd + eps);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (t < per) v[t] = v[t] * rs * to_f(nw[lane + 32 * t]);
  }
  const int hp = per / 2;
  float o[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int t = 0; t < 2; ++t)
    if (t < hp) {
      const float2 cs = rope_row[lane + 32 * t];
      o[t] = v[t] * cs.x - v[t + hp] * cs.y;
      o[t + hp] = v[t + hp] * cs.x + v[t] * cs.y;
    }
#pragma unroll
  for (int t = 0; t < 4; ++t) v[t] = o[t];
}

// ------------------------------------------------------------------------- q/k/v
template <typename TW>
__global__ void k_post_qkv(int M, int S, const float *ws, int Q, int nq, int nkv, int hd,
                           float *qkv, const int32_t *ctx_len, const float2 *rope, const TW *q_norm,
                           const TW *k_norm, float eps) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  const int w = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int heads = nq + 2 * nkv;
  if (w >= M * heads) return;
  const int m = w / heads, h = w % heads;
  const int N = heads * hd, per = hd / 32;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (t < per) v[t] = psum(ws, S, M, N, m, h * hd + lane + 32 * t);
  if (h < nq + nkv) {
    const int b = m / Q, j = m % Q;
    const int pos = ctx_len[b] + j;
    norm_rope_regs<TW>(v, per, h < nq ? q_norm : k_norm, hd, eps, rope + (size_t)pos * (hd / 2), lane);
  }
  float *dst = qkv + (size_t)m * N + (size_t)h * hd;
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (t < per) dst[lane + 32 * t] = v[t];
}

cudaError_t launch_post_qkv(int dtype, const ModelDims &m, int B, const float *ws, int S, float *qkv,
                            const int32_t *ctx_len, const float2 *rope, const void *q_norm,
                            const void *k_norm, cudaStream_t s) {
  const int rows = B * m.Q();
  const int warps = rows * (m.nq + 2 * m.nkv);
  dim3 g((warps + 7) / 8);
  const void *qn = m.qk_norm ? q_norm : nullptr, *kn = m.qk_norm ? k_norm : nullptr;
  if (dtype)
    return launch_pdl(k_post_qkv<bf16>, g, dim3(256), 0, s, rows, S, ws, m.Q(), m.nq, m.nkv, m.hd, qkv,
                      ctx_len, rope, (const bf16 *)qn, (const bf16 *)kn, m.eps);
  return launch_pdl(k_post_qkv<float>, g, dim3(256), 0, s, rows, S, ws, m.Q(), m.nq, m.nkv, m.hd, qkv,
                    ctx_len, rope, (const float *)qn, (const float *)kn, m.eps);
}

// ------------------------------------------------------------------------- residual + RMSNorm
// One 128-thread CTA per row of H <= 8192 (16 float4 per thread in registers). With
// x != nullptr: x[m] += sum (written back), then the norm of x; else the norm of the sum.
// out_skip_k = K > 0 writes the norm only for the K mask rows of each (K+1)-row block, to
// output row b*K + j - 1 (the final norm before the LM head).
// four consecutive weights as floats (one vector load when the address allows it)
__device__ __forceinline__ float4 load4(const bf16 *w) {
  if (((uintptr_t)w & 7u) == 0) {
    const uint2 u = __ldg((const uint2 *)w);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
  }
  return make_float4(to_f(w[0]), to_f(w[1]), to_f(w[2]), to_f(w[3]));
}
__device__ __forceinline__ float4 load4(const float *w) {
  if (((uintptr_t)w & 15u) == 0) return __ldg((const float4 *)w);
  return make_float4(w[0], w[1], w[2], w[3]);
}

constexpr int PN_THREADS = 128;
constexpr int PN_VEC = 16;

template <typename TW>
__global__ void __launch_bounds__(PN_THREADS) k_post_norm(int M, int S, const float *ws, int H,
                                                          float *x, OpOut out, const TW *w,
                                                          float eps, int out_skip_k) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ float red[PN_THREADS / 32];
  const int m = blockIdx.x;
  const int n4 = H / 4;
  float4 v[PN_VEC];
  // residual first, then the partials split by split (all of a split's loads in flight)
#pragma unroll
  for (int t = 0; t < PN_VEC; ++t) {
    const int i = threadIdx.x + t * PN_THREADS;
    v[t] = (x && i < n4) ? ((const float4 *)(x + (size_t)m * H))[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int s = 0; s < S; ++s) {
    const float4 *src = (const float4 *)(ws + ((size_t)s * M + m) * H);
    float4 p[PN_VEC];
#pragma unroll
    for (int t = 0; t < PN_VEC; ++t) {
      const int i = threadIdx.x + t * PN_THREADS;
      p[t] = i < n4 ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int t = 0; t < PN_VEC; ++t) {
      v[t].x += p[t].x; v[t].y += p[t].y; v[t].z += p[t].z; v[t].w += p[t].w;
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < PN_VEC; ++t) {
    const int i = threadIdx.x + t * PN_THREADS;
    if (i < n4) {
      if (x) ((float4 *)(x + (size_t)m * H))[i] = v[t];
      ss += v[t].x * v[t].x + v[t].y * v[t].y + v[t].z * v[t].z + v[t].w * v[t].w;
    }
  }
  int orow = m;
  if (out_skip_k > 0) {
    const int Q = out_skip_k + 1, b = m / Q, j = m % Q;
    if (j == 0) return;                       // the anchor row yields no candidate
    orow = b * out_skip_k + j - 1;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < PN_THREADS / 32; ++i) tot += red[i];
  const float rs = rsqrtf(tot / (float)H + eps);
  const size_t o = (size_t)orow * H;
#pragma unroll
  for (int t = 0; t < PN_VEC; ++t) {
    const int i = threadIdx.x + t * PN_THREADS;
    if (i < n4) {
      const int e = 4 * i;
      const float4 wv = load4(w + e);
      write_op4(out, o + e, make_float4(v[t].x * rs * wv.x, v[t].y * rs * wv.y, v[t].z * rs * wv.z, v[t].w * rs * wv.w));
    }
  }
}

cudaError_t launch_post_norm(int dtype, int M, int H, const float *ws, int S, float *x, OpOut out,
                             const void *w, float eps, int out_skip_k, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (H % 4 || H > PN_THREADS * 4 * PN_VEC) return cudaErrorInvalidValue;
  if (dtype)
    return launch_pdl(k_post_norm<bf16>, dim3(M), dim3(PN_THREADS), 0, s, M, S, ws, H, x, out,
                      (const bf16 *)w, eps, out_skip_k);
  return launch_pdl(k_post_norm<float>, dim3(M), dim3(PN_THREADS), 0, s, M, S, ws, H, x, out,
                    (const float *)w, eps, out_skip_k);
}

// ------------------------------------------------------------------------- SwiGLU
__global__ void k_post_swiglu(int M, int S, const float *ws, int I, OpOut h) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)M * I) return;
  const int m = (int)(i / I), c = (int)(i % I);
  const float g = psum(ws, S, M, 2 * I, m, c), u = psum(ws, S, M, 2 * I, m, I + c);
  write_op(h, i, g / (1.f + expf(-g)) * u);
}

cudaError_t launch_post_swiglu(int M, int I, const float *ws, int S, OpOut h, cudaStream_t s) {
  const long n = (long)M * I;
  if (n == 0) return cudaSuccess;
  return launch_pdl(k_post_swiglu, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, M, S, ws, I, h);
}

// ------------------------------------------------------------------------- injection into the cache
struct KNorms { const void *p[16]; };

template <typename T>
__global__ void k_post_kv(int Trows, int S, const float *ws, int L, int nkv, int hd,
                          const int32_t *slot, const int32_t *pos, const float2 *rope, KNorms kn,
                          int qk_norm, float eps, T *pool) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  const int w = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= Trows * L * nkv) return;
  const int t = w / (L * nkv), rem = w % (L * nkv);
  const int l = rem / nkv, h = rem % nkv;
  const int kv_dim = nkv * hd, N = L * 2 * kv_dim, per = hd / 32;
  const int kcol = l * 2 * kv_dim + h * hd, vcol = kcol + kv_dim;
  float k[4] = {0.f, 0.f, 0.f, 0.f}, v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i < per) {
      k[i] = psum(ws, S, Trows, N, t, kcol + lane + 32 * i);
      v[i] = psum(ws, S, Trows, N, t, vcol + lane + 32 * i);
    }
  norm_rope_regs<T>(k, per, qk_norm ? (const T *)kn.p[l] : nullptr, hd, eps,
                    rope + (size_t)pos[t] * (hd / 2), lane);
  const int sl = slot[t], page = sl / KV_PAGE, off = sl % KV_PAGE;
  T *dk = pool + kv_block(page, l, 0, h, L, nkv, hd) + (size_t)off * hd;
  T *dv = pool + kv_block(page, l, 1, h, L, nkv, hd) + off;     // V stored [hd][64]
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i < per) {
      dk[lane + 32 * i] = from_f<T>(k[i]);
      dv[(size_t)(lane + 32 * i) * KV_PAGE] = from_f<T>(v[i]);
    }
}

cudaError_t launch_post_kv(int dtype, const ModelDims &m, int T, const float *ws, int S,
                           const int32_t *slot, const int32_t *pos, const float2 *rope,
                           const void *const *k_norms, void *pool, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  KNorms kn{};
  for (int l = 0; l < m.L && l < 16; ++l) kn.p[l] = k_norms[l];
  const long warps = (long)T * m.L * m.nkv;
  dim3 g((unsigned)((warps + 7) / 8));
  if (dtype)
    return launch_pdl(k_post_kv<bf16>, g, dim3(256), 0, s, T, S, ws, m.L, m.nkv, m.hd, slot, pos, rope,
                      kn, m.qk_norm, m.eps, (bf16 *)pool);
  return launch_pdl(k_post_kv<float>, g, dim3(256), 0, s, T, S, ws, m.L, m.nkv, m.hd, slot, pos, rope,
                    kn, m.qk_norm, m.eps, (float *)pool);
}

// ------------------------------------------------------------------------- embedding + first norm
// x[b*(K+1) + j] = embed[token] * scale (token = anchor for j = 0, else the mask id), and
// the first layer's input norm of that row as an operand.
template <typename TW>
__global__ void __launch_bounds__(PN_THREADS) k_embed_norm(int H, int Q, int V, const int32_t *anchors,
                                                           int mask_id, float scale, const TW *embed,
                                                           const TW *mask_emb, float *x, OpOut out,
                                                           const TW *w, float eps, int *err) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ float red[PN_THREADS / 32];
  const int r = blockIdx.x, b = r / Q, j = r % Q;
  int tok = j == 0 ? anchors[b] : mask_id;
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) raise_err(err, DEV_ERR_TOKEN);
    tok = 0;
  }
  // a trained mask embedding, when given, replaces the word embedding of the mask rows
  const TW *__restrict__ src = (j > 0 && mask_emb) ? mask_emb : embed + (size_t)tok * H;
  float vals[4 * PN_VEC];
  // all loads first (the row is read once), then the stores
#pragma unroll
  for (int t = 0; t < 4 * PN_VEC; ++t) {
    const int i = threadIdx.x + t * PN_THREADS;
    vals[t] = i < H ? to_f(src[i]) * scale : 0.f;
  }
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < 4 * PN_VEC; ++t) {
    const int i = threadIdx.x + t * PN_THREADS;
    if (i < H) {
      x[(size_t)r * H + i] = vals[t];
      ss += vals[t] * vals[t];
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < PN_THREADS / 32; ++i) tot += red[i];
  const float rs = rsqrtf(tot / (float)H + eps);
#pragma unroll
  for (int t = 0; t < 4 * PN_VEC; ++t) {
    const int i = threadIdx.x + t * PN_THREADS;
    if (i < H) write_op(out, (size_t)r * H + i, vals[t] * rs * to_f(w[i]));
  }
}

cudaError_t launch_embed_norm(int dtype, const ModelDims &m, int B, const int32_t *anchors, int mask_id,
                              const void *embed, const void *mask_emb, float *x, OpOut out, const void *w,
                              int *err, cudaStream_t s) {
  if (m.H > 4 * PN_VEC * PN_THREADS) return cudaErrorInvalidValue;
  dim3 g(B * m.Q());
  if (dtype)
    return launch_pdl(k_embed_norm<bf16>, g, dim3(PN_THREADS), 0, s, m.H, m.Q(), m.V, anchors, mask_id,
                      m.emb_scale, (const bf16 *)embed, (const bf16 *)mask_emb, x, out, (const bf16 *)w,
                      m.eps, err);
  return launch_pdl(k_embed_norm<float>, g, dim3(PN_THREADS), 0, s, m.H, m.Q(), m.V, anchors, mask_id,
                    m.emb_scale, (const float *)embed, (const float *)mask_emb, x, out, (const float *)w,
                    m.eps, err);
}

// ---------------------------------------------------------------------- row gather
// Packs the counted rows of the target's verify blocks: out[f][r] = in[f][src[r]] for every
// feature tensor f; one CTA per (row, feature), 16-byte words when the row allows them.
struct RowPtrs { const void *p[8]; };

__global__ void k_gather_rows(int rows, long row_bytes, long out_stride, const int32_t *src, RowPtrs in,
                              uint8_t *out) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, f = blockIdx.y;
  const uint8_t *a = (const uint8_t *)in.p[f] + (size_t)src[r] * row_bytes;
  uint8_t *d = out + (size_t)f * out_stride + (size_t)r * row_bytes;
  if (((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(d) | (uintptr_t)row_bytes) & 15) == 0) {
    for (long i = threadIdx.x; i < row_bytes / 16; i += blockDim.x)
      reinterpret_cast<uint4 *>(d)[i] = reinterpret_cast<const uint4 *>(a)[i];
  } else {
    for (long i = threadIdx.x; i < row_bytes; i += blockDim.x) d[i] = a[i];
  }
}

cudaError_t launch_gather_rows(int n_feat, int rows, long row_bytes, const int32_t *src,
                               const void *const *in, void *out, long out_stride, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (n_feat < 1 || n_feat > 8) return cudaErrorInvalidValue;
  RowPtrs ip{};
  for (int f = 0; f < n_feat; ++f) ip.p[f] = in[f];
  return launch_pdl(k_gather_rows, dim3((unsigned)rows, (unsigned)n_feat), dim3(256), 0, s, rows, row_bytes,
                    out_stride, src, ip, (uint8_t *)out);
}

}  // namespace dflash
