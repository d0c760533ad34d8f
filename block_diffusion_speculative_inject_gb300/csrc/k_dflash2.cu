// DFlash 2 modules ("DFlash 2 块扩散投机解码技术详解" §3.1 the path selector, §3.2.3 the
// two-tap dynamic depthwise convolution).
//
// Convolution over the K+1 block rows of each request (row t = m % (K+1) of row m):
//   y_t = k_t0 * x_t + k_t1 * x_{t-1},  x_{-1} = 0,
//   k_ti[c] = base[i][c] + corr[t][i*G + c/16],  corr = x P^T  (P [2G, H], G = H/16),
// the correction coming from a GEMM over the convolution's own input rows. Two kernels:
//   conv_in        on a sublayer's input: the input operand (the norm's output) -> the
//                  convolved operand of the sublayer's first GEMM;
//   conv_out_norm  on a sublayer's output (a GEMM product): x += conv(out), then the next
//                  RMSNorm as the next GEMM's operand (the post_norm step with the
//                  convolution folded in).
// to_op turns a GEMM product into an operand (the correction GEMM's input).
//
// Selector: per (request, position t) one CTA scores every (predecessor, candidate) pair,
//   T_t[a][b] = unary[t][b] + sum_r A(a)[r] g_t[r] B(b)[r],
// with predecessors the anchor (t = 0) or the candidates of t-1; a warp per request then
// walks the tables from the anchor.
#include <climits>

#include "../../include/dflash.h"
#include "kernels.h"

namespace dflash {

__device__ __forceinline__ float read_op(const OpOut &o, size_t idx) {
  if (o.lo) return __bfloat162float(((const bf16 *)o.hi)[idx]) + __bfloat162float(((const bf16 *)o.lo)[idx]);
  return ((const float *)o.hi)[idx];
}

// ------------------------------------------------------------------------- convolution, input side
template <typename TW>
__global__ void k_conv_in(int M, int Q, int H, OpOut in, const float *__restrict__ corr,
                          const TW *__restrict__ base, OpOut out) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)M * H) return;
  const int m = (int)(i / H), c = (int)(i % H), G = H / 16;
  const bool first = m % Q == 0;
  const float xt = read_op(in, i), xp = first ? 0.f : read_op(in, i - H);
  const float *cr = corr + (size_t)m * 2 * G;
  const float k0 = to_f(base[c]) + cr[c / 16], k1 = to_f(base[H + c]) + cr[G + c / 16];
  write_op(out, i, k0 * xt + k1 * xp);
}

cudaError_t launch_conv_in(int dtype, int M, int Q, int H, OpOut in, const float *corr, const void *base,
                           OpOut out, cudaStream_t s) {
  const long n = (long)M * H;
  if (n == 0) return cudaSuccess;
  if (H % 16) return cudaErrorInvalidValue;
  const dim3 g((unsigned)((n + 255) / 256));
  if (dtype)
    return launch_pdl(k_conv_in<bf16>, g, dim3(256), 0, s, M, Q, H, in, corr, (const bf16 *)base, out);
  return launch_pdl(k_conv_in<float>, g, dim3(256), 0, s, M, Q, H, in, corr, (const float *)base, out);
}

__global__ void k_to_op(long n, const float *__restrict__ src, OpOut out) {
  pdl_trigger();
  pdl_wait();
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) write_op(out, i, src[i]);
}

cudaError_t launch_to_op(long n, const float *src, OpOut out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(k_to_op, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, n, src, out);
}

// ------------------------------------------------------------------------- convolution, output side
// One 128-thread CTA per row (H <= 8192: 16 float4 per thread): x[m] += conv(y)[m], then
// RMSNorm(x[m]) * w as an operand; out_skip_k = K > 0 writes only the K mask rows of each
// block, to row b*K + j - 1 (the final norm).
constexpr int CV_THREADS = 128;
constexpr int CV_VEC = 16;

template <typename TW>
__global__ void __launch_bounds__(CV_THREADS) k_conv_out_norm(int M, int Q, int H, const float *__restrict__ y,
                                                              const float *__restrict__ corr,
                                                              const TW *__restrict__ base, float *x, OpOut out,
                                                              const TW *__restrict__ w, float eps, int out_skip_k) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[CV_THREADS / 32];
  const int m = blockIdx.x, n4 = H / 4, G = H / 16;
  const bool first = m % Q == 0;
  const float *cr = corr + (size_t)m * 2 * G;
  const float4 *yt = (const float4 *)(y + (size_t)m * H);
  const float4 *yp = first ? yt : (const float4 *)(y + (size_t)(m - 1) * H);
  float4 v[CV_VEC];
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < CV_VEC; ++t) {
    const int i = threadIdx.x + t * CV_THREADS;
    v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n4) {
      const int e = 4 * i;
      const float4 a = __ldg(yt + i), p = first ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldg(yp + i);
      const float c0 = cr[e / 16], c1 = cr[G + e / 16];     // the 4 channels share a group
      const float4 r = ((const float4 *)(x + (size_t)m * H))[i];
      v[t].x = r.x + ((to_f(base[e + 0]) + c0) * a.x + (to_f(base[H + e + 0]) + c1) * p.x);
      v[t].y = r.y + ((to_f(base[e + 1]) + c0) * a.y + (to_f(base[H + e + 1]) + c1) * p.y);
      v[t].z = r.z + ((to_f(base[e + 2]) + c0) * a.z + (to_f(base[H + e + 2]) + c1) * p.z);
      v[t].w = r.w + ((to_f(base[e + 3]) + c0) * a.w + (to_f(base[H + e + 3]) + c1) * p.w);
      ((float4 *)(x + (size_t)m * H))[i] = v[t];
      ss += v[t].x * v[t].x + v[t].y * v[t].y + v[t].z * v[t].z + v[t].w * v[t].w;
    }
  }
  int orow = m;
  if (out_skip_k > 0) {
    const int b = m / Q, j = m % Q;
    if (j == 0) return;                       // the anchor row yields no candidate
    orow = b * out_skip_k + j - 1;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < CV_THREADS / 32; ++i) tot += red[i];
  const float rs = rsqrtf(tot / (float)H + eps);
  const size_t o = (size_t)orow * H;
#pragma unroll
  for (int t = 0; t < CV_VEC; ++t) {
    const int i = threadIdx.x + t * CV_THREADS;
    if (i < n4) {
      const int e = 4 * i;
      write_op(out, o + e + 0, v[t].x * rs * to_f(w[e + 0]));
      write_op(out, o + e + 1, v[t].y * rs * to_f(w[e + 1]));
      write_op(out, o + e + 2, v[t].z * rs * to_f(w[e + 2]));
      write_op(out, o + e + 3, v[t].w * rs * to_f(w[e + 3]));
    }
  }
}

cudaError_t launch_conv_out_norm(int dtype, int M, int Q, int H, const float *y, const float *corr,
                                 const void *base, float *x, OpOut out, const void *w, float eps,
                                 int out_skip_k, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (H % 16 || H > CV_THREADS * 4 * CV_VEC) return cudaErrorInvalidValue;
  if (dtype)
    return launch_pdl(k_conv_out_norm<bf16>, dim3(M), dim3(CV_THREADS), 0, s, M, Q, H, y, corr,
                      (const bf16 *)base, x, out, (const bf16 *)w, eps, out_skip_k);
  return launch_pdl(k_conv_out_norm<float>, dim3(M), dim3(CV_THREADS), 0, s, M, Q, H, y, corr,
                    (const float *)base, x, out, (const float *)w, eps, out_skip_k);
}

// ------------------------------------------------------------------------- path selector
constexpr int SEL_THREADS = 256;
constexpr int SEL_MAX_R = 512;
constexpr int SEL_MAX_KC = 32;

__host__ __device__ inline size_t sel_smem(int kc, int r) { return (size_t)2 * kc * (r + 4) * sizeof(float); }

// tab [n][K][kc][kc]: row a = predecessor (t = 0: row 0 is the anchor), column b = candidate.
// Tokens outside [0, V) read as zero codebook rows.
template <typename TW>
__global__ void __launch_bounds__(SEL_THREADS) k_sel_table(int K, int kc, int r, int V, const int32_t *__restrict__ anchors,
                                                          const int32_t *__restrict__ cand_tok,
                                                          const float *__restrict__ unary,
                                                          const float *__restrict__ gate, const TW *__restrict__ pred,
                                                          const TW *__restrict__ succ, float *__restrict__ tab) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float4 sel_sm[];
  const int t = blockIdx.x, b = blockIdx.y, rs = r + 4;
  float *As = (float *)sel_sm, *Ws = As + (size_t)kc * rs;
  const int32_t *ct = cand_tok + ((size_t)b * K + t) * kc;
  const int32_t *cp = t > 0 ? ct - kc : nullptr;
  const int na = t > 0 ? kc : 1;
  const float *g = gate + ((size_t)b * K + t) * r;
  for (int i = threadIdx.x; i < na * r; i += SEL_THREADS) {
    const int a = i / r, c = i % r;
    const int tok = t > 0 ? cp[a] : anchors[b];
    As[a * rs + c] = (tok >= 0 && tok < V) ? to_f(pred[(size_t)tok * r + c]) : 0.f;
  }
  for (int i = threadIdx.x; i < kc * r; i += SEL_THREADS) {
    const int j = i / r, c = i % r, tok = ct[j];
    Ws[j * rs + c] = (tok >= 0 && tok < V) ? g[c] * to_f(succ[(size_t)tok * r + c]) : 0.f;
  }
  __syncthreads();
  const float *u = unary + ((size_t)b * K + t) * kc;
  float *out = tab + ((size_t)b * K + t) * kc * kc;
  for (int p = threadIdx.x; p < na * kc; p += SEL_THREADS) {
    const int a = p / kc, j = p % kc;
    const float4 *x4 = (const float4 *)(As + a * rs), *w4 = (const float4 *)(Ws + j * rs);
    float acc = 0.f;
    for (int c = 0; c < r / 4; ++c) {
      const float4 x = x4[c], w = w4[c];
      acc = fmaf(x.x, w.x, acc);
      acc = fmaf(x.y, w.y, acc);
      acc = fmaf(x.z, w.z, acc);
      acc = fmaf(x.w, w.w, acc);
    }
    out[a * kc + j] = u[j] + acc;
  }
}

// One warp per request: lane j holds candidate j's score; the best (first on ties) is taken.
__global__ void k_sel_walk(int n, int K, int kc, const int32_t *__restrict__ cand_tok, const float *__restrict__ tab,
                           int32_t *__restrict__ selected, float *__restrict__ scores) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  if (b >= n) return;
  int prev = 0;
  for (int t = 0; t < K; ++t) {
    const float *row = tab + (((size_t)b * K + t) * kc + prev) * kc;
    float v = lane < kc ? row[lane] : -INFINITY;
    if (scores && lane < kc) scores[((size_t)b * K + t) * kc + lane] = v;
    int idx = lane < kc ? lane : SEL_MAX_KC;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ov > v || (ov == v && oi < idx)) {
        v = ov;
        idx = oi;
      }
    }
    if (lane == 0) selected[(size_t)b * K + t] = cand_tok[((size_t)b * K + t) * kc + idx];
    prev = idx;
  }
}

// Sampling mode: position t's candidates get q = softmax(T_t[prev] / temperature); the token
// is drawn by inverse CDF in vocabulary order against u[b][t] (the first candidate, by token
// id, whose running mass exceeds u times the total; if rounding leaves none, the largest
// token with q > 0); q goes out as lists of stride SMP_K (q_tok, q_p, q_n), the form the
// sampling verification reads.
__global__ void k_sel_walk_sample(int n, int K, int kc, const int32_t *__restrict__ cand_tok,
                                  const float *__restrict__ tab, float temperature, const float *__restrict__ u,
                                  int32_t *__restrict__ selected, int32_t *__restrict__ q_tok,
                                  float *__restrict__ q_p, int32_t *__restrict__ q_n) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  if (b >= n) return;
  int prev = 0;
  for (int t = 0; t < K; ++t) {
    const size_t bt = (size_t)b * K + t;
    const float *row = tab + (bt * kc + prev) * kc;
    const bool in = lane < kc;
    const float v = in ? row[lane] : -INFINITY;
    const int32_t tok = in ? cand_tok[bt * kc + lane] : INT_MAX;
    const float mx = warp_max(v);
    const float e = in ? expf((v - mx) / temperature) : 0.f;
    const float q = e / warp_sum(e);
    q_tok[bt * SMP_K + lane] = in ? tok : -1;
    q_p[bt * SMP_K + lane] = q;
    if (lane == 0) q_n[bt] = kc;
    float before = 0.f;                      // mass of the candidates with a smaller token id
    for (int i = 0; i < 32; ++i) {
      const float qi = __shfl_sync(0xffffffffu, q, i);
      const int32_t ti = __shfl_sync(0xffffffffu, tok, i);
      if (ti < tok) before += qi;
    }
    const float thr = u[bt] * warp_sum(q);
    const bool hit = in && q > 0.f && before + q > thr;
    int32_t pick = __reduce_min_sync(0xffffffffu, hit ? tok : INT_MAX);
    if (pick == INT_MAX) pick = __reduce_max_sync(0xffffffffu, in && q > 0.f ? tok : INT_MIN);
    prev = max(0, __ffs(__ballot_sync(0xffffffffu, tok == pick)) - 1);   // 0 if scores were NaN
    if (lane == 0) selected[bt] = pick;
  }
}

cudaError_t launch_select_path(int dtype, int n, int K, int kc, int r, int V, const int32_t *anchors,
                               const int32_t *cand_tok, const float *unary, const float *gate, const void *pred,
                               const void *succ, float *tab, int32_t *selected, float *scores, cudaStream_t s,
                               const SelSample *smp) {
  if (n == 0) return cudaSuccess;
  if (smp && !(smp->temperature > 0.f)) return cudaErrorInvalidValue;
  if (K < 1 || kc < 1 || kc > SEL_MAX_KC || r < 32 || r > SEL_MAX_R || r % 32) return cudaErrorInvalidValue;
  static bool smem_opt_in[2] = {false, false};
  const size_t smem = sel_smem(kc, r);
  cudaError_t e;
  if (!smem_opt_in[dtype ? 1 : 0]) {
    e = dtype ? cudaFuncSetAttribute(k_sel_table<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sel_smem(SEL_MAX_KC, SEL_MAX_R))
              : cudaFuncSetAttribute(k_sel_table<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sel_smem(SEL_MAX_KC, SEL_MAX_R));
    if (e != cudaSuccess) return e;
    smem_opt_in[dtype ? 1 : 0] = true;
  }
  const dim3 g(K, n);
  e = dtype ? launch_pdl(k_sel_table<bf16>, g, dim3(SEL_THREADS), smem, s, K, kc, r, V, anchors, cand_tok,
                         unary, gate, (const bf16 *)pred, (const bf16 *)succ, tab)
            : launch_pdl(k_sel_table<float>, g, dim3(SEL_THREADS), smem, s, K, kc, r, V, anchors, cand_tok,
                         unary, gate, (const float *)pred, (const float *)succ, tab);
  if (e != cudaSuccess) return e;
  if (smp)
    return launch_pdl(k_sel_walk_sample, dim3(n), dim3(32), 0, s, n, K, kc, cand_tok, tab, smp->temperature, smp->u,
                      selected, smp->q_tok, smp->q_p, smp->q_n);
  return launch_pdl(k_sel_walk, dim3(n), dim3(32), 0, s, n, K, kc, cand_tok, tab, selected, scores);
}

}  // namespace dflash

using namespace dflash;

extern "C" dflash_status dflash_select_path(void *stream, int32_t n_req, int32_t K, int32_t kc, int32_t r,
                                            int32_t vocab, dflash_dtype dtype, const int32_t *anchors, const int32_t *cand_tok,
                                            const float *unary, const float *gate, const void *pred_codebook,
                                            const void *succ_codebook, int32_t *selected, float *scores) {
  if (n_req < 0 || K < 1 || K > 31 || kc < 1 || kc > SEL_MAX_KC || r < 32 || r > SEL_MAX_R || r % 32 ||
      vocab < 1 || (dtype != DFLASH_F32 && dtype != DFLASH_BF16))
    return DFLASH_ERR_INVALID_ARG;
  if (n_req == 0) return DFLASH_OK;
  if (!anchors || !cand_tok || !unary || !gate || !pred_codebook || !succ_codebook || !selected)
    return DFLASH_ERR_INVALID_ARG;
  float *tab = nullptr;
  if (cudaMallocAsync((void **)&tab, (size_t)n_req * K * kc * kc * sizeof(float), (cudaStream_t)stream) !=
      cudaSuccess)
    return DFLASH_ERR_CUDA;
  cudaError_t e = launch_select_path(dtype == DFLASH_BF16, n_req, K, kc, r, vocab, anchors, cand_tok, unary, gate,
                                     pred_codebook, succ_codebook, tab, selected, scores, (cudaStream_t)stream);
  cudaFreeAsync(tab, (cudaStream_t)stream);
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

extern "C" dflash_status dflash_select_sample(void *stream, int32_t n_req, int32_t K, int32_t kc, int32_t r,
                                              int32_t vocab, dflash_dtype dtype, float temperature,
                                              const int32_t *anchors, const int32_t *cand_tok, const float *unary,
                                              const float *gate, const void *pred_codebook,
                                              const void *succ_codebook, const float *u, int32_t *selected,
                                              int32_t *q_tok, float *q_p, int32_t *q_n) {
  if (n_req < 0 || K < 1 || K > 31 || kc < 1 || kc > SEL_MAX_KC || r < 32 || r > SEL_MAX_R || r % 32 ||
      vocab < 1 || (dtype != DFLASH_F32 && dtype != DFLASH_BF16) || !(temperature > 0.f))
    return DFLASH_ERR_INVALID_ARG;
  if (n_req == 0) return DFLASH_OK;
  if (!anchors || !cand_tok || !unary || !gate || !pred_codebook || !succ_codebook || !u || !selected || !q_tok ||
      !q_p || !q_n)
    return DFLASH_ERR_INVALID_ARG;
  float *tab = nullptr;
  if (cudaMallocAsync((void **)&tab, (size_t)n_req * K * kc * kc * sizeof(float), (cudaStream_t)stream) !=
      cudaSuccess)
    return DFLASH_ERR_CUDA;
  const SelSample smp{temperature, u, q_tok, q_p, q_n};
  cudaError_t e = launch_select_path(dtype == DFLASH_BF16, n_req, K, kc, r, vocab, anchors, cand_tok, unary, gate,
                                     pred_codebook, succ_codebook, tab, selected, nullptr, (cudaStream_t)stream,
                                     &smp);
  cudaFreeAsync(tab, (cudaStream_t)stream);
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}
