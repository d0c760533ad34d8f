// Split-KV GQA attention of the query block over a paged, ragged context.
//
// Per request b the keys are [context positions 0..ctx_len-1 (paged cache) ; the block's
// own K+1 keys], with no mask anywhere ("LLM的推理加速-DFlash" 关键创新 Step 3: target
// features first, block keys after; "DFlash：把串行 Draft 变成并行“填空”" §5.3: non-causal).
// A split CTA handles (split s, kv head, request b): its rows are the G = nq/nkv query heads
// sharing that kv head times the K+1 block rows, its keys the context range
// [s*split_len, min((s+1)*split_len, ctx_len)) (page aligned). It writes an unnormalised
// accumulator, the running max and the running sum, with scores in log2 units
// (q.k * log2(e) / sqrt(hd)). The combine kernel adds the block's own K+1 keys (fp32, from
// the q/k/v rows) and merges the splits in a fixed order. Splits run on the tensor cores
// (k_attention_tc.cu) for bf16 caches with head_dim 128, on the FFMA cores otherwise.
#include "attn_combine.cuh"
#include "kernels.h"

namespace dflash {

constexpr int AT_KT = 32;       // keys per tile (one per lane for the scores)
constexpr int AT_MAXR = 128;    // rows per CTA (G * (K+1))
constexpr int AT_PAGE = 64;

template <typename T, int HD>
__global__ void __launch_bounds__(256) k_attn_split(
    int L, int nq, int nkv, int Q, int layer, const float *qkv, const T *pool,
    const int32_t *ctx_len, const int32_t *n_split, const int32_t *split_len,
    const int32_t *page_off, const int32_t *pages, int max_split, float scale, float *part_o,
    float *part_ml) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  extern __shared__ float sm[];
  float *qs = sm;                              // [R][HD]
  float *ks = qs + AT_MAXR * HD;               // [KT][HD+1]
  float *vs = ks + AT_KT * (HD + 1);           // [KT][HD]
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  if (s >= n_split[b]) return;
  const int G = nq / nkv, R = G * Q;
  const int qkv_dim = (nq + 2 * nkv) * HD;
  const int n_ctx = ctx_len[b];
  const int k_begin = s * split_len[b];
  const int k_end = min(k_begin + split_len[b], n_ctx);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t row0 = (size_t)b * Q;
  const int32_t *pg = pages + page_off[b];

  for (int i = tid; i < R * HD; i += 256) {
    int r = i / HD, d = i % HD;
    int g = r / Q, j = r % Q;
    qs[i] = qkv[(row0 + j) * qkv_dim + (size_t)(kvh * G + g) * HD + d];
  }

  constexpr int DPL = HD / 32;                 // dims per lane in the PV accumulator
  constexpr int RPW = AT_MAXR / 8;             // most rows per warp
  float m_run[RPW], l_run[RPW], acc[RPW][DPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[i][d] = 0.f;
  }

  for (int t0 = k_begin; t0 < k_end; t0 += AT_KT) {
    __syncthreads();
    for (int i = tid; i < AT_KT * HD; i += 256) {
      int kk = i / HD, d = i % HD;
      int key = t0 + kk;
      float kval = 0.f, vval = 0.f;
      if (key < k_end) {
        int page = pg[key / AT_PAGE], off = key % AT_PAGE;
        kval = to_f(pool[kv_block(page, layer, 0, kvh, L, nkv, HD) + (size_t)off * HD + d]);
        vval = to_f(pool[kv_block(page, layer, 1, kvh, L, nkv, HD) + (size_t)d * AT_PAGE + off]);
      }
      ks[kk * (HD + 1) + d] = kval;
      vs[kk * HD + d] = vval;
    }
    __syncthreads();
    const bool valid = t0 + lane < k_end;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      int r = warp + 8 * i;
      if (r >= R) continue;
      const float *qr = qs + r * HD;
      const float *kr = ks + lane * (HD + 1);
      float sc = 0.f;
#pragma unroll 8
      for (int d = 0; d < HD; ++d) sc = fmaf(qr[d], kr[d], sc);
      sc = valid ? sc * scale : -INFINITY;
      float mt = warp_max(sc);
      float m_new = fmaxf(m_run[i], mt);
      float p = valid ? exp2f(sc - m_new) : 0.f;
      float corr = exp2f(m_run[i] - m_new);     // exp2(-inf) = 0 on the first tile
      l_run[i] = l_run[i] * corr + warp_sum(p);
      m_run[i] = m_new;
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[i][d] *= corr;
      for (int kk = 0; kk < AT_KT; ++kk) {
        float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[i][d] = fmaf(pk, vs[kk * HD + lane + 32 * d], acc[i][d]);
      }
    }
  }

  // partial outputs: part_o[((b*Q + j)*nq + h)*max_split + s][HD], part_ml[...][2]
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    int r = warp + 8 * i;
    if (r >= R) continue;
    int g = r / Q, j = r % Q;
    size_t idx = (((size_t)b * Q + j) * nq + (kvh * G + g)) * max_split + s;
#pragma unroll
    for (int d = 0; d < DPL; ++d) part_o[idx * HD + lane + 32 * d] = acc[i][d];
    if (lane == 0) {
      part_ml[idx * 2] = m_run[i];
      part_ml[idx * 2 + 1] = l_run[i];
    }
  }
}

// One CTA per (kv head, request b, chunk of 8 rows), one warp per row (rows are the G query
// heads of the kv head times the K+1 block rows). The block's own K+1 keys and values (fp32
// q/k/v rows) are staged in shared memory; each lane scores one block key against the warp's
// q row (also staged), the context splits' (max, sum) are read one per lane, and the merged
// output is accumulated with each lane owning hd/32 dimensions:
//   o = (sum_s acc_s 2^(m_s - M) + sum_kk 2^(s_kk - M) v_kk) / (sum_s l_s 2^(m_s - M) + sum_kk 2^(s_kk - M))
// The order of every sum is fixed.
constexpr int CB_ROWS = 8;
constexpr int CB_MAX_SPLIT = 16;   // the host plans at most this many context splits

template <int HD, int MS>   // MS >= the batch's largest split count
__global__ void __launch_bounds__(32 * CB_ROWS) k_attn_combine(int nq, int nkv, int Q,
                                                               const int32_t *n_split, int max_split,
                                                               const float *part_o,
                                                               const float *part_ml, const float *qkv,
                                                               float scale_log2, int causal, OpOut o) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ float ks[32 * CombineSmem<HD>::KP];
  __shared__ float vs[32 * HD];
  __shared__ float qs[CB_ROWS][HD];
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int R = (nq / nkv) * Q;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const CombineSmem<HD> sm{ks, vs};
  const int r = blockIdx.z * CB_ROWS + warp;
  const int ns = n_split[b];
  // the block K/V first (its registers are free again before the row's loads go out)
  stage_block_kv<HD>(b, kvh, nq, nkv, Q, qkv, sm, tid, 32 * CB_ROWS);
  CombineRow<HD, MS> cr;
  if (r < R) combine_load<HD, MS, false>(cr, r, b, kvh, nq, nkv, Q, ns, max_split, part_o, part_ml, qkv, qs[warp], lane);
  __syncthreads();
  if (r >= R) return;
  combine_finish<HD, MS>(cr, r, b, kvh, nq, nkv, Q, ns, scale_log2, causal, o, sm, qs[warp], lane);
}

template <typename T, int HD>
static cudaError_t attn_impl(const ModelDims &m, const DraftBatch &bt, int layer, const float *qkv,
                             const void *pool, float *part_o, float *part_ml, OpOut o,
                             const AttnMaps *maps, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  if (bt.max_split > CB_MAX_SPLIT) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  if (bt.max_split > 0) {
    if (maps && maps->valid && HD == 128 && sizeof(T) == 2) {
      e = launch_attn_split_tc(m, bt, layer, qkv, maps, scale_log2, part_o, part_ml, s);
    } else {
      size_t smem = (size_t)(AT_MAXR * HD + AT_KT * (HD + 1) + AT_KT * HD) * sizeof(float);
      e = cudaFuncSetAttribute(k_attn_split<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e != cudaSuccess) return e;
      dim3 g(bt.max_split, m.nkv, bt.B);
      e = launch_pdl(k_attn_split<T, HD>, g, dim3(256), smem, s, m.L, m.nq, m.nkv, m.Q(), layer, qkv,
                     (const T *)pool, bt.ctx_len, bt.n_split, bt.split_len, bt.page_off, bt.pages,
                     bt.max_split, scale_log2, part_o, part_ml);
    }
    if (e != cudaSuccess) return e;
  }
  const int R = (m.nq / m.nkv) * m.Q();
  dim3 g2(m.nkv, bt.B, (R + CB_ROWS - 1) / CB_ROWS);
  auto go = [&](auto kern) {
    return launch_pdl(kern, g2, dim3(32 * CB_ROWS), 0, s, m.nq, m.nkv, m.Q(), bt.n_split, bt.max_split,
                      (const float *)part_o, (const float *)part_ml, qkv, scale_log2, m.causal, o);
  };
  // register room for the partial outputs follows the largest split count
  if (bt.max_split <= 2) return go(k_attn_combine<HD, 2>);
  if (bt.max_split <= 4) return go(k_attn_combine<HD, 4>);
  if (bt.max_split <= 8) return go(k_attn_combine<HD, 8>);
  return go(k_attn_combine<HD, CB_MAX_SPLIT>);
}

cudaError_t launch_attention(int dtype, const ModelDims &m, const DraftBatch &bt, int layer,
                             const float *qkv, const void *pool, float *part_o, float *part_ml,
                             OpOut o, const AttnMaps *maps, cudaStream_t s) {
  if (bt.B <= 0) return cudaSuccess;
  if (m.hd == 128)
    return dtype ? attn_impl<bf16, 128>(m, bt, layer, qkv, pool, part_o, part_ml, o, maps, s)
                 : attn_impl<float, 128>(m, bt, layer, qkv, pool, part_o, part_ml, o, maps, s);
  if (m.hd == 64)
    return dtype ? attn_impl<bf16, 64>(m, bt, layer, qkv, pool, part_o, part_ml, o, maps, s)
                 : attn_impl<float, 64>(m, bt, layer, qkv, pool, part_o, part_ml, o, maps, s);
  return cudaErrorInvalidValue;
}

}  // namespace dflash
