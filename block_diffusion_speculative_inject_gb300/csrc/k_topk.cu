// Top-k selection (values descending, equal values ordered by the lower vocabulary index;
// the argmax is the first entry). Two entry points share one block-wide selector:
//   launch_topk        a row of fp32 logits [V] per CTA (the FFMA path);
//   launch_topk_merge  the per-tile candidates written by the tensor-core LM-head GEMM
//                      epilogue, [tiles][rows][k] (value, index) per row, merged per CTA.
// Each thread keeps a sorted register list of its best TK candidates over a strided slice,
// then the block merges the 256 sorted lists by k rounds of a block-wide best-head pick.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "../../include/dflash.h"
#include "kernels.h"

namespace dflash {

constexpr int TK = 32;         // register list length (>= any requested k)
constexpr int TK_THREADS = 256;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void list_init(float (&lv)[TK], int (&li)[TK]) {
#pragma unroll
  for (int q = 0; q < TK; ++q) {
    lv[q] = -INFINITY;
    li[q] = 0x7fffffff;
  }
}

// Insertion into a thread's sorted register list (unrolled: registers only).
__device__ __forceinline__ void list_insert(float (&lv)[TK], int (&li)[TK], float v, int id) {
  if (!better(v, id, lv[TK - 1], li[TK - 1])) return;
  float cv = v;
  int ci = id;
#pragma unroll
  for (int q = 0; q < TK; ++q) {
    const bool b = better(cv, ci, lv[q], li[q]);
    const float tv = lv[q];
    const int ti = li[q];
    lv[q] = b ? cv : lv[q];
    li[q] = b ? ci : li[q];
    cv = b ? tv : cv;
    ci = b ? ti : ci;
  }
}

__device__ __forceinline__ void block_merge(float (&lv)[TK], int (&li)[TK], int k, int32_t *argmax_out,
                                            int32_t *idx_out, float *val_out);

template <typename Get>
__device__ __forceinline__ void block_topk(int n, int k, Get get, int32_t *argmax_out,
                                           int32_t *idx_out, float *val_out) {
  float lv[TK];
  int li[TK];
  list_init(lv, li);
  for (int i = threadIdx.x; i < n; i += TK_THREADS) {
    float v;
    int id;
    get(i, v, id);
    list_insert(lv, li, v, id);
  }
  block_merge(lv, li, k, argmax_out, idx_out, val_out);
}

// Block-wide merge of the threads' sorted lists into the k best (value desc, index asc).
__device__ __forceinline__ void block_merge(float (&lv)[TK], int (&li)[TK], int k, int32_t *argmax_out,
                                            int32_t *idx_out, float *val_out) {
  const int tid = threadIdx.x;
  // merge: each round every thread offers its current head; warps reduce by shuffles, the
  // eight warp winners through shared memory; the owner of the block winner advances
  __shared__ float wv_s[TK_THREADS / 32];
  __shared__ int wi_s[TK_THREADS / 32], wt_s[TK_THREADS / 32];
  __shared__ int win_t;
  const int lane = tid & 31, warp = tid >> 5;
  int head = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < TK; ++q)
      if (q == head) {
        bv = lv[q];
        bi = li[q];
      }
    int bt = tid;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int ot = __shfl_xor_sync(0xffffffffu, bt, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
        bt = ot;
      }
    }
    if (lane == 0) {
      wv_s[warp] = bv;
      wi_s[warp] = bi;
      wt_s[warp] = bt;
    }
    __syncthreads();
    if (warp == 0) {
      float v = lane < TK_THREADS / 32 ? wv_s[lane] : -INFINITY;
      int i = lane < TK_THREADS / 32 ? wi_s[lane] : 0x7fffffff;
      int t = lane < TK_THREADS / 32 ? wt_s[lane] : 0;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        const int ot = __shfl_xor_sync(0xffffffffu, t, o);
        if (better(ov, oi, v, i)) {
          v = ov;
          i = oi;
          t = ot;
        }
      }
      if (lane == 0) {
        win_t = t;
        if (r == 0) *argmax_out = i;
        if (idx_out) {
          idx_out[r] = i;
          val_out[r] = v;
        }
      }
    }
    __syncthreads();
    if (tid == win_t) ++head;
  }
}

constexpr int ROWS_CAP = 2048;   // gathered candidates per row before falling back

// Online softmax normaliser: (m, s) stands for s * exp(m); merging keeps the larger max.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float M = fmaxf(m, m2);
  s = s * expf(m - M) + s2 * expf(m2 - M);
  m = M;
}

// The block's log(sum exp): every thread holds a partial (m, s); the result (m + log s) is
// returned to all threads. scratch: 2 * (TK_THREADS / 32) floats of shared memory.
__device__ __forceinline__ float block_lse(float m, float s, float *scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  __syncthreads();
  if (lane == 0) {
    scratch[2 * warp] = m;
    scratch[2 * warp + 1] = s;
  }
  __syncthreads();
  float M = -INFINITY, S = 0.f;
  for (int w = 0; w < TK_THREADS / 32; ++w) lse_merge(M, S, scratch[2 * w], scratch[2 * w + 1]);
  return M + logf(S);
}

// The body of the row selection for one row x[V], run by the whole CTA; the shared scratch
// (tmax, pool, n_pool, thr) is the caller's. Writes argmax_out[0] (if non-null) and the
// sorted best k to idx_out / val_out (if non-null); they may point to shared memory.
__device__ __forceinline__ void row_select(const float *x, int V, int k, float *tmax, int2 *pool,
                                           int *n_pool, float *thr, int32_t *argmax_out,
                                           int32_t *idx_out, float *val_out, float *lse_out = nullptr,
                                           float *lse_scratch = nullptr) {
  const bool vec = (V & 3) == 0 && ((uintptr_t)x & 15u) == 0;
  const int n4 = V / 4;
  const float4 *x4 = (const float4 *)x;
  auto scan = [&](auto &&visit) {
    if (vec) {
      for (int b = 0; b < n4; b += TK_THREADS * 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = b + threadIdx.x + j * TK_THREADS;
          v[j] = i < n4 ? x4[i] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = 4 * (b + threadIdx.x + j * TK_THREADS);
          if (i < V) {
            visit(v[j].x, i);
            visit(v[j].y, i + 1);
            visit(v[j].z, i + 2);
            visit(v[j].w, i + 3);
          }
        }
      }
    } else {
      for (int i = threadIdx.x; i < V; i += TK_THREADS) visit(x[i], i);
    }
  };
  // pass 1: per-thread maximum (and, when asked, the running softmax normaliser)
  float mv = -INFINITY;
  if (lse_out) {
    float s = 0.f;
    scan([&](float v, int) {
      if (v == -INFINITY) return;
      if (v > mv) {
        s = (mv == -INFINITY ? 0.f : s * expf(mv - v)) + 1.f;
        mv = v;
      } else {
        s += expf(v - mv);
      }
    });
    const float l = block_lse(mv, s, lse_scratch);
    if (threadIdx.x == 0) *lse_out = l;
  } else {
    scan([&](float v, int) { mv = fmaxf(mv, v); });
  }
  tmax[threadIdx.x] = mv;
  if (threadIdx.x == 0) *n_pool = 0;
  __syncthreads();
  {
    // stable rank of this thread's maximum among all; rank k - 1 is the bound
    int rank = 0;
    for (int j = 0; j < TK_THREADS; ++j) {
      const float u = tmax[j];
      rank += (u > mv) | ((u == mv) & (j < (int)threadIdx.x));
    }
    if (rank == k - 1) *thr = mv;
  }
  __syncthreads();
  const float T = *thr;
  // pass 2: gather the values >= T
  scan([&](float v, int i) {
    if (v >= T) {
      const int slot = atomicAdd(n_pool, 1);
      if (slot < ROWS_CAP) pool[slot] = make_int2(__float_as_int(v), i);
    }
  });
  __syncthreads();
  const int np = *n_pool;
  if (np <= ROWS_CAP) {
    for (int i = threadIdx.x; i < np; i += TK_THREADS) {
      const int2 c = pool[i];
      const float v = __int_as_float(c.x);
      int rank = 0;
      for (int j = 0; j < np; ++j) {
        const int2 d = pool[j];
        rank += better(__int_as_float(d.x), d.y, v, c.y);
      }
      if (rank < k) {
        if (rank == 0 && argmax_out) *argmax_out = c.y;
        if (idx_out) idx_out[rank] = c.y;
        if (val_out) val_out[rank] = v;
      }
    }
  } else {
    int32_t dummy;
    block_topk(V, k, [&](int i, float &v, int &id) { v = x[i]; id = i; },
               argmax_out ? argmax_out : &dummy, idx_out, val_out);
  }
}

// Two passes over the row: (1) every thread's maximum; the k-th best of those maxima is a
// lower bound T of the row's k-th best value (k threads each hold a value >= T); (2) the
// values >= T (a few more than k) are gathered in shared memory and placed by rank: a
// value's output slot is the number of gathered values that beat it. If more than ROWS_CAP
// values reach T (ties), the block-wide list selector ranks the row instead. CTA b takes
// rows b, b + gridDim.x, ...
__global__ void __launch_bounds__(TK_THREADS, 2) k_topk_rows(int rows, int V, int k, const float *logits,
                                                          int32_t *argmax, int32_t *topk_idx,
                                                          float *topk_val, float *lse) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ float tmax[TK_THREADS];
  __shared__ int2 pool[ROWS_CAP];
  __shared__ int n_pool;
  __shared__ float thr;
  __shared__ float lse_scratch[2 * (TK_THREADS / 32)];
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    row_select(logits + (size_t)row * V, V, k, tmax, pool, &n_pool, &thr, argmax + row,
               topk_idx ? topk_idx + (size_t)row * k : nullptr, topk_val ? topk_val + (size_t)row * k : nullptr,
               lse ? lse + row : nullptr, lse_scratch);
    __syncthreads();                   // the shared scratch is reused by the next row
  }
}

// Merge of per-tile sorted candidate lists (each tile's list is its best k in order). With at
// least k tiles, the k-th best of the tiles' first candidates is a lower bound T of the
// row's k-th best value (those k tiles each hold a value >= T), so only candidates >= T can
// be in the result, and only tiles whose first candidate is >= T (about k of them) hold
// any. T comes from warp-level selection rounds (no block barriers); the gathered
// candidates are placed by rank: a candidate's output slot is the number of gathered
// candidates that beat it (value desc, index asc: a strict order, so slots are distinct).
// (With fewer than k tiles, more than MERGE_TILES tiles, or more than MERGE_CAP gathered
// candidates, the block-wide selector ranks every candidate instead.)
constexpr int MERGE_CAP = 1024;
constexpr int MERGE_PER_THREAD = 8;
constexpr int MERGE_TILES = MERGE_PER_THREAD * TK_THREADS;

__global__ void __launch_bounds__(TK_THREADS) k_topk_merge(int tiles, int rows, int k,
                                                           const int2 *cand, int32_t *argmax,
                                                           int32_t *topk_idx, float *topk_val,
                                                           const float2 *lse_part, float *lse) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ int2 pool[MERGE_CAP];
  __shared__ int n_pool;
  __shared__ float warp_best[TK_THREADS / 32][TK];
  __shared__ float thr;
  __shared__ float lse_scratch[2 * (TK_THREADS / 32)];
  if (lse) {
    // the row's softmax normaliser from the tiles' (max, sum exp) partials
    float m = -INFINITY, sum = 0.f;
    for (int t = threadIdx.x; t < tiles; t += TK_THREADS) {
      const float2 pt = lse_part[(size_t)t * rows + blockIdx.x];
      lse_merge(m, sum, pt.x, pt.y);
    }
    const float l = block_lse(m, sum, lse_scratch);
    if (threadIdx.x == 0) lse[blockIdx.x] = l;
  }
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto at = [&](int t, int j) { return cand[((size_t)t * rows + row) * k + j]; };
  int32_t *oi = topk_idx ? topk_idx + (size_t)row * k : nullptr;
  float *ov = topk_val ? topk_val + (size_t)row * k : nullptr;
  auto rank_all = [&]() {
    block_topk(tiles * k, k,
               [&](int i, float &v, int &id) {
                 const int2 c = at(i / k, i % k);
                 v = __int_as_float(c.x);
                 id = c.y;
               },
               argmax + row, oi, ov);
  };
  if (tiles < k || tiles > MERGE_TILES) {
    rank_all();
    return;
  }
  // 1) this thread's tiles' first values; per warp the k best of them by argmax rounds
  float first[MERGE_PER_THREAD];
#pragma unroll
  for (int j = 0; j < MERGE_PER_THREAD; ++j) {
    const int t = threadIdx.x + j * TK_THREADS;
    first[j] = t < tiles ? __int_as_float(at(t, 0).x) : -INFINITY;
  }
  {
    float rest[MERGE_PER_THREAD];
#pragma unroll
    for (int j = 0; j < MERGE_PER_THREAD; ++j) rest[j] = first[j];
    for (int r = 0; r < k; ++r) {
      float bv = rest[0];
      int bj = 0;
#pragma unroll
      for (int j = 1; j < MERGE_PER_THREAD; ++j)
        if (rest[j] > bv) {
          bv = rest[j];
          bj = j;
        }
      float wv = bv;
      int wl = lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov2 = __shfl_xor_sync(0xffffffffu, wv, o);
        const int ol = __shfl_xor_sync(0xffffffffu, wl, o);
        if (ov2 > wv || (ov2 == wv && ol < wl)) {
          wv = ov2;
          wl = ol;
        }
      }
      if (lane == wl) {
#pragma unroll
        for (int j = 0; j < MERGE_PER_THREAD; ++j)
          if (j == bj) rest[j] = -INFINITY;
      }
      if (lane == 0) warp_best[warp][r] = wv;
    }
  }
  if (threadIdx.x == 0) n_pool = 0;
  __syncthreads();
  // 2) T = the k-th best of the warps' k best values (the k-th best tile first overall)
  const int nw = (TK_THREADS / 32) * k;
  if (threadIdx.x < nw) {
    const float v = warp_best[threadIdx.x / k][threadIdx.x % k];
    int above = 0, tie_before = 0;
    for (int i = 0; i < nw; ++i) {
      const float u = warp_best[i / k][i % k];
      above += u > v;
      tie_before += (u == v) & (i < (int)threadIdx.x);
    }
    if (above + tie_before == k - 1) thr = v;
  }
  __syncthreads();
  const float T = thr;
  // 3) gather the candidates >= T of the tiles whose first is >= T
#pragma unroll
  for (int j = 0; j < MERGE_PER_THREAD; ++j) {
    const int t = threadIdx.x + j * TK_THREADS;
    if (t >= tiles || first[j] < T) continue;
    for (int q = 0; q < k; ++q) {
      const int2 c = at(t, q);
      if (__int_as_float(c.x) < T) break;            // the tile's list is sorted
      const int slot = atomicAdd(&n_pool, 1);
      if (slot < MERGE_CAP) pool[slot] = c;
    }
  }
  __syncthreads();
  const int np = n_pool;
  if (np > MERGE_CAP) {
    rank_all();
    return;
  }
  // 4) place by rank
  for (int i = threadIdx.x; i < np; i += TK_THREADS) {
    const int2 c = pool[i];
    const float v = __int_as_float(c.x);
    int rank = 0;
    for (int j = 0; j < np; ++j) {
      const int2 d = pool[j];
      rank += better(__int_as_float(d.x), d.y, v, c.y);
    }
    if (rank < k) {
      if (rank == 0) argmax[row] = c.y;
      if (oi) {
        oi[rank] = c.y;
        ov[rank] = v;
      }
    }
  }
}

cudaError_t launch_topk(int rows, int V, int k, const float *logits, int32_t *argmax,
                        int32_t *topk_idx, float *topk_val, float *lse, int max_ctas, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (k < 1 || k > TK) return cudaErrorInvalidValue;
  const int g = max_ctas > 0 ? std::min(rows, max_ctas) : rows;
  return launch_pdl(k_topk_rows, dim3(g), dim3(TK_THREADS), 0, s, rows, V, k, logits, argmax, topk_idx,
                    topk_val, lse);
}

cudaError_t launch_topk_merge(int tiles, int rows, int k, const int2 *cand, int32_t *argmax,
                              int32_t *topk_idx, float *topk_val, const float2 *lse_part, float *lse,
                              cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (k < 1 || k > TK) return cudaErrorInvalidValue;
  return launch_pdl(k_topk_merge, dim3(rows), dim3(TK_THREADS), 0, s, tiles, rows, k, cand, argmax,
                    topk_idx, topk_val, lse_part, lse);
}

// ------------------------------------------------------------------------- sampling mode
// Truncated sampling distributions and the sampling verification (DFlash 2 块扩散投机解码技术
// 详解 §2.3 rejection sampling, §3.3 the same top-k / top-p truncation on the draft and the
// target side, §4.2 the fallback to p when the residual vanishes). A row's distribution:
// logits / temperature, the top_k largest kept (ties to the lower index), softmax over them,
// then the shortest prefix in descending order whose mass reaches top_p, renormalised. It
// is stored as at most SMP_K (token, probability) pairs in descending order. Draws are
// inverse-CDF over the kept tokens in vocabulary order against a caller-supplied uniform.

// Inverse-CDF draw over n (token, p) pairs: the pairs are visited in token order (insertion
// sort of at most SMP_K entries, single thread), the first token whose running sum exceeds
// u times the total is drawn (the last kept token if rounding leaves none).
__device__ __forceinline__ int32_t draw_in_vocab_order(const int32_t *tok, const float *p, int n, float u) {
  int32_t t[SMP_K];
  float q[SMP_K];
  for (int i = 0; i < n; ++i) {
    int j = i;
    while (j > 0 && t[j - 1] > tok[i]) {
      t[j] = t[j - 1];
      q[j] = q[j - 1];
      --j;
    }
    t[j] = tok[i];
    q[j] = p[i];
  }
  float total = 0.f;
  for (int i = 0; i < n; ++i) total += q[i];
  float acc = 0.f;
  for (int i = 0; i < n; ++i) {
    acc += q[i];
    if (acc > u * total) return t[i];
  }
  return n > 0 ? t[n - 1] : 0;
}

// One CTA per row (rows b, b + gridDim.x, ...): the row's truncated distribution into
// dist_tok / dist_p / dist_n ([rows][SMP_K], [rows]; skipped when dist_tok is null); with u
// non-null also a draw per row into draw.
__global__ void __launch_bounds__(TK_THREADS, 2) k_trunc_dist(int rows, int V, float temperature, int top_k,
                                                           float top_p, const float *logits, const float *u,
                                                           int32_t *draw, int32_t *dist_tok, float *dist_p,
                                                           int32_t *dist_n) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ float tmax[TK_THREADS];
  __shared__ int2 pool[ROWS_CAP];
  __shared__ int n_pool;
  __shared__ float thr;
  __shared__ int32_t sidx[TK];
  __shared__ float sval[TK];
  const int k = min(top_k, V);
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    row_select(logits + (size_t)row * V, V, k, tmax, pool, &n_pool, &thr, nullptr, sidx, sval);
    __syncthreads();
    if (threadIdx.x == 0) {
      // softmax of the kept values at the temperature, in descending order
      float p[SMP_K];
      const float z0 = sval[0] / temperature;
      float sum = 0.f;
      for (int i = 0; i < k; ++i) {
        p[i] = expf(sval[i] / temperature - z0);
        sum += p[i];
      }
      for (int i = 0; i < k; ++i) p[i] /= sum;
      int n = k;
      if (top_p < 1.f) {
        float mass = 0.f;
        for (n = 1; n <= k; ++n) {
          mass += p[n - 1];
          if (mass >= top_p) break;
        }
        if (n > k) n = k;
        float kept = 0.f;
        for (int i = 0; i < n; ++i) kept += p[i];
        for (int i = 0; i < n; ++i) p[i] /= kept;
      }
      if (dist_tok) {
        for (int i = 0; i < n; ++i) {
          dist_tok[(size_t)row * SMP_K + i] = sidx[i];
          dist_p[(size_t)row * SMP_K + i] = p[i];
        }
        dist_n[row] = n;
      }
      if (u) draw[row] = draw_in_vocab_order(sidx, p, n, u[row]);
    }
    __syncthreads();                   // the shared scratch is reused by the next row
  }
}

__device__ __forceinline__ float dist_lookup(const int32_t *tok, const float *p, int n, int32_t t) {
  for (int i = 0; i < n; ++i)
    if (tok[i] == t) return p[i];
  return 0.f;
}

// One thread per request: position j accepts draft[j] when u_accept[j] < min(1, p(d)/q(d))
// (q(d) = 0 accepts iff p(d) > 0); the first rejection emits a draw from norm(max(p - q, 0))
// (from p when that is all zero) and ends the round; with all K accepted a bonus is drawn
// from p at position K. Target rows are [B][K+1], draft rows [B][K] of the distributions.
__global__ void k_verify_sample(int B, int K, const int32_t *ptok, const float *pp, const int32_t *pn,
                                const int32_t *qtok, const float *qp, const int32_t *qn,
                                const int32_t *draft, const float *u_accept, const float *u_resample,
                                int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int32_t *o = out_tokens + (size_t)b * (K + 1);
  int a = K;
  int32_t last = -1;
  for (int j = 0; j < K; ++j) {
    const size_t pr = (size_t)b * (K + 1) + j, qr = (size_t)b * K + j;
    const int32_t *Pt = ptok + pr * SMP_K, *Qt = qtok + qr * SMP_K;
    const float *Pp = pp + pr * SMP_K, *Qp = qp + qr * SMP_K;
    const int np_ = pn[pr], nq_ = qn[qr];
    const int32_t d = draft[qr];
    const float pd = dist_lookup(Pt, Pp, np_, d), qd = dist_lookup(Qt, Qp, nq_, d);
    const float ratio = qd > 0.f ? pd / qd : (pd > 0.f ? 1.f : 0.f);
    if (u_accept[qr] < fminf(1.f, ratio)) {
      o[j] = d;
      continue;
    }
    // residual max(p - q, 0): only tokens with p > 0 can carry mass
    float r[SMP_K];
    float tot = 0.f;
    for (int i = 0; i < np_; ++i) {
      r[i] = fmaxf(Pp[i] - dist_lookup(Qt, Qp, nq_, Pt[i]), 0.f);
      tot += r[i];
    }
    if (tot > 0.f) {
      for (int i = 0; i < np_; ++i) r[i] /= tot;
      last = draw_in_vocab_order(Pt, r, np_, u_resample[b]);
    } else {
      last = draw_in_vocab_order(Pt, Pp, np_, u_resample[b]);
    }
    o[j] = last;
    a = j;
    break;
  }
  if (a == K) {
    const size_t pr = (size_t)b * (K + 1) + K;
    last = draw_in_vocab_order(ptok + pr * SMP_K, pp + pr * SMP_K, pn[pr], u_resample[b]);
    o[K] = last;
  }
  for (int j = a + 1; j <= K; ++j) o[j] = -1;
  accept_len[b] = a;
  next_anchor[b] = last;
}

cudaError_t launch_trunc_dist(int rows, int V, float temperature, int top_k, float top_p,
                              const float *logits, const float *u, int32_t *draw, int32_t *dist_tok,
                              float *dist_p, int32_t *dist_n, int max_ctas, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (top_k < 1 || top_k > SMP_K || !(temperature > 0.f) || !(top_p > 0.f) || top_p > 1.f)
    return cudaErrorInvalidValue;
  const int g = max_ctas > 0 ? std::min(rows, max_ctas) : rows;
  return launch_pdl(k_trunc_dist, dim3(g), dim3(TK_THREADS), 0, s, rows, V, temperature, top_k, top_p,
                    logits, u, draw, dist_tok, dist_p, dist_n);
}

cudaError_t launch_verify_sample(int B, int K, const int32_t *ptok, const float *pp, const int32_t *pn,
                                 const int32_t *qtok, const float *qp, const int32_t *qn,
                                 const int32_t *draft, const float *u_accept, const float *u_resample,
                                 int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor,
                                 cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(k_verify_sample, dim3((B + 127) / 128), dim3(128), 0, s, B, K, ptok, pp, pn, qtok, qp,
                    qn, draft, u_accept, u_resample, accept_len, out_tokens, next_anchor);
}

// ------------------------------------------------------------------------- no-allocation variant
// dflash_topk_noalloc (declared in dflash.h) ranks rows of fp32 logits like the LM-head path:
// per-chunk candidates first, then the same cross-chunk merge. Its candidates live in the
// file-scope device array below instead of memory the caller or a context allocates, for
// callers that must not touch the CUDA allocator (code recorded into a CUDA graph, runtimes
// that own a fixed device-memory budget). The array is shared by every call in the process
// and keeps the last call's contents.
constexpr int NA_CHUNK = 4096;                      // logits per candidate chunk
constexpr long NA_MAX_CAND = 1L << 19;              // 4 MiB of (value, index) candidates
static __device__ __align__(256) int2 g_topk_scratch[NA_MAX_CAND];

__global__ void __launch_bounds__(TK_THREADS) k_topk_chunks(int V, int k, int chunks, int rows,
                                                            const float *logits, int2 *cand) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ int32_t idx[32];
  __shared__ float val[32];
  __shared__ int32_t first;
  const int row = blockIdx.x, chunk = blockIdx.y;      // rows on x: up to 2^31 - 1 of them
  const int v0 = chunk * NA_CHUNK, n = min(NA_CHUNK, V - v0);
  const float *x = logits + (size_t)row * V + v0;
  block_topk(n, k, [&](int i, float &v, int &id) { v = x[i]; id = v0 + i; }, &first, idx, val);
  __syncthreads();
  if (threadIdx.x < k)
    cand[((size_t)chunk * rows + row) * k + threadIdx.x] = make_int2(__float_as_int(val[threadIdx.x]), idx[threadIdx.x]);
}

namespace {
std::mutex g_na_mu;
int2 *g_na_ptr[128] = {};    // device address of g_topk_scratch, per device, set up once
}  // namespace

}  // namespace dflash

using namespace dflash;

extern "C" dflash_status dflash_topk_noalloc(void *stream, int32_t rows, int32_t vocab, int32_t k,
                                             const float *logits, int32_t *argmax,
                                             int32_t *topk_idx, float *topk_val, char *msg,
                                             int32_t msg_len) {
  auto fail = [&](dflash_status st, const char *why) {
    if (msg && msg_len > 0) snprintf(msg, (size_t)msg_len, "%s", why);
    return st;
  };
  if (msg && msg_len > 0) msg[0] = 0;
  if (rows < 0 || vocab < 1 || k < 1 || k > TK || k > vocab)
    return fail(DFLASH_ERR_INVALID_ARG, "need rows >= 0 and 1 <= k <= min(32, vocab)");
  if (rows == 0) return DFLASH_OK;
  if (!logits || !argmax || ((topk_idx == nullptr) != (topk_val == nullptr)))
    return fail(DFLASH_ERR_INVALID_ARG, "logits and argmax are required; topk_idx/topk_val both or neither");
  const long chunks = (vocab + NA_CHUNK - 1) / NA_CHUNK;
  if (chunks > 65535) return fail(DFLASH_ERR_INVALID_ARG, "vocab above 65535 * 4096 entries");
  if ((long)rows * chunks * k > NA_MAX_CAND) {
    char why[200];
    snprintf(why, sizeof why, "rows * ceil(vocab/%d) * k = %ld exceeds the fixed scratch of %ld candidates",
             NA_CHUNK, (long)rows * chunks * k, NA_MAX_CAND);
    return fail(DFLASH_ERR_INVALID_ARG, why);
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
    return fail(DFLASH_ERR_CUDA, "no current CUDA device");
  int2 *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!g_na_ptr[dev]) {
      // once per device: the host-side symbol is only a stand-in, the kernels need the
      // device address of this device's copy of the array
      int2 *ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress((void **)&ptr, g_topk_scratch);
      if (e != cudaSuccess || !ptr) return fail(DFLASH_ERR_CUDA, "cudaGetSymbolAddress of the top-k scratch failed");
      g_na_ptr[dev] = ptr;
    }
    scratch = g_na_ptr[dev];
  }
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_pdl(k_topk_chunks, dim3((unsigned)rows, (unsigned)chunks), dim3(TK_THREADS), 0, s,
                             (int)vocab, (int)k, (int)chunks, (int)rows, logits, scratch);
  if (e == cudaSuccess)
    e = launch_topk_merge((int)chunks, rows, k, scratch, argmax, topk_idx, topk_val, nullptr, nullptr, s);
  if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, cudaGetErrorString(e));
  return DFLASH_OK;
}
