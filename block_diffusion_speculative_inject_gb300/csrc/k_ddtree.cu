// Draft trees ("DDTree" §2.3 Algorithm 1 and Proposition 2, §3.3 the ancestor-only mask,
// §3.5 the verifier walk): from each block position's best candidates (log-probabilities,
// best first), the `budget` most likely prefixes form a prefix-closed tree, found best-first
// from a frontier of prefixes: a popped prefix becomes a node and is replaced by its next
// sibling (same parent, next candidate) and its first child (best candidate of the next
// position). Ties pop by (log-probability desc, depth asc, parent asc, rank asc).
//
// One CTA per request; its first warp builds the tree. The frontier is a set of 64-bit keys
// held in that warp's registers (FPL slots per lane), ordered so that the largest key pops
// first:
//   high word: the log-probability's bits mapped to an unsigned order;
//   low word: (31 - depth) << 16 | (2047 - (parent + 1)) << 5 | (31 - rank).
// A pop is a two-word warp max (redux.sync); the owner lane puts the sibling in the popped
// slot, the child goes to a fresh slot. Every pop but the last adds at most one slot, so
// budget slots always suffice. The loop touches shared memory only; afterwards the whole CTA
// writes the nodes and forms each mask row by walking its node's parent chain.
#include <cstdio>

#include "../../include/dflash.h"
#include "kernels.h"

namespace dflash {

constexpr int DDT_MAX_BUDGET = 1024;

__device__ __forceinline__ uint32_t ord_f32(float x) {
  const uint32_t u = __float_as_uint(x == 0.f ? 0.f : x);      // -0 orders as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unord_f32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__device__ __forceinline__ uint64_t ddt_key(float lp, int depth, int parent, int rank) {
  const uint32_t lo = (uint32_t)(31 - depth) << 16 | (uint32_t)(2047 - (parent + 1)) << 5 | (uint32_t)(31 - rank);
  return (uint64_t)ord_f32(lp) << 32 | lo;
}

// Shared memory: cand_lp [L*kc] f32, cand_tok [L*kc] i32, node_lp [budget] f32, node_parent
// [budget] i32, node_dr [budget] i32 (depth << 8 | rank), the node count, then (with a mask)
// the rows [(budget + 1) * words] u32.
__host__ __device__ inline size_t ddt_smem(int L, int kc, int budget, int words, bool mask) {
  return (size_t)(2 * L * kc + 3 * budget + 1) * 4 + (mask ? (size_t)(budget + 1) * words * 4 : 0);
}

constexpr int DDT_THREADS = 128;

template <int N>
__device__ __forceinline__ uint64_t max_of(const uint64_t (&v)[N]) {
  uint64_t t[N];
#pragma unroll
  for (int j = 0; j < N; ++j) t[j] = v[j];
#pragma unroll
  for (int h = N / 2; h >= 1; h /= 2)
#pragma unroll
    for (int j = 0; j < h; ++j) t[j] = t[j] > t[j + h] ? t[j] : t[j + h];
  return t[0];
}

// cand_tok / cand_logp [n][L][kc], cand_lse [n][L] or null (subtracted from cand_logp); outputs
// [n][budget] (unused slots: token -1, parent -1, depth 0, log-probability -inf), n_nodes [n],
// mask [n][budget + 1][words] (row i: index 0 = the root, node j = index j + 1; bit j of a row
// set when index j is visible).
template <int FPL>
__global__ void __launch_bounds__(DDT_THREADS) k_ddtree_build(int n, int L, int kc, int budget,
                                                              const int32_t *cand_tok, const float *cand_logp,
                                                              const float *cand_lse, int32_t *tree_tok,
                                                              int32_t *tree_parent, int32_t *tree_depth,
                                                              float *tree_logp, int32_t *n_nodes, uint32_t *mask,
                                                              int words) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  extern __shared__ float ddt_sm[];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  if (b >= n) return;
  float *c_lp = ddt_sm;
  int32_t *c_tok = reinterpret_cast<int32_t *>(c_lp + L * kc);
  float *node_lp = reinterpret_cast<float *>(c_tok + L * kc);
  int32_t *node_par = reinterpret_cast<int32_t *>(node_lp + budget);
  int32_t *node_dr = node_par + budget;
  int32_t *node_cnt = node_dr + budget;
  uint32_t *rows = reinterpret_cast<uint32_t *>(node_cnt + 1);
  for (int i = tid; i < L * kc; i += DDT_THREADS) {
    const float v = cand_logp[(size_t)b * L * kc + i];
    c_lp[i] = cand_lse ? v - cand_lse[(size_t)b * L + i / kc] : v;
    c_tok[i] = cand_tok[(size_t)b * L * kc + i];
  }
  __syncthreads();

  if (tid < 32) {
    uint64_t keys[FPL];
#pragma unroll
    for (int j = 0; j < FPL; ++j) keys[j] = 0;
    if (lane == 0) keys[0] = ddt_key(c_lp[0], 1, -1, 0);
    uint64_t best = keys[0];
    int slots = 1, nodes = 0;
    while (nodes < budget) {
      const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
      const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32) == hi ? (uint32_t)best : 0u);
      if (hi == 0 && lo == 0) break;                                // the frontier is empty
      const uint64_t key = (uint64_t)hi << 32 | lo;
      const float lp = unord_f32(hi);
      const int depth = 31 - (int)(lo >> 16), parent = 2047 - (int)((lo >> 5) & 2047) - 1;
      const int rank = 31 - (int)(lo & 31);
      const int me = nodes++;
      if (lane == 0) {
        node_lp[me] = lp;
        node_par[me] = parent;
        node_dr[me] = depth << 8 | rank;
      }
      // the popped slot takes the next sibling (or empties); the child takes a fresh slot
      const bool last = nodes == budget;
      uint64_t sib = 0, child = 0;
      if (!last && rank + 1 < kc)
        sib = ddt_key((parent < 0 ? 0.f : node_lp[parent]) + c_lp[(depth - 1) * kc + rank + 1], depth, parent,
                      rank + 1);
      if (!last && depth < L) child = ddt_key(lp + c_lp[depth * kc], depth + 1, me, 0);
      if (best == key) {
#pragma unroll
        for (int j = 0; j < FPL; ++j) keys[j] = keys[j] == key ? sib : keys[j];
        best = max_of(keys);
      }
      if (child) {
        const int s = slots++;
        const bool mine = lane == (s & 31);
#pragma unroll
        for (int j = 0; j < FPL; ++j) keys[j] = (mine && j == (s >> 5)) ? child : keys[j];
        if (mine) best = child > best ? child : best;
      }
      __syncwarp();
    }
    if (lane == 0) *node_cnt = nodes;
  }
  __syncthreads();

  const int nodes = *node_cnt;
  int32_t *otok = tree_tok + (size_t)b * budget, *opar = tree_parent + (size_t)b * budget;
  int32_t *odep = tree_depth + (size_t)b * budget;
  float *olp = tree_logp + (size_t)b * budget;
  for (int i = tid; i < budget; i += DDT_THREADS) {
    const bool used = i < nodes;
    const int dr = used ? node_dr[i] : 0;
    otok[i] = used ? c_tok[((dr >> 8) - 1) * kc + (dr & 255)] : -1;
    opar[i] = used ? node_par[i] : -1;
    odep[i] = used ? dr >> 8 : 0;
    olp[i] = used ? node_lp[i] : -INFINITY;
  }
  if (tid == 0) n_nodes[b] = nodes;
  if (!mask) return;
  // row i sees index i, its ancestors and the root (index 0); the chain's indices fall, so the
  // row's words are written once each, from the last to the first
  for (int i = tid; i <= budget; i += DDT_THREADS) {
    uint32_t *row = rows + (size_t)i * words;
    int a = i <= nodes ? i - 1 : -1, w = words - 1;
    uint32_t acc = 0;
    for (;;) {
      const int bit = a + 1, wb = bit >> 5;
      for (; w > wb; --w) {
        row[w] = acc;
        acc = 0;
      }
      acc |= 1u << (bit & 31);
      if (a < 0) break;
      a = node_par[a];
    }
    for (; w >= 0; --w) {
      row[w] = acc;
      acc = 0;
    }
  }
  __syncthreads();
  uint32_t *m = mask + (size_t)b * (budget + 1) * words;
  for (int i = tid; i < (budget + 1) * words; i += DDT_THREADS) m[i] = rows[i];
}

// Greedy walk: target_next [n][budget + 1] (index 0: after the root, index i + 1: after node
// i). Outputs accept_len [n], out_tokens [n][L + 1] (the matched tokens, the target's token
// where the walk stopped, then -1), next_anchor [n]. One warp per request scans the nodes 32
// at a time for the first child of the current node with the target's token.
__global__ void __launch_bounds__(32) k_ddtree_walk(int n, int L, int budget, const int32_t *tree_tok,
                                                    const int32_t *tree_parent, const int32_t *n_nodes,
                                                    const int32_t *target_next, int32_t *accept_len,
                                                    int32_t *out_tokens, int32_t *next_anchor) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  if (b >= n) return;
  const int32_t *tok = tree_tok + (size_t)b * budget, *par = tree_parent + (size_t)b * budget;
  const int32_t *tn = target_next + (size_t)b * (budget + 1);
  int32_t *o = out_tokens + (size_t)b * (L + 1);
  const int nn = n_nodes[b];
  int cur = -1, a = 0;
  int32_t t = tn[0];
  for (;;) {
    int child = -1;
    for (int base = 0; base < nn; base += 32) {
      const int i = base + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, i < nn && par[i] == cur && tok[i] == t);
      if (hit) {
        child = base + __ffs(hit) - 1;
        break;
      }
    }
    if (lane == 0) o[a] = t;
    if (child < 0 || a >= L) break;
    ++a;
    cur = child;
    t = tn[cur + 1];
  }
  for (int j = a + 1 + lane; j <= L; j += 32) o[j] = -1;
  if (lane == 0) {
    accept_len[b] = a;
    next_anchor[b] = t;
  }
}

struct BuildArgs {
  int n, L, kc, budget;
  const int32_t *cand_tok;
  const float *cand_logp, *cand_lse;
  int32_t *tree_tok, *tree_parent, *tree_depth;
  float *tree_logp;
  int32_t *n_nodes;
  uint32_t *mask;
  int words;
};

template <int FPL>
cudaError_t launch_build(const BuildArgs &x, cudaStream_t s) {
  static bool smem_opt_in = false;     // the largest tree's shared memory, once per instance
  if (!smem_opt_in) {
    const cudaError_t e = cudaFuncSetAttribute(k_ddtree_build<FPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)ddt_smem(31, 32, DDT_MAX_BUDGET, (DDT_MAX_BUDGET + 32) / 32, true));
    if (e != cudaSuccess) return e;
    smem_opt_in = true;
  }
  return launch_pdl(k_ddtree_build<FPL>, dim3(x.n), dim3(DDT_THREADS), ddt_smem(x.L, x.kc, x.budget, x.words, x.mask),
                    s, x.n, x.L, x.kc, x.budget, x.cand_tok, x.cand_logp, x.cand_lse, x.tree_tok, x.tree_parent,
                    x.tree_depth, x.tree_logp, x.n_nodes, x.mask, x.words);
}

}  // namespace dflash

using namespace dflash;

extern "C" dflash_status dflash_ddtree_build(void *stream, int32_t n_req, int32_t L, int32_t kc, int32_t budget,
                                             const int32_t *cand_tok, const float *cand_logp,
                                             const float *cand_lse, int32_t *tree_tok, int32_t *tree_parent, int32_t *tree_depth,
                                             float *tree_logp, int32_t *n_nodes, uint32_t *mask) {
  if (n_req < 0 || L < 1 || L > 31 || kc < 1 || kc > 32 || budget < 1 || budget > DDT_MAX_BUDGET)
    return DFLASH_ERR_INVALID_ARG;
  if (n_req == 0) return DFLASH_OK;
  if (!cand_tok || !cand_logp || !tree_tok || !tree_parent || !tree_depth || !tree_logp || !n_nodes)
    return DFLASH_ERR_INVALID_ARG;
  const int words = (budget + 1 + 31) / 32;
  const int fpl = (budget + 31) / 32;
  const BuildArgs x{(int)n_req, (int)L, (int)kc, (int)budget, cand_tok, cand_logp, cand_lse, tree_tok,
                    tree_parent, tree_depth, tree_logp, n_nodes, mask, words};
  const cudaStream_t st = (cudaStream_t)stream;
  const cudaError_t e = fpl <= 1 ? launch_build<1>(x, st) : fpl <= 2 ? launch_build<2>(x, st)
                      : fpl <= 4 ? launch_build<4>(x, st) : fpl <= 8 ? launch_build<8>(x, st)
                      : fpl <= 16 ? launch_build<16>(x, st) : launch_build<32>(x, st);
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

extern "C" dflash_status dflash_ddtree_walk(void *stream, int32_t n_req, int32_t L, int32_t budget,
                                            const int32_t *tree_tok, const int32_t *tree_parent,
                                            const int32_t *n_nodes, const int32_t *target_next,
                                            int32_t *accept_len, int32_t *out_tokens, int32_t *next_anchor) {
  if (n_req < 0 || L < 1 || L > 31 || budget < 1 || budget > DDT_MAX_BUDGET) return DFLASH_ERR_INVALID_ARG;
  if (n_req == 0) return DFLASH_OK;
  if (!tree_tok || !tree_parent || !n_nodes || !target_next || !accept_len || !out_tokens || !next_anchor)
    return DFLASH_ERR_INVALID_ARG;
  cudaError_t e = launch_pdl(k_ddtree_walk, dim3(n_req), dim3(32), 0, (cudaStream_t)stream,
                             (int)n_req, (int)L, (int)budget, tree_tok, tree_parent, n_nodes, target_next,
                             accept_len, out_tokens, next_anchor);
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}
