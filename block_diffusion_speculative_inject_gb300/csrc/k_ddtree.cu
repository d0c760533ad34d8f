// Draft trees ("DDTree" §2.3 Algorithm 1 and Proposition 2, §3.3 the ancestor-only mask,
// §3.5 the verifier walk): from each block position's best candidates (log-probabilities,
// best first), the `budget` most likely prefixes form a prefix-closed tree, found best-first
// with a max-heap of rank tuples: a popped prefix becomes a node and pushes its next sibling
// (same parent, next candidate) and its first child (best candidate of the next position).
// One CTA builds one request's tree on one thread (the heap holds at most budget + 1
// entries, in shared memory); ties pop by (log-probability desc, depth asc, parent asc, rank
// asc).
#include <cstdio>

#include "../../include/dflash.h"
#include "kernels.h"

namespace dflash {

constexpr int DDT_MAX_BUDGET = 1024;

struct HeapEnt {
  float lp;
  int16_t depth, parent, rank, pad;
};

__device__ __forceinline__ bool pops_first(const HeapEnt &a, const HeapEnt &b) {
  if (a.lp != b.lp) return a.lp > b.lp;
  if (a.depth != b.depth) return a.depth < b.depth;
  if (a.parent != b.parent) return a.parent < b.parent;
  return a.rank < b.rank;
}

__device__ __forceinline__ void heap_push(HeapEnt *h, int &n, HeapEnt e) {
  int i = n++;
  while (i > 0) {
    const int p = (i - 1) / 2;
    if (!pops_first(e, h[p])) break;
    h[i] = h[p];
    i = p;
  }
  h[i] = e;
}

__device__ __forceinline__ HeapEnt heap_pop(HeapEnt *h, int &n) {
  const HeapEnt top = h[0];
  const HeapEnt last = h[--n];
  int i = 0;
  for (;;) {
    int c = 2 * i + 1;
    if (c >= n) break;
    if (c + 1 < n && pops_first(h[c + 1], h[c])) ++c;
    if (!pops_first(h[c], last)) break;
    h[i] = h[c];
    i = c;
  }
  if (n > 0) h[i] = last;
  return top;
}

// cand_tok / cand_logp [n][L][kc]; outputs [n][budget] (unused slots: token -1, parent -1,
// depth 0), n_nodes [n], mask [n][budget + 1][words] (row i: index 0 = the root, node j =
// index j + 1; bit j of a row set when index j is visible).
__global__ void k_ddtree_build(int n, int L, int kc, int budget, const int32_t *cand_tok,
                               const float *cand_logp, int32_t *tree_tok, int32_t *tree_parent,
                               int32_t *tree_depth, float *tree_logp, int32_t *n_nodes, uint32_t *mask,
                               int words) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  extern __shared__ HeapEnt heap[];    // budget + 1 entries
  const int b = blockIdx.x;
  if (b >= n || threadIdx.x != 0) return;
  const int32_t *tok = cand_tok + (size_t)b * L * kc;
  const float *lpv = cand_logp + (size_t)b * L * kc;
  int32_t *otok = tree_tok + (size_t)b * budget, *opar = tree_parent + (size_t)b * budget;
  int32_t *odep = tree_depth + (size_t)b * budget;
  float *olp = tree_logp + (size_t)b * budget;
  uint32_t *m = mask ? mask + (size_t)b * (budget + 1) * words : nullptr;
  int hn = 0, nodes = 0;
  heap_push(heap, hn, HeapEnt{lpv[0], 1, -1, 0, 0});
  while (hn > 0 && nodes < budget) {
    const HeapEnt e = heap_pop(heap, hn);
    const int me = nodes++;
    otok[me] = tok[(e.depth - 1) * kc + e.rank];
    opar[me] = e.parent;
    odep[me] = e.depth;
    olp[me] = e.lp;
    const float base = e.parent < 0 ? 0.f : olp[e.parent];
    if (e.rank + 1 < kc)
      heap_push(heap, hn, HeapEnt{base + lpv[(e.depth - 1) * kc + e.rank + 1], e.depth, e.parent,
                                  (int16_t)(e.rank + 1), 0});
    if (e.depth < L)
      heap_push(heap, hn, HeapEnt{e.lp + lpv[e.depth * kc], (int16_t)(e.depth + 1), (int16_t)me, 0, 0});
  }
  for (int i = nodes; i < budget; ++i) {
    otok[i] = -1;
    opar[i] = -1;
    odep[i] = 0;
    olp[i] = -INFINITY;
  }
  n_nodes[b] = nodes;
  if (m) {
    // the root sees itself; a node sees what its parent sees plus itself
    for (int w = 0; w < words; ++w) m[w] = w == 0 ? 1u : 0u;
    for (int i = 0; i < budget; ++i) {
      uint32_t *row = m + (size_t)(i + 1) * words;
      const uint32_t *prow = m + (size_t)(i < nodes ? opar[i] + 1 : 0) * words;
      for (int w = 0; w < words; ++w) row[w] = i < nodes ? prow[w] : (w == 0 ? 1u : 0u);
      if (i < nodes) row[(i + 1) / 32] |= 1u << ((i + 1) % 32);
    }
  }
}

// Greedy walk: target_next [n][budget + 1] (index 0: after the root, index i + 1: after node
// i). Outputs accept_len [n], out_tokens [n][L + 1] (the matched tokens, the target's token
// where the walk stopped, then -1), next_anchor [n].
__global__ void k_ddtree_walk(int n, int L, int budget, const int32_t *tree_tok, const int32_t *tree_parent,
                              const int32_t *n_nodes, const int32_t *target_next, int32_t *accept_len,
                              int32_t *out_tokens, int32_t *next_anchor) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= n) return;
  const int32_t *tok = tree_tok + (size_t)b * budget, *par = tree_parent + (size_t)b * budget;
  const int32_t *tn = target_next + (size_t)b * (budget + 1);
  int32_t *o = out_tokens + (size_t)b * (L + 1);
  const int nn = n_nodes[b];
  int cur = -1, a = 0;
  int32_t t = tn[0];
  for (;;) {
    int child = -1;
    for (int i = 0; i < nn; ++i)
      if (par[i] == cur && tok[i] == t) {
        child = i;
        break;
      }
    o[a] = t;
    if (child < 0 || a >= L) break;
    ++a;
    cur = child;
    t = tn[cur + 1];
  }
  for (int j = a + 1; j <= L; ++j) o[j] = -1;
  accept_len[b] = a;
  next_anchor[b] = t;
}

}  // namespace dflash

using namespace dflash;

extern "C" dflash_status dflash_ddtree_build(void *stream, int32_t n_req, int32_t L, int32_t kc, int32_t budget,
                                             const int32_t *cand_tok, const float *cand_logp,
                                             int32_t *tree_tok, int32_t *tree_parent, int32_t *tree_depth,
                                             float *tree_logp, int32_t *n_nodes, uint32_t *mask) {
  if (n_req < 0 || L < 1 || L > 31 || kc < 1 || kc > 32 || budget < 1 || budget > DDT_MAX_BUDGET)
    return DFLASH_ERR_INVALID_ARG;
  if (n_req == 0) return DFLASH_OK;
  if (!cand_tok || !cand_logp || !tree_tok || !tree_parent || !tree_depth || !tree_logp || !n_nodes)
    return DFLASH_ERR_INVALID_ARG;
  const int words = (budget + 1 + 31) / 32;
  cudaError_t e = launch_pdl(k_ddtree_build, dim3(n_req), dim3(32), (size_t)(budget + 1) * sizeof(HeapEnt),
                             (cudaStream_t)stream,
                             (int)n_req, (int)L, (int)kc, (int)budget, cand_tok, cand_logp, tree_tok, tree_parent,
                             tree_depth, tree_logp, n_nodes, mask, words);
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
  cudaError_t e = launch_pdl(k_ddtree_walk, dim3((n_req + 63) / 64), dim3(64), 0, (cudaStream_t)stream,
                             (int)n_req, (int)L, (int)budget, tree_tok, tree_parent, n_nodes, target_next,
                             accept_len, out_tokens, next_anchor);
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}
