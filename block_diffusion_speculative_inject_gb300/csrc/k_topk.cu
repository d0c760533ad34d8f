// Row-wise top-k over fp32 logits: values descending, equal values ordered by the lower
// vocabulary index; the argmax is the first entry. One CTA per row: every thread keeps a
// sorted register list of its best TK candidates over a strided slice of the row, then
// the block merges the 256 sorted lists by k rounds of a block-wide "best head" pick.
#include "kernels.h"

namespace dflash {

constexpr int TK = 32;         // register list length (>= any requested k)
constexpr int TK_THREADS = 256;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(TK_THREADS) k_topk_rows(int V, int k, const float *logits,
                                                          int32_t *argmax, int32_t *topk_idx,
                                                          float *topk_val) {
  __shared__ float hv[TK_THREADS];
  __shared__ int hi[TK_THREADS];
  __shared__ int ht[TK_THREADS];
  const int row = blockIdx.x, tid = threadIdx.x;
  const float *x = logits + (size_t)row * V;
  float lv[TK];
  int li[TK];
#pragma unroll
  for (int q = 0; q < TK; ++q) {
    lv[q] = -INFINITY;
    li[q] = 0x7fffffff;
  }
  for (int i = tid; i < V; i += TK_THREADS) {
    float v = x[i];
    if (!better(v, i, lv[TK - 1], li[TK - 1])) continue;
    // insertion into the sorted list (unrolled, registers only)
    float cv = v;
    int ci = i;
#pragma unroll
    for (int q = 0; q < TK; ++q) {
      bool b = better(cv, ci, lv[q], li[q]);
      float tv = lv[q];
      int ti = li[q];
      lv[q] = b ? cv : lv[q];
      li[q] = b ? ci : li[q];
      cv = b ? tv : cv;
      ci = b ? ti : ci;
    }
  }
  // merge: each round every thread offers its current head; the block best is emitted
  int head = 0;
  for (int r = 0; r < k; ++r) {
    float myv = -INFINITY;
    int myi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < TK; ++q)
      if (q == head) {
        myv = lv[q];
        myi = li[q];
      }
    hv[tid] = myv;
    hi[tid] = myi;
    ht[tid] = tid;
    __syncthreads();
    for (int st = TK_THREADS / 2; st > 0; st >>= 1) {
      if (tid < st && better(hv[tid + st], hi[tid + st], hv[tid], hi[tid])) {
        hv[tid] = hv[tid + st];
        hi[tid] = hi[tid + st];
        ht[tid] = ht[tid + st];
      }
      __syncthreads();
    }
    float bv = hv[0];
    int bi = hi[0], bt = ht[0];
    __syncthreads();
    if (tid == bt) ++head;
    if (tid == 0) {
      if (r == 0) argmax[row] = bi;
      if (topk_idx) {
        topk_idx[(size_t)row * k + r] = bi;
        topk_val[(size_t)row * k + r] = bv;
      }
    }
  }
}

cudaError_t launch_topk(int rows, int V, int k, const float *logits, int32_t *argmax,
                        int32_t *topk_idx, float *topk_val, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (k < 1 || k > TK) return cudaErrorInvalidValue;
  k_topk_rows<<<rows, TK_THREADS, 0, s>>>(V, k, logits, argmax, topk_idx, topk_val);
  return cudaGetLastError();
}

}  // namespace dflash
