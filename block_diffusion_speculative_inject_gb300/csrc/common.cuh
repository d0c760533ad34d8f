// Shared device helpers and the internal launcher interface of libdflash.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace dflash {

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// Storage rounding of an fp32 value (the value a store of type T would keep).
template <typename T> __device__ __forceinline__ float round_st(float x) { return to_f(from_f<T>(x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Device error codes latched into the mapped host flag (bit set).
enum : int { DEV_ERR_TOKEN = 1, DEV_ERR_BOUNDS = 2, DEV_ERR_TIMEOUT = 4 };

// The flag lives in mapped pinned host memory; a plain volatile store is enough (any
// nonzero value reports an error; the code bits are a hint).
__device__ __forceinline__ void raise_err(int *flag, int code) {
  if (flag) *(volatile int *)flag = code;
}

// ---------------------------------------------------------------- GEMM description
// Y[M, N] = epilogue( X[M, K] . W[N, K]^T ), X and W of the storage type.
// X may be split along K into segments with separate base pointers (the fc fusion reads
// the n_feat feature tensors in place); W may be split along N into segments (e.g. the
// q/k/v or the per-layer k/v weights) each [rows, K] row-major with row stride K.
enum GemmEpi : int {
  EPI_STORE = 0,   // Y = round(acc)                                 (storage type)
  EPI_RESID = 1,   // Y = round(R + round(acc))   (R may alias Y)     (storage type)
  EPI_F32 = 2,     // Yf = acc                                       (fp32)
  EPI_SWIGLU = 3,  // W = [gate; up] halves: Y[:, n] = round(silu(round(g)) * round(u)), N = 2*I
};

constexpr int GEMM_MAX_XSEG = 8;
constexpr int GEMM_MAX_WSEG = 16;

struct GemmDesc {
  int M, N, K;
  int n_xseg;
  const void *x[GEMM_MAX_XSEG];
  int x_k0[GEMM_MAX_XSEG + 1];   // K offset where segment s starts; x_k0[n_xseg] = K
  int ldx[GEMM_MAX_XSEG];        // row stride (elements) of each X segment
  int n_wseg;
  const void *w[GEMM_MAX_WSEG];
  int w_n0[GEMM_MAX_WSEG + 1];   // N offset where segment s starts; w_n0[n_wseg] = N
  int epi;
  void *y;                       // output [M, ldy] (storage type, or fp32 for EPI_F32)
  int ldy;
  const void *resid;             // EPI_RESID input [M, ldy]
};

}  // namespace dflash
