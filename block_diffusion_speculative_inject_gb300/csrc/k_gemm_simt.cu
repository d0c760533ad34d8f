// FFMA GEMM: Y = epilogue(X . W^T), fp32 accumulation on the CUDA cores.
//
// This is the fp32-storage path (where tensor-core TF32 would not meet fp32 accuracy) and
// the reference kernel the tensor-core path is checked against. Tile 32 (rows of X) x 64
// (rows of W) x 32 (K), 256 threads, each thread 2 x 4 outputs. X may be split along K
// into segments (the fc fusion reads each feature tensor in place) and may be a bf16
// hi/lo pair; W may be split along N.
#include "kernels.h"

namespace dflash {

constexpr int SB_M = 32, SB_N = 64, SB_K = 32;

template <typename T>
__device__ __forceinline__ float load_x(const GemmDesc &d, int s, size_t idx) {
  if (!d.x_bf16) return ((const float *)d.x[s])[idx];
  float v = to_f(((const bf16 *)d.x[s])[idx]);
  if (d.x_lo[s]) v += to_f(((const bf16 *)d.x_lo[s])[idx]);
  if (s == 0 && d.x_lo2) v += to_f(((const bf16 *)d.x_lo2)[idx]);
  return v;
}

template <typename T>
__global__ void __launch_bounds__(256) k_gemm_simt(GemmDesc d) {
  pdl_trigger();                       // dependents may launch and prefetch; they still wait
  pdl_wait();
  __shared__ float xs[SB_K][SB_M + 1];
  __shared__ float ws[SB_K][SB_N + 1];
  const int m0 = blockIdx.y * SB_M, n0 = blockIdx.x * SB_N;
  const int tid = threadIdx.x;
  const int tm = tid / 16, tn = tid % 16;   // thread owns rows tm*2.., cols tn + 16*j

  // W segment of this N tile (tiles never straddle segments: boundaries are multiples of 64)
  int ws_i = 0;
  while (ws_i + 1 < d.n_wseg && n0 >= d.w_n0[ws_i + 1]) ++ws_i;
  const T *wbase = (const T *)d.w[ws_i];
  const int wn_off = d.w_n0[ws_i], wn_end = d.w_n0[ws_i + 1];

  float acc[2][4] = {};
  for (int k0 = 0; k0 < d.K; k0 += SB_K) {
    int xs_i = 0;
    while (xs_i + 1 < d.n_xseg && k0 >= d.x_k0[xs_i + 1]) ++xs_i;
    const int xk = k0 - d.x_k0[xs_i], ldx = d.ldx[xs_i];
    // X tile: 32 x 32
    for (int i = tid; i < SB_M * SB_K; i += 256) {
      int r = i / SB_K, c = i % SB_K;
      int m = m0 + r;
      xs[c][r] = m < d.M ? load_x<T>(d, xs_i, (size_t)m * ldx + xk + c) : 0.f;
    }
    // W tile: 64 x 32
    for (int i = tid; i < SB_N * SB_K; i += 256) {
      int r = i / SB_K, c = i % SB_K;
      int n = n0 + r;
      ws[c][r] = n < wn_end ? to_f(wbase[(size_t)(n - wn_off) * d.K + k0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < SB_K; ++k) {
      float a0 = xs[k][tm * 2], a1 = xs[k][tm * 2 + 1];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float b = ws[k][tn + 16 * j];
        acc[0][j] = fmaf(a0, b, acc[0][j]);
        acc[1][j] = fmaf(a1, b, acc[1][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    int m = m0 + tm * 2 + i;
    if (m >= d.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tn + 16 * j;
      if (n >= d.N) continue;
      float a = acc[i][j];
      size_t o = (size_t)m * d.ldy + n;
      d.y[o] = d.epi == EPI_RESID ? d.resid[o] + a : a;
    }
  }
}

cudaError_t gemm_simt(int dtype, const GemmDesc &d_in, cudaStream_t s) {
  if (d_in.M <= 0 || d_in.N <= 0) return cudaSuccess;
  GemmDesc d = d_in;
  if (d.part) {                 // partials mode: one split, the product itself
    d.y = d.part;
    d.ldy = d.N;
    d.epi = EPI_STORE;
  }
  dim3 g((d.N + SB_N - 1) / SB_N, (d.M + SB_M - 1) / SB_M);
  if (dtype) return launch_pdl(k_gemm_simt<bf16>, g, dim3(256), 0, s, d);
  return launch_pdl(k_gemm_simt<float>, g, dim3(256), 0, s, d);
}

}  // namespace dflash
