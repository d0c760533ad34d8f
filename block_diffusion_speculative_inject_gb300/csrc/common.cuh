// Shared device helpers and the internal launcher interface of libdflash.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

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

// Programmatic dependent launch: every kernel of the path is launched so that it may start
// while its predecessor drains. pdl_trigger lets the next kernel be scheduled; pdl_wait
// blocks until the predecessor grids have completed and their writes are visible. A kernel
// reads nothing its predecessors write, and writes nothing they read, before pdl_wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with the programmatic-stream-serialization attribute (and an optional cluster).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Device error codes latched into the mapped host flag (bit set).
enum : int { DEV_ERR_TOKEN = 1, DEV_ERR_BOUNDS = 2, DEV_ERR_TIMEOUT = 4 };

// The flag lives in mapped pinned host memory; a plain volatile store is enough (any
// nonzero value reports an error; the code bits are a hint). flag[1..3] hold the detail of
// an expired wait: the wait site, the CTA (x | y << 10 | z << 20) and the thread;
// flag[4..5] the progress of the CTA's other roles where the kernel tracks it.
__device__ __forceinline__ void raise_err(int *flag, int code) {
  if (flag) *(volatile int *)flag = code;
}
__device__ __forceinline__ void raise_wait_err(int *flag, int site, const volatile int *aux = nullptr) {
  if (!flag) return;
  volatile int *f = flag;
  if (f[1] == 0) {
    f[1] = site;
    f[2] = (int)(blockIdx.x | (blockIdx.y << 10) | (blockIdx.z << 20));
    f[3] = (int)threadIdx.x;
    f[4] = aux ? aux[0] : 0;
    f[5] = aux ? aux[1] : 0;
  }
  f[0] = DEV_ERR_TIMEOUT;
}
// wait sites reported in flag[1]
enum : int {
  SITE_GEMM_EMPTY = 0x101, SITE_GEMM_FULL = 0x102, SITE_GEMM_ACC = 0x103,
  SITE_GEMM_CFULL = 0x104, SITE_GEMM_CEMPTY = 0x105,
  SITE_ATT_EMPTY = 0x201, SITE_ATT_FULL = 0x202, SITE_ATT_PFULL = 0x203, SITE_ATT_SFULL = 0x204,
  SITE_ATT_PVDONE = 0x205, SITE_ATT_OFULL = 0x206, SITE_ATT_COMBINE = 0x207,
};

// ---------------------------------------------------------------- paged KV pool
// A page holds 64 positions of every layer: [L][K|V][nkv][block], one block per (layer,
// K or V, kv head) of 64 x hd values. K blocks are position-major [64][hd] (hd contiguous);
// V blocks are stored transposed, [hd][64] (positions contiguous), so that both attention
// products read their operands K-major.
constexpr int KV_PAGE = 64;
__host__ __device__ __forceinline__ size_t kv_block(int page, int l, int kv, int h, int L, int nkv,
                                                    int hd) {
  return ((((size_t)page * L + l) * 2 + kv) * nkv + h) * (size_t)(KV_PAGE * hd);
}

// ---------------------------------------------------------------- activation operands
// Activations are fp32. Where an activation is the X operand of a GEMM it is written as
// an "operand": fp32 for fp32 weights, or for bf16 weights an exact pair of bf16 planes
// hi = bf16(v), lo = bf16(v - hi), so a bf16 tensor-core product W.hi + W.lo carries the
// activation to ~2^-17 relative precision. The fused context feature g, whose K/V
// projection is rounded to the storage type when cached, takes a third plane
// lo2 = bf16(v - hi - lo) (~2^-25 relative): with two planes the cached values land on
// the other neighbour of their rounding often enough to move the logits by ~2e-3.
struct OpOut {
  void *hi;              // fp32 [rows, ld] when lo == nullptr, else bf16 [rows, ld]
  void *lo;              // bf16 [rows, ld] or nullptr
  void *lo2 = nullptr;   // bf16 [rows, ld] third plane, or nullptr
};

__device__ __forceinline__ void write_op(const OpOut &o, size_t idx, float v) {
  if (o.lo) {
    const bf16 h = __float2bfloat16_rn(v);
    const float r = v - __bfloat162float(h);           // exact in fp32
    const bf16 l = __float2bfloat16_rn(r);
    ((bf16 *)o.hi)[idx] = h;
    ((bf16 *)o.lo)[idx] = l;
    if (o.lo2) ((bf16 *)o.lo2)[idx] = __float2bfloat16_rn(r - __bfloat162float(l));
  } else {
    ((float *)o.hi)[idx] = v;
  }
}

// Four consecutive operand values (idx a multiple of 4): one 8-byte store per bf16 plane.
__device__ __forceinline__ void write_op4(const OpOut &o, size_t idx, float4 v) {
  if (!o.lo) {
    *(float4 *)((float *)o.hi + idx) = v;
    return;
  }
  const float a[4] = {v.x, v.y, v.z, v.w};
  uint16_t h[4], l[4], l2[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bf16 hb = __float2bfloat16_rn(a[j]);
    const float r = a[j] - __bfloat162float(hb);
    const bf16 lb = __float2bfloat16_rn(r);
    h[j] = __bfloat16_as_ushort(hb);
    l[j] = __bfloat16_as_ushort(lb);
    l2[j] = __bfloat16_as_ushort(__float2bfloat16_rn(r - __bfloat162float(lb)));
  }
  auto pack = [](const uint16_t (&q)[4]) {
    return make_uint2((uint32_t)q[0] | ((uint32_t)q[1] << 16), (uint32_t)q[2] | ((uint32_t)q[3] << 16));
  };
  *(uint2 *)((bf16 *)o.hi + idx) = pack(h);
  *(uint2 *)((bf16 *)o.lo + idx) = pack(l);
  if (o.lo2) *(uint2 *)((bf16 *)o.lo2 + idx) = pack(l2);
}

// ---------------------------------------------------------------- GEMM description
// Y[M, N] = epilogue( X[M, K] . W[N, K]^T ) with fp32 output. W has the storage type.
// X is fp32, bf16, or a bf16 hi/lo pair (x_lo non-null). X may be split along K into
// segments with separate base pointers (the fc fusion reads the n_feat feature tensors in
// place); W may be split along N into segments (the q/k/v weights, the per-layer k/v
// weights, gate/up) each [rows, K] row-major with row stride K.
enum GemmEpi : int {
  EPI_STORE = 0,   // Y = acc
  EPI_RESID = 1,   // Y = R + acc   (R may alias Y)
  EPI_TOPK = 2,    // per 128-row weight tile and token: the tile's top-k (value, index)
                   // into cand[tile][m][k]; Y = acc as well when y != nullptr
  EPI_QKV = 3,     // q/k/v projection (head_dim 128: one head per 128-row tile): q and k
                   // heads get their RMSNorm (if q_norm/k_norm) and RoPE at ctx_len[b] + j
  EPI_SWIGLU = 4,  // W = [gate; up] ([2I, K] as two segments of I rows): a tile holds 64 gate
                   // and the same 64 up rows; out = silu(gate) * up as an operand [M, I]
  EPI_RESNORM = 5, // residual add with the next RMSNorm left to the consumer: Y = Y + acc (in
                   // place; Y null: no residual, Y stands for acc), out = Y * norm_w as an operand, ss_part[tile][m] = the tile's sum
                   // of Y^2 for row m; the consuming GEMM scales its rows by
                   // rsqrt(sum_tiles ss_part / dim + eps) (rs_part below)
  EPI_KVCACHE = 6, // injection: W = [Wk_0; Wv_0; Wk_1; ...] (kv_dim rows each, head_dim 128: one
                   // head per tile); K heads get the layer's k-norm (if any) and RoPE at
                   // kv_pos[m], and K and V go to the paged cache at slot kv_slot[m] in the
                   // storage type
};

constexpr int GEMM_MAX_XSEG = 8;
constexpr int GEMM_MAX_WSEG = 16;

struct GemmDesc {
  int M, N, K;
  int x_bf16;                    // 1: X planes are bf16, 0: fp32
  int n_xseg;
  const void *x[GEMM_MAX_XSEG];
  const void *x_lo[GEMM_MAX_XSEG];   // lo plane (bf16 pair) or nullptr
  const void *x_lo2;             // third plane of segment 0 (with x_lo[0]) or nullptr
  int exact_acc;                 // 1: accumulate in short chunks summed in fp32 (round to nearest)
                                 // on the CUDA cores, for products that are rounded to the storage
                                 // type afterwards (the tensor core's own accumulation truncates)
  int x_k0[GEMM_MAX_XSEG + 1];   // K offset where segment s starts; x_k0[n_xseg] = K
  int ldx[GEMM_MAX_XSEG];        // row stride (elements) of each X segment
  int n_wseg;
  const void *w[GEMM_MAX_WSEG];
  int w_n0[GEMM_MAX_WSEG + 1];   // N offset where segment s starts; w_n0[n_wseg] = N
  int epi;
  float *y;                      // output [M, ldy] fp32
  int ldy;
  const float *resid;            // EPI_RESID input [M, ldy]
  int topk;                      // EPI_TOPK: k
  int2 *cand;                    // EPI_TOPK: [ceil(N/128)][M][k] (float bits, index)
  float *part;                   // partials mode: write the split-K partials [S][M][N] here
                                 // (S = 1: the plain product) instead of Y; a post-op sums them
  // EPI_QKV
  const int32_t *ctx_len;        // per request: position of its first query row
  const float2 *rope;            // [position][hd / 2] (cos, sin)
  const void *q_norm, *k_norm;   // bf16 [hd] or nullptr (no q/k norm)
  float eps;
  int rows_per_req;              // K + 1 query rows per request
  int q_dim, kv_dim;             // column ranges [0, q_dim) q, [q_dim, q_dim + kv_dim) k
  // EPI_SWIGLU
  OpOut out;                     // [M, ldo] operand planes
  int ldo;
  // EPI_TOPK: logits *= out_mult, then out_cap * tanh(logits / out_cap) when out_cap > 0,
  // applied before ranking (out_xf = 0: untouched)
  int out_xf;
  float out_mult, out_cap;
  float2 *lse_part;              // EPI_TOPK: [tiles][M] (max, sum exp) of each tile column, or null
  // EPI_RESNORM
  const void *norm_w;            // bf16 [N] RMSNorm weight
  float *ss_part;                // [N / 128][M]
  // any epilogue: X holds unnormalised rows x * w; row m of the product is first scaled by
  // rsqrt(sum_{t < rs_tiles} rs_part[t][m] / rs_dim + eps) (null: no scaling)
  const float *rs_part;
  int rs_tiles, rs_dim;
  int out_skip_k;                // EPI_RESNORM: K > 0 keeps only the K mask rows of each
                                 // (K+1)-row block (operand and sums at row b*K + j - 1)
  // EPI_KVCACHE (also uses rope, eps, kv_dim)
  const int32_t *kv_slot, *kv_pos;   // [M] cache slot (page * 64 + offset) and position
  void *kv_pool;                     // bf16 paged cache [pages][L][2][nkv][64][hd] (V as [hd][64])
  const void *kv_knorm[8];           // bf16 [hd] per layer, or null (no k-norm)
  int kv_L, kv_nkv;
};

__device__ __forceinline__ float logit_xform(float x, float mult, float cap) {
  x *= mult;
  return cap > 0.f ? cap * tanhf(x / cap) : x;
}

}  // namespace dflash
