// Split-KV attention of the query block over the paged context on the tensor cores.
//
// One CTA = (split s, kv head, request b). Its rows are the G query heads of the kv head
// times the K+1 block rows (R = G (K+1) <= 128, padded to the UMMA M of 128); its keys are
// the context positions of split s, one 64-position page per tile. Per tile:
//   S[128 rows, 64 keys]  = Q . K_tile^T          (tcgen05, A = Q in smem, B = K page)
//   P = 2^(S - m)         (one thread per row: max, exp2, row sum; P written to smem)
//   O[128 rows, 128 hd]  += P . V_tile            (tcgen05, A = P, B = V page stored [hd][64])
// Q (fp32) and P (fp32) enter the tensor core as exact bf16 hi/lo pairs, so each product
// is two MMAs against the same staged K or V tile; the cache K/V are exact bf16 already.
// Scores are in log2 units (log2(e)/sqrt(hd) folded into Q). The running max is updated
// lazily: O in TMEM is rescaled only when a row's max grows by more than 8 (2^8 headroom).
// The result per row is the unnormalised O, the max and the row sum, merged by the combine
// kernel with the other splits and the block's own keys.
//
// Roles (192 threads): warp 0 lane 0 issues TMA (K page: two boxes of 64 x 64, V page: one
// box of 64 x 128) into a 3-stage ring; warp 1 owns TMEM (S at columns 0 and 64, O at 128)
// and its lane 0 issues the MMAs; warps 2-5 fill Q, run the softmax (TMEM lane quarter
// warp % 4) and write the partials. The S of the next tile is computed into a second TMEM
// buffer while the softmax of the current one runs. All waits are bounded in time.
#include "kernels.h"
#include "tc_ptx.cuh"

namespace dflash {

constexpr int AT_TC_THREADS = 192;
constexpr int AT_TC_STAGES = 3;
constexpr uint32_t AQ_SUB = 128 * 128;            // [128 rows x 64 hd] bf16
constexpr uint32_t AQ_BYTES = 4 * AQ_SUB;         // [hi, lo] x [hd 0..63, 64..127]
constexpr uint32_t AP_SUB = 128 * 128;            // [128 rows x 64 keys] bf16
constexpr uint32_t AP_BYTES = 2 * AP_SUB;         // hi, lo
constexpr uint32_t AK_SUB = 64 * 128;             // [64 keys x 64 hd] bf16
constexpr uint32_t AK_BYTES = 2 * AK_SUB;
constexpr uint32_t AV_BYTES = 128 * 128;          // [128 hd x 64 keys] bf16
constexpr uint32_t A_STAGE = AK_BYTES + AV_BYTES;
constexpr size_t AT_TC_SMEM = 1024 + AQ_BYTES + AP_BYTES + AT_TC_STAGES * A_STAGE + 256;
constexpr uint32_t AT_TMEM_COLS = 256;
constexpr uint32_t AT_TMEM_O = 128;               // O accumulator column offset

struct AttnTcParams {
  CUtensorMap kmap, vmap;
  const float *qkv;
  const int32_t *ctx_len, *n_split, *split_len, *page_off, *pages;
  int L, nq, nkv, Q, layer, max_split;
  float scale_log2;
  float *part_o, *part_ml;
  int *err;
};

// byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled tile of 128-byte rows
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void split8(const float (&v)[8], uint4 &hi, uint4 &lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bf16 h0 = __float2bfloat16_rn(v[2 * i]), h1 = __float2bfloat16_rn(v[2 * i + 1]);
    const bf16 l0 = __float2bfloat16_rn(v[2 * i] - __bfloat162float(h0));
    const bf16 l1 = __float2bfloat16_rn(v[2 * i + 1] - __bfloat162float(h1));
    h[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
    l[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(AT_TC_THREADS, 1) k_attn_split_tc(const __grid_constant__ AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_trigger();
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int ns = p.n_split[b];                           // descriptor: staged before the chain
  if (s >= ns) return;                                   // uniform for the CTA
  const int n_ctx = p.ctx_len[b];
  const int k_begin = s * p.split_len[b];
  const int k_end = min(k_begin + p.split_len[b], n_ctx);
  const int n_tiles = (k_end - k_begin + 63) / 64;
  const int G = p.nq / p.nkv, R = G * p.Q;
  const int32_t *pg = p.pages + p.page_off[b];

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t qs = base, ps = base + AQ_BYTES, st0 = ps + AP_BYTES;
  uint64_t *bars = (uint64_t *)(gbase + AQ_BYTES + AP_BYTES + AT_TC_STAGES * A_STAGE);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * AT_TC_STAGES;
  const uint32_t s_full0 = empty0 + 8u * AT_TC_STAGES;   // S buffer b ready: s_full0 + 8 b
  const uint32_t p_full = s_full0 + 16u;                   // P of the current tile written
  const uint32_t pv_done = p_full + 8u;                    // P.V of a tile retired
  const uint32_t o_full = pv_done + 8u;                    // all P.V retired
  uint32_t *tmem_slot = (uint32_t *)(bars + 2 * AT_TC_STAGES + 5);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < AT_TC_STAGES; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, 1);
    }
    mbar_init(s_full0, 1);
    mbar_init(s_full0 + 8u, 1);
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), AT_TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();                                            // q comes from the previous kernel
  if (warp >= 2) {
    // Q rows (scaled, split into hi/lo) in the 128-byte-swizzled K-major layout
    const int r = threadIdx.x - 64;
    const int qkv_dim = (p.nq + 2 * p.nkv) * 128;
    const float *src = nullptr;
    if (r < R) {
      const int g = r / p.Q, j = r % p.Q;
      src = p.qkv + ((size_t)b * p.Q + j) * qkv_dim + (size_t)(kvh * G + g) * 128;
    }
    float4 raw[32];                                  // the whole row in one round trip
#pragma unroll
    for (int i = 0; i < 32; ++i) raw[i] = src ? *(const float4 *)(src + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float4 a = raw[2 * c], d = raw[2 * c + 1];
      float v[8] = {a.x, a.y, a.z, a.w, d.x, d.y, d.z, d.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] *= p.scale_log2;
      uint4 hi, lo;
      split8(v, hi, lo);
      const int half = c >> 3, cc = c & 7;
      *(uint4 *)(gbase + (0 * 2 + half) * AQ_SUB + sw128_off(r, cc)) = hi;
      *(uint4 *)(gbase + (1 * 2 + half) * AQ_SUB + sw128_off(r, cc)) = lo;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int issued = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int stg = i % AT_TC_STAGES, u = i / AT_TC_STAGES;
      if (u > 0 && !mbar_wait(empty0 + 8u * stg, (u - 1) & 1, abort_flag, p.err)) break;
      const int page = pg[(k_begin + 64 * i) / 64];
      const int blk = (page * p.L + p.layer) * 2 * p.nkv;
      const int krow = (blk + kvh) * 64;               // K view: rows of 128 values
      const int vrow = (blk + p.nkv + kvh) * 128;      // V view: rows of 64 values
      const uint32_t st = st0 + (uint32_t)stg * A_STAGE;
      const uint32_t fb = full0 + 8u * stg;
      mbar_expect_tx(fb, A_STAGE);
      tma_load_2d(st, &p.kmap, 0, krow, fb);
      tma_load_2d(st + AK_SUB, &p.kmap, 64, krow, fb);
      tma_load_2d(st + AK_BYTES, &p.vmap, 0, vrow, fb);
      issued = i + 1;
    }
    for (int i = 0; i < AT_TC_STAGES && i < issued; ++i) {
      const int last = i + AT_TC_STAGES * ((issued - 1 - i) / AT_TC_STAGES);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(full0 + 8u * i, (last / AT_TC_STAGES) & 1) &&
             global_ns() - t0 < TC_WAIT_NS) {
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: S of tile i+1 is computed while the softmax of tile i
    // runs (two S buffers in TMEM), then P.V of tile i
    constexpr uint32_t idS = idesc_bf16(128, 64);
    constexpr uint32_t idO = idesc_bf16(128, 128);
    auto issue_s = [&](int i) {
      const int stg = i % AT_TC_STAGES, u = i / AT_TC_STAGES;
      if (!mbar_wait(full0 + 8u * stg, u & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      const uint32_t kst = st0 + (uint32_t)stg * A_STAGE;
      const uint32_t dS = tmem + (uint32_t)((i & 1) * 64);
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int pl = 0; pl < 2; ++pl)
            umma_bf16(dS, sw128_desc(qs + (pl * 2 + half) * AQ_SUB + kk * 32),
                      sw128_desc(kst + half * AK_SUB + kk * 32), idS, (half | kk | pl) ? 1u : 0u);
      umma_commit(s_full0 + 8u * (i & 1));
      return true;
    };
    bool go = n_tiles > 0 && issue_s(0);
    for (int i = 0; go && i < n_tiles; ++i) {
      if (i + 1 < n_tiles && !issue_s(i + 1)) break;
      if (!mbar_wait(p_full, i & 1, abort_flag, p.err)) break;
      tc_fence_after();
      const int stg = i % AT_TC_STAGES;
      const uint32_t vst = st0 + (uint32_t)stg * A_STAGE + AK_BYTES;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int pl = 0; pl < 2; ++pl)
          umma_bf16(tmem + AT_TMEM_O, sw128_desc(ps + pl * AP_SUB + kk * 32),
                    sw128_desc(vst + kk * 32), idO, (i | kk | pl) ? 1u : 0u);
      umma_commit(empty0 + 8u * stg);      // K and V of this tile are no longer read
      umma_commit(pv_done);
    }
    umma_commit(o_full);
  } else if (warp >= 2) {
    // ---------------- softmax, one thread per row (TMEM lane)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < n_tiles && ok; ++i) {
      ok = __all_sync(0xffffffffu, mbar_wait(s_full0 + 8u * (i & 1), (i >> 1) & 1, abort_flag, p.err));
      tc_fence_after();
      const int nvalid = min(64, k_end - (k_begin + 64 * i));
      float sc[64];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) {
        uint32_t t[16];
        tmem_ld16(lane_base + (uint32_t)((i & 1) * 64) + c0, t);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) sc[c0 + j] = c0 + j < nvalid ? __uint_as_float(t[j]) : -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) mt = fmaxf(mt, sc[c]);
      if (i > 0) {
        // P.V of the previous tile must have retired: O is stable and the P buffer is free
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (i - 1) & 1, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
      }
      if (i == 0) {
        m_used = mt;
      } else if (__any_sync(0xffffffffu, mt > m_used + 8.f)) {
        const float m_new = fmaxf(m_used, mt);
        const float corr = exp2f(m_used - m_new);
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 16) {
          uint32_t t[16];
          tmem_ld16(lane_base + AT_TMEM_O + c0, t);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) t[j] = __float_as_uint(__uint_as_float(t[j]) * corr);
          tmem_st16(lane_base + AT_TMEM_O + c0, t);
        }
        tmem_st_wait();
        l *= corr;
        m_used = m_new;
      }
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        sc[c] = exp2f(sc[c] - m_used);
        rs += sc[c];
      }
      l += rs;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = sc[8 * cc + j];
        uint4 hi, lo;
        split8(v, hi, lo);
        *(uint4 *)(gbase + AQ_BYTES + sw128_off(r, cc)) = hi;
        *(uint4 *)(gbase + AQ_BYTES + AP_SUB + sw128_off(r, cc)) = lo;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    ok = __all_sync(0xffffffffu, ok && mbar_wait(o_full, 0, abort_flag, p.err));
    tc_fence_after();
    if (r < R) {
      const int g = r / p.Q, j = r % p.Q;
      const size_t idx = (((size_t)b * p.Q + j) * p.nq + (kvh * G + g)) * p.max_split + s;
      p.part_ml[idx * 2] = ok ? m_used : -INFINITY;
      p.part_ml[idx * 2 + 1] = ok ? l : 0.f;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 16) {
      uint32_t t[16];
      tmem_ld16(lane_base + AT_TMEM_O + c0, t);
      tmem_ld_wait();
      if (r < R) {
        const int g = r / p.Q, j = r % p.Q;
        const size_t idx = (((size_t)b * p.Q + j) * p.nq + (kvh * G + g)) * p.max_split + s;
        float4 *dst = (float4 *)(p.part_o + idx * 128 + c0);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4)
          dst[j4] = ok ? make_float4(__uint_as_float(t[4 * j4]), __uint_as_float(t[4 * j4 + 1]),
                                     __uint_as_float(t[4 * j4 + 2]), __uint_as_float(t[4 * j4 + 3]))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, AT_TMEM_COLS);
  }
}

cudaError_t launch_attn_split_tc(const ModelDims &m, const DraftBatch &bt, int layer,
                                 const float *qkv, const AttnMaps *maps, float scale_log2,
                                 float *part_o, float *part_ml, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_split_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)AT_TC_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  AttnTcParams p;
  memset(&p, 0, sizeof(p));
  p.kmap = maps->k;
  p.vmap = maps->v;
  p.qkv = qkv;
  p.ctx_len = bt.ctx_len;
  p.n_split = bt.n_split;
  p.split_len = bt.split_len;
  p.page_off = bt.page_off;
  p.pages = bt.pages;
  p.L = m.L;
  p.nq = m.nq;
  p.nkv = m.nkv;
  p.Q = m.Q();
  p.layer = layer;
  p.max_split = bt.max_split;
  p.scale_log2 = scale_log2;
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.err = maps->err;
  dim3 g(bt.max_split, m.nkv, bt.B);
  return launch_pdl(k_attn_split_tc, g, dim3(AT_TC_THREADS), AT_TC_SMEM, s, p);
}

}  // namespace dflash
