// Split-KV attention of the query block over the paged context on the tensor cores.
//
// One CTA = (split s, kv head, request b). Its rows are the G query heads of the kv head
// times the K+1 block rows (R = G (K+1) <= 128, padded to the UMMA M of 128); its keys are
// the context positions of split s, two 64-position pages per tile (a split's last tile may
// hold one; its second page is then the first again, masked). Per tile:
//   S[128 rows, 128 keys] = Q . K_tile^T          (tcgen05, A = Q in TMEM, B = K pages in smem)
//   P = 2^(S - m)         (two threads per row: max, exp2, row sum; P written over S in TMEM)
//   O[128 rows, 128 hd]  += P . V_tile            (tcgen05, A = P in TMEM, B = V pages [hd][64])
// (128-key tiles: N = 128 MMAs run at the full tensor rate, N = 64 ones at ~70%, measured.)
// Q (fp32) and P (fp32) enter the tensor core as exact bf16 hi/lo pairs, so each product
// is two MMAs against the same staged K or V tile; the cache K/V are exact bf16 already.
// With both A operands in tensor memory the MMAs read only the K/V pages from shared
// memory, and shared memory holds nothing but a 3-stage K/V ring (64 KB per stage).
// Scores are in log2 units (log2(e)/sqrt(hd) folded into Q). The running max is updated
// lazily: O in TMEM is rescaled only when a row's max grows by more than 8 (2^8 headroom).
// The result per row is the unnormalised O, the max and the row sum, merged by the combine
// kernel with the other splits and the block's own keys.
//
// TMEM (512 columns): S/P buffers at 0 and 128 (tile parity), O at 256, Q hi at 384, Q lo
// at 448. A P buffer holds, for the 64 keys owned by each half of a row, 32 columns of hi
// words then 32 of lo words, inside the S columns of those same keys.
//
// Roles (320 threads): warp 0 lane 0 issues TMA (per page, K: two boxes of 64 x 64, V: one
// box of 64 x 128); warp 1 owns TMEM and its lane 0 issues the MMAs; warps 2-9 fill Q, run
// the softmax and write the partials. A row is shared by warps w and w + 4 (TMEM lane
// quarter w % 4): each owns 64 of the tile's 128 keys and 64 of O's 128 columns, and the
// pair exchanges its row maxima through shared memory once per tile. The S of the next
// tile is computed while the softmax of the current one runs; the softmax waits for the
// previous tile's P.V only when it rescales O. All waits are bounded in time.
#include "kernels.h"
#include "tc_ptx.cuh"

namespace dflash {

constexpr int AT_TC_THREADS = 320;
constexpr int AT_TC_STAGES = 3;
constexpr int AT_KT = 128;                        // keys per tile (two pages)
constexpr uint32_t AK_SUB = 64 * 128;             // [64 keys x 64 hd] bf16: one page, one hd half
constexpr uint32_t AK_HALF = 2 * AK_SUB;          // [128 keys x 64 hd]: both pages, one hd half
constexpr uint32_t AK_BYTES = 2 * AK_HALF;
constexpr uint32_t AV_PAGE = 128 * 128;           // [128 hd x 64 keys] bf16: one page
constexpr uint32_t AV_BYTES = 2 * AV_PAGE;
constexpr uint32_t A_STAGE = AK_BYTES + AV_BYTES;
constexpr uint32_t AX_BYTES = (4 * 128 + 2 * 128 + 16 + 2) * 4;   // row-max, row-sum, status, progress
constexpr size_t AT_TC_SMEM = 1024 + AT_TC_STAGES * A_STAGE + 256 + AX_BYTES;
constexpr uint32_t AT_TMEM_COLS = 512;
constexpr uint32_t AT_TMEM_O = 256;               // O accumulator
constexpr uint32_t AT_TMEM_Q = 384;               // Q hi (64 columns), then Q lo

struct AttnTcParams {
  CUtensorMap kmap, vmap;
  const float *qkv;
  const int32_t *ctx_len, *n_split, *split_len, *page_off, *pages;
  int L, nq, nkv, Q, layer, max_split;
  float scale_log2;
  float *part_o, *part_ml;
  int *err;
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// barrier of the two softmax warps that share a TMEM lane quarter (ids 1..4, 64 threads)
__device__ __forceinline__ void bar_pair(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi); two values per 32-bit word (a in the
// low half), each pair rounded by one paired conversion
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

__global__ void __launch_bounds__(AT_TC_THREADS, 1) k_attn_split_tc(const __grid_constant__ AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_trigger();
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int ns = p.n_split[b];                           // descriptor: staged before the chain
  if (s >= ns) {                                         // uniform for the CTA
    pdl_wait();        // this grid must not complete before its predecessor has
    return;
  }
  const int n_ctx = p.ctx_len[b];
  const int k_begin = s * p.split_len[b];
  const int k_end = min(k_begin + p.split_len[b], n_ctx);
  const int n_tiles = (k_end - k_begin + AT_KT - 1) / AT_KT;
  const int G = p.nq / p.nkv, R = G * p.Q;
  const int32_t *pg = p.pages + p.page_off[b];

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t st0 = base;
  uint64_t *bars = (uint64_t *)(gbase + AT_TC_STAGES * A_STAGE);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * AT_TC_STAGES;
  // Per tile parity b: S ready (s_full0 + 8 b) and P written (p_full0 + 8 b). P has its own
  // pair: the softmax may write P of tile i + 1 before the issuer has seen P of tile i.
  const uint32_t s_full0 = empty0 + 8u * AT_TC_STAGES;
  const uint32_t p_full0 = s_full0 + 16u;
  const uint32_t pv_done = p_full0 + 16u;                  // P.V of a tile retired
  const uint32_t o_full = pv_done + 8u;                    // all P.V retired
  uint32_t *tmem_slot = (uint32_t *)(bars + 2 * AT_TC_STAGES + 6);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
  // exchange between the two warps of a row: maxima [parity][half][row], sums [half][row],
  // status [parity][half][quarter]
  float *xmax = (float *)(gbase + AT_TC_STAGES * A_STAGE + 256);
  float *xsum = xmax + 4 * 128;
  volatile int *xok = (volatile int *)(xsum + 2 * 128);
  // progress of the MMA issuer and of softmax warp 2, reported if the producer's wait expires
  volatile int *prog = xok + 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < AT_TC_STAGES; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, 1);
    }
    mbar_init(s_full0, 1);
    mbar_init(s_full0 + 8u, 1);
    mbar_init(p_full0, 8);
    mbar_init(p_full0 + 8u, 8);
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
    *abort_flag = 0;
    prog[0] = prog[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), AT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer. The pages were written by earlier kernels of the stream
    // (context injection), which a programmatic launch does not order before this point.
    tma_prefetch_map(&p.kmap);
    tma_prefetch_map(&p.vmap);
    pdl_wait();
    int issued = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int stg = i % AT_TC_STAGES, u = i / AT_TC_STAGES;
      if (u > 0 && !mbar_wait(empty0 + 8u * stg, (u - 1) & 1, abort_flag, p.err, SITE_ATT_EMPTY, prog)) break;
      const int pos = k_begin + AT_KT * i;
      const uint32_t st = st0 + (uint32_t)stg * A_STAGE;
      const uint32_t fb = full0 + 8u * stg;
      mbar_expect_tx(fb, A_STAGE);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        // page x of the tile; a missing second page repeats the first (finite data, masked)
        const int page = pg[(pos + (pos + 64 * x < k_end ? 64 * x : 0)) / 64];
        const int blk = (page * p.L + p.layer) * 2 * p.nkv;
        const int krow = (blk + kvh) * 64;             // K view: rows of 128 values
        const int vrow = (blk + p.nkv + kvh) * 128;    // V view: rows of 64 values
        tma_load_2d(st + x * AK_SUB, &p.kmap, 0, krow, fb);
        tma_load_2d(st + AK_HALF + x * AK_SUB, &p.kmap, 64, krow, fb);
        tma_load_2d(st + AK_BYTES + x * AV_PAGE, &p.vmap, 0, vrow, fb);
      }
      issued = i + 1;
    }
    for (int i = 0; i < AT_TC_STAGES && i < issued; ++i) {
      const int last = i + AT_TC_STAGES * ((issued - 1 - i) / AT_TC_STAGES);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(full0 + 8u * i, (last / AT_TC_STAGES) & 1) &&
             global_ns() - t0 < TC_WAIT_NS) {
      }
    }
  } else if (warp == 1) {
    // Q rows are written to TMEM by the softmax warps after the previous kernel finished
    __syncwarp();
    pdl_wait();
    asm volatile("bar.sync 5, 288;" ::: "memory");   // warps 1-9: Q is in TMEM
    tc_fence_after();
    if (lane == 0) {
      prog[0] = 1;
      // ---------------- MMA issuer: S of tile i+1 is computed while the softmax of tile i
      // runs, then P.V of tile i
      constexpr uint32_t idS = idesc_bf16(128, AT_KT);
      constexpr uint32_t idO = idesc_bf16(128, 128);
      auto issue_s = [&](int i) {
        const int stg = i % AT_TC_STAGES, u = i / AT_TC_STAGES;
        if (!mbar_wait(full0 + 8u * stg, u & 1, abort_flag, p.err, SITE_ATT_FULL)) return false;
        tc_fence_after();
        const uint32_t kst = st0 + (uint32_t)stg * A_STAGE;
        const uint32_t dS = tmem + (uint32_t)((i & 1) * AT_KT);
#pragma unroll
        for (int pl = 0; pl < 2; ++pl)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)           // hd in steps of 16: 8 TMEM columns of Q
            umma_bf16_ts(dS, tmem + AT_TMEM_Q + 64 * pl + 8 * kk,
                         sw128_desc(kst + (kk >> 2) * AK_HALF + (kk & 3) * 32), idS, (pl | kk) ? 1u : 0u);
        umma_commit(s_full0 + 8u * (i & 1));
        return true;
      };
      bool go = n_tiles > 0 && issue_s(0);
      for (int i = 0; go && i < n_tiles; ++i) {
        prog[0] = 16 + 4 * i;
        if (i + 1 < n_tiles && !issue_s(i + 1)) break;
        prog[0] = 16 + 4 * i + 1;
        if (!mbar_wait(p_full0 + 8u * (i & 1), (i >> 1) & 1, abort_flag, p.err, SITE_ATT_PFULL)) break;
        prog[0] = 16 + 4 * i + 2;
        tc_fence_after();
        const int stg = i % AT_TC_STAGES;
        const uint32_t vst = st0 + (uint32_t)stg * A_STAGE + AK_BYTES;
        const uint32_t pbuf = tmem + (uint32_t)((i & 1) * AT_KT);
#pragma unroll
        for (int pl = 0; pl < 2; ++pl)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)           // keys in steps of 16 (kk >> 2: the page)
            umma_bf16_ts(tmem + AT_TMEM_O, pbuf + 64 * (kk >> 2) + 32 * pl + 8 * (kk & 3),
                         sw128_desc(vst + (kk >> 2) * AV_PAGE + (kk & 3) * 32), idO, (i | kk | pl) ? 1u : 0u);
        umma_commit(empty0 + 8u * stg);      // K and V of this tile are no longer read
        umma_commit(pv_done);
      }
      umma_commit(o_full);
    }
  } else if (warp >= 2) {
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    if (warp == 2 && lane == 0) prog[1] = 1;
    pdl_wait();                                        // q comes from the previous kernel
    if (warp == 2 && lane == 0) prog[1] = 2;
    {
      // Q row r, dims [64 half, 64 half + 64): scaled, split into hi/lo words in TMEM
      const int qkv_dim = (p.nq + 2 * p.nkv) * 128;
      const float *src = nullptr;
      if (r < R) {
        const int g = r / p.Q, j = r % p.Q;
        src = p.qkv + ((size_t)b * p.Q + j) * qkv_dim + (size_t)(kvh * G + g) * 128 + 64 * half;
      }
      float4 raw4[16];                                 // the half row in one round trip
#pragma unroll
      for (int i = 0; i < 16; ++i) raw4[i] = src ? *(const float4 *)(src + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t hw[16], lw[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 a = raw4[8 * c + i];
          split2(a.x * p.scale_log2, a.y * p.scale_log2, hw[2 * i], lw[2 * i]);
          split2(a.z * p.scale_log2, a.w * p.scale_log2, hw[2 * i + 1], lw[2 * i + 1]);
        }
        tmem_st16(lane_base + AT_TMEM_Q + 32 * half + 16 * c, hw);
        tmem_st16(lane_base + AT_TMEM_Q + 64 + 32 * half + 16 * c, lw);
      }
      tmem_st_wait();
      tc_fence_before();
    }
    asm volatile("bar.sync 5, 288;" ::: "memory");   // warps 1-9: Q is in TMEM
    if (warp == 2 && lane == 0) prog[1] = 3;

    // ---------------- softmax: warps w and w + 4 share the rows of lane quarter w % 4
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int par = i & 1;
      if (warp == 2 && lane == 0) prog[1] = 16 + 8 * i;
      // the pair runs the same number of exchanges: a failed wait is passed to the partner
      // through the status word and both leave the loop together
      const bool got = __all_sync(0xffffffffu, ok && mbar_wait(s_full0 + 8u * par, (i >> 1) & 1, abort_flag, p.err, SITE_ATT_SFULL));
      const uint32_t sa = lane_base + (uint32_t)(par * AT_KT + half * 64);   // my 64 keys
      float sc[64];
      float mt = -INFINITY;
      if (got) {
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t t0[16], t1[16];
          tmem_ld16(sa + c0, t0);
          tmem_ld16(sa + c0 + 16, t1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            sc[c0 + j] = __uint_as_float(t0[j]);
            sc[c0 + 16 + j] = __uint_as_float(t1[j]);
          }
        }
        const int nvalid = min(AT_KT, k_end - (k_begin + AT_KT * i)) - 64 * half;
        if (nvalid < 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c) sc[c] = c < nvalid ? sc[c] : -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < 64; ++c) mt = fmaxf(mt, sc[c]);
      }
      xmax[(par * 2 + half) * 128 + r] = mt;
      if (lane == 0) xok[(par * 2 + half) * 4 + q] = got ? 1 : 0;
      bar_pair(1 + q);
      const float mp = xmax[(par * 2 + (half ^ 1)) * 128 + r];
      ok = got && xok[(par * 2 + (half ^ 1)) * 4 + q] != 0;
      if (!ok) break;
      if (warp == 2 && lane == 0) prog[1] = 16 + 8 * i + 1;
      mt = fmaxf(mt, mp);
      // lazy max: rescale only when a row's max grows by more than 8 (the pair decides alike)
      if (i == 0) {
        m_used = mt;
      } else if (__any_sync(0xffffffffu, mt > m_used + 8.f)) {
        const float m_new = fmaxf(m_used, mt);
        const float corr = ex2_approx(m_used - m_new);
        m_used = m_new;
        // P.V of the previous tile must have retired before O is rescaled (the tile before
        // it has: its completion preceded this tile's S)
        if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (i - 1) & 1, abort_flag, p.err, SITE_ATT_PVDONE))) {
          ok = false;                      // the partner learns of it at the next exchange
          continue;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t t[16];
          tmem_ld16(lane_base + AT_TMEM_O + 64 * half + c0, t);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) t[j] = __float_as_uint(__uint_as_float(t[j]) * corr);
          tmem_st16(lane_base + AT_TMEM_O + 64 * half + c0, t);
        }
        l *= corr;
      }
      // P over this thread's own S columns: 32 words of hi pairs, then 32 of lo pairs
#pragma unroll
      for (int c0 = 0; c0 < 32; c0 += 16) {
        uint32_t ph[16], pw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float e0 = ex2_approx(sc[2 * (c0 + c)] - m_used), e1 = ex2_approx(sc[2 * (c0 + c) + 1] - m_used);
          l += e0 + e1;
          split2(e0, e1, ph[c], pw[c]);
        }
        tmem_st16(sa + c0, ph);
        tmem_st16(sa + 32 + c0, pw);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full0 + 8u * par);
      if (warp == 2 && lane == 0) prog[1] = 16 + 8 * i + 3;
    }
    // row sum over both halves (one more exchange, run by both warps of the pair)
    xsum[half * 128 + r] = l;
    bar_pair(1 + q);
    const float l_row = l + xsum[(half ^ 1) * 128 + r];
    ok = __all_sync(0xffffffffu, ok && mbar_wait(o_full, 0, abort_flag, p.err, SITE_ATT_OFULL));
    tc_fence_after();
    const int g = r / p.Q, j = r % p.Q;
    const size_t idx = (((size_t)b * p.Q + j) * p.nq + (kvh * G + g)) * p.max_split + s;
    if (r < R && half == 0) {
      p.part_ml[idx * 2] = ok ? m_used : -INFINITY;
      p.part_ml[idx * 2 + 1] = ok ? l_row : 0.f;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t t[16];
      tmem_ld16(lane_base + AT_TMEM_O + 64 * half + c0, t);
      tmem_ld_wait();
      if (r < R) {
        float4 *dst = (float4 *)(p.part_o + idx * 128 + 64 * half + c0);
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
