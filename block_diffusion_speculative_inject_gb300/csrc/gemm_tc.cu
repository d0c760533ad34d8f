// Tensor-core GEMM on sm_103a: tcgen05.mma with the accumulator in TMEM, operands staged
// in shared memory by TMA (cp.async.bulk.tensor, 128-byte swizzle), an mbarrier pipeline.
//
//   Y[m, n] = sum_k X[m, k] * W[n, k]      (W: bf16 weights [N, K]; X: bf16 activations)
//
// The draft step multiplies few token rows (16 at batch 1) by large weight matrices, so
// the product is computed transposed ("swap AB"): a CTA owns 128 weight rows (the UMMA M
// dimension) and BN token rows (the UMMA N dimension, 16..128), and streams its weight
// slab through the pipeline once. When X is an exact bf16 hi/lo pair (an fp32 activation;
// hi/lo/lo2 for the injected context feature), every plane is multiplied by the same staged
// weight tile and accumulates into the same TMEM columns, so the weights are read from HBM
// once. Small grids are split along K
// (split-K, S <= 8) so every SM streams weights; the S CTAs of one output tile form a
// thread-block cluster, stage their fp32 partial tiles in their own shared memory, and each
// rank sums a share of the tile's columns over all ranks through distributed shared memory,
// in rank order, and applies the epilogue — no partials go through HBM and the sum order
// is fixed.
//
// Roles (192 threads): warp 0 lane 0 issues TMA loads, warp 1 owns the TMEM allocation and
// its lane 0 issues the MMAs, warps 2-5 (one per 32-lane TMEM quarter) run the epilogue.
// Every mbarrier wait is bounded in time; on expiry the kernel raises the device error
// flag, drains its own TMA loads and frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <cstdio>
#include <map>
#include <set>
#include <tuple>
#include <vector>

#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace dflash {

constexpr int TC_BM = 128;            // weight rows per tile (UMMA M)
constexpr int TC_BK = 64;             // K per pipeline stage: 64 bf16 = one 128-byte row
constexpr int TC_MAX_WSEG = 16;
constexpr int TC_MAX_XMAP = 8;
constexpr int TC_THREADS = 192;          // few-token instances: TMA warp, MMA warp, 4 epilogue warps
// Threads of an instance: the big-tile instances run one CTA per SM, so their epilogue gets
// 12 warps (three per TMEM lane quarter, splitting the columns) to hide its memory latencies
// (4 -> 8 -> 12 warps: q4b_b128 step 6.5 -> 5.5 -> 5.2 ms).
template <int BN>
constexpr int tc_threads() { return BN <= 32 ? TC_THREADS : 64 + 32 * 12; }

struct TcParams {
  CUtensorMap wmap[TC_MAX_WSEG];      // one per weight segment, box {64, 128}
  CUtensorMap xmap[TC_MAX_XMAP];      // X segments (box {64, BN}); planes > 1: [0] hi, [1] lo, [2] lo2
  int n_wseg;
  int w_n0[TC_MAX_WSEG + 1];
  int n_xseg;
  int x_k0[TC_MAX_XMAP + 1];
  int planes;                         // X planes: 1, or 2 / 3 for a split fp32 activation
  int chunk;                          // > 0: k-blocks per partial accumulator (folded in fp32)
  int M, N, K;
  int kb_total, kb_per, S;
  int n_tiles;                        // 128-row weight tiles of N
  int stages;
  int epi;
  float *y;
  int ldy;
  const float *resid;
  int topk;                           // EPI_TOPK
  int2 *cand;                         // EPI_TOPK: [n_tiles][M][topk]
  const int32_t *ctx_len;             // EPI_QKV
  const float2 *rope;
  const bf16 *q_norm, *k_norm;
  float eps;
  int rows_per_req, q_dim, kv_dim;
  OpOut out;                          // EPI_SWIGLU
  int ldo;
  int out_xf;                         // EPI_TOPK: logit scale / soft cap
  float out_mult, out_cap;
  float2 *lse_part;                   // EPI_TOPK: per (tile, token) (max, sum exp) or null
  const bf16 *norm_w;                 // EPI_RESNORM
  float *ss_part;
  const float *rs_part;               // row scales of an unnormalised X (or null)
  int rs_tiles, rs_dim;
  int out_skip_k;                     // EPI_RESNORM: operand rows for the K mask rows only
  const int32_t *kv_slot, *kv_pos;    // EPI_KVCACHE
  bf16 *kv_pool;
  const bf16 *kv_knorm[8];
  int kv_L, kv_nkv;
  int *err;
};
static_assert(sizeof(TcParams) <= 4096, "kernel parameters above 4 KB");



template <int BN>
constexpr int tmem_cols() {
  return BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
}

// One warp: the best k of a tile column held as 4 values per lane (value desc, lower index
// first), by k rounds of warp arg-max; lane 0 writes (value bits, index) pairs to out.
__device__ __forceinline__ void warp_tile_topk(float (&v)[4], int (&id)[4], int k, int lane, int2 *out) {
  for (int rr = 0; rr < k; ++rr) {
    float bv = v[0];
    int bi = id[0];
#pragma unroll
    for (int j = 1; j < 4; ++j)
      if (v[j] > bv || (v[j] == bv && id[j] < bi)) {
        bv = v[j];
        bi = id[j];
      }
    float wv = bv;
    int wi = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
      if (ov > wv || (ov == wv && oi < wi)) {
        wv = ov;
        wi = oi;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (id[j] == wi) {      // the winner leaves the race
        v[j] = -INFINITY;
        id[j] = 0x7fffffff;
      }
    if (lane == 0) out[rr] = make_int2(__float_as_int(wv), wi);
  }
}

// The same for T token columns at once (column t: v[t], id[t]); the T arg-max chains of a
// round are independent, so their shuffle latencies overlap. Columns with out[t] == nullptr
// are skipped.
template <int T>
__device__ __forceinline__ void warp_tile_topk_multi(float (&v)[T][4], int (&id)[T][4], int k, int lane,
                                                     int2 *const (&out)[T]) {
  for (int rr = 0; rr < k; ++rr) {
    float wv[T];
    int wi[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      wv[t] = v[t][0];
      wi[t] = id[t][0];
#pragma unroll
      for (int j = 1; j < 4; ++j)
        if (v[t][j] > wv[t] || (v[t][j] == wv[t] && id[t][j] < wi[t])) {
          wv[t] = v[t][j];
          wi[t] = id[t][j];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float ov = __shfl_xor_sync(0xffffffffu, wv[t], o);
        const int oi = __shfl_xor_sync(0xffffffffu, wi[t], o);
        if (ov > wv[t] || (ov == wv[t] && oi < wi[t])) {
          wv[t] = ov;
          wi[t] = oi;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (id[t][j] == wi[t]) {      // the winner leaves the race
          v[t][j] = -INFINITY;
          id[t][j] = 0x7fffffff;
        }
      if (lane == 0 && out[t]) out[t][rr] = make_int2(__float_as_int(wv[t]), wi[t]);
    }
  }
}

// Softmax normaliser partial of one tile column held as 4 values per lane (-inf outside the
// tile): (max, sum exp(v - max)), written by lane 0 to *out when out is non-null.
__device__ __forceinline__ void warp_tile_lse(const float (&v)[4], int lane, float2 *out) {
  float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
  mx = warp_max(mx);
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) s += v[j] == -INFINITY ? 0.f : expf(v[j] - mx);
  s = warp_sum(s);
  if (lane == 0 && out) *out = make_float2(mx, s);
}

// Staged partial tiles [tokens][128 weight rows] (fp32): the four rows a lane reduces and
// finishes (l, l + 32, l + 64, l + 96) are one 16-byte word, so the split-K reduction reads
// each rank's values with one 16-byte load per lane; within the word the rows are rotated by
// a lane-dependent XOR, which keeps the warp's staging stores free of bank conflicts.
__device__ __forceinline__ int stage_idx(int c, int n) {
  const int l = n & 31, q = n >> 5;
  return c * TC_BM + 4 * l + (q ^ ((l >> 3) & 3));
}
// element of the staged word of lane `lane` that holds row lane + 32 j
__device__ __forceinline__ float stage_pick(const float4 &v, int j, int lane) {
  const int e = j ^ ((lane >> 3) & 3);
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// ------------------------------------------------------------------------- the kernel
// FN: the fused-norm epilogue pieces (EPI_RESNORM, rs_part), compiled into the few-token
// instances only so that the others keep their code
// WM: 128-row weight tiles per CTA (1 or 2); with 2 the tiles share every staged activation
// tile, which halves the activation bytes read from L2 per weight byte (the big-M instance).
// CH: chunked (exact) accumulation, see below.
template <int BN, bool FN = false, int WM = 1, bool CH = false>
__global__ void __launch_bounds__(tc_threads<BN>(), BN <= 32 ? 3 : 1) k_gemm_tc(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_trigger();
  constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;          // one 128-row weight tile
  constexpr uint32_t B_BYTES = BN * TC_BK * 2;
  const uint32_t stage_bytes = WM * A_BYTES + B_BYTES * p.planes;
  const int stages = p.stages;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t tiles = (raw + 1023u) & ~1023u;           // 1024-byte aligned tile base
  uint8_t *gen_tiles = smem_raw + (tiles - raw);
  uint64_t *bars = (uint64_t *)(gen_tiles + (size_t)stages * stage_bytes);
  const uint32_t full0 = smem_u32(bars);                   // full[s]  = full0 + 8 s
  const uint32_t empty0 = full0 + 8u * stages;             // empty[s] = empty0 + 8 s
  const uint32_t accf = empty0 + 8u * stages;
  const uint32_t cfull0 = accf + 8u;                       // chunk buffer b written: cfull0 + 8 b
  const uint32_t cempty0 = accf + 24u;                     // chunk buffer b folded: cempty0 + 8 b
  uint32_t *tmem_slot = (uint32_t *)(bars + 2 * stages + 5);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BN, split = blockIdx.z;
  const int n0 = (int)blockIdx.y * WM * TC_BM;             // first weight row of weight tile 0
  const int wm_live = WM == 1 ? 1 : min(WM, p.n_tiles - (int)blockIdx.y * WM);   // weight tiles inside N
  // (the one-split top-k epilogue stages its own layout and scales by rs_lane)
  const bool staged = p.S > 1 || p.epi == EPI_QKV || p.epi == EPI_SWIGLU ||
                      (FN && (p.epi == EPI_RESNORM || p.epi == EPI_KVCACHE || (p.rs_part && p.epi != EPI_TOPK)));
  const int kb0 = split * p.kb_per;
  const int nkb = min(p.kb_total, kb0 + p.kb_per) - kb0;
  // Chunked accumulation: chunk c of `chunk` k-blocks accumulates from zero into TMEM buffer
  // c % 2 (columns [(c % 2) BNW, ...)), the epilogue warps add it into the sum region at 2 BNW
  // in fp32 and hand the buffer back; the epilogue then reads the sum instead of one long
  // tensor-core accumulation (whose additions truncate: ~2e-5 relative at K = 20480).
  constexpr int BNW = BN * WM;
  constexpr int NW = BN <= 32 ? 4 : 12;                     // epilogue warps
  const int CK = CH ? p.chunk : 1;                         // k-blocks per chunk
  const int n_chunks = CH ? (nkb + CK - 1) / CK : 0;
  constexpr uint32_t ncols = !CH ? (uint32_t)tmem_cols<BNW>()
                                 : 3 * BNW <= 64 ? 64 : 3 * BNW <= 128 ? 128 : 3 * BNW <= 256 ? 256 : 512;
  static_assert(!CH || 3 * BNW <= 512, "chunked accumulation needs three accumulator regions");

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(accf, 1);
    if (CH) {
      mbar_init(cfull0, 1);
      mbar_init(cfull0 + 8u, 1);
      mbar_init(cempty0, 32 * NW);
      mbar_init(cempty0 + 8u, 32 * NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (!(warp == 0 && lane == 0 && nkb > 0)) pdl_wait();   // the producer waits after its prefetch
  float2 qk_cs[4][2] = {};               // EPI_QKV epilogue warps: RoPE rows, loaded early

  if (warp == 0 && lane == 0 && nkb > 0) {
    // ---------------- TMA producer
    const bool glu = p.epi == EPI_SWIGLU;                  // rows 0-63 gate, 64-127 up
    const CUtensorMap *wm[WM];
    int wrow[WM];
    for (int w = 0; w < WM; ++w) {
      const int ty = (int)blockIdx.y * WM + w, n0w = ty * TC_BM;
      int ws = 0;
      while (ws + 1 < p.n_wseg && n0w >= p.w_n0[ws + 1]) ++ws;
      wm[w] = &p.wmap[glu ? 0 : ws];
      wrow[w] = glu ? ty * 64 : n0w - p.w_n0[ws];
    }
    const uint32_t tx = wm_live * A_BYTES + B_BYTES * p.planes;   // bytes landing per stage
    auto load_w = [&](uint32_t st, int k, uint32_t fb) {
      for (int w = 0; w < wm_live; ++w) {
        tma_load_2d(st + w * A_BYTES, wm[w], k, wrow[w], fb);
        if (glu) tma_load_2d(st + w * A_BYTES + 64 * 128, &p.wmap[1], k, wrow[w], fb);
      }
    };
    // the activation maps are first used after the dependency wait: fetch them now
    for (int w = 0; w < wm_live; ++w) tma_prefetch_map(wm[w]);
    if (glu) tma_prefetch_map(&p.wmap[1]);
    for (int i = 0; i < (p.planes > 1 ? p.planes : p.n_xseg); ++i) tma_prefetch_map(&p.xmap[i]);
    // the first stages' weight tiles do not depend on the previous kernel: start streaming
    // them before waiting for it
    const int pre = min(stages, nkb);
    for (int i = 0; i < pre; ++i) {
      const uint32_t fb = full0 + 8u * i;
      mbar_expect_tx(fb, tx);
      load_w(tiles + (uint32_t)i * stage_bytes, (kb0 + i) * TC_BK, fb);
    }
    pdl_wait();
    int issued = 0;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % stages, u = i / stages;
      const uint32_t st = tiles + (uint32_t)s * stage_bytes;
      const uint32_t fb = full0 + 8u * s;
      const int k = (kb0 + i) * TC_BK;
      if (i >= pre) {
        if (u > 0 && !mbar_wait(empty0 + 8u * s, (u - 1) & 1, abort_flag, p.err, SITE_GEMM_EMPTY)) break;
        mbar_expect_tx(fb, tx);
        load_w(st, k, fb);
      }
      const uint32_t xb = st + WM * A_BYTES;
      if (p.planes > 1) {
        for (int pl = 0; pl < p.planes; ++pl) tma_load_2d(xb + pl * B_BYTES, &p.xmap[pl], k, m0, fb);
      } else {
        int xs = 0;
        while (xs + 1 < p.n_xseg && k >= p.x_k0[xs + 1]) ++xs;
        tma_load_2d(xb, &p.xmap[xs], k - p.x_k0[xs], m0, fb);
      }
      issued = i + 1;
    }
    if (issued < pre) issued = pre;
    // drain: every load this thread issued has landed before the CTA may exit
    for (int s = 0; s < stages && s < issued; ++s) {
      const int last = s + stages * ((issued - 1 - s) / stages);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(full0 + 8u * s, (last / stages) & 1) && global_ns() - t0 < TC_WAIT_NS) {
      }
    }
  } else if (warp == 1 && lane == 0 && nkb > 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(TC_BM, BN);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % stages, u = i / stages;
      // chunked: k-block i goes to buffer (i / CH) % 2, which the epilogue must have folded
      // (chunk i / CH - 2) before the chunk's first MMA overwrites it
      const int ci = CH ? i / CK : 0;
      const bool first = CH ? i % CK == 0 : i == 0;
      if (CH && first && ci >= 2 &&
          !mbar_wait(cempty0 + 8u * (ci & 1), ((ci >> 1) - 1) & 1, abort_flag, p.err, SITE_GEMM_CEMPTY))
        break;
      if (!mbar_wait(full0 + 8u * s, u & 1, abort_flag, p.err, SITE_GEMM_FULL)) break;
      tc_fence_after();
      const uint32_t b = tiles + (uint32_t)s * stage_bytes + WM * A_BYTES;
      const uint32_t dbuf = tmem + (uint32_t)(CH ? (ci & 1) * BNW : 0);
      for (int w = 0; w < wm_live; ++w) {
        // weight tile w accumulates into TMEM columns [w BN, (w + 1) BN) of the buffer
        const uint32_t a = tiles + (uint32_t)s * stage_bytes + w * A_BYTES, d = dbuf + (uint32_t)(w * BN);
        if constexpr (CH) {
          // the small planes first: in the chunk's fresh accumulator only the hi plane's
          // additions truncate at the full magnitude of the sum
          for (int pl = p.planes - 1; pl >= 0; --pl) {
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk)
              umma_bf16(d, sw128_desc(a + kk * 32), sw128_desc(b + pl * B_BYTES + kk * 32), idesc,
                        (!first || kk > 0 || pl != p.planes - 1) ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            umma_bf16(d, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), idesc, (!first || kk > 0) ? 1u : 0u);
          for (int pl = 1; pl < p.planes; ++pl) {
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk)
              umma_bf16(d, sw128_desc(a + kk * 32), sw128_desc(b + pl * B_BYTES + kk * 32), idesc, 1u);
          }
        }
      }
      umma_commit(empty0 + 8u * s);       // frees the stage once these MMAs have read it
      if (CH && (i % CK == CK - 1 || i == nkb - 1)) umma_commit(cfull0 + 8u * (ci & 1));
    }
    umma_commit(accf);                    // accumulator complete (all MMAs issued above)
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> registers -> global
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int ew = warp - 2;              // epilogue warp 0..NW-1
    const int eh = ew >> 2;               // which of the quarter's NW / 4 warps (column share)
    if (p.epi == EPI_QKV && n0 < p.q_dim + p.kv_dim) {
      // RoPE (cos, sin) of the first tokens this warp finishes, fetched while the MMAs run
      const int rank = (int)cluster_ctarank();
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = rank + p.S * ew + NW * p.S * u, m = m0 + c;
        if (c < BN && m < p.M) {
          const int pos = __ldg(p.ctx_len + m / p.rows_per_req) + m % p.rows_per_req;
          qk_cs[u][0] = __ldg(p.rope + (size_t)pos * 64 + lane);
          qk_cs[u][1] = __ldg(p.rope + (size_t)pos * 64 + lane + 32);
        }
      }
    }
    // the unstaged top-k epilogue scales token column c by the row scale held by lane c
    float rs_lane = 1.f;
    if (FN && p.rs_part && p.epi == EPI_TOPK && m0 + lane < p.M) {
      float ss = 0.f;
      for (int t = 0; t < p.rs_tiles; ++t) ss += __ldg(p.rs_part + (size_t)t * p.M + m0 + lane);
      rs_lane = rsqrtf(ss / (float)p.rs_dim + p.eps);
    }
    bool ok = nkb > 0;
    if constexpr (!CH) {
      ok = ok && mbar_wait(accf, 0, abort_flag, p.err, SITE_GEMM_ACC);
      tc_fence_after();
    } else {
      // fold chunk c (buffer c % 2) into the sum region in fp32, then hand the buffer back
      const uint32_t lanes = (uint32_t)(q * 32) << 16;
      for (int c = 0; ok && c < n_chunks; ++c) {
        // warp-uniform, so that the aligned TMEM loads below run on every lane or none
        ok = __all_sync(0xffffffffu, mbar_wait(cfull0 + 8u * (c & 1), (c >> 1) & 1, abort_flag, p.err,
                                               SITE_GEMM_CFULL));
        tc_fence_after();
        if (ok) {
          const uint32_t part = tmem + lanes + (uint32_t)((c & 1) * BNW), sum = tmem + lanes + (uint32_t)(2 * BNW);
#pragma unroll 1
          for (int c0 = 16 * eh; c0 < BNW; c0 += 16 * (NW / 4)) {
            uint32_t r[16], t[16];
            tmem_ld16(part + c0, r);
            if (c > 0) tmem_ld16(sum + c0, t);
            tmem_ld_wait();
            if (c > 0) {
#pragma unroll
              for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(t[j]));
            }
            tmem_st16(sum + c0, r);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(cempty0 + 8u * (c & 1));
      }
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    // the accumulator the epilogue reads: the sum region when chunked
    const uint32_t tacc = tmem + (uint32_t)(CH ? 2 * BNW : 0);
    // the top-k epilogue stages the tile [BN tokens][128 rows] in the (now idle) stage memory;
    // the staged epilogues [WM][BN][128]
    float *tile = (float *)gen_tiles;
    constexpr int TP = TC_BM + 1;
#pragma unroll 1
    for (int cw = 16 * eh; cw < BN * wm_live; cw += 16 * (NW / 4)) {
      const int w = cw / BN, c0 = cw % BN;
      const int n = n0 + w * TC_BM + q * 32 + lane;
      uint32_t r[16];
      tmem_ld16(tacc + ((uint32_t)(q * 32) << 16) + (uint32_t)cw, r);
      tmem_ld_wait();
      if (p.epi == EPI_TOPK && p.S == 1) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = m0 + c0 + j;
          const bool valid = ok && n < p.N && m < p.M;
          float acc = __uint_as_float(r[j]);
          if (FN && p.rs_part) acc *= __shfl_sync(0xffffffffu, rs_lane, (c0 + j) & 31);
          const float v = p.out_xf ? logit_xform(acc, p.out_mult, p.out_cap) : acc;
          tile[(c0 + j) * TP + q * 32 + lane] = valid ? v : -INFINITY;
          if (valid && p.y) p.y[(size_t)m * p.ldy + n] = v;
        }
        continue;
      }
      if (staged) {
        // stage this CTA's (partial) tile [BN][128] for the split-K reduction and the
        // per-token epilogues
#pragma unroll
        for (int j = 0; j < 16; ++j) tile[stage_idx(cw + j, q * 32 + lane)] = ok ? __uint_as_float(r[j]) : 0.f;
        continue;
      }
      if (!ok || n >= p.N) continue;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = m0 + c0 + j;
        if (m >= p.M) break;
        const float v = __uint_as_float(r[j]);
        const size_t o = (size_t)m * p.ldy + n;
        p.y[o] = p.epi == EPI_RESID ? p.resid[o] + v : v;
      }
    }
    if (p.epi == EPI_TOPK && p.S == 1) {
      // per token: the tile's best topk (value desc, lower index first) by warp arg-max rounds
      asm volatile("bar.sync 1, %0;" ::"n"(32 * NW) : "memory");
      if constexpr (BN <= 32) {
        // this warp's token columns (c = ew + NW t), four at a time in interleaved passes
        constexpr int T = 4;
#pragma unroll 1
        for (int t0 = 0; NW * t0 < BN; t0 += T) {
          float v[T][4];
          int id[T][4];
          int2 *out[T];
#pragma unroll
          for (int t = 0; t < T; ++t) {
            const int c = ew + NW * (t0 + t), m = m0 + c;
            const bool live = ok && c < BN && m < p.M;
            out[t] = live ? p.cand + ((size_t)blockIdx.y * p.M + m) * p.topk : nullptr;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              v[t][j] = live ? tile[c * TP + lane + 32 * j] : -INFINITY;
              id[t][j] = n0 + lane + 32 * j;
            }
          }
          if (p.lse_part) {
#pragma unroll
            for (int t = 0; t < T; ++t) {
              const int c = ew + NW * (t0 + t), m = m0 + c;
              warp_tile_lse(v[t], lane, out[t] ? p.lse_part + (size_t)blockIdx.y * p.M + m : nullptr);
            }
          }
          warp_tile_topk_multi<T>(v, id, p.topk, lane, out);
        }
      } else {
        for (int c = ew; c < BN; c += NW) {
          const int m = m0 + c;
          if (m >= p.M || !ok) continue;
          float v[4];
          int id[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[j] = tile[c * TP + lane + 32 * j];
            id[j] = n0 + lane + 32 * j;
          }
          if (p.lse_part) warp_tile_lse(v, lane, p.lse_part + (size_t)blockIdx.y * p.M + m);
          warp_tile_topk(v, id, p.topk, lane, p.cand + ((size_t)blockIdx.y * p.M + m) * p.topk);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (staged) {
    // every split's partial tile is staged; rank r owns columns (tokens) r, r + S, ...: each
    // epilogue warp takes one of them at a time, sums its 128 rows over all ranks in rank
    // order (lane l: rows l, l + 32, l + 64, l + 96) and applies the epilogue
    constexpr int U = BN <= 32 ? 2 : 4;        // tokens per warp per round: loads in flight
    const int rank = (int)cluster_ctarank();
    const int ew = warp - 2;
    // The epilogue's inputs that do not depend on the accumulator (the residual / stream
    // rows, the RMSNorm sums of the row scale) for this warp's first round, loaded before
    // the cluster barrier so that their latency overlaps the wait for the slowest split.
    float pre_y[U][4], pre_ss[U];
    if (warp >= 2) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = rank + p.S * ew + NW * p.S * u, m = m0 + c;
        pre_ss[u] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) pre_y[u][j] = 0.f;
        if (c >= BN || m >= p.M) continue;
        if (FN && p.rs_part)
          for (int t = lane; t < p.rs_tiles; t += 32) pre_ss[u] += __ldg(p.rs_part + (size_t)t * p.M + m);
        const float *src = (FN && p.epi == EPI_RESNORM) ? p.y : p.epi == EPI_RESID ? p.resid : nullptr;
        if (src) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int n = n0 + lane + 32 * j;
            if (n < p.N) pre_y[u][j] = src[(size_t)m * p.ldy + n];
          }
        }
      }
    }
    if (p.S > 1) cluster_sync_all();
    if (warp >= 2) {
     for (int w = 0; w < wm_live; ++w) {
      // weight tile w: rows n0w.. of the output, staged at [w][BN][128]
      const int ty = (int)blockIdx.y * WM + w, n0w = ty * TC_BM;
      const uint32_t base = smem_u32(gen_tiles) + (uint32_t)(w * BN * TC_BM * 4);
      const float *own = (const float *)gen_tiles + (size_t)w * BN * TC_BM;
      const int part = n0w < p.q_dim ? 0 : (n0w < p.q_dim + p.kv_dim ? 1 : 2);   // EPI_QKV
      for (int cb = rank + p.S * ew; cb < BN; cb += NW * U * p.S) {
        const bool pre = w == 0 && cb == rank + p.S * ew;   // this round's inputs are loaded
        float a[U][4];
        float2 cs[U][2];
        int mu[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = cb + NW * p.S * u;
          mu[u] = (c < BN && m0 + c < p.M) ? m0 + c : -1;
          if (mu[u] < 0) continue;
          if (p.S == 1) {
            const float4 t = *(const float4 *)(own + c * TC_BM + 4 * lane);
#pragma unroll
            for (int j = 0; j < 4; ++j) a[u][j] = stage_pick(t, j, lane);
          } else {
            // every rank's partial of these four rows, summed in rank order
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const uint32_t src = base + (uint32_t)((c * TC_BM + 4 * lane) * 4);
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) {
              if (rk < p.S) {
                const float4 t = dsmem_ld4(dsmem_addr(src, (uint32_t)rk));
                acc.x += t.x;
                acc.y += t.y;
                acc.z += t.z;
                acc.w += t.w;
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) a[u][j] = stage_pick(acc, j, lane);
          }
          if (p.epi == EPI_QKV && part < 2) {
            if (w == 0 && cb == rank + p.S * ew) {
              cs[u][0] = qk_cs[u][0];
              cs[u][1] = qk_cs[u][1];
            } else {
              const int m = mu[u];
              const int pos = __ldg(p.ctx_len + m / p.rows_per_req) + m % p.rows_per_req;
              cs[u][0] = __ldg(p.rope + (size_t)pos * 64 + lane);
              cs[u][1] = __ldg(p.rope + (size_t)pos * 64 + lane + 32);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int m = mu[u];
          if (m < 0) continue;
          float *x = a[u];
          if (FN && p.rs_part) {
            // the producer left the RMSNorm's row scale: lane t holds tile t's sum of squares
            float ss = pre ? pre_ss[u] : 0.f;
            if (!pre)
              for (int t = lane; t < p.rs_tiles; t += 32) ss += __ldg(p.rs_part + (size_t)t * p.M + m);
            const float rs = rsqrtf(warp_sum(ss) / (float)p.rs_dim + p.eps);
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] *= rs;
          }
          if (FN && p.epi == EPI_KVCACHE) {
            // this tile is one head: K (norm + RoPE) or V of layer l, into the paged cache
            const int seg = n0w / p.kv_dim, l = seg >> 1, h = (n0w % p.kv_dim) >> 7;
            const int slot = __ldg(p.kv_slot + m), page = slot / KV_PAGE, off = slot % KV_PAGE;
            if ((seg & 1) == 0) {
              const bf16 *kn = p.kv_knorm[l];
              if (kn) {
                const float rk =
                    rsqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]) / 128.f + p.eps);
#pragma unroll
                for (int j = 0; j < 4; ++j) x[j] = x[j] * rk * __bfloat162float(kn[lane + 32 * j]);
              }
              const int pos = __ldg(p.kv_pos + m);
              const float2 c0 = __ldg(p.rope + (size_t)pos * 64 + lane), c1 = __ldg(p.rope + (size_t)pos * 64 + lane + 32);
              const float o0 = x[0] * c0.x - x[2] * c0.y, o2 = x[2] * c0.x + x[0] * c0.y;
              const float o1 = x[1] * c1.x - x[3] * c1.y, o3 = x[3] * c1.x + x[1] * c1.y;
              bf16 *dk = p.kv_pool + kv_block(page, l, 0, h, p.kv_L, p.kv_nkv, 128) + (size_t)off * 128;
              dk[lane] = __float2bfloat16_rn(o0);
              dk[lane + 32] = __float2bfloat16_rn(o1);
              dk[lane + 64] = __float2bfloat16_rn(o2);
              dk[lane + 96] = __float2bfloat16_rn(o3);
            } else {
              bf16 *dv = p.kv_pool + kv_block(page, l, 1, h, p.kv_L, p.kv_nkv, 128) + off;
#pragma unroll
              for (int j = 0; j < 4; ++j) dv[(size_t)(lane + 32 * j) * KV_PAGE] = __float2bfloat16_rn(x[j]);
            }
            continue;
          }
          if (FN && p.epi == EPI_RESNORM) {
            // out_skip_k = K: only the K mask rows of each (K+1)-row block go on, to row
            // b*K + j - 1 of the operand and of the sums (the final norm before the LM head)
            int orow = m, ldss = p.M;
            if (p.out_skip_k > 0) {
              const int Q = p.out_skip_k + 1, jj = m % Q;
              if (jj == 0) continue;
              orow = (m / Q) * p.out_skip_k + jj - 1;
              ldss = p.M / Q * p.out_skip_k;
            }
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int n = n0w + lane + 32 * j;
              const size_t o = (size_t)m * p.ldy + n;
              const float y = p.y ? (pre ? pre_y[u][j] : p.y[o]) + x[j] : x[j];   // no residual: the norm alone
              if (p.y) p.y[o] = y;
              write_op(p.out, (size_t)orow * p.ldo + n, y * __bfloat162float(p.norm_w[n]));
              ss += y * y;
            }
            ss = warp_sum(ss);
            if (lane == 0) p.ss_part[(size_t)ty * ldss + orow] = ss;
            continue;
          }
          if (p.epi == EPI_TOPK) {
            // split-K LM head: the reduced column's best topk of this tile
            float v[4];
            int id[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int n = n0w + lane + 32 * j;
              if (p.out_xf) x[j] = logit_xform(x[j], p.out_mult, p.out_cap);
              v[j] = n < p.N ? x[j] : -INFINITY;
              id[j] = n;
              if (n < p.N && p.y) p.y[(size_t)m * p.ldy + n] = x[j];
            }
            if (p.lse_part) warp_tile_lse(v, lane, p.lse_part + (size_t)ty * p.M + m);
            warp_tile_topk(v, id, p.topk, lane, p.cand + ((size_t)ty * p.M + m) * p.topk);
            continue;
          }
          if (p.epi == EPI_SWIGLU) {
            // rows lane, lane + 32 are gate; lane + 64, lane + 96 the matching up rows
            const size_t o = (size_t)m * p.ldo + (size_t)ty * 64 + lane;
            write_op(p.out, o, x[0] / (1.f + expf(-x[0])) * x[2]);
            write_op(p.out, o + 32, x[1] / (1.f + expf(-x[1])) * x[3]);
            continue;
          }
          if (p.epi == EPI_QKV && part < 2) {
            // one head of 128: RMSNorm (if weights), then RoPE on (l, l + 64), (l + 32, l + 96)
            const bf16 *nw = part == 0 ? p.q_norm : p.k_norm;
            if (nw) {
              const float rs =
                  rsqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]) / 128.f + p.eps);
#pragma unroll
              for (int j = 0; j < 4; ++j) x[j] = x[j] * rs * __bfloat162float(nw[lane + 32 * j]);
            }
            const float2 c0 = cs[u][0], c1 = cs[u][1];
            const float o0 = x[0] * c0.x - x[2] * c0.y, o2 = x[2] * c0.x + x[0] * c0.y;
            const float o1 = x[1] * c1.x - x[3] * c1.y, o3 = x[3] * c1.x + x[1] * c1.y;
            x[0] = o0;
            x[1] = o1;
            x[2] = o2;
            x[3] = o3;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int n = n0w + lane + 32 * j;
            if (n < p.N) {
              const size_t o = (size_t)m * p.ldy + n;
              p.y[o] = p.epi == EPI_RESID ? (pre ? pre_y[u][j] : p.resid[o]) + x[j] : x[j];
            }
          }
        }
      }
     }
    }
    // peers keep their shared memory until all have read it; this barrier orders nothing
    // else, so its arrive is relaxed (the epilogue's global stores need not drain first)
    if (p.S > 1) cluster_sync_relaxed();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ------------------------------------------------------------------------- host side
struct TcGemm {
  int device = 0, num_sms = 0;
  int *err = nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  std::map<std::tuple<const void *, long, long, long, int>, CUtensorMap> maps;
  int generation = 0;
  bool attr_set[16] = {};
  bool wide = true;                   // two weight tiles per CTA for big M (DFLASH_GEMM_WM1=1: one)
  std::map<std::tuple<const void *, int, long>, int> occ;   // cluster occupancy per instance
  bool debug_plan = false;            // DFLASH_DEBUG_PLAN=1: print each new GEMM plan to stderr
  double ovh = -1;                    // big-tile split-K model: per-CTA cost override (k-blocks)
  std::set<std::tuple<const void *, int, long>> printed;
};

cudaError_t tc_gemm_create(TcGemm **out, int device, int num_sms, int *err_flag) {
  *out = nullptr;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
  TcGemm *t = new TcGemm();
  t->device = device;
  t->num_sms = num_sms;
  t->encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  t->err = err_flag;
  const char *wm1 = getenv("DFLASH_GEMM_WM1");
  t->wide = !(wm1 && wm1[0] == '1');
  if (const char *o = getenv("DFLASH_GEMM_OVH")) t->ovh = atof(o);
  const char *dbg = getenv("DFLASH_DEBUG_PLAN");
  t->debug_plan = dbg && dbg[0] == '1';
  *out = t;
  return cudaSuccess;
}

void tc_gemm_destroy(TcGemm *t) {
  if (!t) return;
  delete t;
}

// bf16 2-D tensor map over a row-major [rows, cols] matrix with row stride ld (elements),
// box {64, box_rows}, 128-byte swizzle, zero fill out of bounds.
static bool get_map(TcGemm *t, const void *ptr, long rows, long cols, long ld, int box_rows,
                    CUtensorMap *out) {
  auto key = std::make_tuple(ptr, rows, cols, ld, box_rows);
  auto it = t->maps.find(key);
  if (it != t->maps.end()) {
    *out = it->second;
    return true;
  }
  CUtensorMap m;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = t->encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (t->maps.size() > 4096) t->maps.clear();
  t->maps.emplace(key, m);
  *out = m;
  return true;
}

bool tc_encode_2d(TcGemm *t, const void *ptr, unsigned long long rows, unsigned long long cols,
                  unsigned long long ld, unsigned box_cols, unsigned box_rows, void *map_out) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = t->encode((CUtensorMap *)map_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void *>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Plan {
  int bn, wm, t_tiles, n_tiles, grid_y, kb, kb_per, S, stages;
  size_t smem;
};

// Few-token instances (FN: the fused-norm / cache-write epilogues) or the wide big-M
// instance (two weight tiles per CTA) — the kernel instance a GEMM launches with.
static bool fn_instance(const GemmDesc &d) { return d.rs_part || d.epi == EPI_RESNORM || d.epi == EPI_KVCACHE; }

static Plan plan_for(const TcGemm *t, const GemmDesc &d) {
  Plan p{};
  p.bn = d.M <= 16 ? 16 : d.M <= 32 ? 32 : d.M <= 64 ? 64 : 128;
  p.t_tiles = (d.M + p.bn - 1) / p.bn;
  p.n_tiles = (d.N + TC_BM - 1) / TC_BM;
  p.kb = d.K / TC_BK;
  // more token rows than one tile: two weight tiles per CTA share the staged activations
  // (the activation planes are the larger part of a stage at 128 tokens)
  const bool wide = t->wide && p.bn == 128 && !fn_instance(d) && p.n_tiles >= 2 && !d.exact_acc &&
                    (d.epi == EPI_STORE || d.epi == EPI_RESID || d.epi == EPI_QKV || d.epi == EPI_SWIGLU);
  p.wm = wide ? 2 : 1;
  p.grid_y = (p.n_tiles + p.wm - 1) / p.wm;
  const int planes = 1 + (d.x_lo[0] ? 1 : 0) + (d.x_lo2 ? 1 : 0);
  const size_t stage = (size_t)p.wm * TC_BM * TC_BK * 2 + (size_t)p.bn * TC_BK * 2 * planes;
  // Few token rows: a short pipeline and many resident CTAs per SM stream weights fastest
  // (measured); more token rows: a longer pipeline in a CTA of its own.
  if (p.bn <= 32)
    p.stages = 3;
  else if (p.wm == 1)
    p.stages = (int)std::max<size_t>(2, std::min<size_t>(8, (200 * 1024) / stage));
  else
    p.stages = (int)std::max<size_t>(2, std::min<size_t>(4, (220 * 1024) / stage));
  p.smem = p.stages * stage + 1024 + 8 * (2 * p.stages + 5) + 16;
  p.S = 1;
  p.kb_per = p.kb;
  return p;
}

// Split-K factor of the few-token instances: as many parts as keep the grid within one wave
// of resident CTAs (more CTAs in flight streamed faster than balancing the bytes per SM,
// measured).
static int splits_few(const TcGemm *t, const Plan &p) {
  const int per_sm = std::max(1, std::min(4, (int)((228 * 1024) / (p.smem + 1024))));
  const int base = p.t_tiles * p.grid_y;
  const int s_max = std::max(1, std::min(8, p.kb / 4));    // a portable cluster holds 8 CTAs
  return std::max(1, std::min((per_sm * t->num_sms) / base, s_max));
}

// Split-K factor of the big-M instances: the CTAs of a launch run in waves of as many
// clusters as fit on the GPU at once (the driver's cluster occupancy for this instance and
// shared-memory size), so the launch takes about waves x (k-blocks per split + a fixed
// per-CTA cost); splitting K evens out a last wave that would run nearly empty (e.g. 160
// tiles on 152 SMs).
static int splits_wide(TcGemm *t, const void *fn, int threads, const Plan &p) {
  const int tiles = p.t_tiles * p.grid_y;
  const int s_max = std::max(1, std::min(8, p.kb / 8));
  // fixed cost of a CTA, in k-blocks of its pipeline (DFLASH_GEMM_OVH: tuning override)
  const double ovh = t->ovh >= 0 ? t->ovh : p.wm == 2 ? 5.0 : 8.0;
  int best_S = 1;
  double best = 0;
  for (int S = 1; S <= s_max; ++S) {
    auto key = std::make_tuple(fn, S, (long)p.smem);
    auto it = t->occ.find(key);
    int occ;
    if (it != t->occ.end()) {
      occ = it->second;
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, 1, S);
      cfg.blockDim = dim3(threads);
      cfg.dynamicSmemBytes = p.smem;
      cudaLaunchAttribute a;
      a.id = cudaLaunchAttributeClusterDimension;
      a.val.clusterDim.x = 1;
      a.val.clusterDim.y = 1;
      a.val.clusterDim.z = S;
      cfg.attrs = &a;
      cfg.numAttrs = 1;
      occ = 0;
      if (cudaOccupancyMaxActiveClusters(&occ, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        occ = 0;
      }
      t->occ.emplace(key, occ);
    }
    if (occ <= 0) continue;
    const int kb_per = (p.kb + S - 1) / S;
    const double cost = (double)((tiles + occ - 1) / occ) * (kb_per + ovh);
    if (S == 1 || cost < 0.97 * best) {
      best = cost;
      best_S = S;
    }
  }
  return best_S;
}

int tc_gemm_generation(const TcGemm *t) { return t ? t->generation : 0; }

int tc_gemm_splits(const TcGemm *, const GemmDesc &) { return 1; }   // reduced in-cluster

int tc_gemm_launches(const TcGemm *, const GemmDesc &) { return 1; }

template <int BN, bool FN = false, int WM = 1, bool CH = false>
static cudaError_t launch_bn(TcGemm *t, int slot, TcParams &p, Plan pl, cudaStream_t s) {
  const void *fn = (const void *)k_gemm_tc<BN, FN, WM, CH>;
  if (!t->attr_set[slot]) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<BN, FN, WM, CH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    t->attr_set[slot] = true;
  }
  const int S = BN <= 32 ? splits_few(t, pl) : splits_wide(t, fn, tc_threads<BN>(), pl);
  pl.kb_per = (pl.kb + S - 1) / S;
  pl.S = (pl.kb + pl.kb_per - 1) / pl.kb_per;    // every split non-empty
  p.kb_per = pl.kb_per;
  p.S = pl.S;
  if (t->debug_plan) {
    auto key = std::make_tuple((const void *)nullptr, p.M * 131071 + p.N, (long)p.K * 16 + p.epi);
    if (t->printed.insert(key).second)
      fprintf(stderr, "[dflash gemm] M %d N %d K %d epi %d planes %d chunk %d: BN %d WM %d grid %d x %d x %d stages %d smem %zu\n",
              p.M, p.N, p.K, p.epi, p.planes, p.chunk, BN, WM, pl.t_tiles, pl.grid_y, pl.S, pl.stages, pl.smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.t_tiles, pl.grid_y, pl.S);
  cfg.blockDim = dim3(tc_threads<BN>());
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = pl.S;      // the S splits of one output tile
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_gemm_tc<BN, FN, WM, CH>, p);
}

cudaError_t tc_gemm_run(TcGemm *t, const GemmDesc &d, cudaStream_t s) {
  if (d.M <= 0 || d.N <= 0) return cudaSuccess;
  if (d.epi == EPI_TOPK && (d.topk < 1 || d.topk > 32 || !d.cand)) return cudaErrorInvalidValue;
  if (!d.x_bf16 || d.K % TC_BK || d.n_wseg > TC_MAX_WSEG || d.n_xseg > TC_MAX_XMAP ||
      (d.x_lo[0] && d.n_xseg != 1) || (d.x_lo2 && !d.x_lo[0]))
    return cudaErrorInvalidValue;
  const Plan pl = plan_for(t, d);
  TcParams p;   // kernel parameters (copied at launch)
  memset(&p, 0, sizeof(p));
  if (d.epi == EPI_SWIGLU &&
      (d.n_wseg != 2 || d.w_n0[1] * 2 != d.N || d.w_n0[1] % 64 || d.part || !d.out.lo))
    return cudaErrorInvalidValue;
  if (d.epi == EPI_QKV && (d.q_dim % TC_BM || d.kv_dim % TC_BM || !d.ctx_len || !d.rope || d.part ||
                           d.rows_per_req < 1))
    return cudaErrorInvalidValue;
  if (d.epi == EPI_RESNORM && (d.N % TC_BM || !d.out.lo || !d.norm_w || !d.ss_part || d.part))
    return cudaErrorInvalidValue;
  if (d.rs_part && (d.rs_tiles < 1 || d.rs_dim < 1)) return cudaErrorInvalidValue;
  if (d.epi == EPI_RESNORM && d.out_skip_k > 0 && d.M % (d.out_skip_k + 1)) return cudaErrorInvalidValue;
  if (d.epi == EPI_KVCACHE && (d.kv_dim % TC_BM || d.kv_L < 1 || d.kv_L > 8 || d.kv_nkv * TC_BM != d.kv_dim ||
                               d.N != d.kv_L * 2 * d.kv_dim || !d.kv_slot || !d.kv_pos || !d.kv_pool || !d.rope ||
                               d.part))
    return cudaErrorInvalidValue;
  p.n_wseg = d.n_wseg;
  for (int i = 0; i < d.n_wseg; ++i) {
    const long rows = d.w_n0[i + 1] - d.w_n0[i];
    const int box = d.epi == EPI_SWIGLU ? 64 : TC_BM;        // gate/up: half tiles of each
    if (!get_map(t, d.w[i], rows, d.K, d.K, box, &p.wmap[i])) return cudaErrorInvalidValue;
    p.w_n0[i] = d.w_n0[i];
  }
  p.w_n0[d.n_wseg] = d.w_n0[d.n_wseg];
  p.planes = 1 + (d.x_lo[0] ? 1 : 0) + (d.x_lo2 ? 1 : 0);
  p.n_xseg = d.n_xseg;
  if (p.planes > 1) {
    if (!get_map(t, d.x[0], d.M, d.K, d.ldx[0], pl.bn, &p.xmap[0]) ||
        !get_map(t, d.x_lo[0], d.M, d.K, d.ldx[0], pl.bn, &p.xmap[1]) ||
        (d.x_lo2 && !get_map(t, d.x_lo2, d.M, d.K, d.ldx[0], pl.bn, &p.xmap[2])))
      return cudaErrorInvalidValue;
    p.x_k0[0] = 0;
    p.x_k0[1] = d.K;
  } else {
    for (int i = 0; i < d.n_xseg; ++i) {
      const long cols = d.x_k0[i + 1] - d.x_k0[i];
      if (cols % TC_BK) return cudaErrorInvalidValue;
      if (!get_map(t, d.x[i], d.M, cols, d.ldx[i], pl.bn, &p.xmap[i])) return cudaErrorInvalidValue;
      p.x_k0[i] = d.x_k0[i];
    }
    p.x_k0[d.n_xseg] = d.x_k0[d.n_xseg];
  }
  p.M = d.M;
  p.N = d.N;
  p.K = d.K;
  p.kb_total = pl.kb;
  p.n_tiles = pl.n_tiles;
  p.chunk = d.exact_acc ? 1 : 0;       // one k-block (64 products) per partial accumulator
  p.stages = pl.stages;
  p.epi = d.epi;
  p.topk = d.topk;
  p.cand = d.cand;
  p.y = d.y;
  p.ldy = d.ldy;
  p.resid = d.resid;
  p.ctx_len = d.ctx_len;
  p.rope = d.rope;
  p.q_norm = (const bf16 *)d.q_norm;
  p.k_norm = (const bf16 *)d.k_norm;
  p.eps = d.eps;
  p.rows_per_req = d.rows_per_req;
  p.q_dim = d.q_dim;
  p.kv_dim = d.kv_dim;
  p.out = d.out;
  p.ldo = d.ldo;
  p.out_xf = d.out_xf;
  p.lse_part = d.lse_part;
  p.norm_w = (const bf16 *)d.norm_w;
  p.ss_part = d.ss_part;
  p.rs_part = d.rs_part;
  p.rs_tiles = d.rs_tiles;
  p.rs_dim = d.rs_dim;
  p.out_skip_k = d.out_skip_k;
  p.kv_slot = d.kv_slot;
  p.kv_pos = d.kv_pos;
  p.kv_pool = (bf16 *)d.kv_pool;
  for (int l = 0; l < 8; ++l) p.kv_knorm[l] = (const bf16 *)d.kv_knorm[l];
  p.kv_L = d.kv_L;
  p.kv_nkv = d.kv_nkv;
  p.out_mult = d.out_mult;
  p.out_cap = d.out_cap;
  p.err = t->err;
  if (d.part) {
    // partials mode: the (already reduced) product goes to the caller's buffer [M][N]
    p.y = d.part;
    p.ldy = d.N;
    p.epi = EPI_STORE;
  }
  cudaError_t e;
  if (fn_instance(d)) {
    if (pl.bn > 32) return cudaErrorInvalidValue;      // few-token instances only
    if (p.chunk)
      return pl.bn == 16 ? launch_bn<16, true, 1, true>(t, 7, p, pl, s) : launch_bn<32, true, 1, true>(t, 8, p, pl, s);
    return pl.bn == 16 ? launch_bn<16, true>(t, 4, p, pl, s) : launch_bn<32, true>(t, 5, p, pl, s);
  }
  if (p.chunk) {
    // exact accumulation of the injection GEMMs (one weight tile per CTA)
    switch (pl.bn) {
      case 16: return launch_bn<16, false, 1, true>(t, 9, p, pl, s);
      case 32: return launch_bn<32, false, 1, true>(t, 10, p, pl, s);
      case 64: return launch_bn<64, false, 1, true>(t, 11, p, pl, s);
      default: return launch_bn<128, false, 1, true>(t, 12, p, pl, s);
    }
  }
  switch (pl.bn) {
    case 16: e = launch_bn<16>(t, 0, p, pl, s); break;
    case 32: e = launch_bn<32>(t, 1, p, pl, s); break;
    case 64: e = launch_bn<64>(t, 2, p, pl, s); break;
    default: e = pl.wm == 2 ? launch_bn<128, false, 2>(t, 6, p, pl, s) : launch_bn<128>(t, 3, p, pl, s); break;
  }
  return e;
}

}  // namespace dflash
